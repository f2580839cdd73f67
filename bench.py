"""Benchmark of the Mamba-2 chunked SSD forward pass on GB300.

One step = one mamba2_ssd_fwd over one batch of the long-sequence workload
(batch 4, L 8192, 64 heads x headdim 64, state 128, 1 group, chunk 256, bf16,
carried fp32 initial state), i.e. every stage of the path: chunk cumsum, state
pass, chunk output.  Inputs are seeded synthetic tensors already resident in
HBM; a 256 MiB buffer is written between timed steps so each step starts with
a cold L2.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Under torchrun (N > 1) every rank runs an independent replica of the workload
(the path has no exchange step), the step time is the max over ranks and the
value is the tokens of all ranks over that time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Mamba-2 SSD fwd tokens/s and TFLOP/s at 1 GB300; % of tensor/HBM roofline"
DEFAULT_WORKLOAD = "long_seq_carried_state"
FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end loop")
    p.add_argument("--soak-s", type=float, default=1.0,
                   help="seconds of untimed steps run under the clock sampler before the timed region")
    p.add_argument("--no-decode", action="store_true", help="skip the decode-step measurement")
    p.add_argument("--cpu-pairs", type=int, default=256,
                   help="(batch, head) pairs the oracle runs for the CPU baseline sample")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the extra workloads (the other configurations and the sweep)")
    p.add_argument("--extra-steps", type=int, default=10, help="timed steps per extra workload")
    return p.parse_args()


# ----------------------------------------------------------------- ranks
def max_over_ranks(value, device="cuda"):
    """The largest `value` over all ranks of the default process group (the
    job's time is its slowest rank's); `value` itself with one process.  The
    only collective of the benchmark: the replicas exchange no data."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms_per_step):
    """Whole-job throughput: the tokens all ranks processed in one step over
    the step time of the slowest rank."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


# --------------------------------------------------------------------- work
def work_counts(w):
    """Algorithmic FLOPs and bytes of one forward pass.

    FLOPs count the causal half of every T x T product and C B^T once per
    group: N [G (T+1) S + nh (T+1) H + 4 nh S H].  Compulsory bytes: x read,
    y written, B, C, dt read, final state written, initial state read."""
    N = w.batch * w.seqlen
    e = 2 if w.dtype == "bf16" else 4
    T, S, H, nh, G = w.chunk_size, w.dstate, w.headdim, w.nheads, w.ngroups
    flop = N * (G * (T + 1) * S + nh * (T + 1) * H + 4 * nh * S * H)
    flop_dense = N * (2 * G * T * S + 2 * nh * T * H + 4 * nh * S * H)
    state = 4 * w.batch * nh * S * H
    bytes_min = N * (2 * nh * H * e + 2 * G * S * e + 4 * nh) + state * (2 if w.init_state else 1)
    return flop, flop_dense, bytes_min


def kernel_bytes(w):
    """Algorithmic bytes of one launch of each stage kernel (what it must read
    and write once): cumsum reads dt (and A) and writes G; the state pass reads
    x, dt, B, G (and the initial state) and writes every chunk state and the
    final state; the output kernel reads x, dt, G, B, C, D and the chunk states
    and writes y."""
    N = w.batch * w.seqlen
    e = 2 if w.dtype == "bf16" else 4
    S, H, nh, G = w.dstate, w.headdim, w.nheads, w.ngroups
    xb = N * nh * H * e
    bcb = N * G * S * e
    dtb = gb = 4 * N * nh
    state = 4 * w.batch * nh * S * H
    csb = w.batch * nh * w.nchunks * S * H * e
    return {
        "chunk_cumsum": dtb + gb + 4 * nh,
        "state_pass": xb + dtb + bcb + gb + csb + state * (2 if w.init_state else 1),
        "chunk_out": xb + dtb + gb + 2 * bcb + csb + xb + 4 * nh,
    }


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def load_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary of
    this workload, or None when there is none or the kernel's source has
    changed since the counters were taken (the summary records its hash)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"ncu_{kernel}_{workload}.md")
    try:
        fields = {}
        for line in open(path):
            if ":" in line and not line.startswith((" ", "|", "#")):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        src = os.path.join(ROOT, fields["source"])
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if sha != fields["source_sha256_16"]:
            return None
        return float(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


def load_ncu_dram(kernel, workload):
    """(duration in us, DRAM throughput in % of peak) of `kernel` from the
    committed ncu summary of this workload, or None when there is none or the
    kernel's source has changed since it was captured."""
    if load_traffic(kernel, workload) is None:
        return None
    path = os.path.join(ROOT, "profiles", f"ncu_{kernel}_{workload}.md")
    dur = pct = None
    try:
        for line in open(path):
            if line.startswith("|") and "`gpu__time_duration.sum`" in line:
                dur = float(line.split("|")[2])
            if line.startswith("|") and "`gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed`" in line:
                pct = float(line.split("|")[2])
    except Exception:
        return None
    return None if dur is None or pct is None else (dur, pct)


def step_ncu_dram(kernels, workload):
    """ncu's DRAM throughput over the pass, time-weighted across its kernels
    (each kernel's own capture: serialised, cold L2), or None unless every
    kernel has a summary of its current source."""
    got = {k: load_ncu_dram(k, workload) for k in kernels}
    if any(v is None for v in got.values()):
        return None
    total = sum(d for d, _ in got.values())
    return {"dram_pct_of_peak_time_weighted": sum(d * p for d, p in got.values()) / total,
            "per_kernel": {k: {"us": d, "dram_pct": p} for k, (d, p) in got.items()},
            "source": f"profiles/ncu_<kernel>_{workload}.md (ncu gpu__dram_throughput, "
                      "% of the hardware's peak)"}


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            self.path = os.path.join(tempfile.gettempdir(), f"bench_clocks_{os.getpid()}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows),
                "window": "soak of the same step, then the timed region"}


# ------------------------------------------------------------ CPU baseline
def _pick_pairs(batch, nheads, n):
    step = max(1, (batch * nheads) // max(1, n))
    pairs = [(i // nheads, i % nheads) for i in range(0, batch * nheads, step)][:n]
    return pairs


def oracle_sample_problem(w, inp, npairs):
    """The sampled (batch, head) sequences gathered into one fp64 problem of
    batch 1 whose heads are the sampled pairs, each its own group (a head only
    reads its own group's B and C, so this is the same arithmetic)."""
    import numpy as np
    import torch
    pairs = _pick_pairs(w.batch, w.nheads, npairs)
    r = w.nheads // w.ngroups
    dev = inp["x"].device
    bi = torch.tensor([b for b, _ in pairs], device=dev)
    hi = torch.tensor([h for _, h in pairs], device=dev)
    gi = hi // r
    f64 = lambda t: np.ascontiguousarray(t.cpu().to(torch.float64).numpy())  # noqa: E731
    prob = {
        "x": f64(inp["x"][bi, :, hi].permute(1, 0, 2).unsqueeze(0)),
        "dt": f64(inp["dt"][bi, :, hi].permute(1, 0).unsqueeze(0)),
        "A": f64(inp["A"][hi]),
        "B": f64(inp["B"][bi, :, gi].permute(1, 0, 2).unsqueeze(0)),
        "C": f64(inp["C"][bi, :, gi].permute(1, 0, 2).unsqueeze(0)),
        "D": f64(inp["D"][hi]),
        "init": None if inp["initial_state"] is None else f64(inp["initial_state"][bi, hi].unsqueeze(0)),
    }
    return pairs, prob


def run_oracle_sample(w, inp, npairs, prepared=None):
    """The fp64 oracle recurrence, as it stands, on the host cores, over a
    bounded sample: `npairs` (batch, head) sequences of the workload at full
    length (inputs widened to fp64 before the clock starts).  Reported as
    whole-workload tokens/s: the sample's share of the heads times batch*L
    tokens, over the wall time of the oracle call."""
    import oracle
    pairs, prob = prepared if prepared is not None else oracle_sample_problem(w, inp, npairs)
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.ssd_recurrence(prob["x"], prob["dt"], prob["A"], prob["B"], prob["C"], D=prob["D"],
                          init=prob["init"], nthreads=cores)
    dt = time.perf_counter() - t0
    frac = len(pairs) / (w.batch * w.nheads)
    return {"value": frac * w.tokens / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "seconds": dt,
            "sample": f"{len(pairs)} of {w.batch * w.nheads} (batch, head) sequences at full length "
                      f"L={w.seqlen}; fp64 token-by-token recurrence, pthreads over sequences; "
                      f"tokens/s scaled by the fraction of sequences covered"}


def decode_bytes(w):
    """Algorithmic bytes of one decode step: the fp32 state read and written,
    x read and y written, B, C, dt read (A, D are negligible)."""
    e = 2 if w.dtype == "bf16" else 4
    state = 4 * w.batch * w.nheads * w.dstate * w.headdim
    return 2 * state + 2 * w.batch * w.nheads * w.headdim * e + 2 * w.batch * w.ngroups * w.dstate * e \
        + 4 * w.batch * w.nheads


# ----------------------------------------------------------------- GPU arm
def run_decode(args, w, peaks):
    """mamba2_ssd_step on `w` (seqlen 1), state updated in place, L2 flushed
    before each timed step; returns the decode_step object of the JSON line."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    inp = make_inputs(w)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    x, dt, B, C = (d[k][:, 0].contiguous() for k in ("x", "dt", "B", "C"))
    state = d["initial_state"]
    y = torch.empty_like(x)
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()

    def step():
        bd.mamba2_ssd_step(x, dt, d["A"], B, C, state_in=state, D=d["D"], state_out=state, y=y)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ms = []
    for _ in range(max(args.steps, 10)):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        ms.append((a, b))
    torch.cuda.synchronize()
    bd.mamba2_check_device_status()
    t = statistics.mean(a.elapsed_time(b) for a, b in ms)
    nbytes = decode_bytes(w)
    achieved = nbytes / (t * 1e-3) / 1e9
    return {"workload": w.name, "batch": w.batch, "nheads": w.nheads, "headdim": w.headdim,
            "dstate": w.dstate, "ngroups": w.ngroups, "dtype": w.dtype,
            "value": w.batch / (t * 1e-3), "unit": "tokens/s", "ms_per_step": t,
            "roofline": {"kernel": "k_ssd_step", "bound": "hbm", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "algorithmic_bytes": nbytes, "traffic": load_traffic("ssd_step", w.name)},
            "l2": "flushed before every timed step; state updated in place"}



def run_gpu(args, w, rank, world):
    import torch
    import torch.distributed as dist
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300 import build_lib
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    build_lib.build()
    bd.load_library()
    inp = make_inputs(w, seed=w.seed + rank)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    stream = torch.cuda.current_stream()
    shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
    ws = torch.empty(max(bd.mamba2_ssd_fwd_workspace_size(shape), 1), device="cuda", dtype=torch.uint8)
    # the chunk the forward pass runs this shape with (the per-stage timings
    # below launch the stages at that chunk, as the pass does)
    run_chunk = bd.mamba2_ssd_fwd_chunk_size(shape)
    wr = w.with_(chunk_size=run_chunk)
    y = torch.empty_like(d["x"])
    fin = torch.empty(w.batch, w.nheads, w.dstate, w.headdim, device="cuda", dtype=torch.float32)
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)

    def step():
        bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                          initial_state=d["initial_state"], y=y, final_state=fin, workspace=ws)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    bd.mamba2_check_device_status()

    # ---- clocks are sampled from a short soak of the same step through the
    # end of the timed region (the timed region alone is shorter than the
    # sampler's 200 ms period)
    clocks = ClockSampler(local)
    clocks.start()
    t_end = time.perf_counter() + args.soak_s
    while time.perf_counter() < t_end:
        for _ in range(20):
            flush.zero_()
            step()
        torch.cuda.synchronize()

    # ---- timed region: K steps, cold L2 before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    barrier()
    clock_info = clocks.stop()
    bd.mamba2_check_device_status()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms))

    # ---- host time of one call: the public call enqueues the whole pass and
    # returns; timed on the host clock, without synchronising, over a burst of
    # calls (the GPU runs behind them)
    host_us = []
    for _ in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(20):
            step()
        host_us.append((time.perf_counter() - t0) / 20 * 1e6)
    torch.cuda.synchronize()
    host_us_per_call = min(host_us)

    # ---- per-kernel durations: the same launches through the per-stage entry
    # points, at the chunk the forward pass runs
    kev = {k: [] for k in ("chunk_cumsum", "state_pass", "chunk_out")}
    G = ws[: 4 * w.batch * w.nheads * w.seqlen].view(torch.float32).view(w.batch, w.nheads, w.seqlen)
    cs = torch.empty(w.batch, w.nheads, wr.nchunks, w.dstate, w.headdim, device="cuda", dtype=d["x"].dtype)
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        bd.mamba2_chunk_cumsum(d["dt"], d["A"], run_chunk, G=G)
        e[1].record(stream)
        bd.mamba2_state_pass(d["x"], d["dt"], d["B"], G, run_chunk, initial_state=d["initial_state"],
                             chunk_states=cs, final_state=fin)
        e[2].record(stream)
        bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], G, cs, run_chunk, D=d["D"], y=y)
        e[3].record(stream)
        if i >= args.warmup:
            kev["chunk_cumsum"].append((e[0], e[1]))
            kev["state_pass"].append((e[1], e[2]))
            kev["chunk_out"].append((e[2], e[3]))
    torch.cuda.synchronize()
    kernel_ms = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in kev.items()}

    if args.no_e2e:
        return {"total_ms": total_ms, "step_ms": step_ms, "kernel_ms": kernel_ms, "clocks": clock_info,
                "e2e_ms": None, "h2d": 0, "d2h": 0, "inp": inp, "host_us": host_us_per_call,
                "run_chunk": run_chunk}

    # ---- end to end through the public API with host buffers, pipelined as a
    # server runs it: two sets of device buffers; step i's inputs are copied in
    # on one stream while step i-1 computes on another and step i-2's outputs
    # are copied out on a third (copy engines in both directions and the SMs
    # busy at once).  The timed region runs from the first copy-in to the last
    # copy-out, so every step's copies and compute are inside it; the inputs
    # (larger than L2) come from pinned host memory every step.
    host = {k: (v.pin_memory() if v is not None else None) for k, v in inp.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = y.numel() * y.element_size() + fin.numel() * fin.element_size()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    sets = [dict(d={k: (torch.empty_like(v) if v is not None else None) for k, v in d.items()},
                 y=torch.empty_like(y), fin=torch.empty_like(fin), ws=torch.empty_like(ws),
                 y_host=torch.empty(y.shape, dtype=y.dtype).pin_memory(),
                 fin_host=torch.empty(fin.shape, dtype=fin.dtype).pin_memory(),
                 in_done=ev(), comp_done=ev(), out_done=ev()) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        for i in range(n):
            S = sets[i % 2]
            if i >= 2:
                s_in.wait_event(S["comp_done"])  # step i-2 has read this set's inputs
            with torch.cuda.stream(s_in):
                for k, v in host.items():
                    if v is not None:
                        S["d"][k].copy_(v, non_blocking=True)
            S["in_done"].record(s_in)
            stream.wait_event(S["in_done"])
            if i >= 2:
                stream.wait_event(S["out_done"])  # step i-2's outputs have left this set
            bd.mamba2_ssd_fwd(S["d"]["x"], S["d"]["dt"], S["d"]["A"], S["d"]["B"], S["d"]["C"], w.chunk_size,
                              D=S["d"]["D"], initial_state=S["d"]["initial_state"], y=S["y"],
                              final_state=S["fin"], workspace=S["ws"], stream=stream)
            S["comp_done"].record(stream)
            s_out.wait_event(S["comp_done"])
            with torch.cuda.stream(s_out):
                S["y_host"].copy_(S["y"], non_blocking=True)
                S["fin_host"].copy_(S["fin"], non_blocking=True)
            S["out_done"].record(s_out)
        s_out.wait_event(sets[(n - 1) % 2]["comp_done"])
        end.record(s_out)
        end.synchronize()
        return start.elapsed_time(end)

    pipelined(max(args.warmup, 2))
    barrier()
    e2e_ms = [pipelined(args.steps)]
    bd.mamba2_check_device_status()
    e2e_total = max_over_ranks(sum(e2e_ms))
    return {"total_ms": total_ms, "step_ms": step_ms, "kernel_ms": kernel_ms, "clocks": clock_info,
            "e2e_ms": e2e_total, "h2d": h2d, "d2h": d2h, "inp": inp, "host_us": host_us_per_call,
            "run_chunk": run_chunk}


EXTRA_WORKLOADS = ("mamba2_1p3b_layer", "large_state", "blog_example", "long_seq_fp32_t128")


def run_extra(args, w, peaks, cpu_pairs):
    """One more workload, measured like the headline one (inputs resident,
    256 MiB L2 flush before every timed step, CUDA events on the launching
    stream), with the oracle timed on a small sample of it.  Inputs are drawn
    on the GPU (different values than the CPU generator, same distributions)."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    d = make_inputs(w, device="cuda")
    shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
    ws = torch.empty(max(bd.mamba2_ssd_fwd_workspace_size(shape), 1), device="cuda", dtype=torch.uint8)
    y = torch.empty_like(d["x"])
    fin = torch.empty(w.batch, w.nheads, w.dstate, w.headdim, device="cuda", dtype=torch.float32)
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()

    def step():
        bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                          initial_state=d["initial_state"], y=y, final_state=fin, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    ev = []
    for _ in range(args.extra_steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    bd.mamba2_check_device_status()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    run_chunk = bd.mamba2_ssd_fwd_chunk_size(shape)
    flop, flop_dense, bytes_min = work_counts(w.with_(chunk_size=run_chunk))
    out = {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
           "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups, "chunk_size": w.chunk_size,
           "run_chunk_size": run_chunk,
           "seed": w.seed, "tokens_per_s": w.tokens / (ms * 1e-3), "ms_per_step": ms,
           "tflops": flop / (ms * 1e-3) / 1e12,
           "hbm_frac": bytes_min / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
           "tensor_frac": flop / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], "bytes_min": bytes_min}
    if cpu_pairs:
        cb = run_oracle_sample(w, d, min(cpu_pairs, w.batch * w.nheads))
        out["oracle_tokens_per_s"] = cb["value"]
        out["oracle_sample"] = f"{min(cpu_pairs, w.batch * w.nheads)} (batch, head) sequences, {cb['cores']} cores"
    del d, ws, y, fin, flush
    return out


def main():
    args = parse_args()
    from mamba_chunked_ssd_gb300.synthetic import WORKLOADS
    w = WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return main_reference(args, w, rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_gpu(args, w, rank, world)
    if rank != 0:
        return
    # FLOPs and per-kernel bytes at the chunk the forward pass runs
    wr = w.with_(chunk_size=r["run_chunk"])
    flop, flop_dense, bytes_min = work_counts(wr)
    peaks = load_peaks()
    ms = r["total_ms"] / args.steps
    tokens = w.tokens * world
    value = job_tokens_per_s(w.tokens, world, ms)
    kb = kernel_bytes(wr)
    top = max(r["kernel_ms"], key=r["kernel_ms"].get)
    achieved = kb[top] / (r["kernel_ms"][top] * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
                   "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups,
                   "chunk_size": w.chunk_size, "run_chunk_size": r["run_chunk"],
                   "initial_state": w.init_state,
                   "l2": "flushed: 256 MiB buffer written before every timed step",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tflops": flop / (ms * 1e-3) / 1e12 * world,
        "tflops_dense_convention": flop_dense / (ms * 1e-3) / 1e12 * world,
        "step_roofline": {"bytes_min": bytes_min, "flop_alg": flop,
                          "hbm_frac": bytes_min / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                          "tensor_frac": flop / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                          "peaks": peaks["source"]},
        "roofline": {"kernel": top, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": load_traffic(top, w.name), "algorithmic_bytes": kb[top]},
        "step_ncu": step_ncu_dram(list(r["kernel_ms"]), w.name),
        "kernel_ms": r["kernel_ms"],
        "host_us_per_call": r["host_us"],
        "gpu_launches": 3 * args.steps,
        "e2e": None if r["e2e_ms"] is None else {
            "value": tokens / (r["e2e_ms"] / args.steps * 1e-3), "unit": "tokens/s",
            "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
            "mode": "pipelined: two buffer sets; copy-in of step i, compute of step i-1 and copy-out of "
                    "step i-2 overlap on three streams; timed from the first copy-in to the last copy-out; "
                    "inputs larger than L2, no flush"},
        "clocks": r["clocks"],
    }
    if not args.no_decode and w.seqlen > 1:
        out["decode_step"] = run_decode(args, WORKLOADS["decode_b256"], peaks)
    if not args.no_extra:
        from mamba_chunked_ssd_gb300.synthetic import sweep_workloads
        pairs = 0 if args.no_cpu_baseline else 8
        out["other_workloads"] = [run_extra(args, WORKLOADS[n], peaks, pairs)
                                  for n in EXTRA_WORKLOADS if n != w.name]
        out["sweep"] = [run_extra(args, sw, peaks, 0) for sw in sweep_workloads(seeds=(0,))]
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = run_oracle_sample(w, r["inp"], args.cpu_pairs)
        out["cpu_baseline"].pop("seconds", None)
    print(json.dumps(out), flush=True)


def main_reference(args, w, rank):
    """The reference arm: the fp64 CPU oracle, as it stands, on host cores.
    Each step is a bounded sample of the workload (see run_oracle_sample)."""
    if rank != 0:
        return
    from mamba_chunked_ssd_gb300.synthetic import make_inputs
    inp = make_inputs(w)
    prepared = oracle_sample_problem(w, inp, args.cpu_pairs)
    small = oracle_sample_problem(w, inp, max(1, args.cpu_pairs // 8))
    for _ in range(args.warmup):
        run_oracle_sample(w, inp, 0, prepared=small)
    runs = [run_oracle_sample(w, inp, args.cpu_pairs, prepared=prepared) for _ in range(args.steps)]
    secs = sum(r["seconds"] for r in runs)
    frac_tokens = sum(r["value"] * r["seconds"] for r in runs)
    value = frac_tokens / secs
    ms = secs / args.steps * 1e3
    cb = {k: v for k, v in runs[0].items() if k != "seconds"}
    cb["value"] = value
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
                      "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups,
                      "chunk_size": w.chunk_size, "initial_state": w.init_state},
           "cpu_baseline": cb,
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
