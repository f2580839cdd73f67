"""Times the alternatives behind the library's per-shape kernel choices.

The library picks, per problem shape, among kernels that all compute the same
result (host dispatch in csrc/dispatch.cu and the launchers).  Where a choice
has more than one candidate that fits, an environment override forces one of
them, and this tool times each candidate on the GPU so the dispatch rule can
be checked against measurements:

  MAMBA2_CHUNK_OUT_HEAD_SPLIT = 1 | 2   stage 3 with heads of 128 columns
      whole (one 128-wide MMA per head) or split into two 64-wide virtual
      heads sharing the head's decays; a forced variant that does not fit
      runs stage 3 on the CUDA-core kernel instead (its time is shown).
  MAMBA2_FWD_PATH = staged | fused      the whole forward pass as separate
      stages or with the fused state-pass + output kernel (where it fits:
      bf16, head dim 64 in pairs of one group, state 128, chunk 128 or 256).
  MAMBA2_STATE_SEGMENTS = 1             the forward pass's state pass in one
      pass over each sequence, instead of over sequence segments where the
      (batch, head) pairs are few.
  MAMBA2_FP32_PATH = simt               an fp32 forward pass on the CUDA
      cores instead of the split-bf16 tensor-core kernels (where they fit:
      head dim 64 or 128, state 64 or 128; run at chunk 128).
  MAMBA2_FWD_CHUNK = given | 64 | 128 | 256   the chunk the forward pass
      runs with: the caller's, or a fixed one (the result does not depend on
      it; the default picks one per shape).
  MAMBA2_STATE_PAIRS = 0 | 1            the state pass with heads of 64
      columns one per CTA, or two of one group per CTA as one head of 128
      columns (where the head count and the group size are even).
  MAMBA2_CHUNK_OUT_PERSISTENT = 0       stage 3 with one CTA per work item
      instead of one CTA per SM taking an equal share of the work (where
      every chunk is one 128-row block: chunks of 128, and of 64 in pairs).

Usage (one GPU):  python -m mamba_chunked_ssd_gb300.tune [--steps K] [--json]
Each line: workload, candidate, mean stage time in microseconds (CUDA events
on the launching stream, a 256 MiB L2 flush before every timed launch), and
the candidate the default rule picks.  Inputs are seeded synthetic tensors
drawn on the GPU.

    python -m mamba_chunked_ssd_gb300.tune --profile WORKLOAD [--steps K]
runs K forward passes (default 3) of one named workload and nothing else,
for a profiler's launch list.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FLUSH_BYTES = 256 << 20
HEAD_SPLIT_ENV = "MAMBA2_CHUNK_OUT_HEAD_SPLIT"
FWD_PATH_ENV = "MAMBA2_FWD_PATH"
SEGMENTS_ENV = "MAMBA2_STATE_SEGMENTS"
FP32_ENV = "MAMBA2_FP32_PATH"
FWD_CHUNK_ENV = "MAMBA2_FWD_CHUNK"
PAIRS_ENV = "MAMBA2_STATE_PAIRS"
PERSISTENT_ENV = "MAMBA2_CHUNK_OUT_PERSISTENT"


def _time(fn, steps, warmup, flush, stream):
    import torch
    for _ in range(warmup):
        flush.zero_()
        fn()
    ev = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3


def head_split_rows(workloads, steps=10, warmup=3):
    """Stage-3 time of every candidate head split, per workload with 128-wide
    heads (others have one candidate)."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    bd.load_library()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    rows = []
    saved = os.environ.pop(HEAD_SPLIT_ENV, None)
    try:
        for w in workloads:
            if w.headdim != 128 or w.dtype != "bf16":
                continue
            d = make_inputs(w, device="cuda")
            G = bd.mamba2_chunk_cumsum(d["dt"], d["A"], w.chunk_size)
            cs, _ = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], G, w.chunk_size,
                                         initial_state=d["initial_state"], want_final_state=False)
            y = torch.empty_like(d["x"])
            fn = lambda: bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], G, cs, w.chunk_size,  # noqa: E731
                                             D=d["D"], y=y)
            times = {}
            for cand in ("1", "2"):
                os.environ[HEAD_SPLIT_ENV] = cand
                times[cand] = _time(fn, steps, warmup, flush, stream)
            os.environ.pop(HEAD_SPLIT_ENV, None)
            default_us = _time(fn, steps, warmup, flush, stream)
            bd.mamba2_check_device_status()
            rows.append({"workload": w.name, "seqlen": w.seqlen, "dstate": w.dstate, "headdim": w.headdim,
                         "chunk_size": w.chunk_size, "whole_us": times["1"], "split_us": times["2"],
                         "default_us": default_us})
            del d, G, cs, y
    finally:
        if saved is not None:
            os.environ[HEAD_SPLIT_ENV] = saved
    return rows


def fused_fits(w):
    """The fused kernel's shape range (mirrors ssd_fused_fits in the library)."""
    return (w.dtype == "bf16" and w.headdim == 64 and w.dstate == 128 and w.chunk_size in (128, 256)
            and w.nheads % 2 == 0 and (w.nheads // w.ngroups) % 2 == 0)


def fwd_path_rows(workloads, steps=10, warmup=3):
    """Whole-pass time (mamba2_ssd_fwd) on the separate stages and on the fused
    kernel, per workload the fused kernel covers."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    bd.load_library()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    rows = []
    saved = os.environ.pop(FWD_PATH_ENV, None)
    try:
        for w in workloads:
            if not fused_fits(w):
                continue
            d = make_inputs(w, device="cuda")
            shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
            ws = torch.empty(max(bd.mamba2_ssd_fwd_workspace_size(shape), 1), device="cuda", dtype=torch.uint8)
            y = torch.empty_like(d["x"])
            fin = torch.empty(w.batch, w.nheads, w.dstate, w.headdim, device="cuda", dtype=torch.float32)
            fn = lambda: bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size,  # noqa: E731
                                           D=d["D"], initial_state=d["initial_state"], y=y, final_state=fin,
                                           workspace=ws)
            times = {}
            for cand in ("staged", "fused"):
                os.environ[FWD_PATH_ENV] = cand
                times[cand] = _time(fn, steps, warmup, flush, stream)
            os.environ.pop(FWD_PATH_ENV, None)
            bd.mamba2_check_device_status()
            rows.append({"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
                         "chunk_size": w.chunk_size, "staged_us": times["staged"], "fused_us": times["fused"]})
            del d, ws, y, fin
    finally:
        if saved is not None:
            os.environ[FWD_PATH_ENV] = saved
    return rows


def segment_rows(workloads, steps=10, warmup=3):
    """Whole-pass time with the state pass over sequence segments (the
    default where it applies) and in one pass, per workload where the
    default splits the sequences."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    bd.load_library()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    rows = []
    saved = os.environ.pop(SEGMENTS_ENV, None)
    try:
        for w in workloads:
            if w.dtype != "bf16":
                continue
            d = make_inputs(w, device="cuda")
            shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
            need = bd.mamba2_ssd_fwd_workspace_size(shape)
            os.environ[SEGMENTS_ENV] = "1"
            one = bd.mamba2_ssd_fwd_workspace_size(shape)
            os.environ.pop(SEGMENTS_ENV, None)
            if need == one:  # the default runs one pass: nothing to compare
                del d
                continue
            ws = torch.empty(need, device="cuda", dtype=torch.uint8)
            y = torch.empty_like(d["x"])
            fn = lambda: bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size,  # noqa: E731
                                           D=d["D"], initial_state=d["initial_state"], y=y, workspace=ws)
            seg_us = _time(fn, steps, warmup, flush, stream)
            os.environ[SEGMENTS_ENV] = "1"
            one_us = _time(fn, steps, warmup, flush, stream)
            os.environ.pop(SEGMENTS_ENV, None)
            bd.mamba2_check_device_status()
            rows.append({"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
                         "chunk_size": w.chunk_size, "segments_us": seg_us, "one_pass_us": one_us})
            del d, ws, y
    finally:
        os.environ.pop(SEGMENTS_ENV, None)
        if saved is not None:
            os.environ[SEGMENTS_ENV] = saved
    return rows


def fp32_rows(workloads, steps=5, warmup=2):
    """Whole-pass time of fp32 workloads on the tensor cores (split bf16) and
    on the CUDA cores."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    bd.load_library()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    rows = []
    saved = os.environ.pop(FP32_ENV, None)
    try:
        for w in workloads:
            if w.dtype != "fp32":
                continue
            d = make_inputs(w, device="cuda")
            shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
            times = {}
            for cand in ("tc", "simt"):
                if cand == "simt":
                    os.environ[FP32_ENV] = "simt"
                ws = torch.empty(max(bd.mamba2_ssd_fwd_workspace_size(shape), 1), device="cuda", dtype=torch.uint8)
                y = torch.empty_like(d["x"])
                fn = lambda: bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size,  # noqa: E731
                                               D=d["D"], initial_state=d["initial_state"], y=y, workspace=ws)
                times[cand] = _time(fn, steps, warmup, flush, stream)
                os.environ.pop(FP32_ENV, None)
                del ws, y
            bd.mamba2_check_device_status()
            rows.append({"workload": w.name, "tensor_cores_us": times["tc"], "cuda_cores_us": times["simt"]})
            del d
    finally:
        os.environ.pop(FP32_ENV, None)
        if saved is not None:
            os.environ[FP32_ENV] = saved
    return rows


def chunk_rows(workloads, steps=10, warmup=3):
    """Whole-pass time (mamba2_ssd_fwd) with each chunk the forward pass can
    run (64, 128, 256), and the one the default rule picks."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    bd.load_library()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    rows = []
    saved = os.environ.pop(FWD_CHUNK_ENV, None)
    try:
        for w in workloads:
            d = make_inputs(w, device="cuda")
            shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
            default = bd.mamba2_ssd_fwd_chunk_size(shape)
            y = torch.empty_like(d["x"])
            times = {}
            for cand in ("64", "128", "256"):
                os.environ[FWD_CHUNK_ENV] = cand
                ws = torch.empty(max(bd.mamba2_ssd_fwd_workspace_size(shape), 1), device="cuda", dtype=torch.uint8)
                fn = lambda: bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size,  # noqa: E731
                                               D=d["D"], initial_state=d["initial_state"], y=y, workspace=ws)
                times[cand] = _time(fn, steps, warmup, flush, stream)
                del ws
            os.environ.pop(FWD_CHUNK_ENV, None)
            bd.mamba2_check_device_status()
            rows.append({"workload": w.name, "chunk_size": w.chunk_size, "default_chunk": default,
                         **{f"chunk{k}_us": v for k, v in times.items()}})
            del d, y
    finally:
        if saved is not None:
            os.environ[FWD_CHUNK_ENV] = saved
    return rows


def profile_run(name, steps):
    """`steps` forward passes of one named workload, synchronised at the end."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import WORKLOADS, make_inputs

    w = WORKLOADS[name]
    d = make_inputs(w, device="cuda")
    shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
    ws = torch.empty(max(bd.mamba2_ssd_fwd_workspace_size(shape), 1), device="cuda", dtype=torch.uint8)
    y = torch.empty_like(d["x"])
    for _ in range(steps):
        bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                          initial_state=d["initial_state"], y=y, workspace=ws)
    torch.cuda.synchronize()
    bd.mamba2_check_device_status()
    print(f"{name}: {steps} forward passes")


def env_rows(workloads, env, values, steps=10, warmup=3):
    """Whole-pass time of each workload with the environment variable `env`
    set to each of `values` in turn, and with it unset (the default)."""
    import torch
    from mamba_chunked_ssd_gb300 import binding as bd
    from mamba_chunked_ssd_gb300.synthetic import make_inputs

    bd.load_library()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    rows = []
    saved = os.environ.pop(env, None)
    try:
        for w in workloads:
            d = make_inputs(w, device="cuda")
            shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
            ws = torch.empty(max(bd.mamba2_ssd_fwd_workspace_size(shape), 1), device="cuda", dtype=torch.uint8)
            y = torch.empty_like(d["x"])
            fn = lambda: bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size,  # noqa: E731
                                           D=d["D"], initial_state=d["initial_state"], y=y, workspace=ws)
            r = {"workload": w.name}
            for v in values:
                os.environ[env] = v
                r[v] = _time(fn, steps, warmup, flush, stream)
            os.environ.pop(env, None)
            r["default"] = _time(fn, steps, warmup, flush, stream)
            bd.mamba2_check_device_status()
            rows.append(r)
            del d, ws, y
    finally:
        os.environ.pop(env, None)
        if saved is not None:
            os.environ[env] = saved
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--json", action="store_true")
    ap.add_argument("--profile", metavar="WORKLOAD", default=None)
    args = ap.parse_args()
    if args.profile:
        profile_run(args.profile, args.steps or 3)
        return
    args.steps = args.steps or 10
    from mamba_chunked_ssd_gb300.synthetic import WORKLOADS, sweep_workloads
    ws = [WORKLOADS["large_state"], WORKLOADS["long_seq_carried_state"], WORKLOADS["mamba2_1p3b_layer"],
          WORKLOADS["blog_example"]] + sweep_workloads(seeds=(0,))
    from mamba_chunked_ssd_gb300.synthetic import Workload
    seg_ws = [WORKLOADS["blog_example"],
              Workload("few_heads_t256", 1, 32768, 4, 64, 128, 1, 256),
              Workload("few_heads_h128", 2, 16384, 4, 128, 128, 1, 128)]
    chunks = chunk_rows([w for w in ws if w.dtype == "bf16"], steps=args.steps)
    rows = head_split_rows(ws, steps=args.steps)
    paths = fwd_path_rows(ws, steps=args.steps)
    segs = segment_rows(seg_ws, steps=args.steps)
    f32 = fp32_rows([WORKLOADS["long_seq_fp32_t128"],
                     Workload("fp32_h128_s64", 2, 4096, 16, 128, 64, 2, 128, dtype="fp32")])
    h64 = [w for w in ws if w.dtype == "bf16" and w.headdim == 64 and w.nheads % 2 == 0
           and (w.nheads // w.ngroups) % 2 == 0]
    pairs = env_rows(h64, PAIRS_ENV, ("0", "1"), steps=args.steps)
    persist = env_rows([w for w in ws if w.dtype == "bf16"], PERSISTENT_ENV, ("0",), steps=args.steps)
    if args.json:
        print(json.dumps({"chunk": chunks, "head_split": rows, "fwd_path": paths, "segments": segs,
                          "fp32": f32, "state_pairs": pairs, "persistent": persist}))
        return
    print("Whole forward pass at each chunk it can run:")
    print("| workload (caller's chunk) | 64 (µs) | 128 (µs) | 256 (µs) | default |")
    print("|---|---|---|---|---|")
    for r in chunks:
        print(f"| {r['workload']} ({r['chunk_size']}) | {r['chunk64_us']:.1f} | {r['chunk128_us']:.1f} | "
              f"{r['chunk256_us']:.1f} | {r['default_chunk']} |")
    print()
    print("Stage 3, heads of 128 columns:")
    print("| workload | whole heads (µs) | split heads (µs) | default (µs) |")
    print("|---|---|---|---|")
    for r in rows:
        print(f"| {r['workload']} | {r['whole_us']:.1f} | {r['split_us']:.1f} | {r['default_us']:.1f} |")
    print()
    print("Whole forward pass where the fused kernel fits:")
    print("| workload | separate stages (µs) | fused (µs) |")
    print("|---|---|---|")
    for r in paths:
        print(f"| {r['workload']} | {r['staged_us']:.1f} | {r['fused_us']:.1f} |")
    print()
    print("State pass over sequence segments vs one pass (whole forward pass):")
    print("| workload | segments (µs) | one pass (µs) |")
    print("|---|---|---|")
    for r in segs:
        print(f"| {r['workload']} | {r['segments_us']:.1f} | {r['one_pass_us']:.1f} |")
    print()
    print("fp32 forward pass, split-bf16 tensor cores vs CUDA cores:")
    print("| workload | tensor cores (µs) | CUDA cores (µs) |")
    print("|---|---|---|")
    for r in f32:
        print(f"| {r['workload']} | {r['tensor_cores_us']:.1f} | {r['cuda_cores_us']:.1f} |")
    print()
    print("State pass with heads of 64 columns single or in pairs (whole forward pass):")
    print("| workload | single (µs) | pairs (µs) | default (µs) |")
    print("|---|---|---|---|")
    for r in pairs:
        print(f"| {r['workload']} | {r['0']:.1f} | {r['1']:.1f} | {r['default']:.1f} |")
    print()
    print("Stage 3 with one CTA per work item vs persistent CTAs (whole forward pass):")
    print("| workload | one CTA per item (µs) | default (µs) |")
    print("|---|---|---|")
    for r in persist:
        print(f"| {r['workload']} | {r['0']:.1f} | {r['default']:.1f} |")


if __name__ == "__main__":
    main()
