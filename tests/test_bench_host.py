"""Host logic of bench.py, on the CPU: the algorithmic work and byte counts
that the reported rooflines divide by, the link from a kernel to its committed
ncu traffic (which must drop to None once the kernel source changes), and the
JSON line of the reference arm.

The counts are checked against independent tallies: FLOPs by walking the
causal pairs of every chunk, bytes by summing the sizes of the tensors each
kernel reads and writes once.
"""
import json
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mamba_chunked_ssd_gb300.synthetic import WORKLOADS, Workload  # noqa: E402


def _causal_pairs(L, T):
    """(i, j) pairs with j <= i inside each chunk, the last chunk ragged."""
    n = 0
    for c0 in range(0, L, T):
        t = min(T, L - c0)
        n += t * (t + 1) // 2
    return n


@pytest.mark.parametrize("w", [WORKLOADS["long_seq_carried_state"], WORKLOADS["mamba2_1p3b_layer"],
                               Workload("ragged", 2, 300, 4, 16, 8, 2, 64)],
                         ids=["bench", "1p3b", "ragged"])
def test_work_counts_against_a_tally(w):
    flop, _, bytes_min = bench.work_counts(w)
    e = 2 if w.dtype == "bf16" else 4
    pairs = w.batch * _causal_pairs(w.seqlen, w.chunk_size)
    N = w.batch * w.seqlen
    # C B^T per group and (CB . decay) X per head over the causal pairs, 2 flops
    # per multiply-add; the state terms C h and B^T (w x): 2 S H each per token and head
    tally = 2 * pairs * (w.ngroups * w.dstate + w.nheads * w.headdim) + 4 * N * w.nheads * w.dstate * w.headdim
    if w.seqlen % w.chunk_size == 0:
        assert flop == tally
    else:
        assert flop >= tally  # the formula counts every chunk as full
    state = 4 * w.batch * w.nheads * w.dstate * w.headdim
    tensors = (2 * N * w.nheads * w.headdim * e          # x in, y out
               + 2 * N * w.ngroups * w.dstate * e        # B, C in
               + 4 * N * w.nheads                        # dt in
               + state * (2 if w.init_state else 1))     # final state out, initial in
    assert bytes_min == tensors


def test_kernel_bytes_bench_workload():
    w = WORKLOADS["long_seq_carried_state"]
    kb = bench.kernel_bytes(w)
    N = w.batch * w.seqlen
    x = N * w.nheads * w.headdim * 2
    bc = N * w.ngroups * w.dstate * 2
    dt = g = 4 * N * w.nheads
    cs = w.batch * w.nheads * w.nchunks * w.dstate * w.headdim * 2
    state = 4 * w.batch * w.nheads * w.dstate * w.headdim
    assert kb["chunk_cumsum"] == dt + g + 4 * w.nheads
    assert kb["state_pass"] == x + dt + bc + g + cs + 2 * state
    assert kb["chunk_out"] == 2 * x + dt + g + 2 * bc + cs + 4 * w.nheads
    assert kb["chunk_out"] == 704_643_328  # the figure the bench line and the design notes quote


@pytest.mark.parametrize("kernel", ["chunk_out", "state_pass", "chunk_cumsum"])
def test_traffic_link_follows_the_committed_summary(kernel):
    """The recorded DRAM bytes while the kernel source still has the hash the
    summary names; None (no traffic claim) once the source has changed."""
    import hashlib
    t = bench.load_traffic(kernel, "long_seq_carried_state")
    path = os.path.join(ROOT, "profiles", f"ncu_{kernel}_long_seq_carried_state.md")
    fields = dict(ln.split(":", 1) for ln in open(path)
                  if ln.startswith(("traffic_bytes_per_launch:", "source:", "source_sha256_16:")))
    src = os.path.join(ROOT, fields["source"].strip())
    same = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] == fields["source_sha256_16"].strip()
    if same:
        assert t == float(fields["traffic_bytes_per_launch"])
    else:
        assert t is None


def test_traffic_link_drops_when_the_source_changes(tmp_path, monkeypatch):
    """A summary whose recorded source hash no longer matches gives None."""
    (tmp_path / "profiles").mkdir()
    src_dir = tmp_path / "mamba_chunked_ssd_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    import hashlib
    src = os.path.join(ROOT, "mamba_chunked_ssd_gb300", "csrc", "k_chunk_out_tc.cu")
    shutil.copy(src, src_dir)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    with open(tmp_path / "profiles" / "ncu_chunk_out_long_seq_carried_state.md", "w") as f:
        f.write("# summary\n\ntraffic_bytes_per_launch: 12345\n"
                "source: mamba_chunked_ssd_gb300/csrc/k_chunk_out_tc.cu\n"
                f"source_sha256_16: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("chunk_out", "long_seq_carried_state") is not None
    with open(src_dir / "k_chunk_out_tc.cu", "a") as f:
        f.write("\n// changed\n")
    assert bench.load_traffic("chunk_out", "long_seq_carried_state") is None
    assert bench.load_traffic("no_such_kernel", "long_seq_carried_state") is None


def test_reference_arm_json_line():
    """--impl reference on a tiny workload: one JSON line with the contract's
    keys, the oracle as both the value and the cpu_baseline, no host copies."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_fp32", "--steps", "1", "--warmup", "1", "--cpu-pairs", "2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 1
    assert d["config"]["workload"] == "tiny_fp32"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_step_ncu_dram_weights_the_committed_summaries(tmp_path, monkeypatch):
    """The pass's ncu DRAM throughput is each kernel's figure weighted by its
    captured duration, and no figure at all once any kernel's source has
    changed since its capture."""
    import hashlib
    (tmp_path / "profiles").mkdir()
    src_dir = tmp_path / "csrc"
    src_dir.mkdir()
    figures = {"a": (10.0, 20.0), "b": (30.0, 60.0)}
    for k, (us, pct) in figures.items():
        src = src_dir / f"{k}.cu"
        src.write_text(f"// kernel {k}\n")
        sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
        with open(tmp_path / "profiles" / f"ncu_{k}_wl.md", "w") as f:
            f.write("# summary\n\n| counter | value | unit |\n|---|---|---|\n"
                    f"| duration (`gpu__time_duration.sum`) | {us} | us |\n"
                    f"| DRAM throughput (`gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed`) | {pct} | % |\n"
                    "\ntraffic_bytes_per_launch: 1000\n"
                    f"source: csrc/{k}.cu\nsource_sha256_16: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    r = bench.step_ncu_dram(["a", "b"], "wl")
    assert r["dram_pct_of_peak_time_weighted"] == pytest.approx((10 * 20 + 30 * 60) / 40)
    assert r["per_kernel"]["b"] == {"us": 30.0, "dram_pct": 60.0}
    with open(src_dir / "b.cu", "a") as f:
        f.write("// changed\n")
    assert bench.step_ncu_dram(["a", "b"], "wl") is None
