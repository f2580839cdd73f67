"""The fused state-pass + output kernel (mamba2_ssd_fwd's path for 64-wide
heads in pairs of one group with state 128 and chunks of 128 or 256 tokens)
against the fp64 recurrence, element by element, and against the three-stage
path on the same inputs.  MAMBA2_FWD_PATH forces a path; shapes outside the
fused kernel's range keep the staged path whatever the override says.
"""
import pytest
import torch

import oracle
from gpu_helpers import TOL, Guarded, np64, oracle_pairs, rel_err, sample_pairs, strong_decay, to_dev
from mamba_chunked_ssd_gb300 import binding as bd
from mamba_chunked_ssd_gb300.synthetic import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mamba_chunked_ssd_gb300 import build_lib
    build_lib.build()
    bd.load_library()


def _fwd(d, w, D=True, final=True):
    y, fin = bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size,
                               D=d["D"] if D else None, initial_state=d["initial_state"],
                               want_final_state=final)
    bd.mamba2_check_device_status()
    return y, fin


FUSED = [
    Workload("fused_t256_two_chunks", 2, 512, 4, 64, 128, 1, 256, init_state=True),
    Workload("fused_t128", 1, 640, 6, 64, 128, 1, 128, init_state=True),
    Workload("fused_t256_ragged", 2, 777, 2, 64, 128, 1, 256),
    Workload("fused_t128_ragged_groups", 1, 333, 8, 64, 128, 2, 128, init_state=True),
    Workload("fused_one_block", 1, 100, 2, 64, 128, 1, 256, init_state=True),
    Workload("fused_t256_single_token_tail", 1, 513, 4, 64, 128, 2, 256, init_state=True),
]


@pytest.mark.parametrize("w", FUSED, ids=[w.name for w in FUSED])
def test_fused_matches_oracle(w, monkeypatch):
    monkeypatch.setenv("MAMBA2_FWD_PATH", "fused")
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert torch.isfinite(y.float()).all()
    assert rel_err(np64(y), r["y"]) <= TOL["bf16"]
    assert rel_err(np64(fin), r["final_state"]) <= TOL["bf16"]
    for h in range(w.nheads):
        assert rel_err(np64(y[:, :, h]), r["y"][:, :, h]) <= TOL["bf16"], h


@pytest.mark.parametrize("w", FUSED[:3], ids=[w.name for w in FUSED[:3]])
def test_fused_matches_staged_path(w, monkeypatch):
    """The two paths compute the same function: their difference is within
    the rounding of either against the oracle."""
    inp = make_inputs(w)
    d = to_dev(inp)
    monkeypatch.setenv("MAMBA2_FWD_PATH", "fused")
    y_f, fin_f = _fwd(d, w)
    monkeypatch.setenv("MAMBA2_FWD_PATH", "staged")
    y_s, fin_s = _fwd(d, w)
    assert rel_err(np64(y_f), np64(y_s)) <= TOL["bf16"]
    assert rel_err(np64(fin_f), np64(fin_s)) <= TOL["bf16"]


@pytest.mark.parametrize("w", FUSED[:2], ids=[w.name for w in FUSED[:2]])
def test_fused_optional_pointers_and_guards(w, monkeypatch):
    """D = NULL, final_state = NULL, no initial state; outputs between guard
    regions."""
    monkeypatch.setenv("MAMBA2_FWD_PATH", "fused")
    inp = make_inputs(w)
    inp["initial_state"] = None
    d = to_dev(inp)
    shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
    y = Guarded(d["x"].shape, d["x"].dtype)
    ws = Guarded((bd.mamba2_ssd_fwd_workspace_size(shape),), torch.uint8)
    bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=None, y=y.t,
                      want_final_state=False, workspace=ws.t)
    bd.mamba2_check_device_status()
    assert y.intact() and ws.intact()
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=None, init=None)
    assert rel_err(np64(y.t), r["y"]) <= TOL["bf16"]
    fin = Guarded((w.batch, w.nheads, w.dstate, w.headdim), torch.float32)
    y2 = Guarded(d["x"].shape, d["x"].dtype)
    bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"], y=y2.t,
                      final_state=fin.t)
    bd.mamba2_check_device_status()
    assert y2.intact() and fin.intact()
    r2 = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"], init=None)
    assert rel_err(np64(y2.t), r2["y"]) <= TOL["bf16"]
    assert rel_err(np64(fin.t), r2["final_state"]) <= TOL["bf16"]


STRONG = [
    Workload("fused_strong_t256", 2, 768, 6, 64, 128, 1, 256, init_state=True),
    Workload("fused_strong_t128_ragged", 1, 650, 6, 64, 128, 3, 128),
]


@pytest.mark.parametrize("w", STRONG, ids=[w.name for w in STRONG])
def test_fused_strong_decay(w, monkeypatch):
    monkeypatch.setenv("MAMBA2_FWD_PATH", "fused")
    inp = strong_decay(make_inputs(w))
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert torch.isfinite(y.float()).all()
    assert rel_err(np64(fin), r["final_state"]) <= TOL["bf16"]
    for h in range(w.nheads):
        assert rel_err(np64(y[:, :, h]), r["y"][:, :, h]) <= TOL["bf16"], h


def test_fused_exact_properties(monkeypatch):
    """Causality on the fused path: a change at token tp leaves every output
    of the 128-token blocks before tp's block bit-exactly unchanged, and the
    earlier outputs of tp's own block unchanged up to rounding (the kernel
    picks each block's decay split from the block's first and last G, so
    their rounding, not their value, depends on the whole block).  dt = 0
    keeps the state bit-exactly."""
    monkeypatch.setenv("MAMBA2_FWD_PATH", "fused")
    w = Workload("fused_exact", 1, 512, 2, 64, 128, 1, 256, init_state=True)
    inp = make_inputs(w)
    base, _ = _fwd(to_dev(inp), w)
    for tp in (5, 127, 128, 255, 256, 400):
        q = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
        q["x"][:, tp] += 1.0
        q["B"][:, tp] -= 0.5
        q["C"][:, tp] *= 2.0
        q["dt"][:, tp] += 0.05
        y, _ = _fwd(to_dev(q), w)
        blk = tp - tp % 128
        assert torch.equal(y[:, :blk], base[:, :blk]), tp
        if tp > blk:
            assert rel_err(np64(y[:, blk:tp]), np64(base[:, blk:tp])) <= 1e-2, tp
        assert not torch.equal(y[:, tp], base[:, tp])
    inp["dt"].zero_()
    d = to_dev(inp)
    _, fin = _fwd(d, w)
    assert torch.equal(fin, d["initial_state"])


def test_fused_long_sequence_full_size(monkeypatch):
    """The long-sequence workload at full size on the fused path, sampled
    (batch, head) pairs against the recurrence."""
    monkeypatch.setenv("MAMBA2_FWD_PATH", "fused")
    w = WORKLOADS["long_seq_carried_state"]
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    pairs = sample_pairs(w.batch, w.nheads, 8, seed=11)
    ref = oracle_pairs(inp, pairs)
    for b, h in pairs:
        assert rel_err(np64(y[b, :, h]), ref[(b, h)][0]) <= TOL["bf16"], (b, h)
        assert rel_err(np64(fin[b, h]), ref[(b, h)][1]) <= TOL["bf16"], (b, h)


def _fused_sweep():
    from mamba_chunked_ssd_gb300.synthetic import sweep_workloads
    return [w for w in sweep_workloads(seeds=(0, 1, 2)) if w.dstate == 128 and w.headdim == 64]


FUSED_SWEEP = _fused_sweep()


@pytest.mark.parametrize("w", FUSED_SWEEP, ids=[f"{w.name}_seed{w.seed}" for w in FUSED_SWEEP])
def test_fused_sweep_shape_sampled(w, monkeypatch):
    """The sweep points the fused kernel covers (state 128, head dim 64; every
    length, both chunks, seeds 0-2) at full size on the fused path, inputs
    drawn on the GPU; four (batch, head) pairs per point against the fp64
    recurrence."""
    monkeypatch.setenv("MAMBA2_FWD_PATH", "fused")
    inp = make_inputs(w, device="cuda")
    y, fin = _fwd(inp, w)
    pairs = sample_pairs(w.batch, w.nheads, 4, seed=7 * w.seqlen + 1000 * w.seed + w.chunk_size)
    ref = oracle_pairs(inp, pairs)
    bi = torch.tensor([b for b, _ in pairs], device="cuda")
    hi = torch.tensor([h for _, h in pairs], device="cuda")
    ys = y[bi, :, hi].cpu()
    fs = fin[bi, hi].cpu()
    for i, p in enumerate(pairs):
        assert rel_err(np64(ys[i]), ref[p][0]) <= TOL["bf16"], p
        assert rel_err(np64(fs[i]), ref[p][1]) <= TOL["bf16"], p
    assert torch.isfinite(y.float()).all()
