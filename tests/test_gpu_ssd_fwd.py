"""End-to-end GPU parity of mamba2_ssd_fwd against the fp64 recurrence.

Small shapes (several tiles and ragged tails) are compared in full; the named
workloads at full size, launched exactly as the benchmark launches them, are
compared on sampled (batch, head) pairs that the oracle computes one by one.
Bit-exact properties: causality, equal heads give equal outputs, dt = 0 keeps
the state.  Edge cases: empty sequence, empty batch, misaligned pointers.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, Guarded, np64, oracle_pairs, rel_err, sample_pairs, strong_decay, to_dev
import oracle
from mamba_chunked_ssd_gb300 import binding as bd
from mamba_chunked_ssd_gb300.synthetic import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mamba_chunked_ssd_gb300 import build_lib
    build_lib.build()
    bd.load_library()


def _fwd(d, w):
    y, fin = bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                               initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    return y, fin


SMALL = [
    Workload("fp32_tiny", 1, 256, 2, 16, 16, 1, 64, dtype="fp32"),
    Workload("fp32_ragged_groups", 2, 150, 4, 32, 32, 2, 32, dtype="fp32", init_state=True),
    Workload("bf16_t256_two_chunks", 2, 512, 4, 64, 128, 1, 256, init_state=True),
    Workload("bf16_t256_ragged", 1, 777, 3, 64, 128, 1, 256),
    Workload("bf16_t128_groups", 2, 640, 8, 64, 64, 4, 128, init_state=True),
    Workload("bf16_h128_s256", 1, 384, 8, 128, 256, 2, 128, dt_mu=-4.0, init_state=True),
    Workload("bf16_t64", 1, 320, 2, 64, 128, 1, 64, init_state=True),
    # one X/h stage with two head streams in the output kernel
    Workload("bf16_t256_s256_h64", 1, 700, 6, 64, 256, 1, 256, init_state=True),
    Workload("bf16_t256_s256_h64_4heads_per_cta", 2, 512, 8, 64, 256, 2, 256),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_full_compare(w):
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert rel_err(np64(y), r["y"]) <= TOL[w.dtype]
    assert rel_err(np64(fin), r["final_state"]) <= TOL[w.dtype]


# The forward pass may run another chunk than the caller's (the result does
# not depend on it); each forced chunk on shapes where it is not the given one.
CHUNK_SHAPES = [w for w in SMALL if w.dtype == "bf16"]


@pytest.mark.parametrize("chunk", ["given", "64", "128", "256"])
@pytest.mark.parametrize("w", CHUNK_SHAPES, ids=[w.name for w in CHUNK_SHAPES])
def test_forward_pass_chunk_override(w, chunk, monkeypatch):
    monkeypatch.setenv("MAMBA2_FWD_CHUNK", chunk)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert rel_err(np64(y), r["y"]) <= TOL[w.dtype]
    assert rel_err(np64(fin), r["final_state"]) <= TOL[w.dtype]


@pytest.mark.parametrize("name,chunk", [("tiny_fp32", None), ("mamba2_1p3b_layer", None),
                                        ("long_seq_carried_state", None), ("large_state", None),
                                        ("blog_example", None), ("long_seq_fp32_t128", None),
                                        # the caller's chunk (256) rather than the pass's own
                                        ("long_seq_carried_state", "given"), ("mamba2_1p3b_layer", "given")])
def test_named_workload_full_size(name, chunk, monkeypatch):
    if chunk:
        monkeypatch.setenv("MAMBA2_FWD_CHUNK", chunk)
    w = WORKLOADS[name]
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    pairs = sample_pairs(w.batch, w.nheads, 6, seed=1)
    ref = oracle_pairs(inp, pairs)
    y_c, fin_c = y.cpu(), fin.cpu()
    ys = np.stack([np64(y_c[b, :, h]) for b, h in pairs])
    yr = np.stack([ref[p][0] for p in pairs])
    fs = np.stack([np64(fin_c[b, h]) for b, h in pairs])
    fr = np.stack([ref[p][1] for p in pairs])
    assert rel_err(ys, yr) <= TOL[w.dtype]
    assert rel_err(fs, fr) <= TOL[w.dtype]
    assert torch.isfinite(y.float()).all()


def test_causality_is_exact():
    w = Workload("causal", 1, 512, 2, 64, 128, 1, 256, init_state=True)
    inp = make_inputs(w)
    base, _ = _fwd(to_dev(inp), w)
    for tp in (5, 255, 256, 400):
        q = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
        q["x"][:, tp] += 1.0
        q["B"][:, tp] -= 0.5
        q["C"][:, tp] *= 2.0
        q["dt"][:, tp] += 0.05
        y, _ = _fwd(to_dev(q), w)
        assert torch.equal(y[:, :tp], base[:, :tp]), tp
        assert not torch.equal(y[:, tp], base[:, tp])


def test_equal_heads_give_equal_outputs():
    w = Workload("heads", 2, 384, 4, 64, 64, 1, 128, init_state=True)
    inp = make_inputs(w)
    for k in ("x", "dt"):
        inp[k][:, :, 3] = inp[k][:, :, 1]
    inp["A"][3] = inp["A"][1]
    inp["D"][3] = inp["D"][1]
    inp["initial_state"][:, 3] = inp["initial_state"][:, 1]
    y, fin = _fwd(to_dev(inp), w)
    assert torch.equal(y[:, :, 3], y[:, :, 1])
    assert torch.equal(fin[:, 3], fin[:, 1])


def test_dt_zero_keeps_state_exactly():
    w = Workload("dt0", 2, 512, 4, 64, 128, 1, 256, init_state=True)
    inp = make_inputs(w)
    inp["dt"].zero_()
    d = to_dev(inp)
    _, fin = _fwd(d, w)
    assert torch.equal(fin, d["initial_state"])


def test_split_sequence_handoff():
    w = Workload("split", 2, 1024, 4, 64, 128, 1, 256, init_state=True)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    L1 = 512
    first = {k: (v[:, :L1].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    y1, f1 = _fwd(first, w)
    second = {k: (v[:, L1:].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    second["initial_state"] = f1
    y2, f2 = _fwd(second, w)
    assert rel_err(np64(torch.cat([y1, y2], 1)), np64(y)) <= TOL["bf16"]
    assert rel_err(np64(f2), np64(fin)) <= TOL["bf16"]


def test_empty_sequence_copies_state():
    w = Workload("empty", 2, 0, 4, 64, 128, 1, 256, init_state=True)
    d = to_dev(make_inputs(w))
    y, fin = _fwd(d, w)
    assert y.numel() == 0
    assert torch.equal(fin, d["initial_state"])
    w0 = w.with_(init_state=False)
    d0 = to_dev(make_inputs(w0))
    _, fin0 = _fwd(d0, w0)
    assert not fin0.any()


def test_empty_batch_is_a_no_op():
    w = Workload("nobatch", 0, 256, 4, 64, 128, 1, 256)
    d = to_dev(make_inputs(w))
    y, fin = _fwd(d, w)
    assert y.numel() == 0 and fin.numel() == 0


def test_misaligned_device_pointer_rejected():
    w = Workload("mis", 1, 256, 2, 64, 64, 1, 128)
    d = to_dev(make_inputs(w))
    flat = torch.empty(d["x"].numel() + 1, dtype=d["x"].dtype, device="cuda")
    x_off = flat[1:].view(d["x"].shape)  # 2-byte offset
    with pytest.raises(bd.Mamba2Error) as e:
        bd.mamba2_ssd_fwd(x_off, d["dt"], d["A"], d["B"], d["C"], w.chunk_size)
    assert e.value.code == 1


def _sweep_ids():
    from mamba_chunked_ssd_gb300.synthetic import sweep_workloads
    return sweep_workloads(seeds=(0, 1, 2))


SWEEP = _sweep_ids()


@pytest.mark.parametrize("w", SWEEP, ids=[f"{w.name}_seed{w.seed}" for w in SWEEP])
def test_sweep_shape_sampled(w):
    """Every point of the bf16 sweep (L, S, H, T) at seeds 0-2, full size, with
    inputs drawn on the GPU; four (batch, head) pairs per point, always the
    first and the last, are checked against the fp64 recurrence."""
    inp = make_inputs(w, device="cuda")
    y, fin = _fwd(inp, w)
    pairs = sample_pairs(w.batch, w.nheads, 4, seed=w.seqlen + 1000 * w.seed + w.dstate + w.headdim + w.chunk_size)
    ref = oracle_pairs(inp, pairs)
    bi = torch.tensor([b for b, _ in pairs], device="cuda")
    hi = torch.tensor([h for _, h in pairs], device="cuda")
    ys = y[bi, :, hi].cpu()
    fs = fin[bi, hi].cpu()
    for i, p in enumerate(pairs):
        assert rel_err(np64(ys[i]), ref[p][0]) <= TOL[w.dtype], p
        assert rel_err(np64(fs[i]), ref[p][1]) <= TOL[w.dtype], p
    assert torch.isfinite(y.float()).all()


# Shapes that take the tensor-core kernels of every stage.
TC_SHAPES = [
    Workload("tc_t256_h64", 2, 640, 4, 64, 128, 1, 256, init_state=True),
    Workload("tc_t128_h128_s256_g2", 1, 384, 4, 128, 256, 2, 128, init_state=True),
    Workload("tc_t128_h64_s64_ragged", 2, 333, 6, 64, 64, 3, 128, init_state=True),
    Workload("tc_t64_h64_odd_chunks", 2, 300, 4, 64, 128, 1, 64, init_state=True),
]


@pytest.mark.parametrize("w", TC_SHAPES, ids=[w.name for w in TC_SHAPES])
def test_optional_pointers_null(w):
    """D = NULL (no skip term) and final_state = NULL (not written) on the
    tensor-core path, each against the oracle."""
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=None,
                               initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=None,
                              init=inp["initial_state"])
    assert rel_err(np64(y), r["y"]) <= TOL[w.dtype]
    assert rel_err(np64(fin), r["final_state"]) <= TOL[w.dtype]
    y2, none = bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                                 initial_state=d["initial_state"], want_final_state=False)
    bd.mamba2_check_device_status()
    assert none is None
    r2 = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                               init=inp["initial_state"])
    assert rel_err(np64(y2), r2["y"]) <= TOL[w.dtype]


# Per-head decay rates cycled over the heads: mild heads keep every row of a
# 32-row quadrant inside the split-decay range; the strong ones put the later
# rows of each quadrant past it (a mixed warp), and the strongest make almost
# every row take the direct per-entry weight, with decays that underflow.
STRONG_SHAPES = [
    Workload("strong_t256_h64", 2, 768, 6, 64, 128, 1, 256, init_state=True),
    Workload("strong_t128_h64", 1, 512, 6, 64, 64, 2, 128, init_state=True),
    Workload("strong_t128_h128_s256", 1, 384, 6, 128, 256, 3, 128, init_state=True),
    Workload("strong_t256_ragged", 1, 650, 6, 64, 128, 1, 256),
    Workload("strong_t64_h64", 1, 500, 6, 64, 128, 2, 64, init_state=True),
]


@pytest.mark.parametrize("w", STRONG_SHAPES, ids=[w.name for w in STRONG_SHAPES])
def test_strong_decay_rows(w):
    """Decays far beyond the chunk-internal split range (A down to -1200, so a
    quadrant spans hundreds of log2 units), compared element by element with
    the fp64 recurrence: the direct-weight rows, the mixed warps and the
    weight clamp are all exercised."""
    inp = strong_decay(make_inputs(w))
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert torch.isfinite(y.float()).all()
    assert rel_err(np64(y), r["y"]) <= TOL[w.dtype]
    assert rel_err(np64(fin), r["final_state"]) <= TOL[w.dtype]
    # per head as well: the strong heads' outputs are small, so a slip there
    # would hide under the mild heads' scale
    for h in range(w.nheads):
        assert rel_err(np64(y[:, :, h]), r["y"][:, :, h]) <= TOL[w.dtype], h


GUARD_SHAPES = [
    Workload("guard_fp32_ragged", 2, 150, 4, 32, 32, 2, 32, dtype="fp32", init_state=True),
    Workload("guard_bf16_t256_ragged", 1, 777, 3, 64, 128, 1, 256, init_state=True),
    Workload("guard_bf16_t128_h128", 2, 200, 4, 128, 256, 2, 128),
    Workload("guard_bf16_t64", 1, 320, 2, 64, 128, 1, 64, init_state=True),
    # few (batch, head) pairs: the state pass runs over sequence segments
    Workload("guard_bf16_segments", 1, 2048, 2, 64, 128, 1, 128, init_state=True),
]


@pytest.mark.parametrize("w", GUARD_SHAPES, ids=[w.name for w in GUARD_SHAPES])
def test_outputs_stay_inside_their_buffers(w):
    """Every output and the workspace sit between guard regions filled with a
    byte pattern; after the pass (and after each stage entry point) the guards
    are unchanged and the result still matches the oracle."""
    inp = make_inputs(w)
    d = to_dev(inp)
    shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
    y = Guarded(d["x"].shape, d["x"].dtype)
    fin = Guarded((w.batch, w.nheads, w.dstate, w.headdim), torch.float32)
    ws = Guarded((bd.mamba2_ssd_fwd_workspace_size(shape),), torch.uint8)
    bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                      initial_state=d["initial_state"], y=y.t, final_state=fin.t, workspace=ws.t)
    bd.mamba2_check_device_status()
    assert y.intact() and fin.intact() and ws.intact()
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert rel_err(np64(y.t), r["y"]) <= TOL[w.dtype]
    assert rel_err(np64(fin.t), r["final_state"]) <= TOL[w.dtype]
    G = Guarded((w.batch, w.nheads, w.seqlen), torch.float32)
    cs = Guarded((w.batch, w.nheads, w.nchunks, w.dstate, w.headdim), d["x"].dtype)
    fin2 = Guarded((w.batch, w.nheads, w.dstate, w.headdim), torch.float32)
    y2 = Guarded(d["x"].shape, d["x"].dtype)
    bd.mamba2_chunk_cumsum(d["dt"], d["A"], w.chunk_size, G=G.t)
    bd.mamba2_state_pass(d["x"], d["dt"], d["B"], G.t, w.chunk_size, initial_state=d["initial_state"],
                         chunk_states=cs.t, final_state=fin2.t)
    bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], G.t, cs.t, w.chunk_size, D=d["D"], y=y2.t)
    bd.mamba2_check_device_status()
    assert G.intact() and cs.intact() and fin2.intact() and y2.intact()
    assert rel_err(np64(y2.t), r["y"]) <= TOL[w.dtype]


# Stage 3 with one row block per chunk runs one CTA per SM, each taking an
# equal share of the (batch, chunk, virtual head) triples and running it as
# items of consecutive heads of one chunk and group.  These shares start and
# end inside chunks and inside groups; a 128-wide head is two virtual heads,
# so a share may start at its second half; chunks of 64 run in pairs; the
# sequences end ragged.
SHARE_SHAPES = [
    Workload("share_h128_groups_ragged", 2, 33 * 128 - 37, 24, 128, 128, 3, 128, init_state=True),
    Workload("share_h64_groups", 3, 20 * 128 + 5, 40, 64, 128, 5, 128, init_state=True),
    Workload("share_t64_pairs", 3, 41 * 64 - 9, 36, 64, 64, 3, 64, init_state=True),
]


@pytest.mark.parametrize("w", SHARE_SHAPES, ids=[w.name for w in SHARE_SHAPES])
def test_persistent_shares(w, monkeypatch):
    """Sampled (batch, head) pairs against the fp64 recurrence, and the same
    pass with one CTA per work item gives the same y bit for bit (each head's
    products and epilogue do not depend on which CTA runs them)."""
    monkeypatch.setenv("MAMBA2_FWD_CHUNK", "given")
    inp = make_inputs(w, device="cuda")
    y, fin = _fwd(inp, w)
    pairs = sample_pairs(w.batch, w.nheads, 12, seed=3)
    ref = oracle_pairs(inp, pairs)
    for (b, h) in pairs:
        ry, rs = ref[(b, h)]
        assert rel_err(np64(y[b, :, h]), ry) <= TOL[w.dtype], (b, h)
        assert rel_err(np64(fin[b, h]), rs) <= TOL[w.dtype], (b, h)
    monkeypatch.setenv("MAMBA2_CHUNK_OUT_PERSISTENT", "0")
    y0, fin0 = _fwd(inp, w)
    assert torch.equal(y, y0) and torch.equal(fin, fin0)


def test_more_chunks_than_a_grid_y_dimension():
    """65 600 chunks of 128 tokens (8.4 M tokens, ragged end): more chunks than
    a grid's y or z dimension holds.  The carried state forgets a prefix of
    thousands of tokens (sum of A dt over 4096 tokens is about -245 here), so
    the last 1024 outputs and the final state equal, to far below the
    tolerance, the recurrence run from a zero state over the last 5120
    tokens alone; the same holds for a window just past chunk 65 535."""
    w = Workload("many_chunks", 1, 128 * 65600 - 77, 2, 64, 64, 1, 128)
    inp = make_inputs(w, device="cuda")
    y, fin = _fwd(inp, w)
    assert torch.isfinite(y.float()).all()
    for end in (w.seqlen, 128 * 65537 + 40):
        lo = end - 5120
        sub = {k: (v[:, lo:end] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
        sub["initial_state"] = None
        r = oracle.ssd_recurrence(*(sub[k].cpu() for k in ("x", "dt", "A", "B", "C")), D=sub["D"].cpu())
        assert rel_err(np64(y[:, end - 1024:end]), r["y"][:, -1024:]) <= TOL[w.dtype], end
        if end == w.seqlen:
            assert rel_err(np64(fin), r["final_state"]) <= TOL[w.dtype]


# Few (batch, head) pairs: the forward pass runs stage 2 over sequence
# segments (a summary pass from zero states, the carry of the entering states
# by the jump formula, then every segment from its entering state).  Each
# shape has 4 to 10 segments; ragged ends, chunk 64/128/256, both head widths,
# a 256-wide state (two state tiles), and the decay stress.
SEGMENT_SHAPES = [
    Workload("seg_t128_h64_init", 1, 4096, 2, 64, 128, 1, 128, init_state=True),
    Workload("seg_t256_s64_ragged", 2, 8192 - 77, 2, 64, 64, 1, 256, init_state=True),
    Workload("seg_t64_h128_s256_groups", 1, 3000, 2, 128, 256, 2, 64),
    Workload("seg_t128_h128_s128", 1, 3333, 3, 128, 128, 1, 128, init_state=True),
]


@pytest.mark.parametrize("w", SEGMENT_SHAPES, ids=[w.name for w in SEGMENT_SHAPES])
def test_sequence_segments(w):
    """y and the final state against the fp64 recurrence, in full."""
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert rel_err(np64(y), r["y"]) <= TOL[w.dtype]
    assert rel_err(np64(fin), r["final_state"]) <= TOL[w.dtype]


@pytest.mark.parametrize("w", [w for w in SEGMENT_SHAPES if w.headdim == 64] +
                         [Workload("seg_pairs_groups_strong", 1, 3000, 4, 64, 128, 2, 128, init_state=True)],
                         ids=lambda w: w.name)
def test_sequence_segments_head_pairs(w, monkeypatch):
    """The summary and segment passes with heads of 64 columns in pairs (each
    half's entering and end states in its own head's rows) give the same y and
    final state as single heads, bit for bit, also under strong decay."""
    inp = strong_decay(make_inputs(w)) if "strong" in w.name else make_inputs(w)
    d = to_dev(inp)
    monkeypatch.setenv("MAMBA2_STATE_PAIRS", "0")
    y0, fin0 = _fwd(d, w)
    monkeypatch.setenv("MAMBA2_STATE_PAIRS", "1")
    y1, fin1 = _fwd(d, w)
    assert torch.equal(y0, y1) and torch.equal(fin0, fin1)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert rel_err(np64(y1), r["y"]) <= TOL[w.dtype]


def test_sequence_segments_strong_decay():
    w = Workload("seg_strong", 1, 2048, 6, 64, 128, 1, 128, init_state=True)
    inp = strong_decay(make_inputs(w))
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert torch.isfinite(y.float()).all()
    for h in range(w.nheads):
        assert rel_err(np64(y[:, :, h]), r["y"][:, :, h]) <= TOL[w.dtype], h
        assert rel_err(np64(fin[:, h]), r["final_state"][:, h]) <= TOL[w.dtype], h


def test_sequence_segments_match_one_pass():
    """The segmented forward pass and the stage entry points (stage 2 in one
    pass over each sequence) give the same outputs up to rounding: both are
    within the tolerance of the oracle and within it of each other."""
    w = Workload("seg_vs_stages", 2, 4096, 2, 64, 128, 1, 256, init_state=True)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    G = bd.mamba2_chunk_cumsum(d["dt"], d["A"], w.chunk_size)
    cs, fin1 = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], G, w.chunk_size, initial_state=d["initial_state"])
    y1 = bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], G, cs, w.chunk_size, D=d["D"])
    bd.mamba2_check_device_status()
    assert rel_err(np64(y), np64(y1)) <= TOL[w.dtype]
    assert rel_err(np64(fin), np64(fin1)) <= TOL[w.dtype]


def test_sequence_segments_override_gives_one_pass(monkeypatch):
    """MAMBA2_STATE_SEGMENTS=1 (one pass over each sequence) and the default
    (segments) agree within the tolerance, and both match the oracle."""
    w = Workload("seg_override", 1, 4096, 2, 64, 128, 1, 128, init_state=True)
    inp = make_inputs(w)
    d = to_dev(inp)
    y_seg, fin_seg = _fwd(d, w)
    monkeypatch.setenv("MAMBA2_STATE_SEGMENTS", "1")
    y_one, fin_one = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    for y, fin in ((y_seg, fin_seg), (y_one, fin_one)):
        assert rel_err(np64(y), r["y"]) <= TOL[w.dtype]
        assert rel_err(np64(fin), r["final_state"]) <= TOL[w.dtype]
    assert rel_err(np64(y_seg), np64(y_one)) <= TOL[w.dtype]


# fp32 problems with chunks of 128, head dim 64 or 128 and state 64 or 128
# run stage 3 on the tensor cores with split-bf16 operands (three products per
# product); each is compared in full with the fp64 recurrence at the fp32
# tolerance, and with the CUDA-core path.
F32_TC_SHAPES = [
    Workload("fp32_tc_h64_s128_groups", 2, 384, 4, 64, 128, 2, 128, dtype="fp32", init_state=True),
    Workload("fp32_tc_h128_s64_ragged", 1, 333, 3, 128, 64, 1, 128, dtype="fp32", init_state=True),
    Workload("fp32_tc_32_heads", 1, 256, 32, 64, 64, 1, 128, dtype="fp32"),
    Workload("fp32_tc_h128_s128", 2, 300, 2, 128, 128, 2, 128, dtype="fp32", init_state=True),
    # other chunks: the forward pass runs these at chunk 128 on the tensor cores
    Workload("fp32_tc_given_t256", 1, 600, 4, 64, 128, 1, 256, dtype="fp32", init_state=True),
    Workload("fp32_tc_given_t64", 2, 200, 2, 128, 64, 2, 64, dtype="fp32"),
]


@pytest.mark.parametrize("w", F32_TC_SHAPES, ids=[w.name for w in F32_TC_SHAPES])
def test_fp32_tensor_core_path(w, monkeypatch):
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert rel_err(np64(y), r["y"]) <= TOL["fp32"]
    assert rel_err(np64(fin), r["final_state"]) <= TOL["fp32"]
    for h in range(w.nheads):
        assert rel_err(np64(y[:, :, h]), r["y"][:, :, h]) <= TOL["fp32"], h
    monkeypatch.setenv("MAMBA2_FP32_PATH", "simt")
    y_simt, _ = _fwd(d, w)
    assert rel_err(np64(y), np64(y_simt)) <= TOL["fp32"]


def test_fp32_tensor_core_path_strong_decay():
    w = Workload("fp32_tc_strong", 1, 512, 6, 64, 128, 1, 128, dtype="fp32", init_state=True)
    inp = strong_decay(make_inputs(w))
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert torch.isfinite(y).all()
    for h in range(w.nheads):
        assert rel_err(np64(y[:, :, h]), r["y"][:, :, h]) <= TOL["fp32"], h
    assert rel_err(np64(fin), r["final_state"]) <= TOL["fp32"]


def test_fp32_tensor_core_path_stays_in_its_buffers():
    w = Workload("fp32_tc_guard", 1, 300, 4, 64, 128, 2, 128, dtype="fp32", init_state=True)
    inp = make_inputs(w)
    d = to_dev(inp)
    shape = bd.shape_of(d["x"], d["B"], w.chunk_size)
    y = Guarded(d["x"].shape, d["x"].dtype)
    fin = Guarded((w.batch, w.nheads, w.dstate, w.headdim), torch.float32)
    ws = Guarded((bd.mamba2_ssd_fwd_workspace_size(shape),), torch.uint8)
    bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                      initial_state=d["initial_state"], y=y.t, final_state=fin.t, workspace=ws.t)
    bd.mamba2_check_device_status()
    assert y.intact() and fin.intact() and ws.intact()
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert rel_err(np64(y.t), r["y"]) <= TOL["fp32"]
