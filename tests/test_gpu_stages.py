"""Per-stage GPU parity: each C-ABI stage against the fp64 oracle, fed the
same inputs (the oracle's own intermediates where a stage needs them).

Stage 1 (chunk_cumsum): |G - G_ref| <= 1e-5 max(1, |G_ref|), plus a bit-exact
layout check.  Stages 2 and 3: max|err| / max|ref| <= 2e-2 (bf16) / 1e-4
(fp32), plus the exact special cases (dt = 0, B = C = 0, chunk 0's state).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, np64, rel_err, strong_decay, to_dev
from mamba_chunked_ssd_gb300 import binding as bd
from mamba_chunked_ssd_gb300.synthetic import Workload, make_inputs

pytestmark = pytest.mark.gpu

# name, b, L, nh, H, S, G, T, dtype, init
SHAPES = [
    ("fp32_tiny", 1, 256, 2, 16, 16, 1, 64, "fp32", False),
    ("fp32_ragged", 2, 203, 3, 16, 32, 1, 64, "fp32", True),
    ("fp32_small_chunk", 1, 100, 4, 32, 16, 2, 16, "fp32", True),
    # fp32 chunks of 128: stage 3 runs the split-bf16 tensor-core kernel
    ("fp32_t128_tc", 2, 300, 4, 64, 128, 2, 128, "fp32", True),
    ("fp32_t128_h128_s64", 1, 256, 2, 128, 64, 1, 128, "fp32", False),
    ("bf16_t128", 2, 384, 4, 64, 64, 2, 128, "bf16", True),
    ("bf16_t256", 1, 512, 3, 64, 128, 1, 256, "bf16", True),
    ("bf16_t256_ragged", 2, 700, 2, 64, 128, 1, 256, "bf16", False),
    ("bf16_h128_s256", 1, 256, 4, 128, 256, 2, 128, "bf16", True),
    ("bf16_t128_ragged", 1, 333, 4, 128, 64, 4, 128, "bf16", True),
    # chunks of 64 run in pairs in the tensor-core output kernel: an even and
    # an odd chunk count (the last pair then holds one chunk), 128-wide heads
    ("bf16_t64_pairs", 2, 384, 4, 64, 128, 2, 64, "bf16", True),
    ("bf16_t64_odd_chunks", 1, 300, 3, 64, 64, 1, 64, "bf16", False),
    ("bf16_t64_h128_s256", 1, 256, 4, 128, 256, 2, 64, "bf16", True),
]


def _w(name, b, L, nh, H, S, G, T, dtype, init, seed=0):
    return Workload(name, b, L, nh, H, S, G, T, dtype=dtype, init_state=init, seed=seed)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mamba_chunked_ssd_gb300 import build_lib
    build_lib.build()
    bd.load_library()


@pytest.mark.parametrize("spec", SHAPES, ids=[s[0] for s in SHAPES])
def test_chunk_cumsum_matches_oracle(spec):
    w = _w(*spec)
    inp = make_inputs(w)
    d = to_dev(inp)
    G = bd.mamba2_chunk_cumsum(d["dt"], d["A"], w.chunk_size)
    bd.mamba2_check_device_status()
    Gref = oracle.chunk_cumsum(inp["dt"], inp["A"], w.chunk_size)
    err = np.abs(np64(G) - Gref) / np.maximum(1.0, np.abs(Gref))
    assert err.max() <= 1e-5, err.max()


@pytest.mark.parametrize("nh", [37, 36, 64])
def test_chunk_cumsum_bit_exact_layout(nh):
    """With A a power of two and dt on a 2^-12 grid every partial sum is exact
    in fp32, so G = fl(sum * log2e) exactly: any indexing or layout slip shows.
    A head count divisible by 4 takes the 16-byte load path, 37 the scalar one."""
    b, L, T = 2, 300, 64
    g = torch.Generator().manual_seed(5)
    dt = (torch.randint(1, 64, (b, L, nh), generator=g).float() / 4096.0)
    A = torch.tensor([-(2.0 ** (k % 3)) for k in range(nh)], dtype=torch.float32)
    G = bd.mamba2_chunk_cumsum(dt.cuda(), A.cuda(), T).cpu()
    a = (A[None, None, :] * dt).double().numpy()  # exact
    ref = np.zeros((b, nh, L), dtype=np.float32)
    for c0 in range(0, L, T):
        run = np.cumsum(a[:, c0:c0 + T], axis=1)  # exact sums of grid values
        ref[:, :, c0:c0 + T] = (run.astype(np.float32) * np.float32(1.4426950408889634)).transpose(0, 2, 1)
    assert np.array_equal(G.numpy(), ref)


def _oracle_stage_inputs(inp, w):
    """Oracle G rounded to fp32 (what the GPU stages consume) and the oracle's
    chunk states computed from that same G."""
    G32 = oracle.chunk_cumsum(inp["dt"], inp["A"], w.chunk_size).astype(np.float32)
    cs, fin = oracle.state_pass(inp["x"], inp["dt"], inp["B"], G32, w.chunk_size,
                                init=inp["initial_state"])
    return G32, cs, fin


@pytest.mark.parametrize("spec", SHAPES, ids=[s[0] for s in SHAPES])
def test_state_pass_matches_oracle(spec):
    w = _w(*spec)
    inp = make_inputs(w)
    d = to_dev(inp)
    G32, cs_ref, fin_ref = _oracle_stage_inputs(inp, w)
    cs, fin = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], torch.from_numpy(G32).cuda(),
                                   w.chunk_size, initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    tol = TOL[w.dtype]
    assert rel_err(np64(cs), cs_ref) <= tol
    assert rel_err(np64(fin), fin_ref) <= tol


@pytest.mark.parametrize("spec", SHAPES, ids=[s[0] for s in SHAPES])
def test_chunk_out_matches_oracle(spec):
    w = _w(*spec)
    inp = make_inputs(w)
    d = to_dev(inp)
    G32, cs_ref, _ = _oracle_stage_inputs(inp, w)
    cs_dev = torch.from_numpy(cs_ref).to(d["x"].dtype).cuda()  # rounded like stored states
    y = bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], torch.from_numpy(G32).cuda(), cs_dev,
                            w.chunk_size, D=d["D"])
    bd.mamba2_check_device_status()
    y_ref = oracle.chunk_out(inp["x"], inp["dt"], inp["B"], inp["C"], G32, cs_dev.cpu(), w.chunk_size,
                             D=inp["D"])
    assert rel_err(np64(y), y_ref) <= TOL[w.dtype]


# Heads of 64 columns run in pairs in the state pass (two heads of one group
# per CTA, as one head of 128 columns) where there are enough (batch, head)
# pairs; MAMBA2_STATE_PAIRS=1 forces the pairs on these small shapes: chunks
# of 64, 128 and 256, states of 64, 128 and 256, ragged ends, groups of two
# and four heads, with and without a carried state.
PAIR_SHAPES = [
    ("pairs_t128_s128_init", 2, 640, 4, 64, 128, 1, 128, "bf16", True),
    ("pairs_t256_s64_groups_ragged", 1, 777, 8, 64, 64, 2, 256, "bf16", False),
    ("pairs_t64_s256_groups_init", 1, 300, 6, 64, 256, 3, 64, "bf16", True),
]


@pytest.mark.parametrize("spec", PAIR_SHAPES, ids=[s[0] for s in PAIR_SHAPES])
def test_state_pass_head_pairs(spec, monkeypatch):
    """Chunk states and final state against the oracle, and equal bit for bit
    to one head per CTA: each element of the pair's product, fold and scan
    takes the same operations in the same order as for a single head."""
    w = _w(*spec)
    inp = make_inputs(w)
    d = to_dev(inp)
    G32, cs_ref, fin_ref = _oracle_stage_inputs(inp, w)
    G = torch.from_numpy(G32).cuda()
    monkeypatch.setenv("MAMBA2_STATE_PAIRS", "1")
    cs, fin = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], G, w.chunk_size, initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    assert rel_err(np64(cs), cs_ref) <= TOL[w.dtype]
    assert rel_err(np64(fin), fin_ref) <= TOL[w.dtype]
    monkeypatch.setenv("MAMBA2_STATE_PAIRS", "0")
    cs1, fin1 = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], G, w.chunk_size, initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    assert torch.equal(cs, cs1) and torch.equal(fin, fin1)


@pytest.mark.parametrize("spec", [s for s in SHAPES if s[-1]], ids=[s[0] for s in SHAPES if s[-1]])
def test_state_pass_exact_cases(spec):
    """dt = 0 leaves the state untouched (exp2(0) = 1, added terms exactly 0),
    and chunk 0's stored state is the initial state rounded to dtype."""
    w = _w(*spec)
    inp = make_inputs(w)
    d = to_dev(inp)
    zero_dt = torch.zeros_like(d["dt"])
    G = bd.mamba2_chunk_cumsum(zero_dt, d["A"], w.chunk_size)
    cs, fin = bd.mamba2_state_pass(d["x"], zero_dt, d["B"], G, w.chunk_size,
                                   initial_state=d["initial_state"])
    assert torch.equal(fin, d["initial_state"])
    G = bd.mamba2_chunk_cumsum(d["dt"], d["A"], w.chunk_size)
    cs, _ = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], G, w.chunk_size,
                                 initial_state=d["initial_state"])
    assert torch.equal(cs[:, :, 0], d["initial_state"].to(cs.dtype))


@pytest.mark.parametrize("spec", SHAPES, ids=[s[0] for s in SHAPES])
def test_chunk_out_skip_only_is_exact(spec):
    """B = C = 0 leaves only the skip term: y = fl(D x), rounded once to dtype."""
    w = _w(*spec)
    inp = make_inputs(w)
    d = to_dev(inp)
    zB = torch.zeros_like(d["B"])
    G = bd.mamba2_chunk_cumsum(d["dt"], d["A"], w.chunk_size)
    cs = torch.randn(w.batch, w.nheads, w.nchunks, w.dstate, w.headdim, device="cuda").to(d["x"].dtype)
    y = bd.mamba2_chunk_out(d["x"], d["dt"], zB, zB, G, cs, w.chunk_size, D=d["D"])
    ref = (d["D"][None, None, :, None] * d["x"].float()).to(d["x"].dtype)
    assert torch.equal(y, ref)


@pytest.mark.parametrize("spec", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("term", ["carried_state_only", "interaction_only"])
def test_chunk_out_single_term(spec, term):
    """One term of the output at a time: x = 0 leaves exp2(G_i) C_i^T h_c
    (the carried-state product); zero states leave the decayed, masked
    interaction term plus the skip."""
    w = _w(*spec)
    inp = make_inputs(w)
    if term == "carried_state_only":
        inp["x"].zero_()
    d = to_dev(inp)
    G32, cs_ref, _ = _oracle_stage_inputs(inp, w)
    if term == "interaction_only":
        cs_ref = np.zeros_like(cs_ref)
    cs_dev = torch.from_numpy(cs_ref).to(d["x"].dtype).cuda()
    y = bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], torch.from_numpy(G32).cuda(), cs_dev,
                            w.chunk_size, D=d["D"])
    bd.mamba2_check_device_status()
    y_ref = oracle.chunk_out(inp["x"], inp["dt"], inp["B"], inp["C"], G32, cs_dev.cpu(), w.chunk_size,
                             D=inp["D"])
    assert rel_err(np64(y), y_ref) <= TOL[w.dtype]


# Tensor-core shapes of stages 2 and 3 (both row blocks of a 256-token chunk,
# both head-dim variants) fed decay rates far beyond the split-decay range.
STRONG = [
    ("strong_t256", 2, 512, 6, 64, 128, 1, 256, "bf16", True),
    ("strong_t128_h128", 1, 384, 6, 128, 256, 2, 128, "bf16", True),
    ("strong_t256_ragged", 1, 600, 6, 64, 64, 3, 256, "bf16", False),
    ("strong_t64_pairs", 1, 448, 6, 64, 128, 1, 64, "bf16", True),
]


@pytest.mark.parametrize("spec", STRONG, ids=[s[0] for s in STRONG])
def test_stages_under_strong_decay(spec):
    """Stage 2 and stage 3 each against the oracle (stage 3 given the oracle's
    states) with decays that leave the split-decay range: the direct-weight
    rows, mixed warps, the weight clamp and underflowing decays all run."""
    w = _w(*spec)
    inp = strong_decay(make_inputs(w))
    d = to_dev(inp)
    G32, cs_ref, fin_ref = _oracle_stage_inputs(inp, w)
    Gd = torch.from_numpy(G32).cuda()
    cs, fin = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], Gd, w.chunk_size, initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    assert rel_err(np64(cs), cs_ref) <= TOL[w.dtype]
    assert rel_err(np64(fin), fin_ref) <= TOL[w.dtype]
    cs_dev = torch.from_numpy(cs_ref).to(d["x"].dtype).cuda()
    y = bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], Gd, cs_dev, w.chunk_size, D=d["D"])
    bd.mamba2_check_device_status()
    y_ref = oracle.chunk_out(inp["x"], inp["dt"], inp["B"], inp["C"], G32, cs_dev.cpu(), w.chunk_size,
                             D=inp["D"])
    assert torch.isfinite(y.float()).all()
    for h in range(w.nheads):
        assert rel_err(np64(y[:, :, h]), y_ref[:, :, h]) <= TOL[w.dtype], h


@pytest.mark.parametrize("spec", [s for s in STRONG if s[4] == 64], ids=[s[0] for s in STRONG if s[4] == 64])
def test_state_pass_head_pairs_strong_decay(spec, monkeypatch):
    """Heads in pairs whose two heads decay at very different rates (each
    pair mixes a mild head with a strong one): each half keeps its own
    weights and decay.  Against the oracle, and bit for bit against single
    heads."""
    w = _w(*spec)
    inp = strong_decay(make_inputs(w))
    d = to_dev(inp)
    G32, cs_ref, fin_ref = _oracle_stage_inputs(inp, w)
    Gd = torch.from_numpy(G32).cuda()
    monkeypatch.setenv("MAMBA2_STATE_PAIRS", "1")
    cs, fin = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], Gd, w.chunk_size, initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    assert rel_err(np64(cs), cs_ref) <= TOL[w.dtype]
    assert rel_err(np64(fin), fin_ref) <= TOL[w.dtype]
    monkeypatch.setenv("MAMBA2_STATE_PAIRS", "0")
    cs1, fin1 = bd.mamba2_state_pass(d["x"], d["dt"], d["B"], Gd, w.chunk_size, initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    assert torch.equal(cs, cs1) and torch.equal(fin, fin1)


# Heads of 128 columns in stage 3: whole (one 128-wide MMA per head) or split
# into two 64-wide virtual heads; the override selects the variant where it
# fits, and both must match the oracle.  State 256 with chunk 256 fits only
# split.
SPLIT = [
    ("h128_t128_s256", 1, 384, 4, 128, 256, 2, 128, "bf16", True),
    ("h128_t256_s128", 2, 512, 2, 128, 128, 1, 256, "bf16", False),
    ("h128_t256_s256_ragged", 1, 700, 3, 128, 256, 1, 256, "bf16", True),
    ("h128_t128_s64_groups", 2, 300, 8, 128, 64, 2, 128, "bf16", True),
    ("h128_t64_s64_pairs", 1, 320, 2, 128, 64, 1, 64, "bf16", True),
]


@pytest.mark.parametrize("variant", ["1", "2"])
@pytest.mark.parametrize("spec", SPLIT, ids=[s[0] for s in SPLIT])
def test_chunk_out_head_split_variants(spec, variant, monkeypatch):
    monkeypatch.setenv("MAMBA2_CHUNK_OUT_HEAD_SPLIT", variant)
    w = _w(*spec)
    inp = make_inputs(w)
    d = to_dev(inp)
    G32, cs_ref, _ = _oracle_stage_inputs(inp, w)
    cs_dev = torch.from_numpy(cs_ref).to(d["x"].dtype).cuda()
    y = bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], torch.from_numpy(G32).cuda(), cs_dev,
                            w.chunk_size, D=d["D"])
    bd.mamba2_check_device_status()
    y_ref = oracle.chunk_out(inp["x"], inp["dt"], inp["B"], inp["C"], G32, cs_dev.cpu(), w.chunk_size,
                             D=inp["D"])
    assert rel_err(np64(y), y_ref) <= TOL[w.dtype]
    for h in range(w.nheads):
        assert rel_err(np64(y[:, :, h]), y_ref[:, :, h]) <= TOL[w.dtype], h


@pytest.mark.parametrize("spec", [s for s in SHAPES if s[8] == "bf16"], ids=[s[0] for s in SHAPES if s[8] == "bf16"])
def test_chunk_out_reads_every_chunk_state(spec):
    """Random chunk states that no state pass would produce (each chunk's
    independent of its neighbours) with x = 0: y is the carried-state term
    alone, so every chunk must use its own state, including the second chunk
    of a pair of 64-token chunks."""
    w = _w(*spec)
    inp = make_inputs(w)
    inp["x"].zero_()
    d = to_dev(inp)
    G32, _, _ = _oracle_stage_inputs(inp, w)
    g = torch.Generator().manual_seed(7)
    cs = torch.randn(w.batch, w.nheads, w.nchunks, w.dstate, w.headdim, generator=g).to(d["x"].dtype)
    y = bd.mamba2_chunk_out(d["x"], d["dt"], d["B"], d["C"], torch.from_numpy(G32).cuda(), cs.cuda(),
                            w.chunk_size, D=d["D"])
    bd.mamba2_check_device_status()
    y_ref = oracle.chunk_out(inp["x"], inp["dt"], inp["B"], inp["C"], G32, cs, w.chunk_size, D=inp["D"])
    assert rel_err(np64(y), y_ref) <= TOL[w.dtype]
