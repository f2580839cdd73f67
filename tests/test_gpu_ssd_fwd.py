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

from gpu_helpers import TOL, np64, oracle_pairs, rel_err, sample_pairs, to_dev
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


@pytest.mark.parametrize("name", ["tiny_fp32", "mamba2_1p3b_layer", "long_seq_carried_state",
                                  "large_state"])
def test_named_workload_full_size(name):
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


def _sweep_cover():
    """One sweep shape for every (S, H, T) combination; the sequence lengths
    rotate so that each (H, T) pair meets three of the four lengths and each
    length appears three times."""
    from mamba_chunked_ssd_gb300.synthetic import sweep_workloads
    by_name = {w.name: w for w in sweep_workloads(seeds=(0,))}
    Ls = (1024, 4096, 16384, 32768)
    combos = [(S, H, T) for S in (64, 128, 256) for H in (64, 128) for T in (128, 256)]
    return [by_name[f"sweep_L{Ls[(i + i // 4) % 4]}_S{S}_H{H}_T{T}"] for i, (S, H, T) in enumerate(combos)]


SWEEP = _sweep_cover()


@pytest.mark.parametrize("w", SWEEP, ids=[w.name for w in SWEEP])
def test_sweep_shape_sampled(w):
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = _fwd(d, w)
    pairs = sample_pairs(w.batch, w.nheads, 3, seed=w.seqlen)
    ref = oracle_pairs(inp, pairs)
    y_c, fin_c = y.cpu(), fin.cpu()
    for b, h in pairs:
        assert rel_err(np64(y_c[b, :, h]), ref[(b, h)][0]) <= TOL[w.dtype], (b, h)
        assert rel_err(np64(fin_c[b, h]), ref[(b, h)][1]) <= TOL[w.dtype], (b, h)
    assert torch.isfinite(y.float()).all()
