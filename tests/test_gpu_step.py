"""GPU parity of the decode step mamba2_ssd_step against the fp64 oracle.

Shapes cover both thread layouts (H a multiple of 4 and not), the largest
state (S = H = 256), groups, fp32 and bf16, a missing D and a zero initial
state.  The hand-off case runs mamba2_ssd_fwd over a prefix and then decode
steps in place, against the recurrence over the whole sequence.  Exact
properties: in place == out of place bit for bit, dt = 0 leaves the state
unchanged.
"""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, np64, rel_err, to_dev
import oracle
from mamba_chunked_ssd_gb300 import binding as bd
from mamba_chunked_ssd_gb300.synthetic import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mamba_chunked_ssd_gb300 import build_lib
    build_lib.build()
    bd.load_library()


def step_inputs(w: Workload, seed=None):
    """The workload's seeded inputs for one token, in the step's layouts."""
    inp = make_inputs(dataclasses.replace(w, seqlen=1), seed=seed)
    return {"x": inp["x"][:, 0].contiguous(), "dt": inp["dt"][:, 0].contiguous(), "A": inp["A"],
            "B": inp["B"][:, 0].contiguous(), "C": inp["C"][:, 0].contiguous(), "D": inp["D"],
            "state": inp["initial_state"]}


STEP_SHAPES = [
    Workload("bf16_s128_h64", 3, 1, 8, 64, 128, 1, 1, init_state=True),
    Workload("bf16_s64_h128_groups", 2, 1, 8, 128, 64, 4, 1, init_state=True),
    Workload("bf16_s256_h256", 2, 1, 2, 256, 256, 2, 1, init_state=True),
    Workload("fp32_h30_odd_cols", 2, 1, 4, 30, 16, 2, 1, dtype="fp32", init_state=True),
    Workload("fp32_s7_h5", 1, 1, 3, 5, 7, 1, 1, dtype="fp32", init_state=True),
    Workload("bf16_zero_state", 4, 1, 4, 64, 128, 2, 1),
]


@pytest.mark.parametrize("w", STEP_SHAPES, ids=[w.name for w in STEP_SHAPES])
def test_step_matches_oracle(w):
    s = step_inputs(w)
    d = to_dev(s)
    y, h = bd.mamba2_ssd_step(d["x"], d["dt"], d["A"], d["B"], d["C"], state_in=d["state"], D=d["D"])
    bd.mamba2_check_device_status()
    y_ref, h_ref = oracle.ssd_step(s["x"], s["dt"], s["A"], s["B"], s["C"], state=s["state"], D=s["D"])
    assert rel_err(np64(y), y_ref) <= TOL[w.dtype]
    assert rel_err(np64(h), h_ref) <= TOL["fp32"]  # the state is carried in fp32 on both paths


def test_step_without_skip_term():
    w = STEP_SHAPES[0]
    s = step_inputs(w)
    d = to_dev(s)
    y, _ = bd.mamba2_ssd_step(d["x"], d["dt"], d["A"], d["B"], d["C"], state_in=d["state"])
    y_ref, _ = oracle.ssd_step(s["x"], s["dt"], s["A"], s["B"], s["C"], state=s["state"])
    assert rel_err(np64(y), y_ref) <= TOL[w.dtype]


def test_prefill_then_decode_in_place():
    """mamba2_ssd_fwd over 300 tokens, then 5 in-place steps, against the
    recurrence over all 305 tokens."""
    w = Workload("handoff", 2, 305, 8, 64, 128, 2, 128, init_state=True)
    inp = make_inputs(w)
    d = to_dev(inp)
    P = 300
    _, state = bd.mamba2_ssd_fwd(d["x"][:, :P].contiguous(), d["dt"][:, :P].contiguous(), d["A"],
                                 d["B"][:, :P].contiguous(), d["C"][:, :P].contiguous(), w.chunk_size,
                                 D=d["D"], initial_state=d["initial_state"])
    ys = []
    for t in range(P, w.seqlen):
        y, _ = bd.mamba2_ssd_step(d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["A"],
                                  d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), state_in=state,
                                  D=d["D"], state_out=state)
        ys.append(np64(y))
    bd.mamba2_check_device_status()
    ref = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                                init=inp["initial_state"])
    assert rel_err(np.stack(ys, axis=1), ref["y"][:, P:]) <= TOL["bf16"]
    assert rel_err(np64(state), ref["final_state"]) <= TOL["bf16"]


def test_in_place_equals_out_of_place():
    w = STEP_SHAPES[1]
    d = to_dev(step_inputs(w))
    y1, h1 = bd.mamba2_ssd_step(d["x"], d["dt"], d["A"], d["B"], d["C"], state_in=d["state"], D=d["D"])
    st = d["state"].clone()
    y2, h2 = bd.mamba2_ssd_step(d["x"], d["dt"], d["A"], d["B"], d["C"], state_in=st, D=d["D"], state_out=st)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(h1, h2)


def test_dt_zero_keeps_state_exactly():
    w = STEP_SHAPES[2]
    s = step_inputs(w)
    s["dt"] = torch.zeros_like(s["dt"])
    d = to_dev(s)
    y, h = bd.mamba2_ssd_step(d["x"], d["dt"], d["A"], d["B"], d["C"], state_in=d["state"], D=d["D"])
    torch.cuda.synchronize()
    assert torch.equal(h, d["state"])
    y_ref, _ = oracle.ssd_step(s["x"], s["dt"], s["A"], s["B"], s["C"], state=s["state"], D=s["D"])
    assert rel_err(np64(y), y_ref) <= TOL[w.dtype]


def test_step_equals_one_token_forward_pass():
    """The step and mamba2_ssd_fwd on a one-token sequence compute the same thing."""
    w = STEP_SHAPES[0]
    inp = make_inputs(dataclasses.replace(w, seqlen=1, chunk_size=128))
    d = to_dev(inp)
    y_f, h_f = bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], 128, D=d["D"],
                                 initial_state=d["initial_state"])
    y_s, h_s = bd.mamba2_ssd_step(d["x"][:, 0].contiguous(), d["dt"][:, 0].contiguous(), d["A"],
                                  d["B"][:, 0].contiguous(), d["C"][:, 0].contiguous(),
                                  state_in=d["initial_state"], D=d["D"])
    torch.cuda.synchronize()
    assert rel_err(np64(y_s), np64(y_f[:, 0])) <= TOL["bf16"]
    assert rel_err(np64(h_s), np64(h_f)) <= TOL["bf16"]


def test_empty_batch_is_a_no_op():
    x = torch.empty(0, 4, 64, device="cuda", dtype=torch.bfloat16)
    dt = torch.empty(0, 4, device="cuda")
    A = torch.full((4,), -1.0, device="cuda")
    B = torch.empty(0, 1, 128, device="cuda", dtype=torch.bfloat16)
    y, h = bd.mamba2_ssd_step(x, dt, A, B, B.clone())
    torch.cuda.synchronize()
    assert y.shape == (0, 4, 64) and h.shape == (0, 4, 128, 64)
