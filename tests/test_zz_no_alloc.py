"""The allocation-free entry point, mamba2_ssd_fwd_noalloc, against the
regular mamba2_ssd_fwd.

Callers that cannot allocate device memory (an allocator-free runtime, code
under a custom pool) use mamba2_ssd_fwd_noalloc, whose intermediates live in
a fixed device array inside the library.  Two calls in a row (different
shapes, dtypes and data) must each match mamba2_ssd_fwd on the same inputs
within the parity tolerance, so nothing left in the shared array by the first
call leaks into the second.  This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, np64, rel_err, to_dev
from mamba_chunked_ssd_gb300 import binding as bd
from mamba_chunked_ssd_gb300.synthetic import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mamba_chunked_ssd_gb300 import build_lib
    build_lib.build()
    bd.load_library()


def _both(w):
    d = to_dev(make_inputs(w))
    y_ref, f_ref = bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                                     initial_state=d["initial_state"])
    y = torch.full_like(d["x"], float("nan"))
    f = torch.full((w.batch, w.nheads, w.dstate, w.headdim), float("nan"), device="cuda")
    bd.mamba2_ssd_fwd_noalloc(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                              initial_state=d["initial_state"], y=y, final_state=f)
    bd.mamba2_check_device_status()
    return (y, f), (y_ref, f_ref)


def test_noalloc_matches_ssd_fwd_on_two_calls_in_a_row():
    calls = [
        Workload("noalloc_bf16", 2, 1024, 8, 64, 128, 1, 256, init_state=True, seed=3),
        Workload("noalloc_fp32", 1, 200, 4, 32, 16, 2, 64, dtype="fp32", seed=4),
    ]
    for w in calls:
        (y, f), (y_ref, f_ref) = _both(w)
        assert torch.isfinite(y.float()).all() and torch.isfinite(f).all()
        assert rel_err(np64(y), np64(y_ref)) <= TOL[w.dtype]
        assert rel_err(np64(f), np64(f_ref)) <= TOL[w.dtype]


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = Workload("too_big", 4, 8192, 64, 64, 128, 1, 256)  # needs ~142 MB of intermediates
    shape = bd.make_shape(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk_size,
                          bd.MAMBA2_BF16)
    assert bd.mamba2_ssd_fwd_workspace_size(shape) > 32 << 20
    x = torch.empty(w.batch, w.seqlen, w.nheads, w.headdim, device="cuda", dtype=torch.bfloat16)
    dt = torch.empty(w.batch, w.seqlen, w.nheads, device="cuda")
    A = torch.empty(w.nheads, device="cuda")
    B = torch.empty(w.batch, w.seqlen, 1, w.dstate, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(bd.Mamba2Error) as e:
        bd.mamba2_ssd_fwd_noalloc(x, dt, A, B, B.clone(), w.chunk_size)
    assert e.value.code == 2
