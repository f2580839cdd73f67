"""Failure handling on the GPU, in the permitted form: a bounded wait that is
made to run out on a barrier nothing completes, never a fault or a hang.

mamba2_selftest_wait_timeout enqueues a kernel that holds tensor memory, lets
one waiter give up after a short limit (recording MAMBA2_ERR_TIMEOUT in the
device status word and raising the kernel's abort flag) and a second waiter
leave through that flag, frees the tensor memory and returns.  The test checks
the status the host reads, that the kernel returned in about the limit (not
the second waiter's own 0.5 s limit), and that the context is still usable:
a full forward pass, whose CTAs allocate all of their SM's tensor memory,
afterwards matches the oracle.
"""
import pytest
import torch

import oracle
from gpu_helpers import TOL, np64, rel_err, to_dev
from mamba_chunked_ssd_gb300 import binding as bd
from mamba_chunked_ssd_gb300.synthetic import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mamba_chunked_ssd_gb300 import build_lib
    build_lib.build()
    bd.load_library()


def test_bounded_wait_runs_out_and_is_reported():
    bd.mamba2_check_device_status()  # start from a clear status word
    stream = torch.cuda.current_stream()
    limit_ns = 2_000_000
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    bd.mamba2_selftest_wait_timeout(limit_ns)
    e1.record(stream)
    with pytest.raises(bd.Mamba2Error) as err:
        bd.mamba2_check_device_status()
    assert err.value.code == 4  # MAMBA2_ERR_TIMEOUT
    ms = e0.elapsed_time(e1)
    assert limit_ns / 1e6 <= ms < 250.0, ms
    bd.mamba2_check_device_status()  # the word was cleared by the read

    w = Workload("after_timeout", 2, 512, 8, 64, 128, 1, 256, init_state=True)
    inp = make_inputs(w)
    d = to_dev(inp)
    y, fin = bd.mamba2_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], w.chunk_size, D=d["D"],
                               initial_state=d["initial_state"])
    bd.mamba2_check_device_status()
    r = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                              init=inp["initial_state"])
    assert rel_err(np64(y), r["y"]) <= TOL[w.dtype]
    assert rel_err(np64(fin), r["final_state"]) <= TOL[w.dtype]


def test_two_timeouts_in_a_row():
    """The self-test leaves nothing behind: a second run reports again."""
    for _ in range(2):
        bd.mamba2_selftest_wait_timeout(1_000_000)
        with pytest.raises(bd.Mamba2Error) as err:
            bd.mamba2_check_device_status()
        assert err.value.code == 4
    bd.mamba2_check_device_status()
