"""C-ABI checks that need no GPU: the library loads, exports every function
include/mamba2_ssd.h declares, and rejects bad arguments on the host before
any CUDA call (fake pointer values are never dereferenced on these paths)."""
import ctypes

import pytest

from mamba_chunked_ssd_gb300 import binding as bd

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    from mamba_chunked_ssd_gb300 import build_lib
    build_lib.build()
    return bd.load_library()


def test_exports_every_declared_function(lib):
    names = bd.header_functions()
    assert len(names) == 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in the header but not exported"


def test_version_and_status_strings(lib):
    assert lib.mamba2_version() == 10200
    for code in range(5):
        s = lib.mamba2_status_string(code).decode()
        assert s.startswith(bd.STATUS[code])


def _shape(**kw):
    d = dict(batch=1, seqlen=64, nheads=2, headdim=16, dstate=16, ngroups=1, chunk_size=64, dtype_code=0)
    d.update(kw)
    return bd.make_shape(d["batch"], d["seqlen"], d["nheads"], d["headdim"], d["dstate"],
                         d["ngroups"], d["chunk_size"], d["dtype_code"])


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def _p(v):
    return ctypes.c_void_p(v)


def _cumsum(lib, shape, dt=FAKE, A=FAKE * 2, G=FAKE * 64):
    return lib.mamba2_chunk_cumsum(ctypes.byref(shape) if shape is not None else None,
                                   _p(dt), _p(A), _p(G), None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype_code=7), INVALID),
    (dict(nheads=3, ngroups=2), INVALID),
    (dict(chunk_size=0), INVALID),
    (dict(headdim=0), INVALID),
    (dict(batch=-1), INVALID),
    (dict(seqlen=-5), INVALID),
    (dict(headdim=512), UNSUPPORTED),
    (dict(dstate=300), UNSUPPORTED),
    (dict(chunk_size=512), UNSUPPORTED),
    (dict(batch=70000), UNSUPPORTED),
])
def test_shape_validation(lib, kw, code):
    assert _cumsum(lib, _shape(**kw)) == code


def test_null_shape(lib):
    assert _cumsum(lib, None) == INVALID
    assert lib.mamba2_ssd_fwd_workspace_size(None) == 0


def test_reserved_must_be_zero(lib):
    s = _shape()
    s.reserved = 1
    assert _cumsum(lib, s) == INVALID


def test_null_and_misaligned_pointers(lib):
    s = _shape()
    assert _cumsum(lib, s, dt=0) == INVALID
    assert _cumsum(lib, s, G=FAKE * 64 + 4) == INVALID
    assert _cumsum(lib, s, A=FAKE * 2 + 8) == INVALID


def test_output_aliasing_input_is_rejected(lib):
    s = _shape()
    # G [1, 2, 64] fp32 = 512 bytes written over dt's bytes
    assert _cumsum(lib, s, dt=FAKE, G=FAKE + 256) == INVALID


def test_chunk_out_rejects_y_aliasing_x(lib):
    s = _shape(dtype_code=1)
    args = [ctypes.byref(s)] + [_p(FAKE * (i + 1) * 16) for i in range(7)] + [_p(FAKE * 16), None]
    assert lib.mamba2_chunk_out(*args) == INVALID


def test_workspace_size(lib):
    s = _shape(batch=2, seqlen=100, nheads=4, headdim=16, dstate=8, chunk_size=32, dtype_code=1)
    nc = 4
    g_bytes = 2 * 4 * 100 * 4
    cs_bytes = 2 * 4 * nc * 8 * 16 * 2
    up = lambda v: (v + 255) // 256 * 256
    assert lib.mamba2_ssd_fwd_workspace_size(ctypes.byref(s)) == up(g_bytes) + up(cs_bytes)


def test_workspace_size_with_sequence_segments(lib):
    """Two (batch, head) pairs of bf16 heads fill few SMs, so the forward
    pass splits each sequence of 32 chunks into 8 segments of 4 chunks and
    keeps the states of the first 7 segments (fp32 S x H each) in the
    workspace after G and the chunk states."""
    s = _shape(batch=1, seqlen=4096, nheads=2, headdim=64, dstate=128, chunk_size=128, dtype_code=1)
    up = lambda v: (v + 255) // 256 * 256
    g_bytes = 1 * 2 * 4096 * 4
    cs_bytes = 1 * 2 * 32 * 128 * 64 * 2
    seg_bytes = 1 * 2 * 7 * 128 * 64 * 4
    assert lib.mamba2_ssd_fwd_workspace_size(ctypes.byref(s)) == up(g_bytes) + up(cs_bytes) + up(seg_bytes)
    # many (batch, head) pairs: one pass, no segment states
    s = _shape(batch=4, seqlen=4096, nheads=64, headdim=64, dstate=128, chunk_size=128, dtype_code=1)
    assert lib.mamba2_ssd_fwd_workspace_size(ctypes.byref(s)) == up(4 * 64 * 4096 * 4) + up(4 * 64 * 32 * 128 * 64 * 2)


def test_ssd_fwd_rejects_small_or_misaligned_workspace(lib):
    s = _shape()
    need = lib.mamba2_ssd_fwd_workspace_size(ctypes.byref(s))
    ptrs = [_p(FAKE * (i + 1) * 64) for i in range(9)]
    small = lib.mamba2_ssd_fwd(ctypes.byref(s), *ptrs, _p(FAKE * 4096), need - 1, None)
    assert small == INVALID
    misaligned = lib.mamba2_ssd_fwd(ctypes.byref(s), *ptrs, _p(FAKE * 4096 + 16), need, None)
    assert misaligned == INVALID


def _step(lib, shape, x=FAKE, dt=FAKE * 2, A=FAKE * 3, B=FAKE * 4, C=FAKE * 5, D=None,
          state_in=FAKE * 8, state_out=FAKE * 16, y=FAKE * 6):
    return lib.mamba2_ssd_step(ctypes.byref(shape), _p(x), _p(dt), _p(A), _p(B), _p(C),
                               _p(D) if D else None, _p(state_in) if state_in else None,
                               _p(state_out) if state_out else None, _p(y), None)


def test_step_requires_one_token(lib):
    assert _step(lib, _shape(seqlen=2)) == INVALID
    assert _step(lib, _shape(seqlen=0)) == INVALID


def test_step_requires_state_out(lib):
    assert _step(lib, _shape(seqlen=1), state_out=None) == INVALID


def test_step_rejects_partial_state_overlap(lib):
    # state [1, 2, 16, 16] fp32 = 2048 bytes; a 16-byte shift overlaps
    assert _step(lib, _shape(seqlen=1), state_in=FAKE * 16, state_out=FAKE * 16 + 16) == INVALID


def test_step_rejects_y_over_state(lib):
    assert _step(lib, _shape(seqlen=1), y=FAKE * 16 + 64) == INVALID


def test_step_rejects_misaligned(lib):
    assert _step(lib, _shape(seqlen=1), x=FAKE + 8) == INVALID


@pytest.mark.parametrize("limit", [0, 999, 100000001, -5])
def test_selftest_rejects_out_of_range_limits(lib, limit):
    """Checked on the host: nothing is launched for a bad limit."""
    assert lib.mamba2_selftest_wait_timeout(limit, None) == INVALID


def test_workspace_size_fp32_tensor_core_path(lib, monkeypatch):
    """An fp32 problem whose stages 2 and 3 run on the tensor cores (head dim
    64, state 128) keeps G, the fp32 chunk states at chunk 128 and B as bf16
    hi/lo planes (the bytes of fp32 B) in the workspace, whatever chunk the
    caller gives (the forward pass runs chunk 128 there); with
    MAMBA2_FWD_CHUNK=given a chunk of 32 runs on the CUDA cores and keeps G
    and the fp32 chunk states at chunk 32 only."""
    up = lambda v: (v + 255) // 256 * 256
    g_bytes = 2 * 4 * 1000 * 4
    cs_bytes = 2 * 4 * 8 * 128 * 64 * 4
    b_bytes = 2 * 1000 * 1 * 128 * 4
    for T in (128, 32, 256):
        s = _shape(batch=2, seqlen=1000, nheads=4, headdim=64, dstate=128, chunk_size=T, dtype_code=0)
        assert lib.mamba2_ssd_fwd_workspace_size(ctypes.byref(s)) == up(g_bytes) + up(cs_bytes) + up(b_bytes)
    monkeypatch.setenv("MAMBA2_FWD_CHUNK", "given")
    s = _shape(batch=2, seqlen=1000, nheads=4, headdim=64, dstate=128, chunk_size=32, dtype_code=0)
    cs_bytes = 2 * 4 * 32 * 128 * 64 * 4
    assert lib.mamba2_ssd_fwd_workspace_size(ctypes.byref(s)) == up(g_bytes) + up(cs_bytes)


def test_forward_pass_chunk_choice(lib, monkeypatch):
    """The forward pass's chunk (seen through the workspace's chunk-state
    bytes): bf16 tensor-core shapes run chunk 128 whatever the caller's chunk,
    except with fewer than 16 (batch, head) pairs, which keep the caller's
    (64 becomes 128); CUDA-core shapes keep the caller's; MAMBA2_FWD_CHUNK
    forces one."""
    up = lambda v: (v + 255) // 256 * 256

    def ws(b, L, nh, H, S, T):
        s = _shape(batch=b, seqlen=L, nheads=nh, headdim=H, dstate=S, chunk_size=T, dtype_code=1)
        return lib.mamba2_ssd_fwd_workspace_size(ctypes.byref(s))

    def expect(b, L, nh, H, S, Trun):
        nc = -(-L // Trun)
        return up(b * nh * L * 4) + up(b * nh * nc * S * H * 2)

    assert ws(4, 4096, 64, 64, 256, 256) == expect(4, 4096, 64, 64, 256, 128)
    assert ws(4, 4096, 64, 128, 128, 256) == expect(4, 4096, 64, 128, 128, 128)
    assert ws(2, 4096, 64, 64, 128, 64) == expect(2, 4096, 64, 64, 128, 128)
    assert ws(1, 1024, 8, 64, 128, 256) == expect(1, 1024, 8, 64, 128, 256)     # 8 pairs
    assert ws(1, 1024, 8, 64, 128, 64) == expect(1, 1024, 8, 64, 128, 128)      # 64 -> 128
    assert ws(4, 4096, 64, 16, 16, 32) == expect(4, 4096, 64, 16, 16, 32)       # CUDA cores
    monkeypatch.setenv("MAMBA2_FWD_CHUNK", "given")
    assert ws(4, 4096, 64, 64, 256, 256) == expect(4, 4096, 64, 64, 256, 256)
    monkeypatch.setenv("MAMBA2_FWD_CHUNK", "64")
    assert ws(4, 4096, 64, 64, 256, 256) == expect(4, 4096, 64, 64, 256, 64)


def test_forward_pass_chunk_size_query(lib, monkeypatch):
    """mamba2_ssd_fwd_chunk_size reports the chunk the forward pass runs
    with: 0 for an invalid shape, the rule's choice, or the forced one."""
    assert lib.mamba2_ssd_fwd_chunk_size(None) == 0
    s = _shape(batch=4, seqlen=4096, nheads=64, headdim=64, dstate=256, chunk_size=256, dtype_code=1)
    assert lib.mamba2_ssd_fwd_chunk_size(ctypes.byref(s)) == 128
    s = _shape(batch=4, seqlen=4096, nheads=64, headdim=128, dstate=128, chunk_size=64, dtype_code=1)
    assert lib.mamba2_ssd_fwd_chunk_size(ctypes.byref(s)) == 128
    s = _shape(batch=1, seqlen=4096, nheads=4, headdim=64, dstate=128, chunk_size=256, dtype_code=1)
    assert lib.mamba2_ssd_fwd_chunk_size(ctypes.byref(s)) == 256
    s = _shape(batch=1, seqlen=64, nheads=2, headdim=16, dstate=16, chunk_size=48, dtype_code=0)
    assert lib.mamba2_ssd_fwd_chunk_size(ctypes.byref(s)) == 48
    monkeypatch.setenv("MAMBA2_FWD_CHUNK", "given")
    s = _shape(batch=4, seqlen=4096, nheads=64, headdim=64, dstate=256, chunk_size=256, dtype_code=1)
    assert lib.mamba2_ssd_fwd_chunk_size(ctypes.byref(s)) == 256
