"""The C-ABI library builds, loads and exports every symbol the header declares (CPU only);
host-side argument validation rejects bad calls before anything reaches a GPU."""
import ctypes
import os
import re

import pytest

import zero_sum_prefix_gb300 as zs
from zero_sum_prefix_gb300 import build as zbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "zeros.h")


@pytest.fixture(scope="module")
def lib():
    zbuild.build()
    return zs.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zeros_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(zs.EXPORTS)


def test_version_and_strings(lib):
    assert lib.zeros_version() >= 100
    assert zs.status_string(0) == "ok"
    assert "invalid" in zs.status_string(1)


def test_state_sizes(lib):
    for d in (32, 64, 128):
        rb = zs.record_bytes(d)
        assert rb % 256 == 0 and rb >= 32 + 8 * d + 12 * d * d
        assert zs.state_bytes(3, 5, d) == 256 + 15 * rb
    assert lib.zeros_state_bytes(1, 1, 48) == 0
    assert lib.zeros_state_record_bytes(16) == 0


def _fwd(lib, ptr=16, B=1, H=1, N=8, d=64, causal=1, rope=0, dtype=0, base=1e4, path=0,
         g0=None):
    p = ctypes.c_void_p(ptr) if ptr is not None else None
    g = ctypes.c_void_p(g0) if g0 is not None else None
    return lib.zeros_fwd_ex(p, p, p, p, p, p, g, p, p, p, B, H, N, d, causal, rope, dtype, base,
                            path, None, None, None, None, None, None)


def test_host_validation_without_gpu(lib):
    # Every rejection below happens before any CUDA call, so it runs on a CPU-only host.
    assert _fwd(lib, d=48) == zs.ZEROS_ERR_UNSUPPORTED
    assert _fwd(lib, B=-1) == zs.ZEROS_ERR_INVALID
    assert _fwd(lib, ptr=None) == zs.ZEROS_ERR_INVALID
    assert _fwd(lib, ptr=18) == zs.ZEROS_ERR_INVALID  # misaligned
    assert "aligned" in lib.zeros_last_error_message().decode()
    assert _fwd(lib, dtype=7) == zs.ZEROS_ERR_INVALID
    assert _fwd(lib, causal=2) == zs.ZEROS_ERR_INVALID
    assert _fwd(lib, rope=1, base=0.0) == zs.ZEROS_ERR_INVALID
    assert _fwd(lib, path=9) == zs.ZEROS_ERR_INVALID
    assert _fwd(lib, g0=20) == zs.ZEROS_ERR_INVALID  # optional zero-order gate misaligned
    assert _fwd(lib, N=1 << 24) == zs.ZEROS_ERR_UNSUPPORTED
    # empty problems are valid no-ops and touch nothing
    assert _fwd(lib, ptr=None, B=0) == zs.ZEROS_OK
    assert _fwd(lib, ptr=None, N=0, H=3) == zs.ZEROS_OK
    # a final state is a causal-mode concept
    p = ctypes.c_void_p(16)
    assert lib.zeros_fwd_ex(p, p, p, p, p, p, None, p, p, p, 1, 1, 4, 64, 0, 0, 0, 1e4, 0, p,
                            None, None, None, None, None) == zs.ZEROS_ERR_INVALID
    # decode on a state this process never created is rejected by the explicit-shape entry
    assert lib.zeros_decode_step_ex(p, 1, 1, 64, *([p] * 6), None, p, None, None, None, None,
                                    None) == zs.ZEROS_ERR_INVALID
    assert lib.zeros_state_init(None, p, p, 1, 1, 64, 0, 0, 1e4, None) == zs.ZEROS_ERR_INVALID
    # backward: rejected arguments never reach the GPU
    def bwd(ptr=16, d=64, g0=None, dg0=None, rope=0, base=1e4):
        x = ctypes.c_void_p(ptr) if ptr is not None else None
        g = ctypes.c_void_p(g0) if g0 is not None else None
        dg = ctypes.c_void_p(dg0) if dg0 is not None else None
        return lib.zeros_bwd(x, x, x, x, x, x, g, x, x, x, x, x, x, x, x, x, dg, x, x,
                             1, 1, 8, d, rope, 0, base, None)
    assert bwd(d=48) == zs.ZEROS_ERR_UNSUPPORTED
    assert bwd(ptr=None) == zs.ZEROS_ERR_INVALID
    assert bwd(ptr=24) == zs.ZEROS_ERR_INVALID
    assert bwd(dg0=16) == zs.ZEROS_ERR_INVALID       # dg0 without the gate
    assert bwd(rope=1, base=-1.0) == zs.ZEROS_ERR_INVALID
    def bwd_ex(d=64, path=0):
        x = ctypes.c_void_p(16)
        return lib.zeros_bwd_ex(x, x, x, x, x, x, None, x, x, x, x, x, x, x, x, x, None, x, x,
                                1, 1, 8, d, 0, 0, 1e4, path, None)
    assert bwd_ex(path=7) == zs.ZEROS_ERR_INVALID
    assert bwd_ex(d=32, path=2) == zs.ZEROS_ERR_UNSUPPORTED  # chunked: d = 64 only
    # output LayerNorm: epsilon and gain/bias pointers are checked before any CUDA call
    def fwd_ln(eps=1e-5, w=None, b=None, d=64):
        wp = ctypes.c_void_p(w) if w is not None else None
        bp = ctypes.c_void_p(b) if b is not None else None
        return lib.zeros_fwd_ln(p, p, p, p, p, p, None, p, p, wp, bp, eps, p, 1, 1, 4, d, 1, 0,
                                0, 1e4, 0, None, None)
    assert fwd_ln(eps=-1.0) == zs.ZEROS_ERR_INVALID
    assert fwd_ln(eps=float("inf")) == zs.ZEROS_ERR_INVALID
    assert fwd_ln(eps=float("nan")) == zs.ZEROS_ERR_INVALID
    assert fwd_ln(w=20) == zs.ZEROS_ERR_INVALID
    assert fwd_ln(b=36) == zs.ZEROS_ERR_INVALID
    assert fwd_ln(d=48) == zs.ZEROS_ERR_UNSUPPORTED
    assert lib.zeros_decode_step_ln(p, 1, 1, 64, *([p] * 6), None, None, None, 1e-5, p,
                                    None) == zs.ZEROS_ERR_INVALID
    # ZeroS-SM: bf16 and d in {64, 128} only; the usual argument checks
    def sm(d=64, dtype=0, ptr=16, rope=0, base=1e4, N=8, causal=1):
        x = ctypes.c_void_p(ptr) if ptr is not None else None
        return lib.zeros_sm_fwd(x, x, x, x, x, None, x, 1, 1, N, d, causal, rope, dtype, base,
                                None)
    assert sm(d=32) == zs.ZEROS_ERR_UNSUPPORTED
    assert sm(dtype=1) == zs.ZEROS_ERR_UNSUPPORTED
    assert sm(ptr=None) == zs.ZEROS_ERR_INVALID
    assert sm(ptr=40) == zs.ZEROS_ERR_INVALID
    assert sm(rope=1, base=0.0) == zs.ZEROS_ERR_INVALID
    assert sm(causal=3) == zs.ZEROS_ERR_INVALID
    assert sm(N=65535 * 128 + 1) == zs.ZEROS_ERR_UNSUPPORTED
    assert sm(ptr=None, N=0) == zs.ZEROS_OK
