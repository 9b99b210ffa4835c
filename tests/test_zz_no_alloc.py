"""The allocation-free forward, zeros_fwd_noalloc, against the regular entry point.

Some callers cannot allocate device memory at all: for example a runtime whose memory is all
handed out up front by its own allocator, or a server that forbids cudaMalloc once it is up.
For them the library offers one entry point whose only scratch (the rotary table) sits in a
fixed device array compiled into the library.  It runs the same rotary-table kernel and the same
token-sequential forward kernel as zeros_fwd_ex on the token-sequential path, so its output must
be bit-identical to that call's.  These tests call it through the C ABI three times in a row,
with a different rotary base in the middle call (so the shared table must be rebuilt by every
call), and compare each output with the regular entry point bit for bit.  This file is named to
be collected last.
"""
import ctypes

import pytest
import torch

import zeros_inputs as zi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import zero_sum_prefix_gb300 as m
    m.load()
    return m


def _call(zs, inp, w, out, status, N=None):
    lib = zs.load()
    B, H, n, d = inp["q"].shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.zeros_fwd_noalloc(
        p(inp["q"]), p(inp["k"]), p(inp["v"]), p(inp["u"]), p(inp["g1"]), p(inp["gh"]),
        p(inp["mu"]), p(inp["tau"]), p(out), B, H, n if N is None else N, d, int(w.causal),
        int(w.rope), zs.ZEROS_F32 if w.dtype == "f32" else zs.ZEROS_BF16, float(w.rope_base),
        p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype,causal,rope,d", [("f32", True, True, 32), ("bf16", True, True, 64),
                                                 ("bf16", False, False, 64),
                                                 ("bf16", True, True, 128)])
def test_noalloc_matches_regular_entry_bitexact(zs, dtype, causal, rope, d):
    w = zi.Workload("noalloc", 2, 3, 301, d, dtype=dtype, causal=causal, rope=rope,
                    rope_base=500.0, seed=9090 + d)
    inp = zi.make(w, "cuda")
    refs = {}
    for base in (500.0, 10000.0):
        refs[base] = zs.fwd(inp["q"], inp["k"], inp["v"], inp["u"], inp["g1"], inp["gh"],
                            inp["mu"], inp["tau"], causal=causal, rope=rope, rope_base=base,
                            path="simt")
    assert zs.get_status() == 0
    if rope:  # the two bases give different outputs, so a stale table would be seen
        assert not torch.equal(refs[500.0], refs[10000.0])
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for base in (500.0, 10000.0, 500.0):  # every call rewrites the shared scratch
        out = torch.full_like(inp["q"], float("nan"))
        assert _call(zs, inp, w.with_(rope_base=base), out, status) == zs.ZEROS_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, refs[base]), base


def test_noalloc_rejects_sizes_beyond_its_scratch(zs):
    w = zi.Workload("noalloc-big", 1, 1, 16, 64, rope=True, seed=1)
    inp = zi.make(w, "cuda")
    out = torch.empty_like(inp["q"])
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    # N * d / 2 = 4097 * 32 > 131072: refused on the host before anything runs
    assert _call(zs, inp, w, out, status, N=4097) == zs.ZEROS_ERR_UNSUPPORTED
    assert "scratch" in zs.load().zeros_last_error_message().decode()
