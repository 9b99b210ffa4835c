"""GB300-native hot path of ZeroS (zero-sum linear attention).

A thin Python binding of the C ABI in ``include/zeros.h``: it checks tensor shapes and
dtypes, passes raw device pointers and the current CUDA stream to ``libzeros.so`` and turns
nonzero status codes into exceptions.  Every step of the computation runs in the library's
CUDA kernels; there is no Python or CPU fallback.  PyTorch is used only for device memory and
streams.

Build the library first with ``python -m zero_sum_prefix_gb300.build`` (or
``__graft_entry__.build()``); importing the binding does not compile anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libzeros.so")

ZEROS_OK, ZEROS_ERR_INVALID, ZEROS_ERR_UNSUPPORTED, ZEROS_ERR_RANGE, ZEROS_ERR_TIMEOUT, \
    ZEROS_ERR_CUDA = range(6)
ZEROS_BF16, ZEROS_F32 = 0, 1
PATHS = {"auto": 0, "simt": 1, "chunk": 2}

EXPORTS = ["zeros_fwd", "zeros_fwd_ex", "zeros_state_bytes", "zeros_state_record_bytes",
           "zeros_state_init", "zeros_decode_step", "zeros_decode_step_ex", "zeros_get_status",
           "zeros_status_string", "zeros_last_error_message", "zeros_version",
           "zeros_kernel_launches", "zeros_fwd_noalloc", "zeros_bwd", "zeros_fwd_ln",
           "zeros_decode_step_ln", "zeros_sm_fwd", "zeros_bwd_ex", "zeros_debug_walk"]

_lock = threading.Lock()
_lib = None


class ZerosError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        msg = f"{where}: status {code} ({status_string(code)})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


def load():
    """Load libzeros.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m zero_sum_prefix_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.zeros_fwd.argtypes = [vp] * 9 + [i] * 6 + [vp]
        lib.zeros_fwd.restype = i
        lib.zeros_fwd_ex.argtypes = [vp] * 10 + [i] * 7 + [f, i, vp, vp, vp, vp, vp, vp]
        lib.zeros_fwd_ex.restype = i
        lib.zeros_state_bytes.argtypes = [i, i, i]
        lib.zeros_state_bytes.restype = sz
        lib.zeros_state_record_bytes.argtypes = [i]
        lib.zeros_state_record_bytes.restype = sz
        lib.zeros_state_init.argtypes = [vp, vp, vp, i, i, i, i, i, f, vp]
        lib.zeros_state_init.restype = i
        lib.zeros_decode_step.argtypes = [vp] * 9
        lib.zeros_decode_step.restype = i
        lib.zeros_decode_step_ex.argtypes = [vp, i, i, i] + [vp] * 13
        lib.zeros_decode_step_ex.restype = i
        lib.zeros_get_status.argtypes = [vp]
        lib.zeros_get_status.restype = i
        lib.zeros_status_string.argtypes = [i]
        lib.zeros_status_string.restype = ctypes.c_char_p
        lib.zeros_last_error_message.restype = ctypes.c_char_p
        lib.zeros_version.restype = i
        lib.zeros_kernel_launches.restype = ctypes.c_ulonglong
        lib.zeros_debug_walk.argtypes = [ctypes.c_longlong, i]
        lib.zeros_debug_walk.restype = i
        lib.zeros_fwd_noalloc.argtypes = [vp] * 9 + [i] * 7 + [f, vp, vp]
        lib.zeros_bwd.argtypes = [vp] * 19 + [i] * 6 + [f, vp]
        lib.zeros_bwd.restype = i
        lib.zeros_fwd_ln.argtypes = [vp] * 11 + [f, vp] + [i] * 7 + [f, i, vp, vp]
        lib.zeros_fwd_ln.restype = i
        lib.zeros_decode_step_ln.argtypes = [vp, i, i, i] + [vp] * 9 + [f, vp, vp]
        lib.zeros_decode_step_ln.restype = i
        lib.zeros_bwd_ex.argtypes = [vp] * 19 + [i] * 6 + [f, i, vp]
        lib.zeros_bwd_ex.restype = i
        lib.zeros_sm_fwd.argtypes = [vp] * 7 + [i] * 7 + [f, vp]
        lib.zeros_sm_fwd.restype = i
        lib.zeros_fwd_noalloc.restype = i
        _lib = lib
        return lib


def kernel_launches() -> int:
    """Kernels launched through the library by this process so far."""
    return int(load().zeros_kernel_launches())


def debug_walk(wait_limit_cycles: int = 0, skip_one_arrive: bool = False):
    """Testing hook of the d = 64 tensor-core forward's failure path (zeros_debug_walk): the
    bound of its waits in SM cycles (0 = default) and whether one warp per CTA withholds an
    arrival so that a wait runs out.  Process-wide; set only while no forward runs."""
    rc = load().zeros_debug_walk(int(wait_limit_cycles), int(bool(skip_one_arrive)))
    if rc != ZEROS_OK:
        raise ZerosError(rc, "zeros_debug_walk")


def status_string(code: int) -> str:
    return load().zeros_status_string(int(code)).decode()


def _check(rc: int, where: str):
    if rc != ZEROS_OK:
        raise ZerosError(rc, where, load().zeros_last_error_message().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ZEROS_BF16
    if t.dtype == torch.float32:
        return ZEROS_F32
    raise TypeError(f"q, k, v, u must be bfloat16 or float32, got {t.dtype}")


def _need(t, name, shape, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ln_args(ln, ln_w, ln_b, H, d):
    if ln_w is not None:
        _need(ln_w, "ln_w", (H, d), torch.float32)
    if ln_b is not None:
        _need(ln_b, "ln_b", (H, d), torch.float32)
    return bool(ln) or ln_w is not None or ln_b is not None


def fwd(q, k, v, u, g1, gh, mu, tau, *, causal=True, rope=False, rope_base=10000.0, out=None,
        final_state=None, debug=False, path="auto", stream=None, g0=None, ln=False, ln_w=None,
        ln_b=None, ln_eps=1e-5):
    """ZeroS forward.  q, k, v, u: [B, H, N, d] bf16 or fp32 (same dtype); g1, gh: [B, H, N]
    fp32 gate logits; mu: [H, d] fp32; tau: [H] fp32; g0: optional [B, H, N] fp32 zero-order
    gate logits of a first layer.  ``ln`` (implied by ``ln_w`` / ``ln_b``, [H, d] fp32) fuses
    the output LayerNorm of each head's rows.  Returns ``out`` (same dtype as q), or
    ``(out, dbg)`` with ``dbg = dict(s, E, P, m)`` ([B, H, N] fp32) when ``debug``."""
    B, H, N, d = q.shape
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("u", u)):
        _need(t, name, (B, H, N, d), dt)
    _need(g1, "g1", (B, H, N), torch.float32)
    _need(gh, "gh", (B, H, N), torch.float32)
    if g0 is not None:
        _need(g0, "g0", (B, H, N), torch.float32)
    _need(mu, "mu", (H, d), torch.float32)
    _need(tau, "tau", (H,), torch.float32)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (B, H, N, d), dt)
    if final_state is not None:
        _need(final_state, "final_state", (state_bytes(B, H, d),), torch.uint8)
    lib = load()
    if _ln_args(ln, ln_w, ln_b, H, d):
        if debug:
            raise ValueError("debug outputs are not available with the output LayerNorm")
        rc = lib.zeros_fwd_ln(_ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(g1), _ptr(gh), _ptr(g0),
                              _ptr(mu), _ptr(tau), _ptr(ln_w), _ptr(ln_b), float(ln_eps),
                              _ptr(out), B, H, N, d, int(bool(causal)), int(bool(rope)),
                              _dtype_code(q), float(rope_base), PATHS[path], _ptr(final_state),
                              _stream(stream))
        _check(rc, "zeros_fwd_ln")
        return out
    dbg = None
    if debug:
        dbg = {n: torch.empty((B, H, N), device=q.device, dtype=torch.float32)
               for n in ("s", "E", "P", "m")}
    rc = lib.zeros_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(g1), _ptr(gh), _ptr(g0),
                          _ptr(mu), _ptr(tau), _ptr(out), B, H, N, d, int(bool(causal)),
                          int(bool(rope)),
                          _dtype_code(q), float(rope_base), PATHS[path], _ptr(final_state),
                          *(None if dbg is None else _ptr(dbg[n]) for n in ("s", "E", "P", "m")),
                          _stream(stream))
    _check(rc, "zeros_fwd_ex")
    return (out, dbg) if debug else out


def sm_fwd(q, k, v, g1, gh, *, causal=True, rope=False, rope_base=10000.0, g0=None, out=None,
           stream=None):
    """ZeroS-SM (the zero-sum reweighting of standard softmax attention): q, k, v [B, H, N, d]
    bf16, d in {64, 128}; g1, gh (g0 optional) [B, H, N] fp32.  Returns ``out`` (bf16)."""
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, (B, H, N, d), torch.bfloat16)
    _need(g1, "g1", (B, H, N), torch.float32)
    _need(gh, "gh", (B, H, N), torch.float32)
    if g0 is not None:
        _need(g0, "g0", (B, H, N), torch.float32)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (B, H, N, d), torch.bfloat16)
    rc = load().zeros_sm_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g1), _ptr(gh), _ptr(g0), _ptr(out),
                             B, H, N, d, int(bool(causal)), int(bool(rope)), ZEROS_BF16,
                             float(rope_base), _stream(stream))
    _check(rc, "zeros_sm_fwd")
    return out


def bwd(q, k, v, u, g1, gh, mu, tau, dout, *, rope=False, rope_base=10000.0, g0=None,
        stream=None, path="auto"):
    """Backward of the causal forward: gradients of sum(out * dout).  Inputs as in ``fwd``
    (causal mode); ``dout`` has the shape and dtype of q.  Returns a dict of fp32 tensors
    dq, dk, dv, du [B, H, N, d], dg1, dgh [B, H, N], dmu [H, d], dtau [H] (and dg0 when
    ``g0`` is given)."""
    B, H, N, d = q.shape
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("u", u), ("dout", dout)):
        _need(t, name, (B, H, N, d), dt)
    _need(g1, "g1", (B, H, N), torch.float32)
    _need(gh, "gh", (B, H, N), torch.float32)
    if g0 is not None:
        _need(g0, "g0", (B, H, N), torch.float32)
    _need(mu, "mu", (H, d), torch.float32)
    _need(tau, "tau", (H,), torch.float32)
    f32 = dict(device=q.device, dtype=torch.float32)
    g = {n: torch.empty((B, H, N, d), **f32) for n in ("dq", "dk", "dv", "du")}
    g["dg1"] = torch.empty((B, H, N), **f32)
    g["dgh"] = torch.empty((B, H, N), **f32)
    g["dmu"] = torch.empty((H, d), **f32)
    g["dtau"] = torch.empty((H,), **f32)
    if g0 is not None:
        g["dg0"] = torch.empty((B, H, N), **f32)
    rc = load().zeros_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(g1), _ptr(gh),
                             _ptr(g0), _ptr(mu), _ptr(tau), _ptr(dout), _ptr(g["dq"]),
                             _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["du"]), _ptr(g["dg1"]),
                             _ptr(g["dgh"]), _ptr(g.get("dg0")), _ptr(g["dmu"]),
                             _ptr(g["dtau"]), B, H, N, d, int(bool(rope)), _dtype_code(q),
                             float(rope_base), PATHS[path], _stream(stream))
    _check(rc, "zeros_bwd_ex")
    return g


def state_bytes(B: int, H: int, d: int) -> int:
    n = load().zeros_state_bytes(B, H, d)
    if n == 0:
        raise ValueError(f"unsupported state dimensions B={B} H={H} d={d}")
    return int(n)


def record_bytes(d: int) -> int:
    return int(load().zeros_state_record_bytes(d))


def new_state(mu, tau, B: int, *, dtype=torch.bfloat16, rope=False, rope_base=10000.0,
              stream=None) -> torch.Tensor:
    """Allocate (with torch) and initialise an empty recurrent state for B x H sequences."""
    H, d = mu.shape
    _need(mu, "mu", (H, d), torch.float32)
    _need(tau, "tau", (H,), torch.float32)
    st = torch.empty(state_bytes(B, H, d), dtype=torch.uint8, device=mu.device)
    rc = load().zeros_state_init(_ptr(st), _ptr(mu), _ptr(tau), B, H, d,
                                 ZEROS_BF16 if dtype == torch.bfloat16 else ZEROS_F32,
                                 int(bool(rope)), float(rope_base), _stream(stream))
    _check(rc, "zeros_state_init")
    return st


def decode_step(state, q, k, v, u, g1, gh, *, out=None, debug=False, stream=None, g0=None,
                ln=False, ln_w=None, ln_b=None, ln_eps=1e-5):
    """One recurrent step for every sequence: q, k, v, u [B, H, d]; g1, gh [B, H]; g0
    optional [B, H] zero-order gate logits; ``ln`` / ``ln_w`` / ``ln_b`` as in ``fwd``."""
    B, H, d = q.shape
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("u", u)):
        _need(t, name, (B, H, d), dt)
    _need(g1, "g1", (B, H), torch.float32)
    _need(gh, "gh", (B, H), torch.float32)
    if g0 is not None:
        _need(g0, "g0", (B, H), torch.float32)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (B, H, d), dt)
    lib = load()
    if _ln_args(ln, ln_w, ln_b, H, d):
        if debug:
            raise ValueError("debug outputs are not available with the output LayerNorm")
        rc = lib.zeros_decode_step_ln(_ptr(state), B, H, d, _ptr(q), _ptr(k), _ptr(v), _ptr(u),
                                      _ptr(g1), _ptr(gh), _ptr(g0), _ptr(ln_w), _ptr(ln_b),
                                      float(ln_eps), _ptr(out), _stream(stream))
        _check(rc, "zeros_decode_step_ln")
        return out
    if debug or g0 is not None:
        dbg = None
        if debug:
            dbg = {n: torch.empty((B, H), device=q.device, dtype=torch.float32)
                   for n in ("s", "E", "P", "m")}
        rc = lib.zeros_decode_step_ex(_ptr(state), B, H, d, _ptr(q), _ptr(k), _ptr(v), _ptr(u),
                                      _ptr(g1), _ptr(gh), _ptr(g0), _ptr(out),
                                      *(None if dbg is None else _ptr(dbg[n])
                                        for n in ("s", "E", "P", "m")),
                                      _stream(stream))
        _check(rc, "zeros_decode_step_ex")
        return (out, dbg) if debug else out
    rc = lib.zeros_decode_step(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(g1),
                               _ptr(gh), _ptr(out), _stream(stream))
    _check(rc, "zeros_decode_step")
    return out


def get_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word (0 = ok)."""
    return int(load().zeros_get_status(_stream(stream)))


def check_status(where="device", stream=None):
    rc = get_status(stream)
    if rc != ZEROS_OK:
        raise ZerosError(rc, where)


def state_view(state: torch.Tensor, B: int, H: int, d: int) -> dict:
    """Named views into a state blob (for tests and checkpoint tooling); layout in zeros.h."""
    rb = record_bytes(d)
    recs = state[256:256 + B * H * rb].view(B * H, rb)
    f = recs.view(torch.float32).view(B * H, rb // 4)
    i = recs.view(torch.int32).view(B * H, rb // 4)
    o = 8
    return dict(t=i[:, 0], mC=f[:, 1], EC=f[:, 2], CP=f[:, 3], etau=f[:, 4], ml=f[:, 5],
                El=f[:, 6], LP=f[:, 7], C=f[:, o:o + d], L=f[:, o + d:o + 2 * d],
                mu=f[:, o + 2 * d:o + 3 * d],
                F=f[:, o + 3 * d:o + 3 * d + d * d].view(B * H, d, d),
                G=f[:, o + 3 * d + d * d:o + 3 * d + 2 * d * d].view(B * H, d, d),
                H=f[:, o + 3 * d + 2 * d * d:o + 3 * d + 3 * d * d].view(B * H, d, d))
