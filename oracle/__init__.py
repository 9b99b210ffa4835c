"""fp64 CPU oracle for the ZeroS (zero-sum linear attention) layer.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()`` and by the
CPU-baseline / reference legs of ``bench.py``; never by the product package.  It shares no
code with the CUDA path.

The arithmetic lives in ``zeros_oracle.cpp`` (plain C++17, fp64, one thread per (b, h)
sequence); this module only compiles it with g++ and marshals numpy arrays through ctypes.
See that file's header for the pages and sections each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zeros_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libzeros_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, so: str = _SO) -> str:
    """Compile the oracle source ``src`` into the shared library ``so`` (host architecture)."""
    os.makedirs(os.path.dirname(so), exist_ok=True)
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        tmp = so + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", src, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, so)
    return so


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _unpack(q, k, v, u, g1, gh, mu, tau):
    q, k, v, u = (_f64(t) for t in (q, k, v, u))
    g1, gh, mu, tau = (_f64(t) for t in (g1, gh, mu, tau))
    B, H, N, d = q.shape
    for t in (k, v, u):
        assert t.shape == (B, H, N, d)
    assert g1.shape == (B, H, N) and gh.shape == (B, H, N)
    assert mu.shape == (H, d) and tau.shape == (H,)
    return q, k, v, u, g1, gh, mu, tau, (B, H, N, d)


def _gate(g, shape):
    if g is None:
        return None
    g = _f64(g)
    assert g.shape == shape
    return g


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.zs_oracle_fwd.argtypes = [dp] * 9 + [i] * 6 + [ctypes.c_double, ctypes.c_double,
                                                         i, dp, dp, dp, dp]
        lib.zs_oracle_fwd.restype = i
        lib.zs_oracle_brute.argtypes = [dp] * 9 + [i] * 6 + [ctypes.c_double, i, dp, dp, dp]
        lib.zs_oracle_brute.restype = i
        lib.zs_oracle_threads.restype = i
        lib.zs_oracle_sm.argtypes = [dp] * 7 + [i] * 6 + [ctypes.c_double, i, dp]
        lib.zs_oracle_sm.restype = i
        lib.zs_oracle_layer_norm.argtypes = [dp] * 3 + [ctypes.c_double, dp] + [i] * 4
        lib.zs_oracle_layer_norm.restype = i
        self.lib = lib

    def threads(self) -> int:
        """Hardware threads the oracle uses by default."""
        return self.lib.zs_oracle_threads()

    def forward(self, q, k, v, u, g1, gh, mu, tau, *, causal=True, rope=False,
                rope_base=10000.0, pos0=0.0, nthreads=0, debug=False, g0=None):
        """Recurrent fp64 forward (five prefix states).  Layouts: q,k,v,u [B,H,N,d],
        g1,gh [B,H,N], mu [H,d], tau [H] (numpy arrays or CPU/GPU torch tensors); g0 [B,H,N]
        (optional) are the zero-order gate logits of a first layer.

        Returns ``out`` [B,H,N,d] float64, or ``(out, s, E, P)`` when ``debug`` is true
        (each [B,H,N]: the logit s_t and the prefix sums E_t, P_t at every step)."""
        q, k, v, u, g1, gh, mu, tau, (B, H, N, d) = _unpack(q, k, v, u, g1, gh, mu, tau)
        g0 = _gate(g0, (B, H, N))
        out = np.zeros((B, H, N, d), np.float64)
        s = E = P = None
        if debug:
            s, E, P = (np.zeros((B, H, N), np.float64) for _ in range(3))
        rc = self.lib.zs_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(g1), _ptr(gh),
                                    _ptr(mu), _ptr(tau), _ptr(out), B, H, N, d, int(causal),
                                    int(rope), float(rope_base), float(pos0), int(nthreads),
                                    _ptr(s), _ptr(E), _ptr(P), _ptr(g0))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return (out, s, E, P) if debug else out

    def brute(self, q, k, v, u, g1, gh, mu, tau, *, causal=True, rope=False,
              rope_base=10000.0, nthreads=0, g0=None):
        """O(N^2 d) fp64 evaluation of the definition.  Returns ``(out, wsum, wabsmax)`` with
        ``wsum[b,h,t] = sum_i w_{t,i}`` and ``wabsmax[b,h,t] = max_i |w_{t,i}|``."""
        q, k, v, u, g1, gh, mu, tau, (B, H, N, d) = _unpack(q, k, v, u, g1, gh, mu, tau)
        g0 = _gate(g0, (B, H, N))
        out = np.zeros((B, H, N, d), np.float64)
        ws = np.zeros((B, H, N), np.float64)
        wm = np.zeros((B, H, N), np.float64)
        rc = self.lib.zs_oracle_brute(_ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(g1), _ptr(gh),
                                      _ptr(mu), _ptr(tau), _ptr(out), B, H, N, d, int(causal),
                                      int(rope), float(rope_base), int(nthreads), _ptr(ws),
                                      _ptr(wm), _ptr(g0))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return out, ws, wm


    def sm(self, q, k, v, g1, gh, *, causal=True, rope=False, rope_base=10000.0, nthreads=0,
           g0=None, wsum=False):
        """ZeroS-SM (the zero-sum reweighting of standard softmax attention), O(N^2 d) fp64.
        q, k, v [B,H,N,d]; g1, gh, g0 [B,H,N].  Returns ``out``, or ``(out, wsum)``."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, d = q.shape
        assert k.shape == q.shape and v.shape == q.shape
        g1, gh, g0 = _gate(g1, (B, H, N)), _gate(gh, (B, H, N)), _gate(g0, (B, H, N))
        out = np.zeros((B, H, N, d), np.float64)
        ws = np.zeros((B, H, N), np.float64) if wsum else None
        if self.lib.zs_oracle_sm(_ptr(q), _ptr(k), _ptr(v), _ptr(g1), _ptr(gh), _ptr(g0),
                                 _ptr(out), B, H, N, d, int(causal), int(rope),
                                 float(rope_base), int(nthreads), _ptr(ws)) != 0:
            raise ValueError("oracle rejected its arguments")
        return (out, ws) if wsum else out

    def layer_norm(self, o, w=None, b=None, eps=1e-5):
        """Output LayerNorm of every head's row over its d channels: o [B,H,N,d]; w, b [H,d]
        (None: gain 1, bias 0).  Returns a new float64 array."""
        o = _f64(o)
        B, H, N, d = o.shape
        w, b = _gate(w, (H, d)), _gate(b, (H, d))
        y = np.zeros_like(o)
        if self.lib.zs_oracle_layer_norm(_ptr(o), _ptr(w), _ptr(b), float(eps), _ptr(y),
                                         B, H, N, d) != 0:
            raise ValueError("oracle rejected its arguments")
        return y


def default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def threads() -> int:
    return default().threads()


def forward(*args, **kw):
    return default().forward(*args, **kw)


def brute(*args, **kw):
    return default().brute(*args, **kw)


def layer_norm(*args, **kw):
    return default().layer_norm(*args, **kw)


def sm(*args, **kw):
    return default().sm(*args, **kw)
