"""fp64 CPU oracle for RetNet retention -- TEST INFRASTRUCTURE ONLY.

Nothing in the product path imports this package.  It is loaded only by the
test suite, by the smoke check (to check one small GPU run) and by the
benchmark's CPU-baseline leg.  It shares no code with the CUDA library: the
arithmetic lives in ``retention_oracle.c`` (plain C, fp64, one OpenMP loop over
heads) and this module only compiles that file with gcc and marshals numpy
arrays into it.

Functions (see the C file for the formulas and the page sections they follow):
  gamma(h)                     per-head decay, 0-based h
  parallel(q, k, v, gamma)     parallel form, returns out
  parallel_rows(q, k, v, g, rows)  selected rows of the parallel form, one head
  recurrent(q, k, v, gamma, state=None)  recurrent form, returns (out, state)
  chunkwise(q, k, v, gamma, chunk, state_in=None)  returns (out, state)
  groupnorm(r, weight=None, bias=None, eps=1e-6)  per-(token, head)
                               normalisation, heads concatenated per token
  rotate(x, theta, n0=0)       position phase rotation of queries or keys
  backward(q, k, v, gamma, dout, dstate=None, state_in=None)
                               gradients of the forward (with optional
                               starting state) for output and final-state
                               gradients; returns (dq, dk, dv, dstate_in)

Every function here is pinned by tests/test_oracle.py against closed forms,
hand-expanded sums, a library-routine special case and the three-form
equality that the pages state.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "retention_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C source into a shared library (gcc, -O2, OpenMP)."""
    stale = (not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src))
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-std=c11", "-shared", "-fPIC",
               "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _f64(a) -> np.ndarray:
    """Contiguous float64 copy/view of a numpy array or a CPU torch tensor."""
    if hasattr(a, "detach"):  # torch tensor: exact widening to float64
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _dims(q, v):
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    return B, H, N, dk, dv


class Oracle:
    """numpy front end over one compiled copy of retention_oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_gamma.restype = ctypes.c_double
        lib.oracle_gamma.argtypes = [ctypes.c_int]
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_threads.argtypes = []
        lib.oracle_parallel.restype = None
        lib.oracle_parallel.argtypes = [_dp, _dp, _dp, _dp, _dp] + [ctypes.c_int] * 5
        lib.oracle_parallel_rows.restype = None
        lib.oracle_parallel_rows.argtypes = [_dp, _dp, _dp, ctypes.c_double,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             _ip, ctypes.c_int, _dp]
        lib.oracle_recurrent.restype = None
        lib.oracle_recurrent.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp] + [ctypes.c_int] * 5
        lib.oracle_chunkwise.restype = None
        lib.oracle_chunkwise.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp] + [ctypes.c_int] * 6
        lib.oracle_rotate.restype = None
        lib.oracle_rotate.argtypes = [_dp, _dp, _dp] + [ctypes.c_int] * 4 + [ctypes.c_long]
        lib.oracle_groupnorm.restype = None
        lib.oracle_groupnorm.argtypes = [_dp, _dp, _dp, _dp] + [ctypes.c_int] * 4 + [ctypes.c_double]
        lib.oracle_backward.restype = None
        lib.oracle_backward.argtypes = [_dp] * 11 + [ctypes.c_int] * 5
        self.lib = lib

    def threads(self) -> int:
        """Number of OpenMP threads the oracle's loops use."""
        return int(self.lib.oracle_threads())

    def gamma(self, h):
        """Per-head decay gamma_h = 1 - 2^(-5-h), 0-based h; scalar or array."""
        if np.isscalar(h):
            return float(self.lib.oracle_gamma(int(h)))
        return np.array([self.lib.oracle_gamma(int(x)) for x in np.asarray(h).ravel()],
                        dtype=np.float64)

    def parallel(self, q, k, v, gammas) -> np.ndarray:
        """Parallel form over [B,H,N,d] arrays; returns out [B,H,N,dv] (fp64)."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gammas)
        B, H, N, dk, dv = _dims(q, v)
        out = np.zeros((B, H, N, dv), dtype=np.float64)
        self.lib.oracle_parallel(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out),
                                 B, H, N, dk, dv)
        return out

    def parallel_rows(self, q_head, k_head, v_head, g: float, rows) -> np.ndarray:
        """Rows `rows` of the parallel form for one head ([N,d] inputs)."""
        q, k, v = _f64(q_head), _f64(k_head), _f64(v_head)
        N, dk = q.shape
        dv = v.shape[-1]
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        out = np.zeros((r.size, dv), dtype=np.float64)
        self.lib.oracle_parallel_rows(_ptr(q), _ptr(k), _ptr(v), float(g), N, dk, dv,
                                      r.ctypes.data_as(_ip), int(r.size), _ptr(out))
        return out

    def recurrent(self, q, k, v, gammas, state=None):
        """Recurrent form; returns (out [B,H,N,dv], final state [B,H,dk,dv])."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gammas)
        B, H, N, dk, dv = _dims(q, v)
        S = (np.zeros((B, H, dk, dv), dtype=np.float64) if state is None
             else _f64(state).copy())
        out = np.zeros((B, H, N, dv), dtype=np.float64)
        self.lib.oracle_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S), _ptr(out),
                                  B, H, N, dk, dv)
        return out, S

    def chunkwise(self, q, k, v, gammas, chunk: int, state_in=None):
        """Chunkwise recurrent form; returns (out [B,H,N,dv], final state)."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gammas)
        B, H, N, dk, dv = _dims(q, v)
        out = np.zeros((B, H, N, dv), dtype=np.float64)
        S = np.zeros((B, H, dk, dv), dtype=np.float64)
        s_in = None if state_in is None else _f64(state_in)
        self.lib.oracle_chunkwise(_ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                  None if s_in is None else _ptr(s_in),
                                  _ptr(out), _ptr(S), B, H, N, dk, dv, int(chunk))
        return out, S


    def groupnorm(self, r, weight=None, bias=None, eps: float = 1e-6) -> np.ndarray:
        """Per-(token, head) normalisation of retention outputs r [B,H,N,dv]
        with heads concatenated per token: returns y [B,N,H,dv] (fp64)."""
        r = _f64(r)
        B, H, N, dv = r.shape
        w = None if weight is None else _f64(weight)
        b = None if bias is None else _f64(bias)
        y = np.zeros((B, N, H, dv), dtype=np.float64)
        self.lib.oracle_groupnorm(_ptr(r), None if w is None else _ptr(w), None if b is None else _ptr(b),
                                  _ptr(y), B, H, N, dv, float(eps))
        return y


    def rotate(self, x, theta, n0: int = 0) -> np.ndarray:
        """Position phase rotation of x [B,H,N,d]: pair j of token n turned by
        (n0 + n) theta_j; returns y [B,H,N,d] (fp64)."""
        x, th = _f64(x), _f64(theta)
        B, H, N, d = x.shape
        y = np.zeros_like(x)
        self.lib.oracle_rotate(_ptr(x), _ptr(th), _ptr(y), B, H, N, d, int(n0))
        return y

    def backward(self, q, k, v, gammas, dout, dstate=None, state_in=None):
        """Gradients of sum(dout * out) + sum(dstate * S_N) with respect to q,
        k, v and the starting state, for the forward started from state_in
        (zero if None).  Returns (dq, dk, dv, dstate_in), all fp64."""
        q, k, v, g, do = _f64(q), _f64(k), _f64(v), _f64(gammas), _f64(dout)
        B, H, N, dk, dv = _dims(q, v)
        s0 = None if state_in is None else _f64(state_in)
        ds = None if dstate is None else _f64(dstate)
        dq = np.zeros((B, H, N, dk), dtype=np.float64)
        dkk = np.zeros((B, H, N, dk), dtype=np.float64)
        dvv = np.zeros((B, H, N, dv), dtype=np.float64)
        ds0 = np.zeros((B, H, dk, dv), dtype=np.float64)
        self.lib.oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 None if s0 is None else _ptr(s0), _ptr(do),
                                 None if ds is None else _ptr(ds),
                                 _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(ds0), B, H, N, dk, dv)
        return dq, dkk, dvv, ds0


def default() -> Oracle:
    """The oracle compiled from retention_oracle.c beside this file."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def threads() -> int:
    return default().threads()


def gamma(h):
    return default().gamma(h)


def parallel(q, k, v, gammas):
    return default().parallel(q, k, v, gammas)


def parallel_rows(q_head, k_head, v_head, g, rows):
    return default().parallel_rows(q_head, k_head, v_head, g, rows)


def recurrent(q, k, v, gammas, state=None):
    return default().recurrent(q, k, v, gammas, state)


def chunkwise(q, k, v, gammas, chunk, state_in=None):
    return default().chunkwise(q, k, v, gammas, chunk, state_in)


def groupnorm(r, weight=None, bias=None, eps=1e-6):
    return default().groupnorm(r, weight, bias, eps)


def rotate(x, theta, n0=0):
    return default().rotate(x, theta, n0)


def backward(q, k, v, gammas, dout, dstate=None, state_in=None):
    return default().backward(q, k, v, gammas, dout, dstate, state_in)
