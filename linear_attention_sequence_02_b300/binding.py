"""ctypes binding of libretention.so: argument marshalling only.

Each function has the name of the C entry point it calls (include/retention.h)
and does nothing but check that the torch tensors it is given match what the
C function expects (device, dtype, shape, contiguity), allocate the outputs
the caller did not pass, and pass raw device pointers plus the current CUDA
stream.  Every step of the computation runs in the library's CUDA kernels.
If the library is missing the call raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libretention.so")
_lock = threading.Lock()
_lib = None

RET_OK = 0
RET_ERR_INVALID = -1
RET_ERR_UNSUPPORTED = -2
RET_ERR_CUDA = -3
RET_DEV_WAIT_TIMEOUT = 0x1

_vp = ctypes.c_void_p
_i = ctypes.c_int
_fp = ctypes.POINTER(ctypes.c_float)

# name -> argument types (all return int status unless noted)
_SIGNATURES = {
    "retention_chunkwise": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
    "retention_chunkwise_from_state": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
    "retention_chunkwise_rotated": [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
    "retention_step_rotated": [_vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _vp],
    "retention_chunkwise_groupnorm": [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _i, _i, _i, _i, _i,
                                      _i, _vp],
    "retention_chunkwise_ws": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp,
                               ctypes.c_size_t, _vp],
    "retention_chunkwise_noalloc": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
    "retention_chunkwise_workspace_size": [_i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)],
    "retention_chunkwise_host": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, ctypes.c_size_t, _vp],
    "retention_chunkwise_host_buffer_size": [_i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)],
    "retention_chunkwise_launches": [_i, _i, _i, _i, _i, _i, ctypes.POINTER(_i)],
    "retention_chunkwise_f32": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
    "retention_parallel": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp],
    "retention_parallel_f32": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp],
    "retention_groupnorm": [_vp, _vp, _vp, _vp, _i, _i, _i, _i, ctypes.c_float, _vp],
    "retention_rotate": [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp],
    "retention_backward": [_vp] * 11 + [_i] * 5 + [_vp],
    "retention_backward_f32": [_vp] * 11 + [_i] * 5 + [_vp],
    "retention_backward_launches": [_i] * 8 + [ctypes.POINTER(_i)],
    "retention_step": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp],
    "retention_step_f32": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp],
    "retention_gamma_schedule": [_i, _fp],
    "retention_device_status": [ctypes.POINTER(ctypes.c_uint), _i],
    "retention_test_stall_waits": [ctypes.c_uint],
    "retention_status_string": [_i],
    "retention_version": [],
}


class RetentionError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: status {status} ({text})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RetentionError("load", RET_ERR_CUDA,
                                     f"{LIB_PATH} is missing; build it with "
                                     "linear_attention_sequence_02_b300.build.build()")
            l = ctypes.CDLL(LIB_PATH)
            for name, args in _SIGNATURES.items():
                fn = getattr(l, name)
                fn.argtypes = args
                fn.restype = ctypes.c_char_p if name == "retention_status_string" else ctypes.c_int
            _lib = l
    return _lib


def _check(fn: str, status: int):
    if status != RET_OK:
        raise RetentionError(fn, status, lib().retention_status_string(status).decode())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _p(t) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gamma_schedule(H: int) -> torch.Tensor:
    """CPU float32 tensor [H]: gamma_h = 1 - 2^(-5-h) as the library computes it."""
    out = (ctypes.c_float * H)()
    _check("retention_gamma_schedule", lib().retention_gamma_schedule(H, out))
    return torch.tensor(list(out), dtype=torch.float32)


def test_stall_waits(microseconds: int) -> None:
    """Failure-path test setting: > 0 makes every later chunkwise launch give
    up one wait after `microseconds` (see retention_test_stall_waits); 0 off."""
    _check("retention_test_stall_waits", lib().retention_test_stall_waits(int(microseconds)))


def device_status(clear: bool = True) -> int:
    flags = ctypes.c_uint(0)
    _check("retention_device_status", lib().retention_device_status(ctypes.byref(flags), int(clear)))
    return int(flags.value)


def _seq_dims(q, v):
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, N, dk = q.shape
    return B, H, N, dk, v.shape[-1]


def _sequence_call(fn, dtype, q, k, v, gamma, out, state_out, want_state, extra, stream):
    B, H, N, dk, dv = _seq_dims(q, v)
    _need(q, "q", dtype, (B, H, N, dk))
    _need(k, "k", dtype, (B, H, N, dk))
    _need(v, "v", dtype, (B, H, N, dv))
    _need(gamma, "gamma", torch.float32, (H,))
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=dtype, device=q.device)
    _need(out, "out", dtype, (B, H, N, dv))
    if state_out is None and want_state:
        state_out = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    if state_out is not None:
        _need(state_out, "state_out", torch.float32, (B, H, dk, dv))
    args = [_p(q), _p(k), _p(v), _p(gamma), _p(out)]
    if state_out is not None or fn.startswith("retention_chunkwise"):
        args.append(_p(state_out))
    args += [B, H, N, dk, dv, *extra]
    return args, out, state_out


def retention_chunkwise(q, k, v, gamma, chunk: int, out=None, state_out=None,
                        want_state: bool = True, stream=None):
    """bf16 chunkwise forward; returns (out, state_out or None)."""
    args, out, state_out = _sequence_call("retention_chunkwise", torch.bfloat16, q, k, v, gamma,
                                          out, state_out, want_state, [int(chunk)], stream)
    _check("retention_chunkwise", lib().retention_chunkwise(*args, _stream(stream)))
    return out, state_out


def retention_chunkwise_from_state(q, k, v, gamma, chunk: int, state_in, out=None, state_out=None,
                                   want_state: bool = True, stream=None):
    """bf16 chunkwise forward continued from `state_in` (float32 [B, H, dk, dv]
    CUDA tensor, or None for zero); returns (out, state_out or None)."""
    args, out, state_out = _sequence_call("retention_chunkwise", torch.bfloat16, q, k, v, gamma,
                                          out, state_out, want_state, [int(chunk)], stream)
    if state_in is not None:
        B, H, _, dk = q.shape
        _need(state_in, "state_in", torch.float32, (B, H, dk, v.shape[-1]))
    # (q, k, v, gamma, state_in, out, state_out, ...)
    args = args[:4] + [_p(state_in)] + args[4:]
    _check("retention_chunkwise_from_state",
           lib().retention_chunkwise_from_state(*args, _stream(stream)))
    return out, state_out


def retention_chunkwise_rotated(q, k, v, gamma, theta, n0: int, chunk: int, state_in=None, out=None,
                                state_out=None, want_state: bool = True, stream=None):
    """bf16 chunkwise forward of q and k turned by the position phase rotation
    (theta float32 [dk/2], token 0 at position n0), the rotation fused into
    the kernels; optional starting state.  Returns (out, state_out or None)."""
    args, out, state_out = _sequence_call("retention_chunkwise", torch.bfloat16, q, k, v, gamma,
                                          out, state_out, want_state, [int(chunk)], stream)
    B, H, N, dk, dv = _seq_dims(q, v)
    _need(theta, "theta", torch.float32, (dk // 2,))
    if state_in is not None:
        _need(state_in, "state_in", torch.float32, (B, H, dk, dv))
    _check("retention_chunkwise_rotated",
           lib().retention_chunkwise_rotated(_p(q), _p(k), _p(v), _p(gamma), _p(theta), int(n0), _p(state_in),
                                             _p(out), _p(state_out), B, H, N, dk, dv, int(chunk), _stream(stream)))
    return out, state_out


def retention_chunkwise_groupnorm(q, k, v, gamma, chunk: int, weight=None, bias=None, eps: float = 1e-6,
                                  out=None, state_out=None, want_state: bool = True, stream=None):
    """bf16 chunkwise forward with the per-(token, head) GroupNorm fused into its
    epilogue; returns (y [B, N, H, dv], state_out or None)."""
    B, H, N, dk, dv = _seq_dims(q, v)
    _need(q, "q", torch.bfloat16, (B, H, N, dk))
    _need(k, "k", torch.bfloat16, (B, H, N, dk))
    _need(v, "v", torch.bfloat16, (B, H, N, dv))
    _need(gamma, "gamma", torch.float32, (H,))
    for t, name in ((weight, "weight"), (bias, "bias")):
        if t is not None:
            _need(t, name, torch.float32, (H * dv,))
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, N, H, dv))
    if state_out is None and want_state:
        state_out = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    if state_out is not None:
        _need(state_out, "state_out", torch.float32, (B, H, dk, dv))
    _check("retention_chunkwise_groupnorm",
           lib().retention_chunkwise_groupnorm(_p(q), _p(k), _p(v), _p(gamma), _p(weight), _p(bias), float(eps),
                                               _p(out), _p(state_out), B, H, N, dk, dv, int(chunk),
                                               _stream(stream)))
    return out, state_out


def retention_chunkwise_ws(q, k, v, gamma, chunk: int, workspace, out=None, state_out=None,
                           want_state: bool = True, stream=None):
    """bf16 chunkwise forward with a caller-owned uint8 CUDA workspace tensor."""
    args, out, state_out = _sequence_call("retention_chunkwise_ws", torch.bfloat16, q, k, v, gamma,
                                          out, state_out, want_state, [int(chunk)], stream)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("retention_chunkwise_ws", lib().retention_chunkwise_ws(*args, ws_ptr, ws_bytes,
                                                                  _stream(stream)))
    return out, state_out


def retention_chunkwise_noalloc(q, k, v, gamma, chunk: int, out=None, state_out=None,
                                want_state: bool = True, stream=None):
    """bf16 chunkwise forward that allocates nothing: the library's static
    device scratch holds the segment states (callers allocate out/state_out)."""
    args, out, state_out = _sequence_call("retention_chunkwise_noalloc", torch.bfloat16, q, k, v,
                                          gamma, out, state_out, want_state, [int(chunk)], stream)
    _check("retention_chunkwise_noalloc", lib().retention_chunkwise_noalloc(*args, _stream(stream)))
    return out, state_out


def _need_host(t, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}")


def chunkwise_host_buffer_size(B, H, N, dk, dv, chunk) -> int:
    n = ctypes.c_size_t(0)
    _check("retention_chunkwise_host_buffer_size",
           lib().retention_chunkwise_host_buffer_size(B, H, N, dk, dv, chunk, ctypes.byref(n)))
    return int(n.value)


def retention_chunkwise_host(q, k, v, gamma, chunk: int, out=None, state_out=None, want_state: bool = True,
                             buffer=None, stream=None):
    """bf16 chunkwise forward of host (CPU, preferably pinned) q, k, v into host
    out / state_out (allocated pinned when None); gamma is a CUDA tensor.  The
    call only enqueues work: synchronise `stream` before reading the outputs.
    `buffer`: optional uint8 CUDA tensor of chunkwise_host_buffer_size bytes."""
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q and v must be [B, H, N, d]")
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    _need_host(q, "q", torch.bfloat16, (B, H, N, dk))
    _need_host(k, "k", torch.bfloat16, (B, H, N, dk))
    _need_host(v, "v", torch.bfloat16, (B, H, N, dv))
    _need(gamma, "gamma", torch.float32, (H,))
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.bfloat16).pin_memory()
    _need_host(out, "out", torch.bfloat16, (B, H, N, dv))
    if state_out is None and want_state:
        state_out = torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory()
    if state_out is not None:
        _need_host(state_out, "state_out", torch.float32, (B, H, dk, dv))
    buf_p = None if buffer is None else buffer.data_ptr()
    buf_n = 0 if buffer is None else buffer.numel() * buffer.element_size()
    _check("retention_chunkwise_host",
           lib().retention_chunkwise_host(_p(q), _p(k), _p(v), _p(gamma), _p(out), _p(state_out), B, H, N, dk, dv,
                                          int(chunk), buf_p, buf_n, _stream(stream)))
    return out, state_out


def chunkwise_workspace_size(B, H, N, dk, dv, chunk) -> int:
    n = ctypes.c_size_t(0)
    _check("retention_chunkwise_workspace_size",
           lib().retention_chunkwise_workspace_size(B, H, N, dk, dv, chunk, ctypes.byref(n)))
    return int(n.value)


def chunkwise_launches(B, H, N, dk, dv, chunk) -> int:
    n = ctypes.c_int(0)
    _check("retention_chunkwise_launches",
           lib().retention_chunkwise_launches(B, H, N, dk, dv, chunk, ctypes.byref(n)))
    return int(n.value)


def retention_chunkwise_f32(q, k, v, gamma, chunk: int, out=None, state_out=None,
                            want_state: bool = True, stream=None):
    """fp32 chunkwise forward on the CUDA cores; returns (out, state_out or None)."""
    args, out, state_out = _sequence_call("retention_chunkwise_f32", torch.float32, q, k, v, gamma,
                                          out, state_out, want_state, [int(chunk)], stream)
    _check("retention_chunkwise_f32", lib().retention_chunkwise_f32(*args, _stream(stream)))
    return out, state_out


def _parallel(fn, dtype, q, k, v, gamma, out, stream):
    B, H, N, dk, dv = _seq_dims(q, v)
    _need(q, "q", dtype, (B, H, N, dk))
    _need(k, "k", dtype, (B, H, N, dk))
    _need(v, "v", dtype, (B, H, N, dv))
    _need(gamma, "gamma", torch.float32, (H,))
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=dtype, device=q.device)
    _need(out, "out", dtype, (B, H, N, dv))
    _check(fn, getattr(lib(), fn)(_p(q), _p(k), _p(v), _p(gamma), _p(out), B, H, N, dk, dv,
                                  _stream(stream)))
    return out


def retention_parallel(q, k, v, gamma, out=None, stream=None):
    """bf16 parallel form; returns out."""
    return _parallel("retention_parallel", torch.bfloat16, q, k, v, gamma, out, stream)


def retention_parallel_f32(q, k, v, gamma, out=None, stream=None):
    """fp32 parallel form; returns out."""
    return _parallel("retention_parallel_f32", torch.float32, q, k, v, gamma, out, stream)


def retention_groupnorm(r, weight=None, bias=None, eps: float = 1e-6, out=None, stream=None):
    """Per-(token, head) normalisation of bf16 retention outputs r [B, H, N, dv];
    returns y [B, N, H, dv] (heads concatenated per token)."""
    if r.dim() != 4:
        raise ValueError("r must be [B, H, N, dv]")
    B, H, N, dv = r.shape
    _need(r, "r", torch.bfloat16, (B, H, N, dv))
    for t, name in ((weight, "weight"), (bias, "bias")):
        if t is not None:
            _need(t, name, torch.float32, (H * dv,))
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=r.device)
    _need(out, "out", torch.bfloat16, (B, N, H, dv))
    _check("retention_groupnorm", lib().retention_groupnorm(_p(r), _p(weight), _p(bias), _p(out), B, H, N,
                                                            dv, float(eps), _stream(stream)))
    return out


def retention_rotate(x, theta, n0: int = 0, out=None, stream=None):
    """Position phase rotation of bf16 queries or keys x [B, H, N, d] with
    frequencies theta (float32 [d/2] CUDA tensor); out may be x (in place)."""
    if x.dim() != 4:
        raise ValueError("x must be [B, H, N, d]")
    B, H, N, d = x.shape
    _need(x, "x", torch.bfloat16, (B, H, N, d))
    _need(theta, "theta", torch.float32, (d // 2,))
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, (B, H, N, d))
    _check("retention_rotate", lib().retention_rotate(_p(x), _p(theta), _p(out), B, H, N, d, int(n0),
                                                      _stream(stream)))
    return out


def _backward(fn, dtype, q, k, v, gamma, dout, dstate, state_in, want_dstate_in, grads, stream):
    B, H, N, dk, dv = _seq_dims(q, v)
    _need(q, "q", dtype, (B, H, N, dk))
    _need(k, "k", dtype, (B, H, N, dk))
    _need(v, "v", dtype, (B, H, N, dv))
    _need(dout, "dout", dtype, (B, H, N, dv))
    _need(gamma, "gamma", torch.float32, (H,))
    for t, name in ((state_in, "state_in"), (dstate, "dstate")):
        if t is not None:
            _need(t, name, torch.float32, (B, H, dk, dv))
    dq, dk_, dv_, ds0 = grads if grads is not None else (None, None, None, None)
    dq = torch.empty_like(q) if dq is None else dq
    dk_ = torch.empty_like(k) if dk_ is None else dk_
    dv_ = torch.empty_like(v) if dv_ is None else dv_
    if ds0 is None and want_dstate_in:
        ds0 = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    _need(dq, "dq", dtype, (B, H, N, dk))
    _need(dk_, "dk", dtype, (B, H, N, dk))
    _need(dv_, "dv", dtype, (B, H, N, dv))
    if ds0 is not None:
        _need(ds0, "dstate_in", torch.float32, (B, H, dk, dv))
    _check(fn, getattr(lib(), fn)(_p(q), _p(k), _p(v), _p(gamma), _p(state_in), _p(dout), _p(dstate),
                                  _p(dq), _p(dk_), _p(dv_), _p(ds0), B, H, N, dk, dv, _stream(stream)))
    return dq, dk_, dv_, ds0


def retention_backward(q, k, v, gamma, dout, dstate=None, state_in=None, want_dstate_in: bool = True,
                       grads=None, stream=None):
    """Gradients of <dout, out> + <dstate, final state> for the bf16 forward
    started from state_in (zero if None); returns (dq, dk, dv, dstate_in),
    dstate_in None when not wanted.  `grads` may pass the four output tensors."""
    return _backward("retention_backward", torch.bfloat16, q, k, v, gamma, dout, dstate, state_in,
                     want_dstate_in, grads, stream)


def backward_launches(B: int, H: int, N: int, dk: int, dv: int, has_state_in: bool = False,
                      has_dstate: bool = False, want_dstate_in: bool = False) -> int:
    """Kernels one bf16 retention_backward call with these sizes enqueues."""
    n = _i(0)
    _check("retention_backward_launches",
           lib().retention_backward_launches(B, H, N, dk, dv, int(has_state_in), int(has_dstate),
                                             int(want_dstate_in), ctypes.byref(n)))
    return n.value


def retention_backward_f32(q, k, v, gamma, dout, dstate=None, state_in=None, want_dstate_in: bool = True,
                           grads=None, stream=None):
    """retention_backward with fp32 q, k, v, dout and gradients."""
    return _backward("retention_backward_f32", torch.float32, q, k, v, gamma, dout, dstate, state_in,
                     want_dstate_in, grads, stream)


def _step(fn, dtype, q, k, v, state, out, stream):
    if q.dim() != 3:
        raise ValueError("q, k, v must be [B, H, d] for a step")
    B, H, dk = q.shape
    dv = v.shape[-1]
    _need(q, "q", dtype, (B, H, dk))
    _need(k, "k", dtype, (B, H, dk))
    _need(v, "v", dtype, (B, H, dv))
    _need(state, "state", torch.float32, (B, H, dk, dv))
    if out is None:
        out = torch.empty((B, H, dv), dtype=dtype, device=q.device)
    _need(out, "out", dtype, (B, H, dv))
    _check(fn, getattr(lib(), fn)(_p(q), _p(k), _p(v), _p(state), _p(out), B, H, dk, dv,
                                  _stream(stream)))
    return out


def retention_step(q, k, v, state, out=None, stream=None):
    """One bf16 decode step; updates `state` in place and returns out."""
    return _step("retention_step", torch.bfloat16, q, k, v, state, out, stream)


def retention_step_rotated(q, k, v, theta, pos: int, state, out=None, stream=None):
    """One bf16 decode step of the token at position `pos`, q and k turned by
    the position phase rotation first; updates `state` in place, returns out."""
    if q.dim() != 3:
        raise ValueError("q, k, v must be [B, H, d] for a step")
    B, H, dk = q.shape
    dv = v.shape[-1]
    _need(q, "q", torch.bfloat16, (B, H, dk))
    _need(k, "k", torch.bfloat16, (B, H, dk))
    _need(v, "v", torch.bfloat16, (B, H, dv))
    _need(theta, "theta", torch.float32, (dk // 2,))
    _need(state, "state", torch.float32, (B, H, dk, dv))
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, H, dv))
    _check("retention_step_rotated",
           lib().retention_step_rotated(_p(q), _p(k), _p(v), _p(theta), int(pos), _p(state), _p(out), B, H, dk, dv,
                                        _stream(stream)))
    return out


def retention_step_f32(q, k, v, state, out=None, stream=None):
    """One fp32 decode step; updates `state` in place and returns out."""
    return _step("retention_step_f32", torch.float32, q, k, v, state, out, stream)
