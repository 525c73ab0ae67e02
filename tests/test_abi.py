"""C-ABI checks that need no GPU: the library builds, loads and exports every
symbol include/retention.h declares; host-side validation rejects bad
arguments before touching the device; the decay schedule is 1 - 2^(-5-h)."""
import ctypes
import os
import re

import numpy as np
import pytest

from linear_attention_sequence_02_b300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "retention.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(retention_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_symbols()
    for must in ("retention_chunkwise", "retention_parallel", "retention_step",
                 "retention_chunkwise_f32", "retention_parallel_f32", "retention_step_f32"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_symbols()) <= set(binding._SIGNATURES)


def test_version_and_status_strings(lib):
    assert lib.retention_version() >= 100
    for st in (0, -1, -2, -3):
        assert lib.retention_status_string(st)


def test_gamma_schedule_matches_oracle(lib, orc):
    H = 24
    g = binding.gamma_schedule(H).numpy()
    want = np.array([orc.gamma(h) for h in range(H)], dtype=np.float64).astype(np.float32)
    assert np.array_equal(g, want)
    # exact in fp32 up to h = 19: the schedule is the formula, not an approximation
    assert np.array_equal(g[:20].astype(np.float64), orc.gamma(np.arange(20)))


P = ctypes.c_void_p(0x1000)       # 16-byte aligned dummy device address (never dereferenced)
P_ODD = ctypes.c_void_p(0x1004)   # misaligned dummy


@pytest.mark.parametrize("args, want", [
    ((None, P, P, P, P, None, 1, 1, 8, 128, 128, 64), binding.RET_ERR_INVALID),   # null q
    ((P, P, P, P, P, None, 0, 1, 8, 128, 128, 64), binding.RET_ERR_INVALID),      # B = 0
    ((P, P, P, P, P, None, 1, -1, 8, 128, 128, 64), binding.RET_ERR_INVALID),     # H < 0
    ((P, P, P, P, P, None, 1, 1, -2, 128, 128, 64), binding.RET_ERR_INVALID),     # N < 0
    ((P, P, P, P, P, None, 1, 1, 8, 0, 128, 64), binding.RET_ERR_INVALID),        # dk = 0
    ((P_ODD, P, P, P, P, None, 1, 1, 8, 128, 128, 64), binding.RET_ERR_INVALID),  # misaligned q
    ((P, P, P, P, P_ODD, None, 1, 1, 8, 128, 128, 64), binding.RET_ERR_INVALID),  # misaligned out
    ((P, P, P, P, P, P_ODD, 1, 1, 8, 128, 128, 64), binding.RET_ERR_INVALID),     # misaligned state
])
def test_chunkwise_rejects_bad_arguments_on_host(lib, args, want):
    assert lib.retention_chunkwise(*args, None) == want
    assert lib.retention_chunkwise_ws(*args, None, 0, None) == want


@pytest.mark.parametrize("dk,dv,chunk,want", [
    (128, 128, 64, binding.RET_OK),
    (16, 16, 32, binding.RET_OK),              # narrowest widths, chunk 32
    (256, 1024, 128, binding.RET_OK),          # widest
    (192, 208, 64, binding.RET_OK),            # multiples of 16 below the tiles
    (128, 128, 16, binding.RET_ERR_UNSUPPORTED),    # chunk outside {32, 64, 128}
    (128, 128, 96, binding.RET_ERR_UNSUPPORTED),
    (128, 128, 256, binding.RET_ERR_UNSUPPORTED),
    (72, 128, 64, binding.RET_ERR_UNSUPPORTED),     # d_k not a multiple of 16
    (8, 128, 64, binding.RET_ERR_UNSUPPORTED),
    (528, 128, 64, binding.RET_ERR_UNSUPPORTED),    # d_k above 512
    (128, 24, 64, binding.RET_ERR_UNSUPPORTED),     # d_v not a multiple of 16
    (128, 1040, 64, binding.RET_ERR_UNSUPPORTED),   # d_v above 1024
])
def test_chunkwise_shape_support(lib, dk, dv, chunk, want):
    """The bf16 chunkwise shapes: chunk 32, 64 or 128; d_k a multiple of 16 up
    to 256; d_v a multiple of 16 up to 1024; anything else is refused on the
    host with RET_ERR_UNSUPPORTED (checked through the host-only planning
    calls, which share the chunkwise calls' shape rules)."""
    size = ctypes.c_size_t(0)
    n = ctypes.c_int(0)
    assert lib.retention_chunkwise_workspace_size(2, 4, 1000, dk, dv, chunk, ctypes.byref(size)) == want
    assert lib.retention_chunkwise_launches(2, 4, 1000, dk, dv, chunk, ctypes.byref(n)) == want
    if want == binding.RET_OK:
        assert n.value in (1, 2)


def test_backward_launch_counts(lib):
    """Kernels per bf16 gradient call: tensor-core widths run three forwards
    (plus the state kernels when states are given); other widths take one
    CUDA-core launch."""
    n = ctypes.c_int(0)
    f = lib.retention_backward_launches
    assert f(4, 8, 2048, 128, 128, 0, 0, 0, ctypes.byref(n)) == binding.RET_OK and n.value == 3
    assert f(4, 8, 2048, 128, 128, 1, 1, 1, ctypes.byref(n)) == binding.RET_OK and n.value == 6
    assert f(1, 16, 16384, 128, 256, 0, 0, 0, ctypes.byref(n)) == binding.RET_OK and n.value >= 4
    # the 7B widths: dq's and dk's forwards in two 256-column parts each, plus their sums
    assert f(8, 16, 8192, 256, 512, 0, 0, 0, ctypes.byref(n)) == binding.RET_OK and n.value >= 3 * 1 + 2 * 2
    assert f(1, 2, 100, 40, 24, 1, 1, 1, ctypes.byref(n)) == binding.RET_OK and n.value == 1
    assert f(1, 2, 0, 128, 128, 0, 0, 1, ctypes.byref(n)) == binding.RET_OK and n.value == 1
    assert f(0, 2, 10, 128, 128, 0, 0, 1, ctypes.byref(n)) == binding.RET_ERR_INVALID


def test_f32_and_parallel_and_step_validation(lib):
    assert lib.retention_chunkwise_f32(P, P, P, P, P, None, 1, 1, 8, 32, 32, 0, None) == binding.RET_ERR_INVALID
    assert lib.retention_chunkwise_f32(P, P, P, P, P, None, 1, 1, 8, 32, 32, 129, None) == binding.RET_ERR_UNSUPPORTED
    assert lib.retention_chunkwise_f32(P, P, P, P, P, None, 1, 1, 8, 300, 32, 32, None) == binding.RET_ERR_UNSUPPORTED
    assert lib.retention_parallel(None, P, P, P, P, 1, 1, 8, 32, 32, None) == binding.RET_ERR_INVALID
    assert lib.retention_parallel_f32(P, P, P, P, P, 1, 1, 8, 32, 512, None) == binding.RET_ERR_UNSUPPORTED
    assert lib.retention_step(P, P, P, None, P, 1, 1, 32, 32, None) == binding.RET_ERR_INVALID
    assert lib.retention_step(P, P, P, P, P, 1, 1, 32, 30, None) == binding.RET_ERR_UNSUPPORTED
    assert lib.retention_step_f32(P, P, P, P, P_ODD, 1, 1, 32, 32, None) == binding.RET_ERR_INVALID
    assert lib.retention_gamma_schedule(0, None) == binding.RET_ERR_INVALID
    assert lib.retention_device_status(None, 0) == binding.RET_ERR_INVALID


def test_chunkwise_from_state_validation(lib):
    """Checked on the host before anything is enqueued: the starting state must
    be 16-byte aligned and must not be the state_out buffer; the checks of
    retention_chunkwise apply as well."""
    P2 = ctypes.c_void_p(0x2000)
    fs = lib.retention_chunkwise_from_state
    # (q, k, v, gamma, state_in, out, state_out, B, H, N, dk, dv, chunk, stream)
    assert fs(P, P, P, P, P_ODD, P, P2, 1, 1, 8, 128, 128, 64, None) == binding.RET_ERR_INVALID
    assert fs(P, P, P, P, P2, P, P2, 1, 1, 8, 128, 128, 64, None) == binding.RET_ERR_INVALID
    assert fs(None, P, P, P, P2, P, None, 1, 1, 8, 128, 128, 64, None) == binding.RET_ERR_INVALID
    assert fs(P, P, P, P, P2, P_ODD, None, 1, 1, 8, 128, 128, 64, None) == binding.RET_ERR_INVALID


def test_groupnorm_validation(lib):
    gn = lib.retention_groupnorm
    # (r, weight, bias, y, B, H, N, dv, eps, stream)
    assert gn(None, None, None, P, 1, 1, 4, 128, 1e-6, None) == binding.RET_ERR_INVALID
    assert gn(P_ODD, None, None, P, 1, 1, 4, 128, 1e-6, None) == binding.RET_ERR_INVALID
    assert gn(P, None, None, P, 1, 1, 4, 128, -1.0, None) == binding.RET_ERR_INVALID
    assert gn(P, None, None, P, 1, 1, 4, 128, float("nan"), None) == binding.RET_ERR_INVALID
    assert gn(P, None, None, P, 0, 1, 4, 128, 1e-6, None) == binding.RET_ERR_INVALID
    assert gn(P, ctypes.c_void_p(0x1002), None, P, 1, 1, 4, 128, 1e-6, None) == binding.RET_ERR_INVALID
    assert gn(P, None, None, P, 1, 1, 4, 130, 1e-6, None) == binding.RET_ERR_UNSUPPORTED
    assert gn(P, None, None, P, 1, 1, 4, 2048, 1e-6, None) == binding.RET_ERR_UNSUPPORTED


def test_rotate_validation(lib):
    rot = lib.retention_rotate
    # (x, theta, y, B, H, N, d, n0, stream)
    assert rot(None, P, P, 1, 1, 4, 128, 0, None) == binding.RET_ERR_INVALID
    assert rot(P_ODD, P, P, 1, 1, 4, 128, 0, None) == binding.RET_ERR_INVALID
    assert rot(P, P, P, 1, 1, 4, 128, -1, None) == binding.RET_ERR_INVALID
    assert rot(P, P, P, 1, 1, 4, 124, 0, None) == binding.RET_ERR_UNSUPPORTED
    assert rot(P, P, P, 1, 1, 4, 128, (1 << 24) - 3, None) == binding.RET_ERR_UNSUPPORTED


def test_chunkwise_groupnorm_validation(lib):
    fn = lib.retention_chunkwise_groupnorm
    # (q, k, v, gamma, weight, bias, eps, out, state_out, B, H, N, dk, dv, chunk, stream)
    assert fn(P, P, P, P, None, None, -1.0, P, None, 1, 1, 8, 128, 128, 64, None) == binding.RET_ERR_INVALID
    assert fn(P, P, P, P, ctypes.c_void_p(0x1008), None, 1e-6, P, None, 1, 1, 8, 128, 128, 64, None) == \
        binding.RET_ERR_INVALID
    assert fn(None, P, P, P, None, None, 1e-6, P, None, 1, 1, 8, 128, 128, 64, None) == binding.RET_ERR_INVALID


def test_backward_validation(lib):
    """Host checks of the gradient call: required pointers present and
    aligned, the starting-state gradient not written over dstate or state_in,
    no gradient overlapping an input or another gradient, widths above 512
    or not a multiple of 4 refused."""
    # distinct, non-overlapping fake device addresses (never dereferenced)
    Q, K, V, G, DO, DQ, DK, DV = (ctypes.c_void_p((i + 1) << 32) for i in range(8))
    P2, P3 = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    for fn in (lib.retention_backward, lib.retention_backward_f32):
        # (q, k, v, gamma, state_in, dout, dstate, dq, dk, dv, dstate_in, B, H, N, dk, dv, stream)
        def call(q=Q, k=K, v=V, gm=G, s0=None, do=DO, ds=None, dq=DQ, dk_=DK, dv_=DV, ds0=None,
                 B=1, H=1, N=8, dk=64, dv=64):
            return fn(q, k, v, gm, s0, do, ds, dq, dk_, dv_, ds0, B, H, N, dk, dv, None)
        assert call(q=None) == binding.RET_ERR_INVALID
        assert call(do=None) == binding.RET_ERR_INVALID
        assert call(dq=None) == binding.RET_ERR_INVALID
        assert call(dv_=P_ODD) == binding.RET_ERR_INVALID
        assert call(s0=P_ODD) == binding.RET_ERR_INVALID
        assert call(ds=P2, ds0=P2) == binding.RET_ERR_INVALID
        assert call(s0=P3, ds=P2, ds0=P3) == binding.RET_ERR_INVALID
        assert call(H=0) == binding.RET_ERR_INVALID
        assert call(N=-1) == binding.RET_ERR_INVALID
        # a gradient written over an input, or over another gradient, in whole or in part
        for bad in (dict(dq=Q), dict(dk_=K), dict(dv_=V), dict(dv_=DO), dict(dq=DO), dict(dk_=DQ),
                    dict(dv_=ctypes.c_void_p(Q.value + 16)), dict(dq=ctypes.c_void_p(DV.value + 512))):
            assert call(**bad) == binding.RET_ERR_INVALID, bad
        # adjacent but disjoint ranges are fine (fails only later, on the width)
        q_bytes = 8 * 64 * (2 if fn is lib.retention_backward else 4)
        assert call(dq=ctypes.c_void_p(Q.value + q_bytes), dk=64, dv=640) == binding.RET_ERR_UNSUPPORTED
        assert call(dv=640) == binding.RET_ERR_UNSUPPORTED
        assert call(dk=1024) == binding.RET_ERR_UNSUPPORTED
        assert call(dk=66) == binding.RET_ERR_UNSUPPORTED
        # nothing to do: no tokens and no starting-state gradient wanted
        assert fn(None, None, None, None, None, None, None, None, None, None, None, 1, 1, 0, 64, 64, None) == \
            binding.RET_OK


def test_host_entry_validation_and_buffer_size(lib):
    """retention_chunkwise_host rejects missing or misaligned arguments before
    it touches the device; its buffer size covers three slab slots."""
    f = lib.retention_chunkwise_host
    assert f(None, P, P, P, P, None, 1, 1, 8, 64, 64, 64, None, 0, None) == binding.RET_ERR_INVALID
    assert f(P, P, P, P, P, None, 0, 1, 8, 64, 64, 64, None, 0, None) == binding.RET_ERR_INVALID
    assert f(P, P, P, P, P, None, 1, 1, 8, 64, 64, 64, P_ODD, 1 << 20, None) == binding.RET_ERR_INVALID
    n = ctypes.c_size_t(0)
    g = lib.retention_chunkwise_host_buffer_size
    assert g(8, 16, 8192, 256, 512, 128, ctypes.byref(n)) == binding.RET_OK
    # one batch row a slab: q, k, v, out and the state of 16 heads, three times
    per_slot = 16 * 8192 * (2 * 256 + 2 * 512) * 2 + 16 * 256 * 512 * 4
    assert 3 * per_slot <= n.value < 3 * per_slot + (64 << 20)
    assert g(1, 2, 100, 72, 64, 64, ctypes.byref(n)) == binding.RET_ERR_UNSUPPORTED
    assert g(1, 2, 100, 64, 64, 64, None) == binding.RET_ERR_INVALID
