"""GPU parity of retention_chunkwise_host (q, k, v and outputs in host memory,
slabs of (batch row, head) pairs pipelined over three streams) against the
fp64 oracle: whole-row slabs, slabs of one row's heads (each reading its own
heads' decays), a last short slab, slot reuse, pageable host memory, a caller
buffer, the empty sequence, and the mid workload at full size."""
import numpy as np
import pytest
import torch

from _compare import TOL_BF16, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _host_call(q, k, v, g, C, pin=True, buffer=None):
    if pin:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    out = torch.empty(B, H, N, dv, dtype=torch.bfloat16)
    st = torch.empty(B, H, dk, dv, dtype=torch.float32)
    if pin:
        out, st = out.pin_memory(), st.pin_memory()
    out, st = binding.retention_chunkwise_host(q, k, v, g.to(DEV), C, out=out, state_out=st, buffer=buffer)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return out, st


@pytest.mark.parametrize("B,H,N,dk,dv,C", [
    (3, 2, 300, 128, 128, 64),    # three whole-row slabs, ragged tail
    (1, 16, 520, 64, 128, 128),   # one row: eight slabs of two heads, slots reused
    (9, 2, 130, 128, 64, 64),     # two rows a slab, the last slab one row
    (2, 3, 2048, 256, 192, 128),  # slabs split into segments, padded widths
])
def test_host_matches_oracle(orc, B, H, N, dk, dv, C):
    q, k, v = inputs.qkv(B, H, N, dk, dv, 11, torch.bfloat16)
    gen = torch.Generator().manual_seed(11)
    g = 0.8 + 0.2 * torch.rand(H, generator=gen)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    out, st = _host_call(q, k, v, g, C)
    assert_close(out, ref_out, TOL_BF16, "host out")
    assert_close(st, ref_state, TOL_BF16, "host state")


def test_host_pageable_and_caller_buffer_match():
    B, H, N, dk, dv, C = 2, 4, 700, 128, 128, 64
    q, k, v = inputs.qkv(B, H, N, dk, dv, 12, torch.bfloat16)
    g = binding.gamma_schedule(H)
    o1, s1 = _host_call(q, k, v, g, C)
    o2, s2 = _host_call(q, k, v, g, C, pin=False)
    nbytes = binding.chunkwise_host_buffer_size(B, H, N, dk, dv, C)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o3, s3 = _host_call(q, k, v, g, C, buffer=buf)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    assert torch.equal(o1, o3) and torch.equal(s1, s3)
    with pytest.raises(binding.RetentionError) as e:
        _host_call(q, k, v, g, C, buffer=buf[: nbytes // 2])
    assert e.value.status == binding.RET_ERR_INVALID


def test_host_empty_sequence_zero_state():
    B, H, dk, dv = 2, 3, 128, 64
    z = torch.empty(B, H, 0, dk, dtype=torch.bfloat16)
    zv = torch.empty(B, H, 0, dv, dtype=torch.bfloat16)
    st = torch.full((B, H, dk, dv), 5.0).pin_memory()
    binding.retention_chunkwise_host(z, z, zv, binding.gamma_schedule(H).to(DEV), 64, state_out=st)
    torch.cuda.synchronize()
    assert torch.all(st == 0)


def test_host_mid_workload_full(orc):
    """B=4, H=8, N=2048, d_k=d_v=128, chunk 64 through host buffers, every output and state."""
    B, H, N, dk, dv, C = 4, 8, 2048, 128, 128, 64
    q, k, v = inputs.qkv(B, H, N, dk, dv, 0, torch.bfloat16)
    g = binding.gamma_schedule(H)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    out, st = _host_call(q, k, v, g, C)
    assert_close(out, ref_out, TOL_BF16, "mid host out")
    assert_close(st, ref_state, TOL_BF16, "mid host state")
