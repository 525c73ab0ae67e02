"""GPU parity of retention_rotate (the position phase rotation of queries and
keys) against the fp64 oracle, and of rotation followed by chunkwise retention
against the oracle doing both.

Frequencies are the usual rotary schedule theta_j = 10000^(-2j/d) and random
ones; starting positions 0, 1000 and 100000 exercise the angle reduction (at
position 1e5 the raw angle is 1e5 rad).  The gate for the rotation alone is
4e-3 of max|ref| (one bf16 rounding of values of the input's size).
"""
import numpy as np
import pytest
import torch

from _compare import TOL_BF16, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_ROT = 4e-3


def _theta(d, kind, seed=0):
    if kind == "rope":
        return torch.tensor([10000.0 ** (-2.0 * j / d) for j in range(d // 2)], dtype=torch.float32)
    return torch.from_numpy(np.abs(np.random.default_rng(seed).standard_normal(d // 2))).float()


@pytest.mark.parametrize("B,H,N,d,kind,n0", [
    (4, 8, 2048, 128, "rope", 0),     # the mid workload's queries
    (1, 3, 77, 64, "random", 0),
    (2, 2, 33, 256, "rope", 1000),
    (1, 16, 5, 24, "random", 100000),  # three chunks per row, large positions
    (1, 2, 300, 128, "rope", 100000),
])
def test_rotate_matches_oracle(orc, B, H, N, d, kind, n0):
    x = inputs.qkv(B, H, N, d, d, 3, torch.bfloat16)[0]
    th = _theta(d, kind)
    ref = orc.rotate(x, th.double(), n0)
    y = binding.retention_rotate(x.to(DEV), th.to(DEV), n0)
    torch.cuda.synchronize()
    assert_close(y.cpu(), ref, TOL_ROT, f"rotation ({kind}, n0 {n0})")


def test_rotate_in_place():
    x = inputs.qkv(2, 3, 100, 128, 128, 4, torch.bfloat16)[0].to(DEV)
    th = _theta(128, "rope").to(DEV)
    y = binding.retention_rotate(x, th, 17)
    x2 = x.clone()
    binding.retention_rotate(x2, th, 17, out=x2)
    torch.cuda.synchronize()
    assert torch.equal(y, x2)


def test_rotation_then_chunkwise_retention(orc):
    """Rotated queries and keys through retention_chunkwise match the oracle
    rotating the original inputs and running the chunkwise form on them."""
    B, H, N, dk, dv, C = 1, 4, 520, 128, 128, 64
    q, k, v = inputs.qkv(B, H, N, dk, dv, 6, torch.bfloat16)
    g = binding.gamma_schedule(H)
    th = _theta(dk, "rope")
    ref_out, ref_state = orc.chunkwise(orc.rotate(q, th.double(), 0), orc.rotate(k, th.double(), 0), v,
                                       g.double(), C)
    qr = binding.retention_rotate(q.to(DEV), th.to(DEV), 0)
    kr = binding.retention_rotate(k.to(DEV), th.to(DEV), 0)
    out, st = binding.retention_chunkwise(qr, kr, v.to(DEV), g.to(DEV), C)
    torch.cuda.synchronize()
    assert_close(out.cpu(), ref_out, TOL_BF16, "rotated chunkwise out")
    assert_close(st.cpu(), ref_state, TOL_BF16, "rotated chunkwise state")
