"""GPU parity of retention_groupnorm (the per-(token, head) normalisation of the
retention outputs, heads concatenated per token) against the fp64 oracle.

Inputs are seeded bf16 tensors in the retention output layout with a random
per-row offset and scale (so the mean and the variance both matter), every
lane-count variant of the kernel (dv up to 128, 256, 512 and 1024, including
rows that leave lanes idle), with and without the affine, and the mid
workload's output shape.  The gate is 4e-3 of max|ref| (one bf16 rounding of
outputs of order one; the statistics are fp32), tighter than the general bf16
tolerance.
"""
import numpy as np
import pytest
import torch

from _compare import assert_close
from linear_attention_sequence_02_b300 import binding

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_GN = 4e-3


def _rows(B, H, N, dv, seed):
    rng = np.random.default_rng(seed)
    r = rng.standard_normal((B, H, N, dv)) * rng.uniform(0.1, 30.0, (B, H, N, 1)) \
        + rng.standard_normal((B, H, N, 1)) * 5.0
    return torch.from_numpy(r).to(torch.bfloat16)


@pytest.mark.parametrize("B,H,N,dv", [
    (1, 3, 77, 24),     # 4 lanes a row, the last lane partly idle
    (1, 3, 77, 64),     # 8 lanes a row
    (1, 2, 41, 100),    # not a multiple of 8: a warp a row, 4 channels a lane
    (2, 1, 19, 36),     # not a multiple of 8, most lanes idle
    (2, 2, 33, 192),    # two groups per lane, the second partly idle
    (1, 2, 50, 256),
    (1, 16, 5, 512),
    (1, 1, 9, 1000),    # eight groups per lane, the last partly idle
    (4, 8, 2048, 128),  # the mid workload's output shape
])
def test_groupnorm_matches_oracle(orc, B, H, N, dv):
    r = _rows(B, H, N, dv, 0)
    rng = np.random.default_rng(1)
    w = torch.from_numpy(rng.standard_normal(H * dv)).float()
    b = torch.from_numpy(rng.standard_normal(H * dv)).float()
    ref = orc.groupnorm(r, w.double(), b.double(), 1e-6)
    y = binding.retention_groupnorm(r.to(DEV), w.to(DEV), b.to(DEV), 1e-6)
    torch.cuda.synchronize()
    assert y.shape == (B, N, H, dv)
    assert_close(y.cpu(), ref, TOL_GN, "groupnorm")


def test_groupnorm_without_affine_and_large_eps(orc):
    B, H, N, dv = 2, 4, 100, 128
    r = _rows(B, H, N, dv, 2)
    for eps in (1e-6, 0.5):
        ref = orc.groupnorm(r, None, None, eps)
        y = binding.retention_groupnorm(r.to(DEV), None, None, eps)
        torch.cuda.synchronize()
        assert_close(y.cpu(), ref, TOL_GN, f"groupnorm, no affine, eps {eps}")


def test_groupnorm_empty_sequence_is_a_no_op():
    r = torch.empty(1, 2, 0, 128, dtype=torch.bfloat16, device=DEV)
    y = binding.retention_groupnorm(r)
    torch.cuda.synchronize()
    assert y.shape == (1, 0, 2, 128)
