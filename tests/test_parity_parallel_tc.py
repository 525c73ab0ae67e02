"""GPU parity of the tensor-core parallel form (retention_parallel with bf16
tensors and widths that are multiples of 16) against the fp64 oracle's
parallel form: several query and key tiles with ragged tails, every compiled
(d_k tile, value tile) variant, decays from 0 to 1 (including those whose far
key tiles are skipped as exact zeros), and the mid and long-context workloads
(mid on every head, long on every head at sampled rows plus two whole heads).
"""
import numpy as np
import pytest
import torch

from _compare import TOL_BF16, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_parallel(q, k, v, g):
    out = binding.retention_parallel(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV))
    torch.cuda.synchronize()
    assert binding.device_status() == 0, "device wait timed out"
    return out.cpu()


@pytest.mark.parametrize("B,H,N,dk,dv", [
    (1, 2, 300, 128, 128),    # three query tiles, ragged last one; value tile 128
    (2, 2, 257, 64, 48),      # d_k padded to 128, value tile 64 (padded)
    (1, 2, 400, 128, 256),    # value tile 256
    (1, 1, 200, 128, 512),    # two value tiles of 256
    (1, 2, 333, 256, 128),    # d_k 256: value tiles of 64
    (1, 1, 128, 16, 16),      # exactly one tile, narrowest widths
    (1, 2, 1, 128, 128),      # one token
])
def test_parallel_tc_cases(orc, B, H, N, dk, dv):
    q, k, v = inputs.qkv(B, H, N, dk, dv, 11, torch.bfloat16)
    g = binding.gamma_schedule(H)
    ref = orc.parallel(q, k, v, g.double())
    assert_close(run_parallel(q, k, v, g), ref, TOL_BF16, f"parallel tc {B}x{H}x{N} {dk}/{dv}")


def test_parallel_tc_any_decay(orc):
    """Decays 0 (diagonal only), 0.3 and 0.5 (far key tiles exactly zero in
    fp32, skipped), 0.9, 0.99 and 1 (no decay), over eight key tiles."""
    gam = [0.0, 0.3, 0.5, 0.9, 0.99, 1.0]
    H, N, dk, dv = len(gam), 1000, 128, 128
    g = torch.tensor(gam, dtype=torch.float32)
    q, k, v = inputs.qkv(1, H, N, dk, dv, 12, torch.bfloat16)
    ref = orc.parallel(q, k, v, g.double())
    assert_close(run_parallel(q, k, v, g), ref, TOL_BF16, "parallel tc, any decay")


def test_parallel_tc_mid_workload(orc):
    """The mid workload (B=4, H=8, N=2048, d_k=d_v=128) on every head."""
    B, H, N, dk, dv = 4, 8, 2048, 128, 128
    q, k, v = inputs.qkv(B, H, N, dk, dv, 0, torch.bfloat16)
    g = binding.gamma_schedule(H)
    ref = orc.parallel(q, k, v, g.double())
    assert_close(run_parallel(q, k, v, g), ref, TOL_BF16, "parallel tc, mid workload")


def test_parallel_tc_long_workload(orc):
    """The long-context workload (B=1, H=16, N=16384, d_k=128, d_v=256): every
    head at rows spread over the sequence (tile edges included), and heads 0
    and 15 whole against the oracle's chunkwise form (pinned equal to the
    parallel form)."""
    B, H, N, dk, dv = 1, 16, 16384, 128, 256
    q, k, v = inputs.qkv(B, H, N, dk, dv, 0, torch.bfloat16)
    g = binding.gamma_schedule(H)
    out = run_parallel(q, k, v, g)
    rows = [0, 1, 127, 128, 129, 4095, 8191, 8192, 12000, 16254, 16255, 16256, 16383]
    for h in range(H):
        ref = orc.parallel_rows(q[0, h], k[0, h], v[0, h], float(g[h]), rows)
        assert_close(out[0, h, rows], ref, TOL_BF16, f"parallel tc, long workload, head {h} rows")
    heads = [0, H - 1]
    ref, _ = orc.chunkwise(q[:, heads], k[:, heads], v[:, heads], g[heads].double(), 128)
    assert_close(out[:, heads], ref, TOL_BF16, "parallel tc, long workload, whole heads")
