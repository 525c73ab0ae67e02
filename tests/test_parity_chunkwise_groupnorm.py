"""GPU parity of retention_chunkwise_groupnorm (chunkwise retention with the
per-(token, head) GroupNorm in its output epilogue) against the fp64 oracle
applying its GroupNorm to its chunkwise output.

Cases cover both chunk sizes, value widths 64 and 128 (a head's row in one
CTA), d_k = 256, a sequence split into segments, decays on both sides of the
rescaled/direct switch and the mid workload; the state must equal
retention_chunkwise's bit for bit (same state path), and a head wider than
one value tile must be refused.
"""
import numpy as np
import pytest
import torch

from _compare import TOL_BF16, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _affine(H, dv, seed):
    rng = np.random.default_rng(seed)
    w = torch.from_numpy(1.0 + 0.5 * rng.standard_normal(H * dv)).float()
    b = torch.from_numpy(0.5 * rng.standard_normal(H * dv)).float()
    return w, b


@pytest.mark.parametrize("B,H,N,dk,dv,C", [
    (1, 2, 300, 128, 128, 64),
    (2, 3, 520, 128, 64, 128),
    (1, 2, 2048, 128, 128, 64),   # segments
    (1, 2, 300, 256, 128, 128),   # d_k = 256
    (1, 2, 333, 256, 64, 64),
    (4, 8, 2048, 128, 128, 64),   # the mid workload
    (2, 80, 1024, 64, 64, 64),    # more heads than SMs: the last wave's heads cut into segments
])
def test_chunkwise_groupnorm_matches_oracle(orc, B, H, N, dk, dv, C):
    q, k, v = inputs.qkv(B, H, N, dk, dv, 11, torch.bfloat16)
    g = binding.gamma_schedule(H)
    w, b = _affine(H, dv, 12)
    ref_r, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    ref = orc.groupnorm(ref_r, w.double(), b.double(), 1e-6)
    qd, kd, vd, gd = q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)
    y, st = binding.retention_chunkwise_groupnorm(qd, kd, vd, gd, C, w.to(DEV), b.to(DEV), 1e-6)
    _, st_plain = binding.retention_chunkwise(qd, kd, vd, gd, C)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert y.shape == (B, N, H, dv)
    assert_close(y.cpu(), ref, TOL_BF16, "fused groupnorm out")
    assert_close(st.cpu(), ref_state, TOL_BF16, "fused groupnorm state")
    assert torch.equal(st, st_plain)


def test_chunkwise_groupnorm_any_decay_no_affine(orc):
    gam = [0.0, 0.5, 0.85, 0.9, 0.93, 0.99, 1.0]
    H, N, dk, dv, C = len(gam), 300, 128, 128, 64
    g = torch.tensor(gam, dtype=torch.float32)
    q, k, v = inputs.qkv(1, H, N, dk, dv, 13, torch.bfloat16)
    ref_r, _ = orc.chunkwise(q, k, v, g.double(), C)
    ref = orc.groupnorm(ref_r, None, None, 1e-6)
    y, _ = binding.retention_chunkwise_groupnorm(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), C)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert_close(y.cpu(), ref, TOL_BF16, "fused groupnorm, any decay")


def test_chunkwise_groupnorm_refuses_wide_heads():
    q = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device=DEV)
    v = torch.zeros(1, 1, 64, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(binding.RetentionError) as e:
        binding.retention_chunkwise_groupnorm(q, q, v, binding.gamma_schedule(1).to(DEV), 64)
    assert e.value.status == binding.RET_ERR_UNSUPPORTED
    # a head's row must be a whole value tile without padding: d_v 64 or 128 only
    for dv in (48, 96):
        v = torch.zeros(1, 1, 64, dv, dtype=torch.bfloat16, device=DEV)
        with pytest.raises(binding.RetentionError) as e:
            binding.retention_chunkwise_groupnorm(q, q, v, binding.gamma_schedule(1).to(DEV), 64)
        assert e.value.status == binding.RET_ERR_UNSUPPORTED
