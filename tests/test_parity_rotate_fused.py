"""GPU parity of the fused position phase rotation: retention_chunkwise_rotated
(q and k turned in shared memory inside the chunkwise kernels) against the
fp64 oracle's rotation followed by its chunkwise form, and
retention_step_rotated (q and k turned as the decode step loads them) against
the oracle's rotation followed by its recurrent form.  Cases cover both chunk
lengths, d_k 128 and 256 and widths padded to the tiles, the segment split
(state-only pre-pass, which turns the keys), a non-zero start position, a
starting state, decays in both the rescaled and the direct form, the mid
workload, and a prefill continued by rotated decode steps."""
import numpy as np
import pytest
import torch

from _compare import TOL_BF16, TOL_F32, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def theta_of(dk, base=10000.0):
    return torch.tensor([base ** (-2.0 * j / dk) for j in range(dk // 2)], dtype=torch.float32)


def oracle_rotated(orc, q, k, v, g, th, n0, C, s0=None):
    rq, rk = orc.rotate(q, th.double(), n0), orc.rotate(k, th.double(), n0)
    return orc.chunkwise(rq, rk, v, g.double(), C, state_in=s0)


@pytest.mark.parametrize("B,H,N,dk,dv,C,n0", [
    (1, 2, 300, 128, 128, 64, 0),      # ragged tail
    (2, 2, 333, 128, 256, 128, 17),    # two value tiles (q, k turned by a separate pass), start position 17
    (1, 2, 300, 256, 128, 64, 5),      # d_k 256: two halves per chunk
    (1, 2, 400, 256, 128, 128, 0),     # d_k 256, chunk 128 (one chunk of Q/K in the ring)
    (1, 3, 250, 64, 96, 64, 1000),     # widths padded to the tiles
    (1, 2, 2048, 128, 128, 64, 3),     # segments on 64-token tiles: the state-only pre-pass turns the keys
    (1, 1, 3000, 256, 64, 128, 77),    # segments with d_k 256
    (2, 80, 1024, 64, 64, 64, 9),      # more heads than SMs: the last wave's heads cut into segments
])
def test_chunkwise_rotated_matches_oracle(orc, B, H, N, dk, dv, C, n0):
    q, k, v = inputs.qkv(B, H, N, dk, dv, 31, torch.bfloat16)
    g = binding.gamma_schedule(H)
    th = theta_of(dk)
    ref_out, ref_st = oracle_rotated(orc, q, k, v, g, th, n0, C)
    out, st = binding.retention_chunkwise_rotated(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), th.to(DEV), n0, C)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert_close(out.cpu(), ref_out, TOL_BF16, "rotated chunkwise out")
    assert_close(st.cpu(), ref_st, TOL_BF16, "rotated chunkwise state")


def test_chunkwise_rotated_any_decay_and_state(orc):
    """Heads in the direct form (decays 0, 0.3, 0.85) and the rescaled form,
    with a starting state, on both chunk lengths."""
    gam = [0.0, 0.3, 0.85, 0.93, 0.99, 1.0]
    H, N, dk, dv = len(gam), 300, 128, 128
    g = torch.tensor(gam, dtype=torch.float32)
    q, k, v = inputs.qkv(1, H, N, dk, dv, 32, torch.bfloat16)
    s0 = inputs.normal((1, H, dk, dv), 33, torch.float32)
    th = theta_of(dk)
    for C in (64, 128):
        ref_out, ref_st = oracle_rotated(orc, q, k, v, g, th, 40, C, s0)
        out, st = binding.retention_chunkwise_rotated(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), th.to(DEV), 40, C,
                                                      state_in=s0.to(DEV))
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        assert_close(out.cpu(), ref_out, TOL_BF16, f"rotated chunkwise out, any decay, chunk {C}")
        assert_close(st.cpu(), ref_st, TOL_BF16, f"rotated chunkwise state, any decay, chunk {C}")


def test_chunkwise_rotated_equals_separate_rotation():
    """The fused call and retention_rotate on q and k followed by
    retention_chunkwise compute the same function; both round the turned
    pairs to bf16, so they agree far inside the oracle tolerance."""
    B, H, N, dk, dv, C = 2, 4, 1000, 128, 128, 64
    q, k, v = (x.to(DEV) for x in inputs.qkv(B, H, N, dk, dv, 34, torch.bfloat16))
    g = binding.gamma_schedule(H).to(DEV)
    th = theta_of(dk).to(DEV)
    fused, st_f = binding.retention_chunkwise_rotated(q, k, v, g, th, 9, C)
    rq, rk = binding.retention_rotate(q, th, 9), binding.retention_rotate(k, th, 9)
    sep, st_s = binding.retention_chunkwise(rq, rk, v, g, C)
    torch.cuda.synchronize()
    assert_close(fused.cpu(), sep.cpu().double(), 5e-3, "fused against separate rotation")
    assert_close(st_f.cpu(), st_s.cpu().double(), 5e-3, "fused against separate rotation, state")


def test_chunkwise_rotated_mid_workload(orc):
    """The mid workload (B=4, H=8, N=2048, d=128, chunk 64), every head."""
    B, H, N, dk, dv, C = 4, 8, 2048, 128, 128, 64
    q, k, v = inputs.qkv(B, H, N, dk, dv, 0, torch.bfloat16)
    g = binding.gamma_schedule(H)
    th = theta_of(dk)
    ref_out, ref_st = oracle_rotated(orc, q, k, v, g, th, 0, C)
    out, st = binding.retention_chunkwise_rotated(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), th.to(DEV), 0, C)
    torch.cuda.synchronize()
    assert_close(out.cpu(), ref_out, TOL_BF16, "rotated chunkwise, mid workload")
    assert_close(st.cpu(), ref_st, TOL_BF16, "rotated chunkwise state, mid workload")


def test_prefill_then_rotated_decode_steps(orc):
    """A rotated chunkwise prefill of 200 tokens, then 24 rotated decode steps
    at positions 200..223: outputs and final state against the oracle's
    rotation of the whole sequence followed by its recurrent form."""
    B, H, dk, dv, C, P, T = 2, 4, 128, 256, 64, 200, 24
    q, k, v = inputs.qkv(B, H, P + T, dk, dv, 35, torch.bfloat16)
    g = binding.gamma_schedule(H)
    th = theta_of(dk)
    _, st = binding.retention_chunkwise_rotated(q[:, :, :P].contiguous().to(DEV), k[:, :, :P].contiguous().to(DEV),
                                                v[:, :, :P].contiguous().to(DEV), g.to(DEV), th.to(DEV), 0, C)
    outs = []
    for t in range(T):
        outs.append(binding.retention_step_rotated(q[:, :, P + t].contiguous().to(DEV),
                                                   k[:, :, P + t].contiguous().to(DEV),
                                                   v[:, :, P + t].contiguous().to(DEV), th.to(DEV), P + t, st))
    torch.cuda.synchronize()
    rq, rk = orc.rotate(q, th.double(), 0), orc.rotate(k, th.double(), 0)
    ref_out, ref_st = orc.recurrent(rq, rk, v, g.double())
    assert_close(torch.stack(outs, 2).cpu(), ref_out[:, :, P:], TOL_BF16, "rotated decode outputs")
    assert_close(st.cpu(), ref_st, TOL_BF16, "rotated decode state")


def test_rotated_validation():
    q = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device=DEV)
    g = binding.gamma_schedule(1).to(DEV)
    th = theta_of(128).to(DEV)
    with pytest.raises(binding.RetentionError) as e:
        binding.retention_chunkwise_rotated(q, q, q, g, th, -1, 64)
    assert e.value.status == binding.RET_ERR_INVALID
    with pytest.raises(binding.RetentionError) as e:
        binding.retention_chunkwise_rotated(q, q, q, g, th, (1 << 24) - 10, 64)
    assert e.value.status == binding.RET_ERR_UNSUPPORTED
    s = torch.zeros(1, 1, 128, 128, device=DEV)
    x = torch.zeros(1, 1, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(binding.RetentionError) as e:
        binding.retention_step_rotated(x, x, x, th, 1 << 24, s)
    assert e.value.status == binding.RET_ERR_UNSUPPORTED
