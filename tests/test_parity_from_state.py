"""GPU parity of retention_chunkwise_from_state, the chunkwise forward
continued from a given state (chunked prefill), against the fp64 oracle.

The main check splits a sequence at `cut`: the GPU runs only the suffix,
started from the oracle's state after the prefix (rounded to float32), and must
reproduce the oracle's outputs on the suffix of the whole sequence and its
final state.  Cases cover both chunk sizes, d_k = 256, value tiles of 64 and
128, ragged cuts, suffixes long enough to be split into segments, and decays
on both sides of the rescaled/direct switch.  A random starting state is
checked against the oracle's own state_in path, a zero state against
retention_chunkwise bit for bit, and an empty sequence against a copy.
"""
import numpy as np
import pytest
import torch

from _compare import TOL_BF16, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _suffix(x, cut):
    return x[:, :, cut:].contiguous().to(DEV)


CASES = [
    # B, H, N, cut, dk, dv, C
    (1, 2, 300, 128, 128, 128, 64),    # cut on a chunk boundary
    (1, 2, 300, 100, 128, 128, 64),    # ragged cut
    (2, 3, 520, 200, 128, 128, 128),   # C = 128
    (1, 2, 300, 77, 256, 128, 64),     # d_k = 256
    (1, 1, 333, 65, 128, 192, 64),     # three value tiles of 64
    (1, 2, 4096, 1000, 128, 128, 64),  # the suffix is split into segments
    (1, 1, 3000, 1100, 256, 64, 128),  # segments, d_k = 256, value tile 64
]


@pytest.mark.parametrize("B,H,N,cut,dk,dv,C", CASES)
def test_from_state_continues_the_sequence(orc, B, H, N, cut, dk, dv, C):
    q, k, v = inputs.qkv(B, H, N, dk, dv, 5, torch.bfloat16)
    g = binding.gamma_schedule(H)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    _, pre_state = orc.chunkwise(q[:, :, :cut], k[:, :, :cut], v[:, :, :cut], g.double(), C)
    state_in = torch.from_numpy(pre_state).float().to(DEV)
    out, st = binding.retention_chunkwise_from_state(_suffix(q, cut), _suffix(k, cut), _suffix(v, cut),
                                                     g.to(DEV), C, state_in)
    torch.cuda.synchronize()
    assert binding.device_status() == 0, "device wait timed out"
    assert_close(out.cpu(), ref_out[:, :, cut:], TOL_BF16, "continued outputs")
    assert_close(st.cpu(), ref_state, TOL_BF16, "continued state")


# decays on both sides of the rescaled/direct switch for both chunk sizes
ANY_GAMMAS = [0.0, 0.5, 0.85, 0.9, 0.93, 0.99, 1.0]


@pytest.mark.parametrize("N,cut,dv,C", [(300, 90, 128, 64), (2048, 700, 64, 64), (520, 260, 128, 128)])
def test_from_state_any_decay(orc, N, cut, dv, C):
    H, dk = len(ANY_GAMMAS), 128
    g = torch.tensor(ANY_GAMMAS, dtype=torch.float32)
    q, k, v = inputs.qkv(1, H, N, dk, dv, 7, torch.bfloat16)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    _, pre_state = orc.chunkwise(q[:, :, :cut], k[:, :, :cut], v[:, :, :cut], g.double(), C)
    out, st = binding.retention_chunkwise_from_state(_suffix(q, cut), _suffix(k, cut), _suffix(v, cut),
                                                     g.to(DEV), C, torch.from_numpy(pre_state).float().to(DEV))
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert_close(out.cpu(), ref_out[:, :, cut:], TOL_BF16, "continued outputs, any decay")
    assert_close(st.cpu(), ref_state, TOL_BF16, "continued state, any decay")


def test_from_random_state(orc):
    """A starting state unrelated to the inputs (seeded, std 30), against the
    oracle's own state_in path; with segments (N = 2048 at H = 2)."""
    B, H, N, dk, dv, C = 1, 2, 2048, 128, 128, 64
    q, k, v = inputs.qkv(B, H, N, dk, dv, 8, torch.bfloat16)
    g = binding.gamma_schedule(H)
    s0 = 30.0 * np.random.default_rng(9).standard_normal((B, H, dk, dv))
    s0 = s0.astype(np.float32).astype(np.float64)  # exactly what the GPU reads
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C, state_in=s0)
    out, st = binding.retention_chunkwise_from_state(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), C,
                                                     torch.from_numpy(s0).float().to(DEV))
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert_close(out.cpu(), ref_out, TOL_BF16, "outputs from a random state")
    assert_close(st.cpu(), ref_state, TOL_BF16, "state from a random state")


@pytest.mark.parametrize("N", [300, 2048])
def test_zero_state_matches_retention_chunkwise(N):
    """No starting state, or a zero one, gives retention_chunkwise bit for bit."""
    B, H, dk, dv, C = 1, 2, 128, 128, 64
    q, k, v = (x.to(DEV) for x in inputs.qkv(B, H, N, dk, dv, 10, torch.bfloat16))
    g = binding.gamma_schedule(H).to(DEV)
    o1, s1 = binding.retention_chunkwise(q, k, v, g, C)
    o2, s2 = binding.retention_chunkwise_from_state(q, k, v, g, C, None)
    o3, s3 = binding.retention_chunkwise_from_state(q, k, v, g, C, torch.zeros(B, H, dk, dv, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    assert torch.equal(o1, o3) and torch.equal(s1, s3)


def test_from_state_empty_sequence_copies_the_state():
    B, H, dk, dv = 1, 2, 128, 128
    z = torch.empty(B, H, 0, dk, dtype=torch.bfloat16, device=DEV)
    zv = torch.empty(B, H, 0, dv, dtype=torch.bfloat16, device=DEV)
    s0 = torch.randn(B, H, dk, dv, device=DEV)
    out, st = binding.retention_chunkwise_from_state(z, z, zv, binding.gamma_schedule(H).to(DEV), 64, s0)
    torch.cuda.synchronize()
    assert out.shape == (B, H, 0, dv) and torch.equal(st, s0)
