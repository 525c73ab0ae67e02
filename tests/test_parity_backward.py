"""GPU parity of retention_backward (gradients of the forward with respect to
q, k, v and the starting state) against the fp64 oracle's derivatives.

bf16 calls with d_k, d_v multiples of 16 up to 256 run on the tensor cores
(each gradient a chunkwise forward of permuted operands); the others, and
the fp32 twin, on the CUDA cores.  Cases cover several internal chunks with a ragged last one, widths that are
not multiples of the 32-column slab, d_k != d_v, the widest rows (d_k 256,
d_v 512), a starting state and a final-state gradient (each present or
absent), decays 0, 0.5, 0.9 and 1, the fp32 twin, an empty sequence, and the
mid workload (4 x 8 heads, N 2048, d 128), compared on a subset of heads:
heads are independent, so the oracle on those heads alone gives their exact
gradients.
"""
import pytest
import torch

from _compare import TOL_BF16, TOL_F32, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, H, N, dk, dv, seed, dtype, states):
    q, k, v = inputs.qkv(B, H, N, dk, dv, seed, dtype)
    dout = inputs.normal((B, H, N, dv), 1000 + seed, dtype)
    s0 = inputs.normal((B, H, dk, dv), 2000 + seed, torch.float32) if states else None
    ds = inputs.normal((B, H, dk, dv), 3000 + seed, torch.float32) if states else None
    return q, k, v, dout, s0, ds


def _gpu(x):
    return None if x is None else x.to(DEV)


def _check(orc, q, k, v, g, dout, s0, ds, tol, f32=False, what=""):
    ref = orc.backward(q, k, v, g.double(), dout, ds, s0)
    fn = binding.retention_backward_f32 if f32 else binding.retention_backward
    got = fn(_gpu(q), _gpu(k), _gpu(v), _gpu(g), _gpu(dout), _gpu(ds), _gpu(s0))
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv", "dstate_in"), got, ref):
        assert_close(a.cpu(), b, tol, f"{what} {name}")


@pytest.mark.parametrize("B,H,N,dk,dv,states", [
    (1, 2, 300, 128, 128, False),   # ten internal chunks, ragged last one
    (1, 2, 300, 128, 128, True),
    (2, 3, 77, 64, 32, True),
    (1, 2, 200, 32, 96, True),      # d_k != d_v
    (1, 2, 130, 40, 24, True),      # slabs of 8 columns at the edge
    (1, 1, 100, 256, 512, True),    # widest rows
    (1, 2, 1, 128, 128, True),      # one token
    (1, 2, 4500, 128, 256, True),   # tensor cores, d_k != d_v: two forward shapes, 128-token tiles, segments
    (2, 2, 700, 256, 128, True),    # tensor cores, d_k = 256
    (1, 3, 333, 48, 80, False),     # tensor cores, widths padded to the tiles
    (1, 2, 300, 256, 512, True),    # tensor cores, the 7B widths: dq's and dk's forwards have 512-wide queries
    (1, 2, 1100, 512, 128, True),   # tensor cores, d_k = 512: the dv forward's queries, segments
    (1, 60, 2048, 64, 64, True),    # tensor cores, more heads than a third of the SMs: the time-reversed
                                    # forwards cut their last wave's heads into segments
])
def test_backward_matches_oracle(orc, B, H, N, dk, dv, states):
    q, k, v, dout, s0, ds = _case(B, H, N, dk, dv, 5, torch.bfloat16, states)
    g = binding.gamma_schedule(H)
    _check(orc, q, k, v, g, dout, s0, ds, TOL_BF16, what=f"bf16 {B}x{H}x{N} {dk}/{dv}")


@pytest.mark.parametrize("N", [170, 1000])  # 1000: the time-reversed forwards run in segments
def test_backward_any_decay_and_one_state(orc, N):
    gam = [0.0, 0.5, 0.9, 1.0]
    H, dk, dv = len(gam), 64, 64
    g = torch.tensor(gam, dtype=torch.float32)
    q, k, v, dout, s0, ds = _case(1, H, N, dk, dv, 6, torch.bfloat16, True)
    _check(orc, q, k, v, g, dout, s0, None, TOL_BF16, what="any decay, starting state only")
    _check(orc, q, k, v, g, dout, None, ds, TOL_BF16, what="any decay, final-state gradient only")


@pytest.mark.parametrize("B,H,N,dk,dv", [(1, 2, 150, 64, 64), (1, 3, 65, 32, 48)])
def test_backward_f32_matches_oracle(orc, B, H, N, dk, dv):
    q, k, v, dout, s0, ds = _case(B, H, N, dk, dv, 7, torch.float32, True)
    g = binding.gamma_schedule(H)
    _check(orc, q, k, v, g, dout, s0, ds, TOL_F32, f32=True, what="fp32")


def test_backward_empty_sequence():
    B, H, dk, dv = 1, 2, 64, 32
    z = torch.zeros(B, H, 0, dk, dtype=torch.bfloat16, device=DEV)
    zv = torch.zeros(B, H, 0, dv, dtype=torch.bfloat16, device=DEV)
    ds = inputs.normal((B, H, dk, dv), 9, torch.float32).to(DEV)
    g = binding.gamma_schedule(H).to(DEV)
    _, _, _, ds0 = binding.retention_backward(z, z, zv, g, zv, ds)
    torch.cuda.synchronize()
    assert torch.equal(ds0, ds)
    _, _, _, ds0 = binding.retention_backward(z, z, zv, g, zv)
    torch.cuda.synchronize()
    assert torch.count_nonzero(ds0) == 0


def test_backward_mid_workload_sampled_heads(orc):
    """Full mid workload on the GPU; the oracle's gradients for heads 0 and 7
    of every batch row (the fastest and slowest decay)."""
    B, H, N, dk, dv = 4, 8, 2048, 128, 128
    q, k, v, dout, s0, ds = _case(B, H, N, dk, dv, 8, torch.bfloat16, True)
    g = binding.gamma_schedule(H)
    got = binding.retention_backward(_gpu(q), _gpu(k), _gpu(v), _gpu(g), _gpu(dout), _gpu(ds), _gpu(s0))
    torch.cuda.synchronize()
    heads = [0, H - 1]
    ref = orc.backward(q[:, heads], k[:, heads], v[:, heads], g[heads].double(), dout[:, heads],
                       ds[:, heads], s0[:, heads])
    for name, a, b in zip(("dq", "dk", "dv", "dstate_in"), got, ref):
        assert_close(a[:, heads].cpu(), b, TOL_BF16, f"mid workload {name}")
