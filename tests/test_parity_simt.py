"""GPU parity of the CUDA-core paths against the fp64 oracle:
fp32 chunkwise / parallel / step (the tiny fp32 workload and edge cases),
bf16 parallel, and the bf16 decode step at the full decode workload
(64 sequences x 16 heads, d_k = 128, d_v = 256, 1024 sequential steps)."""
import numpy as np
import pytest
import torch

from _compare import TOL_BF16, TOL_F32, assert_close, norm_err
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def gammas(H):
    return binding.gamma_schedule(H)


def run_f32_forms(q, k, v, g, chunk):
    qd, kd, vd, gd = q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)
    out_c, st_c = binding.retention_chunkwise_f32(qd, kd, vd, gd, chunk)
    out_p = binding.retention_parallel_f32(qd, kd, vd, gd)
    torch.cuda.synchronize()
    return out_c.cpu(), st_c.cpu(), out_p.cpu()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fp32_three_forms(orc, seed):
    """B=1, H=2, N=256, d_k=d_v=32, chunk=32, fp32: chunkwise, parallel and the
    step loop (recurrent form) each match the fp64 oracle within 1e-4."""
    B, H, N, dk, dv, C = 1, 2, 256, 32, 32, 32
    q, k, v = inputs.qkv(B, H, N, dk, dv, seed, torch.float32)
    g = gammas(H)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    ref_par = orc.parallel(q, k, v, g.double())
    ref_rec, ref_rec_state = orc.recurrent(q, k, v, g.double())
    assert norm_err(ref_par, ref_out) < 1e-12 and norm_err(ref_rec, ref_out) < 1e-12
    out_c, st_c, out_p = run_f32_forms(q, k, v, g, C)
    assert_close(out_c, ref_out, TOL_F32, "chunkwise_f32 out")
    assert_close(st_c, ref_state, TOL_F32, "chunkwise_f32 state")
    assert_close(out_p, ref_out, TOL_F32, "parallel_f32 out")
    # recurrent form: N calls of the step kernel from a zero state
    state = torch.zeros(B, H, dk, dv, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    outs = [binding.retention_step_f32(qd[:, :, n].contiguous(), kd[:, :, n].contiguous(),
                                       vd[:, :, n].contiguous(), state) for n in range(N)]
    torch.cuda.synchronize()
    out_r = torch.stack(outs, dim=2).cpu()
    assert_close(out_r, ref_rec, TOL_F32, "step_f32 outputs")
    assert_close(state.cpu(), ref_rec_state, TOL_F32, "step_f32 state")


@pytest.mark.parametrize("B,H,N,dk,dv,C", [
    (2, 3, 300, 32, 32, 32),    # ragged tail (300 = 9*32 + 12)
    (1, 2, 77, 48, 20, 16),     # dk != dv, odd sizes
    (1, 1, 1, 32, 32, 32),      # single token
    (1, 2, 130, 64, 64, 1),     # chunk 1 is the recurrent form
    (1, 2, 200, 64, 32, 128),   # one full chunk of 128 plus a tail
    (2, 2, 96, 256, 256, 16),   # largest head dims
])
def test_fp32_chunkwise_and_parallel_shapes(orc, B, H, N, dk, dv, C):
    q, k, v = inputs.qkv(B, H, N, dk, dv, 11, torch.float32)
    g = gammas(H)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    out_c, st_c, out_p = run_f32_forms(q, k, v, g, C)
    assert_close(out_c, ref_out, TOL_F32, "chunkwise_f32 out")
    assert_close(st_c, ref_state, TOL_F32, "chunkwise_f32 state")
    assert_close(out_p, ref_out, TOL_F32, "parallel_f32 out")


def test_fp32_empty_sequence_gives_zero_state():
    B, H, dk, dv = 1, 2, 32, 32
    z = torch.empty(B, H, 0, dk, device=DEV)
    zv = torch.empty(B, H, 0, dv, device=DEV)
    st = torch.full((B, H, dk, dv), 7.0, device=DEV)
    out, st = binding.retention_chunkwise_f32(z, z, zv, gammas(H).to(DEV), 32, state_out=st)
    torch.cuda.synchronize()
    assert out.shape == (B, H, 0, dv) and torch.all(st == 0)


def test_fp32_state_continuation(orc):
    """chunkwise on a prefix, then the step kernel on the rest == oracle on the whole."""
    B, H, N, dk, dv, C, cut = 1, 4, 200, 32, 32, 32, 150
    q, k, v = inputs.qkv(B, H, N, dk, dv, 5, torch.float32)
    g = gammas(H)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    _, st = binding.retention_chunkwise_f32(qd[:, :, :cut].contiguous(), kd[:, :, :cut].contiguous(),
                                            vd[:, :, :cut].contiguous(), g.to(DEV), C)
    outs = [binding.retention_step_f32(qd[:, :, n].contiguous(), kd[:, :, n].contiguous(),
                                       vd[:, :, n].contiguous(), st) for n in range(cut, N)]
    torch.cuda.synchronize()
    assert_close(torch.stack(outs, 2).cpu(), ref_out[:, :, cut:], TOL_F32, "continued outputs")
    assert_close(st.cpu(), ref_state, TOL_F32, "continued state")


@pytest.mark.parametrize("B,H,N,dk,dv", [(2, 4, 200, 64, 96), (1, 16, 130, 128, 256)])
def test_bf16_parallel(orc, B, H, N, dk, dv):
    q, k, v = inputs.qkv(B, H, N, dk, dv, 3, torch.bfloat16)
    g = gammas(H)
    ref = orc.parallel(q, k, v, g.double())
    out = binding.retention_parallel(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV))
    torch.cuda.synchronize()
    assert_close(out.cpu(), ref, TOL_BF16, "parallel bf16")


# ---- decode step at the full decode workload ---------------------------------

DEC = dict(T=1024, B=64, H=16, dk=128, dv=256)


@pytest.fixture(scope="module")
def decode_run():
    T, B, H, dk, dv = DEC["T"], DEC["B"], DEC["H"], DEC["dk"], DEC["dv"]
    q, k, v = inputs.decode_steps(T, B, H, dk, dv, 0)
    s0 = inputs.decode_state(B, H, dk, dv, 0)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    state = s0.to(DEV)
    outs = torch.empty(T, B, H, dv, dtype=torch.bfloat16, device=DEV)
    for t in range(T):
        binding.retention_step(qd[t], kd[t], vd[t], state, out=outs[t])
    torch.cuda.synchronize()
    return q, k, v, s0, outs.cpu(), state.cpu()


def test_decode_step_full_workload(orc, decode_run):
    """Every (sequence, head) of the decode workload, all 1024 steps: each
    step's output and the final state against the fp64 recurrent form, in
    groups of 8 sequences (128 heads) so the fp64 outputs stay small."""
    q, k, v, s0, outs, state = decode_run
    g = gammas(DEC["H"]).double()
    per = 8
    for b0 in range(0, DEC["B"], per):
        sl = slice(b0, b0 + per)
        qh, kh, vh = (x[:, sl].permute(1, 2, 0, 3).contiguous() for x in (q, k, v))
        ref_o, ref_s = orc.recurrent(qh, kh, vh, g, state=s0[sl])
        assert_close(outs[:, sl].permute(1, 2, 0, 3), ref_o, TOL_BF16, f"decode outputs, sequences {b0}..{b0 + per - 1}")
        assert_close(state[sl], ref_s, TOL_F32, f"decode state, sequences {b0}..{b0 + per - 1}")


def test_decode_step_is_in_place_and_batched():
    """Heads are independent: one step on a sub-batch equals the same rows of the full step."""
    B, H, dk, dv = 4, 16, 128, 256
    q, k, v = (x[0] for x in inputs.decode_steps(1, B, H, dk, dv, 9))
    s = inputs.decode_state(B, H, dk, dv, 9)
    full_s = s.to(DEV)
    o_full = binding.retention_step(q.to(DEV), k.to(DEV), v.to(DEV), full_s)
    part_s = s[1:3].contiguous().to(DEV)
    o_part = binding.retention_step(q[1:3].contiguous().to(DEV), k[1:3].contiguous().to(DEV),
                                    v[1:3].contiguous().to(DEV), part_s)
    torch.cuda.synchronize()
    assert torch.equal(o_full[1:3].cpu(), o_part.cpu())
    assert torch.equal(full_s[1:3].cpu(), part_s.cpu())
