"""GPU parity of the tensor-core chunkwise forward (bf16 q/k/v/out, fp32 state)
against the fp64 oracle: multi-tile cases with ragged tails over every
compiled (chunk, d_k, value-tile) variant, the segment-split path, guard
bands around the outputs, continuation into the decode step, and the three
bf16 workloads at full size (mid and long-context on every head, 7B-shaped on
two whole batch rows and sampled rows of every other head)."""
import numpy as np
import pytest
import torch

from _compare import TOL_BF16, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gammas(H):
    return binding.gamma_schedule(H)


def run_chunkwise(q, k, v, g, chunk):
    out, st = binding.retention_chunkwise(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), chunk)
    torch.cuda.synchronize()
    assert binding.device_status() == 0, "device wait timed out"
    return out.cpu(), st.cpu()


CASES = [
    # B, H, N, dk, dv, chunk
    (1, 2, 293, 128, 128, 64),    # C=64, value tile 128, ragged tail
    (1, 2, 300, 128, 64, 64),     # C=64, value tile 64
    (2, 3, 520, 128, 128, 128),   # C=128, two value tiles, ragged
    (1, 2, 300, 256, 128, 64),    # d_k = 256, C=64
    (1, 2, 300, 256, 128, 128),   # d_k = 256, C=128 (single stage)
    (1, 1, 64, 128, 192, 64),     # exactly one chunk, three value tiles
    (1, 1, 1, 128, 64, 128),      # one token
    (1, 2, 2048, 128, 128, 64),   # split into segments (pre-pass + combine)
    (1, 2, 4096, 128, 256, 128),  # segments with C=128 and two value tiles
    (1, 1, 3000, 256, 64, 128),   # segments, d_k = 256, ragged
    # widths below the kernel's tiles (zero-padded by the loads) and chunk 32
    (1, 2, 300, 64, 64, 64),      # d_k = 64: half of each 128-column Q/K box is padding
    (2, 2, 333, 16, 16, 64),      # the narrowest widths
    (1, 3, 250, 192, 96, 128),    # d_k = 192 on the 256 tiles; d_v = 96: second value tile half padding
    (1, 2, 2100, 48, 208, 64),    # segments, d_v = 208 (four 64-wide tiles, the last one 16 wide)
    (1, 2, 301, 128, 128, 32),    # chunk 32 (runs on 64-token tiles)
    (1, 1, 2500, 80, 144, 32),    # chunk 32 with segments and padded widths
    # query/key widths above 256: 512-wide tiles, 64-token and 64-wide value tiles
    (1, 2, 300, 512, 128, 128),   # chunk 128 asked for, run on 64-token tiles
    (2, 2, 333, 384, 64, 64),     # d_k = 384: the last 128 columns padding
    (1, 1, 2100, 512, 80, 64),    # segments, padded value tile
]


@pytest.mark.parametrize("B,H,N,dk,dv,C", CASES)
def test_chunkwise_bf16_cases(orc, B, H, N, dk, dv, C):
    q, k, v = inputs.qkv(B, H, N, dk, dv, 1, torch.bfloat16)
    g = gammas(H)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    out, st = run_chunkwise(q, k, v, g, C)
    assert_close(out, ref_out, TOL_BF16, "chunkwise out")
    assert_close(st, ref_state, TOL_BF16, "chunkwise state")


# Decays outside the schedule.  Each head takes the rescaled form when
# gamma^chunk >= 2^-14 and the direct form otherwise; the values straddle that
# switch for both chunk sizes (2^(-14/64) = 0.8595, 2^(-14/128) = 0.9270) and
# include the ends of [0, 1].
ANY_GAMMAS = [0.0, 0.3, 0.5, 0.85, 0.9, 0.92, 0.93, 0.99, 1.0]


@pytest.mark.parametrize("N,dk,dv,C", [
    (300, 128, 128, 64),
    (520, 128, 128, 128),
    (300, 256, 128, 128),
    (2048, 128, 64, 64),   # split into segments: state-only pre-pass in both forms
])
def test_chunkwise_any_decay(orc, N, dk, dv, C):
    H = len(ANY_GAMMAS)
    g = torch.tensor(ANY_GAMMAS, dtype=torch.float32)
    q, k, v = inputs.qkv(1, H, N, dk, dv, 3, torch.bfloat16)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    out, st = run_chunkwise(q, k, v, g, C)
    assert_close(out, ref_out, TOL_BF16, "chunkwise out, any decay")
    assert_close(st, ref_state, TOL_BF16, "chunkwise state, any decay")


def test_chunkwise_empty_sequence_zero_state():
    B, H, dk, dv = 1, 2, 128, 128
    z = torch.empty(B, H, 0, dk, dtype=torch.bfloat16, device=DEV)
    zv = torch.empty(B, H, 0, dv, dtype=torch.bfloat16, device=DEV)
    st = torch.full((B, H, dk, dv), 3.0, device=DEV)
    out, st = binding.retention_chunkwise(z, z, zv, gammas(H).to(DEV), 64, state_out=st)
    torch.cuda.synchronize()
    assert out.shape == (B, H, 0, dv) and torch.all(st == 0)


def test_chunkwise_unsupported_shapes_are_rejected():
    """Widths that are not multiples of 16 and chunks outside {32, 64, 128}."""
    q = torch.zeros(1, 1, 64, 72, dtype=torch.bfloat16, device=DEV)
    v = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(binding.RetentionError) as e:
        binding.retention_chunkwise(q, q, v, gammas(1).to(DEV), 64)
    assert e.value.status == binding.RET_ERR_UNSUPPORTED
    q = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(binding.RetentionError) as e:
        binding.retention_chunkwise(q, q, v, gammas(1).to(DEV), 16)
    assert e.value.status == binding.RET_ERR_UNSUPPORTED


def test_chunkwise_guard_bands_untouched():
    """Outputs written through TMA stay inside their tensors (ragged tail included)."""
    B, H, N, dk, dv, C = 1, 3, 333, 128, 128, 64
    q, k, v = (x.to(DEV) for x in inputs.qkv(B, H, N, dk, dv, 2, torch.bfloat16))
    guard = 4096
    n_out = B * H * N * dv
    buf = torch.full((guard + n_out + guard,), -7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[guard:guard + n_out].view(B, H, N, dv)
    n_st = B * H * dk * dv
    sbuf = torch.full((guard + n_st + guard,), -7.0, dtype=torch.float32, device=DEV)
    st = sbuf[guard:guard + n_st].view(B, H, dk, dv)
    binding.retention_chunkwise(q, k, v, gammas(H).to(DEV), C, out=out, state_out=st)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == -7.0) and torch.all(buf[guard + n_out:] == -7.0)
    assert torch.all(sbuf[:guard] == -7.0) and torch.all(sbuf[guard + n_st:] == -7.0)
    assert torch.isfinite(out.float()).all()


def test_workspace_variant_matches():
    B, H, N, dk, dv, C = 1, 2, 2048, 128, 128, 64
    q, k, v = (x.to(DEV) for x in inputs.qkv(B, H, N, dk, dv, 4, torch.bfloat16))
    g = gammas(H).to(DEV)
    nbytes = binding.chunkwise_workspace_size(B, H, N, dk, dv, C)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o1, s1 = binding.retention_chunkwise(q, k, v, g, C)
    o2, s2 = binding.retention_chunkwise_ws(q, k, v, g, C, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    with pytest.raises(binding.RetentionError):
        binding.retention_chunkwise_ws(q, k, v, g, C, ws[: nbytes // 2])


def test_last_wave_split(orc):
    """More (head, value tile) units than SMs, not a whole number of waves: the
    units of the last wave are cut into segments (state-only pre-pass, then
    the main pass), the others run whole.  The same call with no workspace
    runs every unit whole; with a starting state; and through the static
    scratch entry point."""
    B, H, N, dk, dv, C = 2, 80, 3072, 64, 64, 64
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = B * H
    q, k, v = inputs.qkv(B, H, N, dk, dv, 5, torch.bfloat16)
    gen = torch.Generator().manual_seed(5)
    g = 0.8 + 0.2 * torch.rand(H, generator=gen)
    g[0], g[1], g[2] = 0.0, 1.0, 0.5
    if units > sms and units % sms and sms // (units % sms) >= 2:
        assert binding.chunkwise_launches(B, H, N, dk, dv, C) == 2
        assert binding.chunkwise_workspace_size(B, H, N, dk, dv, C) > 0
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    out, st = run_chunkwise(q, k, v, g, C)
    assert_close(out, ref_out, TOL_BF16, "last-wave split out")
    assert_close(st, ref_state, TOL_BF16, "last-wave split state")
    qd, kd, vd, gd = q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)
    o2, s2 = binding.retention_chunkwise_ws(qd, kd, vd, gd, C, None)
    o3, s3 = binding.retention_chunkwise_noalloc(qd, kd, vd, gd, C)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert_close(o2.cpu(), ref_out, TOL_BF16, "every unit whole, out")
    assert_close(s2.cpu(), ref_state, TOL_BF16, "every unit whole, state")
    assert torch.equal(o3.cpu(), out) and torch.equal(s3.cpu(), st)
    # continued from a state: the prefix's state feeds the rest of the sequence
    cut = 1024
    _, s_pre = binding.retention_chunkwise(qd[:, :, :cut].contiguous(), kd[:, :, :cut].contiguous(),
                                           vd[:, :, :cut].contiguous(), gd, C)
    o4, s4 = binding.retention_chunkwise_from_state(qd[:, :, cut:].contiguous(), kd[:, :, cut:].contiguous(),
                                                    vd[:, :, cut:].contiguous(), gd, C, s_pre)
    torch.cuda.synchronize()
    assert_close(o4.cpu(), ref_out[:, :, cut:], TOL_BF16, "continued out")
    assert_close(s4.cpu(), ref_state, TOL_BF16, "continued state")


def test_chunkwise_then_decode_continuation(orc):
    """state_out of a prefix, advanced by retention_step, reproduces the whole sequence."""
    B, H, N, dk, dv, C, cut = 1, 4, 200, 128, 256, 64, 160
    q, k, v = inputs.qkv(B, H, N, dk, dv, 6, torch.bfloat16)
    g = gammas(H)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    out_pre, st = binding.retention_chunkwise(qd[:, :, :cut].contiguous(), kd[:, :, :cut].contiguous(),
                                              vd[:, :, :cut].contiguous(), g.to(DEV), C)
    outs = [binding.retention_step(qd[:, :, n].contiguous(), kd[:, :, n].contiguous(),
                                   vd[:, :, n].contiguous(), st) for n in range(cut, N)]
    torch.cuda.synchronize()
    assert_close(out_pre.cpu(), ref_out[:, :, :cut], TOL_BF16, "prefix")
    assert_close(torch.stack(outs, 2).cpu(), ref_out[:, :, cut:], TOL_BF16, "continued outputs")
    assert_close(st.cpu(), ref_state, TOL_BF16, "continued state")


# ---- the three bf16 workloads at full size --------------------------------------

def test_mid_workload_full(orc):
    """B=4, H=8, N=2048, d_k=d_v=128, chunk=64: every output and state checked."""
    B, H, N, dk, dv, C = 4, 8, 2048, 128, 128, 64
    for seed in (0, 1, 2):
        q, k, v = inputs.qkv(B, H, N, dk, dv, seed, torch.bfloat16)
        g = gammas(H)
        ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
        out, st = run_chunkwise(q, k, v, g, C)
        assert_close(out, ref_out, TOL_BF16, f"mid out seed {seed}")
        assert_close(st, ref_state, TOL_BF16, f"mid state seed {seed}")


def _sampled_heads_check(orc, q, k, v, g, out, st, C, heads, rows_per_other=6, rng_seed=0):
    """Full oracle on `heads`; single rows (parallel-form definition) on every other head."""
    B, H = q.shape[:2]
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref_o, ref_s = orc.chunkwise(q[sl], k[sl], v[sl], g[h:h + 1].double(), C)
        assert_close(out[sl], ref_o, TOL_BF16, f"out ({b},{h})")
        assert_close(st[sl], ref_s, TOL_BF16, f"state ({b},{h})")
    rng = np.random.default_rng(rng_seed)
    N = q.shape[2]
    for b in range(B):
        for h in range(H):
            rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, rows_per_other)]))
            ref = orc.parallel_rows(q[b, h], k[b, h], v[b, h], float(g[h]), rows)
            assert_close(out[b, h, rows], ref, TOL_BF16, f"rows ({b},{h})", per_head=False)


def test_long_context_workload_full(orc):
    """B=1, H=16, N=16384, d_k=128, d_v=256, chunk=128: every output and state
    of every head against the oracle's chunkwise form."""
    B, H, N, dk, dv, C = 1, 16, 16384, 128, 256, 128
    q, k, v = inputs.qkv(B, H, N, dk, dv, 0, torch.bfloat16)
    g = gammas(H)
    out, st = run_chunkwise(q, k, v, g, C)
    ref_out, ref_state = orc.chunkwise(q, k, v, g.double(), C)
    assert_close(out, ref_out, TOL_BF16, "long out")
    assert_close(st, ref_state, TOL_BF16, "long state")


def test_7b_shaped_workload(orc):
    """B=8, H=16, N=8192, d_k=256, d_v=512, chunk=128: batch rows 0 and 7 in
    full (all 16 heads, every token and state), and rows of every other head
    against the parallel-form definition."""
    B, H, N, dk, dv, C = 8, 16, 8192, 256, 512, 128
    q, k, v = inputs.qkv(B, H, N, dk, dv, 0, torch.bfloat16)
    g = gammas(H)
    out, st = run_chunkwise(q, k, v, g, C)
    for b in (0, B - 1):
        sl = slice(b, b + 1)
        ref_o, ref_s = orc.chunkwise(q[sl], k[sl], v[sl], g.double(), C)
        assert_close(out[sl], ref_o, TOL_BF16, f"7B out, batch row {b}")
        assert_close(st[sl], ref_s, TOL_BF16, f"7B state, batch row {b}")
    _sampled_heads_check(orc, q, k, v, g, out, st, C, heads=[], rows_per_other=3)
