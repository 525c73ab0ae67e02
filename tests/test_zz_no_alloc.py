"""retention_chunkwise_noalloc, the entry point for callers that cannot
allocate device memory (for example serving runtimes with a fixed, pre-planned
device memory budget): it must give the same results as retention_chunkwise
while taking its segment-state scratch from the library's static device array.

Kept in a file that pytest collects last, so a failure here cannot hide the
result of any other test; it passes alone in a fresh process as well as after
the rest of the suite.
"""
import pytest
import torch

from _compare import TOL_BF16, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
STATIC_SCRATCH_BYTES = 8 << 20


def _data(B, H, N, dk, dv, seed):
    q, k, v = (x.to(DEV) for x in inputs.qkv(B, H, N, dk, dv, seed, torch.bfloat16))
    return q, k, v, binding.gamma_schedule(H).to(DEV)


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    # The mid workload: the plan splits each head into segments, so the
    # kernels do use the scratch (a few MiB of segment states).
    B, H, N, dk, dv, C = 4, 8, 2048, 128, 128, 64
    need = binding.chunkwise_workspace_size(B, H, N, dk, dv, C)
    assert 0 < need <= STATIC_SCRATCH_BYTES
    for seed in (0, 1):  # two calls in a row, different inputs
        q, k, v, g = _data(B, H, N, dk, dv, seed)
        ref_out, ref_st = binding.retention_chunkwise(q, k, v, g, C)
        out, st = binding.retention_chunkwise_noalloc(q, k, v, g, C)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        assert_close(out.cpu(), ref_out.cpu(), TOL_BF16, f"noalloc out, call {seed}")
        assert_close(st.cpu(), ref_st.cpu(), TOL_BF16, f"noalloc state, call {seed}")


def test_noalloc_rejects_plans_beyond_static_scratch():
    # Nine wide heads (d_k 256, d_v 1024: 72 value tiles) split into two
    # segments: 9 x 256 x 1024 float32 states, 9.4 MB, beyond the 8 MiB array.
    B, H, N, dk, dv, C = 1, 9, 2048, 256, 1024, 128
    assert binding.chunkwise_workspace_size(B, H, N, dk, dv, C) > STATIC_SCRATCH_BYTES
    q = torch.empty(B, H, N, dk, dtype=torch.bfloat16, device=DEV)
    v = torch.empty(B, H, N, dv, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(binding.RetentionError) as e:
        binding.retention_chunkwise_noalloc(q, q, v, binding.gamma_schedule(H).to(DEV), C)
    assert e.value.status == binding.RET_ERR_UNSUPPORTED
