"""The failure path of the tensor-core chunkwise kernel on the GPU, without a
fault: retention_test_stall_waits makes one barrier wait in each CTA target a
barrier that nothing completes, with a short limit.  The wait must give up,
the kernel must unwind and return (no trap, no hang), the device status word
must report RET_DEV_WAIT_TIMEOUT, and the next call, with the setting off,
must be clean and correct: the context and the tensor memory are still
usable."""
import pytest
import torch

from _compare import TOL_BF16, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("N", [300, 2048])  # one pass; segments (state-only pre-pass + main pass)
def test_bounded_wait_gives_up_then_next_call_is_clean(orc, N):
    B, H, dk, dv, C = 1, 2, 128, 128, 64
    q, k, v = inputs.qkv(B, H, N, dk, dv, 21, torch.bfloat16)
    g = binding.gamma_schedule(H)
    qd, kd, vd, gd = q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV)
    binding.device_status(clear=True)
    binding.test_stall_waits(2000)  # 2 ms
    try:
        binding.retention_chunkwise(qd, kd, vd, gd, C)
        torch.cuda.synchronize()
    finally:
        binding.test_stall_waits(0)
    assert binding.device_status(clear=True) & binding.RET_DEV_WAIT_TIMEOUT
    out, st = binding.retention_chunkwise(qd, kd, vd, gd, C)
    torch.cuda.synchronize()
    assert binding.device_status(clear=True) == 0
    ref_out, ref_st = orc.chunkwise(q, k, v, g.double(), C)
    assert_close(out.cpu(), ref_out, TOL_BF16, "chunkwise out after a timed-out call")
    assert_close(st.cpu(), ref_st, TOL_BF16, "chunkwise state after a timed-out call")


def test_stall_setting_validation():
    with pytest.raises(binding.RetentionError):
        binding.test_stall_waits(20_000_000)
    binding.test_stall_waits(0)
