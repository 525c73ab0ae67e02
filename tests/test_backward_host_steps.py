"""CPU check of backward_kernel's index arithmetic (no GPU).

tests/host_steps/backward_steps.cu includes csrc/backward.cu and runs the
kernel's phase functions (they are __host__ __device__) for every CTA and
thread index on the CPU, phase by phase as the kernel's barriers order them,
under AddressSanitizer and with NaN-filled shared memory.  Its gradients are
compared with the fp64 oracle at the GPU tests' tolerances, so a wrong index,
an overrun of a shared-memory region or a read of an unwritten slot fails
here before the kernel runs on a GPU.  This is a test of the kernel source;
the library never runs its kernels on the CPU.
"""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest
import torch

from _compare import TOL_BF16, TOL_F32, assert_close
from linear_attention_sequence_02_b300 import binding, inputs

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "host_steps", "backward_steps.cu")
CSRC = os.path.join(ROOT, "linear_attention_sequence_02_b300", "csrc")
NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"


@pytest.fixture(scope="module")
def stepper(tmp_path_factory):
    if not os.path.exists(NVCC):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("host_steps")
    obj, exe = str(d / "backward_steps.o"), str(d / "backward_steps")
    subprocess.run([NVCC, "-std=c++17", "-O1", "-g", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-Xcompiler", "-fsanitize=address,-fno-omit-frame-pointer",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-c", SRC, "-o", obj], check=True)
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(NVCC))), "lib64")
    subprocess.run(["g++", "-fsanitize=address", obj, "-o", exe, "-L", cuda_lib, "-lcudart_static",
                    "-ldl", "-lpthread", "-lrt"], check=True)
    return exe, d


def _run(stepper, q, k, v, dout, g, s0, ds, bf16):
    exe, d = stepper
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    inp, out = str(d / "in.bin"), str(d / "out.bin")
    with open(inp, "wb") as f:
        f.write(struct.pack("8i", int(bf16), B, H, N, dk, dv, int(s0 is not None), int(ds is not None)))
        for a in (q, k, v, dout, g) + tuple(x for x in (s0, ds) if x is not None):
            f.write(np.ascontiguousarray(a.float().numpy(), dtype=np.float32).tobytes())
    # bounds checks only: leak detection needs ptrace, which sandboxes may refuse
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:abort_on_error=0")
    p = subprocess.run([exe, inp, out], capture_output=True, text=True, env=env)
    assert p.returncode == 0, p.stderr[-4000:]
    raw = np.fromfile(out, dtype=np.float32)
    nq, nv = B * H * N * dk, B * H * N * dv
    return (raw[:nq].reshape(B, H, N, dk), raw[nq:2 * nq].reshape(B, H, N, dk),
            raw[2 * nq:2 * nq + nv].reshape(B, H, N, dv), raw[2 * nq + nv:].reshape(B, H, dk, dv))


@pytest.mark.parametrize("B,H,N,dk,dv,bf16,states", [
    (1, 2, 300, 128, 128, True, False),   # ragged last chunk
    (2, 3, 77, 64, 32, True, True),
    (1, 2, 130, 40, 24, True, True),      # edge slabs of 8 columns
    (1, 1, 70, 256, 512, True, True),     # widest rows
    (1, 2, 1, 128, 128, True, True),      # one token
    (1, 3, 65, 32, 48, False, True),      # fp32 twin
    (1, 1, 70, 8, 12, False, True),       # narrower than one float4 group per lane
])
def test_backward_phases_on_cpu_match_oracle(orc, stepper, B, H, N, dk, dv, bf16, states):
    dt = torch.bfloat16 if bf16 else torch.float32
    q, k, v = inputs.qkv(B, H, N, dk, dv, 21, dt)
    dout = inputs.normal((B, H, N, dv), 22, dt)
    s0 = inputs.normal((B, H, dk, dv), 23) if states else None
    ds = inputs.normal((B, H, dk, dv), 24) if states else None
    g = binding.gamma_schedule(H) if H > 1 else torch.tensor([0.9])
    got = _run(stepper, q, k, v, dout, g, s0, ds, bf16)
    ref = orc.backward(q, k, v, g.double(), dout, ds, s0)
    tol = TOL_BF16 if bf16 else TOL_F32
    for name, a, b in zip(("dq", "dk", "dv", "dstate_in"), got, ref):
        assert_close(a, b, tol, f"host steps {name}")


def test_backward_phases_any_decay(orc, stepper):
    gam = torch.tensor([0.0, 0.5, 1.0], dtype=torch.float32)
    q, k, v = inputs.qkv(1, 3, 90, 32, 32, 25, torch.bfloat16)
    dout = inputs.normal((1, 3, 90, 32), 26, torch.bfloat16)
    ds = inputs.normal((1, 3, 32, 32), 27)
    got = _run(stepper, q, k, v, dout, gam, None, ds, True)
    ref = orc.backward(q, k, v, gam.double(), dout, ds, None)
    for name, a, b in zip(("dq", "dk", "dv", "dstate_in"), got, ref):
        assert_close(a, b, TOL_BF16, f"host steps, any decay, {name}")
