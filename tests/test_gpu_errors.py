"""GPU error paths, none of which faults, traps or hangs the GPU.

The bounded-wait self-test kernel waits on an mbarrier nothing arrives at,
gives up after a short limit and records MMACT_ERR_TIMEOUT; the host reads it
through mmact_get_last_error, and the context stays usable afterwards.
Argument errors are rejected on the host before anything is enqueued.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_epilogue_gb300 import build, mmact, synth
from parity import check, fp32_to_device, host, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    mmact.load()


def test_timeout_is_reported_and_context_survives():
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    mmact.mmact_selftest_wait_timeout(2_000_000)     # 2 ms
    assert mmact.mmact_get_last_error() == mmact.MMACT_ERR_TIMEOUT
    # read-and-clear
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    # the context still runs real work correctly
    rng = np.random.default_rng(1)
    A = synth.to_codes(rng.uniform(-1, 1, (128, 64)), "bf16")
    B = synth.to_codes(rng.uniform(-1, 1, (64, 64)), "bf16")
    C = torch.empty((128, 64), dtype=torch.float32, device="cuda")
    mmact.mmact_gemm(to_device(A, "bf16"), to_device(B, "bf16"), None, C, "relu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(C), oracle.get().gemm(A, B, "bf16", None, "relu"), "f32", "after timeout")


def test_binding_rejects_bad_tensors():
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):
        mmact.mmact_gemm(A.cpu(), B, None, C)
    with pytest.raises(ValueError):
        mmact.mmact_gemm(A.t(), B, None, C)                       # not contiguous
    with pytest.raises(ValueError):
        mmact.mmact_gemm(A, B[:32], None, C)                      # K mismatch
    with pytest.raises(mmact.MmactError) as ei:
        mmact.mmact_gemm(A[:, :60].contiguous(), B[:60], None, C)  # K % 8 != 0
    assert ei.value.status == mmact.MMACT_ERR_UNSUPPORTED
    with pytest.raises(TypeError):
        mmact.mmact_gemm(A.int(), B.int(), None, C)                # integer operands
    with pytest.raises(ValueError):
        mmact.mmact_gemm(A.float(), B, None, C)                    # fp32 A with bf16 B
    torch.cuda.synchronize()
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK


def test_calls_on_a_side_stream(tmp_path):
    s = torch.cuda.Stream()
    rng = np.random.default_rng(2)
    A = synth.to_codes(rng.uniform(-1, 1, (256, 128)), "f16")
    B = synth.to_codes(rng.uniform(-1, 1, (128, 192)), "f16")
    bias = rng.uniform(-1, 1, 192).astype(np.float32)
    with torch.cuda.stream(s):
        dA, dB, db = to_device(A, "f16"), to_device(B, "f16"), fp32_to_device(bias)
        C = torch.empty((256, 192), dtype=torch.float16, device="cuda")
        mmact.mmact_gemm(dA, dB, db, C, "leaky_relu", 0.01, stream=s)
    assert mmact.mmact_get_last_error(s) == mmact.MMACT_OK
    check(host(C), oracle.get().gemm(A, B, "f16", bias, "leaky_relu", 0.01), "f16", "side stream")
