"""The no-allocation variant of the two-kernel GEMM path, through the C ABI.

mmact_gemm_split_noalloc exists for callers that cannot allocate device
memory when they call the library (they are handed only their input and
output buffers, or a framework allocator owns the device budget, or a
cudaMalloc / cudaFree could stall their latency-critical loop).  It runs the
same two kernels as mmact_gemm_split with the fp32 intermediate in a scratch
array built into the library.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from conv_activation_epilogue_gb300 import build, mmact, synth
from parity import check, fp32_to_device, host, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mmact.load()


def _call_noalloc(lib, A, B, bias, C, act, alpha):
    M, K = A.shape
    N = B.shape[1]
    stream = torch.cuda.current_stream().cuda_stream or None
    return lib.mmact_gemm_split_noalloc(A.data_ptr(), B.data_ptr(),
                                        None if bias is None else bias.data_ptr(), C.data_ptr(),
                                        M, N, K, mmact.DTYPE[A.dtype], mmact.DTYPE[C.dtype],
                                        mmact.ACT[act], ctypes.c_float(alpha), stream)


def test_noalloc_matches_split_entry_point_on_two_calls(lib):
    # two calls in a row, different shapes and data: the second must not see
    # anything the first left in the shared scratch array
    for call, (M, N, K, ab, cd, act, alpha) in enumerate([
            (512, 1024, 256, "bf16", "bf16", "leaky_relu", 0.2),
            (300, 264, 136, "f16", "f32", "tanh", 0.0)]):
        rng = np.random.default_rng(500 + call)
        A = to_device(synth.to_codes(rng.uniform(-1, 1, (M, K)), ab), ab)
        B = to_device(synth.to_codes(rng.uniform(-1, 1, (K, N)), ab), ab)
        bias = fp32_to_device(rng.uniform(-1, 1, N).astype(np.float32))
        out_dtype = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[cd]
        ref = torch.empty((M, N), dtype=out_dtype, device="cuda")
        ws = torch.empty((M * N,), dtype=torch.float32, device="cuda")
        mmact.mmact_gemm_split(A, B, bias, ref, ws, act, alpha)
        got = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        assert _call_noalloc(lib, A, B, bias, got, act, alpha) == mmact.MMACT_OK
        assert mmact.mmact_get_last_error() == mmact.MMACT_OK
        check(host(got), host(ref), cd, f"no-alloc call {call + 1}")


def test_noalloc_at_its_size_limit_matches_split_entry_point(lib):
    # M*N == MMACT_NOALLOC_MAX_ELEMENTS uses every element of the scratch array
    M = N = 2048
    assert M * N == mmact.NOALLOC_MAX_ELEMENTS
    rng = np.random.default_rng(610)
    A = to_device(synth.to_codes(rng.uniform(-1, 1, (M, 128)), "bf16"), "bf16")
    B = to_device(synth.to_codes(rng.uniform(-1, 1, (128, N)), "bf16"), "bf16")
    bias = fp32_to_device(rng.uniform(-1, 1, N).astype(np.float32))
    ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty((M * N,), dtype=torch.float32, device="cuda")
    mmact.mmact_gemm_split(A, B, bias, ref, ws, "sigmoid", 0.0)
    got = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, A, B, bias, got, "sigmoid", 0.0) == mmact.MMACT_OK
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(got), host(ref), "f32", "no-alloc at the limit")
    # one past the limit is refused before anything runs
    C = torch.zeros((2048, 2056), dtype=torch.bfloat16, device="cuda")
    B2 = torch.zeros((128, 2056), dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(lib, A, B2, None, C, "relu", 0.0) == mmact.MMACT_ERR_UNSUPPORTED


def test_noalloc_skinny_split_k_shape_matches_oracle(lib):
    # 128 x 4096 x 4096: few output tiles and a long K loop, so the first kernel
    # is the split-K cluster kernel when the device fits its clusters
    import oracle
    M, N, K = 128, 4096, 4096
    rng = np.random.default_rng(611)
    a = synth.to_codes(rng.uniform(-1, 1, (M, K)), "bf16")
    b = synth.to_codes(rng.uniform(-1, 1, (K, N)), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    split_k = mmact.mmact_gemm_split_k_choice(M, N, K)
    got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(lib, to_device(a, "bf16"), to_device(b, "bf16"), fp32_to_device(bias), got,
                         "leaky_relu", 0.2) == mmact.MMACT_OK
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    ref = oracle.get().gemm(a, b, "bf16", bias, "leaky_relu", 0.2)
    check(host(got), ref, "bf16", f"no-alloc skinny (split-K factor {split_k})")
    assert split_k == 4      # 16 tiles of 128 x 256, 64 K blocks: clusters of 4 on a GB300


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # rejected on the host before anything is enqueued
    A = torch.zeros((2048, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 4096), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((2048, 4096), dtype=torch.bfloat16, device="cuda")   # M*N = 2 x the maximum
    assert 2048 * 4096 > mmact.NOALLOC_MAX_ELEMENTS
    assert _call_noalloc(lib, A, B, None, C, "relu", 0.0) == mmact.MMACT_ERR_UNSUPPORTED
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
