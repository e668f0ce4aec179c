"""GPU parity: the CTA-pair GEMM kernel (256 x 256 tiles, one M = 256
tcgen05.mma per pair of SMs) against the oracle.

The mode switch forces the kernel onto small shapes with ragged M / N / K
tails (a pair whose second CTA lies wholly past M, a last tile partly past
N), every output dtype and activation, with and without a residual, and onto
the full-size square workloads on sampled outputs; the automatic choice is
checked on the workload shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_epilogue_gb300 import build, mmact, synth
from parity import TORCH, check, fp32_to_device, host, sample_points, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    mmact.load()
    mmact.mmact_set_wait_timeout_ns(200_000_000)
    mmact.mmact_set_gemm_pair(2)
    mmact.mmact_set_gemm_split_k(1)
    yield
    mmact.mmact_set_gemm_pair(0)
    mmact.mmact_set_gemm_split_k(0)
    mmact.mmact_set_wait_timeout_ns(0)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def rand_codes(rng, shape, dtype, lo=-1.0, hi=1.0):
    return synth.to_codes(rng.uniform(lo, hi, size=shape), dtype)


def run(A, B, bias, ab, cd, act, alpha, R=None):
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), float("nan"), dtype=TORCH[cd], device="cuda")
    if R is None:
        mmact.mmact_gemm(to_device(A, ab), to_device(B, ab), fp32_to_device(bias), C, act, alpha)
    else:
        dR = fp32_to_device(R) if cd == "f32" else to_device(R, cd)
        mmact.mmact_gemm_residual(to_device(A, ab), to_device(B, ab), fp32_to_device(bias), dR, C, act, alpha)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    return C


SHAPES = [(256, 256, 64), (128, 256, 128), (300, 264, 136), (512, 512, 520), (1, 8, 8), (700, 1000, 256)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pair_kernel_matches_oracle(orc, shape):
    M, N, K = shape
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    for ab, cd, act, alpha in [("bf16", "bf16", "leaky_relu", 0.2), ("f16", "f32", "relu", 0.0),
                               ("bf16", "f16", "tanh", 0.0), ("f16", "bf16", "gelu", 0.0)]:
        A = rand_codes(rng, (M, K), ab)
        B = rand_codes(rng, (K, N), ab)
        bias = rng.uniform(-1, 1, N).astype(np.float32)
        C = run(A, B, bias, ab, cd, act, alpha)
        check(host(C), orc.gemm(A, B, ab, bias, act, alpha), cd, f"pair {shape} {ab}->{cd} {act}")


def test_pair_kernel_residual(orc):
    rng = np.random.default_rng(11)
    M, N, K = 384, 520, 256
    A = rand_codes(rng, (M, K), "bf16")
    B = rand_codes(rng, (K, N), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    R = rand_codes(rng, (M, N), "bf16")
    C = run(A, B, bias, "bf16", "bf16", "sigmoid", 0.0, R=R)
    check(host(C), orc.gemm(A, B, "bf16", bias, "sigmoid", residual=R, res_dtype="bf16"), "bf16", "pair residual")


@pytest.mark.parametrize("cd", ["bf16", "f32"])
def test_pair_kernel_residual_in_place(orc, cd):
    # R is C itself: each element is read before its own unit's store writes it
    rng = np.random.default_rng(21 + len(cd))
    M, N, K = 512, 512, 512
    A = rand_codes(rng, (M, K), "bf16")
    B = rand_codes(rng, (K, N), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    if cd == "f32":
        R = rng.uniform(-1, 1, (M, N)).astype(np.float32)
        C = fp32_to_device(R).clone()
    else:
        R = rand_codes(rng, (M, N), cd)
        C = to_device(R, cd).clone()
    mmact.mmact_gemm_residual(to_device(A, "bf16"), to_device(B, "bf16"), fp32_to_device(bias), C, C,
                              "gelu", 0.0)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(C), orc.gemm(A, B, "bf16", bias, "gelu", residual=R, res_dtype=cd), cd, f"pair in place {cd}")


@pytest.mark.parametrize("name", ["gemm_relu_4096x4096x4096_bf16", "gemm_leakyrelu_8192x8192x8192_bf16"])
def test_pair_kernel_workload(orc, name):
    wl = synth.WORKLOADS[name]
    inp = wl.inputs()
    C = run(inp["A"], inp["B"], inp["bias"], wl.ab_dtype, wl.c_dtype, wl.act, wl.alpha)
    got = host(C).ravel()
    pts = sample_points(wl.M * wl.N, wl.M, wl.N, 4000, seed=wl.seed + 2)
    ref = orc.gemm(inp["A"], inp["B"], wl.ab_dtype, inp["bias"], wl.act, wl.alpha, points=pts)
    check(got[pts], ref, wl.c_dtype, wl.name)


def test_automatic_choice():
    mmact.mmact_set_gemm_pair(0)
    mmact.mmact_set_gemm_split_k(0)
    try:
        assert mmact.mmact_gemm_kernel_choice(8192, 8192, 8192) == "pair"
        assert mmact.mmact_gemm_kernel_choice(4096, 4096, 4096) == "pair"
        assert mmact.mmact_gemm_kernel_choice(16384, 4096, 1024) == "pair"
        assert mmact.mmact_gemm_kernel_choice(1024, 640, 256) == "persistent"   # narrow tiles fill more SMs
        assert mmact.mmact_gemm_kernel_choice(128, 8192, 8192) == "split_k"
        assert mmact.mmact_gemm_kernel_choice(0, 64, 64) == "none"
        assert mmact.mmact_gemm_kernel_choice(8192, 8192, 8192, residual=True) == "pair"
        assert mmact.mmact_gemm_kernel_choice(16384, 4096, 1024, residual=True) == "pair"   # TMA-staged residual
        mmact.mmact_set_gemm_tile_n(256)
        assert mmact.mmact_gemm_kernel_choice(8192, 8192, 8192) == "persistent"  # a fixed tile width
        mmact.mmact_set_gemm_tile_n(0)
        mmact.mmact_set_gemm_pair(1)
        assert mmact.mmact_gemm_kernel_choice(8192, 8192, 8192) == "persistent"
    finally:
        mmact.mmact_set_gemm_tile_n(0)
        mmact.mmact_set_gemm_pair(2)
        mmact.mmact_set_gemm_split_k(1)


@pytest.mark.parametrize("shape", [(1024, 1024, 512), (700, 1000, 256)], ids=lambda s: "x".join(map(str, s)))
def test_l2_policy_changes_no_value(orc, shape):
    """The L2 eviction hints rank lines for eviction only: the output with and
    without them is bit-identical and matches the oracle."""
    M, N, K = shape
    rng = np.random.default_rng(M + N)
    A = rand_codes(rng, (M, K), "bf16")
    B = rand_codes(rng, (K, N), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    try:
        mmact.mmact_set_gemm_l2_policy(0)
        plain = host(run(A, B, bias, "bf16", "bf16", "leaky_relu", 0.2))
        mmact.mmact_set_gemm_l2_policy(1)
        hinted = host(run(A, B, bias, "bf16", "bf16", "leaky_relu", 0.2))
    finally:
        mmact.mmact_set_gemm_l2_policy(1)
    assert np.array_equal(plain, hinted)
    check(hinted, orc.gemm(A, B, "bf16", bias, "leaky_relu", 0.2), "bf16", f"pair with L2 hints {shape}")
