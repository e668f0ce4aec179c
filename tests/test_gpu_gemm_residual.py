"""GPU parity: the fused GEMM with a residual tensor, C = act(A x B + bias + R),
against the oracle.  R has C's shape and dtype and is added to the fp32
accumulator before the activation; R may be C itself (in-place update).
Small shapes are compared element by element (several tiles, ragged M/N/K
tails, every tile width, all three output dtypes); the 4096^3 workload shape
on seeded samples."""
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
    yield
    mmact.mmact_set_gemm_tile_n(0)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def residual_codes(rng, shape, cd, lo=-2.0, hi=2.0):
    v = rng.uniform(lo, hi, size=shape)
    return v.astype(np.float32) if cd == "f32" else synth.to_codes(v, cd)


def residual_device(R, cd):
    return fp32_to_device(R) if cd == "f32" else to_device(R, cd)


def run(A, B, bias, R, ab, cd, act, alpha, inplace=False):
    M, K = A.shape
    N = B.shape[1]
    dA, dB = to_device(A, ab), to_device(B, ab)
    dR = residual_device(R, cd)
    if inplace:
        C = dR.clone()
        mmact.mmact_gemm_residual(dA, dB, fp32_to_device(bias), C, C, act, alpha)
    else:
        C = torch.full((M, N), float("nan"), dtype=TORCH[cd], device="cuda")
        mmact.mmact_gemm_residual(dA, dB, fp32_to_device(bias), dR, C, act, alpha)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    return host(C), host(dR)


SHAPES = [(128, 64, 64), (7, 24, 40), (129, 72, 200), (300, 264, 136), (64, 1000, 64)]


@pytest.mark.parametrize("tile_n", [64, 224, 256])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_residual_small_shapes(orc, tile_n, shape):
    M, N, K = shape
    rng = np.random.default_rng(M + 3 * N + 7 * K + tile_n)
    mmact.mmact_set_gemm_tile_n(tile_n)
    for ab, cd, act, alpha in [("bf16", "bf16", "relu", 0.0), ("f16", "f32", "leaky_relu", 0.1),
                               ("bf16", "f16", "tanh", 0.0), ("f16", "bf16", "none", 0.0)]:
        A = synth.to_codes(rng.uniform(-1, 1, (M, K)), ab)
        B = synth.to_codes(rng.uniform(-1, 1, (K, N)), ab)
        bias = rng.uniform(-1, 1, N).astype(np.float32)
        R = residual_codes(rng, (M, N), cd)
        got, _ = run(A, B, bias, R, ab, cd, act, alpha)
        ref = orc.gemm(A, B, ab, bias, act, alpha, residual=R, res_dtype=cd)
        check(got, ref, cd, f"{shape} tile {tile_n} {ab}->{cd} {act}")
    mmact.mmact_set_gemm_tile_n(0)


@pytest.mark.parametrize("cd", ["bf16", "f32"])
def test_residual_in_place(orc, cd):
    # R == C: every element is read before the same element is written
    rng = np.random.default_rng(31)
    M, N, K = 300, 520, 192
    A = synth.to_codes(rng.uniform(-1, 1, (M, K)), "bf16")
    B = synth.to_codes(rng.uniform(-1, 1, (K, N)), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    R = residual_codes(rng, (M, N), cd)
    got, _ = run(A, B, bias, R, "bf16", cd, "gelu", 0.0, inplace=True)
    check(got, orc.gemm(A, B, "bf16", bias, "gelu", residual=R, res_dtype=cd), cd, "in place")


def test_residual_changes_only_the_preactivation(orc):
    # R = 0 gives mmact_gemm's result exactly (same kernel, same order)
    rng = np.random.default_rng(32)
    M, N, K = 256, 512, 256
    A = to_device(synth.to_codes(rng.uniform(-1, 1, (M, K)), "bf16"), "bf16")
    B = to_device(synth.to_codes(rng.uniform(-1, 1, (K, N)), "bf16"), "bf16")
    bias = fp32_to_device(rng.uniform(-1, 1, N).astype(np.float32))
    C0 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C1 = torch.empty_like(C0)
    mmact.mmact_gemm(A, B, bias, C0, "tanh")
    mmact.mmact_gemm_residual(A, B, bias, torch.zeros_like(C0), C1, "tanh")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    assert torch.equal(C0, C1)


def test_residual_empty_contraction(orc):
    rng = np.random.default_rng(33)
    M, N = 5, 24
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    R = residual_codes(rng, (M, N), "f16")
    dA = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    dB = torch.empty((0, N), dtype=torch.float16, device="cuda")
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    mmact.mmact_gemm_residual(dA, dB, fp32_to_device(bias), to_device(R, "f16"), C, "sigmoid")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    A0 = np.zeros((M, 0), dtype=np.uint16)
    B0 = np.zeros((0, N), dtype=np.uint16)
    check(host(C), orc.gemm(A0, B0, "f16", bias, "sigmoid", residual=R, res_dtype="f16"), "f16", "K=0")


def test_residual_workload_shape(orc):
    # the 4096^3 ReLU workload with a residual, compared on seeded samples
    wl = synth.WORKLOADS["gemm_relu_4096x4096x4096_bf16"]
    inp = wl.inputs()
    rng = np.random.default_rng(34)
    R = residual_codes(rng, (wl.M, wl.N), wl.c_dtype)
    got, _ = run(inp["A"], inp["B"], inp["bias"], R, wl.ab_dtype, wl.c_dtype, wl.act, wl.alpha)
    pts = sample_points(wl.M * wl.N, wl.M, wl.N, 4000, seed=wl.seed)
    ref = orc.gemm(inp["A"], inp["B"], wl.ab_dtype, inp["bias"], wl.act, wl.alpha, points=pts,
                   residual=R, res_dtype=wl.c_dtype)
    check(got.ravel()[pts], ref, wl.c_dtype, "4096^3 + residual")


def test_residual_binding_rejects_mismatch():
    A = torch.zeros((8, 8), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((8, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        mmact.mmact_gemm_residual(A, A, None, torch.zeros((8, 16), dtype=torch.bfloat16, device="cuda"), C)
    with pytest.raises(ValueError):
        mmact.mmact_gemm_residual(A, A, None, torch.zeros((8, 8), dtype=torch.float32, device="cuda"), C)
