"""GPU parity of fp32 inputs in split precision (MMACT_F32) against the oracle,
at the stated tolerance with no operand-rounding allowance.

The inputs are full-precision fp32 values (not representable in 16 bits or
in tf32).  Covered: the GEMM (any K and N, every activation and output dtype,
no bias, residual, the two-kernel split and its workspace), the NCHW conv
(strides, pads, dilations, ragged tiles, residual, split) and a cancellation
case whose exact result is the small difference of large products -- one
16-bit or tf32 rounding of the operands moves it by more than the bound, so
passing it shows that both halves of every operand reach the tensor cores.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_epilogue_gb300 import build, mmact
from parity import TORCH, check, fp32_to_device, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    mmact.load()


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def dev32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


GEMM_CASES = [
    # (M, N, K, out)
    (128, 128, 64, "f32"),
    (300, 200, 100, "f32"),          # K and N not multiples of 8
    (257, 520, 1000, "bf16"),
    (1024, 640, 256, "f32"),         # the MatmulLeakyRelu sample's shape, fp32 inputs
    (64, 72, 4096, "f16"),           # long K
]


@pytest.mark.parametrize("case", GEMM_CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("act", ["none", "relu", "leaky_relu", "tanh", "sigmoid", "gelu"])
def test_fp32_gemm(orc, case, act):
    M, N, K, od = case
    rng = np.random.default_rng(M + N + K)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    C = torch.full((M, N), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_gemm(dev32(A), dev32(B), fp32_to_device(bias), C, act, 0.1)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(C), orc.gemm(A, B, "f32", bias, act, 0.1), od, f"fp32 gemm {case} {act}")


def test_fp32_gemm_without_bias_and_with_residual(orc):
    M, N, K = 200, 136, 300
    rng = np.random.default_rng(5)
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    B = rng.normal(0, 1, (K, N)).astype(np.float32)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_gemm(dev32(A), dev32(B), None, C, "tanh")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(C), orc.gemm(A, B, "f32", None, "tanh"), "f32", "fp32 gemm, no bias")
    R = rng.uniform(-2, 2, (M, N)).astype(np.float32)
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    mmact.mmact_gemm_residual(dev32(A), dev32(B), fp32_to_device(bias), dev32(R), C, "gelu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(C), orc.gemm(A, B, "f32", bias, "gelu", residual=R, res_dtype="f32"), "f32",
          "fp32 gemm residual")


def test_fp32_gemm_split_and_workspace(orc):
    M, N, K = 384, 264, 520
    rng = np.random.default_rng(6)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.full((M * N,), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_gemm_split(dev32(A), dev32(B), fp32_to_device(bias), C, ws, "sigmoid")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(C), orc.gemm(A, B, "f32", bias, "sigmoid"), "bf16", "fp32 split")
    check(host(ws).reshape(M, N), orc.gemm(A, B, "f32", bias, "none"), "f32", "fp32 split workspace")


def test_fp32_split_precision_resolves_cancellation(orc):
    # C[m][n] = v_m * 1 + (-(v_m - d_m)) * 1 = d_m: the products are ~4, the result ~0.01.
    # Rounding the operands to bf16 (8 bits) or tf32 (11 bits) moves it by up to
    # 2 * 4 * 2^-9 or 2 * 4 * 2^-12 -- several times the bound 2e-3 + 2e-3 |d| -- while
    # split precision (about 16 bits per operand) stays far inside it.
    M, N = 256, 64
    rng = np.random.default_rng(8)
    v = rng.uniform(3.0, 4.0, M).astype(np.float32)
    d = rng.uniform(-0.01, 0.01, M).astype(np.float32)
    A = np.stack([v, -(v - d).astype(np.float32)], axis=1).astype(np.float32)
    B = np.ones((2, N), dtype=np.float32)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_gemm(dev32(A), dev32(B), None, C, "none")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    ref = orc.gemm(A, B, "f32", None, "none")
    # a one-pass 16-bit product would miss by more than the bound on most rows
    hi_only = (A.astype(np.float64) @ B.astype(np.float64))
    assert np.max(np.abs(ref - hi_only)) < 1e-12          # the oracle is exact here
    worst = check(host(C), ref, "f32", "fp32 cancellation")
    assert worst < 0.05


CONV_CASES = [
    # (N, C, H, W, Co, kh, kw, stride, pads, dilation, out)
    (1, 8, 8, 8, 16, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f32"),
    (2, 16, 12, 20, 32, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "bf16"),
    (2, 24, 17, 13, 40, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "f32"),
    (3, 3, 11, 9, 5, 3, 2, (2, 1), (1, 0, 2, 1), (1, 2), "f16"),
    (1, 64, 16, 16, 130, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f32"),   # ragged channel tile
    (2, 72, 9, 15, 8, 5, 5, (1, 2), (2, 2, 1, 3), (1, 1), "bf16"),
    (1, 16, 30, 30, 64, 7, 7, (2, 2), (3, 3, 3, 3), (1, 1), "f32"),
    (2, 16, 64, 64, 64, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), "f16"),
]


def conv_inputs(case, seed):
    Nb, C, H, W, Co, kh, kw, st, pd, dl, od = case
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (Nb, C, H, W)).astype(np.float32)
    w = rng.normal(0, (1.0 / (C * kh * kw)) ** 0.5, (Co, C, kh, kw)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    return rng, x, w, bias


@pytest.mark.parametrize("case", CONV_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}{c[6]}")
@pytest.mark.parametrize("act", ["tanh", "relu", "gelu"])
def test_fp32_conv_nchw(orc, case, act):
    Nb, C, H, W, Co, kh, kw, st, pd, dl, od = case
    assert mmact.mmact_conv2d_producer(Nb, C, H, W, Co, kh, kw, st, pd, dl, torch.float32, TORCH[od]) == "gather"
    _, x, w, bias = conv_inputs(case, 40 + C + Co)
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl)
    y = torch.full((Nb, Co, Ho, Wo), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_conv2d(dev32(x), dev32(w), fp32_to_device(bias), y, st, pd, dl, act)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(y), orc.conv2d(x, w, "f32", bias, st, pd, dl, act), od, f"fp32 conv {case} {act}")


def test_fp32_conv_nchw_residual_and_split(orc):
    case = CONV_CASES[1]
    Nb, C, H, W, Co, kh, kw, st, pd, dl, od = case
    rng, x, w, bias = conv_inputs(case, 77)
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl)
    R = rng.uniform(-1, 1, (Nb, Co, Ho, Wo)).astype(np.float32)
    y = dev32(R)                               # in place
    mmact.mmact_conv2d_residual(dev32(x), dev32(w), fp32_to_device(bias), y, y, st, pd, dl, "relu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(y), orc.conv2d(x, w, "f32", bias, st, pd, dl, "relu", residual=R, res_dtype="f32"), "f32",
          "fp32 conv residual in place")
    y2 = torch.full((Nb, Co, Ho, Wo), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.full((y2.numel(),), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_conv2d_split(dev32(x), dev32(w), fp32_to_device(bias), y2, ws, st, pd, dl, "tanh")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(y2), orc.conv2d(x, w, "f32", bias, st, pd, dl, "tanh"), "bf16", "fp32 conv split")


def test_tf32_is_refused_where_no_tf32_path_exists():
    A = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    L = mmact.load()
    st = L.mmact_gemm(A.data_ptr(), A.data_ptr(), None, A.data_ptr(), 8, 8, 8, mmact.MMACT_TF32,
                      mmact.DTYPE[torch.float32], mmact.ACT["relu"], 0.0, None)
    assert st == mmact.MMACT_ERR_UNSUPPORTED
