"""GPU parity: the channels-last fused conv (mmact_conv2d_nhwc) against the oracle.

The oracle computes NCHW convolution; these tests draw NCHW inputs, hand the
kernel their NHWC / [Co,kh,kw,C] transposes and transpose its NHWC output
back before comparing -- pure data movement on the host, no arithmetic.
Geometries cover stride, dilation, asymmetric padding, channel counts that
leave a partial 64-channel block, several output-channel tiles and pixel
tiles spanning image boundaries, plus the three conv workloads' shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_epilogue_gb300 import build, mmact, synth
from parity import ACT_SLOPE, TF32_REL, TORCH, check, fp32_to_device, host, sample_points, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    mmact.load()


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def run_nhwc(x, w, bias, dt, od, stride, pads, dil, act, alpha=0.0):
    """x [N,C,H,W], w [Co,C,kh,kw] codes (NCHW); returns y as NCHW float64."""
    Nb, C, H, W = x.shape
    Co, _, kh, kw = w.shape
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, stride, pads, dil)
    dx = to_device(np.ascontiguousarray(x.transpose(0, 2, 3, 1)), dt)
    dw = to_device(np.ascontiguousarray(w.transpose(0, 2, 3, 1)), dt)
    y = torch.full((Nb, Ho, Wo, Co), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_conv2d_nhwc(dx, dw, fp32_to_device(bias), y, stride, pads, dil, act, alpha)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    return host(y).transpose(0, 3, 1, 2)


CASES = [
    # (N, C, H, W, Co, kh, kw, stride, pads, dilation, dtype, out)
    (1, 64, 8, 8, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),
    (2, 16, 13, 11, 24, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "bf16", "bf16"),   # partial channel block
    (3, 72, 9, 10, 40, 5, 3, (1, 2), (2, 0, 1, 3), (1, 2), "bf16", "f32"),     # C = 72: 2 blocks
    (2, 32, 17, 19, 200, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), "f16", "bf16"),   # Co = 200: 2 tiles
    (1, 8, 30, 30, 8, 7, 7, (2, 2), (3, 3, 3, 3), (1, 1), "bf16", "bf16"),
    (4, 128, 7, 7, 264, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),     # several N tiles
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}{c[6]}s{c[7][0]}{c[7][1]}")
@pytest.mark.parametrize("act", ["tanh", "leaky_relu", "gelu"])
def test_small_geometries(orc, case, act):
    Nb, C, H, W, Co, kh, kw, stride, pads, dil, dt, od = case
    rng = np.random.default_rng(Nb * 100 + C + Co)
    x = synth.to_codes(rng.normal(0, 1, (Nb, C, H, W)), dt)
    w = synth.to_codes(rng.normal(0, (1.0 / (C * kh * kw)) ** 0.5, (Co, C, kh, kw)), dt)
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    y = run_nhwc(x, w, bias, dt, od, stride, pads, dil, act, 0.1)
    check(y, orc.conv2d(x, w, dt, bias, stride, pads, dil, act, 0.1), od, f"nhwc {case} {act}")


def test_rejects_channel_counts_that_are_not_multiples_of_8():
    x = torch.zeros((1, 4, 4, 12), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 3, 3, 12), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, 2, 2, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mmact.MmactError) as ei:
        mmact.mmact_conv2d_nhwc(x, w, None, y)
    assert ei.value.status == mmact.MMACT_ERR_UNSUPPORTED


CONV_WORKLOADS = [w for w in synth.WORKLOADS.values() if w.kind == "conv"]


@pytest.mark.parametrize("wl", CONV_WORKLOADS, ids=lambda w: w.name)
def test_workload_shapes_channels_last(orc, wl):
    inp = wl.inputs()
    y = run_nhwc(inp["x"], inp["w"], inp["bias"], wl.dtype, wl.out_dtype, wl.stride, wl.pads,
                 wl.dilation, wl.act, wl.alpha).ravel()
    # every output element against the oracle
    ref = orc.conv2d(inp["x"], inp["w"], wl.dtype, inp["bias"], wl.stride, wl.pads, wl.dilation,
                     wl.act, wl.alpha).ravel()
    check(y, ref, wl.out_dtype, f"nhwc {wl.name}")


# ---------------------------------------------------------------- fp32 inputs --
def run_nhwc_f32(x, w, bias, od, stride, pads, dil, act, alpha=0.0, tf32=False):
    """fp32 x [N,C,H,W], w [Co,C,kh,kw] (NCHW), computed as tf32 or in split precision;
    returns y as NCHW float64."""
    Nb, C, H, W = x.shape
    Co, _, kh, kw = w.shape
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, stride, pads, dil)
    dx = torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 3, 1))).cuda()
    dw = torch.from_numpy(np.ascontiguousarray(w.transpose(0, 2, 3, 1))).cuda()
    y = torch.full((Nb, Ho, Wo, Co), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_conv2d_nhwc(dx, dw, fp32_to_device(bias), y, stride, pads, dil, act, alpha, tf32=tf32)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    return host(y).transpose(0, 3, 1, 2)


def tf32_allowance(orc, x, w, stride, pads, dil, points=None):
    """1.2 * 2^-9 * sum_k |x_k w_k| per output: the oracle's conv of |x| and |w|."""
    s = orc.conv2d(np.abs(x), np.abs(w), "f32", None, stride, pads, dil, "none", points=points)
    return ACT_SLOPE * TF32_REL * s


F32_CASES = [
    # (N, C, H, W, Co, kh, kw, stride, pads, dilation, out)
    (1, 32, 8, 8, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f32"),
    (2, 36, 13, 11, 24, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "bf16"),    # partial 32-channel block
    (3, 72, 9, 10, 40, 5, 3, (1, 2), (2, 0, 1, 3), (1, 2), "f32"),
    (2, 16, 17, 19, 136, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), "f16"),
    (1, 8, 30, 30, 8, 7, 7, (2, 2), (3, 3, 3, 3), (1, 1), "f32"),
]


def f32_inputs(case):
    Nb, C, H, W, Co, kh, kw, stride, pads, dil, od = case
    rng = np.random.default_rng(Nb * 100 + C + Co + 7)
    # full-precision fp32 values (not representable in 16 bits or in tf32)
    x = rng.normal(0, 1, (Nb, C, H, W)).astype(np.float32)
    w = rng.normal(0, (1.0 / (C * kh * kw)) ** 0.5, (Co, C, kh, kw)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    return x, w, bias


CASE_ID = lambda c: f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}{c[6]}s{c[7][0]}{c[7][1]}"  # noqa: E731


@pytest.mark.parametrize("case", F32_CASES, ids=CASE_ID)
@pytest.mark.parametrize("act", ["tanh", "relu", "gelu"])
def test_tf32_inputs_small_geometries(orc, case, act):
    # one-pass tf32: the stated bound plus the tf32 operand-rounding allowance
    Nb, C, H, W, Co, kh, kw, stride, pads, dil, od = case
    x, w, bias = f32_inputs(case)
    y = run_nhwc_f32(x, w, bias, od, stride, pads, dil, act, tf32=True)
    ref = orc.conv2d(x, w, "f32", bias, stride, pads, dil, act)
    check(y, ref, od, f"nhwc tf32 {case} {act}", extra=tf32_allowance(orc, x, w, stride, pads, dil))


@pytest.mark.parametrize("case", F32_CASES, ids=CASE_ID)
@pytest.mark.parametrize("act", ["tanh", "relu", "gelu"])
def test_fp32_split_precision_small_geometries(orc, case, act):
    # split precision: the stated bound 2e-3 + 2e-3 |y| (+ 1 output ulp), no allowance
    Nb, C, H, W, Co, kh, kw, stride, pads, dil, od = case
    x, w, bias = f32_inputs(case)
    y = run_nhwc_f32(x, w, bias, od, stride, pads, dil, act)
    ref = orc.conv2d(x, w, "f32", bias, stride, pads, dil, act)
    check(y, ref, od, f"nhwc fp32 split {case} {act}")


@pytest.mark.parametrize("tf32", [True, False], ids=["tf32", "split"])
def test_fp32_inputs_workload_shape(orc, tf32):
    # the 3x3 stride-1 workload's values, widened to fp32 (exact), sampled
    wl = synth.WORKLOADS["conv3x3_s1p1d1_tanh_8x64x56x56_f16"]
    inp = wl.inputs()
    x = orc.decode(inp["x"], wl.dtype).astype(np.float32)
    w = orc.decode(inp["w"], wl.dtype).astype(np.float32)
    y = run_nhwc_f32(x, w, inp["bias"], "f32", wl.stride, wl.pads, wl.dilation, wl.act, tf32=tf32).ravel()
    pts = sample_points(y.size, y.size // 56, 56, 8000, wl.seed + 200)
    ref = orc.conv2d(x, w, "f32", inp["bias"], wl.stride, wl.pads, wl.dilation, wl.act, points=pts)
    extra = tf32_allowance(orc, x, w, wl.stride, wl.pads, wl.dilation, points=pts) if tf32 else None
    check(y[pts], ref, "f32", f"nhwc fp32 workload ({'tf32' if tf32 else 'split'})", extra=extra)


@pytest.mark.parametrize("tf32", [True, False], ids=["tf32", "split"])
def test_fp32_rejects_channel_counts_that_are_not_multiples_of_4(tf32):
    x = torch.zeros((1, 4, 4, 6), dtype=torch.float32, device="cuda")
    w = torch.zeros((8, 3, 3, 6), dtype=torch.float32, device="cuda")
    y = torch.zeros((1, 2, 2, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(mmact.MmactError) as ei:
        mmact.mmact_conv2d_nhwc(x, w, None, y, tf32=tf32)
    assert ei.value.status == mmact.MMACT_ERR_UNSUPPORTED
