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
from parity import TORCH, check, fp32_to_device, host, sample_points, to_device

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
    pts = sample_points(y.size, y.size // 64, 64, 20000, wl.seed + 100)
    ref = orc.conv2d(inp["x"], inp["w"], wl.dtype, inp["bias"], wl.stride, wl.pads, wl.dilation,
                     wl.act, wl.alpha, points=pts)
    check(y[pts], ref, wl.out_dtype, f"nhwc {wl.name}")
