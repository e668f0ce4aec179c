"""GPU parity of the NCHW conv kernel whose im2col operand is assembled in
tensor memory (MMACT_CONV_TMEM), against the oracle.

Each case asserts that the planner takes that kernel, then compares every
output element.  The geometries cover what its index arithmetic has to get
right: tiles of 128 consecutive pixels that span several output rows (narrow
outputs) or part of one (Wo > 128), the last partial tile of each image, row
lattices (stride dividing dilation) and strided rows without one, stride 3,
asymmetric pads, 1x1 to 7x7 filters (K-offset table periods 1 to 49), K tails,
output-channel blocks of 64, 128 and 256 with ragged ends, several channel
blocks, an odd pixel count (the per-element store path), fp32 outputs, every
activation, residuals (also in place), and more tiles than SMs (the
accumulator ring wrapping).
"""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_epilogue_gb300 import build, mmact, synth
from parity import TORCH, check, fp32_to_device, host, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    mmact.load()
    mmact.mmact_set_conv_tmem(0)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


CASES = [
    # (N, C, H, W, Co, kh, kw, stride, pads, dilation, dtype, out)
    (2, 64, 56, 56, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),       # the 3x3 s1 geometry
    (2, 128, 64, 64, 256, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "bf16", "bf16"),    # 3x3 s2 d2
    (2, 128, 64, 64, 256, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), "bf16", "bf16"),    # 1x1 s2
    (1, 16, 16, 16, 24, 3, 3, (2, 2), (1, 1, 1, 1), (1, 1), "f16", "f16"),        # strided rows, no lattice
    (2, 8, 40, 200, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "bf16", "f32"),       # Wo = 200
    (1, 16, 40, 8, 16, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "bf16"),        # Wo = 8: 16 rows a tile
    (1, 8, 20, 24, 16, 7, 7, (1, 1), (3, 3, 3, 3), (1, 1), "f16", "f16"),         # 49 taps
    (1, 24, 19, 48, 72, 3, 5, (1, 2), (0, 3, 2, 1), (2, 1), "bf16", "f32"),       # asymmetric
    (2, 32, 24, 40, 48, 2, 2, (1, 1), (0, 1, 1, 0), (1, 1), "f16", "f16"),        # 2x2
    (1, 40, 13, 16, 40, 5, 5, (2, 1), (2, 2, 2, 2), (1, 1), "bf16", "bf16"),      # K = 1000
    (1, 16, 7, 16, 16, 3, 3, (2, 1), (1, 1, 2, 2), (1, 2), "bf16", "f16"),        # dh not a multiple of sh
    (1, 8, 30, 32, 8, 3, 3, (3, 3), (1, 1, 1, 1), (1, 1), "f16", "f16"),          # stride 3
    (1, 16, 15, 16, 32, 3, 3, (1, 1), (1, 1, 0, 1), (1, 1), "f16", "f16"),        # P = 225 (odd)
    (1, 32, 16, 16, 300, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "bf16", "bf16"),     # Co = 300: 2 blocks of 256
    (3, 16, 20, 24, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),        # P = 480 per image
    (16, 8, 64, 64, 256, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "bf16", "bf16"),     # 512 tiles, BN = 256
    (16, 8, 64, 64, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),       # 512 tiles, BN = 128
    (8, 16, 56, 56, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f32"),        # 200 tiles, BN = 64
]


def case_id(c):
    return f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}{c[6]}s{c[7][0]}{c[7][1]}d{c[9][0]}{c[9][1]}-{c[11]}"


def inputs(case, seed):
    Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, od = case
    rng = np.random.default_rng(seed)
    x = synth.to_codes(rng.normal(0, 1, (Nb, C, H, W)), dt)
    w = synth.to_codes(rng.normal(0, (1.0 / (C * kh * kw)) ** 0.5, (Co, C, kh, kw)), dt)
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    return rng, x, w, bias


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_tmem_kernel_geometries(orc, case):
    Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, od = case
    assert mmact.mmact_conv2d_producer(Nb, C, H, W, Co, kh, kw, st, pd, dl, TORCH[dt], TORCH[od]) == "tmem"
    _, x, w, bias = inputs(case, 3000 + Co + C)
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl)
    y = torch.full((Nb, Co, Ho, Wo), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_conv2d(to_device(x, dt), to_device(w, dt), fp32_to_device(bias), y, st, pd, dl, "tanh")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(y), orc.conv2d(x, w, dt, bias, st, pd, dl, "tanh"), od, case_id(case))


@pytest.mark.parametrize("act", ["none", "relu", "leaky_relu", "tanh", "sigmoid", "gelu"])
@pytest.mark.parametrize("od", ["f16", "bf16", "f32"])
def test_tmem_kernel_activations_and_outputs(orc, act, od):
    case = (2, 24, 12, 16, 40, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "bf16", od)
    Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, _ = case
    _, x, w, bias = inputs(case, 71)
    y = torch.full((Nb, Co, H, W), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_conv2d(to_device(x, dt), to_device(w, dt), fp32_to_device(bias), y, st, pd, dl, act, 0.3)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(y), orc.conv2d(x, w, dt, bias, st, pd, dl, act, 0.3), od, f"{act} {od}")


def test_tmem_kernel_without_bias(orc):
    case = (1, 16, 16, 16, 32, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16")
    _, x, w, _ = inputs(case, 5)
    y = torch.full((1, 32, 16, 16), float("nan"), dtype=torch.float16, device="cuda")
    mmact.mmact_conv2d(to_device(x, "f16"), to_device(w, "f16"), None, y, (1, 1), (1, 1, 1, 1), (1, 1), "relu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(y), orc.conv2d(x, w, "f16", None, (1, 1), (1, 1, 1, 1), (1, 1), "relu"), "f16", "no bias")


@pytest.mark.parametrize("in_place", [False, True], ids=["separate", "in_place"])
@pytest.mark.parametrize("case", [CASES[0], CASES[12], CASES[13], CASES[7]], ids=case_id)
def test_tmem_kernel_residual(orc, case, in_place):
    Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, od = case
    rng, x, w, bias = inputs(case, 900 + Co)
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl)
    rv = rng.uniform(-1.5, 1.5, size=(Nb, Co, Ho, Wo))
    R = rv.astype(np.float32) if od == "f32" else synth.to_codes(rv, od)
    dR = fp32_to_device(R) if od == "f32" else to_device(R, od)
    y = dR.clone() if in_place else torch.full((Nb, Co, Ho, Wo), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_conv2d_residual(to_device(x, dt), to_device(w, dt), fp32_to_device(bias), y if in_place else dR,
                                y, st, pd, dl, "gelu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    ref = orc.conv2d(x, w, dt, bias, st, pd, dl, "gelu", residual=R, res_dtype=od)
    check(host(y), ref, od, f"residual {case_id(case)}")


def test_tmem_kernel_split_variant(orc):
    # the two-kernel ablation's first kernel is this kernel with an fp32 output and no activation
    case = CASES[1]
    Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, od = case
    _, x, w, bias = inputs(case, 17)
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl)
    y = torch.full((Nb, Co, Ho, Wo), float("nan"), dtype=TORCH[od], device="cuda")
    ws = torch.full((y.numel(),), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_conv2d_split(to_device(x, dt), to_device(w, dt), fp32_to_device(bias), y, ws, st, pd, dl, "tanh")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(y), orc.conv2d(x, w, dt, bias, st, pd, dl, "tanh"), od, "split")
    check(host(ws).reshape(y.shape), orc.conv2d(x, w, dt, bias, st, pd, dl, "none"), "f32", "split workspace")
