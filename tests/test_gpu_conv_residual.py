"""GPU parity: conv2d with a residual tensor, y = act(conv2d(x, w) + bias + R),
in both layouts, against the oracle.  R has y's shape and dtype and is added to
the fp32 accumulator before the activation; R may be y itself.  The NCHW cases
cover each of the three B-tile producers (asserted), the NHWC cases both input
precisions."""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_epilogue_gb300 import build, mmact, synth
from parity import ACT_SLOPE, TF32_REL, TORCH, check, fp32_to_device, host, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    mmact.load()


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def residual_values(rng, shape, od):
    v = rng.uniform(-1.5, 1.5, size=shape)
    return v.astype(np.float32) if od == "f32" else synth.to_codes(v, od)


def residual_device(R, od):
    return fp32_to_device(R) if od == "f32" else to_device(R, od)


NCHW_CASES = [
    # (N, C, H, W, Co, kh, kw, stride, pads, dilation, dtype, out, producer)
    (2, 64, 24, 24, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16", "window"),
    (2, 16, 64, 64, 96, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "bf16", "bf16", "window"),   # Wo = 32
    (1, 40, 19, 48, 72, 3, 5, (1, 2), (0, 3, 2, 1), (2, 1), "f16", "f32", "window"),     # Wo = 24
    (2, 24, 64, 64, 200, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), "bf16", "f32", "vector"),
    (2, 24, 17, 13, 40, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "bf16", "bf16", "gather"),   # odd Wo
    (3, 3, 11, 9, 5, 3, 2, (2, 1), (1, 0, 2, 1), (1, 2), "f16", "f32", "gather"),
]


@pytest.fixture(params=["tmem", "legacy"])
def conv_mode(request):
    mmact.mmact_set_conv_tmem(0 if request.param == "tmem" else 1)
    yield request.param
    mmact.mmact_set_conv_tmem(0)


@pytest.mark.parametrize("case", NCHW_CASES, ids=lambda c: f"{c[-1]}-{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}{c[6]}")
@pytest.mark.parametrize("act", ["tanh", "relu"])
def test_nchw_residual(orc, case, act, conv_mode):
    Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, od, producer = case
    got_producer = mmact.mmact_conv2d_producer(Nb, C, H, W, Co, kh, kw, st, pd, dl, TORCH[dt], TORCH[od])
    if conv_mode == "legacy":
        assert got_producer == producer
    else:
        assert got_producer == ("tmem" if producer in ("window", "vector") else producer)
    rng = np.random.default_rng(Nb * 7 + C + Co)
    x = synth.to_codes(rng.normal(0, 1, (Nb, C, H, W)), dt)
    w = synth.to_codes(rng.normal(0, (1.0 / (C * kh * kw)) ** 0.5, (Co, C, kh, kw)), dt)
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl)
    R = residual_values(rng, (Nb, Co, Ho, Wo), od)
    y = torch.full((Nb, Co, Ho, Wo), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_conv2d_residual(to_device(x, dt), to_device(w, dt), fp32_to_device(bias),
                                residual_device(R, od), y, st, pd, dl, act)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    ref = orc.conv2d(x, w, dt, bias, st, pd, dl, act, residual=R, res_dtype=od)
    check(host(y), ref, od, f"nchw residual {case} {act}")


def test_nchw_residual_in_place(orc, conv_mode):
    rng = np.random.default_rng(41)
    Nb, C, H, W, Co = 2, 32, 20, 40, 64
    x = synth.to_codes(rng.normal(0, 1, (Nb, C, H, W)), "bf16")
    w = synth.to_codes(rng.normal(0, (1.0 / (C * 9)) ** 0.5, (Co, C, 3, 3)), "bf16")
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    R = residual_values(rng, (Nb, Co, H, W), "bf16")
    y = residual_device(R, "bf16").clone()
    mmact.mmact_conv2d_residual(to_device(x, "bf16"), to_device(w, "bf16"), fp32_to_device(bias), y, y,
                                (1, 1), (1, 1, 1, 1), (1, 1), "gelu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    ref = orc.conv2d(x, w, "bf16", bias, (1, 1), (1, 1, 1, 1), (1, 1), "gelu", residual=R, res_dtype="bf16")
    check(host(y), ref, "bf16", "nchw residual in place")


NHWC_CASES = [
    # (N, C, H, W, Co, kh, kw, stride, pads, dilation, dtype, out)
    (1, 64, 8, 8, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),
    (2, 16, 13, 11, 24, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "bf16", "f32"),
    (2, 32, 17, 19, 200, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), "f16", "bf16"),
    (1, 36, 10, 12, 40, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f32", "f32"),     # fp32 inputs as tf32
]


@pytest.mark.parametrize("case", NHWC_CASES, ids=lambda c: f"{c[-2]}-{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}{c[6]}")
def test_nhwc_residual(orc, case):
    Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, od = case
    rng = np.random.default_rng(Nb * 11 + C + Co)
    xv = rng.normal(0, 1, (Nb, C, H, W))
    wv = rng.normal(0, (1.0 / (C * kh * kw)) ** 0.5, (Co, C, kh, kw))
    if dt == "f32":
        x, w = xv.astype(np.float32), wv.astype(np.float32)
        dx = torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 3, 1))).cuda()
        dw = torch.from_numpy(np.ascontiguousarray(w.transpose(0, 2, 3, 1))).cuda()
    else:
        x, w = synth.to_codes(xv, dt), synth.to_codes(wv, dt)
        dx = to_device(np.ascontiguousarray(x.transpose(0, 2, 3, 1)), dt)
        dw = to_device(np.ascontiguousarray(w.transpose(0, 2, 3, 1)), dt)
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl)
    R = residual_values(rng, (Nb, Co, Ho, Wo), od)                  # NCHW for the oracle
    R_nhwc = np.ascontiguousarray(R.transpose(0, 2, 3, 1))
    y = torch.full((Nb, Ho, Wo, Co), float("nan"), dtype=TORCH[od], device="cuda")
    mmact.mmact_conv2d_nhwc_residual(dx, dw, fp32_to_device(bias), residual_device(R_nhwc, od), y,
                                     st, pd, dl, "tanh", tf32=dt == "f32")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    ref = orc.conv2d(x, w, dt, bias, st, pd, dl, "tanh", residual=R, res_dtype=od)
    extra = None
    if dt == "f32":
        extra = ACT_SLOPE * TF32_REL * orc.conv2d(np.abs(x), np.abs(w), "f32", None, st, pd, dl, "none")
    check(host(y).transpose(0, 3, 1, 2), ref, od, f"nhwc residual {case}", extra=extra)


def test_residual_binding_rejects_mismatch():
    x = torch.zeros((1, 8, 8, 8), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 8, 3, 3), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, 8, 6, 6), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        mmact.mmact_conv2d_residual(x, w, None, torch.zeros((1, 8, 6, 7), dtype=torch.bfloat16,
                                                            device="cuda"), y)
