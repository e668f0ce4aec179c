"""GPU parity: the fused implicit-GEMM conv2d kernel (and its ablation) against the oracle.

Small geometries sweep stride, padding (asymmetric too), dilation, kernel
size, channel counts that leave ragged K / Co / pixel tiles, and the
fallback paths (filter rows whose pitch rules out TMA, outputs whose pitch
rules out TMA stores), each under both NCHW kernel families (the tensor-memory
im2col kernel where it applies, and the window / vector / gather producers).
The full workloads are compared element by element.
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


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.fixture(params=["tmem", "legacy"])
def conv_mode(request):
    """NCHW kernel family: the tensor-memory im2col kernel where it applies, or
    the window / vector / gather producers everywhere."""
    mmact.mmact_set_conv_tmem(0 if request.param == "tmem" else 1)
    yield request.param
    mmact.mmact_set_conv_tmem(0)


@pytest.fixture
def legacy_mode():
    mmact.mmact_set_conv_tmem(1)
    yield
    mmact.mmact_set_conv_tmem(0)


def run_conv(x, w, bias, dt, od, stride, pads, dil, act, alpha=0.0, split=False):
    Nb, C, H, W = x.shape
    Co, _, kh, kw = w.shape
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, stride, pads, dil)
    dx, dw = to_device(x, dt), to_device(w, dt)
    y = torch.full((Nb, Co, Ho, Wo), float("nan"), dtype=TORCH[od], device="cuda")
    if split:
        ws = torch.full((y.numel(),), float("nan"), dtype=torch.float32, device="cuda")
        mmact.mmact_conv2d_split(dx, dw, fp32_to_device(bias), y, ws, stride, pads, dil, act, alpha)
    else:
        mmact.mmact_conv2d(dx, dw, fp32_to_device(bias), y, stride, pads, dil, act, alpha)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    return y


CASES = [
    # (N, C, H, W, Co, kh, kw, stride, pads, dilation, dtype, out)
    (1, 8, 8, 8, 16, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),
    (2, 16, 12, 20, 32, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "bf16", "bf16"),
    (2, 24, 17, 13, 40, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "bf16", "bf16"),
    (1, 8, 16, 16, 8, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), "bf16", "f32"),
    (3, 3, 11, 9, 5, 3, 2, (2, 1), (1, 0, 2, 1), (1, 2), "f16", "f32"),      # K = 18: gathered filter
    (1, 64, 16, 16, 130, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),  # ragged Co tile
    (2, 72, 9, 15, 8, 5, 5, (1, 2), (2, 2, 1, 3), (1, 1), "bf16", "bf16"),   # K not a multiple of 64
    (1, 16, 30, 30, 64, 7, 7, (2, 2), (3, 3, 3, 3), (1, 1), "f16", "f16"),
    (1, 4, 5, 5, 3, 5, 5, (1, 1), (0, 0, 0, 0), (1, 1), "f16", "bf16"),      # one output pixel
    (16, 16, 64, 64, 128, 1, 1, (1, 1), (0, 0, 0, 0), (1, 1), "f16", "f16"), # one K block, several tiles a CTA
]


# Geometries that take the vectorised producer (input width a multiple of 8,
# horizontal stride 1 or 2, filter pitch a multiple of 16 bytes): ragged output
# rows and columns, several column tiles, exactly-32-wide outputs, asymmetric
# pads, dilation, fp32 output, ragged channel tiles and K tails.
VEC_CASES = [
    (2, 64, 24, 24, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16"),
    (1, 32, 40, 144, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), "bf16", "bf16"),    # Wo = 144: 3 col tiles
    (2, 16, 64, 64, 96, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), "bf16", "bf16"),     # Wo = 32 exactly
    (2, 24, 64, 64, 200, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), "bf16", "f32"),     # 1x1 s2, Co ragged
    (1, 40, 19, 48, 72, 3, 5, (1, 2), (0, 3, 2, 1), (2, 1), "f16", "f32"),       # asymmetric
    (3, 8, 10, 16, 24, 5, 5, (1, 1), (2, 2, 2, 2), (1, 1), "f16", "bf16"),       # K = 200
    (1, 16, 7, 16, 16, 3, 3, (2, 1), (1, 1, 2, 2), (1, 2), "bf16", "f16"),       # Wo = 16, Ho = 4
    (1, 64, 32, 32, 64, 1, 1, (1, 1), (0, 0, 0, 0), (1, 1), "f16", "f16"),       # 1x1: global loads
    (2, 20, 24, 40, 48, 2, 2, (1, 1), (0, 1, 1, 0), (1, 1), "bf16", "bf16"),     # 2x2: 17-channel window
    (1, 16, 20, 24, 16, 7, 7, (1, 1), (3, 3, 3, 3), (1, 1), "f16", "f32"),       # 7x7 window
]

# Producer each vectorised case takes (both vectorised producers must be covered).
VEC_PRODUCERS = ["window", "window", "window", "vector", "window", "window", "window", "vector",
                 "window", "window"]


def test_vectorised_cases_cover_both_producers(legacy_mode):
    for case, want in zip(VEC_CASES, VEC_PRODUCERS, strict=True):
        Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, od = case
        assert mmact.mmact_conv2d_producer(Nb, C, H, W, Co, kh, kw, st, pd, dl, TORCH[dt], TORCH[od]) == want, case
    for case in CASES:
        Nb, C, H, W, Co, kh, kw, st, pd, dl, dt, od = case
        assert mmact.mmact_conv2d_producer(Nb, C, H, W, Co, kh, kw, st, pd, dl, TORCH[dt], TORCH[od]) in (
            "gather", "window", "vector")


@pytest.mark.parametrize("case", VEC_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}{c[6]}s{c[7][0]}{c[7][1]}")
@pytest.mark.parametrize("act", ["tanh", "relu", "sigmoid", "gelu"])
def test_vectorised_geometries(orc, case, act, conv_mode):
    test_small_geometries(orc, case, act, conv_mode)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}{c[6]}s{c[7][0]}{c[7][1]}")
@pytest.mark.parametrize("act", ["tanh", "leaky_relu", "sigmoid", "gelu"])
def test_small_geometries(orc, case, act, conv_mode):
    Nb, C, H, W, Co, kh, kw, stride, pads, dil, dt, od = case
    rng = np.random.default_rng(Nb * 1000 + C * 10 + Co)
    x = synth.to_codes(rng.normal(0, 1, (Nb, C, H, W)), dt)
    w = synth.to_codes(rng.normal(0, (1.0 / (C * kh * kw)) ** 0.5, (Co, C, kh, kw)), dt)
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    y = run_conv(x, w, bias, dt, od, stride, pads, dil, act, 0.1)
    ref = orc.conv2d(x, w, dt, bias, stride, pads, dil, act, 0.1)
    check(host(y), ref, od, f"{case} {act}")


def test_split_small(orc):
    rng = np.random.default_rng(77)
    x = synth.to_codes(rng.normal(0, 1, (2, 16, 12, 12)), "bf16")
    w = synth.to_codes(rng.normal(0, 0.08, (24, 16, 3, 3)), "bf16")
    bias = rng.uniform(-0.1, 0.1, 24).astype(np.float32)
    y = run_conv(x, w, bias, "bf16", "bf16", (1, 1), (1, 1, 1, 1), (1, 1), "tanh", split=True)
    check(host(y), orc.conv2d(x, w, "bf16", bias, (1, 1), (1, 1, 1, 1), (1, 1), "tanh"), "bf16", "split")


def test_zero_input_channels_gives_act_of_bias(orc):
    bias = np.array([0.5, -1.5, 2.0], dtype=np.float32)
    dx = torch.empty((2, 0, 4, 4), dtype=torch.float16, device="cuda")
    dw = torch.empty((3, 0, 3, 3), dtype=torch.float16, device="cuda")
    y = torch.full((2, 3, 4, 4), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_conv2d(dx, dw, fp32_to_device(bias), y, (1, 1), (1, 1, 1, 1), (1, 1), "tanh")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    exp = np.broadcast_to(np.tanh(bias.astype(np.float64))[None, :, None, None], (2, 3, 4, 4))
    check(host(y), exp, "f32", "C=0")


CONV_WORKLOADS = [w for w in synth.WORKLOADS.values() if w.kind == "conv"]


_FULL_REF = {}


def workload_reference(orc, wl, inp):
    """Every output element of a conv workload from the oracle (computed once per run)."""
    if wl.name not in _FULL_REF:
        _FULL_REF[wl.name] = orc.conv2d(inp["x"], inp["w"], wl.dtype, inp["bias"], wl.stride, wl.pads,
                                        wl.dilation, wl.act, wl.alpha).ravel()
    return _FULL_REF[wl.name]


@pytest.mark.parametrize("wl", CONV_WORKLOADS, ids=lambda w: w.name)
@pytest.mark.parametrize("split", [False, True], ids=["fused", "split"])
def test_workload_parity(orc, wl, split, conv_mode):
    # every output element of the workload against the oracle (1.8e9-4.8e9 fp64 MACs each)
    inp = wl.inputs()
    if conv_mode == "tmem":
        assert mmact.mmact_conv2d_producer(wl.N, wl.C, wl.H, wl.W, wl.Co, wl.kh, wl.kw, wl.stride, wl.pads,
                                           wl.dilation, TORCH[wl.dtype], TORCH[wl.out_dtype]) == "tmem"
    y = run_conv(inp["x"], inp["w"], inp["bias"], wl.dtype, wl.out_dtype, wl.stride, wl.pads,
                 wl.dilation, wl.act, wl.alpha, split=split)
    check(host(y).ravel(), workload_reference(orc, wl, inp), wl.out_dtype, wl.name)
