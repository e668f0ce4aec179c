"""Pins that tie the oracle to something other than itself.

Each check takes an ``oracle.Oracle`` instance and raises AssertionError when
the oracle disagrees with what the pages and the mathematics fix: hand-worked
fixtures, closed forms, special cases that reduce to a library routine, and
brute force against torch's float64 CPU operators on tiny shapes.  The same
checks run against the committed oracle (they must all pass) and against
deliberately broken copies of it (at least one must fail), which shows that a
plausible mistake anywhere in the oracle is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f16_codes(values) -> np.ndarray:
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_codes(values) -> np.ndarray:
    # exact for the small integers / dyadic values the pins use
    v = np.asarray(values, dtype=np.float32)
    u = v.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "pin value not exact in bfloat16"
    return (u >> 16).astype(np.uint16)


def codes(values, dtype):
    return f16_codes(values) if dtype == "f16" else bf16_codes(values)


def act_ref(z, act, alpha):
    """Activation written independently with numpy, for brute-force checks."""
    z = np.asarray(z, dtype=np.float64)
    if act == "none":
        return z
    if act == "relu":
        return np.where(z > 0, z, 0.0)
    if act == "leaky_relu":
        return np.where(z > 0, z, alpha * z)
    if act == "tanh":
        return np.tanh(z)
    if act == "sigmoid":
        return scipy.special.expit(z)
    if act == "gelu":
        return z * scipy.special.ndtr(z)
    raise ValueError(act)


# ---------------------------------------------------------------- decoding --
def check_decode_f16(orc):
    # values fixed by the binary16 definition, worked by hand
    hand = {0x0000: 0.0, 0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0400: 2.0 ** -14,
            0x0001: 2.0 ** -24, 0x3555: 0.333251953125, 0x3800: 0.5, 0xBC01: -(1 + 2.0 ** -10)}
    for c, v in hand.items():
        got = float(orc.decode([c], "f16")[0])
        assert got == v, (hex(c), got, v)
    # every finite code against numpy's float16 (library cross-check)
    allc = np.arange(0, 1 << 16, 97, dtype=np.uint16)
    ref = allc.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    got = orc.decode(allc[fin], "f16")
    assert np.array_equal(got, ref[fin])


def check_decode_bf16(orc):
    hand = {0x3F80: 1.0, 0xC000: -2.0, 0x4049: 3.140625, 0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126,
            0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127, 0x3E80: 0.25, 0xBF81: -(1 + 2.0 ** -7)}
    for c, v in hand.items():
        got = float(orc.decode([c], "bf16")[0])
        assert got == v, (hex(c), got, v)
    allc = np.arange(0, 1 << 16, 89, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        ref = (allc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fin = np.isfinite(ref)
    got = orc.decode(allc[fin], "bf16")
    assert np.array_equal(got, ref[fin])


# ------------------------------------------------------------- activations --
def check_act_points(orc):
    pts = [-2.0, -1e-3, -0.0, 0.0, 1e-3, 2.0]
    # ReLU: z > 0 ? z : 0
    assert list(orc.act(pts, "relu")) == [0.0, 0.0, 0.0, 0.0, 1e-3, 2.0]
    # LeakyReLU with alpha 0.01: negatives scaled, positives kept
    got = orc.act(pts, "leaky_relu", 0.01)
    exp = [-0.02, -1e-5, 0.0, 0.0, 1e-3, 2.0]
    assert np.allclose(got, exp, rtol=0, atol=1e-18), got
    # alpha = 1 is the identity, alpha = 0 is ReLU
    assert list(orc.act(pts, "leaky_relu", 1.0)) == pts
    assert list(orc.act(pts, "leaky_relu", 0.0)) == list(orc.act(pts, "relu"))
    assert list(orc.act(pts, "none")) == pts
    # alpha = 0.2 at -5 gives -1
    assert float(orc.act([-5.0], "leaky_relu", 0.2)[0]) == -1.0


def check_tanh(orc):
    zs = np.concatenate([np.linspace(-30, 30, 1201), [1e-12, -1e-9, 0.5, 19.999, 20.001, 700.0, -1e4]])
    for z in zs:
        got = orc.tanh(z)
        ref = math.tanh(z)
        assert abs(got - ref) <= 1e-15 + 4e-15 * abs(ref), (z, got, ref)
        assert orc.tanh(-z) == -got                      # odd
        assert abs(got) <= 1.0 and not math.isnan(got)
    assert orc.tanh(0.0) == 0.0
    assert orc.tanh(25.0) == 1.0 and orc.tanh(-25.0) == -1.0
    # the act switch routes to it
    assert float(orc.act([0.75], "tanh")[0]) == orc.tanh(0.75)


def check_sigmoid(orc):
    lib = orc.lib
    assert lib.oracle_sigmoid(0.0) == 0.5
    for z in np.concatenate([np.linspace(-40, 40, 801), [1e-9, -3e-7, 700.0, -700.0]]):
        got = lib.oracle_sigmoid(float(z))
        assert abs(got - scipy.special.expit(z)) <= 1e-16 + 4e-16 * abs(got), (z, got)
        # sigma(z) + sigma(-z) = 1 and sigma(z) = (1 + tanh(z/2)) / 2
        assert abs(got + lib.oracle_sigmoid(float(-z)) - 1.0) <= 5e-16
        assert abs(got - 0.5 * (1.0 + math.tanh(z / 2))) <= 5e-16
        assert 0.0 <= got <= 1.0
    assert float(orc.act([1.5], "sigmoid")[0]) == lib.oracle_sigmoid(1.5)


def check_gelu(orc):
    lib = orc.lib
    assert lib.oracle_gelu(0.0) == 0.0
    for z in np.concatenate([np.linspace(-12, 12, 481), [1e-9, -2e-6]]):
        got = lib.oracle_gelu(float(z))
        # z * Phi(z), Phi the standard normal CDF (library)
        assert abs(got - z * scipy.special.ndtr(z)) <= 1e-15 + 4e-15 * abs(got), (z, got)
        # GELU(z) - GELU(-z) = z (Phi(z) + Phi(-z) = 1)
        assert abs(got - lib.oracle_gelu(float(-z)) - z) <= 1e-14 * max(1.0, abs(z))
    assert abs(lib.oracle_gelu(10.0) - 10.0) < 1e-15 and abs(lib.oracle_gelu(-10.0)) < 1e-20
    assert float(orc.act([0.3], "gelu")[0]) == lib.oracle_gelu(0.3)


# -------------------------------------------------------------------- GEMM --
def _rand_codes(rng, shape, dtype, scale=1.0):
    v = rng.uniform(-scale, scale, size=shape)
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def check_gemm_identity(orc):
    rng = np.random.default_rng(11)
    for dtype in ("f16", "bf16"):
        M, K = 5, 7
        A = _rand_codes(rng, (M, K), dtype)
        B = codes(np.eye(K), dtype)
        bias = rng.uniform(-1, 1, K).astype(np.float32)
        Ad = orc.decode(A, dtype)
        for act, alpha in (("none", 0), ("relu", 0), ("leaky_relu", 0.3)):
            got = orc.gemm(A, B, dtype, bias, act, alpha)
            exp = act_ref(Ad + bias.astype(np.float64)[None, :], act, alpha)
            assert np.array_equal(got, exp), (dtype, act)


def check_gemm_permutation(orc):
    rng = np.random.default_rng(12)
    M, K, N = 4, 6, 9
    A = _rand_codes(rng, (M, K), "bf16")
    src = rng.integers(0, K, size=N)            # column j of C copies column src[j] of A
    P = np.zeros((K, N))
    P[src, np.arange(N)] = 1.0
    B = codes(P, "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    got = orc.gemm(A, B, "bf16", bias, "none")
    exp = orc.decode(A, "bf16")[:, src] + bias.astype(np.float64)[None, :]
    assert np.array_equal(got, exp)


def check_gemm_ones(orc):
    for (M, N, K) in ((3, 5, 7), (1, 1, 1), (2, 8, 64)):
        A = codes(np.ones((M, K)), "f16")
        B = codes(np.ones((K, N)), "f16")
        bias = np.arange(N, dtype=np.float32) - 2.5
        got = orc.gemm(A, B, "f16", bias, "none")
        assert np.array_equal(got, np.broadcast_to(K + bias.astype(np.float64), (M, N)))
    # no bias means zero bias
    got = orc.gemm(codes(np.ones((2, 3)), "f16"), codes(np.ones((3, 4)), "f16"), "f16", None, "none")
    assert np.array_equal(got, np.full((2, 4), 3.0))


def check_gemm_bruteforce(orc):
    rng = np.random.default_rng(13)
    for trial in range(12):
        M, N, K = (int(v) for v in rng.integers(1, 10, size=3))
        dtype = ("f16", "bf16")[trial % 2]
        act, alpha = [("none", 0), ("relu", 0), ("leaky_relu", 0.2), ("tanh", 0), ("sigmoid", 0),
                      ("gelu", 0)][trial % 6]
        A = _rand_codes(rng, (M, K), dtype, 2.0)
        B = _rand_codes(rng, (K, N), dtype, 2.0)
        bias = rng.uniform(-1, 1, N).astype(np.float32)
        At = torch.from_numpy(orc.decode(A, dtype))
        Bt = torch.from_numpy(orc.decode(B, dtype))
        z = (torch.matmul(At, Bt) + torch.from_numpy(bias.astype(np.float64))).numpy()
        exp = act_ref(z, act, alpha)
        got = orc.gemm(A, B, dtype, bias, act, alpha)
        assert got.shape == (M, N)
        assert np.allclose(got, exp, rtol=1e-12, atol=1e-12), (M, N, K, act)


def check_gemm_points(orc):
    rng = np.random.default_rng(14)
    M, N, K = 7, 11, 5
    A = _rand_codes(rng, (M, K), "bf16")
    B = _rand_codes(rng, (K, N), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    full = orc.gemm(A, B, "bf16", bias, "leaky_relu", 0.2)
    pts = rng.integers(0, M * N, size=20)
    part = orc.gemm(A, B, "bf16", bias, "leaky_relu", 0.2, points=pts, threads=3)
    assert np.array_equal(part, full.ravel()[pts])


def check_gemm_golden(orc):
    with open(os.path.join(GOLDEN, "gemm_2x2x3_leakyrelu.json")) as f:
        g = json.load(f)
    A = codes(g["A"], g["dtype"])
    B = codes(g["B"], g["dtype"])
    bias = np.asarray(g["bias"], dtype=np.float32)
    z = orc.gemm(A, B, g["dtype"], bias, "none")
    assert np.array_equal(z, np.asarray(g["z"]))
    got = orc.gemm(A, B, g["dtype"], bias, g["act"], g["alpha"])
    assert np.allclose(got, np.asarray(g["expected"]), rtol=1e-15, atol=0)


def _res_values(R, res_dtype):
    """Residual codes / values as float64, decoded with numpy (independent of the oracle)."""
    R = np.asarray(R)
    if res_dtype == "f32":
        return R.astype(np.float32).astype(np.float64)
    if res_dtype == "f16":
        return R.astype(np.uint16).view(np.float16).astype(np.float64)
    return (R.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_gemm_residual_identity(orc):
    # B = I: the contraction is a copy, so C = act(A + bias + R) exactly
    rng = np.random.default_rng(15)
    M, K = 6, 5
    for dtype, res_dtype in (("f16", "f16"), ("bf16", "bf16"), ("bf16", "f32")):
        A = _rand_codes(rng, (M, K), dtype)
        B = codes(np.eye(K), dtype)
        bias = rng.uniform(-1, 1, K).astype(np.float32)
        R = (rng.uniform(-2, 2, (M, K)).astype(np.float32) if res_dtype == "f32"
             else _rand_codes(rng, (M, K), res_dtype, 2.0))
        Ad = orc.decode(A, dtype)
        for act, alpha in (("none", 0), ("relu", 0), ("leaky_relu", 0.3)):
            got = orc.gemm(A, B, dtype, bias, act, alpha, residual=R, res_dtype=res_dtype)
            exp = act_ref(Ad + bias.astype(np.float64)[None, :] + _res_values(R, res_dtype), act, alpha)
            assert np.array_equal(got, exp), (dtype, res_dtype, act)


def check_gemm_residual_golden(orc):
    with open(os.path.join(GOLDEN, "gemm_2x2x2_residual_relu.json")) as f:
        g = json.load(f)
    A = codes(g["A"], g["dtype"])
    B = codes(g["B"], g["dtype"])
    R = codes(g["residual"], g["res_dtype"])
    bias = np.asarray(g["bias"], dtype=np.float32)
    z = orc.gemm(A, B, g["dtype"], bias, "none", residual=R, res_dtype=g["res_dtype"])
    assert np.array_equal(z, np.asarray(g["z"]))
    got = orc.gemm(A, B, g["dtype"], bias, g["act"], residual=R, res_dtype=g["res_dtype"])
    assert np.array_equal(got, np.asarray(g["expected"]))


def check_gemm_f32_inputs(orc):
    # fp32 inputs are used exactly: brute force against torch float64 of the same values,
    # and identity B copies A
    rng = np.random.default_rng(16)
    for (M, N, K) in ((3, 5, 7), (6, 2, 9)):
        A = rng.uniform(-2, 2, (M, K)).astype(np.float32)
        B = rng.uniform(-2, 2, (K, N)).astype(np.float32)
        bias = rng.uniform(-1, 1, N).astype(np.float32)
        z = (torch.from_numpy(A.astype(np.float64)) @ torch.from_numpy(B.astype(np.float64))).numpy()
        exp = act_ref(z + bias.astype(np.float64)[None, :], "leaky_relu", 0.1)
        got = orc.gemm(A, B, "f32", bias, "leaky_relu", 0.1)
        assert np.allclose(got, exp, rtol=1e-13, atol=1e-13)
    A = np.float32([[1.0 + 2.0 ** -20, -3.25], [0.1, 7.0]])       # not representable in 16 bits
    got = orc.gemm(A, np.eye(2, dtype=np.float32), "f32", None, "none")
    assert np.array_equal(got, A.astype(np.float64))


# -------------------------------------------------------------------- conv --
def check_conv_shape(orc):
    # the workloads' own shapes
    assert orc.conv_out_dim(56, 3, 1, 1, 1, 1) == 56
    assert orc.conv_out_dim(64, 3, 2, 2, 2, 2) == 32
    assert orc.conv_out_dim(64, 1, 2, 0, 0, 1) == 32
    # the rule against torch on a sweep of tiny geometries
    for size in (1, 2, 5, 7, 8):
        for k in (1, 2, 3):
            for s in (1, 2, 3):
                for p in (0, 1, 2):
                    for d in (1, 2):
                        x = torch.zeros(1, 1, size, size, dtype=torch.float64)
                        w = torch.zeros(1, 1, k, k, dtype=torch.float64)
                        span = size + 2 * p - d * (k - 1) - 1
                        got = orc.conv_out_dim(size, k, s, p, p, d)
                        if span < 0:
                            assert got == 0
                            continue
                        ref = F.conv2d(x, w, stride=s, padding=p, dilation=d).shape[-1]
                        assert got == ref, (size, k, s, p, d, got, ref)
    # asymmetric pads add
    assert orc.conv_out_dim(5, 3, 1, 2, 0, 1) == 5


def _torch_conv(orc, x, w, dtype, bias, stride, pads, dil):
    if dtype == "f32":
        xt = torch.from_numpy(np.asarray(x, dtype=np.float32).astype(np.float64))
        wt = torch.from_numpy(np.asarray(w, dtype=np.float32).astype(np.float64))
    else:
        xt = torch.from_numpy(orc.decode(x, dtype))
        wt = torch.from_numpy(orc.decode(w, dtype))
    pt, pb, pl, pr = pads
    xt = F.pad(xt, (pl, pr, pt, pb))
    bt = None if bias is None else torch.from_numpy(bias.astype(np.float64))
    return F.conv2d(xt, wt, bt, stride=stride, dilation=dil).numpy()


def check_conv_bruteforce(orc):
    rng = np.random.default_rng(21)
    for trial in range(40):
        Nb = int(rng.integers(1, 3))
        C = int(rng.integers(1, 4))
        Co = int(rng.integers(1, 4))
        H = int(rng.integers(1, 8))
        W = int(rng.integers(1, 8))
        kh = int(rng.integers(1, 4))
        kw = int(rng.integers(1, 4))
        stride = (int(rng.integers(1, 4)), int(rng.integers(1, 4)))
        pads = tuple(int(v) for v in rng.integers(0, 3, size=4))
        dil = (int(rng.integers(1, 3)), int(rng.integers(1, 3)))
        Ho = orc.conv_out_dim(H, kh, stride[0], pads[0], pads[1], dil[0])
        Wo = orc.conv_out_dim(W, kw, stride[1], pads[2], pads[3], dil[1])
        if Ho <= 0 or Wo <= 0:
            continue
        dtype = ("f16", "bf16")[trial % 2]
        act, alpha = [("none", 0), ("tanh", 0), ("relu", 0), ("leaky_relu", 0.1)][trial % 4]
        x = _rand_codes(rng, (Nb, C, H, W), dtype, 2.0)
        w = _rand_codes(rng, (Co, C, kh, kw), dtype, 1.0)
        bias = rng.uniform(-1, 1, Co).astype(np.float32) if trial % 3 else None
        z = _torch_conv(orc, x, w, dtype, bias, stride, pads, dil)
        exp = act_ref(z, act, alpha)
        got = orc.conv2d(x, w, dtype, bias, stride, pads, dil, act, alpha)
        assert got.shape == exp.shape, (got.shape, exp.shape)
        assert np.allclose(got, exp, rtol=1e-12, atol=1e-12), (trial, Nb, C, H, W, Co, kh, kw,
                                                                stride, pads, dil)


def check_conv_delta(orc):
    """A one-hot filter tap over an identity channel map shifts x by (r*d - p, q*d - p)."""
    rng = np.random.default_rng(22)
    C, H, W = 2, 6, 7
    x = _rand_codes(rng, (1, C, H, W), "bf16")
    xd = orc.decode(x, "bf16")
    for (r, q, s, p, d) in ((0, 0, 1, 0, 1), (1, 2, 1, 1, 1), (2, 1, 2, 2, 2), (1, 1, 1, 2, 2)):
        k = 3
        w = np.zeros((C, C, k, k))
        for c in range(C):
            w[c, c, r, q] = 1.0
        bias = np.array([0.5, -0.25], dtype=np.float32)
        got = orc.conv2d(x, codes(w, "bf16"), "bf16", bias, (s, s), (p, p, p, p), (d, d), "none")
        Ho, Wo = got.shape[2], got.shape[3]
        exp = np.zeros_like(got)
        for c in range(C):
            for oh in range(Ho):
                for ow in range(Wo):
                    ih, iw = oh * s - p + r * d, ow * s - p + q * d
                    v = xd[0, c, ih, iw] if (0 <= ih < H and 0 <= iw < W) else 0.0
                    exp[0, c, oh, ow] = v + float(bias[c])
        assert np.array_equal(got, exp), (r, q, s, p, d)


def check_conv_as_gemm(orc):
    """conv == the GEMM oracle applied to an explicitly built im2col matrix."""
    rng = np.random.default_rng(23)
    Nb, C, H, W, Co, kh, kw = 2, 3, 6, 5, 4, 3, 2
    stride, pads, dil = (2, 1), (1, 0, 2, 1), (1, 2)
    x = _rand_codes(rng, (Nb, C, H, W), "f16")
    w = _rand_codes(rng, (Co, C, kh, kw), "f16")
    bias = rng.uniform(-1, 1, Co).astype(np.float32)
    y = orc.conv2d(x, w, "f16", bias, stride, pads, dil, "leaky_relu", 0.2)
    Ho, Wo = y.shape[2], y.shape[3]
    for n in range(Nb):
        cols = np.zeros((C * kh * kw, Ho * Wo), dtype=np.uint16)       # code 0 is +0.0
        for ci in range(C):
            for r in range(kh):
                for q in range(kw):
                    k = (ci * kh + r) * kw + q
                    for oh in range(Ho):
                        for ow in range(Wo):
                            ih = oh * stride[0] - pads[0] + r * dil[0]
                            iw = ow * stride[1] - pads[2] + q * dil[1]
                            if 0 <= ih < H and 0 <= iw < W:
                                cols[k, oh * Wo + ow] = x[n, ci, ih, iw]
        # GEMM view: [Co x K] . [K x P]; bias runs along rows here, so add it after
        g = orc.gemm(w.reshape(Co, -1), cols, "f16", None, "none")
        exp = act_ref(g + bias.astype(np.float64)[:, None], "leaky_relu", 0.2)
        assert np.allclose(y[n].reshape(Co, -1), exp, rtol=1e-13, atol=1e-13)


def check_conv_points(orc):
    rng = np.random.default_rng(24)
    x = _rand_codes(rng, (2, 3, 7, 6), "bf16")
    w = _rand_codes(rng, (5, 3, 3, 3), "bf16")
    bias = rng.uniform(-1, 1, 5).astype(np.float32)
    full = orc.conv2d(x, w, "bf16", bias, (1, 2), (1, 1, 0, 2), (2, 1), "tanh")
    pts = rng.integers(0, full.size, size=25)
    part = orc.conv2d(x, w, "bf16", bias, (1, 2), (1, 1, 0, 2), (2, 1), "tanh", points=pts, threads=4)
    assert np.array_equal(part, full.ravel()[pts])


def check_conv_golden(orc):
    for name in ("conv_3x3_k2_s2_p1_tanh.json", "conv_4x4_k2_d2_none.json"):
        with open(os.path.join(GOLDEN, name)) as f:
            g = json.load(f)
        x = codes(g["x"], g["dtype"])
        w = codes(g["w"], g["dtype"])
        bias = np.asarray(g["bias"], dtype=np.float32)
        z = orc.conv2d(x, w, g["dtype"], bias, tuple(g["stride"]), tuple(g["pads"]),
                       tuple(g["dilation"]), "none")
        assert np.array_equal(z, np.asarray(g["z"], dtype=np.float64)), name
        y = orc.conv2d(x, w, g["dtype"], bias, tuple(g["stride"]), tuple(g["pads"]),
                       tuple(g["dilation"]), g["act"])
        exp = np.vectorize(math.tanh)(z) if g["act"] == "tanh" else z
        assert np.allclose(y, exp, rtol=4e-15, atol=1e-15), name


def check_conv_f32_inputs(orc):
    rng = np.random.default_rng(26)
    x = rng.uniform(-2, 2, (2, 3, 7, 6)).astype(np.float32)
    w = rng.uniform(-1, 1, (4, 3, 3, 2)).astype(np.float32)
    bias = rng.uniform(-1, 1, 4).astype(np.float32)
    for stride, pads, dil in (((1, 1), (1, 1, 1, 1), (1, 1)), ((2, 1), (0, 2, 1, 0), (1, 2))):
        got = orc.conv2d(x, w, "f32", bias, stride, pads, dil, "none")
        ref = _torch_conv(orc, x, w, "f32", bias, stride, pads, dil)
        assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


def check_conv_residual(orc):
    # with no activation the residual enters linearly, element by element in y's own order
    rng = np.random.default_rng(25)
    x = _rand_codes(rng, (2, 3, 6, 7), "f16")
    w = _rand_codes(rng, (4, 3, 3, 2), "f16")
    bias = rng.uniform(-1, 1, 4).astype(np.float32)
    geo = ((2, 1), (1, 0, 1, 1), (1, 2))
    base = orc.conv2d(x, w, "f16", bias, *geo, "none")
    R = _rand_codes(rng, base.shape, "bf16", 2.0)
    got = orc.conv2d(x, w, "f16", bias, *geo, "none", residual=R, res_dtype="bf16")
    assert np.array_equal(got, base + _res_values(R, "bf16"))
    # and before the activation: tanh(z + R)
    got = orc.conv2d(x, w, "f16", bias, *geo, "tanh", residual=R, res_dtype="bf16")
    assert np.allclose(got, np.tanh(base + _res_values(R, "bf16")), rtol=4e-15, atol=1e-15)


ALL_CHECKS = [
    check_decode_f16, check_decode_bf16, check_act_points, check_tanh, check_sigmoid, check_gelu,
    check_gemm_identity, check_gemm_permutation, check_gemm_ones, check_gemm_bruteforce,
    check_gemm_points, check_gemm_golden, check_gemm_residual_identity, check_gemm_residual_golden,
    check_gemm_f32_inputs,
    check_conv_shape, check_conv_bruteforce, check_conv_delta, check_conv_as_gemm,
    check_conv_points, check_conv_golden, check_conv_residual, check_conv_f32_inputs,
]
