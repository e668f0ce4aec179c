"""GPU parity: the fused GEMM kernel (and its two-kernel ablation) against the oracle.

Small shapes are compared element by element over every output; they cover
several tiles in M and N, ragged M/N/K tails, every tile width, both input
dtypes, all three output dtypes and all activations.  The full-size
workloads, in the launch configuration the benchmark times, are compared on
seeded samples of output elements that the oracle evaluates one by one.
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
    yield
    mmact.mmact_set_gemm_tile_n(0)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def run_gemm(A, B, bias, ab, cd, act, alpha, split=False):
    M, K = A.shape
    N = B.shape[1]
    dA, dB = to_device(A, ab), to_device(B, ab)
    db = fp32_to_device(bias)
    C = torch.full((M, N), float("nan"), dtype=TORCH[cd], device="cuda")
    ws = None
    if split:
        ws = torch.full((M * N,), float("nan"), dtype=torch.float32, device="cuda")
        mmact.mmact_gemm_split(dA, dB, db, C, ws, act, alpha)
    else:
        mmact.mmact_gemm(dA, dB, db, C, act, alpha)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    return C, ws


def rand_codes(rng, shape, dtype, lo=-1.0, hi=1.0):
    return synth.to_codes(rng.uniform(lo, hi, size=shape), dtype)


SMALL = [  # (M, N, K)
    (128, 64, 64), (1, 8, 8), (7, 24, 40), (129, 72, 200), (300, 264, 136), (256, 512, 520),
    (64, 1000, 64),
]


@pytest.mark.parametrize("tile_n", [64, 128, 192, 224, 256])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_all_tiles(orc, tile_n, shape):
    M, N, K = shape
    rng = np.random.default_rng(M * 7 + N * 13 + K + tile_n)
    mmact.mmact_set_gemm_tile_n(tile_n)
    for ab, cd, act, alpha in [("bf16", "bf16", "leaky_relu", 0.2), ("f16", "f32", "relu", 0.0),
                               ("bf16", "f16", "tanh", 0.0), ("f16", "bf16", "none", 0.0),
                               ("bf16", "f32", "sigmoid", 0.0), ("f16", "bf16", "gelu", 0.0)]:
        A = rand_codes(rng, (M, K), ab)
        B = rand_codes(rng, (K, N), ab)
        bias = rng.uniform(-1, 1, N).astype(np.float32)
        C, _ = run_gemm(A, B, bias, ab, cd, act, alpha)
        ref = orc.gemm(A, B, ab, bias, act, alpha)
        check(host(C), ref, cd, f"{shape} tile {tile_n} {ab}->{cd} {act}")
    mmact.mmact_set_gemm_tile_n(0)


@pytest.mark.parametrize("shape", [(200, 136, 72), (384, 256, 1024)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("act", ["relu", "leaky_relu", "tanh", "none", "sigmoid", "gelu"])
def test_split_matches_oracle_and_workspace_holds_z(orc, shape, act):
    M, N, K = shape
    rng = np.random.default_rng(5 + M)
    A = rand_codes(rng, (M, K), "bf16")
    B = rand_codes(rng, (K, N), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    C, ws = run_gemm(A, B, bias, "bf16", "bf16", act, 0.2, split=True)
    check(host(C), orc.gemm(A, B, "bf16", bias, act, 0.2), "bf16", f"split {act}")
    check(host(ws).reshape(M, N), orc.gemm(A, B, "bf16", bias, "none"), "f32", "workspace z")


def test_no_bias_means_zero_bias(orc):
    rng = np.random.default_rng(3)
    A = rand_codes(rng, (130, 64), "f16")
    B = rand_codes(rng, (64, 80), "f16")
    C, _ = run_gemm(A, B, None, "f16", "f32", "leaky_relu", 0.01)
    check(host(C), orc.gemm(A, B, "f16", None, "leaky_relu", 0.01), "f32", "no bias")


def test_empty_contraction_gives_act_of_bias(orc):
    # K == 0: every output is act(bias[j])
    rng = np.random.default_rng(4)
    bias = rng.uniform(-2, 2, 24).astype(np.float32)
    A = np.zeros((5, 0), dtype=np.uint16)
    B = np.zeros((0, 24), dtype=np.uint16)
    for act in ("relu", "leaky_relu", "tanh", "sigmoid", "gelu"):
        dA = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
        dB = torch.empty((0, 24), dtype=torch.bfloat16, device="cuda")
        C = torch.full((5, 24), float("nan"), dtype=torch.float32, device="cuda")
        mmact.mmact_gemm(dA, dB, fp32_to_device(bias), C, act, 0.3)
        assert mmact.mmact_get_last_error() == mmact.MMACT_OK
        check(host(C), orc.gemm(A, B, "bf16", bias, act, 0.3), "f32", f"K=0 {act}")


def test_empty_output_is_a_no_op():
    dA = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    dB = torch.zeros((64, 32), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((0, 32), dtype=torch.bfloat16, device="cuda")
    mmact.mmact_gemm(dA, dB, None, C, "relu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK


def test_extreme_preactivation_saturates_tanh(orc):
    # large |z|: tanh must be +-1, not NaN (the ratio-of-exponentials form is overflow-safe)
    M, N, K = 128, 64, 256
    A = synth.to_codes(np.full((M, K), 8.0), "bf16")
    B = synth.to_codes(np.where(np.arange(N)[None, :] % 2 == 0, 1.0, -1.0) * np.ones((K, N)), "bf16")
    C, _ = run_gemm(A, B, None, "bf16", "f32", "tanh", 0.0)
    got = host(C)
    assert np.all(np.isfinite(got))
    check(got, orc.gemm(A, B, "bf16", None, "tanh"), "f32", "tanh saturation")
    assert np.all(np.abs(got) == 1.0)


def test_identity_B_returns_act_of_A_plus_bias(orc):
    rng = np.random.default_rng(9)
    M, K = 256, 128
    A = rand_codes(rng, (M, K), "bf16", -4, 4)
    B = synth.to_codes(np.eye(K), "bf16")
    bias = rng.uniform(-1, 1, K).astype(np.float32)
    C, _ = run_gemm(A, B, bias, "bf16", "f32", "none", 0.0)
    # exact: one product per element, fp32 accumulate of bf16 values plus an fp32 bias
    Ad = orc.decode(A, "bf16")
    exp = (Ad.astype(np.float32) + bias[None, :]).astype(np.float64)
    assert np.array_equal(host(C), exp)


GEMM_WORKLOADS = [w for w in synth.WORKLOADS.values() if w.kind == "gemm"]


_REF = {}


def workload_points(wl):
    """Output elements compared for a GEMM workload: all of them, except for the 8192^3 one
    (5.5e11 fp64 MACs), where every element of 512 seeded random rows and of 512 seeded
    random columns is compared (8.4 million elements)."""
    M, N = wl.M, wl.N
    if M * N * wl.K <= 2 ** 37:
        return None
    rng = np.random.default_rng(wl.seed)
    rows = rng.choice(M, 512, replace=False)
    cols = rng.choice(N, 512, replace=False)
    pts = np.concatenate([(rows[:, None] * N + np.arange(N)[None, :]).ravel(),
                          (np.arange(M)[:, None] * N + cols[None, :]).ravel()])
    return np.unique(pts.astype(np.int64))


@pytest.mark.parametrize("wl", GEMM_WORKLOADS, ids=lambda w: w.name)
@pytest.mark.parametrize("split", [False, True], ids=["fused", "split"])
def test_workload_parity(orc, wl, split):
    inp = wl.inputs()
    C, _ = run_gemm(inp["A"], inp["B"], inp["bias"], wl.ab_dtype, wl.c_dtype, wl.act, wl.alpha,
                    split=split)
    got = host(C).ravel()
    pts = workload_points(wl)
    if wl.name not in _REF:       # the oracle's values, shared by the fused and split runs
        _REF[wl.name] = orc.gemm(inp["A"], inp["B"], wl.ab_dtype, inp["bias"], wl.act, wl.alpha,
                                 points=pts).ravel()
    check(got if pts is None else got[pts], _REF[wl.name], wl.c_dtype, wl.name)
