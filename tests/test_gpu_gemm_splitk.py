"""GPU parity: the split-K cluster GEMM kernel against the oracle.

For GEMMs with few output tiles each 128 x 256 tile is computed by a cluster
of 2 or 4 CTAs, each over its share of the K blocks, and the fp32 partial
tiles are summed across the cluster before the bias + activation epilogue.
The mode switch forces the kernel onto small shapes that span several tiles,
ragged M / N / K tails, K-block counts not divisible by the split factor
(down to one block per CTA), every output dtype and every activation, with
and without a residual (also in place); the skinny full-size workload is
checked through the automatic choice.
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
    yield
    mmact.mmact_set_gemm_split_k(0)
    mmact.mmact_set_gemm_tile_n(0)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def rand_codes(rng, shape, dtype, lo=-1.0, hi=1.0):
    return synth.to_codes(rng.uniform(lo, hi, size=shape), dtype)


def run(A, B, bias, ab, cd, act, alpha, split=False):
    M, K = A.shape
    N = B.shape[1]
    dA, dB = to_device(A, ab), to_device(B, ab)
    C = torch.full((M, N), float("nan"), dtype=TORCH[cd], device="cuda")
    ws = None
    if split:
        ws = torch.full((M * N,), float("nan"), dtype=torch.float32, device="cuda")
        mmact.mmact_gemm_split(dA, dB, fp32_to_device(bias), C, ws, act, alpha)
    else:
        mmact.mmact_gemm(dA, dB, fp32_to_device(bias), C, act, alpha)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    return C, ws


SHAPES = [  # (M, N, K)
    (128, 256, 512),     # one tile, 8 K blocks
    (1, 8, 512),         # one row, one 8-column group
    (200, 392, 1000),    # ragged M, N (second tile partial) and K (16 blocks, last partial)
    (384, 1024, 2048),   # 3 x 4 tiles
    (130, 520, 576),     # 9 K blocks: uneven shares
    (64, 264, 256),      # 4 K blocks: one per CTA when S = 4
]

COMBOS = [("bf16", "bf16", "leaky_relu", 0.2), ("f16", "f32", "relu", 0.0),
          ("bf16", "f16", "tanh", 0.0), ("f16", "bf16", "none", 0.0),
          ("bf16", "f32", "sigmoid", 0.0), ("f16", "bf16", "gelu", 0.0)]


@pytest.mark.parametrize("S", [2, 4])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_forced_split_k_matches_oracle(orc, S, shape):
    M, N, K = shape
    mmact.mmact_set_gemm_split_k(S)
    try:
        assert mmact.mmact_gemm_split_k_choice(M, N, K) == S
        rng = np.random.default_rng(M * 11 + N * 3 + K + S)
        for ab, cd, act, alpha in COMBOS:
            A = rand_codes(rng, (M, K), ab)
            B = rand_codes(rng, (K, N), ab)
            bias = rng.uniform(-1, 1, N).astype(np.float32)
            C, _ = run(A, B, bias, ab, cd, act, alpha)
            check(host(C), orc.gemm(A, B, ab, bias, act, alpha), cd, f"{shape} S={S} {ab}->{cd} {act}")
    finally:
        mmact.mmact_set_gemm_split_k(0)


@pytest.mark.parametrize("S", [2, 4])
def test_forced_split_k_without_bias_and_two_kernel_path(orc, S):
    rng = np.random.default_rng(40 + S)
    M, N, K = 256, 512, 1024
    A = rand_codes(rng, (M, K), "bf16")
    B = rand_codes(rng, (K, N), "bf16")
    mmact.mmact_set_gemm_split_k(S)
    try:
        C, _ = run(A, B, None, "bf16", "f32", "leaky_relu", 0.1)
        check(host(C), orc.gemm(A, B, "bf16", None, "leaky_relu", 0.1), "f32", f"S={S} no bias")
        bias = rng.uniform(-1, 1, N).astype(np.float32)
        C, ws = run(A, B, bias, "bf16", "bf16", "tanh", 0.0, split=True)
        check(host(C), orc.gemm(A, B, "bf16", bias, "tanh"), "bf16", f"S={S} two-kernel")
        check(host(ws).reshape(M, N), orc.gemm(A, B, "bf16", bias, "none"), "f32", f"S={S} workspace z")
    finally:
        mmact.mmact_set_gemm_split_k(0)


def test_cancellation_across_cluster_partials(orc):
    # the two halves of K (one per CTA of the pair) contribute +x and -x, so
    # the exact result is the bias alone; a partial tile dropped or added
    # twice leaves an error of the order of |x| (several units here)
    M, N, K = 128, 256, 1024
    rng = np.random.default_rng(77)
    half = rand_codes(rng, (M, K // 2), "bf16")
    A = np.concatenate([half, half], axis=1)
    Bh = rand_codes(rng, (K // 2, N), "bf16")
    B = np.concatenate([Bh, Bh ^ np.uint16(0x8000)], axis=0)   # the second half negated
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    mmact.mmact_set_gemm_split_k(2)
    try:
        C, _ = run(A, B, bias, "bf16", "f32", "none", 0.0)
    finally:
        mmact.mmact_set_gemm_split_k(0)
    ref = orc.gemm(A, B, "bf16", bias, "none")
    assert np.array_equal(ref, np.broadcast_to(bias.astype(np.float64), (M, N)))
    check(host(C), ref, "f32", "cancellation")


@pytest.mark.parametrize("S", [2, 4])
@pytest.mark.parametrize("cd", ["bf16", "f32"])
def test_forced_split_k_residual(orc, S, cd):
    # C = act(A @ B + bias + R), R in the output dtype; ragged M and N
    rng = np.random.default_rng(50 + S + len(cd))
    M, N, K = 200, 392, 1024
    A = rand_codes(rng, (M, K), "bf16")
    B = rand_codes(rng, (K, N), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    R = rand_codes(rng, (M, N), cd) if cd != "f32" else rng.uniform(-1, 1, (M, N)).astype(np.float32)
    mmact.mmact_set_gemm_split_k(S)
    try:
        assert mmact.mmact_gemm_split_k_choice(M, N, K) == S
        C = torch.full((M, N), float("nan"), dtype=TORCH[cd], device="cuda")
        mmact.mmact_gemm_residual(to_device(A, "bf16"), to_device(B, "bf16"), fp32_to_device(bias),
                                  fp32_to_device(R) if cd == "f32" else to_device(R, cd), C, "relu", 0.0)
        assert mmact.mmact_get_last_error() == mmact.MMACT_OK
        check(host(C), orc.gemm(A, B, "bf16", bias, "relu", 0.0, residual=R, res_dtype=cd), cd,
              f"S={S} residual {cd}")
    finally:
        mmact.mmact_set_gemm_split_k(0)


@pytest.mark.parametrize("S", [2, 4])
def test_forced_split_k_residual_in_place(orc, S):
    # R is C itself: every element is read before its own unit's store writes it
    rng = np.random.default_rng(60 + S)
    M, N, K = 256, 512, 512
    A = rand_codes(rng, (M, K), "bf16")
    B = rand_codes(rng, (K, N), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    R = rand_codes(rng, (M, N), "bf16")
    mmact.mmact_set_gemm_split_k(S)
    try:
        C = to_device(R, "bf16").clone()
        mmact.mmact_gemm_residual(to_device(A, "bf16"), to_device(B, "bf16"), fp32_to_device(bias), C, C,
                                  "gelu", 0.0)
        assert mmact.mmact_get_last_error() == mmact.MMACT_OK
        check(host(C), orc.gemm(A, B, "bf16", bias, "gelu", residual=R, res_dtype="bf16"), "bf16",
              f"S={S} in place")
    finally:
        mmact.mmact_set_gemm_split_k(0)


def test_mode_switch_rejects_other_factors():
    for bad in (-1, 3, 5, 8):
        with pytest.raises(Exception):
            mmact.mmact_set_gemm_split_k(bad)
    mmact.mmact_set_gemm_split_k(1)
    try:
        assert mmact.mmact_gemm_split_k_choice(128, 8192, 8192) == 0
    finally:
        mmact.mmact_set_gemm_split_k(0)


def test_automatic_choice_takes_split_k_only_for_few_tiles():
    assert mmact.mmact_gemm_split_k_choice(8192, 8192, 8192) == 0
    assert mmact.mmact_gemm_split_k_choice(1024, 640, 256) == 0      # 4 K blocks: too few
    assert mmact.mmact_gemm_split_k_choice(128, 8192, 8192) in (2, 4)
    assert mmact.mmact_gemm_split_k_choice(128, 16384, 4096) == 0    # 64 tiles, 32 K blocks per CTA at S=2
    assert mmact.mmact_gemm_split_k_choice(128, 8192, 1024) == 0     # 16 K blocks: too few
    mmact.mmact_set_gemm_tile_n(128)
    try:
        assert mmact.mmact_gemm_split_k_choice(128, 8192, 8192) == 0  # a fixed tile width
    finally:
        mmact.mmact_set_gemm_tile_n(0)


def test_skinny_workload_through_automatic_choice(orc):
    wl = synth.WORKLOADS["gemm_leakyrelu_128x8192x8192_bf16"]
    assert mmact.mmact_gemm_split_k_choice(wl.M, wl.N, wl.K) != 0
    inp = wl.inputs()
    C, _ = run(inp["A"], inp["B"], inp["bias"], wl.ab_dtype, wl.c_dtype, wl.act, wl.alpha)
    got = host(C).ravel()
    pts = sample_points(wl.M * wl.N, wl.M, wl.N, 6000, seed=wl.seed + 1)
    ref = orc.gemm(inp["A"], inp["B"], wl.ab_dtype, inp["bias"], wl.act, wl.alpha, points=pts)
    check(got[pts], ref, wl.c_dtype, wl.name)
