"""GPU checks of the host-side tensor-map cache: a call that repeats an earlier
call's tensors and shapes reuses its encoded maps, and a call whose tensors,
shapes or dtypes differ encodes new ones and still matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_epilogue_gb300 import build, mmact, synth
from parity import check, fp32_to_device, host, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    mmact.load()


def gemm_inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = synth.to_codes(rng.uniform(-1, 1, (M, K)), "bf16")
    b = synth.to_codes(rng.uniform(-1, 1, (K, N)), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    return a, b, bias


def test_repeated_call_reuses_maps_and_new_tensors_encode():
    orc = oracle.get()
    M, N, K = 256, 192, 128
    a, b, bias = gemm_inputs(M, N, K, 1)
    A, B, db = to_device(a, "bf16"), to_device(b, "bf16"), fp32_to_device(bias)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mmact.mmact_gemm(A, B, db, C, "relu")
    h0, e0 = mmact.mmact_tensor_map_cache_stats()
    for _ in range(5):
        mmact.mmact_gemm(A, B, db, C, "relu")
    h1, e1 = mmact.mmact_tensor_map_cache_stats()
    assert e1 == e0, "a repeated call must not encode"
    assert h1 - h0 >= 15, "A, B and C maps are reused on each of the five calls"
    check(host(C), orc.gemm(a, b, "bf16", bias, "relu"), "bf16", "cached maps")

    # a new output tensor: its map is encoded, the others are reused
    C2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mmact.mmact_gemm(A, B, db, C2, "tanh")
    h2, e2 = mmact.mmact_tensor_map_cache_stats()
    assert e2 == e1 + 1 and h2 >= h1 + 2
    check(host(C2), orc.gemm(a, b, "bf16", bias, "tanh"), "f32", "new output map")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK


def test_same_address_other_shape_is_not_confused():
    """Free and reallocate: the caching allocator hands back the same address
    for a tensor of another shape; the key holds the shape, so the result is
    still right."""
    orc = oracle.get()
    K = 128
    for M, N in ((256, 192), (192, 256), (128, 384)):
        a, b, bias = gemm_inputs(M, N, K, M + N)
        A, B, db = to_device(a, "bf16"), to_device(b, "bf16"), fp32_to_device(bias)
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        mmact.mmact_gemm(A, B, db, C, "sigmoid")
        check(host(C), orc.gemm(a, b, "bf16", bias, "sigmoid"), "f16", f"reused address {M}x{N}")
        del A, B, db, C
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK


def test_conv_repeated_call_reuses_maps():
    orc = oracle.get()
    rng = np.random.default_rng(4)
    x = synth.to_codes(rng.normal(0, 1, (2, 64, 16, 16)), "f16")
    w = synth.to_codes(rng.normal(0, 1 / 24, (128, 64, 3, 3)), "f16")
    bias = rng.uniform(-0.1, 0.1, 128).astype(np.float32)
    dx, dw, db = to_device(x, "f16"), to_device(w, "f16"), fp32_to_device(bias)
    y = torch.empty((2, 128, 16, 16), dtype=torch.float16, device="cuda")
    st, pd, dl = (1, 1), (1, 1, 1, 1), (1, 1)
    mmact.mmact_conv2d(dx, dw, db, y, st, pd, dl, "tanh")
    _, e0 = mmact.mmact_tensor_map_cache_stats()
    for _ in range(3):
        mmact.mmact_conv2d(dx, dw, db, y, st, pd, dl, "tanh")
    _, e1 = mmact.mmact_tensor_map_cache_stats()
    assert e1 == e0
    check(host(y), orc.conv2d(x, w, "f16", bias, st, pd, dl, "tanh"), "f16", "conv cached maps")
