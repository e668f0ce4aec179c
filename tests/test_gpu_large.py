"""GPU parity at sizes whose outputs exceed 2^31 elements (64-bit indexing):
a GEMM with a 65536 x 65536 output and a conv with 3.3e9 output elements, in
both layouts.  Seeded samples are gathered on the device and compared with the
oracle element by element."""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_epilogue_gb300 import build, mmact, synth
from parity import check, fp32_to_device, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    mmact.load()
    yield
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def sampled(y: torch.Tensor, pts: np.ndarray) -> np.ndarray:
    idx = torch.from_numpy(pts).cuda()
    return y.reshape(-1)[idx].float().cpu().numpy().astype(np.float64)


def test_gemm_output_beyond_2_31_elements(orc):
    M = N = 65536
    K = 64
    rng = np.random.default_rng(61)
    A = synth.to_codes(rng.uniform(-1, 1, (M, K)), "bf16")
    B = synth.to_codes(rng.uniform(-1, 1, (K, N)), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mmact.mmact_gemm(to_device(A, "bf16"), to_device(B, "bf16"), fp32_to_device(bias), C, "relu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    pts = np.concatenate([rng.integers(0, M * N, 3000, dtype=np.int64),
                          np.array([M * N - 1, (M - 1) * N, 2 ** 31, 2 ** 31 - 1, 2 ** 32 - N], dtype=np.int64)])
    ref = orc.gemm(A, B, "bf16", bias, "relu", points=pts)
    check(sampled(C, pts), ref, "bf16", "65536^2 x 64")
    del C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layout", ["nchw", "nchw_window", "nhwc"])
def test_conv_output_beyond_2_31_elements(orc, layout):
    Nb, C, H, W, Co = 8192, 64, 56, 56, 128
    rng = np.random.default_rng(62)
    # 64 distinct seeded images, repeated 128 times (host codes for the oracle, device copy expanded on the GPU)
    base = synth.to_codes(rng.normal(0, 1, (64, C, H, W)), "f16")
    x = np.tile(base, (Nb // 64, 1, 1, 1))
    w = synth.to_codes(rng.normal(0, (1.0 / 576) ** 0.5, (Co, C, 3, 3)), "f16")
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    st, pd, dl = (1, 1), (1, 1, 1, 1), (1, 1)
    total = Nb * Co * H * W
    pts = np.concatenate([rng.integers(0, total, 3000, dtype=np.int64),
                          np.array([total - 1, 2 ** 31, 2 ** 31 - 1, 3 * 2 ** 30], dtype=np.int64)])
    if layout.startswith("nchw"):
        # the tensor-memory im2col kernel by default; the window producer when it is turned off
        mmact.mmact_set_conv_tmem(1 if layout == "nchw_window" else 0)
        try:
            assert mmact.mmact_conv2d_producer(Nb, C, H, W, Co, 3, 3, st, pd, dl, torch.float16,
                                               torch.float16) == ("window" if layout == "nchw_window" else "tmem")
            y = torch.empty((Nb, Co, H, W), dtype=torch.float16, device="cuda")
            xd = to_device(base, "f16").repeat(Nb // 64, 1, 1, 1)
            mmact.mmact_conv2d(xd, to_device(w, "f16"), fp32_to_device(bias), y, st, pd, dl, "tanh")
            del xd
        finally:
            mmact.mmact_set_conv_tmem(0)
        got = sampled(y, pts)
    else:
        xd = to_device(base, "f16").permute(0, 2, 3, 1).contiguous().repeat(Nb // 64, 1, 1, 1)
        wd = to_device(w, "f16").permute(0, 2, 3, 1).contiguous()
        y = torch.empty((Nb, H, W, Co), dtype=torch.float16, device="cuda")
        mmact.mmact_conv2d_nhwc(xd, wd, fp32_to_device(bias), y, st, pd, dl, "tanh")
        del xd, wd
        # NCHW flat index -> NHWC flat index of the same element
        n, rem = np.divmod(pts, Co * H * W)
        co, rem = np.divmod(rem, H * W)
        oh, ow = np.divmod(rem, W)
        got = sampled(y, ((n * H + oh) * W + ow) * Co + co)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    ref = orc.conv2d(x, w, "f16", bias, st, pd, dl, "tanh", points=pts)
    check(got, ref, "f16", f"conv 8192x64x56x56 {layout}")
    del y
    torch.cuda.empty_cache()
