"""GPU checks of the run-time fused/split decision (mmact_gemm_auto,
mmact_conv2d_auto) against the oracle and against the clock.

For a shape on each side of the rule the test (1) checks which path ran --
the two-kernel path leaves z = conv/GEMM + bias in the caller's workspace, the
fused path leaves the workspace untouched -- (2) compares the output with the
oracle, and (3) times both paths as CUDA-graph replays and requires the
chosen one not to be slower than the other by more than 10 %.
"""
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


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def graph_ms(fn, reps=20):
    """Per-call milliseconds of fn() replayed as a CUDA graph of `reps` calls (median of 5 replays)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for _ in range(reps):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    times = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / reps)
    return float(np.median(times))


GEMM_CASES = [
    # (M, N, K, act, expected choice)
    (64, 64, 64, "gelu", "split"),
    (256, 256, 512, "gelu", "split"),
    (4096, 4096, 64, "gelu", "fused"),
    (1024, 1024, 512, "relu", "fused"),
    (256, 256, 64, "tanh", "fused"),
]


@pytest.mark.parametrize("case", GEMM_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}")
def test_gemm_auto(orc, case):
    M, N, K, act, want = case
    assert mmact.mmact_gemm_auto_choice(M, N, K, torch.bfloat16, torch.bfloat16, act) == want
    rng = np.random.default_rng(M + K)
    a = synth.to_codes(rng.uniform(-1, 1, (M, K)), "bf16")
    b = synth.to_codes(rng.uniform(-1, 1, (K, N)), "bf16")
    bias = rng.uniform(-1, 1, N).astype(np.float32)
    A, B, db = to_device(a, "bf16"), to_device(b, "bf16"), fp32_to_device(bias)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.full((M * N,), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_gemm_auto(A, B, db, C, act, 0.0, workspace=ws)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    pts = None if M * N <= 1 << 20 else np.random.default_rng(3).integers(0, M * N, 20000)
    ref = orc.gemm(a, b, "bf16", bias, act, points=pts)
    got = host(C).ravel()
    check(got if pts is None else got[pts], ref, "bf16", f"auto {case}")
    wsh = host(ws)
    if want == "split":
        z = orc.gemm(a, b, "bf16", bias, "none", points=pts)
        check(wsh if pts is None else wsh[pts], z, "f32", "auto split workspace")
    else:
        assert np.all(np.isnan(wsh)), "the fused path must not touch the workspace"
    fused = graph_ms(lambda: mmact.mmact_gemm(A, B, db, C, act))
    split = graph_ms(lambda: mmact.mmact_gemm_split(A, B, db, C, ws, act))
    chosen, other = (split, fused) if want == "split" else (fused, split)
    assert chosen <= 1.1 * other, f"{case}: chosen {want} {chosen * 1e3:.2f} us, other {other * 1e3:.2f} us"


CONV_CASES = [
    # (N, C, H, W, Co, k, stride, pad, act, out, expected choice)
    (8, 64, 28, 28, 128, 1, 2, 0, "relu", "f16", "split"),     # 14 x 14 output: 392-byte rows
    (8, 16, 56, 56, 64, 3, 1, 1, "gelu", "f16", "split"),
    (8, 64, 56, 56, 128, 3, 1, 1, "tanh", "f16", "fused"),
]


@pytest.mark.parametrize("case", CONV_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}k{c[5]}s{c[6]}-{c[8]}")
def test_conv_auto(orc, case):
    Nb, C, H, W, Co, k, st, pd, act, od, want = case
    stride, pads, dil = (st, st), (pd,) * 4, (1, 1)
    tod = {"f16": torch.float16, "f32": torch.float32}[od]
    assert mmact.mmact_conv2d_auto_choice(Nb, C, H, W, Co, k, k, stride, pads, dil, torch.float16, tod, act) == want
    rng = np.random.default_rng(C + Co + k)
    x = synth.to_codes(rng.normal(0, 1, (Nb, C, H, W)), "f16")
    w = synth.to_codes(rng.normal(0, (1.0 / (C * k * k)) ** 0.5, (Co, C, k, k)), "f16")
    bias = rng.uniform(-0.1, 0.1, Co).astype(np.float32)
    dx, dw, db = to_device(x, "f16"), to_device(w, "f16"), fp32_to_device(bias)
    Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, k, k, stride, pads, dil)
    y = torch.full((Nb, Co, Ho, Wo), float("nan"), dtype=tod, device="cuda")
    ws = torch.full((y.numel(),), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_conv2d_auto(dx, dw, db, y, stride, pads, dil, act, 0.0, workspace=ws)
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(y), orc.conv2d(x, w, "f16", bias, stride, pads, dil, act), od, f"auto {case}")
    if want == "split":
        check(host(ws), orc.conv2d(x, w, "f16", bias, stride, pads, dil, "none").ravel(), "f32",
              "auto split workspace")
    else:
        assert np.all(np.isnan(host(ws)))
    fused = graph_ms(lambda: mmact.mmact_conv2d(dx, dw, db, y, stride, pads, dil, act))
    split = graph_ms(lambda: mmact.mmact_conv2d_split(dx, dw, db, y, ws, stride, pads, dil, act))
    chosen, other = (split, fused) if want == "split" else (fused, split)
    assert chosen <= 1.1 * other, f"{case}: chosen {want} {chosen * 1e3:.2f} us, other {other * 1e3:.2f} us"


def test_auto_without_workspace_runs_fused(orc):
    M = N = K = 64
    rng = np.random.default_rng(9)
    a = synth.to_codes(rng.uniform(-1, 1, (M, K)), "bf16")
    b = synth.to_codes(rng.uniform(-1, 1, (K, N)), "bf16")
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    mmact.mmact_gemm_auto(to_device(a, "bf16"), to_device(b, "bf16"), None, C, "gelu")
    assert mmact.mmact_get_last_error() == mmact.MMACT_OK
    check(host(C), orc.gemm(a, b, "bf16", None, "gelu"), "f32", "auto, no workspace")
