"""Shared helpers for the parity tests: device transfer and the tolerance.

Tolerance (the fused operator's accuracy contract): for fp32 outputs
|gpu - oracle| <= 2e-3 + 2e-3 * |oracle|; for fp16 / bf16 outputs one unit in
the last place of the output dtype at |oracle| is added to that bound.
"""
from __future__ import annotations

import numpy as np
import torch

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
ATOL = 2e-3
RTOL = 2e-3


def to_device(codes: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """16-bit codes (uint16) -> CUDA tensor of that dtype, bit for bit."""
    t = torch.from_numpy(np.ascontiguousarray(codes).view(np.int16))
    return t.view(TORCH[dtype]).to(device)


def fp32_to_device(a, device="cuda"):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def ulp(o: np.ndarray, dtype: str) -> np.ndarray:
    a = np.abs(o)
    if dtype == "f32":
        return np.zeros_like(a)
    mant, min_exp, sub = (10, -14, 2.0 ** -24) if dtype == "f16" else (7, -126, 2.0 ** -133)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    spacing = np.exp2(e - mant)
    return np.where(a < 2.0 ** min_exp, sub, spacing)


def bound(o: np.ndarray, dtype: str) -> np.ndarray:
    return ATOL + RTOL * np.abs(o) + ulp(o, dtype)


# tf32 operands keep 10 fraction bits: each operand is off by < 2^-10 of itself,
# a product by < 2^-9 of itself (to first order), a dot product by < 2^-9 times
# the sum of |products|.  The activations used here change by at most 1.2x
# their argument's change (GELU's slope peaks near 1.13).
TF32_REL = 2.0 ** -9
ACT_SLOPE = 1.2


def check(gpu: np.ndarray, ref: np.ndarray, dtype: str, what: str = "", extra=None) -> float:
    """Assert every element is within the bound (plus `extra`, a per-element
    allowance, when given); returns the worst |err| / bound."""
    gpu = np.asarray(gpu, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    err = np.abs(gpu - ref)
    b = bound(ref, dtype)
    if extra is not None:
        b = b + np.asarray(extra, dtype=np.float64).ravel()
    ratio = err / b
    worst = int(np.argmax(ratio)) if ratio.size else 0
    assert ratio.size == 0 or ratio[worst] <= 1.0, (
        f"{what}: element {worst} gpu={gpu[worst]!r} oracle={ref[worst]!r} "
        f"|err|={err[worst]:.3e} bound={b[worst]:.3e} ({int(np.sum(ratio > 1))} over)")
    return float(ratio.max()) if ratio.size else 0.0


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def sample_points(total: int, rows: int, cols: int, n: int, seed: int) -> np.ndarray:
    """Seeded flat indices: random ones plus the four corners and the last row/column ends."""
    rng = np.random.default_rng(seed)
    pts = rng.integers(0, total, size=n)
    extra = [0, cols - 1, (rows - 1) * cols, total - 1]
    return np.unique(np.concatenate([pts, np.array(extra, dtype=np.int64)]))
