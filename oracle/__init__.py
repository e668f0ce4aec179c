"""Plain CPU oracle for C = act(A x B + bias) and y = act(conv2d(x, w, bias)).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference leg of ``bench.py`` may import this package.  The
product library never links, imports or calls it, and it shares no code with
the CUDA path: both sides only consume the same seeded input bytes.

The arithmetic lives in ``mmact_oracle.c`` (plain C, fp64, one output element
at a time from its definition).  This module compiles it with gcc on first use
and marshals numpy arrays through ctypes.  ctypes releases the GIL during the
foreign call, so large requests are split across a thread pool; every element
is still computed independently by the same C routine, so the split changes
no value.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mmact_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

DTYPES = {"f16": 0, "bf16": 1, "f32": 2}
RES_DTYPES = {"f16": 0, "bf16": 1, "f32": 2}
ACTS = {"none": 0, "relu": 1, "leaky_relu": 2, "tanh": 3, "sigmoid": 4, "gelu": 5}

_build_lock = threading.Lock()


def build(source: str = SOURCE, output: str = LIBRARY, defines: tuple = ()) -> str:
    """Compile the oracle into a shared library (plain gcc, no vector flags)."""
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
           *[f"-D{d}" for d in defines], source, "-o", output, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def _needs_build(src: str, lib: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)


class Oracle:
    """ctypes front end over one compiled copy of the oracle."""

    def __init__(self, lib_path: str = LIBRARY, source: str = SOURCE):
        if lib_path == LIBRARY:
            with _build_lock:
                if _needs_build(source, lib_path):
                    build(source, lib_path)
        self.lib = ctypes.CDLL(lib_path)
        L = self.lib
        i64, dbl, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        L.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        L.oracle_decode_f16.restype = dbl
        L.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        L.oracle_decode_bf16.restype = dbl
        L.oracle_tanh.argtypes = [dbl]
        L.oracle_tanh.restype = dbl
        L.oracle_sigmoid.argtypes = [dbl]
        L.oracle_sigmoid.restype = dbl
        L.oracle_gelu.argtypes = [dbl]
        L.oracle_gelu.restype = dbl
        L.oracle_act.argtypes = [dbl, ci, dbl]
        L.oracle_act.restype = dbl
        L.oracle_conv_out_dim.argtypes = [i64] * 6
        L.oracle_conv_out_dim.restype = i64
        L.oracle_gemm.argtypes = [vp, vp, ci, vp, i64, i64, i64, ci, dbl, vp, i64, vp]
        L.oracle_gemm.restype = ci
        L.oracle_conv2d.argtypes = [vp, vp, ci, vp] + [i64] * 15 + [ci, dbl, vp, i64, vp]
        L.oracle_conv2d.restype = ci
        L.oracle_gemm_res.argtypes = [vp, vp, ci, vp, vp, ci, i64, i64, i64, ci, dbl, vp, i64, vp]
        L.oracle_gemm_res.restype = ci
        L.oracle_conv2d_res.argtypes = [vp, vp, ci, vp, vp, ci] + [i64] * 15 + [ci, dbl, vp, i64, vp]
        L.oracle_conv2d_res.restype = ci

    # -- scalar pieces -----------------------------------------------------
    def decode(self, codes, dtype: str) -> np.ndarray:
        fn = self.lib.oracle_decode_bf16 if dtype == "bf16" else self.lib.oracle_decode_f16
        flat = np.asarray(codes, dtype=np.uint16).ravel()
        return np.array([fn(int(c)) for c in flat], dtype=np.float64).reshape(np.shape(codes))

    def act(self, z, act: str, alpha: float = 0.0) -> np.ndarray:
        flat = np.asarray(z, dtype=np.float64).ravel()
        a = ACTS[act]
        return np.array([self.lib.oracle_act(float(v), a, float(alpha)) for v in flat]).reshape(np.shape(z))

    def tanh(self, z: float) -> float:
        return self.lib.oracle_tanh(float(z))

    def conv_out_dim(self, size, k, stride, pad_lo, pad_hi, dil) -> int:
        return int(self.lib.oracle_conv_out_dim(size, k, stride, pad_lo, pad_hi, dil))

    # -- full operators ----------------------------------------------------
    @staticmethod
    def _run_chunks(call, points: np.ndarray, threads: int) -> np.ndarray:
        out = np.empty(points.shape[0], dtype=np.float64)
        if points.shape[0] == 0:
            return out
        threads = max(1, min(threads, points.shape[0]))
        bounds = np.linspace(0, points.shape[0], threads + 1).astype(np.int64)

        def work(k):
            lo, hi = int(bounds[k]), int(bounds[k + 1])
            if hi > lo:
                rc = call(points[lo:hi], out[lo:hi])
                if rc != 0:
                    raise ValueError("oracle rejected its arguments")

        if threads == 1:
            work(0)
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                list(ex.map(work, range(threads)))
        return out

    @staticmethod
    def _residual(residual, res_dtype, count):
        """(pointer, dtype code, keep-alive array) of an optional residual tensor."""
        if residual is None:
            return None, 0, None
        if res_dtype == "f32":
            r = np.ascontiguousarray(residual, dtype=np.float32)
        else:
            r = np.ascontiguousarray(residual, dtype=np.uint16)
        if r.size != count:
            raise ValueError("residual has the wrong number of elements")
        return r.ctypes.data, RES_DTYPES[res_dtype], r

    @staticmethod
    def _inputs(dtype, *arrays):
        """16-bit codes as uint16, fp32 inputs as float32 (C-contiguous)."""
        kind = np.float32 if dtype == "f32" else np.uint16
        return [np.ascontiguousarray(a, dtype=kind) for a in arrays]

    def gemm(self, A, B, dtype: str, bias, act: str, alpha: float = 0.0,
             points=None, threads: int | None = None, residual=None,
             res_dtype: str = "f32") -> np.ndarray:
        """act(A @ B + bias [+ residual]) in fp64 from 16-bit codes.

        A: [M, K]; B: [K, N] -- uint16 codes for dtype f16 / bf16, float32
        values for dtype f32; bias: float32 [N] or None.
        residual: [M, N] uint16 codes (res_dtype f16 / bf16) or float32 values
        (res_dtype f32), or None.
        points: flat indices i*N + j to evaluate (None = every element, returned
        as [M, N]).
        """
        A, B = self._inputs(dtype, A, B)
        M, K = A.shape
        K2, N = B.shape
        if K2 != K:
            raise ValueError("inner dimensions differ")
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        if b is not None and b.shape[0] != N:
            raise ValueError("bias length != N")
        full = points is None
        pts = np.arange(M * N, dtype=np.int64) if full else np.ascontiguousarray(points, dtype=np.int64)
        threads = threads or os.cpu_count() or 1
        bp = None if b is None else b.ctypes.data
        rp, rd, _keep = self._residual(residual, res_dtype, M * N)

        def call(p, o):
            return self.lib.oracle_gemm_res(A.ctypes.data, B.ctypes.data, DTYPES[dtype], bp, rp, rd,
                                            M, N, K, ACTS[act], float(alpha), p.ctypes.data,
                                            p.shape[0], o.ctypes.data)

        out = self._run_chunks(call, pts, threads)
        return out.reshape(M, N) if full else out

    def conv2d(self, x, w, dtype: str, bias, stride, pads, dilation, act: str,
               alpha: float = 0.0, points=None, threads: int | None = None, residual=None,
               res_dtype: str = "f32") -> np.ndarray:
        """act(conv2d(x, w) + bias [+ residual]) in fp64 from 16-bit codes.

        residual: [N, Co, Ho, Wo] in res_dtype (codes or float32 values), or None.

        x: [N, C, H, W]; w: [Co, C, kh, kw] -- codes for f16 / bf16, float32
        values for f32; bias float32 [Co] or None;
        stride = (sh, sw); pads = (top, bottom, left, right); dilation = (dh, dw).
        points: flat indices into y [N, Co, Ho, Wo] (None = all, returned 4-D).
        """
        x, w = self._inputs(dtype, x, w)
        Nb, C, H, W = x.shape
        Co, C2, kh, kw = w.shape
        if C2 != C:
            raise ValueError("channel mismatch")
        sh, sw = stride
        pt, pb, pl, pr = pads
        dh, dw = dilation
        Ho = self.conv_out_dim(H, kh, sh, pt, pb, dh)
        Wo = self.conv_out_dim(W, kw, sw, pl, pr, dw)
        if Ho < 0 or Wo < 0:
            raise ValueError("bad conv geometry")
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        full = points is None
        total = Nb * Co * Ho * Wo
        pts = np.arange(total, dtype=np.int64) if full else np.ascontiguousarray(points, dtype=np.int64)
        threads = threads or os.cpu_count() or 1
        bp = None if b is None else b.ctypes.data
        rp, rd, _keep = self._residual(residual, res_dtype, total)

        def call(p, o):
            return self.lib.oracle_conv2d_res(x.ctypes.data, w.ctypes.data, DTYPES[dtype], bp, rp, rd,
                                              Nb, C, H, W, Co, kh, kw, sh, sw, pt, pb, pl, pr, dh, dw,
                                              ACTS[act], float(alpha), p.ctypes.data, p.shape[0],
                                              o.ctypes.data)

        out = self._run_chunks(call, pts, threads)
        return out.reshape(Nb, Co, Ho, Wo) if full else out


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from the committed source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
