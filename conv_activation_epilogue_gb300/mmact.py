"""Thin Python binding over libmmact.so (the C ABI in include/mmact.h).

Argument marshalling only: every function here checks that the torch tensors
it is handed are CUDA, contiguous and of a supported dtype, turns them into
raw device pointers and sizes, calls the C entry point of the same name and
raises MmactError on a non-OK status.  All arithmetic runs in the library's
CUDA kernels; there is no CPU path.  If the library is not built, the first
call raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libmmact.so")

MMACT_OK, MMACT_ERR_INVALID_ARG, MMACT_ERR_UNSUPPORTED, MMACT_ERR_CUDA, MMACT_ERR_TIMEOUT = range(5)
ACT = {"none": 0, "relu": 1, "leaky_relu": 2, "tanh": 3, "sigmoid": 4, "gelu": 5}
DTYPE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}
MMACT_TF32 = 3   # fp32 inputs computed as tf32 (one pass); float32 tensors default to split precision

_lib = None

# Exported C symbols, as declared in include/mmact.h.
SYMBOLS = [
    "mmact_gemm", "mmact_gemm_residual", "mmact_gemm_split", "mmact_gemm_split_noalloc", "mmact_conv2d",
    "mmact_conv2d_split", "mmact_conv2d_residual", "mmact_conv2d_nhwc_residual",
    "mmact_conv2d_nhwc",
    "mmact_conv2d_out_shape", "mmact_conv2d_producer", "mmact_get_last_error",
    "mmact_set_wait_timeout_ns",
    "mmact_selftest_wait_timeout", "mmact_set_gemm_tile_n", "mmact_set_gemm_split_k",
    "mmact_gemm_split_k_choice", "mmact_set_gemm_pair", "mmact_gemm_kernel_choice", "mmact_set_conv_tmem",
    "mmact_gemm_auto", "mmact_gemm_auto_choice", "mmact_conv2d_auto", "mmact_conv2d_auto_choice",
    "mmact_set_gemm_l2_policy", "mmact_tensor_map_cache_stats", "mmact_status_string", "mmact_version",
]


class MmactError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load(path: str = LIBRARY) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libmmact.so not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    L = ctypes.CDLL(path)
    vp, i64, i32, f32, u64, ci = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                  ctypes.c_uint64, ctypes.c_int)
    p_i32 = ctypes.POINTER(i32)
    L.mmact_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, f32, vp]
    L.mmact_gemm_residual.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, f32, vp]
    L.mmact_gemm_residual.restype = ci
    L.mmact_gemm_split.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, f32, vp, vp]
    L.mmact_gemm_split_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, f32, vp]
    L.mmact_gemm_split_noalloc.restype = ci
    conv = [vp, vp, vp, vp] + [i64] * 7 + [p_i32, p_i32, p_i32, ci, ci, ci, f32]
    L.mmact_conv2d.argtypes = conv + [vp]
    L.mmact_conv2d_split.argtypes = conv + [vp, vp]
    L.mmact_conv2d_auto.argtypes = conv + [vp, vp]
    L.mmact_conv2d_auto.restype = ci
    L.mmact_conv2d_auto_choice.argtypes = [i64] * 7 + [p_i32, p_i32, p_i32, ci, ci, ci, ctypes.POINTER(ci)]
    L.mmact_conv2d_auto_choice.restype = ci
    L.mmact_gemm_auto.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, f32, vp, vp]
    L.mmact_gemm_auto.restype = ci
    L.mmact_gemm_auto_choice.argtypes = [i64, i64, i64, ci, ci, ci, ctypes.POINTER(ci)]
    L.mmact_gemm_auto_choice.restype = ci
    L.mmact_conv2d_nhwc.argtypes = conv + [vp]
    L.mmact_conv2d_nhwc.restype = ci
    conv_res = [vp, vp, vp, vp, vp] + [i64] * 7 + [p_i32, p_i32, p_i32, ci, ci, ci, f32, vp]
    L.mmact_conv2d_residual.argtypes = conv_res
    L.mmact_conv2d_residual.restype = ci
    L.mmact_conv2d_nhwc_residual.argtypes = conv_res
    L.mmact_conv2d_nhwc_residual.restype = ci
    L.mmact_conv2d_out_shape.argtypes = [i64, i64, i64, i64, p_i32, p_i32, p_i32,
                                         ctypes.POINTER(i64), ctypes.POINTER(i64)]
    L.mmact_conv2d_producer.argtypes = [i64] * 7 + [p_i32, p_i32, p_i32, ci, ci]
    L.mmact_conv2d_producer.restype = ci
    L.mmact_get_last_error.argtypes = [vp]
    L.mmact_set_wait_timeout_ns.argtypes = [u64]
    L.mmact_set_wait_timeout_ns.restype = None
    L.mmact_selftest_wait_timeout.argtypes = [u64, vp]
    L.mmact_set_gemm_tile_n.argtypes = [ci]
    L.mmact_set_gemm_split_k.argtypes = [ci]
    L.mmact_set_gemm_pair.argtypes = [ci]
    L.mmact_set_conv_tmem.argtypes = [ci]
    L.mmact_set_gemm_l2_policy.argtypes = [ci]
    L.mmact_set_gemm_l2_policy.restype = ci
    L.mmact_gemm_kernel_choice.argtypes = [i64, i64, i64, ci, ctypes.POINTER(ci)]
    L.mmact_gemm_split_k_choice.argtypes = [i64, i64, i64, ctypes.POINTER(ci)]
    L.mmact_tensor_map_cache_stats.argtypes = [ctypes.POINTER(u64), ctypes.POINTER(u64)]
    L.mmact_tensor_map_cache_stats.restype = ci
    L.mmact_status_string.argtypes = [ci]
    L.mmact_status_string.restype = ctypes.c_char_p
    L.mmact_version.argtypes = []
    for name in ("mmact_gemm", "mmact_gemm_split", "mmact_conv2d", "mmact_conv2d_split",
                 "mmact_conv2d_out_shape", "mmact_get_last_error", "mmact_selftest_wait_timeout",
                 "mmact_set_gemm_tile_n", "mmact_set_gemm_split_k", "mmact_gemm_split_k_choice",
                 "mmact_set_gemm_pair", "mmact_gemm_kernel_choice", "mmact_set_conv_tmem",
                 "mmact_version"):
        getattr(L, name).restype = ci
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().mmact_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MMACT_OK:
        raise MmactError(status, where)


# the current stream's raw handle without building a torch.cuda.Stream object
# (a few microseconds per call on small launches); torch's public route otherwise
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_CUR_DEVICE = getattr(torch._C, "_cuda_getDevice", None)


def _stream_handle(stream) -> int | None:
    if stream is None:
        if _RAW_STREAM is not None and _CUR_DEVICE is not None:
            return _RAW_STREAM(_CUR_DEVICE()) or None
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _dev(t: torch.Tensor, name: str, dtypes) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} dtype {t.dtype} not in {dtypes}")
    return t.data_ptr()


_IN = (torch.float16, torch.bfloat16, torch.float32)   # float32 inputs: split precision
_OUT = (torch.float16, torch.bfloat16, torch.float32)


def _bias_ptr(bias, n: int):
    if bias is None:
        return None
    _dev(bias, "bias", (torch.float32,))
    if bias.numel() != n:
        raise ValueError(f"bias must have {n} elements")
    return bias.data_ptr()


def _gemm_args(A, B, bias, C):
    pa = _dev(A, "A", _IN)
    pb = _dev(B, "B", _IN)
    pc = _dev(C, "C", _OUT)
    if A.dim() != 2 or B.dim() != 2 or C.dim() != 2:
        raise ValueError("A, B, C must be 2-D")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N) or B.dtype != A.dtype:
        raise ValueError("shape/dtype mismatch: A [M,K], B [K,N], C [M,N], A and B same dtype")
    return pa, pb, _bias_ptr(bias, N), pc, M, N, K


def mmact_gemm(A, B, bias, C, act: str = "none", alpha: float = 0.0, stream=None) -> None:
    """C = act(A @ B + bias) in one fused kernel (see include/mmact.h)."""
    L = load()
    pa, pb, pbias, pc, M, N, K = _gemm_args(A, B, bias, C)
    _check(L.mmact_gemm(pa, pb, pbias, pc, M, N, K, DTYPE[A.dtype], DTYPE[C.dtype], ACT[act],
                        float(alpha), _stream_handle(stream)), "mmact_gemm")


def mmact_gemm_residual(A, B, bias, R, C, act: str = "none", alpha: float = 0.0, stream=None) -> None:
    """C = act(A @ B + bias + R) in one fused kernel; R [M,N] has C's dtype and
    may be C itself (see include/mmact.h)."""
    L = load()
    pa, pb, pbias, pc, M, N, K = _gemm_args(A, B, bias, C)
    pr = _dev(R, "R", _OUT)
    if tuple(R.shape) != (M, N) or R.dtype != C.dtype:
        raise ValueError("R must be [M,N] with C's dtype")
    _check(L.mmact_gemm_residual(pa, pb, pbias, pr, pc, M, N, K, DTYPE[A.dtype], DTYPE[C.dtype],
                                 ACT[act], float(alpha), _stream_handle(stream)), "mmact_gemm_residual")


def mmact_gemm_split(A, B, bias, C, workspace, act: str = "none", alpha: float = 0.0,
                     stream=None) -> None:
    """Two-kernel ablation: workspace (fp32 [M,N]) = A @ B + bias, then C = act(workspace)."""
    L = load()
    pa, pb, pbias, pc, M, N, K = _gemm_args(A, B, bias, C)
    pw = _dev(workspace, "workspace", (torch.float32,))
    if workspace.numel() < M * N:
        raise ValueError("workspace must hold M*N fp32 elements")
    _check(L.mmact_gemm_split(pa, pb, pbias, pc, M, N, K, DTYPE[A.dtype], DTYPE[C.dtype], ACT[act],
                              float(alpha), pw, _stream_handle(stream)), "mmact_gemm_split")


def mmact_gemm_auto(A, B, bias, C, act: str = "none", alpha: float = 0.0, workspace=None, stream=None) -> None:
    """Fused or two-kernel GEMM, decided per shape (see include/mmact.h); the split path
    needs `workspace` (fp32, at least M*N elements) and is never taken without one."""
    L = load()
    pa, pb, pbias, pc, M, N, K = _gemm_args(A, B, bias, C)
    pw = None
    if workspace is not None:
        pw = _dev(workspace, "workspace", (torch.float32,))
        if workspace.numel() < M * N:
            raise ValueError("workspace must hold M*N fp32 elements")
    _check(L.mmact_gemm_auto(pa, pb, pbias, pc, M, N, K, DTYPE[A.dtype], DTYPE[C.dtype], ACT[act],
                             float(alpha), pw, _stream_handle(stream)), "mmact_gemm_auto")


def mmact_gemm_auto_choice(M, N, K, ab_dtype, c_dtype, act: str) -> str:
    """"split" or "fused": the path mmact_gemm_auto takes with a workspace (dtypes: torch dtypes)."""
    out = ctypes.c_int(-1)
    _check(load().mmact_gemm_auto_choice(int(M), int(N), int(K), DTYPE[ab_dtype], DTYPE[c_dtype], ACT[act],
                                         ctypes.byref(out)), "mmact_gemm_auto_choice")
    return "split" if out.value == 1 else "fused"


NOALLOC_MAX_ELEMENTS = 4194304   # MMACT_NOALLOC_MAX_ELEMENTS in include/mmact.h


def mmact_gemm_split_noalloc(A, B, bias, C, act: str = "none", alpha: float = 0.0,
                             stream=None) -> None:
    """mmact_gemm_split using the library's built-in scratch array instead of a
    caller-provided workspace (for callers that cannot allocate; M*N is limited)."""
    L = load()
    pa, pb, pbias, pc, M, N, K = _gemm_args(A, B, bias, C)
    _check(L.mmact_gemm_split_noalloc(pa, pb, pbias, pc, M, N, K, DTYPE[A.dtype], DTYPE[C.dtype],
                                      ACT[act], float(alpha), _stream_handle(stream)),
           "mmact_gemm_split_noalloc")


# ctypes int32 arrays for strides / pads / dilations, kept per value tuple: a call
# site that repeats its geometry reuses them (the library only reads them during
# the call)
_I32_ARRAYS: dict = {}


def _i32(vals, n):
    vals = tuple(int(v) for v in vals)
    if len(vals) != n:
        raise ValueError(f"expected {n} values")
    arr = _I32_ARRAYS.get(vals)
    if arr is None:
        if len(_I32_ARRAYS) > 1024:
            _I32_ARRAYS.clear()
        arr = _I32_ARRAYS[vals] = (ctypes.c_int32 * n)(*vals)
    return arr


_OUT_SHAPES: dict = {}


def mmact_conv2d_out_shape(H, W, kh, kw, stride, pads, dilation) -> tuple:
    """(Ho, Wo) from the library's output-size rule (answers kept per geometry)."""
    key = (int(H), int(W), int(kh), int(kw), tuple(stride), tuple(pads), tuple(dilation))
    hit = _OUT_SHAPES.get(key)
    if hit is not None:
        return hit
    L = load()
    ho, wo = ctypes.c_int64(), ctypes.c_int64()
    _check(L.mmact_conv2d_out_shape(H, W, kh, kw, _i32(stride, 2), _i32(pads, 4),
                                    _i32(dilation, 2), ctypes.byref(ho), ctypes.byref(wo)),
           "mmact_conv2d_out_shape")
    if len(_OUT_SHAPES) > 1024:
        _OUT_SHAPES.clear()
    _OUT_SHAPES[key] = (ho.value, wo.value)
    return ho.value, wo.value


CONV_PRODUCER = {0: "gather", 1: "vector", 2: "window", 3: "tmem"}


def mmact_conv2d_producer(N, C, H, W, Co, kh, kw, stride, pads, dilation, in_dtype, out_dtype) -> str:
    """Which B-tile producer mmact_conv2d uses for this NCHW geometry (a name
    from CONV_PRODUCER); dtypes are torch dtypes."""
    r = load().mmact_conv2d_producer(N, C, H, W, Co, kh, kw, _i32(stride, 2), _i32(pads, 4),
                                     _i32(dilation, 2), DTYPE[in_dtype], DTYPE[out_dtype])
    if r not in CONV_PRODUCER:
        raise ValueError("mmact_conv2d_producer: invalid arguments")
    return CONV_PRODUCER[r]


def _conv_args(x, w, bias, y, stride, pads, dilation):
    px = _dev(x, "x", _IN)
    pw = _dev(w, "w", _IN)
    py = _dev(y, "y", _OUT)
    if x.dim() != 4 or w.dim() != 4 or y.dim() != 4:
        raise ValueError("x, w, y must be 4-D (NCHW / [Co,C,kh,kw])")
    N, C, H, W = x.shape
    Co, C2, kh, kw = w.shape
    if C2 != C or w.dtype != x.dtype:
        raise ValueError("w must be [Co, C, kh, kw] with x's dtype")
    Ho, Wo = mmact_conv2d_out_shape(H, W, kh, kw, stride, pads, dilation)
    if tuple(y.shape) != (N, Co, Ho, Wo):
        raise ValueError(f"y must be {(N, Co, Ho, Wo)}")
    return (px, pw, _bias_ptr(bias, Co), py, N, C, H, W, Co, kh, kw, _i32(stride, 2),
            _i32(pads, 4), _i32(dilation, 2))


def mmact_conv2d(x, w, bias, y, stride=(1, 1), pads=(0, 0, 0, 0), dilation=(1, 1),
                 act: str = "tanh", alpha: float = 0.0, stream=None) -> None:
    """y = act(conv2d(x, w) + bias), NCHW, pads = (top, bottom, left, right)."""
    L = load()
    args = _conv_args(x, w, bias, y, stride, pads, dilation)
    _check(L.mmact_conv2d(*args, DTYPE[x.dtype], DTYPE[y.dtype], ACT[act], float(alpha),
                          _stream_handle(stream)), "mmact_conv2d")


def _residual_ptr(R, y):
    pr = _dev(R, "R", _OUT)
    if tuple(R.shape) != tuple(y.shape) or R.dtype != y.dtype:
        raise ValueError("R must have y's shape and dtype")
    return pr


def mmact_conv2d_residual(x, w, bias, R, y, stride=(1, 1), pads=(0, 0, 0, 0), dilation=(1, 1),
                          act: str = "tanh", alpha: float = 0.0, stream=None) -> None:
    """y = act(conv2d(x, w) + bias + R), NCHW; R has y's shape and dtype and may be y."""
    L = load()
    px, pw, pb, py, *rest = _conv_args(x, w, bias, y, stride, pads, dilation)
    pr = _residual_ptr(R, y)
    _check(L.mmact_conv2d_residual(px, pw, pb, pr, py, *rest, DTYPE[x.dtype], DTYPE[y.dtype], ACT[act],
                                   float(alpha), _stream_handle(stream)), "mmact_conv2d_residual")


def mmact_conv2d_split(x, w, bias, y, workspace, stride=(1, 1), pads=(0, 0, 0, 0),
                       dilation=(1, 1), act: str = "tanh", alpha: float = 0.0, stream=None) -> None:
    """Two-kernel ablation of mmact_conv2d through an fp32 workspace shaped like y."""
    L = load()
    args = _conv_args(x, w, bias, y, stride, pads, dilation)
    pws = _dev(workspace, "workspace", (torch.float32,))
    if workspace.numel() < y.numel():
        raise ValueError("workspace must hold y.numel() fp32 elements")
    _check(L.mmact_conv2d_split(*args, DTYPE[x.dtype], DTYPE[y.dtype], ACT[act], float(alpha), pws,
                                _stream_handle(stream)), "mmact_conv2d_split")


def _in_code(x, tf32: bool) -> int:
    if tf32:
        if x.dtype != torch.float32:
            raise ValueError("tf32=True needs float32 x and w")
        return MMACT_TF32
    return DTYPE[x.dtype]


def mmact_conv2d_auto(x, w, bias, y, stride=(1, 1), pads=(0, 0, 0, 0), dilation=(1, 1),
                      act: str = "tanh", alpha: float = 0.0, workspace=None, stream=None) -> None:
    """NCHW fused or two-kernel conv, decided per geometry (see include/mmact.h)."""
    L = load()
    args = _conv_args(x, w, bias, y, stride, pads, dilation)
    pws = None
    if workspace is not None:
        pws = _dev(workspace, "workspace", (torch.float32,))
        if workspace.numel() < y.numel():
            raise ValueError("workspace must hold y.numel() fp32 elements")
    _check(L.mmact_conv2d_auto(*args, DTYPE[x.dtype], DTYPE[y.dtype], ACT[act], float(alpha), pws,
                               _stream_handle(stream)), "mmact_conv2d_auto")


def mmact_conv2d_auto_choice(N, C, H, W, Co, kh, kw, stride, pads, dilation, in_dtype, out_dtype,
                             act: str) -> str:
    """"split" or "fused": the path mmact_conv2d_auto takes with a workspace."""
    out = ctypes.c_int(-1)
    _check(load().mmact_conv2d_auto_choice(N, C, H, W, Co, kh, kw, _i32(stride, 2), _i32(pads, 4),
                                           _i32(dilation, 2), DTYPE[in_dtype], DTYPE[out_dtype], ACT[act],
                                           ctypes.byref(out)), "mmact_conv2d_auto_choice")
    return "split" if out.value == 1 else "fused"


def mmact_conv2d_nhwc(x, w, bias, y, stride=(1, 1), pads=(0, 0, 0, 0), dilation=(1, 1),
                      act: str = "tanh", alpha: float = 0.0, stream=None, tf32: bool = False) -> None:
    """Channels-last y = act(conv2d(x, w) + bias): x [N,H,W,C], w [Co,kh,kw,C], y [N,Ho,Wo,Co].
    float32 x and w run in split precision (fp32 accuracy), or as tf32 (one pass) with
    tf32=True (see include/mmact.h)."""
    L = load()
    px, pw, pb, py, *rest = _nhwc_args(x, w, bias, y, stride, pads, dilation)
    _check(L.mmact_conv2d_nhwc(px, pw, pb, py, *rest, _in_code(x, tf32), DTYPE[y.dtype], ACT[act],
                               float(alpha), _stream_handle(stream)), "mmact_conv2d_nhwc")


def _nhwc_args(x, w, bias, y, stride, pads, dilation):
    px = _dev(x, "x", _OUT)
    pw = _dev(w, "w", _OUT)
    py = _dev(y, "y", _OUT)
    if x.dim() != 4 or w.dim() != 4 or y.dim() != 4:
        raise ValueError("x, w, y must be 4-D (NHWC / [Co,kh,kw,C] / NHWC)")
    N, H, W, C = x.shape
    Co, kh, kw, C2 = w.shape
    if C2 != C or w.dtype != x.dtype:
        raise ValueError("w must be [Co, kh, kw, C] with x's dtype")
    Ho, Wo = mmact_conv2d_out_shape(H, W, kh, kw, stride, pads, dilation)
    if tuple(y.shape) != (N, Ho, Wo, Co):
        raise ValueError(f"y must be {(N, Ho, Wo, Co)}")
    return (px, pw, _bias_ptr(bias, Co), py, N, C, H, W, Co, kh, kw, _i32(stride, 2), _i32(pads, 4),
            _i32(dilation, 2))


def mmact_conv2d_nhwc_residual(x, w, bias, R, y, stride=(1, 1), pads=(0, 0, 0, 0), dilation=(1, 1),
                               act: str = "tanh", alpha: float = 0.0, stream=None, tf32: bool = False) -> None:
    """Channels-last y = act(conv2d(x, w) + bias + R); R has y's shape [N,Ho,Wo,Co] and dtype."""
    L = load()
    px, pw, pb, py, *rest = _nhwc_args(x, w, bias, y, stride, pads, dilation)
    pr = _residual_ptr(R, y)
    _check(L.mmact_conv2d_nhwc_residual(px, pw, pb, pr, py, *rest, _in_code(x, tf32), DTYPE[y.dtype],
                                        ACT[act], float(alpha), _stream_handle(stream)),
           "mmact_conv2d_nhwc_residual")


def mmact_get_last_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word's verdict."""
    return int(load().mmact_get_last_error(_stream_handle(stream)))


def mmact_set_wait_timeout_ns(ns: int) -> None:
    load().mmact_set_wait_timeout_ns(int(ns))


def mmact_selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(load().mmact_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream)),
           "mmact_selftest_wait_timeout")


def mmact_set_gemm_tile_n(tile_n: int) -> None:
    _check(load().mmact_set_gemm_tile_n(int(tile_n)), "mmact_set_gemm_tile_n")


def mmact_set_gemm_split_k(split_k: int) -> None:
    """0: split-K chosen per shape; 1: never; 2 or 4: whenever legal."""
    _check(load().mmact_set_gemm_split_k(int(split_k)), "mmact_set_gemm_split_k")


def mmact_set_gemm_pair(mode: int) -> None:
    """CTA-pair GEMM kernel: 0 chosen per shape; 1 never; 2 always (when split-K is not taken)."""
    _check(load().mmact_set_gemm_pair(int(mode)), "mmact_set_gemm_pair")


def mmact_set_conv_tmem(mode: int) -> None:
    """NCHW conv with the im2col operand in tensor memory: 0 where it applies (default); 1 never."""
    _check(load().mmact_set_conv_tmem(int(mode)), "mmact_set_conv_tmem")


def mmact_set_gemm_l2_policy(mode: int) -> None:
    """CTA-pair GEMM: 1 A evict-last and C evict-first in L2 (default); 0 no cache hints."""
    _check(load().mmact_set_gemm_l2_policy(int(mode)), "mmact_set_gemm_l2_policy")


def mmact_tensor_map_cache_stats() -> tuple[int, int]:
    """(hits, encodes) of the library's host-side tensor-map cache, process-wide."""
    h, e = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(load().mmact_tensor_map_cache_stats(ctypes.byref(h), ctypes.byref(e)), "mmact_tensor_map_cache_stats")
    return int(h.value), int(e.value)


GEMM_KERNELS = {0: "none", 1: "persistent", 2: "pair", 3: "split_k"}


def mmact_gemm_kernel_choice(M: int, N: int, K: int, residual: bool = False) -> str:
    """The kernel a GEMM of this shape would run: "none", "persistent", "pair" or "split_k"."""
    out = ctypes.c_int(-1)
    _check(load().mmact_gemm_kernel_choice(int(M), int(N), int(K), 1 if residual else 0,
                                           ctypes.byref(out)), "mmact_gemm_kernel_choice")
    return GEMM_KERNELS[out.value]


def mmact_gemm_split_k_choice(M: int, N: int, K: int) -> int:
    """Split-K factor (0, 2 or 4) a GEMM of this shape would use on the current device."""
    out = ctypes.c_int(-1)
    _check(load().mmact_gemm_split_k_choice(int(M), int(N), int(K), ctypes.byref(out)),
           "mmact_gemm_split_k_choice")
    return out.value


def mmact_status_string(status: int) -> str:
    return status_string(status)


def mmact_version() -> int:
    return int(load().mmact_version())
