"""The C ABI library loads and exports every symbol include/mmact.h declares,
and its host-only paths (argument validation, output shape) behave.  No GPU
is needed: every call here returns before any CUDA work."""
import ctypes
import os
import re
import subprocess

import pytest

from conv_activation_epilogue_gb300 import build, mmact
import oracle

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mmact.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mmact_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mmact.load()


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(mmact.SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIBRARY], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(set(re.findall(r"\b(mmact_[a-z0-9_]+)$", out, flags=re.M)))
    assert exported == declared_functions()


def test_version_and_status_strings(lib):
    assert mmact.mmact_version() == 1
    for s in range(5):
        assert mmact.mmact_status_string(s).startswith("MMACT_")
    assert "unknown" in mmact.mmact_status_string(99)


def test_tile_override_validation(lib):
    for bad in (1, 32, 96, 512, -64):
        assert lib.mmact_set_gemm_tile_n(bad) == mmact.MMACT_ERR_INVALID_ARG
    for good in (64, 128, 192, 224, 256, 0):
        assert lib.mmact_set_gemm_tile_n(good) == mmact.MMACT_OK


def test_kernel_mode_validation(lib):
    # split-K factor: 0 automatic, 1 never, 2 or 4 forced; pair kernel: 0 automatic, 1 never, 2 forced
    for bad in (-1, 3, 5, 8):
        assert lib.mmact_set_gemm_split_k(bad) == mmact.MMACT_ERR_INVALID_ARG
    for good in (1, 2, 4, 0):
        assert lib.mmact_set_gemm_split_k(good) == mmact.MMACT_OK
    for bad in (-1, 3, 4):
        assert lib.mmact_set_gemm_pair(bad) == mmact.MMACT_ERR_INVALID_ARG
    for good in (1, 2, 0):
        assert lib.mmact_set_gemm_pair(good) == mmact.MMACT_OK


def test_kernel_choice_queries_reject_bad_arguments(lib):
    out = ctypes.c_int(-7)
    assert lib.mmact_gemm_kernel_choice(-1, 8, 8, 0, ctypes.byref(out)) == mmact.MMACT_ERR_INVALID_ARG
    assert lib.mmact_gemm_kernel_choice(8, 8, 8, 0, None) == mmact.MMACT_ERR_INVALID_ARG
    assert lib.mmact_gemm_split_k_choice(8, -8, 8, ctypes.byref(out)) == mmact.MMACT_ERR_INVALID_ARG
    assert lib.mmact_gemm_split_k_choice(8, 8, 8, None) == mmact.MMACT_ERR_INVALID_ARG
    assert out.value == -7


def test_out_shape_matches_oracle(lib):
    orc = oracle.get()
    for (H, W, kh, kw, st, pd, dl) in [(56, 56, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1)),
                                       (64, 64, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2)),
                                       (64, 64, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1)),
                                       (7, 5, 3, 2, (2, 1), (1, 0, 2, 1), (1, 2)),
                                       (1, 1, 1, 1, (3, 3), (0, 0, 0, 0), (1, 1))]:
        Ho, Wo = mmact.mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl)
        assert Ho == orc.conv_out_dim(H, kh, st[0], pd[0], pd[1], dl[0])
        assert Wo == orc.conv_out_dim(W, kw, st[1], pd[2], pd[3], dl[1])


def test_conv_producer_choice(lib):
    import torch
    f16, bf16, f32 = torch.float16, torch.bfloat16, torch.float32
    P = mmact.mmact_conv2d_producer
    try:
        # default: the tensor-memory im2col kernel wherever it applies -- the three conv workloads
        assert P(8, 64, 56, 56, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), f16, f16) == "tmem"
        assert P(16, 128, 64, 64, 256, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), bf16, bf16) == "tmem"
        assert P(16, 128, 64, 64, 256, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), bf16, bf16) == "tmem"
        assert P(1, 16, 7, 16, 16, 3, 3, (2, 1), (1, 1, 2, 2), (1, 2), bf16, f16) == "tmem"
        # it does not apply: input width not a multiple of 8, K not a multiple of 8, 11x11 taps
        assert P(2, 24, 17, 13, 40, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), bf16, bf16) == "gather"
        assert P(3, 3, 11, 16, 5, 3, 2, (2, 1), (1, 0, 2, 1), (1, 2), f16, f32) == "gather"
        assert P(1, 8, 64, 64, 8, 11, 11, (1, 1), (5, 5, 5, 5), (1, 1), f16, f16) == "window"
        # with it turned off: the window / vector / gather producers
        mmact.mmact_set_conv_tmem(1)
        assert P(8, 64, 56, 56, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), f16, f16) == "window"
        assert P(16, 128, 64, 64, 256, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), bf16, bf16) == "window"
        # 1x1, 64 channels per K block: the window would be 72 x 8 x 64 x 2 B > 24 KB
        assert P(16, 128, 64, 64, 256, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), bf16, bf16) == "vector"
        # input width not a multiple of 8, horizontal stride 3, K not a multiple of 8
        assert P(2, 24, 17, 13, 40, 3, 3, (2, 2), (2, 2, 2, 2), (2, 2), bf16, bf16) == "gather"
        assert P(1, 8, 16, 48, 8, 3, 3, (1, 3), (1, 1, 1, 1), (1, 1), f16, f16) == "gather"
        assert P(3, 3, 11, 16, 5, 3, 2, (2, 1), (1, 0, 2, 1), (1, 2), f16, f32) == "gather"
        # dh not a multiple of sh: the window keeps every input row
        assert P(1, 16, 7, 16, 16, 3, 3, (2, 1), (1, 1, 2, 2), (1, 2), bf16, f16) == "window"
    finally:
        mmact.mmact_set_conv_tmem(0)
    with pytest.raises(ValueError):
        P(1, 8, 8, 8, 8, 0, 3, (1, 1), (0, 0, 0, 0), (1, 1), f16, f16)


def test_conv_tmem_mode_validation(lib):
    for bad in (-1, 2, 3):
        assert lib.mmact_set_conv_tmem(bad) == mmact.MMACT_ERR_INVALID_ARG
    for good in (1, 0):
        assert lib.mmact_set_conv_tmem(good) == mmact.MMACT_OK


def test_out_shape_rejects_bad_geometry(lib):
    for args in [(5, 5, 0, 3, (1, 1), (0, 0, 0, 0), (1, 1)),
                 (5, 5, 3, 3, (0, 1), (0, 0, 0, 0), (1, 1)),
                 (5, 5, 3, 3, (1, 1), (-1, 0, 0, 0), (1, 1)),
                 (5, 5, 3, 3, (1, 1), (0, 0, 0, 0), (0, 1)),
                 (2, 2, 3, 3, (1, 1), (0, 0, 0, 0), (1, 1))]:   # empty output
        with pytest.raises(mmact.MmactError) as ei:
            mmact.mmact_conv2d_out_shape(*args)
        assert ei.value.status == mmact.MMACT_ERR_INVALID_ARG


# Fake, never-dereferenced device addresses: every call below is rejected on
# the host before any CUDA call, or is a no-op (empty problem).
P16 = 0x7f0000000000
P_MIS = P16 + 2


def gemm(lib, A=P16, B=P16, bias=None, C=P16, M=64, N=64, K=64, ab=1, cd=1, act=2, ws=None,
         split=False):
    if split:
        return lib.mmact_gemm_split(A, B, bias, C, M, N, K, ab, cd, act, ctypes.c_float(0.1), ws, None)
    return lib.mmact_gemm(A, B, bias, C, M, N, K, ab, cd, act, ctypes.c_float(0.1), None)


def test_gemm_host_validation(lib):
    E, U, OK = mmact.MMACT_ERR_INVALID_ARG, mmact.MMACT_ERR_UNSUPPORTED, mmact.MMACT_OK
    assert gemm(lib, A=None) == E
    assert gemm(lib, B=None) == E
    assert gemm(lib, C=None) == E
    assert gemm(lib, M=-1) == E
    assert gemm(lib, K=-8) == E
    assert gemm(lib, N=1 << 31) == E
    assert gemm(lib, ab=3) == U             # one-pass tf32 operands: channels-last conv only
    assert gemm(lib, ab=4) == E
    assert gemm(lib, ab=7) == E
    assert gemm(lib, ab=2, A=P16 + 2) == U  # fp32 operands (split precision) need 4-byte alignment
    assert gemm(lib, ab=2, M=0) == OK       # ... and may have any K and N; empty is a no-op
    assert gemm(lib, cd=5) == E
    assert gemm(lib, act=6) == E
    assert gemm(lib, act=-1) == E
    assert gemm(lib, bias=P16 + 1) == E     # bias must be 4-byte aligned
    assert gemm(lib, A=P_MIS) == U
    assert gemm(lib, C=P_MIS) == U
    assert gemm(lib, K=60) == U             # row pitch of A not a multiple of 16 bytes
    assert gemm(lib, N=60) == U
    assert gemm(lib, A=None, M=0) == OK     # an empty tensor may have a null pointer
    assert gemm(lib, M=0) == OK             # empty: nothing enqueued
    assert gemm(lib, N=0) == OK
    assert gemm(lib, split=True, ws=None) == E
    assert gemm(lib, split=True, ws=P_MIS) == U
    assert gemm(lib, split=True, ws=P16, M=0) == OK


def test_noalloc_checks_arguments_before_its_size_limit(lib):
    # the same checks as mmact_gemm_split come first: a bad argument is reported
    # as such even when M*N is beyond the scratch array; then the size limit
    E, U, OK = mmact.MMACT_ERR_INVALID_ARG, mmact.MMACT_ERR_UNSUPPORTED, mmact.MMACT_OK
    big_m, big_n = 4096, 4096                  # 4 x MMACT_NOALLOC_MAX_ELEMENTS

    def na(A=P16, C=P16, M=64, N=64, K=64, ab=1, cd=1, act=2):
        return lib.mmact_gemm_split_noalloc(A, P16, None, C, M, N, K, ab, cd, act, ctypes.c_float(0.1), None)

    assert na(act=9, M=big_m, N=big_n) == E
    assert na(ab=4, M=big_m, N=big_n) == E
    assert na(A=None, M=big_m, N=big_n) == E
    assert na(M=-1) == E
    assert na(A=P_MIS, M=big_m, N=big_n) == U   # alignment, as for mmact_gemm_split
    assert na(M=big_m, N=big_n) == U            # valid arguments, beyond the scratch array
    assert na(M=2048, N=2056) == U              # just past the limit (2048 x 2048 is the largest square)
    assert na(M=0) == OK                        # empty: nothing enqueued, no set-up


def test_gemm_residual_host_validation(lib):
    E, U, OK = mmact.MMACT_ERR_INVALID_ARG, mmact.MMACT_ERR_UNSUPPORTED, mmact.MMACT_OK

    def res(R=P16 + 4096, C=P16, M=16, N=16, K=16, cd=1):
        return lib.mmact_gemm_residual(P16, P16, None, R, C, M, N, K, 1, cd, 1, ctypes.c_float(0), None)

    assert res(R=None) == E                  # the residual is required
    assert res(R=None, M=0) == OK            # ... unless the output is empty
    assert res(R=P_MIS) == U                 # 16-byte alignment
    assert res(R=P16 + 16) == E              # partial overlap with C (16x16 bf16 = 512 B)
    assert res(M=-1) == E


def test_conv_host_validation(lib):
    E, U = mmact.MMACT_ERR_INVALID_ARG, mmact.MMACT_ERR_UNSUPPORTED
    i32 = lambda *v: (ctypes.c_int32 * len(v))(*v)  # noqa: E731

    def conv(x=P16, w=P16, y=P16, N=1, C=4, H=8, W=8, Co=4, kh=3, kw=3, st=(1, 1),
             pd=(1, 1, 1, 1), dl=(1, 1), i=1, o=1, act=3):
        return lib.mmact_conv2d(x, w, None, y, N, C, H, W, Co, kh, kw, i32(*st), i32(*pd), i32(*dl),
                                i, o, act, ctypes.c_float(0), None)

    assert conv(x=None) == E
    assert conv(y=None) == E
    assert conv(N=-1) == E
    assert conv(kh=0) == E
    assert conv(st=(0, 1)) == E
    assert conv(pd=(0, -1, 0, 0)) == E
    assert conv(dl=(1, 0)) == E
    assert conv(H=1, pd=(0, 0, 0, 0)) == E   # 3x3 filter on a 1-row input: empty output
    assert conv(i=3) == E                    # one-pass tf32: channels-last only
    assert conv(i=4) == E
    assert conv(o=3) == E
    assert conv(act=9) == E
    assert conv(x=P_MIS) == U
    assert lib.mmact_conv2d(P16, P16, None, P16, 1, 4, 8, 8, 4, 3, 3, None, i32(0, 0, 0, 0),
                            i32(1, 1), 1, 1, 3, ctypes.c_float(0), None) == E


def test_auto_choice_follows_the_measured_rule(lib):
    import torch
    bf16, f16, f32 = torch.bfloat16, torch.float16, torch.float32
    G = mmact.mmact_gemm_auto_choice
    assert G(64, 64, 64, bf16, bf16, "gelu") == "split"        # GELU on a small output
    assert G(256, 256, 1024, bf16, bf16, "gelu") == "split"
    assert G(256, 264, 64, bf16, bf16, "gelu") == "fused"       # more than 64 Ki outputs
    assert G(8192, 8192, 64, bf16, bf16, "gelu") == "fused"
    assert G(64, 64, 64, bf16, bf16, "relu") == "fused"         # every other activation: fused
    assert G(64, 64, 64, bf16, bf16, "tanh") == "fused"
    assert G(64, 64, 64, f32, f32, "gelu") == "fused"          # fp32 inputs: split precision, fused
    Cv = mmact.mmact_conv2d_auto_choice
    # 1x1 stride 2 on 28 x 28: a 14 x 14 output (392-byte rows) would be stored element by element
    assert Cv(8, 64, 28, 28, 128, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), f16, f16, "relu") == "split"
    assert Cv(8, 64, 28, 28, 128, 1, 1, (2, 2), (0, 0, 0, 0), (1, 1), f16, f32, "relu") == "fused"
    assert Cv(8, 16, 56, 56, 64, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), f16, f16, "gelu") == "split"
    assert Cv(32, 16, 32, 32, 32, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), f16, f16, "gelu") == "fused"
    assert Cv(8, 64, 56, 56, 128, 3, 3, (1, 1), (1, 1, 1, 1), (1, 1), f16, f16, "tanh") == "fused"
    out = ctypes.c_int(-5)
    assert lib.mmact_gemm_auto_choice(-1, 8, 8, 1, 1, 1, ctypes.byref(out)) == mmact.MMACT_ERR_INVALID_ARG
    assert lib.mmact_gemm_auto_choice(8, 8, 8, 1, 1, 9, ctypes.byref(out)) == mmact.MMACT_ERR_INVALID_ARG
    assert lib.mmact_gemm_auto_choice(8, 8, 8, 1, 1, 1, None) == mmact.MMACT_ERR_INVALID_ARG
    assert out.value == -5
