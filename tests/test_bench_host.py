"""Host-side arithmetic of bench.py: algorithmic flops and bytes per workload and the
roofline object of the bench line (which bound, which peak, which fraction).  No GPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from conv_activation_epilogue_gb300 import build, mmact, synth  # noqa: E402

PEAKS = {"bf16_tflops": 1918.4, "hbm_gbs": 6779.7}


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mmact.load()


def test_gemm_flops_and_bytes():
    wl = synth.WORKLOADS["gemm_leakyrelu_8192x8192x8192_bf16"]
    assert bench.workload_flops(None, wl) == 2.0 * 8192 ** 3
    # A and B bf16, bias fp32 [N], C bf16
    assert bench.workload_bytes(None, wl) == 2.0 * (2 * 8192 * 8192) + 4.0 * 8192 + 2.0 * 8192 * 8192
    wl = synth.WORKLOADS["matmul_leakyrelu_1024x640x256_f16"]   # fp32 output
    assert bench.workload_bytes(None, wl) == 2.0 * (1024 * 256 + 256 * 640) + 4.0 * 640 + 4.0 * 1024 * 640


def test_conv_flops_and_bytes(lib):
    wl = synth.WORKLOADS["conv3x3_s2p2d2_tanh_16x128x64x64_bf16"]
    Ho, Wo = mmact.mmact_conv2d_out_shape(wl.H, wl.W, wl.kh, wl.kw, wl.stride, wl.pads, wl.dilation)
    assert (Ho, Wo) == (32, 32)     # (64 + 2 + 2 - 2 * 2 - 1) // 2 + 1
    assert bench.workload_flops(mmact, wl) == 2.0 * 16 * 32 * 32 * 256 * 128 * 9
    # stride 2, dilation 2, pad 2: outputs read only the even input rows and columns (32 of 64 each)
    assert bench.workload_bytes(mmact, wl) == (2.0 * (16 * 128 * 32 * 32 + 256 * 128 * 9) + 4.0 * 256
                                              + 2.0 * 16 * 256 * 32 * 32)


def test_conv_input_lines_read():
    # 3x3, stride 1, pad 1 on 56: every line; 1x1 stride 2 on 64: the 32 even lines;
    # 3x3 stride 2 dilation 2 pad 2 on 64: the even lines; 3x3 stride 2 pad 1: every line
    assert bench.conv_lines_read(56, 3, 1, 1, 1, 56) == 56
    assert bench.conv_lines_read(64, 1, 2, 0, 1, 32) == 32
    assert bench.conv_lines_read(64, 3, 2, 2, 2, 32) == 32
    assert bench.conv_lines_read(64, 3, 2, 1, 1, 32) == 64
    # a 1x1 stride-2 conv needs a quarter of x
    wl = synth.WORKLOADS["conv1x1_s2_tanh_16x128x64x64_bf16"]
    x_needed = 2.0 * 16 * 128 * 32 * 32
    assert bench.workload_bytes(lib_free_shape(wl), wl) == (x_needed + 2.0 * 256 * 128 + 4.0 * 256
                                                            + 2.0 * 16 * 256 * 32 * 32)


def lib_free_shape(wl):
    """Stand-in for the library's output-shape call (the formula, for these tests only)."""
    class Shape:
        @staticmethod
        def mmact_conv2d_out_shape(H, W, kh, kw, st, pd, dl):
            return ((H + pd[0] + pd[1] - dl[0] * (kh - 1) - 1) // st[0] + 1,
                    (W + pd[2] + pd[3] - dl[1] * (kw - 1) - 1) // st[1] + 1)
    return Shape


def test_tensor_capacity_fractions():
    # burst against the capacity at the maximum clock, sustained against the sampled clock
    rec = bench.tensor_capacity(1872.0, 152, 1537.0, 2070.0, sustained_tflops=1700.0)
    cap_max = 152 * 8192 * 2070e6 / 1e12
    cap = 152 * 8192 * 1537e6 / 1e12
    assert rec["peak_tflops_at_max_clock"] == pytest.approx(cap_max)
    assert rec["frac_at_max_clock"] == pytest.approx(1872.0 / cap_max)
    assert rec["peak_tflops_at_sampled_clock"] == pytest.approx(cap)
    assert rec["sustained_frac_at_sampled_clock"] == pytest.approx(1700.0 / cap)
    assert rec["frac_of_nominal"] == pytest.approx(1872.0 / 2250.0)
    assert "sustained_frac_at_sampled_clock" not in bench.tensor_capacity(1872.0, 152, 1537.0, 2070.0)


def test_roofline_bound_follows_the_ridge_point():
    ridge = PEAKS["bf16_tflops"] * 1e12 / (PEAKS["hbm_gbs"] * 1e9)      # about 283 flop/byte
    # the square workload is far above the ridge: tensor-bound, fraction of the bf16 peak
    wl = synth.WORKLOADS["gemm_leakyrelu_8192x8192x8192_bf16"]
    f, b = bench.workload_flops(None, wl), bench.workload_bytes(None, wl)
    assert f / b > ridge
    r = bench.roofline_record(f, b, 0.5731, PEAKS, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == PEAKS["bf16_tflops"]
    assert r["achieved"] == pytest.approx(f / 0.5731e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["bf16_tflops"])
    # the 128-row workload is below it: HBM-bound on algorithmic bytes
    wl = synth.WORKLOADS["gemm_leakyrelu_128x8192x8192_bf16"]
    f, b = bench.workload_flops(None, wl), bench.workload_bytes(None, wl)
    assert f / b < ridge
    r = bench.roofline_record(f, b, 0.0300, PEAKS, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == PEAKS["hbm_gbs"]
    assert r["achieved"] == pytest.approx(b / 0.0300e-3 / 1e9)
    assert r["alg_bytes_per_launch"] == b


def test_traffic_records_follow_their_kernels_sources(tmp_path, monkeypatch):
    """A stored DRAM figure is reported only while every source its kernel depends on is
    unchanged: each kernel hashes its own file plus the shared headers and the host planner."""
    hashes = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_FILES}
    assert len(set(hashes.values())) == len(hashes)            # one hash per kernel
    assert bench.kernel_source_hash("no_such_kernel") == bench.kernel_source_hash(None)
    # every record committed in profiles/traffic.json matches the current sources
    import json
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for key, ent in rec.items():
        kernel, workload = key.split("/")
        assert kernel in bench.KERNEL_FILES and workload in synth.WORKLOADS
        assert ent["dram_bytes_per_launch"] == ent["dram_read_bytes"] + ent["dram_write_bytes"]
        assert bench.traffic_per_launch(kernel, workload) == ent["dram_bytes_per_launch"]
    # a changed source voids the record: point the hash at a copy of the sources with one edit
    src = os.path.join(bench.ROOT, "conv_activation_epilogue_gb300", "csrc")
    fake = tmp_path / "conv_activation_epilogue_gb300" / "csrc"
    fake.mkdir(parents=True)
    for name in os.listdir(src):
        if name.endswith((".cu", ".cuh", ".h")):
            data = open(os.path.join(src, name), "rb").read()
            if name == "gemm_pair.cu":
                data += b"\n// edited\n"
            (fake / name).write_bytes(data)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_source_hash("gemm_pair_kernel") != hashes["gemm_pair_kernel"]
    assert bench.kernel_source_hash("conv_tmem_kernel") == hashes["conv_tmem_kernel"]
