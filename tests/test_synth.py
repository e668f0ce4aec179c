"""The seeded input generator (CPU only)."""
import numpy as np

from conv_activation_epilogue_gb300 import synth


def test_splitmix64_published_sequence():
    # first outputs of SplitMix64 seeded with 0, as published with the generator
    got = [int(v) for v in synth.splitmix64(0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_prefix_property():
    a = synth.splitmix64(99, 10)
    b = synth.splitmix64(99, (1 << 22) + 5)
    assert np.array_equal(a, b[:10])


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to the even code 0x3F80
    assert synth.to_codes(np.array([1 + 2.0 ** -8]), "bf16")[0] == 0x3F80
    # 1 + 3*2^-8 ties between 1+2^-7 (odd, 0x3F81) and 1+2^-6 (even, 0x3F82)
    assert synth.to_codes(np.array([1 + 3 * 2.0 ** -8]), "bf16")[0] == 0x3F82
    assert synth.to_codes(np.array([-2.0]), "bf16")[0] == 0xC000
    assert synth.to_codes(np.array([1.0]), "f16")[0] == 0x3C00


def test_distributions():
    u = synth.uniform(7, (200000,), -1.0, 1.0)
    assert u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 0.01 and abs(u.std() - (1 / 3) ** 0.5) < 0.01
    g = synth.normal(8, (200001,), 0.5)
    assert abs(g.mean()) < 0.01 and abs(g.std() - 0.5) < 0.01


def test_workloads_deterministic_and_shaped():
    w = synth.WORKLOADS["matmul_leakyrelu_1024x640x256_f16"]
    a = w.inputs()
    b = w.inputs()
    assert a["A"].shape == (1024, 256) and a["B"].shape == (256, 640) and a["bias"].shape == (640,)
    assert np.array_equal(a["A"], b["A"]) and np.array_equal(a["bias"], b["bias"])
    assert a["A"].dtype == np.uint16 and a["bias"].dtype == np.float32
    c = synth.WORKLOADS["conv3x3_s2p2d2_tanh_16x128x64x64_bf16"]
    d = synth.WORKLOADS["conv1x1_s2_tanh_16x128x64x64_bf16"]
    # the 1x1 workload reuses the same input features
    assert c.seed == d.seed and c.x_seed == d.x_seed
    assert c.w_tensor != d.w_tensor
    assert synth.HEADLINE in synth.WORKLOADS
