"""The seeded input generator: determinism, counter independence, rounding."""
import math

import numpy as np

from exact_attention_28_gb300 import inputs


def test_splitmix64_reference_values():
    # First outputs of SplitMix64 seeded with 0 (values of the published
    # generator: state += 0x9E3779B97F4A7C15, then the 64-bit finaliser).
    out = inputs.splitmix64(0, 0, 3)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_slices_agree():
    whole = inputs.splitmix64(1234, 0, 1000)
    part = inputs.splitmix64(1234, 400, 100)
    assert np.array_equal(whole[400:500], part)
    a = inputs.normal_bf16(7, (3, 1001), 1.0)
    b = inputs.normal_bf16(7, (3, 1001), 1.0, chunk_pairs=17)
    assert np.array_equal(a, b)


def test_deterministic_and_seed_sensitive():
    a = inputs.normal_bf16(11, (64, 64))
    assert np.array_equal(a, inputs.normal_bf16(11, (64, 64)))
    assert not np.array_equal(a, inputs.normal_bf16(12, (64, 64)))


def test_distribution_moments():
    x = inputs.bf16_bits_to_fp32(inputs.normal_bf16(99, (1 << 20,), 2.0)).astype(np.float64)
    assert abs(x.mean()) < 0.01
    assert abs(x.std() - 2.0) < 0.01
    # tail mass beyond 3 sigma of a normal: 0.0027
    assert abs(np.mean(np.abs(x) > 6.0) - 0.0027) < 0.0005


def test_bf16_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e-40], dtype=np.float32)
    got = inputs.bf16_bits_to_fp32(inputs.fp32_to_bf16_bits(vals))
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6: goes to 1+2^-6.
    assert list(got[:4]) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0]
    assert got[4] == -2.5


def test_workloads_table():
    w = inputs.WORKLOADS["b2_h16_n4096_d128"]
    assert w.flops == 274877906944 and w.algorithmic_bytes == 134742016
    w = inputs.WORKLOADS["causal_h32_n16384_d128_sigma2"]
    assert w.flops == 2199023255552 and w.sigma_q == 2.0
    assert inputs.WORKLOADS["b8_h32_q128_kv8229_d128"].Nk == 8229
    assert inputs.WORKLOADS["single_head_n256_d64"].scale == np.float32(1 / math.sqrt(64))
