"""Pins of the FP8 oracle (oracle/fp8.py) against facts that do not come from
the oracle itself: the E4M3 format's defining values, PyTorch's float8
conversion, the Hadamard matrix of scipy, exact arithmetic on small integers,
orthogonality, and the plain bf16 oracle on inputs both formats hold exactly.
CPU only."""
import math

import numpy as np
import pytest

import oracle
from oracle import fp8
from exact_attention_28_gb300 import inputs

torch = pytest.importorskip("torch")


def test_e4m3_defining_values():
    # 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; subnormals; S.1111.111 = NaN
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
             0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}
    for code, value in cases.items():
        assert fp8.decode_e4m3(code) == value, hex(code)
    assert np.isnan(fp8.decode_e4m3(0x7F)) and np.isnan(fp8.decode_e4m3(0xFF))
    assert np.signbit(fp8.decode_e4m3(0x80)) and fp8.decode_e4m3(0x80) == 0.0
    finite = fp8.E4M3[np.isfinite(fp8.E4M3)]
    assert finite.max() == 448.0 and finite.size == 254


def test_decode_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fp8.E4M3
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.encode_e4m3(fp8.decode_e4m3(codes)), codes)


def test_encode_ties_go_to_the_even_code_and_large_values_saturate():
    mags = fp8.E4M3[:127]
    mids = 0.5 * (mags[:-1] + mags[1:])                  # exact midpoints in fp64
    got = fp8.encode_e4m3(mids)
    lo = np.arange(126)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, expect.astype(np.uint8))
    assert np.array_equal(fp8.encode_e4m3(np.array([448.0, 449.0, 1e6, -1e6])),
                          np.array([0x7E, 0x7E, 0x7E, 0xFE], dtype=np.uint8))


def test_encode_matches_torch_float8_conversion():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1.0, 30.0, 200.0)])
    x = x[np.abs(x) < 440].astype(np.float32)            # inside the finite range (no saturation question)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode_e4m3(x), ref)


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_is_the_hadamard_product(d):
    from scipy.linalg import hadamard
    rng = np.random.default_rng(d)
    x = rng.integers(-50, 50, size=(7, d)).astype(np.float32)     # small integers: fp32 adds exact
    assert np.array_equal(fp8.fwht_f32(x).astype(np.float64), x.astype(np.float64) @ hadamard(d))


def test_rotation_is_orthogonal_and_keeps_scores():
    rng = np.random.default_rng(1)
    signs = rng.choice([-1.0, 1.0], size=128)
    M = fp8.rotation_matrix(signs)
    assert np.abs(M @ M.T - np.eye(128)).max() < 1e-14
    q, k = rng.standard_normal((5, 128)), rng.standard_normal((9, 128))
    assert np.abs((q @ M) @ (k @ M).T - q @ k.T).max() < 1e-12


def _bits(shape, seed, sigma=1.0):
    return inputs.normal_bf16(seed, shape, sigma)


@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_error_is_within_half_a_step(rotate):
    x = _bits((2, 3, 50, 64), 11)
    signs = np.random.default_rng(2).choice([-1.0, 1.0], size=64) if rotate else None
    codes, descale = fp8.quantize(x, signs)
    target = oracle.bf16_bits_to_f64(x)
    if rotate:
        target = target @ fp8.rotation_matrix(signs)
    deq = fp8.dequantize(codes, descale)
    # relative half step 2^-4 for normal codes, absolute 2^-10 * step scale below 2^-6
    unit = descale.astype(np.float64)[:, :, None, None] * (math.sqrt(64) if rotate else 1.0)
    bound = np.maximum(np.abs(target) * 2.0 ** -4, unit * 2.0 ** -10 / (math.sqrt(64) if rotate else 1.0))
    assert np.all(np.abs(deq - target) <= bound * (1 + 1e-6) + 1e-12)
    # the largest magnitude of each head maps to 448
    assert np.all(np.abs(fp8.decode_e4m3(codes)).reshape(2, 3, -1).max(axis=2) == 448.0)


def test_quantize_zero_head_and_transposed_layout():
    x = _bits((1, 2, 37, 64), 12)
    x[0, 1] = 0
    codes, descale = fp8.quantize(x)
    assert np.all(codes[0, 1] == 0) and descale[0, 1] == 1.0
    t, descale_t = fp8.quantize(x, transpose=True)
    assert t.shape == (1, 2, 64, 48) and np.array_equal(descale_t, descale)
    assert np.array_equal(t[:, :, :, :37], codes.transpose(0, 1, 3, 2)) and np.all(t[:, :, :, 37:] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_attention_equals_the_bf16_oracle_on_shared_values(causal):
    # codes whose values bf16 holds exactly, descale 1: both oracles see the same numbers
    rng = np.random.default_rng(4)
    B, H, N, d = 1, 2, 45, 64
    pick = lambda shape: fp8.encode_e4m3(rng.standard_normal(shape))
    q8, k8, v8 = pick((B, H, N, d)), pick((B, H, N, d)), pick((B, H, N, d))
    ones = np.ones((B, H), dtype=np.float32)
    vt8 = np.zeros((B, H, d, 48), dtype=np.uint8)
    vt8[:, :, :, :N] = v8.transpose(0, 1, 3, 2)
    O1, L1 = fp8.attention_fp8(q8, k8, vt8, ones, ones, ones, 0.125, causal, nk=N)
    as_bf16 = lambda c: inputs.fp32_to_bf16_bits(fp8.decode_e4m3(c).astype(np.float32))
    O2, L2 = oracle.attention_rows(as_bf16(q8), as_bf16(k8), as_bf16(v8), 0.125, causal)
    assert np.abs(O1 - O2).max() < 1e-12 and np.abs(L1 - L2).max() < 1e-12


def test_incoherent_processing_reduces_error_with_outlier_channels():
    # a few channels of Q and K 30x larger: without the rotation those channels
    # set the scale and the rest lose precision ("9.4 FlashAttention 与 FlashMLA" 9.4.4)
    B, H, N, d = 1, 2, 128, 64
    rng = np.random.default_rng(5)
    q = oracle.bf16_bits_to_f64(_bits((B, H, N, d), 31))
    k = oracle.bf16_bits_to_f64(_bits((B, H, N, d), 32))
    v = _bits((B, H, N, d), 33)
    for ch in (3, 17, 40):
        q[..., ch] *= 30.0
        k[..., ch] *= 30.0
    qb = inputs.fp32_to_bf16_bits(q.astype(np.float32))
    kb = inputs.fp32_to_bf16_bits(k.astype(np.float32))
    scale = 1.0 / math.sqrt(d) / 8
    O_ref, _ = oracle.attention_rows(qb, kb, v, scale, False)
    signs = rng.choice([-1.0, 1.0], size=d)
    errs = []
    for s in (None, signs):
        q8, dq = fp8.quantize(qb, s)
        k8, dk = fp8.quantize(kb, s)
        vt8, dv = fp8.quantize(v, transpose=True)
        O, _ = fp8.attention_fp8(q8, k8, vt8, dq, dk, dv, scale, False, nk=N)
        errs.append(np.abs(O - O_ref).mean())
    assert errs[1] < 0.7 * errs[0], errs


MUTATIONS = {
    "exponent bias 8": ("2.0 ** (e - 7)", "2.0 ** (e - 8)"),
    "subnormal scale 2^-7": ("2.0 ** (1 - 7)", "2.0 ** (0 - 7)"),
    "ties to the lower code": ("score = cand * (1 + even[None, :])", "score = cand * 1"),
    "rounds toward zero": ("dist = np.abs(a[:, None] - mags[None, :])",
                           "dist = np.where(mags[None, :] <= a[:, None], a[:, None] - mags[None, :], np.inf)"),
    "sign dropped": ("out[c0:c0 + chunk] = code | (neg.astype(np.uint8) << 7)", "out[c0:c0 + chunk] = code"),
    "butterfly reversed": ("np.stack([a + b, a - b], axis=-2)", "np.stack([a + b, b - a], axis=-2)"),
    "1/sqrt(d) not folded": ("descale * np.float32(1.0 / math.sqrt(d))", "descale * np.float32(1.0)"),
    "amax maps to 240": ("np.float32(E4M3_MAX) / np.where", "np.float32(240.0) / np.where"),
    "V left transposed": ("v = v[:, :, :, :n].transpose(0, 1, 3, 2)", "v = v[:, :, :n, :]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name):
    """Each mistake, planted in a copy of oracle/fp8.py, fails at least one
    of the facts the pins above check."""
    import importlib.util
    import os
    import types
    old, new = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fp8.py"), encoding="utf-8").read()
    assert src.count(old) == 1, name
    mod = types.ModuleType("fp8_mutant")
    mod.__dict__["__name__"] = "oracle.fp8_mutant"
    mod.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(old, new), "fp8_mutant.py", "exec"), mod.__dict__)
    m = mod

    def facts():
        yield m.decode_e4m3(0x01) == 2.0 ** -9 and m.decode_e4m3(0x38) == 1.0 and m.decode_e4m3(0x7E) == 448.0
        codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
        yield np.array_equal(m.encode_e4m3(m.decode_e4m3(codes)), codes)
        mags = m.E4M3[:127]
        mids = 0.5 * (mags[:-1] + mags[1:])
        lo = np.arange(126)
        yield np.array_equal(m.encode_e4m3(mids), np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8))
        yield m.encode_e4m3(np.array([1e6]))[0] == 0x7E
        from scipy.linalg import hadamard
        xi = np.arange(-32, 32, dtype=np.float32).reshape(1, 64)
        yield np.array_equal(m.fwht_f32(xi).astype(np.float64), xi.astype(np.float64) @ hadamard(64))
        x = _bits((1, 2, 40, 64), 11)
        signs = np.random.default_rng(2).choice([-1.0, 1.0], size=64)
        codes, descale = m.quantize(x, signs)
        target = oracle.bf16_bits_to_f64(x) @ fp8.rotation_matrix(signs)
        yield np.all(np.abs(m.dequantize(codes, descale) - target) <= np.abs(target) * 2.0 ** -4 + 1e-3)
        rng = np.random.default_rng(4)
        pick = lambda shape: fp8.encode_e4m3(rng.standard_normal(shape))
        q8, k8, v8 = pick((1, 1, 20, 64)), pick((1, 1, 20, 64)), pick((1, 1, 20, 64))
        ones = np.ones((1, 1), dtype=np.float32)
        vt8 = np.zeros((1, 1, 64, 32), dtype=np.uint8)
        vt8[:, :, :, :20] = v8.transpose(0, 1, 3, 2)
        try:
            O1, _ = m.attention_fp8(q8, k8, vt8, ones, ones, ones, 0.125, False, nk=20)
        except (ValueError, IndexError):
            yield False
            return
        as_bf16 = lambda c: inputs.fp32_to_bf16_bits(fp8.decode_e4m3(c).astype(np.float32))
        O2, _ = oracle.attention_rows(as_bf16(q8), as_bf16(k8), as_bf16(v8), 0.125, False)
        yield np.abs(O1 - O2).max() < 1e-12

    assert not all(facts()), f"planted mistake not caught: {name}"
