"""GPU parity of the E4M3 path: fa_quantize_fp8 against the oracle's quantiser
(bit-exact codes and scales), and fa_fwd_fp8 against exact attention on the
dequantised codes (oracle/fp8.py), both fed the oracle's codes.

Tolerance of the forward (the pages give none for FP8; derived from the
arithmetic): the kernel rounds each weight p_k of P V to E4M3 (relative error
delta_k, |delta_k| <= 2^-4, zero-mean under round-to-nearest-even) and
normalises by the sum of the rounded weights, so with w_k = p_k / sum p
    O_kernel - O  ~=  sum_k w_k delta_k (v_k - O),
a sum of independent zero-mean terms of variance at most
    sigma^2 = (2^-8 / 3) * sum_k w_k^2 (v_k - O)^2
per output element, plus the bf16 rounding of O (2^-9 |O|).  Small weights
fall into E4M3's subnormal range, where the step is 2^-9 absolute: the
kernel scales P so that its row maximum is at least 2^4, so such a weight
moves by at most 2^-10 / 2^4 = 2^-14 * w_max (rounded, or flushed to zero),
which adds at most (2^-14 w_max)^2 * sum_k (v_k - O)^2.  The test checks that
the errors scaled by the total spread have mean square <= 1.5 and stay within
7 spreads, and that LSE (computed from the unrounded sums) is within 1e-3.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from oracle import fp8  # noqa: E402
from exact_attention_28_gb300 import inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_28_gb300 import build, ops as _ops
    build.build()
    _ops.load_library()
    return _ops


def bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def u8_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def signs_for(d, seed):
    return np.random.default_rng(seed).choice([-1.0, 1.0], size=d).astype(np.float32)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("transpose", [False, True])
def test_quantize_is_bit_exact(ops, d, rotate, transpose):
    for N, sigma in ((300, 1.0), (1000, 3.0), (64, 0.01)):
        x = inputs.normal_bf16(700 + N + d, (2, 3, N, d), sigma)
        signs = signs_for(d, N) if rotate else None
        codes, descale = fp8.quantize(x, signs, transpose)
        g_codes, g_descale = ops.quantize_fp8(bf16_dev(x), None if signs is None else torch.from_numpy(signs).cuda(),
                                              transpose)
        ops.check_device_status()
        assert np.array_equal(g_codes.cpu().numpy(), codes), (N, sigma)
        assert np.array_equal(g_descale.cpu().numpy().view(np.uint32), descale.view(np.uint32)), (N, sigma)


def test_quantize_zero_head(ops):
    x = inputs.normal_bf16(9, (1, 2, 100, 128))
    x[0, 0] = 0
    g_codes, g_descale = ops.quantize_fp8(bf16_dev(x))
    ops.check_device_status()
    assert int(g_codes[0, 0].abs().sum()) == 0 and float(g_descale[0, 0]) == 1.0


def exact_weights(Q, K, V, scale, causal, rows):
    """w (softmax weights) and O for the listed flat rows, fp64 (test-side, for the spread)."""
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    out_w, out_o, vis_v = [], [], []
    for r in rows:
        bh, i = divmod(int(r), Nq)
        b, h = divmod(bh, H)
        n = min(Nk, i + 1) if causal else Nk
        s = scale * (K[b, h, :n] @ Q[b, h, i])
        w = np.exp(s - s.max())
        w /= w.sum()
        out_w.append(w)
        vis_v.append(V[b, h, :n])
        out_o.append(w @ V[b, h, :n])
    return out_w, vis_v, np.array(out_o)


def check_fp8_forward(ops, q_bits, k_bits, v_bits, scale, causal, signs=None, nrows=None, tag=""):
    B, H, Nq, d = q_bits.shape
    Nk = k_bits.shape[2]
    q8, dq = fp8.quantize(q_bits, signs)
    k8, dk = fp8.quantize(k_bits, signs)
    vt8, dv = fp8.quantize(v_bits, transpose=True)
    o, lse = ops.fa_fwd_fp8(u8_dev(q8), u8_dev(k8), u8_dev(vt8), torch.from_numpy(dq).cuda(),
                            torch.from_numpy(dk).cuda(), torch.from_numpy(dv).cuda(), scale=scale, causal=causal)
    ops.check_device_status()
    total = B * H * Nq
    rows = np.arange(total) if nrows is None or nrows >= total else \
        np.random.default_rng(1).choice(total, nrows, replace=False)
    O_ref, L_ref = fp8.attention_fp8(q8, k8, vt8, dq, dk, dv, scale, causal, nk=Nk, rows=rows)
    o = o.float().cpu().numpy().reshape(total, d)[rows].astype(np.float64)
    l = lse.cpu().numpy().reshape(total)[rows].astype(np.float64)
    assert np.abs(l - L_ref).max() <= 1e-3, f"{tag}: LSE {np.abs(l - L_ref).max():.3e}"
    Qh, Kh = fp8.dequantize(q8, dq), fp8.dequantize(k8, dk)
    Vh = fp8.dequantize(vt8, dv, transposed=True, n=Nk)
    ws, vs, O_chk = exact_weights(Qh, Kh, Vh, float(np.float32(scale)), causal, rows)
    assert np.abs(O_chk - O_ref).max() < 1e-9                       # same definition, two routes
    var = np.array([(w[:, None] ** 2 * (v - o_row) ** 2).sum(axis=0) for w, v, o_row in zip(ws, vs, O_ref)])
    sub = np.array([(2.0 ** -14 * w.max()) ** 2 * ((v - o_row) ** 2).sum(axis=0) for w, v, o_row in zip(ws, vs, O_ref)])
    spread = np.sqrt(var * 2.0 ** -8 / 3 + sub + (2.0 ** -9 * np.abs(O_ref)) ** 2 + 1e-10)
    z = (o - O_ref) / spread
    assert np.mean(z ** 2) <= 1.5 and np.abs(z).max() <= 7.0, \
        f"{tag}: mean z^2 {np.mean(z ** 2):.3f} max |z| {np.abs(z).max():.2f} max err {np.abs(o - O_ref).max():.3e}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 300, 333), (2, 2, 512, 512), (1, 1, 128, 128), (1, 3, 77, 1000)])
def test_fp8_forward_parity(ops, causal, shape):
    B, H, Nq, Nk = shape
    q, k, v = inputs.custom_inputs(4000 + Nq + Nk, B, H, Nq, Nk, 128)
    check_fp8_forward(ops, q, k, v, 1 / math.sqrt(128), causal, tag=f"{shape} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_rotated_inputs(ops, causal):
    q, k, v = inputs.custom_inputs(4100, 2, 2, 256, 384, 128, sigma=(2.0, 2.0, 1.0))
    check_fp8_forward(ops, q, k, v, 1 / math.sqrt(128), causal, signs=signs_for(128, 5), tag="rotated")


def test_fp8_forward_bench_shape_sampled(ops):
    w = inputs.WORKLOADS["b2_h16_n4096_d128"]
    q, k, v, scale = inputs.make_inputs(w)
    check_fp8_forward(ops, q, k, v, scale, False, signs=signs_for(128, 6), nrows=1024, tag="b2_h16_n4096")


def test_fp8_forward_causal_long_sampled(ops):
    q, k, v = inputs.custom_inputs(4200, 1, 4, 4096, 4096, 128, sigma=(2.0, 2.0, 1.0))
    check_fp8_forward(ops, q, k, v, 1 / math.sqrt(128), True, nrows=1024, tag="causal 4096")


def test_fp8_scale_sign_and_descale_are_applied(ops):
    q, k, v = inputs.custom_inputs(4300, 1, 2, 130, 200, 128)
    check_fp8_forward(ops, q, k, v, -0.3, False, tag="negative scale")
    check_fp8_forward(ops, q, k, v, 0.0, True, tag="zero scale")


def test_end_to_end_rotation_lowers_error_with_outlier_channels(ops):
    # quantise on the GPU, attend on the GPU, compare with exact attention on
    # the original bf16 inputs: the rotation must reduce the error
    B, H, N, d = 1, 4, 512, 128
    q = oracle.bf16_bits_to_f64(inputs.normal_bf16(4400, (B, H, N, d)))
    k = oracle.bf16_bits_to_f64(inputs.normal_bf16(4401, (B, H, N, d)))
    v = inputs.normal_bf16(4402, (B, H, N, d))
    for ch in (5, 77, 100):
        q[..., ch] *= 30.0
        k[..., ch] *= 30.0
    qb = inputs.fp32_to_bf16_bits(q.astype(np.float32))
    kb = inputs.fp32_to_bf16_bits(k.astype(np.float32))
    scale = 1 / math.sqrt(d) / 8
    O_ref, _ = oracle.attention_rows(qb, kb, v, scale, False)
    signs = torch.from_numpy(signs_for(d, 8)).cuda()
    errs = []
    for s in (None, signs):
        q8, dq = ops.quantize_fp8(bf16_dev(qb), s)
        k8, dk = ops.quantize_fp8(bf16_dev(kb), s)
        vt8, dv = ops.quantize_fp8(bf16_dev(v), transpose=True)
        o, _ = ops.fa_fwd_fp8(q8, k8, vt8, dq, dk, dv, scale=scale)
        ops.check_device_status()
        errs.append(np.abs(o.float().cpu().numpy().reshape(-1, d) - O_ref).mean())
    assert errs[1] < 0.7 * errs[0], errs
