"""Pins for the oracle: checks against what the pages and the mathematics fix.

None of these re-derives the oracle from itself.  They use closed forms, a
library softmax/logsumexp on tiny cases, invariants the pages prove, a second
independent algorithm (the pages' blocked/online recurrences in numpy against
the three-pass C code), and brute force over every block split.  The last
section plants plausible mistakes into copies of the oracle and checks that
each one is caught by at least one pin.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
from scipy.special import expit, logsumexp, softmax

import oracle
from oracle import online
from exact_attention_28_gb300.inputs import bf16_bits_to_fp32, custom_inputs, fp32_to_bf16_bits

HERE = os.path.dirname(os.path.abspath(__file__))


def bits(x):
    """fp32-representable values -> bf16 bits (exact for the values used here)."""
    b = fp32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    assert np.array_equal(bf16_bits_to_fp32(b), np.asarray(x, dtype=np.float32)), "value not bf16-exact"
    return b


def f64(b):
    return oracle.bf16_bits_to_f64(b)


def run(lib, Q, K, V, scale, causal):
    return oracle.attention(Q, K, V, scale, causal, nthreads=2, lib=lib)


# ---------------------------------------------------------------------------
# Pin functions for the C three-pass oracle.  Each takes the library so the
# mutation tests below can run them against planted mistakes.
# ---------------------------------------------------------------------------

def pin_two_key_closed_form(lib):
    # q = [1], keys [0] and [2], scale 1: p = (1, e^2) / (1 + e^2) -> a logistic.
    Q = bits([[[[1.0]]]])
    K = bits([[[[0.0], [2.0]]]])
    V = bits([[[[1.0], [3.0]]]])
    O, L = run(lib, Q, K, V, 1.0, False)
    p1 = expit(2.0)
    assert abs(O[0, 0, 0, 0] - ((1 - p1) * 1.0 + p1 * 3.0)) < 1e-15
    assert abs(L[0, 0, 0] - math.log1p(math.exp(2.0))) < 1e-15
    # scale 0.5 halves the logit
    O, L = run(lib, Q, K, V, 0.5, False)
    assert abs(O[0, 0, 0, 0] - (1.0 + 2.0 * expit(1.0))) < 1e-15
    assert abs(L[0, 0, 0] - math.log1p(math.exp(1.0))) < 1e-15


def pin_identity_values_give_softmax(lib, causal):
    # With V = I (d = Nk), O is the probability matrix P itself; compare it to
    # scipy's softmax of the scaled scores and LSE to scipy's logsumexp.
    Nq = Nk = 12
    q, k, _ = custom_inputs(77, 1, 2, Nq, Nk, Nk)
    V = bits(np.broadcast_to(np.eye(Nk, dtype=np.float32), (1, 2, Nk, Nk)).copy())
    scale = float(np.float32(0.37))
    O, L = run(lib, q, k, V, scale, causal)
    S = np.einsum("bhid,bhjd->bhij", f64(q), f64(k)) * scale
    if causal:
        S = np.where(np.tril(np.ones((Nq, Nk), dtype=bool)), S, -np.inf)
    P = softmax(S, axis=-1)
    assert np.max(np.abs(O - P)) < 1e-14
    assert np.max(np.abs(O.sum(-1) - 1.0)) < 1e-14        # rows of P sum to 1
    assert np.max(np.abs(L - logsumexp(S, axis=-1))) < 1e-13
    if causal:
        assert np.all(O[..., np.triu_indices(Nq, 1)[0], np.triu_indices(Nq, 1)[1]] == 0.0)


def pin_equal_scores(lib, causal):
    # Q = 0: every visible score is 0, O_i is the mean of visible V rows and
    # LSE_i = ln |J_i| (ln Nk, or ln(i+1) under causal).
    B, H, Nq, Nk, d = 1, 2, 9, 13, 8
    _, k, v = custom_inputs(5, B, H, Nq, Nk, d)
    Q = np.zeros((B, H, Nq, d), dtype=np.uint16)
    O, L = run(lib, Q, k, v, 0.125, causal)
    Vf = f64(v)
    for i in range(Nq):
        n = min(Nk, i + 1) if causal else Nk
        assert np.max(np.abs(O[:, :, i] - Vf[:, :, :n].mean(axis=2))) < 1e-14
        assert np.max(np.abs(L[:, :, i] - math.log(n))) < 1e-14


def pin_dominant_logit(lib):
    # One key with a margin >= 40 over all others picks its V row:
    # |O_i - v_j*| <= Nk e^{-40} max|v|, LSE_i = s_j* + O(Nk e^{-40}).
    Nk, d = 16, 4
    jstar = 11
    Kx = np.zeros((1, 1, Nk, d), dtype=np.float32)
    Kx[0, 0, jstar, 0] = 64.0
    Qx = np.zeros((1, 1, 3, d), dtype=np.float32)
    Qx[0, 0, :, 0] = [1.0, 2.0, 4.0]
    _, _, v = custom_inputs(9, 1, 1, 3, Nk, d)
    scale = 1.0
    O, L = run(lib, bits(Qx), bits(Kx), v, scale, False)
    Vf = f64(v)
    for i, qv in enumerate([1.0, 2.0, 4.0]):
        s_star = 64.0 * qv
        bound = Nk * math.exp(-s_star) * np.max(np.abs(Vf))
        assert np.max(np.abs(O[0, 0, i] - Vf[0, 0, jstar])) <= bound + 1e-15
        assert abs(L[0, 0, i] - s_star) <= Nk * math.exp(-s_star) + 1e-13


def pin_permutation(lib):
    # Non-causal attention does not depend on the order of the (k_j, v_j) pairs.
    q, k, v = custom_inputs(31, 2, 2, 7, 19, 16)
    perm = np.random.default_rng(3).permutation(19)
    O1, L1 = run(lib, q, k, v, 0.25, False)
    O2, L2 = run(lib, q, k[:, :, perm], v[:, :, perm], 0.25, False)
    assert np.max(np.abs(O1 - O2)) < 1e-14 and np.max(np.abs(L1 - L2)) < 1e-14


def pin_causal_sees_only_the_past(lib):
    # Under causal masking, row i ignores keys j > i (top-left alignment): row 0
    # is exactly v_0 with LSE s_00, and rewriting keys/values after i changes
    # nothing in row i.
    q, k, v = custom_inputs(41, 1, 1, 10, 10, 8)
    scale = float(np.float32(0.3))
    O1, L1 = run(lib, q, k, v, scale, True)
    assert np.array_equal(O1[0, 0, 0], f64(v)[0, 0, 0])
    s00 = scale * float(np.dot(f64(q)[0, 0, 0], f64(k)[0, 0, 0]))
    assert abs(L1[0, 0, 0] - s00) < 1e-13
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 6:] = bits(np.full((1, 1, 4, 8), 8.0, dtype=np.float32))
    v2[:, :, 6:] = bits(np.full((1, 1, 4, 8), -100.0, dtype=np.float32))
    O2, L2 = run(lib, q, k2, v2, scale, True)
    assert np.array_equal(O1[0, 0, :6], O2[0, 0, :6]) and np.array_equal(L1[0, 0, :6], L2[0, 0, :6])
    assert not np.allclose(O1[0, 0, 6:], O2[0, 0, 6:])


def pin_scale_homogeneity(lib):
    # scale * <2q, k> == (2 scale) * <q, k>: doubling Q (exact in bf16) equals
    # doubling the scale.
    q, k, v = custom_inputs(51, 1, 2, 5, 6, 8)
    q2 = bits(2.0 * bf16_bits_to_fp32(q))
    O1, L1 = run(lib, q2, k, v, 0.25, False)
    O2, L2 = run(lib, q, k, v, 0.5, False)
    assert np.max(np.abs(O1 - O2)) < 1e-14 and np.max(np.abs(L1 - L2)) < 1e-14


def pin_rows_and_sampling(lib):
    # Rows computed one by one equal the same rows of the full computation,
    # and sampled rows land at the right (batch, head, query) position.
    q, k, v = custom_inputs(61, 2, 3, 11, 9, 8)
    O, L = run(lib, q, k, v, 0.2, True)
    rows = np.array([0, 5, 11 * 3 + 4, 2 * 3 * 11 - 1])
    Os, Ls = oracle.attention_rows(q, k, v, 0.2, True, rows=rows, nthreads=3, lib=lib)
    assert np.array_equal(Os, O.reshape(-1, 8)[rows]) and np.array_equal(Ls, L.reshape(-1)[rows])


def pin_against_blocked(lib, causal, Nq, Nk):
    # Two independent algorithms (three-pass C vs the pages' blocked online
    # recurrence in numpy) agree.
    q, k, v = custom_inputs(71 + Nq + 100 * Nk, 1, 1, Nq, Nk, 8)
    scale = float(np.float32(0.35))
    O, L = run(lib, q, k, v, scale, causal)
    Ob, _, _, lse = online.blocked_attention(f64(q)[0, 0], f64(k)[0, 0], f64(v)[0, 0], scale, causal, 3, 4)
    assert np.max(np.abs(O[0, 0] - Ob)) < 1e-12 and np.max(np.abs(L[0, 0] - lse)) < 1e-12


ALL_PINS = [
    pin_two_key_closed_form,
    lambda lib: pin_identity_values_give_softmax(lib, False),
    lambda lib: pin_identity_values_give_softmax(lib, True),
    lambda lib: pin_equal_scores(lib, False),
    lambda lib: pin_equal_scores(lib, True),
    pin_dominant_logit,
    pin_permutation,
    pin_causal_sees_only_the_past,
    pin_scale_homogeneity,
    pin_rows_and_sampling,
    lambda lib: pin_against_blocked(lib, True, 10, 10),
    lambda lib: pin_against_blocked(lib, False, 7, 13),
]


@pytest.mark.parametrize("pin", range(len(ALL_PINS)))
def test_c_oracle_pins(pin):
    ALL_PINS[pin](oracle.load())


def test_argument_errors():
    lib = oracle.load()
    q, k, v = custom_inputs(1, 1, 1, 4, 4, 8)
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, k, v, 1.0, False, rows=[16], lib=lib)   # row out of range
    with pytest.raises(TypeError):
        oracle.attention_rows(q.astype(np.float32), k, v, 1.0, False, lib=lib)


# ---------------------------------------------------------------------------
# Online softmax, block recurrence, blocked attention, merge.
# ---------------------------------------------------------------------------

def test_three_pass_softmax_matches_scipy():
    rng = np.random.default_rng(0)
    for n in [1, 2, 7, 64]:
        x = rng.normal(0, 30, n)
        assert np.max(np.abs(online.three_pass_softmax(x) - softmax(x))) < 1e-15
    # the overflow case the page starts from: elements around 1000
    x = np.array([1000.0, 999.0, 990.0])
    y = online.three_pass_softmax(x)
    assert np.all(np.isfinite(y)) and abs(y.sum() - 1) < 1e-15


@pytest.mark.parametrize("spread", [1.0, 30.0, 1000.0])
def test_online_softmax_1d_equals_three_pass(spread):
    rng = np.random.default_rng(int(spread))
    for n in [1, 2, 3, 17, 100]:
        x = rng.normal(0, spread, n)
        y, m, l, steps = online.online_softmax_1d(x, trace=True)
        ref = online.three_pass_softmax(x)
        assert np.max(np.abs(y - ref) / np.maximum(ref, 1e-300)) < 1e-13
        assert m == np.max(x)
        # invariant after every element: l_k = sum_{j<=k} exp(x_j - m_k)
        for kk, (mk, lk) in enumerate(steps):
            assert mk == np.max(x[: kk + 1])
            direct = sum(math.exp(xj - mk) for xj in x[: kk + 1])
            assert abs(lk - direct) <= 1e-13 * direct


def test_online_softmax_page_listing_bug_is_caught():
    # Planted mistake: the section 1.3 listing's "l += exp(m - val)" on a new
    # maximum (adds where the recurrence multiplies).  The equality pin fails.
    def buggy(x):
        m, l = -math.inf, 0.0
        for v in x:
            if v > m:
                l += math.exp(m - v)
                m = v
            l += math.exp(v - m)
        return np.array([math.exp(v - m) / l for v in x])
    x = np.array([0.0, 1.0, 3.0, 2.0])
    assert np.max(np.abs(buggy(x) - online.three_pass_softmax(x))) > 1e-3


@pytest.mark.parametrize("block", [1, 2, 5, 16])
def test_block_recurrence_invariant(block):
    rng = np.random.default_rng(block)
    x = rng.normal(0, 8, 37)
    m, l, steps = online.online_softmax_blocks(x, block)
    for kk, (mk, lk) in enumerate(steps):
        seen = x[: min(len(x), (kk + 1) * block)]
        assert mk == np.max(seen)
        direct = float(np.sum(np.exp(seen - mk)))
        assert abs(lk - direct) <= 1e-13 * direct          # l^(k) = sum exp(x_j - m^(k))
    assert abs(m + math.log(l) - logsumexp(x)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 5), (5, 1), (6, 6), (9, 4), (4, 11), (17, 17)])
def test_blocked_every_split_equals_three_pass(causal, Nq, Nk):
    """Brute force over every (Br, Bc) in [1..Nq] x [1..Nk]."""
    q, k, v = custom_inputs(1000 + 31 * Nq + Nk, 1, 1, Nq, Nk, 4)
    scale = float(np.float32(0.5))
    O, L = oracle.attention(q, k, v, scale, causal, nthreads=1)
    Q, K, V = f64(q)[0, 0], f64(k)[0, 0], f64(v)[0, 0]
    for Br in range(1, Nq + 1):
        for Bc in range(1, Nk + 1):
            Ob, l, m, lse = online.blocked_attention(Q, K, V, scale, causal, Br, Bc)
            assert np.max(np.abs(Ob - O[0, 0])) < 1e-12, (Br, Bc)
            assert np.max(np.abs(lse - L[0, 0])) < 1e-12, (Br, Bc)
            assert np.max(np.abs(m + np.log(l) - lse)) == 0.0


def test_merge_of_any_split_equals_whole():
    q, k, v = custom_inputs(808, 1, 1, 3, 40, 8)
    scale = float(np.float32(0.4))
    O, L = oracle.attention(q, k, v, scale, False, nthreads=1)
    Q, K, V = f64(q)[0, 0], f64(k)[0, 0], f64(v)[0, 0]
    for i in range(3):
        for cuts in [(20,), (1,), (39,), (7, 13, 31), tuple(range(1, 40))]:
            edges = [0, *cuts, 40]
            parts = [online.block_partial(Q[i], K[a:b], V[a:b], scale) for a, b in zip(edges, edges[1:])]
            o, m, l = online.merge_partials(parts)
            assert np.max(np.abs(o - O[0, 0, i])) < 1e-13
            assert abs(m + math.log(l) - L[0, 0, i]) < 1e-13
            # the merge is order independent (tree or sequential reduction)
            o2, m2, l2 = online.merge_partials(parts[::-1])
            assert np.max(np.abs(o2 - o)) < 1e-13


def test_wrong_merge_differs_and_page_constant():
    # Section 13.3's wrong merge keeps the first block's maximum; with block
    # maxima 10 and 20 it weighs the second block by exp(20 - 10) ~ 22026, the
    # number the page prints, and its result differs from the correct merge.
    golden = {}
    with open(os.path.join(HERE, "golden", "page_constants.txt"), encoding="utf-8") as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                name, value, _ = [s.strip() for s in line.split("|", 2)]
                golden.setdefault(name, value)
    assert round(math.exp(10)) == int(golden["exp10"])

    def wrong_merge(parts):
        m, l, o = parts[0]
        o = np.array(o, dtype=np.float64)
        for m_j, l_j, o_j in parts[1:]:
            l = l + l_j * np.exp(m_j - m)
            o = o + np.asarray(o_j) * np.exp(m_j - m)
        return o / l
    parts = [(10.0, 1.5, np.array([1.0, 2.0])), (20.0, 1.2, np.array([-3.0, 0.5]))]
    assert abs(math.exp(parts[1][0] - parts[0][0]) - 22026) < 1
    # In real arithmetic the stale-maximum merge gives the same ratio (both
    # numerator and denominator carry the same factor); what breaks is the
    # range: once the maxima differ by more than ~709 the factor overflows.
    right, _, _ = online.merge_partials(parts)
    assert np.max(np.abs(wrong_merge(parts) - right)) < 1e-12
    parts_big = [(0.0, 1.0, np.array([1.0])), (800.0, 1.0, np.array([2.0]))]
    with np.errstate(over="ignore", invalid="ignore"):
        bad = wrong_merge(parts_big)
    good, _, _ = online.merge_partials(parts_big)
    assert abs(good[0] - 2.0) < 1e-15 and not np.isfinite(bad).all()


# ---------------------------------------------------------------------------
# Planted mistakes in copies of the C oracle: each must fail some pin.
# ---------------------------------------------------------------------------

MUTATIONS = {
    "scale dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "max not subtracted in the sum": ("l += exp(s[j] - m);", "l += exp(s[j]);"),
    "causal off by one": ("if (jb->causal && i + 1 < nvis) nvis = i + 1;",
                          "if (jb->causal && i < nvis) nvis = i;"),
    "causal never applied": ("if (jb->causal && i + 1 < nvis)", "if (0 && i + 1 < nvis)"),
    "K used as the value operand": ("o[c] += p * widen_bf16(V[j * d + c]);",
                                    "o[c] += p * widen_bf16(K[j * d + c]);"),
    "keys read in reverse order": ("widen_bf16(K[j * d + c])", "widen_bf16(K[(nvis - 1 - j) * d + c])"),
    "log dropped from LSE": ("*lse = m + log(l);", "*lse = m + l;"),
    "log base 2 in LSE": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "bf16 widened with a wrong shift": ("(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    "wrong head stride for K/V": ("jb->K + bh * jb->Nk * jb->d", "jb->K + (bh / 2) * jb->Nk * jb->d"),
    "first key skipped": ("for (int64_t j = 0; j < nvis; ++j)\n        l += exp",
                          "for (int64_t j = 1; j < nvis; ++j)\n        l += exp"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attention.c"), encoding="utf-8").read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    mutated = tmp_path / "attention.c"
    mutated.write_text(src.replace(old, new), encoding="utf-8")
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(mutated), "-lm"], check=True)
    lib = oracle.load(str(so))
    caught = 0
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(lib)
        except (AssertionError, RuntimeError, ValueError, IndexError):
            caught += 1
    assert caught >= 1, f"no pin catches: {name}"


@pytest.mark.parametrize("tau", [0.0, 8 * math.log(2.0), 20.0])
@pytest.mark.parametrize("block", [1, 7, 128])
def test_lagged_reference_softmax_equals_logsumexp(tau, block):
    """The kernel's reading of the online softmax: the reference is raised only
    when a block maximum exceeds it by more than tau (alpha is exactly 1
    otherwise).  Any reference keeps l = sum exp(x - r), so r + ln l is the
    log-sum-exp, and every term stays below exp(tau)."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(int(tau * 10) + block)
    for x in (rng.standard_normal(1000) * 3, np.sort(rng.standard_normal(500) * 10),   # rising maxima
              np.linspace(50, -50, 300), np.array([0.0])):
        r, l, steps = online.online_softmax_lagged(x, block, tau)
        assert abs((r + math.log(l)) - logsumexp(x)) < 1e-12 * max(1.0, abs(logsumexp(x)))
        for k, (rk, lk, alpha) in enumerate(steps):   # the invariant at every block boundary
            seen = x[:min(len(x), (k + 1) * block)]
            assert abs(lk - np.sum(np.exp(seen - rk))) <= 1e-12 * lk
            assert np.max(seen) - rk <= tau + 1e-12
            if k > 0 and rk == steps[k - 1][0]:
                assert alpha == 1.0


def test_lagged_reference_with_a_dropped_rescale_is_caught():
    # planted mistake: raising the reference without rescaling the old sum
    x = np.sort(np.random.default_rng(9).standard_normal(400) * 8)
    r, l, _ = online.online_softmax_lagged(x, 16, 2.0)
    rr, ll = -math.inf, 0.0
    for start in range(0, len(x), 16):
        xb = x[start:start + 16]
        if np.max(xb) > rr + 2.0:
            rr = float(np.max(xb))                     # (alpha forgotten)
        ll = ll + float(np.sum(np.exp(xb - rr)))
    from scipy.special import logsumexp
    assert abs(r + math.log(l) - logsumexp(x)) < 1e-12
    assert abs(rr + math.log(ll) - logsumexp(x)) > 1e-3
