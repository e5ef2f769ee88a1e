"""Pins for the backward oracle: finite differences, the blocked section-7.2
recomputation, and closed forms."""
import math

import numpy as np
import pytest

import oracle
from oracle import backward


def rand(shape, seed, s=1.0):
    return np.random.default_rng(seed).normal(0, s, shape)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk,d", [(3, 5, 4), (6, 6, 3), (5, 2, 2)])
def test_gradients_match_central_differences(causal, Nq, Nk, d):
    # L = sum(dO * O(Q, K, V)); its numerical gradient must equal the oracle's.
    Q, K, V, dO = rand((Nq, d), 1), rand((Nk, d), 2), rand((Nk, d), 3), rand((Nq, d), 4)
    scale = 0.7
    dQ, dK, dV = backward.attention_backward(Q, K, V, dO, scale, causal)
    loss = lambda q, k, v: float(np.sum(dO * backward.attention_forward(q, k, v, scale, causal)[0]))
    h = 1e-6
    for X, G, which in ((Q, dQ, 0), (K, dK, 1), (V, dV, 2)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (up - loss(*args)) / (2 * h)
        assert np.max(np.abs(num - G)) < 1e-7, which


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Br,Bc", [(1, 1), (2, 3), (4, 4), (7, 5)])
def test_blocked_recomputation_equals_definition(causal, Br, Bc):
    Q, K, V, dO = rand((9, 6), 5), rand((9, 6), 6), rand((9, 6), 7), rand((9, 6), 8)
    ref = backward.attention_backward(Q, K, V, dO, 0.4, causal)
    got = backward.blocked_backward(Q, K, V, dO, 0.4, causal, Br, Bc)
    for a, b in zip(ref, got):
        assert np.max(np.abs(a - b)) < 1e-12


def test_forward_used_by_the_backward_matches_the_c_oracle():
    # the fp64 forward here agrees with the pinned C oracle on bf16-exact inputs
    from exact_attention_28_gb300.inputs import custom_inputs
    q, k, v = custom_inputs(5, 1, 1, 7, 11, 8)
    f = oracle.bf16_bits_to_f64
    O_ref, L_ref = oracle.attention(q, k, v, 0.3, True, nthreads=1)
    O, _, _, lse = backward.attention_forward(f(q)[0, 0], f(k)[0, 0], f(v)[0, 0], float(np.float32(0.3)), True)
    assert np.max(np.abs(O - O_ref[0, 0])) < 1e-13 and np.max(np.abs(lse - L_ref[0, 0])) < 1e-13


def test_closed_forms():
    Q, K, V = rand((4, 3), 9), rand((5, 3), 10), rand((5, 3), 11)
    # zero upstream gradient: zero gradients
    for g in backward.attention_backward(Q, K, V, np.zeros((4, 3)), 0.5, False):
        assert np.all(g == 0)
    # dV = P^T dO: with dO = e_0 (one row of ones at query 0), dV_j = P_0j * 1
    dO = np.zeros((4, 3)); dO[0] = 1.0
    _, _, dV = backward.attention_backward(Q, K, V, dO, 0.5, False)
    S = 0.5 * Q @ K.T
    P0 = np.exp(S[0] - S[0].max()); P0 /= P0.sum()
    assert np.max(np.abs(dV - P0[:, None] * np.ones((1, 3)))) < 1e-15
    # adding a constant to every V row leaves dQ, dK unchanged (softmax weights sum to 1)
    dO = rand((4, 3), 12)
    a = backward.attention_backward(Q, K, V, dO, 0.5, True)
    b = backward.attention_backward(Q, K, V + 3.0, dO, 0.5, True)
    assert np.max(np.abs(a[0] - b[0])) < 1e-12 and np.max(np.abs(a[1] - b[1])) < 1e-12
    # causal: keys after the last query get no gradient when Nq < Nk
    dQ, dK, dV = backward.attention_backward(Q, K, V, dO, 0.5, True)
    assert np.all(dK[4:] == 0) and np.all(dV[4:] == 0)


def fd_gradients(Q, K, V, dO, scale, causal, h=1e-6):
    loss = lambda q, k, v: float(np.sum(dO * backward.attention_forward(q, k, v, scale, causal)[0]))
    out = []
    for which, X in enumerate((Q, K, V)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (up - loss(*args)) / (2 * h)
        out.append(num)
    return out


def test_planted_mistakes_are_caught_by_finite_differences():
    Q, K, V, dO = rand((4, 3), 21), rand((5, 3), 22), rand((5, 3), 23), rand((4, 3), 24)
    scale = 0.6
    fd = fd_gradients(Q, K, V, dO, scale, False)

    def grads(variant):
        S = scale * Q @ K.T
        P = np.exp(S - S.max(axis=1, keepdims=True)); P /= P.sum(axis=1, keepdims=True)
        dP = dO @ V.T
        dS = P * (dP - np.sum(dP * P, axis=1, keepdims=True))
        dQ, dK, dV = scale * dS @ K, scale * dS.T @ Q, P.T @ dO
        if variant == "no rowsum term":
            dS = P * dP; dQ, dK = scale * dS @ K, scale * dS.T @ Q
        if variant == "scale dropped in dQ":
            dQ = dS @ K
        if variant == "unnormalised P in dV":
            dV = np.exp(S - S.max(axis=1, keepdims=True)).T @ dO
        return dQ, dK, dV

    for variant in ["no rowsum term", "scale dropped in dQ", "unnormalised P in dV"]:
        g = grads(variant)
        assert max(np.max(np.abs(a - b)) for a, b in zip(g, fd)) > 1e-3, variant
    assert max(np.max(np.abs(a - b)) for a, b in zip(grads("none"), fd)) < 1e-7
