"""Backward of attention in fp64: the oracle for the gradient kernels.

TEST INFRASTRUCTURE ONLY (imported by the tests and the bench's CPU leg, never
by the product path).

Two independent routines, both following the pages' statement of the
gradients ("6. FlashAttention 分块逻辑" section 7.1; "9.4 FlashAttention 与
FlashMLA" section 9.4.3):

  S = scale Q K^T,  P = softmax(S) over the visible keys,  O = P V
  dV = P^T dO
  dP = dO V^T
  dS = P * (dP - rowsum(dP * P))
  dQ = scale dS K,   dK = scale dS^T Q

* ``attention_backward`` -- the definition above, per head, with numpy
  matrix products as steps.
* ``blocked_backward`` -- the per-block recomputation of section 7.2: for
  every (Q block, K/V block) pair, recompute S_ij, recover P_ij from the
  forward's saved row maximum m and sum l (P_ij = exp(S_ij - m_i) / l_i), and
  accumulate dV_j, dK_j and dQ_i block by block.
"""
from __future__ import annotations

import math

import numpy as np


def _visible(Nq, Nk, causal):
    if not causal:
        return np.ones((Nq, Nk), dtype=bool)
    return np.arange(Nk)[None, :] <= np.arange(Nq)[:, None]


def attention_forward(Q, K, V, scale, causal):
    """fp64 forward of one head (for the backward's own use): O, m, l, LSE."""
    S = scale * (Q @ K.T)
    S = np.where(_visible(Q.shape[0], K.shape[0], causal), S, -math.inf)
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])
    l = E.sum(axis=1)
    return (E / l[:, None]) @ V, m, l, m + np.log(l)


def attention_backward(Q, K, V, dO, scale, causal):
    """dQ, dK, dV of one head (fp64 arrays [N, d]) from the definition."""
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    S = scale * (Q @ K.T)
    vis = _visible(Q.shape[0], K.shape[0], causal)
    S = np.where(vis, S, -math.inf)
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    dV = P.T @ dO
    dP = dO @ V.T
    dS = P * (dP - np.sum(dP * P, axis=1, keepdims=True))
    return scale * (dS @ K), scale * (dS.T @ Q), dV


def blocked_backward(Q, K, V, dO, scale, causal, Br, Bc):
    """Section 7.2: block-pair recomputation from the saved m and l."""
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    Nq, Nk = Q.shape[0], K.shape[0]
    O, m, l, _ = attention_forward(Q, K, V, scale, causal)
    D = np.sum(dO * O, axis=1)                  # rowsum(dP * P) written as rowsum(dO * O)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for i0 in range(0, Nq, Br):
        i1 = min(Nq, i0 + Br)
        for j0 in range(0, Nk, Bc):
            j1 = min(Nk, j0 + Bc)
            if causal and j0 > i1 - 1:
                continue                         # block entirely above the diagonal
            Sij = scale * (Q[i0:i1] @ K[j0:j1].T)
            if causal:
                Sij = np.where(np.arange(j0, j1)[None, :] <= np.arange(i0, i1)[:, None], Sij, -math.inf)
            Pij = np.exp(Sij - m[i0:i1, None]) / l[i0:i1, None]
            dV[j0:j1] += Pij.T @ dO[i0:i1]
            dPij = dO[i0:i1] @ V[j0:j1].T
            dSij = Pij * (dPij - D[i0:i1, None])
            dQ[i0:i1] += scale * (dSij @ K[j0:j1])
            dK[j0:j1] += scale * (dSij.T @ Q[i0:i1])
    return dQ, dK, dV


def backward_heads(Q, K, V, dO, scale, causal):
    """Backward over [B, H, N, d] fp64 arrays, head by head."""
    B, H = Q.shape[:2]
    dQ, dK, dV = np.empty_like(Q), np.empty_like(K), np.empty_like(V)
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h] = attention_backward(Q[b, h], K[b, h], V[b, h], dO[b, h], scale, causal)
    return dQ, dK, dV
