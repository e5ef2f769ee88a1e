"""Online-softmax pieces of the oracle, in fp64 numpy / plain Python.

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and
the bench's CPU-baseline leg, never by the product path.  Shares nothing with
the CUDA code.

Each function follows one passage of the FlashAttention pages, step by step,
in the pages' order and notation (m = running maximum, l = running sum of
exponentials relative to m, O = unnormalised output):

* ``three_pass_softmax``  -- "6. FlashAttention 分块逻辑", section 1.1 (find the
  maximum, sum exp(x - m), divide); "9.4 FlashAttention 与 FlashMLA", 9.4.2.
* ``online_softmax_1d``   -- "6. FlashAttention 分块逻辑", section 1.2: one pass
  that rescales l by exp(m_old - x) when a new maximum x appears, then a final
  normalising pass.  The page's section 1.3 listing adds where the recurrence
  multiplies and stores exp(x_i - m) with a stale m; this follows the text and
  its proof (l_{k+1} = l_k * e^{m_k - m_{k+1}} + e^{x_{k+1} - m_{k+1}}) instead.
* ``online_softmax_blocks`` -- "9.4 FlashAttention 与 FlashMLA", 9.4.2: block
  recurrence with local statistics m_local, l_local, returning the (m^(k), l^(k))
  pair after every block so the invariant l^(k) = sum exp(x_j - m^(k)) can be
  checked at each block boundary.
* ``blocked_attention``   -- "6. FlashAttention 分块逻辑", sections 3.1 (Q-outer,
  KV-inner loops with deferred normalisation), 4.1/4.2 (causal block classes:
  skip fully masked blocks, mask partial ones), 6 (return O together with the
  final l and m).  LSE = m + ln l as in "9.4 FlashAttention 与 FlashMLA", 9.4.5.
* ``merge_partials``      -- "6. FlashAttention 分块逻辑", sections 11.3 (stage 2)
  and 13.2: merge per-block (m_j, l_j, o_j) triples with the online-softmax
  reduction, o = o_global / l_global.
"""
from __future__ import annotations

import math

import numpy as np


def three_pass_softmax(x):
    """Safe softmax by three passes over a 1-D vector (fp64)."""
    x = np.asarray(x, dtype=np.float64)
    m = -math.inf
    for v in x:                      # pass 1: maximum
        if v > m:
            m = v
    l = 0.0
    for v in x:                      # pass 2: sum of exp(x - m)
        l += math.exp(v - m)
    return np.array([math.exp(v - m) / l for v in x])   # pass 3: divide


def online_softmax_1d(x, trace=False):
    """One streaming pass for (m, l), then one normalising pass.

    Returns (y, m, l) and, with ``trace``, the list of (m_k, l_k) after each
    element.
    """
    x = np.asarray(x, dtype=np.float64)
    m = -math.inf
    l = 0.0
    steps = []
    for v in x:
        if v > m:
            # a new maximum: bring the old sum to the new reference, then add e^0
            l = l * math.exp(m - v) + 1.0
            m = v
        else:
            l = l + math.exp(v - m)
        if trace:
            steps.append((m, l))
    y = np.array([math.exp(v - m) / l for v in x])
    if trace:
        return y, m, l, steps
    return y, m, l


def online_softmax_blocks(x, block):
    """Block recurrence of section 9.4.2.  Returns (m, l, [(m^(k), l^(k)), ...])."""
    x = np.asarray(x, dtype=np.float64)
    m = -math.inf                     # m^(0)
    l = 0.0                           # l^(0)
    steps = []
    for start in range(0, len(x), block):
        xb = x[start:start + block]
        m_local = float(np.max(xb))
        l_local = float(np.sum(np.exp(xb - m_local)))
        m_next = max(m, m_local)
        l = l * math.exp(m - m_next) + l_local * math.exp(m_local - m_next)
        m = m_next
        steps.append((m, l))
    return m, l, steps


def online_softmax_lagged(x, block, tau):
    """The block recurrence with a lagging reference value (the reading of
    "9.4 FlashAttention 与 FlashMLA" section 9.4.2 the GPU kernel uses): the
    reference r is raised to a block's maximum only when that maximum exceeds
    r by more than tau; otherwise the block is summed against the old r and the
    rescale factor alpha is exactly 1.  The section's invariant
    l^(k) = sum_{j <= k} exp(x_j - r^(k)) holds for any reference value, so the
    result r + ln l equals the plain log-sum-exp; tau only bounds the terms,
    exp(x - r) <= exp(tau).  Returns (r, l, [(r^(k), l^(k), alpha^(k)), ...])."""
    x = np.asarray(x, dtype=np.float64)
    r = -math.inf
    l = 0.0
    steps = []
    for start in range(0, len(x), block):
        xb = x[start:start + block]
        m_block = float(np.max(xb))
        alpha = 1.0
        if m_block > r + tau:
            alpha = math.exp(r - m_block)      # 0 on the first block
            r = m_block
        l = l * alpha + float(np.sum(np.exp(xb - r)))
        steps.append((r, l, alpha))
    return r, l, steps


def blocked_attention(Q, K, V, scale, causal, Br, Bc):
    """Tiled attention forward for one head, fp64.

    Q [Nq, d], K and V [Nk, d].  Returns O [Nq, d], l [Nq], m [Nq], LSE [Nq].
    The loops are the pages' Q-block-outer / KV-block-inner loops; the running
    statistics are m (row maximum so far) and l (row sum relative to m); O is
    normalised once, after the last KV block.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Nq, d = Q.shape
    Nk = K.shape[0]
    O = np.zeros((Nq, d))
    L = np.zeros(Nq)
    M = np.full(Nq, -math.inf)

    Tr = (Nq + Br - 1) // Br
    Tc = (Nk + Bc - 1) // Bc
    for i in range(Tr):
        q_start = i * Br
        q_end = min(Nq, q_start + Br)
        Qi = Q[q_start:q_end]
        Oi = np.zeros((q_end - q_start, d))
        li = np.zeros((q_end - q_start, 1))
        mi = np.full((q_end - q_start, 1), -math.inf)
        for j in range(Tc):
            k_start = j * Bc
            k_end = min(Nk, k_start + Bc)
            if causal and k_start >= q_end:
                continue                      # fully masked block: skip
            Kj = K[k_start:k_end]
            Vj = V[k_start:k_end]
            Sij = (Qi @ Kj.T) * scale
            if causal and k_end > q_start:    # partially visible block: mask
                q_pos = np.arange(q_start, q_end)[:, None]
                k_pos = np.arange(k_start, k_end)[None, :]
                Sij = np.where(q_pos >= k_pos, Sij, -math.inf)
            row_max = Sij.max(axis=1, keepdims=True)
            mi_new = np.maximum(mi, row_max)
            # a row with no visible key so far keeps m = -inf; its factors are
            # defined as (alpha = 1, p = 0) instead of exp(-inf - (-inf))
            finite = np.isfinite(mi_new)
            safe_new = np.where(finite, mi_new, 0.0)
            alpha = np.where(finite, np.exp(mi - safe_new), 1.0)
            Pij = np.where(finite, np.exp(Sij - safe_new), 0.0)
            Oi = Oi * alpha
            li = li * alpha
            li = li + Pij.sum(axis=1, keepdims=True)
            Oi = Oi + Pij @ Vj
            mi = mi_new
        O[q_start:q_end] = Oi / li
        L[q_start:q_end] = li[:, 0]
        M[q_start:q_end] = mi[:, 0]
    return O, L, M, M + np.log(L)


def merge_partials(parts):
    """Merge [(m_j, l_j, o_j), ...] partial results of disjoint key blocks.

    Each o_j is the unnormalised sum_k exp(s_k - m_j) v_k of its block.  Returns
    (o, m, l) with o = o_global / l_global.
    """
    m_g = -math.inf
    l_g = 0.0
    o_g = 0.0
    for m_j, l_j, o_j in parts:
        m_new = max(m_g, m_j)
        l_g = l_g * math.exp(m_g - m_new) + l_j * math.exp(m_j - m_new)
        o_g = o_g * math.exp(m_g - m_new) + np.asarray(o_j, dtype=np.float64) * math.exp(m_j - m_new)
        m_g = m_new
    return o_g / l_g, m_g, l_g


def block_partial(q, K, V, scale):
    """Stage-1 triple (m_j, l_j, o_j) for one query vector over one key block."""
    s = (np.asarray(K, dtype=np.float64) @ np.asarray(q, dtype=np.float64)) * scale
    m_j = float(np.max(s))
    p = np.exp(s - m_j)
    return m_j, float(np.sum(p)), p @ np.asarray(V, dtype=np.float64)
