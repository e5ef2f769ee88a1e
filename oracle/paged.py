"""Attention over a paged key/value cache, fp64: the oracle for fa_fwd_paged.

TEST INFRASTRUCTURE ONLY (imported by the tests, never by the product path).

Follows "6. FlashAttention 分块逻辑" section 12.2: for each sequence, walk its
logical blocks in order, look up each one's physical block in the block table,
skip unallocated blocks (negative entries), and take the keys and values of
the allocated blocks up to the sequence length; then the three-pass softmax
attention of section 1.1 over those keys.  The Nq queries are the last Nq
positions of the sequence, so under the causal mask query i sees key positions
k <= i + seq_len - Nq (for prefill, Nq = seq_len, this is the usual k <= i).
A row that sees no key gets O = 0 and LSE = -inf.
"""
from __future__ import annotations

import math

import numpy as np

from . import bf16_bits_to_f64


def gather(k_cache, v_cache, table_row, seq_len, h):
    """Key positions kept, and their K and V rows (fp64), for one sequence and head."""
    block_size = k_cache.shape[2]
    pos, ks, vs = [], [], []
    for lb in range((seq_len + block_size - 1) // block_size):
        phy = int(table_row[lb])
        if phy < 0:
            continue                                   # unallocated: skipped
        n = min(block_size, seq_len - lb * block_size)
        pos.extend(range(lb * block_size, lb * block_size + n))
        ks.append(bf16_bits_to_f64(k_cache[phy, h, :n]))
        vs.append(bf16_bits_to_f64(v_cache[phy, h, :n]))
    d = k_cache.shape[3]
    if not ks:
        return np.zeros(0, dtype=np.int64), np.zeros((0, d)), np.zeros((0, d))
    return np.array(pos), np.concatenate(ks), np.concatenate(vs)


def paged_attention(q, k_cache, v_cache, block_table, seq_lens, scale, causal):
    """q uint16 [B,H,Nq,d]; caches uint16 [num_blocks,H,block_size,d];
    block_table int [B,max_blocks]; seq_lens int [B].  Returns O, LSE (fp64)."""
    B, H, Nq, d = q.shape
    scale = float(np.float32(scale))
    O = np.zeros((B, H, Nq, d))
    LSE = np.full((B, H, Nq), -math.inf)
    cap = block_table.shape[1] * k_cache.shape[2]
    Q = bf16_bits_to_f64(q)
    for b in range(B):
        seq = int(min(max(int(seq_lens[b]), 0), cap))
        for h in range(H):
            pos, Kb, Vb = gather(k_cache, v_cache, block_table[b], seq, h)
            for i in range(Nq):
                vis = pos <= i + seq - Nq if causal else np.ones(len(pos), dtype=bool)
                if not vis.any():
                    continue
                s = scale * (Kb[vis] @ Q[b, h, i])
                m = s.max()
                e = np.exp(s - m)
                l = e.sum()
                O[b, h, i] = (e / l) @ Vb[vis]
                LSE[b, h, i] = m + math.log(l)
    return O, LSE
