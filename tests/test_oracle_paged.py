"""Pins for the paged-cache oracle against the pinned dense oracle."""
import numpy as np
import pytest

import oracle
from oracle import paged
from exact_attention_28_gb300.inputs import custom_inputs, normal_bf16


def dense_to_cache(k, block_size):
    """[1,H,N,d] dense keys -> cache [N/bs, H, bs, d] with identity block table."""
    _, H, N, d = k.shape
    nb = N // block_size
    return np.ascontiguousarray(k[0].reshape(H, nb, block_size, d).transpose(1, 0, 2, 3))


@pytest.mark.parametrize("bs", [4, 8])
def test_identity_table_prefill_equals_dense_causal(bs):
    q, k, v = custom_inputs(3, 1, 2, 32, 32, 8)
    kc, vc = dense_to_cache(k, bs), dense_to_cache(v, bs)
    table = np.arange(32 // bs)[None, :]
    O, L = paged.paged_attention(q, kc, vc, table, [32], 0.3, True)
    Od, Ld = oracle.attention(q, k, v, 0.3, True, nthreads=1)
    assert np.max(np.abs(O - Od)) < 1e-13 and np.max(np.abs(L - Ld)) < 1e-13


def test_permuted_blocks_change_nothing():
    q, k, v = custom_inputs(4, 1, 2, 24, 32, 8)
    kc, vc = dense_to_cache(k, 8), dense_to_cache(v, 8)
    perm = np.array([2, 0, 3, 1])                     # logical l lives in physical perm[l]
    kp, vp = np.empty_like(kc), np.empty_like(vc)
    kp[perm], vp[perm] = kc, vc
    a = paged.paged_attention(q, kc, vc, np.arange(4)[None, :], [32], 0.3, False)
    b = paged.paged_attention(q, kp, vp, perm[None, :], [32], 0.3, False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_unallocated_blocks_are_skipped():
    q, k, v = custom_inputs(5, 1, 1, 6, 32, 8)
    kc, vc = dense_to_cache(k, 8), dense_to_cache(v, 8)
    table = np.array([[0, -1, 2, 3]])                 # block 1 (keys 8..15) unallocated
    O, L = paged.paged_attention(q, kc, vc, table, [30], 0.3, False)
    keep = np.r_[0:8, 16:30]
    Od, Ld = oracle.attention(q, np.ascontiguousarray(k[:, :, keep]), np.ascontiguousarray(v[:, :, keep]), 0.3,
                              False, nthreads=1)
    assert np.max(np.abs(O - Od)) < 1e-13 and np.max(np.abs(L - Ld)) < 1e-13


@pytest.mark.parametrize("seq", [1, 17, 40])
def test_last_positions_causal_equals_truncated_dense(seq):
    # query i sees keys k <= i + seq - Nq: the dense non-causal oracle on that prefix
    Nq = 5
    q, k, v = custom_inputs(6, 1, 2, Nq, 40, 8)
    kc, vc = dense_to_cache(k, 8), dense_to_cache(v, 8)
    O, L = paged.paged_attention(q, kc, vc, np.arange(5)[None, :], [seq], 0.4, True)
    for i in range(Nq):
        n = i + seq - Nq + 1
        if n <= 0:
            assert np.all(O[0, :, i] == 0) and np.all(L[0, :, i] == -np.inf)
            continue
        Od, Ld = oracle.attention(np.ascontiguousarray(q[:, :, i:i + 1]), np.ascontiguousarray(k[:, :, :n]),
                                  np.ascontiguousarray(v[:, :, :n]), 0.4, False, nthreads=1)
        assert np.max(np.abs(O[0, :, i] - Od[0, :, 0])) < 1e-13 and np.max(np.abs(L[0, :, i] - Ld[0, :, 0])) < 1e-13


def test_sequences_are_independent():
    q = normal_bf16(1, (2, 1, 3, 8))
    kc, vc = normal_bf16(2, (6, 1, 8, 8)), normal_bf16(3, (6, 1, 8, 8))
    table = np.array([[0, 1, 2], [3, 4, 5]])
    both = paged.paged_attention(q, kc, vc, table, [20, 9], 0.3, False)
    one = paged.paged_attention(q[1:], kc, vc, table[1:], [9], 0.3, False)
    assert np.array_equal(both[0][1:], one[0]) and np.array_equal(both[1][1:], one[1])
