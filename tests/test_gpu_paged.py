"""GPU parity of fa_fwd_paged (paged key/value cache) against the paged oracle.

Same tolerances as the dense forward: O max |err| <= 2e-2, mean <= 2e-3,
LSE max |err| <= 1e-3; rows that see no key must come back as O = 0,
LSE = -inf.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import paged  # noqa: E402
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


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def make_case(seed, seq_lens, H, Nq, d, block_size, holes=0):
    rng = np.random.default_rng(seed)
    B = len(seq_lens)
    max_blocks = max(1, max((s + block_size - 1) // block_size for s in seq_lens)) + 1
    num_blocks = B * max_blocks + 3
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    phys = rng.permutation(num_blocks)
    n = 0
    for b, s in enumerate(seq_lens):
        for lb in range((s + block_size - 1) // block_size):
            table[b, lb] = phys[n]
            n += 1
    for _ in range(holes):   # unallocated blocks inside sequences
        b = rng.integers(0, B)
        used = (seq_lens[b] + block_size - 1) // block_size
        if used > 1:
            table[b, rng.integers(0, used)] = -1
    q = inputs.normal_bf16(seed + 1, (B, H, Nq, d))
    kc = inputs.normal_bf16(seed + 2, (num_blocks, H, block_size, d))
    vc = inputs.normal_bf16(seed + 3, (num_blocks, H, block_size, d))
    return q, kc, vc, table, np.array(seq_lens, dtype=np.int32)


def run_and_check(ops, q, kc, vc, table, seq_lens, causal, tag, num_splits=None):
    d = q.shape[-1]
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = ops.fa_fwd_paged(to_dev(q), to_dev(kc), to_dev(vc), torch.from_numpy(table).cuda(),
                              torch.from_numpy(seq_lens).cuda(), scale=scale, causal=causal, num_splits=num_splits)
    ops.check_device_status()
    O_ref, L_ref = paged.paged_attention(q, kc, vc, table, seq_lens, scale, causal)
    o = o.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    empty = ~np.isfinite(L_ref)
    assert np.all(o[empty] == 0) and np.all(l[empty] == -np.inf), tag
    err = np.abs(o - O_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, f"{tag}: O {err.max():.3e} {err.mean():.3e}"
    if (~empty).any():
        assert np.abs(l[~empty] - L_ref[~empty]).max() <= 1e-3, tag


@pytest.mark.parametrize("block_size", [16, 64, 128, 256])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_prefill_and_decode(ops, block_size, d, causal):
    seq_lens = [300, 1, 129, 700]
    for Nq in (1, 100):
        q, kc, vc, table, sl = make_case(block_size + d + Nq, seq_lens, 2, Nq, d, block_size)
        run_and_check(ops, q, kc, vc, table, sl, causal, f"bs={block_size} d={d} Nq={Nq} causal={causal}")


@pytest.mark.parametrize("block_size", [16, 128])
def test_paged_unallocated_blocks(ops, block_size):
    q, kc, vc, table, sl = make_case(77, [500, 640, 257], 2, 64, 128, block_size, holes=4)
    run_and_check(ops, q, kc, vc, table, sl, False, "holes")
    run_and_check(ops, q, kc, vc, table, sl, True, "holes causal")


# 16-key pages are copied by the producer lanes into the swizzled tile layout
# by hand, larger ones by TMA boxes: both must give the dense forward's bits
@pytest.mark.parametrize("bs,d", [(128, 128), (16, 128), (16, 64), (32, 64)])
def test_paged_full_prefill_equals_dense_forward(ops, bs, d):
    # identity table, Nq = seq_len: the paged call equals the dense causal forward
    B, H, N = 1, 4, 512
    q, k, v = inputs.custom_inputs(21, B, H, N, N, d)
    kc = np.ascontiguousarray(k[0].reshape(H, N // bs, bs, d).transpose(1, 0, 2, 3))
    vc = np.ascontiguousarray(v[0].reshape(H, N // bs, bs, d).transpose(1, 0, 2, 3))
    table = torch.arange(N // bs, dtype=torch.int32, device="cuda")[None, :].contiguous()
    seq = torch.tensor([N], dtype=torch.int32, device="cuda")
    o1, l1 = ops.fa_fwd_paged(to_dev(q), to_dev(kc), to_dev(vc), table, seq, causal=True)
    o2, l2 = ops.fa_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True)
    ops.check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("block_size", [16, 128])
def test_paged_out_of_range_entries_read_zero_keys(ops, block_size):
    # entries >= num_blocks read as zero keys and values: the oracle sees them
    # as blocks of zeros appended to the cache
    q, kc, vc, table, sl = make_case(88, [400, 333], 2, 40, 128, block_size)
    num_blocks = kc.shape[0]
    rng = np.random.default_rng(5)
    table = table.copy()
    for b, s_len in enumerate(sl):
        used = (int(s_len) + block_size - 1) // block_size
        for lb in rng.choice(used, size=2, replace=False):
            table[b, lb] = num_blocks + int(rng.integers(0, 4))
    zeros = np.zeros((4,) + kc.shape[1:], dtype=kc.dtype)
    kc_ext, vc_ext = np.concatenate([kc, zeros]), np.concatenate([vc, zeros])
    for causal in (False, True):
        o, lse = ops.fa_fwd_paged(to_dev(q), to_dev(kc), to_dev(vc), torch.from_numpy(table).cuda(),
                                  torch.from_numpy(sl).cuda(), scale=float(np.float32(1 / math.sqrt(128))),
                                  causal=causal)
        ops.check_device_status()
        O_ref, L_ref = paged.paged_attention(q, kc_ext, vc_ext, table, sl, float(np.float32(1 / math.sqrt(128))), causal)
        err = np.abs(o.float().cpu().numpy().astype(np.float64) - O_ref)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (block_size, causal, err.max(), err.mean())
        assert np.abs(lse.cpu().numpy().astype(np.float64) - L_ref).max() <= 1e-3


@pytest.mark.parametrize("num_splits", [2, 3, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_split_keys(ops, num_splits, causal):
    # an empty sequence, a one-key one and long ones; slices of a short
    # sequence are empty and must carry no weight in the merge
    seq_lens = [0, 1, 300, 1000]
    for Nq in (1, 5):
        for bs in (16, 64):
            q, kc, vc, table, sl = make_case(500 + bs + Nq, seq_lens, 2, Nq, 128, bs, holes=2)
            run_and_check(ops, q, kc, vc, table, sl, causal, f"splits={num_splits} bs={bs} Nq={Nq} causal={causal}",
                          num_splits=num_splits)


def test_paged_split_decode_shape(ops):
    # one query per head against 32768 keys in 64-key pages, slices chosen by the library
    q, kc, vc, table, sl = make_case(901, [32768], 32, 1, 128, 64)
    run_and_check(ops, q, kc, vc, table, sl, False, "decode auto splits", num_splits=0)
    run_and_check(ops, q, kc, vc, table, sl, True, "decode auto splits causal", num_splits=0)


def test_paged_split_one_slice_is_the_paged_forward(ops):
    q, kc, vc, table, sl = make_case(33, [200, 450], 2, 64, 64, 32)
    args = (to_dev(q), to_dev(kc), to_dev(vc), torch.from_numpy(table).cuda(), torch.from_numpy(sl).cuda())
    o1, l1 = ops.fa_fwd_paged(*args, causal=True)
    o2, l2 = ops.fa_fwd_paged(*args, causal=True, num_splits=1)
    ops.check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
