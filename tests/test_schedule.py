"""The persistent kernel's work list, enumerated on the host (no GPU).

Every (batch*head, 128-row query tile) must be computed exactly once, each
with the key/value tiles its rows can see (all of them, or those up to the
diagonal under the causal mask), and the rounds must balance across CTAs.
Key/value tiles hold 128 keys at head dimension 128 and 64 keys at head
dimension 64, where two persistent CTAs share each SM.
"""
import math

import numpy as np
import pytest

import __graft_entry__  # noqa: F401
from exact_attention_28_gb300 import build, ops


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    ops.load_library()


def expand(items):
    """(cta, round, bh, q0, kv0, end0, end1, split) -> list of (bh, q_start, kv0, end, split)."""
    tiles = []
    for cta, rnd, bh, q0, kv0, e0, e1, split in items.tolist():
        tiles.append((bh, q0, kv0, e0, split))
        if e1 >= 0:                      # -1: the item holds one query tile
            tiles.append((bh, q0 + 128, kv0, e1, split))
    return tiles


def kv_keys(d):
    return 64 if d == 64 else 128


def ctas_per_sm(d):
    return 2 if d == 64 else 1


def visible_tiles(Nq, Nk, causal, q, d):
    bc = kv_keys(d)
    Tc = math.ceil(Nk / bc)
    return min(Tc, (min(Nq, q + 128) - 1) // bc + 1) if causal else Tc


SHAPES = [
    (1, 1, 256, 256, 64, False), (4, 16, 1024, 1024, 64, True), (2, 16, 4096, 4096, 128, False),
    (1, 32, 16384, 16384, 128, True), (8, 32, 128, 8192, 128, False), (8, 32, 128, 8229, 128, False),
    (1, 3, 300, 1000, 64, True), (1, 3, 1000, 300, 128, True), (2, 5, 129, 129, 64, False), (1, 1, 1, 1, 64, True),
    (3, 7, 640, 129, 128, True), (8, 64, 200, 160, 64, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", SHAPES)
@pytest.mark.parametrize("sms", [1, 7, 148, 152])
def test_every_tile_exactly_once_with_its_kv_range(B, H, Nq, Nk, d, causal, sms):
    items = ops.schedule(B, H, Nq, Nk, d, causal, sms)
    tiles = expand(items)
    Tr = math.ceil(Nq / 128)
    assert len(tiles) == B * H * Tr
    assert len(set((bh, q) for bh, q, *_ in tiles)) == B * H * Tr
    for bh, q, kv0, end, split in tiles:
        assert 0 <= bh < B * H and q % 128 == 0 and q < Nq and kv0 == 0 and split == 0
        assert end == visible_tiles(Nq, Nk, causal, q, d), (bh, q, end)
    # each CTA walks consecutive rounds 0, 1, 2, ...
    for cta in np.unique(items[:, 0]):
        rounds = np.sort(items[items[:, 0] == cta, 1])
        assert np.array_equal(rounds, np.arange(len(rounds)))
    assert items[:, 0].max() < ctas_per_sm(d) * sms


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", SHAPES)
@pytest.mark.parametrize("splits", [2, 3, 8, 64])
def test_key_slices_partition_each_tiles_range(B, H, Nq, Nk, d, causal, splits):
    items = ops.schedule(B, H, Nq, Nk, d, causal, 152, splits)
    by_tile = {}
    for bh, q, kv0, end, split in expand(items):
        by_tile.setdefault((bh, q), []).append((split, kv0, end))
    assert len(by_tile) == B * H * math.ceil(Nq / 128)
    for (bh, q), parts in by_tile.items():
        assert sorted(s for s, _, _ in parts) == list(range(splits))   # every slice once
        covered = []
        for _, kv0, end in parts:
            covered.extend(range(kv0, max(kv0, end)))
        assert sorted(covered) == list(range(visible_tiles(Nq, Nk, causal, q, d))), (bh, q)


def cta_loads(items, key=lambda nk: 1):
    load = {}
    for cta, _, _, _, kv0, nk0, nk1, _ in items.tolist():
        load[cta] = load.get(cta, 0) + key(nk0 - kv0) + (key(nk1 - kv0) if nk1 >= 0 else 0)
    return np.array(list(load.values()), dtype=np.float64)


def test_noncausal_rounds_fill_the_machine():
    # 1024 query tiles on 152 SMs: no CTA gets more than ceil(1024/152) = 7 tiles
    items = ops.schedule(2, 16, 4096, 4096, 128, False, 152)
    assert cta_loads(items).max() == 7


def test_causal_load_balance():
    # the long causal workload: KV-tile work per CTA within 10% of the mean
    items = ops.schedule(1, 32, 16384, 16384, 128, True, 152)
    load = cta_loads(items, key=lambda nk: nk)
    assert load.max() / load.mean() < 1.10


def test_causal_single_tiles_pair_heavy_with_light():
    # 4 x 16 x 1024 causal at d = 64: 512 single-tile items (64-key tiles, 2 to
    # 16 key steps each) on 304 CTAs.  Listing each pair index's upper tiles
    # first makes the snake's second round give the lightest items to the CTAs
    # with the heaviest first items: at most 16 key steps per CTA (the optimum:
    # the heaviest item alone has 16; the mean is 15.2).
    items = ops.schedule(4, 16, 1024, 1024, 64, True, 152)
    assert np.all(items[:, 6] == -1)                       # all single-tile items
    load = cta_loads(items, key=lambda nk: nk)
    assert len(load) == 304 and load.max() == 16
    # the work list is heaviest first inside each round's snake
    first_round = items[items[:, 1] == 0]
    assert (first_round[:, 5] - first_round[:, 4]).max() == 16


def test_schedule_argument_errors():
    n = ops.ctypes.c_int64(0)
    lib = ops.load_library()
    assert lib.fa_schedule(1, 1, 128, 128, 96, 0, 152, 1, None, 0, ops.ctypes.byref(n)) == ops.FA_ERR_UNSUPPORTED
    assert lib.fa_schedule(0, 1, 128, 128, 64, 0, 152, 1, None, 0, ops.ctypes.byref(n)) == ops.FA_ERR_INVALID_ARG
    assert lib.fa_schedule(1, 1, 128, 128, 64, 0, 0, 1, None, 0, ops.ctypes.byref(n)) == ops.FA_ERR_INVALID_ARG
    assert lib.fa_schedule(1, 1, 128, 128, 64, 0, 152, 0, None, 0, ops.ctypes.byref(n)) == ops.FA_ERR_INVALID_ARG


def test_splitkv_workspace_size():
    ns, nb = ops.splitkv_workspace(8, 32, 128, 8192, 128, False, num_splits=4)
    o_bytes = 4 * 8 * 32 * 128 * 128 * 4
    assert ns == 4 and nb == o_bytes + 4 * 8 * 32 * 128 * 4
