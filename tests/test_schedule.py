"""The backward kernel's static work schedule, read through the C ABI on the
host (no GPU): the very mapping the kernel runs (its item function is
compiled for both sides) gives every K/V tile of every head to exactly one
CTA, and balances the CTAs' shares of the Q-tile walk."""

import ctypes
import math
import os

import pytest

from exact_attention_fattn_gb300 import _lib
from exact_attention_fattn_gb300.attention import (fattn_bwd_pair_schedule_items, fattn_bwd_schedule,
                                                   fattn_bwd_schedule_items)

L2 = 126 * 2**20  # an L2 of GB300's size (the head sections are sized from it)
SMS = 152


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from exact_attention_fattn_gb300 import build

        build.build()
    return _lib.load()


def walk(n_tiles, causal):
    """Q tiles that K/V tile j walks (causal: j..n_tiles-1)."""
    return [n_tiles - j if causal else n_tiles for j in range(n_tiles)]


def grid_for(B, H, N):
    return min(SMS, B * H * math.ceil(N / 128))


CASES = [
    # B, H, N, d, causal, deterministic
    (2, 32, 4096, 128, True, False),    # causal bench shape: paired + tail
    (1, 16, 16384, 128, True, False),   # long causal
    (1, 2, 65536, 64, True, False),     # few heads, long walks
    (8, 16, 4096, 128, False, False),   # unmasked, head sections
    (2, 32, 4096, 128, True, True),     # ordered dQ: one section, unpaired
    (1, 3, 1920, 128, True, False),     # odd tile count: unpaired causal
    (1, 1, 128, 64, True, False),       # one item
    (3, 5, 2000, 64, True, False),      # ragged N, small grid
    (4, 8, 1024, 128, False, True),
    (16, 16, 1024, 128, True, False),
    # the size-limit shapes of the GPU parity tests (just under 2^31 elements)
    (128, 128, 1023, 128, False, False),
    (128, 128, 1023, 128, True, False),
    (256, 128, 1023, 64, False, False),
]


@pytest.mark.parametrize("B,H,N,d,causal,det", CASES)
def test_every_item_exactly_once(B, H, N, d, causal, det):
    grid = grid_for(B, H, N)
    item_cta, q_tiles = fattn_bwd_schedule(B, H, N, d, causal, grid, L2, deterministic=det)
    assert item_cta.min().item() >= 0, "a K/V tile is missing or scheduled twice"
    assert item_cta.max().item() < grid
    n_tiles = math.ceil(N / 128)
    total = B * H * sum(walk(n_tiles, causal))
    assert q_tiles.sum().item() == total
    # the CTA's share is the sum of its items' walks
    per_cta = [0] * grid
    for bh in range(B * H):
        for j in range(n_tiles):
            per_cta[item_cta[bh, j].item()] += walk(n_tiles, causal)[j]
    assert per_cta == q_tiles.tolist()


def pairs_only_makespan(BH, n_tiles, grid):
    n_pairs = n_tiles // 2 * BH
    return -(-n_pairs // grid) * (n_tiles + 1)


@pytest.mark.parametrize("B,H,N,expect_max", [
    # (bound) the most loaded CTA walks at most this many Q tiles
    (2, 32, 4096, 224),     # 33792 Q tiles over 152 CTAs: 222.3 on average; whole pairs give 231
    (1, 16, 16384, 880),    # average 869.1; whole pairs 903
    (1, 4, 32768, 890),     # average 865.7; whole pairs 1028
    (2, 16, 4096, 114),     # average 111.2; whole pairs 132
])
def test_causal_tail_balances(B, H, N, expect_max):
    grid = grid_for(B, H, N)
    _, q_tiles = fattn_bwd_schedule(B, H, N, 128, True, grid, L2)
    n_tiles = N // 128
    assert q_tiles.max().item() <= expect_max
    assert q_tiles.max().item() < pairs_only_makespan(B * H, n_tiles, grid)
    assert q_tiles.sum().item() == B * H * n_tiles * (n_tiles + 1) // 2


@pytest.mark.parametrize("B,H,N,d", [(2, 32, 4096, 128), (4, 8, 1024, 64), (1, 12, 2048, 128)])
def test_causal_never_worse_than_pairs(B, H, N, d):
    grid = grid_for(B, H, N)
    _, q_tiles = fattn_bwd_schedule(B, H, N, d, True, grid, L2)
    assert q_tiles.max().item() <= pairs_only_makespan(B * H, N // 128, grid)


def test_unmasked_shares_differ_by_at_most_one_item():
    B, H, N = 8, 16, 4096
    _, q_tiles = fattn_bwd_schedule(B, H, N, 128, False, SMS, L2)
    assert q_tiles.max().item() - q_tiles.min().item() <= N // 128


def test_schedule_rejects_bad_arguments():
    lib = _lib.load()
    buf = (ctypes.c_int * 64)()
    assert lib.fattn_bwd_schedule(1, 1, 128, 128, 1, 0, 0, L2, buf, None) == _lib.FATTN_ERR_INVALID_ARG
    assert lib.fattn_bwd_schedule(1, 1, 128, 128, 1, 0, 2, L2, buf, None) == _lib.FATTN_ERR_INVALID_ARG
    assert lib.fattn_bwd_schedule(1, 1, 128, 128, 1, 0, 1, L2, None, None) == _lib.FATTN_ERR_INVALID_ARG
    assert lib.fattn_bwd_schedule(1, 1, 128, 96, 1, 0, 1, L2, buf, None) == _lib.FATTN_ERR_UNSUPPORTED
    assert lib.fattn_bwd_schedule(1, 1, 128, 128, 1, 0, 1, L2, buf, None) == _lib.FATTN_OK
    assert buf[0] == 0


def test_schedule_fuzz():
    """Seeded random shapes, masks, modes and grids: every K/V tile exactly
    once, shares summing to the total walk."""
    import random

    rng = random.Random(20261202)
    for _ in range(60):
        B = rng.randint(1, 4)
        H = rng.randint(1, 40)
        N = rng.choice([1, 127, 128, 129, 256, 384, 1000, 2048, 2176, 4096, 8192])
        d = rng.choice([64, 128])
        causal = rng.random() < 0.7
        det = rng.random() < 0.2
        n_tiles = math.ceil(N / 128)
        items = B * H * n_tiles
        grid = rng.randint(1, min(SMS, items))
        l2 = rng.choice([0, 32 * 2**20, L2])
        item_cta, q_tiles = fattn_bwd_schedule(B, H, N, d, causal, grid, l2, deterministic=det)
        assert item_cta.min().item() >= 0, (B, H, N, d, causal, det, grid, l2)
        assert item_cta.max().item() < grid
        assert q_tiles.sum().item() == B * H * sum(walk(n_tiles, causal))


# ---------------------------------------------------------------------------
# The ordered (deterministic) dQ reduction: the reduce warp of the CTA that
# holds K/V tile j of head bh adds its dQ tile into Q tile i only once tile
# i's counter shows that K/V tiles 0..j-1 of bh have added theirs, and each
# CTA serves its steps strictly in order.  With every CTA of the grid
# resident, that makes progress if and only if the simulation below, which
# replays exactly those rules on the schedule the kernel runs, finishes.

def visits(entry, n_tiles, causal):
    bh, j, i0, n_it, rot = entry
    if causal:
        return [(bh, i0 + it, j) for it in range(n_it)]
    return [(bh, (rot + it) % n_tiles, j) for it in range(n_it)]


def ordered_reduction_finishes(per_cta, n_tiles, causal):
    """Replay the counter waits; True if every CTA gets through its steps."""
    queues = [[v for e in items for v in visits(e, n_tiles, causal)] for items in per_cta]
    pos = [0] * len(queues)
    counter = {}
    pending = sum(len(q) for q in queues)
    while pending:
        moved = False
        for c, q in enumerate(queues):
            while pos[c] < len(q):
                bh, i, j = q[pos[c]]
                if counter.get((bh, i), 0) != j:
                    break
                counter[(bh, i)] = j + 1
                pos[c] += 1
                pending -= 1
                moved = True
        if not moved:
            return False
    return True


DET_CASES = [
    (2, 32, 4096, 128, True),
    (1, 4, 1024, 128, True),
    (2, 3, 777, 64, False),
    (1, 2, 1000, 128, False),
    (2, 32, 2048, 128, True),
    (4, 8, 1024, 128, False),
    (1, 16, 16384, 128, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", DET_CASES)
def test_ordered_reduction_always_progresses(B, H, N, d, causal):
    grid = grid_for(B, H, N)
    per_cta = fattn_bwd_schedule_items(B, H, N, d, causal, grid, L2, deterministic=True)
    n_tiles = math.ceil(N / 128)
    assert sum(len(x) for x in per_cta) == B * H * n_tiles
    assert ordered_reduction_finishes(per_cta, n_tiles, causal)


@pytest.mark.parametrize("seed", range(12))
def test_ordered_reduction_fuzz(seed):
    rng = __import__("random").Random(seed)
    B, H = rng.randint(1, 4), rng.randint(1, 12)
    N = rng.randint(1, 3000)
    d = rng.choice((64, 128))
    causal = rng.random() < 0.5
    n_tiles = math.ceil(N / 128)
    grid = rng.randint(1, min(SMS, B * H * n_tiles))
    per_cta = fattn_bwd_schedule_items(B, H, N, d, causal, grid, L2, deterministic=True)
    assert ordered_reduction_finishes(per_cta, n_tiles, causal)


def test_the_simulation_detects_a_cycle():
    """The check itself, on hand-made two-CTA schedules of one head with two
    K/V tiles (entries (bh, j, i0, n_it, rot), causal visit order)."""
    # each CTA walks its tile over both Q tiles: progresses
    assert ordered_reduction_finishes([[(0, 0, 0, 2, 0)], [(0, 1, 0, 2, 0)]], 2, True)
    # CTA 0 runs tile 1 on Q0 first, which needs tile 0 on Q0 -- last on
    # CTA 1, behind tile 1 on Q1, which needs tile 0 on Q1 -- last on CTA 0
    cyc = [[(0, 1, 0, 1, 0), (0, 0, 1, 1, 0)], [(0, 1, 1, 1, 0), (0, 0, 0, 1, 0)]]
    assert not ordered_reduction_finishes(cyc, 2, True)


# ---------------------------------------------------------------------------
# The CTA-pair backward: units of two K/V tiles dealt to clusters of two CTAs.

PAIR_CASES = [
    (2, 32, 4096, True),      # bench shape: paired units and a balancing tail
    (1, 16, 16384, True),
    (8, 16, 4096, False),     # head sections
    (1, 3, 1920, True),       # 15 tiles: the last unit's second tile is past N
    (1, 1, 128, False),       # one unit
    (3, 5, 2000, True),
    (4, 20, 512, True),
]


@pytest.mark.parametrize("B,H,N,causal", PAIR_CASES)
def test_pair_schedule_every_unit_once(B, H, N, causal):
    n_tiles = math.ceil(N / 128)
    n_units = (n_tiles + 1) // 2
    clusters = min(SMS // 2, B * H * n_units)
    per = fattn_bwd_pair_schedule_items(B, H, N, causal, clusters, L2)
    seen = {}
    steps = []
    for c, items in enumerate(per):
        walked = 0
        for bh, j, i0, n_it, rot in items:
            assert j % 2 == 0 and 0 <= j < n_tiles
            key = (bh, j // 2)
            assert key not in seen, f"unit {key} scheduled twice"
            seen[key] = c
            assert n_it == (n_tiles - j if causal else n_tiles)
            assert i0 == (j if causal else 0)
            walked += n_it
        steps.append(walked)
    assert len(seen) == B * H * n_units
    # the static deal leaves no cluster far behind the others
    total = sum(steps)
    if clusters > 1 and total >= 8 * clusters:
        assert max(steps) <= 1.1 * total / clusters + n_tiles + 2
