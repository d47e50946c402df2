"""The persistent kernels' work schedule, checked on the host (no GPU).

sgemm_test_schedule() walks every CTA's work items with the same functions
the kernels run (plan_schedule, cursor_init, next_item, tile_coords_b,
sk_first_cta, sk_last_cta, sk_slot). For every shape and policy here:
  - every (tile, slab) of the product is computed exactly once;
  - whole tiles precede the stream-K region, whose items are slab ranges;
  - the parts of a tile split among several CTAs come from exactly the
    consecutive CTAs first .. last that the kernels add in that order, and
    the first of them holds the tile's first slab;
  - no two parts write the same partial-sum slot in one launch, and every
    slot lies inside the 2 x sk_ctas slots of the workspace;
  - tile coordinates are distinct and inside the tile grid of each entry;
  - each CTA's items follow one another in order of iteration.
"""

import itertools

import numpy as np
import pytest

import dense_fp32_matrix_07_gb300 as sg

AUTO, WHOLE, STREAM_K, TAIL_SPLIT = 0, 1, 2, 3

SHAPES = [
    # M, N, K, bm, bn, bk, slots, batch
    (4096, 4096, 4096, 128, 256, 32, 152, 1),
    (4097, 3001, 2049, 128, 256, 32, 152, 1),
    (1024, 1024, 1024, 128, 128, 32, 152, 1),
    (1024, 1024, 1024, 128, 64, 32, 304, 1),
    (256, 256, 256, 128, 64, 32, 304, 1),
    (1, 1, 1 << 16, 128, 64, 32, 304, 1),
    (300, 260, 130, 128, 256, 32, 152, 4),
    (64, 96, 48, 128, 64, 32, 304, 40),
    (4096, 4096, 4096, 256, 256, 16, 76, 1),      # cluster-pair tensor tiles
    (16384, 1000, 33, 128, 128, 32, 152, 1),
    (129, 129, 129, 128, 128, 32, 7, 3),
    (5000, 7, 9000, 128, 128, 32, 151, 2),
]


def _check(M, N, K, bm, bn, bk, slots, batch, policy):
    items, info = sg.sgemm_test_schedule(M, N, K, bm, bn, bk, slots, policy, batch)
    tiles_m, tiles_n, nk = info["tiles_m"], info["tiles_n"], info["nk"]
    assert tiles_m == -(-M // bm) and tiles_n == -(-N // bn) and nk == -(-K // bk)
    tiles = info["tiles"]
    assert tiles == tiles_m * tiles_n * batch
    grid, dp_tiles, sk_ctas = info["grid"], info["dp_tiles"], info["sk_ctas"]
    assert 1 <= grid <= max(slots, 1) and 0 <= sk_ctas <= grid and 0 <= dp_tiles <= tiles
    cta, tile, kb0, kb1, b, tm, tn, first, last, slot = (items[:, i] for i in range(10))
    assert np.all((0 <= cta) & (cta < grid))
    assert np.all((0 <= kb0) & (kb0 < kb1) & (kb1 <= nk))

    # Exactly-once coverage of every (tile, slab).
    cover = np.zeros((tiles, nk), dtype=np.int32)
    for t, a, e in zip(tile, kb0, kb1):
        cover[t, a:e] += 1
    assert np.all(cover == 1), (policy, np.argwhere(cover != 1)[:3])

    # Whole tiles below dp_tiles; coordinates distinct and in range.
    assert np.all((kb0 == 0) & (kb1 == nk) | (tile >= dp_tiles))
    assert np.all((0 <= b) & (b < batch) & (0 <= tm) & (tm < tiles_m) & (0 <= tn) & (tn < tiles_n))
    coords = {}
    for t, bb, r, c in zip(tile, b, tm, tn):
        coords.setdefault(int(t), (int(bb), int(r), int(c)))
        assert coords[int(t)] == (bb, r, c)
    assert len(set(coords.values())) == tiles

    # Parts of split tiles.
    pieces = {}
    for g, t, a, e, f, l, sl in zip(cta, tile, kb0, kb1, first, last, slot):
        pieces.setdefault(int(t), []).append((int(a), int(e), int(g), int(f), int(l), int(sl)))
    used_slots = set()
    for t, ps in pieces.items():
        if len(ps) == 1:
            assert ps[0][3:] == (-1, -1, -1)               # one CTA computes the whole tile
            continue
        ctas = sorted(p[2] for p in ps)
        f, l = ps[0][3], ps[0][4]
        assert all((p[3], p[4]) == (f, l) for p in ps), (t, ps)
        assert ctas == list(range(f, l + 1)), (t, ctas, f, l)
        assert [p[2] for p in ps if p[0] == 0] == [f]       # the first part starts the tile
        for a, _, g, _, _, sl in ps:
            assert sl == 2 * g + (1 if a == 0 else 0)
            assert 0 <= sl < 2 * sk_ctas
            assert sl not in used_slots, (t, sl)
            used_slots.add(sl)

    # Each CTA's items in increasing order of (tile, slab) iteration.
    for g in range(grid):
        mine = items[cta == g]
        seq = [int(t) * nk + int(a) for t, a in zip(mine[:, 1], mine[:, 2])]
        assert seq == sorted(seq)


@pytest.mark.parametrize("policy", [AUTO, WHOLE, STREAM_K, TAIL_SPLIT],
                         ids=["auto", "whole_tiles", "stream_k", "tail_split"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}x{s[1]}x{s[2]}_t{s[3]}x{s[4]}_s{s[6]}_b{s[7]}" for s in SHAPES])
def test_schedule_invariants(shape, policy):
    _check(*shape, policy)


def test_schedule_invariants_random():
    rng = np.random.default_rng(5)
    for _ in range(60):
        M, N, K = (int(x) for x in rng.integers(1, 3000, 3))
        bm, bn = int(rng.choice([64, 128, 256])), int(rng.choice([64, 128, 256]))
        bk = int(rng.choice([16, 32]))
        slots = int(rng.integers(1, 400))
        batch = int(rng.integers(1, 4))
        for policy in (AUTO, WHOLE, STREAM_K, TAIL_SPLIT):
            _check(M, N, K, bm, bn, bk, slots, batch, policy)


def test_auto_policy_choices():
    # 4096^3 on 128x256 tiles: three whole-tile waves, then stream-K over the
    # 56 leftover tiles (at least a third of the 152 slots).
    _, info = sg.sgemm_test_schedule(4096, 4096, 4096, 128, 256, 32, 152, AUTO)
    assert info["dp_tiles"] == 456 and info["sk_ctas"] == 152
    # 4096 x 3001 x 2049 on 128x128 tiles: 8 leftover tiles are under a third
    # of the slots, so the last full wave joins the stream-K region.
    _, info = sg.sgemm_test_schedule(4096, 3001, 2049, 128, 128, 32, 152, AUTO)
    assert info["dp_tiles"] == 4 * 152 and info["sk_ctas"] == 152
    # 16384^3: the last wave is 99.8 % full, so whole tiles only.
    _, info = sg.sgemm_test_schedule(16384, 16384, 16384, 128, 256, 32, 152, AUTO)
    assert info["sk_ctas"] == 0 and info["dp_tiles"] == info["tiles"]
    # 1536^3 on 128x128 tiles: one wave, 94.7 % full, stays whole tiles (>= 90 %).
    _, info = sg.sgemm_test_schedule(1536, 1536, 1536, 128, 128, 32, 152, AUTO)
    assert info["sk_ctas"] == 0
    # 8192^3 on 128x256 tiles: 13.47 waves, 96.2 % of the slots busy under
    # whole tiles; after a full wave that is evened out: 13 whole-tile waves,
    # then stream-K over the 72 leftover tiles.
    _, info = sg.sgemm_test_schedule(8192, 8192, 8192, 128, 256, 32, 152, AUTO)
    assert info["dp_tiles"] == 13 * 152 and info["sk_ctas"] == 152
