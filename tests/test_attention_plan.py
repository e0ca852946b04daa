"""Host-side work split of the TMA-staged attention kernel (kvo_plan_attention).

Properties every plan must have, whatever the shape: the work items cover
each group's sparse tiles and then its window tiles exactly once, in order;
no item crosses a part boundary; the CTA ranges are contiguous, in order and
start on a multiple of the CTA's 4 warps; and no range costs much more than
an equal share (a tile costs 1, a work-item epilogue 12).
"""
import random

import pytest

from sparse_kv_cache_landmark_gb300 import kvo
from sparse_kv_cache_landmark_gb300.kvo import KvoError

TILE, WARPS, ITEM_COST = 16, 4, 12


def _check_plan(G, sp_tok, w_tok, grid):
    items, cta = kvo.plan_attention(G, sp_tok, w_tok, grid)
    items, cta = items.tolist(), cta.tolist()
    sp_t = -(-sp_tok // TILE)
    w_t = -(-w_tok // TILE)
    per_g = sp_t + w_t
    T = per_g * G
    used = len(cta) - 1
    assert used == max(1, min(grid, T))
    assert cta[0] == 0 and cta[-1] == len(items)
    assert all(a <= b for a, b in zip(cta, cta[1:]))
    # coverage: the items, in order, walk the global tile sequence once
    nxt = 0
    for g, part, t0, n in items:
        assert 0 <= g < G and part in (0, 1) and n >= 1 and t0 >= 0
        plen = sp_t if part == 0 else w_t
        assert t0 + n <= plen, "an item crosses a part boundary"
        start = g * per_g + (t0 if part == 0 else sp_t + t0)
        assert start == nxt, "tiles skipped or repeated"
        nxt = start + n
    assert nxt == T
    # ranges start on a warp multiple; cost balance
    n_parts = G * ((sp_t > 0) + (w_t > 0))
    share = (T + ITEM_COST * n_parts) / used
    for j in range(used):
        rng = items[cta[j]:cta[j + 1]]
        if not rng:
            continue
        g, part, t0, _ = rng[0]
        start = g * per_g + (t0 if part == 0 else sp_t + t0)
        assert start % WARPS == 0
        cost = sum(n + ITEM_COST for *_, n in rng)
        # rounding a bound down to the warp multiple moves it by < 4 tiles, each of
        # which may start a part (1 + ITEM_COST each); plus one item that continues a part
        # (its epilogue is not among the split's cost points) and integer division
        slack = (WARPS - 1) * (1 + ITEM_COST) + ITEM_COST + 1
        assert cost <= share + slack, (G, sp_tok, w_tok, grid, j, cost, share)
    return items, cta


def test_llama_layer_plan():
    # 128 groups x (64 blocks x 32 tokens + 512 window): 20,480 tiles over the step plan's 228 CTAs
    items, cta = _check_plan(128, 64 * 32, 512, 228)
    assert len(cta) == 229
    assert sum(n for *_, n in items) == 128 * (128 + 32)


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes(seed):
    rnd = random.Random(seed)
    for _ in range(60):
        G = rnd.choice([1, 2, 3, 7, 16, 64, 128, 320, 512])
        k = rnd.choice([1, 3, 8, 16, 64, 128, 400])
        B = rnd.choice([1, 16, 32, 64])
        W = rnd.choice([0, 1, 15, 16, 64, 512, 543])
        grid = rnd.choice([1, 2, 3, 38, 152, 228, 304, 5000])
        _check_plan(G, k * B, W, grid)


def test_window_only_and_sparse_only():
    _check_plan(5, 0, 100, 7)
    _check_plan(5, 64, 0, 7)


def test_more_ctas_than_tiles():
    items, cta = _check_plan(1, 16, 0, 50)
    assert len(cta) == 2 and items == [[0, 0, 0, 1]]


@pytest.mark.parametrize("args", [(0, 64, 16, 4), (4, 0, 0, 4), (4, -1, 16, 4), (4, 64, 16, 0)])
def test_bad_shapes_are_rejected(args):
    with pytest.raises(KvoError):
        kvo.plan_attention(*args)
