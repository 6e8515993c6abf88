"""The host's item plan for the persistent d = 128 forward (no GPU needed).

The plan lists, per CTA, the (head, query tile) items it runs.  These tests check what the kernel
relies on and what the plan is for: every item exactly once; each CTA's planned work (key tiles plus a
fixed cost of two tiles per item) within one item of every other CTA's when it takes its last item
(greedy list scheduling); heads taken in groups whose K/V streams total at most 32 MiB, a group's
items all planned before the next group's, heaviest causal tile first within a group.
"""

import numpy as np
import pytest

from differential_attention_03_gb300 import binding as da
from differential_attention_03_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    da.lib()


def _tiles(qt, n, causal):
    nt = (n + 127) // 128
    return min(nt, qt + 1) if causal else nt


CASES = [  # grid, units, nqt, qt0, n, causal, kv bytes per unit
    (152, 24, 32, 0, 4096, True, 4096 * 1024),     # two batches x 12 heads, n = 4096, d = 128: 3 groups of 8
    (148, 24, 32, 0, 4096, True, 4096 * 1024),
    (152, 12, 64, 0, 8192, True, 8192 * 1024),     # 96 MiB: 3 groups of 4
    (152, 40, 8, 0, 1024, False, 1024 * 1024),     # 40 MiB: 2 groups of 20, not causal
    (152, 12, 8, 24, 4096, True, 4096 * 1024),     # a token range of the host pipeline (tiles 24 .. 31)
    (7, 3, 3, 0, 300, True, 300 * 1024),           # fewer items than SMs would give: tiny grid
]


@pytest.mark.parametrize("grid,units,nqt,qt0,n,causal,kvb", CASES)
def test_plan_is_a_balanced_grouped_permutation(grid, units, nqt, qt0, n, causal, kvb):
    res = da.debug_item_plan(grid, units, nqt, qt0, n, causal, kvb)
    assert res is not None
    first, items = res
    assert first[0] == 0 and int(first[grid]) == units * nqt
    assert np.all(np.diff(first.astype(np.int64)) >= 0)
    # every item exactly once
    assert sorted(items.tolist()) == list(range(units * nqt))
    cost = lambda it: _tiles(qt0 + nqt - 1 - it % nqt, n, causal) + 2  # noqa: E731
    # greedy: when a CTA took its last item, no other CTA had less planned work than its start
    loads = []
    for c in range(grid):
        lst = items[first[c]:first[c + 1]].tolist()
        loads.append(sum(cost(i) for i in lst))
    biggest = max(cost(i) for i in range(units * nqt))
    assert max(loads) - min(loads) <= biggest
    # groups: sizes from the 32 MiB budget, planned in order, heaviest tile first inside a group
    budget = 32 << 20
    ngroups = max(1, -(-units * kvb // budget))
    ug = -(-units // ngroups)
    order = np.empty(units * nqt, dtype=np.int64)  # the position at which each item was planned
    # reconstruct the planning sequence: items are planned in the order group, tile (heaviest first), unit
    seq = [u * nqt + (nqt - 1 - ql) for g0 in range(0, units, ug) for ql in range(nqt - 1, -1, -1)
           for u in range(g0, min(units, g0 + ug))]
    order[np.array(seq)] = np.arange(len(seq))
    for c in range(grid):
        lst = items[first[c]:first[c + 1]]
        assert np.all(np.diff(order[lst]) > 0), "a CTA's list follows the planning sequence"
        groups = (lst // nqt) // ug
        assert np.all(np.diff(groups) >= 0), "a CTA finishes its items of a group before the next group's"


def test_plan_declines_launches_too_large():
    assert da.debug_item_plan(300, 24, 32, 0, 4096, True, 4096 * 1024) is None  # more than 256 CTAs
    assert da.debug_item_plan(152, 200, 32, 0, 4096, True, 4096 * 1024) is None  # more than 4096 items
