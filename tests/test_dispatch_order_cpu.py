"""The work-item order of the tile list (host logic mirrored by the tests that read
moe_dispatch's tile list): every tile in exactly one item, groups self-consistent, and
the experts with several items spread evenly between those with one."""
import numpy as np
import pytest

from support import cluster_items, dispatch_items, dispatch_order, dispatch_tile_first


@pytest.mark.parametrize("seed", range(8))
def test_dispatch_items_is_a_regrouping_of_the_expert_order(seed):
    """Every tile in exactly one item, each expert's tiles consecutive from its first
    tile, its group its pairs then its single, groups in the dispatch order."""
    rng = np.random.default_rng(seed)
    nt = list(rng.choice([0, 1, 1, 1, 2, 3, 4, 7], size=int(rng.integers(1, 300))))
    got = dispatch_items(nt)
    assert len(got) == len(cluster_items(nt))
    tiles = sorted(t for it in got for t in it[:2] if t >= 0)
    assert tiles == list(range(sum(nt)))
    first, order = dispatch_tile_first(nt), dispatch_order(nt)
    assert sorted(order) == [e for e, n in enumerate(nt) if n > 0]
    k = 0
    for e in order:                         # groups: consecutive, sizes and firsts agree
        gc = nt[e] // 2 + nt[e] % 2
        assert all(got[k + j][2:4] == [k, gc] for j in range(gc))
        for j in range(gc):
            pair = j < nt[e] // 2
            assert got[k + j][:2] == [first[e] + 2 * j, first[e] + 2 * j + 1 if pair else -1]
            assert got[k + j][4] == int(pair)
        k += gc
    assert k == len(got)


def test_multi_item_experts_are_spread_evenly():
    nt = [1] * 90 + [4] * 10 + [2] * 50 + [5] * 5      # 140 one-item experts, 15 multi
    got = dispatch_items(nt)
    sizes, k = [], 0
    while k < len(got):
        sizes.append(got[k][3])
        k += got[k][3]
    multi_at = [i for i, g in enumerate(sizes) if g >= 2]
    gaps = np.diff(multi_at) - 1                         # one-item groups in between
    assert len(multi_at) == 15 and gaps.min() >= 140 // 15 - 1 and gaps.max() <= 140 // 15 + 1


def test_all_one_kind():
    """With one kind of expert only, the order is the expert order (cluster_items)."""
    for nt in ([1] * 7, [3] * 7, [2, 0, 2], []):
        assert dispatch_items(nt) == cluster_items(nt)
