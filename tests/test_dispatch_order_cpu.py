"""The work-item order of the tile list (host logic mirrored by the tests that read
moe_dispatch's tile list): every tile in exactly one item, groups self-consistent, and
the experts with several items spread evenly between those with one."""
import numpy as np
import pytest

from support import cluster_items, dispatch_items


@pytest.mark.parametrize("seed", range(8))
def test_dispatch_items_is_a_regrouping_of_the_expert_order(seed):
    rng = np.random.default_rng(seed)
    nt = list(rng.choice([0, 1, 1, 1, 2, 3, 4, 7], size=int(rng.integers(1, 300))))
    got, ref = dispatch_items(nt), cluster_items(nt)
    assert sorted(map(tuple, (it[:2] + it[4:] for it in got))) == \
        sorted(map(tuple, (it[:2] + it[4:] for it in ref)))
    k = 0
    while k < len(got):                     # groups: consecutive, sizes and firsts agree
        f, gc = got[k][2], got[k][3]
        assert f == k and all(got[k + j][2:4] == [f, gc] for j in range(gc))
        k += gc


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
    for nt in ([1] * 7, [3] * 7, [2, 0, 2], []):
        assert sorted(map(tuple, dispatch_items(nt))) == sorted(map(tuple, cluster_items(nt)))
