"""EPLB placement planner (moe_eplb_plan): the oracle pinned to brute force, closed
forms and invariants; the library's host planner bit-exact against the oracle; the
load recorder that re-plans periodically.  CPU only."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

from combine_moe_route_03_gb300 import _lib, api
from oracle import eplb as oeplb


@pytest.fixture(scope="module")
def L():
    from combine_moe_route_03_gb300 import build
    build.build()
    return _lib.load()


def skewed_load(rng, N, s=1.2, scale=1000):
    """Zipf-like loads over a seeded permutation of the experts (the skew workload's
    shape), plus noise; some experts cold (0)."""
    r = np.arange(1, N + 1, dtype=np.float64)
    v = scale * r ** -s
    v = np.floor(v * rng.uniform(0.5, 1.5, N)).astype(np.int64)
    v[rng.random(N) < 0.1] = 0
    return v[rng.permutation(N)]


def check_invariants(m, load, N_log, N_phys, n_group, n_nodes, n_gpus, max_rep):
    l2p, rep, p2l = (np.asarray(a) for a in m)
    assert rep.sum() == N_phys and rep.min() >= 1 and rep.max() <= max_rep
    # every physical slot holds one logical expert; e appears rep[e] times
    assert np.array_equal(np.bincount(p2l, minlength=N_log), rep)
    for e in range(N_log):
        ids = np.flatnonzero(p2l == e)
        assert np.array_equal(l2p[e, : rep[e]], ids)
        assert np.all(l2p[e, rep[e]:] == ids[0])
    if n_nodes > 1 and n_group % n_nodes == 0:
        # hierarchical: a group's replicas all sit on one node, n_group / n_nodes per node
        gs, per = N_log // n_group, N_phys // n_nodes
        node_of_group = []
        for g in range(n_group):
            nodes = {int(p) // per for e in range(g * gs, (g + 1) * gs) for p in np.flatnonzero(p2l == e)}
            assert len(nodes) == 1
            node_of_group.append(nodes.pop())
        assert np.all(np.bincount(node_of_group, minlength=n_nodes) == n_group // n_nodes)


# ------------------------------------------------------------------ oracle pins
@pytest.mark.parametrize("seed", range(40))
def test_replication_is_the_min_max_optimum(seed):
    """Step 2 gives each spare slot to the largest load per replica; for min over rep of
    max_e load[e] / rep[e] (sum rep = slots, 1 <= rep <= max_rep) that greedy is
    optimal.  Brute force over every rep vector on tiny inputs."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 6))
    max_rep = int(rng.integers(1, 5))
    slots = int(rng.integers(n, n * max_rep + 1))
    load = [int(v) for v in rng.integers(0, 50, n)]
    rep = oeplb.replicate(load, list(range(n)), slots, max_rep)
    got = max(Fraction(load[e], rep[e]) for e in range(n))
    best = min(max(Fraction(load[e], r[e]) for e in range(n))
               for r in itertools.product(range(1, max_rep + 1), repeat=n) if sum(r) == slots)
    assert sum(rep.values()) == slots and got == best


def test_group_packing_worked_example():
    """Two nodes, four groups of loads 5, 4, 3, 2: 5 -> node 0, 4 -> node 1, 3 -> node 1
    (4 < 5), node 1 is full, 2 -> node 0: {5, 2} and {4, 3}, both 7."""
    assert oeplb.node_groups([5, 4, 3, 2], 2) == [[0, 3], [1, 2]]
    # equal loads: the lighter node first, ties to the lower node
    assert oeplb.node_groups([1, 1, 1, 1], 2) == [[0, 2], [1, 3]]


def test_uniform_load_is_perfectly_balanced():
    """Equal loads, no spare slots, N_phys a multiple of the GPUs: every GPU carries
    the same load (balance exactly 1), experts in index order on each GPU's turn."""
    m, bal = oeplb.plan([7] * 32, 32, 32, n_group=4, n_nodes=2, n_gpus=8, max_rep=2)
    assert bal == 1.0
    check_invariants(m, [7] * 32, 32, 32, 4, 2, 8, 2)


def test_one_slot_per_gpu_balance_closed_form():
    """One slot per GPU: each GPU holds one replica, so the balance is the mean over
    the max of the replica loads load[e] / rep[e].  The two spare slots go to 12
    (12 > 9) and then 9 (9 > 12/2 = 6 = load of expert 4)."""
    load = [12, 3, 0, 9, 6, 1]
    m, bal = oeplb.plan(load, 6, 8, n_gpus=8, max_rep=3)
    l2p, rep, p2l = m
    assert rep == [2, 1, 1, 2, 1, 1]
    w = [Fraction(load[e], rep[e]) for e in p2l]
    assert abs(bal - float(sum(w) / len(w) / max(w))) < 1e-15


def test_identity_plan_without_spare_slots():
    """N_phys = N_log on one GPU: one replica each, placed heaviest first."""
    load = [4, 9, 9, 1, 0]
    (l2p, rep, p2l), bal = oeplb.plan(load, 5, 5)
    assert rep == [1] * 5 and p2l == [1, 2, 0, 3, 4] and bal == 1.0


@pytest.mark.parametrize("seed", range(12))
def test_oracle_plan_invariants(seed):
    rng = np.random.default_rng(seed)
    n_group = [1, 4, 8][seed % 3]
    N = 8 * n_group * int(rng.integers(1, 4))
    n_nodes = [1, 2, 4][seed % 3]
    n_gpus = n_nodes * int(rng.integers(1, 4))
    spg = int(rng.integers(N // n_gpus + 1, N // n_gpus + 4)) if N % n_gpus == 0 else 0
    if not spg:
        pytest.skip("shape")
    P = spg * n_gpus
    max_rep = int(rng.integers(2, 6))
    if P > N * max_rep:
        pytest.skip("shape")
    load = skewed_load(rng, N)
    m, bal = oeplb.plan(load, N, P, n_group, n_nodes, n_gpus, max_rep)
    check_invariants(m, load, N, P, n_group, n_nodes, n_gpus, max_rep)
    assert 0.0 < bal <= 1.0


# --------------------------------------------------------- library vs oracle
SHAPES = [  # N_log, N_phys, n_group, n_nodes, n_gpus, max_rep
    (256, 288, 8, 4, 32, 2),     # the pages' 256 -> 288 on 4 nodes
    (256, 288, 8, 4, 36, 4),
    (256, 288, 8, 1, 8, 8),      # flat
    (256, 256, 8, 2, 16, 1),     # placement only
    (32, 40, 4, 2, 4, 4),        # the reduced EPLB workload
    (64, 96, 8, 3, 12, 3),       # 8 groups on 3 nodes: not divisible -> flat
    (12, 24, 3, 3, 6, 8),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("seed", range(3))
def test_library_plan_matches_oracle(L, shape, seed):
    N, P, G, nodes, gpus, R = shape
    rng = np.random.default_rng(100 + seed)
    load = skewed_load(rng, N, s=[0.8, 1.2, 2.0][seed], scale=[10**3, 10**6, 10**9][seed])
    got, gbal = api.eplb_plan(load, N, P, G, nodes, gpus, R)
    ref, rbal = oeplb.plan(load, N, P, G, nodes, gpus, R)
    for g, r in zip(got, ref):
        assert np.array_equal(g, np.asarray(r, np.int32))
    assert abs(gbal - rbal) <= 1e-12
    check_invariants(got, load, N, P, G, nodes, gpus, R)


def test_replication_improves_balance_on_skew(L):
    """The pages' case: spare slots holding copies of the hot experts raise the
    balance (mean / max GPU load) over placement without replicas."""
    load = skewed_load(np.random.default_rng(7), 256, s=1.2, scale=10**6)
    _, b0 = api.eplb_plan(load, 256, 256, 8, 4, 32, 1)
    _, b1 = api.eplb_plan(load, 256, 288, 8, 4, 36, 4)
    assert b1 > b0


def test_plan_rejects_bad_shapes(L):
    load = np.ones(16, np.int64)
    bad = [
        (16, 15, 1, 1, 1, 2),   # fewer slots than experts
        (16, 40, 1, 1, 1, 2),   # more slots than 2 replicas each
        (16, 18, 3, 1, 1, 2),   # groups do not divide the experts
        (16, 18, 1, 2, 3, 2),   # GPUs not a multiple of the nodes
        (16, 18, 1, 1, 4, 2),   # slots not a multiple of the GPUs
        (16, 16, 1, 1, 1, 9),   # max_rep above 8
    ]
    for N, P, G, nodes, gpus, R in bad:
        with pytest.raises(_lib.MoEError):
            api.eplb_plan(load, N, P, G, nodes, gpus, R)
    with pytest.raises(_lib.MoEError):
        api.eplb_plan(np.full(16, 1 << 40, np.int64), 16, 16)


# ------------------------------------------------------------------ recorder
def test_recorder_plans_every_period_from_the_recorded_loads(L):
    rng = np.random.default_rng(3)
    rec = api.EplbRecorder(32, 40, period=3, n_group=4, n_nodes=2, n_gpus=4, max_rep=4)
    total = np.zeros(32, np.int64)
    for step in range(3):
        c = rng.integers(0, 50, 32).astype(np.int32)
        total += c
        assert not rec.due()
        rec.observe(c)
    assert rec.due()
    m, bal = rec.plan()
    ref, rbal = oeplb.plan(total, 32, 40, 4, 2, 4, 4)
    assert all(np.array_equal(g, np.asarray(r, np.int32)) for g, r in zip(m, ref))
    assert not rec.due() and rec.load.sum() == 0          # a fresh window
    with pytest.raises(ValueError):
        rec.observe(np.zeros(31, np.int32))


# -------------------------------------------------------------- map validation
@pytest.mark.parametrize("seed", range(8))
def test_maps_from_both_builders_pass_the_layer_check(L, seed):
    """Every map the fixed builder and the planner make (library and oracle) is
    accepted when a layer installs it."""
    from combine_moe_route_03_gb300 import configs
    import oracle
    rng = np.random.default_rng(seed)
    for N, P in ((32, 40), (256, 288), (256, 256), (8, 16), (512, 1024)):
        counts = rng.integers(0, 5, N) * rng.integers(0, 3, N)
        api.check_eplb_map(api.eplb_build_map(counts, N, P), N, P)
        api.check_eplb_map(oracle.eplb_build_map(counts, N, P), N, P)
    for shape in SHAPES:
        N, P, G, nodes, gpus, R = shape
        load = skewed_load(rng, N)
        api.check_eplb_map(api.eplb_plan(load, N, P, G, nodes, gpus, R)[0], N, P)
    cfg = configs.SMALL_EPLB
    api.check_eplb_map(api.eplb_plan(skewed_load(rng, cfg.N) * 50, cfg.N, cfg.N_phys,
                                     cfg.n_group, 2, 4, 4)[0], cfg.N, cfg.N_phys)


def test_layer_check_rejects_broken_maps(L):
    l2p, rep, p2l = api.eplb_plan(skewed_load(np.random.default_rng(1), 32), 32, 40, 4, 2, 4, 4)[0]
    api.check_eplb_map((l2p, rep, p2l), 32, 40)
    hot = int(np.argmax(rep))
    broken = []
    r = rep.copy(); r[hot] -= 1; broken.append((l2p, r, p2l))            # counts short of the slots
    p = p2l.copy(); p[l2p[hot, 1]] = (hot + 1) % 32; broken.append((l2p, rep, p))   # disagree
    m = l2p.copy(); m[0, 0] = 40; broken.append((m, rep, p2l))           # slot out of range
    p = p2l.copy(); p[0] = -1; broken.append((l2p, rep, p))              # expert out of range
    broken.append((l2p[:31], rep[:31], p2l))                              # shape
    for b in broken:
        with pytest.raises(ValueError):
            api.check_eplb_map(b, 32, 40)
    with pytest.raises(ValueError):
        api.check_eplb_map((l2p, rep, p2l), 32, 48)                       # wrong slot count


@pytest.mark.parametrize("shape", [(32, 40, 4, 2, 4, 4), (16, 16, 1, 1, 1, 1), (8, 64, 2, 2, 8, 8),
                                   (1, 1, 1, 1, 1, 1), (1, 8, 1, 1, 8, 8)])
def test_degenerate_loads_and_shapes(L, shape):
    """All-zero loads (a window with no tokens) and extreme shapes (one expert, one slot
    per GPU, eight replicas each): the library equals the oracle, the map is valid, and
    an idle window's balance is 1 (no GPU is the maximum)."""
    N, P, G, nodes, gpus, R = shape
    for load in (np.zeros(N, np.int64), np.arange(1, N + 1, dtype=np.int64)):
        got, gbal = api.eplb_plan(load, N, P, G, nodes, gpus, R)
        ref, rbal = oeplb.plan(list(load), N, P, G, nodes, gpus, R)
        for g, r in zip(got, ref):
            assert np.array_equal(g, np.asarray(r, np.int32))
        assert abs(gbal - rbal) <= 1e-12
        check_invariants(got, load, N, P, G, nodes, gpus, R)
        api.check_eplb_map(got, N, P)
        if not load.any():
            assert gbal == 1.0
