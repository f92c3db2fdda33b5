"""Pins of the CPU oracle against facts outside it (CPU only).

Each test ties one oracle function to something the oracle does not compute
itself: a library routine on a special case, a closed form, a brute-force search
on tiny inputs, an invariant, or a value printed by the pages.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_03_gb300 import configs, inputs


def f32(v):
    return float(np.float32(v))


def ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = a.astype(np.float32).view(np.int32).astype(np.int64)
    ib = b.astype(np.float32).view(np.int32).astype(np.int64)
    return np.abs(ia - ib)


# ------------------------------------------------------------------ exp / sigmoid
def test_exp_within_2ulp_of_fp64():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-87.0, 88.0, 400_000), rng.uniform(-2, 2, 200_000),
                        np.linspace(-87.3, 88.7, 100_001)]).astype(np.float32)
    got = oracle.exp_array(x)
    ref = np.exp(x.astype(np.float64)).astype(np.float32)   # correctly rounded ref (fp64 exp)
    assert ulp_diff(got, ref).max() <= 2
    assert oracle.exp(0.0) == 1.0
    assert oracle.exp(100.0) == math.inf and oracle.exp(-200.0) == 0.0


def test_exp_subnormal_range_and_monotone():
    x = np.linspace(-103.9, -87.0, 50_001).astype(np.float32)
    got = oracle.exp_array(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    # subnormal results: absolute error within two steps of the smallest subnormal
    assert np.all(np.abs(got - ref) <= 2 * 2.0 ** -149 + 4e-7 * ref)
    xs = np.sort(np.random.default_rng(2).uniform(-30, 30, 100_000).astype(np.float32))
    ys = oracle.exp_array(xs)
    assert np.all(np.diff(ys) >= 0)


def test_sigmoid_against_fp64():
    z = np.random.default_rng(3).normal(0, 4, 300_000).astype(np.float32)
    got = oracle.sigmoid_array(z)
    ref = (1.0 / (1.0 + np.exp(-z.astype(np.float64)))).astype(np.float32)
    assert ulp_diff(got, ref).max() <= 3
    assert oracle.sigmoid(0.0) == 0.5
    # symmetry sigma(-z) = 1 - sigma(z), up to a few ulp of 1
    assert np.abs(oracle.sigmoid_array(-z).astype(np.float64) + got - 1.0).max() < 4e-7


# --------------------------------------------------------------------------- e4m3
def test_e4m3_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def _e4m3_cases():
    vals = np.sort(np.unique(np.abs(oracle.e4m3_table()[~np.isnan(oracle.e4m3_table())])))
    mids = (vals[1:] + vals[:-1]) / 2
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)   # midpoints are exact in fp32
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(0))
    rnd = np.random.default_rng(4).uniform(0, 448, 2_000_000).astype(np.float32)
    small = np.random.default_rng(5).uniform(0, 2.0 ** -5, 500_000).astype(np.float32)
    pos = np.concatenate([vals.astype(np.float32), m32, up, dn, rnd, small])
    return np.concatenate([pos, -pos])


def test_e4m3_encode_matches_torch_rne_in_range():
    v = _e4m3_cases()
    got = oracle.e4m3_encode_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_e4m3_encode_every_fp32_pattern():
    """All 2^32 binary32 bit patterns: below 448 in magnitude the code is torch's
    round-to-nearest-even cast to float8_e4m3fn; from 448 up, infinities included, it
    saturates to the largest finite code of the same sign; NaN keeps its sign on the NaN
    code.  (Chunks on a thread pool: the oracle's C loop runs without the GIL.)"""
    from concurrent.futures import ThreadPoolExecutor
    step = 1 << 22
    base = np.arange(step, dtype=np.uint32)

    def chunk(lo):
        u = base + np.uint32(lo)
        v = u.view(np.float32)
        got = oracle.e4m3_encode_array(v)
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        big = ~(np.abs(v) < 448)                    # |v| >= 448, infinities, NaN
        sat = (((u >> 24).astype(np.uint8) & 0x80) |
               np.where(np.isnan(v), 0x7F, 0x7E).astype(np.uint8))
        return np.array_equal(got, np.where(big, sat, ref))

    with ThreadPoolExecutor(min(8, os.cpu_count() or 1)) as ex:
        bad = [lo for lo, ok in zip(range(0, 1 << 32, step),
                                    ex.map(chunk, range(0, 1 << 32, step))) if not ok]
    assert not bad, [hex(b) for b in bad[:4]]


def test_e4m3_encode_brute_force_nearest_ties_even():
    """Nearest representable value by exhaustive search; ties -> even code."""
    table = oracle.e4m3_table()
    fin = [c for c in range(256) if not np.isnan(table[c])]
    v = _e4m3_cases()[::37]
    got = oracle.e4m3_encode_array(v)
    tv = table[fin]
    for x, c in zip(v.astype(np.float64), got):
        d = np.abs(tv - x)
        best = np.flatnonzero(d == d.min())
        cand = [fin[i] for i in best]
        # equal distance: both signs of zero, or a genuine tie -> even mantissa
        if len(cand) > 1:
            cand = [k for k in cand if (k & 1) == 0 and (k & 0x80) == (0x80 if math.copysign(1, x) < 0 else 0)] or cand
        assert c in cand, (x, c, cand)


def test_e4m3_saturates_and_keeps_sign():
    for v in (448.0, 449.0, 464.0, 1e6, math.inf):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-(2.0 ** -11)) == 0x80      # rounds to -0
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00          # tie between 0 and 2^-9 -> even (0)
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02      # tie between 1 and 2 (x2^-9) -> 2


# ------------------------------------------------------------------- UE8M0 scale
def test_scale_exp_is_smallest_power_of_two():
    rng = np.random.default_rng(6)
    amax = np.concatenate([rng.uniform(0, 1, 20000) * 2.0 ** rng.integers(-60, 60, 20000),
                           448.0 * 2.0 ** np.arange(-30, 30),
                           np.nextafter(448.0 * 2.0 ** np.arange(-30, 30), np.inf)])
    amax = amax.astype(np.float32)
    for a in amax[::7]:
        a = float(a)
        if a == 0:
            continue
        e = oracle.scale_exp(a)
        assert a <= 448.0 * 2.0 ** e and a > 448.0 * 2.0 ** (e - 1), (a, e)
    assert oracle.scale_exp(0.0) == 0
    assert oracle.scale_exp(448.0) == 0 and oracle.scale_exp(f32(448.0 * (1 + 2 ** -20))) == 1
    assert oracle.scale_exp(2.0 ** -140) == -127 and oracle.scale_exp(3e38) == 120   # 448*2^119 < 3e38 <= 448*2^120


def test_quantize_row_round_trip_and_bound():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((64, 512)) * 2.0 ** rng.integers(-20, 20, (64, 1))).astype(np.float32)
    q, sf = oracle.quantize_rows(v)
    table = oracle.e4m3_table()
    blocks = np.abs(v).reshape(64, 4, 128).max(-1)
    e = sf.astype(np.int32) - 127
    assert np.all(blocks <= 448.0 * 2.0 ** e) and np.all(blocks > 448.0 * 2.0 ** (e - 1))
    deq = table[q].reshape(64, 4, 128) * 2.0 ** e[:, :, None]
    # relative error of an e4m3 RNE is at most 2^-4 of the value (normal range)
    err = np.abs(deq - v.reshape(64, 4, 128))
    assert np.all(err <= np.maximum(np.abs(v.reshape(64, 4, 128)) * 2.0 ** -4,
                                    2.0 ** -10 * 2.0 ** e[:, :, None]))
    # values that are exactly e4m3 * 2^e with amax = 448 * 2^e survive unchanged
    codes = rng.integers(0, 0x7E, (8, 256)).astype(np.uint8)
    codes[:, ::128] = 0x7E
    exact = (table[codes] * 2.0 ** -3).astype(np.float32)
    q2, sf2 = oracle.quantize_rows(exact)
    assert np.array_equal(q2, codes) and np.all(sf2 == 124)


def test_quantize_f32_scale_is_amax_over_448_and_codes_follow():
    """Binary32 scales: s = fp32(amax / 448) exactly as NumPy's float32 division gives
    it, q = e4m3 of NumPy's float32 quotient x / s (the encoder pinned above), a zero
    block gets s = 1 and zero codes, and each block's largest |x| lands on code 448."""
    rng = np.random.default_rng(8)
    v = (rng.standard_normal((32, 512)) * 2.0 ** rng.integers(-30, 30, (32, 1))).astype(np.float32)
    v[3, 128:256] = 0.0
    q, s = oracle.quantize_rows_f32(v)
    blocks = v.reshape(32, 4, 128)
    amax = np.abs(blocks).max(-1)
    want = np.where(amax == 0, np.float32(1), amax / np.float32(448)).astype(np.float32)
    assert want.dtype == np.float32 and np.array_equal(s, want)
    quot = (blocks / s[:, :, None]).astype(np.float32)       # float32 division, RNE
    assert np.array_equal(q.reshape(32, 4, 128), oracle.e4m3_encode_array(quot))
    assert np.all(q[3, 128:256] == 0) and s[3, 1] == 1.0
    table = oracle.e4m3_table()
    top = np.take_along_axis(q.reshape(32, 4, 128), np.abs(blocks).argmax(-1)[..., None], -1)
    assert np.all((np.abs(table[top]) == 448.0)[amax > 0])


def test_quantize_f32_round_trip_bound_and_power_of_two_case():
    """e4m3 RNE keeps |q s - x| within 2^-4 |x| (normal range) or 2^-10 s (subnormal
    codes); when every block's amax is 448 * 2^e the binary32 scale is exactly 2^e and
    the codes equal the power-of-two path's."""
    rng = np.random.default_rng(9)
    v = (rng.standard_normal((16, 384)) * 2.0 ** rng.integers(-10, 10, (16, 1))).astype(np.float32)
    q, s = oracle.quantize_rows_f32(v)
    deq = oracle.dequant_rows_f32(q, s).reshape(16, 3, 128)
    x = v.reshape(16, 3, 128).astype(np.float64)
    assert np.all(np.abs(deq - x) <= np.maximum(np.abs(x) * 2.0 ** -4,
                                                2.0 ** -10 * s[:, :, None].astype(np.float64)))
    table = oracle.e4m3_table()
    codes = rng.integers(0, 0x7E, (8, 256)).astype(np.uint8)
    codes[:, ::128] = 0x7E                                    # 448 in every block
    exact = (table[codes] * 2.0 ** -3).astype(np.float32)
    q2, s2 = oracle.quantize_rows_f32(exact)
    q3, sf3 = oracle.quantize_rows(exact)
    assert np.all(s2 == 2.0 ** -3) and np.array_equal(q2, codes) and np.array_equal(q2, q3)


def test_ffn_f32_scales_reduce_to_power_of_two_path():
    """With inputs whose 1x128 blocks have amax = 448 * 2^e, the binary32-scale FFN
    sees the same a as the power-of-two FFN; the two paths then differ only through h's
    scales (amax/448 against the next power of two), so y agrees within the e4m3 step of
    h and exactly wherever h's block amax is itself 448 * 2^e."""
    rng = np.random.default_rng(16)
    W13, W13_sf, W2, W2_sf = _tiny_expert(rng, H=256, I=256)
    table = oracle.e4m3_table()
    codes = rng.integers(0, 0x7E, (6, 256)).astype(np.uint8)
    codes[:, ::128] = 0x7E
    x = (table[codes] * 2.0 ** 2).astype(np.float32)
    q0, sf0 = oracle.quantize_rows(x)
    q1, s1 = oracle.quantize_rows_f32(x)
    assert np.array_equal(q0, q1) and np.all(s1 == 4.0)
    y0 = oracle.bf16_to_f32(oracle.expert_ffn(q0, sf0, W13, W13_sf, W2, W2_sf)).astype(np.float64)
    y1, hq, hs, h = oracle.expert_ffn(q1, s1, W13, W13_sf, W2, W2_sf, want_h=True, scale_fmt=1)
    y1 = oracle.bf16_to_f32(y1).astype(np.float64)
    assert np.abs(y1 - y0).max() <= 2.0 ** -3 * np.abs(y0).max()
    # h requantised with binary32 scales: the definition applied to the fp32 h
    hq2, hs2 = oracle.quantize_rows_f32(h.astype(np.float32))
    assert np.array_equal(hq, hq2) and np.array_equal(hs, hs2)


# -------------------------------------------------------------------------- logits
def _tiny_cfg(**kw):
    base = dict(name="t", B=1, H=128, N=8, K=2, I=128)
    base.update(kw)
    return configs.MoEConfig(**base)


def test_logits_are_sequential_fma_in_k_order():
    """x = [2^24, 1, -2^24, 0...], w = 1: in k order the 1 is absorbed (result 0);
    any other order that adds 1 after the cancellation would give 1."""
    cfg = _tiny_cfg(N=2, K=1)
    x = np.zeros((1, 128), np.float32)
    x[0, :3] = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    W = np.zeros((2, 128), np.float32)
    W[0, :3] = 1.0
    W[1, :3] = [1.0, 1.0, 0.0]
    _, _, lg = oracle.route(inputs.bf16_bits(x), W, None, cfg, want_logits=True)
    assert lg[0, 0] == 0.0 and lg[0, 1] == 2.0 ** 24


def test_logits_exact_on_integer_data_and_within_fp32_bound():
    rng = np.random.default_rng(8)
    cfg = _tiny_cfg(H=256, N=16, K=4)
    xi = rng.integers(-8, 9, (5, 256)).astype(np.float32)
    Wi = rng.integers(-8, 9, (16, 256)).astype(np.float32)
    _, _, lg = oracle.route(inputs.bf16_bits(xi), Wi, None, cfg, want_logits=True)
    assert np.array_equal(lg, (xi.astype(np.int64) @ Wi.T.astype(np.int64)).astype(np.float32))
    x = inputs.bf16_bits(rng.standard_normal((5, 256)).astype(np.float32))
    W = rng.standard_normal((16, 256)).astype(np.float32)
    _, _, lg = oracle.route(x, W, None, cfg, want_logits=True)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    ref = xf @ W.astype(np.float64).T
    bound = 256 * 2.0 ** -24 * (np.abs(xf) @ np.abs(W.astype(np.float64)).T)
    assert np.all(np.abs(lg - ref) <= bound * 1.01)


# --------------------------------------------------------------------------- top-k
def _dominates(c, S, eligible):
    """S ranks before every eligible expert outside it (score desc, index asc)."""
    for a in S:
        for b in eligible:
            if b in S:
                continue
            if not (c[a] > c[b] or (c[a] == c[b] and a < b)):
                return False
    return True


def _rank_ordered(c, idx):
    return all(c[idx[i]] > c[idx[i + 1]] or (c[idx[i]] == c[idx[i + 1]] and idx[i] < idx[i + 1])
               for i in range(len(idx) - 1))


def _brute_topk(c, eligible, K):
    sols = [S for S in itertools.combinations(eligible, K) if _dominates(c, set(S), eligible)]
    assert len(sols) == 1
    return set(sols[0])


@pytest.mark.parametrize("ties", [False, True])
def test_softmax_topk_brute_force(ties):
    """Plain top-K over N=8 (the tiny workload's router), all C(8,K) subsets."""
    rng = np.random.default_rng(9 + ties)
    cfg = _tiny_cfg(N=8, K=2)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    if ties:
        x = np.round(x)
    W = rng.standard_normal((8, 128)).astype(np.float32)
    if ties:
        W = np.round(W)
        W[3] = W[5]
    for K in (1, 2, 3, 8):
        c2 = cfg.with_(K=K)
        idx, w, lg = oracle.route(inputs.bf16_bits(x), W, None, c2, want_logits=True)
        for t in range(x.shape[0]):
            assert set(idx[t]) == _brute_topk(lg[t], list(range(8)), K)
            assert _rank_ordered(lg[t], idx[t])
            # softmax probabilities, not renormalised: w = exp(z-m)/sum exp(z-m)
            p = np.exp(lg[t].astype(np.float64) - lg[t].max())
            p /= p.sum()
            assert np.allclose(w[t], p[idx[t]], rtol=2e-6, atol=1e-9)
        if K == 8:
            assert np.allclose(w.sum(1), 1.0, atol=1e-5)


def test_group_limited_topk_brute_force():
    """N=8 in 2 groups of 4, keep 1 group, K=2; and N=12 in 4 groups of 3, keep 2."""
    rng = np.random.default_rng(11)
    for N, G, TG, K in ((8, 2, 1, 2), (12, 4, 2, 3), (16, 4, 2, 4)):
        cfg = _tiny_cfg(N=N, K=K, n_group=G, topk_group=TG, score_fn=configs.SIGMOID,
                        renorm=1, route_scale=2.5)
        x = rng.standard_normal((40, 128)).astype(np.float32)
        W = (rng.standard_normal((N, 128)) * 0.1).astype(np.float32)
        bias = (rng.standard_normal(N) * 0.1).astype(np.float32)
        bias[1] = bias[2]
        idx, w, lg = oracle.route(inputs.bf16_bits(x), W, bias, cfg, want_logits=True)
        gs = N // G
        for t in range(40):
            s = oracle.sigmoid_array(lg[t])
            c = (s + bias).astype(np.float32)
            gscore = [np.float32(np.sort(c[j * gs:(j + 1) * gs])[-1]) +
                      np.float32(np.sort(c[j * gs:(j + 1) * gs])[-2]) for j in range(G)]
            keep = _brute_topk(np.array(gscore, np.float32), list(range(G)), TG)
            elig = [e for e in range(N) if e // gs in keep]
            assert set(idx[t]) == _brute_topk(c, elig, K)
            assert _rank_ordered(c, idx[t])
            sel = s[idx[t]].astype(np.float64)
            assert np.allclose(w[t], 2.5 * sel / sel.sum(), rtol=1e-6)
            assert abs(w[t].astype(np.float64).sum() - 2.5) < 1e-5


def test_one_group_equals_plain_topk():
    rng = np.random.default_rng(12)
    x = inputs.bf16_bits(rng.standard_normal((50, 128)).astype(np.float32))
    W = rng.standard_normal((16, 128)).astype(np.float32)
    b = (rng.standard_normal(16) * 0.1).astype(np.float32)
    a = _tiny_cfg(N=16, K=4, score_fn=1, renorm=1, route_scale=2.5, n_group=1, topk_group=1)
    g = a.with_(n_group=4, topk_group=4)       # all groups kept == no group limit
    assert np.array_equal(oracle.route(x, W, b, a)[0], oracle.route(x, W, b, g)[0])


def test_bias_steers_choice_not_weight():
    rng = np.random.default_rng(13)
    cfg = _tiny_cfg(N=8, K=2, score_fn=1, renorm=0, route_scale=1.0)
    x = inputs.bf16_bits(rng.standard_normal((20, 128)).astype(np.float32))
    W = rng.standard_normal((8, 128)).astype(np.float32)
    bias = np.zeros(8, np.float32)
    bias[6] = 10.0                              # expert 6 always chosen
    idx, w, lg = oracle.route(x, W, bias, cfg, want_logits=True)
    assert np.all(idx[:, 0] == 6)
    assert np.array_equal(w[:, 0], oracle.sigmoid_array(lg[:, 6]))   # weight ignores the bias


# ---------------------------------------------------------------------------- EPLB
def test_eplb_map_replicates_hottest():
    counts = np.array([5, 9, 9, 1, 0, 7, 9, 3])
    l2p, rep, p2l = oracle.eplb_build_map(counts, 8, 11)
    assert list(np.flatnonzero(rep == 2)) == [1, 2, 6]
    assert l2p[1, 1] == 8 and l2p[2, 1] == 9 and l2p[6, 1] == 10   # ties -> lower index first
    assert list(p2l) == list(range(8)) + [1, 2, 6]
    for e in range(8):
        assert l2p[e, 0] == e and (rep[e] == 2 or l2p[e, 1] == e)
    l2p, rep, p2l = oracle.eplb_build_map(counts, 8, 8)
    assert np.all(rep == 1)


# ------------------------------------------------------------------------ dispatch
@pytest.mark.parametrize("name", ["tiny", "small_contig", "small_masked", "small_eplb"])
def test_dispatch_invariants(name):
    cfg = configs.ALL[name]
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    idx, w = oracle.route(x, W, bias, cfg)
    l2p = rep = None
    if cfg.N_phys != cfg.N:
        l2p, rep, _ = oracle.eplb_build_map(oracle.expert_counts(idx, cfg.N), cfg.N, cfg.N_phys)
    check_dispatch(cfg, x, idx, l2p, rep)


@pytest.mark.parametrize("layout", [configs.CONTIG, configs.MASKED])
def test_dispatch_invariants_with_planned_replicas(layout):
    """A planned map with up to 4 replicas per expert (4 columns in log2phys): token t
    of logical expert e lands on replica t mod rep[e] and every other invariant holds.
    The skewed loads make the planner give the hottest experts 3 or 4 replicas."""
    from oracle import eplb as oeplb
    cfg = configs.SMALL_EPLB.with_(layout=layout, cap=512 if layout else 0, n_phys=56)
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    idx, _ = oracle.route(x, W, bias, cfg)
    load = oracle.expert_counts(idx, cfg.N).astype(np.int64)
    load[int(np.argmax(load))] *= 50
    (l2p, rep, _), _ = oeplb.plan(load, cfg.N, cfg.N_phys, n_group=cfg.n_group, max_rep=4)
    l2p, rep = np.asarray(l2p, np.int32), np.asarray(rep, np.int32)
    assert l2p.shape == (cfg.N, 4) and rep.max() >= 3
    check_dispatch(cfg, x, idx, l2p, rep)


def check_dispatch(cfg, x, idx, l2p, rep):
    d = oracle.dispatch(x, idx, cfg, l2p, rep)
    B, K = idx.shape
    assert d["cnt"].sum() == B * K
    assert np.array_equal(np.bincount(d["phys"].reshape(-1), minlength=cfg.N_phys), d["cnt"])
    ro = d["row_of"]
    assert np.all(ro >= 0) and len(np.unique(ro)) == B * K
    assert np.array_equal(d["src_of"][ro], np.repeat(np.arange(B), K).reshape(B, K))
    assert (d["src_of"] >= 0).sum() == B * K
    q, sf = oracle.quantize_rows(oracle.bf16_to_f32(x))
    assert np.array_equal(d["A"][ro.reshape(-1)], np.repeat(q, K, axis=0))
    assert np.array_equal(d["sf"][ro.reshape(-1)], np.repeat(sf, K, axis=0))
    base = d["seg_start"] if cfg.layout == 0 else np.arange(cfg.N_phys + 1) * cfg.cap
    if cfg.layout == 0:
        assert np.all(base % 128 == 0)
        assert np.array_equal(np.diff(base), (d["cnt"] + 127) // 128 * 128)
    for p in range(cfg.N_phys):
        pos = np.argwhere(d["phys"] == p)           # (t, k) pairs in ascending order
        assert np.array_equal(ro[pos[:, 0], pos[:, 1]], base[p] + np.arange(len(pos)))
    if l2p is not None:
        for t in range(B):
            for k in range(K):
                e = idx[t, k]
                assert d["phys"][t, k] == l2p[e, t % rep[e]]


def test_dispatch_capacity_drop():
    cfg = configs.SMALL_MASKED
    x = inputs.make_x(cfg)
    idx = np.zeros((cfg.B, cfg.K), np.int32)
    idx[:] = np.arange(cfg.K)                     # every token -> experts 0..K-1
    d = oracle.dispatch(x, idx, cfg, cap=16)
    assert d["dropped"]
    assert np.all(d["row_of"][:16] >= 0) and np.all(d["row_of"][16:] == -1)


def test_bf16_pass_through_round_trip_is_exact():
    """K=1, w=1, identity expert: dispatch(bf16) then combine returns x bit-exactly."""
    cfg = configs.SMALL_CONTIG.with_(K=1)
    x = inputs.make_x(cfg)
    idx = (np.arange(cfg.B) % cfg.N).astype(np.int32).reshape(-1, 1)
    d = oracle.dispatch(x, idx, cfg, fmt=1)
    Y = d["A"].view(np.uint16)
    out = oracle.combine(Y, d["row_of"], np.ones((cfg.B, 1), np.float32))
    assert np.array_equal(out, x)


def test_identity_expert_combine_is_weighted_sum():
    cfg = configs.SMALL_CONTIG
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    idx, w = oracle.route(x, W, bias, cfg)
    d = oracle.dispatch(x, idx, cfg, fmt=1)
    out = oracle.bf16_to_f32(oracle.combine(d["A"].view(np.uint16), d["row_of"], w))
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    ref = xf * w.astype(np.float64).sum(1, keepdims=True)
    assert np.allclose(out, ref, rtol=2 ** -7, atol=1e-6)     # one bf16 rounding


def test_combine_exact_sum_with_shared_and_dropped_rows():
    """Integer rows, power-of-two weights and an integer shared-expert row make every fp32
    partial sum exact, so out[t] must be bf16-RNE (torch) of the exact sum of w * Y over
    the rows that token t's row_of names (scattered, some dropped), plus S[t] once."""
    rng = np.random.default_rng(16)
    B, K, H = 24, 3, 128
    rows = B * K + 5
    Yv = rng.integers(-600, 600, (rows, H)).astype(np.float32)      # beyond bf16's 8 bits
    Sv = rng.integers(-600, 600, (B, H)).astype(np.float32)
    Yv = torch.from_numpy(Yv).bfloat16().float().numpy()              # bf16-exact inputs
    Sv = torch.from_numpy(Sv).bfloat16().float().numpy()
    to_bits = lambda a: torch.from_numpy(a).bfloat16().view(torch.int16).numpy().view(np.uint16)
    row_of = rng.permutation(rows)[: B * K].reshape(B, K).astype(np.int32)
    row_of[rng.random((B, K)) < 0.15] = -1                            # dropped copies
    w = (2.0 ** rng.integers(-3, 3, (B, K))).astype(np.float32)
    for S in (None, Sv):
        out = oracle.bf16_to_f32(oracle.combine(to_bits(Yv), row_of, w,
                                                None if S is None else to_bits(S)))
        ref = np.zeros((B, H))
        for t in range(B):
            for k in range(K):
                if row_of[t, k] >= 0:
                    ref[t] += float(w[t, k]) * Yv[row_of[t, k]].astype(np.float64)
            if S is not None:
                ref[t] += S[t]
        assert np.all(np.abs(ref) < 2 ** 24)                          # exact in fp32
        want = torch.from_numpy(ref.astype(np.float32)).bfloat16().float().numpy()
        assert np.array_equal(out, want)


# ----------------------------------------------------------------------------- FFN
def _tiny_expert(rng, H=128, I=128):
    W13, W13_sf = inputs.make_fp8_matrix(2 * I, H, (int(rng.integers(1 << 30)), 99, 0))
    W2, W2_sf = inputs.make_fp8_matrix(H, I, (int(rng.integers(1 << 30)), 98, 0))
    return W13, W13_sf, W2, W2_sf


def test_ffn_brute_force_exact_rationals():
    """Tiny expert by explicit loops in exact rational arithmetic (sigmoid via math.exp)."""
    rng = np.random.default_rng(14)
    W13, W13_sf, W2, W2_sf = _tiny_expert(rng)
    xr = rng.standard_normal((2, 128)).astype(np.float32)
    q, sf = oracle.quantize_rows(xr)
    y, hq, hsf, h = oracle.expert_ffn(q, sf, W13, W13_sf, W2, W2_sf, want_h=True)
    T = oracle.e4m3_table()
    for r in range(2):
        a = [Fraction(T[q[r, k]]) * Fraction(2) ** (int(sf[r, 0]) - 127) for k in range(128)]
        for j in range(0, 128, 17):
            g = sum(a[k] * Fraction(T[W13[j, k]]) * Fraction(2) ** (int(W13_sf[0, 0]) - 127)
                    for k in range(128))
            u = sum(a[k] * Fraction(T[W13[128 + j, k]]) * Fraction(2) ** (int(W13_sf[1, 0]) - 127)
                    for k in range(128))
            ref = float(g) / (1.0 + math.exp(-float(g))) * float(u)
            assert abs(h[r, j] - ref) <= 1e-12 * max(1.0, abs(ref))
        hv = [Fraction(T[hq[r, k]]) * Fraction(2) ** (int(hsf[r, 0]) - 127) for k in range(128)]
        for o in range(0, 128, 13):
            yv = float(sum(hv[k] * Fraction(T[W2[o, k]]) * Fraction(2) ** (int(W2_sf[0, 0]) - 127)
                           for k in range(128)))
            assert oracle.f32_to_bf16(np.array([yv], np.float32))[0] == y[r, o]


def test_ffn_scaling_invariants():
    """Power-of-two block scales act exactly: W2 scale +1 doubles y; the up half's
    scale +1 doubles h (gate/up not swapped); a zero up projection gives y = 0."""
    rng = np.random.default_rng(15)
    W13, W13_sf, W2, W2_sf = _tiny_expert(rng, H=256, I=256)
    q, sf = oracle.quantize_rows(rng.standard_normal((6, 256)).astype(np.float32))
    y = oracle.bf16_to_f32(oracle.expert_ffn(q, sf, W13, W13_sf, W2, W2_sf)).astype(np.float64)
    y2 = oracle.bf16_to_f32(oracle.expert_ffn(q, sf, W13, W13_sf, W2, W2_sf + 1))
    assert np.array_equal(y2, 2 * y)
    up_sf = W13_sf.copy()
    up_sf[2:] += 1
    y3 = oracle.bf16_to_f32(oracle.expert_ffn(q, sf, W13, up_sf, W2, W2_sf))
    assert np.array_equal(y3, 2 * y)
    W13z = W13.copy()
    W13z[256:] = 0
    assert np.all(oracle.bf16_to_f32(oracle.expert_ffn(q, sf, W13z, W13_sf, W2, W2_sf)) == 0)


def test_layer_composition_by_power_of_two_experts():
    """Expert e is one base expert with its down scale raised by s[e], so its output for
    token t is exactly 2^s[e] y_t, y_t the base output (power-of-two scales act exactly);
    the shared expert is the base with scale +1, i.e. 2 y_t.  The whole layer must equal
    the combine of rows y_t with weights w[t,k] 2^s[idx[t,k]] (also exact), token by
    token: a wrong expert, token or weight pairing in the gather or scatter breaks it.
    Dropped copies leave their term out."""
    rng = np.random.default_rng(17)
    cfg = _tiny_cfg(B=40, H=256, N=16, K=4, n_group=4, topk_group=2, score_fn=configs.SIGMOID,
                    renorm=1, route_scale=2.5)
    x = inputs.bf16_bits(rng.standard_normal((cfg.B, cfg.H)).astype(np.float32))
    W = (rng.standard_normal((cfg.N, cfg.H)) * 0.1).astype(np.float32)
    bias = (rng.standard_normal(cfg.N) * 0.1).astype(np.float32)
    W13, W13_sf, W2, W2_sf = _tiny_expert(rng, H=256, I=128)
    shift = rng.integers(0, 4, cfg.N)
    up = lambda d: (W2_sf.astype(np.int64) + int(d)).astype(np.uint8)
    get = lambda e: (W13, W13_sf, W2, up(shift[e]))
    q, sf = oracle.quantize_rows(oracle.bf16_to_f32(x))
    y = oracle.expert_ffn(q, sf, W13, W13_sf, W2, W2_sf)
    two_y = oracle.expert_ffn(q, sf, W13, W13_sf, W2, up(1))
    assert np.array_equal(oracle.bf16_to_f32(two_y), 2 * oracle.bf16_to_f32(y))
    idx, w = oracle.route(x, W, bias, cfg)
    assert len(np.unique(shift[idx])) > 1
    w_scaled = (w * 2.0 ** shift[idx]).astype(np.float32)
    tok_rows = np.repeat(np.arange(cfg.B, dtype=np.int32)[:, None], cfg.K, 1)
    dropped = rng.random((cfg.B, cfg.K)) < 0.2
    for drop in (None, dropped):
        got = oracle.layer_tokens(cfg, x, W, bias, get, shared=(W13, W13_sf, W2, up(1)),
                                  dropped=drop)
        assert np.array_equal(got["topk_idx"], idx)
        ro = tok_rows if drop is None else np.where(drop, -1, tok_rows).astype(np.int32)
        assert np.array_equal(got["out"], oracle.combine(y, ro, w_scaled, two_y))
    sub = [5, 0, 39, 17]                     # a token list gives those tokens' rows
    got = oracle.layer_tokens(cfg, x, W, bias, get, shared=(W13, W13_sf, W2, up(1)), tokens=sub)
    assert np.array_equal(got["out"], oracle.combine(y, tok_rows, w_scaled, two_y)[sub])


# --------------------------------------------------------------------------- golden
def test_golden_decode_dispatch_volume():
    """Per-rank decode dispatch volume b*K*H*s printed by the DeepEP page."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "decode_dispatch_volume.txt")
    vals = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = float(v)
    cfg = configs.DECODE
    b = vals["b"]
    assert (b, vals["K"], vals["H"]) == (cfg.B, cfg.K, cfg.H)
    # the e4m3 row bytes the oracle's dispatch writes for the decode workload
    from support import host_workload
    cfg, x, W, bias = host_workload("decode")
    idx, _ = oracle.route(x, W, bias, cfg)
    d = oracle.dispatch(x, idx, cfg)
    rows = int((d["row_of"] >= 0).sum())
    assert rows == cfg.B * cfg.K                     # nothing dropped at capacity 128
    code_bytes = rows * cfg.H * vals["s"]
    assert np.count_nonzero(d["A"][d["row_of"][d["row_of"] >= 0]]) > 0.9 * code_bytes
    assert abs(code_bytes / 1e6 - vals["MB"]) < 0.05
    assert abs(vals["MB"] * 1e-3 / (vals["budget_us"] * 1e-6) - vals["GBps"]) / vals["GBps"] < 0.05
