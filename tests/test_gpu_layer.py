"""Parity of route / dispatch / combine / whole layer with the CPU oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_03_gb300 import api, configs, inputs
from support import (bf16_dev, bits, device_weights, dispatch_items, dispatch_tile_first,
                     getter, host_experts,
                     host_workload, shared_of, to_dev, unpack_sf_atoms, within_tol)

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "small_contig", "small_masked", "small_eplb", "small_sbo"]


def eplb_for(cfg, idx_host):
    if cfg.N_phys == cfg.N:
        return None
    return oracle.eplb_build_map(oracle.expert_counts(idx_host, cfg.N), cfg.N, cfg.N_phys)


# ------------------------------------------------------------------- route
@pytest.mark.parametrize("name", SMALL + ["decode", "sbo"])
def test_route_bit_exact(dev, name):
    cfg, x, W, bias = host_workload(name)
    r = api.route(cfg, bf16_dev(x), to_dev(W), to_dev(bias))
    torch.cuda.synchronize()
    idx, w, lg = oracle.route(x, W, bias, cfg, want_logits=True)
    got_lg = r["logits"][: cfg.B * cfg.N * 4].view(torch.float32).cpu().numpy().reshape(cfg.B, cfg.N)
    assert np.array_equal(got_lg.view(np.uint32), lg.view(np.uint32))
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx)
    assert np.array_equal(r["topk_w"].cpu().numpy().view(np.uint32), w.view(np.uint32))
    assert np.array_equal(r["counts"].cpu().numpy(), oracle.expert_counts(idx, cfg.N))


def _tie_workload(cfg, seed):
    """Router inputs full of exact ties: W repeats 16 distinct rows (every group holds the
    same logits), bias repeats three levels, and the batch mixes zero tokens (every logit
    0), tokens scaled by 2^12 (sigmoid saturates to exactly 0 or 1 for most experts) and
    plain normal tokens."""
    rng = np.random.default_rng(seed)
    base = (rng.standard_normal((16, cfg.H)) / np.sqrt(cfg.H)).astype(np.float32)
    W = base[np.arange(cfg.N) % 16]
    bias = (0.01 * (np.arange(cfg.N) % 3)).astype(np.float32)
    xf = rng.standard_normal((cfg.B, cfg.H)).astype(np.float32)
    xf[0::3] = 0.0
    xf[1::3] *= 4096.0
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)      # truncate to bf16
    return x, W, bias


@pytest.mark.parametrize("grouped", [True, False])
def test_route_ties_and_saturated_scores(dev, grouped):
    """Exact ties everywhere (equal logits across experts and groups, equal biased
    scores, sigmoid saturated to 0 or 1): the GPU's ids, weights, counts and logits equal
    the oracle's bit for bit, so both break every tie to the lower index alike."""
    if grouped:
        cfg = configs.MoEConfig("ties", B=96, H=256, N=256, K=8, I=128, n_group=8,
                                topk_group=4, score_fn=configs.SIGMOID, renorm=1,
                                route_scale=2.5)
    else:
        cfg = configs.MoEConfig("ties_softmax", B=96, H=256, N=32, K=4, I=128)
    x, W, bias = _tie_workload(cfg, 21)
    if not grouped:
        bias = None
    r = api.route(cfg, bf16_dev(x), to_dev(W), to_dev(bias))
    torch.cuda.synchronize()
    idx, w, lg = oracle.route(x, W, bias, cfg, want_logits=True)
    got_lg = r["logits"][: cfg.B * cfg.N * 4].view(torch.float32).cpu().numpy().reshape(cfg.B, cfg.N)
    assert np.array_equal(got_lg.view(np.uint32), lg.view(np.uint32))
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx)
    assert np.array_equal(r["topk_w"].cpu().numpy().view(np.uint32), w.view(np.uint32))
    assert np.array_equal(r["counts"].cpu().numpy(), oracle.expert_counts(idx, cfg.N))
    assert (idx[0] == np.sort(idx[0])).all() or grouped       # all-zero token: lowest ids
    assert len(np.unique(idx, axis=0)) < cfg.B                # ties really repeat choices


@pytest.mark.parametrize("N,G,TG,K", [(24, 8, 3, 4), (48, 6, 2, 5), (64, 1, 1, 6)])
def test_route_bit_exact_other_group_shapes(dev, N, G, TG, K):
    """Group shapes that do not fill whole lanes (the generic selection path)."""
    cfg = configs.MoEConfig("odd", B=77, H=256, N=N, K=K, I=128, n_group=G, topk_group=TG,
                            score_fn=configs.SIGMOID, renorm=1, route_scale=2.5,
                            bias_init="normal", seed=3)
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    r = api.route(cfg, bf16_dev(x), to_dev(W), to_dev(bias))
    torch.cuda.synchronize()
    idx, w = oracle.route(x, W, bias, cfg)
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx)
    assert np.array_equal(r["topk_w"].cpu().numpy().view(np.uint32), w.view(np.uint32))


@pytest.mark.parametrize("B,N,H", [(10000, 256, 256), (4000, 512, 256), (1000, 256, 256),
                                   (700, 512, 192), (300, 256, 160), (77, 64, 160),
                                   (201, 256, 384), (129, 40, 256)])
def test_route_logits_kernel_shapes(dev, B, N, H):
    """The logits kernel is chosen from B, N and H.  On 152 SMs these shapes take, in
    order: the fp32-widened 8x8 tile past the token-sliced range (256 experts) and at
    512 experts, the 2x2 tile with 64-wide chunks (H a multiple of 128, and of 64 only),
    the 32-wide-chunk kernel (H a multiple of 32 only) for a wide and a ragged batch,
    and the two-token tile of decode-size batches for an odd batch (its last token pair
    half empty) and an expert count that leaves a ragged expert tile.  All logits, ids
    and weights bit-exact."""
    kw = (dict(n_group=8, topk_group=3, K=16) if N == 512 else
          dict(n_group=8, topk_group=4, K=8) if N == 256 else dict(n_group=4, topk_group=2, K=6))
    cfg = configs.MoEConfig("shape", B=B, H=H, N=N, I=128, score_fn=configs.SIGMOID, renorm=1,
                            route_scale=2.5, bias_init="normal", seed=5, **kw)
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    r = api.route(cfg, bf16_dev(x), to_dev(W), to_dev(bias))
    torch.cuda.synchronize()
    idx, w, lg = oracle.route(x, W, bias, cfg, want_logits=True)
    got_lg = r["logits"][: B * N * 4].view(torch.float32).cpu().numpy().reshape(B, N)
    assert np.array_equal(got_lg.view(np.uint32), lg.view(np.uint32))
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx)
    assert np.array_equal(r["topk_w"].cpu().numpy().view(np.uint32), w.view(np.uint32))
    assert np.array_equal(r["counts"].cpu().numpy(), oracle.expert_counts(idx, N))

@pytest.mark.parametrize("name,B", [("prefill", 0), ("skew", 0), ("prefill", 6100),
                                    ("prefill", 9700), ("prefill", 3000), ("prefill", 5000)])
def test_route_full_size_sampled(dev, name, B):
    """Full B: routing of a sample of tokens bit-exact, counts consistent at any size.
    The batch sizes take the token-sliced logits kernel with 3 (3000), 4 (4096), 5
    (5000), 6 (6100), 7 (8192) and 8 (9700) tokens per warp (odd counts: token pairs
    plus one token on scalar fmas), with ragged last slices."""
    cfg, x, W, bias = host_workload(name)
    if B:
        cfg = cfg.with_(B=B)
        x = inputs.make_x(cfg)
    r = api.route(cfg, bf16_dev(x), to_dev(W), to_dev(bias))
    torch.cuda.synchronize()
    gi = r["topk_idx"].cpu().numpy()
    tok = np.random.default_rng(0).choice(cfg.B, 384, replace=False)
    tok = np.concatenate([tok, [0, cfg.B - 1]]).astype(np.int32)
    idx, w = oracle.route(x, W, bias, cfg, tokens=tok)
    assert np.array_equal(gi[tok], idx)
    assert np.array_equal(r["topk_w"].cpu().numpy()[tok].view(np.uint32), w.view(np.uint32))
    assert np.array_equal(r["counts"].cpu().numpy(), np.bincount(gi.reshape(-1), minlength=cfg.N))
    assert all(len(set(row)) == cfg.K for row in gi)   # K distinct experts per token


# ---------------------------------------------------------------- dispatch
def check_dispatch(cfg, x, idx, d, ref, fmt=api.FMT_FP8):
    rows = d["rows"]
    assert np.array_equal(d["counts"].cpu().numpy(), ref["cnt"])
    ro = d["row_of"].cpu().numpy()
    assert np.array_equal(ro, ref["row_of"])
    assert np.array_equal(d["src_of"].cpu().numpy(), ref["src_of"][:rows])
    valid = ro[ro >= 0]
    A = d["A"].cpu().numpy()
    if fmt == api.FMT_FP8:
        assert np.array_equal(A[valid], ref["A"][valid])
        sf = unpack_sf_atoms(d["A_sf"].cpu().numpy(), rows, cfg.H // 128)
        assert np.array_equal(sf[valid], ref["sf"][valid])
    else:
        assert np.array_equal(A[valid], ref["A"][valid])
    t = d["tiles"].cpu().numpy()
    nt = t[0]
    cnt = np.minimum(ref["cnt"], cfg.cap) if cfg.layout == configs.MASKED else ref["cnt"]
    assert nt == int(((cnt + 127) // 128).sum())
    ntp = (cnt + 127) // 128
    assert list(t[2:5]) == [int((ntp // 2).sum()), int((ntp % 2).sum()),
                            len(dispatch_items(list(ntp)))]
    tl = t[8: 8 + 8 * nt].reshape(nt, 8)
    first = dispatch_tile_first(list(ntp))     # tiles in the dispatch order, rows not
    for p in range(cfg.N_phys):
        base = ref["seg_start"][p] if cfg.layout == configs.CONTIG else p * cfg.cap
        for j in range(ntp[p]):
            assert list(tl[first[p] + j]) == [base + 128 * j, p, min(128, cnt[p] - 128 * j),
                                              first[p], ntp[p], 0, 0, 0]
    items = dispatch_items(list(ntp))
    mt = d["max_tiles"]
    got = t[8 + 8 * mt: 8 + 8 * mt + 8 * len(items)].reshape(-1, 8)
    assert [list(r[:5]) for r in got] == items


@pytest.mark.parametrize("name", SMALL + ["decode", "sbo"])
def test_dispatch_bit_exact(dev, name):
    cfg, x, W, bias = host_workload(name)
    idx, _ = oracle.route(x, W, bias, cfg)
    emap = eplb_for(cfg, idx)
    ref = oracle.dispatch(x, idx, cfg, *(emap[:2] if emap else (None, None)))
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx), *(map(to_dev, emap[:2]) if emap else (None, None)),
                     shared=cfg.shared)
    torch.cuda.synchronize()
    assert api.read_status(d["status"]) == 0
    check_dispatch(cfg, x, idx, d, ref)
    if cfg.shared:
        q, sf = oracle.quantize_rows(oracle.bf16_to_f32(x))
        assert np.array_equal(d["As"].cpu().numpy()[: cfg.B], q)
        srows = d["As"].shape[0]
        got_sf = unpack_sf_atoms(d["As_sf"].cpu().numpy(), srows, cfg.H // 128)
        assert np.array_equal(got_sf[: cfg.B], sf)


def _every_finite_bf16(seed: int) -> np.ndarray:
    """All 65280 finite bf16 patterns twice, as [128][1024]: first sorted by magnitude
    (a 128-column block holds neighbouring magnitudes, so its scale spreads them over
    the e4m3 range: subnormal codes, saturation at 448, scales clamped at 2^-127), then
    shuffled (tiny values beside huge ones flush to zero); zeros pad the last row."""
    b = np.arange(1 << 16, dtype=np.uint32)
    fin = b[np.isfinite((b << 16).view(np.float32))]
    mag = np.abs((fin << 16).view(np.float32))
    v = np.concatenate([fin[np.argsort(mag, kind="stable")],
                        np.random.default_rng(seed).permutation(fin)]).astype(np.uint16)
    return np.concatenate([v, np.zeros(128 * 1024 - v.size, np.uint16)]).reshape(128, 1024)


@pytest.mark.parametrize("fmt", [api.FMT_FP8, api.FMT_FP8_F32])
def test_dispatch_quantises_every_finite_bf16(dev, fmt):
    """Every finite bf16 value through the dispatch's quantiser, with power-of-two and
    with binary32 scales: the routed copies' codes and scales and the shared expert's
    token-order rows equal the oracle's bit for bit."""
    cfg = configs.MoEConfig("bf16_all", B=128, H=1024, N=8, K=2, I=128, shared=True)
    x = _every_finite_bf16(12)
    t = np.arange(cfg.B)
    idx = np.stack([t % 8, (t + 3) % 8], 1).astype(np.int32)
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx), fmt=fmt, shared=True)
    torch.cuda.synchronize()
    assert api.read_status(d["status"]) == 0
    xf = oracle.bf16_to_f32(x)
    if fmt == api.FMT_FP8:
        check_dispatch(cfg, x, idx, d, oracle.dispatch(x, idx, cfg))
        q, sf = oracle.quantize_rows(xf)
        got_sf = unpack_sf_atoms(d["As_sf"].cpu().numpy(), d["As"].shape[0], cfg.H // 128)
        assert np.array_equal(d["As"].cpu().numpy()[: cfg.B], q)
        assert np.array_equal(got_sf[: cfg.B], sf)
        assert (q[:64] != 0).mean() > 0.9 and sf.min() == 0     # codes used, 2^-127 reached
    else:
        q, s = oracle.quantize_rows_f32(xf)
        ro = d["row_of"].cpu().numpy()
        tt, kk = np.nonzero(ro >= 0)
        A = d["A"].cpu().numpy()
        sfa = d["A_sf"].cpu().numpy().view(np.float32).reshape(d["A"].shape[0], cfg.H // 128)
        assert np.array_equal(A[ro[tt, kk]], q[tt])
        assert np.array_equal(sfa[ro[tt, kk]].view(np.uint32), s[tt].view(np.uint32))
        As = d["As"].cpu().numpy()[: cfg.B]
        Ssf = d["As_sf"].cpu().numpy().view(np.float32).reshape(-1, cfg.H // 128)[: cfg.B]
        assert np.array_equal(As, q) and np.array_equal(Ssf.view(np.uint32), s.view(np.uint32))


@pytest.mark.parametrize("name", ["prefill", "skew"])
def test_dispatch_full_size(dev, name):
    """Full-size dispatch on the oracle's full routing (the oracle routes all B tokens)."""
    cfg, x, W, bias = host_workload(name)
    idx, _ = oracle.route(x, W, bias, cfg)
    ref = oracle.dispatch(x, idx, cfg)
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx))
    torch.cuda.synchronize()
    check_dispatch(cfg, x, idx, d, ref)


def test_dispatch_capacity_overflow_sets_status(dev):
    cfg = configs.SMALL_MASKED
    x = inputs.make_x(cfg)
    idx = np.tile(np.arange(cfg.K, dtype=np.int32), (cfg.B, 1))      # all tokens -> experts 0..K-1
    ref = oracle.dispatch(x, idx, cfg)
    assert ref["dropped"]
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx))
    torch.cuda.synchronize()
    assert api.read_status(d["status"]) & 1
    check_dispatch(cfg, x, idx, d, ref)


def test_dispatch_bad_index_sets_status(dev):
    cfg = configs.SMALL_CONTIG
    x = inputs.make_x(cfg)
    idx = np.tile(np.arange(cfg.K, dtype=np.int32), (cfg.B, 1))
    idx[5, 1] = cfg.N + 3
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx))
    torch.cuda.synchronize()
    assert api.read_status(d["status"]) & 4
    assert d["row_of"].cpu().numpy()[5, 1] == -1


def test_empty_batch(dev):
    cfg = configs.SMALL_CONTIG.with_(B=0)
    x = torch.empty((0, cfg.H), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((0, cfg.K), dtype=torch.int32, device=dev)
    d = api.dispatch(cfg, x, idx)
    torch.cuda.synchronize()
    assert d["tiles"][0].item() == 0 and int(d["counts"].sum()) == 0


@pytest.mark.parametrize("name", ["small_contig", "small_masked", "small_sbo"])
def test_empty_batch_layer(dev, name):
    """B = 0 through the whole layer: every stage returns at once or runs with no work,
    the status stays clean, and the output has no rows."""
    cfg, _, W, bias = host_workload(name)
    cfg = cfg.with_(B=0)
    lay = api.MoELayer(cfg, to_dev(W), to_dev(bias), device_weights(host_experts(name)))
    out = lay.forward(torch.empty((0, cfg.H), dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    assert tuple(out.shape) == (0, cfg.H)
    assert int(lay.counts.sum()) == 0 and lay.tiles[0].item() == 0


@pytest.mark.parametrize("B", [1, 37, 300])
def test_route_at_the_largest_expert_count(dev, B):
    """512 experts in 8 groups of 64, top-3 groups, K = 16 (the largest K), sigmoid +
    bias: logits, ids, weights and counts bit-exact, for one token, a ragged batch and
    a wider one."""
    cfg = configs.MoEConfig("n512", B=B, H=512, N=512, K=16, I=128, n_group=8, topk_group=3,
                            score_fn=configs.SIGMOID, renorm=1, route_scale=2.5,
                            bias_init="normal", seed=9)
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    r = api.route(cfg, bf16_dev(x), to_dev(W), to_dev(bias))
    torch.cuda.synchronize()
    idx, w, lg = oracle.route(x, W, bias, cfg, want_logits=True)
    got_lg = r["logits"][: B * cfg.N * 4].view(torch.float32).cpu().numpy().reshape(B, cfg.N)
    assert np.array_equal(got_lg.view(np.uint32), lg.view(np.uint32))
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx)
    assert np.array_equal(r["topk_w"].cpu().numpy().view(np.uint32), w.view(np.uint32))
    assert np.array_equal(r["counts"].cpu().numpy(), oracle.expert_counts(idx, cfg.N))


@pytest.mark.parametrize("layout", [configs.CONTIG, configs.MASKED])
def test_dispatch_at_the_largest_physical_expert_count(dev, layout):
    """1024 physical experts (the scan's limit) behind 512 logical ones with an EPLB
    map of two columns, K = 16: rows, slots, tile list and bytes as the oracle's."""
    cfg = configs.MoEConfig("p1024", B=300, H=256, N=512, K=16, I=128, n_phys=1024,
                            layout=layout, cap=128, seed=3)
    rng = np.random.default_rng(4)
    x = inputs.make_x(cfg)
    idx = np.stack([rng.choice(cfg.N, cfg.K, replace=False) for _ in range(cfg.B)]).astype(np.int32)
    emap = oracle.eplb_build_map(oracle.expert_counts(idx, cfg.N), cfg.N, cfg.N_phys)
    ref = oracle.dispatch(x, idx, cfg, emap[0], emap[1])
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx), to_dev(emap[0]), to_dev(emap[1]))
    torch.cuda.synchronize()
    assert api.read_status(d["status"]) == 0
    check_dispatch(cfg, x, idx, d, ref)


def test_single_token_layer(dev):
    """B = 1 through the whole layer (one row per chosen expert, the shared expert's
    single row, a 128-row tile holding one valid row each)."""
    name = "small_masked"
    cfg, x, W, bias = host_workload(name)
    cfg1 = cfg.with_(B=1, shared=True)
    x1 = np.ascontiguousarray(x[:1])
    ex = host_experts(name)
    if "W13s" not in ex:
        s = inputs.make_shared_expert(cfg1)
        ex = dict(ex, W13s=s[0], W13s_sf=s[1], W2s=s[2], W2s_sf=s[3])
    lay, out = run_layer(cfg1, x1, W, bias, ex, None)
    ref = oracle.layer_tokens(cfg1, x1, W, bias, getter(ex), shared_of(ex))
    ok, err, bound = within_tol(oracle.bf16_to_f32(out), oracle.bf16_to_f32(ref["out"]))
    assert ok, (err, bound)


# ----------------------------------------------------------------- combine
@pytest.mark.parametrize("name", ["small_contig", "small_masked", "decode"])
def test_combine_bit_exact(dev, name):
    cfg, x, W, bias = host_workload(name)
    idx, w = oracle.route(x, W, bias, cfg)
    ref = oracle.dispatch(x, idx, cfg)
    rng = np.random.default_rng(3)
    Y = inputs.bf16_bits(rng.standard_normal((ref["rows"], cfg.H)).astype(np.float32))
    S = inputs.bf16_bits(rng.standard_normal((cfg.B, cfg.H)).astype(np.float32))
    out_ref = oracle.combine(Y, ref["row_of"], w, S)
    out = api.combine(bf16_dev(Y), to_dev(ref["row_of"]), to_dev(w), shared=bf16_dev(S))
    assert np.array_equal(bits(out), out_ref)
    out_ref = oracle.combine(Y, ref["row_of"], w)
    out = api.combine(bf16_dev(Y), to_dev(ref["row_of"]), to_dev(w))
    assert np.array_equal(bits(out), out_ref)


@pytest.mark.parametrize("K", [8, 16])
def test_combine_bit_exact_at_the_extremes(dev, K):
    """Rows drawn from every finite bf16 pattern (subnormals to 3.39e38), weights from
    fp32 subnormals to 1, a shared row, some ranks dropped: sums that underflow into
    fp32 subnormals (no flush to zero), overflow to infinity, or round to bf16's largest
    finite value or past it -- the GPU's bytes equal the oracle's."""
    rng = np.random.default_rng(31 + K)
    B, H, rows = 96, 512, 700
    b = np.arange(1 << 16, dtype=np.uint32)
    fin = b[np.isfinite((b << 16).view(np.float32))].astype(np.uint16)
    Y = rng.choice(fin, (rows, H))
    Y[:100] = (Y[:100] & 0x007F) | 0x7F00               # positive, exponent 2^127: sums overflow
    Y[100:200] &= 0x807F                                # subnormal rows (exponent 0)
    S = rng.choice(fin, (B, H))
    S[: B // 4] = 0
    w = rng.uniform(0, 1, (B, K)).astype(np.float32)
    w[:, 0] = 2.0 ** rng.integers(-149, 0, B)           # down to the smallest subnormal
    w[B // 2:, -1] = 1.0
    row_of = rng.integers(0, rows, (B, K)).astype(np.int32)
    row_of[B // 4: B // 2, :K // 2] = rng.integers(0, 100, (B // 4, K // 2))    # huge rows
    row_of[B // 2: 3 * B // 4] = rng.integers(100, 200, (B // 4, K))          # subnormal
    row_of[::7, 1] = -1                                 # dropped ranks
    for shared in (S, None):
        ref = oracle.combine(Y, row_of, w, shared)
        out = api.combine(bf16_dev(Y), to_dev(row_of), to_dev(w),
                          shared=None if shared is None else bf16_dev(shared))
        assert np.array_equal(bits(out), ref)
    f = oracle.bf16_to_f32(ref)                         # the cases occur (no shared row)
    sub = (ref & 0x7F80) == 0
    assert np.isinf(f).any() and not np.isnan(f).any()
    assert sub.sum() > 1000 and ((ref[sub] & 0x7F) != 0).sum() > 1000


def test_bf16_round_trip_is_exact(dev):
    cfg = configs.SMALL_CONTIG.with_(K=1)
    x = inputs.make_x(cfg)
    idx = (np.arange(cfg.B) % cfg.N).astype(np.int32).reshape(-1, 1)
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx), fmt=api.FMT_BF16)
    Y = d["A"].view(torch.bfloat16)
    out = api.combine(Y, d["row_of"], torch.ones((cfg.B, 1), dtype=torch.float32, device=dev))
    assert np.array_equal(bits(out), x)


def test_combine_poll_times_out_without_hanging(dev):
    cfg = configs.SMALL_MASKED
    x = inputs.make_x(cfg)
    idx = np.tile(np.arange(cfg.K, dtype=np.int32), (cfg.B, 1))
    rows = cfg.N * 256
    sig = torch.zeros(rows // 64, dtype=torch.int32, device=dev)        # nothing sets it
    row_of = to_dev(oracle.dispatch(x, idx, cfg, cap=256)["row_of"][:16])
    Y = torch.zeros((rows, cfg.H), dtype=torch.bfloat16, device=dev)
    st = api.new_status(dev)
    w = torch.ones((16, cfg.K), dtype=torch.float32, device=dev)
    api.combine(Y, row_of, w, signal=sig, threshold=4, timeout_ns=2_000_000, status=st)
    torch.cuda.synchronize()
    assert api.read_status(st) & 2


# ------------------------------------------------------------------- layer
def run_layer(cfg, x, W, bias, ex, emap=None, **kw):
    lay = api.MoELayer(cfg, to_dev(W), to_dev(bias), device_weights(ex), eplb_map=emap, **kw)
    out = lay.forward(bf16_dev(x))
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    return lay, bits(out)


@pytest.mark.parametrize("name", SMALL)
def test_layer_matches_oracle(dev, name):
    cfg, x, W, bias = host_workload(name)
    ex = host_experts(name)
    idx, _ = oracle.route(x, W, bias, cfg)
    emap = eplb_for(cfg, idx)
    lay, out = run_layer(cfg, x, W, bias, ex, emap)
    ref = oracle.layer_tokens(cfg, x, W, bias, getter(ex), shared_of(ex))
    ok, err, bound = within_tol(oracle.bf16_to_f32(out), oracle.bf16_to_f32(ref["out"]))
    assert ok, (err, bound)
    # determinism: a second run gives the same bytes
    out2 = bits(lay.forward())
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("name", ["small_masked", "small_contig", "small_sbo"])
def test_layer_graph_replay_matches_eager(dev, name):
    """A captured layer graph replays the same bytes as eager calls, on new inputs too
    (the graph reads the layer's x buffer at every launch)."""
    cfg, x, W, bias = host_workload(name)
    ex = host_experts(name)
    idx, _ = oracle.route(x, W, bias, cfg)
    lay, out_a = run_layer(cfg, x, W, bias, ex, eplb_for(cfg, idx))
    x2 = inputs.make_x(cfg.with_(seed=cfg.seed + 11))
    lay.forward(bf16_dev(x2))
    out_b = bits(lay.out)
    st = torch.cuda.Stream(device=dev)
    st.wait_stream(torch.cuda.current_stream())
    g = api.LayerGraph(lay, st)
    for xi, want in ((x, out_a), (x2, out_b), (x, out_a)):
        lay.x.copy_(bf16_dev(xi))
        st.wait_stream(torch.cuda.current_stream())
        lay.out.zero_()
        st.wait_stream(torch.cuda.current_stream())
        g.launch(st)
        torch.cuda.current_stream().wait_stream(st)
        torch.cuda.synchronize()
        assert np.array_equal(bits(lay.out), want)
    assert api.read_status(lay.status) == 0
    g.close()


def test_two_layers_on_two_streams(dev):
    """Two layers enqueued on two streams at once, three times over, give the bytes each
    gives alone: the library keeps no device state shared between calls (tensor maps
    travel as launch parameters, every scratch buffer is the caller's), and the input
    copy of ``forward(x, stream=s)`` is ordered on ``s``."""
    lays, alone = [], {}
    for name in ("small_contig", "small_masked"):
        cfg, x, W, bias = host_workload(name)
        lay = api.MoELayer(cfg, to_dev(W, dev), to_dev(bias, dev),
                           device_weights(host_experts(name), dev), device=dev)
        xd = bf16_dev(x, dev)
        alone[name] = lay.forward(xd).clone()
        lays.append((name, lay, xd))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(dev) for _ in lays]
    for rep in range(3):
        for (name, lay, xd), s in zip(lays, streams):
            lay.x.zero_()              # on the current stream: s orders its copy after it
            lay.forward(xd, stream=s)
        torch.cuda.synchronize()
        for name, lay, _ in lays:
            assert api.read_status(lay.status) == 0
            assert torch.equal(lay.out, alone[name]), (name, rep)


def test_layer_host_graph_matches_forward_host(dev):
    """A graph that includes the pinned host copies gives forward_host's bytes."""
    cfg, x, W, bias = host_workload("small_masked")
    ex = host_experts("small_masked")
    lay, out_a = run_layer(cfg, x, W, bias, ex)
    xh = torch.from_numpy(x).view(torch.bfloat16).pin_memory()
    oh = torch.zeros(cfg.B, cfg.H, dtype=torch.bfloat16).pin_memory()
    st = torch.cuda.Stream(device=dev)
    st.wait_stream(torch.cuda.current_stream())
    g = api.LayerGraph(lay, st, xh, oh)
    for _ in range(2):
        oh.zero_()
        g.launch(st)
        st.synchronize()
        assert np.array_equal(oh.view(torch.int16).numpy().view(np.uint16), out_a)
    g.close()


def test_layouts_and_eplb_agree_bitwise(dev):
    """Masked = contiguous, EPLB on = off: same rows, same weights -> same bytes."""
    base = configs.SMALL_EPLB
    cfg, x, W, bias = host_workload("small_eplb")
    ex = host_experts("small_eplb")
    idx, _ = oracle.route(x, W, bias, cfg)
    outs = []
    for c, em in ((base, eplb_for(base, idx)), (base.with_(n_phys=0), None),
                  (base.with_(n_phys=0, layout=configs.MASKED, cap=384), None)):
        outs.append(run_layer(c, x, W, bias, ex, em)[1])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def planned_map(cfg, idx_host, seed_shift=0, max_rep=4):
    """An EPLB map from the planner (the reduced EPLB workload on 2 nodes x 2 GPUs) for
    the recorded loads with the hottest expert's load x50, so it gets max_rep copies."""
    load = oracle.expert_counts(idx_host, cfg.N).astype(np.int64)
    load[np.argmax(load)] *= 50
    if seed_shift:
        load = np.roll(load, seed_shift)
    return api.eplb_plan(load, cfg.N, cfg.N_phys, cfg.n_group, 2, 4, max_rep)[0]


def test_dispatch_with_planned_replicas_bit_exact(dev):
    """Up to four replicas per expert (log2phys of four columns): the same rows,
    slots, counts and bytes as the oracle's dispatch with that map."""
    cfg, x, W, bias = host_workload("small_eplb")
    idx, _ = oracle.route(x, W, bias, cfg)
    emap = planned_map(cfg, idx)
    assert emap[1].max() == 4
    ref = oracle.dispatch(x, idx, cfg, emap[0], emap[1])
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx), to_dev(emap[0]), to_dev(emap[1]))
    torch.cuda.synchronize()
    assert api.read_status(d["status"]) == 0
    check_dispatch(cfg, x, idx, d, ref)


@pytest.mark.parametrize("layout", [configs.CONTIG, configs.MASKED])
@pytest.mark.parametrize("B", [1, 77, 128, 129])
def test_single_chunk_dispatch_with_planned_map(dev, B, layout):
    """Up to 128 tokens are counted inside the scan's block (one launch fewer); 129
    tokens take the separate count launch.  Both, with a planned map of four columns
    and in both layouts, give the oracle's rows, slots, tile list and bytes."""
    cfg0, x, W, bias = host_workload("small_eplb")
    cfg = cfg0.with_(B=B, layout=layout, cap=256 if layout == configs.MASKED else 0)
    xb = np.ascontiguousarray(x[:B])
    idx, _ = oracle.route(xb, W, bias, cfg)
    emap = planned_map(cfg, idx)
    assert emap[0].shape == (cfg.N, 4)
    ref = oracle.dispatch(xb, idx, cfg, emap[0], emap[1])
    d = api.dispatch(cfg, bf16_dev(xb), to_dev(idx), to_dev(emap[0]), to_dev(emap[1]))
    torch.cuda.synchronize()
    assert api.read_status(d["status"]) == 0
    check_dispatch(cfg, xb, idx, d, ref)

def test_layer_with_planned_eplb_and_map_swap_matches_no_eplb(dev):
    """Planned replicas read their logical expert's weights, so the layer output is
    the same bytes as without EPLB, before and after installing a new map."""
    base = configs.SMALL_EPLB
    cfg, x, W, bias = host_workload("small_eplb")
    ex = host_experts("small_eplb")
    idx, _ = oracle.route(x, W, bias, cfg)
    ref = run_layer(base.with_(n_phys=0), x, W, bias, ex, None)[1]
    lay, out = run_layer(base, x, W, bias, ex, planned_map(base, idx))
    assert np.array_equal(out, ref)
    lay.set_eplb_map(planned_map(base, idx, seed_shift=5))
    out2 = bits(lay.forward())
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    assert np.array_equal(out2, ref)


@pytest.mark.parametrize("name", ["small_masked", "small_sbo"])
def test_pipelined_host_steps_match_forward_host(dev, name):
    """Five host batches through the pipelined entry point (copies of neighbouring
    steps overlapping the layer, two device buffer pairs alternating) give each batch
    the bytes of a plain host-buffer call; inputs and outputs never cross steps."""
    cfg, x, W, bias = host_workload(name)
    ex = host_experts(name)
    lay = api.MoELayer(cfg, to_dev(W), to_dev(bias), device_weights(ex))
    rng = np.random.default_rng(5)
    batches = [x] + [np.ascontiguousarray(x[rng.permutation(cfg.B)]) for _ in range(4)]
    xh = [torch.from_numpy(b).view(torch.bfloat16).pin_memory() for b in batches]
    ref = []
    for h in xh:
        o = torch.empty_like(h).pin_memory()
        lay.forward_host(h, o)
        torch.cuda.synchronize()
        ref.append(o.view(torch.int16).numpy().copy())
    st = torch.cuda.Stream()
    outs = [torch.zeros_like(h).pin_memory() for h in xh]
    lay.forward_host_pipelined(xh, outs, stream=st)
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    for i in range(len(xh)):
        assert np.array_equal(outs[i].view(torch.int16).numpy(), ref[i]), i
    assert not np.array_equal(ref[0], ref[1])   # the batches differ


@pytest.mark.parametrize("name", ["small_contig", "small_eplb", "small_sbo"])
def test_layer_with_2sm_gemms_matches_single_cta(dev, name):
    """The whole layer with both GEMMs on the 2-SM kernel equals the one-CTA layer bit
    for bit."""
    cfg, x, W, bias = host_workload(name)
    ex = host_experts(name)
    idx, _ = oracle.route(x, W, bias, cfg)
    emap = eplb_for(cfg, idx)
    lay = api.MoELayer(cfg, to_dev(W), to_dev(bias), device_weights(ex), eplb_map=emap,
                       gemm_pairs=1)
    a = bits(lay.forward(bf16_dev(x)))
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    _, b = run_layer(cfg, x, W, bias, ex, emap, gemm_pairs=-1)
    assert np.array_equal(a, b)


def test_sbo_equals_sequential(dev):
    cfg, x, W, bias = host_workload("small_sbo")
    ex = host_experts("small_sbo")
    _, a = run_layer(cfg, x, W, bias, ex)
    _, b = run_layer(cfg.with_(sbo=False), x, W, bias, ex)
    assert np.array_equal(a, b)
