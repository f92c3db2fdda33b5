"""Grouped FP8 GEMM (tcgen05) against the oracle's dequantised fp64 products."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_03_gb300 import api, inputs
from support import bits, cluster_items, within_tol

pytestmark = pytest.mark.gpu


def pack_sf_atoms(sf: np.ndarray) -> np.ndarray:
    """UE8M0 bytes [rows][kb] -> SF atoms [rows/128][ceil(kb/4)][512] (layout of
    include/moe.h; bytes past the last column block are 0)."""
    rows, kb = sf.shape
    kg = (kb + 3) // 4
    p = np.zeros((rows, 4 * kg), np.uint8)
    p[:, :kb] = sf
    a = p.reshape(rows // 128, 4, 32, kg, 4).transpose(0, 3, 2, 1, 4)  # mb, g, r%32, r/32, j
    return a.reshape(-1).copy()


def dense_tiles(rows: int, experts_of_tiles=None) -> np.ndarray:
    mt = rows // 128
    t = np.zeros(8 + 8 * mt, np.int32)
    t[0], t[1] = mt, rows
    ex = np.zeros(mt, np.int32) if experts_of_tiles is None else np.asarray(experts_of_tiles)
    for i in range(mt):
        first = int(np.flatnonzero(ex == ex[i])[0])
        t[8 + 8 * i: 8 + 8 * i + 5] = [128 * i, ex[i], 128, first, int((ex == ex[i]).sum())]
    return t


def activations(rows, k, seed, spread=True):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((rows, k)).astype(np.float32)
    if spread:   # per-row and per-block magnitudes differ, so every scale byte matters
        v *= (2.0 ** rng.integers(-6, 7, (rows, k // 128))).repeat(128, axis=1).astype(np.float32)
    return oracle.quantize_rows(v)


@pytest.mark.parametrize("rows,n,k,E", [(128, 256, 128, 1), (256, 512, 512, 1), (384, 256, 1024, 3)])
def test_down_gemm_matches_fp64(dev, rows, n, k, E):
    q, sf = activations(rows, k, 1)
    W, Wsf = zip(*[inputs.make_fp8_matrix(n, k, (5, 77, e)) for e in range(E)])
    W, Wsf = np.stack(W), np.stack(Wsf)
    ex = np.arange(rows // 128) % E
    tiles = dense_tiles(rows, ex)
    # tiles of one expert must be consecutive: reorder rows by expert
    order = np.argsort(ex, kind="stable")
    tiles = dense_tiles(rows, ex[order])
    qo = q.reshape(-1, 128, k)[order].reshape(rows, k)
    sfo = sf.reshape(-1, 128, k // 128)[order].reshape(rows, k // 128)
    A = torch.from_numpy(qo).to(dev)
    A_sf = torch.from_numpy(pack_sf_atoms(sfo)).to(dev)
    Wd = torch.from_numpy(W).to(dev)
    Wsf_atoms = api.pack_weight_scales(torch.from_numpy(Wsf).to(dev))
    st = api.new_status(dev)
    out = api.grouped_gemm_fp8(api.GEMM_DOWN, A, A_sf, Wd, Wsf_atoms,
                               torch.from_numpy(tiles).to(dev), rows // 128, status=st)
    torch.cuda.synchronize()
    assert api.read_status(st) == 0
    got = oracle.bf16_to_f32(bits(out)).astype(np.float64)
    a = oracle.dequant_rows(qo, sfo)
    exs = ex[order].repeat(128)
    for e in range(E):
        m = exs == e
        ref = a[m] @ oracle.dequant_blocks(W[e], Wsf[e]).T
        refb = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
        # fp32 accumulation vs fp64: at most a bf16 rounding step apart
        assert np.all(np.abs(got[m] - refb) <= np.abs(refb) * 2.0 ** -7 + 1e-30 + 1e-6 * np.abs(ref).max()), e


def test_gateup_swiglu_matches_oracle(dev):
    rows, I, H = 256, 256, 512
    q, sf = activations(rows, H, 2, spread=False)
    W13, W13sf = inputs.make_fp8_matrix(2 * I, H, (6, 1, 0))
    tiles = dense_tiles(rows)
    A = torch.from_numpy(q).to(dev)
    A_sf = torch.from_numpy(pack_sf_atoms(sf)).to(dev)
    st = api.new_status(dev)
    H1, H1_sf = api.grouped_gemm_fp8(api.GEMM_GATEUP_SWIGLU, A, A_sf,
                                     torch.from_numpy(W13[None]).to(dev),
                                     api.pack_weight_scales(torch.from_numpy(W13sf[None]).to(dev)),
                                     torch.from_numpy(tiles).to(dev), rows // 128, status=st)
    torch.cuda.synchronize()
    assert api.read_status(st) == 0
    hq = H1.cpu().numpy()
    hsf = support_unpack(H1_sf.cpu().numpy(), rows, I // 128)
    a = oracle.dequant_rows(q, sf)
    gu = a @ oracle.dequant_blocks(W13, W13sf).T
    g, u = gu[:, :I], gu[:, I:]
    h = g / (1 + np.exp(-g)) * u
    hq_ref, hsf_ref = oracle.quantize_rows(h.astype(np.float32))
    # scale exponents: equal except where amax sits on a power-of-two boundary
    assert np.mean(hsf == hsf_ref) > 0.99 and np.all(np.abs(hsf.astype(int) - hsf_ref) <= 1)
    got = oracle.dequant_rows(hq, hsf)
    ok, err, bound = within_tol(got, h, rel=2 ** -4, abs_=0)
    assert ok, (err, bound)
    # most codes identical (fp32 vs fp64 h only moves values across rounding ties)
    assert np.mean(hq == hq_ref) > 0.98


def support_unpack(atoms, rows, kb):
    from support import unpack_sf_atoms
    return unpack_sf_atoms(atoms, rows, kb)


@pytest.mark.parametrize("kb", [1, 4, 5, 56])
def test_pack_unpack_sf_atoms_inverse(kb):
    sf = np.random.default_rng(0).integers(0, 255, (384, kb)).astype(np.uint8)
    atoms = pack_sf_atoms(sf)
    assert atoms.size == 384 // 128 * ((kb + 3) // 4) * 512
    assert np.array_equal(support_unpack(atoms, 384, kb), sf)
    # row 130, block 5: atom (1, 1), word 16*(2 % 32) + 4*(2 // 32), byte 1
    if kb > 5:
        assert atoms[(1 * ((kb + 3) // 4) + 1) * 512 + 32 + 1] == sf[130, 5]


def cluster_tile_list(tiles_per_expert, nvalid_of) -> np.ndarray:
    """Tile list (entries + cluster item table) for consecutive experts with the given
    M-tile counts; tile j of an expert holds nvalid_of(j) rows."""
    mt = sum(tiles_per_expert)
    t = np.zeros(8 + 16 * mt, np.int32)
    i = 0
    for e, c in enumerate(tiles_per_expert):
        for j in range(c):
            t[8 + 8 * (i + j): 8 + 8 * (i + j) + 5] = [128 * (i + j), e, nvalid_of(j), i, c]
        i += c
    items = cluster_items(tiles_per_expert)
    t[0:5] = [mt, 128 * mt, sum(c // 2 for c in tiles_per_expert),
              sum(c % 2 for c in tiles_per_expert), len(items)]
    for k, it in enumerate(items):
        t[8 + 8 * mt + 8 * k: 8 + 8 * mt + 8 * k + 5] = it
    return t


# valid rows of tile j of an expert: singles of 108-128 rows (M=256 pair MMAs with the
# odd CTA idle) or of 1-64 rows (M=128 pair MMAs), ragged pairs in both
NVALID = {"long_singles": lambda j: 128 - 5 * j, "short_singles": lambda j: [64, 100, 37, 128, 1][j]}


@pytest.mark.parametrize("pattern", sorted(NVALID))
@pytest.mark.parametrize("op", [0, 1])
def test_2sm_gemm_equals_single_cta(dev, op, pattern):
    """The 2-SM kernel (an expert's tile pairs on M=256 pair MMAs, its odd last tile in
    the same launch as an M=128 or M=256 pair MMA) gives the same bytes as one CTA per
    tile, for experts with 1, 2, 3 and 5 M tiles."""
    tiles_per_expert = [1, 2, 3, 5, 2]
    E = len(tiles_per_expert)
    k, n = (512, 512) if op == 0 else (256, 768)
    mt = sum(tiles_per_expert)
    rows = 128 * mt
    q, sf = activations(rows, k, 7)
    W, Wsf = zip(*[inputs.make_fp8_matrix(n, k, (9, 55, e)) for e in range(E)])
    W, Wsf = np.stack(W), np.stack(Wsf)
    t = cluster_tile_list(tiles_per_expert, NVALID[pattern])
    A = torch.from_numpy(q).to(dev)
    A_sf = torch.from_numpy(pack_sf_atoms(sf)).to(dev)
    Wd = torch.from_numpy(W).to(dev)
    Wa = api.pack_weight_scales(torch.from_numpy(Wsf).to(dev))
    tl = torch.from_numpy(t).to(dev)
    outs = []
    for pairs in (0, 1):
        st = api.new_status(dev)
        o = api.grouped_gemm_fp8(op, A, A_sf, Wd, Wa, tl, mt, status=st, pair_tiles=pairs)
        torch.cuda.synchronize()
        assert api.read_status(st) == 0
        outs.append(o)
    res = [o.view(torch.int16) if op == 1 else o[0] for o in outs]
    for i0 in range(mt):                      # rows each tile stores
        nvalid = t[8 + 8 * i0 + 2]
        assert torch.equal(res[0][128 * i0: 128 * i0 + nvalid],
                           res[1][128 * i0: 128 * i0 + nvalid]), i0
    if op == 0:                               # and the h scales of those rows
        from support import unpack_sf_atoms
        valid = np.zeros(rows, bool)
        for i0 in range(mt):
            valid[128 * i0: 128 * i0 + t[8 + 8 * i0 + 2]] = True
        sfs = [unpack_sf_atoms(o[1].cpu().numpy(), rows, n // 256) for o in outs]
        assert np.array_equal(sfs[0][valid], sfs[1][valid])


@pytest.mark.parametrize("pattern", sorted(NVALID))
@pytest.mark.parametrize("k", [512, 2048])
def test_down_224_column_tiles_equal_single_cta(dev, k, pattern):
    """The DOWN GEMM on 224-column tiles with two accumulators (tile_n 224, weight scales
    as tile-aligned images), on one CTA per tile and on CTA pairs (every tile at M=256),
    gives the bytes of one CTA per tile on 256-column tiles, for experts with 1, 2, 3
    and 5 M tiles."""
    tiles_per_expert = [1, 2, 3, 5, 2]
    E, n = len(tiles_per_expert), 1792           # 8 tiles of 224, 7 of 256
    mt = sum(tiles_per_expert)
    q, sf = activations(128 * mt, k, 17)
    W = np.stack([inputs.make_fp8_matrix(n, k, (19, 5, e))[0] for e in range(E)])
    Wsf = np.random.default_rng(23).integers(117, 138, (E, n // 128, k // 128)).astype(np.uint8)
    t = cluster_tile_list(tiles_per_expert, NVALID[pattern])
    A, A_sf = torch.from_numpy(q).to(dev), torch.from_numpy(pack_sf_atoms(sf)).to(dev)
    Wd, Wsf_d = torch.from_numpy(W).to(dev), torch.from_numpy(Wsf).to(dev)
    tl = torch.from_numpy(t).to(dev)
    outs = []
    tiled = api.pack_weight_scales_tiled(Wsf_d, 224)
    for pairs, tile_n, scales in ((0, 0, api.pack_weight_scales(Wsf_d)), (1, 224, tiled),
                                  (0, 224, tiled)):
        st = api.new_status(dev)
        outs.append(api.grouped_gemm_fp8(api.GEMM_DOWN, A, A_sf, Wd, scales, tl, mt, status=st,
                                         pair_tiles=pairs, tile_n=tile_n))
        torch.cuda.synchronize()
        assert api.read_status(st) == 0
    for o in outs[1:]:
        for i0 in range(mt):
            nvalid = t[8 + 8 * i0 + 2]
            assert torch.equal(outs[0][128 * i0: 128 * i0 + nvalid].view(torch.int16),
                               o[128 * i0: 128 * i0 + nvalid].view(torch.int16)), i0


def test_tiled_weight_scale_images(dev):
    """moe_pack_weight_scales_tiled: image h of tile j holds, for tile row 128h + r, the
    scale of W row 224j + 128h + r (zero past the tile), in the SF atom layout."""
    E, n, k = 2, 1792, 640
    Wsf = np.random.default_rng(29).integers(0, 255, (E, n // 128, k // 128)).astype(np.uint8)
    img = api.pack_weight_scales_tiled(torch.from_numpy(Wsf).to(dev), 224).cpu().numpy()
    kg = (k // 128 + 3) // 4
    nt = n // 224
    img = img.reshape(E, nt, kg, 2, 512)
    from support import unpack_sf_atoms
    for e in range(E):
        for j in range(nt):
            got = np.concatenate([unpack_sf_atoms(img[e, j, :, h].reshape(-1), 128, k // 128)
                                  for h in range(2)])          # [256][kb]
            rows = 224 * j + np.arange(224)
            assert np.array_equal(got[:224], Wsf[e, rows // 128])
            assert not got[224:].any()


@pytest.mark.parametrize("k", [768, 4352])
@pytest.mark.parametrize("mode", ["one_cta", "pairs", "pairs_224", "one_cta_224"])
@pytest.mark.parametrize("last", [128, 50])
def test_weight_scale_bytes_per_block(dev, mode, k, last):
    """Weight scale bytes drawn per 128x128 block over 21 binades, K of 6 and 34
    k-blocks: the down GEMM still equals the fp64 product of the dequantised operands
    in every scheduling mode (a scale atom read for the wrong block, k-block or row
    half moves an output by a power of two), with full last tiles and with 50-row last
    tiles (the 2-SM kernel's M=128 singles)."""
    pairs, tile_n = int(mode.startswith("pairs")), 224 if mode.endswith("224") else 0
    tiles_per_expert = [2, 3, 1]
    E, n = len(tiles_per_expert), 1792 if tile_n else 512
    mt = sum(tiles_per_expert)
    rows = 128 * mt
    q, sf = activations(rows, k, 11)
    W = np.stack([inputs.make_fp8_matrix(n, k, (12, 3, e))[0] for e in range(E)])
    Wsf = np.random.default_rng(13).integers(117, 138, (E, n // 128, k // 128)).astype(np.uint8)
    nv = {}
    i = 0
    for c in tiles_per_expert:
        for j in range(c):
            nv[i + j] = last if j == c - 1 else 128
        i += c
    t = cluster_tile_list(tiles_per_expert, lambda j: 128)
    for i0, v in nv.items():
        t[8 + 8 * i0 + 2] = v
    st = api.new_status(dev)
    out = api.grouped_gemm_fp8(api.GEMM_DOWN, torch.from_numpy(q).to(dev),
                               torch.from_numpy(pack_sf_atoms(sf)).to(dev),
                               torch.from_numpy(W).to(dev),
                               (api.pack_weight_scales_tiled if tile_n else
                                api.pack_weight_scales)(torch.from_numpy(Wsf).to(dev)),
                               torch.from_numpy(t).to(dev), mt, status=st, pair_tiles=pairs,
                               tile_n=tile_n)
    torch.cuda.synchronize()
    assert api.read_status(st) == 0
    got = oracle.bf16_to_f32(bits(out)).astype(np.float64)
    a = oracle.dequant_rows(q, sf)
    i = 0
    for e, c in enumerate(tiles_per_expert):
        wd = oracle.dequant_blocks(W[e], Wsf[e])
        for j in range(c):
            m = slice(128 * (i + j), 128 * (i + j) + nv[i + j])
            ref = a[m] @ wd.T
            refb = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
            # bf16 rounding of the fp32 sum, plus fp32 accumulation error growing ~ sqrt(k)
            tol = np.abs(refb) * 2.0 ** -7 + 2e-6 * np.sqrt(k / 768) * np.abs(ref).max()
            assert np.all(np.abs(got[m] - refb) <= tol), (e, j)
        i += c


def test_layer_down_224_column_tiles(dev):
    """A layer whose hidden size is a multiple of 224 (CTA pairs, then one CTA per tile): the
    down GEMM on 224-column tiles gives the layer the same bytes as on 256-column tiles,
    and the oracle's output for sampled tokens."""
    from combine_moe_route_03_gb300 import configs
    from support import bf16_dev, getter, shared_of, to_dev, within_tol
    cfg = configs.MoEConfig("mid224", B=2300, H=1792, N=32, K=4, I=512, n_group=4, topk_group=2,
                            score_fn=configs.SIGMOID, renorm=1, route_scale=2.5, shared=True,
                            bias_init="normal")
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    ex = inputs.make_all_experts(cfg)
    s = inputs.make_shared_expert(cfg)
    ex.update(W13s=s[0], W13s_sf=s[1], W2s=s[2], W2s_sf=s[3])
    wdev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in ex.items()}
    outs = []
    for d224, pairs in ((False, 1), (True, 1), (True, 0)):
        lay = api.MoELayer(cfg, to_dev(W, dev), to_dev(bias, dev), wdev, device=dev, down224=d224,
                           gemm_pairs=pairs)
        assert (lay.W2_sf_t224 is not None) == d224
        outs.append(bits(lay.forward(bf16_dev(x, dev))))
        torch.cuda.synchronize()
        assert api.read_status(lay.status) == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    tok = np.array([0, 1, 777, 1500, cfg.B - 1])
    ref = oracle.layer_tokens(cfg, x, W, bias, getter(ex), shared_of(ex), tokens=tok)
    ok, err, bound = within_tol(oracle.bf16_to_f32(outs[1][tok]), oracle.bf16_to_f32(ref["out"]))
    assert ok, (err, bound)
