"""Binary32-scale mode (1x128 activation scales amax/448, per-k-block promotion in
software: the 1d2d scaling of the "Single Batch Overlap (SBO)" PR, §3, with float
scales) against the oracle: dispatch bit for bit, both GEMMs against fp64 products of
the dequantised operands, and whole layers within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_03_gb300 import api, configs, inputs
from support import (bf16_dev, bits, device_weights, getter, host_experts, host_workload,
                     shared_of, to_dev, within_tol)

pytestmark = pytest.mark.gpu

SMALL = ["small_contig", "small_masked", "small_eplb", "small_sbo"]


def _emap(cfg, idx):
    if cfg.N_phys == cfg.N:
        return None
    return oracle.eplb_build_map(oracle.expert_counts(idx, cfg.N), cfg.N, cfg.N_phys)


@pytest.mark.parametrize("name", SMALL + ["decode"])
def test_dispatch_f32_bit_exact(dev, name):
    """Rows and binary32 scales equal the oracle's quantize_rows_f32 of the token rows,
    placed by the oracle's permutation; the shared copy likewise."""
    cfg, x, W, bias = host_workload(name)
    idx, _ = oracle.route(x, W, bias, cfg)
    emap = _emap(cfg, idx)
    l2p, rep = (None, None) if emap is None else emap[:2]
    d = api.dispatch(cfg, bf16_dev(x), to_dev(idx), to_dev(l2p), to_dev(rep),
                     fmt=api.FMT_FP8_F32, shared=True)
    torch.cuda.synchronize()
    ref = oracle.dispatch(x, idx, cfg, log2phys=l2p, rep=rep)
    q, s = oracle.quantize_rows_f32(oracle.bf16_to_f32(x))
    ro = d["row_of"].cpu().numpy()
    assert np.array_equal(ro, ref["row_of"])
    assert np.array_equal(d["counts"].cpu().numpy(), ref["cnt"])
    rows = d["A"].shape[0]
    A = d["A"].cpu().numpy()
    sf = d["A_sf"].cpu().numpy().view(np.float32).reshape(rows, cfg.H // 128)
    t, k = np.nonzero(ro >= 0)
    assert np.array_equal(A[ro[t, k]], q[t])
    assert np.array_equal(sf[ro[t, k]].view(np.uint32), s[t].view(np.uint32))
    As = d["As"].cpu().numpy()[: cfg.B]
    Ssf = d["As_sf"].cpu().numpy().view(np.float32).reshape(-1, cfg.H // 128)[: cfg.B]
    assert np.array_equal(As, q) and np.array_equal(Ssf.view(np.uint32), s.view(np.uint32))


def _tiles(counts):
    """Dense tile list (no item table) for consecutive experts of 128-row tiles."""
    mt = sum(counts)
    t = np.zeros(8 + 16 * mt, np.int32)
    t[0], t[1] = mt, 128 * mt
    i = 0
    for e, c in enumerate(counts):
        for j in range(c):
            t[8 + 8 * (i + j): 8 + 8 * (i + j) + 5] = [128 * (i + j), e, 128 - 17 * (j == c - 1), i, c]
        i += c
    return t


@pytest.mark.parametrize("k", [512, 2048])
def test_down_gemm_f32_matches_fp64(dev, k):
    """Per-row binary32 activation scales over 13 binades and per-block weight scales:
    every stored row equals the fp64 product of the dequantised operands within a bf16
    rounding plus fp32 accumulation error."""
    counts, n = [2, 1, 3], 512
    E, mt = len(counts), sum(counts)
    rows = 128 * mt
    rng = np.random.default_rng(21)
    v = rng.standard_normal((rows, k)).astype(np.float32)
    v *= (2.0 ** rng.integers(-6, 7, (rows, k // 128))).repeat(128, axis=1).astype(np.float32)
    q, s = oracle.quantize_rows_f32(v)
    W = np.stack([inputs.make_fp8_matrix(n, k, (12, 4, e))[0] for e in range(E)])
    Wsf = rng.integers(117, 138, (E, n // 128, k // 128)).astype(np.uint8)
    t = _tiles(counts)
    st = api.new_status(dev)
    out = api.grouped_gemm_fp8(api.GEMM_DOWN, torch.from_numpy(q).to(dev),
                               torch.from_numpy(s).to(dev), torch.from_numpy(W).to(dev),
                               api.weight_scales_f32(torch.from_numpy(Wsf).to(dev)),
                               torch.from_numpy(t).to(dev), mt, status=st,
                               scale_fmt=api.SCALE_F32)
    torch.cuda.synchronize()
    assert api.read_status(st) == 0
    got = oracle.bf16_to_f32(bits(out)).astype(np.float64)
    a = oracle.dequant_rows_f32(q, s)
    i = 0
    for e, c in enumerate(counts):
        wd = oracle.dequant_blocks(W[e], Wsf[e])
        for j in range(c):
            nv = t[8 + 8 * (i + j) + 2]
            m = slice(128 * (i + j), 128 * (i + j) + nv)
            ref = a[m] @ wd.T
            refb = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
            tol = np.abs(refb) * 2.0 ** -7 + 2e-6 * np.sqrt(k / 512) * np.abs(ref).max()
            assert np.all(np.abs(got[m] - refb) <= tol), (e, j)
        i += c


def test_gateup_f32_matches_oracle(dev):
    """SwiGLU of the promoted products, requantised with binary32 scales: the scales are
    amax/448 of the GPU's own h within one e4m3 step of the fp64 h, and the dequantised
    h agrees with the fp64 h within the e4m3 step."""
    rows, I, H = 256, 256, 1024
    rng = np.random.default_rng(22)
    q, s = oracle.quantize_rows_f32(rng.standard_normal((rows, H)).astype(np.float32))
    W13, W13sf = inputs.make_fp8_matrix(2 * I, H, (6, 2, 0))
    t = _tiles([2])
    t[8 + 8 + 2] = 128
    st = api.new_status(dev)
    H1, H1_sf = api.grouped_gemm_fp8(api.GEMM_GATEUP_SWIGLU, torch.from_numpy(q).to(dev),
                                     torch.from_numpy(s).to(dev),
                                     torch.from_numpy(W13[None]).to(dev),
                                     api.weight_scales_f32(torch.from_numpy(W13sf[None]).to(dev)),
                                     torch.from_numpy(t).to(dev), 2, status=st,
                                     scale_fmt=api.SCALE_F32)
    torch.cuda.synchronize()
    assert api.read_status(st) == 0
    hq = H1.cpu().numpy()
    hs = H1_sf.cpu().numpy().view(np.float32).reshape(rows, I // 128)
    a = oracle.dequant_rows_f32(q, s)
    gu = a @ oracle.dequant_blocks(W13, W13sf).T
    g, u = gu[:, :I], gu[:, I:]
    h = g / (1 + np.exp(-g)) * u
    _, hs_ref = oracle.quantize_rows_f32(h.astype(np.float32))
    assert np.all(np.abs(hs - hs_ref) <= 2.0 ** -4 * hs_ref)
    ok, err, bound = within_tol(oracle.dequant_rows_f32(hq, hs), h, rel=2 ** -4, abs_=0)
    assert ok, (err, bound)


@pytest.mark.parametrize("name", SMALL + ["decode"])
def test_layer_f32_matches_oracle(dev, name):
    """The whole layer with binary32 scales against the oracle's layer with the same
    scales (every token at the reduced shapes, 64 at decode); deterministic."""
    cfg, x, W, bias = host_workload(name)
    cfg = cfg.with_(scale_fmt=1)
    ex = host_experts(name)
    idx, _ = oracle.route(x, W, bias, cfg)
    emap = _emap(cfg, idx)
    lay = api.MoELayer(cfg, to_dev(W), to_dev(bias), device_weights(ex), eplb_map=emap)
    out = bits(lay.forward(bf16_dev(x)))
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    tok = np.arange(cfg.B) if cfg.B <= 512 and name != "decode" else \
        np.sort(np.random.default_rng(3).choice(cfg.B, 64, replace=False))
    ref = oracle.layer_tokens(cfg, x, W, bias, getter(ex), shared_of(ex), tokens=tok,
                              scale_fmt=1)
    ok, err, bound = within_tol(oracle.bf16_to_f32(out[tok]), oracle.bf16_to_f32(ref["out"]))
    assert ok, (name, err, bound)
    assert np.array_equal(out, bits(lay.forward()))


def test_layer_f32_rejects_pairs(dev):
    cfg, x, W, bias = host_workload("small_contig")
    cfg = cfg.with_(scale_fmt=1)
    ex = host_experts("small_contig")
    lay = api.MoELayer(cfg, to_dev(W), to_dev(bias), device_weights(ex), gemm_pairs=1)
    with pytest.raises(Exception):
        lay.forward(bf16_dev(x))
