"""The combine fused into the down GEMM ("DeepEP 完全拆解", §为什么 combine 比 dispatch 慢:
combine is a move plus a reduce; here the reduce is done by the GEMM that stores the
rows): its output equals the oracle's combine of the same Y bit for bit, in every GEMM
form (one CTA, CTA pairs with M=256 and M=128 units, binary32 scales), with ranks left
out by capacity, tokens left with no row at all, shared rows, and EPLB replicas."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_03_gb300 import api, configs
from support import bf16_dev, bits, device_weights, host_experts, host_workload, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pair_tiles,scale_fmt", [(0, 0), (1, 0), (0, 1)])
def test_fused_down_gemm_equals_combine(dev, pair_tiles, scale_fmt):
    """Masked layout, capacity 128: experts 1-3 receive all 200 tokens and expert 0 150,
    so tokens 178-199 lose every rank and tokens 128-177 keep one; expert 4 holds 50
    rows (a single tile of at most 64 rows: the M=128 pair form).  No shared expert."""
    cfg = configs.SMALL_MASKED.with_(shared=False)
    B, H, K = cfg.B, cfg.H, cfg.K
    _, x, _, _ = host_workload("small_masked")
    idx = np.tile(np.arange(K, dtype=np.int32), (B, 1))
    idx[:50, 0] = 4
    w = np.random.default_rng(5).uniform(0.1, 1.0, (B, K)).astype(np.float32)
    ex = host_experts("small_masked")
    wd = device_weights({k: ex[k] for k in ("W13", "W13_sf", "W2", "W2_sf")}, dev)
    scales = api.weight_scales_f32 if scale_fmt else api.pack_weight_scales
    st = api.new_status(dev)
    d = api.dispatch(cfg, bf16_dev(x, dev), to_dev(idx, dev),
                     fmt=api.FMT_FP8_F32 if scale_fmt else api.FMT_FP8, status=st)
    H1, H1_sf = api.grouped_gemm_fp8(api.GEMM_GATEUP_SWIGLU, d["A"], d["A_sf"], wd["W13"],
                                     scales(wd["W13_sf"]), d["tiles"], d["max_tiles"],
                                     status=st, pair_tiles=pair_tiles, scale_fmt=scale_fmt)
    out = torch.full((B, H), 7.0, dtype=torch.bfloat16, device=dev)   # overwritten
    fc = dict(row_of=d["row_of"], topk_w=to_dev(w, dev), src_of=d["src_of"],
              pending=torch.empty((B, H // 128), dtype=torch.int32, device=dev), out=out)
    api.fused_combine_prep(**fc)
    Y = api.grouped_gemm_fp8(api.GEMM_DOWN, H1, H1_sf, wd["W2"], scales(wd["W2_sf"]),
                             d["tiles"], d["max_tiles"], status=st, pair_tiles=pair_tiles,
                             scale_fmt=scale_fmt, combine=fc)
    torch.cuda.synchronize()
    assert api.read_status(st) == api._lib.STATUS_CAPACITY      # the drops, nothing else
    ro = d["row_of"].cpu().numpy()
    none = (ro < 0).all(1)
    assert none.sum() == 22 and ((ro >= 0).sum(1) == 1).sum() == 50
    got = bits(out)
    ref = oracle.combine(bits(Y), ro, w)
    assert np.array_equal(got, ref)
    assert np.array_equal(got, bits(api.combine(Y, d["row_of"], fc["topk_w"])))
    assert (got[none] == 0).all() and (got[~none] != 0).any()


@pytest.mark.parametrize("name", ["small_contig", "small_masked", "small_eplb"])
def test_layer_fused_equals_layer(dev, name):
    """The layer with the fused combine gives the bytes of the layer with the separate
    combine (and of the oracle's combine of its own Y), run after run."""
    cfg, x, W, bias = host_workload(name)
    ex = host_experts(name)
    wdev = device_weights(ex, dev)
    emap = None
    if cfg.N_phys != cfg.N:
        idx, _ = oracle.route(x, W, bias, cfg)
        emap = oracle.eplb_build_map(oracle.expert_counts(idx, cfg.N), cfg.N, cfg.N_phys)
    outs = []
    for fused in (False, True):
        lay = api.MoELayer(cfg.with_(fuse_combine=fused), to_dev(W, dev), to_dev(bias, dev), wdev,
                           eplb_map=emap, device=dev)
        outs.append(bits(lay.forward(bf16_dev(x, dev))))
        torch.cuda.synchronize()
        assert api.read_status(lay.status) == 0
    assert np.array_equal(outs[0], outs[1])
    Y = bits(lay.Y)
    ref = oracle.combine(Y, lay.row_of.cpu().numpy(), lay.topk_w.cpu().numpy(),
                         Y[lay.rows: lay.rows + cfg.B])
    assert np.array_equal(outs[1], ref)
    assert np.array_equal(outs[1], bits(lay.forward()))


@pytest.mark.parametrize("name", ["decode", "prefill", "skew"])
def test_layer_fused_full_size(dev, name):
    """Full-size workloads (CTA pairs at prefill and skew, one CTA per tile at decode):
    every token's output equals the oracle's combine of the layer's own Y."""
    cfg, x, W, bias = host_workload(name)
    cfg = cfg.with_(fuse_combine=True)
    lay = api.MoELayer(cfg, to_dev(W, dev), to_dev(bias, dev), device_weights(host_experts(name), dev),
                       device=dev)
    out = bits(lay.forward(bf16_dev(x, dev)))
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    Y = bits(lay.Y)
    ref = oracle.combine(Y, lay.row_of.cpu().numpy(), lay.topk_w.cpu().numpy(),
                         Y[lay.rows: lay.rows + cfg.B])
    assert np.array_equal(out, ref)


def test_layer_fused_rejects_sbo(dev):
    cfg, x, W, bias = host_workload("small_sbo")
    lay = api.MoELayer(cfg.with_(fuse_combine=True), to_dev(W, dev), to_dev(bias, dev),
                       device_weights(host_experts("small_sbo"), dev), device=dev)
    with pytest.raises(api._lib.MoEError):
        lay.forward(bf16_dev(x, dev))
