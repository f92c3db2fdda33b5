"""The four DeepSeek-V3-shaped workloads at full size, through moe_layer_forward,
against the oracle on sampled tokens (the oracle's FFN is fp64 NumPy and too slow
for every token; routing, counts and tile lists are checked at any size)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_03_gb300 import api, configs
from support import (bf16_dev, bits, device_weights, getter, host_experts, host_workload,
                     shared_of, to_dev, within_tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv3_dev(dev):
    ex = host_experts("decode")
    return ex, device_weights(ex, dev)


@pytest.mark.parametrize("name", ["decode", "sbo", "prefill", "skew", "skew_eplb"])
def test_full_layer_sampled(dev, dsv3_dev, name):
    cfg, x, W, bias = host_workload(name)
    ex, wdev = dsv3_dev
    emap = None
    rng = np.random.default_rng(1)
    tok = np.sort(rng.choice(cfg.B, 3, replace=False)).astype(np.int32)
    if cfg.N_phys != cfg.N:
        idx_all, _ = oracle.route(x, W, bias, cfg)
        emap = oracle.eplb_build_map(oracle.expert_counts(idx_all, cfg.N), cfg.N, cfg.N_phys)
    lay = api.MoELayer(cfg, to_dev(W), to_dev(bias), wdev, eplb_map=emap)
    out = bits(lay.forward(bf16_dev(x)))
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    gi = lay.topk_idx.cpu().numpy()
    idx, w = oracle.route(x, W, bias, cfg, tokens=tok)
    assert np.array_equal(gi[tok], idx)
    counts = lay.counts.cpu().numpy()
    assert counts.sum() == cfg.B * cfg.K
    t = lay.tiles.cpu().numpy()
    if cfg.layout == configs.MASKED:
        assert t[0] == int(((np.minimum(counts, cfg.cap) + 127) // 128).sum())
    else:
        assert t[0] == int(((counts + 127) // 128).sum())
    ref = oracle.layer_tokens(cfg, x, W, bias, getter(ex), shared_of(ex), tokens=tok)
    ok, err, bound = within_tol(oracle.bf16_to_f32(out[tok]), oracle.bf16_to_f32(ref["out"]))
    assert ok, (name, err, bound)
    assert np.isfinite(oracle.bf16_to_f32(out)).all()
