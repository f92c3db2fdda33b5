"""The seeded input recipe (CPU only): any expert regenerates alone to the same bytes
as the bulk fill, seeds are independent, and the stored weights, activations and router
follow the stated distributions."""
import numpy as np

import oracle
from combine_moe_route_03_gb300 import configs, inputs


def test_an_expert_regenerates_alone_to_the_bulk_bytes():
    cfg = configs.SMALL_CONTIG
    bulk = inputs.make_all_experts(cfg)
    for e in (0, 7, cfg.N - 1):
        W13, W13_sf, W2, W2_sf = inputs.make_expert(cfg, e)
        assert np.array_equal(bulk["W13"][e], W13) and np.array_equal(bulk["W13_sf"][e], W13_sf)
        assert np.array_equal(bulk["W2"][e], W2) and np.array_equal(bulk["W2_sf"][e], W2_sf)


def test_seeds_and_tags_are_independent():
    cfg = configs.SMALL_CONTIG
    assert np.array_equal(inputs.make_x(cfg), inputs.make_x(cfg))
    assert not np.array_equal(inputs.make_x(cfg), inputs.make_x(cfg, seed=cfg.seed + 1))
    a, b = inputs.make_expert(cfg, 3), inputs.make_expert(cfg, 4)
    assert not np.array_equal(a[0], b[0])
    s = inputs.make_shared_expert(cfg)
    assert not np.array_equal(s[0], a[0])


def _block_variances(W, sf, fan_in):
    v = oracle.dequant_blocks(W, sf)
    blocks = v.reshape(W.shape[0] // 128, 128, W.shape[1] // 128, 128)
    return v, blocks.var(axis=(1, 3)) * fan_in


def test_weights_are_normal_with_variance_about_one_over_fan_in():
    """Dequantised, every 128x128 block has mean ~0 and one variance (the codes' scale
    compensates the per-block exponent jitter, so the block exponents vary but the
    values do not); that variance is 1/fan_in up to the power-of-two rounding of the
    base exponent: within a factor of 2 at any fan_in, within 20 % at the DeepSeek
    shapes (fan_in 7168 and 2048)."""
    cfg = configs.SMALL_CONTIG
    W13, W13_sf, W2, W2_sf = inputs.make_expert(cfg, 5)
    for W, sf, fan_in in ((W13, W13_sf, cfg.H), (W2, W2_sf, cfg.I)):
        v, var = _block_variances(W, sf, fan_in)
        assert np.all((var > 0.5) & (var < 2.0)), var
        assert var.max() / var.min() < 1.15                  # one variance for all blocks
        assert abs(float(v.mean())) < 3.0 / np.sqrt(v.size / fan_in)
        assert len(np.unique(sf)) > 1
    d = configs.DECODE
    W13, W13_sf, W2, W2_sf = inputs.make_expert(d, 5)
    for W, sf, fan_in in ((W13[:512], W13_sf[:4], d.H), (W2[:512], W2_sf[:4], d.I)):
        _, var = _block_variances(W, sf, fan_in)
        assert np.all(np.abs(var - 1.0) < 0.2), var


def test_activations_and_router_follow_the_recipe():
    cfg = configs.PREFILL.with_(B=256)
    x = oracle.bf16_to_f32(inputs.make_x(cfg)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0) < 0.01
    W, bias = inputs.make_router(cfg)              # uniform, variance 1/H, no bias
    a = np.sqrt(3.0 / cfg.H)
    assert W.min() >= -a and W.max() <= a and abs(W.var() * cfg.H - 1.0) < 0.01
    assert bias is None or not np.any(bias)
    d = configs.DECODE
    Wd, bd = inputs.make_router(d)                  # normal, variance 1/H; bias variance 0.01
    assert abs(Wd.var() * d.H - 1.0) < 0.01 and abs(bd.var() - 0.01) < 0.004
