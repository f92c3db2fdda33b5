"""The bench's algorithmic work per stage, tied to the arrays each stage reads or writes
in a small layer (sizes taken from the oracle's own outputs and the stored weights, not
from the formulas), and its roofline bookkeeping.  CPU only."""
import numpy as np
import pytest

import bench
import oracle
from combine_moe_route_03_gb300 import configs, inputs


@pytest.mark.parametrize("name", ["small_contig", "small_masked", "tiny"])
def test_stage_bytes_are_the_arrays_each_stage_moves(name):
    cfg = configs.ALL[name]
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    idx, w = oracle.route(x, W, bias, cfg)
    d = oracle.dispatch(x, idx, cfg)
    work = bench.stage_work(cfg, d["cnt"])
    B, sh = cfg.B, cfg.shared
    live = d["row_of"] >= 0
    R = int(live.sum())                                   # routed rows that exist (drops out)
    q, sf = oracle.quantize_rows(oracle.bf16_to_f32(x[:1]))
    a_row = q[0].nbytes + sf[0].nbytes                    # e4m3 codes + one byte per block
    experts = [inputs.make_expert(cfg, int(e)) for e in np.flatnonzero(d["cnt"] > 0)]
    if sh:
        experts.append(inputs.make_shared_expert(cfg))
    w13 = sum(e[0].nbytes + e[1].nbytes for e in experts)   # each touched expert once
    w2 = sum(e[2].nbytes + e[3].nbytes for e in experts)
    hq, hsf = oracle.quantize_rows(np.ones((1, cfg.I), np.float32))
    h_row = hq[0].nbytes + hsf[0].nbytes
    y_row = 2 * cfg.H                                     # bf16
    rows = R + (B if sh else 0)
    ints = d["row_of"].itemsize + d["src_of"].itemsize
    assert work["route"]["bytes"] == x.nbytes + W.nbytes + idx.nbytes + w.nbytes
    assert work["route"]["flops"] == 2 * B * cfg.H * cfg.N
    assert work["dispatch"]["bytes"] == x.nbytes + R * (a_row + ints) + (B * a_row if sh else 0)
    assert work["gateup"]["bytes"] == w13 + rows * (a_row + h_row)
    assert work["gateup"]["flops"] == 2 * rows * cfg.H * 2 * cfg.I
    assert work["down"]["bytes"] == w2 + rows * (h_row + y_row)
    assert work["down"]["flops"] == 2 * rows * cfg.I * cfg.H
    assert work["combine"]["bytes"] == (R * (y_row + d["row_of"].itemsize + w.itemsize)
                                        + (B * y_row if sh else 0) + B * y_row)


def test_replicas_read_their_logical_experts_weights_once():
    """With an EPLB map, physical counts fold onto logical experts: a replicated hot
    expert's weights are counted once, as when the map is absent."""
    cfg = configs.SMALL_EPLB
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    idx, _ = oracle.route(x, W, bias, cfg)
    counts = oracle.expert_counts(idx, cfg.N)
    l2p, rep, p2l = oracle.eplb_build_map(counts, cfg.N, cfg.N_phys)
    d = oracle.dispatch(x, idx, cfg, l2p, rep)
    with_map = bench.physical_work(cfg, d["cnt"], p2l)
    without = bench.stage_work(cfg.with_(n_phys=0), counts)
    assert with_map == without


def test_stage_summary_fractions():
    work = {"route": dict(bytes=0, flops=10), "dispatch": dict(bytes=6_000_000, flops=0),
            "gateup": dict(bytes=8_000_000, flops=4 * 10**12), "down": dict(bytes=1, flops=0),
            "combine": dict(bytes=3_000_000, flops=0)}
    ms = {"route": 1.0, "dispatch": 0.001, "gateup": 2.0, "down": 0.0, "combine": 0.001}
    s = bench.stage_summary(work, ms, hbm_gbs=6000.0, fp8_tflops=4000.0)
    assert set(s) == {"dispatch", "gateup", "combine"}     # no bytes, or no time: left out
    assert s["dispatch"]["GBps"] == 6000.0 and s["dispatch"]["hbm_frac"] == 1.0
    assert s["dispatch"]["hbm_frac_nominal"] == 0.75 and "fp8_frac" not in s["dispatch"]
    assert s["gateup"]["TFLOPs"] == 2000.0 and s["gateup"]["fp8_frac"] == 0.5
    assert s["gateup"]["fp8_frac_nominal"] == round(2000.0 / 4500.0, 3)
    assert s["combine"]["GBps"] == 3000.0


def test_expert_balance():
    assert bench.expert_balance([7, 7, 7])["mean_over_max"] == 1.0
    b = bench.expert_balance(np.array([4, 2, 0, 2], np.int32))
    assert b == {"mean_over_max": 0.5, "max_rows": 4, "min_rows": 0, "experts": 4}
    assert bench.expert_balance([0, 0])["mean_over_max"] is None
    import json
    json.dumps(b)
