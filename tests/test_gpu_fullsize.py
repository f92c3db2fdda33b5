"""The DeepSeek-V3-shaped workloads at full size, through moe_layer_forward, against the
oracle: routing of every token bit for bit; every row of several whole experts (the
hottest, one whose odd last tile holds at most 64 rows, one whose odd last tile holds
more, the one with the fewest rows) and of the shared expert over at least 256 tokens,
each against the oracle's FFN on the oracle's own dispatched rows; and the layer output
of 64 tokens; then the same layer twice more, every byte of Y and of the output equal to
the first run's.  The oracle's FFN is fp64 NumPy and costs about a second per expert
(dequantising its weights), so the 64 tokens are chosen to share experts."""
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


def pick_experts(cnt: np.ndarray, cap: int) -> list[int]:
    """Physical experts whose rows are compared in full: the hottest, one whose odd last
    tile has 1-64 rows and one whose odd last tile has 65-128 (the 2-SM kernel's two
    single-tile forms), and the one with the fewest rows (at least one)."""
    c = np.minimum(cnt, cap) if cap else cnt
    nt = (c + 127) // 128
    tail = c - 128 * (nt - 1)
    picks = [int(np.argmax(c))]
    for lo, hi in ((1, 64), (65, 128)):
        sel = np.flatnonzero((nt % 2 == 1) & (tail >= lo) & (tail <= hi) & (c > 0))
        if sel.size:
            picks.append(int(sel[np.argmax(c[sel])]))
    live = np.flatnonzero(c > 0)
    picks.append(int(live[np.argmin(c[live])]))
    return sorted(set(picks))


def pick_tokens(idx: np.ndarray, n: int, start: set) -> np.ndarray:
    """n tokens chosen greedily so that their experts add as few new ones as possible."""
    sets = [set(r.tolist()) for r in idx]
    have, chosen = set(start), []
    free = np.ones(len(sets), bool)
    for _ in range(n):
        best, bn = -1, 1 << 30
        for t in np.flatnonzero(free):
            k = len(sets[t] - have)
            if k < bn:
                best, bn = t, k
                if k == 0:
                    break
        chosen.append(best)
        free[best] = False
        have |= sets[best]
    return np.sort(np.array(chosen, np.int32))


@pytest.mark.parametrize("name", ["prefill", "skew", "skew_eplb", "sbo", "decode"])
def test_full_layer_experts_and_tokens(dev, dsv3_dev, name):
    cfg, x, W, bias = host_workload(name)
    ex, wdev = dsv3_dev
    idx, w = oracle.route(x, W, bias, cfg)                     # every token
    l2p = rep = p2l = None
    emap = None
    if cfg.N_phys != cfg.N:
        emap = oracle.eplb_build_map(oracle.expert_counts(idx, cfg.N), cfg.N, cfg.N_phys)
        l2p, rep, p2l = emap
    lay = api.MoELayer(cfg, to_dev(W), to_dev(bias), wdev, eplb_map=emap)
    out_dev = lay.forward(bf16_dev(x)).clone()
    torch.cuda.synchronize()
    assert api.read_status(lay.status) == 0
    out = bits(out_dev)
    Y_dev = lay.Y.clone()

    # routing and dispatch, every token
    assert np.array_equal(lay.topk_idx.cpu().numpy(), idx)
    assert np.array_equal(lay.topk_w.cpu().numpy().view(np.uint32), w.view(np.uint32))
    d = oracle.dispatch(x, idx, cfg, log2phys=l2p, rep=rep)
    assert np.array_equal(lay.counts.cpu().numpy(), d["cnt"])
    row_of = lay.row_of.cpu().numpy()
    assert np.array_equal(row_of, d["row_of"])

    # whole experts: GPU Y rows against the oracle FFN on the oracle's dispatched rows
    Y = bits(lay.Y)
    get = getter(ex)
    picks = pick_experts(d["cnt"], cfg.cap if cfg.layout == configs.MASKED else 0)
    assert len(picks) >= 2
    for p in picks:
        rows = np.sort(row_of[d["phys"] == p])
        rows = rows[rows >= 0]
        assert rows.size > 0
        e = int(p2l[p]) if p2l is not None else p
        ref = oracle.expert_ffn(d["A"][rows], d["sf"][rows], *get(e))
        ok, err, bound = within_tol(oracle.bf16_to_f32(Y[rows]), oracle.bf16_to_f32(ref))
        assert ok, (name, "expert", p, rows.size, err, bound)

    # the shared expert: its rows follow the routed rows, in token order
    q, sf = oracle.quantize_rows(oracle.bf16_to_f32(x))
    ts = np.arange(min(cfg.B, 256))
    if cfg.B > 256:
        ts = np.concatenate([ts, np.arange(cfg.B - 128, cfg.B)])  # and the last tile
    S_ref = oracle.expert_ffn(q[ts], sf[ts], *shared_of(ex))
    ok, err, bound = within_tol(oracle.bf16_to_f32(Y[lay.rows + ts]), oracle.bf16_to_f32(S_ref))
    assert ok, (name, "shared", err, bound)

    # the layer output of 64 tokens, each through its K experts and the shared one
    logical = {int(p2l[p]) if p2l is not None else p for p in picks}
    tok = pick_tokens(idx, 64, logical)
    ref = oracle.layer_tokens(cfg, x, W, bias, get, shared_of(ex), tokens=tok)
    ok, err, bound = within_tol(oracle.bf16_to_f32(out[tok]), oracle.bf16_to_f32(ref["out"]))
    assert ok, (name, "out", err, bound)
    assert np.isfinite(oracle.bf16_to_f32(out)).all()

    # the launch configuration the bench times, run again: every row of Y and every
    # output byte repeat (a race between CTAs, warps or the streams would show here)
    for _ in range(2):
        again = lay.forward()
        torch.cuda.synchronize()
        assert api.read_status(lay.status) == 0
        assert torch.equal(again, out_dev) and torch.equal(lay.Y, Y_dev)
