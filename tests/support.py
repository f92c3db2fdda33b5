"""Test helpers: seeded workloads on host and device, SF-atom unpacking, tolerances."""
from __future__ import annotations

import functools

import numpy as np
import torch

from combine_moe_route_03_gb300 import configs, inputs

# Layer output tolerance: max |gpu - oracle| <= REL * max |oracle| + ABS (bf16 outputs).
REL, ABS = 2e-2, 1e-3


def unpack_sf_atoms(atoms: np.ndarray, rows: int, kb: int) -> np.ndarray:
    """SF atoms [rows/128][ceil(kb/4)][512] -> UE8M0 bytes [rows][kb] (the layout of
    include/moe.h: byte j of the word at 16*(r%32) + 4*(r/32) of group g holds row r's
    scale for column block 4g + j)."""
    kg = (kb + 3) // 4
    a = np.asarray(atoms, dtype=np.uint8).reshape(rows // 128, kg, 32, 4, 4)  # r%32, r/32, j
    # a[mb, g, r%32, r/32, j] -> row = mb*128 + (r/32)*32 + r%32, block = 4g + j
    full = a.transpose(0, 3, 2, 1, 4).reshape(rows, kg * 4)
    return full[:, :kb].copy()


def within_tol(got: np.ndarray, ref: np.ndarray, rel=REL, abs_=ABS) -> tuple[bool, float, float]:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    bound = rel * float(np.max(np.abs(ref))) + abs_ if ref.size else abs_
    return err <= bound, err, bound


@functools.lru_cache(maxsize=None)
def host_workload(name: str):
    cfg = configs.ALL[name]
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    return cfg, x, W, bias


def host_experts(name: str) -> dict:
    """All routed experts (+ shared expert) of a workload, host numpy, stored form.
    Workloads of the same model (shapes and seed) share one copy."""
    c = configs.ALL[name]
    return _experts(c.N, c.H, c.I, c.shared, c.seed)


@functools.lru_cache(maxsize=2)
def _experts(N, H, I, shared, seed) -> dict:
    cfg = configs.MoEConfig("model", B=1, H=H, N=N, K=1, I=I, shared=shared, seed=seed)
    ex = inputs.make_all_experts(cfg)
    if cfg.shared:
        s = inputs.make_shared_expert(cfg)
        ex.update(W13s=s[0], W13s_sf=s[1], W2s=s[2], W2s_sf=s[3])
    return ex


def getter(ex: dict):
    return lambda e: (ex["W13"][e], ex["W13_sf"][e], ex["W2"][e], ex["W2_sf"][e])


def shared_of(ex: dict):
    if "W13s" not in ex:
        return None
    return ex["W13s"], ex["W13s_sf"], ex["W2s"], ex["W2s_sf"]


def to_dev(a, dev="cuda", dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(dev)


def device_weights(ex: dict, dev="cuda") -> dict:
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in ex.items()}


def bf16_dev(x_bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits)).view(torch.bfloat16).to(dev)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 device tensor -> uint16 numpy bits."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dispatch_order(ntiles):
    """The order of the experts' tiles and item groups in moe_dispatch's tile list: the
    experts with two or more items (three or more tiles) spread evenly between those
    with one (multi-item expert i of nm, in expert order, goes before single-item expert
    floor((2i + 1) n1 / (2 nm)) of n1); experts without tiles take no place."""
    gcs = [n // 2 + n % 2 for n in ntiles]
    multi = [e for e, g in enumerate(gcs) if g >= 2]
    single = [e for e, g in enumerate(gcs) if g == 1]
    nm, n1 = len(multi), len(single)
    order, i = [], 0
    for s, e in enumerate(single):
        while i < nm and (2 * i + 1) * n1 // (2 * nm) <= s:
            order.append(multi[i])
            i += 1
        order.append(e)
    return order + multi[i:]


def dispatch_tile_first(ntiles):
    """Each expert's first tile index in the dispatch order (0 for experts without)."""
    first, t = [0] * len(ntiles), 0
    for e in dispatch_order(ntiles):
        first[e], t = t, t + ntiles[e]
    return first


def dispatch_items(ntiles):
    """cluster_items in the group order moe_dispatch writes (dispatch_order), the tiles
    numbered in that order too."""
    first = dispatch_tile_first(ntiles)
    items = []
    for e in dispatch_order(ntiles):
        n = ntiles[e]
        npair, gc = n // 2, n // 2 + n % 2
        f_item = len(items)
        items += [[first[e] + 2 * j, first[e] + 2 * j + 1 if j < npair else -1, f_item, gc,
                   1 if j < npair else 0] for j in range(gc)]
    return items


def cluster_items(ntiles):
    """Expected work items of a tile list for tile counts per expert (in expert order):
    an expert's pairs [t, t+1, group first, group size, 1], then its odd last tile
    [t, -1, group first, group size, 0], all in one group."""
    items, first = [], 0
    for n in ntiles:
        npair, gc, f_item = n // 2, n // 2 + n % 2, len(items)
        for j in range(gc):
            pair = j < npair
            items.append([first + 2 * j, first + 2 * j + 1 if pair else -1, f_item, gc,
                          1 if pair else 0])
        first += n
    return items
