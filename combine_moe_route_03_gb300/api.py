"""Python face of libmoe: same names as the C entry points, torch tensors in and out.

Only marshalling happens here (shape checks, output allocation through torch,
pointer passing); each step of the layer runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib
from ._lib import (FMT_BF16, FMT_FP8, FMT_FP8_F32, GEMM_DOWN, GEMM_GATEUP_SWIGLU, SCALE_F32,
                   SCALE_UE8M0, CombineCfg, DispatchCfg, EplbCfg, FusedCombine, GemmArgs, Layer,
                   RouteCfg, check, load, ptr, stream_ptr)
from .configs import MASKED, MoEConfig

__all__ = ["route", "eplb_build_map", "eplb_plan", "check_eplb_map", "EplbRecorder", "dispatch", "dispatch_sizes", "pack_weight_scales",
           "grouped_gemm_fp8", "combine", "read_status", "new_status", "MoELayer",
           "FMT_FP8", "FMT_BF16", "FMT_FP8_F32", "SCALE_UE8M0", "SCALE_F32", "GEMM_GATEUP_SWIGLU",
           "GEMM_DOWN", "num_sms", "scale_bytes", "weight_scales_f32"]


def num_sms() -> int:
    return load().moe_num_sms()


def _ordered(stream, *temps) -> int:
    """The handle of the stream a call runs on.  A ``stream`` other than the caller's
    current stream first waits for the current one, where the call's inputs and the
    buffers this module allocates for it were made (torch's caching allocator ties a
    fresh buffer to the current stream); ``temps`` -- buffers freed when the call
    returns -- are kept from reuse until ``stream`` is done with them."""
    if stream is not None:
        cur = torch.cuda.current_stream(stream.device)
        if stream != cur:
            stream.wait_stream(cur)
            for t in temps:
                if t is not None:
                    t.record_stream(stream)
    return stream_ptr(stream)


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def read_status(status: torch.Tensor) -> int:
    v = ctypes.c_int32(0)
    check(load().moe_read_status(ptr(status), ctypes.addressof(v)), "moe_read_status")
    return int(v.value)


_BF16 = (torch.bfloat16, torch.int16)   # bf16 values, or their bits viewed as int16


def _expect(t, what: str, dtypes, shape) -> None:
    """Shape and dtype of a tensor argument against the configuration (None in
    `shape`: any extent); a mismatch would make a kernel read past a buffer."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: a torch tensor is required")
    if t.dtype not in dtypes:
        raise ValueError(f"{what}: dtype {t.dtype}, expected one of {dtypes}")
    if t.dim() != len(shape) or any(w is not None and g != w for g, w in zip(t.shape, shape)):
        raise ValueError(f"{what}: shape {tuple(t.shape)}, expected {shape}")


def _route_cfg(cfg: MoEConfig, B: int | None = None) -> RouteCfg:
    return RouteCfg(cfg.B if B is None else B, cfg.H, cfg.N, cfg.K, cfg.n_group, cfg.topk_group,
                    cfg.score_fn, cfg.renorm, cfg.route_scale)


def route(cfg: MoEConfig, x: torch.Tensor, W: torch.Tensor, bias: torch.Tensor | None,
          stream=None, counts: bool = True) -> dict:
    """moe_route: x bf16 [B][H], W fp32 [N][H], bias fp32 [N] -> topk_idx, topk_w, counts."""
    _expect(x, "x", _BF16, (None, cfg.H))
    _expect(W, "W", (torch.float32,), (cfg.N, cfg.H))
    if bias is not None:
        _expect(bias, "bias", (torch.float32,), (cfg.N,))
    B = x.shape[0]
    rc = _route_cfg(cfg, B)
    dev = x.device
    idx = torch.empty((B, cfg.K), dtype=torch.int32, device=dev)
    w = torch.empty((B, cfg.K), dtype=torch.float32, device=dev)
    cnt = torch.empty(cfg.N, dtype=torch.int32, device=dev) if counts else None
    L = load()
    ws = torch.empty(max(1, L.moe_route_workspace_size(ctypes.byref(rc))), dtype=torch.uint8,
                     device=dev)
    check(L.moe_route(ctypes.byref(rc), ptr(x), ptr(W), ptr(bias), ptr(idx), ptr(w), ptr(cnt),
                      ptr(ws), ws.numel(), _ordered(stream)), "moe_route")
    return dict(topk_idx=idx, topk_w=w, counts=cnt, logits=ws)


def eplb_build_map(counts: np.ndarray, N_log: int, N_phys: int):
    """Host EPLB map -> (log2phys [N_log][2], rep [N_log], phys2log [N_phys]) int32 numpy."""
    c = np.ascontiguousarray(counts, dtype=np.int64)
    l2p = np.empty((N_log, 2), np.int32)
    rep = np.empty(N_log, np.int32)
    p2l = np.empty(N_phys, np.int32)
    check(load().eplb_build_map(c.ctypes.data, N_log, N_phys, l2p.ctypes.data, rep.ctypes.data,
                                p2l.ctypes.data), "eplb_build_map")
    return l2p, rep, p2l


def eplb_plan(load_counts: np.ndarray, N_log: int, N_phys: int, n_group: int = 1,
              n_nodes: int = 1, n_gpus: int = 1, max_rep: int = 2):
    """moe_eplb_plan (host): recorded loads -> (log2phys [N_log][max_rep], rep [N_log],
    phys2log [N_phys]) int32 numpy, and the plan's balance (mean / max GPU load)."""
    c = np.ascontiguousarray(load_counts, dtype=np.int64)
    if c.shape != (N_log,):
        raise ValueError("one load per logical expert")
    cfg = EplbCfg(N_log, n_group, N_phys, n_nodes, n_gpus, max_rep)
    l2p = np.empty((N_log, max_rep), np.int32)
    rep = np.empty(N_log, np.int32)
    p2l = np.empty(N_phys, np.int32)
    bal = ctypes.c_double()
    check(load().moe_eplb_plan(ctypes.byref(cfg), c.ctypes.data, p2l.ctypes.data,
                               l2p.ctypes.data, rep.ctypes.data, ctypes.byref(bal)),
          "moe_eplb_plan")
    return (l2p, rep, p2l), bal.value


def check_eplb_map(eplb_map, N_log: int, N_phys: int) -> None:
    """Raises ValueError unless (log2phys [N_log][R], rep [N_log], phys2log [N_phys]) is
    a map as eplb_build_map and eplb_plan make it: every logical expert has 1..R
    replicas, the replica counts fill the physical slots, and every entry of a row of
    log2phys (the tail repeats the first) is a slot that phys2log maps back to it."""
    l2p, rep, p2l = (np.asarray(a) for a in eplb_map)
    if l2p.ndim != 2 or l2p.shape[0] != N_log or not 1 <= l2p.shape[1] <= 64 \
            or rep.shape != (N_log,) or p2l.shape != (N_phys,):
        raise ValueError("EPLB map: shapes must be [N_log][R] (R <= 64), [N_log], [N_phys]")
    if rep.min() < 1 or rep.max() > l2p.shape[1] or int(rep.sum()) != N_phys:
        raise ValueError("EPLB map: replica counts must be 1..R and fill the physical slots")
    if p2l.min() < 0 or p2l.max() >= N_log or l2p.min() < 0 or l2p.max() >= N_phys:
        raise ValueError("EPLB map: expert index out of range")
    if not np.array_equal(p2l[l2p], np.broadcast_to(np.arange(N_log)[:, None], l2p.shape)):
        raise ValueError("EPLB map: log2phys and phys2log disagree")
    if not np.array_equal(np.bincount(p2l, minlength=N_log), rep):
        raise ValueError("EPLB map: a logical expert's replica count differs from its slots")


class EplbRecorder:
    """Periodic rebalancing from measured loads: adds each step's per-expert token
    counts (the route's expert_counts) and, every ``period`` steps, plans a new map
    from the loads recorded since the last plan ("Large-scale EP ...", §EPLB: the
    dynamic mode re-measures and rebalances while running)."""

    def __init__(self, N_log: int, N_phys: int, period: int, **plan_kw):
        if period < 1:
            raise ValueError("period >= 1")
        self.N_log, self.N_phys, self.period, self.plan_kw = N_log, N_phys, period, plan_kw
        self.load = np.zeros(N_log, np.int64)
        self.steps = 0

    def observe(self, expert_counts) -> None:
        c = expert_counts.cpu().numpy() if isinstance(expert_counts, torch.Tensor) else expert_counts
        c = np.asarray(c, np.int64)
        if c.shape != (self.N_log,) or np.any(c < 0):
            raise ValueError("expert counts: one non-negative count per logical expert")
        self.load += c
        self.steps += 1

    def due(self) -> bool:
        return self.steps >= self.period

    def plan(self, group=None):
        """The map for the loads recorded so far; the recorder then starts afresh.

        With a torch.distributed process group, the ranks' recorded loads are summed
        first (one all-reduce of N_log counts on the host side), so every rank of the
        group plans the same map from the whole job's loads."""
        load = self.load
        if group is not None:
            t = torch.from_numpy(self.load.copy())
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM, group=group)
            load = t.numpy()
        m, bal = eplb_plan(load, self.N_log, self.N_phys, **self.plan_kw)
        self.load[:] = 0
        self.steps = 0
        return m, bal


def _dispatch_cfg(cfg: MoEConfig, B: int, fmt: int, cap: int | None = None,
                  max_rep: int = 0) -> DispatchCfg:
    return DispatchCfg(B, cfg.H, cfg.K, cfg.N, cfg.N_phys, cfg.layout,
                       cfg.cap if cap is None else cap, fmt, max_rep)


def dispatch_sizes(cfg: MoEConfig, B: int | None = None, fmt: int = FMT_FP8,
                   cap: int | None = None) -> dict:
    dc = _dispatch_cfg(cfg, cfg.B if B is None else B, fmt, cap)
    L = load()
    return dict(rows=L.moe_dispatch_rows(ctypes.byref(dc)),
                max_tiles=L.moe_dispatch_max_tiles(ctypes.byref(dc)),
                ws=L.moe_dispatch_workspace_size(ctypes.byref(dc)))


def dispatch(cfg: MoEConfig, x: torch.Tensor, topk_idx: torch.Tensor, log2phys=None, rep=None,
             fmt: int = FMT_FP8, shared: bool = False, status: torch.Tensor | None = None,
             cap: int | None = None, stream=None, out: dict | None = None) -> dict:
    """moe_dispatch -> A, A_sf, counts, row_of, src_of, tiles (+ shared copy).
    log2phys [N][max_rep] / rep [N]: an EPLB map (max_rep = its column count)."""
    _expect(x, "x", _BF16, (None, cfg.H))
    B, H = x.shape
    _expect(topk_idx, "topk_idx", (torch.int32,), (B, cfg.K))
    if (log2phys is None) != (rep is None):
        raise ValueError("log2phys and rep go together")
    if log2phys is not None:
        _expect(log2phys, "log2phys", (torch.int32,), (cfg.N, None))
        _expect(rep, "rep", (torch.int32,), (cfg.N,))
    dev = x.device
    dc = _dispatch_cfg(cfg, B, fmt, cap, 0 if log2phys is None else log2phys.shape[1])
    sz = dispatch_sizes(cfg, B, fmt, cap)
    rows, mt = sz["rows"], sz["max_tiles"]
    if rows <= 0:
        raise ValueError("unsupported dispatch configuration")
    o = out if out is not None else {}
    if "A" not in o:
        o["A"] = torch.empty((rows, H * (2 if fmt == FMT_BF16 else 1)), dtype=torch.uint8, device=dev)
        o["A_sf"] = torch.empty(scale_bytes(rows, H, fmt), dtype=torch.uint8, device=dev)
        o["counts"] = torch.empty(cfg.N_phys, dtype=torch.int32, device=dev)
        o["row_of"] = torch.empty((B, cfg.K), dtype=torch.int32, device=dev)
        o["src_of"] = torch.empty(rows, dtype=torch.int32, device=dev)
        o["tiles"] = torch.empty(8 + 16 * mt, dtype=torch.int32, device=dev)
        o["ws"] = torch.empty(max(1, sz["ws"]), dtype=torch.uint8, device=dev)
        if shared:
            srows = (B + 127) // 128 * 128
            o["As"] = torch.empty((srows, H), dtype=torch.uint8, device=dev)
            o["As_sf"] = torch.empty(scale_bytes(srows, H, fmt), dtype=torch.uint8, device=dev)
            o["shared_tiles"] = torch.empty(8 + 16 * (srows // 128), dtype=torch.int32, device=dev)
    st = status if status is not None else new_status(dev)
    check(load().moe_dispatch(ctypes.byref(dc), ptr(x), ptr(topk_idx), ptr(log2phys), ptr(rep),
                              ptr(o["A"]), ptr(o["A_sf"]), ptr(o["counts"]), ptr(o["row_of"]),
                              ptr(o.get("src_of")), ptr(o["tiles"]), ptr(o.get("As")),
                              ptr(o.get("As_sf")), ptr(o.get("shared_tiles")), ptr(o["ws"]),
                              o["ws"].numel(), ptr(st), _ordered(stream)), "moe_dispatch")
    o.update(rows=rows, max_tiles=mt, status=st)
    return o


def scale_bytes(rows: int, k: int, fmt: int = 0) -> int:
    """Bytes of the scales of an activation tensor [rows][k] in format fmt (FMT_FP8: SF
    atoms; FMT_FP8_F32: float [rows][k/128]) (moe_scale_bytes)."""
    n = load().moe_scale_bytes(rows, k, FMT_FP8_F32 if fmt == FMT_FP8_F32 else FMT_FP8)
    if n == 0:
        raise ValueError(f"scale atoms need rows and k multiples of 128 (got {rows}, {k})")
    return n


def weight_scales_f32(W_sf: torch.Tensor, stream=None) -> torch.Tensor:
    """UE8M0 bytes [E][n/128][k/128] (device) -> float 2^(byte-127), same shape (the
    weight scales of the binary32-scale mode)."""
    E, nb, kb = W_sf.shape
    out = torch.empty((E, nb, kb), dtype=torch.float32, device=W_sf.device)
    check(load().moe_weight_scales_f32(E, nb * 128, kb * 128, ptr(W_sf), ptr(out),
                                       _ordered(stream)), "moe_weight_scales_f32")
    return out


def pack_weight_scales(W_sf: torch.Tensor, stream=None) -> torch.Tensor:
    """UE8M0 bytes [E][n/128][k/128] (device) -> SF atoms [E][n/128][k/128][512]."""
    E, nb, kb = W_sf.shape
    L = load()
    nbytes = L.moe_packed_scale_bytes(E, nb * 128, kb * 128)
    out = torch.empty(nbytes, dtype=torch.uint8, device=W_sf.device)
    check(L.moe_pack_weight_scales(E, nb * 128, kb * 128, ptr(W_sf), ptr(out),
                                   _ordered(stream)), "moe_pack_weight_scales")
    return out


def pack_weight_scales_tiled(W_sf: torch.Tensor, tile_n: int = 224, stream=None) -> torch.Tensor:
    """UE8M0 bytes [E][n/128][k/128] (device) -> two 128-row images per tile_n-row weight
    tile and group of four k-blocks, [E][n/tile_n][ceil(k/512)][2][512] (the DOWN GEMM's
    scales with tile_n 224)."""
    E, nb, kb = W_sf.shape
    L = load()
    nbytes = L.moe_tiled_scale_bytes(E, nb * 128, kb * 128, tile_n)
    if nbytes == 0:
        raise ValueError(f"no {tile_n}-row tiles for n={nb * 128}")
    out = torch.empty(nbytes, dtype=torch.uint8, device=W_sf.device)
    check(L.moe_pack_weight_scales_tiled(E, nb * 128, kb * 128, tile_n, ptr(W_sf), ptr(out),
                                         _ordered(stream)), "moe_pack_weight_scales_tiled")
    return out


def grouped_gemm_fp8(op: int, A: torch.Tensor, A_sf: torch.Tensor, W: torch.Tensor,
                     W_sf_atoms: torch.Tensor, tiles: torch.Tensor, max_tiles: int,
                     out: torch.Tensor | None = None, out_sf: torch.Tensor | None = None,
                     phys2log: torch.Tensor | None = None, signal: torch.Tensor | None = None,
                     block_m_signal: int = 64, num_sms_: int = 0,
                     status: torch.Tensor | None = None, stream=None,
                     tiles2: torch.Tensor | None = None, row_offset2: int = 0, expert2: int = 0,
                     pair_tiles: int = 0, scale_fmt: int = SCALE_UE8M0,
                     combine: dict | None = None, tile_n: int = 0):
    """moe_grouped_gemm_fp8.  W e4m3 [E][n][k]; A e4m3 [rows][k]; scale_fmt SCALE_F32:
    A_sf float [rows][k/128] and W_sf_atoms the float [E][n/128][k/128] scales.
    combine (DOWN): the fused combine's tensors, as fused_combine_prep takes them.
    tile_n 224 (DOWN): 224-column tiles with two accumulators; W_sf_atoms then from
    pack_weight_scales_tiled."""
    E, n, k = W.shape
    rows = A.shape[0]
    dev = A.device
    if op == GEMM_GATEUP_SWIGLU:
        I = n // 2
        if out is None:
            out = torch.empty((rows, I), dtype=torch.uint8, device=dev)
            out_sf = torch.empty(scale_bytes(rows, I, FMT_FP8_F32 if scale_fmt else FMT_FP8),
                                 dtype=torch.uint8, device=dev)
    elif out is None:
        out = torch.empty((rows, n), dtype=torch.bfloat16, device=dev)
    st = status if status is not None else new_status(dev)
    g = GemmArgs(op, n, k, rows, max_tiles, E, ptr(A), ptr(A_sf), ptr(W), ptr(W_sf_atoms),
                 ptr(phys2log), ptr(tiles), ptr(tiles2), row_offset2, expert2, ptr(out),
                 ptr(out_sf), ptr(signal), block_m_signal, num_sms_, pair_tiles, scale_fmt,
                 ptr(st))
    g.tile_n = tile_n
    if combine is not None:
        fc = _fused_combine_args(**combine)
        g.combine = ctypes.pointer(fc)
    check(load().moe_grouped_gemm_fp8(ctypes.byref(g), _ordered(stream, st)),
          "moe_grouped_gemm_fp8")
    return (out, out_sf) if op == GEMM_GATEUP_SWIGLU else out


def _fused_combine_args(row_of, topk_w, src_of, pending, out, shared_row0: int = -1):
    _expect(row_of, "row_of", (torch.int32,), (None, None))
    B, K = row_of.shape
    _expect(topk_w, "topk_w", (torch.float32,), (B, K))
    _expect(src_of, "src_of", (torch.int32,), (None,))
    _expect(out, "out", _BF16, (B, None))
    _expect(pending, "pending", (torch.int32,), (B, out.shape[1] // 128))
    return FusedCombine(B, K, ptr(row_of), ptr(topk_w), ptr(src_of), src_of.numel(),
                        ptr(pending), shared_row0, ptr(out))


def fused_combine_prep(row_of: torch.Tensor, topk_w: torch.Tensor, src_of: torch.Tensor,
                       pending: torch.Tensor, out: torch.Tensor, shared_row0: int = -1,
                       stream=None) -> None:
    """moe_fused_combine_prep: the pending counts of a fused-combine DOWN GEMM (and
    zeros in out for tokens without rows).  out bf16 [B][H], pending int32 [B][H/128]."""
    fc = _fused_combine_args(row_of, topk_w, src_of, pending, out, shared_row0)
    check(load().moe_fused_combine_prep(ctypes.byref(fc), out.shape[1], _ordered(stream)),
          "moe_fused_combine_prep")


def combine(Y: torch.Tensor, row_of: torch.Tensor, topk_w: torch.Tensor,
            shared: torch.Tensor | None = None, out: torch.Tensor | None = None,
            signal: torch.Tensor | None = None, threshold: int = 0, block_m_signal: int = 64,
            timeout_ns: int = 1_000_000_000, num_ctas: int = 0, shared_row0: int = 0,
            status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """moe_combine: Y bf16 [rows][H] -> out bf16 [B][H]."""
    _expect(row_of, "row_of", (torch.int32,), (None, None))
    B, K = row_of.shape
    _expect(topk_w, "topk_w", (torch.float32,), (B, K))
    _expect(Y, "Y", _BF16 + (torch.uint8,), (None, None))
    H = Y.shape[1] if Y.element_size() == 2 else Y.shape[1] // 2
    if shared is not None:
        _expect(shared, "shared", _BF16, (B, H))
    if out is not None:
        _expect(out, "out", _BF16, (B, H))
    if out is None:
        out = torch.empty((B, H), dtype=torch.bfloat16, device=Y.device)
    cc = CombineCfg(B, H, K, ptr(signal), threshold, block_m_signal, timeout_ns, num_ctas,
                    shared_row0)
    st = status if status is not None else new_status(Y.device)
    check(load().moe_combine(ctypes.byref(cc), ptr(Y), ptr(row_of), ptr(topk_w), ptr(shared),
                             ptr(out), ptr(st), _ordered(stream, st)), "moe_combine")
    return out


class MoELayer:
    """All device buffers of one MoE layer plus the moe_layer_forward chain.

    ``weights``: dict of device uint8 tensors W13 [N][2I][H], W13_sf [N][2I/128][H/128],
    W2 [N][H][I], W2_sf [N][H/128][I/128] (raw UE8M0 bytes; packed here once), and
    for a shared expert W13s/W13s_sf/W2s/W2s_sf (one expert, batched or not).  The
    shared expert is stored as expert N of the layer's weight tensors, and its rows
    follow the routed rows in the row buffers (see moe_layer in include/moe.h).
    """

    def __init__(self, cfg: MoEConfig, W_router: torch.Tensor, bias: torch.Tensor | None,
                 weights: dict, eplb_map=None, num_sms_: int = 0, combine_ctas: int = 0,
                 timeout_ns: int = 1_000_000_000, device="cuda", gemm_pairs: int = 0,
                 down224: bool = False):
        self.cfg = cfg
        dev = torch.device(device)
        B, H, I, K = cfg.B, cfg.H, cfg.I, cfg.K
        L = load()
        t = lambda *s, dtype=torch.uint8: torch.empty(s, dtype=dtype, device=dev)  # noqa: E731
        self.x = t(B, H, dtype=torch.bfloat16)
        self.W_router, self.bias = W_router, bias
        self.has_shared = cfg.shared
        ne = cfg.N + (1 if cfg.shared else 0)
        if cfg.shared:
            def cat(a, b, *shape):
                out = t(ne, *shape)
                out[: cfg.N].copy_(a.reshape(cfg.N, *shape))
                out[cfg.N].copy_(b.reshape(*shape))
                return out
            self.W13 = cat(weights["W13"], weights["W13s"], 2 * I, H)
            self.W2 = cat(weights["W2"], weights["W2s"], H, I)
            W13_sf = cat(weights["W13_sf"], weights["W13s_sf"], 2 * I // 128, H // 128)
            W2_sf = cat(weights["W2_sf"], weights["W2s_sf"], H // 128, I // 128)
        else:
            self.W13, self.W2 = weights["W13"], weights["W2"]
            W13_sf, W2_sf = weights["W13_sf"], weights["W2_sf"]
        if cfg.scale_fmt:       # binary32 scales, read per k-block by the epilogue
            self.W13_sf = weight_scales_f32(W13_sf)
            self.W2_sf = weight_scales_f32(W2_sf)
        else:                   # SF atoms for the tensor core's block scaling
            self.W13_sf = pack_weight_scales(W13_sf)
            self.W2_sf = pack_weight_scales(W2_sf)
        # the down GEMM's scales for 224-column tiles (CTA pairs, two accumulators)
        self.W2_sf_t224 = (pack_weight_scales_tiled(W2_sf, 224)
                           if down224 and not cfg.scale_fmt and H % 224 == 0 else None)
        afmt = FMT_FP8_F32 if cfg.scale_fmt else FMT_FP8
        self.log2phys = self.rep = self.phys2log = None
        if eplb_map is not None:
            check_eplb_map(eplb_map, cfg.N, cfg.N_phys)
            l2p, rep, p2l = eplb_map
            self.log2phys = torch.from_numpy(np.ascontiguousarray(l2p, np.int32)).to(dev)
            self.rep = torch.from_numpy(np.ascontiguousarray(rep, np.int32)).to(dev)
            self.phys2log = torch.from_numpy(np.ascontiguousarray(p2l, np.int32)).to(dev)
        sz = dispatch_sizes(cfg)
        self.rows, self.max_tiles = sz["rows"], sz["max_tiles"]
        self.srows = (B + 127) // 128 * 128 if cfg.shared else 0
        rows = self.rows + self.srows
        self.topk_idx = t(B, K, dtype=torch.int32)
        self.topk_w = t(B, K, dtype=torch.float32)
        self.expert_counts = t(cfg.N, dtype=torch.int32)
        self.counts = t(cfg.N_phys, dtype=torch.int32)
        self.row_of = t(B, K, dtype=torch.int32)
        self.tiles = t(8 + 16 * self.max_tiles, dtype=torch.int32)
        self.shared_tiles = t(8 + 16 * (self.srows // 128), dtype=torch.int32) if cfg.shared else None
        self.A = t(rows, H)
        self.A_sf = t(scale_bytes(rows, H, afmt))
        self.H1 = t(rows, I)
        self.H1_sf = t(scale_bytes(rows, I, afmt))
        self.Y = t(rows, H, dtype=torch.bfloat16)
        self.S = self.Y[self.rows:] if cfg.shared else None
        self.signal = t(rows // cfg.block_m_signal, dtype=torch.int32) if cfg.sbo else None
        self.src_of = t(self.rows, dtype=torch.int32) if cfg.fuse_combine else None
        self.pending = t(B, H // 128, dtype=torch.int32) if cfg.fuse_combine else None
        self.out = t(B, H, dtype=torch.bfloat16)
        rcfg = _route_cfg(cfg)
        self.route_ws = t(max(1, L.moe_route_workspace_size(ctypes.byref(rcfg))))
        self.dispatch_ws = t(max(1, sz["ws"]))
        self.status = new_status(dev)
        self.stream2 = torch.cuda.Stream(device=dev) if cfg.sbo else None
        lay = Layer()
        lay.route = rcfg
        lay.N_phys, lay.layout, lay.cap, lay.I = cfg.N_phys, cfg.layout, cfg.cap, I
        lay.has_shared, lay.sbo, lay.block_m_signal = int(cfg.shared), int(cfg.sbo), cfg.block_m_signal
        lay.rows, lay.max_tiles, lay.timeout_ns = self.rows, self.max_tiles, timeout_ns
        lay.num_sms = num_sms_ or num_sms()
        lay.combine_ctas = combine_ctas
        lay.gemm_pairs = gemm_pairs
        lay.eplb_max_rep = 0 if self.log2phys is None else self.log2phys.shape[1]
        lay.scale_fmt = cfg.scale_fmt
        lay.fuse_combine = int(cfg.fuse_combine)
        names = ["x", "W_router", "bias", "log2phys", "rep", "phys2log", "W13", "W13_sf", "W2",
                 "W2_sf", "topk_idx", "topk_w", "expert_counts", "counts", "row_of", "tiles",
                 "shared_tiles", "signal", "A", "A_sf", "H1", "H1_sf", "Y", "out", "route_ws",
                 "dispatch_ws", "status", "src_of", "pending", "W2_sf_t224"]
        for n in names:
            setattr(lay, n, ptr(getattr(self, n)))
        lay.route_ws_bytes = self.route_ws.numel()
        lay.dispatch_ws_bytes = self.dispatch_ws.numel()
        lay.stream2 = self.stream2.cuda_stream if self.stream2 is not None else None
        self.layer = lay

    def set_eplb_map(self, eplb_map) -> None:
        """Installs a new EPLB map of the same physical expert count (a replica reads
        its logical expert's weights through phys2log, so no weight moves on one GPU).
        Call between steps: a captured graph keeps the map buffers, not their values,
        so it uses the new map from its next replay when the column count is kept."""
        if self.log2phys is None:
            raise ValueError("the layer was built without an EPLB map")
        check_eplb_map(eplb_map, self.cfg.N, self.cfg.N_phys)
        l2p, rep, p2l = (np.ascontiguousarray(a, np.int32) for a in eplb_map)
        if l2p.shape != tuple(self.log2phys.shape) or p2l.shape != tuple(self.phys2log.shape) \
                or rep.shape != tuple(self.rep.shape):
            raise ValueError("the new map must keep the layer's shapes")
        self.log2phys.copy_(torch.from_numpy(l2p))
        self.rep.copy_(torch.from_numpy(rep))
        self.phys2log.copy_(torch.from_numpy(p2l))

    def forward(self, x: torch.Tensor | None = None, stream=None, events=None) -> torch.Tensor:
        """Runs the layer on self.x (copied from ``x`` first when given) on ``stream``
        (default: the current stream).  The copy is ordered after the caller's current
        stream and runs on ``stream``, ahead of the layer.

        ``events``: optional list of moe_layer.events torch.cuda.Event recorded at the
        stage boundaries."""
        if x is not None:
            cur = torch.cuda.current_stream(self.x.device)
            s = stream if stream is not None else cur
            if s != cur:
                s.wait_stream(cur)      # x was produced on the caller's stream
                x.record_stream(s)
            with torch.cuda.stream(s):
                self.x.copy_(x)
        keep = None
        if events is not None:
            keep = (ctypes.c_void_p * _lib.LAYER_EVENTS)(*[e.cuda_event for e in events])
            self.layer.events = ctypes.cast(keep, ctypes.c_void_p)
        try:
            check(load().moe_layer_forward(ctypes.byref(self.layer), stream_ptr(stream)),
                  "moe_layer_forward")
        finally:
            self.layer.events = None
        return self.out

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, stream=None) -> None:
        """x from (pinned) host memory, out back to host memory, through the C ABI."""
        check(load().moe_layer_forward_host(ctypes.byref(self.layer), ptr(x_host, host=True),
                                            ptr(out_host, host=True), stream_ptr(stream)),
              "moe_layer_forward_host")

    def forward_host_pipelined(self, x_hosts, out_hosts, stream=None, copy_stream=None) -> None:
        """moe_layer_forward_host_pipelined: len(x_hosts) steps, each copying x_hosts[i]
        (pinned bf16 [B][H]) in and the output to out_hosts[i] (pinned), the copies of
        neighbouring steps on ``copy_stream`` overlapping the layer on ``stream``.  The
        second pair of device buffers is allocated on first use."""
        n = len(x_hosts)
        if n != len(out_hosts) or n < 1:
            raise ValueError("one output buffer per input batch")
        if getattr(self, "_x2", None) is None:
            self._x2 = torch.empty_like(self.x)
            self._out2 = torch.empty_like(self.out)
        if copy_stream is None:
            if getattr(self, "_copy_stream", None) is None:
                self._copy_stream = torch.cuda.Stream(device=self.x.device)
            copy_stream = self._copy_stream
        xs = (ctypes.c_void_p * n)(*[ptr(t, host=True) for t in x_hosts])
        outs = (ctypes.c_void_p * n)(*[ptr(t, host=True) for t in out_hosts])
        check(load().moe_layer_forward_host_pipelined(
            ctypes.byref(self.layer), ptr(self._x2), ptr(self._out2), xs, outs, n,
            stream_ptr(stream), stream_ptr(copy_stream)), "moe_layer_forward_host_pipelined")


class LayerGraph:
    """One captured layer call (moe_layer_graph_create), replayed by launch().

    The graph keeps the layer's buffers and, for a host graph, the pinned host buffers
    it was captured with; keep them alive and unchanged while the graph is used."""

    def __init__(self, layer: "MoELayer", stream: torch.cuda.Stream,
                 x_host: torch.Tensor | None = None, out_host: torch.Tensor | None = None):
        self._keep = (layer, x_host, out_host)
        h = ctypes.c_void_p()
        check(load().moe_layer_graph_create(ctypes.byref(layer.layer), ptr(x_host, host=True),
                                            ptr(out_host, host=True),
                                            stream_ptr(stream), ctypes.byref(h)),
              "moe_layer_graph_create")
        self.handle = h

    def launch(self, stream) -> None:
        check(load().moe_layer_graph_launch(self.handle, stream_ptr(stream)),
              "moe_layer_graph_launch")

    def close(self) -> None:
        if self.handle:
            check(load().moe_layer_graph_destroy(self.handle), "moe_layer_graph_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
