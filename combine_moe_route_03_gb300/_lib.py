"""ctypes binding of libmoe.so: argument marshalling only.

Every function here hands raw device pointers (from torch tensors) and sizes to
the C entry points declared in include/moe.h; all arithmetic of the layer runs
in the library's CUDA kernels.  There is no fallback: if libmoe.so is missing or
cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
ERRORS = {-1: "MOE_ERR_INVALID", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_CUDA"}
STATUS_CAPACITY, STATUS_TIMEOUT, STATUS_BAD_INDEX = 1, 2, 4
GEMM_GATEUP_SWIGLU, GEMM_DOWN = 0, 1
FMT_FP8, FMT_BF16, FMT_FP8_F32 = 0, 1, 2
SCALE_UE8M0, SCALE_F32 = 0, 1   # moe_gemm_args.scale_fmt / moe_layer.scale_fmt

_c_int, _c_i64, _c_sz, _vp, _f = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float


class RouteCfg(ctypes.Structure):
    _fields_ = [("B", _c_int), ("H", _c_int), ("N", _c_int), ("K", _c_int),
                ("n_group", _c_int), ("topk_group", _c_int), ("score_fn", _c_int),
                ("renorm", _c_int), ("route_scale", _f)]


class DispatchCfg(ctypes.Structure):
    _fields_ = [("B", _c_int), ("H", _c_int), ("K", _c_int), ("N_log", _c_int),
                ("N_phys", _c_int), ("layout", _c_int), ("cap", _c_int), ("fmt", _c_int),
                ("max_rep", _c_int)]


class EplbCfg(ctypes.Structure):
    _fields_ = [("N_log", _c_int), ("n_group", _c_int), ("N_phys", _c_int),
                ("n_nodes", _c_int), ("n_gpus", _c_int), ("max_rep", _c_int)]


class FusedCombine(ctypes.Structure):
    _fields_ = [("B", _c_int), ("K", _c_int), ("row_of", _vp), ("topk_w", _vp),
                ("src_of", _vp), ("src_rows", _c_i64), ("pending", _vp),
                ("shared_row0", _c_i64), ("out", _vp)]


class GemmArgs(ctypes.Structure):
    _fields_ = [("op", _c_int), ("n", _c_int), ("k", _c_int), ("rows", _c_i64),
                ("max_tiles", _c_i64), ("num_experts", _c_int), ("A", _vp), ("A_sf", _vp),
                ("W", _vp), ("W_sf", _vp), ("phys2log", _vp), ("tiles", _vp), ("tiles2", _vp),
                ("row_offset2", _c_i64), ("expert2", _c_int), ("out", _vp),
                ("out_sf", _vp), ("signal", _vp), ("block_m_signal", _c_int),
                ("num_sms", _c_int), ("pair_tiles", _c_int), ("scale_fmt", _c_int),
                ("status", _vp), ("combine", ctypes.POINTER(FusedCombine)),
                ("tile_n", _c_int)]


class CombineCfg(ctypes.Structure):
    _fields_ = [("B", _c_int), ("H", _c_int), ("K", _c_int), ("signal", _vp),
                ("threshold", _c_int), ("block_m_signal", _c_int), ("timeout_ns", _c_i64),
                ("num_ctas", _c_int), ("shared_row0", _c_i64)]


class Layer(ctypes.Structure):
    _fields_ = [("route", RouteCfg), ("N_phys", _c_int), ("layout", _c_int), ("cap", _c_int),
                ("I", _c_int), ("has_shared", _c_int), ("sbo", _c_int),
                ("block_m_signal", _c_int), ("rows", _c_i64), ("max_tiles", _c_i64),
                ("timeout_ns", _c_i64), ("num_sms", _c_int), ("combine_ctas", _c_int),
                ("gemm_pairs", _c_int)] + [
        (n, _vp) for n in (
            "x", "W_router", "bias", "log2phys", "rep", "phys2log", "W13", "W13_sf", "W2",
            "W2_sf", "topk_idx", "topk_w", "expert_counts", "counts", "row_of", "tiles",
            "shared_tiles", "signal", "A", "A_sf", "H1", "H1_sf", "Y", "out", "route_ws",
            "dispatch_ws")] + [("route_ws_bytes", _c_sz), ("dispatch_ws_bytes", _c_sz),
                               ("status", _vp), ("stream2", _vp), ("events", _vp),
                               ("eplb_max_rep", _c_int), ("scale_fmt", _c_int),
                               ("fuse_combine", _c_int), ("src_of", _vp), ("pending", _vp),
                               ("W2_sf_t224", _vp)]

LAYER_EVENTS = 6
STAGES = ("route", "dispatch", "gateup", "down", "combine")


#: Every symbol include/moe.h declares, with (restype, argtypes).
SIGNATURES = {
    "moe_route_workspace_size": (_c_sz, [ctypes.POINTER(RouteCfg)]),
    "moe_route": (_c_int, [ctypes.POINTER(RouteCfg), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_sz, _vp]),
    "eplb_build_map": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _vp]),
    "moe_eplb_plan": (_c_int, [ctypes.POINTER(EplbCfg), _vp, _vp, _vp, _vp, _vp]),
    "moe_dispatch_rows": (_c_i64, [ctypes.POINTER(DispatchCfg)]),
    "moe_dispatch_max_tiles": (_c_i64, [ctypes.POINTER(DispatchCfg)]),
    "moe_dispatch_workspace_size": (_c_sz, [ctypes.POINTER(DispatchCfg)]),
    "moe_dispatch": (_c_int, [ctypes.POINTER(DispatchCfg)] + [_vp] * 14 + [_c_sz, _vp, _vp]),
    "moe_dispatch_noalloc": (_c_int, [ctypes.POINTER(DispatchCfg)] + [_vp] * 15),
    "moe_grouped_gemm_fp8": (_c_int, [ctypes.POINTER(GemmArgs), _vp]),
    "moe_packed_scale_bytes": (_c_sz, [_c_int, _c_int, _c_int]),
    "moe_scale_bytes": (_c_sz, [_c_i64, _c_int, _c_int]),
    "moe_pack_weight_scales": (_c_int, [_c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "moe_weight_scales_f32": (_c_int, [_c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "moe_tiled_scale_bytes": (_c_sz, [_c_int, _c_int, _c_int, _c_int]),
    "moe_pack_weight_scales_tiled": (_c_int, [_c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "moe_fused_combine_prep": (_c_int, [ctypes.POINTER(FusedCombine), _c_int, _vp]),
    "moe_combine": (_c_int, [ctypes.POINTER(CombineCfg), _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_read_status": (_c_int, [_vp, _vp]),
    "moe_last_cuda_error": (_c_int, []),
    "moe_num_sms": (_c_int, []),
    "moe_layer_forward": (_c_int, [ctypes.POINTER(Layer), _vp]),
    "moe_layer_forward_host": (_c_int, [ctypes.POINTER(Layer), _vp, _vp, _vp]),
    "moe_layer_forward_host_pipelined": (_c_int, [ctypes.POINTER(Layer), _vp, _vp, _vp, _vp,
                                                  _c_int, _vp, _vp]),
    "moe_layer_graph_create": (_c_int, [ctypes.POINTER(Layer), _vp, _vp, _vp,
                                        ctypes.POINTER(ctypes.c_void_p)]),
    "moe_layer_graph_launch": (_c_int, [_vp, _vp]),
    "moe_layer_graph_destroy": (_c_int, [_vp]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (built by ``combine_moe_route_03_gb300.build``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libmoe.so not found at {path}: build it with "
                               "`python -m combine_moe_route_03_gb300.build` (no fallback path)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class MoEError(RuntimeError):
    pass


def check(rc: int, what: str) -> None:
    if rc != MOE_OK:
        extra = ""
        if rc == -3:
            extra = f" (cudaError {load().moe_last_cuda_error()})"
        raise MoEError(f"{what} failed: {ERRORS.get(rc, rc)}{extra}")


def ptr(t, host: bool = False) -> int | None:
    """Address of a contiguous tensor (or a raw address) for a pointer parameter.

    Device parameters take CUDA tensors on the current device (the library's kernels
    would otherwise dereference host or another GPU's addresses); host parameters
    (``host=True``: the pinned buffers of the host-copy entry points) take CPU
    tensors."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            raise ValueError("tensors passed to libmoe must be contiguous")
        if host:
            if t.is_cuda:
                raise ValueError("a host buffer parameter got a CUDA tensor")
        elif not t.is_cuda or t.device.index != torch.cuda.current_device():
            raise ValueError(f"a device parameter got a tensor on {t.device}; libmoe runs on "
                             f"the current CUDA device")
        return t.data_ptr()
    return int(t)


def stream_ptr(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream
