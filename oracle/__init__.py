"""CPU oracle for the MoE layer hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the product package, which must
fail loudly rather than fall back here.

The routing, EPLB map, quantisation, dispatch and combine definitions live in
``moe_oracle.c`` (strict binary32 C, built by :func:`build`); the expert FFN is
``ffn.py`` (fp64 NumPy).  Every function cites the passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_f32p = np.ctypeslib.ndpointer(np.float32, flags="C")
_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE: no contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu99", "-ffp-contract=off", "-fno-fast-math",
                               "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_exp.argtypes = [ctypes.c_float]
        L.oracle_exp.restype = ctypes.c_float
        L.oracle_sigmoid.argtypes = [ctypes.c_float]
        L.oracle_sigmoid.restype = ctypes.c_float
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = ctypes.c_float
        L.oracle_scale_exp.argtypes = [ctypes.c_float]
        L.oracle_scale_exp.restype = ctypes.c_int
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_quantize_rows.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, _u8p, _u8p]
        L.oracle_quantize_rows.restype = None
        L.oracle_quantize_rows_f32.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, _u8p, _f32p]
        L.oracle_quantize_rows_f32.restype = None
        L.oracle_scale_f32.argtypes = [ctypes.c_float]
        L.oracle_scale_f32.restype = ctypes.c_float
        L.oracle_route.argtypes = [_u16p, _f32p, ctypes.c_void_p] + [ctypes.c_int] * 7 + [
            ctypes.c_float, ctypes.c_void_p, ctypes.c_int, _i32p, _f32p, ctypes.c_void_p,
            ctypes.c_int]
        L.oracle_route.restype = ctypes.c_int
        L.oracle_eplb_build_map.argtypes = [_i64p, ctypes.c_int, ctypes.c_int, _i32p, _i32p, _i32p]
        L.oracle_eplb_build_map.restype = ctypes.c_int
        L.oracle_dispatch.argtypes = [_u16p, _i32p, ctypes.c_void_p, ctypes.c_void_p] + [
            ctypes.c_int] * 8 + [_i32p, _i32p, _i32p, _i32p, _i32p, ctypes.c_int64, _u8p, _u8p]
        L.oracle_dispatch.restype = ctypes.c_int
        L.oracle_combine.argtypes = [_u16p, _i32p, _f32p, ctypes.c_void_p] + [ctypes.c_int] * 3 + [_u16p]
        L.oracle_combine.restype = None
        L.oracle_f32_to_bf16_array.argtypes = [_f32p, ctypes.c_int64, _u16p]
        L.oracle_f32_to_bf16_array.restype = None
        L.oracle_num_threads.restype = ctypes.c_int
        for nm, ot in (("oracle_e4m3_encode_array", _u8p), ("oracle_exp_array", _f32p),
                       ("oracle_sigmoid_array", _f32p)):
            getattr(L, nm).argtypes = [_f32p, ctypes.c_int64, ot]
            getattr(L, nm).restype = None
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- scalars
def exp(x: float) -> float:
    return lib().oracle_exp(x)


def sigmoid(x: float) -> float:
    return lib().oracle_sigmoid(x)


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(v)


def e4m3_decode(c: int) -> float:
    return lib().oracle_e4m3_decode(c)


def scale_exp(amax: float) -> int:
    return lib().oracle_scale_exp(amax)


def _map(name, v, otype):
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, otype)
    getattr(lib(), name)(v.reshape(-1), v.size, out.reshape(-1))
    return out


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    return _map("oracle_e4m3_encode_array", v, np.uint8)


def exp_array(v: np.ndarray) -> np.ndarray:
    return _map("oracle_exp_array", v, np.float32)


def sigmoid_array(v: np.ndarray) -> np.ndarray:
    return _map("oracle_sigmoid_array", v, np.float32)


def e4m3_table() -> np.ndarray:
    """fp64 value of each of the 256 e4m3 codes (NaN for the two NaN codes)."""
    return np.array([lib().oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def num_threads() -> int:
    return lib().oracle_num_threads()


# ---------------------------------------------------------------- arrays
def quantize_rows(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """1x128-block e4m3 quantisation of fp32 rows -> (codes, UE8M0 bytes)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    rows, n = v.shape
    q = np.empty((rows, n), np.uint8)
    sf = np.empty((rows, n // 128), np.uint8)
    lib().oracle_quantize_rows(v, rows, n, q, sf)
    return q, sf


def quantize_rows_f32(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """1x128-block e4m3 quantisation with binary32 scales amax/448 -> (codes, scales)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    rows, n = v.shape
    q = np.empty((rows, n), np.uint8)
    s = np.empty((rows, n // 128), np.float32)
    lib().oracle_quantize_rows_f32(v, rows, n, q, s)
    return q, s


def scale_f32(amax: float) -> float:
    return lib().oracle_scale_f32(amax)


def f32_to_bf16(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_f32_to_bf16_array(v.reshape(-1), v.size, out.reshape(-1))
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def route(x: np.ndarray, W: np.ndarray, bias, cfg, tokens=None, nthreads: int = 0,
          want_logits: bool = False):
    """Top-K routing of tokens (all, or the listed ones): (topk_idx, topk_w[, logits])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = x.shape[0] if tok is None else tok.shape[0]
    idx = np.empty((n, cfg.K), np.int32)
    w = np.empty((n, cfg.K), np.float32)
    lg = np.empty((n, cfg.N), np.float32) if want_logits else None
    rc = lib().oracle_route(x, W, _ptr(b), cfg.H, cfg.N, cfg.K, cfg.n_group, cfg.topk_group,
                            cfg.score_fn, cfg.renorm, cfg.route_scale, _ptr(tok), n, idx, w,
                            _ptr(lg), nthreads)
    if rc != 0:
        raise ValueError("oracle_route: unsupported routing shape")
    return (idx, w, lg) if want_logits else (idx, w)


def expert_counts(topk_idx: np.ndarray, N: int) -> np.ndarray:
    return np.bincount(topk_idx.reshape(-1), minlength=N).astype(np.int32)


def eplb_build_map(counts: np.ndarray, N_log: int, N_phys: int):
    """(log2phys [N_log][2], rep [N_log], phys2log [N_phys])."""
    c = np.ascontiguousarray(counts, dtype=np.int64)
    l2p = np.empty((N_log, 2), np.int32)
    rep = np.empty(N_log, np.int32)
    p2l = np.empty(N_phys, np.int32)
    if lib().oracle_eplb_build_map(c, N_log, N_phys, l2p, rep, p2l) != 0:
        raise ValueError("eplb map: N_phys - N_log must lie in [0, N_log]")
    return l2p, rep, p2l


def contig_rows_alloc(B: int, K: int, N_phys: int) -> int:
    """Upper bound on rows of the contiguous layout: every segment padded to 128."""
    return ((B * K + N_phys * 127) + 127) // 128 * 128


def dispatch(x: np.ndarray, topk_idx: np.ndarray, cfg, log2phys=None, rep=None,
             fmt: int = 0, cap: int | None = None) -> dict:
    """Expert-major permutation + 1x128 e4m3 quantisation (see moe_oracle.c).
    log2phys [N_log][R] / rep: an EPLB map of R columns (eplb_build_map: R = 2)."""
    B, K, H = x.shape[0], topk_idx.shape[1], x.shape[1]
    Np = cfg.N_phys
    layout = cfg.layout
    cap = cfg.cap if cap is None else cap
    rows = contig_rows_alloc(B, K, Np) if layout == 0 else Np * cap
    phys = np.empty((B, K), np.int32)
    cnt = np.empty(Np, np.int32)
    seg = np.zeros(Np + 1, np.int32)
    row_of = np.empty((B, K), np.int32)
    src_of = np.empty(rows, np.int32)
    A = np.zeros((rows, H * (2 if fmt == 1 else 1)), np.uint8)
    sf = np.zeros((rows, H // 128), np.uint8)
    rc = lib().oracle_dispatch(np.ascontiguousarray(x, dtype=np.uint16),
                               np.ascontiguousarray(topk_idx, dtype=np.int32),
                               _ptr(None if log2phys is None else np.ascontiguousarray(log2phys, np.int32)),
                               _ptr(None if rep is None else np.ascontiguousarray(rep, np.int32)),
                               0 if log2phys is None else np.shape(log2phys)[1],
                               B, H, K, Np, layout, cap, fmt, phys, cnt, seg, row_of, src_of,
                               rows, A, sf)
    return dict(phys=phys, cnt=cnt, seg_start=seg, row_of=row_of, src_of=src_of, A=A, sf=sf,
                dropped=bool(rc & 2), rows=rows)


def combine(Y: np.ndarray, row_of: np.ndarray, w: np.ndarray, S=None) -> np.ndarray:
    """out[t] = bf16(sum_k w[t,k] * Y[row_of[t,k]] (+ S[t])), fp32 fma in k order."""
    B, K = row_of.shape
    H = Y.shape[1]
    out = np.empty((B, H), np.uint16)
    s = None if S is None else np.ascontiguousarray(S, dtype=np.uint16)
    lib().oracle_combine(np.ascontiguousarray(Y, dtype=np.uint16),
                         np.ascontiguousarray(row_of, dtype=np.int32),
                         np.ascontiguousarray(w, dtype=np.float32), _ptr(s), B, H, K, out)
    return out


from .ffn import (dequant_blocks, dequant_rows, dequant_rows_f32, expert_ffn,  # noqa: E402,F401
                  layer_tokens)
