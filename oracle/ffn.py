"""Expert FFN of the oracle (TEST INFRASTRUCTURE ONLY), dequantised, in fp64.

Per expert ("DeepEP 完全拆解", §专家并行: each token goes through its K expert FFNs),
with the FP8 "1d2d" scaling of the "Single Batch Overlap (SBO)" PR, §3
(1x128 activation blocks, 128x128 weight blocks):

    a      = e4m3(A) * 2^(sf_A - 127)                 per 1x128 block of a row
    W      = e4m3(W) * 2^(sf_W - 127)                 per 128x128 block
    [g|u]  = a @ W13^T                                 (rows [0,I) gate, [I,2I) up)
    h      = g * sigmoid(g) * u                        (SwiGLU)
    h32    = fp32(h); (hq, sf_h) = 1x128 e4m3 quantisation of h32 (same rule as x)
    y      = bf16(fp32(dequant(hq) @ W2^T))

The matmuls are NumPy fp64 (a library primitive as one step); the dequantised
operands are exact in fp64 and each product of two e4m3 values is exact, so the
only rounding before the fp32/bf16 roundings is fp64 summation.

With scale_fmt = 1 the activations (x and h) carry binary32 scales amax/448 per 1x128
block instead of powers of two (quantize_rows_f32); a = e4m3(A) * s is again exact in
fp64, and the weights keep their 128x128 power-of-two scales (exact binary32 values).
"""
from __future__ import annotations

import numpy as np

from . import (bf16_to_f32, combine, e4m3_table, f32_to_bf16, quantize_rows, quantize_rows_f32,
               route)

_TABLE = None


def _table() -> np.ndarray:
    global _TABLE
    if _TABLE is None:
        _TABLE = e4m3_table()
    return _TABLE


def _pow2(sf: np.ndarray) -> np.ndarray:
    return np.ldexp(1.0, sf.astype(np.int32) - 127)


def dequant_rows(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """[m][n] e4m3 codes with [m][n/128] UE8M0 bytes -> fp64."""
    m, n = codes.shape
    v = _table()[codes].reshape(m, n // 128, 128)
    return (v * _pow2(sf)[:, :, None]).reshape(m, n)


def dequant_rows_f32(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    """[m][n] e4m3 codes with [m][n/128] binary32 scales -> fp64."""
    m, n = codes.shape
    v = _table()[codes].reshape(m, n // 128, 128)
    return (v * np.asarray(s, np.float64)[:, :, None]).reshape(m, n)


def dequant_blocks(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """[r][c] e4m3 codes with [r/128][c/128] UE8M0 bytes -> fp64."""
    r, c = codes.shape
    v = _table()[codes].reshape(r // 128, 128, c // 128, 128)
    return (v * _pow2(sf)[:, None, :, None]).reshape(r, c)


def expert_ffn(a_codes, a_sf, W13, W13_sf, W2, W2_sf, want_h: bool = False, scale_fmt: int = 0):
    """SwiGLU expert on quantised rows -> y as bf16 bits [m][H].  a_sf: UE8M0 bytes
    (scale_fmt 0) or binary32 scales (scale_fmt 1) per 1x128 block."""
    I = W13.shape[0] // 2
    a = dequant_rows(a_codes, a_sf) if scale_fmt == 0 else dequant_rows_f32(a_codes, a_sf)
    gu = a @ dequant_blocks(W13, W13_sf).T
    g, u = gu[:, :I], gu[:, I:]
    h = g / (1.0 + np.exp(-g)) * u
    if scale_fmt == 0:
        hq, hsf = quantize_rows(h.astype(np.float32))
        hd = dequant_rows(hq, hsf)
    else:
        hq, hsf = quantize_rows_f32(h.astype(np.float32))
        hd = dequant_rows_f32(hq, hsf)
    y = hd @ dequant_blocks(W2, W2_sf).T
    yb = f32_to_bf16(y.astype(np.float32))
    return (yb, hq, hsf, h) if want_h else yb


def layer_tokens(cfg, x, W_router, bias, get_expert, shared=None, tokens=None,
                 dropped=None, nthreads: int = 0, scale_fmt: int = 0):
    """The whole layer for a list of tokens (default: all), output bf16 bits.

    ``get_expert(e)`` returns (W13, W13_sf, W2, W2_sf) of logical expert e; replicas
    of an expert share its weights, so the output does not depend on the EPLB map
    or the layout.  ``dropped`` (bool [ntok][K]) marks rows a masked layout dropped
    for capacity; they are left out of the sum.
    """
    tok = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    idx, w = route(x, W_router, bias, cfg, tokens=tok, nthreads=nthreads)
    xs = bf16_to_f32(x[tok])
    q, sf = quantize_rows(xs) if scale_fmt == 0 else quantize_rows_f32(xs)
    ntok = tok.shape[0]
    Y = np.zeros((ntok * cfg.K, cfg.H), np.uint16)
    row_of = np.arange(ntok * cfg.K, dtype=np.int32).reshape(ntok, cfg.K)
    if dropped is not None:
        row_of = np.where(dropped, -1, row_of).astype(np.int32)
    for e in np.unique(idx):
        sel = np.argwhere(idx == e)
        if sel.size == 0:
            continue
        ws = get_expert(int(e))
        y = expert_ffn(q[sel[:, 0]], sf[sel[:, 0]], *ws, scale_fmt=scale_fmt)
        Y[sel[:, 0] * cfg.K + sel[:, 1]] = y
    S = expert_ffn(q, sf, *shared, scale_fmt=scale_fmt) if shared is not None else None
    out = combine(Y, row_of, w, S)
    return dict(out=out, topk_idx=idx, topk_w=w, S=S, Y=Y)
