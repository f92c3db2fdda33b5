"""Seeded synthetic inputs for the MoE layer.

This module draws random numbers and nothing else: it holds none of the layer's
arithmetic (no routing, no quantisation rule, no GEMM).  The CPU oracle and the
CUDA path both take their inputs from here, so the two sides see the same bytes.

Recipe (all draws from NumPy PCG64 streams keyed by ``(seed, tag, index)``):

* ``x``         N(0, 1) float32, cast to bf16 by torch's round-to-nearest-even cast.
* router ``W``  fp32 ``[N][H]``: N(0, 1/H), or U(-sqrt(3/H), sqrt(3/H)) for the
                near-balanced prefill workload.
* ``bias``      fp32 ``[N]``: N(0, 0.01) (variance 0.01), or a Zipf profile
                ``bias[perm[r-1]] = -tau * s * ln r`` over a seeded permutation.
* expert weights are produced directly in their stored form, e4m3 codes plus one
                UE8M0 exponent byte per 128x128 block.  Codes are inverse-CDF samples
                of N(0, sigma_c^2) (sigma_c = 96 * 2^-j, torch's e4m3 cast of 65536
                normal quantiles), and the block exponent is ``e_base(fan_in) + j`` with
                j in {0, 1, 2} drawn per block.  The dequantised weight is then
                N(0, ~1/fan_in) in every block while the per-block exponents vary along
                both the N and the K direction.
Each expert is keyed separately, so any single expert can be regenerated alone.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from .configs import MoEConfig

_SIGMA_CODE = 96.0
_J_PROBS = (0.5, 0.3, 0.2)

TAG_X, TAG_ROUTER, TAG_BIAS, TAG_W13, TAG_W2, TAG_W13S, TAG_W2S, TAG_PERM = range(8)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16) via torch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def make_x(cfg: MoEConfig, seed: int | None = None, B: int | None = None) -> np.ndarray:
    """Token activations x, bf16 bits ``[B][H]``."""
    s = cfg.seed if seed is None else seed
    b = cfg.B if B is None else B
    return bf16_bits(_rng(s, TAG_X).standard_normal((b, cfg.H), dtype=np.float32))


def make_router(cfg: MoEConfig, seed: int | None = None) -> tuple[np.ndarray, np.ndarray | None]:
    """Router weight ``[N][H]`` fp32 and bias ``[N]`` fp32 (or None)."""
    s = cfg.seed if seed is None else seed
    r = _rng(s, TAG_ROUTER)
    if cfg.router_init == "uniform":
        a = math.sqrt(3.0 / cfg.H)
        W = r.uniform(-a, a, (cfg.N, cfg.H)).astype(np.float32)
    else:
        W = (r.standard_normal((cfg.N, cfg.H), dtype=np.float32)
             * np.float32(1.0 / math.sqrt(cfg.H))).astype(np.float32)
    if cfg.bias_init == "none":
        return W, None
    if cfg.bias_init == "normal":
        bias = (_rng(s, TAG_BIAS).standard_normal(cfg.N) * 0.1).astype(np.float32)
    elif cfg.bias_init == "zipf":
        perm = _rng(s, TAG_PERM).permutation(cfg.N)
        ranks = np.arange(1, cfg.N + 1, dtype=np.float64)
        bias = np.empty(cfg.N, np.float32)
        bias[perm] = (-cfg.zipf_tau * cfg.zipf_s * np.log(ranks)).astype(np.float32)
    else:
        raise ValueError(cfg.bias_init)
    return W, bias


_TABLES: np.ndarray | None = None


def _code_tables() -> np.ndarray:
    """uint8 [3][65536]: e4m3 codes of the 65536 quantiles of N(0, (96*2^-j)^2)."""
    global _TABLES
    if _TABLES is None:
        p = (torch.arange(65536, dtype=torch.float64) + 0.5) / 65536.0
        q = torch.special.ndtri(p)
        rows = []
        for j in range(3):
            v = (q * (_SIGMA_CODE * 2.0 ** -j)).clamp(-448.0, 448.0).to(torch.float32)
            rows.append(v.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        _TABLES = np.stack(rows).reshape(-1).copy()
    return _TABLES


def _e_base(fan_in: int) -> int:
    return int(round(math.log2(1.0 / (_SIGMA_CODE * math.sqrt(fan_in)))))


def make_fp8_matrix(rows: int, cols: int, key: tuple[int, ...],
                    out_codes: np.ndarray | None = None,
                    out_sf: np.ndarray | None = None) -> tuple[np.ndarray, np.ndarray]:
    """One weight matrix ``[rows][cols]`` (fan_in = cols) in stored form.

    Returns e4m3 codes (uint8 ``[rows][cols]``) and UE8M0 exponent bytes
    (uint8 ``[rows/128][cols/128]``, value = 2^(byte-127)).
    """
    assert rows % 128 == 0 and cols % 128 == 0
    nb, kb = rows // 128, cols // 128
    r = _rng(*key)
    j = r.choice(3, size=(nb, kb), p=_J_PROBS).astype(np.int32)
    idx = r.integers(0, 65536, size=(nb, 128, kb, 128), dtype=np.uint16)
    flat = (j[:, None, :, None] << 16) + idx.astype(np.int32)
    codes = _code_tables()[flat].reshape(rows, cols)
    sf = (127 + _e_base(cols) + j).astype(np.uint8)
    if out_codes is not None:
        out_codes[...] = codes
        codes = out_codes
    if out_sf is not None:
        out_sf[...] = sf
        sf = out_sf
    return codes, sf


def make_expert(cfg: MoEConfig, e: int, seed: int | None = None):
    """Weights of routed expert ``e``: (W13, W13_sf, W2, W2_sf).

    W13 ``[2I][H]`` rows [0, I) are the gate projection, rows [I, 2I) the up
    projection; W2 ``[H][I]`` is the down projection.
    """
    s = cfg.seed if seed is None else seed
    W13, W13_sf = make_fp8_matrix(2 * cfg.I, cfg.H, (s, TAG_W13, e))
    W2, W2_sf = make_fp8_matrix(cfg.H, cfg.I, (s, TAG_W2, e))
    return W13, W13_sf, W2, W2_sf


def make_shared_expert(cfg: MoEConfig, seed: int | None = None):
    s = cfg.seed if seed is None else seed
    W13, W13_sf = make_fp8_matrix(2 * cfg.I, cfg.H, (s, TAG_W13S, 0))
    W2, W2_sf = make_fp8_matrix(cfg.H, cfg.I, (s, TAG_W2S, 0))
    return W13, W13_sf, W2, W2_sf


def alloc_expert_weights(cfg: MoEConfig, pin: bool = False) -> dict:
    """Host buffers for all routed experts' stored weights."""
    def empty(*shape):
        return torch.empty(shape, dtype=torch.uint8, pin_memory=pin)
    N, H, I = cfg.N, cfg.H, cfg.I
    return dict(W13=empty(N, 2 * I, H), W13_sf=empty(N, 2 * I // 128, H // 128),
                W2=empty(N, H, I), W2_sf=empty(N, H // 128, I // 128))


def fill_expert_weights(cfg: MoEConfig, bufs: dict, seed: int | None = None,
                        threads: int | None = None) -> dict:
    """Fill the host buffers from :func:`alloc_expert_weights` with every expert."""
    s = cfg.seed if seed is None else seed
    n = [t.numpy() for t in (bufs["W13"], bufs["W13_sf"], bufs["W2"], bufs["W2_sf"])]

    def one(e):
        make_fp8_matrix(2 * cfg.I, cfg.H, (s, TAG_W13, e), n[0][e], n[1][e])
        make_fp8_matrix(cfg.H, cfg.I, (s, TAG_W2, e), n[2][e], n[3][e])

    with ThreadPoolExecutor(threads or min(32, (torch.get_num_threads() or 8))) as ex:
        list(ex.map(one, range(cfg.N)))
    return bufs


def make_all_experts(cfg: MoEConfig, seed: int | None = None) -> dict:
    """numpy dict of all routed experts' stored weights (small workloads)."""
    bufs = fill_expert_weights(cfg, alloc_expert_weights(cfg), seed)
    return {k: v.numpy() for k, v in bufs.items()}
