"""Named MoE-layer workloads (shapes and input recipes only, no arithmetic).

Notation follows the MoE layer definition in "DeepEP 完全拆解" (§专家并行): B tokens,
N routed experts, top-K experts per token, hidden size H; I is the expert FFN's
intermediate size.  Group-limited gating ("DeepEP 完全拆解", §group-limited gating)
adds n_group groups of which topk_group survive.

The five workloads are the ones the method is measured on:

* ``tiny``      B=64, H=256, N=8, K=2, softmax router, contiguous layout.
* ``decode``    B=128, DeepSeek-V3-shaped layer (H=7168, 256 experts in 8 groups of
                32, top-4 groups, K=8, sigmoid + bias, weights normalised and x2.5,
                I=2048, one shared expert), masked layout with capacity 128.
* ``prefill``   B=8192 (4 sequences x 2048) of the same layer, contiguous layout,
                uniform router weights.
* ``skew``      B=4096 of the same layer, Zipf(1.2) router bias, run with 256
                physical experts and with 288 (EPLB, 32 replicas).
* ``sbo``       B=256 of the same layer, masked capacity 256, down GEMM signals
                per (expert, 64-row block) that the combine polls.

``small_*`` workloads are reduced shapes used by the parity tests: they keep the
structure (groups, bias, layouts, EPLB, ragged tails) at sizes the CPU oracle
finishes in seconds.
"""
from __future__ import annotations

import dataclasses

SOFTMAX = 0
SIGMOID = 1
CONTIG = 0
MASKED = 1


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    B: int                 # tokens
    H: int                 # hidden size
    N: int                 # logical routed experts
    K: int                 # experts per token
    I: int                 # expert FFN intermediate size
    n_group: int = 1
    topk_group: int = 1
    score_fn: int = SOFTMAX
    renorm: int = 0
    route_scale: float = 1.0
    shared: bool = False   # one shared expert of intermediate size I
    layout: int = CONTIG
    cap: int = 0           # masked capacity per physical expert (multiple of 128)
    n_phys: int = 0        # physical experts (0 -> N, no EPLB replicas)
    sbo: bool = False      # down GEMM signals + polling combine
    block_m_signal: int = 64
    router_init: str = "normal"   # "normal" N(0,1/H) or "uniform" U(-sqrt(3/H), sqrt(3/H))
    bias_init: str = "none"       # "none", "normal" (variance 0.01) or "zipf"
    zipf_s: float = 1.2
    zipf_tau: float = 0.05
    seed: int = 0
    scale_fmt: int = 0     # 0: UE8M0 power-of-two scales; 1: binary32 scales amax/448
    fuse_combine: bool = False  # the down GEMM reduces Y into out (no combine launch)

    @property
    def N_phys(self) -> int:
        return self.n_phys if self.n_phys else self.N

    @property
    def R(self) -> int:
        """Routed rows B*K."""
        return self.B * self.K

    def with_(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


_DSV3 = dict(H=7168, N=256, K=8, I=2048, n_group=8, topk_group=4, score_fn=SIGMOID,
             renorm=1, route_scale=2.5, shared=True)

TINY = MoEConfig("tiny", B=64, H=256, N=8, K=2, I=128, layout=CONTIG)
DECODE = MoEConfig("decode", B=128, layout=MASKED, cap=128, bias_init="normal", **_DSV3)
PREFILL = MoEConfig("prefill", B=8192, layout=CONTIG, router_init="uniform", **_DSV3)
SKEW = MoEConfig("skew", B=4096, layout=CONTIG, bias_init="zipf", **_DSV3)
SKEW_EPLB = SKEW.with_(name="skew_eplb", n_phys=288)
SBO = MoEConfig("sbo", B=256, layout=MASKED, cap=256, bias_init="normal", sbo=True, **_DSV3)

NAMED = {c.name: c for c in (TINY, DECODE, PREFILL, SKEW, SKEW_EPLB, SBO)}

# Reduced shapes with the same structure: 32 experts in 4 groups of 8, top-2 groups,
# K=4, sigmoid + bias; H and I span several 128-wide blocks; B is ragged.
_SMALL = dict(H=1024, N=32, K=4, I=512, n_group=4, topk_group=2, score_fn=SIGMOID,
              renorm=1, route_scale=2.5, shared=True, bias_init="normal")
SMALL_CONTIG = MoEConfig("small_contig", B=300, layout=CONTIG, **_SMALL)
SMALL_MASKED = MoEConfig("small_masked", B=200, layout=MASKED, cap=128, **_SMALL)
SMALL_EPLB = MoEConfig("small_eplb", B=333, layout=CONTIG, n_phys=40,
                       **{**_SMALL, "bias_init": "zipf"})
SMALL_SBO = MoEConfig("small_sbo", B=160, layout=MASKED, cap=256, sbo=True, **_SMALL)

SMALL = {c.name: c for c in (SMALL_CONTIG, SMALL_MASKED, SMALL_EPLB, SMALL_SBO)}
ALL = {**NAMED, **SMALL}

# Profiling shapes: the decode and prefill layers with 64 experts (8 groups of 8),
# so a profiler capture holds about 3 GB of weights instead of 11 GB while each
# expert keeps the full-size per-expert row counts (prefill: B*K/N = 256 rows).
_DSV3_64 = {**_DSV3, "N": 64}
DECODE_N64 = MoEConfig("decode_n64", B=128, layout=MASKED, cap=128, bias_init="normal",
                       **_DSV3_64)
PREFILL_N64 = MoEConfig("prefill_n64", B=2048, layout=CONTIG, router_init="uniform", **_DSV3_64)
PROFILE = {c.name: c for c in (DECODE_N64, PREFILL_N64)}
ALL.update(PROFILE)

# The SBO workload run sequentially (down GEMM on every SM, then the combine): the
# comparison arm of single-batch overlap.
SBO_SEQ = SBO.with_(name="sbo_seq", sbo=False)
# The decode layer with binary32 activation scales (1d2d with float scales, promoted per
# k-block in software) instead of power-of-two ones.
DECODE_F32 = DECODE.with_(name="decode_f32", scale_fmt=1)
# The combine fused into the down GEMM (each (token, 128 columns) reduced by the warp
# that stores its last row) instead of a separate pass over Y.
PREFILL_FC = PREFILL.with_(name="prefill_fc", fuse_combine=True)
SKEW_FC = SKEW.with_(name="skew_fc", fuse_combine=True)
DECODE_FC = DECODE.with_(name="decode_fc", fuse_combine=True)
VARIANTS = {c.name: c for c in (SBO_SEQ, DECODE_F32, PREFILL_FC, SKEW_FC, DECODE_FC)}
ALL.update(VARIANTS)
