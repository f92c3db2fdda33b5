"""MoE-layer throughput on GB300: route -> dispatch -> grouped FP8 FFN -> combine.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|prefill|...]
    python bench.py --impl reference ...     # the CPU oracle, timed on the host cores

One step = one pass of the whole layer (moe_layer_forward: route, dispatch, shared
expert, gate/up + SwiGLU, down, combine) over one batch of seeded synthetic input,
inputs resident in HBM; the K timed steps run as one CUDA graph of K passes, every
8th recording its stage events (their averages give each stage's duration).  `e2e` runs
K steps through the library's pipelined
host-buffer call (each step's x copied in from pinned host memory and its output copied
back, the copies of neighbouring steps overlapping the layer on a copy stream; all copies
inside the timed region).  Prints one JSON line (rank 0): the rates, the dominant
kernel against its roofline (`roofline`), every stage against the measured and nominal
peaks (`stages`), the step's expert balance, clocks, the oracle's rate on a sample of
the same workload (`cpu_baseline`) and, at one GPU, the other workloads timed the same
way after it (`workloads`: prefill, decode and skew with the combine fused into the down
GEMM, decode, SBO with and without the overlap, decode with binary32 scales, skew with
and without EPLB, tiny).  Under
torchrun each rank runs its own independent batch (weak scaling, no collective on the
data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from combine_moe_route_03_gb300 import _lib, api, configs, inputs  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 GB300; GEMM % FP8 peak; dispatch/combine % HBM BW"
UNIT = "tokens/s"
STAGES = _lib.STAGES


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def max_over_ranks(ms: float, dist, device) -> float:
    """Wall time of the slowest rank (every rank gets it)."""
    if dist is None:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Tokens/s of the whole job: every rank processes its own batch each step."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch recorded by an ncu capture (profiles/traffic.txt), or None
    when none exists or the GEMM sources changed since it was taken."""
    import hashlib
    csrc = os.path.join(ROOT, "combine_moe_route_03_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    sha = h.hexdigest()[:16]
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split("#")[0].split()
        if len(f) == 4 and f[0] == workload and f[1] == kernel and f[2] == sha:
            return int(f[3])
    return None


def describe(cfg) -> str:
    lay = "masked cap %d" % cfg.cap if cfg.layout == configs.MASKED else "contiguous"
    s = (f"{cfg.name}: B={cfg.B} H={cfg.H} N={cfg.N} K={cfg.K} I={cfg.I} "
         f"groups={cfg.n_group}/top{cfg.topk_group} {'sigmoid+bias' if cfg.score_fn else 'softmax'} "
         f"{lay}")
    if cfg.shared:
        s += " +1 shared expert"
    if cfg.N_phys != cfg.N:
        s += f" EPLB {cfg.N}->{cfg.N_phys}"
    if cfg.sbo:
        s += " SBO signals"
    return s


def stage_work(cfg, counts: np.ndarray) -> dict:
    """Algorithmic bytes and flops per launch of each stage (the minimum a stage must
    move: padding rows, unused capacity and scale replication not counted; a 1x128 or
    128x128 block's scale is one byte wherever it is written or read)."""
    B, H, N, K, I = cfg.B, cfg.H, cfg.N, cfg.K, cfg.I
    R = int(np.minimum(counts, cfg.cap).sum()) if cfg.layout == configs.MASKED else B * K
    Hb, Ib = H // 128, I // 128
    touched = counts > 0
    nt = int(touched.sum())
    w13 = 2 * I * H + (2 * I // 128) * Hb          # codes + one UE8M0 byte per block
    w2 = H * I + Hb * Ib
    sh = 1 if cfg.shared else 0
    work = {
        "route": dict(bytes=B * H * 2 + N * H * 4 + B * K * 8, flops=2 * B * H * N, bound="alu"),
        "dispatch": dict(bytes=B * H * 2 + R * (H + Hb + 8) + sh * B * (H + Hb), flops=0,
                         bound="hbm"),
        # the shared expert's B rows run inside the routed GEMM launches
        "gateup": dict(bytes=(nt + sh) * w13 + (R + sh * B) * (H + Hb + I + Ib),
                       flops=2 * (R + sh * B) * H * 2 * I, bound="hbm"),
        "down": dict(bytes=(nt + sh) * w2 + (R + sh * B) * (I + Ib + H * 2),
                     flops=2 * (R + sh * B) * I * H, bound="hbm"),
        "combine": dict(bytes=R * H * 2 + sh * B * H * 2 + R * 8 + B * H * 2, flops=0, bound="hbm"),
    }
    if cfg.fuse_combine:    # the down GEMM does the combine's work too
        work["down"]["bytes"] += work["combine"]["bytes"]
        work["combine"] = dict(bytes=0, flops=0, bound="hbm")
    return work


# Nominal GB300 figures, the secondary denominators (the measured ones are primary):
# HBM3e about 8 TB/s; dense e4m3 tensor throughput 4.5 PFLOP/s.
NOMINAL_HBM_GBS = 8000.0
NOMINAL_FP8_TFLOPS = 4500.0


def stage_summary(work: dict, stage_ms: dict, hbm_gbs: float, fp8_tflops: float) -> dict:
    """Per-stage duration, GB/s and TFLOP/s from the algorithmic work, as fractions of
    the measured HBM and e4m3 peaks and of the nominal ones."""
    out = {}
    for s in STAGES:
        d = stage_ms[s] * 1e-3
        if d <= 0 or not work[s]["bytes"]:
            continue
        gbs = work[s]["bytes"] / d / 1e9
        tfs = work[s]["flops"] / d / 1e12
        out[s] = {"ms": round(stage_ms[s], 4), "GBps": round(gbs, 1),
                  "hbm_frac": round(gbs / hbm_gbs, 3),
                  "hbm_frac_nominal": round(gbs / NOMINAL_HBM_GBS, 3),
                  "TFLOPs": round(tfs, 1)}
        if s in ("gateup", "down"):
            out[s]["fp8_frac"] = round(tfs / fp8_tflops, 3)
            out[s]["fp8_frac_nominal"] = round(tfs / NOMINAL_FP8_TFLOPS, 3)
    return out


def expert_balance(counts) -> dict:
    """Rows per physical expert in the last step: mean / max (1 = perfectly even), the
    balance measure the EPLB pages use, with the extremes."""
    c = np.asarray(counts, np.float64)
    top = float(c.max()) if c.size else 0.0
    return {"mean_over_max": round(float(c.mean()) / top, 4) if top > 0 else None,
            "max_rows": int(top), "min_rows": int(c.min()) if c.size else 0,
            "experts": int(c.size)}


def physical_work(cfg, counts_phys, phys2log) -> dict:
    """stage_work for an EPLB layout: replicas read their logical expert's weights."""
    logical = np.zeros(cfg.N, np.int64)
    np.add.at(logical, phys2log, counts_phys)
    return stage_work(cfg.with_(n_phys=0), logical)


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.p = gpu, None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def load_workload(cfg, dev):
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    host = inputs.fill_expert_weights(cfg, inputs.alloc_expert_weights(cfg))
    wdev = {k: v.to(dev) for k, v in host.items()}
    shared = None
    if cfg.shared:
        s = inputs.make_shared_expert(cfg)
        shared = s
        for k, v in zip(("W13s", "W13s_sf", "W2s", "W2s_sf"), s):
            wdev[k] = torch.from_numpy(v).to(dev)
    return x, W, bias, host, shared, wdev


def cpu_oracle_rate(cfg, x, W, bias, host, shared, ntok: int, seed: int = 0):
    """The oracle as it stands, full layer for `ntok` sampled tokens -> tokens/s."""
    import oracle
    oracle.build()
    ex = {k: v.numpy() for k, v in host.items()}
    get = lambda e: (ex["W13"][e], ex["W13_sf"][e], ex["W2"][e], ex["W2_sf"][e])  # noqa: E731
    tok = np.sort(np.random.default_rng(seed).choice(cfg.B, ntok, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    oracle.layer_tokens(cfg, x, W, bias, get, shared, tokens=tok)
    dt = time.perf_counter() - t0
    return ntok / dt, dt, tok


REF_BUDGET_S = 60.0  # timed oracle seconds the reference arm spends at most (about)


def streamed_weight_bytes(cfg, counts=None) -> int:
    """e4m3 weight bytes (+ one scale byte per block) the two GEMMs read per step: the
    touched experts' W13 and W2, and the shared expert's.  Without counts, every
    expert counts as touched (the bound for a large batch)."""
    touched = cfg.N if counts is None else int((np.asarray(counts) > 0).sum())
    per = 2 * cfg.I * cfg.H + cfg.H * cfg.I + 3 * (cfg.I // 128) * (cfg.H // 128)
    return (touched + (1 if cfg.shared else 0)) * per


def run_config(cfg, world):
    """The JSON line's `config`, the same for both arms: the reference arm times a
    sample of this workload (its cpu_baseline says which)."""
    per_mb = streamed_weight_bytes(cfg.with_(N=1, shared=False), None) / 1e6
    top_gb = streamed_weight_bytes(cfg, None) / 1e9
    return {"workload": describe(cfg), "global_batch": world * cfg.B,
            "parallelism": f"dp{world} (independent batch per GPU)",
            "l2": (f"inputs larger than L2 (129 MB): each step streams from HBM the e4m3 "
                   f"weights of the experts its batch touches ({per_mb:.1f} MB per expert, "
                   f"at most {top_gb:.1f} GB; weights_streamed_gb gives the step's figure)"
                   if top_gb > 0.129 else
                   f"weights ({top_gb * 1e3:.1f} MB) fit in L2 and stay resident between "
                   f"steps (no flush)")}


def measure(lay, st, K, warmup, dist=None, dev=None, sampler=None):
    """The timed region: one CUDA graph of K layer passes (the decode serving form:
    launches replayed, no host work per step), replayed once between CUDA events after
    `warmup` passes.  Every EVERY-th pass records its stage events as graph nodes; their
    averages give the per-kernel durations (an event node costs a few microseconds, so
    not every pass has them).  Returns (max over ranks of the total ms, stage ms)."""
    EVERY = 8
    sampled = list(range(0, K, EVERY))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(_lib.LAYER_EVENTS)]
           for _ in sampled]
    for row in evs:                      # torch creates the CUDA event on first record
        for e in row:
            e.record(st)
    torch.cuda.synchronize()
    steps_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(steps_graph, stream=st):
        for i in range(K):
            lay.forward(stream=st, events=evs[i // EVERY] if i % EVERY == 0 else None)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
        time.sleep(0.2)
    for _ in range(warmup):                         # the GPU idled while the sampler started
        lay.forward(stream=st)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):                     # replay() launches on the current stream
        t0.record(st)
        steps_graph.replay()
        t1.record(st)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    stage_ms = {s: float(np.mean([row[j].elapsed_time(row[j + 1]) for row in evs]))
                for j, s in enumerate(STAGES)}
    return ms_total, stage_ms


def roofline(cfg, work, stage_ms, pk, mhz, sms):
    """The dominant stage against its roofline: the tensor peak for a GEMM at (or within
    a quarter of) the ridge, HBM otherwise, FFMA units for the router."""
    # e4m3 = 2x bf16 (the nominal dense ratio 4.5 / 2.25 PFLOP/s); the burst figure, as
    # each GEMM launch is timed alone (well under a second), the sustained one beside it
    fp8_peak, fp8_peak_sus = 2.0 * pk["bf16"], 2.0 * pk["bf16_sus"]
    dom = max((s for s in STAGES if work[s]["bytes"]), key=lambda s: stage_ms[s])
    w = work[dom]
    dur = stage_ms[dom] * 1e-3
    t_hbm = w["bytes"] / (pk["hbm"] * 1e9)
    t_tc = w["flops"] / (fp8_peak * 1e12) if dom != "route" else 0.0
    if dom == "route":
        roof = {"bound": "alu", "achieved": w["flops"] / dur / 1e12, "unit": "TFLOP/s",
                "peak": sms * 128 * 2 * (mhz or 1900.0) * 1e6 / 1e12}  # FFMA units x clock
    elif t_tc >= 0.75 * t_hbm:
        roof = {"bound": "tensor", "achieved": w["flops"] / dur / 1e12, "peak": fp8_peak,
                "unit": "TFLOP/s", "frac_of_sustained": w["flops"] / dur / 1e12 / fp8_peak_sus}
    else:
        roof = {"bound": "hbm", "achieved": w["bytes"] / dur / 1e9, "peak": pk["hbm"],
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dom
    roof["peak_source"] = f"{pk['src']} ({'burst bf16 x2 for e4m3' if roof['bound'] == 'tensor' else 'hbm_gbs' if roof['bound'] == 'hbm' else 'FFMA units x clock'})"
    return roof


# Workloads timed after the headline one in the same run (at one GPU): the other named
# configurations, the combine fused into the down GEMM (prefill, decode, skew), the SBO
# workload run sequentially and the decode layer with binary32 scales; passes per
# workload.
EXTRAS = (("prefill_fc", 20), ("decode", 100), ("decode_fc", 100), ("sbo", 100),
          ("sbo_seq", 100), ("decode_f32", 100), ("skew", 20), ("skew_fc", 20),
          ("skew_eplb", 20), ("tiny", 100))


def run_extra(name, steps, base_cfg, wdev, dev, pk, mhz, sms, rank):
    """Times one more workload on the same box (its own inputs; the expert weights of
    the headline workload when the shapes and seed agree).  -> summary dict."""
    cfg = {**configs.NAMED, **configs.PROFILE, **configs.VARIANTS}[name]
    cfg = cfg.with_(seed=cfg.seed + rank)
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    same = (cfg.N, cfg.H, cfg.I, cfg.seed, cfg.shared) == (base_cfg.N, base_cfg.H, base_cfg.I,
                                                           base_cfg.seed, base_cfg.shared)
    wd = wdev if same else load_workload(cfg, dev)[5]
    Wd = torch.from_numpy(W).to(dev)
    bd = None if bias is None else torch.from_numpy(bias).to(dev)
    xd = torch.from_numpy(x).view(torch.bfloat16).to(dev)
    emap = None
    if cfg.N_phys != cfg.N:
        r = api.route(cfg, xd, Wd, bd)
        emap = api.eplb_build_map(r["counts"].cpu().numpy(), cfg.N, cfg.N_phys)
    lay = api.MoELayer(cfg, Wd, bd, wd, eplb_map=emap, device=dev)
    lay.x.copy_(xd)
    st = torch.cuda.Stream(device=dev)
    st.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        lay.forward(stream=st)
    torch.cuda.synchronize()
    status = api.read_status(lay.status)
    ms_total, stage_ms = measure(lay, st, steps, 3)
    counts = lay.counts.cpu().numpy()
    work = stage_work(cfg, counts) if emap is None else physical_work(cfg, counts, emap[2])
    roof = roofline(cfg, work, stage_ms, pk, mhz, sms)
    out = {"workload": describe(cfg), "ms_per_step": round(ms_total / steps, 5),
           "tokens_per_s": round(cfg.B / (ms_total / steps * 1e-3), 1), "steps": steps,
           "status": status,
           "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
           "dominant": {k: (round(v, 4) if isinstance(v, float) else v) for k, v in roof.items()
                        if k in ("kernel", "bound", "achieved", "peak", "unit", "frac")}}
    if name.startswith("skew"):
        out["expert_balance"] = expert_balance(counts)
    del lay
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_reference(args, cfg):
    """--impl reference: the CPU oracle on the host cores, one sampled token per step.

    An oracle token costs seconds (it dequantises its experts' whole weights to fp64),
    so the run is bounded: min(--warmup, 3) warm-up tokens, then timed tokens until
    `--steps` are done or about REF_BUDGET_S seconds of oracle time have accrued (at least
    one token); the line reports the tokens actually timed.  Expert weights are generated outside the
    timed region, as each token needs them."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x = inputs.make_x(cfg)
    W, bias = inputs.make_router(cfg)
    import oracle
    oracle.build()
    nwarm = max(1, min(args.warmup, 3))
    nmax = nwarm + args.steps
    tok = np.random.default_rng(7).choice(cfg.B, nmax, replace=nmax > cfg.B).astype(np.int32)
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = inputs.make_expert(cfg, e)
        return cache[e]
    shared = inputs.make_shared_expert(cfg) if cfg.shared else None
    idx, _ = oracle.route(x, W, bias, cfg, tokens=tok)
    times = []
    for i in range(nmax):
        for e in np.unique(idx[i]):          # untimed: this token's experts, generated
            get(int(e))
        t0 = time.perf_counter()
        oracle.layer_tokens(cfg, x, W, bias, get, shared, tokens=tok[i:i + 1])
        if i >= nwarm:                       # the first nwarm tokens warm up
            times.append(time.perf_counter() - t0)
            if sum(times) >= REF_BUDGET_S:
                break
        if len(cache) > 64:                  # bound host memory: keep the latest experts
            for e in list(cache)[:-32]:
                del cache[e]
    total = sum(times)
    n = len(times)
    value = n / total
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": n, "requested_steps": args.steps, "warmup": nwarm, "ms_per_step": 1e3 * total / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": run_config(cfg, int(os.environ.get("WORLD_SIZE", args.gpus))),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{n} sampled tokens of {cfg.name}, one per step through the "
                                       f"whole layer ({total:.1f} s of oracle time)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill",
                    choices=sorted(configs.NAMED) + sorted(configs.PROFILE) +
                    sorted(configs.VARIANTS))
    ap.add_argument("--cpu-tokens", type=int, default=12,
                    help="tokens of the CPU-oracle baseline sample (0 = skip)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="time only the chosen workload (not the others beside it)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    cfg = {**configs.NAMED, **configs.PROFILE, **configs.VARIANTS}[args.workload]
    if args.impl == "reference":
        return run_reference(args, cfg)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    cfg = cfg.with_(seed=cfg.seed + rank)           # independent batch per rank

    x, W, bias, host, shared, wdev = load_workload(cfg, dev)
    emap = None
    if cfg.N_phys != cfg.N:                          # EPLB map from an unreplicated pass
        r = api.route(cfg, torch.from_numpy(x).view(torch.bfloat16).to(dev),
                      torch.from_numpy(W).to(dev), torch.from_numpy(bias).to(dev))
        emap = api.eplb_build_map(r["counts"].cpu().numpy(), cfg.N, cfg.N_phys)
    lay = api.MoELayer(cfg, torch.from_numpy(W).to(dev),
                       None if bias is None else torch.from_numpy(bias).to(dev), wdev,
                       eplb_map=emap, device=dev)
    torch.cuda.empty_cache()
    lay.x.copy_(torch.from_numpy(x).view(torch.bfloat16).to(dev))
    st = torch.cuda.Stream(device=dev)              # graphs capture on a created stream
    st.wait_stream(torch.cuda.current_stream())
    for _ in range(args.warmup):
        lay.forward(stream=st)
    torch.cuda.synchronize()
    if api.read_status(lay.status) != 0:
        raise RuntimeError(f"device status {api.read_status(lay.status)}")

    sampler = ClockSampler(local)
    ms_total, stage_ms = measure(lay, st, args.steps, args.warmup, dist, dev, sampler)
    clocks = sampler.stop()
    K = args.steps
    ms_step = ms_total / K
    value = whole_job_rate(world, cfg.B, ms_step)

    # end to end through the library's pipelined host-buffer call: K steps, each copying
    # its batch in from pinned host memory and its output back, the copies of
    # neighbouring steps overlapping the layer (moe_layer_forward_host_pipelined)
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(x).view(torch.bfloat16).pin_memory()
        ohs = [torch.empty_like(xh).pin_memory() for _ in range(2)]
        cs = torch.cuda.Stream(device=dev)
        lay.forward_host_pipelined([xh] * 3, [ohs[i % 2] for i in range(3)], stream=st,
                                   copy_stream=cs)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        lay.forward_host_pipelined([xh] * K, [ohs[i % 2] for i in range(K)], stream=st,
                                   copy_stream=cs)
        b.record(st)
        torch.cuda.synchronize()
        ms = max_over_ranks(a.elapsed_time(b), dist, dev)
        e2e = {"value": whole_job_rate(world, cfg.B, ms / K), "unit": UNIT,
               "h2d_bytes_per_step": xh.numel() * 2, "d2h_bytes_per_step": ohs[0].numel() * 2}
    st = api.read_status(lay.status)
    if st != 0:
        raise RuntimeError(f"device status {st}")

    counts = lay.counts.cpu().numpy()
    work = (stage_work(cfg, counts) if emap is None
            else physical_work(cfg, counts, emap[2]))
    pk = peaks()
    fp8_peak = 2.0 * pk["bf16"]
    sms = _lib.load().moe_num_sms()
    roof = roofline(cfg, work, stage_ms, pk, clocks.get("sm_mhz"), sms)
    dom = roof["kernel"]
    roof["traffic"] = recorded_traffic(cfg.name, dom) if dom in ("gateup", "down") else None
    per_stage = stage_summary(work, stage_ms, pk["hbm"], fp8_peak)

    # route (logits, select), dispatch (count + scan fused into one launch for a
    # batch of one 128-token chunk, then scatter), gate/up, down, combine
    fused = cfg.B <= 128 and 4 * (8 * cfg.N_phys + 2 * 128 * cfg.K) <= 24 * 1024
    launches_per_step = 2 + (2 if fused else 3) + 2 + 1
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic (seeded; random-init weights stored as e4m3 + UE8M0 128x128 scales)",
            "config": run_config(cfg, world),
            "weights_streamed_gb": round(streamed_weight_bytes(
                cfg, counts if emap is None else np.bincount(emap[2][counts > 0], minlength=cfg.N)) / 1e9, 3),
            "clocks": clocks, "gpu_launches": launches_per_step * K, "roofline": roof,
            "stages": per_stage, "expert_balance": expert_balance(counts), "e2e": e2e}
    if rank == 0 and world == 1 and args.cpu_tokens > 0:
        rate, dt, tok = cpu_oracle_rate(cfg, x, W, bias, host, shared, args.cpu_tokens)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{len(tok)} sampled tokens of {cfg.name} through the "
                                          f"whole layer ({dt:.1f} s)"}
    if world == 1 and not args.no_extras:
        # the other workloads, timed on the same box after the headline one (reported
        # beside it; they do not enter value, ms_per_step or roofline)
        del lay
        torch.cuda.empty_cache()
        line["workloads"] = {
            name: run_extra(name, n, cfg, wdev, dev, pk, clocks.get("sm_mhz"), sms, rank)
            for name, n in EXTRAS if name != args.workload}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
