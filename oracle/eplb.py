"""Oracle of the EPLB placement planner (moe_eplb_plan).

TEST INFRASTRUCTURE ONLY (see the package docstring).

DeepSeek's EPLB as the pages describe it, step by step in plain Python with exact
fractions: "Large-scale EP: DeepEP, EPLB and two-batch overlap", §EPLB — the
algorithm is hierarchical: expert groups are first packed onto nodes, then the
experts are placed within each node, so that a node's experts come from the same
groups; the mapping is recomputed from measured loads.  "SGLang开源首个对标官方性能的
DeepSeek-V3/R1 H100部署方案", §专家并行负载均衡器 — redundant slots (256 experts in
288 slots) hold extra copies of the most used experts, cold experts are stacked with
medium ones on one GPU, and balance is the mean over the maximum of the per-GPU
load.  The pages give no formulas; the plain readings taken here (greedy steps, a
replica carrying load / rep, ties to the lower index) are listed with the planner's
declaration in include/moe.h.
"""
from __future__ import annotations

from fractions import Fraction


def node_groups(group_load: list[int], n_nodes: int) -> list[list[int]]:
    """Step 1: the groups, heaviest first (ties: lower group), each to the lightest
    node (ties: lower node) among those holding fewer than G / n_nodes groups."""
    G = len(group_load)
    cap = G // n_nodes
    order = sorted(range(G), key=lambda g: (-group_load[g], g))
    held = [[] for _ in range(n_nodes)]
    node_load = [0] * n_nodes
    for g in order:
        open_nodes = [n for n in range(n_nodes) if len(held[n]) < cap]
        n = min(open_nodes, key=lambda n: (node_load[n], n))
        held[n].append(g)
        node_load[n] += group_load[g]
    return [sorted(h) for h in held]


def replicate(load: list[int], experts: list[int], slots: int, max_rep: int) -> dict[int, int]:
    """Step 2: one slot per expert, then each spare slot to the expert with the largest
    load per replica (ties: lower expert) that is below max_rep replicas."""
    rep = {e: 1 for e in experts}
    for _ in range(slots - len(experts)):
        cand = [e for e in experts if rep[e] < max_rep]
        best = max(cand, key=lambda e: (Fraction(load[e], rep[e]), -e))
        rep[best] += 1
    return rep


def pack(load: list[int], experts: list[int], rep: dict[int, int], n_gpus: int,
         slots_per_gpu: int):
    """Step 3: replicas (each load / rep), heaviest first (ties: lower expert), each to
    the lightest GPU with a free slot (ties: lower GPU).  Returns, per GPU, its
    experts in slot order, and the per-GPU loads."""
    items = [(Fraction(load[e], rep[e]), e) for e in experts for _ in range(rep[e])]
    items.sort(key=lambda it: (-it[0], it[1]))
    gpus = [[] for _ in range(n_gpus)]
    gload = [Fraction(0)] * n_gpus
    for w, e in items:
        free = [j for j in range(n_gpus) if len(gpus[j]) < slots_per_gpu]
        j = min(free, key=lambda j: (gload[j], j))
        gpus[j].append(e)
        gload[j] += w
    return gpus, gload


def plan(load, N_log: int, N_phys: int, n_group: int = 1, n_nodes: int = 1, n_gpus: int = 1,
         max_rep: int = 2):
    """(log2phys [N_log][max_rep], rep [N_log], phys2log [N_phys]) as lists, and the
    balance mean / max of the per-GPU loads."""
    load = [int(v) for v in load]
    hier = n_nodes > 1 and n_group % n_nodes == 0
    nodes = n_nodes if hier else 1
    gpn = n_gpus // nodes
    spg = N_phys // n_gpus
    if hier:
        gs = N_log // n_group
        glo = [sum(load[g * gs:(g + 1) * gs]) for g in range(n_group)]
        members = [[e for g in gl for e in range(g * gs, (g + 1) * gs)]
                   for gl in node_groups(glo, nodes)]
    else:
        members = [list(range(N_log))]
    rep = [1] * N_log
    phys2log = [None] * N_phys
    all_loads = []
    for n, experts in enumerate(members):
        r = replicate(load, experts, N_phys // nodes, max_rep)
        for e, v in r.items():
            rep[e] = v
        gpus, gload = pack(load, experts, r, gpn, spg)
        all_loads += gload
        for j, slot_experts in enumerate(gpus):
            for i, e in enumerate(slot_experts):
                phys2log[(n * gpn + j) * spg + i] = e
    log2phys = []
    for e in range(N_log):
        ids = [p for p in range(N_phys) if phys2log[p] == e]
        log2phys.append(ids + [ids[0]] * (max_rep - len(ids)))
    mx = max(all_loads)
    balance = float(sum(all_loads) / len(all_loads) / mx) if mx else 1.0
    return (log2phys, rep, phys2log), balance
