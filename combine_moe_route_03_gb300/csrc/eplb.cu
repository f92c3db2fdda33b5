// moe_eplb_plan: expert placement from recorded loads — DeepSeek's EPLB algorithm as
// the pages describe it ("Large-scale EP: DeepEP, EPLB and two-batch overlap", §EPLB:
// hierarchical, expert groups packed onto nodes first and the experts placed within
// each node; "SGLang开源首个对标官方性能的DeepSeek-V3/R1 H100部署方案",
// §专家并行负载均衡器: copies of the most used experts in the redundant slots, cold
// experts stacked with medium ones on one GPU, balance = mean / max GPU load).
// Host code only; the rules (order, ties, slot numbering) are those of include/moe.h.
#include <algorithm>
#include <vector>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kEplbMaxRep = 8;
constexpr int64_t kRepLcm = 840;       // lcm(1..8): load * (840 / rep) is exact
constexpr int64_t kMaxLoad = 1ll << 40;

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_eplb_plan(const moe_eplb_cfg *c, const int64_t *load, int32_t *phys2log,
                             int32_t *log2phys, int32_t *rep, double *balance) {
  if (!c || !load || !phys2log || !log2phys || !rep) return MOE_ERR_INVALID;
  const int N = c->N_log, G = c->n_group, P = c->N_phys, R = c->max_rep;
  if (N < 1 || G < 1 || N % G || P < N || c->n_nodes < 1 || c->n_gpus < 1 ||
      c->n_gpus % c->n_nodes || P % c->n_gpus || R < 1 || R > kEplbMaxRep || P > 8192)
    return MOE_ERR_INVALID;
  for (int e = 0; e < N; ++e)
    if (load[e] < 0 || load[e] >= kMaxLoad) return MOE_ERR_INVALID;
  const bool hier = c->n_nodes > 1 && G % c->n_nodes == 0;
  const int nodes = hier ? c->n_nodes : 1;
  const int gpn = c->n_gpus / nodes;       // GPUs per node
  const int S = P / c->n_gpus;             // slots per GPU
  const int node_slots = P / nodes;
  const int per_node = N / nodes;          // logical experts per node
  if (node_slots < per_node || node_slots > per_node * R) return MOE_ERR_INVALID;

  // (1) groups -> nodes
  std::vector<std::vector<int>> members(nodes);
  if (hier) {
    const int gs = N / G, cap = G / nodes;
    std::vector<int64_t> gl(G, 0);
    for (int e = 0; e < N; ++e) gl[e / gs] += load[e];
    std::vector<int> order(G);
    for (int g = 0; g < G; ++g) order[g] = g;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return gl[a] > gl[b]; });
    std::vector<int64_t> nl(nodes, 0);
    std::vector<int> ng(nodes, 0);
    std::vector<std::vector<int>> groups(nodes);
    for (int g : order) {
      int best = -1;
      for (int n = 0; n < nodes; ++n)
        if (ng[n] < cap && (best < 0 || nl[n] < nl[best])) best = n;
      groups[best].push_back(g);
      nl[best] += gl[g];
      ++ng[best];
    }
    for (int n = 0; n < nodes; ++n) {
      std::sort(groups[n].begin(), groups[n].end());
      for (int g : groups[n])
        for (int e = g * gs; e < (g + 1) * gs; ++e) members[n].push_back(e);
    }
  } else {
    for (int e = 0; e < N; ++e) members[0].push_back(e);
  }

  for (int e = 0; e < N; ++e) rep[e] = 1;
  std::vector<int64_t> gpu_load(c->n_gpus, 0);
  for (int n = 0; n < nodes; ++n) {
    const std::vector<int> &m = members[n];
    // (2) replicas: each spare slot to the largest load per replica
    for (int extra = node_slots - per_node; extra > 0; --extra) {
      int best = -1;
      for (int e : m) {
        if (rep[e] >= R) continue;
        // load[e] / rep[e] > load[best] / rep[best], exactly
        if (best < 0 || load[e] * rep[best] > load[best] * rep[e]) best = e;
      }
      ++rep[best];
    }
    // (3) replicas onto the node's GPUs, heaviest first, each to the lightest GPU
    struct Item {
      int64_t w;
      int e;
    };
    std::vector<Item> items;
    for (int e : m)
      for (int r = 0; r < rep[e]; ++r) items.push_back({load[e] * (kRepLcm / rep[e]), e});
    std::stable_sort(items.begin(), items.end(), [](const Item &a, const Item &b) {
      return a.w != b.w ? a.w > b.w : a.e < b.e;
    });
    std::vector<int> fill(gpn, 0);
    for (const Item &it : items) {
      int best = -1;
      for (int j = 0; j < gpn; ++j)
        if (fill[j] < S && (best < 0 || gpu_load[n * gpn + j] < gpu_load[n * gpn + best]))
          best = j;
      const int g = n * gpn + best;
      phys2log[g * S + fill[best]] = it.e;
      ++fill[best];
      gpu_load[g] += it.w;
    }
  }
  // log2phys: e's physical experts ascending, the tail repeating the first
  std::vector<int> seen(N, 0);
  for (int p = 0; p < P; ++p) {
    const int e = phys2log[p];
    log2phys[(size_t)e * R + seen[e]++] = p;
  }
  for (int e = 0; e < N; ++e)
    for (int r = rep[e]; r < R; ++r) log2phys[(size_t)e * R + r] = log2phys[(size_t)e * R];
  if (balance) {
    int64_t mx = 0;
    double sum = 0.0;
    for (int64_t v : gpu_load) {
      mx = std::max(mx, v);
      sum += (double)v;
    }
    *balance = mx ? sum / c->n_gpus / (double)mx : 1.0;
  }
  return MOE_OK;
}
