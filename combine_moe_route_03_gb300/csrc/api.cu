// Host-side entry points of libmoe: error and status reporting, the EPLB map
// builder, and the whole-layer chain.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace moe {

static std::atomic<int> g_last_cuda_error{0};

int set_cuda_error(cudaError_t e) {
  g_last_cuda_error.store((int)e);
  return MOE_ERR_CUDA;
}

int device_slot() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  return dev >= 0 && dev < kMaxDevices ? dev : MOE_ERR_UNSUPPORTED;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_last_cuda_error(void) { return g_last_cuda_error.load(); }

extern "C" int moe_num_sms(void) { return device_sm_count(); }

extern "C" int moe_read_status(const int32_t *status, int32_t *host_status) {
  if (!status || !host_status) return MOE_ERR_INVALID;
  cudaError_t e = cudaMemcpy(host_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
}

// Redundant-expert placement: one replica for each of the N_phys - N_log most
// loaded logical experts ("Large-scale EP ...", §EPLB: 256 logical experts in 288
// physical slots, popular experts in several places, each copy taking a share).
extern "C" int eplb_build_map(const int64_t *counts_host, int N_log, int N_phys,
                              int32_t *log2phys, int32_t *rep, int32_t *phys2log) {
  if (!counts_host || !log2phys || !rep || !phys2log || N_log <= 0) return MOE_ERR_INVALID;
  const int extra = N_phys - N_log;
  if (extra < 0 || extra > N_log) return MOE_ERR_INVALID;
  std::vector<int> order(N_log);
  for (int e = 0; e < N_log; ++e) order[e] = e;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return counts_host[a] > counts_host[b]; });
  for (int e = 0; e < N_log; ++e) {
    log2phys[2 * e] = e;
    log2phys[2 * e + 1] = e;
    rep[e] = 1;
    phys2log[e] = e;
  }
  for (int i = 0; i < extra; ++i) {
    const int e = order[i];
    log2phys[2 * e + 1] = N_log + i;
    rep[e] = 2;
    phys2log[N_log + i] = e;
  }
  return MOE_OK;
}

namespace {

std::mutex g_order_mutex;
cudaEvent_t g_order_ev[kMaxDevices][2] = {};

// Makes `waiter` wait for the work enqueued so far on `signaler`, through one of the
// library's two events of the current device (created on first use).  Record and wait
// happen under one lock, so callers on other threads cannot slip their own record in
// between.  Only enqueues (also under stream capture, where it forks or joins streams).
int order_streams(cudaStream_t signaler, cudaStream_t waiter, int which) {
  const int dev = device_slot();
  if (dev < 0) return dev;
  std::lock_guard<std::mutex> lock(g_order_mutex);
  cudaEvent_t &ev = g_order_ev[dev][which];
  cudaError_t e = cudaSuccess;
  if (!ev) {
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      ev = nullptr;
      return set_cuda_error(e);
    }
  }
  e = cudaEventRecord(ev, signaler);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(waiter, ev, 0);
  return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
}

}  // namespace

extern "C" int moe_layer_forward(const moe_layer *L, void *stream) {
  if (!L) return MOE_ERR_INVALID;
  const moe_route_cfg &rc = L->route;
  cudaStream_t st = as_stream(stream);
  // Under stream capture a stage event becomes an event-record node of the graph, so
  // it records at every replay (a plain record would only order the capture).
  unsigned ev_flags = cudaEventRecordDefault;
  if (L->events) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
      ev_flags = cudaEventRecordExternal;
  }
  auto mark = [&](int i) {
    if (L->events) cudaEventRecordWithFlags(static_cast<cudaEvent_t>(L->events[i]), st, ev_flags);
  };
  if (L->has_shared && !L->shared_tiles) return MOE_ERR_INVALID;
  if (L->gemm_pairs < -1 || L->gemm_pairs > 1) return MOE_ERR_INVALID;
  const int sms = L->num_sms > 0 ? L->num_sms : device_sm_count();
  const int sbo_ctas = L->combine_ctas > 0 ? L->combine_ctas : 32;  // SBO consumer CTAs
  if (L->sbo && sbo_ctas >= sms) return MOE_ERR_INVALID;
  if (L->gemm_pairs == 1 && (rc.H % 256 || L->I % 256)) return MOE_ERR_UNSUPPORTED;
  if (L->scale_fmt != 0 && L->scale_fmt != 1) return MOE_ERR_INVALID;
  if (L->scale_fmt == 1 && L->gemm_pairs == 1) return MOE_ERR_UNSUPPORTED;
  if (L->fuse_combine != 0 && L->fuse_combine != 1) return MOE_ERR_INVALID;
  if (L->fuse_combine && (L->sbo || !L->src_of || !L->pending)) return MOE_ERR_INVALID;
  moe_dispatch_cfg dc;
  dc.B = rc.B;
  dc.H = rc.H;
  dc.K = rc.K;
  dc.N_log = rc.N;
  dc.N_phys = L->N_phys;
  dc.layout = L->layout;
  dc.cap = L->cap;
  dc.fmt = L->scale_fmt ? MOE_FMT_FP8_F32 : MOE_FMT_FP8;
  dc.max_rep = L->eplb_max_rep;
  // the row buffers and the tile list must hold what dispatch writes (before any launch)
  const int64_t need_rows = moe_dispatch_rows(&dc);
  if (need_rows > 0 && (L->rows < need_rows || L->max_tiles < need_rows / 128))
    return MOE_ERR_INVALID;
  const int64_t srows = L->has_shared ? ((int64_t)rc.B + 127) / 128 * 128 : 0;
  const int64_t rows_all = L->rows + srows;
  mark(0);
  int rc_ = moe_route(&rc, L->x, L->W_router, L->bias, L->topk_idx, L->topk_w, L->expert_counts,
                      L->route_ws, L->route_ws_bytes, stream);
  if (rc_) return rc_;
  mark(1);
  uint8_t *A = static_cast<uint8_t *>(L->A), *A_sf = static_cast<uint8_t *>(L->A_sf);
  rc_ = moe_dispatch(&dc, L->x, L->topk_idx, L->log2phys, L->rep, A, A_sf, L->counts, L->row_of,
                     L->fuse_combine ? L->src_of : nullptr, L->tiles,
                     L->has_shared ? A + L->rows * rc.H : nullptr,
                     L->has_shared ? A_sf + (L->scale_fmt ? (size_t)L->rows * (rc.H / 128) * 4
                                                          : (size_t)L->rows * sf_groups(rc.H) * 4)
                                   : nullptr,
                     L->has_shared ? L->shared_tiles : nullptr, L->dispatch_ws,
                     L->dispatch_ws_bytes, L->status, stream);
  if (rc_) return rc_;
  // the fused combine's counts, from the row_of just written
  moe_fused_combine fc{};
  if (L->fuse_combine) {
    fc.B = rc.B;
    fc.K = rc.K;
    fc.row_of = L->row_of;
    fc.topk_w = L->topk_w;
    fc.src_of = L->src_of;
    fc.src_rows = L->rows;
    fc.pending = L->pending;
    fc.shared_row0 = L->has_shared ? L->rows : -1;
    fc.out = L->out;
    if ((rc_ = moe_fused_combine_prep(&fc, rc.H, stream))) return rc_;
  }
  mark(2);
  moe_gemm_args g{};
  g.op = MOE_GEMM_GATEUP_SWIGLU;
  g.n = 2 * L->I;
  g.k = rc.H;
  g.rows = rows_all;            // A / H1 / Y hold the routed rows, then the shared rows
  g.max_tiles = L->max_tiles;   // capacity of the routed tile list (as dispatch wrote it)
  g.num_experts = rc.N + (L->has_shared ? 1 : 0);
  g.A = L->A;
  g.A_sf = L->A_sf;
  g.W = L->W13;
  g.W_sf = L->W13_sf;
  g.phys2log = L->phys2log;
  g.tiles = L->tiles;
  if (L->has_shared && srows > 0) {  // (an empty batch has no shared rows)
    g.tiles2 = L->shared_tiles;
    g.row_offset2 = L->rows;
    g.expert2 = rc.N;
  }
  g.out = L->H1;
  g.out_sf = L->H1_sf;
  g.num_sms = sms;
  g.status = L->status;
  // The gate/up GEMM on CTA pairs when experts average at least two M tiles (the long
  // K = H loop is bound by the MMA rate, which the pair form raises 1.5x per SM); one
  // CTA per tile otherwise, where most experts' single tile streams its weights from
  // HBM (decode, and skewed batches).  The down GEMM (K = I) runs one CTA per tile
  // unless pairs are forced: its deeper ring of 128-deep stages measured faster at
  // every batch (prefill 1.06 vs 1.10 ms, skew 0.75 vs 0.87 ms).
  const bool pairs_ok = !L->scale_fmt && rc.H % 256 == 0 && L->I % 256 == 0;
  const bool pairs_up = pairs_ok && (L->gemm_pairs == 1 ||
                                     (L->gemm_pairs == 0 &&
                                      (int64_t)rc.B * rc.K >= 256LL * L->N_phys));
  const bool pairs_down = pairs_ok && L->gemm_pairs == 1;
  g.pair_tiles = pairs_up ? 1 : 0;
  g.scale_fmt = L->scale_fmt;
  if ((rc_ = moe_grouped_gemm_fp8(&g, stream))) return rc_;
  mark(3);
  g.op = MOE_GEMM_DOWN;
  g.n = rc.H;
  g.k = L->I;
  g.A = L->H1;
  g.A_sf = L->H1_sf;
  g.W = L->W2;
  g.W_sf = L->W2_sf;
  g.pair_tiles = pairs_down ? 1 : 0;
  // 224-column tiles with two accumulators, when the layer has their scales
  if (L->W2_sf_t224 && !L->scale_fmt && !L->fuse_combine && !L->sbo && rc.H % 224 == 0) {
    g.tile_n = 224;
    g.W_sf = L->W2_sf_t224;
  }
  g.out = L->Y;
  g.out_sf = nullptr;
  moe_combine_cfg cc{};
  cc.B = rc.B;
  cc.H = rc.H;
  cc.K = rc.K;
  const void *S = L->has_shared ? static_cast<uint8_t *>(L->Y) + (size_t)L->rows * rc.H * 2
                                : nullptr;
  if (L->sbo) {
    if (!L->signal || !L->stream2 || L->stream2 == stream || L->block_m_signal <= 0 ||
        128 % L->block_m_signal)
      return MOE_ERR_INVALID;
    const size_t nsig = (size_t)(rows_all / L->block_m_signal);
    cudaError_t e = cudaMemsetAsync(L->signal, 0, nsig * sizeof(int32_t), st);
    if (e != cudaSuccess) return set_cuda_error(e);
    cudaStream_t st2 = as_stream(L->stream2);
    if ((rc_ = order_streams(st, st2, 0))) return rc_;
    g.signal = L->signal;
    g.block_m_signal = L->block_m_signal;
    g.num_sms = sms - sbo_ctas;  // the consumer's CTAs take SMs of their own
    if ((rc_ = moe_grouped_gemm_fp8(&g, stream))) return rc_;
    mark(4);
    cc.signal = L->signal;
    cc.threshold = rc.H / 256;
    cc.block_m_signal = L->block_m_signal;
    cc.timeout_ns = L->timeout_ns > 0 ? L->timeout_ns : 1000000000ll;
    cc.num_ctas = sbo_ctas;
    cc.shared_row0 = L->rows;
    if ((rc_ = moe_combine(&cc, L->Y, L->row_of, L->topk_w, S, L->out, L->status, L->stream2)))
      return rc_;
    if ((rc_ = order_streams(st2, st, 1))) return rc_;
    mark(5);
    return MOE_OK;
  }
  if (L->fuse_combine) {  // the down GEMM reduces Y into out as it stores it
    g.combine = &fc;
    if ((rc_ = moe_grouped_gemm_fp8(&g, stream))) return rc_;
    mark(4);
    mark(5);
    return MOE_OK;
  }
  if ((rc_ = moe_grouped_gemm_fp8(&g, stream))) return rc_;
  mark(4);
  rc_ = moe_combine(&cc, L->Y, L->row_of, L->topk_w, S, L->out, L->status, stream);
  if (rc_) return rc_;
  mark(5);
  return MOE_OK;
}

extern "C" int moe_layer_forward_host(const moe_layer *L, const void *x_host, void *out_host,
                                      void *stream) {
  if (!L || !x_host || !out_host) return MOE_ERR_INVALID;
  const size_t bytes = (size_t)L->route.B * L->route.H * 2;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(L->x, x_host, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  int rc = moe_layer_forward(L, stream);
  if (rc) return rc;
  e = cudaMemcpyAsync(out_host, L->out, bytes, cudaMemcpyDeviceToHost, st);
  return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
}

// Copies of neighbouring steps overlapped with the layer ("Large-scale EP ...", §TBO:
// data movement hidden behind the other batch's computation).  Per step i (buffer
// b = i % 2): stream waits for x(i) and for out(i-2)'s copy, runs the layer, records
// done(i); copy_stream then copies x(i+1) in (after done(i-1): the last reader of
// that input buffer) and out(i) back (after done(i)).
extern "C" int moe_layer_forward_host_pipelined(const moe_layer *L, void *x2, void *out2,
                                                const void *const *x_host,
                                                void *const *out_host, int n_steps,
                                                void *stream, void *copy_stream) {
  if (!L || !x2 || !out2 || !x_host || !out_host || n_steps < 1 || !copy_stream ||
      copy_stream == stream)
    return MOE_ERR_INVALID;
  for (int i = 0; i < n_steps; ++i)
    if (!x_host[i] || !out_host[i]) return MOE_ERR_INVALID;
  const size_t bytes = (size_t)L->route.B * L->route.H * 2;
  cudaStream_t st = as_stream(stream), cs = as_stream(copy_stream);
  void *xd[2] = {L->x, x2}, *od[2] = {L->out, out2};
  cudaEvent_t in_ready[2], done[2], out_copied[2];
  bool made[3][2] = {};
  cudaError_t e = cudaSuccess;
  int rc = MOE_OK;
  for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
    if ((e = cudaEventCreateWithFlags(&in_ready[b], cudaEventDisableTiming)) == cudaSuccess)
      made[0][b] = true;
    if (e == cudaSuccess &&
        (e = cudaEventCreateWithFlags(&done[b], cudaEventDisableTiming)) == cudaSuccess)
      made[1][b] = true;
    if (e == cudaSuccess &&
        (e = cudaEventCreateWithFlags(&out_copied[b], cudaEventDisableTiming)) == cudaSuccess)
      made[2][b] = true;
  }
  // copy_stream starts after the work already on stream (the caller's inputs may
  // have been prepared there)
  if (e == cudaSuccess) e = cudaEventRecord(done[1], st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, done[1], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(xd[0], x_host[0], bytes, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaEventRecord(in_ready[0], cs);
  for (int i = 0; e == cudaSuccess && i < n_steps; ++i) {
    const int b = i & 1;
    if ((e = cudaStreamWaitEvent(st, in_ready[b], 0)) != cudaSuccess) break;
    if (i >= 2 && (e = cudaStreamWaitEvent(st, out_copied[b], 0)) != cudaSuccess) break;
    moe_layer Lc = *L;
    Lc.x = xd[b];
    Lc.out = od[b];
    if ((rc = moe_layer_forward(&Lc, stream))) break;
    if ((e = cudaEventRecord(done[b], st)) != cudaSuccess) break;
    if (i + 1 < n_steps) {  // the next input, into the buffer step i-1 read
      if (i >= 1 && (e = cudaStreamWaitEvent(cs, done[b ^ 1], 0)) != cudaSuccess) break;
      if ((e = cudaMemcpyAsync(xd[b ^ 1], x_host[i + 1], bytes, cudaMemcpyHostToDevice, cs)) !=
          cudaSuccess)
        break;
      if ((e = cudaEventRecord(in_ready[b ^ 1], cs)) != cudaSuccess) break;
    }
    if ((e = cudaStreamWaitEvent(cs, done[b], 0)) != cudaSuccess) break;
    if ((e = cudaMemcpyAsync(out_host[i], od[b], bytes, cudaMemcpyDeviceToHost, cs)) !=
        cudaSuccess)
      break;
    if ((e = cudaEventRecord(out_copied[b], cs)) != cudaSuccess) break;
  }
  // stream follows the last copy (whatever was enqueued)
  if (made[2][0]) {
    cudaError_t e2 = cudaEventRecord(out_copied[0], cs);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, out_copied[0], 0);
    if (e == cudaSuccess) e = e2;
  }
  for (int k = 0; k < 3; ++k)
    for (int b = 0; b < 2; ++b)
      if (made[k][b]) cudaEventDestroy(k == 0 ? in_ready[b] : k == 1 ? done[b] : out_copied[b]);
  if (rc) return rc;
  return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
}

// Whole-layer CUDA graph ("Large-scale EP ...", §DeepEP: fixed shapes make decode
// replayable as a graph, which keeps launch overhead off each step).  Every call of
// the layer is stream work with no host synchronisation, so it captures as is.
extern "C" int moe_layer_graph_create(const moe_layer *L, const void *x_host, void *out_host,
                                      void *stream, void **graph) {
  if (!L || !graph || !stream) return MOE_ERR_INVALID;  // no capture on the legacy stream
  if ((x_host == nullptr) != (out_host == nullptr)) return MOE_ERR_INVALID;
  *graph = nullptr;
  moe_layer Lc = *L;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return set_cuda_error(e);
  const int rc = x_host ? moe_layer_forward_host(&Lc, x_host, out_host, stream)
                        : moe_layer_forward(&Lc, stream);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(st, &g);
  if (rc || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return rc ? rc : set_cuda_error(e);
  }
  cudaGraphExec_t ex = nullptr;
  e = cudaGraphInstantiate(&ex, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return set_cuda_error(e);
  *graph = ex;
  return MOE_OK;
}

extern "C" int moe_layer_graph_launch(void *graph, void *stream) {
  if (!graph) return MOE_ERR_INVALID;
  cudaError_t e = cudaGraphLaunch(static_cast<cudaGraphExec_t>(graph), as_stream(stream));
  return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
}

extern "C" int moe_layer_graph_destroy(void *graph) {
  if (!graph) return MOE_OK;
  cudaError_t e = cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(graph));
  return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
}
