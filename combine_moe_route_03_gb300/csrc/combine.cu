// moe_combine: weighted gather-reduce of the expert outputs back to token order.
//
// Combine moves every expert output back to its token and reduces the K of them
// with the routing weights ("DeepEP 完全拆解", §专家并行 and §为什么 combine 比
// dispatch 慢).  Here it is a gather: for each token, the K rows of Y are summed in
// fp32 in the fixed rank order k = 0..K-1, so the result is deterministic (the
// page lists DeepEP's non-deterministic BF16 pre-reduction as a limitation,
// §局限).
//
// Single-batch overlap ("Single Batch Overlap (SBO)" PR, §2): with a signal
// array, a row is read only after the down GEMM has published all of its output
// tiles (acquire load of the row block's counter reaching the threshold).  The
// consumer's wait is bounded by one wall-clock limit for the whole launch; rows that
// are not ready by then are skipped and MOE_STATUS_TIMEOUT is raised.
//
// The combine can also run inside the down GEMM (moe_gemm_args.combine); the setup it
// needs, each (token, 128-column chunk)'s count of rows still to arrive, is written by
// moe_fused_combine_prep here.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kCombineWarps = 4;  // small CTAs: an SBO consumer fits beside a GEMM CTA

// One warp owns a task = (token, run of `cpt` consecutive 256-column chunks), so a
// small batch still spreads over many warps and every lane keeps K independent
// 16-byte loads in flight.
template <int KM>  // K <= KM
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(
    const uint16_t *__restrict__ Y, const int32_t *__restrict__ row_of,
    const float *__restrict__ topk_w, const uint16_t *__restrict__ S, uint16_t *__restrict__ out,
    int B, int H, int K, int cpt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = gridDim.x * kCombineWarps;
  const int nch = (H + 255) / 256;
  const int tpt = (nch + cpt - 1) / cpt;  // tasks per token
  const long ntasks = (long)B * tpt;
  for (long task = (long)blockIdx.x * kCombineWarps + warp; task < ntasks; task += nwarps) {
    const int t = (int)(task / tpt);
    const int c0 = (int)(task % tpt) * cpt;
    const int c1 = min(nch, c0 + cpt);
    int my_r = -1;
    float my_w = 0.0f;
    if (lane < K) {
      my_r = row_of[(size_t)t * K + lane];
      my_w = topk_w[(size_t)t * K + lane];
    }
    const bool use_s = S != nullptr;
    int r[KM];
    float w[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      r[k] = __shfl_sync(0xffffffffu, my_r, k);
      w[k] = __shfl_sync(0xffffffffu, my_w, k);
    }
    for (int c = c0; c < c1; ++c) {
      const int h = c * 256 + 8 * lane;
      if (h >= H) continue;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      // all K loads of the chunk first, then the sum in rank order
      uint4 y[KM];
#pragma unroll
      for (int k = 0; k < KM; ++k)
        y[k] = (k < K && r[k] >= 0)
                   ? __ldcg(reinterpret_cast<const uint4 *>(Y + (size_t)r[k] * H + h))
                   : make_uint4(0, 0, 0, 0);
      uint4 sv = make_uint4(0, 0, 0, 0);
      if (use_s) sv = __ldcs(reinterpret_cast<const uint4 *>(S + (size_t)t * H + h));
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        if (k >= K || r[k] < 0) continue;
        const uint4 v = y[k];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = __fmaf_rn(w[k], __uint_as_float(u[i] << 16), acc[2 * i]);
          acc[2 * i + 1] = __fmaf_rn(w[k], __uint_as_float(u[i] & 0xffff0000u), acc[2 * i + 1]);
        }
      }
      if (use_s) {
        const uint4 v = sv;
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(u[i] << 16));
          acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(u[i] & 0xffff0000u));
        }
      }
      uint4 o;
      o.x = f32_to_bf16_bits(acc[0]) | (f32_to_bf16_bits(acc[1]) << 16);
      o.y = f32_to_bf16_bits(acc[2]) | (f32_to_bf16_bits(acc[3]) << 16);
      o.z = f32_to_bf16_bits(acc[4]) | (f32_to_bf16_bits(acc[5]) << 16);
      o.w = f32_to_bf16_bits(acc[6]) | (f32_to_bf16_bits(acc[7]) << 16);
      __stcs(reinterpret_cast<uint4 *>(out + (size_t)t * H + h), o);
    }
  }
}

// Sum of one token's K rows (and its shared row) over 256-column chunks [c0, c1), in
// the rank order k = 0..K-1 (the arithmetic of combine_kernel, bit for bit), with all
// K + 1 loads of a chunk in flight.  r[k] < 0: rank k left out.
template <int KM>
__device__ __forceinline__ void reduce_token(const uint16_t *__restrict__ Y,
                                             const uint16_t *__restrict__ S,
                                             uint16_t *__restrict__ out, int t, int H, int K,
                                             int c0, int c1, const int *r, const float *w,
                                             bool use_s, int lane) {
  for (int c = c0; c < c1; ++c) {
    const int h = c * 256 + 8 * lane;
    if (h >= H) continue;
    uint4 y[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k)
      y[k] = (k < K && r[k] >= 0)
                 ? __ldcg(reinterpret_cast<const uint4 *>(Y + (size_t)r[k] * H + h))
                 : make_uint4(0, 0, 0, 0);
    const uint4 sv =
        use_s ? __ldcs(reinterpret_cast<const uint4 *>(S + (size_t)t * H + h)) : make_uint4(0, 0, 0, 0);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k >= K || r[k] < 0) continue;
      const uint32_t v[4] = {y[k].x, y[k].y, y[k].z, y[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(w[k], __uint_as_float(v[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w[k], __uint_as_float(v[i] & 0xffff0000u), acc[2 * i + 1]);
      }
    }
    if (use_s) {
      const uint32_t v[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(v[i] << 16));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(v[i] & 0xffff0000u));
      }
    }
    uint4 o;
    o.x = f32_to_bf16_bits(acc[0]) | (f32_to_bf16_bits(acc[1]) << 16);
    o.y = f32_to_bf16_bits(acc[2]) | (f32_to_bf16_bits(acc[3]) << 16);
    o.z = f32_to_bf16_bits(acc[4]) | (f32_to_bf16_bits(acc[5]) << 16);
    o.w = f32_to_bf16_bits(acc[6]) | (f32_to_bf16_bits(acc[7]) << 16);
    __stcs(reinterpret_cast<uint4 *>(out + (size_t)t * H + h), o);
  }
}

// The SBO consumer ("Single Batch Overlap (SBO)" PR, §2), launched beside the down GEMM.
// A token is ready once the row blocks of all its K rows (and of its shared row) have
// reached the threshold; a token's rows come from K experts spread over the GEMM's whole
// schedule, so tokens become ready in no useful order.  Each warp therefore owns a set
// of tasks (token, run of cpt 256-column chunks; tasks w, w + warps, ..., 64 at a time)
// and sweeps them without blocking, reducing a task as soon as its token is ready; it
// sleeps briefly only after a sweep that found nothing.  It runs on SMs of its own (the
// producing GEMM's grid leaves them free), so it never holds resources that a GEMM CTA
// it waits for would need.  One wall-clock limit bounds the whole launch: past it
// MOE_STATUS_TIMEOUT is raised and the remaining tasks are reduced without the rows still
// unpublished.
template <int KM>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_sbo_kernel(
    const uint16_t *__restrict__ Y, const int32_t *__restrict__ row_of,
    const float *__restrict__ topk_w, const uint16_t *__restrict__ S, uint16_t *__restrict__ out,
    int B, int H, int K, int cpt, const int32_t *signal, int threshold, int bm,
    int64_t timeout_ns, int64_t shared_row0, int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const int nw = gridDim.x * kCombineWarps;
  const int nch = (H + 255) / 256;
  const int tpt = (nch + cpt - 1) / cpt;  // tasks per token
  const long ntasks = (long)B * tpt;
  const long mine = gw < ntasks ? (ntasks - 1 - gw) / nw + 1 : 0;
  const uint64_t t0 = globaltimer();
  bool late = false;  // past the wall-clock limit
  for (long base = 0; base < mine; base += 64) {
    const int n = (int)min(64L, mine - base);
    uint64_t pending = n == 64 ? ~0ull : ((1ull << n) - 1);
    while (pending) {
      bool progress = false;
      for (uint64_t m = pending; m; m &= m - 1) {
        const int i = __ffsll((long long)m) - 1;
        const long task = gw + (base + i) * nw;
        const int t = (int)(task / tpt);
        const int c0 = (int)(task % tpt) * cpt;
        int my_r = -1;
        float my_w = 0.0f;
        int64_t sr = -1;
        if (lane < K) {
          my_r = row_of[(size_t)t * K + lane];
          my_w = topk_w[(size_t)t * K + lane];
          sr = my_r;
        } else if (lane == K && S) {
          sr = shared_row0 + t;
        }
        const bool ok = sr < 0 || ld_acquire_gpu(signal + sr / bm) >= threshold;
        if (!__all_sync(0xffffffffu, ok) && !late) continue;
        if (!ok) my_r = -1;  // past the limit: the row is left out
        const bool use_s = S && __shfl_sync(0xffffffffu, ok ? 1 : 0, K) != 0;
        int r[KM];
        float w[KM];
#pragma unroll
        for (int k = 0; k < KM; ++k) {
          r[k] = __shfl_sync(0xffffffffu, my_r, k);
          w[k] = __shfl_sync(0xffffffffu, my_w, k);
        }
        reduce_token<KM>(Y, S, out, t, H, K, c0, min(nch, c0 + cpt), r, w, use_s, lane);
        pending &= ~(1ull << i);
        progress = true;
      }
      if (pending && !progress) {
        if (!late && globaltimer() - t0 > (uint64_t)timeout_ns) {
          late = true;
          if (lane == 0) status_or(status, MOE_STATUS_TIMEOUT);
        } else {
          __nanosleep(256);
        }
      }
    }
  }
}

// Setup of the fused combine of the down GEMM (the reduce done where the rows are
// stored): pending[t][c] = 2 x (the ranks of t with a row + its shared row) for every
// 128-column chunk c (a full-width store of a row counts 2, a half-width one 1), and
// out[t] = 0 for a token with no row at all, which no store would ever complete
// (combine_kernel's empty sum).  One warp per token.
__global__ void __launch_bounds__(256) fused_combine_prep_kernel(
    const int32_t *__restrict__ row_of, int32_t *__restrict__ pending, uint16_t *__restrict__ out,
    int B, int K, int nch, int n, int shared) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= B) return;
  const bool has = lane < K && row_of[(size_t)t * K + lane] >= 0;
  const int cnt = __popc(__ballot_sync(0xffffffffu, has)) + (shared ? 1 : 0);
  for (int c = lane; c < nch; c += 32) pending[(size_t)t * nch + c] = 2 * cnt;
  if (cnt == 0)
    for (int h = 8 * lane; h < n; h += 256)
      *reinterpret_cast<uint4 *>(out + (size_t)t * n + h) = make_uint4(0, 0, 0, 0);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_fused_combine_prep(const moe_fused_combine *fc, int n, void *stream) {
  if (!fc || fc->B < 0 || fc->K < 1 || n <= 0) return MOE_ERR_INVALID;
  if (fc->K > 16 || n % 256) return MOE_ERR_UNSUPPORTED;
  if (fc->B == 0) return MOE_OK;
  if (!fc->row_of || !fc->pending || !fc->out || (uintptr_t)fc->out % 16) return MOE_ERR_INVALID;
  fused_combine_prep_kernel<<<(unsigned)((fc->B + 7) / 8), 256, 0, as_stream(stream)>>>(
      fc->row_of, fc->pending, static_cast<uint16_t *>(fc->out), fc->B, fc->K, n / 128, n,
      fc->shared_row0 >= 0 ? 1 : 0);
  return check_launch();
}

extern "C" int moe_combine(const moe_combine_cfg *c, const void *Y, const int32_t *row_of,
                           const float *topk_w, const void *shared, void *out, int32_t *status,
                           void *stream) {
  if (!c || c->B < 0 || c->H <= 0 || c->K <= 0) return MOE_ERR_INVALID;
  if (c->H % 128 || c->K > 16) return MOE_ERR_UNSUPPORTED;
  if (c->B == 0) return MOE_OK;
  if (!Y || !row_of || !topk_w || !out) return MOE_ERR_INVALID;
  if ((uintptr_t)Y % 16 || (uintptr_t)out % 16 || (shared && (uintptr_t)shared % 16))
    return MOE_ERR_INVALID;
  if (c->signal && (c->block_m_signal <= 0 || c->timeout_ns <= 0)) return MOE_ERR_INVALID;
  // chunks per task: enough tasks for ~4 resident warps per SM sub-partition
  const long nch = (c->H + 255) / 256;
  const long want = (long)device_sm_count() * 128;
  long cpt = ((long)c->B * nch) / want;
  cpt = cpt < 1 ? 1 : (cpt > nch ? nch : cpt);
  const long tasks = (long)c->B * ((nch + cpt - 1) / cpt);
  long grid = (tasks + kCombineWarps - 1) / kCombineWarps;
  if (c->num_ctas > 0 && c->num_ctas < grid) grid = c->num_ctas;
  if (c->signal) {  // the SBO consumer: tasks in the order their tokens become ready
    long g = c->num_ctas > 0 ? c->num_ctas : device_sm_count();
    // about two tasks per consumer warp, at least two chunks per task
    const long w = g * kCombineWarps;
    long sc = ((long)c->B * nch + 2 * w - 1) / (2 * w);
    sc = sc < 2 ? 2 : (sc > nch ? nch : sc);
    cpt = sc;
#define MOE_SBO_ARGS                                                                       \
  static_cast<const uint16_t *>(Y), row_of, topk_w, static_cast<const uint16_t *>(shared),   \
      static_cast<uint16_t *>(out), c->B, c->H, c->K, (int)cpt, c->signal, c->threshold,     \
      c->block_m_signal, c->timeout_ns, c->shared_row0, status
    if (c->K <= 8)
      combine_sbo_kernel<8><<<(unsigned)g, kCombineWarps * 32, 0, as_stream(stream)>>>(MOE_SBO_ARGS);
    else
      combine_sbo_kernel<16><<<(unsigned)g, kCombineWarps * 32, 0, as_stream(stream)>>>(MOE_SBO_ARGS);
#undef MOE_SBO_ARGS
    return check_launch();
  }
#define MOE_COMBINE_ARGS                                                                   \
  static_cast<const uint16_t *>(Y), row_of, topk_w, static_cast<const uint16_t *>(shared),   \
      static_cast<uint16_t *>(out), c->B, c->H, c->K, (int)cpt
  if (c->K <= 8)
    combine_kernel<8><<<(unsigned)grid, kCombineWarps * 32, 0, as_stream(stream)>>>(MOE_COMBINE_ARGS);
  else
    combine_kernel<16><<<(unsigned)grid, kCombineWarps * 32, 0, as_stream(stream)>>>(MOE_COMBINE_ARGS);
#undef MOE_COMBINE_ARGS
  return check_launch();
}
