// moe_route: router logits, scores, group-limited top-K and routing weights.
//
// The layer's router ("DeepEP 完全拆解", §专家并行) scores each token against N
// experts and keeps K; DeepSeek-V3's group-limited gating (same page, §group-limited
// gating) first keeps the best groups, then the best experts inside them.
//
// Kernels:
//   route_logits_kernel  z = x . W^T in fp32, each logit one fused multiply-add per
//                        k in order k = 0..H-1 (register-tiled SIMT: the ordering
//                        rule keeps this off the tensor cores, which round inputs
//                        and reorder partial sums).  Small grids.
//   route_logits_wide_kernel  the same arithmetic for wide grids: x widened to fp32
//                        once per CTA, larger per-thread tiles.
//   route_logits_pair_kernel  256 experts, large batches: a warp owns a slice of
//                        tokens against all experts, one CTA of 8 warps per SM; packed
//                        fp32 fmas (__ffma2_rn) advance two tokens' logits per
//                        instruction, each in its own sequential k order; each step's
//                        W and x operands are loaded into registers one step ahead.
//   route_select_kernel  one warp per token: scores, group scores, top-K with the
//                        (score desc, index asc) order, weights, expert counts.
#include <algorithm>
#include <cfloat>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 128;  // 4 warps: 2 (tokens) x 2 (experts)

// Warp tile: lanes as 4 (tokens) x 8 (experts); thread tile TT tokens x TE experts,
// strided by 4 and 8 so the shared-memory reads of one warp hit 4 and 8 distinct
// rows whose pitches (80 B for x, 144 B for W) put them in distinct banks.
// Operands stream through an S-stage cp.async ring of 32-wide k chunks (x stays
// bf16 in shared memory and is widened when read), so even the small decode grids
// keep enough loads in flight to cover the memory latency of each chunk.
template <int TT, int TE, int S, int kRouteBK>
__global__ void __launch_bounds__(kRouteThreads) route_logits_kernel(const uint16_t *__restrict__ x,
                                                                     const float *__restrict__ W,
                                                                     float *__restrict__ logits,
                                                                     int B, int H, int N) {
  constexpr int BT = 2 * 4 * TT;  // tokens per CTA
  constexpr int BE = 2 * 8 * TE;  // experts per CTA
  constexpr int LDX = kRouteBK + 8;  // bf16 per staged x row
  constexpr int LDW = kRouteBK + 4;  // fp32 per staged W row
  constexpr int XST = BT * LDX, WST = BE * LDW;
  extern __shared__ __align__(16) uint8_t route_smem[];
  uint16_t *xs = reinterpret_cast<uint16_t *>(route_smem);                // [S][BT][LDX]
  float *ws = reinterpret_cast<float *>(route_smem + S * XST * 2);        // [S][BE][LDW]

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int tl = lane >> 3, el = lane & 7;
  const int wt = warp >> 1, we = warp & 1;
  const int t0 = blockIdx.y * BT, e0 = blockIdx.x * BE;
  const int nchunks = H / kRouteBK;

  auto load = [&](int c, int buf) {
    const int kc = c * kRouteBK;
    constexpr int XP = kRouteBK / 8, WP = kRouteBK / 4;  // 16-byte pieces per row
    for (int i = tid; i < BT * XP; i += kRouteThreads) {
      const int t = i / XP, k = (i % XP) * 8;
      const bool ok = t0 + t < B;
      const uint16_t *src = x + (size_t)(ok ? t0 + t : 0) * H + kc + k;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                       smem_u32(xs + buf * XST + t * LDX + k)),
                   "l"(src), "r"(ok ? 16 : 0)
                   : "memory");
    }
    for (int i = tid; i < BE * WP; i += kRouteThreads) {
      const int e = i / WP, k = (i % WP) * 4;
      const bool ok = e0 + e < N;
      const float *src = W + (size_t)(ok ? e0 + e : 0) * H + kc + k;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                       smem_u32(ws + buf * WST + e * LDW + k)),
                   "l"(src), "r"(ok ? 16 : 0)
                   : "memory");
    }
  };

  // token pairs (2p, 2p+1) on packed fmas, acc[p][j] = their logits; an odd last
  // token on scalar fmas (acc1)
  constexpr int TP = TT / 2, TS = TT % 2;
  float2 acc[TP > 0 ? TP : 1][TE];
  float acc1[TE];
#pragma unroll
  for (int j = 0; j < TE; ++j) {
#pragma unroll
    for (int p = 0; p < TP; ++p) acc[p][j] = make_float2(0.0f, 0.0f);
    acc1[j] = 0.0f;
  }

#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    if (s < nchunks) load(s, s);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int c = 0; c < nchunks; ++c) {
    asm volatile("cp.async.wait_group %0;" ::"n"(S - 2) : "memory");
    __syncthreads();  // chunk c visible to all; chunk c-1's buffer no longer read
    if (c + S - 1 < nchunks) load(c + S - 1, (c + S - 1) % S);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const uint16_t *xb = xs + (c % S) * XST;
    const float *wb = ws + (c % S) * WST;
    // operands of step k4 + 4 are fetched while step k4's FMAs run
    uint2 xr[TT];
    float4 wr[TE];
    auto fetch = [&](int k4) {
#pragma unroll
      for (int i = 0; i < TT; ++i)
        xr[i] = *reinterpret_cast<const uint2 *>(xb + (wt * 4 * TT + tl + 4 * i) * LDX + k4);
#pragma unroll
      for (int j = 0; j < TE; ++j)
        wr[j] = *reinterpret_cast<const float4 *>(wb + (we * 8 * TE + el + 8 * j) * LDW + k4);
    };
    fetch(0);
#pragma unroll
    for (int k4 = 0; k4 < kRouteBK; k4 += 4) {
      float4 xv[TT], wv[TE];
#pragma unroll
      for (int i = 0; i < TT; ++i)
        xv[i] = make_float4(__uint_as_float(xr[i].x << 16), __uint_as_float(xr[i].x & 0xffff0000u),
                            __uint_as_float(xr[i].y << 16), __uint_as_float(xr[i].y & 0xffff0000u));
#pragma unroll
      for (int j = 0; j < TE; ++j) wv[j] = wr[j];
      if (k4 + 4 < kRouteBK) fetch(k4 + 4);
      // k order is strictly sequential for every output
#pragma unroll
      for (int j = 0; j < TE; ++j)
        if (TS) {
          acc1[j] = __fmaf_rn(xv[TT - 1].x, wv[j].x, acc1[j]);
          acc1[j] = __fmaf_rn(xv[TT - 1].y, wv[j].y, acc1[j]);
          acc1[j] = __fmaf_rn(xv[TT - 1].z, wv[j].z, acc1[j]);
          acc1[j] = __fmaf_rn(xv[TT - 1].w, wv[j].w, acc1[j]);
        }
#pragma unroll
      for (int p = 0; p < TP; ++p)
#pragma unroll
        for (int j = 0; j < TE; ++j) {
          acc[p][j] = __ffma2_rn(make_float2(xv[2 * p].x, xv[2 * p + 1].x),
                                 make_float2(wv[j].x, wv[j].x), acc[p][j]);
          acc[p][j] = __ffma2_rn(make_float2(xv[2 * p].y, xv[2 * p + 1].y),
                                 make_float2(wv[j].y, wv[j].y), acc[p][j]);
          acc[p][j] = __ffma2_rn(make_float2(xv[2 * p].z, xv[2 * p + 1].z),
                                 make_float2(wv[j].z, wv[j].z), acc[p][j]);
          acc[p][j] = __ffma2_rn(make_float2(xv[2 * p].w, xv[2 * p + 1].w),
                                 make_float2(wv[j].w, wv[j].w), acc[p][j]);
        }
    }
  }
#pragma unroll
  for (int i = 0; i < TT; ++i) {
    const int t = t0 + wt * 4 * TT + tl + 4 * i;
    if (t >= B) continue;
#pragma unroll
    for (int j = 0; j < TE; ++j) {
      const int e = e0 + we * 8 * TE + el + 8 * j;
      if (e < N)
        logits[(size_t)t * N + e] =
            (TS && i == TT - 1) ? acc1[j] : ((i & 1) ? acc[i / 2][j].y : acc[i / 2][j].x);
    }
  }
}

// Wide-grid variant: the same thread and warp tiling and the same k order, but each
// chunk's x is widened from bf16 to fp32 once, into a buffer the whole CTA reads, so
// the inner loop is 128-bit shared loads and fused multiply-adds only (every thread
// that shares a token would otherwise widen the same values again).  Chunk loop of
// one CTA: wait for chunk c | barrier | widen x(c) | refill the ring slot chunk c-1
// used | barrier | FMAs of chunk c.  The first barrier also ends every read of the
// widened buffer by chunk c-1, so one buffer is enough.  Large tiles (up to 8 x 8 per
// thread) pay off once the grid has CTAs to spare; small grids keep the bf16 kernel.
template <int TT, int TE, int S, int BK>
__global__ void __launch_bounds__(kRouteThreads) route_logits_wide_kernel(
    const uint16_t *__restrict__ x, const float *__restrict__ W, float *__restrict__ logits,
    int B, int H, int N) {
  constexpr int BT = 2 * 4 * TT;  // tokens per CTA
  constexpr int BE = 2 * 8 * TE;  // experts per CTA
  constexpr int LDH = BK + 8;     // bf16 per staged x row
  constexpr int LDF = BK + 4;     // fp32 per widened x row and staged W row
  constexpr int XST = BT * LDH, WST = BE * LDF;
  extern __shared__ __align__(16) uint8_t route_smem[];
  float *ws = reinterpret_cast<float *>(route_smem);           // [S][BE][LDF]
  float *xf = ws + S * WST;                                    // [BT][LDF]
  uint16_t *xs = reinterpret_cast<uint16_t *>(xf + BT * LDF);  // [S][BT][LDH]

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int tl = lane >> 3, el = lane & 7;
  const int wt = warp >> 1, we = warp & 1;
  const int t0 = blockIdx.y * BT, e0 = blockIdx.x * BE;
  const int nchunks = H / BK;

  auto load = [&](int c, int buf) {
    const int kc = c * BK;
    constexpr int XP = BK / 8, WP = BK / 4;  // 16-byte pieces per row
    for (int i = tid; i < BT * XP; i += kRouteThreads) {
      const int t = i / XP, k = (i % XP) * 8;
      const bool ok = t0 + t < B;
      const uint16_t *src = x + (size_t)(ok ? t0 + t : 0) * H + kc + k;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                       smem_u32(xs + buf * XST + t * LDH + k)),
                   "l"(src), "r"(ok ? 16 : 0)
                   : "memory");
    }
    for (int i = tid; i < BE * WP; i += kRouteThreads) {
      const int e = i / WP, k = (i % WP) * 4;
      const bool ok = e0 + e < N;
      const float *src = W + (size_t)(ok ? e0 + e : 0) * H + kc + k;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                       smem_u32(ws + buf * WST + e * LDF + k)),
                   "l"(src), "r"(ok ? 16 : 0)
                   : "memory");
    }
  };

  static_assert(TT % 2 == 0, "tokens per thread come in pairs");
  float2 acc[TT / 2][TE];  // packed fmas over token pairs, as in route_logits_kernel
#pragma unroll
  for (int p = 0; p < TT / 2; ++p)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc[p][j] = make_float2(0.0f, 0.0f);

#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    if (s < nchunks) load(s, s);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int c = 0; c < nchunks; ++c) {
    asm volatile("cp.async.wait_group %0;" ::"n"(S - 2) : "memory");
    __syncthreads();
    {  // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 word
      const uint16_t *xb = xs + (c % S) * XST;
      for (int i = tid; i < BT * BK / 8; i += kRouteThreads) {
        const int t = i / (BK / 8), k = (i % (BK / 8)) * 8;
        const uint4 v = *reinterpret_cast<const uint4 *>(xb + t * LDH + k);
        float4 *d = reinterpret_cast<float4 *>(xf + t * LDF + k);
        d[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
        d[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                           __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
      }
    }
    if (c + S - 1 < nchunks) load(c + S - 1, (c + S - 1) % S);
    asm volatile("cp.async.commit_group;" ::: "memory");
    __syncthreads();
    const float *wb = ws + (c % S) * WST;
#pragma unroll
    for (int k4 = 0; k4 < BK; k4 += 4) {
      float4 xv[TT], wv[TE];
#pragma unroll
      for (int i = 0; i < TT; ++i)
        xv[i] = *reinterpret_cast<const float4 *>(xf + (wt * 4 * TT + tl + 4 * i) * LDF + k4);
#pragma unroll
      for (int j = 0; j < TE; ++j)
        wv[j] = *reinterpret_cast<const float4 *>(wb + (we * 8 * TE + el + 8 * j) * LDF + k4);
      // k order is strictly sequential for every output
#pragma unroll
      for (int p = 0; p < TT / 2; ++p)
#pragma unroll
        for (int j = 0; j < TE; ++j) {
          acc[p][j] = __ffma2_rn(make_float2(xv[2 * p].x, xv[2 * p + 1].x),
                                 make_float2(wv[j].x, wv[j].x), acc[p][j]);
          acc[p][j] = __ffma2_rn(make_float2(xv[2 * p].y, xv[2 * p + 1].y),
                                 make_float2(wv[j].y, wv[j].y), acc[p][j]);
          acc[p][j] = __ffma2_rn(make_float2(xv[2 * p].z, xv[2 * p + 1].z),
                                 make_float2(wv[j].z, wv[j].z), acc[p][j]);
          acc[p][j] = __ffma2_rn(make_float2(xv[2 * p].w, xv[2 * p + 1].w),
                                 make_float2(wv[j].w, wv[j].w), acc[p][j]);
        }
    }
  }
#pragma unroll
  for (int i = 0; i < TT; ++i) {
    const int t = t0 + wt * 4 * TT + tl + 4 * i;
    if (t >= B) continue;
#pragma unroll
    for (int j = 0; j < TE; ++j) {
      const int e = e0 + we * 8 * TE + el + 8 * j;
      if (e < N) logits[(size_t)t * N + e] = (i & 1) ? acc[i / 2][j].y : acc[i / 2][j].x;
    }
  }
}

// Token-sliced kernel for wide batches: one CTA of NW warps per SM, and each warp owns
// TT consecutive tokens (TT = B / (NW * SMs), rounded up) against all 32 * TE experts:
// lane l takes experts l, l + 32, ...  Per 4-deep k step a lane loads its TE rows of W
// (distinct addresses) and its tokens' x as warp-wide broadcast loads (half the
// shared-memory cost of a distinct load); the token slicing keeps every SM equally
// loaded (a fixed 2-D tiling of 2^21 logits over 152 SMs leaves a sixth of them idle).
// The token-sliced kernel on packed fp32 fused multiply-adds: __ffma2_rn performs two
// independent binary32 fmas (round to nearest even) in one instruction, so each one
// advances two tokens' logits of one expert, each chain still in the sequential k order
// (bit for bit the scalar kernel's results) while the multiply-add instructions halve.
// A warp's TT tokens form TT/2 pairs plus, for odd TT, one token on scalar fmas.  Each
// warp widens its own tokens' x of a chunk as its pairs, {x_2p(k), x_2p+1(k)} for k = 0,
// 1, ..., then its odd token, so a broadcast 16-byte load yields two k steps of a pair
// (or four of the odd token), and only a warp sync separates that pass from the fmas:
// one CTA barrier per chunk (chunk landed; the ring slot of chunk c-1 free).  W is
// staged and read as in the scalar kernel.  With 8 warps the four SM sub-partitions
// carry equal work.
template <int TT, int TE, int S, int BK, int NW>
__global__ void __launch_bounds__(NW * 32, 1) route_logits_pair_kernel(
    const uint16_t *__restrict__ x, const float *__restrict__ W, float *__restrict__ logits,
    int B, int H) {
  constexpr int TP = TT / 2, TS = TT % 2;
  constexpr int BT = NW * TT, NE = 32 * TE, NT = NW * 32;
  constexpr int LDH = BK + 8, LDF = BK + 4, LDP = 2 * BK + 4;
  constexpr int XW = TP * LDP + TS * LDF;  // one warp's widened x, floats
  constexpr int XST = BT * LDH, WST = NE * LDF;
  extern __shared__ __align__(16) uint8_t route_smem[];
  float *ws = reinterpret_cast<float *>(route_smem);           // [S][NE][LDF]
  float *xp = ws + S * WST;                                    // [NW][XW]
  uint16_t *xs = reinterpret_cast<uint16_t *>(xp + NW * XW);   // [S][BT][LDH]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * BT;
  const int nchunks = H / BK;

  auto load = [&](int c, int buf) {
    const int kc = c * BK;
    constexpr int XP = BK / 8, WP = BK / 4;
    for (int i = tid; i < BT * XP; i += NT) {
      const int t = i / XP, k = (i % XP) * 8;
      const bool ok = t0 + t < B;
      const uint16_t *src = x + (size_t)(ok ? t0 + t : 0) * H + kc + k;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                       smem_u32(xs + buf * XST + t * LDH + k)),
                   "l"(src), "r"(ok ? 16 : 0)
                   : "memory");
    }
    for (int i = tid; i < NE * WP; i += NT) {
      const int e = i / WP, k = (i % WP) * 4;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                       smem_u32(ws + buf * WST + e * LDF + k)),
                   "l"(W + (size_t)e * H + kc + k)
                   : "memory");
    }
  };
  auto widen8 = [](uint32_t u, float &lo, float &hi) {  // bf16 -> fp32 is exact
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
  };

  float2 acc[TP > 0 ? TP : 1][TE];
  float acc1[TE];
#pragma unroll
  for (int j = 0; j < TE; ++j) {
#pragma unroll
    for (int p = 0; p < TP; ++p) acc[p][j] = make_float2(0.0f, 0.0f);
    acc1[j] = 0.0f;
  }
#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    if (s < nchunks) load(s, s);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int c = 0; c < nchunks; ++c) {
    asm volatile("cp.async.wait_group %0;" ::"n"(S - 2) : "memory");
    __syncthreads();
    {  // widen x: each warp its own token pairs (interleaved), then its odd token
      const uint16_t *xb = xs + (c % S) * XST;
      constexpr int R = TP + TS;  // rows per warp
      const int w = warp;
      for (int i = lane; i < R * (BK / 8); i += 32) {
        const int rr = i / (BK / 8), k = (i % (BK / 8)) * 8;
        const int tw = w * TT + 2 * rr;  // first token of the row in the CTA
        const uint4 a = *reinterpret_cast<const uint4 *>(xb + tw * LDH + k);
        const uint32_t ua[4] = {a.x, a.y, a.z, a.w};
        if (rr < TP) {
          const uint4 b = *reinterpret_cast<const uint4 *>(xb + (tw + 1) * LDH + k);
          const uint32_t ub[4] = {b.x, b.y, b.z, b.w};
          float4 *d = reinterpret_cast<float4 *>(xp + w * XW + rr * LDP + 2 * k);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float a0, a1, b0, b1;
            widen8(ua[q], a0, a1);
            widen8(ub[q], b0, b1);
            d[q] = make_float4(a0, b0, a1, b1);
          }
        } else {
          float4 *d = reinterpret_cast<float4 *>(xp + w * XW + TP * LDP + k);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float a0, a1, a2, a3;
            widen8(ua[2 * q], a0, a1);
            widen8(ua[2 * q + 1], a2, a3);
            d[q] = make_float4(a0, a1, a2, a3);
          }
        }
      }
    }
    __syncwarp();  // only this warp reads its widened rows
    if (c + S - 1 < nchunks) load(c + S - 1, (c + S - 1) % S);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const float *wb = ws + (c % S) * WST + lane * LDF;
    const float *xw = xp + warp * XW;
    // operands of step k4 + 4 are loaded while step k4's fmas run
    float4 wn[TE], xn[TP > 0 ? TP : 1][2], x1n;
    auto fetch = [&](int k4) {
#pragma unroll
      for (int j = 0; j < TE; ++j) wn[j] = *reinterpret_cast<const float4 *>(wb + 32 * j * LDF + k4);
#pragma unroll
      for (int p = 0; p < TP; ++p)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          xn[p][h] = *reinterpret_cast<const float4 *>(xw + p * LDP + 2 * k4 + 4 * h);
      if (TS) x1n = *reinterpret_cast<const float4 *>(xw + TP * LDP + k4);
    };
    fetch(0);
#pragma unroll
    for (int k4 = 0; k4 < BK; k4 += 4) {
      float4 wv[TE], xc[TP > 0 ? TP : 1][2], x1;
#pragma unroll
      for (int j = 0; j < TE; ++j) wv[j] = wn[j];
#pragma unroll
      for (int p = 0; p < TP; ++p) {
        xc[p][0] = xn[p][0];
        xc[p][1] = xn[p][1];
      }
      x1 = x1n;
      if (k4 + 4 < BK) fetch(k4 + 4);
      // k order strictly sequential per logit
#pragma unroll
      for (int p = 0; p < TP; ++p) {
        const float2 x0 = make_float2(xc[p][0].x, xc[p][0].y);
        const float2 xk1 = make_float2(xc[p][0].z, xc[p][0].w);
        const float2 x2 = make_float2(xc[p][1].x, xc[p][1].y);
        const float2 x3 = make_float2(xc[p][1].z, xc[p][1].w);
#pragma unroll
        for (int j = 0; j < TE; ++j) {
          acc[p][j] = __ffma2_rn(x0, make_float2(wv[j].x, wv[j].x), acc[p][j]);
          acc[p][j] = __ffma2_rn(xk1, make_float2(wv[j].y, wv[j].y), acc[p][j]);
          acc[p][j] = __ffma2_rn(x2, make_float2(wv[j].z, wv[j].z), acc[p][j]);
          acc[p][j] = __ffma2_rn(x3, make_float2(wv[j].w, wv[j].w), acc[p][j]);
        }
      }
      if (TS) {
#pragma unroll
        for (int j = 0; j < TE; ++j) {
          acc1[j] = __fmaf_rn(x1.x, wv[j].x, acc1[j]);
          acc1[j] = __fmaf_rn(x1.y, wv[j].y, acc1[j]);
          acc1[j] = __fmaf_rn(x1.z, wv[j].z, acc1[j]);
          acc1[j] = __fmaf_rn(x1.w, wv[j].w, acc1[j]);
        }
      }
    }
  }
  const int tw = t0 + warp * TT;
#pragma unroll
  for (int j = 0; j < TE; ++j) {
#pragma unroll
    for (int p = 0; p < TP; ++p) {
      if (tw + 2 * p < B) logits[(size_t)(tw + 2 * p) * NE + 32 * j + lane] = acc[p][j].x;
      if (tw + 2 * p + 1 < B) logits[(size_t)(tw + 2 * p + 1) * NE + 32 * j + lane] = acc[p][j].y;
    }
    if (TS && tw + TT - 1 < B) logits[(size_t)(tw + TT - 1) * NE + 32 * j + lane] = acc1[j];
  }
}

struct Cand {
  float v;  // choice score
  int i;    // expert index (INT_MAX = none)
  float s;  // weight score of that expert
};

// a ranks before b: larger score first, equal scores -> lower index first.
__device__ __forceinline__ bool before(const Cand &a, const Cand &b) {
  if (a.i == INT_MAX) return false;
  if (b.i == INT_MAX) return true;
  return a.v > b.v || (a.v == b.v && a.i < b.i);
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Cand o;
    o.v = __shfl_xor_sync(0xffffffffu, c.v, off);
    o.i = __shfl_xor_sync(0xffffffffu, c.i, off);
    o.s = __shfl_xor_sync(0xffffffffu, c.s, off);
    if (before(o, c)) c = o;
  }
  return c;
}

constexpr int kMaxNI = 16;  // N <= 512
constexpr int kSelWarps = 8;

__global__ void __launch_bounds__(kSelWarps * 32) route_select_kernel(
    const float *__restrict__ logits, const float *__restrict__ bias, int B, int N, int K,
    int n_group, int topk_group, int score_fn, int renorm, float route_scale,
    int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int32_t *__restrict__ counts) {
  __shared__ float sd[kSelWarps][kMaxNI * 32];
  __shared__ float sg[kSelWarps][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kSelWarps + warp;
  if (t >= B) return;
  const int NI = (N + 31) >> 5;

  float c[kMaxNI], s[kMaxNI];
  bool elig[kMaxNI];
#pragma unroll
  for (int i = 0; i < kMaxNI; ++i) {
    const int e = lane + 32 * i;
    elig[i] = (i < NI) && (e < N);
    c[i] = elig[i] ? logits[(size_t)t * N + e] : 0.0f;
  }
  if (score_fn == MOE_SCORE_SOFTMAX) {
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < kMaxNI; ++i)
      if (elig[i]) m = fmaxf(m, c[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
#pragma unroll
    for (int i = 0; i < kMaxNI; ++i)
      if (elig[i]) {
        s[i] = route_exp(__fsub_rn(c[i], m));
        sd[warp][lane + 32 * i] = s[i];
      }
    __syncwarp();
    float S = 0.0f;
    if (lane == 0)
      for (int e = 0; e < N; ++e) S = __fadd_rn(S, sd[warp][e]);  // expert order
    S = __shfl_sync(0xffffffffu, S, 0);
#pragma unroll
    for (int i = 0; i < kMaxNI; ++i)
      if (elig[i]) s[i] = __fdiv_rn(s[i], S);  // choice score stays z
  } else {
#pragma unroll
    for (int i = 0; i < kMaxNI; ++i)
      if (elig[i]) {
        const int e = lane + 32 * i;
        s[i] = route_sigmoid(c[i]);
        c[i] = bias ? __fadd_rn(s[i], __ldg(bias + e)) : s[i];
      }
  }

  if (n_group > 1) {
    const int gs = N / n_group;
    for (int j = 0; j < n_group; ++j) {
      Cand b1{0.0f, INT_MAX, 0.0f};
#pragma unroll
      for (int i = 0; i < kMaxNI; ++i) {
        const int e = lane + 32 * i;
        Cand x{c[i], e, 0.0f};
        if (elig[i] && e / gs == j && before(x, b1)) b1 = x;
      }
      b1 = warp_best(b1);
      Cand b2{0.0f, INT_MAX, 0.0f};
#pragma unroll
      for (int i = 0; i < kMaxNI; ++i) {
        const int e = lane + 32 * i;
        Cand x{c[i], e, 0.0f};
        if (elig[i] && e / gs == j && e != b1.i && before(x, b2)) b2 = x;
      }
      b2 = warp_best(b2);
      if (lane == 0) sg[warp][j] = __fadd_rn(b1.v, b2.v);
    }
    __syncwarp();
    uint32_t keep = 0;
    for (int r = 0; r < topk_group; ++r) {
      int best = -1;
      for (int j = 0; j < n_group; ++j) {
        if (keep >> j & 1) continue;
        if (best < 0 || sg[warp][j] > sg[warp][best]) best = j;  // ties keep the lower j
      }
      keep |= 1u << best;
    }
#pragma unroll
    for (int i = 0; i < kMaxNI; ++i) {
      const int e = lane + 32 * i;
      if (elig[i]) elig[i] = (keep >> (e / gs)) & 1;
    }
  }

  int my_idx = -1;
  float my_s = 0.0f;
  for (int r = 0; r < K; ++r) {
    Cand b{0.0f, INT_MAX, 0.0f};
#pragma unroll
    for (int i = 0; i < kMaxNI; ++i) {
      Cand x{c[i], lane + 32 * i, s[i]};
      if (elig[i] && before(x, b)) b = x;
    }
    b = warp_best(b);
#pragma unroll
    for (int i = 0; i < kMaxNI; ++i)
      if (lane + 32 * i == b.i) elig[i] = false;
    if (lane == r) {  // no candidate only if scores are NaN: report index -1
      my_idx = b.i == INT_MAX ? -1 : b.i;
      my_s = b.s;
    }
  }
  // weights: the normaliser sums the selected scores in rank order
  float sum = 0.0f;
  for (int r = 0; r < K; ++r) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, my_s, r));
  if (lane < K) {
    const float w = renorm ? __fmul_rn(__fdiv_rn(my_s, sum), route_scale)
                           : __fmul_rn(my_s, route_scale);
    topk_idx[(size_t)t * K + lane] = my_idx;
    topk_w[(size_t)t * K + lane] = w;
    if (counts && my_idx >= 0) atomicAdd(counts + my_idx, 1);
  }
}

// Top-2 of two ranked pairs: (a1, a2) <- best two of {a1, a2, b1, b2}.
__device__ __forceinline__ void merge_top2(Cand &a1, Cand &a2, const Cand &b1, const Cand &b2) {
  if (before(b1, a1)) {
    a2 = before(a1, b2) ? a1 : b2;
    a1 = b1;
  } else if (before(b1, a2)) {
    a2 = b1;
  }
}

// Selection with contiguous ownership: lane l holds experts [l*NPL, (l+1)*NPL).
// When a group's experts fill whole lanes (group size a multiple of NPL, a power
// of two of lanes per group), a group's top two are a scan of the lane's own
// values plus log2(lanes per group) butterfly merges, the kept groups follow from
// each group's rank, and each top-K round is a scan of NPL values plus two warp
// reductions (redux).  Same results as route_select_kernel.
template <int NPL>
__global__ void __launch_bounds__(kSelWarps * 32) route_select_lanes_kernel(
    const float *__restrict__ logits, const float *__restrict__ bias, int B, int N, int K,
    int n_group, int topk_group, int score_fn, int renorm, float route_scale,
    int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int32_t *__restrict__ counts) {
  __shared__ float sd[kSelWarps][kMaxNI * 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kSelWarps + warp;
  if (t >= B) return;
  const int base = lane * NPL;
  float c[NPL], s[NPL];
  bool elig[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    elig[i] = base + i < N;
    c[i] = elig[i] ? logits[(size_t)t * N + base + i] : 0.0f;
  }
  if (score_fn == MOE_SCORE_SOFTMAX) {
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (elig[i]) m = fmaxf(m, c[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (elig[i]) {
        s[i] = route_exp(__fsub_rn(c[i], m));
        sd[warp][base + i] = s[i];
      }
    __syncwarp();
    float S = 0.0f;
    if (lane == 0)
      for (int e = 0; e < N; ++e) S = __fadd_rn(S, sd[warp][e]);  // expert order
    S = __shfl_sync(0xffffffffu, S, 0);
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (elig[i]) s[i] = __fdiv_rn(s[i], S);
  } else {
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (elig[i]) {
        s[i] = route_sigmoid(c[i]);
        c[i] = bias ? __fadd_rn(s[i], __ldg(bias + base + i)) : s[i];
      }
  }
  if (n_group > 1) {
    const int gs = N / n_group, L = gs / NPL;
    Cand b1{0.0f, INT_MAX, 0.0f}, b2{0.0f, INT_MAX, 0.0f};
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const Cand x{c[i], base + i, 0.0f};
      if (!elig[i]) continue;
      if (before(x, b1)) {
        b2 = b1;
        b1 = x;
      } else if (before(x, b2)) {
        b2 = x;
      }
    }
    for (int off = 1; off < L; off <<= 1) {
      Cand o1, o2;
      o1.v = __shfl_xor_sync(0xffffffffu, b1.v, off);
      o1.i = __shfl_xor_sync(0xffffffffu, b1.i, off);
      o2.v = __shfl_xor_sync(0xffffffffu, b2.v, off);
      o2.i = __shfl_xor_sync(0xffffffffu, b2.i, off);
      o1.s = o2.s = 0.0f;
      merge_top2(b1, b2, o1, o2);
    }
    // Every lane of a group holds its score now.  A group is kept when fewer than
    // topk_group groups rank before it (higher score; equal scores: lower index).
    const float gsc = __fadd_rn(b1.v, b2.v);
    const int gme = lane / L;
    int ahead = 0;
    for (int j = 0; j < n_group; ++j) {
      const float o = __shfl_sync(0xffffffffu, gsc, j * L);
      ahead += (o > gsc || (o == gsc && j < gme)) ? 1 : 0;
    }
    const bool mine = base < N && gme < n_group && ahead < topk_group;
#pragma unroll
    for (int i = 0; i < NPL; ++i) elig[i] = elig[i] && mine;
  }
  // Top-K rounds as warp reductions on an order-preserving key of the score (+0 for
  // -0, so equal scores tie), ties to the smallest expert index; 0 = not a candidate.
  uint32_t key[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const uint32_t u = __float_as_uint(__fadd_rn(c[i], 0.0f));
    key[i] = elig[i] ? (u & 0x80000000u ? ~u : u | 0x80000000u) : 0u;
  }
  int my_idx = -1;
  float my_s = 0.0f;
  for (int r = 0; r < K; ++r) {
    uint32_t kb = 0;
    int ib = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (key[i] > kb) {  // strict: the lower index keeps a tie
        kb = key[i];
        ib = i;
      }
    const uint32_t km = __reduce_max_sync(0xffffffffu, kb);
    const uint32_t win =
        __reduce_min_sync(0xffffffffu, (km != 0 && kb == km) ? (uint32_t)(base + ib) : 0xffffffffu);
    float sb = 0.0f;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (i == ib) sb = s[i];
    const int owner = win == 0xffffffffu ? 0 : (int)win / NPL;
    const float sw = __shfl_sync(0xffffffffu, sb, owner);
    if (lane == owner && win != 0xffffffffu)
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (i == ib) key[i] = 0u;
    if (lane == r) {
      my_idx = win == 0xffffffffu ? -1 : (int)win;
      my_s = win == 0xffffffffu ? 0.0f : sw;
    }
  }
  float sum = 0.0f;
  for (int r = 0; r < K; ++r) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, my_s, r));
  if (lane < K) {
    const float w = renorm ? __fmul_rn(__fdiv_rn(my_s, sum), route_scale)
                           : __fmul_rn(my_s, route_scale);
    topk_idx[(size_t)t * K + lane] = my_idx;
    topk_w[(size_t)t * K + lane] = w;
    if (counts && my_idx >= 0) atomicAdd(counts + my_idx, 1);
  }
}

template <int TT, int TE, int S, int kRouteBK>
int launch_logits(const uint16_t *x, const float *W, float *lg, int B, int H, int N,
                  cudaStream_t st) {
  constexpr int BT = 8 * TT, BE = 16 * TE;
  constexpr size_t smem = (size_t)S * (BT * (kRouteBK + 8) * 2 + BE * (kRouteBK + 4) * 4);
  static bool attr[kMaxDevices] = {};
  const int dev = device_slot();
  if (dev < 0) return dev;
  if (!attr[dev] && smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_logits_kernel<TT, TE, S, kRouteBK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  attr[dev] = true;
  dim3 grid((N + BE - 1) / BE, (B + BT - 1) / BT);
  route_logits_kernel<TT, TE, S, kRouteBK><<<grid, kRouteThreads, smem, st>>>(x, W, lg, B, H, N);
  return check_launch();
}

template <int TT, int TE, int S, int BK>
int launch_logits_wide(const uint16_t *x, const float *W, float *lg, int B, int H, int N,
                       cudaStream_t st) {
  constexpr int BT = 8 * TT, BE = 16 * TE;
  constexpr size_t smem =
      (size_t)S * (BT * (BK + 8) * 2 + BE * (BK + 4) * 4) + (size_t)BT * (BK + 4) * 4;
  static bool attr[kMaxDevices] = {};
  const int dev = device_slot();
  if (dev < 0) return dev;
  if (!attr[dev] && smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_logits_wide_kernel<TT, TE, S, BK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  attr[dev] = true;
  dim3 grid((N + BE - 1) / BE, (B + BT - 1) / BT);
  route_logits_wide_kernel<TT, TE, S, BK><<<grid, kRouteThreads, smem, st>>>(x, W, lg, B, H, N);
  return check_launch();
}

template <int TT, int TE, int S, int BK, int NW>
int launch_logits_pair(const uint16_t *x, const float *W, float *lg, int B, int H,
                       cudaStream_t st) {
  constexpr int BT = NW * TT;
  constexpr size_t smem = (size_t)S * (BT * (BK + 8) * 2 + 32 * TE * (BK + 4) * 4) +
                          (size_t)NW * ((TT / 2) * (2 * BK + 4) + (TT % 2) * (BK + 4)) * 4;
  static bool attr[kMaxDevices] = {};
  const int dev = device_slot();
  if (dev < 0) return dev;
  if (!attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(route_logits_pair_kernel<TT, TE, S, BK, NW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  attr[dev] = true;
  route_logits_pair_kernel<TT, TE, S, BK, NW><<<(B + BT - 1) / BT, NW * 32, smem, st>>>(x, W, lg,
                                                                                   B, H);
  return check_launch();
}

int route_check(const moe_route_cfg *c) {
  if (!c) return MOE_ERR_INVALID;
  if (c->B < 0 || c->H <= 0 || c->N <= 0 || c->K <= 0) return MOE_ERR_INVALID;
  if (c->H % 32 || c->N > 32 * kMaxNI || c->K > 16 || c->K > c->N)
    return MOE_ERR_UNSUPPORTED;
  if (c->score_fn != MOE_SCORE_SOFTMAX && c->score_fn != MOE_SCORE_SIGMOID)
    return MOE_ERR_INVALID;
  if (c->n_group > 1) {
    if (c->n_group > 32 || c->N % c->n_group || c->N / c->n_group < 2 || c->topk_group < 1 ||
        c->topk_group > c->n_group || c->K > c->topk_group * (c->N / c->n_group))
      return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_workspace_size(const moe_route_cfg *cfg) {
  if (!cfg || cfg->B < 0 || cfg->N <= 0) return 0;
  return ((size_t)cfg->B * cfg->N * sizeof(float) + 255) / 256 * 256;
}

extern "C" int moe_route(const moe_route_cfg *cfg, const void *x, const float *W,
                         const float *bias, int32_t *topk_idx, float *topk_w,
                         int32_t *expert_counts, void *workspace, size_t workspace_bytes,
                         void *stream) {
  int rc = route_check(cfg);
  if (rc) return rc;
  if (cfg->B == 0) return MOE_OK;
  if (!x || !W || !topk_idx || !topk_w || !workspace) return MOE_ERR_INVALID;
  if (workspace_bytes < moe_route_workspace_size(cfg)) return MOE_ERR_INVALID;
  if ((uintptr_t)x % 16 || (uintptr_t)W % 16) return MOE_ERR_INVALID;
  cudaStream_t st = as_stream(stream);
  float *lg = static_cast<float *>(workspace);
  const int B = cfg->B, H = cfg->H, N = cfg->N;
  if (expert_counts) {
    cudaError_t e = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * N, st);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  // Pick the largest per-thread tile that still gives every SM several CTAs.
  const long sms = device_sm_count();
  auto ctas = [&](int tt, int te) {
    return (long)((N + 16 * te - 1) / (16 * te)) * ((B + 8 * tt - 1) / (8 * tt));
  };
  const uint16_t *xb = static_cast<const uint16_t *>(x);
  // 256 experts and 3-8 tokens per warp in one wave of CTAs of 7 or 8 warps: the
  // token-sliced kernel on packed fmas, with the tile whose 4-deep step costs least:
  // the larger of the SM's shared-memory wavefronts (per warp 32 for W, about TT for x)
  // and the busiest sub-partition's fma cycles (ceil(NW/4) warps x TT x 32).  Other wide
  // grids: fp32-widened x and the largest per-thread tile that still leaves every SM
  // one and a half CTAs; small grids: the bf16 kernel below.  The token-sliced kernel
  // stages 64-deep chunks in two buffers (a chunk's fmas outlast the next chunk's load),
  // which halves its barriers and widening passes against 32-deep ones.
  int best_tt = 0, best_nw = 0;
  long best_cost = 0;
  if (N == 256)
    for (int nw = 7; nw <= 8; ++nw)
      for (int tt = 3; tt <= 8; ++tt) {
        // the instantiated tiles: 7 warps for 3-6 tokens (shared-memory-bound steps),
        // 8 warps for 7-8 (fma-bound, so all four sub-partitions get two warps)
        if ((nw == 7) != (tt <= 6) || (long)nw * tt * sms < B) continue;
        const long cost = std::max((long)nw * (32 + tt), (long)((nw + 3) / 4) * tt * 32);
        if (!best_tt || cost < best_cost) {
          best_tt = tt;
          best_nw = nw;
          best_cost = cost;
        }
      }
  if (best_tt && H % 64 == 0 && (long)B * 4 >= 3L * 3 * 7 * sms) {  // ~3 tokens per warp
    switch (best_nw * 16 + best_tt) {
#define MOE_PAIR_CASE(TT, NW) \
  case NW * 16 + TT: rc = launch_logits_pair<TT, 8, 2, 64, NW>(xb, W, lg, B, H, st); break;
      MOE_PAIR_CASE(3, 7) MOE_PAIR_CASE(4, 7) MOE_PAIR_CASE(5, 7) MOE_PAIR_CASE(6, 7)
      MOE_PAIR_CASE(7, 8) MOE_PAIR_CASE(8, 8)
#undef MOE_PAIR_CASE
      default: rc = MOE_ERR_UNSUPPORTED;
    }
  }
  else if (2 * ctas(8, 8) >= 3 * sms)
    rc = launch_logits_wide<8, 8, 3, 32>(xb, W, lg, B, H, N, st);
  else if (2 * ctas(4, 8) >= 3 * sms)
    rc = launch_logits_wide<4, 8, 3, 32>(xb, W, lg, B, H, N, st);
  else if (B >= 128 && B <= 512 && H % 128 == 0)  // two tokens per thread: ILP for the FMA
    rc = launch_logits<2, 1, 8, 128>(xb, W, lg, B, H, N, st);  // chains, half the W reads
  else if (B >= 256 && H % 64 == 0)
    rc = launch_logits_wide<2, 2, 4, 64>(xb, W, lg, B, H, N, st);
  // (a <4,4> tile is never reached here: ctas(4, 4) <= 2 * ctas(4, 8) < 3 * sms)
  else if (ctas(2, 2) >= 4 * sms && H % 64 == 0)
    rc = launch_logits<2, 2, 4, 64>(xb, W, lg, B, H, N, st);
  else if (H % 128 == 0)  // small grid: only the in-flight chunks hide the load latency
    rc = launch_logits<1, 1, 8, 128>(xb, W, lg, B, H, N, st);
  else
    rc = launch_logits<1, 1, 8, 32>(xb, W, lg, B, H, N, st);
  if (rc) return rc;
  // lanes-own-experts selection when every group fills whole lanes, else generic
  int npl = 1;
  while (npl * 32 < N) npl *= 2;
  const int gs = cfg->n_group > 1 ? N / cfg->n_group : 0;
  const int L = gs ? gs / npl : 0;
  const bool lanes_ok = cfg->n_group <= 1 || (gs % npl == 0 && L >= 1 && (L & (L - 1)) == 0 &&
                                             L * cfg->n_group <= 32);
  const dim3 grid((B + kSelWarps - 1) / kSelWarps), block(kSelWarps * 32);
#define MOE_SEL_ARGS                                                                         \
  lg, bias, B, N, cfg->K, cfg->n_group, cfg->topk_group, cfg->score_fn, cfg->renorm,      \
      cfg->route_scale, topk_idx, topk_w, expert_counts
  if (!lanes_ok)
    route_select_kernel<<<grid, block, 0, st>>>(MOE_SEL_ARGS);
  else if (npl == 1)
    route_select_lanes_kernel<1><<<grid, block, 0, st>>>(MOE_SEL_ARGS);
  else if (npl == 2)
    route_select_lanes_kernel<2><<<grid, block, 0, st>>>(MOE_SEL_ARGS);
  else if (npl == 4)
    route_select_lanes_kernel<4><<<grid, block, 0, st>>>(MOE_SEL_ARGS);
  else if (npl == 8)
    route_select_lanes_kernel<8><<<grid, block, 0, st>>>(MOE_SEL_ARGS);
  else
    route_select_lanes_kernel<16><<<grid, block, 0, st>>>(MOE_SEL_ARGS);
#undef MOE_SEL_ARGS
  return check_launch();
}
