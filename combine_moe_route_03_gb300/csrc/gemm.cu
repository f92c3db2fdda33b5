// moe_grouped_gemm_fp8: grouped FP8 GEMMs of the expert FFN on tcgen05 tensor
// cores (sm_100-class), persistent over the M-tile list written by moe_dispatch.
//
// What it computes follows DeepGEMM's grouped GEMMs for the two dispatch layouts
// ("Large-scale EP: DeepEP, EPLB and two-batch overlap", §DeepEP: each mode where
// it belongs) with 1x128 activation and 128x128 weight scaling ("Single Batch
// Overlap (SBO)" PR, §3 "1d2d"), and the SBO producer side: per (expert, block_m)
// completion counters bumped with release atomics (same PR, §2).  How it computes
// is Blackwell-specific: the scales are powers of two (UE8M0), so the tensor core
// applies them itself (kind::mxf8f6f4 block scaling, one scale per 32 K values,
// each 1x128 / 128x128 scale repeated over its four 32-wide sub-blocks) and the
// fp32 accumulator stays in tensor memory for the whole K loop.
//
// Two kernels over the same tile list, both persistent with 11 warps per CTA:
//   grouped_gemm_kernel (one CTA per M tile, 128x256 MMAs; with binary32 scales the
//   k-blocks' partial products are promoted in the epilogue) and grouped_gemm_2sm_kernel
//   (CTA pairs on one TPC: an expert's tile pairs as M=256 cta_group::2 MMAs, its odd
//   last tile as an M=128 or M=256 pair MMA in the same launch; for DOWN optionally on
//   224-column tiles with two accumulators).  The DOWN epilogue can also reduce the
//   stored rows into token order (the fused combine).
//   warp 0  TMA producer: A tile 128x128 e4m3, B tile 256x128 e4m3 (two 128-row
//           boxes: gate and up halves for GATEUP, two output blocks for DOWN),
//           and the matching scale atoms, a ring of stages.
//   warp 1  TMEM owner and MMA issuer: scale atoms -> TMEM (tcgen05.cp), four
//           block-scaled MMAs per 128-deep k-block, commits free the stage.
//   warps 2-9 epilogue: TMEM -> registers (two warps per accumulator row group,
//           half the columns each; TMEM is released before any math), SwiGLU +
//           1x128 requantisation (GATEUP) or bf16 rounding (DOWN), global
//           stores, optional release signals.
//   warp 10 scheduler: decodes the CTA's work units from the tile list (a few
//           dependent global loads each) into a shared-memory ring, kUnitQ units
//           ahead, so no role waits on that latency at a tile boundary.
#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4;
constexpr int kGemmThreads = 352;  // producer, MMA, 8 epilogue warps, scheduler
constexpr int kUnitQ = 8;          // decoded units in flight
constexpr int kEpiThreads = 256;
constexpr uint32_t A_BYTES = BM * BK;   // 16 KB
constexpr uint32_t B_BYTES = BN * BK;   // 32 KB
constexpr uint32_t SFA_BYTES = 512;     // one SF atom
constexpr uint32_t SFB_BYTES = 1024;    // two SF atoms
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr uint32_t OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
// full, empty [STAGES]; accumulator full, empty; binary32-scale mode: partial full [2],
// partial empty [2]
constexpr uint32_t OFF_MISC = OFF_BAR + (2 * STAGES + 6) * 8;
constexpr uint32_t OFF_AMAX = OFF_MISC + 16;  // [2][128] partial row amax of the epilogue
constexpr uint32_t OFF_UNITQ = OFF_AMAX + 2 * 128 * 4;  // [kUnitQ] decoded units
constexpr uint32_t OFF_UBAR = OFF_UNITQ + kUnitQ * 32;  // [kUnitQ] full, [kUnitQ] empty
constexpr uint32_t STAGE_BYTES = 2048;                  // per epilogue warp, see store_bf16_rows
constexpr uint32_t OFF_STAGE = OFF_UBAR + 2 * kUnitQ * 8;
constexpr uint32_t SMEM_BYTES = OFF_STAGE + (kEpiThreads / 32) * STAGE_BYTES + 1024;  // + slack
static_assert(SMEM_BYTES <= 232448, "shared memory of the one-CTA kernel");
constexpr uint32_t TMEM_COLS = 512;
// Scale columns start here: kSfSets rotating sets of 16 columns (A atom at +0, B atoms
// at +4 and +8), one set per group of four k-blocks; a set is rewritten 4 * kSfSets
// k-blocks after its last use.
constexpr uint32_t TMEM_SF = 256;
constexpr int kSfSets = 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct GemmParams {
  int op, n, k, Kb, Kg, n_tiles, I;
  int64_t rows;
  const uint8_t *A_sf, *W_sf;
  const int32_t *phys2log, *tiles, *tiles2;
  int row_offset2, expert2, num_experts, max_tiles;
  uint8_t *out, *out_sf;
  int32_t *signal;
  int bm_signal;
  int32_t *status;
  int scale_fmt;  // 0: UE8M0 SF atoms; 1: binary32 scales, promoted per k-block
  // fused combine (DOWN; fc_B > 0 turns it on): see fused_combine_rows
  int fc_B, fc_K, fc_nch;
  const int32_t *fc_row_of, *fc_src_of;
  const float *fc_w;
  int32_t *fc_pending;
  int64_t fc_src_rows, fc_shared_row0;
  uint16_t *fc_out;
};
constexpr int kFusedKMax = 16;

struct Unit {
  int row0;    // first A / out row of this CTA's tile
  int nvalid;  // rows of that tile that hold data
  int we;      // weight expert
  int ni;      // output column tile
  int band;    // M tiles sharing this unit's weight tile
  bool ok;     // the unit runs (its tile-list entries address memory inside the operands)
  bool end;    // end of the CTA's unit stream
};

static_assert(sizeof(Unit) <= 32, "unit ring slot");
static_assert(TMEM_SF + 16 * kSfSets <= TMEM_COLS, "TMEM columns");

__device__ __forceinline__ bool tile_ok(const GemmParams &P, int row0, int nvalid) {
  return row0 >= 0 && (int64_t)row0 + 128 <= P.rows && row0 % 128 == 0 && nvalid > 0 &&
         nvalid <= 128;
}

// Work unit -> (M tile, N tile).  Units of one expert band (its consecutive M
// tiles) are ordered N-tile-major, M fastest, so CTAs running side by side share
// the same weight tile through L2.  Units of tiles2 come first.
__device__ __forceinline__ Unit get_unit(const GemmParams &P, int unit, int units2) {
  const int32_t *tl = P.tiles;
  int u = unit;
  const bool second = unit < units2;
  if (second)
    tl = P.tiles2;
  else
    u -= units2;
  const int g = u / P.n_tiles;  // some M tile of the right expert band
  const int f = tl[8 + 8 * g + 3], c = tl[8 + 8 * g + 4];
  const int cap = second ? tl[0] : P.max_tiles;
  Unit r;
  // the entry must describe its own band, inside the list
  if (f < 0 || c < 1 || g < f || g >= f + c || f + c > cap) {
    r.ok = r.end = false;
    r.row0 = r.nvalid = r.we = r.ni = r.band = 0;
    return r;
  }
  r.end = false;
  const int local = u - P.n_tiles * f;
  const int mi = f + local % c;
  const int32_t *t = tl + 8 + 8 * mi;
  r.ni = local / c;
  r.band = c;
  r.row0 = t[0] + (second ? P.row_offset2 : 0);
  r.nvalid = t[2];
  r.we = second ? P.expert2 : (P.phys2log ? P.phys2log[t[1]] : t[1]);
  // every role skips a tile entry that would address memory outside the operands
  r.ok = tile_ok(P, r.row0, r.nvalid) && r.we >= 0 && r.we < P.num_experts && r.ni < P.n_tiles;
  return r;
}


__device__ __forceinline__ void fail(int32_t *status, volatile int *abort) {
  *abort = 1;
  status_or(status, MOE_STATUS_TIMEOUT);
}

// 32 rows (one per lane, row `lane` at out_row0 + lane) x 64 bytes of this warp, stored
// so that each instruction writes 8 rows x 64 contiguous bytes: every lane puts its
// row's four 16-byte pieces into the warp's 2 KB staging slot (XOR-swizzled by row, so
// neither the writes nor the reads conflict on banks), then reads back piece lane%4 of
// row 8i + lane/4.  Rows at or past nrows are not stored.
__device__ __forceinline__ void store_rows_64B(uint8_t *stage, const uint4 *w, uint8_t *out_row0,
                                               size_t pitch, int nrows, int lane) {
#pragma unroll
  for (int p = 0; p < 4; ++p)
    *reinterpret_cast<uint4 *>(stage + 64 * lane + 16 * (p ^ ((lane >> 1) & 3))) = w[p];
  __syncwarp();
  const int p = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 8 * i + (lane >> 2);
    const uint4 x = *reinterpret_cast<const uint4 *>(stage + 64 * row + 16 * (p ^ ((row >> 1) & 3)));
    if (row < nrows) *reinterpret_cast<uint4 *>(out_row0 + (size_t)row * pitch + 16 * p) = x;
  }
  __syncwarp();
}

// store_rows_64B of 32 fp32 values per row (float, or their bits as uint32_t), rounded
// to bf16.
__device__ __forceinline__ float as_f32(uint32_t b) { return __uint_as_float(b); }
__device__ __forceinline__ float as_f32(float f) { return f; }
template <class T>
__device__ __forceinline__ void store_bf16_rows(uint8_t *stage, const T *v, uint8_t *out_row0,
                                                size_t pitch, int nrows, int lane) {
  uint4 w[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    w[p].x = f32_to_bf16_bits(as_f32(v[8 * p + 0])) | (f32_to_bf16_bits(as_f32(v[8 * p + 1])) << 16);
    w[p].y = f32_to_bf16_bits(as_f32(v[8 * p + 2])) | (f32_to_bf16_bits(as_f32(v[8 * p + 3])) << 16);
    w[p].z = f32_to_bf16_bits(as_f32(v[8 * p + 4])) | (f32_to_bf16_bits(as_f32(v[8 * p + 5])) << 16);
    w[p].w = f32_to_bf16_bits(as_f32(v[8 * p + 6])) | (f32_to_bf16_bits(as_f32(v[8 * p + 7])) << 16);
  }
  store_rows_64B(stage, w, out_row0, pitch, nrows, lane);
}

// 64 fp32 values of a row times 2^-e, as 64 e4m3 codes (round to nearest even,
// saturating) in four 16-byte pieces.
__device__ __forceinline__ void quantize_64(const uint32_t *v, float inv, uint4 *w) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t *wp = &w[c].x;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int b = 16 * c + 4 * j;
      wp[j] = e4m3x2(__fmul_rn(__uint_as_float(v[b]), inv),
                     __fmul_rn(__uint_as_float(v[b + 1]), inv)) |
              (e4m3x2(__fmul_rn(__uint_as_float(v[b + 2]), inv),
                      __fmul_rn(__uint_as_float(v[b + 3]), inv))
               << 16);
    }
  }
}

// Fused combine ("DeepEP 完全拆解", §为什么 combine 比 dispatch 慢: the reduce of the
// expert outputs, here done by the kernel that makes them).  This warp has stored rows
// [wrow0, wrow0 + nrows) of Y in the 128-column chunk `chunk`: all 128 columns (weight
// 2) or 64 of them (weight 1, the split of the M=128 pair epilogue).  Each lane counts
// its row off the pending count of (its row's token, chunk), after a gpu-scope fence of
// its own stores; a lane whose subtraction empties the count holds the token's last
// missing piece, so every row of that chunk is in memory, and the warp reduces those
// chunks, two at a time (a half-warp each, 8 columns per lane), reading the rows
// through L2: fmas into fp32 in the rank order k = 0..K-1, then the shared row, then
// bf16 -- the arithmetic of moe_combine, bit for bit.  Nothing waits.
__device__ __forceinline__ void fused_combine_rows(const GemmParams &P, int64_t wrow0, int nrows,
                                                   int chunk, int weight, int lane) {
  __threadfence();
  __syncwarp();
  int t = -1;
  bool last = false;
  if (lane < nrows) {
    const int64_t row = wrow0 + lane;
    if (P.fc_shared_row0 >= 0 && row >= P.fc_shared_row0)
      t = row - P.fc_shared_row0 < P.fc_B ? (int)(row - P.fc_shared_row0) : -1;
    else if (row < P.fc_src_rows)
      t = P.fc_src_of[row];
    if (t >= 0 && t < P.fc_B)
      last = atomicSub(P.fc_pending + (size_t)t * P.fc_nch + chunk, weight) == weight;
  }
  unsigned m = __ballot_sync(0xffffffffu, last);
  if (m == 0) return;
  __threadfence();  // the token's other rows were fenced before they were counted
  const int hl = lane & 15;
  const int col = 128 * chunk + 8 * hl;
  const uint16_t *Y = reinterpret_cast<const uint16_t *>(P.out);
  while (m) {
    const int la = __ffs(m) - 1;
    m &= m - 1;
    int lb = la;
    if (m) {
      lb = __ffs(m) - 1;
      m &= m - 1;
    }
    const int ta = __shfl_sync(0xffffffffu, t, la), tb = __shfl_sync(0xffffffffu, t, lb);
    const int tt = lane < 16 ? ta : (lb != la ? tb : -1);
    int my_r = -1;
    float my_w = 0.0f;
    if (tt >= 0 && hl < P.fc_K) {
      my_r = P.fc_row_of[(size_t)tt * P.fc_K + hl];
      my_w = P.fc_w[(size_t)tt * P.fc_K + hl];
    }
    int r[kFusedKMax];
    float w[kFusedKMax];
    uint4 y[kFusedKMax];
#pragma unroll
    for (int k = 0; k < kFusedKMax; ++k) {
      r[k] = __shfl_sync(0xffffffffu, my_r, k, 16);
      w[k] = __shfl_sync(0xffffffffu, my_w, k, 16);
      if (k >= P.fc_K || (uint64_t)r[k] >= (uint64_t)P.rows) r[k] = -1;
    }
    if (tt < 0) continue;
#pragma unroll
    for (int k = 0; k < kFusedKMax; ++k)
      y[k] = r[k] >= 0 ? __ldcg(reinterpret_cast<const uint4 *>(Y + (size_t)r[k] * P.n + col))
                       : make_uint4(0, 0, 0, 0);
    const bool use_s = P.fc_shared_row0 >= 0;
    const uint4 sv =
        use_s ? __ldcg(reinterpret_cast<const uint4 *>(Y + (size_t)(P.fc_shared_row0 + tt) * P.n + col))
              : make_uint4(0, 0, 0, 0);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < kFusedKMax; ++k) {
      if (r[k] < 0) continue;
      const uint32_t u[4] = {y[k].x, y[k].y, y[k].z, y[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(w[k], __uint_as_float(u[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w[k], __uint_as_float(u[i] & 0xffff0000u), acc[2 * i + 1]);
      }
    }
    if (use_s) {
      const uint32_t u[4] = {sv.x, sv.y, sv.z, sv.w};
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
    __stcs(reinterpret_cast<uint4 *>(P.fc_out + (size_t)tt * P.n + col), o);
  }
}

// Epilogue of one 128-row accumulator for this thread's half-row: TMEM ->
// registers, release() (the MMAs may overwrite the accumulator from then on), then
// SwiGLU + 1x128 requantisation (GATEUP) or bf16 rounding (DOWN), global stores and
// the optional per-block_m release signals.  All kEpiThreads epilogue threads call it.
template <class Release>
__device__ __forceinline__ void epilogue_tile(const GemmParams &P, int row0, int valid, int ni,
                                              uint32_t t_row, int half, int row_local, int warp,
                                              int lane, float *amax_x, uint8_t *stage,
                                              Release release) {
  const int64_t r = (int64_t)row0 + row_local;
  const bool store = row_local < valid && r < P.rows;
  if (P.op == MOE_GEMM_GATEUP_SWIGLU) {
    // gate columns [64*half, +64) and the matching up columns [128 + 64*half, +64)
    uint32_t g[64], u[64];
    MOE_TMEM_LD_32x32b_X32(t_row + 64 * half, g);
    MOE_TMEM_LD_32x32b_X32(t_row + 64 * half + 32, (g + 32));
    MOE_TMEM_LD_32x32b_X32(t_row + 128 + 64 * half, u);
    MOE_TMEM_LD_32x32b_X32(t_row + 128 + 64 * half + 32, (u + 32));
    tc_wait_ld();
    tc_fence_before();
    release();
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float gf = __uint_as_float(g[i]), uf = __uint_as_float(u[i]);
      const float v = __fdividef(gf, 1.0f + __expf(-gf)) * uf;  // silu(g) * u
      g[i] = __float_as_uint(v);
      amax = fmaxf(amax, fabsf(v));
    }
    // the 1x128 block of h spans both halves of the row
    amax_x[half * 128 + row_local] = amax;
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    amax = fmaxf(amax, amax_x[(half ^ 1) * 128 + row_local]);
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    const int e = ue8m0_exp(amax);
    uint4 w[4];
    quantize_64(g, pow2i(-e), w);
    if (store && half == 0) P.out_sf[sf_byte_off(r, ni, sf_groups(P.I))] = (uint8_t)(e + 127);
    const int64_t wrow0 = (int64_t)row0 + (row_local - lane);
    const int nrows = (int)min((int64_t)min(valid - (row_local - lane), 32), P.rows - wrow0);
    if (nrows > 0)
      store_rows_64B(stage, w, P.out + (size_t)wrow0 * P.I + (size_t)ni * 128 + 64 * half,
                     (size_t)P.I, nrows, lane);
  } else {
    // output columns [128*half, +128)
    uint32_t v[128];
#pragma unroll
    for (int c = 0; c < 4; ++c) MOE_TMEM_LD_32x32b_X32(t_row + 128 * half + 32 * c, (v + 32 * c));
    tc_wait_ld();
    tc_fence_before();
    release();
    // this warp's 32 rows (row_local - lane onwards), 32 columns at a time
    const int64_t wrow0 = (int64_t)row0 + (row_local - lane);
    const int nrows = (int)min((int64_t)min(valid - (row_local - lane), 32), P.rows - wrow0);
    if (nrows > 0) {
      uint8_t *dst = P.out + ((size_t)wrow0 * P.n + (size_t)ni * 256 + 128 * half) * 2;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        store_bf16_rows(stage, v + 32 * c, dst + 64 * c, (size_t)P.n * 2, nrows, lane);
    }
    if (P.fc_B > 0) fused_combine_rows(P, wrow0, nrows, 2 * ni + half, 2, lane);
    if (P.signal) {
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      if (warp == 2 && lane == 0) {
        for (int j = 0; j * P.bm_signal < BM; ++j)
          if (j * P.bm_signal < valid && row0 + j * P.bm_signal < P.rows)
            red_release_gpu_add(P.signal + (row0 + j * P.bm_signal) / P.bm_signal, 1);
      }
    }
  }
}

// Binary32-scale mode ("Single Batch Overlap (SBO)" PR, §3: the 1d2d scaling with float
// scales, promoted in software): the tensor core computes each 128-deep k-block's
// partial product unscaled (kind::f8f6f4) into one of two TMEM buffers (k-block g of
// the CTA into buffer g % 2), and the epilogue warps fold it into 128 fp32 accumulators
// per thread, acc += (s_a[row][kb] * s_w[block][kb]) * partial, one fma per value with
// the k-blocks in order; then SwiGLU with binary32-scale requantisation of h (s = amax /
// 448, code = e4m3(h / s)) or bf16 rounding, as epilogue_tile.  Returns false when a
// wait gave up.  All kEpiThreads epilogue threads call it.
__device__ __forceinline__ bool epilogue_f32(const GemmParams &P, const Unit &U, uint32_t tmem,
                                             int q, int half, int row_local, int warp, int lane,
                                             float *amax_x, uint8_t *stage, uint32_t bar_pfull,
                                             uint32_t bar_pempty, uint32_t &g,
                                             volatile int *abort) {
  const bool gateup = P.op == MOE_GEMM_GATEUP_SWIGLU;
  const int64_t r = (int64_t)U.row0 + row_local;  // < P.rows: tile_ok holds for the unit
  const bool store = row_local < U.nvalid;
  const float *sa = reinterpret_cast<const float *>(P.A_sf) + (size_t)r * P.Kb;
  const int nb0 = gateup ? U.ni : 2 * U.ni + half, nb1 = gateup ? P.I / 128 + U.ni : nb0;
  const float *sw = reinterpret_cast<const float *>(P.W_sf);
  const float *sw0 = sw + ((size_t)U.we * (P.n / 128) + nb0) * P.Kb;
  const float *sw1 = sw + ((size_t)U.we * (P.n / 128) + nb1) * P.Kb;
  // this thread's columns: gate [64h, +64) and up [128 + 64h, +64), or [128h, +128)
  const int c0 = gateup ? 64 * half : 128 * half, c1 = gateup ? 128 + 64 * half : c0 + 64;
  const uint32_t t_lane = tmem + ((uint32_t)(32 * q) << 16);
  float acc[128];
#pragma unroll
  for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
  // a warp whose 32 rows hold no data (most of a decode tile) only frees the buffers
  const bool busy = row_local - lane < U.nvalid;
  float sa_next = sa[0], w0_next = sw0[0], w1_next = sw1[0];
  for (int kb = 0; kb < P.Kb; ++kb) {
    const int b = g & 1;
    if (!mbar_wait(bar_pfull + 8 * b, (g >> 1) & 1, abort, kWaitLimitNs)) return false;
    tc_fence_after();
    if (busy) {
      const float s0 = __fmul_rn(sa_next, w0_next), s1 = __fmul_rn(sa_next, w1_next);
      if (kb + 1 < P.Kb) {  // the next k-block's scales load while this one folds
        sa_next = sa[kb + 1];
        w0_next = sw0[kb + 1];
        w1_next = sw1[kb + 1];
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // gate (or first 64) columns, then up (or next 64)
        uint32_t v[64];
        const uint32_t col = t_lane + 256 * b + (hh ? c1 : c0);
        MOE_TMEM_LD_32x32b_X32(col, v);
        MOE_TMEM_LD_32x32b_X32(col + 32, (v + 32));
        tc_wait_ld();
        const float sc = hh ? s1 : s0;
#pragma unroll
        for (int i = 0; i < 64; ++i)
          acc[64 * hh + i] = __fmaf_rn(sc, __uint_as_float(v[i]), acc[64 * hh + i]);
      }
    }
    tc_fence_before();
    mbar_arrive(bar_pempty + 8 * b);
    ++g;
  }
  const int64_t wrow0 = (int64_t)U.row0 + (row_local - lane);
  const int nrows = (int)min((int64_t)min(U.nvalid - (row_local - lane), 32), P.rows - wrow0);
  if (gateup) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float v = __fdividef(acc[i], 1.0f + __expf(-acc[i])) * acc[64 + i];  // silu(g) u
      acc[i] = v;
      amax = fmaxf(amax, fabsf(v));
    }
    amax_x[half * 128 + row_local] = amax;  // the 1x128 block of h spans both halves
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    amax = fmaxf(amax, amax_x[(half ^ 1) * 128 + row_local]);
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    float sh = __fdiv_rn(amax, 448.0f);
    if (sh == 0.0f) sh = 1.0f;
    uint4 w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t *wp = &w[c].x;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 16 * c + 4 * j;
        wp[j] = e4m3x2(__fdiv_rn(acc[i], sh), __fdiv_rn(acc[i + 1], sh)) |
                (e4m3x2(__fdiv_rn(acc[i + 2], sh), __fdiv_rn(acc[i + 3], sh)) << 16);
      }
    }
    if (store && half == 0)
      reinterpret_cast<float *>(P.out_sf)[(size_t)r * (P.I / 128) + U.ni] = sh;
    if (nrows > 0)
      store_rows_64B(stage, w, P.out + (size_t)wrow0 * P.I + (size_t)U.ni * 128 + 64 * half,
                     (size_t)P.I, nrows, lane);
  } else {
    if (nrows > 0) {
      uint8_t *dst = P.out + ((size_t)wrow0 * P.n + (size_t)U.ni * 256 + 128 * half) * 2;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        store_bf16_rows(stage, acc + 32 * c, dst + 64 * c, (size_t)P.n * 2, nrows, lane);
    }
    if (P.fc_B > 0) fused_combine_rows(P, wrow0, nrows, 2 * U.ni + half, 2, lane);
    if (P.signal) {
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      if (warp == 2 && lane == 0) {
        for (int j = 0; j * P.bm_signal < BM; ++j)
          if (j * P.bm_signal < U.nvalid && U.row0 + j * P.bm_signal < P.rows)
            red_release_gpu_add(P.signal + (U.row0 + j * P.bm_signal) / P.bm_signal, 1);
      }
    }
  }
  return true;
}

// The DOWN GEMM on 224-column tiles (H = 7168 = 32 x 224): two 224-column accumulators
// and the scale sets fill TMEM exactly, so the MMAs of a unit run while the epilogue
// drains the previous unit's accumulator.
constexpr int BN224 = 224;
constexpr uint32_t TMEM_SF224 = 2 * BN224;
static_assert(TMEM_SF224 + 16 * kSfSets <= TMEM_COLS, "TMEM columns (224-column tiles)");

// Epilogue of a 224-column DOWN accumulator: this thread's lane row, columns [0,128)
// (half 0) or [128,224) (half 1); TMEM -> registers, release(), bf16 rounding and
// stores as in epilogue_tile.
template <class Release>
__device__ __forceinline__ void epilogue_down224(const GemmParams &P, int row0, int valid, int ni,
                                                 uint32_t t_row, int half, int row_local,
                                                 int lane, uint8_t *stage, Release release) {
  uint32_t v[128];
  const int pieces = half ? (BN224 - 128) / 32 : 4;  // 32-column pieces of this thread
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (c < pieces) MOE_TMEM_LD_32x32b_X32(t_row + 128 * half + 32 * c, (v + 32 * c));
  tc_wait_ld();
  tc_fence_before();
  release();
  const int64_t wrow0 = (int64_t)row0 + (row_local - lane);
  const int nrows = (int)min((int64_t)min(valid - (row_local - lane), 32), P.rows - wrow0);
  if (nrows > 0) {
    uint8_t *dst = P.out + ((size_t)wrow0 * P.n + (size_t)ni * BN224 + 128 * half) * 2;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (c < pieces)
        store_bf16_rows(stage, v + 32 * c, dst + 64 * c, (size_t)P.n * 2, nrows, lane);
  }
}

// tmA loads full 128-row A tiles; tmA32 loads 32-row slices, used for tiles with
// fewer valid rows so rows that hold no data are never fetched (the MMA then reads
// stale shared memory for them, which only feeds accumulator rows never stored).
// kF32: binary32-scale mode (see epilogue_f32); otherwise UE8M0 block scaling in the
// tensor core.  kW224: the DOWN GEMM on 224-column tiles with two accumulators (TMEM
// columns [0,224) and [224,448), scale sets from 448; weight scales as tile images).
template <bool kF32, bool kW224 = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmA32,
                        const __grid_constant__ CUtensorMap tmW, const GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bar_full = s_base + OFF_BAR;                 // [STAGES]
  const uint32_t bar_empty = bar_full + 8 * STAGES;           // [STAGES]
  const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  const uint32_t bar_pfull = bar_acc_empty + 8;               // [2], binary32-scale mode
  const uint32_t bar_pempty = bar_pfull + 16;                 // [2]
  const uint32_t bar_unit_full = s_base + OFF_UBAR;          // [kUnitQ]
  const uint32_t bar_unit_empty = bar_unit_full + 8 * kUnitQ; // [kUnitQ]
  Unit *unit_q = reinterpret_cast<Unit *>(smem + OFF_UNITQ);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, kEpiThreads);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_pfull + 8 * b, 1);
      mbar_init(bar_pempty + 8 * b, kEpiThreads);
    }
    for (int q = 0; q < kUnitQ; ++q) {
      mbar_init(bar_unit_full + 8 * q, 1);
      mbar_init(bar_unit_empty + 8 * q, 2 + kEpiThreads / 32);  // producer, MMA, epilogue warps
    }
    *abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmA32);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int units2 = P.tiles2 ? P.tiles2[0] * P.n_tiles : 0;
  const int total = P.tiles[0] * P.n_tiles + units2;
  // The seq-th unit of this CTA from the scheduler's ring (false: timed out / aborted).
  // The caller releases the slot with release_unit once it has copied the unit.
  auto take_unit = [&](int seq, Unit &U) {
    const int slot = seq % kUnitQ;
    if (!mbar_wait(bar_unit_full + 8 * slot, (uint32_t)(seq / kUnitQ) & 1u, abort, kWaitLimitNs))
      return false;
    U = unit_q[slot];
    return true;
  };
  auto release_unit = [&](int seq) { mbar_arrive(bar_unit_empty + 8 * (seq % kUnitQ)); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // A tiles are re-read by every N tile of their expert: keep them in L2.  A
      // weight tile read by one M tile only is streamed (evict first); one shared by
      // several M tiles (read by neighbouring CTAs at about the same time) is kept.
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_normal();
      const uint64_t pol_a = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        Unit U;
        if (!take_unit(seq, U)) {
          fail(P.status, abort);
          ok = false;
          break;
        }
        release_unit(seq);
        if (U.end) break;
        if (!U.ok) {
          status_or(P.status, MOE_STATUS_BAD_INDEX);
          continue;
        }
        const int row0 = U.row0, we = U.we, ni = U.ni;
        const uint64_t pol_w = U.band > 1 ? pol_keep : pol_stream;
        const int a_slices = U.nvalid == BM ? 0 : (U.nvalid + 31) / 32;  // 0: one full box
        const uint32_t a_bytes = a_slices ? a_slices * (A_BYTES / 4) : A_BYTES;
        // a group's scale atoms travel with its first k-block
        const uint32_t tx = a_bytes + (kW224 ? (uint32_t)BN224 * BK : B_BYTES),
                       tx_sf = SFA_BYTES + SFB_BYTES;
        int wrow0, wrow1, nb0, nb1;
        if (kW224) {  // one 224-row box; the tile's two scale images
          wrow0 = wrow1 = we * P.n + ni * BN224;
          nb0 = nb1 = 0;
        } else if (P.op == MOE_GEMM_GATEUP_SWIGLU) {
          wrow0 = we * P.n + ni * 128;
          wrow1 = we * P.n + P.I + ni * 128;
          nb0 = ni;
          nb1 = P.I / 128 + ni;
        } else {
          wrow0 = we * P.n + ni * 256;
          wrow1 = wrow0 + 128;
          nb0 = 2 * ni;
          nb1 = 2 * ni + 1;
        }
        const uint8_t *sfa = P.A_sf + (size_t)(row0 >> 7) * P.Kg * 512;
        // group g's atoms at sfb0 / sfb1 + g * sfb_step (images interleave per group)
        const uint8_t *sfb0 =
            kW224 ? P.W_sf + ((size_t)we * P.n_tiles + ni) * P.Kg * 1024
                  : P.W_sf + ((size_t)we * (P.n / 128) + nb0) * P.Kg * 512;
        const uint8_t *sfb1 =
            kW224 ? sfb0 + 512 : P.W_sf + ((size_t)we * (P.n / 128) + nb1) * P.Kg * 512;
        const size_t sfb_step = kW224 ? 1024 : 512;
        for (int kb = 0; kb < P.Kb; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort, kWaitLimitNs)) {
            fail(P.status, abort);
            ok = false;
            break;
          }
          const uint32_t full = bar_full + 8 * stage;
          const bool sf = !kF32 && (kb & 3) == 0;  // binary32 scales are not staged
          mbar_arrive_expect_tx(full, sf ? tx + tx_sf : tx);
          const uint32_t sa = s_base + OFF_A + stage * A_BYTES;
          const uint32_t sb = s_base + OFF_B + stage * B_BYTES;
          const uint32_t ssfa = s_base + OFF_SFA + stage * SFA_BYTES;
          const uint32_t ssfb = s_base + OFF_SFB + stage * SFB_BYTES;
          if (a_slices == 0)
            tma_load_2d(sa, &tmA, full, kb * BK, row0, pol_a);
          else
            for (int j = 0; j < a_slices; ++j)
              tma_load_2d(sa + j * (A_BYTES / 4), &tmA32, full, kb * BK, row0 + 32 * j, pol_a);
          tma_load_2d(sb, &tmW, full, kb * BK, wrow0, pol_w);
          if (!kW224) tma_load_2d(sb + B_BYTES / 2, &tmW, full, kb * BK, wrow1, pol_w);
          if (sf) {
            bulk_load(ssfa, sfa + (size_t)(kb >> 2) * 512, 512, full);
            bulk_load(ssfb, sfb0 + (size_t)(kb >> 2) * sfb_step, 512, full);
            bulk_load(ssfb + 512, sfb1 + (size_t)(kb >> 2) * sfb_step, 512, full);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA can exit.
        for (int i = 0; i < STAGES && i < issued; ++i) {
          if (--stage < 0) {
            stage = STAGES - 1;
            phase ^= 1;
          }
          volatile int never = 0;
          mbar_wait(bar_full + 8 * stage, phase, &never, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // kind::mxf8f6f4 instruction descriptor: E4M3 x E4M3, K-major A and B,
      // N = 256, UE8M0 scales, M = 128; bits 4-5 / 29-30 select the B / A scale byte.
      const uint32_t idesc_base = ((uint32_t)((kW224 ? BN224 : BN) >> 3) << 17) | (1u << 23) |
                                  ((uint32_t)(BM >> 4) << 24);
      const uint32_t tmem_sf = kW224 ? TMEM_SF224 : TMEM_SF;
      int stage = 0, nacc = 0;  // units accumulated so far (buffer nacc % 2 if kW224)
      uint32_t phase = 0, pg = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        Unit U;
        if (!take_unit(seq, U)) {
          fail(P.status, abort);
          break;
        }
        release_unit(seq);
        if (U.end) break;
        if (!U.ok) continue;
        if constexpr (kF32) {
          // each k-block's unscaled partial into TMEM buffer g % 2, once the epilogue has
          // folded the k-block two before out of it
          const uint32_t idesc_f8 = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
          for (int kb = 0; kb < P.Kb; ++kb) {
            const int b = pg & 1;
            if (!mbar_wait(bar_full + 8 * stage, phase, abort, kWaitLimitNs) ||
                !mbar_wait(bar_pempty + 8 * b, ((pg >> 1) & 1) ^ 1, abort, kWaitLimitNs)) {
              fail(P.status, abort);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = s_base + OFF_A + stage * A_BYTES;
            const uint32_t sb = s_base + OFF_B + stage * B_BYTES;
#pragma unroll
            for (int j = 0; j < BK / 32; ++j)
              tc_mma_f8(tmem + 256 * b, smem_desc(sa + 32 * j, 16, 1024, 2),
                        smem_desc(sb + 32 * j, 16, 1024, 2), idesc_f8, j != 0);
            tc_commit(bar_empty + 8 * stage);
            tc_commit(bar_pfull + 8 * b);
            ++pg;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          continue;
        }
        // buffer 1 of kW224 uses the binary32 mode's (here idle) partial barriers
        const int buf = kW224 ? nacc & 1 : 0;
        const uint32_t acc_phase = (uint32_t)(kW224 ? nacc >> 1 : nacc) & 1u;
        const uint32_t acc = tmem + (kW224 ? (uint32_t)(BN224 * buf) : 0u);
        const uint32_t b_full = buf ? bar_pfull : bar_acc_full;
        const uint32_t b_empty = buf ? bar_pempty : bar_acc_empty;
        if (!mbar_wait(b_empty, acc_phase ^ 1, abort, kWaitLimitNs)) {
          fail(P.status, abort);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < P.Kb; ++kb) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort, kWaitLimitNs)) {
            fail(P.status, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = s_base + OFF_A + stage * A_BYTES;
          const uint32_t sb = s_base + OFF_B + stage * B_BYTES;
          const uint32_t t_sfa = tmem + tmem_sf + 16 * ((kb >> 2) % kSfSets);
          const uint32_t t_sfb = t_sfa + 4;
          if ((kb & 3) == 0) {  // the group's scale atoms, once per four k-blocks
            const uint32_t ssfa = s_base + OFF_SFA + stage * SFA_BYTES;
            const uint32_t ssfb = s_base + OFF_SFB + stage * SFB_BYTES;
            tc_cp_32x128b_x4(t_sfa, smem_desc(ssfa, 16, 128, 0));
            tc_cp_32x128b_x4(t_sfb, smem_desc(ssfb, 16, 128, 0));
            tc_cp_32x128b_x4(t_sfb + 4, smem_desc(ssfb + 512, 16, 128, 0));
          }
          // k-block kb's scales are byte kb % 4 of each atom word, for all four
          // 32-wide MMAs of the block
          const uint32_t idesc = idesc_base | ((uint32_t)(kb & 3) << 29) | ((uint32_t)(kb & 3) << 4);
#pragma unroll
          for (int j = 0; j < BK / 32; ++j) {
            const uint64_t ad = smem_desc(sa + 32 * j, 16, 1024, 2);
            const uint64_t bd = smem_desc(sb + 32 * j, 16, 1024, 2);
            tc_mma_mxf8(acc, ad, bd, idesc, t_sfa, t_sfb, (kb | j) != 0);
          }
          tc_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(b_full);
        ++nacc;
      }
    }
  } else if (warp < 2 + kEpiThreads / 32) {
    // ------------------------------------------------------------ epilogue
    // Eight warps: a warp may read TMEM lanes 32*(warp%4)..+31 (its rows); the two
    // warps of a lane quarter split the columns.  Each thread moves its half-row of
    // the accumulator into registers and releases TMEM at once, so the next tile's
    // MMAs run while these warps finish SwiGLU / quantisation / stores.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_local = 32 * q + lane;
    const uint32_t t_row = tmem + ((uint32_t)(32 * q) << 16);
    float *amax_x = reinterpret_cast<float *>(smem + OFF_AMAX);  // [half][row]
    uint8_t *stage = smem + OFF_STAGE + (warp - 2) * STAGE_BYTES;
    uint32_t pg = 0;
    int nacc = 0;  // as the MMA issuer: buffer nacc % 2 if kW224
    for (int seq = 0;; ++seq) {
      Unit U;
      if (!take_unit(seq, U)) {
        fail(P.status, abort);
        break;
      }
      __syncwarp();
      if (lane == 0) release_unit(seq);
      if (U.end) break;
      if (!U.ok) continue;
      if constexpr (kF32) {
        if (!epilogue_f32(P, U, tmem, q, half, row_local, warp, lane, amax_x, stage, bar_pfull,
                          bar_pempty, pg, abort)) {
          fail(P.status, abort);
          break;
        }
        continue;
      }
      const int buf = kW224 ? nacc & 1 : 0;
      const uint32_t acc_phase = (uint32_t)(kW224 ? nacc >> 1 : nacc) & 1u;
      ++nacc;
      const uint32_t b_full = buf ? bar_pfull : bar_acc_full;
      const uint32_t b_empty = buf ? bar_pempty : bar_acc_empty;
      if (!mbar_wait(b_full, acc_phase, abort, kWaitLimitNs)) {
        fail(P.status, abort);
        break;
      }
      tc_fence_after();
      if constexpr (kW224)
        epilogue_down224(P, U.row0, U.nvalid, U.ni, t_row + (uint32_t)(BN224 * buf), half,
                         row_local, lane, stage, [&] { mbar_arrive(b_empty); });
      else
        epilogue_tile(P, U.row0, U.nvalid, U.ni, t_row, half, row_local, warp, lane, amax_x,
                      stage, [&] { mbar_arrive(b_empty); });
    }
  } else if (lane == 0) {
    // ------------------------------------------------------------ scheduler
    int seq = 0;
    auto push = [&](const Unit &U) {
      const int slot = seq % kUnitQ;
      if (!mbar_wait(bar_unit_empty + 8 * slot, ((uint32_t)(seq / kUnitQ) & 1u) ^ 1u, abort,
                     kWaitLimitNs)) {
        fail(P.status, abort);
        return false;
      }
      unit_q[slot] = U;
      mbar_arrive(bar_unit_full + 8 * slot);  // release: the unit is visible to the waiters
      ++seq;
      return true;
    };
    bool ok = true;
    // Equal rounds: the units are spread over just enough CTAs that every CTA runs the
    // same number of them (the rest run none), so the last round keeps as many CTAs
    // streaming weights as the others (an HBM-bound launch otherwise ends on a partial
    // round that cannot fill the memory system).
    const int rounds = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int ctas = rounds > 0 ? (total + rounds - 1) / rounds : 0;
    for (int unit = blockIdx.x; ok && unit < total && (int)blockIdx.x < ctas; unit += ctas)
      ok = push(get_unit(P, unit, units2));
    if (ok) {
      Unit end = {};
      end.end = true;
      push(end);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------ 2-SM variant
// The two CTAs of a cluster (the two SMs of a TPC) share one weight tile: each holds
// half of it (128 of its 256 rows: the gate or up half for GATEUP, one output block
// for DOWN) and both weight scale atoms, and the even CTA issues tcgen05 cta_group::2
// MMAs that read both halves.  Work units (an item of the tile list's item table at
// one N tile):
//   pair   two M tiles of one expert, one per CTA: M=256 x N=256 block-scaled MMAs;
//          each CTA's TMEM holds its 128 rows' accumulator (lanes = rows, columns = N).
//   single an expert's odd last tile, in the even CTA; with at most 64 valid rows it
//          runs M=128 MMAs (64 rows per CTA; the odd CTA's half is idle), whose
//          accumulator sits in TMEM lanes 0-63 for columns [0,128) and lanes 64-127
//          for columns [128,256) of the same 64 rows; with more rows, M=256 MMAs with
//          the odd CTA's rows idle.
// Scales in TMEM: each 32-lane quarter of the tensor core reads the scales of the
// accumulator lanes it computes from its own TMEM lanes: a row's scale at its lane,
// word (row % 64) / 32 of the A scale columns (M=128; row / 32 at M=256), and output
// column c's weight scale at lane 32 * quarter + c % 32, word (c % 128) / 32 of the
// B scale columns.  So an atom copied with .32x128b.warpx4 (the same 32 lanes in all four
// quarters) serves M=256 (two atoms for the two 128-column halves); at M=128 the quarters holding columns [128,256) need the second
// weight atom in the same columns as the first: those units stage a 128-row image
// (atom 0 in quarters 0-1, atom 1 in quarters 2-3) and copy it unreplicated.  The odd
// CTA could only hold a tile's rows 64-127 at M=128 with their scales moved to words
// 0-1, which no copy can do, hence the M=256 form for longer singles.
// Singles run in the same launch as the pairs and next to them (same item group, N
// tiles interleaved), so they read the weight tiles the pairs just brought into L2.
// The pair instruction issues about 1.5x the FLOPs per SM-cycle of the one-CTA M=128
// form, and each SM moves 16 KB of weights per 128-deep k-block instead of 32 KB.
// Both CTAs' TMA loads complete on the even CTA's stage barrier, and the MMA commits
// free the stage in both.  A stage holds KB2 k-blocks (256 K): the issuing thread
// waits, fences and commits once per eight MMAs, which keeps the pair's tensor pipe fed.
constexpr int KB2 = 2, S2 = 3;              // k-blocks per stage, stages
constexpr uint32_t BH_BYTES = B_BYTES / 2;  // a CTA's half of a k-block's weight tile
constexpr uint32_t O2_A = 0;
constexpr uint32_t O2_B = O2_A + S2 * KB2 * A_BYTES;
constexpr uint32_t O2_SFA = O2_B + S2 * KB2 * BH_BYTES;
constexpr uint32_t O2_SFB = O2_SFA + S2 * SFA_BYTES;  // a group's atoms, in its first stage
constexpr uint32_t O2_BAR = O2_SFB + S2 * SFB_BYTES;  // full, empty [S2]; acc full, empty [2]
constexpr uint32_t O2_MISC = O2_BAR + (2 * S2 + 4) * 8;
constexpr uint32_t O2_AMAX = O2_MISC + 16;
constexpr uint32_t O2_UNITQ = O2_AMAX + 2 * 128 * 4;
constexpr uint32_t O2_UBAR = O2_UNITQ + kUnitQ * 32;
constexpr uint32_t O2_XBUF = O2_UBAR + 2 * kUnitQ * 8;  // [2 halves][32 columns][64 rows] fp32
constexpr uint32_t XBUF_BYTES = 2 * 32 * 64 * 4;
static_assert(XBUF_BYTES >= (kEpiThreads / 32) * STAGE_BYTES, "DOWN staging slots in xbuf");
constexpr uint32_t SMEM2_BYTES = O2_XBUF + XBUF_BYTES + 1024;
constexpr uint32_t TMEM_SF2 = 256;  // kSfSets rotating scale sets of 16 columns, as above
static_assert(TMEM_SF2 + 16 * kSfSets <= TMEM_COLS, "TMEM columns");
static_assert(KB2 == 1 || KB2 == 2 || KB2 == 4, "a scale group (4 k-blocks) starts a stage");
static_assert(SMEM2_BYTES <= 232448, "shared memory of the 2-SM kernel");

struct Unit2 {
  int row0, nvalid;  // this CTA's tile, when active
  int we, ni, band;
  uint32_t tx;       // bytes one stage brings into both CTAs (expected on the even CTA)
  uint32_t tx_sf;    // + the scale atoms, in a stage that starts a group of 4 k-blocks
  bool ok, active, end, m128;
};
static_assert(sizeof(Unit2) <= 32, "unit ring slot");

// Work unit -> the item's 2-SM unit.  Both CTAs decode alike: `rank` only selects which
// tile fills row0 / nvalid / active.  U.ok is false when the entries do not describe
// tiles inside the operands (every role then skips the unit).  kW224: 224-column DOWN
// tiles (112 weight rows per CTA), every single tile at M=256.
template <bool kW224>
__device__ __forceinline__ Unit2 get_2sm_unit(const GemmParams &P, int unit, int units2,
                                              int rank) {
  const int32_t *tl = P.tiles;
  int u = unit;
  const bool second = unit < units2;
  if (second)
    tl = P.tiles2;
  else
    u -= units2;
  Unit2 U = {};
  const int cap = second ? tl[0] : P.max_tiles;
  const int nitems = tl[4];
  const int32_t *items = tl + 8 + 8 * (size_t)cap;
  const int g = u / P.n_tiles;  // some item of the right group
  if (g >= nitems) return U;
  const int gf = items[8 * g + 2], gc = items[8 * g + 3];
  // the item must lie inside the group it names (so local >= 0 below)
  if (gf < 0 || gc < 1 || g < gf || g >= gf + gc || gf + gc > nitems) return U;
  const int local = u - P.n_tiles * gf;
  U.ni = local / gc;
  if (U.ni >= P.n_tiles) return U;
  const int32_t *it = items + 8 * (gf + local % gc);
  const bool pair = it[4] != 0;
  const int tile[2] = {it[0], pair ? it[1] : -1};  // pair: one expert's two tiles
  if (tile[0] < 0 || tile[0] >= cap || (pair && (tile[1] < 0 || tile[1] >= cap))) return U;
  const int32_t *e = tl + 8 + 8 * tile[0];
  U.we = second ? P.expert2 : (P.phys2log ? P.phys2log[e[1]] : e[1]);
  U.band = e[4];
  if (U.we < 0 || U.we >= P.num_experts) return U;
  U.m128 = !kW224 && !pair && e[2] > 0 && e[2] <= 64;
  // both halves of the weight tile
  uint32_t tx = 2 * KB2 * (kW224 ? (uint32_t)(BN224 / 2) * BK : BH_BYTES), tx_sf = 0;
  for (int c = 0; c < 2; ++c) {
    const int mi = tile[c];
    if (mi < 0) continue;
    const int32_t *t = tl + 8 + 8 * mi;
    if (pair && t[1] != e[1]) return U;  // a pair shares one expert's weights
    const int row0 = t[0] + (second ? P.row_offset2 : 0), nv = t[2];
    if (!tile_ok(P, row0, nv)) return U;
    const int slices = nv == BM ? 0 : (nv + 31) / 32;
    tx += KB2 * (slices ? slices * (A_BYTES / 4) : A_BYTES);
    // an M=128 unit's weight scales come as a 128-row image (4 atoms per group)
    tx_sf += SFA_BYTES + (U.m128 ? 2 * SFB_BYTES : SFB_BYTES);
    if (c == rank) {
      U.row0 = row0;
      U.nvalid = nv;
      U.active = true;
    }
  }
  U.tx = tx;
  U.tx_sf = tx_sf;
  U.ok = true;
  return U;
}

// Epilogue of an M=128 pair accumulator in the even CTA (the tile's rows 0-63): TMEM
// lanes 0-63 hold output columns [0,128) of rows 0-63, lanes 64-127 columns
// [128,256) of the same rows; each thread takes 64 of its lane's 128 columns.  For
// GATEUP the lower lanes hold gate, the upper lanes up: the up values pass through
// shared memory (xbuf, 32 columns at a time) to the gate thread of the same row, which
// forms h = silu(g) * u, requantises it and stores it.  All kEpiThreads epilogue
// threads call it.
template <class Release>
__device__ __forceinline__ void epilogue_m128(const GemmParams &P, int row0, int valid, int ni,
                                              uint32_t t_row, int q, int half, int warp,
                                              int lane, float *amax_x, float *xbuf,
                                              uint8_t *stage, Release release) {
  const int m = 32 * (q & 1) + lane;  // row of the tile
  const bool upper = q >= 2;          // columns [128, 256)
  const int64_t r = (int64_t)row0 + m;
  const bool store = m < valid && r < P.rows;
  uint32_t v[64];
  MOE_TMEM_LD_32x32b_X32(t_row + 64 * half, v);
  MOE_TMEM_LD_32x32b_X32(t_row + 64 * half + 32, (v + 32));
  tc_wait_ld();
  tc_fence_before();
  release();
  if (P.op == MOE_GEMM_GATEUP_SWIGLU) {
    // xbuf also holds the warps' staging slots: every warp is done with the previous
    // unit's stores before any up value lands in it
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    float amax = 0.0f;
#pragma unroll
    for (int rd = 0; rd < 2; ++rd) {
      if (upper) {
#pragma unroll
        for (int c = 0; c < 32; ++c) xbuf[(half * 32 + c) * 64 + m] = __uint_as_float(v[32 * rd + c]);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      if (!upper) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float gf = __uint_as_float(v[32 * rd + c]);
          const float uf = xbuf[(half * 32 + c) * 64 + m];
          const float h = __fdividef(gf, 1.0f + __expf(-gf)) * uf;  // silu(g) * u
          v[32 * rd + c] = __float_as_uint(h);
          amax = fmaxf(amax, fabsf(h));
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    }
    // the 1x128 block of h spans both column halves
    if (!upper) amax_x[half * 128 + m] = amax;
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    if (!upper) amax = fmaxf(amax, amax_x[(half ^ 1) * 128 + m]);
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    if (!upper) {  // warp-uniform: the gate lanes hold h
      const int e = ue8m0_exp(amax);
      uint4 w[4];
      quantize_64(v, pow2i(-e), w);
      if (store && half == 0) P.out_sf[sf_byte_off(r, ni, sf_groups(P.I))] = (uint8_t)(e + 127);
      const int64_t wrow0 = (int64_t)row0 + (m - lane);
      const int nrows = (int)min((int64_t)min(valid - (m - lane), 32), P.rows - wrow0);
      if (nrows > 0)
        store_rows_64B(stage, w, P.out + (size_t)wrow0 * P.I + (size_t)ni * 128 + 64 * half,
                       (size_t)P.I, nrows, lane);
    }
  } else {
    const int64_t wrow0 = (int64_t)row0 + (m - lane);
    const int nrows = (int)min((int64_t)min(valid - (m - lane), 32), P.rows - wrow0);
    if (nrows > 0) {
      uint8_t *dst =
          P.out + ((size_t)wrow0 * P.n + (size_t)ni * 256 + (upper ? 128 : 0) + 64 * half) * 2;
#pragma unroll
      for (int c = 0; c < 2; ++c)
        store_bf16_rows(stage, v + 32 * c, dst + 64 * c, (size_t)P.n * 2, nrows, lane);
    }
    if (P.fc_B > 0) fused_combine_rows(P, wrow0, nrows, 2 * ni + (upper ? 1 : 0), 1, lane);
    if (P.signal) {
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      if (warp == 2 && lane == 0) {
        for (int j = 0; j * P.bm_signal < BM; ++j)
          if (j * P.bm_signal < valid && row0 + j * P.bm_signal < P.rows)
            red_release_gpu_add(P.signal + (row0 + j * P.bm_signal) / P.bm_signal, 1);
      }
    }
  }
}

// kW224: the DOWN GEMM on 224-column tiles with two accumulators (see BN224).
template <bool kW224>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmA32,
                            const __grid_constant__ CUtensorMap tmW,
                            const __grid_constant__ CUtensorMap tmSFA,
                            const __grid_constant__ CUtensorMap tmSFW, const GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t s_base = smem_u32(smem);
  const uint32_t bar_full = s_base + O2_BAR;          // [S2], used in the even CTA
  const uint32_t bar_empty = bar_full + 8 * S2;       // [S2]
  const uint32_t bar_acc_full = bar_empty + 8 * S2;  // [2] (one buffer unless kW224)
  const uint32_t bar_acc_empty = bar_acc_full + 16;  // [2], used in the even CTA
  const uint32_t bar_unit_full = s_base + O2_UBAR;
  const uint32_t bar_unit_empty = bar_unit_full + 8 * kUnitQ;
  Unit2 *unit_q = reinterpret_cast<Unit2 *>(smem + O2_UNITQ);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + O2_MISC);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + O2_MISC + 4);
  constexpr uint16_t kBoth = 3;
  const int rank = (int)cluster_ctarank();
  const int first_unit = (int)cluster_id_x();
  const int ustride = (int)cluster_count_x();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S2; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full + 8 * b, 1);
      mbar_init(bar_acc_empty + 8 * b, 2 * (kEpiThreads / 32));  // epilogue warps, both CTAs
    }
    for (int q = 0; q < kUnitQ; ++q) {
      mbar_init(bar_unit_full + 8 * q, 1);
      mbar_init(bar_unit_empty + 8 * q, 2 + kEpiThreads / 32);
    }
    *abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmA32);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmSFA);
    tma_prefetch_desc(&tmSFW);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anything targets them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int units2 = P.tiles2 ? P.tiles2[4] * P.n_tiles : 0;
  const int total = P.tiles[4] * P.n_tiles + units2;
  auto take = [&](int seq, Unit2 &U) {
    const int slot = seq % kUnitQ;
    if (!mbar_wait(bar_unit_full + 8 * slot, (uint32_t)(seq / kUnitQ) & 1u, abort, kWaitLimitNs))
      return false;
    U = unit_q[slot];
    return true;
  };
  auto release_unit = [&](int seq) { mbar_arrive(bar_unit_empty + 8 * (seq % kUnitQ)); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_normal();
      const uint64_t pol_a = policy_evict_last();
      const uint32_t lead_full = mapa_shared(bar_full, 0);  // the even CTA's stage barriers
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        Unit2 U;
        if (!take(seq, U)) {
          fail(P.status, abort);
          ok = false;
          break;
        }
        release_unit(seq);
        if (U.end) break;
        if (!U.ok) {
          status_or(P.status, MOE_STATUS_BAD_INDEX);
          continue;
        }
        const int we = U.we, ni = U.ni;
        // a weight tile read by another unit of the expert (its other pairs or its
        // single, scheduled beside this one) stays in L2
        const uint64_t pol_w = U.band > 2 ? pol_keep : pol_stream;
        const int a_slices = U.nvalid == BM ? 0 : (U.nvalid + 31) / 32;
        int wrow, nb0, nb1;
        if (P.op == MOE_GEMM_GATEUP_SWIGLU) {
          wrow = we * P.n + (rank ? P.I : 0) + ni * 128;  // gate half / up half
          nb0 = ni;
          nb1 = P.I / 128 + ni;
        } else if (kW224) {
          wrow = we * P.n + ni * BN224 + (BN224 / 2) * rank;
          nb0 = nb1 = 0;
        } else {
          wrow = we * P.n + ni * 256 + 128 * rank;
          nb0 = 2 * ni;
          nb1 = 2 * ni + 1;
        }
        const int sfa_atom = (U.row0 >> 7) * P.Kg;
        // atom of group g: 128-row atoms [E][n/128][Kg], or for 224-column tiles the
        // tile's two images [E][n/224][Kg][2]
        const int sfb_tile = (we * P.n_tiles + ni) * P.Kg * 2;
        const int sfb_atom0 = kW224 ? sfb_tile : (we * (P.n / 128) + nb0) * P.Kg;
        const int sfb_atom1 = kW224 ? sfb_tile + 1 : (we * (P.n / 128) + nb1) * P.Kg;
        const int sfb_step = kW224 ? 2 : 1;
        for (int kb = 0; kb < P.Kb; kb += KB2) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort, kWaitLimitNs)) {
            fail(P.status, abort);
            ok = false;
            break;
          }
          const bool sf = (kb & 3) == 0;  // the stage starts a group of 4 k-blocks
          if (rank == 0) mbar_arrive_expect_tx(bar_full + 8 * stage, sf ? U.tx + U.tx_sf : U.tx);
          const uint32_t fb = lead_full + 8 * stage;
          const uint32_t sb = s_base + O2_B + stage * KB2 * BH_BYTES;
#pragma unroll
          for (int h = 0; h < KB2; ++h)
            tma_load_2d_pair(sb + h * BH_BYTES, &tmW, fb, (kb + h) * BK, wrow, pol_w);
          if (U.active) {
            const uint32_t sa = s_base + O2_A + stage * KB2 * A_BYTES;
#pragma unroll
            for (int h = 0; h < KB2; ++h) {
              if (a_slices == 0)
                tma_load_2d_pair(sa + h * A_BYTES, &tmA, fb, (kb + h) * BK, U.row0, pol_a);
              else
                for (int j = 0; j < a_slices; ++j)
                  tma_load_2d_pair(sa + h * A_BYTES + j * (A_BYTES / 4), &tmA32, fb, (kb + h) * BK,
                                   U.row0 + 32 * j, pol_a);
            }
            if (sf) {
              const int g = kb >> 2;
              tma_load_2d_pair(s_base + O2_SFA + stage * SFA_BYTES, &tmSFA, fb, 0, sfa_atom + g,
                               pol_a);
              if (U.m128) {
                // the weight scale image of an M=128 unit: atom 0 in rows 0-63, atom 1 in
                // rows 64-127, in the A slot's upper half (its rows 64-127 are never
                // read); only the even CTA is active here, so its own barrier takes them
                const uint32_t img = sa + A_BYTES / 2;
                const uint8_t *a0 = P.W_sf + (size_t)(sfb_atom0 + g) * 512;
                const uint8_t *a1 = P.W_sf + (size_t)(sfb_atom1 + g) * 512;
                bulk_load(img, a0, 512, bar_full + 8 * stage);
                bulk_load(img + 512, a0, 512, bar_full + 8 * stage);
                bulk_load(img + 1024, a1, 512, bar_full + 8 * stage);
                bulk_load(img + 1536, a1, 512, bar_full + 8 * stage);
              } else {
                const uint32_t ssfb = s_base + O2_SFB + stage * SFB_BYTES;
                tma_load_2d_pair(ssfb, &tmSFW, fb, 0, sfb_atom0 + sfb_step * g, pol_w);
                tma_load_2d_pair(ssfb + 512, &tmSFW, fb, 0, sfb_atom1 + sfb_step * g, pol_w);
              }
            }
          }
          ++issued;
          if (++stage == S2) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA can exit: the even CTA
        // sees them on its stage barriers, the odd CTA waits a fixed grace period.
        if (rank == 0) {
          volatile int never = 0;
          for (int i = 0; i < S2 && i < issued; ++i) {
            if (--stage < 0) {
              stage = S2 - 1;
              phase ^= 1;
            }
            mbar_wait(bar_full + 8 * stage, phase, &never, 100000000ull);
          }
        } else {
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 1000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // N = 256, UE8M0 scales, M = 256 (or 128) over the pair; bits 4-5 / 29-30 pick
      // the scale byte
      const uint32_t idesc_n = ((uint32_t)((kW224 ? BN224 : BN) >> 3) << 17) | (1u << 23);
      const uint32_t tmem_sf = kW224 ? TMEM_SF224 : TMEM_SF2;
      int stage = 0, nacc = 0;  // nacc: units accumulated so far (buffer nacc % 2 if kW224)
      uint32_t phase = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        Unit2 U;
        if (!take(seq, U)) {
          fail(P.status, abort);
          break;
        }
        release_unit(seq);
        if (U.end) break;
        if (!U.ok || rank != 0) continue;  // the odd CTA only follows the unit stream
        const uint32_t idesc_base = idesc_n | ((uint32_t)((U.m128 ? BM : 2 * BM) >> 4) << 24);
        const int buf = kW224 ? nacc & 1 : 0;
        const uint32_t acc_phase = (uint32_t)(kW224 ? nacc >> 1 : nacc) & 1u;
        const uint32_t acc = tmem + (kW224 ? (uint32_t)(BN224 * buf) : 0u);
        if (!mbar_wait_cluster(bar_acc_empty + 8 * buf, acc_phase ^ 1, abort, kWaitLimitNs)) {
          fail(P.status, abort);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < P.Kb; kb += KB2) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort, kWaitLimitNs)) {
            fail(P.status, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          // a stage's scale columns are rewritten S2 stages later, after its refill
          const uint32_t ssfa = s_base + O2_SFA + stage * SFA_BYTES;
          const uint32_t ssfb = s_base + O2_SFB + stage * SFB_BYTES;
          const uint32_t sa = s_base + O2_A + stage * KB2 * A_BYTES;
          const uint32_t sb = s_base + O2_B + stage * KB2 * BH_BYTES;
#pragma unroll
          for (int h = 0; h < KB2; ++h) {
            const int kbh = kb + h;
            const uint32_t t_sfa = tmem + tmem_sf + 16 * ((kbh >> 2) % kSfSets);
            const uint32_t t_sfb = t_sfa + 4;
            if ((kbh & 3) == 0) {  // the group's scale atoms, once per four k-blocks
              tc_cp_pair_32x128b_x4(t_sfa, smem_desc(ssfa, 16, 128, 0));
              if (U.m128) {
                tc_cp_pair_128x128b(t_sfb, smem_desc(sa + h * A_BYTES + A_BYTES / 2, 16, 128, 0));
              } else {
                tc_cp_pair_32x128b_x4(t_sfb, smem_desc(ssfb, 16, 128, 0));
                tc_cp_pair_32x128b_x4(t_sfb + 4, smem_desc(ssfb + 512, 16, 128, 0));
              }
            }
            // k-block kbh's scales are byte kbh % 4 of each atom word
            const uint32_t idesc =
                idesc_base | ((uint32_t)(kbh & 3) << 29) | ((uint32_t)(kbh & 3) << 4);
#pragma unroll
            for (int j = 0; j < BK / 32; ++j) {
              const uint64_t ad = smem_desc(sa + h * A_BYTES + 32 * j, 16, 1024, 2);
              const uint64_t bd = smem_desc(sb + h * BH_BYTES + 32 * j, 16, 1024, 2);
              tc_mma_pair_mxf8(acc, ad, bd, idesc, t_sfa, t_sfb, (kb | h | j) != 0);
            }
          }
          tc_commit_pair_mc(bar_empty + 8 * stage, kBoth);
          if (++stage == S2) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(bar_acc_full + 8 * buf, kBoth);
        ++nacc;
      }
    }
  } else if (warp < 2 + kEpiThreads / 32) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_local = 32 * q + lane;
    const uint32_t t_row = tmem + ((uint32_t)(32 * q) << 16);
    float *amax_x = reinterpret_cast<float *>(smem + O2_AMAX);
    float *xbuf = reinterpret_cast<float *>(smem + O2_XBUF);
    // the DOWN epilogue's staging slots share xbuf (the GATEUP M=128 exchange buffer)
    uint8_t *stage = smem + O2_XBUF + (warp - 2) * STAGE_BYTES;
    const uint32_t lead_acc_empty = mapa_shared(bar_acc_empty, 0);
    int buf = 0, nacc = 0;  // as the MMA issuer: buffer nacc % 2 if kW224
    auto release_acc = [&] {
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead_acc_empty + 8 * buf);
    };
    for (int seq = 0;; ++seq) {
      Unit2 U;
      if (!take(seq, U)) {
        fail(P.status, abort);
        break;
      }
      __syncwarp();
      if (lane == 0) release_unit(seq);
      if (U.end) break;
      if (!U.ok) continue;
      buf = kW224 ? nacc & 1 : 0;
      const uint32_t acc_phase = (uint32_t)(kW224 ? nacc >> 1 : nacc) & 1u;
      ++nacc;
      if (!mbar_wait(bar_acc_full + 8 * buf, acc_phase, abort, kWaitLimitNs)) {
        fail(P.status, abort);
        break;
      }
      tc_fence_after();
      const uint32_t t_acc = t_row + (kW224 ? (uint32_t)(BN224 * buf) : 0u);
      if (!U.active) {  // this CTA's rows of the pair MMA carry no tile
        tc_fence_before();
        release_acc();
      } else if (kW224) {
        epilogue_down224(P, U.row0, U.nvalid, U.ni, t_acc, half, row_local, lane, stage,
                         release_acc);
      } else if (U.m128) {
        epilogue_m128(P, U.row0, U.nvalid, U.ni, t_acc, q, half, warp, lane, amax_x, xbuf,
                      stage, release_acc);
      } else {
        epilogue_tile(P, U.row0, U.nvalid, U.ni, t_acc, half, row_local, warp, lane, amax_x,
                      stage, release_acc);
      }
    }
  } else if (lane == 0) {
    // ------------------------------------------------------------ scheduler
    int seq = 0;
    auto push = [&](const Unit2 &U) {
      const int slot = seq % kUnitQ;
      if (!mbar_wait(bar_unit_empty + 8 * slot, ((uint32_t)(seq / kUnitQ) & 1u) ^ 1u, abort,
                     kWaitLimitNs)) {
        fail(P.status, abort);
        return false;
      }
      unit_q[slot] = U;
      mbar_arrive(bar_unit_full + 8 * slot);
      ++seq;
      return true;
    };
    bool ok = true;
    // U.ok false: every role skips the unit, and the producer records it.  Equal rounds
    // over just enough CTA pairs, as in the one-CTA kernel.
    const int rounds = (total + ustride - 1) / ustride;
    const int pairs = rounds > 0 ? (total + rounds - 1) / rounds : 0;
    for (int unit = first_unit; ok && unit < total && first_unit < pairs; unit += pairs)
      ok = push(get_2sm_unit<kW224>(P, unit, units2, rank));
    if (ok) {
      Unit2 end = {};
      end.end = true;
      push(end);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the even CTA's MMAs read the odd CTA's shared memory to the end
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, TMEM_COLS);
}

// Weight scale bytes [blocks][Kb] -> atoms [blocks][Kg][512]: every word of a group's
// atom holds the group's four k-block bytes (0 past the last k-block).
__global__ void pack_scales_kernel(const uint8_t *__restrict__ sf, uint8_t *__restrict__ atoms,
                                   size_t n_atoms, int Kb, int Kg) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // one 16-byte piece
  if (i >= n_atoms * 32) return;
  const size_t a = i >> 5;
  const int g = (int)(a % Kg);
  const uint8_t *src = sf + (a / Kg) * Kb + 4 * g;
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (4 * g + j < Kb) w |= (uint32_t)src[j] << (8 * j);
  reinterpret_cast<uint4 *>(atoms)[i] = make_uint4(w, w, w, w);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D byte tensor [rows][cols] (cols contiguous), boxes of box_rows x 128 bytes,
// 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
              uint32_t box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale atoms [n_atoms][512 bytes] as a 2-D uint32 tensor [n_atoms][128], box_atoms
// atoms per box, so TMA (which can signal the other CTA of a pair) moves them.
bool make_sf_map(CUtensorMap *m, const void *base, uint64_t n_atoms, uint32_t box_atoms) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || n_atoms == 0 || n_atoms > 0x7fffffffull) return false;
  cuuint64_t dims[2] = {128, n_atoms};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, box_atoms};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-CTA cluster launch of `kernel` on at most one cluster per SM pair, no more
// clusters than can be resident at once (the grid is persistent).
template <class Kernel, class... Args>
int launch_pairs(Kernel kernel, uint32_t smem, int sms, int &max_clusters, cudaStream_t st,
                 Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms / 2 * 2 > 0 ? sms / 2 * 2 : 2));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters == 0) {
    cudaError_t e = cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &cfg);
    if (e != cudaSuccess || max_clusters <= 0)
      return set_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidConfiguration);
  }
  if ((int)cfg.gridDim.x / 2 > max_clusters) cfg.gridDim = dim3((unsigned)(2 * max_clusters));
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return set_cuda_error(e);
  return check_launch();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_packed_scale_bytes(int E, int n, int k) {
  if (E <= 0 || n <= 0 || k <= 0 || n % 128 || k % 128) return 0;
  return (size_t)E * (n / 128) * sf_groups(k) * 512;
}

// Weight scale images of tile_n-row tiles (tile_n <= 256, a multiple of 16): per (expert,
// tile, group of four k-blocks) two 128-row images, image h holding tile rows
// [128h, 128h + 128) in the SF atom layout, each row with its own 128x128 block's scale
// (rows past tile_n zero).  One 16-byte piece (four rows of one lane) per thread.
__global__ void pack_scales_tiled_kernel(const uint8_t *__restrict__ sf, uint8_t *__restrict__ out,
                                         size_t n_atoms, int n, int tile_n, int n_tiles, int Kb,
                                         int Kg) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_atoms * 32) return;
  const size_t a = i >> 5;
  const int lane_row = (int)(i & 31), h = (int)(a & 1);
  const int g = (int)((a >> 1) % Kg);
  const size_t tile = (a >> 1) / Kg;
  const size_t e = tile / n_tiles;
  const int ni = (int)(tile % n_tiles);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int tr = 128 * h + 32 * q + lane_row;
    w[q] = 0;
    if (tr < tile_n) {
      const uint8_t *src = sf + (e * (n / 128) + (size_t)(ni * tile_n + tr) / 128) * Kb + 4 * g;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (4 * g + j < Kb) w[q] |= (uint32_t)src[j] << (8 * j);
    }
  }
  reinterpret_cast<uint4 *>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
}

extern "C" size_t moe_tiled_scale_bytes(int E, int n, int k, int tile_n) {
  if (E <= 0 || n <= 0 || k <= 0 || n % 128 || k % 128 || tile_n <= 128 || tile_n > 256 ||
      tile_n % 16 || n % tile_n)
    return 0;
  return (size_t)E * (n / tile_n) * sf_groups(k) * 1024;
}

extern "C" int moe_pack_weight_scales_tiled(int E, int n, int k, int tile_n, const uint8_t *W_sf,
                                            void *W_sf_tiled, void *stream) {
  const size_t bytes = moe_tiled_scale_bytes(E, n, k, tile_n);
  if (!bytes || !W_sf || !W_sf_tiled || (uintptr_t)W_sf_tiled % 16) return MOE_ERR_INVALID;
  const size_t n_atoms = bytes / 512, pieces = n_atoms * 32;
  pack_scales_tiled_kernel<<<(unsigned)((pieces + 255) / 256), 256, 0, as_stream(stream)>>>(
      W_sf, static_cast<uint8_t *>(W_sf_tiled), n_atoms, n, tile_n, n / tile_n, k / 128,
      sf_groups(k));
  return check_launch();
}

extern "C" size_t moe_scale_bytes(int64_t rows, int k, int fmt) {
  if (rows <= 0 || k <= 0 || rows % 128 || k % 128) return 0;
  if (fmt == MOE_FMT_FP8_F32) return (size_t)rows * (k / 128) * 4;
  if (fmt != MOE_FMT_FP8) return 0;
  return (size_t)(rows / 128) * sf_groups(k) * 512;
}

extern "C" int moe_pack_weight_scales(int E, int n, int k, const uint8_t *W_sf,
                                      void *W_sf_packed, void *stream) {
  const size_t bytes = moe_packed_scale_bytes(E, n, k);
  if (!bytes || !W_sf || !W_sf_packed || (uintptr_t)W_sf_packed % 16) return MOE_ERR_INVALID;
  const size_t n_atoms = bytes / 512;
  const size_t pieces = n_atoms * 32;
  pack_scales_kernel<<<(unsigned)((pieces + 255) / 256), 256, 0, as_stream(stream)>>>(
      W_sf, static_cast<uint8_t *>(W_sf_packed), n_atoms, k / 128, sf_groups(k));
  return check_launch();
}

__global__ void weight_scales_f32_kernel(const uint8_t *__restrict__ sf, float *__restrict__ out,
                                         size_t n) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = pow2i((int)sf[i] - 127);
}

extern "C" int moe_weight_scales_f32(int E, int n, int k, const uint8_t *W_sf, float *W_sf_f32,
                                     void *stream) {
  if (E <= 0 || n <= 0 || k <= 0 || n % 128 || k % 128 || !W_sf || !W_sf_f32)
    return MOE_ERR_INVALID;
  const size_t cnt = (size_t)E * (n / 128) * (k / 128);
  weight_scales_f32_kernel<<<(unsigned)((cnt + 255) / 256), 256, 0, as_stream(stream)>>>(
      W_sf, W_sf_f32, cnt);
  return check_launch();
}

extern "C" int moe_grouped_gemm_fp8(const moe_gemm_args *a, void *stream) {
  if (!a) return MOE_ERR_INVALID;
  if (a->op != MOE_GEMM_GATEUP_SWIGLU && a->op != MOE_GEMM_DOWN) return MOE_ERR_INVALID;
  if (a->pair_tiles != 0 && a->pair_tiles != 1) return MOE_ERR_INVALID;
  if (a->tile_n != 0 && a->tile_n != BN && a->tile_n != BN224) return MOE_ERR_INVALID;
  const bool w224 = a->tile_n == BN224;  // 224-column DOWN tiles with two accumulators
  if (w224) {
    if (a->op != MOE_GEMM_DOWN || a->signal || a->combine || a->scale_fmt)
      return MOE_ERR_INVALID;
    if (a->n % BN224) return MOE_ERR_UNSUPPORTED;
  }
  if (a->scale_fmt != 0 && a->scale_fmt != 1) return MOE_ERR_INVALID;
  if (a->scale_fmt == 1 && a->pair_tiles) return MOE_ERR_UNSUPPORTED;
  if (a->n <= 0 || a->k <= 0 || a->rows <= 0 || a->max_tiles <= 0 || a->num_experts <= 0)
    return MOE_ERR_INVALID;
  if (a->n % 256 || a->k % 128 || a->rows % 128) return MOE_ERR_UNSUPPORTED;
  if (a->pair_tiles && a->k % (KB2 * BK)) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)a->num_experts * a->n > INT32_MAX || a->rows > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (!a->A || !a->A_sf || !a->W || !a->W_sf || !a->tiles || !a->out) return MOE_ERR_INVALID;
  if (a->op == MOE_GEMM_GATEUP_SWIGLU && (!a->out_sf || a->signal)) return MOE_ERR_INVALID;
  if (a->signal && (a->block_m_signal <= 0 || BM % a->block_m_signal)) return MOE_ERR_INVALID;
  if (const moe_fused_combine *fc = a->combine) {
    if (a->op != MOE_GEMM_DOWN || a->signal || fc->B <= 0 || fc->K < 1 ||
        fc->K > kFusedKMax || !fc->row_of || !fc->topk_w || !fc->pending || !fc->out ||
        (uintptr_t)fc->out % 16 || fc->src_rows < 0 || (fc->src_rows > 0 && !fc->src_of) ||
        fc->shared_row0 < -1 ||
        (fc->shared_row0 >= 0 && fc->shared_row0 + fc->B > a->rows))
      return MOE_ERR_INVALID;
  }
  const void *ptrs[] = {a->A, a->A_sf, a->W, a->W_sf, a->out, a->out_sf};
  for (const void *p : ptrs)
    if ((uintptr_t)p % 16) return MOE_ERR_INVALID;
  CUtensorMap mA, mA32, mW;
  if (!make_map(&mA, a->A, (uint64_t)a->rows, (uint64_t)a->k) ||
      !make_map(&mA32, a->A, (uint64_t)a->rows, (uint64_t)a->k, 32) ||
      !make_map(&mW, a->W, (uint64_t)a->num_experts * a->n, (uint64_t)a->k,
                w224 ? (a->pair_tiles ? BN224 / 2 : BN224) : 128))
    return MOE_ERR_CUDA;
  if (a->tiles2 && (a->expert2 < 0 || a->expert2 >= a->num_experts || a->row_offset2 < 0 ||
                    a->row_offset2 % 128 || a->row_offset2 >= a->rows))
    return MOE_ERR_INVALID;
  if (a->max_tiles > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  GemmParams P;
  P.op = a->op;
  P.rows = a->rows;
  P.tiles2 = a->tiles2;
  P.row_offset2 = (int)a->row_offset2;
  P.expert2 = a->expert2;
  P.num_experts = a->num_experts;
  P.max_tiles = (int)a->max_tiles;
  P.n = a->n;
  P.k = a->k;
  P.Kb = a->k / BK;
  P.Kg = sf_groups(a->k);
  P.n_tiles = a->n / (w224 ? BN224 : BN);
  P.I = a->n / 2;
  P.A_sf = static_cast<const uint8_t *>(a->A_sf);
  P.W_sf = static_cast<const uint8_t *>(a->W_sf);
  P.phys2log = a->phys2log;
  P.tiles = a->tiles;
  P.out = static_cast<uint8_t *>(a->out);
  P.out_sf = static_cast<uint8_t *>(a->out_sf);
  P.signal = a->signal;
  P.bm_signal = a->block_m_signal > 0 ? a->block_m_signal : BM;
  P.status = a->status;
  P.scale_fmt = a->scale_fmt;
  P.fc_B = 0;
  if (const moe_fused_combine *fc = a->combine) {
    P.fc_B = fc->B;
    P.fc_K = fc->K;
    P.fc_nch = a->n / 128;
    P.fc_row_of = fc->row_of;
    P.fc_src_of = fc->src_of;
    P.fc_w = fc->topk_w;
    P.fc_pending = fc->pending;
    P.fc_src_rows = fc->src_rows;
    P.fc_shared_row0 = fc->shared_row0;
    P.fc_out = static_cast<uint16_t *>(fc->out);
  }
  static bool attr_set[kMaxDevices] = {};
  static int max_clusters[kMaxDevices] = {}, max_clusters224[kMaxDevices] = {};
  const int dev = device_slot();
  if (dev < 0) return dev;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grouped_gemm_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grouped_gemm_kernel<false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grouped_gemm_2sm_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM2_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grouped_gemm_2sm_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM2_BYTES);
    if (e != cudaSuccess) return set_cuda_error(e);
    attr_set[dev] = true;
  }
  const int sms = a->num_sms > 0 ? a->num_sms : device_sm_count();
  if (a->pair_tiles) {
    CUtensorMap mSFA, mSFW;
    const uint64_t kg = (uint64_t)sf_groups(a->k);
    // weight scales: 128-row atoms, or two images per 224-column tile
    const uint64_t w_atoms = w224
                                 ? (uint64_t)a->num_experts * (a->n / BN224) * kg * 2
                                 : (uint64_t)a->num_experts * (a->n / 128) * kg;
    if (!make_sf_map(&mSFA, a->A_sf, (uint64_t)(a->rows / 128) * kg, 1) ||
        !make_sf_map(&mSFW, a->W_sf, w_atoms, 1))
      return MOE_ERR_CUDA;
    if (w224)
      return launch_pairs(grouped_gemm_2sm_kernel<true>, SMEM2_BYTES, sms, max_clusters224[dev],
                          as_stream(stream), mA, mA32, mW, mSFA, mSFW, P);
    return launch_pairs(grouped_gemm_2sm_kernel<false>, SMEM2_BYTES, sms, max_clusters[dev],
                        as_stream(stream), mA, mA32, mW, mSFA, mSFW, P);
  }
  const int64_t max_units = a->tiles2 ? sms : a->max_tiles * (a->n / BN);
  const int grid = (int)(max_units < sms ? max_units : sms);
  if (a->scale_fmt)
    grouped_gemm_kernel<true><<<grid, kGemmThreads, SMEM_BYTES, as_stream(stream)>>>(mA, mA32, mW, P);
  else if (w224)
    grouped_gemm_kernel<false, true>
        <<<grid, kGemmThreads, SMEM_BYTES, as_stream(stream)>>>(mA, mA32, mW, P);
  else
    grouped_gemm_kernel<false><<<grid, kGemmThreads, SMEM_BYTES, as_stream(stream)>>>(mA, mA32, mW, P);
  return check_launch();
}
