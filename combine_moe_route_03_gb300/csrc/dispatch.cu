// moe_dispatch: the EP all-to-all of one GPU — a stable expert-major permutation
// of the routed (token, k) rows inside HBM, fused with 1x128 FP8 quantisation.
//
// The two layouts are the ones DeepEP's two dispatch modes hand to DeepGEMM
// ("Large-scale EP: DeepEP, EPLB and two-batch overlap", §DeepEP: each mode where
// it belongs): contiguous per-expert segments (normal mode, prefill) and a
// fixed-capacity masked buffer (low-latency mode, decode; fixed shapes that a CUDA
// graph can replay).  DeepEP's normal mode has the CPU wait for a GPU count before
// it can size buffers ("DeepEP 完全拆解", §隐式的 CPU 等待); here the counts, the
// prefix sums and the tile list stay on the device, so no call waits.
//
// Three kernels, no atomics whose order could change a result:
//   dispatch_count_kernel   per chunk of 128 tokens: physical expert of every
//                           (t,k) (EPLB map applied), its rank among the chunk's
//                           rows of that expert in (t,k) order, chunk histogram.
//   dispatch_scan_kernel    one CTA: chunk bases per expert, expert counts,
//                           segment starts, capacity check, M-tile list and work
//                           items (experts with several items spread evenly between
//                           those with one).  A batch of one chunk counts here too.
//   dispatch_scatter_kernel warps over (token, column chunk): quantise each piece of
//                           a row once, write its K copies and their scales,
//                           row_of / src_of.
#include <climits>
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kChunk = 128;  // tokens per count chunk
constexpr int kCountWarps = 8;
constexpr int kScanThreads = 1024;
constexpr int kScatterWarps = 8;

struct DispatchWs {
  int32_t *phys, *rank, *hist, *seg;
};

__host__ __device__ inline size_t align256(size_t b) { return (b + 255) / 256 * 256; }

__host__ __device__ inline DispatchWs carve(void *ws, int B, int K, int N_phys) {
  char *p = static_cast<char *>(ws);
  const int nchunks = (B + kChunk - 1) / kChunk;
  DispatchWs w;
  w.phys = reinterpret_cast<int32_t *>(p);
  p += align256(sizeof(int32_t) * B * K);
  w.rank = reinterpret_cast<int32_t *>(p);
  p += align256(sizeof(int32_t) * B * K);
  w.hist = reinterpret_cast<int32_t *>(p);
  p += align256(sizeof(int32_t) * (size_t)nchunks * N_phys);
  w.seg = reinterpret_cast<int32_t *>(p);
  return w;
}

// Counts of one kChunk-token chunk: each (t, k) pair's physical expert and its rank
// among the chunk's pairs of that expert (ascending (t, k)); the chunk's per-expert
// totals go to ws.hist.  kCountWarps warps do the work; a larger block calls it too
// (every thread reaches the barriers, warps past kCountWarps get no pairs).  sm:
// kCountWarps * N_phys + 2 * kChunk * K ints of shared memory.
__device__ __forceinline__ void count_chunk(int chunk, const int32_t *__restrict__ topk_idx,
                                            const int32_t *__restrict__ log2phys,
                                            const int32_t *__restrict__ rep, int max_rep,
                                            int B, int K, int N_log, int N_phys,
                                            const DispatchWs &ws, int32_t *status,
                                            int32_t *sm) {
  int32_t *whist = sm;                              // [kCountWarps][N_phys]
  int32_t *pp = whist + kCountWarps * N_phys;       // [kChunk*K]
  int32_t *lr = pp + kChunk * K;                    // [kChunk*K]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t_begin = chunk * kChunk;
  const int ntok = min(kChunk, B - t_begin);
  const int npairs = ntok * K;
  for (int i = tid; i < kCountWarps * N_phys; i += blockDim.x) whist[i] = 0;
  __syncthreads();

  const int per = (npairs + kCountWarps - 1) / kCountWarps;
  const int w_begin = warp * per, w_end = min(npairs, w_begin + per);
  const uint32_t lt_mask = (1u << lane) - 1u;
  // the warp's expert ids, loaded together (up to 4 per lane) before the ranking rounds
  constexpr int kPre = 4;
  int pre[kPre];
#pragma unroll
  for (int r = 0; r < kPre; ++r) {
    const int i = w_begin + 32 * r + lane;
    pre[r] = i < w_end ? topk_idx[(size_t)t_begin * K + i] : 0;
  }
  for (int base = w_begin, round = 0; base < w_end; base += 32, ++round) {
    const int i = base + lane;
    const bool valid = i < w_end;
    int p = -1;
    if (valid) {
      const int t = t_begin + i / K;
      int e = 0;
#pragma unroll
      for (int r = 0; r < kPre; ++r)
        if (round == r) e = pre[r];
      if (round >= kPre) e = topk_idx[(size_t)t_begin * K + i];
      if (e < 0 || e >= N_log) {
        status_or(status, MOE_STATUS_BAD_INDEX);
      } else if (log2phys) {
        const int re = rep[e];
        p = (re >= 1 && re <= max_rep) ? log2phys[(size_t)max_rep * e + (t % re)] : -1;
        if (p < 0 || p >= N_phys) {
          status_or(status, MOE_STATUS_BAD_INDEX);
          p = -1;
        }
      } else {
        p = e < N_phys ? e : -1;
      }
    }
    const int key = valid ? p : -2;
    const uint32_t mask = __match_any_sync(0xffffffffu, key);
    const int leader = __ffs(mask) - 1;
    const int old = (p >= 0) ? whist[warp * N_phys + p] : 0;
    const int r = old + __popc(mask & lt_mask);
    __syncwarp();
    if (p >= 0 && lane == leader) whist[warp * N_phys + p] = old + __popc(mask);
    __syncwarp();
    if (valid) {
      pp[i] = p;
      lr[i] = r;
    }
  }
  __syncthreads();
  for (int p = tid; p < N_phys; p += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kCountWarps; ++w) {
      const int v = whist[w * N_phys + p];
      whist[w * N_phys + p] = run;
      run += v;
    }
    ws.hist[(size_t)chunk * N_phys + p] = run;
  }
  __syncthreads();
  for (int i = tid; i < npairs; i += blockDim.x) {
    const int p = pp[i];
    const int w = i / per;
    ws.phys[(size_t)t_begin * K + i] = p;
    ws.rank[(size_t)t_begin * K + i] = p >= 0 ? whist[w * N_phys + p] + lr[i] : -1;
  }
}

__global__ void __launch_bounds__(kCountWarps * 32) dispatch_count_kernel(
    const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ log2phys,
    const int32_t *__restrict__ rep, int max_rep, int B, int K, int N_log, int N_phys,
    DispatchWs ws, int32_t *status) {
  extern __shared__ int32_t sm[];
  count_chunk(blockIdx.x, topk_idx, log2phys, rep, max_rep, B, K, N_log, N_phys, ws, status,
              sm);
}

// Inclusive block-wide sum (Hillis-Steele) of one value per thread over the CTA's
// kScanThreads threads: shuffles inside each warp, then one warp scans the warp
// totals.  `buf` holds one int per warp.
__device__ __forceinline__ int block_scan(int32_t *buf, int v) {
  const int p = threadIdx.x, lane = p & 31, warp = p >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) buf[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kScanThreads / 32 ? buf[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += o;
    }
    if (lane < kScanThreads / 32) buf[lane] = w;
  }
  __syncthreads();
  const int prefix = warp > 0 ? buf[warp - 1] : 0;
  __syncthreads();  // buf is reused by the next scan
  return v + prefix;
}

// Work items of the 2-SM GEMM: an expert's tile pairs (one weight tile shared by both
// SMs of a pair), then its odd last tile alone, all in one group, so the single runs
// beside the pairs that read the same weight tiles (the groups' order: see the scan).  Item k =
// {tile 0, tile 1 or -1, first item of its group, items in its group, 1 for a pair,
// 0, 0, 0}; a group's units are N-tile-major.
// An 8-int tile-list entry as two 16-byte stores (the list is 16-byte aligned).
__device__ __forceinline__ void put8(int32_t *dst, int a, int b, int c, int d, int e) {
  reinterpret_cast<int4 *>(dst)[0] = make_int4(a, b, c, d);
  reinterpret_cast<int4 *>(dst)[1] = make_int4(e, 0, 0, 0);
}

__device__ __forceinline__ void write_items(int32_t *items, int first, int nt, int item_first) {
  const int np = nt / 2, gc = np + nt % 2;
  for (int j = 0; j < gc; ++j) {
    const bool pair = j < np;
    put8(items + 8 * (size_t)(item_first + j), first + 2 * j, pair ? first + 2 * j + 1 : -1,
         item_first, gc, pair ? 1 : 0);
  }
}

// With a single chunk (small batches) the count runs here first, in this block
// (fused = 1, count_chunk's shared memory as the launch's dynamic shared memory): one
// launch and one round trip of the counts through global memory fewer.
__global__ void __launch_bounds__(kScanThreads) dispatch_scan_kernel(
    int B, int N_phys, int nchunks, int layout, int cap, int64_t rows_alloc, DispatchWs ws,
    int32_t *__restrict__ counts, int32_t *__restrict__ tiles, int32_t *__restrict__ src_of,
    int32_t *__restrict__ shared_tiles, int32_t *status, int fused,
    const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ log2phys,
    const int32_t *__restrict__ rep, int max_rep, int K, int N_log) {
  if (fused) {
    extern __shared__ int32_t sm[];
    count_chunk(0, topk_idx, log2phys, rep, max_rep, B, K, N_log, N_phys, ws, status, sm);
    __syncthreads();  // ws.hist / phys / rank of the chunk, written by this block
  }
  __shared__ int32_t scan[kScanThreads / 32];
  __shared__ int32_t pad_seg[kScanThreads], pad_from[kScanThreads], pad_to[kScanThreads];
  __shared__ int32_t totals[4];  // tiles, pairs, singles, items
  const int p = threadIdx.x;
  int cnt = 0, valid = 0, nt = 0;
  if (p < N_phys) {
    // exclusive prefix over the chunks, 16 loads in flight before their stores
    constexpr int kBatch = 16;
    for (int c0 = 0; c0 < nchunks; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        v[i] = c0 + i < nchunks ? ws.hist[(size_t)(c0 + i) * N_phys + p] : 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (c0 + i < nchunks) ws.hist[(size_t)(c0 + i) * N_phys + p] = cnt;
        cnt += v[i];
      }
    }
    counts[p] = cnt;
    valid = cnt;
    if (layout == MOE_LAYOUT_MASKED && cnt > cap) {
      valid = cap;
      status_or(status, MOE_STATUS_CAPACITY);
    }
    nt = (valid + 127) / 128;
  }
  const int first = block_scan(scan, nt) - nt;
  const int np = nt / 2, ns = nt % 2, gcnt = np + ns;
  // Order of the experts' tiles and item groups (both GEMMs' schedules: the one-CTA
  // kernel walks the tiles, the 2-SM kernel the items): an expert with several items
  // reads each weight tile from HBM once for all of them (the rest come from L2), one
  // with a single item reads a weight tile from HBM per unit.  Spreading the multi-item
  // experts evenly between the single-item ones, in expert order within each kind, keeps
  // the HBM demand of the CTAs running side by side even.  Multi-item expert i of nm
  // goes before single-item expert floor((2i + 1) * n1 / (2 nm)) of n1; experts without
  // tiles take no place.  The rows stay in expert order (segments as `first`).  One scan
  // gives both ranks (counts <= kScanThreads, 11 bits apart), two more each position's
  // first item and first tile.
  const int multi = (p < N_phys && gcnt >= 2) ? 1 : 0;
  const int single = (p < N_phys && gcnt == 1) ? 1 : 0;
  const int kinds_incl = block_scan(scan, multi | (single << 11));
  const int multi_rank = (kinds_incl & 2047) - multi;
  const int single_rank = (kinds_incl >> 11) - single;
  __shared__ int32_t kinds[2];
  __shared__ int32_t by_pos[kScanThreads], by_pos_nt[kScanThreads];
  if (p == kScanThreads - 1) {
    kinds[0] = kinds_incl & 2047;
    kinds[1] = kinds_incl >> 11;
  }
  by_pos[p] = 0;
  by_pos_nt[p] = 0;
  const int singles = __syncthreads_count(ns);  // also orders the writes above
  const int nm = kinds[0], n1 = kinds[1];
  int pos = -1;
  if (multi) {  // (products < 2^22: ranks and counts are at most kScanThreads)
    pos = (2 * multi_rank + 1) * n1 / (2 * nm) + multi_rank;
  } else if (single) {  // after the multi-item experts whose slot is at most single_rank
    const int q = n1 > 0 ? (2 * nm * (single_rank + 1) - 1) / n1 : 0;
    pos = single_rank + min(nm, (q + 1) / 2);
  }
  if (pos >= 0) {
    by_pos[pos] = gcnt;
    by_pos_nt[pos] = nt;
  }
  __syncthreads();
  const int at_pos = p < nm + n1 ? by_pos[p] : 0;
  const int at_pos_nt = p < nm + n1 ? by_pos_nt[p] : 0;
  const int pos_incl = block_scan(scan, at_pos);         // items up to position p
  const int pos_nt_incl = block_scan(scan, at_pos_nt);   // tiles up to position p
  by_pos[p] = pos_incl - at_pos;
  by_pos_nt[p] = pos_nt_incl - at_pos_nt;
  if (p == kScanThreads - 1) {
    totals[0] = first + nt;
    totals[1] = pos_incl - singles;  // pairs: items that are not singles
    totals[2] = singles;
    totals[3] = pos_incl;
  }
  __syncthreads();
  const int item_first = pos >= 0 ? by_pos[pos] : 0;
  const int tile_first = pos >= 0 ? by_pos_nt[pos] : 0;
  const int64_t max_tiles = rows_alloc / 128;
  if (p < N_phys) {
    const int seg = layout == MOE_LAYOUT_CONTIG ? first * 128 : p * cap;
    ws.seg[p] = seg;
    for (int i = 0; i < nt; ++i)
      put8(tiles + 8 + 8 * (size_t)(tile_first + i), seg + 128 * i, p,
           min(128, valid - 128 * i), tile_first, nt);
    write_items(tiles + 8 + 8 * max_tiles, tile_first, nt, item_first);
    pad_seg[p] = seg;  // rows [valid, end) of this expert's segment that no token fills
    pad_from[p] = valid;
    pad_to[p] = layout == MOE_LAYOUT_CONTIG ? nt * 128 : cap;
  }
  __syncthreads();
  if (src_of) {  // one warp per expert, coalesced
    const int lane = p & 31;
    for (int e = p >> 5; e < N_phys; e += kScanThreads / 32)
      for (int j = pad_from[e] + lane; j < pad_to[e]; j += 32) src_of[pad_seg[e] + j] = -1;
  }
  const int total_tiles = totals[0];
  const int64_t used = layout == MOE_LAYOUT_CONTIG ? (int64_t)total_tiles * 128
                                                   : (int64_t)N_phys * cap;
  if (p == 0) {
    tiles[0] = total_tiles;
    tiles[1] = (int32_t)used;
    tiles[2] = totals[1];
    tiles[3] = totals[2];
    tiles[4] = totals[3];
    for (int i = 5; i < 8; ++i) tiles[i] = 0;
  }
  if (src_of)
    for (int64_t r = used + p; r < rows_alloc; r += kScanThreads) src_of[r] = -1;
  if (shared_tiles) {  // one expert, the batch in token order; capacity = its tiles
    const int snt = (B + 127) / 128;
    if (p == 0) {
      shared_tiles[0] = snt;
      shared_tiles[1] = snt * 128;
      shared_tiles[2] = snt / 2;
      shared_tiles[3] = snt % 2;
      shared_tiles[4] = snt / 2 + snt % 2;
      for (int i = 5; i < 8; ++i) shared_tiles[i] = 0;
    }
    // items: snt / 2 pairs, then the odd last tile alone, all in one group
    const int snp = snt / 2, sgc = snp + snt % 2;
    for (int j = p; j < sgc; j += kScanThreads) {
      const bool pair = j < snp;
      put8(shared_tiles + 8 + 8 * (size_t)snt + 8 * (size_t)j, 2 * j, pair ? 2 * j + 1 : -1, 0,
           sgc, pair ? 1 : 0);
    }
    for (int i = p; i < snt; i += kScanThreads)
      put8(shared_tiles + 8 + 8 * (size_t)i, 128 * i, 0, min(128, B - 128 * i), 0, snt);
  }
}

// One warp per task = (token, run of `cpt` chunks of kCols columns): each lane
// quantises kCols/32 values (8 or 16), 128/(kCols/32) lanes share one 128-column
// block's amax, and each lane stores 8 or 16 bytes into each of the K copies.  The
// task holding a token's first chunk also writes row_of / src_of.
template <int kFmt, int kCols>
__global__ void __launch_bounds__(kScatterWarps * 32) dispatch_scatter_kernel(
    const uint16_t *__restrict__ x, int B, int H, int K, int N_phys, int layout, int cap,
    int cpt, DispatchWs ws, uint8_t *__restrict__ A, uint8_t *__restrict__ A_sf,
    int32_t *__restrict__ row_of, int32_t *__restrict__ src_of, uint8_t *__restrict__ As,
    uint8_t *__restrict__ As_sf) {
  constexpr bool kFp8 = kFmt != MOE_FMT_BF16;
  static_assert(kCols == 256 || (kFp8 && kCols == 512), "chunk width");
  constexpr int kPer = kCols / 32;    // columns per lane
  constexpr int kBlk = 128 / kPer;    // lanes per 128-column scale block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = (H + kCols - 1) / kCols;
  const int tpt = (nch + cpt - 1) / cpt;
  const long ntasks = (long)B * tpt;
  const long task = (long)blockIdx.x * kScatterWarps + warp;
  if (task >= ntasks) return;
  const int t = (int)(task / tpt);
  const int c0 = (int)(task % tpt) * cpt, c1 = min(nch, c0 + cpt);
  const int chunk = t / kChunk;
  int64_t my_row = -1;
  if (lane < K) {
    const int p = ws.phys[(size_t)t * K + lane];
    if (p >= 0) {
      const int slot = ws.hist[(size_t)chunk * N_phys + p] + ws.rank[(size_t)t * K + lane];
      if (layout == MOE_LAYOUT_CONTIG)
        my_row = (int64_t)ws.seg[p] + slot;
      else if (slot < cap)
        my_row = (int64_t)p * cap + slot;
    }
    if (c0 == 0) {
      row_of[(size_t)t * K + lane] = (int32_t)my_row;
      if (src_of && my_row >= 0) src_of[my_row] = t;
    }
  }
  int64_t rows[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) rows[k] = __shfl_sync(0xffffffffu, my_row, k);

  const uint16_t *xr = x + (size_t)t * H;
  const int Kg = sf_groups(H);
  for (int c = c0; c < c1; ++c) {
    const int h = c * kCols + kPer * lane;
    const bool act = h < H;
    uint4 v[kPer / 8];
#pragma unroll
    for (int i = 0; i < kPer / 8; ++i)
      v[i] = act ? __ldg(reinterpret_cast<const uint4 *>(xr + h + 8 * i)) : make_uint4(0, 0, 0, 0);
    if constexpr (!kFp8) {
      if (act) {
#pragma unroll
        for (int k = 0; k < 16; ++k)
          if (k < K && rows[k] >= 0)
            *reinterpret_cast<uint4 *>(A + ((size_t)rows[k] * H + h) * 2) = v[0];
      }
      continue;
    } else {
      float f[kPer];
#pragma unroll
      for (int i = 0; i < kPer / 8; ++i) {
        const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
          f[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
        }
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < kPer; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
      for (int off = kBlk / 2; off > 0; off >>= 1)  // the lanes of one 128-column block
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      uint32_t q[kPer / 4];
      uint8_t sfb = 0;
      float sf32 = 1.0f;
      if constexpr (kFmt == MOE_FMT_FP8) {  // power-of-two scale: an exact multiply
        const int e = ue8m0_exp(amax);
        const float inv = pow2i(-e);
#pragma unroll
        for (int i = 0; i < kPer / 4; ++i)
          q[i] = e4m3x2(__fmul_rn(f[4 * i], inv), __fmul_rn(f[4 * i + 1], inv)) |
                 (e4m3x2(__fmul_rn(f[4 * i + 2], inv), __fmul_rn(f[4 * i + 3], inv)) << 16);
        sfb = (uint8_t)(e + 127);
      } else {  // binary32 scale amax / 448 (1 when it is 0), IEEE divisions
        sf32 = __fdiv_rn(amax, 448.0f);
        if (sf32 == 0.0f) sf32 = 1.0f;
#pragma unroll
        for (int i = 0; i < kPer / 4; ++i)
          q[i] = e4m3x2(__fdiv_rn(f[4 * i], sf32), __fdiv_rn(f[4 * i + 1], sf32)) |
                 (e4m3x2(__fdiv_rn(f[4 * i + 2], sf32), __fdiv_rn(f[4 * i + 3], sf32)) << 16);
      }
      const int kb = h >> 7;
      auto put = [&](uint8_t *dst) {
        if constexpr (kPer == 8)
          *reinterpret_cast<uint2 *>(dst) = make_uint2(q[0], q[1]);
        else
          *reinterpret_cast<uint4 *>(dst) = make_uint4(q[0], q[1], q[2], q[3]);
      };
      if (act) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          if (k >= K || rows[k] < 0) continue;
          put(A + (size_t)rows[k] * H + h);
          if ((lane & (kBlk - 1)) == 0) {
            if constexpr (kFmt == MOE_FMT_FP8)
              A_sf[sf_byte_off(rows[k], kb, Kg)] = sfb;
            else
              reinterpret_cast<float *>(A_sf)[(size_t)rows[k] * (H / 128) + kb] = sf32;
          }
        }
        if (As) {
          put(As + (size_t)t * H + h);
          if ((lane & (kBlk - 1)) == 0) {
            if constexpr (kFmt == MOE_FMT_FP8)
              As_sf[sf_byte_off(t, kb, Kg)] = sfb;
            else
              reinterpret_cast<float *>(As_sf)[(size_t)t * (H / 128) + kb] = sf32;
          }
        }
      }
    }
  }
}

// Chunks per scatter task: enough warps for the whole GPU, at most a full row.
inline int scatter_cpt(int B, int H, int cols) {
  const long nch = (H + cols - 1) / cols;
  long cpt = ((long)B * nch) / ((long)device_sm_count() * 128);
  return (int)(cpt < 1 ? 1 : (cpt > nch ? nch : cpt));
}

// The count and scan launches of both dispatch entry points: one fused launch when
// the batch is a single chunk and the count's shared memory fits beside the scan's.
int launch_count_scan(const moe_dispatch_cfg *c, int B, int K, int Np, int nchunks,
                      const int32_t *topk_idx, const int32_t *log2phys, const int32_t *rep,
                      const DispatchWs &ws, int32_t *counts, int32_t *tiles, int32_t *src_of,
                      int32_t *shared_tiles, int32_t *status, cudaStream_t st) {
  const int max_rep = c->max_rep ? c->max_rep : 2;
  const size_t smem = sizeof(int32_t) * ((size_t)kCountWarps * Np + 2 * kChunk * K);
  if (nchunks == 1 && smem <= 24 * 1024) {
    dispatch_scan_kernel<<<1, kScanThreads, smem, st>>>(
        B, Np, nchunks, c->layout, c->cap, moe_dispatch_rows(c), ws, counts, tiles, src_of,
        shared_tiles, status, 1, topk_idx, log2phys, rep, max_rep, K, c->N_log);
    return check_launch();
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(dispatch_count_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  dispatch_count_kernel<<<nchunks, kCountWarps * 32, smem, st>>>(
      topk_idx, log2phys, rep, max_rep, B, K, c->N_log, Np, ws, status);
  int rc = check_launch();
  if (rc) return rc;
  dispatch_scan_kernel<<<1, kScanThreads, 0, st>>>(
      B, Np, nchunks, c->layout, c->cap, moe_dispatch_rows(c), ws, counts, tiles, src_of,
      shared_tiles, status, 0, nullptr, nullptr, nullptr, 0, 0, 0);
  return check_launch();
}

// The scatter launch of both dispatch entry points: fp8 rows in 512-column chunks
// (16-byte stores per lane and copy) when H allows, else 256.
int launch_scatter(const moe_dispatch_cfg *c, int B, int K, int Np, const void *x,
                   const DispatchWs &ws, void *A, void *A_sf, int32_t *row_of, int32_t *src_of,
                   void *As, void *As_sf, cudaStream_t st) {
  const uint16_t *xb = static_cast<const uint16_t *>(x);
  const bool fp8 = c->fmt != MOE_FMT_BF16;
  const int cols = fp8 && c->H % 512 == 0 ? 512 : 256;
  const int cpt = scatter_cpt(B, c->H, cols);
  const long tasks = (long)B * (((c->H + cols - 1) / cols + cpt - 1) / cpt);
  const unsigned grid = (unsigned)((tasks + kScatterWarps - 1) / kScatterWarps);
  uint8_t *a = static_cast<uint8_t *>(A), *asf = static_cast<uint8_t *>(A_sf);
  uint8_t *as = static_cast<uint8_t *>(As), *assf = static_cast<uint8_t *>(As_sf);
#define MOE_SCATTER(FMT, COLS)                                                         \
  dispatch_scatter_kernel<FMT, COLS><<<grid, kScatterWarps * 32, 0, st>>>(               \
      xb, B, c->H, K, Np, c->layout, c->cap, cpt, ws, a, asf, row_of, src_of, as, assf)
  if (!fp8)
    MOE_SCATTER(MOE_FMT_BF16, 256);
  else if (c->fmt == MOE_FMT_FP8 && cols == 512)
    MOE_SCATTER(MOE_FMT_FP8, 512);
  else if (c->fmt == MOE_FMT_FP8)
    MOE_SCATTER(MOE_FMT_FP8, 256);
  else if (cols == 512)
    MOE_SCATTER(MOE_FMT_FP8_F32, 512);
  else
    MOE_SCATTER(MOE_FMT_FP8_F32, 256);
#undef MOE_SCATTER
  return check_launch();
}

}  // namespace
}  // namespace moe

using namespace moe;

static int dispatch_check(const moe_dispatch_cfg *c) {
  if (!c) return MOE_ERR_INVALID;
  if (c->B < 0 || c->H <= 0 || c->K <= 0 || c->N_log <= 0 || c->N_phys <= 0)
    return MOE_ERR_INVALID;
  if (c->H % 128 || c->K > 16 || c->N_phys > kScanThreads) return MOE_ERR_UNSUPPORTED;
  if (c->layout != MOE_LAYOUT_CONTIG && c->layout != MOE_LAYOUT_MASKED) return MOE_ERR_INVALID;
  if (c->fmt != MOE_FMT_FP8 && c->fmt != MOE_FMT_BF16 && c->fmt != MOE_FMT_FP8_F32)
    return MOE_ERR_INVALID;
  if (c->layout == MOE_LAYOUT_MASKED && (c->cap <= 0 || c->cap % 128)) return MOE_ERR_UNSUPPORTED;
  if (c->max_rep < 0 || c->max_rep > 64) return MOE_ERR_INVALID;
  return MOE_OK;
}

extern "C" int64_t moe_dispatch_rows(const moe_dispatch_cfg *c) {
  if (dispatch_check(c)) return 0;
  if (c->layout == MOE_LAYOUT_MASKED) return (int64_t)c->N_phys * c->cap;
  return ((int64_t)c->B * c->K + (int64_t)c->N_phys * 127 + 127) / 128 * 128;
}

extern "C" int64_t moe_dispatch_max_tiles(const moe_dispatch_cfg *c) {
  return moe_dispatch_rows(c) / 128;
}

extern "C" size_t moe_dispatch_workspace_size(const moe_dispatch_cfg *c) {
  if (dispatch_check(c)) return 0;
  const size_t nchunks = (c->B + kChunk - 1) / kChunk;
  return 2 * align256(sizeof(int32_t) * (size_t)c->B * c->K) +
         align256(sizeof(int32_t) * nchunks * c->N_phys) +
         align256(sizeof(int32_t) * (c->N_phys + 1));
}

extern "C" int moe_dispatch(const moe_dispatch_cfg *c, const void *x, const int32_t *topk_idx,
                            const int32_t *log2phys, const int32_t *rep, void *A, void *A_sf,
                            int32_t *counts, int32_t *row_of, int32_t *src_of, int32_t *tiles,
                            void *A_shared, void *A_shared_sf, int32_t *shared_tiles,
                            void *workspace, size_t workspace_bytes, int32_t *status,
                            void *stream) {
  int rc = dispatch_check(c);
  if (rc) return rc;
  cudaStream_t st = as_stream(stream);
  const int B = c->B, K = c->K, Np = c->N_phys;
  if (!counts || !tiles) return MOE_ERR_INVALID;
  if (B == 0) {  // empty batch: no rows, no tiles, zero counts
    cudaError_t e = cudaMemsetAsync(tiles, 0, 8 * sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * Np, st);
    if (e == cudaSuccess && shared_tiles)
      e = cudaMemsetAsync(shared_tiles, 0, 8 * sizeof(int32_t), st);
    return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
  }
  if (!x || !topk_idx || !A || !row_of || !workspace) return MOE_ERR_INVALID;
  if (c->fmt != MOE_FMT_BF16 && !A_sf) return MOE_ERR_INVALID;
  if ((log2phys == nullptr) != (rep == nullptr)) return MOE_ERR_INVALID;
  if (A_shared && (c->fmt == MOE_FMT_BF16 || !A_shared_sf)) return MOE_ERR_INVALID;
  if (workspace_bytes < moe_dispatch_workspace_size(c)) return MOE_ERR_INVALID;
  if ((uintptr_t)x % 16 || (uintptr_t)A % 16 || (A_sf && (uintptr_t)A_sf % 16) ||
      (A_shared && (uintptr_t)A_shared % 16) || (uintptr_t)tiles % 16 ||
      (shared_tiles && (uintptr_t)shared_tiles % 16))
    return MOE_ERR_INVALID;
  const int nchunks = (B + kChunk - 1) / kChunk;
  DispatchWs ws = carve(workspace, B, K, Np);
  if ((rc = launch_count_scan(c, B, K, Np, nchunks, topk_idx, log2phys, rep, ws, counts, tiles,
                              src_of, shared_tiles, status, st)))
    return rc;
  return launch_scatter(c, B, K, Np, x, ws, A, A_sf, row_of, src_of, A_shared, A_shared_sf, st);
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the scratch of the three dispatch kernels lives in this
// file-scope device array instead of a caller-provided workspace.  Host code must
// not pass the symbol itself to a kernel (on the host it only names a stand-in);
// the device address is looked up once per device and cached.
static __device__ __align__(256) uint8_t g_dispatch_scratch[MOE_DISPATCH_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device (set up on first use).
int scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess || !p) return set_cuda_error(e != cudaSuccess ? e : cudaErrorUnknown);
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_dispatch_noalloc(const moe_dispatch_cfg *c, const void *x,
                                    const int32_t *topk_idx, const int32_t *log2phys,
                                    const int32_t *rep, void *A, void *A_sf, int32_t *counts,
                                    int32_t *row_of, int32_t *src_of, int32_t *tiles,
                                    void *A_shared, void *A_shared_sf, int32_t *shared_tiles,
                                    int32_t *status, void *stream) {
  int rc = dispatch_check(c);
  if (rc) return rc;
  const size_t need = moe_dispatch_workspace_size(c);
  if (need > MOE_DISPATCH_STATIC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  const int B = c->B, K = c->K, Np = c->N_phys;
  if (!counts || !tiles) return MOE_ERR_INVALID;
  if (B == 0) {
    cudaError_t e = cudaMemsetAsync(tiles, 0, 8 * sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * Np, st);
    if (e == cudaSuccess && shared_tiles)
      e = cudaMemsetAsync(shared_tiles, 0, 8 * sizeof(int32_t), st);
    return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
  }
  if (!x || !topk_idx || !A || !row_of) return MOE_ERR_INVALID;
  if (c->fmt != MOE_FMT_BF16 && !A_sf) return MOE_ERR_INVALID;
  if ((log2phys == nullptr) != (rep == nullptr)) return MOE_ERR_INVALID;
  if (A_shared && (c->fmt == MOE_FMT_BF16 || !A_shared_sf)) return MOE_ERR_INVALID;
  if ((uintptr_t)x % 16 || (uintptr_t)A % 16 || (A_sf && (uintptr_t)A_sf % 16) ||
      (A_shared && (uintptr_t)A_shared % 16) || (uintptr_t)tiles % 16 ||
      (shared_tiles && (uintptr_t)shared_tiles % 16))
    return MOE_ERR_INVALID;
  void *scratch = nullptr;
  if ((rc = scratch_address(&scratch))) return rc;
  const int nchunks = (B + kChunk - 1) / kChunk;
  DispatchWs ws = carve(scratch, B, K, Np);
  if ((rc = launch_count_scan(c, B, K, Np, nchunks, topk_idx, log2phys, rep, ws, counts, tiles,
                              src_of, shared_tiles, status, st)))
    return rc;
  return launch_scatter(c, B, K, Np, x, ws, A, A_sf, row_of, src_of, A_shared, A_shared_sf, st);
}
