// Shared device helpers of libmoe: status words, bf16 / e4m3 / UE8M0 conversions,
// the routing exp, and thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk)
// and the tcgen05 tensor-core / tensor-memory instructions of sm_100-class GPUs.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------------------ host side
int set_cuda_error(cudaError_t e);  // records e, returns MOE_ERR_CUDA
inline int check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : set_cuda_error(e);
}
inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }
int device_sm_count();
// One-time setup (kernel shared-memory limits, cluster occupancy) is kept per device:
// the current device's ordinal, or a negative MOE_ERR_* code.
constexpr int kMaxDevices = 64;
int device_slot();

// ---------------------------------------------------------------- status word
__device__ __forceinline__ void status_or(int32_t *st, int bits) {
  if (st) atomicOr(st, bits);
}

// ---------------------------------------------------------------------- bf16
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ---------------------------------------------------------------- powers of 2
// Exact 2^n as a binary32, -149 <= n <= 127.
__device__ __forceinline__ float pow2i(int n) {
  uint32_t u = n >= -126 ? (uint32_t)(n + 127) << 23 : 1u << (n + 149);
  return __uint_as_float(u);
}

// --------------------------------------------------------------- routing exp
// exp(x) by Cody-Waite reduction with a two-part ln 2 and the degree-7 Taylor
// polynomial of e^r in Horner form; every step is an explicitly rounded
// binary32 operation, so the result is a fixed function of x.
__device__ __forceinline__ float route_exp(float x) {
  if (x != x) return x;
  if (x > 88.72283172607421875f) return __uint_as_float(0x7f800000u);
  if (x < -103.97208404541015625f) return 0.0f;
  const float t = __fmul_rn(x, 1.44269502162933349609375f);
  const float nf = rintf(t);
  const int n = (int)nf;
  float r = __fmaf_rn(-nf, 0.693145751953125f, x);
  r = __fmaf_rn(-nf, 1.428606765330187045037746429443359375e-06f, r);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  if (n > 127) return __fmul_rn(__fmul_rn(p, pow2i(127)), pow2i(n - 127));
  if (n < -126) return __fmul_rn(__fmul_rn(p, pow2i(n + 126)), pow2i(-126));
  return __fmul_rn(p, pow2i(n));
}

__device__ __forceinline__ float route_sigmoid(float z) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, route_exp(-z)));
}

// ---------------------------------------------------------- e4m3 and UE8M0
// Smallest e with amax <= 448 * 2^e, clamped to [-127, 127]; 0 for amax == 0.
// From the bits: amax = 1.m * 2^(E-127); 448 = 1.75 * 2^8.
__device__ __forceinline__ int ue8m0_exp(float amax) {
  uint32_t b = __float_as_uint(amax) & 0x7fffffffu;
  if (b == 0) return 0;
  int e8 = (int)(b >> 23);
  uint32_t m = b & 0x7fffffu;
  if (e8 == 0) {  // subnormal: normalise the mantissa
    const int p = 31 - __clz((int)m);
    e8 = p - 22;
    m = (m << (23 - p)) & 0x7fffffu;
  }
  int e = (m <= 0x600000u) ? e8 - 135 : e8 - 134;
  return min(max(e, -127), 127);
}

// Two binary32 values -> two e4m3 codes (round to nearest even, saturating to
// +-448), `lo` in bits 0..7 and `hi` in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------ SF atoms
// Scale atoms: one 512-byte atom per (128-row block, group of four 128-column blocks);
// the byte of row r (0..127) for column block 4g + j sits at 16*(r%32) + 4*(r/32) + j.
// Kg = column-block groups per row.
__host__ __device__ __forceinline__ int sf_groups(int k) { return (k / 128 + 3) / 4; }
__device__ __forceinline__ size_t sf_byte_off(int64_t r, int kb, int Kg) {
  return ((size_t)(r >> 7) * Kg + (kb >> 2)) * 512 + 16 * (r & 31) + 4 * ((r & 127) >> 5) +
         (kb & 3);
}

// ------------------------------------------------------------- PTX: memory
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(int32_t *p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------------------------ PTX: mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up (returns
// false) when *abort becomes non-zero or after `limit_ns` of wall time.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          uint64_t limit_ns) {
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ----------------------------------------------------------------- PTX: TMA
__device__ __forceinline__ void tma_prefetch_desc(const void *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, uint32_t bar, int x,
                                            int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------- PTX: tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on this CTA's mbarrier once this thread's earlier tcgen05 operations are
// complete.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T with per-32-K block scales from TMEM.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem,
                                            uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> fp32, no block scaling.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Copy a 32-row x 16-byte matrix from shared memory to TMEM, replicated to all
// four 32-lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------ PTX: 2-CTA (cta_group::2) forms
// A CTA pair = the even and odd CTA of a 2-CTA cluster (one TPC).  The even CTA
// issues the pair's MMAs and scale copies; each operand comes from the shared memory
// of the CTA that owns it, at the same offset in both.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t cta_rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta_rank));
  return r;
}
// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for a barrier that other CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int *abort, uint64_t limit_ns) {
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}
// TMA tile load into this CTA's shared memory whose completion is counted on the
// mbarrier `cluster_bar` of either CTA of the pair (here: the even CTA's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *map,
                                                 uint32_t cluster_bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
      ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(map), "r"(cluster_bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// Collective over the pair: both CTAs' allocating warps execute these, and both get
// the same TMEM address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Scale atom copy issued by the even CTA: each CTA's shared memory -> its own TMEM.
__device__ __forceinline__ void tc_cp_pair_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Scale copy issued by the even CTA without replication: 128 rows of 16 bytes in each
// CTA's shared memory -> TMEM lanes 0-127 of its own TMEM (row r -> lane r).
__device__ __forceinline__ void tc_cp_pair_128x128b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.128x128b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// M = 256 block-scaled MMA over the pair: rows 0-127 from the even CTA's A tile,
// 128-255 from the odd CTA's; B columns 0-127 from the even CTA's B half, 128-255
// from the odd CTA's; each CTA's TMEM holds its rows' accumulator and scales.
__device__ __forceinline__ void tc_mma_pair_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t sfa_tmem,
                                                 uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
// Pair form of tc_commit: arrive on the mbarrier at this shared-memory offset in every
// CTA of cta_mask (an arrival, not a data transfer).
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

#define MOE_TMEM_LD_32x32b_X32(taddr, r)                                                       \
  asm volatile(                                                                                \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, " \
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, " \
      "%28, %29, %30, %31}, [%32];"                                                            \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),             \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),          \
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),          \
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),          \
        "=r"(r[31])                                                                            \
      : "r"(taddr))

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

}  // namespace moe
