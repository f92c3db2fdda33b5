/*
 * libmoe — single-GPU MoE layer hot path for GB300 (sm_103a).
 *
 * route -> (EPLB map) -> dispatch -> grouped FP8 gate/up + SwiGLU -> grouped FP8
 * down -> combine, each a C entry point over caller-owned device memory.
 *
 * The layer ("DeepEP 完全拆解", §专家并行): a router scores each of N experts for
 * every one of B tokens of hidden size H, keeps the top K, sends the token through
 * those K expert FFNs and sums the outputs weighted by the routing weights.  On
 * one GPU the EP all-to-all "dispatch" becomes a permutation of token rows inside
 * HBM, and the "combine" becomes a gather + weighted reduce back to token order.
 *
 * Conventions shared by every call
 *   - All pointers are device pointers unless a parameter says "host".  The
 *     caller allocates and owns all memory; no entry point allocates device
 *     memory.  Sizes of work buffers come from the *_workspace_size queries.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call only enqueues work; none synchronises the host, so sequences of
 *     calls can be captured into a CUDA graph.
 *   - Return value: MOE_OK, or a negative MOE_ERR_* detected on the host before
 *     anything is launched (MOE_ERR_INVALID: null pointer, bad size or
 *     alignment; MOE_ERR_UNSUPPORTED: a shape outside the supported range;
 *     MOE_ERR_CUDA: a CUDA launch or API error, the CUDA error is then available
 *     from moe_last_cuda_error()).
 *   - Errors found on the device are OR-ed into the caller's int32 `status` word
 *     (MOE_STATUS_* bits; sticky until the caller clears it).  moe_read_status()
 *     is the only call that waits for the device.
 *   - Calls run on the calling thread's current CUDA device.  The first call on a
 *     device raises the kernels' shared-memory limits and caches cluster
 *     occupancy for that device (up to 64 devices per process).
 *   - bf16 tensors are passed as void* and hold IEEE bfloat16 bit patterns.
 *   - e4m3 tensors hold OCP FP8 E4M3 ("e4m3fn") codes.  Scales are UE8M0
 *     bytes: value = 2^(byte - 127).
 *
 * Packed scale layout ("SF atoms").  Every FP8 operand of the grouped GEMM
 * carries its 1x128 (activation) or 128x128 (weight) block scales as 512-byte
 * atoms, one per (128-row block, group of four 128-column blocks).  Inside an atom,
 * the scale of row r (0..127 within the block) for column block 4g + j (j = 0..3)
 * sits at byte 16*(r%32) + 4*(r/32) + j; bytes for blocks past the last column block
 * are unused.  With Kg = ceil(k/512) groups, an activation tensor of `rows` rows and
 * `k` columns has atoms [rows/128][Kg][512] (moe_scale_bytes(rows, k) bytes); a
 * weight tensor of E experts x n rows x k columns has atoms [E][n/128][Kg][512]
 * (moe_packed_scale_bytes; all 32 rows' words of a weight atom are equal).
 *
 * Tile list.  moe_dispatch describes the rows it wrote as 128-row "M tiles" in
 * an int32 array `tiles` of 8 + 16*max_tiles entries:
 *   header tiles[0..7] = {M tiles, rows in use (contiguous layout), tile pairs,
 *   singles, work items, 0, 0, 0};
 *   tile i at tiles[8 + 8*i ...]: {first row, physical expert, valid rows (1..128),
 *   first tile of this expert, number of tiles of this expert, 0, 0, 0};
 *   work item k at tiles[8 + 8*max_tiles + 8*k ...]: {tile 0, tile 1 or -1, first
 *   item of its group, items in its group, 1 for a pair of one expert's tiles (0 for
 *   a single tile), 0, 0, 0}.  An expert's tiles form pairs two by two, and an odd
 *   last tile is a single; an expert's pairs and its single form one group.
 * Tiles of one expert are consecutive, and the experts' tiles and groups come in this
 *   order: the experts with two or more items spread evenly between the experts with
 *   one (multi-item expert i of nm, in expert order, before single-item expert
 *   floor((2i + 1) * n1 / (2 nm)) of n1), so CTAs running side by side mix weight tiles
 *   read once for several units with tiles read for one.  The rows themselves stay in
 *   expert order.  The grouped GEMM reads this list on the
 * device, so the host never needs the routing result.
 */
#ifndef LIBMOE_MOE_H
#define LIBMOE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID (-1)
#define MOE_ERR_UNSUPPORTED (-2)
#define MOE_ERR_CUDA (-3)

#define MOE_STATUS_CAPACITY 1  /* a masked-layout expert received more rows than cap */
#define MOE_STATUS_TIMEOUT 2   /* a bounded device-side wait gave up */
#define MOE_STATUS_BAD_INDEX 4 /* an expert index outside [0, N) reached dispatch */

#define MOE_SCORE_SOFTMAX 0
#define MOE_SCORE_SIGMOID 1
#define MOE_LAYOUT_CONTIG 0
#define MOE_LAYOUT_MASKED 1
#define MOE_FMT_FP8 0
#define MOE_FMT_BF16 1
#define MOE_FMT_FP8_F32 2 /* e4m3 with binary32 scales amax/448 per 1x128 block */
#define MOE_GEMM_GATEUP_SWIGLU 0
#define MOE_GEMM_DOWN 1

/* ------------------------------------------------------------------ route */
/*
 * Router ("DeepEP 完全拆解", §专家并行 and §group-limited gating).
 *   logits z[t][e] = sum_k x[t][k] * W[e][k], accumulated in fp32 by one fused
 *     multiply-add per k in order k = 0..H-1 (so results are reproducible bit
 *     for bit);
 *   score_fn SOFTMAX: choice score z; s = softmax(z) over all N (max-shifted,
 *     denominator summed in expert order);
 *   score_fn SIGMOID: s = 1/(1+exp(-z)); choice score c = s + bias (bias may be
 *     NULL = 0);  exp is the library's own Cody-Waite + degree-7 polynomial;
 *   n_group > 1: experts form n_group equal groups; a group scores the sum of
 *     its two best choice scores; the topk_group best groups stay eligible;
 *   top-K eligible experts by (choice score desc, index asc), stored in that
 *     order in topk_idx[t][0..K-1];
 *   topk_w = renorm ? s_k / (s_0+...+s_{K-1}) * route_scale : s_k * route_scale.
 *   expert_counts[e] (nullable) = number of (t,k) routed to e (overwritten).
 * Shapes: x bf16 [B][H], W fp32 [N][H], bias fp32 [N], topk_idx int32 [B][K],
 * topk_w fp32 [B][K].  Limits: H % 32 == 0, N <= 512, K <= 16, n_group <= 32,
 * N % n_group == 0 with at least 2 experts per group.
 */
typedef struct moe_route_cfg {
  int B, H, N, K;
  int n_group, topk_group;
  int score_fn;
  int renorm;
  float route_scale;
} moe_route_cfg;

size_t moe_route_workspace_size(const moe_route_cfg *cfg);
int moe_route(const moe_route_cfg *cfg, const void *x, const float *W, const float *bias,
              int32_t *topk_idx, float *topk_w, int32_t *expert_counts, void *workspace,
              size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------- EPLB */
/*
 * Redundant experts ("Large-scale EP: DeepEP, EPLB and two-batch overlap", §EPLB:
 * 256 logical experts in 288 physical slots, the popular ones copied).  HOST
 * function, deterministic: the N_phys - N_log hottest logical experts by
 * counts_host (ties -> lower index) get one replica each; the i-th hottest gets
 * physical id N_log + i.  Outputs (host arrays): log2phys [N_log][2] (column 0 =
 * e itself, column 1 = its replica or e), rep [N_log] (1 or 2), phys2log
 * [N_phys].  moe_dispatch then sends token t of logical expert e to
 * log2phys[e][t % rep[e]].  Returns MOE_ERR_INVALID unless 0 <= N_phys - N_log <= N_log.
 */
int eplb_build_map(const int64_t *counts_host, int N_log, int N_phys, int32_t *log2phys,
                   int32_t *rep, int32_t *phys2log);

/*
 * EPLB placement from recorded loads: DeepSeek's algorithm as the pages describe it
 * ("Large-scale EP: DeepEP, EPLB and two-batch overlap", §EPLB: hierarchical — the
 * expert groups are packed onto nodes first and the experts placed within each node,
 * so that one node's experts come from the same groups; rebalanced from measured
 * counts; "SGLang开源首个对标官方性能的DeepSeek-V3/R1 H100部署方案", §专家并行负载均衡器:
 * redundant slots hold extra copies of the most used experts, and cold experts
 * share a GPU with medium ones; balance = mean / max of the per-GPU load).  HOST
 * function, deterministic.
 *   load [N_log]: recorded tokens per logical expert, 0 <= load < 2^40.
 *   Groups: expert e belongs to group e / (N_log / n_group).  When n_nodes > 1 and
 *   n_group % n_nodes == 0 the plan is hierarchical: (1) the groups, heaviest
 *   first (ties -> lower group), each go to the lightest node that holds fewer than
 *   n_group / n_nodes groups (ties -> lower node); a node's experts are those of its
 *   groups in ascending order.  Otherwise all experts and GPUs form one node.
 *   (2) Within a node, every expert gets one slot and each remaining slot of the
 *   node (N_phys / nodes in all) goes, one at a time, to the expert with the largest
 *   load per replica, load[e] / rep[e], that has fewer than max_rep replicas (ties
 *   -> lower e).  (3) The node's replicas, each carrying load[e] / rep[e], are taken
 *   heaviest first (ties -> lower e) and each put on the lightest GPU of the node
 *   that has a free slot (ties -> lower GPU), N_phys / n_gpus slots per GPU.
 *   Outputs (host arrays): phys2log [N_phys] — slot j of GPU g is physical expert
 *   g * (N_phys / n_gpus) + j, filled in placement order; log2phys [N_log][max_rep]
 *   — e's physical experts ascending, the unused tail repeating the first; rep
 *   [N_log]; balance (nullable) — mean / max of the per-GPU loads (1 when all are 0).
 *   moe_dispatch sends token t of e to log2phys[e][t % rep[e]] (cfg->max_rep =
 *   max_rep).
 * Returns MOE_ERR_INVALID unless N_log >= 1, n_group >= 1, N_log % n_group == 0,
 * N_phys >= N_log, N_phys <= 8192, n_gpus % n_nodes == 0, N_phys % n_gpus == 0,
 * 1 <= max_rep <= 8, and each node's slots lie between its expert count and max_rep
 * times it.
 */
typedef struct moe_eplb_cfg {
  int N_log;    /* logical experts */
  int n_group;  /* expert groups (1: none) */
  int N_phys;   /* physical expert slots */
  int n_nodes;  /* nodes */
  int n_gpus;   /* GPUs in all */
  int max_rep;  /* replicas of one logical expert at most, 1..8 */
} moe_eplb_cfg;

int moe_eplb_plan(const moe_eplb_cfg *cfg, const int64_t *load, int32_t *phys2log,
                  int32_t *log2phys, int32_t *rep, double *balance);

/* --------------------------------------------------------------- dispatch */
/*
 * Dispatch ("Large-scale EP ...", §DeepEP: each mode where it belongs — the
 * contiguous layout after normal dispatch, the masked fixed-shape layout after
 * low-latency dispatch; "DeepEP 完全拆解", §通信量: each token sent once per
 * chosen expert, FP8 with s = 1 byte).
 *   Rows of one physical expert are taken in ascending (t, k) order.
 *   CONTIG: expert p's segment starts at sum_{q<p} roundup128(count_q); rows
 *     past a segment's count are padding and are never written or read back.
 *   MASKED: expert p's slot j is row p*cap + j; rows with j >= cap are dropped
 *     (row_of = -1, MOE_STATUS_CAPACITY set); cap is a multiple of 128.
 *   FP8: each token row is quantised once in 1x128 blocks — block exponent
 *     e = smallest integer with amax <= 448*2^e (amax == 0 -> 0, clamped to
 *     [-127,127]), code = e4m3_rne_satfinite(x * 2^-e) — and copied to its K
 *     rows of A [rows][H]; the exponents go to A_sf as SF atoms.
 *   FP8_F32: the same rows with binary32 scales ("Single Batch Overlap (SBO)" PR,
 *     §3, 1d2d scaling with float scales): s = amax / 448 per 1x128 block (one IEEE
 *     division; 1 when it is 0), code = e4m3_rne_satfinite(x / s) (IEEE division);
 *     A_sf is float [rows][H/128] (A_shared_sf likewise).
 *   BF16: rows are copied unchanged (A is bf16 [rows][H], A_sf unused).
 *   log2phys [N_log][max_rep] / rep [N_log] (nullable, EPLB) map logical to
 *     physical experts: token t of e goes to log2phys[e][t % rep[e]], and a
 *     rep[e] outside [1, max_rep] or a physical id outside [0, N_phys) sets
 *     MOE_STATUS_BAD_INDEX and drops the pair.
 *   counts [N_phys]: rows routed to each physical expert (before capacity).
 *   row_of [B][K]: A row of (t,k); src_of [rows] (nullable): token of each row,
 *     -1 for padding / empty slots.  tiles: see the tile list above.
 *   A_shared (nullable, FP8 only): the same quantised rows in token order,
 *     [roundup128(B)][H] + SF atoms A_shared_sf, and its tile list shared_tiles
 *     (one expert, id 0) for a shared expert.
 *   status: device int32, MOE_STATUS_* bits OR-ed in.
 * Limits: H % 128 == 0, K <= 16, N_phys <= 1024, rows as returned by
 * moe_dispatch_rows(); x, A, A_sf, A_shared, tiles and shared_tiles 16-byte aligned
 * (else MOE_ERR_INVALID).
 */
typedef struct moe_dispatch_cfg {
  int B, H, K;
  int N_log, N_phys;
  int layout;
  int cap;
  int fmt;
  int max_rep; /* columns of log2phys (0: 2, the eplb_build_map layout), at most 64 */
} moe_dispatch_cfg;

int64_t moe_dispatch_rows(const moe_dispatch_cfg *cfg);      /* rows of A to allocate */
int64_t moe_dispatch_max_tiles(const moe_dispatch_cfg *cfg); /* M tiles in `tiles` */
size_t moe_dispatch_workspace_size(const moe_dispatch_cfg *cfg);
int moe_dispatch(const moe_dispatch_cfg *cfg, const void *x, const int32_t *topk_idx,
                 const int32_t *log2phys, const int32_t *rep, void *A, void *A_sf,
                 int32_t *counts, int32_t *row_of, int32_t *src_of, int32_t *tiles,
                 void *A_shared, void *A_shared_sf, int32_t *shared_tiles, void *workspace,
                 size_t workspace_bytes, int32_t *status, void *stream);

/* Int32 entries of a tile list with room for max_tiles M tiles. */
#define MOE_TILE_LIST_INTS(max_tiles) (8 + 16 * (max_tiles))

/*
 * moe_dispatch for callers that cannot allocate device memory.  (The pages have
 * no counterpart of this entry point; it exists for library users.)
 *
 * Some callers cannot call cudaMalloc at all or at the point where they dispatch:
 * a host framework that owns every byte of device memory through its own
 * pre-reserved pool, a code path that must never make the device synchronise
 * (cudaMalloc and cudaFree may), or a plugin host that forbids allocation while
 * it runs.  This variant takes the same arguments as moe_dispatch except the
 * workspace: its scratch lives in a fixed device array inside this library,
 * MOE_DISPATCH_STATIC_SCRATCH_BYTES (4 MiB) large, which every GPU that loads
 * the library keeps until the process exits.  It allocates nothing.
 *   - A configuration whose workspace (moe_dispatch_workspace_size) exceeds that
 *     size is rejected with MOE_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on each device looks up the array's device address (a
 *     one-time set-up on the then-current device); make that first call before
 *     any stream capture on the device.
 *   - All calls share the one array, and it keeps whatever the last call left:
 *     nothing in it needs to start at zero (every scratch word is written before
 *     it is read within a call), but two calls whose work overlaps on the GPU (on
 *     different streams without ordering between them) race on it and give wrong
 *     results.  Order such calls on one stream or with events.
 */
#define MOE_DISPATCH_STATIC_SCRATCH_BYTES (4u << 20)
int moe_dispatch_noalloc(const moe_dispatch_cfg *cfg, const void *x, const int32_t *topk_idx,
                         const int32_t *log2phys, const int32_t *rep, void *A, void *A_sf,
                         int32_t *counts, int32_t *row_of, int32_t *src_of, int32_t *tiles,
                         void *A_shared, void *A_shared_sf, int32_t *shared_tiles,
                         int32_t *status, void *stream);

/* ------------------------------------------------------------ grouped GEMM */
/*
 * Fused combine for the DOWN GEMM: the expert outputs are reduced back to token order
 * inside the GEMM that makes them ("DeepEP 完全拆解", §为什么 combine 比 dispatch 慢:
 * combine moves and reduces; here the reduce rides in the producing kernel instead of
 * a separate pass over Y).  The result is that of moe_combine, bit for bit: the sum
 * of a token's rows is still formed by one warp in the rank order k = 0..K-1, in fp32,
 * then the shared row added, then rounded to bf16.  What changes is who forms it and
 * when: every warp of the GEMM that stores rows of Y counts them off per (token,
 * 128-column chunk) (an atomic subtraction on `pending`, after a gpu-scope fence of its
 * stores), and the warp that brings a chunk's count to zero -- it stored the token's
 * last row of that chunk -- reduces the chunk right away, reading the other rows
 * through L2.  No warp waits for another.
 *   row_of, topk_w [B][K]: as for moe_combine (row_of < 0: rank left out).
 *   src_of [src_rows]: token of each routed row of Y (moe_dispatch's src_of).
 *   pending int32 [B][n/128]: initialised by moe_fused_combine_prep before each GEMM.
 *   shared_row0: row of Y holding token 0's shared-expert row (token t at
 *     shared_row0 + t), or -1 without a shared expert.
 *   out bf16 [B][n].
 * Limits: 1 <= K <= 16.
 */
typedef struct moe_fused_combine {
  int B, K;
  const int32_t *row_of;
  const float *topk_w;
  const int32_t *src_of;
  int64_t src_rows;
  int32_t *pending;
  int64_t shared_row0;
  void *out;
} moe_fused_combine;

/* Sets pending[t][c] for the fused combine of an n-column DOWN GEMM (twice the rows the
   token has in Y: its ranks with row_of >= 0, plus its shared row) and writes zeros to
   out[t] for a token that has no row at all (moe_combine's result for it).  Enqueued on
   `stream` after the dispatch that wrote row_of and before the GEMM.  Reads row_of and
   shared_row0 of fc (shared_row0 < 0: no shared row); B = 0 enqueues nothing.  Errors,
   before any launch: fc NULL, B < 0, K < 1, n <= 0, or (B > 0) row_of, pending or out
   NULL or out not 16-byte aligned: MOE_ERR_INVALID; K > 16 or n not a multiple of 256:
   MOE_ERR_UNSUPPORTED. */
int moe_fused_combine_prep(const moe_fused_combine *fc, int n, void *stream);

/*
 * Grouped FP8 GEMM over the M tiles of a tile list (DeepGEMM's contiguous and
 * masked grouped GEMMs, "Large-scale EP ...", §DeepEP; FP8 1x128 x 128x128
 * "1d2d" scaling, "Single Batch Overlap (SBO)" PR, §3), on tcgen05 tensor
 * cores with TMEM accumulators, operands fed by TMA.
 *   acc[r][j] = sum_k a[r][k] * w[j][k] with a = e4m3(A)*2^(sfA-127) per 1x128
 *   block and w = e4m3(W)*2^(sfW-127) per 128x128 block, fp32 accumulation.
 *   GATEUP_SWIGLU: W [E][n][k] with n = 2I, rows [0,I) gate and [I,2I) up;
 *     h = silu(g) * u in fp32, quantised per 1x128 block exactly as dispatch
 *     quantises x; out = e4m3 [rows][I], out_sf = SF atoms [rows/128][ceil(I/512)][512].
 *   DOWN: W [E][n][k] with n = H, k = I; out = bf16 [rows][n] (round to nearest
 *     even).  signal (nullable): after the tile (rows R..R+127, any 256 output
 *     columns) is stored, signal[(R + j) / block_m_signal] += 1 (release, gpu
 *     scope) for every block j*block_m_signal of the tile; a row block is
 *     complete when its count reaches n / 256.
 *   The weight expert of physical expert p is phys2log[p] (nullable = p), so
 *   EPLB replicas read the same weights.  Rows past a tile's valid count are
 *   computed but never stored.
 *   W_sf: SF atoms from moe_pack_weight_scales.
 *   tiles2 (nullable): tiles of a second group, e.g. a shared expert whose rows
 *     sit at row_offset2 in A/out and whose weights are expert expert2 of W; its
 *     tiles join the same persistent grid (scheduled before those of `tiles`); its
 *     capacity is its own tile count (as moe_dispatch writes a shared tile list).
 *   num_sms: CTAs of the persistent grid (0 = every SM).
 * Limits: k % 128 == 0, n % 256 == 0, 16-byte aligned pointers.
 */
typedef struct moe_gemm_args {
  int op;
  int n, k;
  int64_t rows;      /* rows of A and out */
  int64_t max_tiles; /* capacity of the tile list */
  int num_experts;   /* experts in W */
  const void *A;
  const void *A_sf;
  const void *W;
  const void *W_sf;
  const int32_t *phys2log;
  const int32_t *tiles;
  const int32_t *tiles2; /* nullable: a second tile list computed in the same launch */
  int64_t row_offset2;   /* added to every row of tiles2 (A and out rows) */
  int expert2;           /* weight expert of every tile of tiles2 (phys2log unused) */
  void *out;
  void *out_sf;
  int32_t *signal;
  int block_m_signal;
  int num_sms;
  int pair_tiles; /* 0: one CTA per M tile (128x256 MMAs).
                     1: CTA pairs on one TPC share each weight tile, half of it in
                        each SM: an expert's tile pairs run as M = 256 pair MMAs and its
                        single tile, in the same launch, as an M = 128 pair MMA (up to 64
                        valid rows) or an M = 256 one with the second half idle; needs
                        k % 256 == 0 (else MOE_ERR_UNSUPPORTED).
                     Other values: MOE_ERR_INVALID.  Both give the same bytes. */
  int scale_fmt;  /* 0: UE8M0 scales as SF atoms, applied by the tensor core (block
                     scaling).  1: binary32 scales (1d2d with float scales, "Single Batch
                     Overlap (SBO)" PR, §3): A_sf float [rows][k/128], W_sf float
                     [E][n/128][k/128] (moe_weight_scales_f32), out_sf (GATEUP) float
                     [rows][I/128] with h's scales amax/448 and codes e4m3(h / s); each
                     128-deep k-block's product is formed unscaled and promoted by
                     acc += (s_a * s_w) * partial in fp32, k-blocks in order.  Needs
                     pair_tiles == 0 (else MOE_ERR_UNSUPPORTED).  Other values:
                     MOE_ERR_INVALID. */
  int32_t *status;
  const moe_fused_combine *combine; /* nullable; DOWN only, and not with signal (else
                                       MOE_ERR_INVALID): reduce Y into combine->out as
                                       the rows are stored (see moe_fused_combine) */
  int tile_n; /* output columns per tile: 0 or 256; or 224 (DOWN only, UE8M0 scales, no
                 signal or combine, else MOE_ERR_INVALID; n % 224 == 0, else
                 MOE_ERR_UNSUPPORTED): two 224-column accumulators in TMEM, so a unit's
                 MMAs overlap the previous unit's epilogue, with W_sf from
                 moe_pack_weight_scales_tiled (tile_n 224); with pair_tiles 1 every tile
                 runs at M = 256.  The same bytes either way. */
} moe_gemm_args;

int moe_grouped_gemm_fp8(const moe_gemm_args *args, void *stream);

/*
 * Weight scales (UE8M0 bytes W_sf [E][n/128][k/128], one per 128x128 block as in the
 * "1d2d" scaling of the "Single Batch Overlap (SBO)" PR, §3) -> SF atoms
 * [E][n/128][ceil(k/512)][512] (moe_packed_scale_bytes bytes; 0 when E, n or k is not
 * positive or n or k not a multiple of 128).  One-time setup, off the hot path.
 */
size_t moe_packed_scale_bytes(int E, int n, int k);
/* Weight scales of tile_n-row weight tiles (128 < tile_n <= 256, tile_n % 16 == 0,
   n % tile_n == 0; 0 otherwise): per (expert, tile, group of four k-blocks) two 128-row
   images in the SF atom layout, image h holding the tile's rows [128h, 128h + 128), each
   row with its own 128x128 block's scale (rows past tile_n zero):
   [E][n/tile_n][ceil(k/512)][2][512] bytes.  The DOWN GEMM with tile_n 224 reads them.  One-time setup, off the hot path. */
size_t moe_tiled_scale_bytes(int E, int n, int k, int tile_n);
/* Errors, before any launch: a shape moe_tiled_scale_bytes rejects (0 bytes), W_sf or
   W_sf_tiled NULL, or W_sf_tiled not 16-byte aligned: MOE_ERR_INVALID. */
int moe_pack_weight_scales_tiled(int E, int n, int k, int tile_n, const uint8_t *W_sf,
                                 void *W_sf_tiled, void *stream);
/* Weight scales for scale_fmt 1: UE8M0 bytes W_sf [E][n/128][k/128] -> float
   2^(byte - 127), same shape (exact).  One-time setup, off the hot path.  E, n or k
   not positive, n or k not a multiple of 128, or a NULL pointer: MOE_ERR_INVALID. */
int moe_weight_scales_f32(int E, int n, int k, const uint8_t *W_sf, float *W_sf_f32,
                          void *stream);
/* Bytes of the scales of an activation tensor of `rows` rows and k columns (rows and k
   multiples of 128; 0 otherwise) in format fmt: MOE_FMT_FP8, SF atoms, rows/128 *
   ceil(k/512) * 512; MOE_FMT_FP8_F32, float [rows][k/128], rows * k/128 * 4. */
size_t moe_scale_bytes(int64_t rows, int k, int fmt);
/* W_sf -> SF atoms (above).  Errors, before any launch: a shape moe_packed_scale_bytes
   rejects (0 bytes), W_sf or W_sf_packed NULL, or W_sf_packed not 16-byte aligned:
   MOE_ERR_INVALID. */
int moe_pack_weight_scales(int E, int n, int k, const uint8_t *W_sf, void *W_sf_packed,
                           void *stream);

/* ----------------------------------------------------------------- combine */
/*
 * Combine ("DeepEP 完全拆解", §专家并行 and §为什么 combine 比 dispatch 慢: move
 * the expert outputs back and reduce them with the routing weights):
 *   acc = 0; for k = 0..K-1: if row_of[t][k] >= 0: acc = fma(topk_w[t][k],
 *   Y[row_of[t][k]], acc); if shared: acc += shared[t]; out[t] = bf16(acc)
 * in fp32, fixed k order (deterministic).  Y bf16 [rows][H], shared bf16 [B][H]
 * (nullable), out bf16 [B][H].
 * Single-batch overlap ("Single Batch Overlap (SBO)" PR, §2): with signal
 * non-NULL, the row r of (t,k) is read only after signal[r / block_m_signal]
 * reaches threshold (acquire load, polled); a poll that lasts longer than
 * timeout_ns gives up, sets MOE_STATUS_TIMEOUT and skips the row (the shared row
 * likewise, see shared_row0).  num_ctas bounds the grid (0 = as many warps as the
 * work splits into); a small grid on its own stream runs beside the producing GEMM.
 * Limits: H % 256 == 0, K <= 16.
 */
typedef struct moe_combine_cfg {
  int B, H, K;
  const int32_t *signal;
  int threshold;
  int block_m_signal;
  int64_t timeout_ns;
  int num_ctas;
  int64_t shared_row0; /* with signal and shared: row (in the signal's row space) of
                          shared[0]; shared[t] is read after signal[(shared_row0 + t) /
                          block_m_signal] reaches threshold */
} moe_combine_cfg;

int moe_combine(const moe_combine_cfg *cfg, const void *Y, const int32_t *row_of,
                const float *topk_w, const void *shared, void *out, int32_t *status,
                void *stream);

/* ------------------------------------------------------------------ status */
/* Copies the device status word to *host_status (synchronous). */
int moe_read_status(const int32_t *status, int32_t *host_status);
/* The last CUDA error an entry point saw (cudaError_t as int). */
int moe_last_cuda_error(void);
/* SM count of the current device. */
int moe_num_sms(void);

/* ------------------------------------------------------------------- layer */
/*
 * The whole layer as one call ("DeepEP 完全拆解", §专家并行: route, send each token
 * to its K experts, run them, weighted sum back): route -> dispatch -> gate/up ->
 * down -> combine, every buffer caller-owned (see the fields).
 * Shared expert (has_shared != 0): its weights are the last expert (index N) of
 * W13 / W13_sf / W2 / W2_sf, which then hold N + 1 experts; its rows (the batch in
 * token order, roundup128(B) rows) follow the `rows` routed rows in A, A_sf, H1,
 * H1_sf and Y, and its tiles (shared_tiles) run inside the routed GEMM launches.
 * With sbo != 0 (masked layout; "Single Batch Overlap (SBO)" PR, §2) the down GEMM
 * publishes per-block signals and the combine runs on stream2 beside it, polling them; stream2 must be a stream
 * other than `stream` (the call orders it after the work before the down GEMM
 * and makes `stream` wait for the combine).
 * moe_layer_forward_host additionally copies x from host memory (pinned for
 * asynchronous copies) to layer->x before, and out to host memory after, all on
 * `stream`; it returns once the work is enqueued.
 */
typedef struct moe_layer {
  moe_route_cfg route;
  int N_phys, layout, cap, I, has_shared, sbo, block_m_signal;
  int64_t rows, max_tiles, timeout_ns; /* rows, max_tiles: at least moe_dispatch_rows and
                                           moe_dispatch_max_tiles of the layer's dispatch
                                           (else MOE_ERR_INVALID before any launch) */
  int num_sms;      /* CTAs of the persistent GEMM grids (0: every SM) */
  int combine_ctas; /* sbo: CTAs of the combine consumer, taken from num_sms for the down
                       GEMM while they run beside it (0: 32; at least one SM must stay
                       for the GEMM, else MOE_ERR_INVALID) */
  int gemm_pairs; /* CTA pairs (pair_tiles 1) for the GEMMs.  0: the gate/up GEMM on
                     pairs when B*K >= 256*N_phys (two M tiles per expert on average) and
                     H and I are multiples of 256, the down GEMM on one CTA per tile; 1:
                     both GEMMs on pairs (MOE_ERR_UNSUPPORTED unless H and I are multiples
                     of 256); -1: both on one CTA per tile; other values: MOE_ERR_INVALID */
  /* inputs and weights */
  void *x;                                         /* bf16 [B][H] */
  const float *W_router, *bias;                    /* [N][H], [N] or NULL */
  const int32_t *log2phys, *rep, *phys2log;        /* EPLB map or NULL */
  const void *W13, *W13_sf, *W2, *W2_sf;           /* e4m3 + SF atoms, N (+1) experts */
  /* outputs and intermediates; row buffers hold rows (+ roundup128(B)) rows */
  int32_t *topk_idx;
  float *topk_w;
  int32_t *expert_counts, *counts, *row_of, *tiles, *shared_tiles;
  int32_t *signal; /* sbo: (rows + shared rows) / block_m_signal counters */
  void *A, *A_sf, *H1, *H1_sf, *Y;
  void *out;
  void *route_ws, *dispatch_ws;
  size_t route_ws_bytes, dispatch_ws_bytes;
  int32_t *status;
  void *stream2;
  /* nullable: MOE_LAYER_EVENTS cudaEvent_t handles, recorded on `stream` at the
     stage boundaries (start, after route, dispatch, gate/up, down, combine) so a
     caller can time each stage of the chain. */
  void *const *events;
  int eplb_max_rep; /* columns of log2phys (0: 2) */
  int scale_fmt;    /* 0: UE8M0 scales (W13_sf / W2_sf as SF atoms, A_sf / H1_sf as SF
                       atoms); 1: binary32 scales (W13_sf / W2_sf float [E][n/128][k/128],
                       A_sf / H1_sf float [rows][k/128]; both GEMMs on one CTA per tile,
                       so gemm_pairs 1 is MOE_ERR_UNSUPPORTED) */
  int fuse_combine; /* 1: the down GEMM reduces Y into out itself (moe_fused_combine; the
                       same bytes as the separate combine); needs src_of and pending, and
                       sbo == 0 (else MOE_ERR_INVALID) */
  int32_t *src_of;  /* fuse_combine: int32 [rows], the token of each routed row */
  int32_t *pending; /* fuse_combine: int32 [B][H/128] */
  const void *W2_sf_t224; /* nullable: W2's scales as moe_pack_weight_scales_tiled images
                             (tile_n 224); with them the down GEMM runs on 224-column
                             tiles (moe_gemm_args.tile_n 224), unless fuse_combine or sbo */
} moe_layer;

#define MOE_LAYER_EVENTS 6

int moe_layer_forward(const moe_layer *layer, void *stream);
int moe_layer_forward_host(const moe_layer *layer, const void *x_host, void *out_host,
                           void *stream);

/*
 * n_steps layer passes over host batches, the copies overlapped with the kernels
 * ("Large-scale EP ...", §TBO: hide data movement behind the other batch's
 * computation, here the host<->device copies of neighbouring steps): step i copies
 * x_host[i] (pinned, bf16 [B][H]) in, runs the layer and copies out to out_host[i]
 * (pinned).  Device input and output buffers alternate between layer->x / layer->out
 * (even steps) and x2 / out2 (odd steps; same sizes, caller-owned).  The copies run on
 * copy_stream (a created stream other than `stream`): step i+1's input is copied
 * while step i computes, step i's output while step i+1 computes; events order a
 * buffer's reuse after its last reader.  On return everything is enqueued and
 * `stream` waits for the last copy, so work or an event recorded on `stream`
 * afterwards follows all n steps.  x_host / out_host entries may repeat (copies to
 * one host buffer are ordered on copy_stream).
 * Errors: MOE_ERR_INVALID for NULL arguments, n_steps < 1, or copy_stream equal to
 * stream; a failing layer call returns its code (work already enqueued stays).
 */
int moe_layer_forward_host_pipelined(const moe_layer *layer, void *x2, void *out2,
                                     const void *const *x_host, void *const *out_host,
                                     int n_steps, void *stream, void *copy_stream);

/*
 * Whole-layer CUDA graph ("Large-scale EP: DeepEP, EPLB and two-batch overlap",
 * §DeepEP: each mode where it belongs -- the fixed-shape low-latency path is the
 * one decode replays as a CUDA graph to keep launch overhead off each step).
 *
 * moe_layer_graph_create captures one moe_layer_forward of L (or, with x_host and
 * out_host both non-NULL, one moe_layer_forward_host: the copies are part of the
 * graph, so the host buffers must be pinned) on `stream` and instantiates it into
 * *graph.  `stream` must be a created stream, not the legacy default stream.  The
 * graph keeps every pointer of L and of the host buffers as they were at capture:
 * launch it only while they stay valid and unchanged; the stage events of L, if any,
 * are recorded at every replay.  Run the layer once eagerly before capturing (first calls
 * set kernel attributes).  moe_layer_graph_launch replays it on `stream` (no host
 * synchronisation); moe_layer_graph_destroy frees it (NULL is a no-op).
 * Errors: MOE_ERR_INVALID for NULL L / graph / stream or only one host buffer; a
 * failing layer call or capture returns its code and leaves *graph NULL.
 */
int moe_layer_graph_create(const moe_layer *L, const void *x_host, void *out_host, void *stream,
                           void **graph);
int moe_layer_graph_launch(void *graph, void *stream);
int moe_layer_graph_destroy(void *graph);

#ifdef __cplusplus
}
#endif
#endif /* LIBMOE_MOE_H */
