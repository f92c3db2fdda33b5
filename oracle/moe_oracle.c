/*
 * CPU oracle for the MoE layer hot path: route -> EPLB map -> dispatch ->
 * (expert FFN, in oracle/ffn.py) -> combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code with the CUDA library.
 *
 * Plain, slow, token-by-token C99 in strict IEEE single precision: compile with
 * -O2 -ffp-contract=off and no fast-math; every fused multiply-add is an explicit
 * fmaf().  Sources of each definition:
 *   MoE layer (router scores N experts, top-K, K expert FFNs, weighted sum):
 *       "DeepEP 完全拆解", §专家并行 (B, N, K, H notation).
 *   Group-limited gating (top groups first, then top-K inside them):
 *       "DeepEP 完全拆解", §group-limited gating.
 *   Redundant experts, logical -> physical (256 -> 288 slots, hot ones copied):
 *       "Large-scale EP: DeepEP, EPLB and two-batch overlap", §EPLB.
 *   Contiguous (per-expert segments) vs masked (fixed capacity) layouts:
 *       same page, §DeepEP: each mode where it belongs.
 *   1x128 activation / 128x128 weight FP8 scaling ("1d2d"):
 *       "Single Batch Overlap (SBO)" PR, §3 Modifications.
 * Readings where the pages are silent (sigmoid + bias scoring, top-2-sum group
 * score, UE8M0 power-of-two scales, tie-breaks, summation orders) are stated at
 * each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ bf16 */

float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest-even from binary32 to bfloat16 (keep the top 16 bits). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN stays a (quiet) NaN */
        return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------ exp, sigmoid */
/*
 * exp in binary32 by Cody-Waite argument reduction (W. J. Cody and W. Waite,
 * "Software Manual for the Elementary Functions", 1980) followed by the degree-7
 * Taylor polynomial of e^r, evaluated by Horner's rule with fmaf:
 *   n = rint(x * log2(e));  r = (x - n*L1) - n*L2  (L1 + L2 = ln 2, L1 short);
 *   p = sum_{i=0..7} r^i / i!;  exp(x) = p * 2^n.
 * |r| <= ln(2)/2 + tiny, so the truncation error is below 1e-8 relative.
 * The GPU routing kernel evaluates the same operations in the same order, so
 * both produce identical bits; only the mathematics is shared, not code.
 */
static const float EXP_LOG2E = 1.44269502162933349609375f;   /* 0x3FB8AA3B */
static const float EXP_L1 = 0.693145751953125f;              /* 0x3F317200 */
static const float EXP_L2 = 1.428606765330187045037746429443359375e-06f; /* 0x35BFBE8E */
static const float EXP_HI = 88.72283172607421875f;
static const float EXP_LO = -103.97208404541015625f;

static float pow2i(int n) /* exact 2^n for -149 <= n <= 127 */
{
    uint32_t u;
    if (n >= -126)
        u = (uint32_t)(n + 127) << 23;
    else
        u = 1u << (n + 149);
    float f;
    memcpy(&f, &u, 4);
    return f;
}

float oracle_exp(float x)
{
    if (x != x)
        return x;
    if (x > EXP_HI)
        return INFINITY;
    if (x < EXP_LO)
        return 0.0f;
    float t = x * EXP_LOG2E;
    float nf = rintf(t);
    int n = (int)nf;
    float r = fmaf(-nf, EXP_L1, x);
    r = fmaf(-nf, EXP_L2, r);
    /* 1/7! .. 1/2!, each rounded to the nearest binary32 */
    float p = 0x1.a01a02p-13f;
    p = fmaf(p, r, 0x1.6c16c2p-10f);
    p = fmaf(p, r, 0x1.111112p-7f);
    p = fmaf(p, r, 0x1.555556p-5f);
    p = fmaf(p, r, 0x1.555556p-3f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    if (n > 127)
        return (p * pow2i(127)) * pow2i(n - 127);
    if (n < -126)
        return (p * pow2i(n + 126)) * pow2i(-126);
    return p * pow2i(n);
}

/* sigma(z) = 1 / (1 + e^{-z}), one rounding per operation. */
float oracle_sigmoid(float z)
{
    float e = oracle_exp(-z);
    return 1.0f / (1.0f + e);
}

/* ------------------------------------------------------------------- e4m3 */
/*
 * OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8; smallest
 * normal 2^-6; subnormals m * 2^-9, m = 1..7.
 */
float oracle_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    float v = (e == 0) ? (float)m * pow2i(-9) : (1.0f + (float)m / 8.0f) * pow2i(e - 7);
    return s ? -v : v;
}

/*
 * Round to nearest, ties to even, saturating finite values to +-448.
 * Written from the definition: find the binade of |v| (the subnormal range
 * shares the quantum of the lowest normal binade), round |v| / quantum to an
 * integer with ties-to-even, and re-encode.  A round-up into the next binade
 * is handled by the re-encoding of the rounded value.
 */
uint8_t oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (v != v)
        return sign | 0x7f;
    float a = fabsf(v);
    if (a >= 448.0f) /* satfinite (includes +-inf) */
        return sign | 0x7e;
    if (a == 0.0f)
        return sign;
    int E;
    frexpf(a, &E);          /* a = f * 2^E, f in [0.5, 1): floor(log2 a) = E - 1 */
    int eb = E - 1;
    if (eb < -6)
        eb = -6;
    float q = pow2i(eb - 3); /* spacing of representable values in this binade */
    float nq = rintf(a / q); /* exact quotient, RNE to an integer */
    float val = nq * q;      /* exact */
    if (val == 0.0f)
        return sign;
    if (val > 448.0f)
        val = 448.0f;
    frexpf(val, &E);
    eb = E - 1;
    if (eb < -6) /* subnormal: val = m * 2^-9 */
        return sign | (uint8_t)(val / pow2i(-9));
    int mant = (int)((val / pow2i(eb) - 1.0f) * 8.0f);
    return sign | (uint8_t)(((eb + 7) << 3) | mant);
}

/*
 * UE8M0 block scale for an amax: the smallest power of two 2^e with
 * amax <= 448 * 2^e (so amax / 2^e fits e4m3 without saturating), clamped to the
 * UE8M0 range e in [-127, 127]; amax == 0 gives e = 0.  Computed exactly from
 * frexp: amax = f * 2^E with f in [0.5, 1) and 448 = 0.875 * 2^9.
 */
int oracle_scale_exp(float amax)
{
    if (amax == 0.0f)
        return 0;
    int E;
    float f = frexpf(amax, &E);
    int e = (f <= 0.875f) ? E - 9 : E - 8;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/*
 * Quantise one row of n values (n a multiple of 128) in 1x128 blocks:
 * e_b = scale_exp(max |v| over block b); q = e4m3(v * 2^-e_b).  The product is
 * one binary32 multiply by an exact power of two, i.e. the correctly rounded
 * v / 2^e_b.  sf_byte[b] = e_b + 127 (UE8M0 encoding).
 */
void oracle_quantize_row(const float *v, int n, uint8_t *q, uint8_t *sf_byte)
{
    for (int b = 0; b < n / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float a = fabsf(v[b * 128 + i]);
            if (a > amax)
                amax = a;
        }
        int e = oracle_scale_exp(amax);
        float inv = pow2i(-e);
        for (int i = 0; i < 128; ++i)
            q[b * 128 + i] = oracle_e4m3_encode(v[b * 128 + i] * inv);
        sf_byte[b] = (uint8_t)(e + 127);
    }
}

void oracle_quantize_rows(const float *v, int rows, int n, uint8_t *q, uint8_t *sf_byte)
{
    for (int r = 0; r < rows; ++r)
        oracle_quantize_row(v + (size_t)r * n, n, q + (size_t)r * n, sf_byte + (size_t)r * (n / 128));
}

/*
 * The same 1x128 quantisation with binary32 scales instead of powers of two (the
 * "1d2d" scaling of the "Single Batch Overlap (SBO)" PR, §3, with its scales kept as
 * floats): s_b = amax_b / 448, one binary32 division rounded to nearest even (1 when it
 * is 0: an all-zero block, or an amax so small that the quotient underflows), and
 * q = e4m3(v / s_b), one binary32 division per value followed by the e4m3 rounding
 * above.  The largest |v| of a block lands at (or rounds to) 448.
 */
float oracle_scale_f32(float amax)
{
    float s = amax / 448.0f;
    return s == 0.0f ? 1.0f : s;
}

void oracle_quantize_rows_f32(const float *v, int rows, int n, uint8_t *q, float *s)
{
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < n / 128; ++b) {
            const float *x = v + (size_t)r * n + b * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i)
                if (fabsf(x[i]) > amax)
                    amax = fabsf(x[i]);
            float sb = oracle_scale_f32(amax);
            for (int i = 0; i < 128; ++i)
                q[(size_t)r * n + b * 128 + i] = oracle_e4m3_encode(x[i] / sb);
            s[(size_t)r * (n / 128) + b] = sb;
        }
}

/* ---------------------------------------------------------------- routing */

/* "a ranks before b": larger score first, equal scores -> lower index first. */
static int ranks_before(float sa, int ia, float sb, int ib)
{
    return sa > sb || (sa == sb && ia < ib);
}

/*
 * Route one token.
 *   logits z_e = sum_k x_k * W[e][k], accumulated as z = fmaf(x_k, W[e][k], z)
 *   for k = 0 .. H-1 in order (this fixes the rounding of every logit).
 * score_fn 0 (softmax): the choice score is z itself; s = softmax(z) over all N
 *   experts: m = max z, d_e = exp(z_e - m), S = d_0 + d_1 + ... (index order),
 *   s_e = d_e / S.
 * score_fn 1 (sigmoid): s_e = sigmoid(z_e); choice score c_e = s_e + bias_e
 *   (bias only steers the choice; weights use s).
 * Group-limited choice (n_group > 1): group j holds experts
 *   [j*N/n_group, (j+1)*N/n_group); its score is c_(1) + c_(2), the two largest
 *   choice scores in the group; the topk_group best groups survive (ties -> lower
 *   group index); experts outside them are not eligible.
 * Top-K: the K eligible experts ranked by (choice score desc, index asc), stored
 *   in that rank order.
 * Weights: renorm ? (s_k / (s_0 + ... + s_{K-1})) * scale : s_k * scale, the sum
 *   taken in rank order, one rounding per operation.
 * logits_out (nullable) receives z.
 */
static void route_token(const uint16_t *x, const float *W, const float *bias, int H, int N,
                        int K, int n_group, int topk_group, int score_fn, int renorm,
                        float scale, int32_t *idx_out, float *w_out, float *logits_out,
                        float *z, float *s, float *c, int *eligible)
{
    for (int e = 0; e < N; ++e) {
        float acc = 0.0f;
        const float *w = W + (size_t)e * H;
        for (int k = 0; k < H; ++k)
            acc = fmaf(oracle_bf16_to_f32(x[k]), w[k], acc);
        z[e] = acc;
        if (logits_out)
            logits_out[e] = acc;
    }
    if (score_fn == 0) {
        float m = z[0];
        for (int e = 1; e < N; ++e)
            if (z[e] > m)
                m = z[e];
        float S = 0.0f;
        for (int e = 0; e < N; ++e) {
            s[e] = oracle_exp(z[e] - m);
            S = S + s[e];
        }
        for (int e = 0; e < N; ++e) {
            s[e] = s[e] / S;
            c[e] = z[e];
        }
    } else {
        for (int e = 0; e < N; ++e) {
            s[e] = oracle_sigmoid(z[e]);
            c[e] = bias ? s[e] + bias[e] : s[e];
        }
    }
    for (int e = 0; e < N; ++e)
        eligible[e] = 1;
    if (n_group > 1) {
        int gs = N / n_group;
        float gscore[64];
        int keep[64];
        for (int j = 0; j < n_group; ++j) {
            int b1 = -1, b2 = -1;
            for (int e = j * gs; e < (j + 1) * gs; ++e) {
                if (b1 < 0 || ranks_before(c[e], e, c[b1], b1)) {
                    b2 = b1;
                    b1 = e;
                } else if (b2 < 0 || ranks_before(c[e], e, c[b2], b2)) {
                    b2 = e;
                }
            }
            gscore[j] = c[b1] + c[b2];
            keep[j] = 0;
        }
        for (int r = 0; r < topk_group; ++r) {
            int best = -1;
            for (int j = 0; j < n_group; ++j)
                if (!keep[j] && (best < 0 || ranks_before(gscore[j], j, gscore[best], best)))
                    best = j;
            keep[best] = 1;
        }
        for (int e = 0; e < N; ++e)
            eligible[e] = keep[e / gs];
    }
    for (int r = 0; r < K; ++r) {
        int best = -1;
        for (int e = 0; e < N; ++e)
            if (eligible[e] && (best < 0 || ranks_before(c[e], e, c[best], best)))
                best = e;
        idx_out[r] = best;
        eligible[best] = 0;
    }
    float sum = 0.0f;
    for (int r = 0; r < K; ++r)
        sum = sum + s[idx_out[r]];
    for (int r = 0; r < K; ++r)
        w_out[r] = renorm ? (s[idx_out[r]] / sum) * scale : s[idx_out[r]] * scale;
}

/*
 * Route tokens tok[0..ntok-1] (tok == NULL: tokens 0..ntok-1) of x [B][H].
 * Outputs are indexed by position in the token list.
 */
int oracle_route(const uint16_t *x, const float *W, const float *bias, int H, int N, int K,
                 int n_group, int topk_group, int score_fn, int renorm, float scale,
                 const int32_t *tok, int ntok, int32_t *topk_idx, float *topk_w,
                 float *logits, int nthreads)
{
    if (N > 1024 || K > N || (n_group > 1 && (N % n_group || n_group > 64 ||
                                                topk_group > n_group || N / n_group < 2 ||
                                                K > topk_group * (N / n_group))))
        return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        float *z = malloc(sizeof(float) * N), *s = malloc(sizeof(float) * N),
              *c = malloc(sizeof(float) * N);
        int *el = malloc(sizeof(int) * N);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int i = 0; i < ntok; ++i) {
            int t = tok ? tok[i] : i;
            route_token(x + (size_t)t * H, W, bias, H, N, K, n_group, topk_group, score_fn,
                        renorm, scale, topk_idx + (size_t)i * K, topk_w + (size_t)i * K,
                        logits ? logits + (size_t)i * N : NULL, z, s, c, el);
        }
        free(z);
        free(s);
        free(c);
        free(el);
    }
    return 0;
}

/* ------------------------------------------------------------------- EPLB */
/*
 * Redundant-expert map: N_phys - N_log extra slots go to the hottest logical
 * experts, one replica each (counts descending, ties -> lower index); the i-th
 * hottest expert's replica is physical expert N_log + i.  A token t routed to
 * logical e goes to log2phys[e][t mod rep[e]].
 *   log2phys [N_log][2], rep [N_log], phys2log [N_phys].
 */
int oracle_eplb_build_map(const int64_t *counts, int N_log, int N_phys, int32_t *log2phys,
                          int32_t *rep, int32_t *phys2log)
{
    int extra = N_phys - N_log;
    if (extra < 0 || extra > N_log)
        return -1;
    int *taken = calloc((size_t)N_log, sizeof(int));
    for (int e = 0; e < N_log; ++e) {
        log2phys[2 * e] = e;
        log2phys[2 * e + 1] = e;
        rep[e] = 1;
        phys2log[e] = e;
    }
    for (int i = 0; i < extra; ++i) {
        int best = -1;
        for (int e = 0; e < N_log; ++e)
            if (!taken[e] && (best < 0 || counts[e] > counts[best]))
                best = e;
        taken[best] = 1;
        log2phys[2 * best + 1] = N_log + i;
        rep[best] = 2;
        phys2log[N_log + i] = best;
    }
    free(taken);
    return 0;
}

/* --------------------------------------------------------------- dispatch */
/*
 * Expert-major permutation of the routed rows, the single-GPU counterpart of the
 * EP all-to-all (each token copied to its K experts).
 *   phys(t,k) = log2phys[e][t mod rep[e]] (or e without a map); log2phys has
 *   max_rep columns.
 *   Within a physical expert, rows are taken in ascending (t, k) order.
 *   layout 0 (contiguous): expert p's segment starts at
 *       sum_{q<p} ceil(cnt_q / 128) * 128; rows_used = that sum over all experts.
 *   layout 1 (masked): expert p's slot j is row p*cap + j; a row with j >= cap is
 *       dropped (row_of = -1) and the return value's bit 1 is set.
 *   A[row] = e4m3 codes of x[t] quantised in 1x128 blocks, sf[row][b] = UE8M0 byte
 *   (fmt 0); fmt 1 copies the bf16 row unchanged (pass-through).
 * Outputs: phys [B][K], cnt [N_phys], seg_start [N_phys+1] (contiguous) ,
 *   row_of [B][K], src_of [rows] (-1 for rows nobody fills), A, sf.
 * Returns 0, or 2 if any row was dropped for capacity.
 */
int oracle_dispatch(const uint16_t *x, const int32_t *topk_idx, const int32_t *log2phys,
                    const int32_t *rep, int max_rep, int B, int H, int K, int N_phys,
                    int layout, int cap,
                    int fmt, int32_t *phys, int32_t *cnt, int32_t *seg_start, int32_t *row_of,
                    int32_t *src_of, int64_t rows_alloc, uint8_t *A, uint8_t *sf)
{
    int ret = 0;
    if (N_phys <= 0 || B < 0 || K <= 0 || H % 128)
        return -1;
    for (int p = 0; p < N_phys; ++p)
        cnt[p] = 0;
    for (int t = 0; t < B; ++t)
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[t * K + k];
            int p = log2phys ? log2phys[max_rep * e + (t % rep[e])] : e;
            phys[t * K + k] = p;
            cnt[p] += 1;
        }
    if (layout == 0) {
        seg_start[0] = 0;
        for (int p = 0; p < N_phys; ++p)
            seg_start[p + 1] = seg_start[p] + (cnt[p] + 127) / 128 * 128;
    }
    for (int64_t r = 0; r < rows_alloc; ++r)
        src_of[r] = -1;
    int32_t *fill = calloc((size_t)N_phys, sizeof(int32_t));
    int Hb = H / 128;
    float *row = malloc(sizeof(float) * H);
    uint8_t *qrow = malloc((size_t)H);
    uint8_t *srow = malloc((size_t)Hb);
    for (int t = 0; t < B; ++t) {
        if (fmt == 0) {
            for (int i = 0; i < H; ++i)
                row[i] = oracle_bf16_to_f32(x[(size_t)t * H + i]);
            oracle_quantize_row(row, H, qrow, srow);
        }
        for (int k = 0; k < K; ++k) {
            int p = phys[t * K + k];
            int j = fill[p]++;
            int64_t r;
            if (layout == 0) {
                r = seg_start[p] + j;
            } else if (j < cap) {
                r = (int64_t)p * cap + j;
            } else {
                row_of[t * K + k] = -1;
                ret = 2;
                continue;
            }
            row_of[t * K + k] = (int32_t)r;
            src_of[r] = t;
            if (fmt == 0) {
                memcpy(A + r * H, qrow, (size_t)H);
                memcpy(sf + r * Hb, srow, (size_t)Hb);
            } else {
                memcpy(A + r * H * 2, x + (size_t)t * H, (size_t)H * 2);
            }
        }
    }
    free(fill);
    free(row);
    free(qrow);
    free(srow);
    return ret;
}

/* ---------------------------------------------------------------- combine */
/*
 * Weighted sum back to token order (the combine step, "DeepEP 完全拆解",
 * §专家并行 / §combine):
 *   acc = 0; for k = 0..K-1 (rank order): if row_of[t][k] >= 0,
 *       acc = fmaf(w[t][k], Y[row_of[t][k]], acc);
 *   if S: acc = acc + S[t];   out[t] = bf16_rne(acc).
 * Y, S and out are bf16 bit patterns.
 */
void oracle_combine(const uint16_t *Y, const int32_t *row_of, const float *w,
                    const uint16_t *S, int B, int H, int K, uint16_t *out)
{
    for (int t = 0; t < B; ++t)
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t r = row_of[t * K + k];
                if (r < 0)
                    continue;
                acc = fmaf(w[t * K + k], oracle_bf16_to_f32(Y[(size_t)r * H + h]), acc);
            }
            if (S)
                acc = acc + oracle_bf16_to_f32(S[(size_t)t * H + h]);
            out[(size_t)t * H + h] = oracle_f32_to_bf16(acc);
        }
}

/* Float32 array -> bf16 bits (RNE), for the FFN's final rounding. */
void oracle_f32_to_bf16_array(const float *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16(v[i]);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Element-wise e4m3 encode/decode of arrays (for the pins' bulk checks). */
void oracle_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_exp_array(const float *v, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_exp(v[i]);
}

void oracle_sigmoid_array(const float *v, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_sigmoid(v[i]);
}
