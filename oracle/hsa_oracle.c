/*
 * hsa_oracle.c -- plain, slow CPU oracle for Hybrid-SWA dual-KV-pool attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  It shares no code, header, table or
 * helper with the CUDA path; the two meet only in the seeded inputs.
 *
 * Sources (page title, section):
 *  [P2 s1]  youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%",
 *           s1 "为什么选择 Hybrid SWA 架构": 70 layers, 10 Full Attention, 60 SWA with a
 *           128-token window; KV storage falls to about 1/7.
 *  [P2 s2]  same page, s2 "KVCache系统重构": Full KV Pool grows on demand and is kept;
 *           SWA KV Pool is a ring buffer sized by the window, storage strictly O(W);
 *           the prefix tree matches by "window-safe length" (the last W tokens of the
 *           match must still hold valid SWA slots).
 *  [P4]     hotdry.top "MiMo-V2.5 ultra-speed inference architecture", section
 *           "Hybrid SWA：用 1/7 计算量捕获长程依赖": 6:1 interleave; match length is cut
 *           back to the window boundary.
 *
 * Readings taken where the pages are silent (each also listed in the design notes):
 *  - A sliding window of W covers W keys including the query itself: a query at
 *    position p attends positions max(0, p-W+1) .. p.
 *  - Query head h reads KV head h / (Hq/Hkv) (contiguous GQA grouping).
 *  - Softmax scale is an input (1/sqrt(d) in every workload); no bias, sink or cap.
 *  - Ring placement: slot = pos mod W; appends are applied in position order, so
 *    after positions [0,E) were appended slot j holds the largest p < E, p = j mod W.
 *  - Window-safe length: the largest L in [0, m] such that every position in
 *    [max(0, L-W), L) is live; "at least W tokens" is taken literally.
 *
 * Arithmetic: bf16 inputs are widened exactly to double; every sum is in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> double, exact (bf16 is the top half of an IEEE binary32). */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* Masked softmax attention [P2 s1]: for one query row q (already widened),
 * o = sum_j softmax_j(scale * q . k_j) v_j over the given key rows.
 * The row maximum is subtracted before exp (same value, no overflow).          */
static void attend_row(const double *q, int d, double scale, int nkeys,
                       const uint16_t *const *krow, const uint16_t *const *vrow,
                       double *score, double *out)
{
    double mx = -INFINITY;
    for (int j = 0; j < nkeys; ++j) {
        double s = 0.0;
        for (int c = 0; c < d; ++c)
            s += q[c] * bf16_to_double(krow[j][c]);
        s *= scale;
        score[j] = s;
        if (s > mx)
            mx = s;
    }
    double den = 0.0;
    for (int j = 0; j < nkeys; ++j) {
        score[j] = exp(score[j] - mx);
        den += score[j];
    }
    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    for (int j = 0; j < nkeys; ++j) {
        double w = score[j] / den;
        for (int c = 0; c < d; ++c)
            out[c] += w * bf16_to_double(vrow[j][c]);
    }
}

/*
 * Attention for new query rows on top of a cached prefix; decode, MTP verify
 * and chunked prefill are all this one computation.
 *
 * Request r owns new rows cu_rows[r] .. cu_rows[r+1]-1; row i of request r sits at
 * position prefix_len[r] + i.  Keys at positions < prefix_len[r] come from the
 * request's history; keys at positions >= prefix_len[r] are the new rows' own K/V
 * (causal among the new rows).  window == 0 means full causal attention; window W
 * restricts a query at p to positions max(0, p-W+1) .. p [P2 s1].
 *
 * History of request r: hist_off[r] .. hist_off[r+1]-1 rows of hist_k/hist_v, each
 * [Hkv, d], holding positions hist_start[r] .. prefix_len[r]-1.
 *
 * Items: if n_items < 0 every (row, head) is computed into out[rows, Hq, d];
 * otherwise item k = (item_row[k], item_head[k]) goes to out[k, d].
 * Returns 0, or -1 if a needed history position is not present, or -2 on bad args.
 */
int orc_attention(int R, const int32_t *cu_rows, const int32_t *prefix_len,
                  int Hq, int Hkv, int d, int window, double scale,
                  const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                  const uint16_t *hist_k, const uint16_t *hist_v,
                  const int64_t *hist_off, const int32_t *hist_start,
                  int64_t n_items, const int32_t *item_row, const int32_t *item_head,
                  double *out, int nthreads)
{
    if (R < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || window < 0)
        return -2;
    const int group = Hq / Hkv;
    const int64_t rows = cu_rows[R];
    const int64_t total = n_items < 0 ? rows * Hq : n_items;
    int status = 0;
    int64_t max_keys = 1;
    for (int r = 0; r < R; ++r) {
        int64_t k = (int64_t)prefix_len[r] + (cu_rows[r + 1] - cu_rows[r]);
        if (k > max_keys)
            max_keys = k;
    }
    if (nthreads <= 0)
        nthreads = 1;

#pragma omp parallel num_threads(nthreads)
    {
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(*krow) * max_keys);
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(*vrow) * max_keys);
        double *score = (double *)malloc(sizeof(double) * max_keys);
        double *qd = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t it = 0; it < total; ++it) {
            int64_t row;
            int h;
            if (n_items < 0) {
                row = it / Hq;
                h = (int)(it % Hq);
            } else {
                row = item_row[it];
                h = item_head[it];
            }
            double *o = out + it * d;
            if (row < 0 || row >= rows || h < 0 || h >= Hq) {
#pragma omp atomic write
                status = -2;
                continue;
            }
            int r = 0; /* request owning this row: plain linear search */
            while (r + 1 < R && cu_rows[r + 1] <= row)
                ++r;
            const int64_t i = row - cu_rows[r];
            const int64_t P = prefix_len[r];
            const int64_t p = P + i;
            const int64_t lo = window > 0 ? (p - window + 1 > 0 ? p - window + 1 : 0) : 0;
            const int kv = h / group;
            int nk = 0, bad = 0;
            for (int64_t x = lo; x <= p; ++x) {
                if (x < P) {
                    if (x < hist_start[r]) {
                        bad = 1;
                        break;
                    }
                    int64_t hr = hist_off[r] + (x - hist_start[r]);
                    krow[nk] = hist_k + (hr * Hkv + kv) * d;
                    vrow[nk] = hist_v + (hr * Hkv + kv) * d;
                } else {
                    int64_t nr = cu_rows[r] + (x - P);
                    krow[nk] = k_new + (nr * Hkv + kv) * d;
                    vrow[nk] = v_new + (nr * Hkv + kv) * d;
                }
                ++nk;
            }
            if (bad) {
#pragma omp atomic write
                status = -1;
                continue;
            }
            for (int c = 0; c < d; ++c)
                qd[c] = bf16_to_double(q[(row * Hq + h) * d + c]);
            attend_row(qd, d, scale, nk, krow, vrow, score, o);
        }
        free(krow);
        free(vrow);
        free(score);
        free(qd);
    }
    return status;
}

/* ------------------------------------------------------------------------- */
/* Placement [P2 s2].  Full KV Pool: a sequence's logical page pos/page_size maps
 * through its block-table row to a physical block; the row within the block is
 * pos mod page_size.  Pool layout [num_blocks, Hkv, page_size, d].            */
int orc_full_place(const int32_t *block_tables, int max_blocks, int num_blocks,
                   int page_size, int seq, int64_t pos, int32_t *block, int32_t *offset)
{
    if (pos < 0 || page_size <= 0)
        return -1;
    int64_t logical = pos / page_size;
    if (logical >= max_blocks)
        return -1;
    int32_t b = block_tables[(int64_t)seq * max_blocks + logical];
    if (b < 0 || b >= num_blocks)
        return -1;
    *block = b;
    *offset = (int32_t)(pos % page_size);
    return 0;
}

/* SWA KV Pool: a ring of W slots per sequence; slot = pos mod W [P2 s2].
 * Ring layout [n_rows, Hkv, W, d].                                             */
int orc_ring_place(const int32_t *ring_row, int n_rows, int W, int seq, int64_t pos,
                   int32_t *row, int32_t *slot)
{
    if (pos < 0 || W <= 0)
        return -1;
    int32_t rr = ring_row[seq];
    if (rr < 0 || rr >= n_rows)
        return -1;
    *row = rr;
    *slot = (int32_t)(pos % W);
    return 0;
}

/*
 * Apply one append call to a host image of a pool.  Request r appends rows
 * cu_rows[r] .. cu_rows[r+1]-1 of k_new/v_new ([rows, Hkv, d]) at positions
 * start_pos[r] + i of sequence seq_idx[r].  Tokens are written one by one in
 * position order, each into its own place; for the ring a later token
 * overwrites an earlier one that shares its slot.
 *   is_ring == 0: pool [num_blocks, Hkv, page_size, d], block_tables [*, max_blocks]
 *   is_ring == 1: pool [n_rows, Hkv, W, d] (num_blocks = n_rows, page_size = W),
 *                 ring_row [*]
 * Returns the number of tokens that could not be placed (out of range).
 */
int64_t orc_append(int is_ring, uint16_t *pool_k, uint16_t *pool_v, int num_blocks,
                   int Hkv, int page_size, int d, const int32_t *block_tables,
                   int max_blocks, const int32_t *ring_row, int R, const int32_t *cu_rows,
                   const int32_t *seq_idx, const int32_t *start_pos,
                   const uint16_t *k_new, const uint16_t *v_new)
{
    int64_t bad = 0;
    for (int r = 0; r < R; ++r) {
        for (int64_t row = cu_rows[r]; row < cu_rows[r + 1]; ++row) {
            int64_t pos = (int64_t)start_pos[r] + (row - cu_rows[r]);
            int32_t blk, off;
            int rc = is_ring
                ? orc_ring_place(ring_row, num_blocks, page_size, seq_idx[r], pos, &blk, &off)
                : orc_full_place(block_tables, max_blocks, num_blocks, page_size,
                                 seq_idx[r], pos, &blk, &off);
            if (rc != 0) {
                ++bad;
                continue;
            }
            for (int h = 0; h < Hkv; ++h) {
                int64_t dst = (((int64_t)blk * Hkv + h) * page_size + off) * d;
                int64_t src = (row * Hkv + h) * d;
                memcpy(pool_k + dst, k_new + src, sizeof(uint16_t) * d);
                memcpy(pool_v + dst, v_new + src, sizeof(uint16_t) * d);
            }
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Window-safe length [P2 s2], [P4]: a prefix match of length L may be reused only
 * if every position in [max(0, L-W), L) still holds a live SWA slot.  The answer
 * is the largest such L in [0, m]; L = 0 is always safe.  Brute force straight
 * from the definition.                                                        */
static int32_t safe_len_scan(int32_t m, int W, const void *ctx,
                             int (*live)(const void *, int64_t))
{
    for (int64_t L = m; L > 0; --L) {
        int64_t lo = L - W > 0 ? L - W : 0;
        int ok = 1;
        for (int64_t p = lo; p < L; ++p) {
            if (!live(ctx, p)) {
                ok = 0;
                break;
            }
        }
        if (ok)
            return (int32_t)L;
    }
    return 0;
}

struct ring_ctx { const int32_t *slot_pos; int W; };
static int ring_live(const void *c, int64_t p)
{
    const struct ring_ctx *rc = (const struct ring_ctx *)c;
    return rc->slot_pos[p % rc->W] == p;
}

struct bitmap_ctx { const uint8_t *live; };
static int bitmap_live(const void *c, int64_t p)
{
    return ((const struct bitmap_ctx *)c)->live[p] != 0;
}

/* Ring form: slot_pos[k*W + j] is the position ring slot j of case k holds
 * (-1 = freed); position p is live iff slot_pos[p mod W] == p.              */
void orc_window_safe_len_ring(int n, int W, const int32_t *match_len,
                              const int32_t *slot_pos, int32_t *out)
{
    for (int k = 0; k < n; ++k) {
        struct ring_ctx c = {slot_pos + (int64_t)k * W, W};
        out[k] = match_len[k] <= 0 ? 0 : safe_len_scan(match_len[k], W, &c, ring_live);
    }
}

/* Bitmap (prefix-tree) form: live[live_off[k] + p] != 0 iff position p of case k
 * still has a valid SWA slot, for p in [0, match_len[k]).                    */
void orc_window_safe_len_bitmap(int n, int W, const int32_t *match_len,
                                const int64_t *live_off, const uint8_t *live, int32_t *out)
{
    for (int k = 0; k < n; ++k) {
        struct bitmap_ctx c = {live + live_off[k]};
        out[k] = match_len[k] <= 0 ? 0 : safe_len_scan(match_len[k], W, &c, bitmap_live);
    }
}

/* ------------------------------------------------------------------------- */
/* KV bytes held for one sequence of length L [P2 s1], [P2 s2]: a full layer keeps
 * all L tokens (Full KV Pool, O(N)); a sliding-window layer keeps min(L, W)
 * (SWA KV Pool, O(W)).  bytes_per_token is per layer (K and V, all KV heads). */
double orc_kv_bytes(int n_layers, const uint8_t *is_full, int W, int64_t L,
                    double bytes_per_token)
{
    double tokens = 0.0;
    for (int l = 0; l < n_layers; ++l)
        tokens += is_full[l] ? (double)L : (double)(L < W ? L : W);
    return tokens * bytes_per_token;
}

/* ------------------------------------------------------------------------- */
/* FP8 KV Pool variant.
 * [P5] hotdry.top "MiMo inference optimization, edge deployment", sections
 *      "KV Cache 量化策略的技术选型" (quantisation groups aligned to the window so
 *      that no group straddles a window boundary) and "边缘部署的工程权衡与参数清单"
 *      (FP8 as a baseline KV format; the newest 128 tokens kept at the original
 *      precision).
 * Readings: the Full KV Pool holds E4M3 codes with one fp32 scale per (position,
 * KV head) row of d values -- a group of one token never crosses a window
 * boundary; the SWA ring, which holds exactly the newest W = 128 tokens, stays
 * bf16.  scale = amax / 448 (fp32 division), code = E4M3 of x / scale (fp32
 * division), all codes 0 and scale 0 for an all-zero row.
 *
 * E4M3 (OCP 8-bit floating point): sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits, subnormals at exponent field 0, no infinities, 0x7F / 0xFF are
 * NaN; the largest finite magnitude is 448.                                    */
double orc_e4m3_value(uint8_t c)
{
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return (c & 0x80) ? -v : v;
}

/* The finite code nearest to x, ties to the code with an even mantissa; beyond
 * the largest finite magnitude the result saturates to +-448.  Plain search over
 * the 127 non-negative finite codes.                                          */
uint8_t orc_e4m3_encode(float x)
{
    const double a = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 126; ++c) {
        const double err = fabs(orc_e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(signbit(x) ? (best | 0x80) : best);
}

/* Quantise rows of d bf16 values: codes [rows, d], scales [rows].            */
void orc_quantize_e4m3(int64_t rows, int d, const uint16_t *x, uint8_t *codes, float *scales)
{
    /* rows are independent groups: spread over the host's threads */
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < d; ++c) {
            const float v = fabsf((float)bf16_to_double(x[r * d + c]));
            if (v > amax)
                amax = v;
        }
        const float scale = amax / 448.0f;
        scales[r] = amax > 0.0f ? scale : 0.0f;
        for (int c = 0; c < d; ++c) {
            const float v = (float)bf16_to_double(x[r * d + c]);
            codes[r * d + c] = amax > 0.0f ? orc_e4m3_encode(v / scale) : 0;
        }
    }
}

/* E5M2 (OCP 8-bit floating point), the second FP8 format [P5 "KV Cache 量化策略的
 * 技术选型" weighs both]: sign bit, 5 exponent bits with bias 15, 2 mantissa bits,
 * subnormals at exponent field 0; exponent field 31 holds the infinities (mantissa
 * 0) and the NaNs; the largest finite magnitude is 57344.  Reading: the same row
 * groups as E4M3, scale = amax / 57344, code = E5M2 of x / scale (round to nearest
 * even, saturating to the largest finite magnitude).                          */
double orc_e5m2_value(uint8_t c)
{
    const int e = (c >> 2) & 31, m = c & 3;
    double v;
    if (e == 31)
        v = m == 0 ? INFINITY : NAN;
    else
        v = e == 0 ? ldexp((double)m / 4.0, -14) : ldexp(1.0 + (double)m / 4.0, e - 15);
    return (c & 0x80) ? -v : v;
}

/* Nearest finite E5M2 code (ties to the even mantissa, saturating): plain search
 * over the 124 non-negative finite codes.                                      */
uint8_t orc_e5m2_encode(float x)
{
    const double a = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 123; ++c) {
        const double err = fabs(orc_e5m2_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(signbit(x) ? (best | 0x80) : best);
}

/* Quantise rows of d bf16 values to E5M2: codes [rows, d], scales [rows].     */
void orc_quantize_e5m2(int64_t rows, int d, const uint16_t *x, uint8_t *codes, float *scales)
{
    /* rows are independent groups: spread over the host's threads */
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < d; ++c) {
            const float v = fabsf((float)bf16_to_double(x[r * d + c]));
            if (v > amax)
                amax = v;
        }
        const float scale = amax / 57344.0f;
        scales[r] = amax > 0.0f ? scale : 0.0f;
        for (int c = 0; c < d; ++c) {
            const float v = (float)bf16_to_double(x[r * d + c]);
            codes[r * d + c] = amax > 0.0f ? orc_e5m2_encode(v / scale) : 0;
        }
    }
}

/* Value of a code of format fmt (0 = E4M3, 1 = E5M2).                          */
static double fp8_value(uint8_t c, int fmt)
{
    return fmt ? orc_e5m2_value(c) : orc_e4m3_value(c);
}

/* attend_row for an FP8 history: keys / values with index < n_hist are
 * (codes, scale) rows dequantised exactly to double; the rest are bf16 rows.   */
static void attend_row_fp8(const double *q, int d, double scale, int nkeys, int n_hist,
                           const uint8_t *const *kc, const float *ks, const uint8_t *const *vc,
                           const float *vs, const uint16_t *const *krow,
                           const uint16_t *const *vrow, int fmt, double *score, double *out)
{
    double mx = -INFINITY;
    for (int j = 0; j < nkeys; ++j) {
        double s = 0.0;
        for (int c = 0; c < d; ++c)
            s += q[c] * (j < n_hist ? fp8_value(kc[j][c], fmt) * (double)ks[j]
                                    : bf16_to_double(krow[j][c]));
        s *= scale;
        score[j] = s;
        if (s > mx)
            mx = s;
    }
    double den = 0.0;
    for (int j = 0; j < nkeys; ++j) {
        score[j] = exp(score[j] - mx);
        den += score[j];
    }
    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    for (int j = 0; j < nkeys; ++j) {
        const double w = score[j] / den;
        for (int c = 0; c < d; ++c)
            out[c] += w * (j < n_hist ? fp8_value(vc[j][c], fmt) * (double)vs[j]
                                      : bf16_to_double(vrow[j][c]));
    }
}

/*
 * Full causal attention of T new rows per sequence on top of an FP8 history:
 * decode / MTP verify on an FP8 Full KV Pool.  Sequence r has prefix_len[r]
 * cached positions, history rows hist_off[r] .. hist_off[r+1]-1 holding positions
 * 0 .. prefix_len[r]-1 as codes [rows, Hkv, d] with scales [rows, Hkv]; its new
 * rows cu_rows[r] .. cu_rows[r+1]-1 (bf16) sit at positions prefix_len[r] + i.
 * fmt: 0 = E4M3 codes, 1 = E5M2.  Items as in orc_attention.  Returns 0, -1 if an
 * asked row's request lacks its history, or -2 on bad arguments.
 */
int orc_attention_fp8hist_fmt(int R, const int32_t *cu_rows, const int32_t *prefix_len,
                              int Hq, int Hkv, int d, double scale, const uint16_t *q,
                              const uint16_t *k_new, const uint16_t *v_new, const uint8_t *hk,
                              const float *hks, const uint8_t *hv, const float *hvs,
                              const int64_t *hist_off, int64_t n_items,
                              const int32_t *item_row, const int32_t *item_head, double *out,
                              int fmt, int nthreads)
{
    if (R < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || (fmt != 0 && fmt != 1))
        return -2;
    const int group = Hq / Hkv;
    const int64_t rows = cu_rows[R];
    const int64_t total = n_items < 0 ? rows * Hq : n_items;
    int status = 0;
    int64_t max_keys = 1;
    for (int r = 0; r < R; ++r) {
        int64_t k = (int64_t)prefix_len[r] + (cu_rows[r + 1] - cu_rows[r]);
        if (k > max_keys)
            max_keys = k;
    }
    if (nthreads <= 0)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        const uint8_t **kc = (const uint8_t **)malloc(sizeof(*kc) * max_keys);
        const uint8_t **vc = (const uint8_t **)malloc(sizeof(*vc) * max_keys);
        float *ks = (float *)malloc(sizeof(float) * max_keys);
        float *vs = (float *)malloc(sizeof(float) * max_keys);
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(*krow) * max_keys);
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(*vrow) * max_keys);
        double *score = (double *)malloc(sizeof(double) * max_keys);
        double *qd = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t it = 0; it < total; ++it) {
            const int64_t row = n_items < 0 ? it / Hq : item_row[it];
            const int h = n_items < 0 ? (int)(it % Hq) : item_head[it];
            double *o = out + it * d;
            if (row < 0 || row >= rows || h < 0 || h >= Hq) {
#pragma omp atomic write
                status = -2;
                continue;
            }
            int r = 0;
            while (r + 1 < R && cu_rows[r + 1] <= row)
                ++r;
            const int64_t P = prefix_len[r];
            const int64_t p = P + (row - cu_rows[r]);
            const int kv = h / group;
            if (hist_off[r + 1] - hist_off[r] != P) {  /* history of 0 .. P-1 missing */
#pragma omp atomic write
                status = -1;
                continue;
            }
            int nk = 0;
            for (int64_t x = 0; x <= p; ++x, ++nk) {
                if (x < P) {
                    const int64_t hr = hist_off[r] + x;
                    kc[nk] = hk + (hr * Hkv + kv) * d;
                    vc[nk] = hv + (hr * Hkv + kv) * d;
                    ks[nk] = hks[hr * Hkv + kv];
                    vs[nk] = hvs[hr * Hkv + kv];
                } else {
                    const int64_t nr = cu_rows[r] + (x - P);
                    krow[nk] = k_new + (nr * Hkv + kv) * d;
                    vrow[nk] = v_new + (nr * Hkv + kv) * d;
                }
            }
            for (int c = 0; c < d; ++c)
                qd[c] = bf16_to_double(q[(row * Hq + h) * d + c]);
            attend_row_fp8(qd, d, scale, nk, (int)P, kc, ks, vc, vs, krow, vrow, fmt, score, o);
        }
        free(kc);
        free(vc);
        free(ks);
        free(vs);
        free(krow);
        free(vrow);
        free(score);
        free(qd);
    }
    return status;
}

/* orc_attention_fp8hist_fmt of an E4M3 history.                                */
int orc_attention_fp8hist(int R, const int32_t *cu_rows, const int32_t *prefix_len, int Hq,
                          int Hkv, int d, double scale, const uint16_t *q,
                          const uint16_t *k_new, const uint16_t *v_new, const uint8_t *hk,
                          const float *hks, const uint8_t *hv, const float *hvs,
                          const int64_t *hist_off, int64_t n_items, const int32_t *item_row,
                          const int32_t *item_head, double *out, int nthreads)
{
    return orc_attention_fp8hist_fmt(R, cu_rows, prefix_len, Hq, Hkv, d, scale, q, k_new, v_new,
                                     hk, hks, hv, hvs, hist_off, n_items, item_row, item_head,
                                     out, 0, nthreads);
}
