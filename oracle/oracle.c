/*
 * oracle.c -- plain, slow, fp64 CPU restatement of fused inference attention
 * over a paged KV cache, and of the work schedules the GPU path publishes.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so, which
 * only the tests, the package smoke check and the CPU-baseline leg of the
 * benchmark load.  It shares no code, header, table or constant with the CUDA
 * library: every formula below is written out again from the pages that define
 * the operators:
 *   [FIA-V5]  "aclnnFusedInferAttentionScoreV5" (formula section; Attention Mask,
 *             Paged Attention, LearnableSink and SoftmaxLSE parameter groups)
 *   [FIA-V4]  "aclnnFusedInferAttentionScoreV4" (common constraints: empty tensors)
 *   [FIA-V2]  "aclnnFusedInferAttentionScoreV2" (softmax_lse restriction, the
 *             page-attention scenario, innerPrecise invalid-row correction)
 *   [KQSAS]   "ops-transformer .../kv_quant_sparse_attn_sharedkv" (formula,
 *             parameter table, constraints)
 *   [SFMLA]   "sparse_flash_mla" (SWA / CSA / HCA modes, metadata, CP example)
 *
 * Every floating-point step is done in IEEE double.  Inputs arrive as bf16 bit
 * patterns (uint16), FP8 E4M3 codes (uint8) with fp32 tile scales, and int32
 * index arrays.  Parallelism is a single OpenMP loop over independent output
 * rows; nothing is blocked, fused or reordered inside a row.
 *
 * Functions whose result is pinned by the CPU test-suite are listed in the
 * package docstring (oracle/__init__.py) together with the pins.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn": no infinities, S.1111.111 is NaN):
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
 * encodes subnormals m/8 * 2^-6.  Decoded from the bit definition, with no
 * table copied from anywhere. */
double oracle_e4m3_to_double(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

double oracle_bf16_to_double(uint16_t h) { return bf16_bits_to_double(h); }

/* OCP E8M0 ("float8_e8m0fnu", the MX scale format [KQSAS] names for the
 * nope_quant_scale): 8 exponent bits, no sign, no mantissa, bias 127; the
 * value is 2^(e - 127) and e = 255 encodes NaN. */
double oracle_e8m0_to_double(uint8_t e)
{
    if (e == 0xFF)
        return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* ------------------------------------------------------------------------ */
/* fused inference attention (FIA)                                          */
/* ------------------------------------------------------------------------ */

enum { OR_LAYOUT_BSND = 0, OR_LAYOUT_TND = 1 };
enum { OR_KV_BF16 = 0, OR_KV_E4M3 = 1 };
enum { OR_MASK_NONE = 0, OR_MASK_ALL = 1, OR_MASK_LUC = 2, OR_MASK_RDC = 3, OR_MASK_BAND = 4 };
enum { OR_KV_BNBSH = 0, OR_KV_BNNBSD = 1 };

typedef struct {
    int32_t B, QN, KVN, D;
    int32_t layout;              /* 0: BSND q [B,S_q,QN,D]; 1: TND q [T,QN,D]   */
    int32_t S_q;                 /* BSND query length                            */
    int32_t T;                   /* TND total query rows                         */
    const uint16_t *q;           /* bf16 bits                                    */
    const int32_t *cu_seqlens_q; /* TND: [B+1] cumulative query lengths          */
    int32_t kv_dtype;            /* 0 bf16, 1 FP8 E4M3 with fp32 tile scales     */
    const void *k, *v;           /* paged pool [nb,bs,KVN,D] or contiguous       */
    const float *k_scale, *v_scale; /* [nb,KVN,bs,D/tile] or [B,KVN,S_kv,D/tile] */
    int32_t quant_tile;
    const int32_t *block_table;  /* [B,max_blocks] or NULL (contiguous)          */
    int32_t max_blocks, block_size;
    int32_t S_kv;                /* contiguous KV [B,S_kv,KVN,D]                 */
    const int32_t *seqused_kv;   /* [B] valid KV length per batch, or NULL       */
    double scale;
    int32_t mask_mode, pre_tokens, next_tokens;
    const float *sinks;          /* [QN] fp32 or NULL                            */
    int32_t kv_layout;           /* paged pools: 0 [nb,bs,KVN,D], 1 [nb,KVN,bs,D] */
    int32_t max_seqlen_q;        /* rows per sequence the decode units cover     */
    const uint8_t *atten_mask;   /* modes 0/1: byte (b, i, j) nonzero = hidden   */
    int64_t mask_batch_stride;   /* bytes between batches (0: shared)            */
    int64_t mask_row_stride;     /* bytes between query rows                     */
} oracle_fia_args;

/* Index of the D-element vector of logical KV row j of batch b, head g, in the
 * KV storage ([FIA-V2] page-attention scenario: blockTable holds block ids,
 * the rows of a block sit contiguously in one pool; [FIA-V5] Paged Attention
 * group: the cache is BnBsH = [nb, bs, KVN*D] or BnNBsD = [nb, KVN, bs, D]).
 * Multiply by D for the first element. */
static int64_t kv_row_base(const oracle_fia_args *a, int b, int64_t j, int g)
{
    if (a->block_table) {
        int64_t blk = a->block_table[(int64_t)b * a->max_blocks + j / a->block_size];
        int64_t jp = j % a->block_size;
        if (a->kv_layout == OR_KV_BNNBSD)
            return (blk * a->KVN + g) * a->block_size + jp;
        return (blk * a->block_size + jp) * a->KVN + g;
    }
    return ((int64_t)b * a->S_kv + j) * a->KVN + g;
}

/* Index of the scale row of logical KV row j of batch b, head g.  The scales
 * are laid out head-major inside each page, as [FIA-V5]'s DequantChecker group
 * gives the page-managed per-token, per-head scale: (blockNum, N, blockSize),
 * here with the D/tile tiles of a row as a last axis; without a block table
 * the page is the whole sequence, (B, N, S_kv), as the non-paged per-token,
 * per-head shape (B, N, KV_S) in the same group. */
static int64_t scale_row(const oracle_fia_args *a, int b, int64_t j, int g)
{
    if (a->block_table) {
        int64_t blk = a->block_table[(int64_t)b * a->max_blocks + j / a->block_size];
        return (blk * a->KVN + g) * a->block_size + j % a->block_size;
    }
    return ((int64_t)b * a->KVN + g) * a->S_kv + j;
}

static double kv_value(const oracle_fia_args *a, const void *pool, const float *scales,
                       int b, int64_t j, int g, int d)
{
    int64_t rh = kv_row_base(a, b, j, g);
    if (a->kv_dtype == OR_KV_BF16)
        return bf16_bits_to_double(((const uint16_t *)pool)[rh * a->D + d]);
    /* FP8: value = decode(code) * scale of the 64-element tile holding d */
    {
        double c = oracle_e4m3_to_double(((const uint8_t *)pool)[rh * a->D + d]);
        int ntile = a->D / a->quant_tile;
        double s = (double)scales[scale_row(a, b, j, g) * ntile + d / a->quant_tile];
        return c * s;
    }
}

static void fia_lengths(const oracle_fia_args *a, int b, int64_t *q_len, int64_t *q_start,
                        int64_t *kv_len)
{
    if (a->layout == OR_LAYOUT_TND) {
        *q_start = a->cu_seqlens_q[b];
        *q_len = (int64_t)a->cu_seqlens_q[b + 1] - a->cu_seqlens_q[b];
    } else {
        *q_start = (int64_t)b * a->S_q;
        *q_len = a->S_q;
    }
    *kv_len = a->seqused_kv ? a->seqused_kv[b] : a->S_kv;
}

/* Visible KV interval [lo, hi] (inclusive) of query row i, per the mask mode
 * ([FIA-V5] Attention Mask group, sparseMode 0-4).  For modes 3 and 4 the
 * query row is aligned to the bottom-right corner of the (q_len x kv_len)
 * score matrix: its position is p = kv_len - q_len + i ([KQSAS] cmp_mask_mode
 * 3 "rightDownCausal", split by the right vertex; the CP example in [SFMLA]
 * derives the query start as kv length minus q length); mode 2 is the causal
 * mask split by the left vertex, p = i.
 *   modes 0, 1: all of [0, kv_len) (the explicit mask then hides single keys)
 *   modes 2, 3: j <= p
 *   mode 4:     p - pre_tokens <= j <= p + next_tokens  ([KQSAS] ori_mask_mode
 *               4 "band", ori_win_left / ori_win_right)
 * Returns 0 when the interval is empty. */
static int fia_visible(const oracle_fia_args *a, int64_t q_len, int64_t kv_len, int64_t i,
                       int64_t *lo, int64_t *hi)
{
    int64_t p = (a->mask_mode == OR_MASK_LUC ? 0 : kv_len - q_len) + i;
    *lo = 0;
    *hi = kv_len - 1;
    if (a->mask_mode == OR_MASK_RDC || a->mask_mode == OR_MASK_LUC) {
        if (p < *hi) *hi = p;
    } else if (a->mask_mode == OR_MASK_BAND) {
        if (p - a->pre_tokens > *lo) *lo = p - a->pre_tokens;
        if (p + a->next_tokens < *hi) *hi = p + a->next_tokens;
    }
    return *hi >= *lo;
}

/* Explicit mask ([FIA-V5] Attention Mask group: attenMask of shape
 * [batch or 1, >= Q_S, >= KV_S], 1 = masked out, 0 = kept): nonzero when key
 * j is hidden from query row i of batch b.  Modes 0 and 1 only. */
static int fia_hidden(const oracle_fia_args *a, int b, int64_t i, int64_t j)
{
    if (!a->atten_mask) return 0;
    return a->atten_mask[(int64_t)b * a->mask_batch_stride + i * a->mask_row_stride + j] != 0;
}

/* One output row: softmax over the visible scores (plus the sink logit, which
 * enters the denominator only), then the probability-weighted sum of V rows.
 * Follows the formula Attention(Q,K,V) = Softmax(QK^T * scale) V of [FIA-V5],
 * and the lse definition of [FIA-V2]: row max, subtract, exp, sum, log, add
 * the max back.  An empty visible set gives O = 0 and lse = +inf ([FIA-V4]
 * empty-tensor rule). */
static void fia_row(const oracle_fia_args *a, int b, int h, int64_t q_row, int64_t q_len,
                    int64_t kv_len, int64_t i, double *o, double *lse, double *s_buf)
{
    int D = a->D, G = a->QN / a->KVN, g = h / G;
    const uint16_t *qv = a->q + (q_row * a->QN + h) * (int64_t)D;
    int64_t lo, hi, j, n, nvis;
    double m, l;
    int d;

    for (d = 0; d < D; ++d) o[d] = 0.0;
    if (kv_len <= 0 || !fia_visible(a, q_len, kv_len, i, &lo, &hi)) {
        *lse = INFINITY;
        return;
    }
    n = hi - lo + 1;
    /* scores of the visible keys (an explicit mask hides single keys) */
    m = -INFINITY;
    nvis = 0;
    for (j = 0; j < n; ++j) {
        double s = 0.0;
        if (fia_hidden(a, b, i, lo + j)) {
            s_buf[j] = -INFINITY;
            continue;
        }
        ++nvis;
        for (d = 0; d < D; ++d)
            s += bf16_bits_to_double(qv[d]) * kv_value(a, a->k, a->k_scale, b, lo + j, g, d);
        s *= a->scale;
        s_buf[j] = s;
        if (s > m) m = s;
    }
    if (nvis == 0) {
        *lse = INFINITY;
        return;
    }
    if (a->sinks && (double)a->sinks[h] > m) m = (double)a->sinks[h];
    /* denominator */
    l = 0.0;
    for (j = 0; j < n; ++j)
        if (s_buf[j] != -INFINITY) l += exp(s_buf[j] - m);
    if (a->sinks) l += exp((double)a->sinks[h] - m);
    /* numerator */
    for (j = 0; j < n; ++j) {
        double w;
        if (s_buf[j] == -INFINITY) continue;
        w = exp(s_buf[j] - m) / l;
        for (d = 0; d < D; ++d)
            o[d] += w * kv_value(a, a->v, a->v_scale, b, lo + j, g, d);
    }
    *lse = m + log(l);
}

/* out: [rows, QN, D] (rows = B*S_q for BSND, T for TND), row-major.
 * lse: BSND [B, QN, S_q]; TND [T, QN]  ([FIA-V5] SoftmaxLSE group shapes with
 * the trailing 1 dropped). */
int oracle_fia(const oracle_fia_args *a, double *out, double *lse, int nthreads)
{
    int64_t rows = a->layout == OR_LAYOUT_TND ? a->T : (int64_t)a->B * a->S_q;
    int64_t total = rows * a->QN, max_kv = 0, t;
    int b;
    if (!a || !out) return 1;
    for (b = 0; b < a->B; ++b) {
        int64_t ql, qs, kl;
        fia_lengths(a, b, &ql, &qs, &kl);
        if (kl > max_kv) max_kv = kl;
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *s_buf = (double *)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
        double lse_dummy;
#pragma omp for schedule(dynamic, 1)
        for (t = 0; t < total; ++t) {
            int64_t row = t / a->QN;
            int h = (int)(t % a->QN);
            int bb = 0;
            int64_t ql, qs, kl, i;
            /* locate the batch owning this query row */
            if (a->layout == OR_LAYOUT_TND) {
                while (bb + 1 <= a->B && a->cu_seqlens_q[bb + 1] <= row) ++bb;
            } else {
                bb = (int)(row / a->S_q);
            }
            fia_lengths(a, bb, &ql, &qs, &kl);
            i = row - qs;
            {
                double *lse_p = &lse_dummy;
                if (lse) {
                    if (a->layout == OR_LAYOUT_TND)
                        lse_p = &lse[row * a->QN + h];
                    else
                        lse_p = &lse[((int64_t)bb * a->QN + h) * a->S_q + i];
                }
                fia_row(a, bb, h, row, ql, kl, i, out + t * a->D, lse_p, s_buf);
            }
        }
        free(s_buf);
    }
    return 0;
}

/* Probabilities of one row (for the "rows of the softmax sum to 1" check):
 * writes the visible interval start into *lo_out and the probabilities of the
 * n visible positions into p (capacity cap); returns n, or -1 if cap is too
 * small.  The sink's own probability is returned in *p_sink (0 without sink). */
int64_t oracle_fia_row_probs(const oracle_fia_args *a, int b, int h, int64_t i, double *p,
                             int64_t cap, int64_t *lo_out, double *p_sink)
{
    int64_t ql, qs, kl, lo, hi, n, j;
    int D = a->D, G = a->QN / a->KVN, g = h / G, d;
    const uint16_t *qv;
    double m = -INFINITY, l = 0.0;
    fia_lengths(a, b, &ql, &qs, &kl);
    *p_sink = 0.0;
    *lo_out = 0;
    if (kl <= 0 || !fia_visible(a, ql, kl, i, &lo, &hi)) return 0;
    n = hi - lo + 1;
    if (n > cap) return -1;
    qv = a->q + ((qs + i) * a->QN + h) * (int64_t)D;
    for (j = 0; j < n; ++j) {
        double s = 0.0;
        if (fia_hidden(a, b, i, lo + j)) {
            p[j] = -INFINITY;
            continue;
        }
        for (d = 0; d < D; ++d)
            s += bf16_bits_to_double(qv[d]) * kv_value(a, a->k, a->k_scale, b, lo + j, g, d);
        p[j] = s * a->scale;
        if (p[j] > m) m = p[j];
    }
    if (m == -INFINITY) {  /* every key hidden: no probabilities */
        for (j = 0; j < n; ++j) p[j] = 0.0;
        *lo_out = lo;
        return n;
    }
    if (a->sinks && (double)a->sinks[h] > m) m = (double)a->sinks[h];
    for (j = 0; j < n; ++j)
        if (p[j] != -INFINITY) l += exp(p[j] - m);
    if (a->sinks) l += exp((double)a->sinks[h] - m);
    for (j = 0; j < n; ++j) p[j] = p[j] == -INFINITY ? 0.0 : exp(p[j] - m) / l;
    if (a->sinks) *p_sink = exp((double)a->sinks[h] - m) / l;
    *lo_out = lo;
    return n;
}

/* ------------------------------------------------------------------------ */
/* shared-KV sparse attention (SWA / CSA / HCA)                             */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t B, N1, D;
    int32_t layout;              /* 0: BSND q [B,S1,N1,D]; 1: TND q [T1,N1,D]  */
    int32_t S1, T1;
    const uint16_t *q;
    const int32_t *cu_seqlens_q; /* TND [B+1]                                   */
    const void *ori_kv;          /* [nb1, bs1, 1, D] bf16 or [nb1, bs1, 1, 640] B */
    const int32_t *ori_block_table;
    int32_t ori_max_blocks, ori_block_size;
    const void *cmp_kv;          /* the same for the compressed rows; NULL: SWA  */
    const int32_t *cmp_block_table;
    int32_t cmp_max_blocks, cmp_block_size;
    const int32_t *cmp_sparse_indices; /* [rows, 1, K2] or NULL (HCA)          */
    int32_t K2;
    const int32_t *seqused_kv;   /* [B] S2 of each batch (ori length)            */
    const float *sinks;          /* [N1] or NULL                                 */
    double scale;
    int32_t cmp_ratio, win_left, win_right;
    int32_t kv_dtype;            /* 0 bf16 rows of D; 1 packed FP8 rows of 640 B */
} oracle_sparse_args;

/* Bytes of one stored K~ row: D bf16 values, or the packed FP8 row of
 * [KQSAS] (constraint on the D of ori_kv / cmp_kv: 640, the rope part, the
 * nope part and its scales in that order, padded to a multiple of 128 B). */
static int64_t sparse_row_bytes(const oracle_sparse_args *a)
{
    return a->kv_dtype == 1 ? 640 : 2 * (int64_t)a->D;
}

/* Element d of a stored K~ row.  Packed FP8 ([KQSAS] constraints: kv_rope
 * bf16 with rope_head_dim 64, then kv_nope E4M3 with nope_head_dim 448, then
 * nope_quant_scale E8M0 with 448 / tile_size = 7 entries, tile_size 64):
 * d < 64 is the rope value; d >= 64 is the nope code times its tile scale. */
static double sparse_value(const oracle_sparse_args *a, const uint8_t *row, int d)
{
    if (a->kv_dtype != 1) {
        uint16_t h = (uint16_t)(row[2 * d] | (row[2 * d + 1] << 8));
        return bf16_bits_to_double(h);
    }
    if (d < 64) {
        uint16_t h = (uint16_t)(row[2 * d] | (row[2 * d + 1] << 8));
        return bf16_bits_to_double(h);
    }
    return oracle_e4m3_to_double(row[128 + (d - 64)]) *
           oracle_e8m0_to_double(row[128 + 448 + (d - 64) / 64]);
}

/* Logical rows of K~ (= V~) for query row i of batch b, in concatenation
 * order: the band window of the original KV, then the compressed rows.
 *   window ([KQSAS] ori_mask_mode 4, ori_win_left, ori_win_right):
 *       ori rows p - win_left .. p + win_right clipped to [0, S2)
 *   compressed ([KQSAS] cmp_mask_mode 3 right-down causal; cmp length is
 *   floor(S2 / cmp_ratio) per the cmp_block_table sizing rule): compressed row
 *   c summarises ori tokens [c*r, (c+1)*r) and is visible iff (c+1)*r <= p+1.
 *       CSA: the listed indices of cmp_sparse_indices, scanned until the first
 *            -1 (valid entries come first, invalid after), each kept if
 *            visible;
 *       HCA: every visible compressed row 0 .. floor((p+1)/r) - 1.
 * Each entry is encoded as  (row << 1) | is_cmp.  Returns the count. */
static int64_t sparse_rows(const oracle_sparse_args *a, int b, int64_t q_len, int64_t q_row,
                           int64_t i, int64_t *list)
{
    int64_t S2 = a->seqused_kv[b];
    int64_t p = S2 - q_len + i, n = 0, j, lo, hi, ncmp_vis;
    lo = p - a->win_left;
    hi = p + a->win_right;
    if (lo < 0) lo = 0;
    if (hi > S2 - 1) hi = S2 - 1;
    for (j = lo; j <= hi; ++j) list[n++] = (j << 1);
    if (!a->cmp_kv) return n;
    ncmp_vis = (p + 1) >= 0 ? (p + 1) / a->cmp_ratio : 0;
    if (a->cmp_sparse_indices) {
        const int32_t *ix = a->cmp_sparse_indices + q_row * (int64_t)a->K2;
        int t;
        for (t = 0; t < a->K2; ++t) {
            int64_t c = ix[t];
            if (c < 0) break;
            if (c < ncmp_vis) list[n++] = (c << 1) | 1;
        }
    } else {
        for (j = 0; j < ncmp_vis; ++j) list[n++] = (j << 1) | 1;
    }
    return n;
}

static const uint8_t *sparse_row_ptr(const oracle_sparse_args *a, int b, int64_t e)
{
    int64_t r = e >> 1, phys;
    if (e & 1) {
        phys = (int64_t)a->cmp_block_table[(int64_t)b * a->cmp_max_blocks + r / a->cmp_block_size] *
                   a->cmp_block_size + r % a->cmp_block_size;
        return (const uint8_t *)a->cmp_kv + phys * sparse_row_bytes(a);
    }
    phys = (int64_t)a->ori_block_table[(int64_t)b * a->ori_max_blocks + r / a->ori_block_size] *
               a->ori_block_size + r % a->ori_block_size;
    return (const uint8_t *)a->ori_kv + phys * sparse_row_bytes(a);
}

/* out: [rows, N1, D]; lse: [rows, N1] (= [B, N2=1, S1, N1] or [N2=1, T1, N1]).
 * O = softmax(Q K~^T * softmax_scale) V~ with K~ = V~ ([KQSAS] formula). */
int oracle_sparse(const oracle_sparse_args *a, double *out, double *lse, int nthreads)
{
    int64_t rows = a->layout == OR_LAYOUT_TND ? a->T1 : (int64_t)a->B * a->S1;
    int64_t total = rows * a->N1, t;
    int64_t cap = (int64_t)a->win_left + a->win_right + 1;
    int b;
    if (a->cmp_kv) {
        if (a->cmp_sparse_indices) {
            cap += a->K2;
        } else {
            int64_t mx = 0;
            for (b = 0; b < a->B; ++b)
                if (a->seqused_kv[b] > mx) mx = a->seqused_kv[b];
            cap += mx / a->cmp_ratio + 1;
        }
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        int64_t *list = (int64_t *)malloc(sizeof(int64_t) * (size_t)cap);
        double *s = (double *)malloc(sizeof(double) * (size_t)cap);
#pragma omp for schedule(dynamic, 1)
        for (t = 0; t < total; ++t) {
            int64_t row = t / a->N1, ql, qs, i, n, j;
            int h = (int)(t % a->N1), bb = 0, d, D = a->D;
            const uint16_t *qv = a->q + t * (int64_t)D;
            double *o = out + t * (int64_t)D, m = -INFINITY, l = 0.0;
            if (a->layout == OR_LAYOUT_TND) {
                while (bb + 1 <= a->B && a->cu_seqlens_q[bb + 1] <= row) ++bb;
                qs = a->cu_seqlens_q[bb];
                ql = (int64_t)a->cu_seqlens_q[bb + 1] - qs;
            } else {
                bb = (int)(row / a->S1);
                qs = (int64_t)bb * a->S1;
                ql = a->S1;
            }
            i = row - qs;
            n = sparse_rows(a, bb, ql, row, i, list);
            for (d = 0; d < D; ++d) o[d] = 0.0;
            if (n == 0) {
                if (lse) lse[t] = INFINITY;
                continue;
            }
            for (j = 0; j < n; ++j) {
                const uint8_t *kr = sparse_row_ptr(a, bb, list[j]);
                double acc = 0.0;
                for (d = 0; d < D; ++d)
                    acc += bf16_bits_to_double(qv[d]) * sparse_value(a, kr, d);
                s[j] = acc * a->scale;
                if (s[j] > m) m = s[j];
            }
            if (a->sinks && (double)a->sinks[h] > m) m = (double)a->sinks[h];
            for (j = 0; j < n; ++j) l += exp(s[j] - m);
            if (a->sinks) l += exp((double)a->sinks[h] - m);
            for (j = 0; j < n; ++j) {
                const uint8_t *vr = sparse_row_ptr(a, bb, list[j]);
                double w = exp(s[j] - m) / l;
                for (d = 0; d < D; ++d) o[d] += w * sparse_value(a, vr, d);
            }
            if (lse) lse[t] = m + log(l);
        }
        free(list);
        free(s);
    }
    return 0;
}

/* Logical K~ rows of one query (for tests of the index gather): same
 * encoding as sparse_rows.  Returns the count or -1 if cap is too small. */
int64_t oracle_sparse_rows(const oracle_sparse_args *a, int b, int64_t i, int64_t *list,
                           int64_t cap)
{
    int64_t ql, qs, row;
    int64_t need = (int64_t)a->win_left + a->win_right + 1 +
                   (a->cmp_kv ? (a->cmp_sparse_indices ? a->K2
                                                       : a->seqused_kv[b] / a->cmp_ratio + 1)
                              : 0);
    if (need > cap) return -1;
    if (a->layout == OR_LAYOUT_TND) {
        qs = a->cu_seqlens_q[b];
        ql = (int64_t)a->cu_seqlens_q[b + 1] - qs;
    } else {
        qs = (int64_t)b * a->S1;
        ql = a->S1;
    }
    row = qs + i;
    return sparse_rows(a, b, ql, row, i, list);
}

/* ------------------------------------------------------------------------ */
/* work schedules (twins of the metadata the GPU path publishes)            */
/* ------------------------------------------------------------------------ */
/*
 * The pages fix only the contract of the metadata step ([SFMLA]: a task list
 * giving each core the batch, head and Q/K block indices where its work starts
 * and ends, in a fixed [1024] int32 buffer; [KQSAS] metadata parameter).  The
 * split policy below is this library's own, restated here from its written
 * definition (include/fia.h, "schedules"), independently of the CUDA code.
 */

#define OR_KV_TILE 128
#define OR_Q_TILE 128

static int64_t or_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* number of 128-wide KV tiles touched by the inclusive interval [lo, hi] */
static int64_t or_tiles(int64_t lo, int64_t hi)
{
    if (hi < lo) return 0;
    return hi / OR_KV_TILE - lo / OR_KV_TILE + 1;
}

/* Decode schedule (query rows per sequence S = max_seqlen_q, 1..16).  The
 * columns of a KV head hk of batch b are its (query row i, query head h of
 * the GQA group) pairs, numbered c = i*G + (h - hk*G); they are taken in
 * groups of GH = 16 (one query row, S = 1, and G > 8) or 8 (otherwise),
 * HG = ceil(S*G/GH) groups per KV head,
 * unit u = (b*KVN + hk)*HG + hg, UPB = KVN*HG units per batch.  Of these, the
 * HA(b) = ceil(q_len(b)*G/GH) first groups of every KV head hold columns
 * ("active"; A(b) = KVN*HA(b) of them, active index a = hk*HA(b) + hg).  All
 * active units of a batch cost the same: 0 when the batch has no query row,
 * else the number of KV tiles its rows can see together (the interval from
 * the first row's lower bound to the last row's upper bound), at least 1.
 * With T the sum of all active units' costs, n CTAs and W chunks per CTA:
 *   C  = max(1, ceil(T / (n*W))),  c2 = ceil(C/k), k = 2 for a bf16 cache
 *   and one query row (S = 1), else 1;
 *   a unit of cost c has n1 = max(0, floor(c/C) - 1) big chunks of C tiles,
 *   then its remaining c - n1*C tiles in small chunks of c2 tiles (the last
 *   one shorter), n2 of them.
 * Outputs (int64 sched[8 + 3(B+1) + B]): C, c2, N (all chunks), F (big
 * chunks), M (batches whose units have more than one chunk), the plan's
 * mark 0x4649414445434F44, B and the CTA count (so that execute can tell a
 * plan of its arguments from anything else in the workspace);
 * Q[b] = sum over b' < b of (n1+n2)(b')*A(b'), then R1[b] (big) and R2[b]
 * (small) the same sums of n1*A and n2*A, each array with B+1 entries; then
 * the M batches with more than one chunk per unit in increasing order,
 * followed by -1 up to B entries.  Chunk i of active unit a of batch b owns
 * partial slot Q[b] + i*A(b) + a.
 * The queue (N entries of four int32) lists for b = 0..B-1, chunk i =
 * 0..n1-1, active unit a = 0..A(b)-1 the entry (b | q_len(b) << 16,
 * i << 16 | u - b*UPB, kv_len(b), first query row of b), then the small
 * chunks in the same
 * nesting with i = n1..n1+n2-1.  Query lengths above S count as S.  Returns
 * N, or -1 if N > cap. */
int64_t oracle_decode_schedule(const oracle_fia_args *a, int32_t num_ctas, int32_t per_cta,
                               int64_t *sched, int32_t *queue, int64_t cap)
{
    int G = a->QN / a->KVN;
    int64_t S = a->max_seqlen_q;
    int GH = (S == 1 && G > 8) ? 16 : 8;
    int64_t HG = or_ceil_div(S * G, GH);
    int B = a->B, b;
    int64_t *Q = sched + 8, *R1 = Q + (B + 1), *R2 = R1 + (B + 1), *SB = R2 + (B + 1);
    int64_t nsplit = 0;
    int64_t *cost = (int64_t *)malloc(sizeof(int64_t) * (B > 0 ? B : 1));
    int64_t *ha = (int64_t *)malloc(sizeof(int64_t) * (B > 0 ? B : 1));
    int64_t T = 0, C, c2, q = 0, r1 = 0, r2 = 0, n = 0;
    for (b = 0; b < B; ++b) {
        int64_t ql, qs, kl, lo, hi, lo1, hi1, c = 0;
        fia_lengths(a, b, &ql, &qs, &kl);
        if (ql > S) ql = S;
        ha[b] = ql > 0 ? or_ceil_div(ql * G, GH) : 0;
        if (ql > 0) {
            if (kl > 0) {
                /* first row's lower bound, last row's upper bound */
                int v0 = fia_visible(a, ql, kl, 0, &lo, &hi);
                int v1 = fia_visible(a, ql, kl, ql - 1, &lo1, &hi1);
                (void)v0;
                (void)v1;
                if (lo < 0) lo = 0;
                if (hi1 > kl - 1) hi1 = kl - 1;
                c = or_tiles(lo, hi1);
            }
            if (c < 1) c = 1;
        }
        cost[b] = c;
        T += c * a->KVN * ha[b];
    }
    C = or_ceil_div(T, (int64_t)num_ctas * per_cta);
    if (C < 1) C = 1;
    {
        int64_t k = (a->kv_dtype == OR_KV_BF16 && S == 1) ? 2 : 1;
        c2 = (C + k - 1) / k;
    }
    for (b = 0; b < B; ++b) {
        int64_t n1 = 0, n2 = 0, A = a->KVN * ha[b];
        if (cost[b] > 0) {
            n1 = cost[b] / C - 1;
            if (n1 < 0) n1 = 0;
            n2 = or_ceil_div(cost[b] - n1 * C, c2);
        }
        Q[b] = q;
        R1[b] = r1;
        R2[b] = r2;
        SB[b] = -1;
        if (n1 + n2 > 1) SB[nsplit++] = b;
        q += (n1 + n2) * A;
        r1 += n1 * A;
        r2 += n2 * A;
    }
    Q[B] = q;
    R1[B] = r1;
    R2[B] = r2;
    sched[0] = C;
    sched[1] = c2;
    sched[2] = q;
    sched[3] = r1;
    sched[4] = nsplit;
    sched[5] = 0x4649414445434F44LL;  /* the plan's mark, then B and the CTA count */
    sched[6] = B;
    sched[7] = num_ctas;
    if (q > cap) {
        free(cost);
        free(ha);
        return -1;
    }
    /* big chunks, then small chunks */
    {
        int pass;
        for (pass = 0; pass < 2; ++pass)
            for (b = 0; b < B; ++b) {
                int64_t A = a->KVN * ha[b], i, k, ql, qs, kl, i0, i1;
                if (A == 0) continue;
                fia_lengths(a, b, &ql, &qs, &kl);
                if (ql > S) ql = S;
                if (pass == 0) {
                    i0 = 0;
                    i1 = (R1[b + 1] - R1[b]) / A;
                } else {
                    i0 = (R1[b + 1] - R1[b]) / A;
                    i1 = i0 + (R2[b + 1] - R2[b]) / A;
                }
                for (i = i0; i < i1; ++i)
                    for (k = 0; k < A; ++k) {
                        int64_t w = (k / ha[b]) * HG + k % ha[b];
                        queue[4 * n] = (int32_t)(b | (ql << 16));
                        queue[4 * n + 1] = (int32_t)((i << 16) | w);
                        queue[4 * n + 2] = (int32_t)kl;
                        queue[4 * n + 3] = (int32_t)qs;
                        ++n;
                    }
            }
    }
    free(cost);
    free(ha);
    return n;
}

/* Prefill work units in canonical order (b, q_tile, hk, pair) and their
 * costs.  Heads of one KV group are taken two at a time (pair = 2 heads;
 * when G is odd a pair holds one head).  The KV interval a 128-row query tile
 * [i0, i1] can see is bounded by its first and last rows: lo = max(0, lo(i0)),
 * hi = min(kv_len-1, hi(i1)) with lo(i) = p(i) - pre_tokens for the band mask
 * and 0 otherwise, hi(i) = p(i) for the causal masks, p(i) + next_tokens for
 * the band and kv_len-1 for modes 0 and 1 (p(i) = kv_len - q_len + i, or i for
 * the left-up causal mask; an explicit mask does not narrow it).  Both bounds
 * are monotone in the row, so this is the union of the rows' intervals.  The
 * cost of a unit is 1 plus the number of KV tiles that interval touches.  The
 * GPU orders units by non-increasing cost (ties in any order).  Writes
 * (b, q_tile, hk, pair) quadruples to units[4*k..] and cost[k]; returns the
 * number of units, or -1 when cap is too small. */
int64_t oracle_prefill_units(const oracle_fia_args *a, int32_t *units, int64_t *cost, int64_t cap)
{
    int G = a->QN / a->KVN;
    int per_pair = (G % 2 == 0) ? 2 : 1;
    int npairs = G / per_pair;
    int64_t n = 0;
    int b;
    for (b = 0; b < a->B; ++b) {
        int64_t ql, qs, kl, t, nt;
        fia_lengths(a, b, &ql, &qs, &kl);
        nt = or_ceil_div(ql, OR_Q_TILE);
        for (t = 0; t < nt; ++t) {
            int64_t i0 = t * OR_Q_TILE, i1 = (t + 1) * OR_Q_TILE - 1;
            int64_t p0, p1, lo, hi, c = 1;
            int hk, pr;
            if (i1 > ql - 1) i1 = ql - 1;
            p0 = (a->mask_mode == OR_MASK_LUC ? 0 : kl - ql) + i0;
            p1 = (a->mask_mode == OR_MASK_LUC ? 0 : kl - ql) + i1;
            lo = a->mask_mode == OR_MASK_BAND ? p0 - a->pre_tokens : 0;
            hi = (a->mask_mode == OR_MASK_RDC || a->mask_mode == OR_MASK_LUC) ? p1
               : a->mask_mode == OR_MASK_BAND ? p1 + a->next_tokens : kl - 1;
            if (lo < 0) lo = 0;
            if (hi > kl - 1) hi = kl - 1;
            if (kl > 0) c += or_tiles(lo, hi);
            for (hk = 0; hk < a->KVN; ++hk)
                for (pr = 0; pr < npairs; ++pr) {
                    if (n >= cap) return -1;
                    units[4 * n + 0] = b;
                    units[4 * n + 1] = (int32_t)t;
                    units[4 * n + 2] = hk;
                    units[4 * n + 3] = pr;
                    cost[n] = c;
                    ++n;
                }
        }
    }
    return n;
}

/* Sparse metadata ([SFMLA] sparse_flash_mla_metadata; fixed [1024] int32).
 * Work items are (query row u, group g of `heads` consecutive query heads),
 * numbered k = u * G + g with G = ceil(N1 / heads).  The weight of an item is
 * its row's chunk count: ceil(W/chunk) window chunks (W = win_left +
 * win_right + 1) plus ceil(kc/chunk) compressed chunks, kc = the visible
 * compressed rows capped at K2 (CSA), all of them (HCA), 0 (SWA).  With P_k
 * the summed weight of the items before k and T the total weight, CTA c
 * takes the items with floor(c*T/n) <= P_k < floor((c+1)*T/n); it begins at
 * item #{k : P_k < floor(c*T/n)}.  Layout:
 *   [0] 0x46534D32  [1] n  [2] rows  [3] chunk  [4] T  [5] B  [6] N1  [7] K2
 *   [8] cmp_ratio (1 without a compressed cache)  [9] win_left
 *   [10] win_right  [11] mode (0 SWA, 1 CSA, 2 HCA)  [12] heads  [13] items
 *   [14] K~ row format (0 bf16, 1 packed FP8)  [15] 0
 *   [16 + c]: first item of CTA c, c = 0..n;  the rest 0.
 * Returns 0, or -1 if n does not fit. */
int oracle_sparse_metadata(const oracle_sparse_args *a, int32_t num_ctas, int32_t chunk,
                           int32_t heads, int32_t *md)
{
    int64_t rows = a->layout == OR_LAYOUT_TND ? a->T1 : (int64_t)a->B * a->S1;
    int64_t W = (int64_t)a->win_left + a->win_right + 1, total = 0, u, c, k;
    int64_t G = or_ceil_div(a->N1, heads), items = rows * G;
    int64_t *P;
    int mode = !a->cmp_kv ? 0 : (a->cmp_sparse_indices ? 1 : 2);
    if (num_ctas < 1 || 17 + (int64_t)num_ctas > 1024) return -1;
    P = (int64_t *)malloc(sizeof(int64_t) * (size_t)(items + 1));
    for (u = 0; u < rows; ++u) {
        int b = 0;
        int64_t ql, qs, i, p, kc = 0, nch, g;
        if (a->layout == OR_LAYOUT_TND) {
            while (b + 1 <= a->B && a->cu_seqlens_q[b + 1] <= u) ++b;
            qs = a->cu_seqlens_q[b];
            ql = (int64_t)a->cu_seqlens_q[b + 1] - qs;
        } else {
            b = (int)(u / a->S1);
            qs = (int64_t)b * a->S1;
            ql = a->S1;
        }
        i = u - qs;
        p = (int64_t)a->seqused_kv[b] - ql + i;
        if (mode != 0) {
            kc = (p + 1) >= 0 ? (p + 1) / a->cmp_ratio : 0;
            if (mode == 1 && kc > a->K2) kc = a->K2;
        }
        nch = or_ceil_div(W, chunk) + or_ceil_div(kc, chunk);
        for (g = 0; g < G; ++g) {
            P[u * G + g] = total;
            total += nch;
        }
    }
    P[items] = total;
    memset(md, 0, sizeof(int32_t) * 1024);
    md[0] = 0x46534D32;
    md[1] = num_ctas;
    md[2] = (int32_t)rows;
    md[3] = chunk;
    md[4] = (int32_t)total;
    md[5] = a->B;
    md[6] = a->N1;
    md[7] = a->K2;
    md[8] = a->cmp_kv ? a->cmp_ratio : 1;  /* no compressed cache: 1 */
    md[9] = a->win_left;
    md[10] = a->win_right;
    md[11] = mode;
    md[12] = heads;
    md[13] = (int32_t)items;
    md[14] = a->kv_dtype;
    for (c = 0; c <= num_ctas; ++c) {
        int64_t theta = c * total / num_ctas, cnt = 0;
        for (k = 0; k < items; ++k) cnt += P[k] < theta;
        md[16 + c] = (int32_t)cnt;
    }
    free(P);
    return 0;
}

/* The same rows as oracle_fia, for a sample of (query row, head) pairs only
 * (full-size parity checks).  out: [n, D]; lse: [n]. */
int oracle_fia_sample(const oracle_fia_args *a, const int64_t *rows, const int32_t *heads,
                      int64_t n, double *out, double *lse, int nthreads)
{
    int64_t max_kv = 0, t;
    int b;
    for (b = 0; b < a->B; ++b) {
        int64_t ql, qs, kl;
        fia_lengths(a, b, &ql, &qs, &kl);
        if (kl > max_kv) max_kv = kl;
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *s_buf = (double *)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
#pragma omp for schedule(dynamic, 1)
        for (t = 0; t < n; ++t) {
            int64_t row = rows[t], ql, qs, kl;
            int bb = 0;
            if (a->layout == OR_LAYOUT_TND) {
                while (bb + 1 <= a->B && a->cu_seqlens_q[bb + 1] <= row) ++bb;
            } else {
                bb = (int)(row / a->S_q);
            }
            fia_lengths(a, bb, &ql, &qs, &kl);
            fia_row(a, bb, heads[t], row, ql, kl, row - qs, out + t * a->D, &lse[t], s_buf);
        }
        free(s_buf);
    }
    return 0;
}
