/*
 * fia.h -- C ABI of libfia: fused inference attention over a paged KV cache
 * for NVIDIA GB300 (sm_103a), and the shared-KV sparse attention variant.
 *
 * Operations
 *   FIA     O = softmax(Q K^T * scale + mask) V, per query head h against KV
 *           head floor(h / G), G = Q_N / KV_N ("aclnnFusedInferAttentionScoreV5",
 *           formula section; "...V2": an incremental branch for short queries
 *           and a prompt branch otherwise -- here a query of at most 16 rows
 *           per sequence runs the split-KV decode kernel, a longer one the
 *           prefill kernel; GQA needs Q_N divisible by KV_N with ratio <= 64).
 *   COMBINE the log-sum-exp join of partial results computed over disjoint
 *           key sets (fia_lse_combine; the softmax_lse use of "...V2" and the
 *           context-parallel example of "sparse_flash_mla").
 *   SPARSE  O = softmax(Q K~^T * softmax_scale) V~ with K~ = V~ gathered from a
 *           band window of the original KV and from compressed KV rows
 *           ("kv_quant_sparse_attn_sharedkv", formula and parameter table;
 *           "sparse_flash_mla", SWA / CSA / HCA modes).
 *
 * Calling convention (two phases, as on the pages: a first call checks the
 * inputs and sizes the workspace, a second call executes):
 *   fia_get_workspace_size -> fia_run        (fia_run = fia_plan + fia_execute)
 *   sparse_attn_metadata   -> sparse_attn_run
 * Every pointer in a params struct is a DEVICE pointer unless stated
 * otherwise.  The caller owns every buffer; the library never allocates,
 * never synchronises the host and launches only on the given stream, so the
 * execute calls can be captured in a CUDA graph.  All functions return a
 * status code; no C++ exception crosses this boundary.  `stream` is a
 * cudaStream_t passed as void* (NULL = the legacy default stream).
 *
 * Readings where the pages are silent (they are restated in the design notes):
 *  - query rows are aligned to the bottom-right corner of the score matrix:
 *    row i of a sequence sits at KV position p = kv_len - q_len + i;
 *  - mask modes: 0 none (or an explicit mask); 1 the explicit mask; 2
 *    left-up causal (j <= i); 3 right-down causal (j <= p); 4 band
 *    (p - pre_tokens <= j <= p + next_tokens);
 *  - a sink is one extra logit per query head that enters the softmax
 *    denominator only (not multiplied by scale, carries no value); lse
 *    includes it;
 *  - a row that sees no key (empty KV, or fully masked) gets O = 0 and
 *    lse = +inf, with or without a sink ("...V4" empty-tensor rule; "...V2"
 *    invalid-row correction);
 *  - FP8 KV: E4M3 codes with one fp32 scale per 64 consecutive elements of D,
 *    value = code * scale; sparse packed FP8 rows carry E8M0 tile scales.
 */
#ifndef FIA_H_
#define FIA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FIA_ABI_VERSION 3

/* Status codes ("...V5" two-phase API: the first phase validates the inputs
 * and reports errors before anything is launched). */
typedef int fia_status;
#define FIA_OK 0
#define FIA_ERR_NULL_ARG 1            /* a required pointer is NULL                  */
#define FIA_ERR_BAD_SHAPE 2           /* a size, stride, alignment or attribute is   */
                                      /* out of range or inconsistent                */
#define FIA_ERR_BAD_DTYPE 3           /* unknown kv_dtype                            */
#define FIA_ERR_UNSUPPORTED 4         /* valid on the pages, not built here          */
#define FIA_ERR_WORKSPACE_TOO_SMALL 5 /* workspace NULL or smaller than required     */
#define FIA_ERR_CUDA 6                /* a CUDA runtime/driver call failed           */

#define FIA_LAYOUT_BSND 0 /* q/out [B, S, N, D]                                   */
#define FIA_LAYOUT_TND 1  /* q/out [T, N, D] with cu_seqlens_q [B+1]               */

#define FIA_KV_BF16 0
#define FIA_KV_FP8_E4M3 1

/* Mask modes ("...V5" Attention Mask group, sparseMode 0-4).  Row i of a
 * sequence with q_len query rows and kv_len keys sees key j (0 <= j < kv_len)
 * when:
 *   0 NONE               every key; with atten_mask, where the mask byte is 0
 *   1 ALL_MASK           where the mask byte is 0 (atten_mask required)
 *   2 LEFT_UP_CAUSAL     j <= i            (the diagonal from the top-left)
 *   3 RIGHT_DOWN_CAUSAL  j <= p, p = kv_len - q_len + i
 *   4 BAND               p - pre_tokens <= j <= p + next_tokens
 * Modes 2-4 are computed from positions; the pages pass them a fixed
 * 2048 x 2048 mask that encodes the same rule, which this library neither
 * needs nor reads (atten_mask must be NULL there). */
#define FIA_MASK_NONE 0
#define FIA_MASK_ALL 1
#define FIA_MASK_LEFT_UP_CAUSAL 2
#define FIA_MASK_RIGHT_DOWN_CAUSAL 3
#define FIA_MASK_BAND 4

/* Paged KV cache layouts ("...V5" Paged Attention group). */
#define FIA_KV_LAYOUT_BNBSH 0  /* [num_blocks, block_size, KV_N, D] (H = KV_N*D)  */
#define FIA_KV_LAYOUT_BNNBSD 1 /* [num_blocks, KV_N, block_size, D]             */

/* Fused inference attention parameters.
 *
 * Shapes and limits ("...V2", restrictions when Q_S > 1: B <= 65536, N <= 256,
 * D <= 512, S <= 20M; GQA ratio <= 64).  Built here: D in {64, 128}.
 *
 * KV cache ("...V2" page-attention scenario; "...V5" Paged Attention group):
 *  - paged (block_table != NULL): k_cache/v_cache are pools
 *    [num_blocks, block_size, KV_N, D] (BnBsH); logical row j of batch b is
 *    pool row block_table[b*max_blocks_per_seq + j/block_size]*block_size
 *    + j%block_size.  Block ids are not validated; table entries past a
 *    sequence's last block are never read.  seqused_kv is required.
 *    block_size: multiple of 16, <= 1024 (FP8: multiple of 32, <= 512).
 *  - contiguous (block_table == NULL): k_cache/v_cache are [B, max_seqlen_kv,
 *    KV_N, D]; seqused_kv optional (default max_seqlen_kv for every batch).
 *  - FP8: k_scale/v_scale fp32, head-major inside each page:
 *    [num_blocks, KV_N, block_size, D/64] (paged) or [B, KV_N, max_seqlen_kv,
 *    D/64] (contiguous; max_seqlen_kv even).  This is the page-managed
 *    per-token, per-head scale shape (blockNum, N, blockSize) of the "V5"
 *    dequantisation parameter group (DequantChecker), and its non-paged form
 *    (B, N, KV_S), with the D/64 tiles of a row as the last axis.
 * Alignment: q, out, k_cache, v_cache, k_scale, v_scale 16-byte aligned;
 * token strides multiples of 8 elements. */
typedef struct fia_params {
    int32_t batch;            /* B                                             */
    int32_t num_q_heads;      /* Q_N                                           */
    int32_t num_kv_heads;     /* KV_N                                          */
    int32_t head_dim;         /* D                                             */
    int32_t layout;           /* FIA_LAYOUT_*                                  */
    int32_t max_seqlen_q;     /* BSND: S_q.  TND: upper bound of the query     */
                              /* lengths (1 selects the decode branch)         */
    int32_t total_q;          /* TND: T (rows of q and out); BSND: ignored     */
    int32_t pad0_;
    const void *q;            /* bf16                                          */
    void *out;                /* bf16, same layout and strides as q            */
    float *lse;               /* fp32, nullable: BSND [B,Q_N,S_q,1],           */
                              /* TND [T,Q_N,1]                                 */
    int64_t q_token_stride;   /* elements between tokens of q (0: Q_N*D)       */
    int64_t out_token_stride; /* elements between tokens of out (0: Q_N*D)     */
    const void *k_cache;
    const void *v_cache;
    const float *k_scale;     /* FP8 only                                      */
    const float *v_scale;     /* FP8 only                                      */
    int32_t kv_dtype;         /* FIA_KV_*                                      */
    int32_t quant_tile;       /* FP8: 64                                       */
    const int32_t *block_table;   /* int32 [B, max_blocks_per_seq] or NULL     */
    int32_t max_blocks_per_seq;
    int32_t block_size;
    int32_t num_blocks;
    int32_t max_seqlen_kv;    /* contiguous KV: S_kv; paged: ignored           */
    const int32_t *cu_seqlens_q;  /* TND: int32 [B+1], non-decreasing, last=T */
    const int32_t *seqused_kv;    /* int32 [B]: KV length of each batch        */
    float scale;              /* multiplies Q K^T (typically 1/sqrt(D))         */
    int32_t mask_mode;        /* FIA_MASK_*                                    */
    int32_t pre_tokens;       /* band: keys before p (may be negative)         */
    int32_t next_tokens;      /* band: keys after p;  pre + next >= 0          */
    const float *sinks;       /* fp32 [Q_N] or NULL                            */
    int32_t num_sms;          /* persistent CTAs; 0 = the device's SM count    */
    int32_t kv_layout;        /* FIA_KV_LAYOUT_* (paged caches)                */
    const uint8_t *atten_mask;    /* modes 0/1: int8/uint8/bool bytes, nonzero  */
                              /* = masked out; element (b, i, j) at            */
                              /* b*mask_batch_stride + i*mask_row_stride + j    */
    int64_t mask_batch_stride;    /* bytes; 0 = one [S_q, S_kv] mask for all B  */
    int64_t mask_row_stride;      /* bytes, a multiple of 16, >= the KV capacity */
                              /* (paged: max_blocks_per_seq * block_size)        */
    int32_t reserved[8];      /* must be 0                                     */
} fia_params;

/* Returns a static string naming a status code. */
const char *fia_status_string(fia_status s);

/* Version of this ABI (FIA_ABI_VERSION). */
int32_t fia_abi_version(void);

/* sizeof(fia_params), sizeof(sparse_attn_params) and sizeof(fia_combine_params)
 * as compiled into the library, so that a binding can check its mirror of the
 * structs. */
size_t fia_sizeof_params(void);
size_t fia_sizeof_sparse_params(void);
size_t fia_sizeof_combine_params(void);

/* Phase 1 ("...V5": the GetWorkspaceSize call validates the inputs and
 * computes the workspace).  Host-only, pure, idempotent: reads only the
 * struct's scalar fields and checks pointers for NULL and alignment (it never
 * dereferences a device pointer).  *bytes receives the workspace size that
 * fia_plan / fia_execute / fia_run need; the size depends only on scalar
 * fields, never on device-side lengths. */
fia_status fia_get_workspace_size(const fia_params *p, size_t *bytes);

/* Phase 2a: launch the tile scheduler on `stream`.  It reads the device-side
 * lengths (seqused_kv, cu_seqlens_q) and writes into `workspace` the balanced
 * split of (batch, kv-head, q-tile, kv-split) work items across persistent
 * CTAs, and resets the counters fia_execute uses.  The plan stays valid for
 * later fia_execute calls with the same shapes and lengths (e.g. every layer
 * of a model step). */
fia_status fia_plan(const fia_params *p, void *workspace, size_t workspace_bytes,
                    void *stream);

/* Phase 2b: launch the attention kernels on `stream` using the plan in
 * `workspace`.  Writes every element of out (and lse when non-NULL).
 * Deterministic: the same inputs give bitwise the same outputs.
 * Device error word: the first int32 of the workspace is 0 after a clean
 * execute; 1 when a bounded wait inside a kernel gave up (about 2 s; the
 * kernel returned early and the outputs are undefined); 2 when the
 * workspace holds no plan of these arguments (never planned, planned with
 * other shapes, or planned for the other branch since: a decode plan clears
 * the prefill plan's mark and a decode execute runs nothing while that mark
 * is set; nothing ran), when a plan entry lies outside these arguments (that
 * entry ran as empty, its loads and stores kept inside their buffers), or
 * when a decode plan held more chunks than the workspace bound (not
 * reachable for validated inputs); 3, only with FIA_DEBUG set in the
 * environment (any value not starting with '0', read on every call), when a
 * block_table entry for a key position the kernels read names a page outside
 * [0, num_blocks) -- those rows are read as zeros either way; the word then
 * stays 3 until the next plan.  Reading it needs a device-to-host copy after
 * the stream has reached the call. */
fia_status fia_execute(const fia_params *p, void *workspace, size_t workspace_bytes,
                       void *stream);

/* Phase 2: fia_plan followed by fia_execute. */
fia_status fia_run(const fia_params *p, void *workspace, size_t workspace_bytes, void *stream);

/* Decode without a workspace.  The pages have no counterpart to this call; it
 * exists for callers that cannot allocate device memory when they run
 * attention (a device fully owned by another component's memory pool, a host
 * process that forbids allocations after start-up, a latency-critical path
 * that must not touch the allocator).  It behaves like fia_run on the decode
 * branch but keeps the scheduler's scratch -- the plan, the split-KV counters
 * and the partial slots -- in a device array of FIA_NOALLOC_SCRATCH_BYTES
 * compiled into the library, which every GPU that loads libfia holds until
 * the process exits.  It allocates nothing.
 *  - status (nullable, a device int32 the caller owns): receives, in stream
 *    order after the kernels, the error word fia_execute documents (0 clean,
 *    1 a bounded wait gave up, 2 a plan problem); 0 when there was nothing to
 *    run.  Without it a failure inside the kernels cannot be seen, since the
 *    word lives in the library's array.
 *  - Returns FIA_ERR_WORKSPACE_TOO_SMALL, before launching anything, when the
 *    decode plan needs more than FIA_NOALLOC_SCRATCH_BYTES (what fia_get_
 *    workspace_size reports for the same params), FIA_ERR_UNSUPPORTED for the
 *    prefill branch, and any status fia_run returns.
 *  - Every call looks up the array's device address in the current context;
 *    the first call on a device loads the library's device code there, so
 *    make that first call before any stream capture.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents; every value that must start at zero is reset by the call.
 *    Calls that overlap on the GPU (unordered streams) race on the array. */
#define FIA_NOALLOC_SCRATCH_BYTES (8u << 20)
fia_status fia_decode_run_noalloc(const fia_params *p, int32_t *status, void *stream);

/* Log-sum-exp combine of partial attention results over disjoint key sets:
 * the use of softmax_lse that "...V2" names (softmax_lse restriction: the
 * ring-attention algorithm), i.e. the exchange step of context parallelism
 * with the KV cut across ranks ("sparse_flash_mla", CP example).  Given
 * n_parts results (O_k, lse_k) of the same query rows against disjoint parts
 * of the keys, it writes the result against their union:
 *   lse = log sum_k exp(lse_k),   O = sum_k exp(lse_k - lse) * O_k.
 * Parts with lse_k = +inf saw no key and are skipped; when every part is
 * skipped, O = 0 and lse = +inf (the empty-row rule).  Sinks: run every part
 * without them and pass them here (fp32 [N], nullable); each enters the sum
 * once as one more logit that carries no value,
 *   lse = log(sum_k exp(lse_k) + exp(sink_h)),
 * which gives the result of one call over all keys with the sinks (a part
 * that kept the sink would lose it whenever that part sees no key).
 * Layouts are those of fia_params' out and lse: O bf16 [tokens, N, D] (BSND
 * tokens = B * S_q, TND tokens = T) and lse fp32 BSND [B, N, S_q] or TND
 * [T, N].  o_parts and lse_parts are HOST arrays of n_parts DEVICE pointers
 * (16-byte aligned O, 4-byte aligned lse); out may alias none of the parts.
 * Deterministic: parts are folded in index order.  Errors: FIA_ERR_NULL_ARG,
 * FIA_ERR_BAD_SHAPE (n_parts outside 1..FIA_COMBINE_MAX_PARTS, D not a
 * multiple of 8 or above 512, sizes out of range, misalignment),
 * FIA_ERR_CUDA for a failed launch. */
#define FIA_COMBINE_MAX_PARTS 16
typedef struct fia_combine_params {
    int32_t n_parts;
    int32_t layout;           /* FIA_LAYOUT_BSND | FIA_LAYOUT_TND              */
    int32_t batch;            /* BSND: B                                       */
    int32_t seqlen_q;         /* BSND: S_q                                     */
    int32_t total_q;          /* TND: T                                        */
    int32_t num_heads;        /* N                                             */
    int32_t head_dim;         /* D                                             */
    int32_t pad0_;
    const void *const *o_parts;     /* host array [n_parts] of device pointers */
    const float *const *lse_parts;  /* host array [n_parts] of device pointers */
    void *out;                /* bf16 [tokens, N, D]                           */
    float *lse;               /* fp32, nullable                                */
    const float *sinks;       /* fp32 [N], nullable                            */
    int32_t reserved[8];      /* must be 0                                     */
} fia_combine_params;
fia_status fia_lse_combine(const fia_combine_params *p, void *stream);

/* Self-test of the bounded wait that every pipeline barrier of this library
 * uses (failure detection without a GPU fault): launches, on `stream`, one
 * warp that waits on a shared-memory barrier nothing ever completes, with a
 * time limit of `limit_ns` (1 ms .. 1 s) instead of the pipelines' 2 s.
 * `status` (device int32 [3], caller-owned) receives: [0] the error word
 * (1 = the wait gave up, as the pipelines report it), [1] microseconds
 * waited, [2] 1 if the wait had completed (never).  The kernel returns after
 * the time-out and the context stays usable.  FIA_ERR_NULL_ARG for a null
 * status, FIA_ERR_BAD_SHAPE for a limit out of range, FIA_ERR_CUDA if the
 * launch fails. */
fia_status fia_selftest_bounded_wait(int32_t *status, uint64_t limit_ns, void *stream);

/* Workspace layout of the plan, for inspection (host-only).
 *
 * Decode schedule (written by fia_plan): the columns of a KV head are its
 * (query row, query head) pairs, S*G of them (S = max_seqlen_q <= 16), taken
 * in groups of GH = 16 (S = 1 and G > 8) or 8 (otherwise); work unit
 * u = (b, kv head, group),
 * UPB = KV_N * ceil(S*G/GH) units per batch, of which the first
 * A(b) = KV_N * ceil(q_len(b)*G/GH) hold columns of batch b ("active", active
 * index a).  Cost of an active unit = KV tiles (128 positions) its rows see
 * together, at least 1 (0 when the batch has no query row).  With T the total
 * cost, n CTAs and W = 5 chunks per CTA, C = max(1, ceil(T / (n W))) and
 * c2 = ceil(C / k), k = 2 for a bf16 cache and S = 1, else 1.  A unit of
 * cost c gets n1 = max(0, floor(c/C) - 1) chunks of C tiles, then chunks of
 * c2 tiles over the rest (at most 2k), so n W + 2k U bounds the chunks of U
 * units.
 * sched holds int64 {C, c2, chunks N, big chunks F, split batches M, plan
 * mark 0x4649414445434F44, B, CTA count}, then Q[B+1] (partial slots before
 * batch b: chunk i of active unit a of batch b owns slot Q[b] + i*A(b) + a),
 * then R1[B+1] and R2[B+1] (big and small chunks before batch b), then the M
 * batches whose units have several chunks (ascending; -1 after).  The claim
 * queue lists the big chunks, batch-major then chunk then active unit,
 * followed by the small chunks in the same order; entry = four int32
 * (b | q_len(b) << 16, i << 16 | u - b*UPB, KV length of b, first token row
 * of b). */
typedef struct fia_plan_layout {
    int32_t branch;           /* 1 decode (split-KV), 2 prefill                */
    int32_t num_ctas;         /* persistent CTAs                               */
    int64_t num_units;        /* decode: units; prefill: bound on units        */
    int64_t max_chunks;       /* decode: partial slots, bound on chunks        */
    int64_t sched_off;        /* decode: int64 [8 + 3(B+1) + B] schedule       */
    int64_t queue_off;        /* decode: int32 [max_chunks][4] claim queue     */
    int64_t unit_list_off;    /* prefill: int32 [num_units][2] ordered units   */
    int64_t total_bytes;
} fia_plan_layout;
fia_status fia_get_plan_layout(const fia_params *p, fia_plan_layout *layout);

/* ------------------------------------------------------------------------ */
/* shared-KV sparse attention                                               */
/* ------------------------------------------------------------------------ */

/* KV row formats of the sparse variant ("kv_quant_sparse_attn_sharedkv",
 * parameter table: kv_quant_mode 1 = per-tile quantised nope part, tile_size,
 * rope_head_dim; constraint on the D of ori_kv / cmp_kv):
 *  - BF16: a row is D bf16 values.
 *  - FP8_PACKED: a row is 640 bytes for a query D of 512: the 64 rope values
 *    as bf16 (128 bytes), then the 448 nope values as E4M3 codes (448 bytes),
 *    then the 7 per-64 nope tile scales as E8M0 bytes (value 2^(e - 127),
 *    e = 255 is NaN), then 57 bytes of padding.  Element d of the row is the
 *    rope value for d < 64 and e4m3(code[d - 64]) * 2^(scale[(d - 64)/64] -
 *    127) after.  The pool is bytes [num_blocks, block_size, 1, 640]. */
#define FIA_SPARSE_KV_BF16 0
#define FIA_SPARSE_KV_FP8_PACKED 1
#define FIA_SPARSE_PACKED_ROW_BYTES 640

/* Parameters ("kv_quant_sparse_attn_sharedkv" parameter table and
 * constraints; "sparse_flash_mla" modes):
 *  - q bf16 BSND [B, S1, N1, D] or TND [T1, N1, D]; out the same; KV_N = 1.
 *  - ori_kv bf16 [ori_num_blocks, ori_block_size, 1, D] with ori_block_table
 *    int32 [B, >= ceil(S2_max/ori_block_size)] (required).
 *  - cmp_kv bf16 [cmp_num_blocks, cmp_block_size, 1, D] with cmp_block_table
 *    int32 [B, >= ceil(floor(S2_max/cmp_ratio)/cmp_block_size)]; NULL for SWA.
 *  - cmp_sparse_indices int32 [rows, 1, topk]: logical compressed rows, valid
 *    entries first, -1 after; NULL with cmp_kv given selects HCA (every
 *    causally visible compressed row).
 *  - seqused_kv int32 [B]: S2 of each batch (required).
 *  - query row i of batch b sits at p = S2 - q_len + i; window rows
 *    p - ori_win_left .. p + ori_win_right of ori_kv; compressed row c is
 *    visible iff (c+1)*cmp_ratio <= p+1.
 *  - sinks fp32 [N1] or NULL; lse fp32 [B, 1, S1, N1] / [1, T1, N1] or NULL.
 * Built here: D = 512 (the pages' only value) and D in {128, 256}; N1 a power
 * of two <= 128; block sizes multiples of 16, <= 1024; topk <= 2048; K~ rows
 * in bf16, or packed FP8 (kv_dtype FIA_SPARSE_KV_FP8_PACKED, D = 512,
 * tile_size = rope_head_dim = 64, ori_kv and cmp_kv bytes [nb, bs, 1, 640]). */
typedef struct sparse_attn_params {
    int32_t batch;            /* B                                             */
    int32_t num_q_heads;      /* N1                                            */
    int32_t head_dim;         /* D                                             */
    int32_t layout;           /* FIA_LAYOUT_BSND | FIA_LAYOUT_TND              */
    int32_t max_seqlen_q;     /* BSND: S1; TND: upper bound of query lengths   */
    int32_t total_q;          /* TND: T1                                       */
    const void *q;
    void *out;
    float *lse;
    const void *ori_kv;
    const int32_t *ori_block_table;
    int32_t ori_max_blocks;
    int32_t ori_block_size;
    int32_t ori_num_blocks;
    int32_t pad0_;
    const void *cmp_kv;
    const int32_t *cmp_block_table;
    int32_t cmp_max_blocks;
    int32_t cmp_block_size;
    int32_t cmp_num_blocks;
    int32_t topk;             /* K2 (CSA)                                      */
    const int32_t *cmp_sparse_indices;
    const int32_t *cu_seqlens_q;  /* TND [B+1]                                 */
    const int32_t *seqused_kv;    /* [B]                                       */
    const float *sinks;
    float softmax_scale;
    int32_t cmp_ratio;        /* 1 for SWA; 4 (CSA) or 128 (HCA) on the pages  */
    int32_t ori_win_left;     /* 127 on the pages                              */
    int32_t ori_win_right;    /* 0 on the pages                                */
    int32_t num_sms;          /* CTAs of the split; 0 = the device's SM count  */
    int32_t kv_dtype;         /* FIA_SPARSE_KV_* (ori_kv and cmp_kv alike)     */
    int32_t tile_size;        /* packed FP8 rows: 64 (nope quantisation tile)  */
    int32_t rope_head_dim;    /* packed FP8 rows: 64                           */
    int32_t reserved[8];      /* must be 0                                     */
} sparse_attn_params;

/* Metadata step ("sparse_flash_mla_metadata": generates, before the main call,
 * the task list of every core; "kv_quant_sparse_attn_sharedkv": metadata
 * int32 [1024]).  Validates p, launches the scheduler kernel on `stream`,
 * which writes `metadata` (device int32 [1024], 16-byte aligned, else
 * FIA_ERR_BAD_SHAPE -- in this call and in sparse_attn_run), and stores the
 * workspace size that sparse_attn_run needs in *workspace_bytes (host; the
 * status word only).  A work item is (query row u, group g of 8 query heads),
 * numbered k = u * G + g with G = ceil(N1 / 8); it weighs its row's chunk
 * count ceil(W/64) + ceil(kc/64) (W = win_left + win_right + 1, kc = visible
 * compressed rows, capped at topk for CSA, 0 for SWA).  With P_k the weight
 * before item k and T the total, CTA c takes the items with
 * floor(c*T/n) <= P_k < floor((c+1)*T/n).  Layout of metadata:
 *   [0] 0x46534D32  [1] n = CTAs  [2] query rows  [3] chunk rows (64)
 *   [4] T  [5] B  [6] N1  [7] topk  [8] cmp_ratio (1 without cmp_kv)
 *   [9] win_left  [10] win_right  [11] mode (0 SWA, 1 CSA, 2 HCA)
 *   [12] heads per item (8)  [13] items  [14] kv_dtype  [15] 0
 *   [16 + c]: first item of CTA c, c = 0..n;  remaining entries 0.
 * A query row's K~ is processed whole by one CTA, in order, so results do
 * not depend on the other rows of the batch ("sparse_flash_mla":
 * deterministic and batch invariant by default).  n is capped at 1007 so
 * that the list fits. */
fia_status sparse_attn_metadata(const sparse_attn_params *p, int32_t *metadata,
                                size_t *workspace_bytes, void *stream);

/* Main call: launches the gather-attention kernel on `stream`; `workspace`
 * needs the size sparse_attn_metadata reported.
 * `metadata` must come from sparse_attn_metadata with the same shapes.  The
 * kernel checks its header (magic, CTA count, rows, B, N1, topk, heads per
 * item, items, kv_dtype) on the device; on a mismatch it writes nothing to out/lse and sets the int32
 * status word at workspace offset 0 to FIA_ERR_BAD_SHAPE (0 otherwise; read
 * it with any device-to-host copy after the call).  With FIA_DEBUG set in the
 * environment the word is also 3 when a window or listed compressed row's
 * page lies outside its block table or pool (such rows are left out either
 * way). */
fia_status sparse_attn_run(const sparse_attn_params *p, const int32_t *metadata,
                           void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FIA_H_ */
