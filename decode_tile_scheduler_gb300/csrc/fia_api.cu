// fia_api.cu -- host side of libfia: the C ABI declared in include/fia.h.
// Validation and workspace sizing follow the two-phase convention of the FIA
// pages ("aclnnFusedInferAttentionScoreV5": GetWorkspaceSize checks the
// inputs and computes the workspace; the execute call runs); launches go to
// the caller's stream only, and nothing here allocates or synchronises.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/fia.h"
#include "internal.h"

using namespace fia;

namespace {

constexpr int64_t kAlign = 256;
int64_t align_up(int64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int gcd_i(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Multiplier and shift with j / d == (j * magic) >> shift for 0 <= j < 2^31,
// 1 <= d <= 2^20: l = ceil(log2 d), magic = floor(2^(31+l) / d) + 1 (the
// round-up method; magic * d - 2^(31+l) <= d <= 2^l keeps it exact, and
// magic < 2^32).
void fast_divisor(int d, uint32_t* magic, int* shift) {
  int l = 0;
  while ((1 << l) < d) ++l;
  *magic = (uint32_t)(((uint64_t)1 << (31 + l)) / (uint64_t)d + 1);
  *shift = 31 + l;
}

// ---------------------------------------------------------------------------
// device properties and the tensor-map encoder (driver entry point)
// ---------------------------------------------------------------------------
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

fia_status get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return FIA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  *fn = g_encode;
  return FIA_OK;
}

fia_status sm_count(int requested, int* n) {
  if (requested > 0) {
    *n = requested;
    return FIA_OK;
  }
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FIA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FIA_ERR_CUDA;
  *n = v;
  return FIA_OK;
}

// 2-D tiled map over a row-major [rows, cols] matrix with 128-byte swizzling.
fia_status make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                    uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
                    uint64_t row_stride_elems,
                    CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  fia_status st = get_encoder(&enc);
  if (st != FIA_OK) return st;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_elems * (uint64_t)esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FIA_OK : FIA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// FIA validation ("...V5" constraint catalogue, the parts this library builds)
// ---------------------------------------------------------------------------
// The decode kernel takes sequences of up to kDecodeMaxRows query rows (the
// incremental branch; multi-token decode); longer ones run on the prefill kernel.
bool is_decode(const fia_params* p) {
  return p->max_seqlen_q >= 1 && p->max_seqlen_q <= kDecodeMaxRows;
}

int64_t q_rows_of(const fia_params* p) {
  return p->layout == FIA_LAYOUT_TND ? (int64_t)p->total_q
                                     : (int64_t)p->batch * p->max_seqlen_q;
}

int64_t kv_capacity_of(const fia_params* p) {
  return p->block_table ? (int64_t)p->max_blocks_per_seq * p->block_size : p->max_seqlen_kv;
}

fia_status validate(const fia_params* p) {
  if (!p) return FIA_ERR_NULL_ARG;
  for (int i = 0; i < 8; ++i)
    if (p->reserved[i] != 0) return FIA_ERR_BAD_SHAPE;
  if (p->batch < 1 || p->batch > 65536) return FIA_ERR_BAD_SHAPE;
  if (p->num_q_heads < 1 || p->num_q_heads > 256) return FIA_ERR_BAD_SHAPE;
  if (p->num_kv_heads < 1 || p->num_kv_heads > 256) return FIA_ERR_BAD_SHAPE;
  if (p->num_q_heads % p->num_kv_heads) return FIA_ERR_BAD_SHAPE;
  if (p->num_q_heads / p->num_kv_heads > 64) return FIA_ERR_BAD_SHAPE;
  if (p->head_dim < 1 || p->head_dim > 512) return FIA_ERR_BAD_SHAPE;
  if (p->layout != FIA_LAYOUT_BSND && p->layout != FIA_LAYOUT_TND) return FIA_ERR_BAD_SHAPE;
  if (p->max_seqlen_q < 0 || p->max_seqlen_q > 20971520) return FIA_ERR_BAD_SHAPE;
  if (p->layout == FIA_LAYOUT_TND) {
    if (p->total_q < 0) return FIA_ERR_BAD_SHAPE;
    if (!p->cu_seqlens_q) return FIA_ERR_NULL_ARG;
  }
  if (p->kv_dtype != FIA_KV_BF16 && p->kv_dtype != FIA_KV_FP8_E4M3) return FIA_ERR_BAD_DTYPE;
  if (p->mask_mode < FIA_MASK_NONE || p->mask_mode > FIA_MASK_BAND) return FIA_ERR_BAD_SHAPE;
  // an explicit mask goes with modes 0 and 1 only; mode 1 needs one
  if (p->mask_mode == FIA_MASK_ALL && !p->atten_mask) return FIA_ERR_NULL_ARG;
  if (p->atten_mask && p->mask_mode != FIA_MASK_NONE && p->mask_mode != FIA_MASK_ALL)
    return FIA_ERR_BAD_SHAPE;
  if (p->atten_mask) {
    if (!aligned16(p->atten_mask) || p->mask_row_stride <= 0 || p->mask_row_stride % 16 ||
        p->mask_batch_stride < 0 || p->mask_batch_stride % 16)
      return FIA_ERR_BAD_SHAPE;
  }
  if (p->kv_layout != FIA_KV_LAYOUT_BNBSH && p->kv_layout != FIA_KV_LAYOUT_BNNBSD)
    return FIA_ERR_BAD_SHAPE;
  if (p->kv_layout == FIA_KV_LAYOUT_BNNBSD && !p->block_table) return FIA_ERR_BAD_SHAPE;
  if (p->mask_mode == FIA_MASK_BAND && (int64_t)p->pre_tokens + p->next_tokens < 0)
    return FIA_ERR_BAD_SHAPE;
  if (!std::isfinite(p->scale)) return FIA_ERR_BAD_SHAPE;
  if (p->num_sms < 0 || p->num_sms > 4096) return FIA_ERR_BAD_SHAPE;
  if (p->q_token_stride < 0 || p->out_token_stride < 0) return FIA_ERR_BAD_SHAPE;
  const int64_t ND = (int64_t)p->num_q_heads * p->head_dim;
  if (p->q_token_stride && (p->q_token_stride < ND || p->q_token_stride % 8)) return FIA_ERR_BAD_SHAPE;
  if (p->out_token_stride && (p->out_token_stride < ND || p->out_token_stride % 8))
    return FIA_ERR_BAD_SHAPE;
  if (!p->q || !p->out || !p->k_cache || !p->v_cache) return FIA_ERR_NULL_ARG;
  if (!aligned16(p->q) || !aligned16(p->out) || !aligned16(p->k_cache) || !aligned16(p->v_cache))
    return FIA_ERR_BAD_SHAPE;
  if (p->lse && (reinterpret_cast<uintptr_t>(p->lse) & 3u)) return FIA_ERR_BAD_SHAPE;
  if (p->kv_dtype == FIA_KV_FP8_E4M3) {
    if (!p->k_scale || !p->v_scale) return FIA_ERR_NULL_ARG;
    if (p->quant_tile != 64) return FIA_ERR_BAD_SHAPE;
    if (p->head_dim % 64) return FIA_ERR_BAD_SHAPE;
    if (!aligned16(p->k_scale) || !aligned16(p->v_scale)) return FIA_ERR_BAD_SHAPE;
    // scale pieces of a contiguous cache are copied in 16-byte units
    if (!p->block_table && (p->max_seqlen_kv & 1)) return FIA_ERR_BAD_SHAPE;
  }
  if (p->block_table) {
    if (!p->seqused_kv) return FIA_ERR_NULL_ARG;
    if (p->block_size <= 0 || p->block_size % 16 || p->block_size > 1024) return FIA_ERR_BAD_SHAPE;
    if (p->kv_dtype == FIA_KV_FP8_E4M3 && (p->block_size % 32 || p->block_size > 512))
      return FIA_ERR_BAD_SHAPE;
    if (p->num_blocks <= 0 || p->max_blocks_per_seq <= 0) return FIA_ERR_BAD_SHAPE;
    if ((int64_t)p->num_blocks * p->block_size *
            (p->kv_layout == FIA_KV_LAYOUT_BNNBSD ? p->num_kv_heads : 1) > INT32_MAX)
      return FIA_ERR_BAD_SHAPE;
    if ((int64_t)p->max_blocks_per_seq * p->block_size > 20971520) return FIA_ERR_BAD_SHAPE;
  } else {
    if (p->max_seqlen_kv < 0 || p->max_seqlen_kv > 20971520) return FIA_ERR_BAD_SHAPE;
    if ((int64_t)p->batch * p->max_seqlen_kv > INT32_MAX) return FIA_ERR_BAD_SHAPE;
  }
  if (p->atten_mask) {
    // every row of a sequence reaches the mask row of its query index, and
    // every key position below the KV capacity
    if (p->mask_row_stride < kv_capacity_of(p)) return FIA_ERR_BAD_SHAPE;
  }
  // what is built
  if (p->head_dim != 64 && p->head_dim != 128) return FIA_ERR_UNSUPPORTED;
  if (p->kv_dtype == FIA_KV_FP8_E4M3 && p->head_dim != 128) return FIA_ERR_UNSUPPORTED;
  return FIA_OK;
}


struct DecodePlan {
  int n;
  int64_t U, max_chunks;
  int64_t off_sched, off_queue, off_part, total;
};

// FIA_DEBUG=1 (or any value not starting with 0) in the environment, read on
// every call: the kernels also report a block_table entry that names a page
// outside the pool for a position they read, with 3 in the error word (they
// read such rows as zeros, or leave them out, either way).
int debug_checks() {
  const char* e = getenv("FIA_DEBUG");
  return e && e[0] && e[0] != '0';
}

// The divisor k of the decode schedule's small chunks (c2 = ceil(C / k)): 2
// for a bf16 cache with one query row per sequence, else 1 (the rest of a
// unit then goes in at most two chunks of at most C tiles).  Every chunk
// costs a fixed set-up and merge, and the FP8 and multi-row units do more
// consumer work per tile, so for them fewer, longer chunks pay more than a
// finer tail (fia_execute: long FP8 decode 139.4 -> 134.8 us, FP8 with 16
// heads per KV head 120.3 -> 113.6 us, 4-row decode 88.2 -> 79.9 us against
// k = 6, 6 and 3; one-row bf16 decode 58.9 -> 58.6 us against k = 3).
int decode_small_div(const fia_params* p) {
  return (p->kv_dtype == FIA_KV_FP8_E4M3 || p->max_seqlen_q > 1) ? 1 : 2;
}

// Decode workspace: [0, 256) error word (offset 0) and the claim counters
// (offset 16); the schedule; the claim queue; the partial slots.  A unit of
// cost c gets at most c/C big chunks (so at most n*W over all units) and at
// most ceil((2C - 1)/c2) <= 2*small_div small ones (the rest it leaves is
// below 2C and c2 >= C/small_div), hence max_chunks = n*W + 2*small_div*U bounds the chunks of any lengths.
fia_status decode_plan(const fia_params* p, DecodePlan* pl) {
  int n;
  fia_status st = sm_count(p->num_sms, &n);
  if (st != FIA_OK) return st;
  const int G = p->num_q_heads / p->num_kv_heads;
  const int cols = p->max_seqlen_q * G;  // (query row, head) columns of a KV head
  const int GH = decode_group_heads(p->max_seqlen_q, cols);
  const int HG = (int)ceil_div(cols, GH);
  pl->n = n;
  pl->U = (int64_t)p->batch * p->num_kv_heads * HG;
  pl->max_chunks = (int64_t)n * kDecodeChunksPerCta + 2 * decode_small_div(p) * pl->U;
  // queue positions and slots are 32-bit in the kernels
  if (pl->max_chunks >= INT32_MAX) return FIA_ERR_BAD_SHAPE;
  int64_t off = kAlign;
  pl->off_sched = off;
  off = align_up(off + 8 * (kSchedHeader + 3 * ((int64_t)p->batch + 1) + p->batch));
  pl->off_queue = off;
  off = align_up(off + 16 * pl->max_chunks);
  pl->off_part = off;
  off = align_up(off + 4 * pl->max_chunks * GH * (p->head_dim + 2));
  pl->total = off;
  return FIA_OK;
}

DecodeArgs decode_args(const fia_params* p, const DecodePlan& pl, void* ws) {
  DecodeArgs a;
  memset(&a, 0, sizeof a);
  const int G = p->num_q_heads / p->num_kv_heads;
  a.B = p->batch;
  a.QN = p->num_q_heads;
  a.KVN = p->num_kv_heads;
  a.D = p->head_dim;
  a.G = G;
  a.GH = decode_group_heads(p->max_seqlen_q, p->max_seqlen_q * G);
  a.HG = (int)ceil_div(p->max_seqlen_q * G, a.GH);
  a.layout = p->layout;
  a.S_q = p->layout == FIA_LAYOUT_BSND ? p->max_seqlen_q : 1;
  a.S_max = p->max_seqlen_q;
  a.kv_layout = p->block_table ? p->kv_layout : 0;
  a.mask = p->atten_mask;
  a.mask_bstride = p->mask_batch_stride;
  a.mask_rstride = p->mask_row_stride;
  a.q = static_cast<const uint16_t*>(p->q);
  a.q_stride = p->q_token_stride ? p->q_token_stride : (int64_t)p->num_q_heads * p->head_dim;
  a.out = static_cast<uint16_t*>(p->out);
  a.out_stride = p->out_token_stride ? p->out_token_stride : (int64_t)p->num_q_heads * p->head_dim;
  a.lse = p->lse;
  a.cu_seqlens_q = p->cu_seqlens_q;
  a.seqused_kv = p->seqused_kv;
  a.S_kv = p->block_table ? (int)kv_capacity_of(p) : p->max_seqlen_kv;
  a.q_rows = p->layout == FIA_LAYOUT_TND ? (int64_t)p->total_q
                                         : (int64_t)p->batch * p->max_seqlen_q;
  a.num_blocks = p->block_table ? p->num_blocks : 0;
  a.block_table = p->block_table;
  a.max_blocks = p->max_blocks_per_seq;
  a.block_size = p->block_table ? p->block_size : 1;
  a.box_rows = p->block_table ? gcd_i(p->block_size, kKvTile) : kKvTile;
  fast_divisor(a.block_size, &a.bs_magic, &a.bs_shift);
  a.k_scale = p->k_scale;
  a.v_scale = p->v_scale;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.mask_mode = p->mask_mode;
  a.pre_tokens = p->pre_tokens;
  a.next_tokens = p->next_tokens;
  a.sinks = p->sinks;
  a.num_ctas = pl.n;
  a.num_units = pl.U;
  a.chunks_per_cta = kDecodeChunksPerCta;
  a.small_div = decode_small_div(p);
  a.max_chunks = pl.max_chunks;
  char* w = static_cast<char*>(ws);
  a.sched = reinterpret_cast<int64_t*>(w + pl.off_sched);
  a.queue = reinterpret_cast<int4*>(w + pl.off_queue);
  a.claim = reinterpret_cast<int*>(w + 16);
  a.prefill_mark = reinterpret_cast<int64_t*>(w + kWsPrefillMarkOff);
  a.partials = reinterpret_cast<float*>(w + pl.off_part);
  a.err = reinterpret_cast<int*>(w);
  a.debug = debug_checks();
  return a;
}

// Tensor maps of the K and V caches: token-major pools (and contiguous
// caches) as a matrix of KV_N * D columns with one row per token, head-major
// pools [num_blocks, KV_N, block_size, D] as one of D columns with one row per
// (block, head, token).
fia_status kv_maps(const fia_params* p, int box_rows, CUtensorMap* tk, CUtensorMap* tv) {
  const bool fp8 = p->kv_dtype == FIA_KV_FP8_E4M3;
  const bool head_major = p->block_table && p->kv_layout == FIA_KV_LAYOUT_BNNBSD;
  const uint64_t cols = head_major ? (uint64_t)p->head_dim
                                   : (uint64_t)p->num_kv_heads * p->head_dim;
  const uint64_t rows = p->block_table
                            ? (uint64_t)p->num_blocks * p->block_size * (head_major ? p->num_kv_heads : 1)
                            : (uint64_t)p->batch * p->max_seqlen_kv;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int es = fp8 ? 1 : 2;
  const uint32_t bc = fp8 ? 128 : 64;
  // One head's slice of a token is D * esize bytes: 256 for bf16 D=128 (two
  // 128-byte boxes, so a 256-byte L2 fill is used in full) but 128 for FP8,
  // where a 256-byte fill would also drag in the next head's slice.
  const CUtensorMapL2promotion promo = (uint64_t)p->head_dim * es >= 256
                                           ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                           : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
  fia_status st = make_map(tk, p->k_cache, dt, es, cols, rows ? rows : 1, bc, (uint32_t)box_rows,
                           cols, promo);
  if (st != FIA_OK) return st;
  return make_map(tv, p->v_cache, dt, es, cols, rows ? rows : 1, bc, (uint32_t)box_rows, cols,
                  promo);
}

struct PrefillPlan {
  int n, per_pair, npairs, max_cost;
  int64_t U_max;
  int64_t off_seq, off_hist, off_list, total;
  // FP8 caches: their fp16 copies [B, cap, KVN, D], the largest scales and
  // the K/V factors [B * KVN * 2] (all 0 for bf16 caches; the queries are
  // converted to fp16 inside the prefill kernel)
  int64_t off_kbf, off_vbf, off_smax, off_kvfac;
};

fia_status prefill_plan(const fia_params* p, PrefillPlan* pl) {
  fia_status st = sm_count(p->num_sms, &pl->n);
  if (st != FIA_OK) return st;
  const int G = p->num_q_heads / p->num_kv_heads;
  pl->per_pair = (G % 2 == 0) ? 2 : 1;
  pl->npairs = G / pl->per_pair;
  const int64_t H = (int64_t)p->num_kv_heads * pl->npairs;
  const int64_t qtiles = p->layout == FIA_LAYOUT_TND
                             ? ceil_div(p->total_q, kQTile) + p->batch
                             : (int64_t)p->batch * ceil_div(p->max_seqlen_q, kQTile);
  pl->U_max = qtiles * H;
  pl->max_cost = (int)(1 + ceil_div(kv_capacity_of(p), kKvTile));
  int64_t off = kAlign;  // [0,4) error word, [8,16) units, [16,24) claim counters,
                         // [24,48) the plan's mark, B and CTA count
  pl->off_seq = off;
  off = align_up(off + 8 * ((int64_t)p->batch + 1));
  pl->off_hist = off;
  off = align_up(off + 4 * ((int64_t)pl->max_cost + 2));
  pl->off_list = off;
  off = align_up(off + 8 * pl->U_max);
  pl->off_kbf = pl->off_vbf = pl->off_smax = pl->off_kvfac = 0;
  if (p->kv_dtype == FIA_KV_FP8_E4M3) {
    const int64_t bytes = 2 * (int64_t)p->batch * kv_capacity_of(p) * p->num_kv_heads * p->head_dim;
    pl->off_kbf = off;
    off = align_up(off + bytes);
    pl->off_vbf = off;
    off = align_up(off + bytes);
    pl->off_smax = off;
    off = align_up(off + 8 * (int64_t)p->batch * p->num_kv_heads);
    pl->off_kvfac = off;
    off = align_up(off + 8 * (int64_t)p->batch * p->num_kv_heads);
  }
  pl->total = off;
  return FIA_OK;
}

// The parameters the tcgen05 prefill kernel runs on: for FP8 caches, their
// fp16 copies in the workspace as contiguous caches [B, cap, KVN, D] (16-bit
// elements move through the same tensor maps; the bf16 queries are converted
// to fp16 by the kernel itself).
fia_params prefill_view(const fia_params* p, const PrefillPlan& pl, void* ws) {
  fia_params v = *p;
  if (p->kv_dtype != FIA_KV_FP8_E4M3) return v;
  char* w = static_cast<char*>(ws);
  v.k_cache = w + pl.off_kbf;
  v.v_cache = w + pl.off_vbf;
  v.max_seqlen_kv = (int32_t)kv_capacity_of(p);
  v.kv_dtype = FIA_KV_BF16;
  v.k_scale = v.v_scale = nullptr;
  v.quant_tile = 0;
  v.block_table = nullptr;
  v.max_blocks_per_seq = v.block_size = v.num_blocks = 0;
  v.kv_layout = FIA_KV_LAYOUT_BNBSH;
  return v;
}

DequantArgs dequant_args(const fia_params* p, const PrefillPlan& pl, void* ws) {
  DequantArgs d;
  memset(&d, 0, sizeof d);
  d.B = p->batch;
  d.KVN = p->num_kv_heads;
  d.D = p->head_dim;
  d.cap = (int)kv_capacity_of(p);
  d.kv_layout = p->block_table ? p->kv_layout : 0;
  d.k = static_cast<const uint8_t*>(p->k_cache);
  d.v = static_cast<const uint8_t*>(p->v_cache);
  d.k_scale = p->k_scale;
  d.v_scale = p->v_scale;
  d.block_table = p->block_table;
  d.max_blocks = p->max_blocks_per_seq;
  d.block_size = p->block_table ? p->block_size : 1;
  d.num_blocks = p->num_blocks;
  d.seqused_kv = p->seqused_kv;
  char* w = static_cast<char*>(ws);
  d.k_out = reinterpret_cast<uint16_t*>(w + pl.off_kbf);
  d.v_out = reinterpret_cast<uint16_t*>(w + pl.off_vbf);
  d.smax = reinterpret_cast<uint32_t*>(w + pl.off_smax);
  d.kvfac = reinterpret_cast<float*>(w + pl.off_kvfac);
  d.err = reinterpret_cast<int*>(w);
  d.debug = debug_checks();
  return d;
}

PrefillArgs prefill_args(const fia_params* p, const PrefillPlan& pl, void* ws) {
  PrefillArgs a;
  memset(&a, 0, sizeof a);
  a.B = p->batch;
  a.QN = p->num_q_heads;
  a.KVN = p->num_kv_heads;
  a.D = p->head_dim;
  a.G = p->num_q_heads / p->num_kv_heads;
  a.npairs = pl.npairs;
  a.per_pair = pl.per_pair;
  a.layout = p->layout;
  a.S_q = p->max_seqlen_q;
  a.kv_layout = p->block_table ? p->kv_layout : 0;
  a.mask = p->atten_mask;
  a.mask_bstride = p->mask_batch_stride;
  a.mask_rstride = p->mask_row_stride;
  a.out = static_cast<uint16_t*>(p->out);
  a.out_stride = p->out_token_stride ? p->out_token_stride : (int64_t)p->num_q_heads * p->head_dim;
  a.lse = p->lse;
  a.cu_seqlens_q = p->cu_seqlens_q;
  a.seqused_kv = p->seqused_kv;
  a.S_kv = p->block_table ? (int)kv_capacity_of(p) : p->max_seqlen_kv;
  a.block_table = p->block_table;
  a.max_blocks = p->max_blocks_per_seq;
  a.block_size = p->block_table ? p->block_size : 1;
  a.box_rows = p->block_table ? gcd_i(p->block_size, kKvTile) : kKvTile;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.mask_mode = p->mask_mode;
  a.pre_tokens = p->pre_tokens;
  a.next_tokens = p->next_tokens;
  a.sinks = p->sinks;
  a.num_ctas = pl.n;
  a.max_cost = pl.max_cost;
  a.num_blocks = p->block_table ? p->num_blocks : 0;
  a.debug = debug_checks();
  char* w = static_cast<char*>(ws);
  a.err = reinterpret_cast<int*>(w);
  a.claim = reinterpret_cast<int*>(w + 16);
  a.num_units = reinterpret_cast<int64_t*>(w + 8);
  a.seq_prefix = reinterpret_cast<int64_t*>(w + pl.off_seq);
  a.hist = reinterpret_cast<int*>(w + pl.off_hist);
  a.unit_list = reinterpret_cast<int2*>(w + pl.off_list);
  a.max_units = pl.U_max;
  return a;
}

fia_status q_map(const fia_params* p, CUtensorMap* tq) {
  const uint64_t cols = (uint64_t)p->num_q_heads * p->head_dim;
  const uint64_t rows = p->layout == FIA_LAYOUT_TND ? (uint64_t)p->total_q
                                                    : (uint64_t)p->batch * p->max_seqlen_q;
  const uint64_t stride = p->q_token_stride ? (uint64_t)p->q_token_stride : cols;
  return make_map(tq, p->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, 64, 128, stride);
}

// ---------------------------------------------------------------------------
// shared-KV sparse attention ("kv_quant_sparse_attn_sharedkv" constraints)
// ---------------------------------------------------------------------------
constexpr int kSparseHeads = 8;       // query heads per work item
constexpr int kSparseMaxCtas = 1007;  // 1024 - 16 - 1 begins fit the metadata

struct SparsePlan {
  int n, mode;
  int64_t rows, total;
};

fia_status sparse_validate(const sparse_attn_params* p) {
  if (!p) return FIA_ERR_NULL_ARG;
  for (int i = 0; i < 8; ++i)
    if (p->reserved[i] != 0) return FIA_ERR_BAD_SHAPE;
  if (p->kv_dtype != FIA_SPARSE_KV_BF16 && p->kv_dtype != FIA_SPARSE_KV_FP8_PACKED)
    return FIA_ERR_BAD_DTYPE;
  if (p->kv_dtype == FIA_SPARSE_KV_FP8_PACKED &&
      (p->head_dim != 512 || p->tile_size != 64 || p->rope_head_dim != 64))
    return FIA_ERR_BAD_SHAPE;
  if (p->batch < 1 || p->batch > 65536) return FIA_ERR_BAD_SHAPE;
  if (p->num_q_heads < 1 || p->num_q_heads > 128 || (p->num_q_heads & (p->num_q_heads - 1)))
    return FIA_ERR_BAD_SHAPE;
  if (p->head_dim < 1 || p->head_dim > 512) return FIA_ERR_BAD_SHAPE;
  if (p->layout != FIA_LAYOUT_BSND && p->layout != FIA_LAYOUT_TND) return FIA_ERR_BAD_SHAPE;
  if (p->max_seqlen_q < 0 || p->total_q < 0) return FIA_ERR_BAD_SHAPE;
  if (p->layout == FIA_LAYOUT_TND && !p->cu_seqlens_q) return FIA_ERR_NULL_ARG;
  if (!p->q || !p->out || !p->ori_kv || !p->ori_block_table || !p->seqused_kv)
    return FIA_ERR_NULL_ARG;
  if (!aligned16(p->q) || !aligned16(p->out) || !aligned16(p->ori_kv)) return FIA_ERR_BAD_SHAPE;
  if (p->ori_block_size <= 0 || p->ori_block_size % 16 || p->ori_block_size > 1024)
    return FIA_ERR_BAD_SHAPE;
  if (p->ori_max_blocks <= 0 || p->ori_num_blocks <= 0) return FIA_ERR_BAD_SHAPE;
  if ((int64_t)p->ori_max_blocks * p->ori_block_size > INT32_MAX) return FIA_ERR_BAD_SHAPE;
  if (p->ori_win_left < 0 || p->ori_win_right < 0 ||
      (int64_t)p->ori_win_left + p->ori_win_right + 1 > 65536)
    return FIA_ERR_BAD_SHAPE;
  if (!std::isfinite(p->softmax_scale)) return FIA_ERR_BAD_SHAPE;
  if (p->num_sms < 0 || p->num_sms > 4096) return FIA_ERR_BAD_SHAPE;
  if (p->cmp_kv) {
    if (!p->cmp_block_table) return FIA_ERR_NULL_ARG;
    if (!aligned16(p->cmp_kv)) return FIA_ERR_BAD_SHAPE;
    if (p->cmp_block_size <= 0 || p->cmp_block_size % 16 || p->cmp_block_size > 1024)
      return FIA_ERR_BAD_SHAPE;
    if (p->cmp_max_blocks <= 0 || p->cmp_num_blocks <= 0) return FIA_ERR_BAD_SHAPE;
    if ((int64_t)p->cmp_max_blocks * p->cmp_block_size > INT32_MAX) return FIA_ERR_BAD_SHAPE;
    if (p->cmp_ratio < 1) return FIA_ERR_BAD_SHAPE;
    if (p->cmp_sparse_indices && (p->topk < 1 || p->topk > 2048)) return FIA_ERR_BAD_SHAPE;
  } else if (p->cmp_sparse_indices) {
    return FIA_ERR_BAD_SHAPE;  // indices without a compressed cache
  }
  if (p->head_dim != 128 && p->head_dim != 256 && p->head_dim != 512) return FIA_ERR_UNSUPPORTED;
  return FIA_OK;
}

fia_status sparse_plan(const sparse_attn_params* p, SparsePlan* pl) {
  fia_status st = sparse_validate(p);
  if (st != FIA_OK) return st;
  int n;
  st = sm_count(p->num_sms, &n);
  if (st != FIA_OK) return st;
  pl->n = n < kSparseMaxCtas ? n : kSparseMaxCtas;
  pl->mode = !p->cmp_kv ? 0 : (p->cmp_sparse_indices ? 1 : 2);
  pl->rows = p->layout == FIA_LAYOUT_TND ? (int64_t)p->total_q
                                         : (int64_t)p->batch * p->max_seqlen_q;
  // the metadata holds the item count and the total item weight as int32
  // (a row's weight is its chunk count: the window's, then the compressed
  // rows' -- for CSA at most topk, for HCA at most the compressed capacity)
  const int64_t W = (int64_t)p->ori_win_left + p->ori_win_right + 1;
  int64_t kc = 0;
  if (pl->mode == 1) kc = p->topk;
  else if (pl->mode == 2) kc = (int64_t)p->cmp_max_blocks * p->cmp_block_size;
  const int64_t items = pl->rows * ((p->num_q_heads + kSparseHeads - 1) / kSparseHeads);
  if (items * (ceil_div(W, 64) + ceil_div(kc, 64)) > INT32_MAX) return FIA_ERR_BAD_SHAPE;
  // workspace: the status word only (a row's chunks all run in one CTA)
  pl->total = kAlign;
  return FIA_OK;
}

SparseArgs sparse_args(const sparse_attn_params* p, const SparsePlan& pl, void* ws) {
  SparseArgs a;
  memset(&a, 0, sizeof a);
  a.B = p->batch;
  a.N1 = p->num_q_heads;
  a.D = p->head_dim;
  a.layout = p->layout;
  a.S1 = p->max_seqlen_q;
  a.q = static_cast<const uint16_t*>(p->q);
  a.out = static_cast<uint16_t*>(p->out);
  a.lse = p->lse;
  a.ori_kv = p->ori_kv;
  a.ori_block_table = p->ori_block_table;
  a.ori_max_blocks = p->ori_max_blocks;
  a.ori_block_size = p->ori_block_size;
  a.ori_num_blocks = p->ori_num_blocks;
  a.cmp_num_blocks = p->cmp_kv ? p->cmp_num_blocks : 0;
  a.cmp_kv = p->cmp_kv;
  a.cmp_block_table = p->cmp_block_table;
  a.cmp_max_blocks = p->cmp_max_blocks;
  a.cmp_block_size = p->cmp_kv ? p->cmp_block_size : 1;
  a.cmp_sparse_indices = p->cmp_sparse_indices;
  a.K2 = pl.mode == 1 ? p->topk : 0;
  a.cu_seqlens_q = p->cu_seqlens_q;
  a.seqused_kv = p->seqused_kv;
  a.sinks = p->sinks;
  a.scale_log2 = p->softmax_scale * 1.4426950408889634f;
  a.cmp_ratio = p->cmp_kv ? p->cmp_ratio : 1;
  a.win_left = p->ori_win_left;
  a.win_right = p->ori_win_right;
  a.mode = pl.mode;
  a.kv_dtype = p->kv_dtype;
  a.rows = pl.rows;
  a.hgs = (p->num_q_heads + kSparseHeads - 1) / kSparseHeads;
  fast_divisor(p->ori_block_size, &a.ori_magic, &a.ori_shift);
  fast_divisor(a.cmp_block_size, &a.cmp_magic, &a.cmp_shift);
  a.num_ctas = pl.n;
  if (ws) a.err = reinterpret_cast<int*>(ws);
  a.debug = debug_checks();
  return a;
}

bool q_empty(const fia_params* p) {
  return p->layout == FIA_LAYOUT_TND ? p->total_q == 0 : p->max_seqlen_q == 0;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

const char* fia_status_string(fia_status s) {
  switch (s) {
    case FIA_OK: return "FIA_OK";
    case FIA_ERR_NULL_ARG: return "FIA_ERR_NULL_ARG";
    case FIA_ERR_BAD_SHAPE: return "FIA_ERR_BAD_SHAPE";
    case FIA_ERR_BAD_DTYPE: return "FIA_ERR_BAD_DTYPE";
    case FIA_ERR_UNSUPPORTED: return "FIA_ERR_UNSUPPORTED";
    case FIA_ERR_WORKSPACE_TOO_SMALL: return "FIA_ERR_WORKSPACE_TOO_SMALL";
    case FIA_ERR_CUDA: return "FIA_ERR_CUDA";
    default: return "FIA_ERR_UNKNOWN";
  }
}

int32_t fia_abi_version(void) { return FIA_ABI_VERSION; }

size_t fia_sizeof_params(void) { return sizeof(fia_params); }
size_t fia_sizeof_sparse_params(void) { return sizeof(sparse_attn_params); }

fia_status fia_get_plan_layout(const fia_params* p, fia_plan_layout* out) {
  if (!out) return FIA_ERR_NULL_ARG;
  fia_status st = validate(p);
  if (st != FIA_OK) return st;
  memset(out, 0, sizeof *out);
  if (q_empty(p)) {
    out->total_bytes = kAlign;
    return FIA_OK;
  }
  if (is_decode(p)) {
    DecodePlan pl;
    st = decode_plan(p, &pl);
    if (st != FIA_OK) return st;
    out->branch = 1;
    out->num_ctas = pl.n;
    out->num_units = pl.U;
    out->max_chunks = pl.max_chunks;
    out->sched_off = pl.off_sched;
    out->queue_off = pl.off_queue;
    out->total_bytes = pl.total;
    return FIA_OK;
  }
  PrefillPlan pp;
  st = prefill_plan(p, &pp);
  if (st != FIA_OK) return st;
  out->branch = 2;
  out->num_ctas = pp.n;
  out->num_units = pp.U_max;
  out->unit_list_off = pp.off_list;
  out->total_bytes = pp.total;
  return FIA_OK;
}

fia_status fia_get_workspace_size(const fia_params* p, size_t* bytes) {
  if (!bytes) return FIA_ERR_NULL_ARG;
  fia_plan_layout l;
  fia_status st = fia_get_plan_layout(p, &l);
  if (st != FIA_OK) return st;
  *bytes = (size_t)l.total_bytes;
  return FIA_OK;
}

fia_status fia_plan(const fia_params* p, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange range("fia_plan");
  fia_plan_layout l;
  fia_status st = fia_get_plan_layout(p, &l);
  if (st != FIA_OK) return st;
  if (!ws || ws_bytes < (size_t)l.total_bytes) return FIA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (q_empty(p)) return FIA_OK;
  if (l.branch == 2) {
    PrefillPlan pp;
    st = prefill_plan(p, &pp);
    if (st != FIA_OK) return st;
    const fia_params v = prefill_view(p, pp, ws);
    PrefillArgs a = prefill_args(&v, pp, ws);
    return launch_prefill_schedule(a, s) == cudaSuccess ? FIA_OK : FIA_ERR_CUDA;
  }
  DecodePlan pl;
  st = decode_plan(p, &pl);
  if (st != FIA_OK) return st;
  DecodeArgs a = decode_args(p, pl, ws);
  return launch_decode_schedule(a, s) == cudaSuccess ? FIA_OK : FIA_ERR_CUDA;
}

fia_status fia_execute(const fia_params* p, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange range("fia_execute");
  fia_plan_layout l;
  fia_status st = fia_get_plan_layout(p, &l);
  if (st != FIA_OK) return st;
  if (!ws || ws_bytes < (size_t)l.total_bytes) return FIA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (q_empty(p)) return FIA_OK;
  if (l.branch == 2) {
    PrefillPlan pp;
    st = prefill_plan(p, &pp);
    if (st != FIA_OK) return st;
    const fia_params v = prefill_view(p, pp, ws);
    PrefillArgs a = prefill_args(&v, pp, ws);
    if (p->kv_dtype == FIA_KV_FP8_E4M3) {
      char* w = static_cast<char*>(ws);
      a.f16 = 1;
      a.kvfac = reinterpret_cast<const float*>(w + pp.off_kvfac);
    }
    // (FP8 caches: the prefill kernel converts each bf16 query tile to fp16
    // itself; the conversion pass covers K and V)
    CUtensorMap tq, tk, tv;
    st = q_map(&v, &tq);
    if (st != FIA_OK) return st;
    st = kv_maps(&v, a.box_rows, &tk, &tv);
    if (st != FIA_OK) return st;
    if (p->kv_dtype == FIA_KV_FP8_E4M3) {
      int n;
      st = sm_count(p->num_sms, &n);
      if (st != FIA_OK) return st;
      if (launch_kv_dequant(dequant_args(p, pp, ws), n, s) != cudaSuccess) return FIA_ERR_CUDA;
    }
    return launch_prefill(a, tq, tk, tv, s) == cudaSuccess ? FIA_OK : FIA_ERR_CUDA;
  }
  DecodePlan pl;
  st = decode_plan(p, &pl);
  if (st != FIA_OK) return st;
  DecodeArgs a = decode_args(p, pl, ws);
  CUtensorMap tk, tv;
  st = kv_maps(p, a.box_rows, &tk, &tv);
  if (st != FIA_OK) return st;
  return launch_decode(a, tk, tv, p->kv_dtype == FIA_KV_FP8_E4M3, s) == cudaSuccess ? FIA_OK
                                                                                     : FIA_ERR_CUDA;
}

fia_status fia_run(const fia_params* p, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange range("fia_run");
  fia_status st = fia_plan(p, ws, ws_bytes, stream);
  if (st != FIA_OK) return st;
  return fia_execute(p, ws, ws_bytes, stream);
}

fia_status sparse_attn_metadata(const sparse_attn_params* p, int32_t* metadata,
                                size_t* workspace_bytes, void* stream) {
  NvtxRange range("sparse_attn_metadata");
  if (!p || !metadata || !workspace_bytes) return FIA_ERR_NULL_ARG;
  if (!aligned16(metadata)) return FIA_ERR_BAD_SHAPE;  // the documented alignment
  SparsePlan pl;
  fia_status st = sparse_plan(p, &pl);
  if (st != FIA_OK) return st;
  *workspace_bytes = (size_t)pl.total;
  SparseArgs a = sparse_args(p, pl, nullptr);
  if (a.rows == 0) return FIA_OK;
  return launch_sparse_metadata(a, metadata, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FIA_OK
             : FIA_ERR_CUDA;
}

fia_status sparse_attn_run(const sparse_attn_params* p, const int32_t* metadata, void* ws,
                           size_t ws_bytes, void* stream) {
  NvtxRange range("sparse_attn_run");
  if (!p || !metadata) return FIA_ERR_NULL_ARG;
  if (!aligned16(metadata)) return FIA_ERR_BAD_SHAPE;
  SparsePlan pl;
  fia_status st = sparse_plan(p, &pl);
  if (st != FIA_OK) return st;
  if (!ws || ws_bytes < (size_t)pl.total) return FIA_ERR_WORKSPACE_TOO_SMALL;
  SparseArgs a = sparse_args(p, pl, ws);
  if (a.rows == 0) return FIA_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // (the kernel clears the status word itself once the metadata checks out,
  // except with FIA_DEBUG, where the host does it first)
  if (a.debug && cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return FIA_ERR_CUDA;
  return launch_sparse(a, metadata, s) == cudaSuccess ? FIA_OK : FIA_ERR_CUDA;
}

}  // extern "C"
