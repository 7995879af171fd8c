// internal.h -- argument blocks shared between the host side of libfia
// (fia_api.cu) and its kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

namespace fia {

// An NVTX range over one C-ABI call (plan, execute, run, the sparse calls,
// the combine, the workspace-free decode): a profiler or tracer sees each
// call with the kernels it launched.  nvtx3 is header-only and finds its
// tool at run time; with none attached a range costs a few nanoseconds.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kKvTile = 128;   // KV positions per tile (one split granule)
constexpr int kQTile = 128;    // query rows per prefill tile
constexpr int kMaxHeadGroup = 16;  // query columns packed per decode unit, at most
constexpr int kDecodeMaxRows = 16; // query rows per sequence the decode kernel takes

// Columns per decode unit: the (query row, query head) pairs of a KV head,
// S rows x G heads of them, in mma N columns of 8.  A unit takes 16 columns
// only for one query row with more than 8 heads per KV head; several query
// rows go in 8-column units, two per KV head for 16 columns, whose chunks sit
// next to each other in the queue and share their K/V tiles through L2 (a
// 4-row GQA-4 decode: 92.2 against 100.4 us per execute while 16-column
// units spilled registers; the same, 88.0 against 88.2 us, once the
// consumers had 208 registers).
inline int decode_group_heads(int rows, int cols) { return (rows == 1 && cols > 8) ? 16 : 8; }

// Everything the decode schedule and the decode kernel read.
struct DecodeArgs {
  int B, QN, KVN, D, G, GH, HG;  // GH columns per unit, HG units per KV head
  int layout;            // 0 BSND, 1 TND
  int S_q;               // BSND query length
  int S_max;             // query rows per sequence the units cover (1..16)
  int kv_layout;         // 0 [nb, bs, KVN, D], 1 [nb, KVN, bs, D]
  const uint8_t* mask;   // explicit mask (modes 0/1) or null
  int64_t mask_bstride, mask_rstride;
  const uint16_t* q;     // bf16
  int64_t q_stride;      // elements between tokens
  uint16_t* out;
  int64_t out_stride;
  float* lse;
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_kv;  // may be null (contiguous: S_kv for every batch)
  int S_kv;
  int64_t q_rows;              // query rows of q/out (B * S_q, or T for TND)
  int64_t num_blocks;          // pages in the pool (paged caches)
  const int32_t* block_table;  // null: contiguous
  int max_blocks, block_size, box_rows;
  uint32_t bs_magic;           // j / block_size == (j * bs_magic) >> bs_shift, 0 <= j < 2^31
  int bs_shift;
  const float* k_scale;
  const float* v_scale;
  float scale_log2;      // scale * log2(e)
  int mask_mode, pre_tokens, next_tokens;
  const float* sinks;
  // plan (workspace)
  int num_ctas;
  int chunks_per_cta;          // W: the chunk size aims at W chunks per CTA
  int small_div;               // small chunks of ceil(C / small_div) tiles (2; 1 for FP8 or rows > 1)
  int64_t num_units;           // B * KVN * HG
  int64_t max_chunks;          // partial slots: a bound on the number of chunks
  int64_t* sched;              // [8 + 3(B+1) + B]: C, c2, chunks, big chunks, split
                               // batches, mark, B, CTAs; the partial-slot prefix Q, the
                               // queue prefixes R1, R2; the split batches (then -1)
  int4* queue;                 // [max_chunks] (b | q_len << 16, chunk << 16 | unit of b,
                               // kv_len, first token row)
  int* claim;                  // [2]: next queue entry, CTAs done with the queue
  int64_t* prefill_mark;       // header word of a prefill plan: a decode plan clears it
  float* partials;             // [max_chunks][GH][D + 2]: acc, then m and l
  int* err;
  int debug;                   // FIA_DEBUG: report page ids outside the pool (error word 3)
};

// Target number of big chunks per persistent CTA in the decode schedule.
constexpr int kDecodeChunksPerCta = 5;
constexpr int kSchedHeader = 8;  // int64 header words of the decode schedule
// header word 5 of a decode plan written by the scheduler (words 6, 7: B and
// the CTA count): fia_execute runs nothing on a workspace without it
constexpr int64_t kDecodePlanMark = 0x4649414445434F44LL;
// the same for a prefill plan, at workspace bytes [24, 48): mark, B, CTA count
constexpr int64_t kPrefillPlanMark = 0x4649415052454649LL;
// The first 256 bytes of a workspace are a header that both branches share:
// [0, 4) error word, [8, 16) prefill unit count, [16, 24) claim counters,
// [24, 48) prefill plan mark, B and CTA count.  A decode plan clears the
// prefill mark, and a decode execute runs nothing while that mark is set, so
// one workspace can serve both branches: an execute after the other branch's
// plan reports 2 in the error word instead of reading a plan that is gone.
constexpr int kWsPrefillMarkOff = 24;

struct PrefillArgs {
  int B, QN, KVN, D, G, npairs, per_pair;  // per_pair query heads per unit (2, or 1 if G odd)
  int layout;
  int S_q;
  int kv_layout;             // 0 [nb, bs, KVN, D], 1 [nb, KVN, bs, D]
  const uint8_t* mask;       // explicit mask (modes 0/1) or null
  int64_t mask_bstride, mask_rstride;
  // fp16 operands (FP8 caches, f16 = 1): the kernel converts each bf16 query
  // row to fp16 times 2^sh (sh per row), so the scores of row (token t, head
  // h) are S' * 2^-sh * kvfac[(b*KVN + hk)*2], the output O' * kvfac[.. + 1]
  int f16;
  const float* kvfac;
  int64_t out_stride;
  uint16_t* out;
  float* lse;
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_kv;
  int S_kv;
  const int32_t* block_table;
  int max_blocks, block_size, box_rows;
  float scale_log2;
  int mask_mode, pre_tokens, next_tokens;
  const float* sinks;
  // plan (workspace)
  int num_ctas;
  int max_cost;           // costs above are clamped (ordering only)
  int64_t* num_units;     // written by the scheduler
  int64_t* seq_prefix;    // [B+1] units before each sequence
  int* hist;              // [max_cost + 2] cost histogram, then offsets
  int2* unit_list;        // [units] (b, q_tile | hk << 18 | pair << 26), cost-descending
  int* claim;             // [2]: next unit to claim, CTAs done claiming
  int* err;
  int64_t max_units;      // bound on the plan's unit count (the unit list's length)
  int64_t num_blocks;     // pages in the pool (paged caches)
  int debug;              // FIA_DEBUG: report page ids outside the pool (error word 3)
};

struct SparseArgs {
  int B, N1, D, layout, S1;
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  const void* ori_kv;    // bf16 rows of D, or packed FP8 rows of 640 bytes
  const int32_t* ori_block_table;
  int ori_max_blocks, ori_block_size;
  int64_t ori_num_blocks;
  const void* cmp_kv;
  const int32_t* cmp_block_table;
  int cmp_max_blocks, cmp_block_size;
  int64_t cmp_num_blocks;
  const int32_t* cmp_sparse_indices;
  int K2;
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_kv;
  const float* sinks;
  float scale_log2;
  int cmp_ratio, win_left, win_right;
  int mode;              // 0 SWA, 1 CSA, 2 HCA
  int kv_dtype;          // 0 bf16 rows, 1 packed FP8 rows (640 bytes, D = 512)
  int64_t rows;
  int64_t hgs;           // groups of 8 query heads per row (work items per row)
  uint32_t ori_magic, cmp_magic;  // j / block_size == (j * magic) >> shift, 0 <= j < 2^31
  int ori_shift, cmp_shift;
  int* err;
  int num_ctas;
  int debug;             // FIA_DEBUG: report page ids outside the pool (error word 3)
};

// host launchers (return cudaSuccess or the launch error)
cudaError_t launch_decode_schedule(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                          int fp8, cudaStream_t s);
size_t decode_smem_bytes(int D, int fp8);

cudaError_t launch_prefill_schedule(const PrefillArgs& a, cudaStream_t s);

// FP8 K/V for the prefill kernel: every visible row of the paged (or
// contiguous) E4M3 caches dequantised once into contiguous fp16 caches
// [B, cap, KVN, D] in the workspace, each (batch, KV head) scaled by a power
// of two that keeps it inside fp16 (the prefill kernel converts the queries
// itself, with a power-of-two shift per (token, head)).
struct DequantArgs {
  int B, KVN, D, cap, kv_layout;
  const uint8_t* k;
  const uint8_t* v;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;  // null: contiguous [B, cap, KVN, D]
  int max_blocks, block_size;
  int64_t num_blocks;
  const int32_t* seqused_kv;   // null: cap for every batch
  uint16_t* k_out;
  uint16_t* v_out;
  uint32_t* smax;              // [B * KVN * 2] largest K and V scale (bits), zeroed first
  float* kvfac;                // [B * KVN * 2] the power of two taken out of K and V
  int* err;                    // the workspace's error word
  int debug;                   // FIA_DEBUG: report page ids outside the pool (error word 3)
};
cudaError_t launch_kv_dequant(const DequantArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t s);

cudaError_t launch_sparse_metadata(const SparseArgs& a, int32_t* md, cudaStream_t s);
cudaError_t launch_sparse(const SparseArgs& a, const int32_t* md, cudaStream_t s);

}  // namespace fia
