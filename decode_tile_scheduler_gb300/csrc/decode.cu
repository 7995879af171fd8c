// decode.cu -- the incremental-inference branch of fused inference attention
// (a few query rows per sequence; "aclnnFusedInferAttentionScoreV2": the
// IncreFlashAttention branch runs when the query S is 1; the quantised
// Decode-MLA rules of "...V5" allow Q_S up to 16 for multi-token decode) over a
// paged KV cache, plus its tile scheduler.
//
// Columns and units: the query side of KV head hk of a sequence is its
// (query row i, query head h of the GQA group) pairs, column c = i*G + h%G,
// S_max*G of them.  A work unit (batch b, KV head hk, column group hg) holds up
// to GH consecutive columns (16 for one query row with G > 8, else 8): they
// form the N columns of every mma.sync, so each KV page is read once for all
// of them (the GQA heads and, for multi-token decode, the query rows too; the
// units of one KV head sit next to each other in the queue and share its
// pages through L2).  Only the groups holding columns of the sequence's own
// rows are scheduled ("active").  A unit owns the KV tiles (128 positions) its rows see together; every column
// is masked with its own row's bounds.
//
// Scheduler (decode_schedule_kernel): cost(u) = visible tiles (>= 1; 0 when
// the batch has no query row).  With T the total cost of the active units and
// n persistent CTAs, the chunk size is C = ceil(T / (n * W)) tiles (W chunks
// per CTA, at least one tile), and a unit of cost c is cut into
// n1 = max(0, floor(c/C) - 1) big chunks of C tiles followed by the remaining
// r = c - n1*C tiles (C <= r < 2C unless c < C) in small chunks of
// c2 = ceil(C/k) tiles, k = 2 for a bf16 cache and one query row, else 1
// (every chunk has a fixed cost, and the FP8 and multi-row units' tiles
// cost the consumers more).  The claim queue lists every big chunk
// (batch-major, then chunk, then active unit of the batch) before every small
// chunk (same order), so the work left at the end is always small pieces.  CTAs claim
// chunks from the queue with one atomic each: an SM that streams faster
// simply takes more chunks.  A unit cut into several chunks is split-KV: each
// chunk writes its (m, l, acc) partial to the slot of its (unit, chunk
// index), and a combine kernel chained behind the decode kernel folds them in
// chunk order (deterministic, whichever CTAs ran them).
//
// Decode kernel: producer warps (two, four with an FP8 cache) stream K and V
// pages with TMA (page rows from block_table) into a ring of shared-memory
// stages, with the rows of an explicit mask when there is one; eight consumer
// warps (two warpgroups, with the registers the producers' warpgroup gives
// up) each take 16 rows of every tile.  The products are computed transposed ("swap AB"):
// S^T = K Q^T with the KV rows as the mma M dimension and the query columns
// as N, then O^T += V^T P^T, where P^T comes out of the S^T accumulators with
// movmatrix.  Softmax is online, in the exp2 domain, per column.  FP8 E4M3
// pages are widened to fp16 in registers (exact); K tile scales multiply the
// per-64-column partial scores and V tile scales are folded into P^T, so the
// dequantised cache is never materialised.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace fia {

namespace {

constexpr int kConsumers = 8;                        // consumer warps
// three warpgroups: the producer's (warp 0 works, warps 1-3 leave at once)
// gives its registers to the two consumer warpgroups (setmaxnreg):
// 128 * kProdRegs + 256 * kConsRegs = 384 * 168, the launch's register file
constexpr int kThreads = 32 * (4 + kConsumers);
constexpr int kProdRegs = 88;
constexpr int kConsRegs = 208;
static_assert(128 * kProdRegs + 256 * kConsRegs <= kThreads * 168, "register split");
constexpr int kRowsPerWarp = kKvTile / kConsumers;  // 16
constexpr int kMaxGH = 16;                           // heads per unit, max

// Row permutation inside each group of 8 KV rows: n -> pi(n) keeps
// pi(2q) = 2q and maps pi(2q+1) = 2q+5 mod 8.  Rows g and g+1 of a fragment
// then differ in bit 2, which keeps the FP8 16-byte shared loads free of bank
// conflicts under the 128-byte swizzle; ldmatrix takes any row order.
__device__ __forceinline__ int pi8(int n) { return (n & 1) ? ((n + 4) & 7) : n; }
// KV row (0..15, within a warp's 16 rows) of fragment row m
__device__ __forceinline__ int rho16(int m) { return (m & 8) + pi8(m & 7); }

template <int D, bool FP8>
struct DecodeCfg {
  static constexpr int kNsub = FP8 ? 1 : D / 64;            // 128-byte slices per row
  static constexpr int kTileBytes = kNsub * kKvTile * 128;  // one of K or V
  static constexpr int kScaleBytes = FP8 ? kKvTile * (D / 64) * 4 : 0;
  // explicit mask: one 128-byte row slice per query row of the unit
  static constexpr int kMaskBytes = kDecodeMaxRows * kKvTile;
  static constexpr int kOffMask = 2 * kTileBytes + 2 * kScaleBytes;  // inside a stage
  static constexpr int kStageBytes = 2 * kTileBytes + 2 * kScaleBytes + kMaskBytes;
  static constexpr int kStages = FP8 ? 5 : (D == 128 ? 3 : 6);
  static constexpr int kQBytes = kMaxGH * D * 2;
  static constexpr int kRedBytes = 4 * kConsumers * 32 * 16;  // merge rounds: [4][8 warps][32] float4
  static constexpr int kRedMlBytes = kConsumers * kMaxGH * 2 * 4;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffRed = kOffQ + 2 * kQBytes;
  static constexpr int kOffRedMl = kOffRed + kRedBytes;
  static constexpr int kOffBar = kOffRedMl + kRedMlBytes;
  static constexpr int kOffMsg = kOffBar + 8 * (2 * kStages + 6);
  static constexpr int kOffMisc = kOffMsg + 2 * 128;
  static constexpr int kSmem = kOffMisc + 64 + 1024;  // + alignment slack
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kSmem <= 232448, "shared memory");
};

struct UnitInfo {
  int b, hk, hg, c0, ncols;  // columns c0 .. c0 + ncols - 1 of KV head hk
  int qrow0, q_len, kv_len;  // the batch's first token row; lengths (q_len <= S_max)
  int lo, hi;                // keys the batch's rows see together
  int lo_last, hi_first;     // the last row's lower bound, the first row's upper
  int tile0, ntiles;
};

// Keys [lo, hi] that query row i of a sequence sees, per the mask mode: modes
// 0 and 1 every key (an explicit mask then hides single keys), 2 the causal
// mask from the top-left corner (p = i), 3 from the bottom-right corner
// (p = kv_len - q_len + i), 4 the band p - pre .. p + next.  Clipped to
// [0, kv_len); hi < lo when the row sees nothing.
__device__ __forceinline__ void row_bounds(const DecodeArgs& a, int q_len, int kv_len, int i,
                                           int* lo, int* hi) {
  const int64_t p = (int64_t)(a.mask_mode == 2 ? 0 : kv_len - q_len) + i;
  int64_t l = 0, h = (int64_t)kv_len - 1;
  if (a.mask_mode == 2 || a.mask_mode == 3) {
    h = min(h, p);
  } else if (a.mask_mode == 4) {
    l = max(l, p - a.pre_tokens);
    h = min(h, p + a.next_tokens);
  }
  *lo = (int)min(l, (int64_t)kv_len);
  *hi = (int)max(h, (int64_t)-1);
}

// Rows of batch b the decode units cover: its query length, at most S_max.
__device__ __forceinline__ int clamp_rows(const DecodeArgs& a, int64_t ql) {
  return (int)min(max(ql, (int64_t)0), (int64_t)a.S_max);
}

// Active column groups of a KV head of a batch with q_len rows.
__device__ __forceinline__ int active_groups(const DecodeArgs& a, int q_len) {
  return q_len > 0 ? (q_len * a.G + a.GH - 1) / a.GH : 0;
}

// Unit w of batch b with the batch's first token row and lengths known.
__device__ __forceinline__ UnitInfo unit_from(const DecodeArgs& a, int b, int w, int qrow0,
                                              int64_t ql, int kv_len) {
  UnitInfo r;
  r.b = b;
  r.hk = w / a.HG;
  r.hg = w % a.HG;
  r.c0 = r.hg * a.GH;
  r.q_len = clamp_rows(a, ql);
  r.ncols = max(0, min(a.GH, r.q_len * a.G - r.c0));
  r.qrow0 = qrow0;
  r.kv_len = kv_len;
  r.lo = r.lo_last = 0;
  r.hi = r.hi_first = -1;
  r.tile0 = r.ntiles = 0;
  if (r.q_len > 0 && kv_len > 0) {
    int lo1, hi0;
    row_bounds(a, r.q_len, kv_len, 0, &r.lo, &hi0);
    row_bounds(a, r.q_len, kv_len, r.q_len - 1, &lo1, &r.hi);
    r.lo_last = lo1;
    r.hi_first = hi0;
    if (r.hi >= r.lo) {
      r.tile0 = r.lo / kKvTile;
      r.ntiles = r.hi / kKvTile - r.lo / kKvTile + 1;
    }
  }
  return r;
}

// First token row, query length and KV length of batch b.
__device__ __forceinline__ void batch_lengths(const DecodeArgs& a, int b, int64_t* qrow,
                                              int64_t* ql, int64_t* kv_len) {
  if (a.layout == 1) {
    *qrow = a.cu_seqlens_q[b];
    *ql = (int64_t)a.cu_seqlens_q[b + 1] - *qrow;
  } else {
    *qrow = (int64_t)b * a.S_q;
    *ql = a.S_q;
  }
  *kv_len = a.seqused_kv ? a.seqused_kv[b] : a.S_kv;
}

// What the producer hands the consumers with each chunk's query rows (one per
// query buffer), so that consumers never wait on global loads between chunks.
struct UnitMsg {
  UnitInfo r;
  int64_t slot;   // partial slot of this chunk: Q[b] + ci * A(b) + active index
  int ci, nch;    // chunk index within the unit, chunks of the unit
  int t_begin, t_end, done;
};
static_assert(sizeof(UnitMsg) <= 128, "message slot");

// Chunking of a unit of `cost` tiles: n1 big chunks of C tiles, then small
// chunks of c2 tiles over the rest.
struct ChunkGeom {
  int n1, nch;
};
// A unit's cost is below 2^31 and C, c2 matter only up to it, so 32-bit
// divisions give the 64-bit results (a 64-bit division costs several times
// more, and this sits on the path to a chunk's first load).
__device__ __forceinline__ ChunkGeom chunk_geom(int64_t cost, int64_t C, int64_t c2) {
  ChunkGeom g;
  const uint32_t c = (uint32_t)cost;
  const uint32_t Cc = (uint32_t)min(C, (int64_t)0x7fffffff);
  const uint32_t c2c = (uint32_t)min(c2, (int64_t)0x7fffffff);
  const uint32_t q = c / Cc;
  const uint32_t n1 = q > 0 ? q - 1 : 0;
  const uint32_t rest = c - n1 * Cc;
  g.n1 = (int)n1;
  g.nch = (int)(n1 + (rest + c2c - 1) / c2c);
  return g;
}

// Cost of every active unit of batch b and its active groups per KV head
// (all active units of a batch see the same tiles).
__device__ __forceinline__ int64_t batch_cost(const DecodeArgs& a, int b, int* ha) {
  int64_t qrow, ql, kv_len;
  batch_lengths(a, b, &qrow, &ql, &kv_len);
  const UnitInfo r = unit_from(a, b, 0, (int)qrow, ql, (int)kv_len);
  *ha = active_groups(a, r.q_len);
  return r.q_len > 0 ? max(1, r.ntiles) : 0;
}

// largest b with prefix[b] <= g (prefix[0] = 0 <= g < prefix[B])
template <typename T>
__device__ __forceinline__ int find_batch(const T* prefix, int B, int64_t g) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

// Page index of logical KV row j (0 <= j < 2^31) of a paged cache: j / block_size
// as one wide multiply and a shift (the multiplier and shift come with the
// arguments).  The producer finds a page per tile, and a 64-bit division there
// costs more issue time than the rest of its per-tile work.
__device__ __forceinline__ int64_t page_index(const DecodeArgs& a, int64_t j) {
  return (int64_t)(((uint64_t)(uint32_t)j * a.bs_magic) >> a.bs_shift);
}
// Pool row and FP8 scale row of logical KV row j of batch b, KV head hk, in
// page blk, with jp = j - block_size * page_index(j) (j's row in its page).
// Token-major pages [pages, page rows, KV_N, D] are a matrix of KV_N * D
// columns whose rows are tokens; head-major pages [pages, KV_N, page rows, D]
// one of D columns whose rows are (page, head, token) ("...V5" Paged
// Attention group: BnBsH and BnNBsD).  FP8 scales are stored head-major inside
// each page, [pages, KV_N, page rows, D/64] (the paged per-token, per-head
// scale shape (blockNum, N, blockSize) of the FIA dequantisation parameters,
// with the 64-element tiles last).
__device__ __forceinline__ int64_t pool_row(const DecodeArgs& a, int b, int hk, int64_t blk,
                                            int64_t j, int64_t jp) {
  if (!a.block_table) return (int64_t)b * a.S_kv + j;
  return a.kv_layout == 1 ? (blk * a.KVN + hk) * a.block_size + jp : blk * a.block_size + jp;
}
__device__ __forceinline__ int64_t scale_row_in(const DecodeArgs& a, int b, int hk, int64_t blk,
                                                int64_t j, int64_t jp) {
  return a.block_table ? (blk * a.KVN + hk) * a.block_size + jp
                       : ((int64_t)b * a.KVN + hk) * a.S_kv + j;
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Final normalisation of one head: sink, 1/l, lse (natural log).
__device__ __forceinline__ void finish_head(const DecodeArgs& a, int h, float M, float L,
                                            float* scl_out, float* lse_out) {
  float scl = 0.f, lse = INFINITY;
  if (M != -INFINITY) {
    float Mp = M;
    if (a.sinks) {
      const float sk = a.sinks[h] * 1.4426950408889634f;
      Mp = fmaxf(M, sk);
      L = L * exp2f(M - Mp) + exp2f(sk - Mp);
    }
    scl = exp2f(M - Mp) / L;
    lse = (Mp + log2f(L)) * 0.6931471805599453f;
  }
  *scl_out = scl;
  *lse_out = lse;
}

}  // namespace

// ---------------------------------------------------------------------------
// scheduler
// ---------------------------------------------------------------------------
// Block-wide exclusive scan of three 32-bit counters; returns the block
// totals in tot[] (every thread).  One barrier after the warp totals are
// stored (each warp then sums the totals before it with a shuffle
// reduction), one before `ws` is reused.
__device__ __forceinline__ void scan3(uint32_t (&x)[3], uint32_t (&tot)[3], uint32_t (*ws)[3]) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
  uint32_t incl[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    uint32_t v = x[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    incl[k] = v;
    if (lane == 31) ws[wid][k] = v;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const uint32_t wv = lane < nw ? ws[lane][k] : 0u;
    uint32_t before = lane < wid ? wv : 0u, all = wv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    tot[k] = all;
    x[k] = before + incl[k] - x[k];
  }
  __syncthreads();
}

constexpr int kSchedSmemBatches = 2048;  // per-batch values kept in shared memory up to this B

// Per-batch cost and active groups in one shared-memory word: the cost is at
// most 20M / 128 tiles (< 2^24), the active groups at most 64.
__device__ __forceinline__ uint32_t pack_cost(int64_t cost, int ha) {
  return (uint32_t)cost | ((uint32_t)ha << 24);
}

__global__ void __launch_bounds__(1024) decode_schedule_kernel(const DecodeArgs a) {
  __shared__ uint32_t ws[32][3];
  __shared__ int64_t ws_total[32];
  // up to kSchedSmemBatches batches: lengths, costs and queue prefixes stay in
  // shared memory, so the batch arrays are read from global memory once
  __shared__ uint32_t s_cost[kSchedSmemBatches];
  __shared__ int s_kv[kSchedSmemBatches], s_qrow[kSchedSmemBatches + 1];
  __shared__ int sR[2][kSchedSmemBatches + 1];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  pdl_trigger();  // the decode kernel may set up while the plan is built
  // The decode kernel's first dependent load after its wait is a chunk's
  // page ids: this block pulls the block table into L2 while it works (four
  // 128-byte lines per thread at most, 512 KB).
  if (a.block_table) {
    const char* bt = reinterpret_cast<const char*>(a.block_table);
    const int64_t lines = ((int64_t)a.B * a.max_blocks * 4 + 127) >> 7;
    for (int64_t k = tid, i = 0; i < 4 && k < lines; ++i, k += blockDim.x)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(bt + (k << 7)));
  }
  const int B = a.B;
  const bool small = B <= kSchedSmemBatches;
  const int HG = a.HG;
  int64_t* sched = a.sched;
  int64_t* Q = sched + kSchedHeader;  // [B+1] partial slots before batch b
  int64_t* R1 = Q + (B + 1);          // [B+1] big-chunk queue positions
  int64_t* R2 = R1 + (B + 1);         // [B+1] small-chunk queue positions
  int64_t* SB = R2 + (B + 1);         // [B] batches cut into several chunks, then -1

  // total cost of the active units (and, for small B, each batch's lengths,
  // cost and active groups)
  int64_t part = 0;
  for (int b = tid; b < B; b += blockDim.x) {
    int64_t qrow, ql, kv_len;
    batch_lengths(a, b, &qrow, &ql, &kv_len);
    const UnitInfo r = unit_from(a, b, 0, (int)qrow, ql, (int)kv_len);
    const int64_t cost = r.q_len > 0 ? max(1, r.ntiles) : 0;
    const int ha = active_groups(a, r.q_len);
    part += cost * a.KVN * ha;
    if (small) {
      s_cost[b] = pack_cost(cost, ha);
      s_kv[b] = (int)kv_len;
      s_qrow[b] = (int)qrow;
    }
  }
  if (small && tid == 0)  // the end of the last batch's rows: query lengths are differences
    s_qrow[B] = a.layout == 1 ? a.cu_seqlens_q[B] : B * a.S_q;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) ws_total[wid] = part;
  __syncthreads();  // (also publishes the shared-memory batch values)
  int64_t total = lane < (int)(blockDim.x >> 5) ? ws_total[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  const int64_t T = total;
  const int64_t per = (int64_t)a.num_ctas * a.chunks_per_cta;
  // C = max(1, ceil(T / per)), with a 32-bit division whenever T allows
  int64_t C = 1;
  if (T > 0)
    C = (T - 1 <= 0xffffffffLL && per <= 0xffffffffLL)
            ? (int64_t)((uint32_t)(T - 1) / (uint32_t)per) + 1
            : (T - 1) / per + 1;
  const int64_t c2 = C <= 0x7fffffffLL
                         ? (int64_t)((uint32_t)(C + a.small_div - 1) / (uint32_t)a.small_div)
                         : (C + a.small_div - 1) / a.small_div;

  // per batch: big and small chunks of its active units and whether it is
  // split -> three exclusive scans (all chunks before b = big + small before b)
  int64_t carry[3] = {0, 0, 0};
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + tid;
    uint32_t x[3] = {0u, 0u, 0u};
    if (b < B) {
      int64_t cost;
      int ha;
      if (small) {
        cost = s_cost[b] & 0xffffffu;
        ha = (int)(s_cost[b] >> 24);
      } else {
        cost = batch_cost(a, b, &ha);
      }
      const uint32_t A = (uint32_t)(a.KVN * ha);
      if (cost > 0 && A > 0) {
        const ChunkGeom gm = chunk_geom(cost, C, c2);
        x[0] = (uint32_t)gm.n1 * A;
        x[1] = (uint32_t)(gm.nch - gm.n1) * A;
        x[2] = gm.nch > 1;
      }
    }
    const bool is_split = x[2] != 0;
    uint32_t tot[3];
    scan3(x, tot, ws);
    if (b < B && is_split) SB[carry[2] + x[2]] = b;
    if (b < B) {
      const int64_t r1 = carry[0] + x[0], r2 = carry[1] + x[1];
      Q[b] = r1 + r2;
      R1[b] = r1;
      R2[b] = r2;
      if (small) {
        sR[0][b] = (int)r1;
        sR[1][b] = (int)r2;
      }
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) carry[k] += tot[k];
  }
  // the list of split batches ends with -1 entries
  for (int64_t b = carry[2] + tid; b < B; b += blockDim.x) SB[b] = -1;
  // N <= n*W + 6*U always holds (the workspace bound); a plan that broke it
  // would run nothing and say so in the error word
  const int64_t n_all = carry[0] + carry[1];
  const bool fits = n_all <= a.max_chunks;
  const int64_t F = fits ? carry[0] : 0, N = fits ? n_all : 0;
  if (tid == 0) {
    Q[B] = n_all;
    R1[B] = carry[0];
    R2[B] = carry[1];
    if (small) {
      sR[0][B] = (int)carry[0];
      sR[1][B] = (int)carry[1];
    }
    sched[0] = C;
    sched[1] = c2;
    sched[2] = N;
    sched[3] = F;
    sched[4] = fits ? carry[2] : 0;  // split batches
    sched[5] = kDecodePlanMark;  // this plan's mark, B and CTA count
    sched[6] = B;
    sched[7] = a.num_ctas;
    a.claim[0] = a.claim[1] = 0;
    *a.prefill_mark = 0;  // the workspace holds no prefill plan any more
    *a.err = fits ? 0 : 2;  // error word of this plan's execution
  }
  __syncthreads();
  // the claim queue: big chunks, then small chunks (queue positions below
  // 2^31, as the workspace bound implies, take 32-bit arithmetic)
  for (int64_t g = tid; g < N; g += blockDim.x) {
    int b;
    int64_t local, r1 = 0;
    if (g < F) {
      b = small ? find_batch(sR[0], B, g) : find_batch(R1, B, g);
      local = g - (small ? sR[0][b] : R1[b]);
    } else {
      b = small ? find_batch(sR[1], B, g - F) : find_batch(R2, B, g - F);
      local = g - F - (small ? sR[1][b] : R2[b]);
      r1 = small ? sR[0][b + 1] - sR[0][b] : R1[b + 1] - R1[b];
    }
    int ha, kv_len, qrow, qlen;
    if (small) {
      ha = (int)(s_cost[b] >> 24);
      kv_len = s_kv[b];
      qrow = s_qrow[b];
      qlen = clamp_rows(a, (int64_t)s_qrow[b + 1] - s_qrow[b]);
    } else {
      int64_t q64, ql, kv64;
      batch_lengths(a, b, &q64, &ql, &kv64);
      qlen = clamp_rows(a, ql);
      ha = active_groups(a, qlen);
      kv_len = (int)kv64;
      qrow = (int)q64;
    }
    // a batch with queue entries has active units, so A >= 1
    const uint32_t A = (uint32_t)max(1, a.KVN * ha);
    const uint32_t qd = (uint32_t)local / A;
    const int act = (int)((uint32_t)local - qd * A);  // active unit index
    const int ci = (int)((uint32_t)r1 / A + qd);
    const int hac = max(ha, 1);
    const int w = (act / hac) * HG + act % hac;      // unit of the batch
    a.queue[g] = make_int4(b | (qlen << 16), (ci << 16) | w, kv_len, qrow);
  }
}

// ---------------------------------------------------------------------------
// split-KV combine helpers: the partials of a unit's chunks are folded in a
// fixed order (deterministic), then the sink and the final normalisation are
// applied.
// ---------------------------------------------------------------------------
// Fold chunk partials k = k0, k0 + step, ... (< nch) of one (unit, head) into
// (M, L, o0, o1) for the d-pair at d, eight loads in flight at a time.
template <int D>
__device__ __forceinline__ void fold_chunks(const float* base, int64_t kstride, int d, int k0,
                                            int step, int nch, float& M, float& L, float& o0,
                                            float& o1) {
  constexpr int NB = 8;  // partials in flight per thread
  for (int kb = k0; kb < nch; kb += NB * step) {
    float2 ml[NB], ov[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int kk = kb + k * step;
      ml[k] = make_float2(-INFINITY, 0.f);
      ov[k] = make_float2(0.f, 0.f);
      if (kk < nch) {
        const float* pp = base + kk * kstride;
        ml[k] = __ldcg(reinterpret_cast<const float2*>(pp + D));  // (m, l)
        ov[k] = __ldcg(reinterpret_cast<const float2*>(pp + d));
      }
    }
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      if (ml[k].x == -INFINITY) continue;
      const float Mn = fmaxf(M, ml[k].x);
      const float fo = M == -INFINITY ? 0.f : exp2f(M - Mn);
      const float fn = exp2f(ml[k].x - Mn);
      L = L * fo + ml[k].y * fn;
      o0 = o0 * fo + ov[k].x * fn;
      o1 = o1 * fo + ov[k].y * fn;
      M = Mn;
    }
  }
}

// Final O and lse of one column (query row i of the sequence, head h) whose
// chunk partials have been folded into (M, L, o0, o1) for the d-pair at d.
__device__ __forceinline__ void combine_store(const DecodeArgs& a, int b, int64_t tok, int i,
                                              int h, int D, int d, float M, float L, float o0,
                                              float o1) {
  float scl, lse;
  finish_head(a, h, M, L, &scl, &lse);
  uint16_t* o = a.out + tok * a.out_stride + (int64_t)h * D + d;
  *reinterpret_cast<uint32_t*>(o) = pack_bf16(o0 * scl, o1 * scl);
  if (a.lse && d == 0) {
    const int64_t li = a.layout == 1 ? tok * a.QN + h : ((int64_t)b * a.QN + h) * a.S_q + i;
    a.lse[li] = lse;
  }
}

// ---------------------------------------------------------------------------
// decode kernel
// ---------------------------------------------------------------------------
// NG: groups of 8 query columns per unit (1 or 2).  MR: the general form --
// several query rows per sequence (each column masked with its own row's
// bounds) or an explicit mask; without it every column of a unit is row 0 of
// its sequence, shares that row's bounds, and the per-column work drops out.
template <int D, bool FP8, int NG, bool MR>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv) {
  using Cfg = DecodeCfg<D, FP8>;
  constexpr int S = Cfg::kStages;
  constexpr int kProdWarps = FP8 ? 4 : 2;  // producer warps (a whole warpgroup is reserved)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* empty = full + S;
  uint64_t* qfull = empty + S;
  uint64_t* qempty = qfull + 2;
  uint64_t* vpost = qempty + 2;  // [2] chunk message posted, for producer warps 1-3
  int* misc = reinterpret_cast<int*>(smem + Cfg::kOffMisc);
  UnitMsg* msg = reinterpret_cast<UnitMsg*>(smem + Cfg::kOffMsg);
  float* red = reinterpret_cast<float*>(smem + Cfg::kOffRed);
  float* red_ml = reinterpret_cast<float*>(smem + Cfg::kOffRedMl);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);  // the K warp's and the V warp's arrivals (with their bytes)
      mbar_init(&empty[s], kConsumers);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], kConsumers + kProdWarps - 1);  // consumers and producer warps 1..
      mbar_init(&vpost[s], 1);
    }
    misc[0] = 0;  // abort flag
    fence_barrier_init();
  }
  if (tid == 0) {
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  __syncthreads();
  pdl_wait();  // the plan (and anything else before us on the stream) is complete

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs) : "memory");
    // ======================= producers =======================
    // Even warps stream the K boxes (and the explicit-mask slices), odd warps
    // the V boxes; with an FP8 cache, warps 0/1 take the even tiles and 2/3
    // the odd ones, without it warps 0/1 take every tile.  Warp 0 also does
    // the chunk bookkeeping (claims, chunk messages, query vectors); the
    // others follow the messages it posts (vpost), walking the same tiles.
    // So the per-tile page lookups, address arithmetic and copy issue are
    // spread over several warps (the FP8 decode's single producer was busy
    // most of its time: 155.8 -> 150.2 us with two warps, 141.8 us with four;
    // the bf16 decodes gain nothing from more than two).  The two warps of a
    // tile wait for its stage and each arrives on the stage's full barrier
    // with its own bytes (count 2).  FP8 scales go with their K or V boxes.
    if (warp >= kProdWarps) return;
    const int isv = warp & 1;
    const int parity_of_mine = warp >> 1;  // (four warps) the tiles (it & 1) == this one
    const int nrb = kKvTile / a.box_rows;
    const int nbox = nrb * Cfg::kNsub;  // boxes of K (or V) per tile, one per lane
    const int sub = lane % Cfg::kNsub;  // 128-byte column slice
    const int rb = lane / Cfg::kNsub;   // page piece
    int it = 0, ucount = 0;             // tiles and chunks issued
    bool aborted = false;
    // K/V pages are read once, unless two units of a KV head share them
    // (several column groups, neighbours in the queue): those keep the
    // default policy so that the second unit finds them in L2
    const bool once = a.HG == 1;
    const uint64_t pol = l2_evict_first_policy();

    // The chunk's page ids, one per lane, with one coalesced load when the
    // chunk spans at most 32 pages: each tile then finds its pages by a
    // shuffle instead of a dependent global load.
    struct Pages {
      int64_t pg0;
      int npg, mypage;
    };
    auto chunk_pages = [&](const UnitInfo& r, int t_begin, int t_end) -> Pages {
      Pages pp{0, 0, 0};
      if (a.block_table && r.ntiles > 0 && t_begin < t_end) {
        const int64_t jlo = (int64_t)(r.tile0 + t_begin) * kKvTile;
        const int64_t jhi = min((int64_t)(r.tile0 + t_end) * kKvTile, (int64_t)r.kv_len);
        pp.pg0 = page_index(a, jlo);
        pp.npg = (int)(page_index(a, jhi - 1) - pp.pg0 + 1);
        if (pp.npg <= 32 && lane < pp.npg)
          pp.mypage = a.block_table[(int64_t)r.b * a.max_blocks + pp.pg0 + lane];
      }
      return pp;
    };
    // One tile's K (isv 0) or V (isv 1) boxes and their FP8 scales, and for
    // K the explicit-mask slices of the unit's query rows; false after a
    // time-out (nothing issued).
    auto issue_tile = [&](const UnitInfo& r, int t, const Pages& pp, int i_first,
                          int i_last) -> bool {
      if (kProdWarps == 4 && (it & 1) != parity_of_mine) {  // the other warp of this kind has it
        ++it;
        return true;
      }
      const int s = it % S;
      const uint32_t par = ((it / S) & 1) ^ 1;
      const int64_t j0 = (int64_t)(r.tile0 + t) * kKvTile;
      const int64_t jb = j0 + (int64_t)rb * a.box_rows;
      const bool mine = lane < nbox && jb < r.kv_len;
      int64_t blk, jp = 0;
      if (a.block_table) {
        const int64_t pj = mine ? page_index(a, jb) : 0;
        jp = jb - pj * a.block_size;
        if (pp.npg > 0 && pp.npg <= 32) {
          blk = __shfl_sync(0xffffffffu, pp.mypage, (int)(pj - pp.pg0));
        } else {
          blk = mine ? (int64_t)a.block_table[(int64_t)r.b * a.max_blocks + pj] : 0;
        }
      } else {
        blk = 0;
      }
      if (a.debug && mine && a.block_table && (blk < 0 || blk >= a.num_blocks))
        atomicExch(a.err, 3);  // (read as zeros by the TMA box all the same)
      const int64_t prow = mine ? pool_row(a, r.b, r.hk, blk, jb, jp) : 0;
      constexpr int NT = D / 64;
      // FP8: the scales of one head inside a page are contiguous rows of NT
      // floats, so each (K or V, page piece) is one bulk copy next to its
      // TMA box.  Pieces are even-length at even rows (block sizes are
      // multiples of 32; contiguous caches have an even length), hence
      // 16-byte aligned.
      // (a page id outside the pool reads zeros through TMA; its FP8
      // scales, which come by plain bulk copy, are not read at all)
      int64_t srow = 0;
      int srows = a.box_rows;
      bool scale_ok = false;
      if constexpr (FP8) {
        scale_ok = mine && (!a.block_table || (blk >= 0 && blk < a.num_blocks));
        if (scale_ok) srow = scale_row_in(a, r.b, r.hk, blk, jb, jp);
        if (!a.block_table) srows = (int)min((int64_t)a.box_rows, (int64_t)a.S_kv - jb);
      }
      int nvalid = 0;
      for (int q = 0; q < nrb; ++q)
        if (j0 + (int64_t)q * a.box_rows < r.kv_len) ++nvalid;
      uint32_t scale_bytes = 0;
      if constexpr (FP8)
        scale_bytes = __reduce_add_sync(0xffffffffu, scale_ok ? (uint32_t)(srows * NT * 4) : 0u);
      // explicit mask (K warp): the tile's slice of each of the unit's query
      // rows, 16-byte pieces up to kv_len (row strides are multiples of 16
      // that cover the KV capacity, so the copy stays inside the row)
      const bool with_mask = MR && a.mask && isv == 0;
      const int mrow_bytes =
          with_mask ? (int)min((int64_t)kKvTile, ((int64_t)r.kv_len - j0 + 15) & ~(int64_t)15) : 0;
      const int nmrows = with_mask ? i_last - i_first + 1 : 0;
      wait_or_abort(&empty[s], par, a.err, misc);
      if (*reinterpret_cast<volatile int*>(misc)) return false;  // issue nothing after a time-out
      uint8_t* st = smem + s * Cfg::kStageBytes;
      if (lane == 0) {
        uint32_t bytes = (uint32_t)(nvalid * Cfg::kNsub * a.box_rows * 128);
        if constexpr (FP8) bytes += scale_bytes;
        bytes += (uint32_t)(nmrows * mrow_bytes);
        mbar_arrive_expect_tx(&full[s], bytes);
      }
      __syncwarp();
      if (with_mask && lane < nmrows)
        bulk_load(st + Cfg::kOffMask + lane * kKvTile,
                  a.mask + (int64_t)r.b * a.mask_bstride + (int64_t)(i_first + lane) * a.mask_rstride +
                      j0,
                  (uint32_t)mrow_bytes, &full[s]);
      if (mine) {
        uint8_t* dst = st + isv * Cfg::kTileBytes + sub * (kKvTile * 128) + rb * a.box_rows * 128;
        const int col = (a.kv_layout == 1 ? 0 : r.hk * D) + (FP8 ? 0 : sub * 64);
        if (once)
          tma_load_2d_hint(dst, isv ? &tv : &tk, &full[s], col, (int)prow, pol);
        else
          tma_load_2d(dst, isv ? &tv : &tk, &full[s], col, (int)prow);
        if constexpr (FP8) {
          float* sdst = reinterpret_cast<float*>(st + 2 * Cfg::kTileBytes) + isv * (kKvTile * NT) +
                        rb * a.box_rows * NT;
          if (scale_ok)
            bulk_load(sdst, (isv ? a.v_scale : a.k_scale) + srow * NT, (uint32_t)(srows * NT * 4),
                      &full[s]);
        }
      }
      ++it;
      return true;
    };
    auto drain = [&]() {
      // a wait timed out: issue nothing more, give the copies already in
      // flight a bounded time to land, and leave (the error word is set)
      for (int k = max(0, it - S); k < it; ++k) mbar_wait(&full[k % S], (k / S) & 1, a.err);
    };

    if (warp != 0) {
      // ---- warps 1..: the chunks warp 0 posts, in order, until the empty one ----
      while (true) {
        const int qs = ucount & 1;
        wait_or_abort(&vpost[qs], (ucount >> 1) & 1, a.err, misc);
        const bool done = msg[qs].done != 0;
        const UnitInfo r = msg[qs].r;
        const int t_begin = msg[qs].t_begin, t_end = msg[qs].t_end;
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[qs]);  // the message is read
        ++ucount;
        if (done || *reinterpret_cast<volatile int*>(misc)) break;
        const Pages pp = chunk_pages(r, t_begin, t_end);
        // the unit's query rows (their explicit-mask slices go with K)
        const int i_first = MR ? r.c0 / a.G : 0;
        const int i_last = MR ? (r.c0 + max(r.ncols, 1) - 1) / a.G : 0;
        for (int t = t_begin; r.ntiles > 0 && t < t_end; ++t)
          if (!issue_tile(r, t, pp, i_first, i_last)) {
            aborted = true;
            break;
          }
        if (aborted) break;
      }
      if (aborted || *reinterpret_cast<volatile int*>(misc)) drain();
      return;
    }

    // ---- K warp ----
    // A plan of these arguments carries the scheduler's mark, B and CTA
    // count, and no prefill plan has been written over the workspace since;
    // without one (execute on a workspace never planned, or planned for the
    // prefill branch last) nothing runs and the error word says 2.  Queue
    // entries and partial slots are range-checked as well, so a plan of
    // other lengths cannot send a load or store out of bounds.
    // (the CTA's first queue entry is loaded beside the plan's header, not
    // after it: entry blockIdx.x lies inside the queue buffer, which holds
    // max_chunks >= gridDim.x entries, and is used only if the plan checks out)
    // (all header words are loaded before any is tested: one round trip)
    const int4 ent0 = a.queue[blockIdx.x];
    int64_t hd[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) hd[k] = a.sched[k];
    const int64_t pmark = *a.prefill_mark;
    const bool plan_ok = (hd[5] == kDecodePlanMark) & (hd[6] == a.B) & (hd[7] == a.num_ctas) &
                         (hd[0] >= 1) & (hd[1] >= 1) & (hd[2] >= 0) & (hd[2] <= a.max_chunks) &
                         (pmark != kPrefillPlanMark);
    if (!plan_ok && lane == 0 && blockIdx.x == 0) atomicExch(a.err, 2);
    const int64_t C = plan_ok ? hd[0] : 1, c2 = plan_ok ? hd[1] : 1;
    const int64_t N = plan_ok ? hd[2] : 0;
    const int UPB = a.KVN * a.HG;
    // CTA c starts with queue entry c (no claim on the way to the first
    // loads); the entries after the first gridDim.x are claimed with the
    // counter, each claim issued one chunk ahead and read only after the
    // chunk's tiles are queued, so its latency hides
    int64_t g = plan_ok ? (int64_t)blockIdx.x : N;
    int4 ent = g < N ? ent0 : make_int4(0, 0, 0, 0);
    while (g < N) {
      // claim the next chunk now; its result and queue entry are read once
      // the first tile of this chunk is queued, so neither latency is exposed
      int gn_l = 0;
      if (lane == 0) gn_l = (int)gridDim.x + atomicAdd(a.claim, 1);
      int64_t gn = N;
      int4 ent_n = make_int4(0, 0, 0, 0);
      bool fetched = false;
      // entry: (b | q_len << 16, chunk << 16 | unit of b, kv_len, first token row)
      const int b = ent.x & 0xffff, ql = (int)((uint32_t)ent.x >> 16);
      const int ci = (int)((uint32_t)ent.y >> 16), w = ent.y & 0xffff;
      bool ent_ok = b < a.B && ql >= 1 && ql <= a.S_max && w < UPB && ent.z >= 0 &&
                    ent.z <= a.S_kv && ent.w >= 0 && (int64_t)ent.w + ql <= a.q_rows;
      const UnitInfo r = unit_from(a, b, w, ent.w, ql, ent.z);
      const int ha = active_groups(a, r.q_len);
      ent_ok = ent_ok && r.hg < ha && r.ncols > 0;  // an active unit of the batch
      if (!ent_ok && lane == 0) atomicExch(a.err, 2);
      const int64_t cost = max(1, r.ntiles);
      const ChunkGeom gm = chunk_geom(cost, C, c2);
      int t_begin, t_end;
      if (ci < gm.n1) {
        t_begin = (int)(ci * C);
        t_end = (int)(t_begin + C);
      } else {
        t_begin = (int)(gm.n1 * C + (ci - gm.n1) * c2);
        t_end = (int)min(cost, t_begin + c2);
      }
      if (!ent_ok || ci >= gm.nch) t_begin = t_end = 0;  // nothing of a bad entry runs
      // query rows of the unit's columns: one row of the sequence per range
      // (without MR every column is row 0)
      const int i_first = MR ? r.c0 / a.G : 0;
      const int i_last = MR ? (r.c0 + max(r.ncols, 1) - 1) / a.G : 0;
      // the chunk's page ids first: their load overlaps the message and the
      // query copies below
      const Pages pp = chunk_pages(r, t_begin, t_end);
      if (ent_ok && ci < gm.nch) {  // chunk description + the columns' query vectors
        const int qs = ucount & 1;
        wait_or_abort(&qempty[qs], ((ucount >> 1) & 1) ^ 1, a.err, misc);
        if (lane == 0) {
          UnitMsg& m = msg[qs];
          m.r = r;
          // partial slot: Q[b] + ci * A(b) + active index (clamped by the consumers)
          m.slot = (int64_t)ci * (a.KVN * ha) + r.hk * ha + r.hg;
          m.ci = ci;
          m.nch = gm.nch;
          m.t_begin = t_begin;
          m.t_end = t_end;
          m.done = 0;
          mbar_arrive(&vpost[qs]);  // producer warps 1-3 may read the message
          mbar_arrive_expect_tx(&qfull[qs], (uint32_t)(r.ncols * D * 2));
        }
        __syncwarp();
        // the columns of query row i are heads cb - i*G .. ce - 1 - i*G of the
        // group, contiguous in q: one bulk copy per row, row i from lane i - i_first
        for (int i = i_first + lane; i <= i_last; i += 32) {
          const int cb = max(r.c0, i * a.G), ce = min(r.c0 + r.ncols, (i + 1) * a.G);
          bulk_load(smem + Cfg::kOffQ + qs * Cfg::kQBytes + (cb - r.c0) * D * 2,
                    a.q + ((int64_t)r.qrow0 + i) * a.q_stride +
                        ((int64_t)r.hk * a.G + cb - i * a.G) * D,
                    (uint32_t)((ce - cb) * D * 2), &qfull[qs]);
        }
        ++ucount;
      }
      for (int t = t_begin; r.ntiles > 0 && t < t_end; ++t) {
        if (!issue_tile(r, t, pp, i_first, i_last)) {
          aborted = true;
          break;
        }
        if (!fetched) {
          gn = __shfl_sync(0xffffffffu, (int64_t)gn_l, 0);
          if (gn < N) ent_n = a.queue[gn];
          fetched = true;
        }
      }
      if (aborted || *reinterpret_cast<volatile int*>(misc)) {
        aborted = true;
        break;
      }
      if (!fetched) {
        gn = __shfl_sync(0xffffffffu, (int64_t)gn_l, 0);
        if (gn < N) ent_n = a.queue[gn];
      }
      g = gn;
      ent = ent_n;
    }
    if (aborted) {
      drain();
      return;
    }
    pdl_trigger();  // this CTA loads nothing more: the combine kernel may launch
    // this CTA claims no more: the last CTA out resets the queue for the
    // next fia_execute with the same plan
    if (lane == 0 && plan_ok) {
      __threadfence();  // this CTA's last claim is performed before it counts out
      if (atomicAdd(a.claim + 1, 1) == a.num_ctas - 1) {
        a.claim[0] = 0;
        a.claim[1] = 0;
      }
    }
    {  // end of the CTA's work: an empty message, for the consumers and warps 1-3
      const int qs = ucount & 1;
      wait_or_abort(&qempty[qs], ((ucount >> 1) & 1) ^ 1, a.err, misc);
      if (lane == 0) {
        msg[qs].done = 1;
        mbar_arrive(&vpost[qs]);
        mbar_arrive(&qfull[qs]);
      }
    }
    return;
  }

  // ======================= consumers =======================
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsRegs) : "memory");
  const int cw = warp - 4;     // 0..7
  const int g = lane >> 2;     // fragment row group
  const int q4 = lane & 3;     // thread in quad
  const int R0 = cw * kRowsPerWarp;
  const int nthr = 32 * kConsumers;
  const uint32_t smem_base = smem_u32(smem);
  constexpr int KS = D / 16;   // k-steps over D (QK)
  constexpr int MT = D / 16;   // m-tiles over D (PV)

  int it = 0, ucount = 0;
  while (true) {
    const int qs = ucount & 1;
    wait_or_abort(&qfull[qs], (ucount >> 1) & 1, a.err, misc);
    // every consumer warp leaves together (the merge meets at a named
    // barrier), so the stop decision is one barrier OR over the consumers
    if (named_bar_or(1, nthr, msg[qs].done || *reinterpret_cast<volatile int*>(misc))) break;
    const UnitInfo r = msg[qs].r;
    const int kvl = r.kv_len;
    // this chunk's partial slot: Q[b] + chunk * A(b) + active index
    const int64_t slot0 = a.sched[kSchedHeader + r.b] + msg[qs].slot;
    const int t_begin = msg[qs].t_begin, t_end = msg[qs].t_end;
    const int nch = msg[qs].nch;
    const bool split = nch > 1;
    const int64_t pstride = (int64_t)a.GH * (D + 2);  // floats per partial slot
    // keys seen by the query rows of accumulator columns 2*q4 + e of each
    // group of 8 (every column its own row; columns past the unit's count
    // take its last one), and their rows among the unit's mask rows
    int loc[NG][2], hic[NG][2], mrow[NG][2];
    if constexpr (MR) {
      const int i_first = r.c0 / a.G;
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = (r.c0 + min(ng * 8 + 2 * q4 + e, max(r.ncols, 1) - 1)) / a.G;
          row_bounds(a, r.q_len, kvl, i, &loc[ng][e], &hic[ng][e]);
          mrow[ng][e] = (i - i_first) * kKvTile;
        }
    } else {
      // one row: the unit's bounds are every column's
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          loc[ng][e] = r.lo;
          hic[ng][e] = r.hi;
          mrow[ng][e] = 0;
        }
    }

    // ---- Q^T fragments (mma B operand: k = d, n = column) ----
    uint32_t qb[NG][KS][2];
    // score factor: scale * log2(e), times 2^-sh on the FP8 path (below)
    float slc = a.scale_log2;
    {
      const uint16_t* qsm = reinterpret_cast<const uint16_t*>(smem + Cfg::kOffQ + qs * Cfg::kQBytes);
      if constexpr (!FP8) {
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          const int head = ng * 8 + g;  // the unit's column in this lane's B fragments
          const bool ok = head < r.ncols;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const int d0 = kk * 16 + 2 * q4;
            qb[ng][kk][0] = ok ? *reinterpret_cast<const uint32_t*>(qsm + head * D + d0) : 0u;
            qb[ng][kk][1] = ok ? *reinterpret_cast<const uint32_t*>(qsm + head * D + d0 + 8) : 0u;
          }
        }
      } else {
        // The FP8 products run in fp16, whose range is far narrower than
        // bf16's.  The unit's queries are multiplied by 2^sh, a power of two
        // chosen from the largest exponent E among them so that the largest
        // element lands at exponent 15 (sh = 15 - E, kept in [-100, 100]):
        // nothing overflows, every element within 2^-29 of the largest
        // converts exactly (smaller ones round to multiples of 2^(E-39),
        // far below the scores' tolerance), and the scores take 2^-sh back
        // in their scale factor.  Powers of two scale exactly.
        // k-step kk = 4*tile + j covers d = 64*tile + 16*q + 4*j + {0..3}:
        // slots 2q,2q+1 <- the first two, slots 2q+8,2q+9 <- the last two
        uint32_t emax = 0;
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          const int head = ng * 8 + g;
          if (head < r.ncols) {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
              const int d0 = (kk >> 2) * 64 + 16 * q4 + 4 * (kk & 3);
              const uint2 v = *reinterpret_cast<const uint2*>(qsm + head * D + d0);
              emax = max(emax, max(max((v.x >> 7) & 0xffu, (v.x >> 23) & 0xffu),
                                   max((v.y >> 7) & 0xffu, (v.y >> 23) & 0xffu)));
            }
          }
        }
        emax = __reduce_max_sync(0xffffffffu, emax);  // over the unit's columns
        const int sh = min(max(142 - (int)emax, -100), 100);  // 15 - (emax - 127)
        const float up = __int_as_float((127 + sh) << 23);
        slc = a.scale_log2 * __int_as_float((127 - sh) << 23);
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          const int head = ng * 8 + g;
          const bool ok = head < r.ncols;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const int d0 = (kk >> 2) * 64 + 16 * q4 + 4 * (kk & 3);
            if (ok) {
              const uint2 v = *reinterpret_cast<const uint2*>(qsm + head * D + d0);
              const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
              const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
              qb[ng][kk][0] = pack_f16(lo.x * up, lo.y * up);
              qb[ng][kk][1] = pack_f16(hi.x * up, hi.y * up);
            } else {
              qb[ng][kk][0] = qb[ng][kk][1] = 0u;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qs]);
      ++ucount;
    }

    // O^T accumulators: m-tile i (16 d rows) x head group ng (8 heads)
    float acc[MT][NG][4];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) acc[i][ng][0] = acc[i][ng][1] = acc[i][ng][2] = acc[i][ng][3] = 0.f;
    float m_r[NG][2], l_r[NG][2];  // per head 2q+e (exp2 domain)
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      m_r[ng][0] = m_r[ng][1] = -INFINITY;
      l_r[ng][0] = l_r[ng][1] = 0.f;
    }
    int vexp[2] = {0, 0};  // FP8: exponent of the V scale reference per d-tile (0: none yet)

    // FP8: the P V of each tile runs one tile late, beside the next tile's
    // Q K^T and softmax (two independent instruction streams per warp)
    struct PendingPV {
      bool valid;
      int s;
      int jw;
      bool tail;
      uint32_t pb[2][NG][2];
      float fct[2][NG][2];
    } prev;
    prev.valid = false;
    auto pv_fp8 = [&](const PendingPV& pp) {
      bool resc = false;
#pragma unroll
      for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) resc |= (pp.fct[t2][ng][0] != 1.f) | (pp.fct[t2][ng][1] != 1.f);
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          const int t2 = i >> 2;
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            acc[i][ng][0] *= pp.fct[t2][ng][0];
            acc[i][ng][1] *= pp.fct[t2][ng][1];
            acc[i][ng][2] *= pp.fct[t2][ng][0];
            acc[i][ng][3] *= pp.fct[t2][ng][1];
          }
        }
      }
      // V codes of KV slots 2q, 2q+1, 2q+8, 2q+9: 8 bytes per d-tile at
      // d = 64*tile + 8*g .. +7 (m-tile i covers d = 64*(i/4) + 8*g + (i%4)
      // in fragment rows 0-7 and +4 in rows 8-15); rows past kv_len -> 0
      const uint8_t* vt = smem + pp.s * Cfg::kStageBytes + Cfg::kTileBytes;
      uint2 w[4][2];
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        const int slot = 2 * q4 + (sl & 1) + (sl >> 1) * 8;
        const int row = R0 + rho16(slot);
        const bool ok = !pp.tail || (pp.jw + rho16(slot) < kvl);
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          uint2 x = *reinterpret_cast<const uint2*>(vt + sw128(row, 4 * t2 + (g >> 1)) + 8 * (g & 1));
          if (!ok) { x.x = 0u; x.y = 0u; }
          w[sl][t2] = x;
        }
      }
#pragma unroll
      for (int t2 = 0; t2 < 2; ++t2) {
#pragma unroll
        for (int ip = 0; ip < 4; ip += 2) {  // m-tiles 4*t2 + ip, +1
          // bytes ip, ip+1 (fragment rows 0-7) and 4+ip, 5+ip (rows 8-15)
          const uint32_t sel = (uint32_t)(ip | (4 + ip) << 4 | (ip + 1) << 8 | (5 + ip) << 12);
          const uint32_t p_lo01 = __byte_perm(w[0][t2].x, w[1][t2].x, sel);  // slots 2q,2q+1
          const uint32_t p_hi01 = __byte_perm(w[0][t2].y, w[1][t2].y, sel);
          const uint32_t p_lo89 = __byte_perm(w[2][t2].x, w[3][t2].x, sel);  // slots 2q+8,2q+9
          const uint32_t p_hi89 = __byte_perm(w[2][t2].y, w[3][t2].y, sel);
          uint32_t va[2][4];  // [h2]: the low and the high halves of the four words
          e4m3x4_to_f16x2x2(p_lo01, va[0][0], va[1][0]);
          e4m3x4_to_f16x2x2(p_hi01, va[0][1], va[1][1]);
          e4m3x4_to_f16x2x2(p_lo89, va[0][2], va[1][2]);
          e4m3x4_to_f16x2x2(p_hi89, va[0][3], va[1][3]);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int ng = 0; ng < NG; ++ng)
              mma_f16(acc[4 * t2 + ip + h2][ng], va[h2], pp.pb[t2][ng][0], pp.pb[t2][ng][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[pp.s]);
    };

    const int ntile_here = r.ntiles == 0 ? 0 : (t_end - t_begin);
    for (int tt = 0; tt < ntile_here; ++tt, ++it) {
      const int t = t_begin + tt;
      const int s = it % S;
      wait_or_abort(&full[s], (it / S) & 1, a.err, misc);
      const uint32_t st = smem_base + s * Cfg::kStageBytes;
      const uint8_t* stp = smem + s * Cfg::kStageBytes;
      // KV positions in 32 bits: lengths are int32, so every position and
      // bound here is below 2^31
      const int jw = (r.tile0 + t) * kKvTile + R0;  // first KV row of this warp
      // rows of this warp some column may not see (every column sees keys
      // lo_last .. hi_first, and hi_first < kv_len, so a tail is an edge)
      const bool edge =
          (jw < r.lo_last) || (jw + kRowsPerWarp - 1 > r.hi_first) || (MR && a.mask != nullptr);
      const bool tail = (jw + kRowsPerWarp > kvl);
      // KV positions of fragment rows g and g+8
      const int jg0 = jw + rho16(g), jg1 = jw + rho16(g + 8);

      // ---------------- S^T = K Q^T  (m = 16 KV rows, n = 8 heads) ----------------
      float sc[NG][4];
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) sc[ng][0] = sc[ng][1] = sc[ng][2] = sc[ng][3] = 0.f;
      if constexpr (!FP8) {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          // matrices: (rows 0-7, lo 8 d), (rows 8-15, lo), (rows 0-7, hi), (rows 8-15, hi)
          const int mi = lane >> 3;
          const int row = R0 + (mi & 1) * 8 + pi8(lane & 7);
          const int chunk = (kk & 3) * 2 + (mi >> 1);
          const uint32_t addr = st + (kk >> 2) * (kKvTile * 128) + sw128(row, chunk);
          uint32_t ka[4];
          ldsm_x4(addr, ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) mma_bf16(sc[ng], ka, qb[ng][kk][0], qb[ng][kk][1]);
        }
      } else {
        constexpr int NT = D / 64;
        float s2[NG][4];
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) s2[ng][0] = s2[ng][1] = s2[ng][2] = s2[ng][3] = 0.f;
        const int rowa = R0 + pi8(g), rowb = R0 + 8 + pi8(g);
#pragma unroll
        for (int tile = 0; tile < NT; ++tile) {
          const uint4 wa = *reinterpret_cast<const uint4*>(stp + sw128(rowa, tile * 4 + q4));
          const uint4 wb = *reinterpret_cast<const uint4*>(stp + sw128(rowb, tile * 4 + q4));
          const uint32_t va[4] = {wa.x, wa.y, wa.z, wa.w};
          const uint32_t vb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t ka[4];
            e4m3x4_to_f16x2x2(va[j], ka[0], ka[2]);
            e4m3x4_to_f16x2x2(vb[j], ka[1], ka[3]);
#pragma unroll
            for (int ng = 0; ng < NG; ++ng) {
              if (tile == 0) mma_f16(sc[ng], ka, qb[ng][tile * 4 + j][0], qb[ng][tile * 4 + j][1]);
              else mma_f16(s2[ng], ka, qb[ng][tile * 4 + j][0], qb[ng][tile * 4 + j][1]);
            }
          }
        }
        // per-row K scales of the two 64-column tiles (rows g and g+8)
        const float* ks = reinterpret_cast<const float*>(stp + 2 * Cfg::kTileBytes);
        float2 k0 = *reinterpret_cast<const float2*>(ks + rowa * NT);
        float2 k1 = *reinterpret_cast<const float2*>(ks + rowb * NT);
        if (tail) {
          if (jg0 >= kvl) k0 = make_float2(0.f, 0.f);
          if (jg1 >= kvl) k1 = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          sc[ng][0] = sc[ng][0] * k0.x + s2[ng][0] * k0.y;
          sc[ng][1] = sc[ng][1] * k0.x + s2[ng][1] * k0.y;
          sc[ng][2] = sc[ng][2] * k1.x + s2[ng][2] * k1.y;
          sc[ng][3] = sc[ng][3] * k1.x + s2[ng][3] * k1.y;
        }
      }

      // ---------------- mask + online softmax per column ----------------
      float corr[NG][2];
      // the reference moves only when a score passes it by more than 8 (log2
      // units): p <= 2^8 stays exact enough in 16-bit P, and the
      // accumulators are rarely rescaled.  One warp vote finds out whether
      // any column needs that; only then are the row maxima reduced.
      float xs[NG][4];
      bool over = false;
      if (!edge) {
#pragma unroll
        for (int ng = 0; ng < NG; ++ng)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            xs[ng][e] = sc[ng][e] * slc;
            xs[ng][2 + e] = sc[ng][2 + e] * slc;
          }
      } else {
        // each column against its own row's bounds, and the explicit mask's
        // bytes of that row (staged with the tile) where there is one
        const uint8_t* mk = stp + Cfg::kOffMask;
        const int ta = R0 + rho16(g), tb = R0 + rho16(g + 8);  // rows within the tile
#pragma unroll
        for (int ng = 0; ng < NG; ++ng)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            bool okA = jg0 >= loc[ng][e] && jg0 <= hic[ng][e];
            bool okB = jg1 >= loc[ng][e] && jg1 <= hic[ng][e];
            if (MR && a.mask) {
              okA = okA && mk[mrow[ng][e] + ta] == 0;
              okB = okB && mk[mrow[ng][e] + tb] == 0;
            }
            xs[ng][e] = okA ? sc[ng][e] * slc : -INFINITY;
            xs[ng][2 + e] = okB ? sc[ng][2 + e] * slc : -INFINITY;
          }
      }
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int e = 0; e < 2; ++e) over |= fmaxf(xs[ng][e], xs[ng][2 + e]) > m_r[ng][e] + 8.f;
      const bool any_over = __any_sync(0xffffffffu, over);
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x0 = xs[ng][e], x1 = xs[ng][2 + e];
          const float mold = m_r[ng][e];
          float mn = mold;
          if (any_over) {
            float mx = fmaxf(x0, x1);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            mn = mx > mold + 8.f ? mx : mold;
          }
          const float mu = mn == -INFINITY ? 0.f : mn;
          corr[ng][e] = mn == mold ? 1.f : (mold == -INFINITY ? 0.f : fast_exp2(mold - mu));
          m_r[ng][e] = mn;
          const float p0 = fast_exp2(x0 - mu), p1 = fast_exp2(x1 - mu);
          sc[ng][e] = p0;
          sc[ng][2 + e] = p1;
          l_r[ng][e] = l_r[ng][e] * corr[ng][e] + p0 + p1;
        }
      }

      // ---------------- O^T += V^T P^T ----------------
      if constexpr (!FP8) {
        // P^T as the B operand: transpose the two 8x8 halves of S^T
        uint32_t pb[NG][2];
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          pb[ng][0] = movmatrix_t(pack_bf16(sc[ng][0], sc[ng][1]));
          pb[ng][1] = movmatrix_t(pack_bf16(sc[ng][2], sc[ng][3]));
        }
        bool resc = false;
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) resc |= (corr[ng][0] != 1.f) | (corr[ng][1] != 1.f);
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int ng = 0; ng < NG; ++ng) {
              acc[i][ng][0] *= corr[ng][0];
              acc[i][ng][1] *= corr[ng][1];
              acc[i][ng][2] *= corr[ng][0];
              acc[i][ng][3] *= corr[ng][1];
            }
        }
        // rows past kv_len may hold anything (even NaN): zero their V lanes
        bool z0 = false, z1 = false, z2 = false, z3 = false;
        if (tail) {
          z0 = jw + rho16(2 * q4) >= kvl;
          z1 = jw + rho16(2 * q4 + 1) >= kvl;
          z2 = jw + rho16(2 * q4 + 8) >= kvl;
          z3 = jw + rho16(2 * q4 + 9) >= kvl;
        }
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          // A = V^T (m = d, k = KV rows): matrices (k 0-7, d lo8), (k 0-7, d hi8),
          // (k 8-15, d lo8), (k 8-15, d hi8) of V[row][d], transposed by ldmatrix
          const int mi = lane >> 3;
          const int row = R0 + (mi >> 1) * 8 + pi8(lane & 7);
          const int dchunk = 2 * i + (mi & 1);
          const uint32_t addr = st + Cfg::kTileBytes + (dchunk >> 3) * (kKvTile * 128) +
                                sw128(row, dchunk & 7);
          uint32_t va[4];
          ldsm_x4_t(addr, va[0], va[1], va[2], va[3]);
          if (tail) {
            if (z0) { va[0] &= 0xffff0000u; va[1] &= 0xffff0000u; }
            if (z1) { va[0] &= 0x0000ffffu; va[1] &= 0x0000ffffu; }
            if (z2) { va[2] &= 0xffff0000u; va[3] &= 0xffff0000u; }
            if (z3) { va[2] &= 0x0000ffffu; va[3] &= 0x0000ffffu; }
          }
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) mma_bf16(acc[i][ng], va, pb[ng][0], pb[ng][1]);
        }
      } else {
        constexpr int NT = D / 64;
        static_assert(NT == 2, "FP8 decode is built for D = 128");
        const float* vs = reinterpret_cast<const float*>(stp + 2 * Cfg::kTileBytes + Cfg::kScaleBytes);
        const int rowa = R0 + pi8(g), rowb = R0 + 8 + pi8(g);
        // V scales of fragment rows g, g+8 (zero past kv_len)
        float2 v0 = *reinterpret_cast<const float2*>(vs + rowa * NT);
        float2 v1 = *reinterpret_cast<const float2*>(vs + rowb * NT);
        if (tail) {
          if (jg0 >= kvl) v0 = make_float2(0.f, 0.f);
          if (jg1 >= kvl) v1 = make_float2(0.f, 0.f);
        }
        // Warp-wide power-of-two reference per d-tile: 2^(e-127) with e the
        // largest exponent of a V scale seen so far (positive floats order
        // like their bit patterns, so one warp max over the bits finds it).
        // P^T * scale / ref then stays below 2^9 in fp16, and moving the
        // reference rescales the accumulators by an exact power of two.
        float ratio[2], iv[2];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          const uint32_t bits = max(__float_as_uint(t2 ? v0.y : v0.x), __float_as_uint(t2 ? v1.y : v1.x));
          const int e = (int)(__reduce_max_sync(0xffffffffu, bits) >> 23);
          const int en = max(vexp[t2], e);
          // 2^(old - new) and 2^(127 - new) built from their exponent bits
          // (a jump past 2^-126 leaves a negligible old sum and gives 0)
          ratio[t2] = (en == vexp[t2] || vexp[t2] == 0)
                          ? 1.f
                          : __int_as_float(max(127 + vexp[t2] - en, 0) << 23);
          vexp[t2] = en;
          iv[t2] = (en > 0 && en < 254) ? __int_as_float((254 - en) << 23) : 1.f;
        }
        // P^T of this tile with the V scales folded in, and the factors the
        // accumulators take before its P V is added
        uint32_t pb[2][NG][2];
        float fct[2][NG][2];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          const float fa = (t2 ? v0.y : v0.x) * iv[t2], fb = (t2 ? v1.y : v1.x) * iv[t2];
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            pb[t2][ng][0] = movmatrix_t(pack_f16(sc[ng][0] * fa, sc[ng][1] * fa));
            pb[t2][ng][1] = movmatrix_t(pack_f16(sc[ng][2] * fb, sc[ng][3] * fb));
            fct[t2][ng][0] = corr[ng][0] * ratio[t2];
            fct[t2][ng][1] = corr[ng][1] * ratio[t2];
          }
        }
        // P V of the previous tile: independent of this tile's work above, so
        // the two interleave (the previous stage is released after it)
        if (prev.valid) pv_fp8(prev);
        prev.valid = true;
        prev.s = s;
        prev.jw = jw;
        prev.tail = tail;
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            prev.pb[t2][ng][0] = pb[t2][ng][0];
            prev.pb[t2][ng][1] = pb[t2][ng][1];
            prev.fct[t2][ng][0] = fct[t2][ng][0];
            prev.fct[t2][ng][1] = fct[t2][ng][1];
          }
        continue;  // the stage stays held until its P V ran
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if constexpr (FP8) {
      if (prev.valid) pv_fp8(prev);  // the chunk's last tile
    }

    // ---------------- merge the eight warps' states ----------------
    if constexpr (FP8) {
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const float f = vexp[i >> 2] > 0 ? __int_as_float(vexp[i >> 2] << 23) : 1.f;  // 2^(e-127)
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          acc[i][ng][0] *= f; acc[i][ng][1] *= f; acc[i][ng][2] *= f; acc[i][ng][3] *= f;
        }
      }
    }
    // d index of accumulator row: m-tile i, fragment row gg (0..15)
    auto drow = [&](int i, int gg) -> int {
      if constexpr (!FP8) return 16 * i + gg;
      else return 64 * (i >> 2) + 8 * (gg & 7) + 4 * (gg >> 3) + (i & 3);
    };
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = l_r[ng][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_r[ng][e] = l;
      }
      if (g == 0) {
        red_ml[(cw * kMaxGH + ng * 8 + 2 * q4) * 2 + 0] = m_r[ng][0];
        red_ml[(cw * kMaxGH + ng * 8 + 2 * q4) * 2 + 1] = l_r[ng][0];
        red_ml[(cw * kMaxGH + ng * 8 + 2 * q4 + 1) * 2 + 0] = m_r[ng][1];
        red_ml[(cw * kMaxGH + ng * 8 + 2 * q4 + 1) * 2 + 1] = l_r[ng][1];
      }
    }
    named_bar_sync(1, nthr);
    // every thread: combined (M, L) of its columns, and its own scale factor
    float Mh[NG][2], Lh[NG][2];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int head = ng * 8 + 2 * q4 + e;
        float M = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < kConsumers; ++w2) M = fmaxf(M, red_ml[(w2 * kMaxGH + head) * 2]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kConsumers; ++w2) {
          const float mw = red_ml[(w2 * kMaxGH + head) * 2];
          L += mw == -INFINITY ? 0.f : red_ml[(w2 * kMaxGH + head) * 2 + 1] * exp2f(mw - Mu);
        }
        Mh[ng][e] = M;
        Lh[ng][e] = L;
        const float f = m_r[ng][e] == -INFINITY ? 0.f : exp2f(m_r[ng][e] - Mu);
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          acc[i][ng][e] *= f;
          acc[i][ng][2 + e] *= f;
        }
      }
    }
    // Reduce-scatter of the scaled accumulators: warp w ends with m-tile w
    // (its 16 d rows) summed over the eight warps.  The m-tiles go through
    // shared memory in rounds of four ([4 slots][8 warps][32 lanes] float4,
    // 16 KB): round r carries m-tiles i = r, r + R, ... (R = MT / 4 rounds),
    // every warp stores those it does not own, then each owner adds the
    // other seven warps' copies of its m-tile to its own.  Lanes keep their
    // fragment layout throughout, so every access is a conflict-free 16-byte
    // one.  red_ml (read above) is rewritten only by the next chunk's merge.
    constexpr int R = MT / 4;
    float4* red4 = reinterpret_cast<float4*>(red);
    const int d0 = drow(cw, g), d1 = drow(cw, g + 8);
    const int64_t slot = min(max(slot0, (int64_t)0), a.max_chunks - 1);
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      float own[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int rnd = 0; rnd < R; ++rnd) {
        if (ng > 0 || rnd > 0) named_bar_sync(1, nthr);  // the previous round's reads are done
#pragma unroll
        for (int i = rnd; i < MT; i += R)
          if (i != cw)
            red4[((i / R) * kConsumers + cw) * 32 + lane] =
                make_float4(acc[i][ng][0], acc[i][ng][1], acc[i][ng][2], acc[i][ng][3]);
        named_bar_sync(1, nthr);
        if (cw < MT && cw % R == rnd) {
#pragma unroll
          for (int i = rnd; i < MT; i += R)
            if (i == cw) {
              own[0] = acc[i][ng][0];
              own[1] = acc[i][ng][1];
              own[2] = acc[i][ng][2];
              own[3] = acc[i][ng][3];
            }
#pragma unroll
          for (int w2 = 0; w2 < kConsumers; ++w2) {
            if (w2 == cw) continue;
            const float4 x = red4[((cw / R) * kConsumers + w2) * 32 + lane];
            own[0] += x.x; own[1] += x.y; own[2] += x.z; own[3] += x.w;
          }
        }
      }
      // the owner warp writes its d rows of this group's columns: the final
      // O (bf16, times the column's 1/L and sink factor) and lse, or the
      // partial slot (fp32 accumulator, then m and l after the D values)
      if (cw < MT) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = ng * 8 + 2 * q4 + e;  // the unit's column
          if (hh >= r.ncols) continue;
          if (!split) {
            const int c = r.c0 + hh;  // column: query row i, head h
            const int i = c / a.G, h = r.hk * a.G + (c - i * a.G);
            const int64_t tok = (int64_t)r.qrow0 + i;
            float scl, lse;
            finish_head(a, h, Mh[ng][e], Lh[ng][e], &scl, &lse);
            uint16_t* o = a.out + tok * a.out_stride + (int64_t)h * D;
            const __nv_bfloat16 v0 = __float2bfloat16_rn(own[e] * scl);
            const __nv_bfloat16 v1 = __float2bfloat16_rn(own[2 + e] * scl);
            o[d0] = *reinterpret_cast<const uint16_t*>(&v0);
            o[d1] = *reinterpret_cast<const uint16_t*>(&v1);
            if (a.lse && cw == 0 && g == 0) {
              const int64_t li =
                  a.layout == 1 ? tok * a.QN + h : ((int64_t)r.b * a.QN + h) * a.S_q + i;
              a.lse[li] = lse;
            }
          } else {
            // (the slot is clamped: a plan of other lengths cannot move the
            // write out of the partial slots; the combine rejects such a
            // plan's prefixes)
            float* col = a.partials + slot * pstride + (int64_t)hh * (D + 2);
            col[d0] = own[e];
            col[d1] = own[2 + e];
            if (cw == 0 && g == 0) {
              col[D] = Mh[ng][e];
              col[D + 1] = Lh[ng][e];
            }
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// split-KV combine, launched right after the decode kernel: one item per
// (batch with several chunks per unit, unit, head), found from the schedule's
// list of such batches; the partials are folded in chunk order.
// ---------------------------------------------------------------------------
struct CombineItem {
  int b, i, h;         // batch, query row of the sequence, query head
  int64_t tok;         // token row of q/out
  int nch;             // chunks of the unit
  int64_t kstride;     // floats between the unit's consecutive chunk partials
  const float* base;   // the column's partial in the unit's first chunk
};

// Columns of a unit the combine visits: at most S_max * G of its GH are ever
// used (one query row with fewer than 8 heads per KV head fills half of an
// 8-column unit), so the items skip the rest and no combine block idles.
__host__ __device__ __forceinline__ int combine_cols(const DecodeArgs& a) {
  return a.GH < a.S_max * a.G ? a.GH : a.S_max * a.G;
}

// Item pr of the combine: (split batch m, active unit index act of it, column
// col of the unit), pr = (m * UPB + act) * GC + col with GC = combine_cols;
// false for indices past the batch's active units or the unit's columns.
__device__ __forceinline__ bool combine_item(const DecodeArgs& a, int64_t pr, int D,
                                             CombineItem* it) {
  const int64_t UPB = (int64_t)a.KVN * a.HG;
  const int64_t* Q = a.sched + kSchedHeader;
  const int64_t* SB = Q + 3 * ((int64_t)a.B + 1);
  const int GC = combine_cols(a);
  const int col = (int)(pr % GC);
  const int64_t ma = pr / GC;
  const int act = (int)(ma % UPB);
  const int64_t b64 = SB[ma / UPB];
  // an entry outside the batches or the partial slots (a plan of other
  // lengths) is skipped: the decode kernel has reported the plan
  if (b64 < 0 || b64 >= a.B) {
    atomicExch(a.err, 2);
    return false;
  }
  const int b = (int)b64;
  int64_t qrow, ql, kv_len;
  batch_lengths(a, b, &qrow, &ql, &kv_len);
  const int qlen = clamp_rows(a, ql);
  const int ha = active_groups(a, qlen);
  const int A = a.KVN * ha;
  if (act >= A) return false;  // past the batch's active units
  const int hk = act / ha, hg = act % ha;
  const int c = hg * a.GH + col;
  if (c >= qlen * a.G || col >= GC) return false;  // past the unit's columns
  if (Q[b] < 0 || Q[b + 1] < Q[b] + A || Q[b + 1] > a.max_chunks || (Q[b + 1] - Q[b]) % A) {
    atomicExch(a.err, 2);
    return false;
  }
  it->b = b;
  it->i = c / a.G;
  it->h = hk * a.G + (c - it->i * a.G);
  it->tok = qrow + it->i;
  it->nch = (int)((Q[b + 1] - Q[b]) / A);
  it->kstride = (int64_t)A * a.GH * (D + 2);
  it->base = a.partials + (Q[b] + act) * (int64_t)a.GH * (D + 2) + col * (D + 2);
  return true;
}

// Few chunks per unit: one thread per (item, d-pair), chunks folded in order.
template <int D>
__global__ void __launch_bounds__(256, 4) decode_combine_flat(const DecodeArgs a) {
  if (a.sched[5] != kDecodePlanMark || a.sched[6] != a.B || a.sched[7] != a.num_ctas ||
      a.sched[4] < 0 || a.sched[4] > a.B || *a.prefill_mark == kPrefillPlanMark)
    return;  // no plan of these arguments: the decode kernel has reported it
  constexpr int TPP = D / 2, PPB = 256 / TPP;
  // The schedule was complete before the decode kernel started its work, so
  // the first item is located while the decode kernel still runs; only the
  // partials need its completion.
  const int64_t items = a.sched[4] * a.KVN * a.HG * combine_cols(a);
  const int d = 2 * (threadIdx.x % TPP);
  int64_t pr = (int64_t)blockIdx.x * PPB + threadIdx.x / TPP;
  CombineItem it;
  bool have = pr < items && combine_item(a, pr, D, &it);
  pdl_wait();  // every partial of the decode kernel is written
  while (pr < items) {
    if (have) {
      float M = -INFINITY, L = 0.f, o0 = 0.f, o1 = 0.f;
      fold_chunks<D>(it.base, it.kstride, d, 0, 1, it.nch, M, L, o0, o1);
      combine_store(a, it.b, it.tok, it.i, it.h, D, d, M, L, o0, o1);
    }
    pr += (int64_t)gridDim.x * PPB;
    have = pr < items && combine_item(a, pr, D, &it);
  }
}

// Many chunks per unit: one CTA per item; NGRP thread groups fold every
// NGRP-th chunk, then group 0 folds the groups in order.
template <int D>
__global__ void __launch_bounds__(256, 4) decode_combine_grouped(const DecodeArgs a) {
  if (a.sched[5] != kDecodePlanMark || a.sched[6] != a.B || a.sched[7] != a.num_ctas ||
      a.sched[4] < 0 || a.sched[4] > a.B || *a.prefill_mark == kPrefillPlanMark)
    return;  // no plan of these arguments: the decode kernel has reported it
  constexpr int TPP = D / 2, NGRP = 256 / TPP;
  __shared__ float4 st[NGRP][TPP];
  const int64_t items = a.sched[4] * a.KVN * a.HG * combine_cols(a);
  const int grp = threadIdx.x / TPP, t = threadIdx.x % TPP, d = 2 * t;
  int64_t pr = blockIdx.x;
  CombineItem it;
  bool have = pr < items && combine_item(a, pr, D, &it);  // the schedule is complete
  pdl_wait();  // every partial of the decode kernel is written
  for (; pr < items; pr += gridDim.x, have = pr < items && combine_item(a, pr, D, &it)) {
    if (!have) continue;  // uniform over the CTA
    float M = -INFINITY, L = 0.f, o0 = 0.f, o1 = 0.f;
    fold_chunks<D>(it.base, it.kstride, d, grp, NGRP, it.nch, M, L, o0, o1);
    st[grp][t] = make_float4(M, L, o0, o1);
    __syncthreads();
    if (grp == 0) {
      for (int g2 = 1; g2 < NGRP; ++g2) {
        const float4 x = st[g2][t];
        if (x.x == -INFINITY) continue;
        const float Mn = fmaxf(M, x.x);
        const float fo = M == -INFINITY ? 0.f : exp2f(M - Mn);
        const float fn = exp2f(x.x - Mn);
        L = L * fo + x.y * fn;
        o0 = o0 * fo + x.z * fn;
        o1 = o1 * fo + x.w * fn;
        M = Mn;
      }
      combine_store(a, it.b, it.tok, it.i, it.h, D, d, M, L, o0, o1);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
size_t decode_smem_bytes(int D, int fp8) {
  if (fp8) return DecodeCfg<128, true>::kSmem;
  return D == 64 ? DecodeCfg<64, false>::kSmem : DecodeCfg<128, false>::kSmem;
}

cudaError_t launch_decode_schedule(const DecodeArgs& a, cudaStream_t s) {
  decode_schedule_kernel<<<1, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, bool FP8, int NG, bool MR>
static cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap& tk,
                                   const CUtensorMap& tv, cudaStream_t s) {
  using Cfg = DecodeCfg<D, FP8>;
  auto kern = decode_kernel<D, FP8, NG, MR>;
  // the shared-memory opt-in is per device and function: set it once for each
  static std::atomic<uint64_t> done_mask[4];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done_mask[(dev >> 6) & 3].load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    done_mask[(dev >> 6) & 3].fetch_or(bit);
  }
  return launch_pdl(kern, dim3(a.num_ctas), dim3(kThreads), Cfg::kSmem, s, a, tk, tv);
}

template <int D, bool FP8, int NG>
static cudaError_t launch_decode_mr(const DecodeArgs& a, const CUtensorMap& tk,
                                    const CUtensorMap& tv, cudaStream_t s) {
  const bool mr = a.S_max > 1 || a.mask != nullptr;
  return mr ? launch_decode_t<D, FP8, NG, true>(a, tk, tv, s)
            : launch_decode_t<D, FP8, NG, false>(a, tk, tv, s);
}

static cudaError_t launch_decode_main(const DecodeArgs& a, const CUtensorMap& tk,
                                      const CUtensorMap& tv, int fp8, cudaStream_t s) {
  const bool two = a.GH > 8;
  if (fp8) return two ? launch_decode_mr<128, true, 2>(a, tk, tv, s)
                      : launch_decode_mr<128, true, 1>(a, tk, tv, s);
  if (a.D == 64) return two ? launch_decode_mr<64, false, 2>(a, tk, tv, s)
                            : launch_decode_mr<64, false, 1>(a, tk, tv, s);
  return two ? launch_decode_mr<128, false, 2>(a, tk, tv, s)
             : launch_decode_mr<128, false, 1>(a, tk, tv, s);
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                          int fp8, cudaStream_t s) {
  cudaError_t e = launch_decode_main(a, tk, tv, fp8, s);
  if (e != cudaSuccess) return e;
  // The plan bounds the chunks by n*W + 6*U, so a unit has about n*W/U + 6;
  // with more than 16 an item gets a whole CTA.  The choice depends on shapes
  // only, so results stay deterministic.
  const int64_t items = a.num_units * combine_cols(a);  // bound: every batch split
  const int64_t est = (int64_t)a.num_ctas * a.chunks_per_cta / a.num_units + 2 * a.small_div;
  if (est > 16) {
    const int grid = (int)std::min<int64_t>(items, (int64_t)a.num_ctas * 8);
    if (a.D == 64) return launch_pdl(decode_combine_grouped<64>, dim3(grid), dim3(256), 0, s, a);
    return launch_pdl(decode_combine_grouped<128>, dim3(grid), dim3(256), 0, s, a);
  }
  const int ppb = 256 / (a.D / 2);
  const int grid = (int)std::min<int64_t>((items + ppb - 1) / ppb, (int64_t)a.num_ctas * 8);
  if (a.D == 64) return launch_pdl(decode_combine_flat<64>, dim3(grid), dim3(256), 0, s, a);
  return launch_pdl(decode_combine_flat<128>, dim3(grid), dim3(256), 0, s, a);
}

}  // namespace fia
