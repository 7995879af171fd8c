// sparse.cu -- shared-KV sparse attention ("kv_quant_sparse_attn_sharedkv":
// O = softmax(Q K~^T * softmax_scale) V~ with K~ = V~; "sparse_flash_mla":
// SWA, CSA and HCA modes and the metadata pre-step), with bf16 K~ rows or the
// packed FP8 rows of the kv_quant page (bf16 rope 64, E4M3 nope 448, E8M0
// tile scales; widened to bf16 in shared memory, exactly: an E4M3 value times
// a power of two is a bf16 value).
//
// K~ of a query row is the band window of the original KV followed by the
// compressed rows (the listed top-k indices for CSA, scanned up to the first
// -1 and kept when causally visible; every visible compressed row for HCA).
// A work item is (query row, group of 8 query heads); the metadata kernel
// hands each CTA a contiguous run of items of balanced weight.  In a CTA eight
// producer warps gather K~ in 64-row chunks (index -> block table -> pool
// row, one bulk copy per row) into a ring of shared-memory stages, and eight
// consumer warps run the whole item: S^T = K~ Q^T and O^T += V~^T P^T with
// mma.sync (the K~ rows are the M dimension, the 8 heads N), the online
// softmax across chunks in the exp2 domain, and the sink and normalisation at
// the end.  A row's chunks all run in one CTA, in order, so nothing is
// combined through global memory and the result does not depend on the rest
// of the batch.
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace fia {

namespace {

constexpr int kChunk = 64;                // K~ rows per stage
constexpr int kHeads = 8;                 // query heads per work item (mma N)
constexpr int kSCons = 8;                 // consumer warps
constexpr int kSProd = 8;                 // producer warps (warp w gathers the rows r of a chunk with r mod kSProd = w)
constexpr int kSThreads = 32 * (kSProd + kSCons);
// four warpgroups: the producers' two give registers to the consumers' two
// (setmaxnreg), 256 * kSProdRegs + 256 * kSConsRegs = 512 * 128, the launch's
constexpr int kSProdRegs = 72;
constexpr int kSConsRegs = 184;
static_assert(32 * kSProd * kSProdRegs + 32 * kSCons * kSConsRegs <= kSThreads * 128,
              "register split");
constexpr int kMdBase = 16;               // metadata: CTA begins from this entry
constexpr int32_t kMdMagic = 0x46534D32;
constexpr int kMaxK2 = 2048;              // longest index list (validated on the host)
constexpr int kPackedRow = 640;           // bytes of a packed FP8 row (D = 512)
constexpr float kSparseRescale = 8.0f;    // the reference moves past this (log2 units)

struct SparseRow {
  int b;
  int64_t i, q_len, S2, p;
  int64_t vis;  // visible compressed rows, floor((p + 1) / cmp_ratio)
  int cost;     // balancing weight: window chunks + capped compressed chunks
};

__device__ __forceinline__ SparseRow sparse_row(const SparseArgs& a, int64_t u) {
  SparseRow r;
  if (a.layout == 1) {
    int lo = 0, hi = a.B;  // largest b with cu[b] <= u
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.cu_seqlens_q[mid] <= u) lo = mid; else hi = mid;
    }
    r.b = lo;
    r.i = u - a.cu_seqlens_q[lo];
    r.q_len = (int64_t)a.cu_seqlens_q[lo + 1] - a.cu_seqlens_q[lo];
  } else {
    r.b = (int)(u / a.S1);
    r.i = u % a.S1;
    r.q_len = a.S1;
  }
  r.S2 = a.seqused_kv[r.b];
  r.p = r.S2 - r.q_len + r.i;
  r.vis = (r.p + 1) >= 0 ? (r.p + 1) / a.cmp_ratio : 0;
  int64_t kc = 0;
  if (a.mode == 1) kc = min(r.vis, (int64_t)a.K2);
  else if (a.mode == 2) kc = r.vis;
  const int64_t W = (int64_t)a.win_left + a.win_right + 1;
  r.cost = (int)((W + kChunk - 1) / kChunk + (kc + kChunk - 1) / kChunk);
  return r;
}

// j / d for 0 <= j < 2^31 with the host's multiplier and shift
__device__ __forceinline__ int64_t fast_div(int64_t j, uint32_t magic, int shift) {
  return (int64_t)(((uint64_t)(uint32_t)j * magic) >> shift);
}

// 2^(e - 127) of an E8M0 scale byte (255 is NaN)
__device__ __forceinline__ float e8m0_value(uint32_t e) {
  if (e == 0xffu) return __int_as_float(0x7fc00000);
  if (e == 0u) return __int_as_float(0x00400000);  // 2^-127, subnormal
  return __int_as_float((int)(e << 23));
}

}  // namespace

// ---------------------------------------------------------------------------
// metadata: item weights -> the first item of every CTA
// ---------------------------------------------------------------------------
// Items k = u * G + g (query row u, head group g, G groups per row) weigh
// cost(u); with P_k the weight before item k and T the total, CTA c begins at
// #{k : P_k < floor(c T / n)}.  Row u's items start at A = G * pre(u) and
// item g of the row at A + g * cost(u), so a threshold t in (A, A + G cost]
// gives the begin u * G + ceil((t - A) / cost).
// Prefetches the 128-byte lines of [p, p + bytes) into L2, at most `cap`
// per thread of the block (a hint: nothing is read).
__device__ __forceinline__ void prefetch_lines(const void* p, int64_t bytes, int cap) {
  if (p == nullptr || bytes <= 0) return;
  const char* c = static_cast<const char*>(p);
  const int64_t lines = (bytes + 127) >> 7;  // (lines - 1) * 128 < bytes
  int64_t k = threadIdx.x;
  for (int i = 0; i < cap && k < lines; ++i, k += blockDim.x)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c + (k << 7)));
}

__global__ void __launch_bounds__(1024) sparse_metadata_kernel(const SparseArgs a, int32_t* md) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nthr = blockDim.x;
  const int64_t n = a.num_ctas, G = a.hgs;
  pdl_trigger();  // the attention kernel may set up while the metadata is built
  // The attention kernel's first dependent loads after its wait are the
  // block tables and the index lists: this block pulls them into L2 while it
  // works (at most 512 KB of each).
  prefetch_lines(a.ori_block_table, (int64_t)a.B * a.ori_max_blocks * 4, 4);
  if (a.mode != 0)
    prefetch_lines(a.cmp_block_table, (int64_t)a.B * a.cmp_max_blocks * 4, 4);
  if (a.mode == 1) prefetch_lines(a.cmp_sparse_indices, a.rows * a.K2 * 4, 4);
  for (int k = tid; k < 1024; k += nthr) md[k] = 0;
  // pass 1: total weight
  if (tid == 0) carry = 0;
  __syncthreads();
  int64_t part = 0;
  for (int64_t u = tid; u < a.rows; u += nthr) part += sparse_row(a, u).cost;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) atomicAdd(reinterpret_cast<unsigned long long*>(&carry), (unsigned long long)part);
  __syncthreads();
  const int64_t T = carry * G;
  __syncthreads();
  // pass 2: running row prefix; each row writes the begins whose threshold
  // falls on its items
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < a.rows; base += nthr) {
    const int64_t u = base + tid;
    const int64_t cost = u < a.rows ? sparse_row(a, u).cost : 0;
    int64_t x = cost;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int64_t w = lane < (nthr >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int64_t pre = carry + (wid ? warp_sums[wid - 1] : 0) + x - cost;
    if (u < a.rows && T > 0) {
      const int64_t A = pre * G, E = A + G * cost;
      // thresholds floor(c T / n) in (A, E]: c from ceil((A + 1) n / T)
      for (int64_t c = ((A + 1) * n + T - 1) / T; c <= n; ++c) {
        const int64_t t = c * T / n;
        if (t > E) break;
        md[kMdBase + c] = (int32_t)(u * G + (t - A + cost - 1) / cost);
      }
    }
    __syncthreads();
    if (tid == nthr - 1) carry = pre + cost;
    __syncthreads();
  }
  if (tid == 0) {
    md[0] = kMdMagic;
    md[1] = (int32_t)n;
    md[2] = (int32_t)a.rows;
    md[3] = kChunk;
    md[4] = (int32_t)T;
    md[5] = a.B;
    md[6] = a.N1;
    md[7] = a.K2;
    md[8] = a.cmp_ratio;
    md[9] = a.win_left;
    md[10] = a.win_right;
    md[11] = a.mode;
    md[12] = kHeads;
    md[13] = (int32_t)(a.rows * G);
    md[14] = a.kv_dtype;
  }
}

// ---------------------------------------------------------------------------
// attention: one (query row, 8 heads) item at a time, K~ streamed in chunks
// ---------------------------------------------------------------------------
template <int D>
struct SparseCfg {
  static constexpr int kRowBytes = D * 2 + 16;  // padded rows: ldmatrix without bank conflicts
  static constexpr int kStageBytes = kChunk * kRowBytes;
  static constexpr int kStages = D == 512 ? 3 : (D == 256 ? 6 : 8);
  static constexpr int kPtStride = kChunk + 8;  // bf16 per head row of P^T (padded)
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffSx = kOffQ + kHeads * kRowBytes;        // [8 warps][4][32] fp32
  static constexpr int kOffMx = kOffSx + kSCons * 4 * 32 * 4;      // [4 row groups][8 heads]
  static constexpr int kOffL = kOffMx + 4 * kHeads * 4;            // [4 row groups][8 heads]
  static constexpr int kOffPt = kOffL + 4 * kHeads * 4;            // [8 heads][kPtStride] bf16
  static constexpr int kOffList = kOffPt + kHeads * kPtStride * 2; // [K2] int32 CSA rows
  static constexpr int kOffHdr = kOffList + kMaxK2 * 4;            // per stage: valid rows, last
  static constexpr int kOffBar = kOffHdr + kStages * 16;
  static constexpr int kOffMisc = kOffBar + 8 * (2 * kStages + 2);
  static constexpr int kSmem = kOffMisc + 16;  // misc: abort flag, -, CSA list length
  static_assert(kStageBytes % 16 == 0 && kOffQ % 16 == 0, "bulk-copy alignment");
  static_assert(D != 512 || kRowBytes >= kPackedRow, "a packed row fits its slot");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(kSmem <= 232448, "shared memory");
};

struct StageHdr {
  uint64_t valid;  // bit r: row r holds a K~ row
  int32_t last;    // the item's last chunk
  int32_t pad;
};

template <int D>
__global__ void __launch_bounds__(kSThreads, 1)
    sparse_attn_kernel(const SparseArgs a, const int32_t* md) {
  using Cfg = SparseCfg<D>;
  constexpr int S = Cfg::kStages;
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Cfg::kOffBar);
  uint64_t* empty = full + S;
  uint64_t* qfull = empty + S;
  uint64_t* qempty = qfull + 1;
  StageHdr* hdr = reinterpret_cast<StageHdr*>(sm + Cfg::kOffHdr);
  int* misc = reinterpret_cast<int*>(sm + Cfg::kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const bool packed = a.kv_dtype == 1;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSCons);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, kSCons);
    misc[0] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // launched behind the metadata kernel with programmatic serialization: the
  // set-up above overlaps it, everything below reads its result (and the
  // inputs of earlier work on the stream).  `md` is a plain pointer: marked
  // __restrict__ its loads could be hoisted above this wait.
  pdl_wait();
  if (md[0] != kMdMagic || md[1] != a.num_ctas || md[2] != (int32_t)a.rows || md[5] != a.B ||
      md[6] != a.N1 || md[7] != a.K2 || md[12] != kHeads || md[13] != (int32_t)(a.rows * a.hgs) ||
      md[14] != a.kv_dtype) {
    if (tid == 0) atomicExch(a.err, 2);
    return;
  }
  // the status word of this call: cleared here (a time-out, the only other
  // error, is reported seconds later), set to 2 above on a metadata mismatch;
  // with FIA_DEBUG the host clears it before the launch instead, since a
  // page reported by another CTA may come before this CTA's clear
  if (c == 0 && tid == 0 && !a.debug) *reinterpret_cast<volatile int*>(a.err) = 0;
  const int64_t k_begin = md[kMdBase + c], k_end = md[kMdBase + c + 1];
  if (k_begin >= k_end) return;
  const int row_src_bytes = packed ? kPackedRow : D * 2;

  if (warp < kSProd) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSProdRegs) : "memory");
    // ======================= producers =======================
    // Every producer warp walks the same items and chunks; warp pw issues
    // the copies of the rows r = pw mod kSProd of each chunk (the copies of one
    // warp are issued one after another, so more warps keep more rows in
    // flight), warp 0 also the query rows, the CSA compaction and the
    // stage header.
    const int pw = warp;
    int32_t* list = reinterpret_cast<int32_t*>(sm + Cfg::kOffList);
    int it = 0, qn = 0;
    bool aborted = false;
    // Gathers chunk positions [base, base + 64) of one part of the row's K~:
    // the window (rows lo + pos of the original cache) or the compressed
    // rows (list entries for CSA, rows 0.. for HCA); cnt = the part's length.
    auto issue_chunk = [&](const SparseRow& r, bool cmp, int64_t lo, int base, int cnt,
                           bool last) {
      const int s = it % S;
      wait_or_abort(&empty[s], ((it / S) & 1) ^ 1, a.err, misc);
      if (*reinterpret_cast<volatile int*>(misc)) {
        aborted = true;
        return;
      }
      uint8_t* st = sm + s * Cfg::kStageBytes;
      int64_t off[2];
      bool ok[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int pos = base + lane + 32 * h2;
        ok[h2] = pos < cnt;
        off[h2] = 0;
        if (ok[h2]) {
          // a row whose page lies outside the block table or the pool (a
          // length or table entry that breaks the caller's contract) is
          // left out instead of read
          if (!cmp) {
            const int64_t j = lo + pos;
            const int64_t pg = fast_div(j, a.ori_magic, a.ori_shift);
            const int64_t blk = pg < a.ori_max_blocks
                                    ? a.ori_block_table[(int64_t)r.b * a.ori_max_blocks + pg] : -1;
            ok[h2] = blk >= 0 && blk < a.ori_num_blocks;
            off[h2] = (blk * a.ori_block_size + (j - pg * a.ori_block_size)) * row_src_bytes;
          } else {
            const int64_t cr = a.mode == 1 ? (int64_t)list[pos] : (int64_t)pos;
            const int64_t pg = fast_div(cr, a.cmp_magic, a.cmp_shift);
            const int64_t blk = pg < a.cmp_max_blocks
                                    ? a.cmp_block_table[(int64_t)r.b * a.cmp_max_blocks + pg] : -1;
            ok[h2] = blk >= 0 && blk < a.cmp_num_blocks;
            off[h2] = (blk * a.cmp_block_size + (cr - pg * a.cmp_block_size)) * row_src_bytes;
          }
          if (a.debug && !ok[h2] && pw == 0) atomicExch(a.err, 3);
        }
      }
      const uint64_t valid = (uint64_t)__ballot_sync(0xffffffffu, ok[0]) |
                             ((uint64_t)__ballot_sync(0xffffffffu, ok[1]) << 32);
      // rows without a K~ row are zeroed: their P is 0, and a zero row keeps
      // P V exact whatever an earlier chunk left there
      // (warp 0 alone, so that its arrival orders the zeros for the consumers)
      for (uint64_t inval = pw == 0 ? ~valid : 0ull; inval; inval &= inval - 1) {
        const int rr = __ffsll((long long)inval) - 1;
        for (int x = lane; x < D / 8; x += 32)
          *reinterpret_cast<uint4*>(st + rr * Cfg::kRowBytes + x * 16) = make_uint4(0, 0, 0, 0);
      }
      if (pw == 0 && lane == 0) {
        hdr[s].valid = valid;
        hdr[s].last = last ? 1 : 0;
      }
      // the zero rows (generic proxy) precede later bulk copies into them
      fence_proxy_async_smem();
      __syncwarp();
      uint64_t* txb = &full[s];
      if (pw == 0 && lane == 0)
        mbar_arrive_expect_tx(txb, (uint32_t)(__popcll(valid) * row_src_bytes));
      __syncwarp();
      const uint8_t* src =
          reinterpret_cast<const uint8_t*>(cmp ? a.cmp_kv : a.ori_kv);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2)
        if (ok[h2] && (lane + 32 * h2) % kSProd == pw)
          bulk_load(st + (lane + 32 * h2) * Cfg::kRowBytes, src + off[h2], row_src_bytes, txb);
      ++it;
    };

    // (for CSA every producer warp reaches the item's barriers, aborted or not)
    for (int64_t k = k_begin; k < k_end && (a.mode == 1 || !aborted); ++k, ++qn) {
      const int64_t u = k / a.hgs;
      const int head0 = (int)(k - u * a.hgs) * kHeads;
      const int nh = min(kHeads, a.N1 - head0);
      const SparseRow r = sparse_row(a, u);
      // ---- the item's query rows (once the consumers hold the last item's) ----
      if (pw == 0) {
        wait_or_abort(qempty, (qn & 1) ^ 1, a.err, misc);
        if (*reinterpret_cast<volatile int*>(misc)) aborted = true;
        uint8_t* qs = sm + Cfg::kOffQ;
        for (int h = nh; h < kHeads; ++h)  // heads past N1 read as zeros
          for (int x = lane; x < D / 8; x += 32)
            *reinterpret_cast<uint4*>(qs + h * Cfg::kRowBytes + x * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
        if (!aborted) {
          if (lane == 0) mbar_arrive_expect_tx(qfull, (uint32_t)(nh * D * 2));
          __syncwarp();
          if (lane < nh)
            bulk_load(qs + lane * Cfg::kRowBytes, a.q + (u * a.N1 + head0 + lane) * (int64_t)D,
                      D * 2, qfull);
        }
      }
      // ---- window rows [lo, hi] of the original cache ----
      const int64_t lo = max((int64_t)0, r.p - a.win_left);
      const int64_t hi = min(r.S2 - 1, r.p + a.win_right);
      const int nw = (int)max((int64_t)0, hi - lo + 1);
      const int nwch = (nw + kChunk - 1) / kChunk;
      // the last window chunk ends the item when no compressed rows follow
      // (known up front except for CSA, whose list is compacted below)
      const bool win_ends = a.mode == 0 || (a.mode == 2 && r.vis == 0);
      bool ended = false;
      for (int ch = 0; ch < nwch && !aborted; ++ch) {
        const bool last = win_ends && ch == nwch - 1;
        issue_chunk(r, false, lo, ch * kChunk, nw, last);
        ended |= last;
      }
      // (for CSA the producer warps stop together at the barriers below)
      if (aborted && a.mode != 1) break;
      // ---- compressed rows ----
      int nk = 0;
      if (a.mode == 1) {
        // every producer warp is done with the previous item's list (and
        // all stop together after a time-out)
        if (named_bar_or(3, 32 * kSProd, aborted)) break;
      }
      if (a.mode == 1 && pw == 0) {
        // CSA: the list up to the first negative entry, visible entries kept
        // in order (warp compaction into shared memory)
        const int32_t* ix = a.cmp_sparse_indices + u * (int64_t)a.K2;
        bool stop = false;
        // 16 entries per lane per round: a list of up to 512 in one round trip
        for (int t0 = 0; t0 < a.K2 && !stop; t0 += 32 * 16) {
          int v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = t0 + 32 * j + lane;
            v[j] = t < a.K2 ? __ldg(ix + t) : -1;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (!stop) {
              const uint32_t neg = __ballot_sync(0xffffffffu, v[j] < 0);
              const int first = neg ? __ffs(neg) - 1 : 32;
              const bool keep = lane < first && (int64_t)v[j] < r.vis;
              const uint32_t km = __ballot_sync(0xffffffffu, keep);
              if (keep) list[nk + __popc(km & ((1u << lane) - 1u))] = v[j];
              nk += __popc(km);
              stop = neg != 0;
            }
          }
        }
        if (lane == 0) misc[2] = nk;
      }
      if (a.mode == 1) {
        // the list and its length are ready for every producer warp
        if (named_bar_or(3, 32 * kSProd, aborted)) break;
        nk = *reinterpret_cast<volatile int*>(misc + 2);
      } else if (a.mode == 2) {
        nk = (int)r.vis;
      }
      const int nkch = (nk + kChunk - 1) / kChunk;
      for (int ch = 0; ch < nkch && !aborted; ++ch) {
        const bool last = ch == nkch - 1;
        issue_chunk(r, true, 0, ch * kChunk, nk, last);
        ended |= last;
      }
      if (!ended && !aborted) issue_chunk(r, true, 0, 0, 0, true);  // nothing visible: one empty chunk
    }
    return;
  }

  // ======================= consumers =======================
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSConsRegs) : "memory");
  // Warp cw: QK rows 16 rg .. 16 rg + 15 of each chunk over half hf of D
  // (the two halves' partial scores are summed through shared memory), and
  // P V for output columns cw * D/8 .. + D/8 over all 64 rows.
  constexpr int KS = D / 32;             // k-steps over half of D
  constexpr int DW = D / kSCons;         // output columns of a warp
  constexpr int MTW = DW / 16;           // their m-tiles
  constexpr int nthr = 32 * kSCons;
  const int cw = warp - kSProd, rg = cw & 3, hf = cw >> 2;
  const int g = lane >> 2, q4 = lane & 3;
  float* sx = reinterpret_cast<float*>(sm + Cfg::kOffSx);
  float* mxs = reinterpret_cast<float*>(sm + Cfg::kOffMx);
  float* lsum = reinterpret_cast<float*>(sm + Cfg::kOffL);
  uint16_t* pt = reinterpret_cast<uint16_t*>(sm + Cfg::kOffPt);
  const uint32_t sm_base = smem_u32(sm);
  const int r0 = 16 * rg + g, r1 = r0 + 8;  // chunk rows of fragment rows g, g+8
  int it = 0, qn = 0;
  for (int64_t k = k_begin; k < k_end; ++k, ++qn) {
    const int64_t u = k / a.hgs;
    const int head0 = (int)(k - u * a.hgs) * kHeads;
    const int nh = min(kHeads, a.N1 - head0);
    // ---- Q^T fragments of this warp's half of D (mma B: k = d, n = head) ----
    wait_or_abort(qfull, qn & 1, a.err, misc);
    uint32_t qb[KS][2];
    {
      const uint16_t* qsm = reinterpret_cast<const uint16_t*>(sm + Cfg::kOffQ);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const int d0 = hf * (D / 2) + kk * 16 + 2 * q4;
        qb[kk][0] = *reinterpret_cast<const uint32_t*>(qsm + g * (Cfg::kRowBytes / 2) + d0);
        qb[kk][1] = *reinterpret_cast<const uint32_t*>(qsm + g * (Cfg::kRowBytes / 2) + d0 + 8);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(qempty);

    float acc[MTW][4];
#pragma unroll
    for (int i = 0; i < MTW; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    // reference of heads 2q, 2q+1 (exp2 domain): no score seen lies more
    // than 2^8 above it (-inf until a head's first visible row)
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};              // this lane's share of the sums (row-group warps)
    bool stop = false;
    while (true) {
      const int s = it % S;
      wait_or_abort(&full[s], (it / S) & 1, a.err, misc);
      const uint64_t valid = hdr[s].valid;
      const bool last = hdr[s].last != 0;
      const uint32_t st = sm_base + s * Cfg::kStageBytes;
      // packed FP8 rows -> bf16 rows in place, this warp's 8 rows in two
      // batches of 4: the rope values are bf16 already; lane l < 28 widens
      // nope codes 16 l .. 16 l + 15 (tile l / 4).  A batch's reads precede
      // its writes (__syncwarp), and the named barrier orders every warp's
      // rows before any warp's reads.
      if constexpr (D == 512) {
        if (packed) {
#pragma unroll
          for (int bt = 0; bt < 2; ++bt) {
            uint4 c16[4];
            uint32_t ex[4];
            bool vr[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int rr = cw * 8 + bt * 4 + j;
              vr[j] = ((valid >> rr) & 1) && lane < 28;
              c16[j] = make_uint4(0, 0, 0, 0);
              ex[j] = 127;
              if (vr[j]) {
                const uint8_t* row = sm + s * Cfg::kStageBytes + rr * Cfg::kRowBytes;
                c16[j] = *reinterpret_cast<const uint4*>(row + 128 + 16 * lane);
                ex[j] = row[128 + 448 + (lane >> 2)];
              }
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (vr[j]) {
                const float f = e8m0_value(ex[j]);
                const uint32_t w4[4] = {c16[j].x, c16[j].y, c16[j].z, c16[j].w};
                uint32_t o[8];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  uint32_t lo2, hi2;
                  e4m3x4_to_f16x2x2(w4[w], lo2, hi2);
                  const float2 fl = __half22float2(*reinterpret_cast<const __half2*>(&lo2));
                  const float2 fh = __half22float2(*reinterpret_cast<const __half2*>(&hi2));
                  o[2 * w] = pack_bf16(fl.x * f, fl.y * f);
                  o[2 * w + 1] = pack_bf16(fh.x * f, fh.y * f);
                }
                uint4* dst = reinterpret_cast<uint4*>(sm + s * Cfg::kStageBytes +
                                                      (cw * 8 + bt * 4 + j) * Cfg::kRowBytes +
                                                      128 + 32 * lane);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
              }
            }
            __syncwarp();
          }
          named_bar_sync(1, nthr);
        }
      }
      // ---- partial S^T = K~ Q^T: rows of this row group, half hf of D ----
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        // A: matrices (rows 0-7, d lo8), (rows 8-15, d lo8), (rows 0-7, hi8), (rows 8-15, hi8)
        const int mi = lane >> 3;
        const int row = 16 * rg + (mi & 1) * 8 + (lane & 7);
        const int col = hf * (D / 2) + kk * 16 + (mi >> 1) * 8;
        uint32_t ka[4];
        ldsm_x4(st + row * Cfg::kRowBytes + col * 2, ka[0], ka[1], ka[2], ka[3]);
        mma_bf16(sc, ka, qb[kk][0], qb[kk][1]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sx[(cw * 4 + e) * 32 + lane] = sc[e];
      // the two halves meet; a time-out anywhere stops every consumer warp here
      if (named_bar_or(1, nthr, *reinterpret_cast<volatile int*>(misc) != 0)) {
        stop = true;
        break;
      }
      float x[4];
      {
        const bool v0 = (valid >> r0) & 1, v1 = (valid >> r1) & 1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float o = sx[((cw ^ 4) * 4 + e) * 32 + lane];
          const float sfull = hf ? o + sc[e] : sc[e] + o;  // the same sum in both warps
          x[e] = ((e < 2) ? v0 : v1) ? sfull * a.scale_log2 : -INFINITY;
        }
      }
      // ---- chunk maxima per head over this warp's 16 rows ----
      float lm[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(x[e], x[2 + e]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        lm[e] = mx;
        if (hf == 0 && g == 0) mxs[rg * kHeads + 2 * q4 + e] = mx;
      }
      // ---- P = exp2(x - m) against the shared reference m, which moves
      // only when a chunk's maximum passes it by more than 2^8 (or with a
      // head's first visible rows).  The row-group warps publish P^T against
      // the current m, and the barrier that publishes it also ORs every
      // warp's vote that m must move; only then (rarely, after an item's
      // first chunk) do all warps take the chunk maxima, move m and write P^T
      // again behind one more barrier. ----
      bool must_move = false;
      float pv[2][2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        must_move |= lm[e] > m[e] + kSparseRescale || (m[e] == -INFINITY && lm[e] != -INFINITY);
        const float mu = m[e] == -INFINITY ? 0.f : m[e];
        pv[e][0] = fast_exp2(x[e] - mu);
        pv[e][1] = fast_exp2(x[2 + e] - mu);
      }
      auto put_p = [&]() {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const __nv_bfloat16 b0 = __float2bfloat16_rn(pv[e][0]), b1 = __float2bfloat16_rn(pv[e][1]);
          pt[(2 * q4 + e) * Cfg::kPtStride + r0] = *reinterpret_cast<const uint16_t*>(&b0);
          pt[(2 * q4 + e) * Cfg::kPtStride + r1] = *reinterpret_cast<const uint16_t*>(&b1);
        }
      };
      if (hf == 0) put_p();
      float corr[2] = {1.f, 1.f};
      if (!named_bar_or(1, nthr, must_move)) {
        if (hf == 0) {
#pragma unroll
          for (int e = 0; e < 2; ++e) l[e] += pv[e][0] + pv[e][1];
        }
      } else {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float mc = mxs[2 * q4 + e];
#pragma unroll
          for (int r2 = 1; r2 < 4; ++r2) mc = fmaxf(mc, mxs[r2 * kHeads + 2 * q4 + e]);
          if (mc > m[e] + kSparseRescale || (m[e] == -INFINITY && mc != -INFINITY)) {
            corr[e] = m[e] == -INFINITY ? 0.f : fast_exp2(m[e] - mc);
            m[e] = mc;
          }
          const float mu = m[e] == -INFINITY ? 0.f : m[e];
          pv[e][0] = fast_exp2(x[e] - mu);
          pv[e][1] = fast_exp2(x[2 + e] - mu);
          if (hf == 0) l[e] = l[e] * corr[e] + pv[e][0] + pv[e][1];
        }
        if (hf == 0) put_p();
        named_bar_sync(1, nthr);
      }
      // ---- O^T += V~^T P^T over this warp's columns ----
      if (__any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
        for (int i = 0; i < MTW; ++i) {
          acc[i][0] *= corr[0]; acc[i][1] *= corr[1];
          acc[i][2] *= corr[0]; acc[i][3] *= corr[1];
        }
      }
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk) {
        // B = P^T (k = rows, n = head): rows 2q, 2q+1 and 2q+8, 2q+9 of head g
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(pt + g * Cfg::kPtStride + kk * 16 + 2 * q4);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(pt + g * Cfg::kPtStride + kk * 16 + 2 * q4 + 8);
#pragma unroll
        for (int i = 0; i < MTW; ++i) {
          // A = V^T (m = d, k = rows), transposed by ldmatrix: matrices
          // (rows 0-7, d lo8), (rows 0-7, d hi8), (rows 8-15, d lo8), (rows 8-15, d hi8)
          const int mi = lane >> 3;
          const int row = kk * 16 + (mi >> 1) * 8 + (lane & 7);
          const int col = cw * DW + i * 16 + (mi & 1) * 8;
          uint32_t va[4];
          ldsm_x4_t(st + row * Cfg::kRowBytes + col * 2, va[0], va[1], va[2], va[3]);
          mma_bf16(acc[i], va, b0, b1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      ++it;
      if (last) break;
    }
    if (stop) break;

    // ---- sink, normalisation, O and lse ----
    if (hf == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float t = l[e];
        t += __shfl_xor_sync(0xffffffffu, t, 4);
        t += __shfl_xor_sync(0xffffffffu, t, 8);
        t += __shfl_xor_sync(0xffffffffu, t, 16);
        if (g == 0) lsum[rg * kHeads + 2 * q4 + e] = t;
      }
    }
    named_bar_sync(1, nthr);
    float scl[2], lse[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hl = 2 * q4 + e;
      float L = 0.f;
#pragma unroll
      for (int r2 = 0; r2 < 4; ++r2) L += lsum[r2 * kHeads + hl];
      scl[e] = 0.f;
      lse[e] = INFINITY;
      if (m[e] != -INFINITY) {
        float Mp = m[e];
        if (a.sinks && hl < nh) {
          const float sk = a.sinks[head0 + hl] * 1.4426950408889634f;
          Mp = fmaxf(m[e], sk);
          L = L * exp2f(m[e] - Mp) + exp2f(sk - Mp);
        }
        scl[e] = exp2f(m[e] - Mp) / L;
        lse[e] = (Mp + log2f(L)) * 0.6931471805599453f;
      }
    }
    // acc[i][0..1]: column d = cw*DW + 16i + g, heads 2q, 2q+1; [2..3]: d + 8.
    // Lanes g and g^1 hold neighbouring columns: even g writes head 2q at
    // (d, d+1), odd g head 2q+1 at (d-1, d), as bf16 pairs.
    uint16_t* orow = a.out + (u * a.N1 + head0) * (int64_t)D;
#pragma unroll
    for (int i = 0; i < MTW; ++i)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const float v0 = acc[i][2 * hr] * scl[0], v1 = acc[i][2 * hr + 1] * scl[1];
        const float w0 = __shfl_xor_sync(0xffffffffu, v0, 4);
        const float w1 = __shfl_xor_sync(0xffffffffu, v1, 4);
        const int d = cw * DW + 16 * i + 8 * hr + g;
        if ((g & 1) == 0) {
          if (2 * q4 < nh)
            *reinterpret_cast<uint32_t*>(orow + (2 * q4) * D + d) = pack_bf16(v0, w0);
        } else {
          if (2 * q4 + 1 < nh)
            *reinterpret_cast<uint32_t*>(orow + (2 * q4 + 1) * D + d - 1) = pack_bf16(w1, v1);
        }
      }
    if (a.lse && cw == 0 && g == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (2 * q4 + e < nh) a.lse[u * a.N1 + head0 + 2 * q4 + e] = lse[e];
    }
  }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
cudaError_t launch_sparse_metadata(const SparseArgs& a, int32_t* md, cudaStream_t s) {
  sparse_metadata_kernel<<<1, 1024, 0, s>>>(a, md);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_sparse_t(const SparseArgs& a, const int32_t* md, cudaStream_t s) {
  using Cfg = SparseCfg<D>;
  auto kern = sparse_attn_kernel<D>;
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
  return launch_pdl(kern, dim3(a.num_ctas), dim3(kSThreads), Cfg::kSmem, s, a, md);
}

cudaError_t launch_sparse(const SparseArgs& a, const int32_t* md, cudaStream_t s) {
  if (a.D == 512) return launch_sparse_t<512>(a, md, s);
  if (a.D == 256) return launch_sparse_t<256>(a, md, s);
  return launch_sparse_t<128>(a, md, s);
}

}  // namespace fia
