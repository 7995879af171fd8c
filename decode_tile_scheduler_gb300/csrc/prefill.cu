// prefill.cu -- the full-inference branch of fused inference attention (query
// length > 1; "aclnnFusedInferAttentionScoreV2": the PromptFlashAttention branch)
// over a paged or contiguous KV cache, on the 5th-generation tensor cores.
//
// Work unit: (batch b, 128-row query tile t, KV head hk, head pair).  Two query
// heads of the same GQA group share every K/V tile, so one unit runs two
// 128 x D query tiles ("slots") against one stream of 128-row K/V tiles.
//
// Scheduler (prefill_schedule_kernel): every unit gets cost 1 + (KV tiles its
// query tile can see); units are ordered by non-increasing cost (a counting
// sort) and persistent CTAs claim them one by one with an atomic counter, so
// the longest units start first (longest-processing-time order).  A unit runs
// entirely in one CTA, so results do not depend on which CTA took it.
//
// Kernel roles (12 warps, one CTA per SM, all 512 TMEM columns):
//   warp 0      producer: TMA loads of the Q tiles and of K/V tiles whose rows
//               come from block_table (128-byte swizzled boxes)
//   warps 1, 3  MMA issuers, one thread each, for query slots 0 and 1:
//               S = Q K^T (both operands in shared memory) and O += P V (P in
//               TMEM, V in shared memory), fp32 accumulators in TMEM; the two
//               slots ping-pong, and each thread's commits and waits overlap
//               the other slot's MMAs
//   warp 2      V guard: zeroes V rows past kv_len in a tail tile, so that a
//               zero probability never meets a NaN in unused cache rows
//   warps 4-7   softmax of slot 0; warps 8-11 softmax of slot 1: one TMEM lane
//               (query row) per thread, online softmax in the exp2 domain with
//               a lazily moved maximum (O is rescaled only when the running
//               maximum grows by more than 2^8), P written back to TMEM as bf16,
//               and the epilogue (sink, 1/l, lse, bf16 store).
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace fia {

namespace {

constexpr int kPWarps = 12;
constexpr int kPThreads = 32 * kPWarps;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct PrefillCfg {
  static constexpr int kNsub = D / 64;                    // 128-byte slices per row
  static constexpr int kTileBytes = kNsub * 128 * 128;    // a 128-row tile of Q, K or V
  static constexpr int kKStages = D == 128 ? 2 : 4;
  static constexpr int kVStages = D == 128 ? 3 : 4;
  static constexpr int kOffQ = 0;                         // 2 slots
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  // barriers: mfull[2] mempty[2] qfull qempty kfull[KS] kempty[KS] vfull[VS]
  // vready[VS] vempty[VS] sfull[2] pfull[2] ofull[2] ofree[2] drain[2] tok[2]
  // qconv[2]
  static constexpr int kNumBars = 4 + 2 + 2 * kKStages + 3 * kVStages + 8 + 2 + 2 + 2;
  static constexpr int kOffMsg = kOffBar + 8 * kNumBars;
  static constexpr int kOffMisc = kOffMsg + 2 * 64;
  static constexpr int kSmem = kOffMisc + 64 + 1024;
  static_assert(kSmem <= 232448, "shared memory");
};

struct PMsg {
  int b, t, hk, nslots, h0, h1;
  int q_len, kv_len, tile0, ntiles, done, pad;
  int64_t q_row0;  // token row of the tile's first query row
};
static_assert(sizeof(PMsg) <= 64, "message slot");

// ex2.approx without `volatile`, so the compiler may schedule it freely.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pair arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void pwait(uint64_t* bar, uint32_t parity, int* err, int* abort_flag) {
  if (*reinterpret_cast<volatile int*>(abort_flag)) return;
  if (!mbar_wait(bar, parity, err)) *reinterpret_cast<volatile int*>(abort_flag) = 1;
}

__device__ __forceinline__ void seq_lengths(const PrefillArgs& a, int b, int64_t* q_start,
                                            int64_t* q_len, int64_t* kv_len) {
  if (a.layout == 1) {
    *q_start = a.cu_seqlens_q[b];
    *q_len = (int64_t)a.cu_seqlens_q[b + 1] - *q_start;
  } else {
    *q_start = (int64_t)b * a.S_q;
    *q_len = a.S_q;
  }
  *kv_len = a.seqused_kv ? a.seqused_kv[b] : a.S_kv;
}

// Position of query row i of a sequence: right-down alignment
// (kv_len - q_len + i) for modes 3 and 4, the row itself for the left-up
// causal mode 2 (modes 0 and 1 do not use it).
__device__ __forceinline__ int64_t row_pos(const PrefillArgs& a, int64_t q_len, int64_t kv_len,
                                           int64_t i) {
  return (a.mask_mode == 2 ? 0 : kv_len - q_len) + i;
}

// KV interval [lo, hi] (clipped) seen by query rows i0..i1 of a sequence, as a
// tile range; returns the number of 128-wide KV tiles (0 if none).  An
// explicit mask narrows nothing here: its bytes are read per row.
__device__ __forceinline__ int tile_span(const PrefillArgs& a, int64_t q_len, int64_t kv_len,
                                         int64_t i0, int64_t i1, int* tile0) {
  const int64_t p0 = row_pos(a, q_len, kv_len, i0), p1 = row_pos(a, q_len, kv_len, i1);
  int64_t lo = a.mask_mode == 4 ? p0 - a.pre_tokens : 0;
  int64_t hi = (a.mask_mode == 2 || a.mask_mode == 3)
                   ? p1
                   : (a.mask_mode == 4 ? p1 + a.next_tokens : kv_len - 1);
  lo = max(lo, (int64_t)0);
  hi = min(hi, kv_len - 1);
  *tile0 = 0;
  if (kv_len <= 0 || hi < lo) return 0;
  *tile0 = (int)(lo / kKvTile);
  return (int)(hi / kKvTile - lo / kKvTile + 1);
}

// Tensor-map row of logical KV row j of batch b, KV head hk: token-major
// pools have one row per token (the head is a column offset), head-major
// pools [nb, KVN, bs, D] one per (page, head, token).
__device__ __forceinline__ int64_t kv_phys_row(const PrefillArgs& a, int b, int hk, int64_t j) {
  if (a.block_table) {
    const int64_t blk = a.block_table[(int64_t)b * a.max_blocks + j / a.block_size];
    if (a.debug && (blk < 0 || blk >= a.num_blocks))
      atomicExch(a.err, 3);  // (read as zeros by the TMA box all the same)
    if (a.kv_layout == 1) return (blk * a.KVN + hk) * a.block_size + j % a.block_size;
    return blk * a.block_size + j % a.block_size;
  }
  return (int64_t)b * a.S_kv + j;
}

}  // namespace

// ---------------------------------------------------------------------------
// scheduler: enumerate units, cost them, counting-sort by non-increasing cost
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) prefill_schedule_kernel(const PrefillArgs a) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  pdl_trigger();  // the prefill kernel may set up while the plan is built
  const int nthr = blockDim.x;
  const int H = a.KVN * a.npairs;
  int64_t* seq_prefix = a.seq_prefix;

  auto block_scan = [&](int64_t v, int64_t* excl_out) {  // returns block total via carry
    int64_t x = v;
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
    *excl_out = carry + (wid ? warp_sums[wid - 1] : 0) + x - v;
    __syncthreads();
    if (tid == nthr - 1) carry = *excl_out + v;
    __syncthreads();
  };

  // 1. units per sequence -> prefix
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < a.B; base += nthr) {
    const int b = base + tid;
    int64_t nu = 0;
    if (b < a.B) {
      int64_t qs, ql, kl;
      seq_lengths(a, b, &qs, &ql, &kl);
      nu = (ql + kQTile - 1) / kQTile * H;
    }
    int64_t ex;
    block_scan(nu, &ex);
    if (b < a.B) seq_prefix[b] = ex;
  }
  const int64_t U = carry;
  if (tid == 0) seq_prefix[a.B] = U;
  // 2. histogram of costs
  const int nb = a.max_cost + 2;
  for (int c = tid; c < nb; c += nthr) a.hist[c] = 0;
  __syncthreads();
  auto unit_of = [&](int64_t k, int* b_out, int* t_out, int* hk_out, int* pr_out, int* cost) {
    int lo = 0, hi = a.B;  // largest b with seq_prefix[b] <= k
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seq_prefix[mid] <= k) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int64_t r = k - seq_prefix[b];
    const int t = (int)(r / H);
    const int hh = (int)(r % H);
    *b_out = b;
    *t_out = t;
    *hk_out = hh / a.npairs;
    *pr_out = hh % a.npairs;
    int64_t qs, ql, kl;
    seq_lengths(a, b, &qs, &ql, &kl);
    const int64_t i0 = (int64_t)t * kQTile, i1 = min(i0 + kQTile, ql) - 1;
    int tile0;
    const int n = tile_span(a, ql, kl, i0, i1, &tile0);
    *cost = min(1 + n, a.max_cost + 1);
  };
  for (int64_t k = tid; k < U; k += nthr) {
    int b, t, hk, pr, cost;
    unit_of(k, &b, &t, &hk, &pr, &cost);
    atomicAdd(&a.hist[cost], 1);
  }
  __syncthreads();
  // 3. offsets in non-increasing cost order: off[c] = sum of hist[c'] for c' > c
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < nb; base += nthr) {
    const int c = nb - 1 - (base + tid);  // high costs first
    const int64_t v = c >= 0 ? a.hist[c] : 0;
    int64_t ex;
    block_scan(v, &ex);
    if (c >= 0) a.hist[c] = (int)ex;
  }
  __syncthreads();
  // 4. scatter
  for (int64_t k = tid; k < U; k += nthr) {
    int b, t, hk, pr, cost;
    unit_of(k, &b, &t, &hk, &pr, &cost);
    const int pos = atomicAdd(&a.hist[cost], 1);
    a.unit_list[pos] = make_int2(b, t | (hk << 18) | (pr << 26));
  }
  if (tid == 0) {
    *a.num_units = U;
    a.num_units[2] = kPrefillPlanMark;  // workspace bytes [24, 48): mark, B, CTA count
    a.num_units[3] = a.B;
    a.num_units[4] = a.num_ctas;
    a.claim[0] = 0;
    a.claim[1] = 0;
    *a.err = 0;
  }
}

// ---------------------------------------------------------------------------
// attention kernel
// ---------------------------------------------------------------------------
// NEG: the softmax scale is negative.  F16: fp16 operands (FP8 caches after
// their conversion): Q' = Q * 2^sh per (token, head), K' and V' divided by a
// power of two per (batch, KV head); every row takes the factors back in its
// score scale and its output.
template <int D, bool NEG, bool F16>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using Cfg = PrefillCfg<D>;
  constexpr int KS = Cfg::kKStages, VS = Cfg::kVStages, NSUB = Cfg::kNsub;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* mfull = bars;
  uint64_t* mempty = mfull + 2;
  uint64_t* qfull = mempty + 2;
  uint64_t* qempty = qfull + 1;
  uint64_t* kfull = qempty + 1;
  uint64_t* kempty = kfull + KS;
  uint64_t* vfull = kempty + KS;
  uint64_t* vready = vfull + VS;
  uint64_t* vempty = vready + VS;
  uint64_t* sfull = vempty + VS;
  uint64_t* pfull = sfull + 2;
  uint64_t* ofull = pfull + 2;
  uint64_t* ofree = ofull + 2;
  uint64_t* drain = ofree + 2;  // [2], one per MMA thread
  uint64_t* tok = drain + 2;    // [2], MMA issue turn of each slot
  uint64_t* qconv = tok + 2;    // [2] (F16) a slot's query tile converted to fp16
  PMsg* msg = reinterpret_cast<PMsg*>(smem + Cfg::kOffMsg);
  int* misc = reinterpret_cast<int*>(smem + Cfg::kOffMisc);  // [0] abort, [1] tmem base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&mfull[s], 1);
      mbar_init(&mempty[s], 5);  // two MMA threads, the V guard, two softmax warpgroups
      mbar_init(&sfull[s], 1);
      mbar_init(&pfull[s], 4);  // one arrival per softmax warp
      mbar_init(&ofull[s], 1);
      mbar_init(&ofree[s], 4);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, 2);  // one commit (or arrival) per MMA thread
    for (int s = 0; s < KS; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 2);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vready[s], 1);
      mbar_init(&vempty[s], 2);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(&tok[0], 1);
    mbar_init(&tok[1], 1);
    mbar_init(&qconv[0], 4);  // one arrival per softmax warp of the slot
    mbar_init(&qconv[1], 4);
    misc[0] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(reinterpret_cast<uint32_t*>(&misc[1]), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[1]);
  // launched behind the scheduler with programmatic serialization: the
  // set-up above overlaps it; the plan and the inputs are read from here on
  pdl_wait();
  // a plan of these arguments carries the scheduler's mark, B and CTA count;
  // without one (execute on a workspace never planned) nothing runs and the
  // error word says 2
  const bool plan_ok = a.num_units[2] == kPrefillPlanMark && a.num_units[3] == a.B &&
                       a.num_units[4] == a.num_ctas && *a.num_units >= 0 &&
                       *a.num_units <= a.max_units;
  if (!plan_ok && tid == 0 && blockIdx.x == 0) atomicExch(a.err, 2);
  const int64_t num_units = plan_ok ? *a.num_units : 0;
  // Register split by warpgroup (each role branch below starts with its
  // part): the producer / MMA / guard warpgroup gives registers to the two
  // softmax warpgroups, which keep a whole row of S (128 fp32) in registers.
  // 128 x 72 + 256 x 216 = 384 x 168, the launch's total.

  if (warp == 0) {
    // ============================ producer ============================
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
    }
    int ucnt = 0, kv_it = 0, q_cnt = 0;
    while (true) {
      int idx = 0;
      if (lane == 0) idx = atomicAdd(a.claim, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      const int ms = ucnt & 1;
      pwait(&mempty[ms], ((ucnt >> 1) & 1) ^ 1, a.err, misc);
      ++ucnt;
      if (idx < 0 || idx >= num_units || *reinterpret_cast<volatile int*>(misc)) {
        if (lane == 0) {
          if (plan_ok && idx >= num_units) {
            // this CTA claims no more: the last CTA out re-arms the counter
            // for the next fia_execute with the same plan
            __threadfence();
            if (atomicAdd(a.claim + 1, 1) == a.num_ctas - 1) {
              a.claim[0] = 0;
              a.claim[1] = 0;
            }
          }
          msg[ms].done = 1;
          mbar_arrive(&mfull[ms]);
        }
        break;
      }
      const int2 pk = a.unit_list[idx];
      PMsg m;
      m.b = pk.x;
      m.t = pk.y & 0x3FFFF;
      m.hk = (pk.y >> 18) & 0xFF;
      int pr = (pk.y >> 26) & 0x3F;
      // an entry that names no unit of these arguments (a unit list of other
      // lengths) runs as an empty unit: nothing is loaded or written
      const bool ent_ok = m.b >= 0 && m.b < a.B && m.hk < a.KVN && pr < a.npairs;
      if (!ent_ok) {
        if (lane == 0) atomicExch(a.err, 2);
        m.b = 0;
        m.hk = 0;
        pr = 0;
      }
      m.nslots = a.per_pair;
      m.h0 = m.hk * a.G + pr * a.per_pair;
      m.h1 = m.h0 + 1;
      int64_t qs, ql, kl;
      seq_lengths(a, m.b, &qs, &ql, &kl);
      const int64_t i0 = (int64_t)m.t * kQTile, i1 = min(i0 + kQTile, ql) - 1;
      if (!ent_ok || i0 >= ql) ql = 0;  // no query row of the tile exists
      m.q_len = (int)ql;
      m.kv_len = (int)kl;
      m.ntiles = ql > 0 ? tile_span(a, ql, kl, i0, i1, &m.tile0) : 0;
      if (ql <= 0) m.tile0 = 0;
      m.q_row0 = qs + i0;
      m.done = 0;
      m.pad = 0;
      if (lane == 0) {
        msg[ms] = m;
        mbar_arrive(&mfull[ms]);
      }
      if (m.ntiles == 0) continue;
      // query tiles of the slots
      pwait(qempty, (q_cnt & 1) ^ 1, a.err, misc);
      ++q_cnt;
      if (lane == 0) mbar_arrive_expect_tx(qfull, (uint32_t)(m.nslots * Cfg::kTileBytes));
      __syncwarp();
      if (lane < m.nslots * NSUB) {
        const int s = lane / NSUB, sub = lane % NSUB;
        const int h = s ? m.h1 : m.h0;
        tma_load_2d(smem + Cfg::kOffQ + s * Cfg::kTileBytes + sub * 16384, &tq, qfull,
                    h * D + sub * 64, (int)m.q_row0);
      }
      // K and V tiles
      const int nrb = kKvTile / a.box_rows;
      for (int j = 0; j < m.ntiles; ++j, ++kv_it) {
        const int64_t j0 = (int64_t)(m.tile0 + j) * kKvTile;
        const int rb = lane / NSUB, sub = lane % NSUB;
        const int64_t jb = j0 + (int64_t)rb * a.box_rows;
        const bool mine = lane < nrb * NSUB && jb < kl;
        const int64_t prow = mine ? kv_phys_row(a, m.b, m.hk, jb) : 0;
        const int kcol = (a.kv_layout == 1 ? 0 : m.hk * D) + sub * 64;
        int nvalid = 0;
        for (int q = 0; q < nrb; ++q)
          if (j0 + (int64_t)q * a.box_rows < kl) ++nvalid;
        const uint32_t bytes = (uint32_t)(nvalid * NSUB * a.box_rows * 128);
        const int ks = kv_it % KS, vs = kv_it % VS;
        pwait(&kempty[ks], ((kv_it / KS) & 1) ^ 1, a.err, misc);
        if (lane == 0) mbar_arrive_expect_tx(&kfull[ks], bytes);
        __syncwarp();
        if (mine)
          tma_load_2d(smem + Cfg::kOffK + ks * Cfg::kTileBytes + sub * 16384 + rb * a.box_rows * 128,
                      &tk, &kfull[ks], kcol, (int)prow);
        pwait(&vempty[vs], ((kv_it / VS) & 1) ^ 1, a.err, misc);
        if (lane == 0) mbar_arrive_expect_tx(&vfull[vs], bytes);
        __syncwarp();
        if (mine)
          tma_load_2d(smem + Cfg::kOffV + vs * Cfg::kTileBytes + sub * 16384 + rb * a.box_rows * 128,
                      &tv, &vfull[vs], kcol, (int)prow);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ========================= MMA issuers =========================
    // Warp 1 issues the MMAs of query slot 0, warp 3 those of slot 1 (one
    // thread each).  tcgen05.mma issue blocks at about the rate the tensor
    // core executes, so a single issuing thread leaves the tensor core idle
    // while it commits and waits between batches; with one thread per slot,
    // one slot's bookkeeping overlaps the other slot's MMAs.  K, V and Q
    // buffers are released when both threads have committed (count 2).
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    const int s = warp == 3 ? 1 : 0;
    if (lane == 0) {
      constexpr uint32_t kIdS = F16 ? idesc_f16(128, 128, false) : idesc_bf16(128, 128, false);
      constexpr uint32_t kIdO = F16 ? idesc_f16(128, D, true) : idesc_bf16(128, D, true);
      const uint32_t sq = smem_u32(smem + Cfg::kOffQ);
      const uint32_t sk = smem_u32(smem + Cfg::kOffK);
      const uint32_t sv = smem_u32(smem + Cfg::kOffV);
      int ucnt = 0, kv_it = 0, q_cnt = 0, p_it = 0, u_cnt = 0, qc_cnt = 0;
      // Issue turns: in units with two slots the threads issue their MMA
      // batches strictly alternately (slot 0, slot 1, slot 0, ...), which
      // keeps the two softmax warpgroups half a period apart (ping-pong);
      // a thread hands the turn over right after its last MMA of a batch.
      int turn = 0;  // batches issued in two-slot units
      auto take_turn = [&](bool paired) {
        if (!paired) return;
        if (s == 0) {
          if (turn > 0) pwait(&tok[0], (uint32_t)((turn - 1) & 1), a.err, misc);
        } else {
          pwait(&tok[1], (uint32_t)(turn & 1), a.err, misc);
        }
      };
      auto pass_turn = [&](bool paired) {
        if (!paired) return;
        mbar_arrive(&tok[1 - s]);
        ++turn;
      };
      // descriptors of every operand buffer, built once; a k-step only adds
      // its byte offset (>> 4) to the start-address field
      const uint64_t qd = smem_desc_sw128(sq, 16, 1024) + (uint64_t)s * (Cfg::kTileBytes >> 4);
      const uint64_t kd0 = smem_desc_sw128(sk, 16, 1024);
      // V is the MN-major B operand of P V: 64-column swizzle atoms 16 KB apart
      // (leading byte offset), 8-row groups along K 1 KB apart (stride offset)
      const uint64_t vd0 = smem_desc_sw128(sv, 16384, 1024);
      constexpr uint64_t kTileUnits = Cfg::kTileBytes >> 4;
      const uint32_t tS = tmem + 256 * s, tO = tmem + 256 * s + 128;
      auto issue_qk = [&](int ks) {
        const uint64_t kd = kd0 + (uint64_t)ks * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_ss(tS, qd + off, kd + off, kIdS, kk > 0);
        }
      };
      auto issue_pv = [&](int vs, bool first_tile) {
        const uint64_t vd = vd0 + (uint64_t)vs * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < kKvTile / 16; ++kk) {
          const uint64_t off = (uint64_t)((kk * 2048) >> 4);
          mma_ts(tO, tS + kk * 8, vd + off, kIdO, (!first_tile || kk > 0) ? 1u : 0u);
        }
      };
      while (true) {
        const int ms = ucnt & 1;
        pwait(&mfull[ms], (ucnt >> 1) & 1, a.err, misc);
        ++ucnt;
        const PMsg m = msg[ms];
        mbar_arrive(&mempty[ms]);
        if (m.done || *reinterpret_cast<volatile int*>(misc)) break;
        const int n = m.ntiles;
        if (n == 0) continue;  // no MMA work: the softmax warps write the zeros
        if (s >= m.nslots) {
          // this slot is idle in the unit (odd GQA group): give the shared
          // buffers this thread's release once each is filled for the unit
          pwait(qfull, q_cnt & 1, a.err, misc);
          ++q_cnt;
          mbar_arrive(qempty);
          for (int j = 0; j < n; ++j) {
            const int it = kv_it + j;
            pwait(&kfull[it % KS], (it / KS) & 1, a.err, misc);
            mbar_arrive(&kempty[it % KS]);
            pwait(&vready[it % VS], (it / VS) & 1, a.err, misc);
            mbar_arrive(&vempty[it % VS]);
          }
          kv_it += n;
          continue;
        }
        // (F16: the slot's softmax warps convert the bf16 query tile to fp16
        // in place once it lands and then release it to the tensor core)
        if constexpr (F16) {
          pwait(&qconv[s], qc_cnt & 1, a.err, misc);
          ++qc_cnt;
        } else {
          pwait(qfull, q_cnt & 1, a.err, misc);
        }
        ++q_cnt;
        const bool paired = m.nslots == 2;
        {
          const int ks0 = kv_it % KS;
          pwait(&kfull[ks0], (kv_it / KS) & 1, a.err, misc);
          take_turn(paired);
          tc_fence_after();
          issue_qk(ks0);
          pass_turn(paired);
          tc_commit(&sfull[s]);
          tc_commit(&kempty[ks0]);
          if (n == 1) tc_commit(qempty);
        }
        for (int j = 0; j < n; ++j) {
          const int it = kv_it + j;
          const int vs = it % VS;
          const int itn = it + 1, ksn = itn % KS;
          pwait(&vready[vs], (it / VS) & 1, a.err, misc);
          if (j + 1 < n) pwait(&kfull[ksn], (itn / KS) & 1, a.err, misc);
          pwait(&pfull[s], p_it & 1, a.err, misc);
          ++p_it;
          if (j == 0) {
            // O of the slot is free once the previous unit's epilogue read
            // it (the first QK above already overlapped that epilogue).
            // Only units with tiles take part in this handshake, so the
            // softmax side can never run two phases ahead of these waits.
            pwait(&ofree[s], (u_cnt & 1) ^ 1, a.err, misc);
            ++u_cnt;
          }
          take_turn(paired);
          tc_fence_after();
          issue_pv(vs, j == 0);
          if (j + 1 < n) issue_qk(ksn);
          pass_turn(paired);
          if (j == n - 1) tc_commit(&ofull[s]);
          tc_commit(&vempty[vs]);
          if (j + 1 < n) {
            tc_commit(&sfull[s]);
            tc_commit(&kempty[ksn]);
            if (j + 1 == n - 1) tc_commit(qempty);
          }
        }
        kv_it += n;
      }
      // everything this thread issued has finished before the TMEM is released
      tc_commit(&drain[s]);
      mbar_wait(&drain[s], 0, a.err);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ============================ V guard ============================
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    int ucnt = 0, kv_it = 0;
    while (true) {
      const int ms = ucnt & 1;
      pwait(&mfull[ms], (ucnt >> 1) & 1, a.err, misc);
      ++ucnt;
      const PMsg m = msg[ms];
      __syncwarp();
      if (lane == 0) mbar_arrive(&mempty[ms]);
      if (m.done || *reinterpret_cast<volatile int*>(misc)) break;
      for (int j = 0; j < m.ntiles; ++j, ++kv_it) {
        const int vs = kv_it % VS;
        pwait(&vfull[vs], (kv_it / VS) & 1, a.err, misc);
        const int64_t j0 = (int64_t)(m.tile0 + j) * kKvTile;
        const int nv = (int)min((int64_t)kKvTile, (int64_t)m.kv_len - j0);
        if (nv < kKvTile) {
          uint8_t* vt = smem + Cfg::kOffV + vs * Cfg::kTileBytes;
          for (int x = nv * 8 + lane; x < kKvTile * 8; x += 32) {  // 16-byte pieces
            const int row = x >> 3, piece = x & 7;
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub)
              *reinterpret_cast<uint4*>(vt + sub * 16384 + row * 128 + piece * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&vready[vs]);
      }
    }
  } else {
    // ============================ softmax + epilogue ============================
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;" ::: "memory");
    const int s = (warp - 4) >> 2;      // slot
    const int row = tid - 128 - 128 * s;  // query row of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + 256 * s;
    const uint32_t tO = tS + 128;
    int ucnt = 0, s_it = 0, o_cnt = 0, qf_cnt = 0;
    while (true) {
      const int ms = ucnt & 1;
      pwait(&mfull[ms], (ucnt >> 1) & 1, a.err, misc);
      ++ucnt;
      const PMsg m = msg[ms];
      named_bar_sync(2 + s, 128);
      if (row == 0) mbar_arrive(&mempty[ms]);
      if (m.done || *reinterpret_cast<volatile int*>(misc)) break;
      const int qf_par = qf_cnt & 1;  // (F16) the query tiles land once per unit with tiles
      if (m.ntiles > 0) ++qf_cnt;
      if (s >= m.nslots) continue;
      const int h = s ? m.h1 : m.h0;
      const int64_t i = (int64_t)m.t * kQTile + row;
      const bool valid = i < m.q_len;
      const int64_t p = row_pos(a, m.q_len, m.kv_len, i);
      int64_t lo = a.mask_mode == 4 ? p - a.pre_tokens : 0;
      int64_t hi = (a.mask_mode == 2 || a.mask_mode == 3)
                       ? p
                       : (a.mask_mode == 4 ? p + a.next_tokens : m.kv_len - 1);
      lo = max(lo, (int64_t)0);
      hi = min(hi, (int64_t)m.kv_len - 1);
      // explicit mask: this row's bytes (1 = hidden) of sequence m.b
      const uint8_t* mrow_ptr =
          (a.mask && valid) ? a.mask + (int64_t)m.b * a.mask_bstride + i * a.mask_rstride : nullptr;
      // score scale of this row (log2 units); fp16 operands take back their
      // powers of two here and in the output
      float sl = a.scale_log2, vfac = 1.f;
      if constexpr (F16) {
        // This thread's row of the slot's bf16 query tile, to fp16 in place
        // times 2^sh, sh = 15 - the exponent of the row's largest element
        // (kept in [-100, 100]): fp16 then holds the row without overflow or
        // lost bits, and 2^-sh goes into the row's score scale.  The row's
        // 128-byte pieces are visited from a different chunk per row, so a
        // warp's accesses spread over the banks; the chunks' order within a
        // row does not matter here.  Then the slot's MMA thread may read it.
        float qfac_row = 1.f;
        if (m.ntiles > 0) {
          pwait(qfull, qf_par, a.err, misc);
          uint8_t* qr = smem + Cfg::kOffQ + s * Cfg::kTileBytes + row * 128;
          uint4 qw[NSUB * 8];
          uint32_t e = 0;
#pragma unroll
          for (int c = 0; c < NSUB * 8; ++c) {
            const int cc = ((c & 7) + row) & 7;
            qw[c] = *reinterpret_cast<const uint4*>(qr + (c >> 3) * 16384 + cc * 16);
            const uint32_t wv[4] = {qw[c].x, qw[c].y, qw[c].z, qw[c].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) e = max(e, max((wv[k] >> 7) & 0xffu, (wv[k] >> 23) & 0xffu));
          }
          const int sh = min(max(142 - (int)e, -100), 100);  // 15 - (e - 127)
          const float up = __int_as_float((127 + sh) << 23);
#pragma unroll
          for (int c = 0; c < NSUB * 8; ++c) {
            const int cc = ((c & 7) + row) & 7;
            const uint32_t wv[4] = {qw[c].x, qw[c].y, qw[c].z, qw[c].w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[k]));
              o[k] = pack_f16(f.x * up, f.y * up);
            }
            *reinterpret_cast<uint4*>(qr + (c >> 3) * 16384 + cc * 16) = make_uint4(o[0], o[1], o[2], o[3]);
          }
          qfac_row = __int_as_float((127 - sh) << 23);
          fence_proxy_async_smem();  // the fp16 tile, for the tensor core
          __syncwarp();
          if (lane == 0) mbar_arrive(&qconv[s]);
        }
        const int64_t hkv = ((int64_t)m.b * a.KVN + m.hk) * 2;
        if (valid) sl *= qfac_row;
        sl *= __ldg(a.kvfac + hkv);
        vfac = __ldg(a.kvfac + hkv + 1);
      }
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < m.ntiles; ++j) {
        // visible columns of this row in the tile: [c0, c1) (tile-local)
        const int64_t j0 = (int64_t)(m.tile0 + j) * kKvTile;
        const int c0 = (int)min(max(lo - j0, (int64_t)0), (int64_t)kKvTile);
        const int c1 = (int)min(max(hi - j0 + 1, (int64_t)0), (int64_t)kKvTile);
        // explicit mask: the tile's bytes of this row, 16 at a time up to the
        // row's visible end (rows are 16-byte multiples covering the KV
        // capacity), as four 32-bit hidden-key bit sets; the loads are issued
        // before the wait for the scores
        uint32_t hidden[4] = {0u, 0u, 0u, 0u};
        if (a.mask) {
          if (mrow_ptr) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              uint4 w = make_uint4(0u, 0u, 0u, 0u);
              if (16 * k < c1) w = __ldg(reinterpret_cast<const uint4*>(mrow_ptr + j0) + k);
              const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                // nonzero bytes -> 0x80 in their top bit, gathered into 4 bits
                const uint32_t nz = (((wv[q] & 0x7f7f7f7fu) + 0x7f7f7f7fu) | wv[q]) & 0x80808080u;
                hidden[k >> 1] |= ((nz * 0x00204081u) >> 28) << (16 * (k & 1) + 4 * q);
              }
            }
          }
        }
        pwait(&sfull[s], s_it & 1, a.err, misc);
        ++s_it;
        tc_fence_after();
        const bool all_full =
            __all_sync(0xffffffffu, c0 == 0 && c1 == kKvTile &&
                                        (hidden[0] | hidden[1] | hidden[2] | hidden[3]) == 0u);
        // masked score: -inf after the scaling for either sign of the scale
        const uint32_t hole = __float_as_uint(NEG ? INFINITY : -INFINITY);
        // the row's 128 scores: four TMEM loads, one wait; they stay in
        // registers for the maximum and the exponentials
        uint32_t v[kKvTile];
#pragma unroll
        for (int c = 0; c < kKvTile / 32; ++c)
          tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
        tmem_wait_ld();
        if (!all_full) {
#pragma unroll
          for (int e = 0; e < kKvTile; ++e)
            if (e < c0 || e >= c1 || ((hidden[e >> 5] >> (e & 31)) & 1u)) v[e] = hole;
        }
        // row maximum of the raw scores (minimum for a negative scale), four
        // three-input chains
        float pm[4] = {__uint_as_float(hole), __uint_as_float(hole), __uint_as_float(hole),
                       __uint_as_float(hole)};
#pragma unroll
        for (int e = 0; e < kKvTile; e += 8)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if constexpr (NEG)
              pm[k] = fmin3(pm[k], __uint_as_float(v[e + k]), __uint_as_float(v[e + 4 + k]));
            else
              pm[k] = fmax3(pm[k], __uint_as_float(v[e + k]), __uint_as_float(v[e + 4 + k]));
          }
        const float best = NEG ? fminf(fminf(pm[0], pm[1]), fminf(pm[2], pm[3]))
                               : fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
        const float mx = isinf(best) ? -INFINITY : best * sl;  // all masked -> -inf
        // lazily moved reference maximum: a row moves it when the new maximum
        // exceeds it by more than 2^8 (or on its first visible key); rows
        // that move it rescale l and their O row.  TMEM loads and stores are
        // warp-collective, so the rescale runs for the whole warp with a
        // factor of 1 on the rows that keep their reference.
        const bool move = mx > m_used + kRescaleThreshold || (m_used == -INFINITY && mx != -INFINITY);
        const bool rescale = move && m_used != -INFINITY;
        float corr = 1.f;
        if (rescale) {
          corr = ex2_approx(m_used - mx);
          l *= corr;
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t w[32];
            tmem_ld32(tO + 32 * c, w);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * corr);
            tmem_st32(tO + 32 * c, w);
          }
          tmem_wait_st();
        }
        if (move) m_used = mx;
        const float nbase = m_used == -INFINITY ? 0.f : -m_used;
        // p = 2^(s * scale * log2e - m), two columns per packed FMA; masked
        // columns hold -inf after the scaling and give 0; P goes back to the
        // first 64 TMEM columns of S as bf16 pairs
        float2 ps[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) ps[k] = make_float2(0.f, 0.f);
        const float2 sl2 = make_float2(sl, sl), nb2 = make_float2(nbase, nbase);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pv[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x = ffma2(make_float2(__uint_as_float(v[64 * c + 2 * e]),
                                               __uint_as_float(v[64 * c + 2 * e + 1])),
                                   sl2, nb2);
            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            ps[e & 3] = fadd2(ps[e & 3], pp);
            pv[e] = F16 ? pack_f16(pp.x, pp.y) : pack_bf16(pp.x, pp.y);
          }
          tmem_st32(tS + 32 * c, pv);
        }
        const float2 s2 = fadd2(fadd2(ps[0], ps[1]), fadd2(ps[2], ps[3]));
        const float sum = s2.x + s2.y;
        tmem_wait_st();
        l += sum;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[s]);
      }
      // ---- epilogue ----
      float scl = 0.f, lse = INFINITY;
      if (m_used != -INFINITY && l > 0.f) {  // l == 0: the row saw no key
        float Mp = m_used, L = l;
        if (a.sinks) {
          const float sk = a.sinks[h] * 1.4426950408889634f;
          Mp = fmaxf(m_used, sk);
          L = l * exp2f(m_used - Mp) + exp2f(sk - Mp);
        }
        scl = exp2f(m_used - Mp) / L * vfac;
        lse = (Mp + log2f(L)) * 0.6931471805599453f;
      }
      uint16_t* orow = a.out + (m.q_row0 + row) * a.out_stride + (int64_t)h * D;
      if (m.ntiles > 0) {
        pwait(&ofull[s], o_cnt & 1, a.err, misc);
        ++o_cnt;
        tc_fence_after();
        // the whole O row into registers, then the slot's O is released (the
        // next unit's first P V may overwrite it) before the global stores
        uint32_t v[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          tmem_ld32(tO + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ofree[s]);
        if (valid) {
          // 32-byte stores where the row allows (a row is D bf16 = 2D bytes)
          const bool wide = (reinterpret_cast<uintptr_t>(orow) & 31) == 0;
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack_bf16(__uint_as_float(v[16 * c + 2 * e]) * scl,
                               __uint_as_float(v[16 * c + 2 * e + 1]) * scl);
            if (wide) {
              asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(orow + 16 * c),
                           "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                           "r"(w[6]), "r"(w[7])
                           : "memory");
            } else {
              *reinterpret_cast<uint4*>(orow + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(orow + 16 * c + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
      } else if (valid) {
#pragma unroll
        for (int e = 0; e < D / 8; ++e)
          *reinterpret_cast<uint4*>(orow + 8 * e) = make_uint4(0u, 0u, 0u, 0u);
      }
      if (valid && a.lse) {
        const int64_t li = a.layout == 1 ? (m.q_row0 + row) * a.QN + h
                                         : ((int64_t)m.b * a.QN + h) * a.S_q + i;
        a.lse[li] = lse;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
cudaError_t launch_prefill_schedule(const PrefillArgs& a, cudaStream_t s) {
  prefill_schedule_kernel<<<1, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, bool NEG, bool F16>
static cudaError_t launch_prefill_t(const PrefillArgs& a, const CUtensorMap& tq,
                                    const CUtensorMap& tk, const CUtensorMap& tv,
                                    cudaStream_t s) {
  using Cfg = PrefillCfg<D>;
  auto kern = prefill_kernel<D, NEG, F16>;
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
  return launch_pdl(kern, dim3(a.num_ctas), dim3(kPThreads), Cfg::kSmem, s, a, tq, tk, tv);
}

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t s) {
  const bool neg = a.scale_log2 < 0.f;
  if (a.f16)  // fp16 operands: FP8 caches, D = 128
    return neg ? launch_prefill_t<128, true, true>(a, tq, tk, tv, s)
               : launch_prefill_t<128, false, true>(a, tq, tk, tv, s);
  if (a.D == 64) return neg ? launch_prefill_t<64, true, false>(a, tq, tk, tv, s)
                            : launch_prefill_t<64, false, false>(a, tq, tk, tv, s);
  return neg ? launch_prefill_t<128, true, false>(a, tq, tk, tv, s)
             : launch_prefill_t<128, false, false>(a, tq, tk, tv, s);
}

}  // namespace fia
