// decode.cu -- the incremental-inference branch of fused inference attention
// (query length 1; "aclnnFusedInferAttentionScoreV2": the IncreFlashAttention
// branch runs when the query S is 1) over a paged KV cache, plus its tile
// scheduler.
//
// Work unit: (batch b, KV head hk, head group hg).  The query heads of one GQA
// group share KV head hk; up to 8 (G <= 8) or 16 of them form the N columns
// of every mma.sync, so each KV page is read from HBM once for the group.  A
// unit owns the KV tiles (128 positions) its query row can see.
//
// Scheduler (decode_schedule_kernel): cost(u) = visible tiles (>= 1; 0 when
// the batch has no query row); CTA c of n persistent CTAs owns the global tile
// interval [floor(c*total/n), floor((c+1)*total/n)) of the units laid end to
// end, so all CTAs get the same number of tiles within one.  A unit cut by a
// CTA boundary is split-KV: each piece writes its (m, l, acc) partial and the
// last piece to finish folds all pieces in CTA order (deterministic).
//
// Decode kernel: one producer warp streams K and V pages with TMA (page rows
// from block_table) into a ring of shared-memory stages; eight consumer warps
// each take 16 rows of every tile.  The products are computed transposed
// ("swap AB"): S^T = K Q^T with the KV rows as the mma M dimension and the
// query heads as N, then O^T += V^T P^T, where P^T comes out of the S^T
// accumulators with movmatrix.  Softmax is online, in the exp2 domain, per
// head (column).  FP8 E4M3 pages are widened to fp16 in registers (exact);
// K tile scales multiply the per-64-column partial scores and V tile scales
// are folded into P^T, so the dequantised cache is never materialised.
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace fia {

namespace {

constexpr int kConsumers = 8;                        // consumer warps
constexpr int kThreads = 32 * (1 + kConsumers);
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
  static constexpr int kStageBytes = 2 * kTileBytes + 2 * kScaleBytes;
  static constexpr int kStages = FP8 ? 5 : (D == 128 ? 3 : 6);
  static constexpr int kQBytes = kMaxGH * D * 2;
  static constexpr int kRedBytes = 4 * 8 * D * 4;           // 4 warps x 8 heads x D
  static constexpr int kRedMlBytes = kConsumers * kMaxGH * 2 * 4;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffRed = kOffQ + 2 * kQBytes;
  static constexpr int kOffRedMl = kOffRed + kRedBytes;
  static constexpr int kOffBar = kOffRedMl + kRedMlBytes;
  static constexpr int kOffMsg = kOffBar + 8 * (2 * kStages + 4);
  static constexpr int kOffMisc = kOffMsg + 2 * 128;
  static constexpr int kSmem = kOffMisc + 64 + 1024;  // + alignment slack
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kSmem <= 232448, "shared memory");
};

struct UnitInfo {
  int b, hk, hg, h0, nrows;
  int64_t qrow;  // token row of q/out
  int64_t kv_len, lo, hi;
  int tile0, ntiles;
};

__device__ __forceinline__ UnitInfo unit_info(const DecodeArgs& a, int64_t u) {
  UnitInfo r;
  const int per_b = a.KVN * a.HG;
  r.b = (int)(u / per_b);
  const int rem = (int)(u % per_b);
  r.hk = rem / a.HG;
  r.hg = rem % a.HG;
  r.h0 = r.hk * a.G + r.hg * a.GH;
  r.nrows = min(a.GH, a.G - r.hg * a.GH);
  int64_t ql;
  if (a.layout == 1) {
    r.qrow = a.cu_seqlens_q[r.b];
    ql = (int64_t)a.cu_seqlens_q[r.b + 1] - r.qrow;
  } else {
    r.qrow = (int64_t)r.b * a.S_q;
    ql = a.S_q;
  }
  r.kv_len = a.seqused_kv ? a.seqused_kv[r.b] : a.S_kv;
  const int64_t p = r.kv_len - 1;  // the single query row sits at the last key
  int64_t lo = 0, hi = r.kv_len - 1;
  if (a.mask_mode == 3) {
    hi = min(hi, p);
  } else if (a.mask_mode == 4) {
    lo = max(lo, p - a.pre_tokens);
    hi = min(hi, p + a.next_tokens);
  }
  r.lo = lo;
  r.hi = hi;
  if (ql <= 0 || r.kv_len <= 0 || hi < lo) {
    r.tile0 = 0;
    r.ntiles = 0;
  } else {
    r.tile0 = (int)(lo / kKvTile);
    r.ntiles = (int)(hi / kKvTile - lo / kKvTile + 1);
  }
  return r;
}

// What the producer hands the consumers with each unit's query rows (one per
// query buffer), so that consumers never wait on global loads between units.
struct UnitMsg {
  UnitInfo r;
  int64_t u, pu, pu1;
  int t_begin, t_end, split, first, done;
};
static_assert(sizeof(UnitMsg) <= 128, "message slot");

// largest u with prefix[u] <= g (prefix[U] > g)
__device__ __forceinline__ int64_t find_unit(const int64_t* prefix, int64_t U, int64_t g) {
  int64_t lo = 0, hi = U;  // invariant prefix[lo] <= g < prefix[hi]
  while (hi - lo > 1) {
    const int64_t mid = (lo + hi) >> 1;
    if (prefix[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int64_t next_unit(const int64_t* prefix, int64_t U, int64_t u) {
  ++u;
  while (u < U && prefix[u + 1] == prefix[u]) ++u;
  return u;
}

// largest c with cta_begin[c] <= g
__device__ __forceinline__ int find_cta(const int64_t* beg, int n, int64_t g) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (beg[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int64_t phys_row(const DecodeArgs& a, int b, int64_t j) {
  if (a.block_table) {
    const int64_t blk = a.block_table[(int64_t)b * a.max_blocks + j / a.block_size];
    return blk * a.block_size + j % a.block_size;
  }
  return (int64_t)b * a.S_kv + j;
}

// Row of the FP8 scale arrays for logical KV row j of batch b, KV head hk:
// scales are stored head-major inside each page, [pages, KV_N, page rows,
// D/64] (the paged per-token, per-head scale shape (blockNum, N, blockSize) of
// the FIA dequantisation parameters, with the 64-element tiles last).
__device__ __forceinline__ int64_t scale_row(const DecodeArgs& a, int b, int hk, int64_t j) {
  if (a.block_table) {
    const int64_t blk = a.block_table[(int64_t)b * a.max_blocks + j / a.block_size];
    return (blk * a.KVN + hk) * a.block_size + j % a.block_size;
  }
  return ((int64_t)b * a.KVN + hk) * a.S_kv + j;
}

// Bounded barrier wait; after the first time-out in the CTA every later wait
// returns at once, so a broken pipeline ends the kernel instead of hanging it.
__device__ __forceinline__ void wait_or_abort(uint64_t* bar, uint32_t parity, int* err,
                                              int* misc) {
  if (*reinterpret_cast<volatile int*>(misc)) return;
  if (!mbar_wait(bar, parity, err)) *reinterpret_cast<volatile int*>(misc) = 1;
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
__global__ void __launch_bounds__(1024) decode_schedule_kernel(const DecodeArgs a) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t carry;
  const int64_t U = a.num_units;
  int64_t* prefix = const_cast<int64_t*>(a.unit_prefix);
  int64_t* beg = const_cast<int64_t*>(a.cta_begin);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < U; base += blockDim.x) {
    const int64_t u = base + tid;
    int64_t cost = 0;
    if (u < U) {
      UnitInfo r = unit_info(a, u);
      int64_t ql;
      if (a.layout == 1) ql = (int64_t)a.cu_seqlens_q[r.b + 1] - a.cu_seqlens_q[r.b];
      else ql = a.S_q;
      cost = ql > 0 ? max(1, r.ntiles) : 0;
      a.counters[u] = 0;
    }
    // block-wide inclusive scan of cost
    int64_t x = cost;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int64_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int64_t excl = carry + (wid ? warp_sums[wid - 1] : 0) + x - cost;
    if (u < U) prefix[u] = excl;
    __syncthreads();
    if (tid == blockDim.x - 1) carry = excl + cost;
    __syncthreads();
  }
  const int64_t total = carry;
  if (tid == 0) {
    prefix[U] = total;
    *a.err = 0;  // error word of this plan's execution
  }
  for (int c = tid; c <= a.num_ctas; c += blockDim.x)
    beg[c] = (int64_t)c * total / a.num_ctas;
}

// ---------------------------------------------------------------------------
// decode kernel
// ---------------------------------------------------------------------------
template <int D, bool FP8, int NG>  // NG: groups of 8 query heads per unit (1 or 2)
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv) {
  using Cfg = DecodeCfg<D, FP8>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* empty = full + S;
  uint64_t* qfull = empty + S;
  uint64_t* qempty = qfull + 2;
  int* misc = reinterpret_cast<int*>(smem + Cfg::kOffMisc);
  UnitMsg* msg = reinterpret_cast<UnitMsg*>(smem + Cfg::kOffMsg);
  float* red = reinterpret_cast<float*>(smem + Cfg::kOffRed);
  float* red_ml = reinterpret_cast<float*>(smem + Cfg::kOffRedMl);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int64_t U = a.num_units;
  const int64_t g0 = a.cta_begin[c], g1 = a.cta_begin[c + 1];

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], kConsumers);
    }
    misc[0] = 0;  // abort flag
    fence_barrier_init();
  }
  __syncthreads();
  if (g0 >= g1) return;

  const int64_t u0 = find_unit(a.unit_prefix, U, g0);

  if (warp == 0) {
    // ======================= producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
    }
    int it = 0, ucount = 0;
    int64_t u = u0;
    UnitInfo r = unit_info(a, u);
    int64_t pu = a.unit_prefix[u], pu1 = a.unit_prefix[u + 1];
    while (true) {
      // the next unit's description is loaded one unit ahead
      const int64_t un = next_unit(a.unit_prefix, U, u);
      const int64_t pun = un < U ? a.unit_prefix[un] : g1;
      const bool has_next = un < U && pun < g1;
      UnitInfo rn = r;
      int64_t pun1 = pu1;
      if (has_next) {
        rn = unit_info(a, un);
        pun1 = a.unit_prefix[un + 1];
      }
      const int t_begin = (int)(max(g0, pu) - pu);
      const int t_end = (int)(min(g1, pu1) - pu);
      {  // unit description + query rows of the group (one bulk copy)
        const int qs = ucount & 1;
        wait_or_abort(&qempty[qs], ((ucount >> 1) & 1) ^ 1, a.err, misc);
        if (lane == 0) {
          UnitMsg& m = msg[qs];
          m.r = r;
          m.u = u;
          m.pu = pu;
          m.pu1 = pu1;
          m.t_begin = t_begin;
          m.t_end = t_end;
          m.split = (pu < g0) || (pu1 > g1);
          m.first = (u == u0);
          m.done = 0;
          const uint32_t bytes = (uint32_t)(r.nrows * D * 2);
          mbar_arrive_expect_tx(&qfull[qs], bytes);
          bulk_load(smem + Cfg::kOffQ + qs * Cfg::kQBytes,
                    a.q + r.qrow * a.q_stride + (int64_t)r.h0 * D, bytes, &qfull[qs]);
        }
        ++ucount;
      }
      for (int t = t_begin; r.ntiles > 0 && t < t_end; ++t, ++it) {
        const int s = it % S;
        const uint32_t par = ((it / S) & 1) ^ 1;
        const int64_t j0 = (int64_t)(r.tile0 + t) * kKvTile;
        const int nrb = kKvTile / a.box_rows;
        const int nbox = nrb * Cfg::kNsub * 2;  // <= 32: one box per lane
        // page lookups first: their latency overlaps the wait for the slot
        const int isv = lane & 1;
        const int sub = (lane >> 1) % Cfg::kNsub;
        const int rb = (lane >> 1) / Cfg::kNsub;
        const int64_t jb = j0 + (int64_t)rb * a.box_rows;
        const bool mine = lane < nbox && jb < r.kv_len;
        const int64_t prow = mine ? phys_row(a, r.b, jb) : 0;
        constexpr int NT = D / 64;
        // FP8: the scales of one head inside a page are contiguous rows of NT
        // floats, so each (K or V, page piece) is one bulk copy next to its
        // TMA box.  Pieces are even-length at even rows (block sizes are
        // multiples of 32; contiguous caches have an even length), hence
        // 16-byte aligned.
        int64_t srow = 0;
        int srows = a.box_rows;
        if constexpr (FP8) {
          if (mine) srow = scale_row(a, r.b, r.hk, jb);
          if (!a.block_table) srows = (int)min((int64_t)a.box_rows, (int64_t)a.S_kv - jb);
        }
        int nvalid = 0, scale_rows = 0;
        for (int q = 0; q < nrb; ++q) {
          const int64_t jq = j0 + (int64_t)q * a.box_rows;
          if (jq < r.kv_len) {
            ++nvalid;
            scale_rows += a.block_table ? a.box_rows : (int)min((int64_t)a.box_rows, (int64_t)a.S_kv - jq);
          }
        }
        wait_or_abort(&empty[s], par, a.err, misc);
        uint8_t* st = smem + s * Cfg::kStageBytes;
        if (lane == 0) {
          uint32_t bytes = (uint32_t)(2 * nvalid * Cfg::kNsub * a.box_rows * 128);
          if constexpr (FP8) bytes += (uint32_t)(2 * scale_rows * NT * 4);
          mbar_arrive_expect_tx(&full[s], bytes);
        }
        __syncwarp();
        if (mine) {
          uint8_t* dst = st + isv * Cfg::kTileBytes + sub * (kKvTile * 128) + rb * a.box_rows * 128;
          const int col = FP8 ? r.hk * D : r.hk * D + sub * 64;
          tma_load_2d(dst, isv ? &tv : &tk, &full[s], col, (int)prow);
          if constexpr (FP8) {
            float* sdst = reinterpret_cast<float*>(st + 2 * Cfg::kTileBytes) +
                          isv * (kKvTile * NT) + rb * a.box_rows * NT;
            bulk_load(sdst, (isv ? a.v_scale : a.k_scale) + srow * NT,
                      (uint32_t)(srows * NT * 4), &full[s]);
          }
        }
      }
      if (!has_next) break;
      u = un;
      r = rn;
      pu = pun;
      pu1 = pun1;
    }
    {  // end of the CTA's work: an empty message
      const int qs = ucount & 1;
      wait_or_abort(&qempty[qs], ((ucount >> 1) & 1) ^ 1, a.err, misc);
      if (lane == 0) {
        msg[qs].done = 1;
        mbar_arrive(&qfull[qs]);
      }
    }
    return;
  }

  // ======================= consumers =======================
  const int cw = warp - 1;     // 0..7
  const int g = lane >> 2;     // fragment row group
  const int q4 = lane & 3;     // thread in quad
  const int R0 = cw * kRowsPerWarp;
  const int nthr = 32 * kConsumers;
  const int ctid = tid - 32;
  const uint32_t smem_base = smem_u32(smem);
  constexpr int KS = D / 16;   // k-steps over D (QK)
  constexpr int MT = D / 16;   // m-tiles over D (PV)

  int it = 0, ucount = 0;
  while (true) {
    const int qs = ucount & 1;
    wait_or_abort(&qfull[qs], (ucount >> 1) & 1, a.err, misc);
    if (msg[qs].done || *reinterpret_cast<volatile int*>(misc)) break;
    const UnitInfo r = msg[qs].r;
    const int64_t u = msg[qs].u, pu = msg[qs].pu, pu1 = msg[qs].pu1;
    const int t_begin = msg[qs].t_begin, t_end = msg[qs].t_end;
    const bool split = msg[qs].split, first = msg[qs].first;

    // ---- Q^T fragments (mma B operand: k = d, n = head) ----
    uint32_t qb[NG][KS][2];
    {
      const uint16_t* qsm = reinterpret_cast<const uint16_t*>(smem + Cfg::kOffQ + qs * Cfg::kQBytes);
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
        const int head = ng * 8 + g;
        const bool ok = head < r.nrows;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          if constexpr (!FP8) {
            const int d0 = kk * 16 + 2 * q4;
            qb[ng][kk][0] = ok ? *reinterpret_cast<const uint32_t*>(qsm + head * D + d0) : 0u;
            qb[ng][kk][1] = ok ? *reinterpret_cast<const uint32_t*>(qsm + head * D + d0 + 8) : 0u;
          } else {
            // k-step kk = 4*tile + j covers d = 64*tile + 16*q + 4*j + {0..3}:
            // slots 2q,2q+1 <- the first two, slots 2q+8,2q+9 <- the last two
            const int d0 = (kk >> 2) * 64 + 16 * q4 + 4 * (kk & 3);
            if (ok) {
              const uint2 v = *reinterpret_cast<const uint2*>(qsm + head * D + d0);
              const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
              const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
              qb[ng][kk][0] = pack_f16(lo.x, lo.y);
              qb[ng][kk][1] = pack_f16(hi.x, hi.y);
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
    float vref[2] = {1.f, 1.f};  // FP8: V scale reference per d-tile

    const int ntile_here = r.ntiles == 0 ? 0 : (t_end - t_begin);
    for (int tt = 0; tt < ntile_here; ++tt, ++it) {
      const int t = t_begin + tt;
      const int s = it % S;
      wait_or_abort(&full[s], (it / S) & 1, a.err, misc);
      const uint32_t st = smem_base + s * Cfg::kStageBytes;
      const uint8_t* stp = smem + s * Cfg::kStageBytes;
      const int64_t jw = (int64_t)(r.tile0 + t) * kKvTile + R0;  // first KV row of this warp
      const bool edge = (jw < r.lo) || (jw + kRowsPerWarp - 1 > r.hi);
      const bool tail = (jw + kRowsPerWarp > r.kv_len);
      // KV positions of fragment rows g and g+8
      const int64_t jg0 = jw + rho16(g), jg1 = jw + rho16(g + 8);

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
            ka[0] = e4m3x2_to_f16x2((uint16_t)(va[j] & 0xffffu));
            ka[1] = e4m3x2_to_f16x2((uint16_t)(vb[j] & 0xffffu));
            ka[2] = e4m3x2_to_f16x2((uint16_t)(va[j] >> 16));
            ka[3] = e4m3x2_to_f16x2((uint16_t)(vb[j] >> 16));
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
          if (jg0 >= r.kv_len) k0 = make_float2(0.f, 0.f);
          if (jg1 >= r.kv_len) k1 = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          sc[ng][0] = sc[ng][0] * k0.x + s2[ng][0] * k0.y;
          sc[ng][1] = sc[ng][1] * k0.x + s2[ng][1] * k0.y;
          sc[ng][2] = sc[ng][2] * k1.x + s2[ng][2] * k1.y;
          sc[ng][3] = sc[ng][3] * k1.x + s2[ng][3] * k1.y;
        }
      }

      // ---------------- mask + online softmax per head ----------------
      const bool ok0 = !(edge || tail) || (jg0 >= r.lo && jg0 <= r.hi);
      const bool ok1 = !(edge || tail) || (jg1 >= r.lo && jg1 <= r.hi);
      float corr[NG][2];
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x0 = ok0 ? sc[ng][e] * a.scale_log2 : -INFINITY;
          const float x1 = ok1 ? sc[ng][2 + e] * a.scale_log2 : -INFINITY;
          float mx = fmaxf(x0, x1);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m_r[ng][e], mx);
          const float mu = mn == -INFINITY ? 0.f : mn;
          corr[ng][e] = m_r[ng][e] == -INFINITY ? 0.f : fast_exp2(m_r[ng][e] - mu);
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
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            acc[i][ng][0] *= corr[ng][0];
            acc[i][ng][1] *= corr[ng][1];
            acc[i][ng][2] *= corr[ng][0];
            acc[i][ng][3] *= corr[ng][1];
          }
        // rows past kv_len may hold anything (even NaN): zero their V lanes
        bool z0 = false, z1 = false, z2 = false, z3 = false;
        if (tail) {
          z0 = jw + rho16(2 * q4) >= r.kv_len;
          z1 = jw + rho16(2 * q4 + 1) >= r.kv_len;
          z2 = jw + rho16(2 * q4 + 8) >= r.kv_len;
          z3 = jw + rho16(2 * q4 + 9) >= r.kv_len;
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
          if (jg0 >= r.kv_len) v0 = make_float2(0.f, 0.f);
          if (jg1 >= r.kv_len) v1 = make_float2(0.f, 0.f);
        }
        // warp-wide reference per d-tile keeps P^T * scale / ref in (0, 1]
        float vmax[2] = {fmaxf(v0.x, v1.x), fmaxf(v0.y, v1.y)};
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          vmax[t2] = fmaxf(vmax[t2], __shfl_xor_sync(0xffffffffu, vmax[t2], 4));
          vmax[t2] = fmaxf(vmax[t2], __shfl_xor_sync(0xffffffffu, vmax[t2], 8));
          vmax[t2] = fmaxf(vmax[t2], __shfl_xor_sync(0xffffffffu, vmax[t2], 16));
          if (!(vmax[t2] > 0.f)) vmax[t2] = vref[t2];
        }
        const float ratio[2] = {vref[0] / vmax[0], vref[1] / vmax[1]};
        vref[0] = vmax[0];
        vref[1] = vmax[1];
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          const int t2 = i >> 2;
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            acc[i][ng][0] *= corr[ng][0] * ratio[t2];
            acc[i][ng][1] *= corr[ng][1] * ratio[t2];
            acc[i][ng][2] *= corr[ng][0] * ratio[t2];
            acc[i][ng][3] *= corr[ng][1] * ratio[t2];
          }
        }
        // P^T per d-tile with the V scales folded in
        uint32_t pb[2][NG][2];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          const float iv = 1.f / vref[t2];
          const float fa = (t2 ? v0.y : v0.x) * iv, fb = (t2 ? v1.y : v1.x) * iv;
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            pb[t2][ng][0] = movmatrix_t(pack_f16(sc[ng][0] * fa, sc[ng][1] * fa));
            pb[t2][ng][1] = movmatrix_t(pack_f16(sc[ng][2] * fb, sc[ng][3] * fb));
          }
        }
        // V codes of KV slots 2q, 2q+1, 2q+8, 2q+9: 8 bytes per d-tile at
        // d = 64*tile + 8*g .. +7 (m-tile i covers d = 64*(i/4) + 8*g + (i%4)
        // in fragment rows 0-7 and +4 in rows 8-15)
        const uint8_t* vt = stp + Cfg::kTileBytes;
        uint2 w[4][2];
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          const int slot = 2 * q4 + (sl & 1) + (sl >> 1) * 8;
          const int row = R0 + rho16(slot);
          const bool ok = !tail || (jw + rho16(slot) < r.kv_len);
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
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t va[4];
              va[0] = e4m3x2_to_f16x2((uint16_t)(h2 ? (p_lo01 >> 16) : (p_lo01 & 0xffffu)));
              va[1] = e4m3x2_to_f16x2((uint16_t)(h2 ? (p_hi01 >> 16) : (p_hi01 & 0xffffu)));
              va[2] = e4m3x2_to_f16x2((uint16_t)(h2 ? (p_lo89 >> 16) : (p_lo89 & 0xffffu)));
              va[3] = e4m3x2_to_f16x2((uint16_t)(h2 ? (p_hi89 >> 16) : (p_hi89 & 0xffffu)));
#pragma unroll
              for (int ng = 0; ng < NG; ++ng)
                mma_f16(acc[4 * t2 + ip + h2][ng], va, pb[t2][ng][0], pb[t2][ng][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---------------- merge the eight warps' states ----------------
    if constexpr (FP8) {
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const float f = vref[i >> 2];
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
    // every thread: combined (M, L) of its heads, and its own scale factor
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
    named_bar_sync(1, nthr);  // red_ml is rewritten below
    // tree sum of the scaled accumulators (8 -> 4 -> 2 -> 1 warps), one head
    // group at a time through a [4][D][8] buffer; slot 0 ends as the result
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
      for (int half = 4; half >= 1; half >>= 1) {
        if (cw >= half && cw < 2 * half) {
          float* bp = red + (size_t)(cw - half) * D * 8;
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            *reinterpret_cast<float2*>(bp + drow(i, g) * 8 + 2 * q4) = make_float2(acc[i][ng][0], acc[i][ng][1]);
            *reinterpret_cast<float2*>(bp + drow(i, g + 8) * 8 + 2 * q4) = make_float2(acc[i][ng][2], acc[i][ng][3]);
          }
        }
        named_bar_sync(1, nthr);
        if (cw < half) {
          const float* bp = red + (size_t)cw * D * 8;
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            const float2 x = *reinterpret_cast<const float2*>(bp + drow(i, g) * 8 + 2 * q4);
            const float2 y = *reinterpret_cast<const float2*>(bp + drow(i, g + 8) * 8 + 2 * q4);
            acc[i][ng][0] += x.x; acc[i][ng][1] += x.y;
            acc[i][ng][2] += y.x; acc[i][ng][3] += y.y;
          }
        }
        named_bar_sync(1, nthr);
      }
      if (cw == 0) {
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          *reinterpret_cast<float2*>(red + drow(i, g) * 8 + 2 * q4) = make_float2(acc[i][ng][0], acc[i][ng][1]);
          *reinterpret_cast<float2*>(red + drow(i, g + 8) * 8 + 2 * q4) = make_float2(acc[i][ng][2], acc[i][ng][3]);
        }
        if (g == 0) {  // (M, L) of this head group into red_ml[0..7]
          red_ml[(2 * q4) * 2 + 0] = Mh[ng][0];
          red_ml[(2 * q4) * 2 + 1] = Lh[ng][0];
          red_ml[(2 * q4 + 1) * 2 + 0] = Mh[ng][1];
          red_ml[(2 * q4 + 1) * 2 + 1] = Lh[ng][1];
        }
      }
      named_bar_sync(1, nthr);
      // all consumer threads: write this head group (final O or a partial)
      const int nh = min(8, r.nrows - ng * 8);
      if (!split) {
        for (int idx = ctid; idx < nh * (D / 2); idx += nthr) {
          const int hh = idx / (D / 2), d = (idx % (D / 2)) * 2;
          const int h = r.h0 + ng * 8 + hh;
          float scl, lse;
          finish_head(a, h, red_ml[hh * 2], red_ml[hh * 2 + 1], &scl, &lse);
          uint16_t* o = a.out + r.qrow * a.out_stride + (int64_t)h * D + d;
          *reinterpret_cast<uint32_t*>(o) = pack_bf16(red[d * 8 + hh] * scl, red[(d + 1) * 8 + hh] * scl);
          if (a.lse && d == 0) {
            const int64_t li = a.layout == 1 ? r.qrow * a.QN + h : ((int64_t)r.b * a.QN + h) * a.S_q;
            a.lse[li] = lse;
          }
        }
      } else {
        const int slot = 2 * c + (first ? 0 : 1);
        float* pp = a.partials + (size_t)slot * kMaxGH * (D + 2);
        for (int idx = ctid; idx < nh * (D + 2); idx += nthr) {
          const int hh = idx / (D + 2), d = idx % (D + 2);
          const float v = d < D ? red[d * 8 + hh] : red_ml[hh * 2 + (d - D)];
          pp[(ng * 8 + hh) * (D + 2) + d] = v;
        }
        __threadfence();
      }
      named_bar_sync(1, nthr);
    }
    if (split) {
      // the last piece of a split unit folds all pieces in CTA order; pieces:
      // CTA cf (the one holding tile pu) and every later CTA up to cl whose
      // interval is non-empty (CTAs with empty intervals hold nothing)
      const int cf = find_cta(a.cta_begin, a.num_ctas, pu);
      const int cl = find_cta(a.cta_begin, a.num_ctas, pu1 - 1);
      int nseg = 1;
      for (int cc = cf + 1; cc <= cl; ++cc) nseg += a.cta_begin[cc] < a.cta_begin[cc + 1];
      if (ctid == 0) {
        const int prev = atomicAdd(&a.counters[u], 1);
        misc[1] = (prev == nseg - 1);
      }
      named_bar_sync(1, nthr);
      if (misc[1]) {
        __threadfence();
        for (int idx = ctid; idx < r.nrows * (D / 2); idx += nthr) {
          const int head = idx / (D / 2);
          const int d = (idx % (D / 2)) * 2;
          float M = -INFINITY;
          for (int cc = cf; cc <= cl; ++cc) {
            if (cc > cf && a.cta_begin[cc] == a.cta_begin[cc + 1]) continue;
            const int slot = 2 * cc + ((cc == cf && a.cta_begin[cc] < pu) ? 1 : 0);
            const float* pp = a.partials + (size_t)slot * kMaxGH * (D + 2) + head * (D + 2);
            M = fmaxf(M, __ldcg(pp + D));
          }
          const float Mu = M == -INFINITY ? 0.f : M;
          float L = 0.f, o0 = 0.f, o1 = 0.f;
          for (int cc = cf; cc <= cl; ++cc) {
            if (cc > cf && a.cta_begin[cc] == a.cta_begin[cc + 1]) continue;
            const int slot = 2 * cc + ((cc == cf && a.cta_begin[cc] < pu) ? 1 : 0);
            const float* pp = a.partials + (size_t)slot * kMaxGH * (D + 2) + head * (D + 2);
            const float mw = __ldcg(pp + D);
            if (mw == -INFINITY) continue;
            const float f = exp2f(mw - Mu);
            L += __ldcg(pp + D + 1) * f;
            o0 += __ldcg(pp + d) * f;
            o1 += __ldcg(pp + d + 1) * f;
          }
          const int h = r.h0 + head;
          float scl, lse;
          finish_head(a, h, M, L, &scl, &lse);
          uint16_t* o = a.out + r.qrow * a.out_stride + (int64_t)h * D + d;
          *reinterpret_cast<uint32_t*>(o) = pack_bf16(o0 * scl, o1 * scl);
          if (a.lse && d == 0) {
            const int64_t li = a.layout == 1 ? r.qrow * a.QN + h : ((int64_t)r.b * a.QN + h) * a.S_q;
            a.lse[li] = lse;
          }
        }
      }
      named_bar_sync(1, nthr);
    }
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

template <int D, bool FP8, int NG>
static cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap& tk,
                                   const CUtensorMap& tv, cudaStream_t s) {
  using Cfg = DecodeCfg<D, FP8>;
  auto kern = decode_kernel<D, FP8, NG>;
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
  kern<<<a.num_ctas, kThreads, Cfg::kSmem, s>>>(a, tk, tv);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                          int fp8, cudaStream_t s) {
  const bool two = a.GH > 8;
  if (fp8) return two ? launch_decode_t<128, true, 2>(a, tk, tv, s)
                      : launch_decode_t<128, true, 1>(a, tk, tv, s);
  if (a.D == 64) return two ? launch_decode_t<64, false, 2>(a, tk, tv, s)
                            : launch_decode_t<64, false, 1>(a, tk, tv, s);
  return two ? launch_decode_t<128, false, 2>(a, tk, tv, s)
             : launch_decode_t<128, false, 1>(a, tk, tv, s);
}

}  // namespace fia
