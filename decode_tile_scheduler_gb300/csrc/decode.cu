// decode.cu -- the incremental-inference branch of fused inference attention
// (query length 1; "aclnnFusedInferAttentionScoreV2": the IncreFlashAttention
// branch runs when the query S is 1) over a paged KV cache, plus its tile
// scheduler.
//
// Work unit: (batch b, KV head hk, head group hg) -- the up to 16 query heads
// of one GQA group that share KV head hk are packed as the M=16 rows of one
// mma.sync, so each KV page is read from HBM once for the whole group.  A unit
// owns the KV tiles (128 positions each) its query row can see.
//
// Scheduler (decode_schedule_kernel): cost(u) = visible tiles (>= 1; 0 when
// the batch has no query row); CTA c of n persistent CTAs owns the global tile
// interval [floor(c*total/n), floor((c+1)*total/n)) of the units laid end to
// end, so every CTA gets the same number of tiles within one.  A unit cut by a
// CTA boundary is a split-KV unit: every piece writes its (m, l, acc) partial
// and the last piece to finish folds all pieces in CTA order (deterministic).
//
// Decode kernel: one producer warp streams K and V pages with TMA (one box per
// 128-byte row slice; page rows come from block_table) into a ring of shared
// memory stages; four consumer warps each take 32 rows of every tile and run
// Q K^T, an online softmax in the exp2 domain and P V with mma.sync.  FP8 E4M3
// pages are converted to fp16 in registers (exact), the K tile scales are
// applied to the per-64-column partial scores and the V tile scales are folded
// into P, so the dequantised cache is never materialised.
#include "common.cuh"
#include "internal.h"

namespace fia {

namespace {

constexpr int kConsumers = 4;            // consumer warps
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kRowsPerWarp = kKvTile / kConsumers;  // 32

// Row permutation inside each group of 8 KV rows (see the bank-conflict note
// at the FP8 K loads): n -> pi(n) keeps pi(2q) = 2q and pi(2q+1) = 2q+5 mod 8.
__device__ __forceinline__ int pi8(int n) { return (n & 1) ? ((n + 4) & 7) : n; }

template <int D, bool FP8>
struct DecodeCfg {
  static constexpr int kNsub = FP8 ? 1 : D / 64;            // 128-byte slices per row
  static constexpr int kTileBytes = kNsub * kKvTile * 128;  // one of K or V
  static constexpr int kScaleBytes = FP8 ? kKvTile * (D / 64) * 4 : 0;
  static constexpr int kStageBytes = 2 * kTileBytes + 2 * kScaleBytes;
  static constexpr int kStages = FP8 ? 5 : (D == 128 ? 3 : 6);
  static constexpr int kQBytes = kHeadGroup * D * 2;
  static constexpr int kRedAccBytes = (kConsumers - 1) * kHeadGroup * D * 4;
  static constexpr int kRedMlBytes = kConsumers * kHeadGroup * 2 * 4;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffRedAcc = kOffQ + 2 * kQBytes;
  static constexpr int kOffRedMl = kOffRedAcc + kRedAccBytes;
  static constexpr int kOffBar = kOffRedMl + kRedMlBytes;
  static constexpr int kOffMisc = kOffBar + 8 * (2 * kStages + 4);
  static constexpr int kSmem = kOffMisc + 64 + 1024;  // + alignment slack
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
};

struct UnitInfo {
  int b, hk, hg, h0, nrows;
  int64_t qrow;      // token row of q/out
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
  r.h0 = r.hk * a.G + r.hg * kHeadGroup;
  r.nrows = min(kHeadGroup, a.G - r.hg * kHeadGroup);
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

// Bounded barrier wait; after the first time-out in the CTA every later wait
// returns at once, so a broken pipeline ends the kernel instead of hanging it.
__device__ __forceinline__ void wait_or_abort(uint64_t* bar, uint32_t parity, int* err,
                                              int* misc) {
  if (*reinterpret_cast<volatile int*>(misc)) return;
  if (!mbar_wait(bar, parity, err)) *reinterpret_cast<volatile int*>(misc) = 1;
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
  if (tid == 0) prefix[U] = total;
  for (int c = tid; c <= a.num_ctas; c += blockDim.x)
    beg[c] = (int64_t)c * total / a.num_ctas;
}

// ---------------------------------------------------------------------------
// decode kernel
// ---------------------------------------------------------------------------
template <int D, bool FP8>
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
  float* red_acc = reinterpret_cast<float*>(smem + Cfg::kOffRedAcc);
  float* red_ml = reinterpret_cast<float*>(smem + Cfg::kOffRedMl);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int64_t U = a.num_units;
  const int64_t g0 = a.cta_begin[c], g1 = a.cta_begin[c + 1];

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], FP8 ? 33 : 1);
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

  int64_t u0 = find_unit(a.unit_prefix, U, g0);

  if (warp == 0) {
    // ======================= producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
    }
    int it = 0, ucount = 0;
    for (int64_t u = u0; u < U && a.unit_prefix[u] < g1; u = next_unit(a.unit_prefix, U, u)) {
      const UnitInfo r = unit_info(a, u);
      const int64_t pu = a.unit_prefix[u];
      const int t_begin = (int)(max(g0, pu) - pu);
      const int t_end = (int)(min(g1, a.unit_prefix[u + 1]) - pu);
      // query rows of the group: one bulk copy
      {
        const int qs = ucount & 1;
        const uint32_t par = ((ucount >> 1) & 1) ^ 1;
        wait_or_abort(&qempty[qs], par, a.err, misc);
        if (lane == 0) {
          const uint32_t bytes = (uint32_t)(r.nrows * D * 2);
          mbar_arrive_expect_tx(&qfull[qs], bytes);
          bulk_load(smem + Cfg::kOffQ + qs * Cfg::kQBytes,
                    a.q + r.qrow * a.q_stride + (int64_t)r.h0 * D, bytes, &qfull[qs]);
        }
        ++ucount;
      }
      if (r.ntiles == 0) continue;
      for (int t = t_begin; t < t_end; ++t, ++it) {
        const int s = it % S;
        const uint32_t par = ((it / S) & 1) ^ 1;
        wait_or_abort(&empty[s], par, a.err, misc);
        uint8_t* st = smem + s * Cfg::kStageBytes;
        const int64_t j0 = (int64_t)(r.tile0 + t) * kKvTile;
        const int nrb = kKvTile / a.box_rows;
        int nvalid = 0;
        for (int rb = 0; rb < nrb; ++rb)
          if (j0 + (int64_t)rb * a.box_rows < r.kv_len) ++nvalid;
        if (lane == 0)
          mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * nvalid * Cfg::kNsub * a.box_rows * 128));
        __syncwarp();
        // one box per (row block, 128-byte slice, K|V)
        const int nbox = nrb * Cfg::kNsub * 2;
        for (int bx = lane; bx < nbox; bx += 32) {
          const int isv = bx & 1;
          const int sub = (bx >> 1) % Cfg::kNsub;
          const int rb = (bx >> 1) / Cfg::kNsub;
          const int64_t j = j0 + (int64_t)rb * a.box_rows;
          if (j >= r.kv_len) continue;
          const int64_t prow = phys_row(a, r.b, j);
          uint8_t* dst = st + isv * Cfg::kTileBytes + sub * (kKvTile * 128) + rb * a.box_rows * 128;
          const int col = FP8 ? r.hk * D : r.hk * D + sub * 64;
          tma_load_2d(dst, isv ? &tv : &tk, &full[s], col, (int)prow);
        }
        if constexpr (FP8) {
          constexpr int NT = D / 64;
          float* ks = reinterpret_cast<float*>(st + 2 * Cfg::kTileBytes);
          float* vs = ks + kKvTile * NT;
          for (int rr = lane; rr < kKvTile; rr += 32) {
            const int64_t j = j0 + rr;
            if (j < r.kv_len) {
              const int64_t off = (phys_row(a, r.b, j) * a.KVN + r.hk) * NT;
#pragma unroll
              for (int t2 = 0; t2 < NT; t2 += 2) {
                cp_async_8(ks + rr * NT + t2, a.k_scale + off + t2);
                cp_async_8(vs + rr * NT + t2, a.v_scale + off + t2);
              }
            }
          }
          cp_async_arrive_noinc(&full[s]);
        }
      }
    }
    return;
  }

  // ======================= consumers =======================
  const int cw = warp - 1;        // 0..3
  const int g = lane >> 2;        // mma row group
  const int q4 = lane & 3;        // thread in quad
  const int wrow0 = cw * kRowsPerWarp;
  const uint32_t smem_base = smem_u32(smem);
  constexpr int KS = D / 16;      // k-steps over D
  constexpr int NDT = D / 8;      // n-tiles over D

  int it = 0, ucount = 0;
  for (int64_t u = u0; u < U && a.unit_prefix[u] < g1; u = next_unit(a.unit_prefix, U, u)) {
    const UnitInfo r = unit_info(a, u);
    const int64_t pu = a.unit_prefix[u], pu1 = a.unit_prefix[u + 1];
    const int t_begin = (int)(max(g0, pu) - pu);
    const int t_end = (int)(min(g1, pu1) - pu);
    const bool split = (pu < g0) || (pu1 > g1);

    // ---- Q fragments (A operand), rows = heads of the group ----
    uint32_t qa[KS][4];
    {
      const int qs = ucount & 1;
      const uint32_t par = (ucount >> 1) & 1;
      wait_or_abort(&qfull[qs], par, a.err, misc);
      const uint16_t* qsm = reinterpret_cast<const uint16_t*>(smem + Cfg::kOffQ + qs * Cfg::kQBytes);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        if constexpr (!FP8) {
          const int d0 = kk * 16 + 2 * q4;
          qa[kk][0] = g < r.nrows ? *reinterpret_cast<const uint32_t*>(qsm + g * D + d0) : 0u;
          qa[kk][1] = g + 8 < r.nrows ? *reinterpret_cast<const uint32_t*>(qsm + (g + 8) * D + d0) : 0u;
          qa[kk][2] = g < r.nrows ? *reinterpret_cast<const uint32_t*>(qsm + g * D + d0 + 8) : 0u;
          qa[kk][3] = g + 8 < r.nrows ? *reinterpret_cast<const uint32_t*>(qsm + (g + 8) * D + d0 + 8) : 0u;
        } else {
          // k-step kk = 4*tile + j covers d = 64*tile + 16*q + 4*j + {0..3}:
          // slots 2q,2q+1 <- first two, slots 2q+8,2q+9 <- last two
          const int d0 = (kk >> 2) * 64 + 16 * q4 + 4 * (kk & 3);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int row = g + 8 * hh;
            if (row < r.nrows) {
              const uint2 v = *reinterpret_cast<const uint2*>(qsm + row * D + d0);
              const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
              const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
              const float2 flo = __bfloat1622float2(lo), fhi = __bfloat1622float2(hi);
              qa[kk][hh] = pack_f16(flo.x, flo.y);
              qa[kk][2 + hh] = pack_f16(fhi.x, fhi.y);
            } else {
              qa[kk][hh] = 0u;
              qa[kk][2 + hh] = 0u;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qs]);
      ++ucount;
    }

    float acc[NDT][4];
#pragma unroll
    for (int i = 0; i < NDT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY};  // rows g, g+8 (exp2 domain)
    float l_r[2] = {0.f, 0.f};
    float vref[2] = {1.f, 1.f};             // FP8: V scale reference per d-tile

    const int ntile_here = r.ntiles == 0 ? 0 : (t_end - t_begin);
    for (int tt = 0; tt < ntile_here; ++tt, ++it) {
      const int t = t_begin + tt;
      const int s = it % S;
      wait_or_abort(&full[s], (it / S) & 1, a.err, misc);
      const uint32_t st = smem_base + s * Cfg::kStageBytes;
      const int64_t j0 = (int64_t)(r.tile0 + t) * kKvTile + wrow0;  // first row of this warp
      const bool edge = (j0 < r.lo) || (j0 + kRowsPerWarp - 1 > r.hi);
      const bool tail = (j0 + kRowsPerWarp > r.kv_len);

      // ---------------- S = Q K^T (M=16 heads, N=32 rows) ----------------
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      if constexpr (!FP8) {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int sub = kk >> 2;  // 64-wide slice
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            // matrices: (nt=2np, lo8), (2np, hi8), (2np+1, lo8), (2np+1, hi8)
            const int mi = lane >> 3;
            const int nt = 2 * np + (mi >> 1);
            const int row = wrow0 + nt * 8 + pi8(lane & 7);
            const int chunk = (kk & 3) * 2 + (mi & 1);
            const uint32_t addr = st + sub * (kKvTile * 128) + sw128(row, chunk);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma_bf16(sc[2 * np], qa[kk], b0, b1);
            mma_bf16(sc[2 * np + 1], qa[kk], b2, b3);
          }
        }
      } else {
        constexpr int NT = D / 64;
        float s2[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int row = wrow0 + nt * 8 + pi8(g);
#pragma unroll
          for (int tile = 0; tile < NT; ++tile) {
            const uint4 w = *reinterpret_cast<const uint4*>(
                smem + s * Cfg::kStageBytes + sw128(row, tile * 4 + q4));
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t b0 = e4m3x2_to_f16x2((uint16_t)(wv[j] & 0xffffu));
              const uint32_t b1 = e4m3x2_to_f16x2((uint16_t)(wv[j] >> 16));
              if (tile == 0) mma_f16(sc[nt], qa[tile * 4 + j], b0, b1);
              else mma_f16(s2[nt], qa[tile * 4 + j], b0, b1);
            }
          }
        }
        // per-row K scales of the two 64-column tiles
        const float* ks = reinterpret_cast<const float*>(smem + s * Cfg::kStageBytes + 2 * Cfg::kTileBytes);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int rrow = wrow0 + nt * 8 + pi8(2 * q4 + e);
            float k0 = ks[rrow * NT + 0], k1 = ks[rrow * NT + 1];
            if (tail && (j0 - wrow0 + rrow >= r.kv_len)) { k0 = 0.f; k1 = 0.f; }
            sc[nt][e] = sc[nt][e] * k0 + s2[nt][e] * k1;
            sc[nt][2 + e] = sc[nt][2 + e] * k0 + s2[nt][2 + e] * k1;
          }
        }
      }

      // ---------------- mask + online softmax (exp2 domain) ----------------
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = sc[nt][e] * a.scale_log2;
          if (edge || tail) {
            const int64_t j = j0 + nt * 8 + pi8(2 * q4 + (e & 1));
            if (j < r.lo || j > r.hi) x = -INFINITY;
          }
          sc[nt][e] = x;
          mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
        mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
      }
      float corr[2], mu[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float mn = fmaxf(m_r[hh], mx[hh]);
        mu[hh] = mn == -INFINITY ? 0.f : mn;
        corr[hh] = m_r[hh] == -INFINITY ? 0.f : fast_exp2(m_r[hh] - mu[hh]);
        m_r[hh] = mn;
      }
      float psum[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pv = fast_exp2(sc[nt][e] - mu[e >> 1]);
          sc[nt][e] = pv;
          psum[e >> 1] += pv;
        }
      }
      l_r[0] = l_r[0] * corr[0] + psum[0];
      l_r[1] = l_r[1] * corr[1] + psum[1];

      // ---------------- O += P V ----------------
      if constexpr (!FP8) {
#pragma unroll
        for (int i = 0; i < NDT; ++i) {
          acc[i][0] *= corr[0];
          acc[i][1] *= corr[0];
          acc[i][2] *= corr[1];
          acc[i][3] *= corr[1];
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          uint32_t pa[4];
          pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
          pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
          pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
          pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
          // rows of this k-step held by the thread (for zeroing past kv_len)
          bool z0 = false, z1 = false, z2 = false, z3 = false;
          if (tail) {
            const int64_t jb = j0 + kk * 16;
            z0 = jb + pi8(2 * q4) >= r.kv_len;
            z1 = jb + pi8(2 * q4 + 1) >= r.kv_len;
            z2 = jb + 8 + pi8(2 * q4) >= r.kv_len;
            z3 = jb + 8 + pi8(2 * q4 + 1) >= r.kv_len;
          }
#pragma unroll
          for (int ndp = 0; ndp < NDT / 2; ++ndp) {
            // matrices: (rows 0-7, d-chunk 2ndp), (rows 8-15, 2ndp),
            //           (rows 0-7, 2ndp+1), (rows 8-15, 2ndp+1)
            const int mi = lane >> 3;
            const int row = wrow0 + kk * 16 + (mi & 1) * 8 + pi8(lane & 7);
            const int dchunk = 2 * ndp + (mi >> 1);
            const uint32_t addr = st + Cfg::kTileBytes + (dchunk >> 3) * (kKvTile * 128) +
                                  sw128(row, dchunk & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(addr, b0, b1, b2, b3);
            if (tail) {
              if (z0) { b0 &= 0xffff0000u; b2 &= 0xffff0000u; }
              if (z1) { b0 &= 0x0000ffffu; b2 &= 0x0000ffffu; }
              if (z2) { b1 &= 0xffff0000u; b3 &= 0xffff0000u; }
              if (z3) { b1 &= 0x0000ffffu; b3 &= 0x0000ffffu; }
            }
            mma_bf16(acc[2 * ndp], pa, b0, b1);
            mma_bf16(acc[2 * ndp + 1], pa, b2, b3);
          }
        }
      } else {
        constexpr int NT = D / 64;
        static_assert(NT == 2, "FP8 decode is built for D = 128");
        const float* vs = reinterpret_cast<const float*>(smem + s * Cfg::kStageBytes +
                                                         2 * Cfg::kTileBytes + Cfg::kScaleBytes);
        // V scales of the 8 rows this thread feeds (2 k-steps x 4 slots)
        float vsc[2][4][2];
        float vmax[2] = {0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            const int rrow = wrow0 + kk * 16 + (sl >> 1) * 8 + pi8(2 * q4 + (sl & 1));
            const bool ok = !tail || (j0 - wrow0 + rrow < r.kv_len);
            const float2 v2 = *reinterpret_cast<const float2*>(vs + rrow * NT);
            vsc[kk][sl][0] = ok ? v2.x : 0.f;
            vsc[kk][sl][1] = ok ? v2.y : 0.f;
            vmax[0] = fmaxf(vmax[0], vsc[kk][sl][0]);
            vmax[1] = fmaxf(vmax[1], vsc[kk][sl][1]);
          }
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          vmax[t2] = fmaxf(vmax[t2], __shfl_xor_sync(0xffffffffu, vmax[t2], 1));
          vmax[t2] = fmaxf(vmax[t2], __shfl_xor_sync(0xffffffffu, vmax[t2], 2));
          if (!(vmax[t2] > 0.f)) vmax[t2] = vref[t2];  // all-zero scales: keep reference
        }
        // rescale acc by the softmax correction and the change of V reference
        float f[2][2];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          const float ratio = vref[t2] / vmax[t2];
          f[t2][0] = corr[0] * ratio;
          f[t2][1] = corr[1] * ratio;
          vref[t2] = vmax[t2];
        }
#pragma unroll
        for (int i = 0; i < NDT; ++i) {
          const int t2 = i >> 3;
          acc[i][0] *= f[t2][0];
          acc[i][1] *= f[t2][0];
          acc[i][2] *= f[t2][1];
          acc[i][3] *= f[t2][1];
        }
        const float inv0 = 1.f / vref[0], inv1 = 1.f / vref[1];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          // P scaled per d-tile: slot sl -> (n-tile 2kk + sl/2, col 2q + sl%2)
          uint32_t pa[2][4];
#pragma unroll
          for (int t2 = 0; t2 < 2; ++t2) {
            const float iv = t2 ? inv1 : inv0;
            pa[t2][0] = pack_f16(sc[2 * kk][0] * vsc[kk][0][t2] * iv, sc[2 * kk][1] * vsc[kk][1][t2] * iv);
            pa[t2][1] = pack_f16(sc[2 * kk][2] * vsc[kk][0][t2] * iv, sc[2 * kk][3] * vsc[kk][1][t2] * iv);
            pa[t2][2] = pack_f16(sc[2 * kk + 1][0] * vsc[kk][2][t2] * iv, sc[2 * kk + 1][1] * vsc[kk][3][t2] * iv);
            pa[t2][3] = pack_f16(sc[2 * kk + 1][2] * vsc[kk][2][t2] * iv, sc[2 * kk + 1][3] * vsc[kk][3][t2] * iv);
          }
          // V codes: 4 rows (slots 2q, 2q+1, 2q+8, 2q+9), 8 bytes per d-tile
          // at d = 64*tile + 8*g .. +7  ->  n-tile 8*tile + e, column g
          const uint8_t* vt = smem + s * Cfg::kStageBytes + Cfg::kTileBytes;
          uint2 w[4][2];
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            const int rrow = wrow0 + kk * 16 + (sl >> 1) * 8 + pi8(2 * q4 + (sl & 1));
            const bool ok = !tail || (j0 - wrow0 + rrow < r.kv_len);
#pragma unroll
            for (int t2 = 0; t2 < 2; ++t2) {
              // d-tile t2: bytes 64*t2 + 8g .. +7 -> chunk 4*t2 + g/2, half g&1
              const uint32_t off = sw128(rrow, 4 * t2 + (g >> 1)) + 8 * (g & 1);
              uint2 x = *reinterpret_cast<const uint2*>(vt + off);
              if (!ok) { x.x = 0u; x.y = 0u; }
              w[sl][t2] = x;
            }
          }
#pragma unroll
          for (int t2 = 0; t2 < 2; ++t2) {
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              // bytes e, e+1 of rows (slot 2q, 2q+1) and (2q+8, 2q+9)
              const uint32_t lo01 = e < 4 ? w[0][t2].x : w[0][t2].y;
              const uint32_t hi01 = e < 4 ? w[1][t2].x : w[1][t2].y;
              const uint32_t lo89 = e < 4 ? w[2][t2].x : w[2][t2].y;
              const uint32_t hi89 = e < 4 ? w[3][t2].x : w[3][t2].y;
              const int sh = (e & 3);
              // select byte sh and sh+1 of each word: (A[sh], B[sh], A[sh+1], B[sh+1])
              const uint32_t sel = (uint32_t)(sh | (4 + sh) << 4 | (sh + 1) << 8 | (4 + sh + 1) << 12);
              const uint32_t p01 = __byte_perm(lo01, hi01, sel);
              const uint32_t p89 = __byte_perm(lo89, hi89, sel);
              const uint32_t b0a = e4m3x2_to_f16x2((uint16_t)(p01 & 0xffffu));
              const uint32_t b0b = e4m3x2_to_f16x2((uint16_t)(p01 >> 16));
              const uint32_t b1a = e4m3x2_to_f16x2((uint16_t)(p89 & 0xffffu));
              const uint32_t b1b = e4m3x2_to_f16x2((uint16_t)(p89 >> 16));
              mma_f16(acc[8 * t2 + e], pa[t2], b0a, b1a);
              mma_f16(acc[8 * t2 + e + 1], pa[t2], b0b, b1b);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---------------- merge the four warps' states ----------------
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      l_r[hh] += __shfl_xor_sync(0xffffffffu, l_r[hh], 1);
      l_r[hh] += __shfl_xor_sync(0xffffffffu, l_r[hh], 2);
    }
    if constexpr (FP8) {
      // bring acc back to absolute V units
#pragma unroll
      for (int i = 0; i < NDT; ++i) {
        const float f = vref[i >> 3];
        acc[i][0] *= f; acc[i][1] *= f; acc[i][2] *= f; acc[i][3] *= f;
      }
    }
    if (q4 == 0) {
      red_ml[(cw * kHeadGroup + g) * 2 + 0] = m_r[0];
      red_ml[(cw * kHeadGroup + g) * 2 + 1] = l_r[0];
      red_ml[(cw * kHeadGroup + g + 8) * 2 + 0] = m_r[1];
      red_ml[(cw * kHeadGroup + g + 8) * 2 + 1] = l_r[1];
    }
    named_bar_sync(1, 32 * kConsumers);
    float fac[2], Mrow[2], Lrow[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = g + 8 * hh;
      float M = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < kConsumers; ++w2) M = fmaxf(M, red_ml[(w2 * kHeadGroup + row) * 2]);
      float L = 0.f;
      const float Mu = M == -INFINITY ? 0.f : M;
#pragma unroll
      for (int w2 = 0; w2 < kConsumers; ++w2) {
        const float mw = red_ml[(w2 * kHeadGroup + row) * 2];
        const float lw = red_ml[(w2 * kHeadGroup + row) * 2 + 1];
        L += mw == -INFINITY ? 0.f : lw * exp2f(mw - Mu);
      }
      Mrow[hh] = M;
      Lrow[hh] = L;
      fac[hh] = m_r[hh] == -INFINITY ? 0.f : exp2f(m_r[hh] - Mu);
    }
    // d index of accumulator element (n-tile i, column 2q+e)
    auto dcol = [&](int i, int e) -> int {
      if constexpr (!FP8) return i * 8 + 2 * q4 + e;
      else return (i >> 3) * 64 + 8 * (2 * q4 + e) + (i & 7);
    };
    if (cw > 0) {
      float* ra = red_acc + (size_t)(cw - 1) * kHeadGroup * D;
#pragma unroll
      for (int i = 0; i < NDT; ++i)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (g < r.nrows) ra[g * D + dcol(i, e)] = acc[i][e] * fac[0];
          if (g + 8 < r.nrows) ra[(g + 8) * D + dcol(i, e)] = acc[i][2 + e] * fac[1];
        }
    }
    named_bar_sync(1, 32 * kConsumers);
    if (cw == 0) {
#pragma unroll
      for (int i = 0; i < NDT; ++i)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = dcol(i, e);
          float x0 = acc[i][e] * fac[0], x1 = acc[i][2 + e] * fac[1];
#pragma unroll
          for (int w2 = 0; w2 < kConsumers - 1; ++w2) {
            const float* ra = red_acc + (size_t)w2 * kHeadGroup * D;
            if (g < r.nrows) x0 += ra[g * D + d];
            if (g + 8 < r.nrows) x1 += ra[(g + 8) * D + d];
          }
          acc[i][e] = x0;
          acc[i][2 + e] = x1;
        }
      if (!split) {
        // finalize: sink, normalise, write O (bf16) and lse
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = g + 8 * hh;
          if (row >= r.nrows) continue;
          const int h = r.h0 + row;
          float M = Mrow[hh], L = Lrow[hh], scl = 0.f, lse = INFINITY;
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
          uint16_t* o = a.out + r.qrow * a.out_stride + (int64_t)h * D;
#pragma unroll
          for (int i = 0; i < NDT; ++i) {
            if constexpr (!FP8) {
              const uint32_t v = pack_bf16(acc[i][2 * hh] * scl, acc[i][2 * hh + 1] * scl);
              *reinterpret_cast<uint32_t*>(o + dcol(i, 0)) = v;
            } else {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                __nv_bfloat16 bv = __float2bfloat16_rn(acc[i][2 * hh + e] * scl);
                o[dcol(i, e)] = *reinterpret_cast<uint16_t*>(&bv);
              }
            }
          }
          if (a.lse && q4 == 0) {
            const int64_t li = a.layout == 1 ? r.qrow * a.QN + h : ((int64_t)r.b * a.QN + h) * a.S_q;
            a.lse[li] = lse;
          }
        }
      } else {
        // partial: slot 2c for the CTA's first unit, 2c+1 otherwise
        const int slot = 2 * c + (u == u0 ? 0 : 1);
        float* pp = a.partials + (size_t)slot * kHeadGroup * (D + 2);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = g + 8 * hh;
          if (row >= r.nrows) continue;
#pragma unroll
          for (int i = 0; i < NDT; ++i)
#pragma unroll
            for (int e = 0; e < 2; ++e) pp[row * (D + 2) + dcol(i, e)] = acc[i][2 * hh + e];
          if (q4 == 0) {
            pp[row * (D + 2) + D] = Mrow[hh];
            pp[row * (D + 2) + D + 1] = Lrow[hh];
          }
        }
        __threadfence();
      }
    }
    named_bar_sync(1, 32 * kConsumers);
    if (split) {
      // the last piece of a split unit folds all pieces in CTA order
      // pieces: CTA cf (the one holding tile pu) and every later CTA up to cl
      // whose interval is non-empty (CTAs with empty intervals hold nothing)
      const int cf = find_cta(a.cta_begin, a.num_ctas, pu);
      const int cl = find_cta(a.cta_begin, a.num_ctas, pu1 - 1);
      int nseg = 1;
      for (int cc = cf + 1; cc <= cl; ++cc) nseg += a.cta_begin[cc] < a.cta_begin[cc + 1];
      if (tid == 32) {
        const int prev = atomicAdd(&a.counters[u], 1);
        misc[1] = (prev == nseg - 1);
      }
      named_bar_sync(1, 32 * kConsumers);
      if (misc[1]) {
        __threadfence();
        const int ctid = tid - 32;
        for (int idx = ctid; idx < r.nrows * (D / 2); idx += 32 * kConsumers) {
          const int row = idx / (D / 2);
          const int d = (idx % (D / 2)) * 2;
          float M = -INFINITY;
          for (int cc = cf; cc <= cl; ++cc) {
            if (cc > cf && a.cta_begin[cc] == a.cta_begin[cc + 1]) continue;
            const int slot = 2 * cc + ((cc == cf && a.cta_begin[cc] < pu) ? 1 : 0);
            const float* pp = a.partials + (size_t)slot * kHeadGroup * (D + 2) + row * (D + 2);
            M = fmaxf(M, __ldcg(pp + D));
          }
          const float Mu = M == -INFINITY ? 0.f : M;
          float L = 0.f, o0 = 0.f, o1 = 0.f;
          for (int cc = cf; cc <= cl; ++cc) {
            if (cc > cf && a.cta_begin[cc] == a.cta_begin[cc + 1]) continue;
            const int slot = 2 * cc + ((cc == cf && a.cta_begin[cc] < pu) ? 1 : 0);
            const float* pp = a.partials + (size_t)slot * kHeadGroup * (D + 2) + row * (D + 2);
            const float mw = __ldcg(pp + D);
            if (mw == -INFINITY) continue;
            const float f = exp2f(mw - Mu);
            L += __ldcg(pp + D + 1) * f;
            o0 += __ldcg(pp + d) * f;
            o1 += __ldcg(pp + d + 1) * f;
          }
          const int h = r.h0 + row;
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
          uint16_t* o = a.out + r.qrow * a.out_stride + (int64_t)h * D + d;
          *reinterpret_cast<uint32_t*>(o) = pack_bf16(o0 * scl, o1 * scl);
          if (a.lse && d == 0) {
            const int64_t li = a.layout == 1 ? r.qrow * a.QN + h : ((int64_t)r.b * a.QN + h) * a.S_q;
            a.lse[li] = lse;
          }
        }
      }
      named_bar_sync(1, 32 * kConsumers);
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

template <int D, bool FP8>
static cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap& tk,
                                   const CUtensorMap& tv, cudaStream_t s) {
  using Cfg = DecodeCfg<D, FP8>;
  auto kern = decode_kernel<D, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<a.num_ctas, kThreads, Cfg::kSmem, s>>>(a, tk, tv);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                          int fp8, cudaStream_t s) {
  if (fp8) return launch_decode_t<128, true>(a, tk, tv, s);
  if (a.D == 64) return launch_decode_t<64, false>(a, tk, tv, s);
  return launch_decode_t<128, false>(a, tk, tv, s);
}

}  // namespace fia
