// sparse.cu -- shared-KV sparse attention ("kv_quant_sparse_attn_sharedkv":
// O = softmax(Q K~^T * softmax_scale) V~ with K~ = V~; "sparse_flash_mla":
// SWA, CSA and HCA modes and the metadata pre-step), bf16 KV.
//
// K~ of a query row is the band window of the original KV followed by the
// compressed rows (the listed top-k indices for CSA, every causally visible
// compressed row for HCA).  It is cut into fixed chunks of kChunk logical
// positions; the metadata kernel balances the (query row, chunk) items over
// the CTAs; the attention kernel gathers each chunk's rows with one bulk copy
// per row (the index -> block_table -> pool row indirection happens in the
// kernel), computes the chunk's (m, l, acc) for all heads with mma.sync, and
// the combine kernel folds the chunks of a row in chunk order and applies the
// sink.  Chunk boundaries do not depend on the rest of the batch, so results
// are batch invariant as well as deterministic.
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace fia {

namespace {

constexpr int kChunk = 64;          // K~ rows per item
constexpr int kSThreads = 256;      // 8 warps: 4 head groups of 16 x 2 halves of D
constexpr int kHeadsPerCta = 64;
constexpr int kMdCtaBase = 16;      // metadata: CTA begins from this entry

struct SparseRow {
  int b;
  int64_t i, q_len, S2, p;
  int ncmp_vis;  // visible compressed rows (before the top-k cap)
  int nchunks;
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
  const int64_t vis = (r.p + 1) >= 0 ? (r.p + 1) / a.cmp_ratio : 0;
  r.ncmp_vis = (int)vis;
  int64_t kc = 0;
  if (a.mode == 1) kc = min(vis, (int64_t)a.K2);
  else if (a.mode == 2) kc = vis;
  const int64_t W = (int64_t)a.win_left + a.win_right + 1;
  r.nchunks = (int)((W + kChunk - 1) / kChunk + (kc + kChunk - 1) / kChunk);
  return r;
}

}  // namespace

// ---------------------------------------------------------------------------
// metadata: per-row chunk counts -> balanced (row, chunk) begins of every CTA
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) sparse_metadata_kernel(const SparseArgs a, int32_t* md) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nthr = blockDim.x;
  const int n = a.num_ctas;
  for (int k = tid; k < 1024; k += nthr) md[k] = 0;
  // pass 1: total number of chunks
  if (tid == 0) carry = 0;
  __syncthreads();
  int64_t part = 0;
  for (int64_t u = tid; u < a.rows; u += nthr) part += sparse_row(a, u).nchunks;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) atomicAdd(reinterpret_cast<unsigned long long*>(&carry), (unsigned long long)part);
  __syncthreads();
  const int64_t total = carry;
  __syncthreads();
  // pass 2: running prefix; every row writes the begins that fall inside it
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < a.rows; base += nthr) {
    const int64_t u = base + tid;
    const int64_t nch = u < a.rows ? sparse_row(a, u).nchunks : 0;
    int64_t x = nch;
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
    const int64_t pre = carry + (wid ? warp_sums[wid - 1] : 0) + x - nch;
    if (u < a.rows && nch > 0 && total > 0) {
      // CTAs c with floor(c * total / n) in [pre, pre + nch)
      int64_t c = (pre * n + total - 1) / total;
      for (; c < n; ++c) {
        const int64_t g = c * total / n;
        if (g >= pre + nch) break;
        md[kMdCtaBase + 2 * c] = (int32_t)u;
        md[kMdCtaBase + 2 * c + 1] = (int32_t)(g - pre);
      }
    }
    __syncthreads();
    if (tid == nthr - 1) carry = pre + nch;
    __syncthreads();
  }
  if (tid == 0) {
    md[0] = 0x46534D31;
    md[1] = n;
    md[2] = (int32_t)a.rows;
    md[3] = kChunk;
    md[4] = (int32_t)total;
    md[5] = a.B;
    md[6] = a.N1;
    md[7] = a.K2;
    md[8] = a.cmp_ratio;
    md[9] = a.win_left;
    md[10] = a.win_right;
    md[11] = a.mode;
    md[kMdCtaBase + 2 * n] = (int32_t)a.rows;
    md[kMdCtaBase + 2 * n + 1] = 0;
    if (total == 0)
      for (int c = 0; c < n; ++c) {
        md[kMdCtaBase + 2 * c] = (int32_t)a.rows;
        md[kMdCtaBase + 2 * c + 1] = 0;
      }
  }
}

// ---------------------------------------------------------------------------
// attention over one (row, chunk) item at a time
// ---------------------------------------------------------------------------
template <int D>
struct SparseCfg {
  static constexpr int kRowBytes = D * 2 + 16;  // padded: ldmatrix rows hit distinct banks
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kHeadsPerCta * kRowBytes;
  static constexpr int kOffS = kOffK + kChunk * kRowBytes;          // [8 warps][16][64] fp32
  static constexpr int kOffRows = kOffS + 8 * 16 * kChunk * 4;     // [64] int64 pool offsets
  static constexpr int kOffBar = kOffRows + kChunk * 8;
  static constexpr int kOffMisc = kOffBar + 16;
  static constexpr int kSmem = kOffMisc + 64;
  static_assert(kSmem <= 232448, "shared memory");
};

template <int D>
__global__ void __launch_bounds__(kSThreads, 1)
    sparse_attn_kernel(const SparseArgs a, const int32_t* __restrict__ md) {
  using Cfg = SparseCfg<D>;
  constexpr int DH = D / 2;      // d range of one warp
  constexpr int KS = DH / 16;    // k-steps of Q K^T over a half
  constexpr int NT = DH / 8;     // n-tiles of P V over a half
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Cfg::kOffBar);
  int64_t* rowoff = reinterpret_cast<int64_t*>(sm + Cfg::kOffRows);
  int* misc = reinterpret_cast<int*>(sm + Cfg::kOffMisc);
  float* sx = reinterpret_cast<float*>(sm + Cfg::kOffS);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q4 = lane & 3;
  const int hgrp = warp & 3, half = warp >> 2;  // 16 heads x D/2
  const int c = blockIdx.x;
  const int head0 = blockIdx.y * kHeadsPerCta;
  const int nheads = min(kHeadsPerCta, a.N1 - head0);
  if (md[0] != 0x46534D31 || md[1] != a.num_ctas || md[2] != (int32_t)a.rows ||
      md[5] != a.B || md[6] != a.N1 || md[7] != a.K2) {
    if (tid == 0) atomicExch(a.err, 2);
    return;
  }
  int64_t u = md[kMdCtaBase + 2 * c];
  int ch = md[kMdCtaBase + 2 * c + 1];
  const int64_t u_end = md[kMdCtaBase + 2 * c + 2];
  const int ch_end = md[kMdCtaBase + 2 * c + 3];
  if (tid == 0) {
    mbar_init(bar, 1);
    misc[0] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const uint32_t sq = smem_u32(sm + Cfg::kOffQ), sk = smem_u32(sm + Cfg::kOffK);
  const int64_t W = (int64_t)a.win_left + a.win_right + 1;
  int phase = 0;
  while (u < u_end || (u == u_end && ch < ch_end)) {
    const SparseRow r = sparse_row(a, u);
    if (ch >= r.nchunks) {  // next row
      ++u;
      ch = 0;
      continue;
    }
    // ---- first -1 of the index list up to this chunk (CSA scan rule) ----
    int first_neg = 0x7fffffff;
    if (a.mode == 1) {
      const int lim = (int)min((int64_t)a.K2, (int64_t)(ch + 1) * kChunk - W);
      const int32_t* ix = a.cmp_sparse_indices + u * (int64_t)a.K2;
      for (int t = tid; t < lim; t += kSThreads)
        if (ix[t] < 0) first_neg = min(first_neg, t);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) first_neg = min(first_neg, __shfl_xor_sync(0xffffffffu, first_neg, o));
      if (lane == 0) misc[1 + warp] = first_neg;
      __syncthreads();
      first_neg = misc[1];
      for (int w2 = 1; w2 < 8; ++w2) first_neg = min(first_neg, misc[1 + w2]);
    }
    // ---- gather: pool offsets of the chunk's 64 K~ rows (-1: no row) ----
    if (tid < kChunk) {
      const int64_t pos = (int64_t)ch * kChunk + tid;
      int64_t off = -1;
      if (pos < W) {
        const int64_t j = r.p - a.win_left + pos;
        if (j >= 0 && j < r.S2) {
          const int64_t blk = a.ori_block_table[(int64_t)r.b * a.ori_max_blocks + j / a.ori_block_size];
          off = (blk * a.ori_block_size + j % a.ori_block_size) * (int64_t)D;
        }
      } else if (a.mode != 0) {
        const int64_t t = pos - W;
        int64_t idx = -1;
        if (a.mode == 1) {
          if (t < a.K2 && t < first_neg) idx = a.cmp_sparse_indices[u * (int64_t)a.K2 + t];
        } else {
          idx = t;
        }
        if (idx >= 0 && idx < r.ncmp_vis) {
          const int64_t blk = a.cmp_block_table[(int64_t)r.b * a.cmp_max_blocks + idx / a.cmp_block_size];
          // compressed rows are flagged by bit 62 so the copy picks the right pool
          off = ((blk * a.cmp_block_size + idx % a.cmp_block_size) * (int64_t)D) | (1ll << 62);
        }
      }
      rowoff[tid] = off;
    }
    __syncthreads();
    // ---- bulk copies: Q rows of the head group and the valid K~ rows ----
    if (warp == 0) {
      // earlier generic-proxy reads and zero-fills of these rows precede the
      // async-proxy copies below
      fence_proxy_async_smem();
      int nvalid = 0;
      for (int rr = 0; rr < kChunk; ++rr) nvalid += rowoff[rr] >= 0;
      if (lane == 0)
        mbar_arrive_expect_tx(bar, (uint32_t)((nheads + nvalid) * D * 2));
      __syncwarp();
      const uint16_t* qrow = a.q + (u * a.N1 + head0) * (int64_t)D;
      for (int h = lane; h < nheads; h += 32)
        bulk_load(sm + Cfg::kOffQ + h * Cfg::kRowBytes, qrow + (int64_t)h * D, D * 2, bar);
      for (int rr = lane; rr < kChunk; rr += 32) {
        const int64_t off = rowoff[rr];
        if (off >= 0) {
          const uint16_t* src = (off >> 62) ? a.cmp_kv + (off & ((1ll << 62) - 1)) : a.ori_kv + off;
          bulk_load(sm + Cfg::kOffK + rr * Cfg::kRowBytes, src, D * 2, bar);
        }
      }
    } else {
      // zero the rows that hold no K~ row (and head rows past N1)
      for (int x = tid - 32; x < kChunk * (D / 8); x += kSThreads - 32) {
        const int rr = x / (D / 8), k = x % (D / 8);
        if (rowoff[rr] < 0)
          *reinterpret_cast<uint4*>(sm + Cfg::kOffK + rr * Cfg::kRowBytes + k * 16) = make_uint4(0, 0, 0, 0);
      }
      for (int x = tid - 32; x < (kHeadsPerCta - nheads) * (D / 8); x += kSThreads - 32) {
        const int h = nheads + x / (D / 8), k = x % (D / 8);
        *reinterpret_cast<uint4*>(sm + Cfg::kOffQ + h * Cfg::kRowBytes + k * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    if (!mbar_wait(bar, phase, a.err)) misc[0] = 1;
    phase ^= 1;
    __syncthreads();

    // ---- partial S = Q K~^T over this warp's half of D (16 heads x 64 rows) ----
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int d0 = half * DH + kk * 16;
      uint32_t qa[4];
      {
        // A: rows = heads (16), k = d: matrices (h 0-7, d lo), (h 8-15, d lo), (h 0-7, d hi), (h 8-15, d hi)
        const int mi = lane >> 3;
        const int hr = hgrp * 16 + (mi & 1) * 8 + (lane & 7);
        const uint32_t addr = sq + hr * Cfg::kRowBytes + (d0 + (mi >> 1) * 8) * 2;
        ldsm_x4(addr, qa[0], qa[1], qa[2], qa[3]);
      }
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        // B: n = K~ rows, k = d: matrices (rows 8np.., d lo), (.., d hi), (rows 8np+8.., lo), (.., hi)
        const int mi = lane >> 3;
        const int rr = np * 16 + (mi >> 1) * 8 + (lane & 7);
        const uint32_t addr = sk + rr * Cfg::kRowBytes + (d0 + (mi & 1) * 8) * 2;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        mma_bf16(sc[2 * np], qa, b0, b1);
        mma_bf16(sc[2 * np + 1], qa, b2, b3);
      }
    }
    // exchange halves: S = S_half0 + S_half1
    float* mine = sx + (size_t)warp * 16 * kChunk;
    const float* other = sx + (size_t)(warp ^ 4) * 16 * kChunk;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      mine[g * kChunk + nt * 8 + 2 * q4] = sc[nt][0];
      mine[g * kChunk + nt * 8 + 2 * q4 + 1] = sc[nt][1];
      mine[(g + 8) * kChunk + nt * 8 + 2 * q4] = sc[nt][2];
      mine[(g + 8) * kChunk + nt * 8 + 2 * q4 + 1] = sc[nt][3];
    }
    __syncthreads();
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      sc[nt][0] += other[g * kChunk + nt * 8 + 2 * q4];
      sc[nt][1] += other[g * kChunk + nt * 8 + 2 * q4 + 1];
      sc[nt][2] += other[(g + 8) * kChunk + nt * 8 + 2 * q4];
      sc[nt][3] += other[(g + 8) * kChunk + nt * 8 + 2 * q4 + 1];
    }
    // ---- softmax of the chunk per head (exp2 domain) ----
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = nt * 8 + 2 * q4 + (e & 1);
        const float x = rowoff[col] >= 0 ? sc[nt][e] * a.scale_log2 : -INFINITY;
        sc[nt][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
    }
    float lsum[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float base = mx[e >> 1] == -INFINITY ? 0.f : mx[e >> 1];
        const float pv = fast_exp2(sc[nt][e] - base);
        sc[nt][e] = pv;
        lsum[e >> 1] += pv;
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      lsum[hh] += __shfl_xor_sync(0xffffffffu, lsum[hh], 1);
      lsum[hh] += __shfl_xor_sync(0xffffffffu, lsum[hh], 2);
    }
    // ---- acc = P V over this warp's half of D ----
    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kChunk / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
      pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
      pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        // B = V rows (k = K~ row, n = d), transposed by ldmatrix:
        // matrices (rows 0-7, d lo), (rows 8-15, d lo), (rows 0-7, d hi), (rows 8-15, d hi)
        const int mi = lane >> 3;
        const int rr = kk * 16 + (mi & 1) * 8 + (lane & 7);
        const int dd = half * DH + np * 16 + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sk + rr * Cfg::kRowBytes + dd * 2, b0, b1, b2, b3);
        mma_bf16(acc[2 * np], pa, b0, b1);
        mma_bf16(acc[2 * np + 1], pa, b2, b3);
      }
    }
    // ---- partial of this item: [N1][D + 2] at slot (row, chunk) ----
    float* pp = a.partials + ((size_t)u * a.max_chunks + ch) * (size_t)a.N1 * (D + 2);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int hl = hgrp * 16 + g + 8 * hh;
      if (hl >= nheads) continue;
      float* ph = pp + (size_t)(head0 + hl) * (D + 2);
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const int d = half * DH + i * 8 + 2 * q4;
        *reinterpret_cast<float2*>(ph + d) = make_float2(acc[i][2 * hh], acc[i][2 * hh + 1]);
      }
      if (half == 0 && q4 == 0) {
        ph[D] = mx[hh];
        ph[D + 1] = lsum[hh];
      }
    }
    __syncthreads();  // shared buffers are reused by the next item
    if (*reinterpret_cast<volatile int*>(misc)) break;
    ++ch;
  }
}

// ---------------------------------------------------------------------------
// combine: fold a row's chunk partials in chunk order, sink, normalise
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) sparse_combine_kernel(const SparseArgs a,
                                                              const int32_t* __restrict__ md) {
  if (md[0] != 0x46534D31 || md[1] != a.num_ctas || md[2] != (int32_t)a.rows ||
      md[5] != a.B || md[6] != a.N1 || md[7] != a.K2)
    return;  // the attention kernel has set the status word
  const int64_t u = blockIdx.x;
  const int h = blockIdx.y;
  const SparseRow r = sparse_row(a, u);
  const float* base = a.partials + ((size_t)u * a.max_chunks) * (size_t)a.N1 * (D + 2) +
                      (size_t)h * (D + 2);
  const size_t cstride = (size_t)a.N1 * (D + 2);
  float M = -INFINITY;
  for (int ch = 0; ch < r.nchunks; ++ch) M = fmaxf(M, base[ch * cstride + D]);
  const float Mu = M == -INFINITY ? 0.f : M;
  float L = 0.f;
  for (int ch = 0; ch < r.nchunks; ++ch) {
    const float mc = base[ch * cstride + D];
    if (mc != -INFINITY) L += base[ch * cstride + D + 1] * exp2f(mc - Mu);
  }
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
  for (int d = threadIdx.x * 2; d < D; d += 256) {
    float o0 = 0.f, o1 = 0.f;
    for (int ch = 0; ch < r.nchunks; ++ch) {
      const float mc = base[ch * cstride + D];
      if (mc == -INFINITY) continue;
      const float f = exp2f(mc - Mu);
      o0 += base[ch * cstride + d] * f;
      o1 += base[ch * cstride + d + 1] * f;
    }
    *reinterpret_cast<uint32_t*>(a.out + (u * a.N1 + h) * (int64_t)D + d) = pack_bf16(o0 * scl, o1 * scl);
  }
  if (a.lse && threadIdx.x == 0) a.lse[u * a.N1 + h] = lse;
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
  dim3 grid(a.num_ctas, (a.N1 + kHeadsPerCta - 1) / kHeadsPerCta);
  kern<<<grid, kSThreads, Cfg::kSmem, s>>>(a, md);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 cgrid((unsigned)a.rows, a.N1);
  sparse_combine_kernel<D><<<cgrid, 128, 0, s>>>(a, md);
  return cudaGetLastError();
}

cudaError_t launch_sparse(const SparseArgs& a, const int32_t* md, cudaStream_t s) {
  if (a.D == 512) return launch_sparse_t<512>(a, md, s);
  if (a.D == 256) return launch_sparse_t<256>(a, md, s);
  return launch_sparse_t<128>(a, md, s);
}

}  // namespace fia
