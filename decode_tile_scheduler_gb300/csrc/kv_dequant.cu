// kv_dequant.cu -- FP8 E4M3 K/V for the prefill branch.
//
// The FIA pages allow FP8 K/V with per-64-element fp32 scales in the prefill
// layouts as well ("aclnnFusedInferAttentionScoreV5", FLOAT8_E4M3FN key/value
// rules and the DequantChecker group).  Prefill is bound by the tensor cores,
// and each K/V tile is read by every 128-row query tile and head pair of its
// sequence, so the visible rows are dequantised once, here, into contiguous
// caches in the workspace, and the tcgen05 prefill kernel runs on those with
// fp16 operands (11 significant bits: a code times its fp32 scale keeps its
// value to 2^-12, where bf16 would lose it at 2^-9 -- too coarse for the
// 1e-3 lse bound).  fp16's range is kept by powers of two that the prefill
// kernel takes back exactly:
//   K', V': every (batch, KV head) divided by 2^E, E the exponent of its
//           largest K (V) scale, so |K'| < 2 * 448;
//   Q':     every (token, head) times 2^sh, sh = 15 - (the exponent of its
//           largest element), kept in [-100, 100] -- the same exact move the
//           FP8 decode kernel makes; the prefill kernel's softmax warps do it
//           to each query tile in shared memory as it lands (a pass here
//           would read and write all of Q once more).
// The scores of row (t, h) are then S' * 2^-sh * 2^EK, and the output O' * 2^EV.
//
// Two passes, short next to the prefill: the largest scale of each (batch,
// KV head) (warp maxima, then atomic maxima over the float bits, positive
// floats ordering like their bit patterns) and the K/V conversion (one thread
// per 16 elements of a (batch, row, head) vector).  Rows at or past a batch's
// KV length are not touched (the prefill kernel masks their scores and
// zeroes their V rows).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fia {

namespace {

// Code offset and scale row of element d0 of (batch b, row j, head hk); false
// when the row's page lies outside the pool.
__device__ __forceinline__ bool locate(const DequantArgs& a, int b, int j, int hk, int d0,
                                       int64_t* code_off, int64_t* scale_row) {
  if (a.block_table) {
    const int64_t blk = a.block_table[(int64_t)b * a.max_blocks + j / a.block_size];
    if (blk < 0 || blk >= a.num_blocks) {
      if (a.debug) atomicExch(a.err, 3);
      return false;
    }
    const int jp = j % a.block_size;
    *code_off = a.kv_layout == 1 ? ((blk * a.KVN + hk) * a.block_size + jp) * a.D + d0
                                 : ((blk * a.block_size + jp) * a.KVN + hk) * a.D + d0;
    *scale_row = (blk * a.KVN + hk) * a.block_size + jp;
  } else {
    *code_off = (((int64_t)b * a.cap + j) * a.KVN + hk) * a.D + d0;
    *scale_row = ((int64_t)b * a.KVN + hk) * a.cap + j;
  }
  return true;
}

// Largest K and V scale of every (batch, KV head) over its visible rows: a
// warp per (batch, KV head, run of 128 rows), a warp maximum, then one
// atomic per warp (an atomic per row serialised on the few addresses).  Each
// row is a page lookup and then its scales, so a warp's runs are a chain of
// dependent loads: short runs and many warps keep the chain short (runs of
// 1024 rows took ~30 us on the varlen FP8 prefill).
constexpr int kScaleRun = 128;
__global__ void __launch_bounds__(256) scale_max_kernel(const DequantArgs a) {
  const int NT = a.D / 64;
  const int lane = threadIdx.x & 31;
  const int nrun = (a.cap + kScaleRun - 1) / kScaleRun;
  const int64_t items = (int64_t)a.B * a.KVN * nrun;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < items; w += nw) {
    const int64_t pair = w / nrun;
    const int run = (int)(w - pair * nrun);
    const int b = (int)(pair / a.KVN), hk = (int)(pair - (int64_t)b * a.KVN);
    const int kv_len = a.seqused_kv ? a.seqused_kv[b] : a.cap;
    const int j_end = min(kv_len, (run + 1) * kScaleRun);
    uint32_t mk = 0, mv = 0;
    for (int j = run * kScaleRun + lane; j < j_end; j += 32) {
      int64_t off, srow;
      if (!locate(a, b, j, hk, 0, &off, &srow)) continue;
      for (int k = 0; k < NT; ++k) {
        mk = max(mk, __float_as_uint(fabsf(__ldg(a.k_scale + srow * NT + k))));
        mv = max(mv, __float_as_uint(fabsf(__ldg(a.v_scale + srow * NT + k))));
      }
    }
    mk = __reduce_max_sync(0xffffffffu, mk);
    mv = __reduce_max_sync(0xffffffffu, mv);
    if (lane == 0 && (mk | mv)) {
      atomicMax(a.smax + pair * 2, mk);
      atomicMax(a.smax + pair * 2 + 1, mv);
    }
  }
}

// 2^-E for the largest scale bits m (E its exponent, kept in [-100, 100]);
// a zero or non-finite maximum takes 1.
__device__ __forceinline__ float inv_pow2_of(uint32_t m) {
  const int e = (int)((m >> 23) & 0xffu);
  if (e == 0 || e == 0xff) return 1.f;
  const int E = min(max(e - 127, -100), 100);
  return __int_as_float((127 - E) << 23);
}

__global__ void __launch_bounds__(256) kv_dequant_kernel(const DequantArgs a) {
  const int per_row = a.KVN * (a.D / 16);  // threads per (batch, row)
  const int64_t total = (int64_t)a.B * a.cap * per_row;
  const int NT = a.D / 64;
  // the factors the prefill kernel multiplies back (thread 0 of the grid)
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < a.B * a.KVN * 2; i += blockDim.x)
      a.kvfac[i] = 1.f / inv_pow2_of(a.smax[i]);
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bj = t / per_row;
    const int rest = (int)(t - bj * per_row);
    const int b = (int)(bj / a.cap);
    const int j = (int)(bj - (int64_t)b * a.cap);
    const int kv_len = a.seqused_kv ? a.seqused_kv[b] : a.cap;
    if (j >= kv_len) continue;
    const int hk = rest / (a.D / 16), d0 = (rest % (a.D / 16)) * 16;
    int64_t code_off, scale_row;
    if (!locate(a, b, j, hk, d0, &code_off, &scale_row)) continue;
    const int64_t out_off = (((int64_t)b * a.cap + j) * a.KVN + hk) * a.D + d0;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const uint8_t* src = kv ? a.v : a.k;
      const float f = inv_pow2_of(__ldg(a.smax + ((int64_t)b * a.KVN + hk) * 2 + kv));
      const float sc = __ldg((kv ? a.v_scale : a.k_scale) + scale_row * NT + d0 / 64) * f;
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(src + code_off));
      const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
      uint32_t o[8];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t lo, hi;
        e4m3x4_to_f16x2x2(cw[w], lo, hi);  // exact: E4M3 values are fp16 values
        const float2 fl = __half22float2(*reinterpret_cast<const __half2*>(&lo));
        const float2 fh = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        o[2 * w] = pack_f16(fl.x * sc, fl.y * sc);
        o[2 * w + 1] = pack_f16(fh.x * sc, fh.y * sc);
      }
      uint16_t* dst = (kv ? a.v_out : a.k_out) + out_off;
      reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
      reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

}  // namespace

cudaError_t launch_kv_dequant(const DequantArgs& a, int num_sms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(a.smax, 0, sizeof(uint32_t) * 2 * (size_t)a.B * a.KVN, s);
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)a.B * a.cap * a.KVN;
  if (rows > 0) {
    const int64_t warps = (int64_t)a.B * a.KVN * ((a.cap + kScaleRun - 1) / kScaleRun);
    const int g1 = (int)std::min<int64_t>((warps + 7) / 8, (int64_t)num_sms * 8);
    scale_max_kernel<<<g1, 256, 0, s>>>(a);
    const int64_t total = rows * (a.D / 16);
    const int g2 = (int)std::min<int64_t>((total + 255) / 256, (int64_t)num_sms * 32);
    kv_dequant_kernel<<<g2, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace fia
