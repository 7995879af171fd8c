// combine.cu -- fia_lse_combine: the log-sum-exp combine of attention results
// computed against disjoint parts of the keys ("aclnnFusedInferAttentionScoreV2",
// softmax_lse restriction: the ring-attention use of the lse output;
// "sparse_flash_mla", CP example: context parallelism across ranks).
//
// For one query row and head with part results (O_k, lse_k), k = 0..n-1:
//   lse = log (sum_k e^{lse_k} + e^{sink}),  O = sum_k e^{lse_k - lse} O_k,
// parts with lse_k = +inf (no visible key) left out, the sink term only with
// a sink, and O = 0, lse = +inf when every part is left out.  One warp per (token, head) row; each lane
// owns 8 consecutive elements of D per pass (16-byte loads and stores), and
// the parts are folded in index order, so the result does not depend on the
// launch shape.  HBM-bound: reads n rows of D bf16 and n lse values, writes
// one row.
#include <algorithm>
#include <cstring>

#include "../../include/fia.h"
#include "common.cuh"
#include "internal.h"

namespace fia {

namespace {

struct CombineArgs {
  const uint16_t* o[FIA_COMBINE_MAX_PARTS];
  const float* l[FIA_COMBINE_MAX_PARTS];
  uint16_t* out;
  float* lse;
  const float* sinks;
  int n, layout, N, D, S_q;
  int64_t rows;  // tokens * N
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(256) lse_combine_kernel(const CombineArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < a.rows;
       r += warps) {
    const int64_t t = r / a.N;
    const int h = (int)(r - t * a.N);
    int64_t li;
    if (a.layout == FIA_LAYOUT_TND) {
      li = r;
    } else {
      const int64_t b = t / a.S_q, i = t - b * a.S_q;
      li = (b * a.N + h) * a.S_q + i;
    }
    // the total: largest finite lse, then the sum of e^{lse_k - max}
    float lk[FIA_COMBINE_MAX_PARTS];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < FIA_COMBINE_MAX_PARTS; ++k) {
      lk[k] = k < a.n ? __ldg(a.l[k] + li) : INFINITY;
      if (lk[k] != INFINITY) M = fmaxf(M, lk[k]);
    }
    // a sink is one more logit with no value, counted once when some part
    // saw a key (a row that sees no key stays 0 / +inf, with a sink too)
    const bool any = M != -INFINITY;
    const float sk = (a.sinks && any) ? __ldg(a.sinks + h) : -INFINITY;
    const float Mx = fmaxf(M, sk);
    float S = 0.f;
    if (any) {
#pragma unroll
      for (int k = 0; k < FIA_COMBINE_MAX_PARTS; ++k)
        if (lk[k] != INFINITY) S += expf(lk[k] - Mx);
      if (sk != -INFINITY) S += expf(sk - Mx);
    }
    const bool empty = !any || !(S > 0.f);
    const float L = empty ? INFINITY : Mx + logf(S);
    uint16_t* orow = a.out + r * a.D;
    for (int d0 = 8 * lane; d0 < a.D; d0 += 256) {
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      if (!empty) {
#pragma unroll
        for (int k = 0; k < FIA_COMBINE_MAX_PARTS; ++k) {
          if (lk[k] == INFINITY) continue;
          const float w = expf(lk[k] - L);
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.o[k] + r * a.D + d0));
          acc[0] += w * bf16_lo(v.x); acc[1] += w * bf16_hi(v.x);
          acc[2] += w * bf16_lo(v.y); acc[3] += w * bf16_hi(v.y);
          acc[4] += w * bf16_lo(v.z); acc[5] += w * bf16_hi(v.z);
          acc[6] += w * bf16_lo(v.w); acc[7] += w * bf16_hi(v.w);
        }
      }
      *reinterpret_cast<uint4*>(orow + d0) =
          make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                     pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
    }
    if (a.lse && lane == 0) a.lse[li] = L;
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace fia

extern "C" size_t fia_sizeof_combine_params(void) { return sizeof(fia_combine_params); }

extern "C" fia_status fia_lse_combine(const fia_combine_params* p, void* stream) {
  fia::NvtxRange range("fia_lse_combine");
  using namespace fia;
  if (!p) return FIA_ERR_NULL_ARG;
  for (int i = 0; i < 8; ++i)
    if (p->reserved[i] != 0) return FIA_ERR_BAD_SHAPE;
  if (p->n_parts < 1 || p->n_parts > FIA_COMBINE_MAX_PARTS) return FIA_ERR_BAD_SHAPE;
  if (p->layout != FIA_LAYOUT_BSND && p->layout != FIA_LAYOUT_TND) return FIA_ERR_BAD_SHAPE;
  if (p->num_heads < 1 || p->num_heads > 256) return FIA_ERR_BAD_SHAPE;
  if (p->head_dim < 8 || p->head_dim > 512 || p->head_dim % 8) return FIA_ERR_BAD_SHAPE;
  int64_t tokens;
  if (p->layout == FIA_LAYOUT_TND) {
    if (p->total_q < 0) return FIA_ERR_BAD_SHAPE;
    tokens = p->total_q;
  } else {
    if (p->batch < 0 || p->batch > 65536 || p->seqlen_q < 0) return FIA_ERR_BAD_SHAPE;
    tokens = (int64_t)p->batch * p->seqlen_q;
  }
  if (!p->o_parts || !p->lse_parts || !p->out) return FIA_ERR_NULL_ARG;
  CombineArgs a;
  memset(&a, 0, sizeof a);
  for (int k = 0; k < p->n_parts; ++k) {
    if (!p->o_parts[k] || !p->lse_parts[k]) return FIA_ERR_NULL_ARG;
    if (!al16(p->o_parts[k]) || (reinterpret_cast<uintptr_t>(p->lse_parts[k]) & 3u))
      return FIA_ERR_BAD_SHAPE;
    if (p->o_parts[k] == p->out) return FIA_ERR_BAD_SHAPE;
    a.o[k] = static_cast<const uint16_t*>(p->o_parts[k]);
    a.l[k] = p->lse_parts[k];
  }
  if (!al16(p->out) || (p->lse && (reinterpret_cast<uintptr_t>(p->lse) & 3u)))
    return FIA_ERR_BAD_SHAPE;
  a.out = static_cast<uint16_t*>(p->out);
  a.lse = p->lse;
  a.sinks = p->sinks;
  a.n = p->n_parts;
  a.layout = p->layout;
  a.N = p->num_heads;
  a.D = p->head_dim;
  a.S_q = p->layout == FIA_LAYOUT_BSND ? p->seqlen_q : 1;
  a.rows = tokens * p->num_heads;
  if (a.rows == 0) return FIA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FIA_ERR_CUDA;
  const int64_t blocks = (a.rows + 7) / 8;
  const int grid = (int)std::min<int64_t>(blocks, (int64_t)sms * 8);
  lse_combine_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? FIA_OK : FIA_ERR_CUDA;
}
