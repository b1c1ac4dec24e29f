// combine.cu -- log-sum-exp merge of split-KV partial results.
//
// Each split j of a row (sequence b, head i) produced a normalised partial
// output o_j over its token range and lse_j = log2 of its softmax
// denominator (log2 domain, scores already scaled by log2 e).  The merged
// output is  sum_j w_j o_j / sum_j w_j  with  w_j = 2^(lse_j - max_k lse_k);
// an empty range (lse = -inf) has weight 0.  A +inf lse marks a range that
// met bad data: the whole row is written as zeros.
//
// One warp per row; lane l owns the float4 columns l, l + 32, ... of the row.
#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();

template <int D, bool kBF16>
__global__ void __launch_bounds__(256) lse_combine_kernel(const CombineParams p) {
  constexpr int kVec = D / 128;  // float4 per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + warp;
  if (row >= p.rows) return;
  const int ns = p.n_split;
  const float* lse = p.part_lse + static_cast<size_t>(row) * ns;

  float mx = kNegInf;
  bool poison = false;
  for (int s = lane; s < ns; s += 32) {
    const float v = lse[s];
    poison |= (v == kPosInf);
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  poison = __any_sync(0xffffffffu, poison);

  uint16_t* out = static_cast<uint16_t*>(p.out) + static_cast<size_t>(row) * D;
  if (poison || mx == kNegInf) {
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      uint2 z = make_uint2(0, 0);
      *reinterpret_cast<uint2*>(out + (v * 32 + lane) * 4) = z;
    }
    return;
  }

  float wsum = 0.f;
  for (int s = lane; s < ns; s += 32) wsum += ex2(lse[s] - mx);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);

  float4 acc[kVec];
#pragma unroll
  for (int v = 0; v < kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* po = reinterpret_cast<const float4*>(p.part_o + static_cast<size_t>(row) * ns * D);
#pragma unroll 4
  for (int s = 0; s < ns; ++s) {
    const float ls = lse[s];
    if (ls == kNegInf) continue;
    const float w = ex2(ls - mx);
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const float4 x = po[static_cast<size_t>(s) * (D / 4) + v * 32 + lane];
      acc[v].x = fmaf(w, x.x, acc[v].x);
      acc[v].y = fmaf(w, x.y, acc[v].y);
      acc[v].z = fmaf(w, x.z, acc[v].z);
      acc[v].w = fmaf(w, x.w, acc[v].w);
    }
  }
  const float inv = 1.f / wsum;
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    uint2 w2;
    w2.x = pack2<kBF16>(acc[v].x * inv, acc[v].y * inv);
    w2.y = pack2<kBF16>(acc[v].z * inv, acc[v].w * inv);
    *reinterpret_cast<uint2*>(out + (v * 32 + lane) * 4) = w2;
  }
}

template <int D, bool kBF16>
cudaError_t launch_d(const CombineParams& p, cudaStream_t stream) {
  constexpr int kWarps = 8;
  const int blocks = (p.rows + kWarps - 1) / kWarps;
  lse_combine_kernel<D, kBF16><<<blocks, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, int d, bool bf16, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  if (d == kHeadDim) return bf16 ? launch_d<kHeadDim, true>(p, stream) : launch_d<kHeadDim, false>(p, stream);
  if (d == kMlaDc) return bf16 ? launch_d<kMlaDc, true>(p, stream) : launch_d<kMlaDc, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace decattn
