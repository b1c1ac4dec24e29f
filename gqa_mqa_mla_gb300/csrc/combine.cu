// combine.cu -- log-sum-exp merge of split-KV partial results.
//
// Each split j of a row (sequence b, head i) produced a normalised partial
// output o_j over its token range and lse_j = log2 of its softmax
// denominator (log2 domain, scores already scaled by log2 e).  The merged
// output is  sum_j w_j o_j / sum_j w_j  with  w_j = 2^(lse_j - max_k lse_k);
// an empty range (lse = -inf) has weight 0.  A +inf lse marks a range that
// met bad data: the whole row is written as zeros.
//
// One CTA of kWarps warps per row.  Warp w accumulates the splits
// j = w, w + kWarps, ... (lane l owns the float4 columns l, l + 32, ...), with
// several splits' loads in flight; the warps' sums meet in shared memory.
#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();
constexpr int kWarps = 4;

template <int D, bool kBF16>
__global__ void __launch_bounds__(kWarps * 32) lse_combine_kernel(const CombineParams p) {
  constexpr int kVec = D / 128;  // float4 per lane
  __shared__ float4 red[kWarps][D / 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x;
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
    for (int c = threadIdx.x; c < D / 4; c += kWarps * 32)
      *reinterpret_cast<uint2*>(out + c * 4) = make_uint2(0, 0);
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
  for (int s = warp; s < ns; s += kWarps) {
    const float w = ex2(lse[s] - mx);  // 0 for an empty split
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const float4 x = po[static_cast<size_t>(s) * (D / 4) + v * 32 + lane];
      acc[v].x = fmaf(w, x.x, acc[v].x);
      acc[v].y = fmaf(w, x.y, acc[v].y);
      acc[v].z = fmaf(w, x.z, acc[v].z);
      acc[v].w = fmaf(w, x.w, acc[v].w);
    }
  }
#pragma unroll
  for (int v = 0; v < kVec; ++v) red[warp][v * 32 + lane] = acc[v];
  __syncthreads();
  const float inv = 1.f / wsum;
  for (int c = threadIdx.x; c < D / 4; c += kWarps * 32) {
    float4 t = red[0][c];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      const float4 u = red[w][c];
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    uint2 w2;
    w2.x = pack2<kBF16>(t.x * inv, t.y * inv);
    w2.y = pack2<kBF16>(t.z * inv, t.w * inv);
    *reinterpret_cast<uint2*>(out + c * 4) = w2;
  }
}

template <int D, bool kBF16>
cudaError_t launch_d(const CombineParams& p, cudaStream_t stream) {
  lse_combine_kernel<D, kBF16><<<p.rows, kWarps * 32, 0, stream>>>(p);
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
