// combine.cu -- log-sum-exp merge of split-KV partial results.
//
// Each split j of a row (sequence b, head i) produced a normalised partial
// output o_j over its token range and lse_j = log2 of its softmax
// denominator (log2 domain, scores already scaled by log2 e).  The merged
// output is  sum_j w_j o_j / sum_j w_j  with  w_j = 2^(lse_j - max_k lse_k);
// an empty range (lse = -inf) has weight 0.  A +inf lse marks a range that
// met bad data: the whole row is written as zeros.
//
// One warp per row, kRowsPerCta rows per CTA.  Lane l owns the float4
// columns l, l + 32, ...; the weights are computed one per lane and
// broadcast, and the loads of all partials are independent of each other,
// so a row costs about two dependent global-load latencies.
#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();
constexpr int kRowsPerCta = 8;
constexpr unsigned kFull = 0xffffffffu;

// Merge ns partial rows into one output row (one warp).  Partial s has its
// lse at lse[row(s)] and its D values at po[row(s) * D].
template <int D, bool kBF16, typename RowOf>
__device__ __forceinline__ void merge_row(const float* lse, const float* po, RowOf row, int ns,
                                          uint16_t* out, int lane) {
  constexpr int kVec = D / 128;  // float4 per lane
  float mx = kNegInf;
  bool poison = false;
  for (int s = lane; s < ns; s += 32) {
    const float v = lse[row(s)];
    poison |= (v == kPosInf);
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
  poison = __any_sync(kFull, poison);
  uint2* dst = reinterpret_cast<uint2*>(out);
  if (poison || mx == kNegInf) {
#pragma unroll
    for (int v = 0; v < kVec; ++v) dst[v * 32 + lane] = make_uint2(0, 0);
    return;
  }
  float4 acc[kVec];
#pragma unroll
  for (int v = 0; v < kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* po4 = reinterpret_cast<const float4*>(po);
  float wsum = 0.f;
  for (int s0 = 0; s0 < ns; s0 += 32) {
    const int cnt = min(32, ns - s0);
    // Weight of partial s0 + lane: 2^(lse - max), 0 for an empty split.
    const float wl = lane < cnt ? ex2(lse[row(s0 + lane)] - mx) : 0.f;
    wsum += wl;
    // All of a row's partial loads in flight at once where registers allow
    // (long context merges 32 splits of 128 values: 16 in flight against 4,
    // 88.9 against 91.7 us for the whole B = 1, S = 131072 call).
    constexpr int kUnroll = kVec == 1 ? 16 : 4;
#pragma unroll kUnroll
    for (int i = 0; i < cnt; ++i) {
      const float w = __shfl_sync(kFull, wl, i);
      const size_t base = row(s0 + i) * (D / 4);
#pragma unroll
      for (int v = 0; v < kVec; ++v) {
        const float4 x = po4[base + v * 32 + lane];
        acc[v].x = fmaf(w, x.x, acc[v].x);
        acc[v].y = fmaf(w, x.y, acc[v].y);
        acc[v].z = fmaf(w, x.z, acc[v].z);
        acc[v].w = fmaf(w, x.w, acc[v].w);
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) wsum += __shfl_xor_sync(kFull, wsum, off);
  const float inv = 1.f / wsum;
#pragma unroll
  for (int v = 0; v < kVec; ++v)
    dst[v * 32 + lane] = make_uint2(pack2<kBF16>(acc[v].x * inv, acc[v].y * inv),
                                    pack2<kBF16>(acc[v].z * inv, acc[v].w * inv));
}

// The combines are launched as programmatic dependents of the partial
// kernel: their CTAs may start while its last CTAs run, and wait here until
// every partial is written (a no-op for an ordinary launch).
__device__ __forceinline__ void wait_for_partials() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Per-sequence split-KV partials: row r's splits are contiguous.
template <int D, bool kBF16>
__global__ void __launch_bounds__(kRowsPerCta * 32) lse_combine_kernel(const CombineParams p) {
  wait_for_partials();
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (r >= p.rows) return;
  const size_t row0 = static_cast<size_t>(r) * p.n_split;
  merge_row<D, kBF16>(p.part_lse, p.part_o, [row0](int s) { return row0 + s; }, p.n_split,
                      static_cast<uint16_t*>(p.out) + static_cast<size_t>(r) * D,
                      threadIdx.x & 31);
}

// MLA partials of a balanced schedule: sequence b's tiles [g0, g1) were cut
// by the pair slices [starts[q], starts[q + 1]) (the partial kernel writes
// the slice starts and every sequence's first cost position after the
// per-sequence first-tile table).  Only the first and the last segment of a
// slice can be partial, and pair q writes them to slots 2 q and 2 q + 1: b's
// piece in its first pair q0 is slot 2 q0 + 1 unless b starts that slice,
// and its piece in every later pair starts that pair's slice (slot 2 q).
// Rows of sequences that one pair covered whole (or that have no tiles)
// were written by the partial kernel and are skipped.  One warp per
// (sequence, head).
template <bool kBF16>
__global__ void __launch_bounds__(kRowsPerCta * 32) mla_combine_kernel(const MlaCombineParams p) {
  wait_for_partials();
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (r >= p.batch * kMlaHeads) return;
  const int b = r / kMlaHeads, h = r % kMlaHeads;
  const int g0 = p.ws_hdr[kHdrPref + b], g1 = p.ws_hdr[kHdrPref + b + 1];
  if (g1 <= g0) return;
  const int* starts = p.ws_hdr + kHdrPref + p.batch + 1;
  const int* cprefs = starts + p.n_pairs + 1;
  // The pair holding tile g is the one whose cost slice holds g's cost
  // position: q = min(c(g) / W, n_pairs - 1), c(b's first tile) = cprefs[b].
  const int W = p.ws_hdr[0], cb = cprefs[b];
  const int q0 = min(cb / W, p.n_pairs - 1), q1 = min((cb + g1 - g0 - 1) / W, p.n_pairs - 1);
  if (q1 == q0) return;
  const int first_slot = 2 * q0 + (g0 == starts[q0] ? 0 : 1);
  auto row = [=](int s) {
    const int slot = s == 0 ? first_slot : 2 * (q0 + s);
    return static_cast<size_t>(slot) * kMlaHeads + h;
  };
  merge_row<kMlaDc, kBF16>(p.part_lse, p.part_o, row, q1 - q0 + 1,
                           static_cast<uint16_t*>(p.out) + static_cast<size_t>(r) * kMlaDc,
                           threadIdx.x & 31);
}

// Launch with programmatic stream serialization: the kernel may begin
// before the previous kernel on the stream has finished, and its
// griddepcontrol.wait holds it until that kernel's memory is visible.
template <typename Params>
cudaError_t launch_dependent(void (*kern)(Params), int ctas, const Params& p,
                             cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kRowsPerCta * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int D, bool kBF16>
cudaError_t launch_d(const CombineParams& p, cudaStream_t stream) {
  const int ctas = (p.rows + kRowsPerCta - 1) / kRowsPerCta;
  return launch_dependent(lse_combine_kernel<D, kBF16>, ctas, p, stream);
}

}  // namespace

cudaError_t launch_mla_combine(const MlaCombineParams& p, bool bf16, cudaStream_t stream) {
  if (p.batch <= 0) return cudaSuccess;
  const int ctas = (p.batch * kMlaHeads + kRowsPerCta - 1) / kRowsPerCta;
  return bf16 ? launch_dependent(mla_combine_kernel<true>, ctas, p, stream)
              : launch_dependent(mla_combine_kernel<false>, ctas, p, stream);
}

cudaError_t launch_combine(const CombineParams& p, int d, bool bf16, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  if (d == kHeadDim) return bf16 ? launch_d<kHeadDim, true>(p, stream) : launch_d<kHeadDim, false>(p, stream);
  if (d == kMlaDc) return bf16 ? launch_d<kMlaDc, true>(p, stream) : launch_d<kMlaDc, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace decattn
