// kv_append.cu -- the decode step's cache write: each sequence's new token
// (its K and V rows, or its MLA latent row) goes into the paged slot
// block_table[b][pos / block_size], pos % block_size.
//
// A token's row is contiguous in the new-token tensor ([B, row]) and in the
// cache (slot-major [num_blocks, block_size, row]), so one CTA per sequence
// moves it in 16-byte pieces; K and V are one launch.  Over an 8-bit cache
// each 16-bit value x of KV head j is stored as the e4m3 code of
// fp32(x) / scale[j] (round to nearest even, saturating at 448): eight
// values in, eight codes out per thread.  The work is a few hundred KB per
// layer, so the launch itself is the cost.
#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Slot row of sequence b's position, or -1 (flagged) when the position lies
// past the block table or its block id is out of range; -2 for a skip.
__device__ __forceinline__ int64_t slot_row(const AppendParams& p, int b) {
  const int pos = p.positions[b];
  if (pos < 0) return -2;
  const int lb = pos >> p.log2_block_size;
  if (lb >= p.max_blocks_per_seq) {
    if (threadIdx.x == 0) flag_error(p.err_flag, kFlagBadSeqLen);
    return -1;
  }
  const int id = p.block_table[static_cast<int64_t>(b) * p.max_blocks_per_seq + lb];
  if (id < 0 || id >= p.num_blocks) {
    if (threadIdx.x == 0) flag_error(p.err_flag, kFlagBadBlock);
    return -1;
  }
  return static_cast<int64_t>(id) * p.block_size + (pos & (p.block_size - 1));
}

// 16-bit rows copied as they are.  row_elems is a multiple of 8.
__global__ void __launch_bounds__(kThreads) append_copy_kernel(const AppendParams p) {
  const int b = blockIdx.x;
  const int64_t row = slot_row(p, b);
  if (row < 0) return;
  const int chunks = p.row_elems / 8;  // 16-byte pieces per row
  const int n = p.v_new ? 2 * chunks : chunks;
  for (int c = threadIdx.x; c < n; c += kThreads) {
    const bool is_v = c >= chunks;
    const int cc = is_v ? c - chunks : c;
    const uint16_t* src = static_cast<const uint16_t*>(is_v ? p.v_new : p.k_new) +
                          static_cast<int64_t>(b) * p.row_elems + cc * 8;
    uint16_t* dst = static_cast<uint16_t*>(is_v ? p.v_cache : p.k_cache) + row * p.row_elems +
                    cc * 8;
    *reinterpret_cast<uint4*>(dst) = ld_nc_v4(src);
  }
}

// 16-bit rows quantised to e4m3 codes with one scale per head_elems-wide head.
template <bool kBF16>
__global__ void __launch_bounds__(kThreads) append_e4m3_kernel(const AppendParams p) {
  const int b = blockIdx.x;
  const int64_t row = slot_row(p, b);
  if (row < 0) return;
  const int chunks = p.row_elems / 8;
  for (int c = threadIdx.x; c < 2 * chunks; c += kThreads) {
    const bool is_v = c >= chunks;
    const int cc = is_v ? c - chunks : c;
    const int e0 = cc * 8;
    const float s = (is_v ? p.v_scale : p.k_scale)[e0 / p.head_elems];
    const uint4 w = ld_nc_v4(static_cast<const uint16_t*>(is_v ? p.v_new : p.k_new) +
                             static_cast<int64_t>(b) * p.row_elems + e0);
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t codes[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float2 a = unpack2<kBF16>(in[2 * h]), c2 = unpack2<kBF16>(in[2 * h + 1]);
      const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(a.x, s), __fdiv_rn(a.y, s));
      const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(c2.x, s), __fdiv_rn(c2.y, s));
      codes[h] = lo | (hi << 16);
    }
    uint8_t* dst = static_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) + row * p.row_elems + e0;
    *reinterpret_cast<uint2*>(dst) = make_uint2(codes[0], codes[1]);
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, bool e4m3, bool bf16, cudaStream_t stream) {
  if (p.batch <= 0) return cudaSuccess;
  if (!e4m3)
    append_copy_kernel<<<p.batch, kThreads, 0, stream>>>(p);
  else if (bf16)
    append_e4m3_kernel<true><<<p.batch, kThreads, 0, stream>>>(p);
  else
    append_e4m3_kernel<false><<<p.batch, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace decattn
