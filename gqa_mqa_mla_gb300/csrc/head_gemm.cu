// head_gemm.cu -- the two GEMMs around absorbed MLA decode, one weight matrix
// per head:
//   q_abs[b, i, :] = q_nope[b, i, :] W_uk^(i)^T   (W_uk^(i): d_c x d_h)
//   out[b, i, :]   = o_lat[b, i, :]  W_uv^(i)     (given as W_uv^(i)^T: d_v x d_c)
// Both are Y_i = X_i W_i^T with W_i [M x K] (K contiguous) and X_i the
// batch's rows of head i.
//
// Decode batches are narrow and the weights are the bytes, so the MMA is
// swapped: D [128 x N] = W_i[m0 : m0 + 128, :] . X_i^T, the weight tile the A
// operand (M = 128 rows of the output dimension), the batch the N side (N =
// the batch rounded up to 16, at most 256 per CTA; TMA zero-fills rows past
// the batch).  One CTA per (M tile, head, N tile): warp 0 streams K in
// 64-element chunks (A 16 KB + B N x 128 B per stage, 128-byte swizzle) into
// a ring, one thread of warp 1 issues tcgen05.mma (K = 16 each) into a TMEM
// accumulator of N fp32 columns, and warps 2-5 read it back (TMEM lane r =
// output row m0 + r, column = batch row), round to 16 bits, stage the tile
// in the (by then idle) ring as [N][128] and write Y[b, i, m0 : m0 + 128]
// with two bulk tensor stores.  Every wait is bounded; a timeout sets the
// error flag, the CTA stops issuing, waits for its copies and MMAs in
// flight, frees TMEM and writes nothing.
//
// The kernel is launched as a programmatic dependent of the previous kernel
// on the stream: its CTAs may start while that kernel finishes.  The
// weights do not depend on it, so the producer requests the first stages'
// weight boxes at once and waits (griddepcontrol.wait) only before the
// activation boxes; every global write follows that wait.  Each CTA lets the
// next kernel start launching as soon as it runs.
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr int kGemmThreads = 192;       // warp 0 TMA, warp 1 MMA (+ TMEM), warps 2-5 epilogue
constexpr int kChunk = 64;              // K elements per stage: one 128-byte swizzle row
constexpr int kATileBytes = 128 * 128;  // 128 weight rows x 128 B

// The ring, also the epilogue's staging area ([n_tile][128] 16-bit values).
__host__ __device__ __forceinline__ int ring_bytes(const HeadGemmParams& p) {
  const int ring = p.stages * (kATileBytes + p.n_tile * 128);
  const int staging = p.n_tile * 256;
  return ring > staging ? ring : staging;
}

// At most 79 registers, so that four CTAs fit an SM's register file (the
// q_abs GEMM's 512 CTAs then run as one wave).
template <bool kBF16>
__global__ void __launch_bounds__(kGemmThreads, 4)
    head_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_y, const HeadGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const int stage_bytes = kATileBytes + p.n_tile * 128;  // a multiple of 1024
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes(p));
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + S);
  const uint32_t done_bar = smem_u32(bars + 2 * S);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 2 * S + 2);

  const int mt = blockIdx.x, head = blockIdx.y, n0 = blockIdx.z * p.n_tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.k / kChunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(done_bar, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_x);
      const int w_row = head * p.m + mt * 128;
      // The first stages' weight boxes need nothing from the previous
      // kernel; its activations (X) may, so they follow griddepcontrol.wait.
      const int first = nk < S ? nk : S;
      for (int c = 0; c < first; ++c) {
        const uint32_t st = smem_u32(smem + c * stage_bytes);
        mbar_arrive_expect_tx(full0 + 8 * c, static_cast<uint32_t>(stage_bytes));
        tma_load_2d(st, &tm_w, c * kChunk, w_row, full0 + 8 * c);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int issued = 0;
      for (int c = 0; c < nk; ++c) {
        const int s = c % S;
        const uint32_t st = smem_u32(smem + s * stage_bytes);
        if (c >= first) {
          if (!mbar_wait_or_abort(empty0 + 8 * s, ((c / S) & 1) ^ 1, p.err_flag, abort)) break;
          mbar_arrive_expect_tx(full0 + 8 * s, static_cast<uint32_t>(stage_bytes));
          tma_load_2d(st, &tm_w, c * kChunk, w_row, full0 + 8 * s);
        }
        tma_load_3d(st + kATileBytes, &tm_x, c * kChunk, head, n0, full0 + 8 * s);
        ++issued;
      }
      // Never leave with copies in flight: wait (bounded) for the last phase
      // of every stage that was filled.
      for (int c = max(0, issued - S); c < issued; ++c)
        if (!mbar_wait(full0 + 8 * (c % S), (c / S) & 1, p.err_flag)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBF16, 128, p.n_tile, false, false);
      for (int c = 0; c < nk; ++c) {
        const int s = c % S;
        if (!mbar_wait_or_abort(full0 + 8 * s, (c / S) & 1, p.err_flag, abort)) break;
        tc_fence_after();
        const uint32_t st = smem_u32(smem + s * stage_bytes);
        const uint64_t da = smem_desc_sw128(st, 16, 1024);
        const uint64_t db = smem_desc_sw128(st + kATileBytes, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks)  // 32 bytes further along K per step
          tc_mma_f16(tmem, da + 2 * ks, db + 2 * ks, idesc, (c | ks) != 0 ? 1u : 0u);
        tc_commit(empty0 + 8 * s);
      }
      // Arrives once every MMA issued above has completed (also after an abort).
      tc_commit(done_bar);
    }
  } else {
    // Epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31.
    const bool ok = mbar_wait_or_abort(done_bar, 0, p.err_flag, abort);
    tc_fence_after();
    if (ok && !*abort) {
      // Every MMA has completed, so the ring is idle: stage the tile there as
      // two boxes [n_tile][64] (output rows m0 .. m0 + 63, m0 + 64 ..), one
      // 16-bit value per (batch row, output row); a warp's 32 lanes write 64
      // contiguous bytes per batch row.
      const int q = warp & 3;
      const int r = q * 32 + lane;  // output row within the tile (TMEM lane)
      const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
      uint16_t* stage = reinterpret_cast<uint16_t*>(smem) + (r >> 6) * (p.n_tile * 64) + (r & 63);
      for (int j = 0; j * 32 < p.n_tile; ++j) {
        float v[32];
        tmem_ld32(tmem + lane_base + j * 32, v);
        tc_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (j * 32 + k < p.n_tile) stage[(j * 32 + k) * 64] = round1<kBF16>(v[k]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (warp == 2 && lane == 0) {
        // Rows past the batch fall outside the tensor and are not written.
        const uint32_t src = smem_u32(smem);
        tma_store_3d(&tm_y, mt * 128, head, n0, src);
        tma_store_3d(&tm_y, mt * 128 + 64, head, n0, src + p.n_tile * 128);
        bulk_commit_group();
        bulk_wait_read_all();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
  if (warp == 2 && lane == 0) bulk_wait_all();
}

}  // namespace

int head_gemm_smem_bytes(const HeadGemmParams& p) {
  const int need = 1024 + ring_bytes(p) + (2 * p.stages + 4) * 8;
  // Keep (resident CTAs) x (TMEM columns) within the SM's 512 columns: ask
  // for enough shared memory that no more than 512 / tmem_cols CTAs fit.
  const int max_ctas = 512 / p.tmem_cols;
  const int floor_bytes = 233472 / (max_ctas + 1) + 1024;
  return need > floor_bytes ? need : floor_bytes;
}

// Raise the kernel's dynamic shared-memory limit once per process and
// device (not per call, so that calls can be captured into CUDA graphs).
template <bool kBF16>
cudaError_t allow_smem() {
  static cudaError_t status[64];
  static bool done[64] = {false};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    status[dev] = cudaFuncSetAttribute(head_gemm_kernel<kBF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    // All of the SM's unified L1 / shared storage as shared memory, so that
    // as many CTAs stay resident as their shared memory and TMEM allow (the
    // default split left 3 of the q_abs GEMM's 42 KB CTAs per SM: two waves).
    if (status[dev] == cudaSuccess)
      status[dev] = cudaFuncSetAttribute(head_gemm_kernel<kBF16>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
    done[dev] = true;
  }
  return status[dev];
}

cudaError_t launch_head_gemm(const HeadGemmParams& p, const CUtensorMap& tm_w,
                             const CUtensorMap& tm_x, const CUtensorMap& tm_y, bool bf16,
                             cudaStream_t stream) {
  if (p.batch <= 0 || p.heads <= 0) return cudaSuccess;
  const int smem = head_gemm_smem_bytes(p);
  if (smem > 232448) return cudaErrorInvalidValue;
  const dim3 grid(p.m / 128, p.heads, (p.batch + p.n_tile - 1) / p.n_tile);
  const cudaError_t e = bf16 ? allow_smem<true>() : allow_smem<false>();
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch (see the kernel's comment).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) return cudaLaunchKernelEx(&cfg, head_gemm_kernel<true>, tm_w, tm_x, tm_y, p);
  return cudaLaunchKernelEx(&cfg, head_gemm_kernel<false>, tm_w, tm_x, tm_y, p);
}

}  // namespace decattn
