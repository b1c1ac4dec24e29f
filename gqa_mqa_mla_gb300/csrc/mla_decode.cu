// mla_decode.cu -- absorbed multi-head latent attention decode, split-KV
// partial kernel on tcgen05 / TMEM, sm_103a.
//
// Absorbed MLA ("MQA, GQA, and MLA", section 5, KEY TRICK; "Why GQA's KV
// Cache Savings Don't Fully Reduce TPOT", "What Makes MLA Different"): the
// 128 query heads arrive pre-multiplied by W_uk (512-d) plus a 64-d
// decoupled-RoPE query; each cached token is one 576-element row (512-d
// latent c_t, then the 64-d RoPE key shared by all heads).  For head i
//     s_t = scale * (q_abs_i . c_t + q_rope_i . kr_t),  out_i = sum_t p_t c_t.
// Both contractions are dense 128-row GEMM tiles: S = Q C^T (K = 576) and
// O = P C_lat (N = 512).
//
// Work split: a cluster of two CTAs handles one (split, sequence).
//   CTA r = 0 holds latent columns [0, 256);
//   CTA r = 1 holds latent columns [256, 512) and the RoPE columns.
// Each CTA loads only its columns of every 32-token cache tile (every byte of
// the cache is read once), computes a partial score tile S_r = Q_r C_r^T into
// TMEM, and sends it to its peer through distributed shared memory
// (st.async, counted on the peer's mbarrier).  Both CTAs then hold the full
// S = S_0 + S_1 (identical bits on both sides), run the same fp32 online
// softmax, and each accumulates its own 256-column half of O = P C_lat in
// TMEM: the latent columns a CTA loads for S are exactly the value columns
// it needs for its half of O.  No FLOP is duplicated.
//
// Per CTA (192 threads):
//   warps 0-3  softmax / epilogue: thread h owns head h = TMEM lane h;
//   warp 4     TMA producer: Q once, then the cache tiles through a
//              3-stage ring, walking the block table;
//   warp 5     TMEM allocator and the single MMA-issuing thread.
// TMEM columns: O [0, 256) fp32, S double buffer [256, 288) and [288, 320).
//
// Online softmax in the log2 domain with lazy rescaling: the running max
// used for the exponentials only moves (and O is rescaled in TMEM) when a new
// score exceeds it by more than 2^8; otherwise p <= 256 stays exact in bf16 /
// fp16 range and the final division by l uses the same stale max.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr int kT = 32;                          // tokens per tile
constexpr int kStages = 3;                      // cache ring depth
constexpr int kChunk = 64;                      // columns per 128-byte swizzle row
constexpr int kQChunkBytes = kMlaHeads * 128;   // [128 heads][64 cols] bf16 = 16 KB
constexpr int kCChunkBytes = kT * 128;          // [32 tokens][64 cols] = 4 KB
constexpr int kMaxChunks = 5;                   // CTA 1: 4 latent chunks + 1 RoPE chunk
constexpr int kStageBytes = kMaxChunks * kCChunkBytes;  // 20 KB
constexpr int kPBytes = kMlaHeads * 128;        // P tile [128 heads][32 tok] in 128-B rows
constexpr int kRecvBytes = kMlaHeads * kT * 4;  // fp32 partial scores [128][32]
constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + kMaxChunks * kQChunkBytes;   // 80 KB
constexpr int kOffP = kOffRing + kStages * kStageBytes;       // +60 KB
constexpr int kOffRecv = kOffP + 2 * kPBytes;                 // +32 KB
constexpr int kOffBars = kOffRecv + 2 * kRecvBytes;           // +32 KB
constexpr int kSmemBytes = 1024 + kOffBars + 256;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kTmemO = 0;
constexpr int kTmemS = 256;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when p could exceed 2^8

// mbarrier slots (8 bytes each) inside the barrier area
enum : int {
  kBarQ = 0,
  kBarKvFull = 1,                    // kStages
  kBarKvEmpty = kBarKvFull + kStages,
  kBarSFull = kBarKvEmpty + kStages, // 2
  kBarSFree = kBarSFull + 2,         // 2
  kBarPFull = kBarSFree + 2,         // 2
  kBarPvDone = kBarPFull + 2,        // 2
  kBarRecv = kBarPvDone + 2,         // 2
  kBarDrain = kBarRecv + 2,
  kNumBars = kBarDrain + 1
};
static_assert(kNumBars * 8 + 16 <= 256, "barrier area");

template <bool kBF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_partial_kernel(const __grid_constant__ CUtensorMap tm_qa,
                       const __grid_constant__ CUtensorMap tm_qr,
                       const __grid_constant__ CUtensorMap tm_c, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBars;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile int* abort_word = reinterpret_cast<volatile int*>(smem + kOffBars + kNumBars * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBars + kNumBars * 8 + 4);

  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int split = blockIdx.x >> 1;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qchunks = rank == 0 ? 4 : 5;  // Q / cache column chunks this CTA holds
  const int col0 = static_cast<int>(rank) * 256;  // first latent column of this CTA

  // ---------------- range and data checks (identical on both CTAs)
  const int seq_len = p.seq_lens[b];
  int bad = 0;
  if (seq_len < 0 || seq_len > p.max_seq_len) {
    bad = 1;
    if (threadIdx.x == 0 && split == 0 && rank == 0) flag_error(p.err_flag, kFlagBadSeqLen);
  }
  const int t_begin = split * p.tokens_per_split;
  const int t_end = bad ? t_begin : min(seq_len, t_begin + p.tokens_per_split);
  if (!bad && t_end > t_begin) {
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const int k1 = (t_end - 1) >> p.log2_block_size;
    for (int k = (t_begin >> p.log2_block_size) + threadIdx.x; k <= k1; k += blockDim.x) {
      const int id = bt[k];
      if (id < 0 || id >= p.num_blocks) {
        bad = 1;
        if (rank == 0) flag_error(p.err_flag, kFlagBadBlock);
      }
    }
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKvFull + s), 1);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSFree + s), 128);
      mbar_init(bar(kBarPFull + s), 128);
      mbar_init(bar(kBarPvDone + s), 1);
      mbar_init(bar(kBarRecv + s), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  bad = __syncthreads_or(bad);
  cluster_sync();  // both CTAs' barriers exist before any remote traffic

  const size_t head0 = static_cast<size_t>(b) * kMlaHeads;
  if (bad || t_end <= t_begin) {
    for (int e = threadIdx.x; e < kMlaHeads * 256; e += blockDim.x) {
      const int h = e >> 8, c = col0 + (e & 255);
      if (p.n_split == 1) {
        static_cast<uint16_t*>(p.out)[(head0 + h) * kMlaDc + c] = 0;
      } else {
        p.part_o[((head0 + h) * p.n_split + split) * kMlaDc + c] = 0.f;
        if (rank == 0 && (e & 255) == 0)
          p.part_lse[(head0 + h) * p.n_split + split] = bad ? DECATTN_POISON_LSE : kNegInf;
      }
    }
    cluster_sync();
    return;
  }

  const int n_tiles = (t_end - t_begin + kT - 1) / kT;

  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_qa);
      tma_prefetch_desc(&tm_qr);
      tma_prefetch_desc(&tm_c);
      const int qy = static_cast<int>(head0);
      mbar_arrive_expect_tx(bar(kBarQ), static_cast<uint32_t>(n_qchunks * kQChunkBytes));
      for (int c = 0; c < 4; ++c)
        tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &tm_qa, col0 + c * kChunk, qy, bar(kBarQ));
      if (rank == 1) tma_load_2d(sbase + kOffQ + 4 * kQChunkBytes, &tm_qr, 0, qy, bar(kBarQ));

      const uint64_t policy = policy_evict_first();
      const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
      const int bs = p.block_size;
      const int rows_per_box = bs < kT ? bs : kT;
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int s = it % kStages;
        if (!mbar_wait_or_abort(bar(kBarKvEmpty + s), ((it / kStages) & 1) ^ 1, p.err_flag,
                                abort_word))
          break;
        const int t0 = t_begin + it * kT;
        const int nval = min(kT, t_end - t0);
        const int nbox = (nval + rows_per_box - 1) / rows_per_box;
        const uint32_t st = sbase + kOffRing + s * kStageBytes;
        mbar_arrive_expect_tx(bar(kBarKvFull + s),
                              static_cast<uint32_t>(nbox * n_qchunks * rows_per_box * 128));
        for (int k = 0; k < nbox; ++k) {
          const int t = t0 + k * rows_per_box;
          const int row = bt[t >> p.log2_block_size] * bs + (t & (bs - 1));
          const uint32_t off = static_cast<uint32_t>(k * rows_per_box * 128);
          for (int c = 0; c < n_qchunks; ++c) {
            const int x = c < 4 ? col0 + c * kChunk : kMlaDc;  // chunk 4 = RoPE columns
            tma_load_2d_hint(st + c * kCChunkBytes + off, &tm_c, x, row, bar(kBarKvFull + s),
                             policy);
          }
        }
        ++issued;
      }
      for (int it = max(0, issued - kStages); it < issued; ++it)
        if (!mbar_wait_or_abort(bar(kBarKvFull + it % kStages), (it / kStages) & 1, p.err_flag,
                                abort_word))
          break;
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBF16, 128, kT, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kBF16, 128, 256, false, true);
      bool ok = mbar_wait_or_abort(bar(kBarQ), 0, p.err_flag, abort_word);
      auto issue_pv = [&](int j) -> bool {
        const int pb = j & 1;
        if (!mbar_wait_or_abort(bar(kBarPFull + pb), (j >> 1) & 1, p.err_flag, abort_word))
          return false;
        tc_fence_after();
        const uint32_t st = sbase + kOffRing + (j % kStages) * kStageBytes;
        const uint32_t pbuf = sbase + kOffP + pb * kPBytes;
#pragma unroll
        for (int ks = 0; ks < kT / 16; ++ks) {
          const uint64_t a = smem_desc_sw128(pbuf + ks * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(st + ks * 2048, kCChunkBytes, 1024);
          tc_mma_f16(tmem + kTmemO, a, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(bar(kBarPvDone + pb));
        tc_commit(bar(kBarKvEmpty + j % kStages));
        return true;
      };
      for (int it = 0; ok && it < n_tiles; ++it) {
        const int s = it % kStages;
        const int sb = it & 1;
        if (!mbar_wait_or_abort(bar(kBarKvFull + s), (it / kStages) & 1, p.err_flag, abort_word) ||
            !mbar_wait_or_abort(bar(kBarSFree + sb), ((it >> 1) & 1) ^ 1, p.err_flag,
                                abort_word)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = sbase + kOffRing + s * kStageBytes;
        for (int c = 0; c < n_qchunks; ++c) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t a = smem_desc_sw128(sbase + kOffQ + c * kQChunkBytes + ks * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(st + c * kCChunkBytes + ks * 32, 16, 1024);
            tc_mma_f16(tmem + kTmemS + sb * kT, a, bd, idesc_s, (c > 0 || ks > 0) ? 1u : 0u);
          }
        }
        tc_commit(bar(kBarSFull + sb));
        if (it > 0 && !issue_pv(it - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) issue_pv(n_tiles - 1);
      // Wait (bounded) until every MMA this thread issued has completed.
      tc_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, p.err_flag);
    }
  } else {
    // ---------------- softmax warps: thread h owns head h
    const int h = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_used = kNegInf, l = 0.f;
    bool ok = true;
    for (int it = 0; it < n_tiles; ++it) {
      const int sb = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      const int nval = min(kT, t_end - (t_begin + it * kT));
      if (!mbar_wait_or_abort(bar(kBarSFull + sb), ph, p.err_flag, abort_word)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[32];
      tmem_ld32(tmem + lane_base + kTmemS + sb * kT, s);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(kBarSFree + sb));

      // Exchange partial scores with the peer CTA (row h, 128 bytes).
      if (h == 0) mbar_arrive_expect_tx(bar(kBarRecv + sb), kRecvBytes);
      {
        const uint32_t dst = sbase + kOffRecv + sb * kRecvBytes + h * 128;
        const uint32_t rb = mapa_shared(bar(kBarRecv + sb), peer);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_async_v4(mapa_shared(dst + ((k ^ (h & 7)) << 4), peer), rb, s[4 * k], s[4 * k + 1],
                      s[4 * k + 2], s[4 * k + 3]);
      }
      if (!mbar_wait_or_abort(bar(kBarRecv + sb), ph, p.err_flag, abort_word, true)) {
        ok = false;
        break;
      }
      {
        const float4* rv =
            reinterpret_cast<const float4*>(smem + kOffRecv + sb * kRecvBytes + h * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 x = rv[k ^ (h & 7)];
          s[4 * k] += x.x;
          s[4 * k + 1] += x.y;
          s[4 * k + 2] += x.z;
          s[4 * k + 3] += x.w;
        }
      }
      // Scale into the log2 domain, mask tokens past the end, tile max.
      float mt = kNegInf;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        s[k] = k < nval ? s[k] * p.scale_log2 : kNegInf;
        mt = fmaxf(mt, s[k]);
      }
      // P buffer (it & 1) was read by PV(it - 2): wait before overwriting it.
      if (it >= 2 &&
          !mbar_wait_or_abort(bar(kBarPvDone + sb), ((it - 2) >> 1) & 1, p.err_flag, abort_word)) {
        ok = false;
        break;
      }
      const bool need = mt > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_used;
        const float factor = need ? ex2(m_used - m_new) : 1.f;  // 0 when m_used = -inf
        if (it > 0) {
          // O must include PV(it - 1) before it is rescaled.
          if (!mbar_wait_or_abort(bar(kBarPvDone + ((it - 1) & 1)), ((it - 1) >> 1) & 1,
                                  p.err_flag, abort_word)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            float o[32];
            tmem_ld32(tmem + lane_base + kTmemO + c, o);
            tc_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= factor;
            tmem_st32(tmem + lane_base + kTmemO + c, o);
          }
          tc_wait_st();
        }
        l *= factor;
        m_used = m_new;
      }
      // p = 2^(s - m_used), row sum, P row in the 128-byte-swizzled K-major tile.
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float p0 = ex2(s[2 * k] - m_used), p1 = ex2(s[2 * k + 1] - m_used);
        l += p0 + p1;
        pk[k] = pack2<kBF16>(p0, p1);
      }
      {
        uint8_t* prow = smem + kOffP + sb * kPBytes + h * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(prow + ((k ^ (h & 7)) << 4)) =
              make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
      if (nval < kT) {
        // Value rows past the sequence end may hold anything (even NaN): zero
        // them so that P = 0 there contributes exactly nothing.
        uint8_t* st = smem + kOffRing + (it % kStages) * kStageBytes;
        for (int e = h; e < (kT - nval) * 4 * 8; e += 128) {
          const int row = nval + e / 32, c = (e / 8) & 3, q = e & 7;
          *reinterpret_cast<uint4*>(st + c * kCChunkBytes + row * 128 + q * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + sb));
    }

    // ---------------- epilogue: O row h (this CTA's 256 columns) / l
    if (ok && mbar_wait_or_abort(bar(kBarPvDone + ((n_tiles - 1) & 1)), ((n_tiles - 1) >> 1) & 1,
                                 p.err_flag, abort_word)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        float o[32];
        tmem_ld32(tmem + lane_base + kTmemO + c, o);
        tc_wait_ld();
        if (p.n_split == 1) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                (head0 + h) * kMlaDc + col0 + c);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[k] = make_uint4(pack2<kBF16>(o[8 * k] * inv, o[8 * k + 1] * inv),
                                pack2<kBF16>(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                                pack2<kBF16>(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                                pack2<kBF16>(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.part_o + ((head0 + h) * p.n_split + split) * kMlaDc + col0 + c);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv,
                                 o[4 * k + 3] * inv);
        }
      }
      if (p.n_split > 1 && rank == 0)
        p.part_lse[(head0 + h) * p.n_split + split] = l > 0.f ? m_used + lg2(l) : kNegInf;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // the peer may still be reading our partial scores until here
}

template <bool kBF16>
cudaError_t launch_t(const MlaParams& p, const CUtensorMap& tqa, const CUtensorMap& tqr,
                     const CUtensorMap& tc, cudaStream_t stream) {
  auto kern = mla_partial_kernel<kBF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * p.n_split, p.batch);
  kern<<<grid, kThreads, kSmemBytes, stream>>>(tqa, tqr, tc, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mla_partial(const MlaParams& p, const CUtensorMap& tm_qa,
                               const CUtensorMap& tm_qr, const CUtensorMap& tm_c, bool bf16,
                               cudaStream_t stream) {
  if (p.block_size > kT && (p.block_size % kT) != 0) return cudaErrorNotSupported;
  return bf16 ? launch_t<true>(p, tm_qa, tm_qr, tm_c, stream)
              : launch_t<false>(p, tm_qa, tm_qr, tm_c, stream);
}

}  // namespace decattn
