// gqa_wide.cu -- split-KV partial kernel for wide query groups (GQA with
// many query heads per KV head, and MQA) over a 16-bit paged KV cache, on
// tcgen05 / TMEM, sm_103a; also over an 8-bit e4m3 cache.
//
// "MQA, GQA, and MLA", section 4: a KV head shared by G query heads serves
// G dot products per cached byte, so the attention arithmetic per byte grows
// with G (MQA: G = h).  Past a few dozen query heads per KV head the two
// contractions per token, not the cache bytes, set the pace of a CUDA-core or
// mma.sync kernel.  Here both run on the tensor cores, with the query group
// as the MMA's M:
//     S = Q_j K^T    M = 64 query heads (the group, zero-padded), N = 64 tokens, K = 128
//     O += P V       M = 64, N = 128 head dims, K = 64 tokens
// One CTA handles one (split, KV head j, sequence b), as the other GQA
// partial kernels, and writes the same outputs (the final rows for one
// split, else fp32 partials for the log-sum-exp combine).
//
// Operand placement:
//   Q_j        shared memory, [2 halves][64 rows][128 B], 128-byte swizzled
//              K-major, written once by the softmax threads    A of S
//   K, V tiles TMA ring (kStages), [2 halves][64 tokens][128 B], 128-byte
//              swizzled, one box per 64-column half and block:
//                                                     K        B of S (K-major)
//                                                     V        B of PV (MN-major)
//   P(j)       shared memory, [64 rows][64 tokens x 2 B], two buffers  A of PV
//   S(j)       TMEM, two buffers of 64 fp32 columns
//   O          TMEM, 128 fp32 columns
// An M = 64 MMA writes rows 0-15 to TMEM lanes 0-15, rows 16-31 to lanes
// 32-47, rows 32-47 to 64-79 and rows 48-63 to 96-111.
//
// Warps (352 threads, two CTAs per SM):
//   0-7  load Q; online softmax of S(j) into P(j); lazy O rescale; epilogue.
//        Warp w reads TMEM lane quarter w % 4 (rows 16 (w % 4) .. + 15) with
//        the 16x32bx2 shape: lanes t and t + 16 own row 16 (w % 4) + t, in
//        the two 32-column halves of S; w / 4 picks the 16 columns of each
//        half (and the 32 of each 64-column half of O) whose exponentials
//        and outputs a thread computes.  The two warps of a quarter both
//        read all 64 score columns of their rows and take the same maximum.
//   8    TMA producer of the K tiles (walks the block table); a K stage is
//        free again once S(j) has read it;
//   10   TMA producer of the V tiles; a V stage is free after PV(j).
//   9    TMEM allocator and MMA issuer (one elected lane): S(j + 1) (its K
//        tile landed, its S buffer read) and O += P(j) V(j) (P(j) written)
//        go in whichever order their operands arrive, S first when both are
//        ready, so that S(j + 1) runs while the softmax works on tile j.
// While an MMA runs, threads touch only TMEM columns and shared memory it
// neither reads nor writes: S(j + 1) (S buffer (j + 1) & 1, K) runs while the
// softmax writes P(j) and zeroes stale V(j) rows; O is rescaled only after
// O += P(j - 1) V(j - 1) has completed, and P(j) is written only after
// O += P(j - 2) V(j - 2) (the last reader of its buffer) has.
//
// An 8-bit (e4m3) cache takes the same pipeline with three changes: the K
// stage, as it lands, is the B operand of S = Q K^T on kind::f8f6f4, whose A
// operand is Q split into e4m3 terms (two for a bf16 query, three for fp16,
// each row scaled by a power of two that the softmax undoes: exact except
// for parts below 2^-18 of the row's largest element); the
// softmax threads convert each landed V tile into one of two 16-bit slabs
// (e4m3 -> f16 is exact) before they publish P(j), the slab being the B
// operand of O += P V on f16; and the rings hold two 8 KB stages.  A
// conversion warp of its own would put the conversion (~1.3k cycles per 8 KB
// tile on one sub-partition) on the serial path; spread over the eight
// softmax warps it is a few hundred cycles.
//
// Online softmax in the log2 domain with lazy rescaling, as the MLA kernel:
// the running max used for the exponentials (and O in TMEM) moves only when
// a new score exceeds it by more than 2^8; the final division by l uses the
// same stale max.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gqa_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr int kM = 64;                            // query heads per CTA (MMA rows)
// K / V ring depth: two stages keep a CTA at ~100 KB of shared memory, so
// that two CTAs share an SM.  One CTA streams about 38 GB/s however deep
// its ring (4 and 6 stages measured the same); two CTAs per SM reach the
// copy rate (70B-shaped layer, 32 query heads per KV head, B = 64: 110.9 us
// with one CTA per SM and 4 stages, 91.9 us with two and 2 stages).
constexpr int kStages = 2;
constexpr int kHalf = kTile * 128;                // one 64-column half of a tile: 8 KB
constexpr int kKvTile = 2 * kHalf;                // a 16-bit K or V tile: 16 KB
constexpr int kF8Tile = kTile * 128;              // an 8-bit K or V tile: 8 KB
constexpr int kF8Stages = 2;                      // 8-bit K / V ring depth
constexpr int kQBytes = 2 * kM * 128;             // 16 KB
constexpr int kPBytes = kM * kTile * 2;           // 8 KB per buffer
constexpr int kBarBytes = 256;
constexpr int kSoftmaxThreads = 256;
constexpr int kWarpProducerK = 8, kWarpMma = 9, kWarpProducerV = 10;
constexpr int kThreads = kSoftmaxThreads + 96;
constexpr int kTmemCols = 256;
constexpr int kTmemO = 0;                         // 128 columns
constexpr int kTmemS = 128;                       // S(j): 128 + 64 (j & 1)
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;         // log2 units: p stays <= 2^8

// Shared-memory layout.  16-bit cache: K and V rings of 16-bit tiles (the
// MMA operands), Q, two P buffers.  8-bit cache: K and V rings of 8-bit
// tiles (the K stage is the score MMA's operand as it lands), two 16-bit V
// slabs (the softmax threads convert each landed V tile into one, f16, the
// operand of O += P V), Q as e4m3 terms, two P buffers — at most ~106 KB, so
// that two CTAs still share an SM.
constexpr int kQTermBytes = kM * 128;             // one e4m3 term of Q: [64 rows][128 codes]
template <bool kBF16, bool kF8>
struct WLayout {
  static constexpr int kRing = kF8 ? kF8Stages : kStages;
  static constexpr int kStageBytes = kF8 ? kF8Tile : kKvTile;
  // e4m3 terms of an 8-bit cache's Q: a bf16 query (8 significant bits) is
  // exactly two terms, an fp16 query (11) three.
  static constexpr int kQTerms = kF8 ? (kBF16 ? 2 : 3) : 0;
  static constexpr int kOffK = 0;                                          // K ring
  static constexpr int kOffV = kOffK + kRing * kStageBytes;                // V ring
  static constexpr int kOffV16 = kOffV + kRing * kStageBytes;              // 8-bit: f16 V
  static constexpr int kOffQ = kOffV16 + (kF8 ? 2 * kKvTile : 0);
  static constexpr int kPBuffers = 2;
  static constexpr int kOffP = kOffQ + (kF8 ? kQTerms * kQTermBytes : kQBytes);
  static constexpr int kOffBars = kOffP + kPBuffers * kPBytes;
  // Row sums of the two column groups, then (8-bit cache) 1 / alpha per row.
  static constexpr int kOffRed = kOffBars + kBarBytes;
  static constexpr int kSmemBytes = 1024 + kOffRed + 3 * kM * 4;
};
static_assert(WLayout<true, false>::kSmemBytes <= 232448 / 2 - 1024, "two 16-bit CTAs per SM");
static_assert(WLayout<false, true>::kSmemBytes <= 232448 / 2 - 1024, "two 8-bit CTAs per SM");

enum : int {
  kBarQ = 0,                        // Q in shared memory (256 arrivals)
  kBarFullK = 1,                    // ring stages: K tile landed (TMA bytes)
  kBarFullV = kBarFullK + kF8Stages,  // ring stages: V tile landed
  kBarEmptyK = kBarFullV + kF8Stages, // ring stages: K stage free (S(j) read it)
  kBarEmptyV = kBarEmptyK + kF8Stages,// ring stages: V stage free (PV(j) read it / converted)
  kBarSFull = kBarEmptyV + kF8Stages, // 2: S(j) computed
  kBarSFree = kBarSFull + 2,        // 2: S(j) read by the softmax (256 arrivals)
  kBarPFull = kBarSFree + 2,        // 2: P(j) written (256 arrivals)
  kBarPvDone = kBarPFull + 2,       // 2: O += P(j) V(j) complete
  kBarSum = kBarPvDone + 2,         // row sums exchanged (256 arrivals)
  kBarDrain = kBarSum + 1,          // every MMA complete
  kNumBars = kBarDrain + 1
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier area");
static_assert(kTmemS + 128 <= kTmemCols, "tensor memory columns");

// Issue the copies of one 64-token K or V tile (16-bit cache) into `dst`,
// called by the whole producer warp: one box per 64-column half (blocks of
// 64 tokens or more: lane 0), or per block and half for smaller blocks (lane
// k copies the tile's block k).  `id` is the block id of the lane's block and
// `bytes` the total the copies complete on `full`, announced by lane 0 first.
__device__ __forceinline__ void load_tile(const CUtensorMap* tm, int id, int nblk, int bs,
                                          int row_in_block, int x0, uint32_t bytes,
                                          uint32_t dst, uint32_t full, uint64_t policy,
                                          int lane) {
  if (lane == 0) mbar_arrive_expect_tx(full, bytes);
  __syncwarp();
  if (lane < nblk) {
    const int row = id * bs + row_in_block;
    const uint32_t off = static_cast<uint32_t>(lane * bs * 128);
    tma_load_2d_hint(dst + off, tm, x0, row, full, policy);
    tma_load_2d_hint(dst + kHalf + off, tm, x0 + 64, row, full, policy);
  }
}

// The same tile of an 8-bit cache: one 128-byte box row per token (the whole
// 128-d head), one box per block (or one 64-row box for blocks of 64 tokens
// or more).
__device__ __forceinline__ void load_tile8(const CUtensorMap* tm, int id, int nblk, int bs,
                                           int row_in_block, int x0, uint32_t bytes,
                                           uint32_t dst, uint32_t full, uint64_t policy,
                                           int lane) {
  if (lane == 0) mbar_arrive_expect_tx(full, bytes);
  __syncwarp();
  if (lane < nblk)
    tma_load_2d_hint(dst + static_cast<uint32_t>(lane * bs * 128), tm, x0,
                     id * bs + row_in_block, full, policy);
}

// Convert one landed 8-bit V tile ([64 tokens][128 codes], 128-byte swizzle)
// into the 16-bit operand layout ([2 halves][64 tokens][128 B], 128-byte
// swizzle), e4m3 -> f16 (exact), by the 256 softmax threads: thread t takes
// the 16-byte code chunks t and t + 256; chunk c of row r (dims 16c .. 16c +
// 15) becomes 16-byte chunks 2 (c % 4) and 2 (c % 4) + 1 of half c / 4.
// Rows outside [zlo, zhi) are written as zeros (tokens before a window or
// past the end, whose slots may hold anything, even NaN codes).
__device__ __forceinline__ void convert_v8(const uint8_t* src, uint8_t* dst, int t, int zlo,
                                           int zhi) {
#pragma unroll
  for (int i = 0; i < (kTile * 8) / kSoftmaxThreads; ++i) {
    const int e = t + kSoftmaxThreads * i;
    const int r = e >> 3, c = e & 7;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
    if (r >= zlo && r < zhi) {
      const uint4 w = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ (r & 7)) << 4));
      e4m3x4_to_f16x2(w.x, lo.x, lo.y);
      e4m3x4_to_f16x2(w.y, lo.z, lo.w);
      e4m3x4_to_f16x2(w.z, hi.x, hi.y);
      e4m3x4_to_f16x2(w.w, hi.z, hi.w);
    }
    uint8_t* row = dst + (c >> 2) * kHalf + r * 128;
    const int c0 = 2 * (c & 3);
    *reinterpret_cast<uint4*>(row + ((c0 ^ (r & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) = hi;
  }
}

// Two floats rounded to e4m3 (nearest even; |x| <= 448 here): the two codes
// (x in the lower byte) and the rounded values.
__device__ __forceinline__ uint32_t e4m3_round2(float x, float y, float& rx, float& ry) {
  const uint32_t c = f32x2_to_e4m3x2(x, y);
  uint32_t h, unused;
  e4m3x4_to_f16x2(c, h, unused);
  const float2 v = unpack2<false>(h);
  rx = v.x;
  ry = v.y;
  return c;
}

// kF8: the cache holds e4m3 codes with per-KV-head scales (K's folds into the
// score scale, V's into the output).  S = Q K^T then runs as kind::f8f6f4 on
// the landed K codes, with Q split into e4m3 terms, and O += P V on f16
// operands (V converted by the softmax threads).
template <bool kBF16, bool kF8>
// (A minimum-blocks bound of 1 here made ptxas cap the registers at 168 and
// spill; without it the kernel takes under 100.)
__global__ void __launch_bounds__(kThreads)
    gqa_wide_kernel(const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const GqaParams p) {
  using L = WLayout<kBF16, kF8>;
  constexpr int kQTerms = L::kQTerms;
  constexpr bool kMmaBF16 = kBF16 && !kF8;  // operand type of O += P V (and 16-bit S)
  constexpr int kRing = L::kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kOffBars;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile int* abort_word = reinterpret_cast<volatile int*>(smem + L::kOffBars + kNumBars * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffBars + kNumBars * 8 + 8);

  const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;

  const GqaSpan span = gqa_span(p, split, j, b);
  const int w0 = span.w0, t_begin = span.t_begin, t_end = span.t_end;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), kSoftmaxThreads);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(bar(kBarFullK + s), 1);
      mbar_init(bar(kBarFullV + s), 1);
      mbar_init(bar(kBarEmptyK + s), 1);
      // 8-bit cache: one arrival per softmax warp once it has converted V(j).
      mbar_init(bar(kBarEmptyV + s), kF8 ? kSoftmaxThreads / 32 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSFree + i), kSoftmaxThreads);
      mbar_init(bar(kBarPFull + i), kSoftmaxThreads);
      mbar_init(bar(kBarPvDone + i), 1);
    }
    mbar_init(bar(kBarSum), kSoftmaxThreads);
    mbar_init(bar(kBarDrain), 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  const int bad = __syncthreads_or(span.bad);
  const size_t row0 = static_cast<size_t>(b) * p.h_q + static_cast<size_t>(j) * G;
  if (bad || t_end <= t_begin) {
    gqa_write_empty(p, row0, G, split, bad);
    return;
  }

  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n = (t_end - t_begin + kTile - 1) / kTile;

  if (warp == kWarpProducerK || warp == kWarpProducerV) {
    // ---------------- TMA producers, one warp for K and one for V (two
    // independent streams of 2 KB boxes for blocks of 16 tokens; one thread
    // issues a box about every 100 cycles).  The lanes hold the block ids of
    // the next 32 blocks, read with one coalesced load, so that no copy waits
    // on a block-table read of its own.
    const bool is_v = warp == kWarpProducerV;
    const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
    if (lane == 0) tma_prefetch_desc(tm);
    const uint64_t policy = policy_evict_first();
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const int x0 = j * kHeadDim;  // element (= byte, for an 8-bit cache) column of head j
    const int bs = p.block_size, lg = p.log2_block_size;
    const int kb_end = ((t_end - 1) >> lg) + 1;  // one past the range's last block
    const int bar_full = is_v ? kBarFullV : kBarFullK, bar_empty = is_v ? kBarEmptyV : kBarEmptyK;
    const uint32_t ring = sbase + (is_v ? L::kOffV : L::kOffK);
    constexpr int kStageBytes = L::kStageBytes;
    int cache0 = -(1 << 30), my_id = 0;
    int issued = 0;
    // Request tile `it` into its ring stage once the stage is free.
    auto request = [&](int it) -> bool {
      const int s = it % kRing;
      const uint32_t ph = static_cast<uint32_t>((it / kRing) & 1) ^ 1u;
      const int t0 = t_begin + it * kTile;
      const int nval = min(kTile, t_end - t0);
      const int kb0 = t0 >> lg;
      const int nblk = bs >= kTile ? 1 : (nval + bs - 1) >> lg;
      if (kb0 + nblk > cache0 + 32) {
        cache0 = kb0;
        my_id = kb0 + lane < kb_end ? bt[kb0 + lane] : 0;
      }
      const int id = __shfl_sync(0xffffffffu, my_id, kb0 - cache0 + min(lane, nblk - 1));
      const int rib = bs >= kTile ? (t0 & (bs - 1)) : 0;
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar(bar_empty + s), ph, p.err_flag, abort_word);
      if (__shfl_sync(0xffffffffu, w ? 1 : 0, 0) == 0) return false;
      if constexpr (kF8) {
        const uint32_t bytes = static_cast<uint32_t>(bs >= kTile ? kF8Tile : nblk * bs * 128);
        load_tile8(tm, id, nblk, bs, rib, x0, bytes, ring + s * kStageBytes, bar(bar_full + s),
                   policy, lane);
      } else {
        const uint32_t bytes = static_cast<uint32_t>(bs >= kTile ? kKvTile : nblk * 2 * bs * 128);
        load_tile(tm, id, nblk, bs, rib, x0, bytes, ring + s * kStageBytes, bar(bar_full + s),
                  policy, lane);
      }
      issued = it + 1;
      return true;
    };
    for (int it = 0; it < n; ++it)
      if (!request(it)) break;
    // Never leave the CTA with copies in flight: wait (bounded) for the
    // last phase of every stage that was filled.
    if (lane == 0)
      for (int it = max(0, issued - kRing); it < issued; ++it)
        if (!mbar_wait(bar(bar_full + it % kRing), (it / kRing) & 1, p.err_flag)) break;
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer: the whole warp runs the loop (uniform
    // operands), lane 0 waits, one elected lane issues and commits.
    const uint64_t dq = smem_desc_sw128(sbase + L::kOffQ, 16, 1024);
    const uint64_t dk = smem_desc_sw128(sbase + L::kOffK, 16, 1024);
    const uint64_t dp = smem_desc_sw128(sbase + L::kOffP, 16, 1024);
    const uint64_t dv = smem_desc_sw128(sbase + (kF8 ? L::kOffV16 : L::kOffV), kHalf, 1024);
    constexpr uint32_t idesc_s =
        kF8 ? idesc_e4m3(kM, kTile) : idesc_f16(kMmaBF16, kM, kTile, false, false);
    constexpr uint32_t idesc_o = idesc_f16(kMmaBF16, kM, kHeadDim, false, true);
    auto wait = [&](int bi, uint32_t parity) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar(bi), parity, p.err_flag, abort_word);
      return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    };
    // S(it) = Q K(it)^T.  16-bit: 8 k-steps of 16 dims; k-step ks sits in
    // half ks / 4 at byte 32 (ks % 4) of the swizzled rows.  8-bit: each of
    // the three Q terms against the landed codes, 4 k-steps of 32 dims at
    // byte 32 ks of the 128-byte rows.  (Descriptor units of 16 B.)  The
    // whole warp computes the operands; one elected lane issues.
    auto issue_s = [&](int it) {
      const int s = it % kRing;
      const uint32_t d = tmem + kTmemS + 64 * (it & 1);
      const uint64_t bk = dk + static_cast<uint64_t>((s * L::kStageBytes) >> 4);
      const uint32_t full = bar(kBarSFull + (it & 1));
      const uint32_t empty = bar(kBarEmptyK + s);
      if (elect_one()) {
        if constexpr (kF8) {
#pragma unroll
          for (int t = 0; t < kQTerms; ++t)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_f8(d, dq + static_cast<uint64_t>((t * kQTermBytes + ks * 32) >> 4),
                        bk + static_cast<uint64_t>((ks * 32) >> 4), idesc_s,
                        (t | ks) > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t off = static_cast<uint64_t>(((ks >> 2) * kHalf + (ks & 3) * 32) >> 4);
            tc_mma_f16(d, dq + off, bk + off, idesc_s, ks > 0 ? 1u : 0u);
          }
        }
        tc_commit(full);
        tc_commit(empty);
      }
      __syncwarp();
    };
    // O += P(it) V(it): 4 k-steps of 16 tokens; V is MN-major (the next 64
    // dims one half = 8 KB on, the next 8 tokens 1 KB on).  16-bit: V(it) is
    // its ring stage; 8-bit: the f16 slab, converted by the softmax threads
    // before they publish P(it).
    auto issue_pv = [&](int it) {
      const int s = it % kRing;  // 16-bit: the V ring stage; 8-bit: the f16 slab (it & 1)
      const uint64_t ap =
          dp + static_cast<uint64_t>(((it & 1) * kPBytes) >> 4);
      const uint64_t bv = dv + static_cast<uint64_t>((s * kKvTile) >> 4);
      const uint32_t done = bar(kBarPvDone + (it & 1));
      const uint32_t acc0 = it > 0 ? 1u : 0u;
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)
          tc_mma_f16(tmem + kTmemO, ap + static_cast<uint64_t>((ks * 32) >> 4),
                     bv + static_cast<uint64_t>((ks * 2048) >> 4), idesc_o, ks > 0 ? 1u : acc0);
        tc_commit(done);
        if constexpr (!kF8) tc_commit(bar(kBarEmptyV + s));
      }
      __syncwarp();
    };
    // Issue in whatever order the operands arrive: S(i) needs its K tile and
    // its S buffer (read by the softmax of tile i - 2), and may run at most
    // one tile ahead of the value GEMM; O += P(i) V(i) needs P(i) (and, for a
    // 16-bit cache, V(i)).  S goes first when both are ready, so that the
    // softmax always has the next scores.  Lane 0 probes the barriers without
    // blocking; the loop gives up (error flag, abort word) after the wait
    // limit without progress.
    auto probe = [&](int bi, uint32_t parity) { return mbar_test_wait(bar(bi), parity); };
    int ns = 0, np = 0;
    bool ok = wait(kBarQ, 0);
    uint64_t t_idle = 0;
    uint32_t spins = 0;
    while (ok && np < n) {
      int act = 0;  // 1: issue S(ns), 2: issue O += P(np) V(np)
      if (lane == 0) {
        if (ns < n && ns <= np + 1 &&
            (ns < 2 || probe(kBarSFree + (ns & 1), ((ns - 2) >> 1) & 1)) &&
            probe(kBarFullK + ns % kRing, (ns / kRing) & 1))
          act = 1;
        else if (np < ns && probe(kBarPFull + (np & 1), (np >> 1) & 1) &&
                 (kF8 || probe(kBarFullV + np % kRing, (np / kRing) & 1)))
          act = 2;
        if (act == 0) {
          if ((++spins & 255u) == 0) {
            const uint64_t now = global_timer_ns();
            if (t_idle == 0) {
              t_idle = now;
            } else if (*abort_word || now - t_idle > kWaitTimeoutNs) {
              if (!*abort_word) flag_error(p.err_flag, kFlagTimeout);
              *abort_word = 1;
              act = -1;
            }
          }
        } else {
          t_idle = 0;
          spins = 0;
        }
      }
      act = __shfl_sync(0xffffffffu, act, 0);
      if (act < 0) {
        ok = false;
      } else if (act == 1) {
        tc_fence_after();
        issue_s(ns++);
      } else if (act == 2) {
        tc_fence_after();
        issue_pv(np++);
      }
    }
    // Wait (bounded) until every MMA this warp issued has completed.
    if (elect_one()) {
      tc_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, p.err_flag);
    }
    __syncwarp();
  } else {
    // ---------------- softmax warps: thread (row r, column half hl, column
    // group cg) owns score columns 32 hl + 16 cg .. + 15 of row r and O
    // columns 64 hl + 32 cg .. + 31 (the 16x32bx2 TMEM access shape: lanes
    // 0-15 and 16-31 read the same 16 TMEM lanes at two column offsets).
    const int quarter = warp & 3, cg = warp >> 2;
    const int hl = lane >> 4;
    const int r = 16 * quarter + (lane & 15);  // CTA row (query head of the group)
    const bool mine = r < G;                   // a real row
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    float* red = reinterpret_cast<float*>(smem + L::kOffRed);  // [2 column groups][64 rows]
    float* qinv = red + 2 * kM;                                 // 8-bit cache: 1 / alpha_r

    // Q_j (rows >= G zero) into the swizzled K-major A tile.
    {
      const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                         row0 * kHeadDim);
#pragma unroll
      for (int i = 0; i < (kM * 16) / kSoftmaxThreads; ++i) {
        const int e = threadIdx.x + i * kSoftmaxThreads;
        const int row = e >> 4, c16 = e & 15;  // 16 threads per row, 8 elements each
        const uint4 v = row < G ? qsrc[row * 16 + c16] : make_uint4(0, 0, 0, 0);
        if constexpr (!kF8) {
          *reinterpret_cast<uint4*>(smem + L::kOffQ + (c16 >> 3) * kHalf + row * 128 +
                                    (((c16 & 7) ^ (row & 7)) << 4)) = v;
        } else {
          // 8-bit cache: row r of Q times alpha_r = 2^k (the largest power of
          // two with max |q_r| alpha_r <= 448) as the sum of e4m3 terms
          // t1 = e4m3(x), t2 = e4m3(x - t1) (, t3 = e4m3(x - t1 - t2)): each
          // residual is a multiple of the query's own last bit no larger than
          // half of the previous term's, so two terms hold a bf16 query (8
          // significant bits) and three an fp16 one (11) exactly, except for
          // parts below 2^-10 (e4m3's subnormal step) of the scaled row; the
          // score row is scaled back by 1 / alpha_r.
          float x[8];
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = unpack2<kBF16>(wv[k]);
            x[2 * k] = f.x;
            x[2 * k + 1] = f.y;
          }
          float m = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(x[k]));
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          const uint32_t mb = __float_as_uint(m);
          const int ex = static_cast<int>((mb >> 23) & 0xffu) - 127;
          const int kexp = min(max(((mb & 0x7fffffu) <= 0x600000u ? 8 : 7) - ex, -126), 126);
          const float alpha = __uint_as_float(static_cast<uint32_t>(kexp + 127) << 23);
          if (c16 == 0) qinv[row] = __uint_as_float(static_cast<uint32_t>(127 - kexp) << 23);
          uint32_t code[kQTerms][2] = {};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float a0 = x[2 * k] * alpha, a1 = x[2 * k + 1] * alpha;
#pragma unroll
            for (int t = 0; t < kQTerms; ++t) {
              float r0, r1;
              code[t][k >> 1] |= e4m3_round2(a0, a1, r0, r1) << (16 * (k & 1));
              a0 -= r0;
              a1 -= r1;
            }
          }
          // Elements 8 c16 .. + 7: bytes 8 (c16 % 2) of 16-byte chunk c16 / 2.
#pragma unroll
          for (int t = 0; t < kQTerms; ++t)
            *reinterpret_cast<uint2*>(smem + L::kOffQ + t * kQTermBytes + row * 128 +
                                      (((c16 >> 1) ^ (row & 7)) << 4) + (c16 & 1) * 8) =
                make_uint2(code[t][0], code[t][1]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kBarQ));
      if constexpr (kF8) named_bar_sync(1, kSoftmaxThreads);  // qinv of every row
    }
    // An 8-bit cache's K scale multiplies every score of KV head j, and the
    // score row r carries Q's alpha_r.
    const float scale = kF8 ? p.scale_log2 * p.k_scale[j] * qinv[r] : p.scale_log2;

    bool ok = true;
    // m_used: the row's running max (the same in all four threads of the
    // row); l: this thread's partial row sum over its columns.
    float m_used = kNegInf, l = 0.f;
    const float lowest = scale >= 0.f ? kNegInf : -kNegInf;
    const int c_own = 32 * hl + 16 * cg, c_oth = 32 * hl + 16 * (cg ^ 1);
    for (int it = 0; ok && it < n; ++it) {
      const int s = it % kStages;
      const int t0 = t_begin + it * kTile;
      const int nval = min(kTile, t_end - t0);
      const int nskip = max(0, w0 - t0);
      const bool ragged = nval < kTile || nskip > 0;
      if (!mbar_wait_or_abort(bar(kBarSFull + (it & 1)), (it >> 1) & 1, p.err_flag, abort_word)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sc[16], so[16];
      const uint32_t sb = tmem + lane_base + kTmemS + 64 * (it & 1);
      tmem_ld16x2_x16<32>(sb + 16 * cg, sc);
      tmem_ld16x2_x16<32>(sb + 16 * (cg ^ 1), so);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(kBarSFree + (it & 1)));
      // Columns outside [nskip, nval) are masked (tokens past the end or
      // before a sliding window); each tile holds at least one valid token.
      if (ragged) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          if (c_own + kk >= nval || c_own + kk < nskip) sc[kk] = lowest;
          if (c_oth + kk >= nval || c_oth + kk < nskip) so[kk] = lowest;
        }
      }
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        so[kk] = scale >= 0.f ? fmaxf(so[kk], sc[kk]) : fminf(so[kk], sc[kk]);
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int kk = 0; kk < w; ++kk)
          so[kk] = scale >= 0.f ? fmaxf(so[kk], so[kk + w]) : fminf(so[kk], so[kk + w]);
      float mr = so[0];
      const float mo = __shfl_xor_sync(0xffffffffu, mr, 16);  // the other 32 columns
      mr = scale >= 0.f ? fmaxf(mr, mo) : fminf(mr, mo);
      const float mt = mr * scale;
      // Rows past the group (zero queries) take part too, so that their P
      // stays finite; they are never written out.
      const bool need = mt > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_used;
        const float factor = need ? ex2(m_used - m_new) : 1.f;  // 0 when m_used = -inf
        if (it > 0) {
          // O += P(it - 1) V(it - 1) must have completed before O is rescaled.
          if (!mbar_wait_or_abort(bar(kBarPvDone + ((it - 1) & 1)), ((it - 1) >> 1) & 1,
                                  p.err_flag, abort_word)) {
            ok = false;
            break;
          }
          tc_fence_after();
          float o[32];
          tmem_ld16x2_x32<64>(tmem + lane_base + kTmemO + 32 * cg, o);
          tc_wait_ld();
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) o[kk] *= factor;
          tmem_st16x2_x32<64>(tmem + lane_base + kTmemO + 32 * cg, o);
          tc_wait_st();
        }
        l *= factor;
        m_used = m_new;
      }
      // p = 2^(s scale - m) for this thread's 16 columns, packed two per word.
      uint32_t pk[8];
      {
        const float neg_m = -m_used;
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          float p0 = ex2(fmaf(sc[2 * kk], scale, neg_m));
          float p1 = ex2(fmaf(sc[2 * kk + 1], scale, neg_m));
          if (ragged) {
            const int cc = c_own + 2 * kk;
            p0 = (cc < nval && cc >= nskip) ? p0 : 0.f;
            p1 = (cc + 1 < nval && cc + 1 >= nskip) ? p1 : 0.f;
          }
          ls[kk & 1] += p0 + p1;
          // bf16 P without the pack conversion (see pack2_bf16_pos); fp16
          // keeps cvt.rn, whose subnormal results an integer form would lose.
          if constexpr (kMmaBF16)
            pk[kk] = pack2_bf16_pos(p0, p1);
          else
            pk[kk] = pack2<false>(p0, p1);
        }
        l += ls[0] + ls[1];
      }
      // P(it)'s buffer (and, for an 8-bit cache, V(it)'s f16 slab) was last
      // read by O += P(it - 2) V(it - 2).
      {
        const int last = it - L::kPBuffers;
        if (last >= 0 && !mbar_wait_or_abort(bar(kBarPvDone + (last & 1)), (last >> 1) & 1,
                                             p.err_flag, abort_word)) {
          ok = false;
          break;
        }
      }
      if constexpr (kF8) {
        // V(it) into f16 slab it % 2 (its last reader, O += P(it - 2) V(it - 2),
        // has completed: the wait above), then its 8-bit stage is free again.
        const int s8 = it % kRing;
        if (!mbar_wait_or_abort(bar(kBarFullV + s8), (it / kRing) & 1, p.err_flag, abort_word)) {
          ok = false;
          break;
        }
        convert_v8(smem + L::kOffV + s8 * kF8Tile, smem + L::kOffV16 + (it & 1) * kKvTile,
                   threadIdx.x, nskip, nval);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarEmptyV + s8));
      }
      {
        // Row r, tokens c_own .. c_own + 15: 16-byte chunks c_own / 8 and + 1.
        uint8_t* prow = smem + L::kOffP + (it & 1) * kPBytes + r * 128;
        const int ch0 = c_own >> 3;
        *reinterpret_cast<uint4*>(prow + ((ch0 ^ (r & 7)) << 4)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(prow + (((ch0 + 1) ^ (r & 7)) << 4)) =
            make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      if (!kF8 && ragged) {
        // V rows outside [nskip, nval) may hold anything (even NaN): zero
        // them once the tile has landed, so that P = 0 there contributes
        // exactly nothing.  O += P(it) V(it) reads them after P(it) is published.
        if (!mbar_wait_or_abort(bar(kBarFullV + s), (it / kStages) & 1, p.err_flag, abort_word)) {
          ok = false;
          break;
        }
        uint8_t* vt = smem + L::kOffV + s * kKvTile;
        const int lo = nskip, hi = kTile - nval;
        for (int e = threadIdx.x; e < (lo + hi) * 16; e += kSoftmaxThreads) {
          const int k = e >> 4, c16 = e & 15;
          const int row = k < lo ? k : nval + (k - lo);
          *reinterpret_cast<uint4*>(vt + (c16 >> 3) * kHalf + row * 128 +
                                    (((c16 & 7) ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + (it & 1)));
    }

    // ---------------- epilogue: O / l (one split) or the fp32 partial
    if (ok) ok = mbar_wait_or_abort(bar(kBarPvDone + ((n - 1) & 1)), ((n - 1) >> 1) & 1, p.err_flag,
                                    abort_word);
    if (ok) {
      l += __shfl_xor_sync(0xffffffffu, l, 16);  // both column halves of this group
      if (lane < 16) red[cg * kM + r] = l;
      mbar_arrive(bar(kBarSum));
      ok = mbar_wait_or_abort(bar(kBarSum), 0, p.err_flag, abort_word);
    }
    if (ok) {
      tc_fence_after();
      const float lsum = red[r] + red[kM + r];
      // An 8-bit cache's V scale multiplies the whole output row.
      const float inv = lsum > 0.f ? (kF8 ? p.v_scale[j] : 1.f) / lsum : 0.f;
      float o[32];
      tmem_ld16x2_x32<64>(tmem + lane_base + kTmemO + 32 * cg, o);
      tc_wait_ld();
      if (mine) {
        const size_t row = row0 + r;
        const int col = 64 * hl + 32 * cg;
        if (p.n_split == 1) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * kHeadDim + col);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[k] = make_uint4(pack2<kBF16>(o[8 * k] * inv, o[8 * k + 1] * inv),
                                pack2<kBF16>(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                                pack2<kBF16>(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                                pack2<kBF16>(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
        } else {
          float4* dst =
              reinterpret_cast<float4*>(p.part_o + (row * p.n_split + split) * kHeadDim + col);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv,
                                 o[4 * k + 3] * inv);
          if (cg == 0 && hl == 0)
            p.part_lse[row * p.n_split + split] = lsum > 0.f ? m_used + lg2(lsum) : kNegInf;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kBF16, bool kF8>
cudaError_t launch_t(const GqaParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t stream) {
  auto kern = gqa_wide_kernel<kBF16, kF8>;
  constexpr int smem = WLayout<kBF16, kF8>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_split, p.h_kv, p.batch);
  kern<<<grid, kThreads, smem, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gqa_wide_partial(const GqaParams& p, const CUtensorMap& tm_k,
                                    const CUtensorMap& tm_v, bool bf16, cudaStream_t stream) {
  if (p.group > kM) return cudaErrorNotSupported;
  return bf16 ? launch_t<true, false>(p, tm_k, tm_v, stream)
              : launch_t<false, false>(p, tm_k, tm_v, stream);
}

cudaError_t launch_gqa_wide_partial_fp8(const GqaParams& p, const CUtensorMap& tm_k,
                                        const CUtensorMap& tm_v, bool bf16, cudaStream_t stream) {
  if (p.group > kM) return cudaErrorNotSupported;
  return bf16 ? launch_t<true, true>(p, tm_k, tm_v, stream)
              : launch_t<false, true>(p, tm_k, tm_v, stream);
}

}  // namespace decattn
