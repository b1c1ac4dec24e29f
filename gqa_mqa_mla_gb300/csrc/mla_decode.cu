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
// Work split: a cluster of two CTAs handles one (split, sequence).  The fp32
// O accumulator for 128 heads x 512 columns would fill all of one SM's
// tensor memory, so CTA r accumulates only O[:, 256 r : 256 r + 256].  Both
// CTAs compute the full score tile S = Q C^T (the same MMA sequence on the
// same bytes, hence the same bits) and the same online softmax, so they need
// to exchange nothing; the cluster only co-schedules the pair so that the
// second load of every cache tile is an L2 hit.  The redundant score GEMM
// costs 1.44x the minimum tensor work, which at 576-d keys still balances
// the HBM stream on GB300.
//
// Tile width: every tcgen05.mma costs at least ~60 SM cycles whatever its
// N, and only N >= 128 reaches the full tensor rate (measured on GB300:
// M = 128, K = 16 bf16 runs at ~1.1k / 2.2k / 3.9k MAC per cycle for N = 32 /
// 64 / 128).  The score GEMM's N is the token count of a tile, so tiles are
// 64 tokens, the widest that fits tensor memory next to O and Q.
//
// Operand placement (per CTA):
//   Q[:, 0:256)    shared memory (TMA), 128-byte swizzled K-major      A of S
//   Q[:, 256:576)  TMEM, 160 columns (two 16-bit values per column)  A of S
//   cache tiles    shared memory ring, 2 stages x 64 tokens x 576     B of S, PV
//   P(j)           TMEM, 32 columns                                  A of PV
// TMEM columns: O [0, 256) fp32 | Q [256, 416) | S [416, 480) | P [480, 512).
//
// Per CTA (320 threads):
//   warps 0-7  load Q, softmax, epilogue: warp w serves heads
//              h = 32 (w % 4) + lane (TMEM lane h) over score columns
//              [32 (w / 4), 32 (w / 4) + 32) and O columns of the same half;
//              the two threads of a row swap their tile maxima through
//              shared memory and keep separate partial row sums;
//   warp 8     TMA producer for the cache ring, walking the block table;
//   warp 9     TMEM allocator and the single MMA-issuing thread: S(j), then
//              O += P(j) C_lat(j) once P(j) is written, then S(j + 1).
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

constexpr int kT = 64;                          // tokens per tile
constexpr int kBoxRows = 32;                    // rows per TMA box (tensor-map box height cap)
constexpr int kStages = 2;                      // cache ring depth
constexpr int kChunk = 64;                      // columns per 128-byte swizzle row
constexpr int kChunks = kMlaWidth / kChunk;     // 9 column chunks per cache row
constexpr int kQSmemChunks = 4;                 // Q columns [0, 256) in shared memory
constexpr int kQChunkBytes = kMlaHeads * 128;   // [128 heads][64 cols] = 16 KB
constexpr int kCChunkBytes = kT * 128;          // [64 tokens][64 cols] = 8 KB
constexpr int kStageBytes = kChunks * kCChunkBytes;  // 72 KB
constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + kQSmemChunks * kQChunkBytes;  // 64 KB
constexpr int kOffBars = kOffRing + kStages * kStageBytes;     // +144 KB
constexpr int kBarBytes = 256;
constexpr int kOffRed = kOffBars + kBarBytes;                  // row maxima / sums exchange
constexpr int kRedBytes = 3 * 2 * kMlaHeads * 4;               // 2 max slots + 1 sum slot
constexpr int kSmemBytes = 1024 + kOffRed + kRedBytes;
constexpr int kSoftmaxThreads = 256;
constexpr int kThreads = kSoftmaxThreads + 64;
constexpr int kTmemCols = 512;
constexpr int kTmemO = 0;
constexpr int kTmemQ = 256;                     // Q columns [256, 576): 160 TMEM columns
constexpr int kTmemS = 416;                     // S tile: 64 columns fp32
constexpr int kTmemP = 480;                     // P tile: 64 bf16 = 32 columns
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when p could exceed 2^8

// mbarrier slots (8 bytes each) inside the barrier area
enum : int {
  kBarQ = 0,                               // Q[:, 256:576) in TMEM (128 arrivals)
  kBarKvFull = 1,                          // kStages: cache tile landed (2 arrivals)
  kBarKvEmptyS = kBarKvFull + kStages,     // kStages: score-only chunks consumed by S
  kBarKvEmptyV = kBarKvEmptyS + kStages,   // kStages: value chunks consumed by PV
  kBarSFull = kBarKvEmptyV + kStages,      // S(j) computed
  kBarSFree = kBarSFull + 1,               // S(j) read by the softmax (128 arrivals)
  kBarPFull = kBarSFree + 1,               // P(j) written (128 arrivals)
  kBarPvDone = kBarPFull + 1,              // O += P(j) C_lat(j) complete
  kBarQs = kBarPvDone + 1,                 // Q[:, 0:256) in shared memory (TMA)
  kBarMax = kBarQs + 1,                    // row tile maxima exchanged (256 arrivals)
  kBarSum = kBarMax + 1,                   // row sums exchanged (256 arrivals)
  kBarDrain = kBarSum + 1,
  kNumBars = kBarDrain + 1
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier area");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kTmemP + kT / 2 <= kTmemCols, "tensor memory columns");

template <bool kBF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_partial_kernel(const __grid_constant__ CUtensorMap tm_qa,
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
  const int split = blockIdx.x >> 1;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col0 = static_cast<int>(rank) * 256;  // this CTA's O columns

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
    mbar_init(bar(kBarQ), kSoftmaxThreads);
    mbar_init(bar(kBarQs), 1);
    mbar_init(bar(kBarMax), kSoftmaxThreads);
    mbar_init(bar(kBarSum), kSoftmaxThreads);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKvFull + s), 2);
      mbar_init(bar(kBarKvEmptyS + s), 1);
      mbar_init(bar(kBarKvEmptyV + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), kSoftmaxThreads);
    mbar_init(bar(kBarPFull), kSoftmaxThreads);
    mbar_init(bar(kBarPvDone), 1);
    mbar_init(bar(kBarDrain), 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  bad = __syncthreads_or(bad);
  cluster_sync();

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

  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_c);
      tma_prefetch_desc(&tm_qa);
      mbar_arrive_expect_tx(bar(kBarQs), kQSmemChunks * kQChunkBytes);
      for (int c = 0; c < kQSmemChunks; ++c)
        tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &tm_qa, c * kChunk,
                    static_cast<int>(head0), bar(kBarQs));
      const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
      const int bs = p.block_size;
      const int rows_per_box = bs < kBoxRows ? bs : kBoxRows;
      // A stage holds all 9 column chunks of a tile.  This CTA's 4 value
      // chunks (latent columns [256 r, 256 r + 256)) stay until PV(j); the
      // other 5 are only read by S(j) and are refilled as soon as S(j) is
      // done, so loads run ahead of the PV that would otherwise gate them.
      auto load_part = [&](int it, bool value_part) -> bool {
        const int s = it % kStages;
        const uint32_t empty = bar((value_part ? kBarKvEmptyV : kBarKvEmptyS) + s);
        if (!mbar_wait_or_abort(empty, ((it / kStages) & 1) ^ 1, p.err_flag, abort_word))
          return false;
        const int t0 = t_begin + it * kT;
        const int nval = min(kT, t_end - t0);
        const int nbox = (nval + rows_per_box - 1) / rows_per_box;
        const uint32_t st = sbase + kOffRing + s * kStageBytes;
        const int nparts = value_part ? 4 : kChunks - 4;
        mbar_arrive_expect_tx(bar(kBarKvFull + s),
                              static_cast<uint32_t>(nbox * nparts * rows_per_box * 128));
        for (int k = 0; k < nbox; ++k) {
          const int t = t0 + k * rows_per_box;
          const int row = bt[t >> p.log2_block_size] * bs + (t & (bs - 1));
          const uint32_t off = static_cast<uint32_t>(k * rows_per_box * 128);
          // Default L2 policy: the peer CTA loads the same tile moments later.
          for (int c = 0; c < kChunks; ++c) {
            const bool is_value = (c >> 2) == static_cast<int>(rank) && c < 8;
            if (is_value != value_part) continue;
            tma_load_2d(st + c * kCChunkBytes + off, &tm_c, c * kChunk, row, bar(kBarKvFull + s));
          }
        }
        return true;
      };
      // The tensor pipe completes PV(j - 2) before S(j - 1), so the value
      // part of tile j is requested before the score part of tile j + 1.
      int issued = 0;
      bool ok = load_part(0, false);
      for (int it = 0; ok && it < n_tiles; ++it) {
        ok = load_part(it, true);
        if (ok) issued = it + 1;
        if (ok && it + 1 < n_tiles) ok = load_part(it + 1, false);
      }
      for (int it = max(0, issued - kStages); it < issued; ++it)
        if (!mbar_wait_or_abort(bar(kBarKvFull + it % kStages), (it / kStages) & 1, p.err_flag,
                                abort_word))
          break;
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBF16, 128, kT, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kBF16, 128, 256, false, true);
      // Shared-memory descriptors are built once; within a swizzle atom and
      // across chunks / stages only the 14-bit start address (16-byte units,
      // low bits of the descriptor) moves, so each MMA is one add + issue.
      const uint64_t dq = smem_desc_sw128(sbase + kOffQ, 16, 1024);
      const uint64_t dr = smem_desc_sw128(sbase + kOffRing, 16, 1024);
      const uint64_t dv = smem_desc_sw128(
          sbase + kOffRing + static_cast<uint32_t>(rank) * 4 * kCChunkBytes, kCChunkBytes, 1024);
      constexpr uint64_t kStageUnits = kStageBytes >> 4;
      constexpr uint64_t kQChunkUnits = kQChunkBytes >> 4;
      constexpr uint64_t kCChunkUnits = kCChunkBytes >> 4;
      // S(i) = Q C(i)^T (M = 128 heads, N = 64 tokens, K = 576).  The S tile
      // is reused: S(i) waits until the softmax has read S(i - 1).
      auto issue_s = [&](int i) -> bool {
        const int s = i % kStages;
        if (!mbar_wait_or_abort(bar(kBarKvFull + s), (i / kStages) & 1, p.err_flag, abort_word))
          return false;
        if (i > 0 &&
            !mbar_wait_or_abort(bar(kBarSFree), (i - 1) & 1, p.err_flag, abort_word))
          return false;
        tc_fence_after();
        const uint64_t db = dr + static_cast<uint64_t>(s) * kStageUnits;
        const uint32_t d = tmem + kTmemS;
#pragma unroll
        for (int c = 0; c < kQSmemChunks; ++c) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc_mma_f16(d, dq + c * kQChunkUnits + 2 * ks, db + c * kCChunkUnits + 2 * ks, idesc_s,
                       (c > 0 || ks > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int c = kQSmemChunks; c < kChunks; ++c) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc_mma_f16_ts(d, tmem + kTmemQ + (c - kQSmemChunks) * 32 + ks * 8,
                          db + c * kCChunkUnits + 2 * ks, idesc_s, 1u);
        }
        tc_commit(bar(kBarSFull));
        tc_commit(bar(kBarKvEmptyS + s));
        return true;
      };
      // O += P(j) C_lat(j) over this CTA's 256 value columns (MN-major B).
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait_or_abort(bar(kBarPFull), j & 1, p.err_flag, abort_word)) return false;
        tc_fence_after();
        const uint64_t db = dv + static_cast<uint64_t>(j % kStages) * kStageUnits;
#pragma unroll
        for (int ks = 0; ks < kT / 16; ++ks)
          tc_mma_f16_ts(tmem + kTmemO, tmem + kTmemP + ks * 8, db + ks * (2048 >> 4), idesc_pv,
                        (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(bar(kBarPvDone));
        tc_commit(bar(kBarKvEmptyV + j % kStages));
        return true;
      };
      // PV(j) goes before S(j + 1): the value chunks of tile j are released
      // (and the load of tile j + 2 starts) as early as possible.
      bool ok = mbar_wait_or_abort(bar(kBarQ), 0, p.err_flag, abort_word) &&
                mbar_wait_or_abort(bar(kBarQs), 0, p.err_flag, abort_word);
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        ok = issue_pv(j);
        if (ok && j + 1 < n_tiles) ok = issue_s(j + 1);
      }
      // Wait (bounded) until every MMA this thread issued has completed.
      tc_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, p.err_flag);
    }
  } else {
    // ---------------- softmax warps: thread (h, ch) owns head h, column half ch
    const int h = (warp & 3) * 32 + lane;
    const int ch = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* red_max = reinterpret_cast<float*>(smem + kOffRed);       // [2 slots][2 halves][128]
    float* red_sum = red_max + 2 * 2 * kMlaHeads;                    // [2 halves][128]
    const float scale = p.scale_log2;
    float m_used = kNegInf, l = 0.f;  // l: this half's partial row sum

    // Q row h, columns [256, 512) and the RoPE part, into TMEM (columns
    // [0, 256) arrive in shared memory by TMA); the two halves split the
    // five 64-column chunks 3 + 2, all loads in flight before any store.
    {
      const uint4* qa = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q_abs) +
                                                       (head0 + h) * kMlaDc) + 32;
      const uint4* qr = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q_rope) +
                                                       (head0 + h) * kMlaDr);
      const int c0 = ch == 0 ? 0 : 3, nc = ch == 0 ? 3 : 2;
      uint4 w[24];
#pragma unroll
      for (int k = 0; k < 24; ++k) {
        const int c = c0 + k / 8;
        if (k < nc * 8) w[k] = c < 4 ? qa[c * 8 + k % 8] : qr[k % 8];
      }
#pragma unroll
      for (int cc = 0; cc < 3; ++cc) {
        if (cc < nc) {
          float v[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            v[4 * k] = __uint_as_float(w[cc * 8 + k].x);
            v[4 * k + 1] = __uint_as_float(w[cc * 8 + k].y);
            v[4 * k + 2] = __uint_as_float(w[cc * 8 + k].z);
            v[4 * k + 3] = __uint_as_float(w[cc * 8 + k].w);
          }
          tmem_st32(tmem + lane_base + kTmemQ + (c0 + cc) * 32, v);
        }
      }
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarQ));
    }

    bool ok = true;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int nval = min(kT, t_end - (t_begin + j * kT));
      const int nv = nval - ch * 32;  // valid columns in this half (may be <= 0 or > 32)
      if (!mbar_wait_or_abort(bar(kBarSFull), j & 1, p.err_flag, abort_word)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[32];
      tmem_ld32(tmem + lane_base + kTmemS + ch * 32, s);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(kBarSFree));  // the MMA thread may now compute S(j + 1)
      // Tile max of the scaled scores over this half (masked columns ignored).
      if (nv < 32) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k >= nv) s[k] = scale >= 0.f ? kNegInf : -kNegInf;
      }
      float mx[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        mx[k] = scale >= 0.f ? fmaxf(s[k], s[k + 16]) : fminf(s[k], s[k + 16]);
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k)
          mx[k] = scale >= 0.f ? fmaxf(mx[k], mx[k + w]) : fminf(mx[k], mx[k + w]);
      float mt = mx[0] * scale;
      if (mt != mt) mt = kNegInf;  // an all-masked half (-inf * 0 cannot occur: scale != 0)
      // Swap halves' maxima: slot j & 1 of the exchange area.
      red_max[((j & 1) * 2 + ch) * kMlaHeads + h] = mt;
      mbar_arrive(bar(kBarMax));
      if (!mbar_wait_or_abort(bar(kBarMax), j & 1, p.err_flag, abort_word)) {
        ok = false;
        break;
      }
      mt = fmaxf(mt, red_max[((j & 1) * 2 + (ch ^ 1)) * kMlaHeads + h]);
      // P(j - 1) must have been consumed (and O updated) before P(j) is
      // written or O is rescaled.
      if (j > 0 && !mbar_wait_or_abort(bar(kBarPvDone), (j - 1) & 1, p.err_flag, abort_word)) {
        ok = false;
        break;
      }
      const bool need = mt > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_used;
        const float factor = need ? ex2(m_used - m_new) : 1.f;  // 0 when m_used = -inf
        if (j > 0) {
          tc_fence_after();
#pragma unroll 1
          for (int c = ch * 128; c < ch * 128 + 128; c += 32) {
            float o[32];
            tmem_ld32(tmem + lane_base + kTmemO + c, o);
            tc_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= factor;
            tmem_st32(tmem + lane_base + kTmemO + c, o);
          }
        }
        l *= factor;
        m_used = m_new;
      }
      // p = 2^(s scale - m_used) (one FFMA + EX2), partial row sum, P(j) half
      // into TMEM (two 16-bit values per column).
      const float neg_m = -m_used;
      uint32_t pk[16];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        float p0 = ex2(fmaf(s[2 * k], scale, neg_m));
        float p1 = ex2(fmaf(s[2 * k + 1], scale, neg_m));
        if (nv < 32) {
          p0 = 2 * k < nv ? p0 : 0.f;
          p1 = 2 * k + 1 < nv ? p1 : 0.f;
        }
        ls[k & 3] += p0 + p1;
        pk[k] = pack2<kBF16>(p0, p1);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tmem_st16(tmem + lane_base + kTmemP + ch * 16, pk);
      if (nval < kT) {
        // Value rows past the sequence end may hold anything (even NaN): zero
        // them so that P = 0 there contributes exactly nothing.
        uint8_t* st = smem + kOffRing + (j % kStages) * kStageBytes + rank * 4 * kCChunkBytes;
        const int t = ch * 128 + h;
        for (int e = t; e < (kT - nval) * 4 * 8; e += kSoftmaxThreads) {
          const int row = nval + e / 32, c = (e / 8) & 3, q = e & 7;
          *reinterpret_cast<uint4*>(st + c * kCChunkBytes + row * 128 + q * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull));
    }

    // ---------------- epilogue: O row h, this thread's 128 columns, / l
    if (ok) {
      red_sum[ch * kMlaHeads + h] = l;
      mbar_arrive(bar(kBarSum));
      ok = mbar_wait_or_abort(bar(kBarSum), 0, p.err_flag, abort_word) &&
           mbar_wait_or_abort(bar(kBarPvDone), (n_tiles - 1) & 1, p.err_flag, abort_word);
    }
    if (ok) {
      const float lt = l + red_sum[(ch ^ 1) * kMlaHeads + h];
      tc_fence_after();
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll 1
      for (int c = ch * 128; c < ch * 128 + 128; c += 32) {
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
      if (p.n_split > 1 && rank == 0 && ch == 0)
        p.part_lse[(head0 + h) * p.n_split + split] = lt > 0.f ? m_used + lg2(lt) : kNegInf;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();
}

template <bool kBF16>
cudaError_t launch_t(const MlaParams& p, const CUtensorMap& tqa, const CUtensorMap& tc,
                     cudaStream_t stream) {
  auto kern = mla_partial_kernel<kBF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * p.n_split, p.batch);
  kern<<<grid, kThreads, kSmemBytes, stream>>>(tqa, tc, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mla_partial(const MlaParams& p, const CUtensorMap& tm_qa,
                               const CUtensorMap& tm_c, bool bf16, cudaStream_t stream) {
  if (p.block_size > kT && (p.block_size % kT) != 0) return cudaErrorNotSupported;
  return bf16 ? launch_t<true>(p, tm_qa, tm_c, stream) : launch_t<false>(p, tm_qa, tm_c, stream);
}

}  // namespace decattn
