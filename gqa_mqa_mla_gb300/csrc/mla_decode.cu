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
// Work split: a cluster of two CTAs streams one share of the batch's tiles
// (see the work schedule below).  The fp32 O accumulator for 128 heads x 512
// columns would fill all of one SM's tensor memory, so CTA r accumulates only
// O[:, 256 r : 256 r + 256].  Both CTAs compute the full score tile
// S = Q C^T (the same MMA sequence on the same bytes, hence the same bits)
// and the same online softmax, so they need to exchange nothing; the cluster
// only co-schedules the pair so that the second load of every cache tile is
// an L2 hit.  The redundant score GEMM costs 1.44x the minimum tensor work.
//
// Tile width: a chain of tcgen05.mma (M = 128, K = 16, bf16) into one
// accumulator costs ~58 SM cycles per instruction for any N <= 64 and only
// N >= 128 reaches the full tensor rate (measured on GB300: ~1.1k / 2.2k /
// 3.9k MAC per cycle for N = 32 / 64 / 128).  The score GEMM's N is the
// token count of a tile, so tiles are 64 tokens, the widest that fits tensor
// memory next to O and Q.
//
// Operand placement (per CTA):
//   Q[:, 0:256)    shared memory (TMA), 128-byte swizzled K-major      A of S
//   Q[:, 256:576)  TMEM, 160 columns (two 16-bit values per column)  A of S
//   cache tiles    shared memory ring, 2 stages x 64 tokens x 576     B of S, PV
//   P(j)           TMEM, 32 columns                                  A of PV
//   epilogue       the cache ring, idle once a segment's MMAs are done
// TMEM columns: O [0, 256) fp32 | Q [256, 416) | S [416, 480) | P [480, 512).
//
// Per CTA (320 threads):
//   warps 0-7  load Q, softmax, epilogue: warp w serves heads
//              h = 32 (w % 4) + lane (TMEM lane h) over score columns
//              [32 (w / 4), 32 (w / 4) + 32) and O columns of the same half;
//              both threads of a row read all 64 score columns and take
//              the same row maximum, and keep separate partial row sums;
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
constexpr int kBoxRows = kT;                    // rows per TMA box: a whole block up to one tile
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
constexpr int kOffRed = kOffBars + kBarBytes;                  // row-sum exchange
constexpr int kRedBytes = 2 * kMlaHeads * 4;                   // row sums (and the scan before)
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
  kBarSum = kBarQs + 1,                    // row sums exchanged (256 arrivals)
  kBarEpiW = kBarSum + 1,                  // epilogue round staged in smem (256 arrivals)
  kBarEpiR = kBarEpiW + 1,                 // epilogue round's bulk stores have read smem
  kBarEpiDone = kBarEpiR + 1,              // segment epilogue done: the ring is free again
  kBarDrain = kBarEpiDone + 1,
  kNumBars = kBarDrain + 1
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier area");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(8 * kQChunkBytes <= kStages * kStageBytes, "epilogue staging must fit the ring");
static_assert(kTmemP + kT / 2 <= kTmemCols, "tensor memory columns");

// Work schedule.  The batch's 64-token tiles, sequence after sequence, form
// one list of T_all tiles (an invalid seq_len counts as 0 tiles); pair p of
// the P CTA pairs takes the slice [p T, p T + T), T = ceil(T_all / P), so
// every pair streams the same number of tiles however ragged the lengths
// are.  The slice is cut at sequence boundaries into segments: a segment
// holding a whole sequence writes its output rows directly; one holding
// part of a sequence writes an fp32 partial (normalised O and log2-sum-exp)
// that the combine merges.  Only a slice's first and last segments can be
// partial; they go to workspace slots 2 p and 2 p + 1.  A sequence with no
// tiles is zeroed by the pair whose slice contains its start.
enum : int { kSegZero = 0, kSegDirect = 1, kSegPartial = 2 };

struct Sched {
  int pair, n_pairs, T, lo, hi;  // this pair's tile slice [lo, hi)
};
struct Cursor {
  int b, pref;  // next sequence to examine and the index of its first tile
};
struct Seg {
  int b, t0, t1, kind;  // tokens [t0, t1) of sequence b
};

__device__ __forceinline__ int seq_tiles(const MlaParams& p, int len) {
  return (len < 0 || len > p.max_seq_len) ? 0 : (len + kT - 1) / kT;
}

// Next segment of this pair's slice (every role walks the same sequence).
__device__ bool next_seg(const MlaParams& p, const Sched& sc, Cursor& cur, Seg& sg) {
  while (cur.b < p.batch) {
    const int b = cur.b, pref = cur.pref;
    const int len = p.seq_lens[b];
    const int n = seq_tiles(p, len);
    if (n == 0) {
      const int owner = min(pref / sc.T, sc.n_pairs - 1);
      if (owner > sc.pair) return false;
      ++cur.b;
      if (owner < sc.pair) continue;
      sg.b = b;
      sg.t0 = sg.t1 = 0;
      sg.kind = kSegZero;
      return true;
    }
    if (pref >= sc.hi) return false;
    ++cur.b;
    cur.pref = pref + n;
    const int g0 = max(pref, sc.lo), g1 = min(pref + n, sc.hi);
    if (g1 <= g0) continue;
    sg.b = b;
    sg.t0 = (g0 - pref) * kT;
    sg.t1 = min(len, (g1 - pref) * kT);
    sg.kind = (g0 == pref && g1 == pref + n) ? kSegDirect : kSegPartial;
    return true;
  }
  return false;
}

template <bool kBF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_partial_kernel(const __grid_constant__ CUtensorMap tm_qa,
                       const __grid_constant__ CUtensorMap tm_c,
                       const __grid_constant__ CUtensorMap tm_c4,
                       const __grid_constant__ CUtensorMap tm_out,
                       const __grid_constant__ CUtensorMap tm_po, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBars;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile int* abort_word = reinterpret_cast<volatile int*>(smem + kOffBars + kNumBars * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBars + kNumBars * 8 + 4);

  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col0 = static_cast<int>(rank) * 256;  // this CTA's O columns

  // ---------------- schedule: block-wide scan of the per-sequence tile counts
  Sched sc;
  sc.pair = static_cast<int>(blockIdx.x >> 1);
  sc.n_pairs = static_cast<int>(gridDim.x >> 1);
  Cursor cur0;
  {
    int* s_warp = reinterpret_cast<int*>(smem + kOffRed);  // [0, 32) totals, [32, 64) scanned
    int* s_misc = s_warp + 64;                              // b_start, its first tile
    constexpr int kWarpsAll = kThreads / 32;
    const int chunk = (p.batch + kThreads - 1) / kThreads;
    const int b_a = min(p.batch, static_cast<int>(threadIdx.x) * chunk);
    const int b_b = min(p.batch, b_a + chunk);
    int sum = 0;
    bool bad_len = false;
    for (int b = b_a; b < b_b; ++b) {
      const int len = p.seq_lens[b];
      bad_len |= (len < 0 || len > p.max_seq_len);
      sum += seq_tiles(p, len);
    }
    if (bad_len && sc.pair == 0 && rank == 0) flag_error(p.err_flag, kFlagBadSeqLen);
    int x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    if (threadIdx.x == 0) s_misc[0] = p.batch;
    __syncthreads();
    if (warp == 0) {
      int v = lane < kWarpsAll ? s_warp[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
      }
      s_warp[32 + lane] = v;
    }
    __syncthreads();
    const int t_all = s_warp[32 + kWarpsAll - 1];
    sc.T = max(1, (t_all + sc.n_pairs - 1) / sc.n_pairs);
    sc.lo = sc.pair * sc.T;
    sc.hi = min(sc.lo + sc.T, t_all);
    // First sequence this pair touches: pref_b + max(n_b, 1) > lo.
    const int excl = (warp > 0 ? s_warp[32 + warp - 1] : 0) + x - sum;
    int pref = excl, cand = p.batch, cand_pref = 0;
    for (int b = b_a; b < b_b; ++b) {
      const int n = seq_tiles(p, p.seq_lens[b]);
      if (cand == p.batch && pref + max(n, 1) > sc.lo) {
        cand = b;
        cand_pref = pref;
      }
      if (p.ws_hdr && sc.pair == 0 && rank == 0) p.ws_hdr[kHdrPref + b] = pref;
      pref += n;
    }
    if (cand < p.batch) atomicMin(&s_misc[0], cand);
    if (p.ws_hdr && sc.pair == 0 && rank == 0 && threadIdx.x == 0) {
      p.ws_hdr[0] = sc.T;
      p.ws_hdr[1] = t_all;
      p.ws_hdr[kHdrPref + p.batch] = t_all;
    }
    __syncthreads();
    if (cand < p.batch && cand == s_misc[0]) s_misc[1] = cand_pref;
    __syncthreads();
    cur0.b = s_misc[0];
    cur0.pref = cur0.b < p.batch ? s_misc[1] : 0;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), kSoftmaxThreads);
    mbar_init(bar(kBarQs), 1);
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
    mbar_init(bar(kBarEpiW), kSoftmaxThreads);
    mbar_init(bar(kBarEpiR), 1);
    mbar_init(bar(kBarEpiDone), 1);
    mbar_init(bar(kBarDrain), 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_c);
      tma_prefetch_desc(&tm_c4);
      tma_prefetch_desc(&tm_qa);
      const int bs = p.block_size;
      const int rows_per_box = bs < kBoxRows ? bs : kBoxRows;
      int g = 0;          // global tile index (ring stage and phase)
      int s_issued = 0;   // tiles whose score part is requested
      int v_issued = 0;   // tiles whose value part is requested
      int q_issued = 0;   // segments whose Q part is requested
      bool ok = true;
      // A stage holds all 9 column chunks of a tile.  This CTA's 4 value
      // chunks (latent columns [256 r, 256 r + 256)) stay until PV(j); the
      // other 5 are only read by S(j) and are refilled as soon as S(j) is
      // done, so loads run ahead of the PV that would otherwise gate them.
      auto load_part = [&](const int32_t* bt, int t_lo, int t_hi, int it, bool value_part) -> bool {
        const int gi = g + it;
        const int s = gi % kStages;
        const uint32_t empty = bar((value_part ? kBarKvEmptyV : kBarKvEmptyS) + s);
        if (!mbar_wait_or_abort(empty, ((gi / kStages) & 1) ^ 1, p.err_flag, abort_word))
          return false;
        const int t0 = t_lo + it * kT;
        const int nval = min(kT, t_hi - t0);
        const int nbox = (nval + rows_per_box - 1) / rows_per_box;
        const uint32_t st = sbase + kOffRing + s * kStageBytes;
        const int nparts = value_part ? 4 : kChunks - 4;
        mbar_arrive_expect_tx(bar(kBarKvFull + s),
                              static_cast<uint32_t>(nbox * nparts * rows_per_box * 128));
        for (int k = 0; k < nbox; ++k) {
          const int t = t0 + k * rows_per_box;
          // A block id outside [0, num_blocks) lands the box outside the
          // cache tensor, where the copy reads zeros; the softmax warps flag
          // the segment and zero its result.
          const int row = bt[t >> p.log2_block_size] * bs + (t & (bs - 1));
          const uint32_t off = static_cast<uint32_t>(k * rows_per_box * 128);
          // Default L2 policy: the peer CTA loads the same tile moments later.
          if (rows_per_box == kT) {
            // One 64-row box per tile: a 3-D copy brings four chunks at once
            // (this CTA's value chunks, or the other CTA's), chunk 8 (RoPE)
            // goes with the score part.
            const int c0 = value_part ? 4 * static_cast<int>(rank) : 4 - 4 * static_cast<int>(rank);
            tma_load_3d(st + c0 * kCChunkBytes, &tm_c4, 0, row, c0, bar(kBarKvFull + s));
            if (!value_part)
              tma_load_2d(st + 8 * kCChunkBytes, &tm_c, 8 * kChunk, row, bar(kBarKvFull + s));
            continue;
          }
          for (int c = 0; c < kChunks; ++c) {
            const bool is_value = (c >> 2) == static_cast<int>(rank) && c < 8;
            if (is_value != value_part) continue;
            tma_load_2d(st + c * kCChunkBytes + off, &tm_c, c * kChunk, row, bar(kBarKvFull + s));
          }
        }
        if (value_part) v_issued = gi + 1; else s_issued = gi + 1;
        return true;
      };
      Cursor cur = cur0;
      Seg sg;
      while (ok && next_seg(p, sc, cur, sg)) {
        if (sg.kind == kSegZero) continue;
        const int n = (sg.t1 - sg.t0 + kT - 1) / kT;
        // Q[:, 0:256) of this segment's sequence, once the previous
        // segment's last S (tile g - 1, the last reader of the Q region) has
        // completed: the previous epilogue stages its output in the ring, so
        // this load overlaps it.
        if (g > 0 && !mbar_wait_or_abort(bar(kBarKvEmptyS + (g - 1) % kStages),
                                         ((g - 1) / kStages) & 1, p.err_flag, abort_word)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarQs), kQSmemChunks * kQChunkBytes);
        for (int c = 0; c < kQSmemChunks; ++c)
          tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &tm_qa, c * kChunk, sg.b * kMlaHeads,
                      bar(kBarQs));
        ++q_issued;
        // This segment's tiles, once the previous segment's epilogue has
        // released the ring.
        if (q_issued > 1 &&
            !mbar_wait_or_abort(bar(kBarEpiDone), (q_issued - 2) & 1, p.err_flag, abort_word)) {
          ok = false;
          break;
        }
        const int32_t* bt = p.block_table + static_cast<size_t>(sg.b) * p.max_blocks_per_seq;
        // The tensor pipe completes PV(j - 2) before S(j - 1), so the value
        // part of tile j is requested before the score part of tile j + 1.
        ok = load_part(bt, sg.t0, sg.t1, 0, false);
        for (int it = 0; ok && it < n; ++it) {
          ok = load_part(bt, sg.t0, sg.t1, it, true);
          if (ok && it + 1 < n) ok = load_part(bt, sg.t0, sg.t1, it + 1, false);
        }
        g += n;
      }
      // Wait for this thread's copies still in flight before the CTA may
      // exit, even when another thread has raised the abort word: a bulk
      // copy must never land in the shared memory of a finished CTA.  A tile
      // whose value part was never requested gets the missing arrival so
      // that its phase completes once the score part has landed.  Each wait
      // is bounded on its own.
      if (v_issued < s_issued) mbar_arrive(bar(kBarKvFull + (s_issued - 1) % kStages));
      for (int it = max(0, s_issued - kStages); it < s_issued; ++it)
        if (!mbar_wait(bar(kBarKvFull + it % kStages), (it / kStages) & 1, p.err_flag)) break;
      if (q_issued > 0) mbar_wait(bar(kBarQs), (q_issued - 1) & 1, p.err_flag);
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
        // Fully unrolled: a rolled chunk loop measurably slows the issue of
        // this 36-MMA chain (1.5 vs 1.2 us per tile on GB300).
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
      // O += P(j) C_lat(j) over this CTA's 256 value columns (MN-major B);
      // the first tile of a segment overwrites O.
      auto issue_pv = [&](int j, bool first) -> bool {
        if (!mbar_wait_or_abort(bar(kBarPFull), j & 1, p.err_flag, abort_word)) return false;
        tc_fence_after();
        const uint64_t db = dv + static_cast<uint64_t>(j % kStages) * kStageUnits;
#pragma unroll
        for (int ks = 0; ks < kT / 16; ++ks)
          tc_mma_f16_ts(tmem + kTmemO, tmem + kTmemP + ks * 8, db + ks * (2048 >> 4), idesc_pv,
                        (!first || ks > 0) ? 1u : 0u);
        tc_commit(bar(kBarPvDone));
        tc_commit(bar(kBarKvEmptyV + j % kStages));
        return true;
      };
      // Per segment: wait for its Q (TMEM part written by the softmax warps
      // after the previous segment's epilogue, so O is free again), then
      // S(j), PV(j), S(j + 1), ...  PV(j) goes before S(j + 1): the value
      // chunks of tile j are released (and the load of tile j + 2 starts) as
      // early as possible.
      bool ok = true;
      int g = 0, k = 0;
      Cursor cur = cur0;
      Seg sg;
      while (ok && next_seg(p, sc, cur, sg)) {
        if (sg.kind == kSegZero) continue;
        const int n = (sg.t1 - sg.t0 + kT - 1) / kT;
        ok = mbar_wait_or_abort(bar(kBarQ), k & 1, p.err_flag, abort_word) &&
             mbar_wait_or_abort(bar(kBarQs), k & 1, p.err_flag, abort_word);
        for (int j = -1; ok && j < n; ++j) {  // j = -1 issues S(0) only
          if (j >= 0) ok = issue_pv(g + j, j == 0);
          if (ok && j + 1 < n) ok = issue_s(g + j + 1);
        }
        g += n;
        ++k;
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
    float* red_sum = reinterpret_cast<float*>(smem + kOffRed);       // [2 halves][128]
    const float scale = p.scale_log2;
    bool ok = true;
    int g = 0, k = 0, epi_round = 0;
    Cursor cur = cur0;
    Seg sg;
    while (ok && next_seg(p, sc, cur, sg)) {
      const size_t head0 = static_cast<size_t>(sg.b) * kMlaHeads;
      uint16_t* out_row = static_cast<uint16_t*>(p.out) + (head0 + h) * kMlaDc + col0 + ch * 128;
      if (sg.kind == kSegZero) {
        // An empty (or invalid-length) sequence: zero output rows.
        uint4* dst = reinterpret_cast<uint4*>(out_row);
#pragma unroll
        for (int q = 0; q < 16; ++q) dst[q] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int n_tiles = (sg.t1 - sg.t0 + kT - 1) / kT;
      float m_used = kNegInf, l = 0.f;  // l: this half's partial row sum

      // Q row h, columns [256, 512) and the RoPE part, into TMEM (columns
      // [0, 256) arrive in shared memory by TMA); the two halves split the
      // five 64-column chunks 3 + 2, all loads in flight before any store.
      // No MMA is in flight here: the previous segment's epilogue waited for
      // its last PV, and this segment's first S waits for kBarQ.
      {
        const uint4* qa = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q_abs) +
                                                         (head0 + h) * kMlaDc) + 32;
        const uint4* qr = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q_rope) +
                                                         (head0 + h) * kMlaDr);
        const int c0 = ch == 0 ? 0 : 3, nc = ch == 0 ? 3 : 2;
        uint4 w[24];
#pragma unroll
        for (int kk = 0; kk < 24; ++kk) {
          const int c = c0 + kk / 8;
          if (kk < nc * 8) w[kk] = c < 4 ? qa[c * 8 + kk % 8] : qr[kk % 8];
        }
#pragma unroll
        for (int cc = 0; cc < 3; ++cc) {
          if (cc < nc) {
            float v[32];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              v[4 * kk] = __uint_as_float(w[cc * 8 + kk].x);
              v[4 * kk + 1] = __uint_as_float(w[cc * 8 + kk].y);
              v[4 * kk + 2] = __uint_as_float(w[cc * 8 + kk].z);
              v[4 * kk + 3] = __uint_as_float(w[cc * 8 + kk].w);
            }
            tmem_st32(tmem + lane_base + kTmemQ + (c0 + cc) * 32, v);
          }
        }
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarQ));
      }
      // Block ids of the segment (needed by the epilogue only, so checked
      // while the first tile is in flight): every warp checks all of them,
      // so the verdict is uniform without a CTA-wide barrier.
      bool seg_bad = false;
      {
        const int32_t* bt = p.block_table + static_cast<size_t>(sg.b) * p.max_blocks_per_seq;
        const int k1 = (sg.t1 - 1) >> p.log2_block_size;
        for (int kb = (sg.t0 >> p.log2_block_size) + lane; kb <= k1; kb += 32) {
          const int id = bt[kb];
          seg_bad |= (id < 0 || id >= p.num_blocks);
        }
        seg_bad = __any_sync(0xffffffffu, seg_bad);
        if (seg_bad && rank == 0 && threadIdx.x == 0) flag_error(p.err_flag, kFlagBadBlock);
      }

      for (int j = 0; ok && j < n_tiles; ++j) {
        const int gj = g + j;
        const int nval = min(kT, sg.t1 - (sg.t0 + j * kT));
        const int nv = nval - ch * 32;  // valid columns in this half (may be <= 0 or > 32)
        if (!mbar_wait_or_abort(bar(kBarSFull), gj & 1, p.err_flag, abort_word)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // This thread's 32 score columns, and the partner half's, from which
        // both threads of the row take the same full-row maximum (no exchange).
        float s[32], so[32];
        tmem_ld32(tmem + lane_base + kTmemS + ch * 32, s);
        tmem_ld32(tmem + lane_base + kTmemS + (ch ^ 1) * 32, so);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kBarSFree));  // the MMA thread may now compute S(j + 1)
        // Tile max of the scaled scores over the row (masked columns ignored).
        const int nvo = nval - (ch ^ 1) * 32;  // valid columns of the partner half
        const float lowest = scale >= 0.f ? kNegInf : -kNegInf;
        if (nv < 32) {
#pragma unroll
          for (int kk = 0; kk < 32; ++kk)
            if (kk >= nv) s[kk] = lowest;
        }
        if (nvo < 32) {
#pragma unroll
          for (int kk = 0; kk < 32; ++kk)
            if (kk >= nvo) so[kk] = lowest;
        }
#pragma unroll
        for (int kk = 0; kk < 32; ++kk)
          so[kk] = scale >= 0.f ? fmaxf(so[kk], s[kk]) : fminf(so[kk], s[kk]);
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
          for (int kk = 0; kk < w; ++kk)
            so[kk] = scale >= 0.f ? fmaxf(so[kk], so[kk + w]) : fminf(so[kk], so[kk + w]);
        float mt = so[0] * scale;
        if (mt != mt) mt = kNegInf;  // an all-masked row (-inf * 0 cannot occur: scale != 0)
        // P(j - 1) must have been consumed (and O updated) before P(j) is
        // written or O is rescaled.  (The previous segment's last PV was
        // waited for by its epilogue.)
        if (j > 0 &&
            !mbar_wait_or_abort(bar(kBarPvDone), (gj - 1) & 1, p.err_flag, abort_word)) {
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
              for (int kk = 0; kk < 32; ++kk) o[kk] *= factor;
              tmem_st32(tmem + lane_base + kTmemO + c, o);
            }
          }
          l *= factor;
          m_used = m_new;
        }
        // p = 2^(s scale - m) (one FFMA + EX2), partial row sum, P packed two
        // 16-bit values per TMEM column.
        uint32_t pk[16];
        float lt_tile;
        {
          const float neg_m = -m_used;
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            float p0 = ex2(fmaf(s[2 * kk], scale, neg_m));
            float p1 = ex2(fmaf(s[2 * kk + 1], scale, neg_m));
            if (nv < 32) {
              p0 = 2 * kk < nv ? p0 : 0.f;
              p1 = 2 * kk + 1 < nv ? p1 : 0.f;
            }
            ls[kk & 3] += p0 + p1;
            pk[kk] = pack2<kBF16>(p0, p1);
          }
          lt_tile = (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        l += lt_tile;
        tmem_st16(tmem + lane_base + kTmemP + ch * 16, pk);
        if (nval < kT) {
          // Value rows past the sequence end may hold anything (even NaN): zero
          // them so that P = 0 there contributes exactly nothing.
          uint8_t* st = smem + kOffRing + (gj % kStages) * kStageBytes + rank * 4 * kCChunkBytes;
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
      if (!ok) break;

      // Pull the next segment's Q row into L2 now; its TMEM load follows
      // this epilogue on the critical path of the segment switch.
      {
        Cursor c2 = cur;
        Seg nx;
        bool have = false;
        while (!have && next_seg(p, sc, c2, nx)) have = nx.kind != kSegZero;
        if (have) {
          const char* row = reinterpret_cast<const char*>(
              static_cast<const uint16_t*>(p.q_abs) + (static_cast<size_t>(nx.b) * kMlaHeads + h) * kMlaDc);
          if (ch == 0) {
            prefetch_l2(row + 512);
            prefetch_l2(row + 640);
            prefetch_l2(row + 768);
          } else {
            prefetch_l2(row + 896);
            prefetch_l2(static_cast<const uint16_t*>(p.q_rope) +
                        (static_cast<size_t>(nx.b) * kMlaHeads + h) * kMlaDr);
          }
        }
      }

      // ---------------- epilogue: O row h, this thread's 128 columns, / l
      red_sum[ch * kMlaHeads + h] = l;
      mbar_arrive(bar(kBarSum));
      ok = mbar_wait_or_abort(bar(kBarSum), k & 1, p.err_flag, abort_word) &&
           mbar_wait_or_abort(bar(kBarPvDone), (g + n_tiles - 1) & 1, p.err_flag, abort_word);
      if (!ok) break;
      const float lt = l + red_sum[(ch ^ 1) * kMlaHeads + h];
      tc_fence_after();
      const float inv = (lt > 0.f && !seg_bad) ? 1.f / lt : 0.f;
      const bool partial = sg.kind == kSegPartial;
      const int slot = 2 * sc.pair + (k == 0 ? 0 : 1);
      if (partial && rank == 0 && ch == 0)
        p.part_lse[static_cast<size_t>(slot) * kMlaHeads + h] =
            seg_bad ? DECATTN_POISON_LSE : (lt > 0.f ? m_used + lg2(lt) : kNegInf);
      // O / l leaves through shared memory and bulk tensor stores, staged in
      // the cache ring (idle: every MMA of the segment has completed, and the
      // producer requests the next segment's tiles only after kBarEpiDone):
      // 128-row boxes of 128-byte rows, 128-byte swizzled (16-byte chunk j of
      // row y at chunk j ^ (y % 8), conflict-free for a warp writing 32 rows).
      // An fp32 partial (this CTA's 256 columns) is 8 boxes of 32 columns, a
      // 16-bit output 4 boxes of 64; either way one round of bulk stores.
      {
        const int nbt = partial ? 4 : 2;  // boxes per thread
#pragma unroll 1
        for (int cc = 0; cc < nbt; ++cc) {
          uint8_t* box = smem + kOffRing + (ch * nbt + cc) * kQChunkBytes;
          uint4 v[8];
          if (partial) {
            float o[32];
            tmem_ld32(tmem + lane_base + kTmemO + ch * 128 + cc * 32, o);
            tc_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              v[q] = make_uint4(__float_as_uint(o[4 * q] * inv), __float_as_uint(o[4 * q + 1] * inv),
                                __float_as_uint(o[4 * q + 2] * inv),
                                __float_as_uint(o[4 * q + 3] * inv));
          } else {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float o[32];
              tmem_ld32(tmem + lane_base + kTmemO + ch * 128 + cc * 64 + half * 32, o);
              tc_wait_ld();
#pragma unroll
              for (int q = 0; q < 4; ++q)
                v[half * 4 + q] = make_uint4(pack2<kBF16>(o[8 * q] * inv, o[8 * q + 1] * inv),
                                             pack2<kBF16>(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                             pack2<kBF16>(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                             pack2<kBF16>(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(box + h * 128 + ((q ^ (h & 7)) << 4)) = v[q];
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarEpiW));
        if (threadIdx.x == 0) {
          ok = mbar_wait_or_abort(bar(kBarEpiW), epi_round & 1, p.err_flag, abort_word);
          if (ok) {
            for (int bi = 0; bi < 2 * nbt; ++bi) {
              const uint32_t src = sbase + kOffRing + bi * kQChunkBytes;
              if (partial)
                tma_store_2d(&tm_po, col0 + bi * 32, slot * kMlaHeads, src);
              else
                tma_store_2d(&tm_out, col0 + bi * 64, static_cast<int>(head0), src);
            }
            bulk_commit_group();
            bulk_wait_read_all();
            mbar_arrive(bar(kBarEpiR));
          }
        }
        if (ok) ok = mbar_wait_or_abort(bar(kBarEpiR), epi_round & 1, p.err_flag, abort_word);
        ++epi_round;
      }
      if (!ok) break;
      if (threadIdx.x == 0) mbar_arrive(bar(kBarEpiDone));
      // This thread's next segment writes Q into TMEM only now, after its
      // own O reads; the MMA thread starts that segment (whose first PV
      // overwrites O) only once all softmax threads have done so.
      g += n_tiles;
      ++k;
    }
  }

  // The epilogue's bulk stores belong to thread 0: let them complete.
  if (threadIdx.x == 0) bulk_wait_all();
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
                     const CUtensorMap& tc4, const CUtensorMap& tout, const CUtensorMap& tpo,
                     cudaStream_t stream) {
  auto kern = mla_partial_kernel<kBF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * p.n_pairs, 1);
  kern<<<grid, kThreads, kSmemBytes, stream>>>(tqa, tc, tc4, tout, tpo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mla_partial(const MlaParams& p, const CUtensorMap& tm_qa,
                               const CUtensorMap& tm_c, const CUtensorMap& tm_c4,
                               const CUtensorMap& tm_out, const CUtensorMap& tm_po, bool bf16,
                               cudaStream_t stream) {
  if (p.block_size > kT && (p.block_size % kT) != 0) return cudaErrorNotSupported;
  return bf16 ? launch_t<true>(p, tm_qa, tm_c, tm_c4, tm_out, tm_po, stream)
              : launch_t<false>(p, tm_qa, tm_c, tm_c4, tm_out, tm_po, stream);
}

}  // namespace decattn
