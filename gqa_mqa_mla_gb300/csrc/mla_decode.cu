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
// S = Q C^T and the same online softmax, so they need to exchange nothing;
// the cluster only co-schedules the pair so that the second load of every
// cache tile is an L2 hit.  The redundant score GEMM costs 1.44x the minimum
// tensor work.  (Each CTA sums the 576 dimensions in its own chunk order, so
// the two CTAs' scores may differ in the last bit; each CTA normalises its
// own columns with its own row sums.)
//
// Tensor-core costs that shape the kernel (measured on GB300 with M = 128,
// K = 16, bf16): one issuing thread cannot issue tcgen05.mma faster than one
// per ~36 cycles (A in TMEM) for any N up to 64 when the whole warp computes
// the operands and one elected lane issues (about 50 cycles from a lane-0
// branch, which needs three times the instructions per MMA); with A in
// shared memory an N = 64 MMA takes 48 cycles (shared-memory bandwidth), an
// N = 256 MMA 128.  So the score chain (36 MMAs of N = 64 per tile) is bound
// by its issue rate, and the value GEMM is issued by a second warp:
// O += P(j) C_lat(j) runs on the tensor pipe while the first warp issues
// S(j + 1), which itself runs while the softmax warps work on tile j.
//
// Chunks: the 576 columns are nine 64-column chunks; CTA r's value chunks are
// 4r..4r+3 (latent columns [256 r, 256 r + 256)), its score chunks the other
// five.  Every CTA keeps its chunks in "position" order: positions 0-4 hold
// the score chunks (4-4r..7-4r, then the RoPE chunk 8) and positions 5-8 the
// value chunks, so that one instruction sequence serves both CTAs.
// Operand placement (per CTA):
//   Q, positions 0-2, 4  TMEM, 128 columns (two 16-bit values per column) A of S
//   Q, positions 3, 5-8  shared memory (TMA), 128-byte swizzled K-major  A of S
//   cache tiles        shared memory ring, 2 stages x 64 tokens x 9     B of S;
//                      chunk slots in position order                    positions 5-8: B of PV
//   S(j), P(j)         TMEM, two 64-column buffers (j % 2): S in fp32,  A of PV (P)
//                      then P(j) (16-bit) over its first 32 columns
//   epilogue           the ring stage of the segment's last tile
// TMEM columns: O [0, 256) | Q [256, 384) | S/P buffer 0 [384, 448) | buffer 1 [448, 512).
// With two S buffers the score chain does not wait for the softmax: S(j + 1)
// runs while the softmax works on S(j); S(j + 2) reuses buffer j % 2 once
// O += P(j) C(j), the last reader of P(j) there, has completed.  While an MMA
// runs, threads touch only TMEM columns it neither reads nor writes: the
// softmax writes P(j) over S(j) only after every softmax thread has loaded
// S(j); O is rescaled only after O += P(j - 1) C(j - 1) has completed (and
// before O += P(j) C(j) is issued, which waits for P(j)).
//
// Per CTA (352 threads):
//   warps 0-7  load Q, softmax, epilogue: warp w serves heads
//              h = 32 (w % 4) + lane (TMEM lane h) over score columns
//              [32 (w / 4), 32 (w / 4) + 32) and O columns of the same half;
//              both threads of a row read all 64 score columns and take
//              the same row maximum, and keep separate partial row sums;
//   warp 8     TMA producer for the cache ring, walking the block table;
//   warp 9     TMEM allocator; issues the score GEMMs (one elected lane);
//   warp 10    issues the value GEMMs (one elected lane).
//
// Ring: a stage holds all 9 column chunks of a 64-token tile.  This CTA's 4
// value chunks (latent columns [256 r, 256 r + 256)) stay until O += P C
// has read them; the other 5 ("score chunks") are read by S only and are
// refilled as soon as S(j) completes.  Each CTA's score chain takes its score
// chunks first and its value chunks last, with a full barrier for each part,
// so that a value part refilled only after O += P(j - 2) C(j - 2) is needed
// as late as possible.  The CTA of rank 0 also pulls tiles into L2 two tiles
// ahead of their loads.
//
// Online softmax in the log2 domain with lazy rescaling: the running max
// used for the exponentials only moves (and O is rescaled in TMEM) when a new
// score exceeds it by more than 2^8; otherwise p <= 256 stays exact in bf16 /
// fp16 range and the final division by l uses the same stale max.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr int kT = 64;                          // tokens per tile
constexpr int kBoxRows = kT;                    // rows per TMA box: a whole block up to one tile
constexpr int kStages = 2;                      // cache ring depth
constexpr int kChunk = 64;                      // columns per 128-byte swizzle row
constexpr int kChunks = kMlaWidth / kChunk;     // 9 column chunks per cache row
constexpr int kQSmemChunks = 5;                 // Q positions 5-8 (value chunks) and 3 in shared memory
constexpr int kQPos3Slot = 4;                   // shared-memory Q chunk slot of position 3
constexpr int kValueSlot = 5;                   // ring slot (position) of the first value chunk
constexpr int kQChunkBytes = kMlaHeads * 128;   // [128 heads][64 cols] = 16 KB
constexpr int kCChunkBytes = kT * 128;          // [64 tokens][64 cols] = 8 KB
constexpr int kStageBytes = kChunks * kCChunkBytes;  // 72 KB
constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + kQSmemChunks * kQChunkBytes;  // 80 KB
constexpr int kOffBars = kOffRing + kStages * kStageBytes;     // +144 KB
constexpr int kBarBytes = 256;
constexpr int kOffRed = kOffBars + kBarBytes;                  // row-sum exchange
constexpr int kRedBytes = 2 * kMlaHeads * 4;                   // row sums (and the scan before)
constexpr int kSmemBytes = 1024 + kOffRed + kRedBytes;
constexpr int kSoftmaxThreads = 256;
constexpr int kWarpProducer = 8, kWarpMmaS = 9, kWarpMmaPv = 10;
constexpr int kThreads = kSoftmaxThreads + 96;
constexpr int kTmemCols = 512;
constexpr int kTmemO = 0;
constexpr int kTmemQ = 256;                     // Q positions 0, 1, 2, 4: 128 TMEM columns
constexpr int kTmemS = 384;                     // two S / P buffers of 64 columns
constexpr int kEpiBoxes = 4;                    // 16 KB output boxes staged per round
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when p could exceed 2^8

// mbarrier slots (8 bytes each) inside the barrier area
enum : int {
  kBarQ = 0,                               // Q's TMEM positions written (256 arrivals)
  kBarFullS = 1,                           // kStages: score chunks landed (TMA bytes)
  kBarFullV = kBarFullS + kStages,         // kStages: value chunks landed (TMA bytes)
  kBarEmptyS = kBarFullV + kStages,        // kStages: score chunks free again
  kBarEmptyV = kBarEmptyS + kStages,       // kStages: value chunks free again
  kBarSFull = kBarEmptyV + kStages,        // 2 (buffer j % 2): S(j) computed
  kBarSRead = kBarSFull + 2,               // 2: S(j) loaded by every softmax thread (256 arrivals)
  kBarPFull = kBarSRead + 2,               // 2: P(j) written (256 arrivals)
  kBarPvDone = kBarPFull + 2,              // 2: O += P(j) C_lat(j) complete
  kBarQs = kBarPvDone + 2,                 // Q's shared-memory chunks landed (TMA)
  kBarQFree = kBarQs + 1,                  // a segment's last S done: Q may be replaced
  kBarSum = kBarQFree + 1,                 // row sums exchanged (256 arrivals)
  kBarEpiW = kBarSum + 1,                  // epilogue round staged in smem (256 arrivals)
  kBarEpiR = kBarEpiW + 1,                 // epilogue round's bulk stores have read smem
  kBarDrainS = kBarEpiR + 1,               // every score MMA complete
  kBarDrainP = kBarDrainS + 1,             // every value MMA complete
  kNumBars = kBarDrainP + 1
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier area");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kEpiBoxes * kQChunkBytes <= kStageBytes, "epilogue staging must fit one stage");
static_assert(kTmemS + 2 * kT <= kTmemCols, "tensor memory columns");

// TMEM slot (32 columns each) of Q position p = 0, 1, 2 or 4.
__host__ __device__ constexpr int q_tmem_slot(int pos) { return pos < 3 ? pos : 3; }

// Work schedule.  The batch's 64-token tiles, sequence after sequence, form
// one list of T_all tiles (an invalid seq_len counts as 0 tiles).  A CTA
// pair's time is its tiles plus a fixed cost for every sequence it starts
// beyond its first (an epilogue, a new Q and a pipeline refill: about
// kSegCost tiles' worth, measured with per-CTA clock stamps), so the list
// is cut in cost units: tile g of the r-th non-empty sequence costs
// position c(g) = g + kSegCost r, and pair p of the P pairs takes the tiles
// with c(g) in [p W, p W + W), W = ceil(c_all / P).  A slice that would
// start in the cost gap before a sequence starts at that sequence's first
// tile.  The slice is cut at sequence boundaries into segments: a segment
// holding a whole sequence writes its output rows directly; one holding
// part of a sequence writes an fp32 partial (normalised O and log2-sum-exp)
// that the combine merges.  Only a slice's first and last segments can be
// partial; they go to workspace slots 2 p and 2 p + 1.  A sequence with no
// tiles is zeroed by the pair whose slice contains its start (at tile
// position t: the pair with lo <= t < the next pair's lo).
enum : int { kSegZero = 0, kSegDirect = 1, kSegPartial = 2 };
constexpr int kSegCost = 9;

struct Sched {
  int pair, n_pairs, lo, hi;  // this pair's tile slice [lo, hi)
  int own_end;                // zero-length sequences at tile positions [lo, own_end) are ours
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

// Cache / Q chunk held at position pos by the CTA of rank r (positions 0-4:
// its score chunks, 5-8: its value chunks), and the position of chunk c.
__host__ __device__ constexpr int chunk_at(int r, int pos) {
  return pos < 4 ? 4 - 4 * r + pos : (pos == 4 ? 8 : 4 * r + pos - kValueSlot);
}
__host__ __device__ constexpr int position_of(int r, int c) {
  return c == 8 ? 4 : ((c >> 2) == r ? kValueSlot + (c & 3) : (c & 3));
}
static_assert(chunk_at(0, 0) == 4 && chunk_at(0, 4) == 8 && chunk_at(0, 5) == 0 && chunk_at(0, 8) == 3,
              "position order, CTA 0");
static_assert(chunk_at(1, 0) == 0 && chunk_at(1, 4) == 8 && chunk_at(1, 5) == 4 && chunk_at(1, 8) == 7,
              "position order, CTA 1");
static_assert(position_of(0, chunk_at(0, 6)) == 6 && position_of(1, chunk_at(1, 2)) == 2 &&
                  position_of(1, chunk_at(1, 7)) == 7 && position_of(0, chunk_at(0, 4)) == 4,
              "positions invert the chunk order");

// Next segment of this pair's slice (every role walks the same sequence).
__device__ __noinline__ bool next_seg(const MlaParams& p, const Sched& sc, Cursor& cur, Seg& sg) {
  while (cur.b < p.batch) {
    const int b = cur.b, pref = cur.pref;
    const int len = p.seq_lens[b];
    const int n = seq_tiles(p, len);
    if (n == 0) {
      if (pref >= sc.own_end) return false;  // a later pair's
      ++cur.b;
      if (pref < sc.lo) continue;            // an earlier pair's
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

// ---------------- producer helpers (out of line: the producer's code is
// kept small so that the four roles' loops share the SM's instruction cache)
struct Producer {
  const MlaParams* p;
  const CUtensorMap* tm_c;
  const CUtensorMap* tm_c4;
  volatile int* abort;
  uint32_t ring, bar0;  // shared-memory addresses: ring base, barrier area
  int rank, rows_per_box;
};

// Request one part of ring tile gi (tokens [t0, t0 + nval) of the sequence
// whose block-table row is bt): the 4 value chunks of this CTA (latent columns
// [256 r, 256 r + 256)) or the 5 others.  Waits until the part's previous
// readers have released the stage.  Returns false when the wait gave up.
__device__ __noinline__ bool load_part(const Producer& pr, const int32_t* bt, int t0, int nval,
                                       int gi, bool value_part) {
  const MlaParams& p = *pr.p;
  const int s = gi % kStages;
  const uint32_t empty = pr.bar0 + 8u * static_cast<uint32_t>((value_part ? kBarEmptyV : kBarEmptyS) + s);
  if (!mbar_wait_or_abort(empty, ((gi / kStages) & 1) ^ 1, p.err_flag, pr.abort)) return false;
  const int bs = p.block_size, rpb = pr.rows_per_box;
  const int nbox = (nval + rpb - 1) / rpb;
  const uint32_t st = pr.ring + s * kStageBytes;
  const uint32_t full = pr.bar0 + 8u * static_cast<uint32_t>((value_part ? kBarFullV : kBarFullS) + s);
  const int nparts = value_part ? 4 : kChunks - 4;
  mbar_arrive_expect_tx(full, static_cast<uint32_t>(nbox * nparts * rpb * 128));
#pragma unroll 1
  for (int k = 0; k < nbox; ++k) {
    const int t = t0 + k * rpb;
    // A block id outside [0, num_blocks) lands the box outside the cache
    // tensor, where the copy reads zeros; the softmax warps flag the segment
    // and zero its result.
    const int row = bt[t >> p.log2_block_size] * bs + (t & (bs - 1));
    const uint32_t off = static_cast<uint32_t>(k * rpb * 128);
    if (rpb == kT) {
      // One 64-row box per tile: a 3-D copy brings four chunks at once (this
      // CTA's value chunks, or the other CTA's); chunk 8 (RoPE) goes with the
      // score part.
      const int c0 = value_part ? 4 * pr.rank : 4 - 4 * pr.rank;
      tma_load_3d(st + (value_part ? kValueSlot : 0) * kCChunkBytes, pr.tm_c4, 0, row, c0, full);
      if (!value_part) tma_load_2d(st + 4 * kCChunkBytes, pr.tm_c, 8 * kChunk, row, full);
      continue;
    }
#pragma unroll 1
    for (int c = 0; c < kChunks; ++c) {
      const int pos = position_of(pr.rank, c);
      if ((pos >= kValueSlot) != value_part) continue;
      tma_load_2d(st + pos * kCChunkBytes + off, pr.tm_c, c * kChunk, row, full);
    }
  }
  return true;
}

// Rank 0 pulls the tile at token t0 into L2 (whole-tile boxes only).
__device__ __noinline__ void prefetch_tile(const Producer& pr, const int32_t* bt, int t0) {
  const MlaParams& p = *pr.p;
  const int id = bt[t0 >> p.log2_block_size];
  if (id < 0 || id >= p.num_blocks) return;
  const int row = id * p.block_size + (t0 & (p.block_size - 1));
  tma_prefetch_l2_3d(pr.tm_c4, 0, row, 0);
  tma_prefetch_l2_3d(pr.tm_c4, 0, row, 4);
  tma_prefetch_l2_2d(pr.tm_c, 8 * kChunk, row);
}

// The score chain S = Q C(stage)^T over the 9 chunk positions: positions
// 0-2 and 4 take Q from TMEM, positions 3 and 5-8 from shared memory.
// `part` 0 issues positions 0-4 (the score chunks; the first MMA overwrites
// S), part 1 positions 5-8 (the value chunks).  Fully unrolled: the issue
// rate of this single thread bounds the chain.
template <bool kBF16>
__device__ __forceinline__ void issue_score_part(int part, uint32_t d, uint32_t tmem, uint64_t dq,
                                                 uint64_t db) {
  constexpr uint32_t idesc = idesc_f16(kBF16, 128, kT, false, false);
  constexpr uint64_t kQChunkUnits = kQChunkBytes >> 4;
  constexpr uint64_t kCChunkUnits = kCChunkBytes >> 4;
  if (part == 0) {
#pragma unroll
    for (int pos = 0; pos < kValueSlot; ++pos)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if (pos == 3)
          tc_mma_f16(d, dq + kQPos3Slot * kQChunkUnits + 2 * ks, db + pos * kCChunkUnits + 2 * ks,
                     idesc, 1u);
        else
          tc_mma_f16_ts(d, tmem + kTmemQ + q_tmem_slot(pos) * 32 + ks * 8,
                        db + pos * kCChunkUnits + 2 * ks, idesc, (pos > 0 || ks > 0) ? 1u : 0u);
      }
  } else {
#pragma unroll
    for (int pos = kValueSlot; pos < kChunks; ++pos)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        tc_mma_f16(d, dq + (pos - kValueSlot) * kQChunkUnits + 2 * ks,
                   db + pos * kCChunkUnits + 2 * ks, idesc, 1u);
  }
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

  // ---------------- schedule: block-wide scan of the per-sequence tile
  // counts and non-empty-sequence counts
  Sched sc;
  sc.pair = static_cast<int>(blockIdx.x >> 1);
  sc.n_pairs = static_cast<int>(gridDim.x >> 1);
  Cursor cur0;
  {
    // [0, 32) / [32, 64): per-warp totals / scanned totals of tiles;
    // [64, 96) / [96, 128): the same for non-empty sequences
    int* s_warp = reinterpret_cast<int*>(smem + kOffRed);
    int* s_misc = s_warp + 128;  // cursor sequence, its first tile, lo, hi
    constexpr int kWarpsAll = kThreads / 32;
    const int chunk = (p.batch + kThreads - 1) / kThreads;
    const int b_a = min(p.batch, static_cast<int>(threadIdx.x) * chunk);
    const int b_b = min(p.batch, b_a + chunk);
    int sum = 0, cnt = 0;
    bool bad_len = false;
    for (int b = b_a; b < b_b; ++b) {
      const int len = p.seq_lens[b];
      bad_len |= (len < 0 || len > p.max_seq_len);
      const int n = seq_tiles(p, len);
      sum += n;
      cnt += n > 0;
    }
    if (bad_len && sc.pair == 0 && rank == 0) flag_error(p.err_flag, kFlagBadSeqLen);
    int x = sum, y = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int xu = __shfl_up_sync(0xffffffffu, x, off);
      const int yu = __shfl_up_sync(0xffffffffu, y, off);
      if (lane >= off) {
        x += xu;
        y += yu;
      }
    }
    if (lane == 31) {
      s_warp[warp] = x;
      s_warp[64 + warp] = y;
    }
    __syncthreads();
    if (warp == 0) {
      int v = lane < kWarpsAll ? s_warp[lane] : 0;
      int u = lane < kWarpsAll ? s_warp[64 + lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int vu = __shfl_up_sync(0xffffffffu, v, off);
        const int uu = __shfl_up_sync(0xffffffffu, u, off);
        if (lane >= off) {
          v += vu;
          u += uu;
        }
      }
      s_warp[32 + lane] = v;
      s_warp[96 + lane] = u;
    }
    __syncthreads();
    const int t_all = s_warp[32 + kWarpsAll - 1];
    const int ne_all = s_warp[96 + kWarpsAll - 1];
    const int64_t c_all = t_all + static_cast<int64_t>(kSegCost) * max(0, ne_all - 1);
    const int64_t W0 = (c_all + sc.n_pairs - 1) / sc.n_pairs;
    const int64_t W = W0 > 1 ? W0 : 1;
    const int excl_t = (warp > 0 ? s_warp[32 + warp - 1] : 0) + x - sum;
    const int excl_r = (warp > 0 ? s_warp[96 + warp - 1] : 0) + y - cnt;
    // Slice starts: the pair whose cost target p W falls on tile g of a
    // sequence starts there; a target in the gap before a sequence starts
    // at its first tile; targets past the last tile start at t_all.
    int* starts = p.ws_hdr ? p.ws_hdr + kHdrPref + p.batch + 1 : nullptr;  // [n_pairs + 1]
    int* cprefs = starts ? starts + sc.n_pairs + 1 : nullptr;               // [batch]
    const bool table = starts && sc.pair == 0 && rank == 0;
    if (threadIdx.x == 0) {
      s_misc[2] = t_all;
      s_misc[3] = t_all;
    }
    if (table)
      for (int q = threadIdx.x; q <= sc.n_pairs; q += kThreads) starts[q] = t_all;
    __syncthreads();
    {
      int pref = excl_t, r = excl_r;
      const int64_t lo_c = sc.pair * W, hi_c = lo_c + W;
      for (int b = b_a; b < b_b; ++b) {
        const int n = seq_tiles(p, p.seq_lens[b]);
        if (table) cprefs[b] = pref + kSegCost * r;  // cost position of b's first tile
        if (n > 0) {
          const int64_t cpref = pref + static_cast<int64_t>(kSegCost) * r;
          const int64_t prev_end = r == 0 ? -1 : cpref - kSegCost - 1;  // previous sequence's last tile
          const int64_t last = cpref + n - 1;
          // tile of this sequence where cost target c starts (c in (prev_end, last])
          auto at = [&](int64_t c) { return pref + static_cast<int>(c > cpref ? c - cpref : 0); };
          if (lo_c > prev_end && lo_c <= last) s_misc[2] = at(lo_c);
          if (hi_c > prev_end && hi_c <= last) s_misc[3] = at(hi_c);
          if (table)
            for (int64_t q = prev_end < 0 ? 0 : prev_end / W + 1; q <= last / W && q <= sc.n_pairs;
                 ++q)
              starts[q] = at(q * W);
          ++r;
        }
        pref += n;
      }
    }
    if (threadIdx.x == 0) s_misc[0] = p.batch;
    __syncthreads();
    sc.lo = s_misc[2];
    sc.hi = sc.pair + 1 < sc.n_pairs ? s_misc[3] : t_all;
    sc.own_end = sc.pair + 1 < sc.n_pairs ? sc.hi : INT_MAX;
    // First sequence this pair touches: pref_b + max(n_b, 1) > lo.
    int pref = excl_t, cand = p.batch, cand_pref = 0;
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
      p.ws_hdr[0] = static_cast<int>(W);
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
    mbar_init(bar(kBarQFree), 1);
    mbar_init(bar(kBarSum), kSoftmaxThreads);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFullS + s), 1);
      mbar_init(bar(kBarFullV + s), 1);
      mbar_init(bar(kBarEmptyS + s), 1);
      mbar_init(bar(kBarEmptyV + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSRead + i), kSoftmaxThreads);
      mbar_init(bar(kBarPFull + i), kSoftmaxThreads);
      mbar_init(bar(kBarPvDone + i), 1);
    }
    mbar_init(bar(kBarEpiW), kSoftmaxThreads);
    mbar_init(bar(kBarEpiR), 1);
    mbar_init(bar(kBarDrainS), 1);
    mbar_init(bar(kBarDrainP), 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMmaS) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpProducer) {
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
      Producer pr;
      pr.p = &p;
      pr.tm_c = &tm_c;
      pr.tm_c4 = &tm_c4;
      pr.abort = abort_word;
      pr.ring = sbase + kOffRing;
      pr.bar0 = bar0;
      pr.rank = static_cast<int>(rank);
      pr.rows_per_box = rows_per_box;
      // A part's chunks are refilled once their last reader has completed
      // (S(j - 2) for the score chunks, O += P(j - 2) C(j - 2) for the value
      // chunks; for a segment's last tile, the epilogue staged there).
      auto load = [&](const Seg& sg, const int32_t* bt, int it, bool value_part) -> bool {
        const int t0 = sg.t0 + it * kT;
        if (!load_part(pr, bt, t0, min(kT, sg.t1 - t0), g + it, value_part)) return false;
        if (value_part) v_issued = g + it + 1; else s_issued = g + it + 1;
        return true;
      };
      const bool do_prefetch = rank == 0 && rows_per_box == kT;
      Cursor cur = cur0;
      Seg sg;
      while (ok && next_seg(p, sc, cur, sg)) {
        if (sg.kind == kSegZero) continue;
        const int n = (sg.t1 - sg.t0 + kT - 1) / kT;
        const int32_t* bt = p.block_table + static_cast<size_t>(sg.b) * p.max_blocks_per_seq;
        // Q's shared-memory chunks (this CTA's value columns and position 3)
        // of this segment's sequence, once the previous segment's last S (the
        // last reader of the Q region) has completed; this overlaps the
        // previous segment's epilogue.
        if (q_issued > 0 &&
            !mbar_wait_or_abort(bar(kBarQFree), (q_issued - 1) & 1, p.err_flag, abort_word)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarQs), kQSmemChunks * kQChunkBytes);
        tma_load_2d(sbase + kOffQ + kQPos3Slot * kQChunkBytes, &tm_qa,
                    chunk_at(static_cast<int>(rank), 3) * kChunk, sg.b * kMlaHeads, bar(kBarQs));
        for (int c = 0; c < 4; ++c)
          tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &tm_qa, (4 * static_cast<int>(rank) + c) * kChunk, sg.b * kMlaHeads,
                      bar(kBarQs));
        ++q_issued;
        if (do_prefetch && n > 1) prefetch_tile(pr, bt, sg.t0 + kT);
        // The value part of tile j is released by O += P(j - 2) C(j - 2),
        // about when S(j - 1) completes and releases the score part of tile
        // j + 1: request them in that order.
        ok = load(sg, bt, 0, false);
        for (int it = 0; ok && it < n; ++it) {
          if (do_prefetch && it + 2 < n) prefetch_tile(pr, bt, sg.t0 + (it + 2) * kT);
          ok = load(sg, bt, it, true);
          if (ok && it + 1 < n) ok = load(sg, bt, it + 1, false);
        }
        g += n;
      }
      // Wait for this thread's copies still in flight before the CTA may
      // exit, even when another thread has raised the abort word: a bulk
      // copy must never land in the shared memory of a finished CTA.  Each
      // wait is bounded on its own.
      for (int it = max(0, s_issued - kStages); it < s_issued; ++it)
        if (!mbar_wait(bar(kBarFullS + it % kStages), (it / kStages) & 1, p.err_flag)) break;
      for (int it = max(0, v_issued - kStages); it < v_issued; ++it)
        if (!mbar_wait(bar(kBarFullV + it % kStages), (it / kStages) & 1, p.err_flag)) break;
      if (q_issued > 0) mbar_wait(bar(kBarQs), (q_issued - 1) & 1, p.err_flag);
    }
  } else if (warp == kWarpMmaS) {
    // ---------------- score GEMM issuer: the whole warp runs the loop and
    // computes the operands (uniform registers), lane 0 waits on the
    // barriers and the elected lane (lane 0: the warp is converged) issues
    // the MMAs and their commits.
    // Shared-memory descriptors are built once; within a swizzle atom and
    // across chunks / stages only the 14-bit start address (16-byte units,
    // low bits of the descriptor) moves.
    const uint64_t dq = smem_desc_sw128(sbase + kOffQ, 16, 1024);
    const uint64_t dr = smem_desc_sw128(sbase + kOffRing, 16, 1024);
    constexpr uint64_t kStageUnits = kStageBytes >> 4;
    auto wait = [&](int b, uint32_t parity) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait_or_abort(bar(b), parity, p.err_flag, abort_word);
      return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    };
    bool ok = true;
    int g = 0, k = 0;
    Cursor cur = cur0;
    Seg sg;
    while (ok && next_seg(p, sc, cur, sg)) {
      if (sg.kind == kSegZero) continue;
      const int n = (sg.t1 - sg.t0 + kT - 1) / kT;
      // This segment's Q: the TMEM part (softmax warps) and the TMA part.
      ok = wait(kBarQ, k & 1) && wait(kBarQs, k & 1);
      for (int j = 0; ok && j < n; ++j) {
        const int gi = g + j;
        const int s = gi % kStages;
        const uint32_t ph = static_cast<uint32_t>(gi / kStages) & 1u;
        // S(gi) goes to buffer gi % 2 once O += P(gi - 2) C(gi - 2) (the last
        // reader of P(gi - 2) there) has completed.
        const uint32_t sbuf = tmem + kTmemS + 64 * (gi & 1);
        ok = (gi < 2 || wait(kBarPvDone + (gi & 1), ((gi - 2) >> 1) & 1)) && wait(kBarFullS + s, ph);
        if (!ok) break;
        tc_fence_after();
        const uint64_t db = dr + static_cast<uint64_t>(s) * kStageUnits;
        if (elect_one()) issue_score_part<kBF16>(0, sbuf, tmem, dq, db);
        __syncwarp();
        ok = wait(kBarFullV + s, ph);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          issue_score_part<kBF16>(1, sbuf, tmem, dq, db);
          tc_commit(bar(kBarSFull + (gi & 1)));
          // Q may be replaced once a segment's last S has completed.
          tc_commit(bar(j + 1 < n ? kBarEmptyS + s : kBarQFree));
        }
        __syncwarp();
      }
      g += n;
      ++k;
    }
    // Wait (bounded) until every MMA this warp issued has completed.
    if (elect_one()) {
      tc_commit(bar(kBarDrainS));
      mbar_wait(bar(kBarDrainS), 0, p.err_flag);
    }
    __syncwarp();
  } else if (warp == kWarpMmaPv) {
    // ---------------- value GEMM issuer (the same warp structure)
    constexpr uint32_t idesc_pv = idesc_f16(kBF16, 128, 256, false, true);
    const uint64_t dv =
        smem_desc_sw128(sbase + kOffRing + kValueSlot * kCChunkBytes, kCChunkBytes, 1024);
    constexpr uint64_t kStageUnits = kStageBytes >> 4;
    bool ok = true;
    int g = 0;
    Cursor cur = cur0;
    Seg sg;
    while (ok && next_seg(p, sc, cur, sg)) {
      if (sg.kind == kSegZero) continue;
      const int n = (sg.t1 - sg.t0 + kT - 1) / kT;
      for (int j = 0; ok && j < n; ++j) {
        const int gi = g + j;
        bool w = true;
        if (lane == 0)
          w = mbar_wait_or_abort(bar(kBarPFull + (gi & 1)), (gi >> 1) & 1, p.err_flag, abort_word);
        ok = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
        if (!ok) break;
        tc_fence_after();
        // O += P(gi) C_lat(gi) over this CTA's 256 value columns (MN-major
        // B); the first tile of a segment overwrites O.
        const uint64_t db = dv + static_cast<uint64_t>(gi % kStages) * kStageUnits;
        if (elect_one()) {
#pragma unroll
          for (int ks = 0; ks < kT / 16; ++ks)
            tc_mma_f16_ts(tmem + kTmemO, tmem + kTmemS + 64 * (gi & 1) + ks * 8,
                          db + ks * (2048 >> 4), idesc_pv,
                          (j > 0 || ks > 0) ? 1u : 0u);
          tc_commit(bar(kBarPvDone + (gi & 1)));
          if (j + 1 < n) tc_commit(bar(kBarEmptyV + gi % kStages));
        }
        __syncwarp();
      }
      g += n;
    }
    if (elect_one()) {
      tc_commit(bar(kBarDrainP));
      mbar_wait(bar(kBarDrainP), 0, p.err_flag);
    }
    __syncwarp();
  } else if (warp < kWarpProducer) {
    // ---------------- softmax warps: thread (h, ch) owns head h, column half ch
    const int h = (warp & 3) * 32 + lane;
    const int ch = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* red_sum = reinterpret_cast<float*>(smem + kOffRed);       // [2 halves][128]
    const float scale = p.scale_log2;
    // Q row h of sequence b at positions 0, 1, 2 and 4 into TMEM (positions
    // 3 and 5-8 arrive in shared memory by TMA); the two halves take two
    // positions each, all loads in flight before any store.  Called only
    // while no MMA reads the Q columns (before the segment's first S, after
    // the previous segment's last S has completed).
    auto load_q_tmem = [&](int b) {
      const size_t row = static_cast<size_t>(b) * kMlaHeads + h;
      const uint4* qa = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q_abs) +
                                                       row * kMlaDc);
      const uint4* qr = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q_rope) +
                                                       row * kMlaDr);
      const int pos2[2] = {ch == 0 ? 0 : 2, ch == 0 ? 1 : 4};
      uint4 w[16];
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const int c = chunk_at(static_cast<int>(rank), pos2[kk / 8]);
        w[kk] = c < 8 ? qa[c * 8 + kk % 8] : qr[kk % 8];
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float v[32];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          v[4 * kk] = __uint_as_float(w[cc * 8 + kk].x);
          v[4 * kk + 1] = __uint_as_float(w[cc * 8 + kk].y);
          v[4 * kk + 2] = __uint_as_float(w[cc * 8 + kk].z);
          v[4 * kk + 3] = __uint_as_float(w[cc * 8 + kk].w);
        }
        tmem_st32(tmem + lane_base + kTmemQ + q_tmem_slot(pos2[cc]) * 32, v);
      }
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarQ));
    };
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
      // The first segment's Q; later segments' Q was loaded right after the
      // previous segment's last tile.
      if (k == 0) load_q_tmem(sg.b);

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
        const int sb = gj & 1;                        // S / P buffer of this tile
        const uint32_t sp_phase = static_cast<uint32_t>(gj >> 1) & 1u;
        if (!mbar_wait_or_abort(bar(kBarSFull + sb), sp_phase, p.err_flag, abort_word)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // This thread's 32 score columns, and the partner half's, from which
        // both threads of the row take the same full-row maximum (no exchange).
        float s[32], so[32];
        tmem_ld32(tmem + lane_base + kTmemS + 64 * sb + ch * 32, s);
        tmem_ld32(tmem + lane_base + kTmemS + 64 * sb + (ch ^ 1) * 32, so);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kBarSRead + sb));  // P(j) may overwrite S(j) once all have loaded it
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
        const bool need = mt > m_used + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mt : m_used;
          const float factor = need ? ex2(m_used - m_new) : 1.f;  // 0 when m_used = -inf
          if (j > 0) {
            // O += P(j - 1) C(j - 1) must have completed before O is rescaled.
            // (The previous segment's last one was waited for by its epilogue.)
            if (!mbar_wait_or_abort(bar(kBarPvDone + ((gj - 1) & 1)), ((gj - 1) >> 1) & 1,
                                    p.err_flag, abort_word)) {
              ok = false;
              break;
            }
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
            // bf16 P without the pack conversion (see pack2_bf16_pos); fp16
            // keeps cvt.rn, whose subnormal results an integer form would lose.
            if constexpr (kBF16)
              pk[kk] = pack2_bf16_pos(p0, p1);
            else
              pk[kk] = pack2<false>(p0, p1);
          }
          lt_tile = (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        l += lt_tile;
        // P(j) over the first 32 columns of S(j)'s buffer, once every softmax
        // thread has loaded S(j) (both threads of a row read all 64 columns).
        if (!mbar_wait_or_abort(bar(kBarSRead + sb), sp_phase, p.err_flag, abort_word)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(tmem + lane_base + kTmemS + 64 * sb + ch * 16, pk);
        if (nval < kT) {
          // Value rows past the sequence end may hold anything (even NaN): zero
          // them so that P = 0 there contributes exactly nothing.  S(j) has
          // already read them; O += P(j) C(j) reads them after P(j) is published.
          uint8_t* st = smem + kOffRing + (gj % kStages) * kStageBytes + kValueSlot * kCChunkBytes;
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
        mbar_arrive(bar(kBarPFull + sb));
        if (j + 2 == n_tiles) {
          // Pull the next segment's Q rows into L2 for its TMEM load.
          Cursor c2 = cur;
          Seg nx;
          bool have = false;
          while (!have && next_seg(p, sc, c2, nx)) have = nx.kind != kSegZero;
          if (have) {
            const char* row = reinterpret_cast<const char*>(
                static_cast<const uint16_t*>(p.q_abs) + (static_cast<size_t>(nx.b) * kMlaHeads + h) * kMlaDc);
            for (int i = 0; i < 2; ++i) {
              const int c = chunk_at(static_cast<int>(rank), i == 0 ? (ch == 0 ? 0 : 2) : (ch == 0 ? 1 : 4));
              if (c < 8)
                prefetch_l2(row + c * 128);
              else
                prefetch_l2(static_cast<const uint16_t*>(p.q_rope) +
                            (static_cast<size_t>(nx.b) * kMlaHeads + h) * kMlaDr);
            }
          }
        }
      }
      if (!ok) break;

      // The segment's last S has completed (it was read above): load the
      // next segment's Q into TMEM now, so that its first S overlaps this
      // epilogue.
      {
        Cursor c2 = cur;
        Seg nx;
        bool have = false;
        while (!have && next_seg(p, sc, c2, nx)) have = nx.kind != kSegZero;
        if (have) load_q_tmem(nx.b);
      }

      // ---------------- epilogue: O row h, this thread's 128 columns, / l
      const int g_last = g + n_tiles - 1;
      red_sum[ch * kMlaHeads + h] = l;
      mbar_arrive(bar(kBarSum));
      ok = mbar_wait_or_abort(bar(kBarSum), k & 1, p.err_flag, abort_word) &&
           mbar_wait_or_abort(bar(kBarPvDone + (g_last & 1)), (g_last >> 1) & 1, p.err_flag,
                              abort_word);
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
      // the ring stage of the segment's last tile (idle: its S and O += P C
      // have completed, and the producer refills it only after this
      // epilogue releases it): 128-row boxes of 128-byte rows, 128-byte
      // swizzled (16-byte chunk j of row y at chunk j ^ (y % 8),
      // conflict-free for a warp writing 32 rows), four boxes per round.  A
      // 16-bit output (this CTA's 256 columns) is 4 boxes of 64 columns, one
      // round; an fp32 partial is 8 boxes of 32 columns, two rounds.
      const uint32_t stage_off = static_cast<uint32_t>(kOffRing + (g_last % kStages) * kStageBytes);
      const int rounds = partial ? 2 : 1;
#pragma unroll 1
      for (int rd = 0; ok && rd < rounds; ++rd) {
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint8_t* box = smem + stage_off + (ch * 2 + cc) * kQChunkBytes;
          uint4 v[8];
          if (partial) {
            float o[32];
            tmem_ld32(tmem + lane_base + kTmemO + ch * 128 + (rd * 2 + cc) * 32, o);
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
            for (int sl = 0; sl < kEpiBoxes; ++sl) {
              const uint32_t src = sbase + stage_off + sl * kQChunkBytes;
              // staging slot sl = 2 ch + cc holds column box (ch, rd, cc)
              if (partial)
                tma_store_2d(&tm_po, col0 + ((sl >> 1) * 4 + rd * 2 + (sl & 1)) * 32,
                             slot * kMlaHeads, src);
              else
                tma_store_2d(&tm_out, col0 + sl * 64, static_cast<int>(head0), src);
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
      // The stage is free again: release both of its parts to the producer.
      if (threadIdx.x == 0) {
        mbar_arrive(bar(kBarEmptyS + g_last % kStages));
        mbar_arrive(bar(kBarEmptyV + g_last % kStages));
      }
      g += n_tiles;
      ++k;
    }
  }

  // The epilogue's bulk stores belong to thread 0: let them complete.
  if (threadIdx.x == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaS) {
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
