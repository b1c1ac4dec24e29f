// gqa_decode.cu -- split-KV partial kernels for MHA / GQA / MQA decode over a
// paged KV cache, sm_103a.
//
// One CTA handles one (split, KV head j, sequence b): the query heads
// j*G .. j*G+G-1 (G = h_q / h_kv) that read KV head j ("MQA, GQA, and MLA",
// section 8: query head i reads KV head i / (h/g), index arithmetic, no
// copy).  Each K/V tile is fetched ONCE from HBM by TMA into shared memory
// and reused by the whole query-head group.
//
// Warp roles:
//   warp 0        producer: walks the block table (token t of sequence b is
//                 slot t % block_size of block block_table[b][t / block_size])
//                 and issues 2-D TMA loads of 64-token K and V tiles into a
//                 multi-stage ring guarded by mbarriers;
//   warps 1..W    consumers: scores, fp32 online softmax (base 2, the scale
//                 folded with log2 e) and the P.V accumulation, each warp on
//                 its own slice of the tile's tokens with its own (m, l, o);
//                 the warps' states are merged through shared memory at the
//                 end and written as the final output (one split) or as an
//                 fp32 partial (o, lse) for the log-sum-exp combine.
//
// Two consumer flavours:
//   CcConsumer<G>    CUDA cores, used for MHA (G = 1): a half-warp holds one
//                    token row (16 lanes x 16 B), warp-shuffle dot products;
//   MmaConsumer<MT>  tensor cores (mma.sync m16n8k16) for 2 <= G <= 16 (wider
//                    groups run on the tcgen05 kernel of gqa_wide.cu): the
//                    query group padded to 16*MT rows is the A operand, K^T / V
//                    the B operand read with ldmatrix from the swizzled tile.
//
// Shared-memory tile layout (written by TMA with 128-byte swizzle): a stage
// holds K then V; each holds 64 token rows of 256 B in groups of
// R = min(block size, 64) rows, one box per cache block, a group being
// [2 column halves][R rows][128 B] (tile_off below); the 16-byte chunk c of a
// 128-byte row r sits at chunk (c ^ (r % 8)) of that row.
//
// 8-bit (e4m3) caches ("Why GQA's KV Cache Savings Don't Fully Reduce TPOT",
// "When the Serving Engineer Doesn't Get to Choose the Model Architecture":
// an fp8 cache halves the bytes, quantised at KV-head granularity): one
// 128-byte swizzle row holds a token's whole 128-d head, so a K or V tile is
// [64 tokens][128 B].  The consumers build fp16 mma fragments straight from
// those bytes (cvt e4m3x2 -> f16x2), with no staging copy; K's scale folds
// into the score scale and V's into the output.  Up to 16 query heads per KV
// head they use the transposed products S^T = K Q^T, O^T += V^T P^T, where
// the group is the mma's N and a group of 8 fills every tile
// (MmaConsumerF8T); wider groups go to the tcgen05 kernel of gqa_wide.cu.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gqa_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace decattn {
namespace {

constexpr int kHalfBytes = kTile * 128;         // one 64-column half of a K or V tile
constexpr int kKvTileBytes = 2 * kHalfBytes;    // 16 KB
constexpr int kStageBytes = 2 * kKvTileBytes;   // K + V: 32 KB
constexpr float kNegInf = -__builtin_huge_valf();

// Byte offset of 16-byte chunk c (0..15) of token row r (0..63) in a 16-bit
// K or V tile.  The tile lands in groups of R = min(block size, 64) rows
// (lg_r = log2 R), one box per group holding both 64-column halves: group
// r / R at (r / R) 2R x 128 B, half c / 8 R x 128 B into it, then row
// r % R; R = 64 is the plain [2 halves][64 rows][128 B] layout.
__device__ __forceinline__ uint32_t tile_off(int r, int c, int lg_r) {
  return static_cast<uint32_t>((((r >> lg_r) + (c >> 3)) << (lg_r + 7)) + r * 128 +
                               (((c & 7) ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ CUDA-core consumer

template <int G, bool kBF16>
struct CcConsumer {
  static constexpr int kCacheBytes = 2;
  static constexpr int kMinBlocks = 1;
  static constexpr int kWarps = 4;
  static constexpr int kRowsPerWarp = G;

  float q[G][8];
  float o[G][8];
  float m[G], l[G];
  int chunk, half, cw, lg_r;

  __device__ __forceinline__ void init(const GqaParams& p, int b, int j, int cw_, int lane) {
    cw = cw_;
    chunk = lane & 15;  // 16-byte chunk of the 256-byte row: d = chunk*8 .. chunk*8+7
    half = lane >> 4;   // the two half-warps take alternate tokens
    lg_r = min(p.log2_block_size, 6);
    const uint16_t* qb = static_cast<const uint16_t*>(p.q);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const size_t row = static_cast<size_t>(b) * p.h_q + j * G + g;
      const uint4 w = *reinterpret_cast<const uint4*>(qb + row * kHeadDim + chunk * 8);
      const float2 a = unpack2<kBF16>(w.x), bb = unpack2<kBF16>(w.y), c = unpack2<kBF16>(w.z),
                   d = unpack2<kBF16>(w.w);
      q[g][0] = a.x; q[g][1] = a.y; q[g][2] = bb.x; q[g][3] = bb.y;
      q[g][4] = c.x; q[g][5] = c.y; q[g][6] = d.x; q[g][7] = d.y;
      m[g] = kNegInf;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] = 0.f;
    }
  }

  __device__ __forceinline__ static void load8(const uint8_t* p, float (&x)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const float2 a = unpack2<kBF16>(w.x), b = unpack2<kBF16>(w.y), c = unpack2<kBF16>(w.z),
                 d = unpack2<kBF16>(w.w);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y; x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
  }

  // Process this warp's 16 tokens (rows cw*16 .. cw*16+15) of one stage;
  // rows >= nval are past the sequence end and rows < nskip before a sliding
  // window: neither is used.
  __device__ __forceinline__ void tile(const uint8_t* stage, int nskip, int nval, float scale_log2) {
    const unsigned span = static_cast<unsigned>(nval - nskip);  // nskip < nval
    const uint8_t* ks = stage;
    const uint8_t* vs = stage + kKvTileBytes;
    float s[8][G];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = cw * 16 + 2 * i + half;
      float k[8];
      load8(ks + tile_off(r, chunk, lg_r), k);
      float part[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(q[g][e], k[e], acc);
        part[g] = acc;
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] += __shfl_xor_sync(0xffffffffu, part[g], off);
      }
      const bool live = static_cast<unsigned>(r - nskip) < span;
#pragma unroll
      for (int g = 0; g < G; ++g) s[i][g] = live ? part[g] * scale_log2 : kNegInf;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mt = s[0][g];
#pragma unroll
      for (int i = 1; i < 8; ++i) mt = fmaxf(mt, s[i][g]);
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
      const float m_new = fmaxf(m[g], mt);
      const float corr = (m_new == kNegInf) ? 1.f : ex2(m[g] - m_new);
      m[g] = m_new;
      l[g] *= corr;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] *= corr;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = cw * 16 + 2 * i + half;
      if (static_cast<unsigned>(r - nskip) < span) {
        float v[8];
        load8(vs + tile_off(r, chunk, lg_r), v);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pr = ex2(s[i][g] - m[g]);
          l[g] += pr;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[g][e] = fmaf(pr, v[e], o[g][e]);
        }
      }
    }
  }

  // Write this warp's (m, l, o) rows to the merge area.
  __device__ __forceinline__ void finish(float* mo, float* mm, float* ml, int lane) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], 16);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
    }
    if (half == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float4* dst = reinterpret_cast<float4*>(mo + (cw * kRowsPerWarp + g) * kHeadDim + chunk * 8);
        dst[0] = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
        dst[1] = make_float4(o[g][4], o[g][5], o[g][6], o[g][7]);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mm[cw * kRowsPerWarp + g] = m[g];
        ml[cw * kRowsPerWarp + g] = l[g];
      }
    }
  }

  // Does consumer warp w hold row r, and at which slot row?
  __device__ __forceinline__ static int slot(int w, int r) { return w * kRowsPerWarp + r; }
  __device__ __forceinline__ static bool covers(int /*w*/, int /*r*/) { return true; }
};

// ------------------------------------------------------------------ tensor-core consumer

template <int MT, bool kBF16>
struct MmaConsumer {
  static constexpr int kCacheBytes = 2;
  static constexpr int kMinBlocks = 1;
  // One m-tile (up to 16 query heads): 4 warps.  Wider groups: 8 warps, so
  // that two warps per SM sub-partition hide each other's latency (the
  // register file then holds one CTA per SM either way).
  static constexpr int kWarps = MT == 1 ? 4 : 8;
  static constexpr int kRowsPerWarp = 16;
  static constexpr int kWarpsPerMtile = kWarps / MT;
  static constexpr int kTokensPerWarp = kTile / kWarpsPerMtile;

  uint32_t qa[8][4];  // A fragments of the padded query group, 8 k-steps of 16
  float o[16][4];     // 16 n-tiles of 8 head dims, rows (lane/4, lane/4+8)
  float m[2], l[2];
  int mt, tok0, cw, lane, lg_r;

  __device__ __forceinline__ void init(const GqaParams& p, int b, int j, int cw_, int lane_) {
    cw = cw_;
    lane = lane_;
    lg_r = min(p.log2_block_size, 6);
    mt = cw % MT;
    tok0 = (cw / MT) * kTokensPerWarp;
    const int G = p.group;
    const int r_lo = mt * 16 + (lane >> 2);
    const int r_hi = r_lo + 8;
    const int kc = (lane & 3) * 2;
    const uint32_t* qb = static_cast<const uint32_t*>(p.q);
    const size_t base = (static_cast<size_t>(b) * p.h_q + static_cast<size_t>(j) * G) * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int k0 = ks * 16 + kc;
      qa[ks][0] = r_lo < G ? qb[(base + r_lo * kHeadDim + k0) >> 1] : 0u;
      qa[ks][1] = r_hi < G ? qb[(base + r_hi * kHeadDim + k0) >> 1] : 0u;
      qa[ks][2] = r_lo < G ? qb[(base + r_lo * kHeadDim + k0 + 8) >> 1] : 0u;
      qa[ks][3] = r_hi < G ? qb[(base + r_hi * kHeadDim + k0 + 8) >> 1] : 0u;
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m[0] = m[1] = kNegInf;
    l[0] = l[1] = 0.f;
  }

  __device__ __forceinline__ void tile(uint8_t* stage, int nskip, int nval, float scale_log2) {
    const unsigned span = static_cast<unsigned>(nval - nskip);  // nskip < nval
    const uint32_t ks_base = smem_u32(stage);
    const uint32_t vs_base = ks_base + kKvTileBytes;
    const int t4 = lane & 3;
#pragma unroll
    for (int c = 0; c < kTokensPerWarp / 16; ++c) {
      const int r0 = tok0 + 16 * c;
      if (r0 >= nval) break;
      if (r0 + 16 <= nskip) continue;  // wholly before a sliding window
      if (r0 + 16 > nval || r0 < nskip) {
        // Rows past the sequence end (or before a sliding window) may hold
        // anything, even NaN; zero their V rows so that P = 0 there
        // contributes exactly nothing.  Both ranges are under 16 rows.
        uint8_t* vs = stage + kKvTileBytes;
        const int lo = max(0, nskip - r0), hi = max(0, r0 + 16 - nval);
        for (int idx = lane; idx < (lo + hi) * 16; idx += 32) {
          const int k = idx >> 4;
          const int r = k < lo ? r0 + k : nval + (k - lo);
          *reinterpret_cast<uint4*>(vs + tile_off(r, idx & 15, lg_r)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // S = Q K^T for 16 tokens: two n-tiles of 8 tokens.
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int mi = lane >> 3;
        const int tok = r0 + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(ks_base + tile_off(tok, 2 * ks + (mi & 1), lg_r), b0, b1, b2, b3);
          mma_16816<kBF16>(s0, qa[ks], b0, b1);
          mma_16816<kBF16>(s1, qa[ks], b2, b3);
        }
      }
      // Scale into the log2 domain and mask tokens outside [nskip, nval).
      // ta, tb count from the window start: valid rows are [0, span).
      const int ta = r0 - nskip + 2 * t4, tb = ta + 8;
      s0[0] = static_cast<unsigned>(ta) < span ? s0[0] * scale_log2 : kNegInf;
      s0[1] = static_cast<unsigned>(ta + 1) < span ? s0[1] * scale_log2 : kNegInf;
      s0[2] = static_cast<unsigned>(ta) < span ? s0[2] * scale_log2 : kNegInf;
      s0[3] = static_cast<unsigned>(ta + 1) < span ? s0[3] * scale_log2 : kNegInf;
      s1[0] = static_cast<unsigned>(tb) < span ? s1[0] * scale_log2 : kNegInf;
      s1[1] = static_cast<unsigned>(tb + 1) < span ? s1[1] * scale_log2 : kNegInf;
      s1[2] = static_cast<unsigned>(tb) < span ? s1[2] * scale_log2 : kNegInf;
      s1[3] = static_cast<unsigned>(tb + 1) < span ? s1[3] * scale_log2 : kNegInf;
      float mx_lo = fmaxf(fmaxf(s0[0], s0[1]), fmaxf(s1[0], s1[1]));
      float mx_hi = fmaxf(fmaxf(s0[2], s0[3]), fmaxf(s1[2], s1[3]));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      // Every chunk holds at least one valid token, so the new maxima are finite.
      const float mn_lo = fmaxf(m[0], mx_lo), mn_hi = fmaxf(m[1], mx_hi);
      const float c_lo = ex2(m[0] - mn_lo), c_hi = ex2(m[1] - mn_hi);
      m[0] = mn_lo;
      m[1] = mn_hi;
      l[0] *= c_lo;
      l[1] *= c_hi;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= c_lo; o[n][1] *= c_lo; o[n][2] *= c_hi; o[n][3] *= c_hi;
      }
      const float p00 = ex2(s0[0] - mn_lo), p01 = ex2(s0[1] - mn_lo);
      const float p02 = ex2(s0[2] - mn_hi), p03 = ex2(s0[3] - mn_hi);
      const float p10 = ex2(s1[0] - mn_lo), p11 = ex2(s1[1] - mn_lo);
      const float p12 = ex2(s1[2] - mn_hi), p13 = ex2(s1[3] - mn_hi);
      l[0] += (p00 + p01) + (p10 + p11);
      l[1] += (p02 + p03) + (p12 + p13);
      const uint32_t pa[4] = {pack2<kBF16>(p00, p01), pack2<kBF16>(p02, p03),
                              pack2<kBF16>(p10, p11), pack2<kBF16>(p12, p13)};
      // O += P V: 16 tokens x 128 dims, V read transposed by ldmatrix.
      {
        const int mi = lane >> 3;
        const int tok = r0 + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(vs_base + tile_off(tok, 2 * dp + (mi >> 1), lg_r), b0, b1, b2, b3);
          mma_16816<kBF16>(o[2 * dp], pa, b0, b1);
          mma_16816<kBF16>(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
  }

  __device__ __forceinline__ void finish(float* mo, float* mm, float* ml, int lane_) {
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], 2);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], 1);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], 2);
    const int rl = lane_ >> 2, t4 = lane_ & 3;
    float* lo = mo + (cw * kRowsPerWarp + rl) * kHeadDim;
    float* hi = mo + (cw * kRowsPerWarp + rl + 8) * kHeadDim;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      *reinterpret_cast<float2*>(lo + n * 8 + 2 * t4) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(hi + n * 8 + 2 * t4) = make_float2(o[n][2], o[n][3]);
    }
    if (t4 == 0) {
      mm[cw * kRowsPerWarp + rl] = m[0];
      ml[cw * kRowsPerWarp + rl] = l[0];
      mm[cw * kRowsPerWarp + rl + 8] = m[1];
      ml[cw * kRowsPerWarp + rl + 8] = l[1];
    }
  }

  __device__ __forceinline__ static bool covers(int w, int r) { return (w % MT) == (r >> 4); }
  __device__ __forceinline__ static int slot(int w, int r) { return w * kRowsPerWarp + (r & 15); }
};

// ------------------------------------------------------------------ 8-bit cache consumers

constexpr int kF8TileBytes = kTile * 128;      // [64 tokens][128 B]: K or V
constexpr int kF8StageBytes = 2 * kF8TileBytes;  // 16 KB

// Byte offset of 16-byte chunk c (0..7) of token row r in an 8-bit tile.
__device__ __forceinline__ uint32_t f8_off(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// CUDA cores, MHA (G = 1): a half-warp holds one token row, lane chunk c
// covers head dims 8c .. 8c + 7 (8 bytes of the row).
template <int G, bool kBF16>
struct CcConsumerF8 {
  static constexpr int kCacheBytes = 1;
  static constexpr int kMinBlocks = 1;
  static constexpr int kWarps = 4;
  static constexpr int kRowsPerWarp = G;

  float q[G][8];
  float o[G][8];
  float m[G], l[G];
  float v_scale;
  int chunk, half, cw;

  __device__ __forceinline__ void init(const GqaParams& p, int b, int j, int cw_, int lane) {
    cw = cw_;
    chunk = lane & 15;
    half = lane >> 4;
    v_scale = p.v_scale[j];
    const uint16_t* qb = static_cast<const uint16_t*>(p.q);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const size_t row = static_cast<size_t>(b) * p.h_q + j * G + g;
      const uint4 w = *reinterpret_cast<const uint4*>(qb + row * kHeadDim + chunk * 8);
      const float2 a = unpack2<kBF16>(w.x), bb = unpack2<kBF16>(w.y), c = unpack2<kBF16>(w.z),
                   d = unpack2<kBF16>(w.w);
      q[g][0] = a.x; q[g][1] = a.y; q[g][2] = bb.x; q[g][3] = bb.y;
      q[g][4] = c.x; q[g][5] = c.y; q[g][6] = d.x; q[g][7] = d.y;
      m[g] = kNegInf;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] = 0.f;
    }
  }

  __device__ __forceinline__ void load8(const uint8_t* tile, int r, float (&x)[8]) const {
    const uint2 w = *reinterpret_cast<const uint2*>(tile + f8_off(r, chunk >> 1) + 8 * (chunk & 1));
    uint32_t h[4];
    e4m3x4_to_f16x2(w.x, h[0], h[1]);
    e4m3x4_to_f16x2(w.y, h[2], h[3]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = unpack2<false>(h[k]);
      x[2 * k] = f.x;
      x[2 * k + 1] = f.y;
    }
  }

  // Process this warp's 16 tokens (rows cw*16 .. cw*16+15) of one stage;
  // rows >= nval are past the sequence end and rows < nskip before a sliding
  // window: neither is used.
  __device__ __forceinline__ void tile(const uint8_t* stage, int nskip, int nval, float scale_log2) {
    const unsigned span = static_cast<unsigned>(nval - nskip);  // nskip < nval
    const uint8_t* ks = stage;
    const uint8_t* vs = stage + kF8TileBytes;
    float s[8][G];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = cw * 16 + 2 * i + half;
      float k[8];
      load8(ks, r, k);
      float part[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(q[g][e], k[e], acc);
        part[g] = acc;
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] += __shfl_xor_sync(0xffffffffu, part[g], off);
      }
      const bool live = static_cast<unsigned>(r - nskip) < span;
#pragma unroll
      for (int g = 0; g < G; ++g) s[i][g] = live ? part[g] * scale_log2 : kNegInf;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mt = s[0][g];
#pragma unroll
      for (int i = 1; i < 8; ++i) mt = fmaxf(mt, s[i][g]);
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
      const float m_new = fmaxf(m[g], mt);
      const float corr = (m_new == kNegInf) ? 1.f : ex2(m[g] - m_new);
      m[g] = m_new;
      l[g] *= corr;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] *= corr;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = cw * 16 + 2 * i + half;
      if (static_cast<unsigned>(r - nskip) < span) {
        float v[8];
        load8(vs, r, v);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pr = ex2(s[i][g] - m[g]);
          l[g] += pr;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[g][e] = fmaf(pr, v[e], o[g][e]);
        }
      }
    }
  }

  // Write this warp's (m, l, o) rows to the merge area; V's scale applies here.
  __device__ __forceinline__ void finish(float* mo, float* mm, float* ml, int lane) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], 16);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
    }
    if (half == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float4* dst = reinterpret_cast<float4*>(mo + (cw * kRowsPerWarp + g) * kHeadDim + chunk * 8);
        dst[0] = make_float4(o[g][0] * v_scale, o[g][1] * v_scale, o[g][2] * v_scale,
                             o[g][3] * v_scale);
        dst[1] = make_float4(o[g][4] * v_scale, o[g][5] * v_scale, o[g][6] * v_scale,
                             o[g][7] * v_scale);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mm[cw * kRowsPerWarp + g] = m[g];
        ml[cw * kRowsPerWarp + g] = l[g];
      }
    }
  }

  __device__ __forceinline__ static int slot(int w, int r) { return w * kRowsPerWarp + r; }
  __device__ __forceinline__ static bool covers(int /*w*/, int /*r*/) { return true; }
};

// Tensor cores for 2..16 query heads per KV head over an 8-bit cache, in the
// transposed form S^T = K Q^T and O^T += V^T P^T: a warp's 16 tokens are the
// mma's M (scores) or its K (values) and the query group is its N, 8 heads
// per n-tile.  A group of 8 then fills every mma -- half the mma work of a
// 16-row padded form (the query group as M), and half its accumulator
// registers, so more warps fit an SM.
//   Scores: ldmatrix gives a thread 4 consecutive head dims (4q .. 4q + 3)
//   of token g = lane / 4 (or g + 8); they fill k-slots (2q, 2q+1) and
//   (2q+8, 2q+9) of the A fragment, and Q^T's B fragments use the same dim
//   order.  The result holds tokens (g, g + 8) x heads (2q, 2q + 1).
//   Values: transposed ldmatrix plus a byte permute give the token pairs
//   (2q, 2q + 1) of dims 2g and 2g + 1 of a 16-dim block: m-tile row g is dim
//   2g, row g + 8 dim 2g + 1.  P^T's B fragment (tokens 2q, 2q+1 of head g) is
//   the score layout transposed: movmatrix per 8 tokens.
template <int NT, bool kBF16>
struct MmaConsumerF8T {
  static constexpr int kCacheBytes = 1;
  static constexpr int kMinBlocks = NT == 1 ? 4 : 2;
  static constexpr int kWarps = 4;
  static constexpr int kRowsPerWarp = 8 * NT;

  uint32_t qb[8][NT][2];  // Q^T B fragments: k-step, n-tile, dims (4q, 4q+1 | 4q+2, 4q+3)
  float o[8][NT][4];      // O^T, 16-dim block b: (2g, 2q) (2g, 2q+1) (2g+1, 2q) (2g+1, 2q+1)
  float m[NT][2], l[NT][2];
  float v_scale;
  int tok0, cw, lane;

  __device__ __forceinline__ void init(const GqaParams& p, int b, int j, int cw_, int lane_) {
    cw = cw_;
    lane = lane_;
    tok0 = cw * 16;
    v_scale = p.v_scale[j];
    const int G = p.group;
    const int g = lane >> 2, q4 = lane & 3;
    const uint16_t* qp = static_cast<const uint16_t*>(p.q);
    const size_t base = (static_cast<size_t>(b) * p.h_q + static_cast<size_t>(j) * G) * kHeadDim;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = 8 * nt + g;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint2 w = make_uint2(0u, 0u);
        if (h < G) w = *reinterpret_cast<const uint2*>(qp + base + h * kHeadDim + ks * 16 + 4 * q4);
        const float2 f0 = unpack2<kBF16>(w.x), f1 = unpack2<kBF16>(w.y);
        qb[ks][nt][0] = pack2<false>(f0.x, f0.y);
        qb[ks][nt][1] = pack2<false>(f1.x, f1.y);
      }
      m[nt][0] = m[nt][1] = kNegInf;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int bb = 0; bb < 8; ++bb) o[bb][nt][0] = o[bb][nt][1] = o[bb][nt][2] = o[bb][nt][3] = 0.f;
    }
  }

  __device__ __forceinline__ void tile(uint8_t* stage, int nskip, int nval, float scale_log2) {
    const unsigned span = static_cast<unsigned>(nval - nskip);  // nskip < nval
    const int r0 = tok0;
    if (r0 >= nval || r0 + 16 <= nskip) return;  // past the end, or before a sliding window
    const uint32_t ks_base = smem_u32(stage);
    const uint32_t vs_base = ks_base + kF8TileBytes;
    if (r0 + 16 > nval || r0 < nskip) {
      // Rows past the sequence end (or before a sliding window) may hold
      // anything, even NaN codes; zero their V rows so that P = 0 there
      // contributes exactly nothing.  Both ranges are under 16 rows.
      uint8_t* vs = stage + kF8TileBytes;
      const int lo = max(0, nskip - r0), hi = max(0, r0 + 16 - nval);
      for (int idx = lane; idx < (lo + hi) * 8; idx += 32) {
        const int k = idx >> 3;
        const int r = k < lo ? r0 + k : nval + (k - lo);
        *reinterpret_cast<uint4*>(vs + f8_off(r, idx & 7)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    const int g = lane >> 2;
    const int mi = lane >> 3;
    const int tok = r0 + ((mi & 1) << 3) + (lane & 7);
    // S^T = K Q^T: one ldmatrix.x4 holds tokens 0-7 and 8-15 of k-steps 2w, 2w + 1.
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t k0, k1, k2, k3;
      ldsm_x4(ks_base + f8_off(tok, 2 * w + (mi >> 1)), k0, k1, k2, k3);
      uint32_t a[4];
      e4m3x4_to_f16x2(k0, a[0], a[2]);
      e4m3x4_to_f16x2(k1, a[1], a[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816<false>(s[nt], a, qb[2 * w][nt][0], qb[2 * w][nt][1]);
      e4m3x4_to_f16x2(k2, a[0], a[2]);
      e4m3x4_to_f16x2(k3, a[1], a[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_16816<false>(s[nt], a, qb[2 * w + 1][nt][0], qb[2 * w + 1][nt][1]);
    }
    // Scale into the log2 domain and mask tokens outside [nskip, nval); ta,
    // tb count from the window start (valid: [0, span)).
    const int ta = r0 + g - nskip, tb = ta + 8;
    const bool la = static_cast<unsigned>(ta) < span, lb = static_cast<unsigned>(tb) < span;
    uint32_t pb[NT][2];
    bool moved = false;
    float cr[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      s[nt][0] = la ? s[nt][0] * scale_log2 : kNegInf;
      s[nt][1] = la ? s[nt][1] * scale_log2 : kNegInf;
      s[nt][2] = lb ? s[nt][2] * scale_log2 : kNegInf;
      s[nt][3] = lb ? s[nt][3] * scale_log2 : kNegInf;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(s[nt][e], s[nt][e + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        // Every chunk holds at least one valid token, so the new maximum is finite.
        const float mn = fmaxf(m[nt][e], mx);
        cr[nt][e] = ex2(m[nt][e] - mn);
        moved |= cr[nt][e] != 1.f;
        m[nt][e] = mn;
        l[nt][e] *= cr[nt][e];
      }
      const float p0 = ex2(s[nt][0] - m[nt][0]), p1 = ex2(s[nt][1] - m[nt][1]);
      const float p2 = ex2(s[nt][2] - m[nt][0]), p3 = ex2(s[nt][3] - m[nt][1]);
      l[nt][0] += p0 + p2;
      l[nt][1] += p1 + p3;
      pb[nt][0] = movmatrix_trans(pack2<false>(p0, p1));  // tokens 0-7
      pb[nt][1] = movmatrix_trans(pack2<false>(p2, p3));  // tokens 8-15
    }
    // Rescale O only when some head's maximum moved (the factors are exactly
    // 1 otherwise): after the first tiles that is rare.
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
      for (int bb = 0; bb < 8; ++bb) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[bb][nt][0] *= cr[nt][0]; o[bb][nt][1] *= cr[nt][1];
          o[bb][nt][2] *= cr[nt][0]; o[bb][nt][3] *= cr[nt][1];
        }
      }
    }
    // O^T += V^T P^T: transposed ldmatrix per 16-dim block pair and token half.
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t v0, v1, v2, v3;  // (tokens 0-7, block 2w), (8-15, 2w), (0-7, 2w+1), (8-15, 2w+1)
      ldsm_x4_trans(vs_base + f8_off(tok, 2 * w + (mi >> 1)), v0, v1, v2, v3);
      uint32_t a[4];
      e4m3x4_to_f16x2(byte_perm(v0, 0u, 0x3120u), a[0], a[1]);
      e4m3x4_to_f16x2(byte_perm(v1, 0u, 0x3120u), a[2], a[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816<false>(o[2 * w][nt], a, pb[nt][0], pb[nt][1]);
      e4m3x4_to_f16x2(byte_perm(v2, 0u, 0x3120u), a[0], a[1]);
      e4m3x4_to_f16x2(byte_perm(v3, 0u, 0x3120u), a[2], a[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816<false>(o[2 * w + 1][nt], a, pb[nt][0], pb[nt][1]);
    }
  }

  // Write this warp's (m, l, o) rows (query heads of the group) to the merge
  // area; V's scale applies here.
  __device__ __forceinline__ void finish(float* mo, float* mm, float* ml, int lane_) {
    const int g = lane_ >> 2, q4 = lane_ & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], 4);
        l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], 8);
        l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], 16);
      }
      const int h0 = cw * kRowsPerWarp + 8 * nt + 2 * q4;
#pragma unroll
      for (int bb = 0; bb < 8; ++bb) {
        const int d0 = 16 * bb + 2 * g;
        *reinterpret_cast<float2*>(mo + h0 * kHeadDim + d0) =
            make_float2(o[bb][nt][0] * v_scale, o[bb][nt][2] * v_scale);
        *reinterpret_cast<float2*>(mo + (h0 + 1) * kHeadDim + d0) =
            make_float2(o[bb][nt][1] * v_scale, o[bb][nt][3] * v_scale);
      }
      if (g == 0) {
        mm[h0] = m[nt][0];
        ml[h0] = l[nt][0];
        mm[h0 + 1] = m[nt][1];
        ml[h0 + 1] = l[nt][1];
      }
    }
  }

  __device__ __forceinline__ static bool covers(int /*w*/, int /*r*/) { return true; }
  __device__ __forceinline__ static int slot(int w, int r) { return w * kRowsPerWarp + r; }
};

// ------------------------------------------------------------------ the kernel

template <class Consumer>
__host__ __device__ constexpr int merge_bytes() {
  return Consumer::kWarps * Consumer::kRowsPerWarp * (kHeadDim + 2) * 4;
}

template <class Consumer>
__host__ __device__ constexpr int stage_bytes() {
  return Consumer::kCacheBytes == 1 ? kF8StageBytes : kStageBytes;
}

template <class Consumer, int kStages>
__host__ __device__ constexpr int smem_bytes() {
  return 1024 /*alignment slack*/ + kStages * stage_bytes<Consumer>() + 256 /*barriers*/;
}

template <class Consumer, bool kBF16, int kStages>
__global__ void __launch_bounds__(32 * (1 + Consumer::kWarps), Consumer::kMinBlocks)
    gqa_partial_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const GqaParams p) {
  constexpr int kStage = stage_bytes<Consumer>();
  static_assert(merge_bytes<Consumer>() <= kStages * kStage, "merge area must fit the ring");
  constexpr int kW = Consumer::kWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStage);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kStages);
  const uint32_t done_bar = smem_u32(bars + 2 * kStages);
  const uint32_t merge_bar = smem_u32(bars + 2 * kStages + 1);

  const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;

  const GqaSpan span = gqa_span(p, split, j, b);
  const int w0 = span.w0, t_begin = span.t_begin, t_end = span.t_end;
  int bad = span.bad;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kW);
    }
    mbar_init(done_bar, kW);
    mbar_init(merge_bar, kW);
    fence_barrier_init();
  }
  bad = __syncthreads_or(bad);

  const size_t row0 = static_cast<size_t>(b) * p.h_q + static_cast<size_t>(j) * G;
  if (bad || t_end <= t_begin) {
    gqa_write_empty(p, row0, G, split, bad);
    return;
  }

  const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;
  const int bs = p.block_size;

  if (warp == 0) {
    // ---------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t policy = policy_evict_first();
      const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
      const int x0 = j * kHeadDim;  // element (= byte, for an 8-bit cache) column of head j
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int s = it % kStages;
        if (!mbar_wait(empty0 + 8 * s, ((it / kStages) & 1) ^ 1, p.err_flag)) break;
        const int t0 = t_begin + it * kTile;
        const int nval = min(kTile, t_end - t0);
        const uint32_t st = smem_u32(smem + s * kStage);
        const uint32_t fb = full0 + 8 * s;
        if constexpr (Consumer::kCacheBytes == 1) {
          // One 128-byte box row per token: K and V tiles of [64][128 B].
          if (bs >= kTile) {
            const int row = bt[t0 >> p.log2_block_size] * bs + (t0 & (bs - 1));
            mbar_arrive_expect_tx(fb, kStage);
            tma_load_2d_hint(st, &tm_k, x0, row, fb, policy);
            tma_load_2d_hint(st + kF8TileBytes, &tm_v, x0, row, fb, policy);
          } else {
            const int nblk = (nval + bs - 1) >> p.log2_block_size;
            const int box = bs * 128;
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nblk * 2 * box));
            for (int k = 0; k < nblk; ++k) {
              const int row = bt[(t0 >> p.log2_block_size) + k] * bs;
              const uint32_t off = static_cast<uint32_t>(k * box);
              tma_load_2d_hint(st + off, &tm_k, x0, row, fb, policy);
              tma_load_2d_hint(st + kF8TileBytes + off, &tm_v, x0, row, fb, policy);
            }
          }
        } else if (bs >= kTile) {
          // One box per tile and tensor: 64 rows x both 64-column halves of
          // KV head j (3-D map [2 h_kv halves][rows][64], half-major landing).
          const int row = bt[t0 >> p.log2_block_size] * bs + (t0 & (bs - 1));
          mbar_arrive_expect_tx(fb, kStageBytes);
          tma_load_3d_hint(st, &tm_k, 0, row, 2 * j, fb, policy);
          tma_load_3d_hint(st + kKvTileBytes, &tm_v, 0, row, 2 * j, fb, policy);
        } else {
          // One box per block and tensor: its bs rows x both halves.
          const int nblk = (nval + bs - 1) >> p.log2_block_size;
          const int box = 2 * bs * 128;
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nblk * 2 * box));
          for (int k = 0; k < nblk; ++k) {
            const int row = bt[(t0 >> p.log2_block_size) + k] * bs;
            const uint32_t off = static_cast<uint32_t>(k * box);
            tma_load_3d_hint(st + off, &tm_k, 0, row, 2 * j, fb, policy);
            tma_load_3d_hint(st + kKvTileBytes + off, &tm_v, 0, row, 2 * j, fb, policy);
          }
        }
        ++issued;
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the
      // last phase of every stage that was filled.
      for (int it = max(0, issued - kStages); it < issued; ++it)
        if (!mbar_wait(full0 + 8 * (it % kStages), (it / kStages) & 1, p.err_flag)) break;
    }
    return;
  }

  // ---------------- consumers
  const int cw = warp - 1;
  Consumer c;
  c.init(p, b, j, cw, lane);
  // An 8-bit cache's K scale multiplies every score of KV head j.
  const float scale_log2 =
      Consumer::kCacheBytes == 1 ? p.scale_log2 * p.k_scale[j] : p.scale_log2;
  bool ok = true;
  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % kStages;
    if (!mbar_wait(full0 + 8 * s, (it / kStages) & 1, p.err_flag)) {
      ok = false;
      break;
    }
    const int t0 = t_begin + it * kTile;
    const int nval = min(kTile, t_end - t0);
    c.tile(smem + s * kStage, max(0, w0 - t0), nval, scale_log2);
    fence_proxy_async_smem();  // order any generic smem writes before the next TMA fill
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }

  // Merge the consumer warps' (m, l, o) through shared memory (the ring is
  // free once every warp has passed the last tile).
  __syncwarp();
  if (lane == 0) mbar_arrive(done_bar);
  if (!ok || !mbar_wait(done_bar, 0, p.err_flag)) return;
  float* mo = reinterpret_cast<float*>(smem);
  float* mm = mo + kW * Consumer::kRowsPerWarp * kHeadDim;
  float* ml = mm + kW * Consumer::kRowsPerWarp;
  c.finish(mo, mm, ml, lane);
  __syncwarp();
  if (lane == 0) mbar_arrive(merge_bar);
  if (!mbar_wait(merge_bar, 0, p.err_flag)) return;

  const int tid = threadIdx.x - 32;
  for (int e = tid; e < G * kHeadDim; e += kW * 32) {
    const int r = e / kHeadDim, d = e % kHeadDim;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kW; ++w)
      if (Consumer::covers(w, r)) M = fmaxf(M, mm[Consumer::slot(w, r)]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      if (!Consumer::covers(w, r)) continue;
      const int sl = Consumer::slot(w, r);
      const float mw = mm[sl];
      if (mw == kNegInf) continue;
      const float f = ex2(mw - M);
      L = fmaf(ml[sl], f, L);
      O = fmaf(mo[sl * kHeadDim + d], f, O);
    }
    const float res = L > 0.f ? O / L : 0.f;
    if (p.n_split == 1) {
      static_cast<uint16_t*>(p.out)[(row0 + r) * kHeadDim + d] = round1<kBF16>(res);
    } else {
      p.part_o[((row0 + r) * p.n_split + split) * kHeadDim + d] = res;
      if (d == 0) p.part_lse[(row0 + r) * p.n_split + split] = L > 0.f ? M + lg2(L) : kNegInf;
    }
  }
}

template <class Consumer, bool kBF16, int kStages>
cudaError_t launch_one(const GqaParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream, unsigned max_cluster) {
  auto kern = gqa_partial_kernel<Consumer, kBF16, kStages>;
  constexpr int smem = smem_bytes<Consumer, kStages>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_split, p.h_kv, p.batch);
  // The CTAs of one (split, sequence) read the same cache blocks, each its
  // KV head's rows of every token (256 B, or 128 B of e4m3 codes); launched
  // as clusters of up to max_cluster KV heads they run at the same time on
  // one GPC, so those reads meet in DRAM.  No cluster feature is used.
  // Measured on GB300 (A/B in one process): 16-bit, clusters of 4: long
  // context B = 4 with 8 splits 313.5 against 317.8 us, B = 1 with 32
  // splits 86.9 against 88.2, the 70B layer and the Llama-3.1-8B layers
  // unchanged; e4m3 70B layer, clusters of 2: 162.6 against 171.9 us and
  // 164.6 against 168.4 on two GPUs (B = 16: 48.1-48.3 against 51.1-51.4).
  unsigned cluster = max_cluster;
  while (cluster > 1 && p.h_kv % cluster != 0) cluster >>= 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(32 * (1 + Consumer::kWarps));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = cluster;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}


template <bool kBF16>
cudaError_t dispatch(const GqaParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t stream) {
  constexpr int S = 3;
  // MHA (one query head per KV head) stays on CUDA cores.  From two query
  // heads per KV head up, the padded 16-row mma tile is faster (measured on
  // the Llama-3.1-8B-shaped GQA layer, 4 heads per KV head: 3.6 TB/s on
  // tensor cores against 2.2 TB/s for the warp-shuffle CUDA-core consumer,
  // which is issue- and latency-bound there).
  if (p.group == 1) return launch_one<CcConsumer<1, kBF16>, kBF16, S>(p, tk, tv, stream, 4);
  if (p.group <= kWideGroup)
    return launch_one<MmaConsumer<1, kBF16>, kBF16, S>(p, tk, tv, stream, 4);
  return launch_gqa_wide_partial(p, tk, tv, kBF16, stream);
}

template <bool kBF16>
cudaError_t dispatch_fp8(const GqaParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                         cudaStream_t stream) {
  constexpr int S = 4;  // 16 KB stages: keep as many cache bytes in flight as the 16-bit ring
  if (p.group == 1) return launch_one<CcConsumerF8<1, kBF16>, kBF16, S>(p, tk, tv, stream, 2);
  // Four CTAs per SM of the transposed consumer: three 16 KB stages each.
  if (p.group <= 8)
    return launch_one<MmaConsumerF8T<1, kBF16>, kBF16, 3>(p, tk, tv, stream, 2);
  if (p.group <= kWideGroup)
    return launch_one<MmaConsumerF8T<2, kBF16>, kBF16, S>(p, tk, tv, stream, 2);
  return launch_gqa_wide_partial_fp8(p, tk, tv, kBF16, stream);
}

}  // namespace

cudaError_t launch_gqa_partial_fp8(const GqaParams& p, const CUtensorMap& tm_k,
                                   const CUtensorMap& tm_v, bool bf16, cudaStream_t stream) {
  return bf16 ? dispatch_fp8<true>(p, tm_k, tm_v, stream)
              : dispatch_fp8<false>(p, tm_k, tm_v, stream);
}

cudaError_t launch_gqa_partial(const GqaParams& p, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, bool bf16, int /*num_sms*/,
                               cudaStream_t stream) {
  return bf16 ? dispatch<true>(p, tm_k, tm_v, stream) : dispatch<false>(p, tm_k, tm_v, stream);
}

}  // namespace decattn
