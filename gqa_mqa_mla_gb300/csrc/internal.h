// internal.h -- parameter blocks and launcher entry points shared between the
// C-ABI front end (api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "decattn.h"

namespace decattn {

constexpr int kHeadDim = 128;      // GQA head dimension supported
constexpr int kTile = 64;          // tokens per pipeline stage
constexpr int kMlaHeads = 128;     // MLA query heads
constexpr int kMlaDc = 512;        // MLA latent width
constexpr int kMlaDr = 64;         // MLA decoupled-RoPE width
constexpr int kMlaWidth = kMlaDc + kMlaDr;

// Marker written into a partial log-sum-exp when the rows it covers met bad
// data (bad block id or seq_len): the combine then writes zeros.
#define DECATTN_POISON_LSE (__builtin_huge_valf())  // +inf

struct GqaParams {
  const void* q;              // [B, h_q, 128]
  const int32_t* block_table; // [B, max_blocks_per_seq]
  const int32_t* seq_lens;    // [B]
  void* out;                  // [B, h_q, 128]      (written when n_split == 1)
  float* part_o;              // [B, h_q, n_split, 128]
  float* part_lse;            // [B, h_q, n_split]  log2 domain
  int* err_flag;
  int batch, h_q, h_kv, group;
  int block_size, log2_block_size, num_blocks, max_blocks_per_seq, max_seq_len;
  int n_split, tokens_per_split;  // tokens_per_split is a multiple of kTile
  float scale_log2;               // scale * log2(e)
  int window;                     // > 0: attend only to the last `window` tokens
  const float* k_scale;           // [h_kv], 8-bit caches only: K value = e4m3 * k_scale[j]
  const float* v_scale;           // [h_kv], 8-bit caches only
};

// MLA workspace (n_pairs > 1): a header of kHdrPref ints (slice width in
// cost units, total tiles), the first-tile index of every sequence (batch + 1
// ints), the first tile of every pair's slice (n_pairs + 1 ints), the cost
// position of every sequence's first tile (batch ints), then the partial
// log2-sum-exps and outputs of 2 n_pairs slots.
constexpr int kHdrPref = 64;

struct MlaParams {
  const void* q_abs;          // [B, 128, 512]
  const void* q_rope;         // [B, 128, 64]
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;                  // [B, 128, 512]
  float* part_o;              // [slots, 128, 512]
  float* part_lse;            // [slots, 128]  log2 domain
  int* ws_hdr;                // header + first-tile table (null when n_pairs == 1)
  int* err_flag;
  int batch;
  int block_size, log2_block_size, num_blocks, max_blocks_per_seq, max_seq_len;
  int n_pairs;                // CTA pairs sharing the batch's tiles
  float scale_log2;
};

struct MlaCombineParams {
  const float* part_o;
  const float* part_lse;
  const int* ws_hdr;
  void* out;
  int batch, n_pairs;
};

// Decode-step cache write: one new row per sequence.
struct AppendParams {
  const void* k_new;          // [B, row_elems] 16-bit (the MLA latent row for mla)
  const void* v_new;          // [B, row_elems] 16-bit, or null (MLA: one cache)
  const int32_t* positions;   // [B] slot index of the new token; < 0 skips
  const int32_t* block_table; // [B, max_blocks_per_seq]
  void* k_cache;              // [num_blocks, block_size, row_elems]
  void* v_cache;
  const float* k_scale;       // [row_elems / head_elems], 8-bit caches only
  const float* v_scale;
  int* err_flag;
  int batch, row_elems, head_elems;
  int block_size, log2_block_size, num_blocks, max_blocks_per_seq;
};

// Per-head batched GEMM Y[b, i, :] = X[b, i, :] W_i^T (MLA absorption).
struct HeadGemmParams {
  void* out;        // [batch, heads, m] 16-bit
  int* err_flag;
  int batch, heads;
  int m, k;         // W_i is [m x k]; m a multiple of 128, k of 64
  int n_tile;       // batch rows per CTA: a multiple of 16, <= 256
  int stages;       // K-chunk ring depth
  int tmem_cols;    // power of two >= max(32, n_tile)
};

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  void* out;
  int rows;      // B * heads
  int n_split;
};

// Kernel launchers (return cudaGetLastError() after the launch).
cudaError_t launch_gqa_partial(const GqaParams& p, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, bool bf16, int num_sms,
                               cudaStream_t stream);
// The same over an e4m3 KV cache (tm_k / tm_v: 8-bit maps, boxes of 128 B x
// min(block_size, 64) rows); q / out in fp16 or bf16.
cudaError_t launch_gqa_partial_fp8(const GqaParams& p, const CUtensorMap& tm_k,
                                   const CUtensorMap& tm_v, bool bf16, cudaStream_t stream);
// Query heads per KV head above which the GQA partials run on the tcgen05
// kernel (gqa_wide.cu); up to it, on the CUDA-core / mma.sync consumers of
// gqa_decode.cu, whose 16-bit tensor maps differ (see api.cu).
constexpr int kWideGroup = 16;

// The tcgen05 partial kernel for wide groups (up to 64 query heads per KV
// head) over a 16-bit cache; the same maps and outputs as launch_gqa_partial.
cudaError_t launch_gqa_wide_partial(const GqaParams& p, const CUtensorMap& tm_k,
                                    const CUtensorMap& tm_v, bool bf16, cudaStream_t stream);
// The same over an e4m3 cache (the 8-bit maps of launch_gqa_partial_fp8).
cudaError_t launch_gqa_wide_partial_fp8(const GqaParams& p, const CUtensorMap& tm_k,
                                        const CUtensorMap& tm_v, bool bf16, cudaStream_t stream);
// tm_out: 16-bit [B * 128, 512] output, boxes of 64 x 128; tm_po: fp32
// [2 n_pairs * 128, 512] partials, boxes of 32 x 128 (both 128-byte swizzle).
// tm_c4: the latent cache viewed as [9 chunks][rows][64] (chunk stride 128 B,
// row stride 1152 B), boxes of 64 x 64 rows x 4 chunks: one copy brings four
// 64-column chunks of a 64-token tile, chunk-major; used when block_size is 64.
cudaError_t launch_mla_partial(const MlaParams& p, const CUtensorMap& tm_qa,
                               const CUtensorMap& tm_c, const CUtensorMap& tm_c4,
                               const CUtensorMap& tm_out, const CUtensorMap& tm_po, bool bf16,
                               cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, int d, bool bf16, cudaStream_t stream);
// tm_w: 2-D [heads * m, k] 16-bit, boxes of 64 x 128; tm_x: 3-D [batch, heads,
// k] (x = k innermost), boxes of 64 x 1 x n_tile; both 128-byte swizzle.
// tm_y: 3-D [batch, heads, m], boxes of 64 x 1 x n_tile, no swizzle.
cudaError_t launch_head_gemm(const HeadGemmParams& p, const CUtensorMap& tm_w,
                             const CUtensorMap& tm_x, const CUtensorMap& tm_y, bool bf16,
                             cudaStream_t stream);
int head_gemm_smem_bytes(const HeadGemmParams& p);
// e4m3: quantise with k_scale / v_scale (bf16 or fp16 input); else a copy.
cudaError_t launch_append(const AppendParams& p, bool e4m3, bool bf16, cudaStream_t stream);
cudaError_t launch_mla_combine(const MlaCombineParams& p, bool bf16, cudaStream_t stream);

// Bounded-wait self test (csrc/selftest.cu).
cudaError_t launch_wait_selftest(int* err_flag, int* result, uint64_t limit_ns,
                                 cudaStream_t stream);

// Token chunk per split: a multiple of kTile covering max_seq_len in at most
// n_split chunks.  Returns the number of chunks actually used.
int resolve_splits(int max_seq_len, int n_split, int* tokens_per_split);
// The longest token range a sliding window of `window` tokens streams
// (max_seq_len when window <= 0).
int window_span(int max_seq_len, int window, int block_size);
// gqa_decode's host-side argument checks, in its order (no CUDA call):
// DECATTN_OK, or the status the call would return.
int gqa_check_args(const void* q, const void* k_cache, const void* v_cache,
                   const float* k_scale, const float* v_scale, bool fp8,
                   const int32_t* block_table, const int32_t* seq_lens, const void* out, int h_q,
                   int h_kv, int d_head, float scale, int window, const decattn_launch* L);

// Planner shared by the front end and the workspace query.
int plan_gqa_splits(int batch, int h_q, int h_kv, int max_seq_len, int num_sms);
int plan_gqa_fp8_splits(int batch, int h_q, int h_kv, int max_seq_len, int num_sms);
int plan_mla_splits(int batch, int max_seq_len, int num_sms);
size_t mla_workspace_bytes(int batch, int n_pairs, size_t* off_lse, size_t* off_o);

}  // namespace decattn
