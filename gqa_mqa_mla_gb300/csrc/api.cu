// api.cu -- the C ABI of libdecattn: argument checks, split planning,
// workspace carving, TMA descriptor construction and kernel dispatch.
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "decattn.h"
#include "internal.h"

namespace decattn {
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D tensor map over a row-major [outer, inner] tensor of element type dt
// whose rows are row_bytes apart; boxes of box_inner x box_outer elements,
// 128-byte swizzle.
bool make_map_2d_t(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same over a 16-bit (fp16 / bf16) tensor.
bool make_map_2d(CUtensorMap* m, const void* base, bool bf16, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_map_2d_t(m, base,
                       bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                       inner, outer, row_bytes, box_inner, box_outer);
}

// 3-D tensor map over a row-major [n2, n1, n0] 16-bit tensor (n0 innermost),
// boxes of b0 x b1 x b2 elements, 128-byte swizzle.
bool make_map_3d(CUtensorMap* m, const void* base, bool bf16, uint64_t n0, uint64_t n1,
                 uint64_t n2, uint32_t b0, uint32_t b1, uint32_t b2,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {n0, n1, n2};
  cuuint64_t strides[2] = {n0 * 2, n0 * n1 * 2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D tensor map with explicit byte strides for dimensions 1 and 2 (they
// need not increase), boxes of b0 x b1 x b2 elements, 128-byte swizzle.
bool make_map_3d_strided(CUtensorMap* m, const void* base, bool bf16, uint64_t n0, uint64_t n1,
                         uint64_t n2, uint64_t stride1, uint64_t stride2, uint32_t b0,
                         uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {n0, n1, n2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = n;
  return n;
}

}  // namespace

// Token chunk per split: a multiple of kTile covering max_seq_len in at most
// n_split chunks.  Returns the number of chunks actually used.
int resolve_splits(int max_seq_len, int n_split, int* tokens_per_split) {
  const int tiles = max_seq_len > 0 ? (max_seq_len + kTile - 1) / kTile : 1;
  if (n_split < 1) n_split = 1;
  if (n_split > tiles) n_split = tiles;
  const int tiles_per = (tiles + n_split - 1) / n_split;
  *tokens_per_split = tiles_per * kTile;
  return (tiles + tiles_per - 1) / tiles_per;
}

// A sliding window of W tokens starts at a block (or 64-token) boundary at
// most min(block_size, 64) - 1 tokens before the window: the longest token
// range any sequence streams.
int window_span(int max_seq_len, int window, int block_size) {
  if (window <= 0) return max_seq_len;
  const int64_t span = static_cast<int64_t>(window) + (block_size < kTile ? block_size : kTile) - 1;
  return span < max_seq_len ? static_cast<int>(span) : max_seq_len;
}

namespace {

// Split count for `units` independent (sequence[, KV head]) work units on
// `slots` resident CTAs, for the latency-bound 8-bit-cache consumers of
// wide groups, which gain from more CTAs in flight: one split per unit once
// there are 1.5 waves of CTAs; otherwise split each sequence until about two
// waves exist, keeping at least two 64-token tiles per split (measured on the
// 70B-shaped layer with the 16-row padded consumer: 2 splits 211 us, 1 split
// 233 us).
int plan_splits(int units, int max_seq_len, int slots) {
  const int tiles = max_seq_len > 0 ? (max_seq_len + kTile - 1) / kTile : 1;
  if (units < 1) units = 1;
  if (slots < 1) slots = 1;
  if (2 * units >= 3 * slots) return 1;
  int ns = (2 * slots + units - 1) / units;
  int cap = tiles / 2 > 1 ? tiles / 2 : 1;
  if (cap > DECATTN_MAX_SPLITS) cap = DECATTN_MAX_SPLITS;
  if (ns > cap) ns = cap;
  int tps = 0;
  return resolve_splits(max_seq_len, ns, &tps);
}

// Split count for the 16-bit GQA partial kernel: fill at most ~85 % of one
// wave of resident CTAs, with at least 8 tiles (512 tokens) per split.  A
// wave that overflows by a few CTAs costs a second pass over the whole
// per-CTA time, and short splits only add partials.  Measured on GB300
// (2 CTAs per SM, 304 slots): B=1 x 8 KV heads at S=131072, 32 splits
// 92.7 us / 38 splits 96.1 / 40 splits 133.9 / 76 splits 109.1; B=4, 8 splits
// 314 us / 10 splits 456 / 19 splits 325; Llama-3.1-8B MQA (16 units,
// S <= 4096), 8 splits 32 us / 32 splits 59; its GQA-8 (128 units), 2-3
// splits 44-45 us / 5 splits 50.
int plan_splits_one_wave(int units, int max_seq_len, int slots, int min_tiles = 8) {
  const int tiles = max_seq_len > 0 ? (max_seq_len + kTile - 1) / kTile : 1;
  if (units < 1) units = 1;
  if (slots < 1) slots = 1;
  int ns = static_cast<int>((static_cast<int64_t>(slots) * 85) / (100 * static_cast<int64_t>(units)));
  int cap = tiles / min_tiles > 1 ? tiles / min_tiles : 1;
  if (cap > DECATTN_MAX_SPLITS) cap = DECATTN_MAX_SPLITS;
  if (ns > cap) ns = cap;
  if (ns < 1) ns = 1;
  int tps = 0;
  return resolve_splits(max_seq_len, ns, &tps);
}

}  // namespace

int plan_gqa_splits(int batch, int h_q, int h_kv, int max_seq_len, int num_sms) {
  // GQA partial kernels: two resident CTAs per SM, both the mma.sync one
  // (3-stage ring of 32 KB, up to 16 query heads per KV head) and the
  // tcgen05 one for wider groups (2-stage K and V rings, ~100 KB).  The
  // tcgen05 kernel's splits may be as short as 4 tiles: with few units
  // (Llama-3.1-8B MQA at B = 16, 16 units, S <= 4096) 16 splits ran 20.7 us
  // against 22.9 for the 8 that 8-tile splits allow (L2 flushed).
  const int group = h_kv > 0 ? h_q / h_kv : 1;
  return plan_splits_one_wave(batch * h_kv, max_seq_len, num_sms * 2, group > kWideGroup ? 4 : 8);
}

int plan_gqa_fp8_splits(int batch, int h_q, int h_kv, int max_seq_len, int num_sms) {
  // Up to 8 query heads per KV head the 8-bit-cache kernel (transposed
  // consumer, 95 registers, three 16 KB stages) runs four CTAs per SM and,
  // like the 16-bit kernel, wants at most one wave (70B-shaped layer, 512
  // units on 608 slots: 1 split 160 us, 2 splits 171, 4 splits 185; at
  // B=16, 4 splits 48.4 us, 3 splits 50.0, 8 splits 55.6).  Groups of 9..16
  // run two CTAs per SM; from ~0.85 of a wave of units on, their
  // latency-bound consumers prefer about two waves.  Wider groups go to the
  // tensor-core kernel (two CTAs per SM), which, like its 16-bit form, wants
  // one wave.
  const int group = h_kv > 0 ? h_q / h_kv : 1;
  const int per_sm = (group >= 2 && group <= 8) ? 4 : 2;
  const int slots = num_sms * per_sm;
  const int64_t units = static_cast<int64_t>(batch) * h_kv;
  // (The tensor-core kernel's splits may again be 4 tiles long: MQA with 32
  // query heads at B = 16, S = 4096, 16 splits 18.7 us against 20.7 for 8.)
  if (per_sm == 4 || group > 16 || units * 100 < static_cast<int64_t>(slots) * 85)
    return plan_splits_one_wave(batch * h_kv, max_seq_len, slots, group > kWideGroup ? 4 : 8);
  return plan_splits(batch * h_kv, max_seq_len, slots);
}

int plan_mla_splits(int batch, int max_seq_len, int num_sms) {
  // MLA partial kernel: one CTA pair per two SMs, all pairs resident at
  // once, each streaming an equal share of the batch's 64-token tiles.  Use
  // every SM pair, but give each pair at least two tiles of the host's
  // upper bound (batch x tiles of max_seq_len) so that tiny batches do not
  // pay a partial + combine for nothing.
  const long long slots = num_sms / 2 > 0 ? num_sms / 2 : 1;
  const long long tiles =
      static_cast<long long>(batch) * (max_seq_len > 0 ? (max_seq_len + kTile - 1) / kTile : 1);
  long long pairs = tiles / 2;
  if (pairs > slots) pairs = slots;
  if (pairs > DECATTN_MAX_SPLITS) pairs = DECATTN_MAX_SPLITS;
  return pairs < 1 ? 1 : static_cast<int>(pairs);
}

size_t mla_workspace_bytes(int batch, int n_pairs, size_t* off_lse, size_t* off_o) {
  if (batch < 1 || n_pairs < 1 || n_pairs > DECATTN_MAX_SPLITS) return 0;
  if (n_pairs == 1) return 0;
  const size_t slots = 2 * static_cast<size_t>(n_pairs);
  // header, per-sequence first tiles (batch + 1), pair slice starts (n_pairs + 1),
  // per-sequence first cost positions (batch)
  const size_t hdr =
      align_up((static_cast<size_t>(kHdrPref) + 2 * batch + 1 + n_pairs + 1) * sizeof(int));
  const size_t lse = align_up(slots * kMlaHeads * sizeof(float));
  const size_t o = align_up(slots * kMlaHeads * kMlaDc * sizeof(float));
  if (off_lse) *off_lse = hdr;
  if (off_o) *off_o = hdr + lse;
  return hdr + lse + o;
}

}  // namespace decattn

using namespace decattn;

extern "C" {

const char* decattn_status_string(int status) {
  switch (status) {
    case DECATTN_OK: return "ok";
    case DECATTN_ERR_INVALID_ARG: return "invalid argument";
    case DECATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case DECATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case DECATTN_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int decattn_version(void) { return 100; }

int decattn_selftest_wait_timeout(int* err_flag, int* result, int limit_us, void* stream) {
  if (!err_flag || !result || !aligned(err_flag, 4) || !aligned(result, 4) || limit_us < 1 ||
      limit_us > 100000)
    return DECATTN_ERR_INVALID_ARG;
  const cudaError_t e = launch_wait_selftest(err_flag, result, static_cast<uint64_t>(limit_us) * 1000,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DECATTN_OK : DECATTN_ERR_CUDA;
}

int64_t decattn_kv_bytes_per_token(int n_layers, int n_kv, int d_head, int bytes) {
  if (n_layers < 0 || n_kv < 0 || d_head < 0 || bytes < 0) return -1;
  return static_cast<int64_t>(n_layers) * n_kv * d_head * 2 * bytes;
}

int64_t decattn_mla_bytes_per_token(int n_layers, int d_c, int d_rope, int bytes) {
  if (n_layers < 0 || d_c < 0 || d_rope < 0 || bytes < 0) return -1;
  return static_cast<int64_t>(n_layers) * (d_c + d_rope) * bytes;
}

size_t gqa_decode_workspace_size(int batch, int h_q, int d_head, int num_splits) {
  if (batch < 1 || h_q < 1 || d_head < 1 || num_splits < 1 || num_splits > DECATTN_MAX_SPLITS)
    return 0;
  if (num_splits == 1) return 0;
  const size_t rows = static_cast<size_t>(batch) * h_q * num_splits;
  return align_up(rows * d_head * sizeof(float)) + align_up(rows * sizeof(float));
}

size_t mla_decode_workspace_size(int batch, int num_splits) {
  return mla_workspace_bytes(batch, num_splits, nullptr, nullptr);
}

int gqa_decode_plan_splits(int batch, int h_q, int h_kv, int d_head, int max_seq_len,
                           int num_sms) {
  if (batch < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0 || d_head < 1 || max_seq_len < 0)
    return DECATTN_ERR_INVALID_ARG;
  if (num_sms <= 0) num_sms = device_sm_count();
  if (num_sms <= 0) return DECATTN_ERR_CUDA;
  return plan_gqa_splits(batch, h_q, h_kv, max_seq_len, num_sms);
}

int gqa_decode_fp8kv_plan_splits(int batch, int h_q, int h_kv, int d_head, int max_seq_len,
                                 int num_sms) {
  if (batch < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0 || d_head < 1 || max_seq_len < 0)
    return DECATTN_ERR_INVALID_ARG;
  if (num_sms <= 0) num_sms = device_sm_count();
  if (num_sms <= 0) return DECATTN_ERR_CUDA;
  return plan_gqa_fp8_splits(batch, h_q, h_kv, max_seq_len, num_sms);
}

int gqa_decode_window_plan_splits(int batch, int h_q, int h_kv, int d_head, int max_seq_len,
                                  int window, int block_size, int kv_bytes, int num_sms) {
  if (batch < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0 || d_head < 1 || max_seq_len < 0 ||
      window < 1 || !is_pow2(block_size) || (kv_bytes != 1 && kv_bytes != 2))
    return DECATTN_ERR_INVALID_ARG;
  if (num_sms <= 0) num_sms = device_sm_count();
  if (num_sms <= 0) return DECATTN_ERR_CUDA;
  const int span = window_span(max_seq_len, window, block_size);
  return kv_bytes == 1 ? plan_gqa_fp8_splits(batch, h_q, h_kv, span, num_sms)
                       : plan_gqa_splits(batch, h_q, h_kv, span, num_sms);
}

int mla_decode_plan_splits(int batch, int max_seq_len, int num_sms) {
  if (batch < 1 || max_seq_len < 0) return DECATTN_ERR_INVALID_ARG;
  if (num_sms <= 0) num_sms = device_sm_count();
  if (num_sms <= 0) return DECATTN_ERR_CUDA;
  return plan_mla_splits(batch, max_seq_len, num_sms);
}

static int check_launch(const decattn_launch* L, bool mla) {
  if (!L) return DECATTN_ERR_INVALID_ARG;
  if (L->batch < 1 || L->num_blocks < 1 || L->max_blocks_per_seq < 1 || L->max_seq_len < 0)
    return DECATTN_ERR_INVALID_ARG;
  if (L->dtype != DECATTN_FP16 && L->dtype != DECATTN_BF16) return DECATTN_ERR_INVALID_ARG;
  if (L->num_splits < 0 || L->num_splits > DECATTN_MAX_SPLITS) return DECATTN_ERR_INVALID_ARG;
  if (!is_pow2(L->block_size)) return DECATTN_ERR_INVALID_ARG;
  if (L->block_size < 8 || L->block_size > (mla ? 64 : 256)) return DECATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(L->max_seq_len) >
      static_cast<int64_t>(L->max_blocks_per_seq) * L->block_size)
    return DECATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(L->num_blocks) * L->block_size > 0x7fffffffLL)
    return DECATTN_ERR_UNSUPPORTED;
  if (L->workspace && !aligned(L->workspace, 16)) return DECATTN_ERR_INVALID_ARG;
  if (L->err_flag && !aligned(L->err_flag, 4)) return DECATTN_ERR_INVALID_ARG;
  return DECATTN_OK;
}

}  // extern "C"

namespace decattn {

int gqa_check_args(const void* q, const void* k_cache, const void* v_cache,
                   const float* k_scale, const float* v_scale, bool fp8,
                   const int32_t* block_table, const int32_t* seq_lens, const void* out, int h_q,
                   int h_kv, int d_head, float scale, int window, const decattn_launch* L) {
  int st = check_launch(L, false);
  if (st != DECATTN_OK) return st;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out)
    return DECATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return DECATTN_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4)))
    return DECATTN_ERR_INVALID_ARG;
  if (h_q < 1 || h_kv < 1 || h_q % h_kv != 0) return DECATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return DECATTN_ERR_INVALID_ARG;
  if (d_head != kHeadDim) return DECATTN_ERR_UNSUPPORTED;
  if (h_q / h_kv > 64) return DECATTN_ERR_UNSUPPORTED;
  if (window < 0) return DECATTN_ERR_INVALID_ARG;
  return DECATTN_OK;
}

}  // namespace decattn

extern "C" {

// gqa_decode and gqa_decode_fp8kv share everything but the cache element type
// (and the 8-bit cache's per-KV-head scales).
static int gqa_decode_impl(const void* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, bool fp8,
                           const int32_t* block_table, const int32_t* seq_lens, void* out,
                           int h_q, int h_kv, int d_head, float scale, int window,
                           const decattn_launch* L) {
  const int st = gqa_check_args(q, k_cache, v_cache, k_scale, v_scale, fp8, block_table,
                                seq_lens, out, h_q, h_kv, d_head, scale, window, L);
  if (st != DECATTN_OK) return st;
  const int span = window_span(L->max_seq_len, window, L->block_size);
  int n_split = L->num_splits;
  if (n_split == 0) {
    const int sms = device_sm_count();
    if (sms <= 0) return DECATTN_ERR_CUDA;
    n_split = fp8 ? plan_gqa_fp8_splits(L->batch, h_q, h_kv, span, sms)
                  : plan_gqa_splits(L->batch, h_q, h_kv, span, sms);
  }
  int tps = 0;
  const int eff = resolve_splits(span, n_split, &tps);

  GqaParams p{};
  p.q = q;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.err_flag = L->err_flag;
  p.batch = L->batch;
  p.h_q = h_q;
  p.h_kv = h_kv;
  p.group = h_q / h_kv;
  p.block_size = L->block_size;
  p.log2_block_size = ilog2(L->block_size);
  p.num_blocks = L->num_blocks;
  p.max_blocks_per_seq = L->max_blocks_per_seq;
  p.max_seq_len = L->max_seq_len;
  p.n_split = eff;
  p.tokens_per_split = tps;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.window = window;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  if (eff > 1) {
    const size_t need = gqa_decode_workspace_size(L->batch, h_q, d_head, eff);
    if (!L->workspace || L->workspace_bytes < need) return DECATTN_ERR_WORKSPACE;
    const size_t rows = static_cast<size_t>(L->batch) * h_q * eff;
    p.part_o = static_cast<float*>(L->workspace);
    p.part_lse = reinterpret_cast<float*>(static_cast<char*>(L->workspace) +
                                          align_up(rows * d_head * sizeof(float)));
  }

  const bool bf16 = L->dtype == DECATTN_BF16;
  const uint64_t rows_total = static_cast<uint64_t>(L->num_blocks) * L->block_size;
  const uint32_t box_rows = static_cast<uint32_t>(L->block_size < kTile ? L->block_size : kTile);
  CUtensorMap tk, tv;
  if (fp8) {
    // One byte per element: a token's 128-d head is one 128-byte box row.
    const uint64_t row_bytes = static_cast<uint64_t>(h_kv) * kHeadDim;
    if (!make_map_2d_t(&tk, k_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, row_bytes, rows_total,
                       row_bytes, kHeadDim, box_rows) ||
        !make_map_2d_t(&tv, v_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, row_bytes, rows_total,
                       row_bytes, kHeadDim, box_rows))
      return DECATTN_ERR_CUDA;
  } else if (h_q / h_kv <= kWideGroup) {
    // The CUDA-core / mma.sync consumers: a 3-D view [2 h_kv halves][rows][64]
    // (strides: a token row, then 128 B per 64-column half), so that one box
    // brings box_rows rows of both halves of a KV head (landing half-major).
    const uint64_t row_bytes = static_cast<uint64_t>(h_kv) * kHeadDim * 2;
    if (!make_map_3d_strided(&tk, k_cache, bf16, 64, rows_total, 2 * static_cast<uint64_t>(h_kv),
                             row_bytes, 128, 64, box_rows, 2) ||
        !make_map_3d_strided(&tv, v_cache, bf16, 64, rows_total, 2 * static_cast<uint64_t>(h_kv),
                             row_bytes, 128, 64, box_rows, 2))
      return DECATTN_ERR_CUDA;
  } else {
    // The tcgen05 kernel of wide groups: 2-D boxes of one 64-column half.
    const uint64_t row_bytes = static_cast<uint64_t>(h_kv) * kHeadDim * 2;
    if (!make_map_2d(&tk, k_cache, bf16, static_cast<uint64_t>(h_kv) * kHeadDim, rows_total,
                     row_bytes, 64, box_rows) ||
        !make_map_2d(&tv, v_cache, bf16, static_cast<uint64_t>(h_kv) * kHeadDim, rows_total,
                     row_bytes, 64, box_rows))
      return DECATTN_ERR_CUDA;
  }

  cudaStream_t stream = static_cast<cudaStream_t>(L->stream);
  const cudaError_t e = fp8 ? launch_gqa_partial_fp8(p, tk, tv, bf16, stream)
                            : launch_gqa_partial(p, tk, tv, bf16, 0, stream);
  if (e != cudaSuccess) return DECATTN_ERR_CUDA;
  if (eff > 1) {
    CombineParams c{p.part_o, p.part_lse, out, L->batch * h_q, eff};
    if (launch_combine(c, kHeadDim, bf16, stream) != cudaSuccess) return DECATTN_ERR_CUDA;
  }
  return DECATTN_OK;
}

int gqa_decode(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_table, const int32_t* seq_lens, void* out, int h_q, int h_kv,
               int d_head, float scale, const decattn_launch* L) {
  return gqa_decode_impl(q, k_cache, v_cache, nullptr, nullptr, false, block_table, seq_lens, out,
                         h_q, h_kv, d_head, scale, 0, L);
}

int gqa_decode_fp8kv(const void* q, const void* k_cache, const void* v_cache,
                     const float* k_scale, const float* v_scale, const int32_t* block_table,
                     const int32_t* seq_lens, void* out, int h_q, int h_kv, int d_head,
                     float scale, const decattn_launch* L) {
  return gqa_decode_impl(q, k_cache, v_cache, k_scale, v_scale, true, block_table, seq_lens, out,
                         h_q, h_kv, d_head, scale, 0, L);
}

int gqa_decode_window(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* seq_lens, void* out, int h_q,
                      int h_kv, int d_head, float scale, int window, const decattn_launch* L) {
  if (window < 1) return DECATTN_ERR_INVALID_ARG;
  return gqa_decode_impl(q, k_cache, v_cache, nullptr, nullptr, false, block_table, seq_lens, out,
                         h_q, h_kv, d_head, scale, window, L);
}

int gqa_decode_fp8kv_window(const void* q, const void* k_cache, const void* v_cache,
                            const float* k_scale, const float* v_scale,
                            const int32_t* block_table, const int32_t* seq_lens, void* out,
                            int h_q, int h_kv, int d_head, float scale, int window,
                            const decattn_launch* L) {
  if (window < 1) return DECATTN_ERR_INVALID_ARG;
  return gqa_decode_impl(q, k_cache, v_cache, k_scale, v_scale, true, block_table, seq_lens, out,
                         h_q, h_kv, d_head, scale, window, L);
}

int mla_decode(const void* q_absorbed, const void* q_rope, const void* latent_cache,
               const int32_t* block_table, const int32_t* seq_lens, void* out, float scale,
               const decattn_launch* L) {
  int st = check_launch(L, true);
  if (st != DECATTN_OK) return st;
  if (!q_absorbed || !q_rope || !latent_cache || !block_table || !seq_lens || !out)
    return DECATTN_ERR_INVALID_ARG;
  if (!aligned(q_absorbed, 16) || !aligned(q_rope, 16) || !aligned(latent_cache, 16) ||
      !aligned(out, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return DECATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return DECATTN_ERR_INVALID_ARG;

  int n_pairs = L->num_splits;
  if (n_pairs == 0) {
    const int sms = device_sm_count();
    if (sms <= 0) return DECATTN_ERR_CUDA;
    n_pairs = plan_mla_splits(L->batch, L->max_seq_len, sms);
  }

  MlaParams p{};
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.err_flag = L->err_flag;
  p.batch = L->batch;
  p.block_size = L->block_size;
  p.log2_block_size = ilog2(L->block_size);
  p.num_blocks = L->num_blocks;
  p.max_blocks_per_seq = L->max_blocks_per_seq;
  p.max_seq_len = L->max_seq_len;
  p.n_pairs = n_pairs;
  p.scale_log2 = scale * 1.4426950408889634f;
  if (n_pairs > 1) {
    size_t off_lse = 0, off_o = 0;
    const size_t need = mla_workspace_bytes(L->batch, n_pairs, &off_lse, &off_o);
    if (!L->workspace || L->workspace_bytes < need) return DECATTN_ERR_WORKSPACE;
    char* ws = static_cast<char*>(L->workspace);
    p.ws_hdr = reinterpret_cast<int*>(ws);
    p.part_lse = reinterpret_cast<float*>(ws + off_lse);
    p.part_o = reinterpret_cast<float*>(ws + off_o);
  }

  const bool bf16 = L->dtype == DECATTN_BF16;
  const uint64_t c_rows = static_cast<uint64_t>(L->num_blocks) * L->block_size;
  const uint64_t q_rows = static_cast<uint64_t>(L->batch) * kMlaHeads;
  CUtensorMap tqa, tc, tc4, tout, tpo;
  if (!make_map_2d(&tqa, q_absorbed, bf16, kMlaDc, q_rows, kMlaDc * 2, 64, kMlaHeads) ||
      !make_map_2d(&tc, latent_cache, bf16, kMlaWidth, c_rows, kMlaWidth * 2, 64,
                   static_cast<uint32_t>(L->block_size < 64 ? L->block_size : 64)) ||
      !make_map_2d(&tout, out, bf16, kMlaDc, q_rows, kMlaDc * 2, 64, kMlaHeads))
    return DECATTN_ERR_CUDA;
  // check_launch caps MLA blocks at 64 rows, so block size 64 is exactly the
  // case in which the kernel takes one 64-row box per tile and copies four
  // chunks at once through tc4.
  if (L->block_size >= 64) {
    if (!make_map_3d_strided(&tc4, latent_cache, bf16, 64, c_rows, kMlaWidth / 64, kMlaWidth * 2,
                             128, 64, 64, 4))
      return DECATTN_ERR_CUDA;
  } else {
    tc4 = tc;  // never used: smaller blocks take one 2-D copy per chunk and block
  }
  if (n_pairs > 1) {
    if (!make_map_2d_t(&tpo, p.part_o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kMlaDc,
                       2ull * n_pairs * kMlaHeads, kMlaDc * 4, 32, kMlaHeads))
      return DECATTN_ERR_CUDA;
  } else {
    tpo = tout;  // never used: every segment of a single pair is whole
  }
  p.q_abs = q_absorbed;
  p.q_rope = q_rope;

  cudaStream_t stream = static_cast<cudaStream_t>(L->stream);
  cudaError_t e = launch_mla_partial(p, tqa, tc, tc4, tout, tpo, bf16, stream);
  if (e == cudaErrorNotSupported) return DECATTN_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return DECATTN_ERR_CUDA;
  if (n_pairs > 1) {
    MlaCombineParams c{p.part_o, p.part_lse, p.ws_hdr, out, L->batch, n_pairs};
    if (launch_mla_combine(c, bf16, stream) != cudaSuccess) return DECATTN_ERR_CUDA;
  }
  return DECATTN_OK;
}

// The decode step's cache write (gqa_kv_append, gqa_kv_append_fp8kv,
// mla_kv_append): host checks, then one launch for K and V.
static int kv_append_impl(const void* k_new, const void* v_new, const float* k_scale,
                          const float* v_scale, bool e4m3, const int32_t* positions,
                          const int32_t* block_table, void* k_cache, void* v_cache, int row_elems,
                          int head_elems, bool mla, const decattn_launch* L) {
  if (!L) return DECATTN_ERR_INVALID_ARG;
  if (L->batch < 1 || L->num_blocks < 1 || L->max_blocks_per_seq < 1)
    return DECATTN_ERR_INVALID_ARG;
  if (L->dtype != DECATTN_FP16 && L->dtype != DECATTN_BF16) return DECATTN_ERR_INVALID_ARG;
  if (!is_pow2(L->block_size)) return DECATTN_ERR_INVALID_ARG;
  if (L->block_size < 8 || L->block_size > (mla ? 64 : 256)) return DECATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(L->num_blocks) * L->block_size > 0x7fffffffLL)
    return DECATTN_ERR_UNSUPPORTED;
  if (!k_new || !k_cache || !positions || !block_table) return DECATTN_ERR_INVALID_ARG;
  if (!mla && (!v_new || !v_cache)) return DECATTN_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(k_cache, 16) || !aligned(positions, 4) ||
      !aligned(block_table, 4) || (v_new && !aligned(v_new, 16)) ||
      (v_cache && !aligned(v_cache, 16)))
    return DECATTN_ERR_INVALID_ARG;
  if (e4m3 && (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4)))
    return DECATTN_ERR_INVALID_ARG;
  if (L->err_flag && !aligned(L->err_flag, 4)) return DECATTN_ERR_INVALID_ARG;

  AppendParams p{};
  p.k_new = k_new;
  p.v_new = mla ? nullptr : v_new;
  p.positions = positions;
  p.block_table = block_table;
  p.k_cache = k_cache;
  p.v_cache = mla ? nullptr : v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err_flag = L->err_flag;
  p.batch = L->batch;
  p.row_elems = row_elems;
  p.head_elems = head_elems;
  p.block_size = L->block_size;
  p.log2_block_size = ilog2(L->block_size);
  p.num_blocks = L->num_blocks;
  p.max_blocks_per_seq = L->max_blocks_per_seq;
  const cudaError_t e = launch_append(p, e4m3, L->dtype == DECATTN_BF16,
                                      static_cast<cudaStream_t>(L->stream));
  return e == cudaSuccess ? DECATTN_OK : DECATTN_ERR_CUDA;
}

int gqa_kv_append(const void* k_new, const void* v_new, const int32_t* positions,
                  const int32_t* block_table, void* k_cache, void* v_cache, int h_kv, int d_head,
                  const decattn_launch* L) {
  if (h_kv < 1 || h_kv > 1024) return DECATTN_ERR_INVALID_ARG;
  if (d_head != kHeadDim) return DECATTN_ERR_UNSUPPORTED;
  return kv_append_impl(k_new, v_new, nullptr, nullptr, false, positions, block_table, k_cache,
                        v_cache, h_kv * kHeadDim, kHeadDim, false, L);
}

int gqa_kv_append_fp8kv(const void* k_new, const void* v_new, const float* k_scale,
                        const float* v_scale, const int32_t* positions,
                        const int32_t* block_table, void* k_cache, void* v_cache, int h_kv,
                        int d_head, const decattn_launch* L) {
  if (h_kv < 1 || h_kv > 1024) return DECATTN_ERR_INVALID_ARG;
  if (d_head != kHeadDim) return DECATTN_ERR_UNSUPPORTED;
  return kv_append_impl(k_new, v_new, k_scale, v_scale, true, positions, block_table, k_cache,
                        v_cache, h_kv * kHeadDim, kHeadDim, false, L);
}

int mla_kv_append(const void* latent_new, const int32_t* positions, const int32_t* block_table,
                  void* latent_cache, const decattn_launch* L) {
  return kv_append_impl(latent_new, nullptr, nullptr, nullptr, false, positions, block_table,
                        latent_cache, nullptr, kMlaWidth, kMlaWidth, true, L);
}

// MLA's absorption GEMMs: Y[b, i, :] = X[b, i, :] W_i^T for every head i.
static int head_gemm_impl(const void* x, const void* w, void* y, int batch, int heads, int m,
                          int k, int dtype, int* err_flag, void* stream) {
  if (!x || !w || !y) return DECATTN_ERR_INVALID_ARG;
  if (batch < 1 || heads < 1 || m < 1 || k < 1) return DECATTN_ERR_INVALID_ARG;
  if (dtype != DECATTN_FP16 && dtype != DECATTN_BF16) return DECATTN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16)) return DECATTN_ERR_INVALID_ARG;
  if (err_flag && !aligned(err_flag, 4)) return DECATTN_ERR_INVALID_ARG;
  if (m % 128 != 0 || k % 64 != 0 || heads > 65535) return DECATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(heads) * m > 0x7fffffffLL ||
      static_cast<int64_t>(batch) * heads * m > (1LL << 40))
    return DECATTN_ERR_UNSUPPORTED;
  HeadGemmParams p{};
  p.out = y;
  p.err_flag = err_flag;
  p.batch = batch;
  p.heads = heads;
  p.m = m;
  p.k = k;
  const int b16 = (batch + 15) / 16 * 16;
  p.n_tile = b16 < 256 ? b16 : 256;
  if ((batch + p.n_tile - 1) / p.n_tile > 65535) return DECATTN_ERR_UNSUPPORTED;
  // Ring stages: up to 8, within ~100 KB of shared memory, so that two CTAs
  // fit an SM and a call launched right after this one (a programmatic
  // dependent) can start streaming its weights while this one finishes
  // (DeepSeek-V2 out GEMM, B = 32, 8 layers' weights in turn: 6.99 us with
  // 8 stages and one CTA per SM).
  const int stage_bytes = 128 * 128 + p.n_tile * 128;
  int stages = (100 * 1024) / stage_bytes;
  stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  p.stages = k / 64 < stages ? k / 64 : stages;
  p.tmem_cols = 32;
  while (p.tmem_cols < p.n_tile) p.tmem_cols *= 2;
  const bool bf16 = dtype == DECATTN_BF16;
  CUtensorMap tw, tx, ty;
  if (!make_map_2d(&tw, w, bf16, static_cast<uint64_t>(k), static_cast<uint64_t>(heads) * m,
                   static_cast<uint64_t>(k) * 2, 64, 128) ||
      !make_map_3d(&tx, x, bf16, static_cast<uint64_t>(k), static_cast<uint64_t>(heads),
                   static_cast<uint64_t>(batch), 64, 1, static_cast<uint32_t>(p.n_tile)) ||
      !make_map_3d(&ty, y, bf16, static_cast<uint64_t>(m), static_cast<uint64_t>(heads),
                   static_cast<uint64_t>(batch), 64, 1, static_cast<uint32_t>(p.n_tile),
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return DECATTN_ERR_CUDA;
  const cudaError_t e = launch_head_gemm(p, tw, tx, ty, bf16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DECATTN_OK : DECATTN_ERR_CUDA;
}

int mla_absorb_q(const void* q_nope, const void* w_uk, void* q_abs, int batch, int n_heads,
                 int d_h, int d_c, int dtype, int* err_flag, void* stream) {
  return head_gemm_impl(q_nope, w_uk, q_abs, batch, n_heads, d_c, d_h, dtype, err_flag, stream);
}

int mla_unabsorb_out(const void* o_lat, const void* w_uv_t, void* out, int batch, int n_heads,
                     int d_c, int d_v, int dtype, int* err_flag, void* stream) {
  return head_gemm_impl(o_lat, w_uv_t, out, batch, n_heads, d_v, d_c, dtype, err_flag, stream);
}

}  // extern "C"
