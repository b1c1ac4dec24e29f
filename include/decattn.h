/*
 * decattn.h -- C ABI of libdecattn: single-token decode attention over a
 * paged KV cache on one GB300 (sm_103a) GPU.
 *
 * Two operations:
 *
 *   gqa_decode  MHA / GQA / MQA.  h_q query heads share h_kv K/V heads;
 *               query head i reads KV head i / (h_q / h_kv) by index
 *               arithmetic, never by copying ("MQA, GQA, and MLA",
 *               section 2 "The three answers" and section 8 "Implementation
 *               notes", GQA in the kernel).  MHA is h_kv = h_q, MQA h_kv = 1.
 *
 *   mla_decode  Multi-head latent attention in its absorbed form: the 128
 *               query heads arrive already multiplied by W_uk (q_absorbed,
 *               512-d) plus a 64-d decoupled-RoPE query; each is scored
 *               against the cached 512-d latent and the cached 64-d RoPE
 *               key, and the latent itself serves as the value ("MQA, GQA,
 *               and MLA", section 5 "MLA, mechanically", KEY TRICK; "Why
 *               GQA's KV Cache Savings Don't Fully Reduce TPOT", "What Makes
 *               MLA Different": 512 + 64 = 576 cached elements per token).
 *
 * For each sequence b and query head i the result is
 *     s_t   = scale * (q_i . k_t)                  for t < seq_lens[b]
 *     p     = softmax(s)  (base e)
 *     out_i = sum_t p_t v_t
 * where k_t / v_t come from the paged cache: token t of sequence b lives in
 * physical block block_table[b][t / block_size], slot t % block_size.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller, row-major and
 *   contiguous, 16-byte aligned.  The library allocates nothing on the call
 *   path; the split-KV workspace is caller-provided (see *_workspace_size).
 * - Calls are asynchronous on launch->stream and return once the kernels are
 *   enqueued.
 * - A negative return is an error: host-side argument checks fail before
 *   anything is launched; DECATTN_ERR_CUDA reports a launch failure.
 * - Bad DATA found on the device (a block id outside [0, num_blocks), a
 *   seq_len outside [0, max_seq_len]) never traps: the kernel ORs a
 *   DECATTN_FLAG_* bit into *launch->err_flag (when non-NULL) and writes
 *   zeros to the affected output rows.  The caller reads the flag after
 *   synchronising.
 * - seq_lens[b] = 0 gives an all-zero output row (an empty softmax).
 * - Cache slots past seq_lens[b] inside a sequence's last block may be
 *   fetched with the block but never affect the result: they may hold
 *   anything, NaN included.  Block table entries past a sequence's last
 *   block are never read.
 */
#ifndef DECATTN_H
#define DECATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DECATTN_OK = 0,
  DECATTN_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer, ... */
  DECATTN_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. d_head != 128) */
  DECATTN_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required   */
  DECATTN_ERR_CUDA = -4         /* a CUDA call or kernel launch failed           */
} decattn_status;

typedef enum { DECATTN_FP16 = 0, DECATTN_BF16 = 1 } decattn_dtype;

/* Bits ORed into *err_flag by the kernels. */
#define DECATTN_FLAG_BAD_BLOCK 1   /* a block id outside [0, num_blocks)          */
#define DECATTN_FLAG_BAD_SEQ_LEN 2 /* seq_lens[b] < 0 or > max_seq_len            */
#define DECATTN_FLAG_TIMEOUT 4     /* a pipeline wait gave up (internal error)    */

/* Largest split count accepted (num_splits) and chosen by the planner. */
#define DECATTN_MAX_SPLITS 256

/*
 * Launch description shared by both operations.
 *   batch              number of sequences B (>= 1)
 *   num_blocks         physical blocks in the cache tensors (>= 1)
 *   block_size         tokens per block (GQA: 8..256 power of two;
 *                      MLA: 8, 16, 32 or 64)
 *   max_blocks_per_seq row length of block_table
 *   max_seq_len        host upper bound on seq_lens[] (sizes the split grid;
 *                      must be <= max_blocks_per_seq * block_size)
 *   num_splits         gqa_decode: split-KV chunks per sequence;
 *                      mla_decode: CTA pairs sharing the batch's KV tiles
 *                      (see mla_decode); 0 = automatic
 *   dtype              element type of every 16-bit tensor (decattn_dtype)
 *   workspace          device scratch of workspace_bytes bytes (may be NULL
 *                      when the required size is 0)
 *   err_flag           device int receiving DECATTN_FLAG_* bits, or NULL
 *   stream             cudaStream_t to launch on (NULL = legacy default)
 */
typedef struct {
  int batch;
  int num_blocks;
  int block_size;
  int max_blocks_per_seq;
  int max_seq_len;
  int num_splits;
  int dtype;
  void* workspace;
  size_t workspace_bytes;
  int* err_flag;
  void* stream;
} decattn_launch;

/*
 * gqa_decode -- MHA / GQA / MQA decode attention, one query token per
 * sequence ("MQA, GQA, and MLA", sections 2, 4 and 8).
 *   q            [batch, h_q, d_head]                       fp16/bf16
 *   k_cache      [num_blocks, block_size, h_kv, d_head]     fp16/bf16
 *   v_cache      [num_blocks, block_size, h_kv, d_head]     fp16/bf16
 *   block_table  [batch, max_blocks_per_seq]                int32
 *   seq_lens     [batch]                                    int32
 *   out          [batch, h_q, d_head]                       fp16/bf16 (written)
 *   h_q, h_kv    query / KV heads; h_q % h_kv == 0, h_q / h_kv <= 64
 *   d_head       head dimension (128)
 *   scale        softmax scale (typically 1/sqrt(d_head))
 * Softmax and accumulation run in fp32; out is rounded to nearest-even.
 */
int gqa_decode(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_table, const int32_t* seq_lens, void* out, int h_q, int h_kv,
               int d_head, float scale, const decattn_launch* launch);

/*
 * gqa_decode_noalloc -- gqa_decode for callers that may not allocate device
 * memory.  The pages have no counterpart: this is an interface convenience.
 *
 * Same arguments, results and statuses as gqa_decode, except that
 * launch->workspace / workspace_bytes are ignored: the split-KV scratch is a
 * fixed 8 MiB (8 * 2^20 bytes) device array inside the library, held by every
 * GPU that loads it until the process exits.  Meant for hosts that cannot
 * call cudaMalloc around a decode call (engines that reserve all free HBM for
 * the KV cache, runtime plugin interfaces that hand over only inputs and
 * outputs, loops that must not pay an allocation's synchronisation).
 *   - A split plan needing more than 8 MiB of scratch returns
 *     DECATTN_ERR_WORKSPACE and launches nothing (the need is
 *     gqa_decode_workspace_size(batch, h_q, d_head, splits)).
 *   - All calls on a device share the array: calls that may overlap on the
 *     GPU (unordered streams) race; serialise them.
 *   - The first call on a device looks up the array's address with that
 *     device current; make it before any stream capture.  The address is
 *     kept for the life of the process, so a device reset (cudaDeviceReset
 *     or a primary-context reset) is not supported after that first call.
 *   - The scratch check uses the split count gqa_decode actually runs (a
 *     requested count is cut to the 64-token tiles of max_seq_len), and it
 *     comes after gqa_decode's own argument checks.
 *   - Nothing in the array needs to start at zero; its contents after a call
 *     are unspecified.
 */
int gqa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* seq_lens, void* out, int h_q,
                       int h_kv, int d_head, float scale, const decattn_launch* launch);

/*
 * gqa_decode_fp8kv -- gqa_decode over an 8-bit KV cache ("Why GQA's KV Cache
 * Savings Don't Fully Reduce TPOT", "When the Serving Engineer Doesn't Get to
 * Choose the Model Architecture": an fp8 cache halves GQA's bytes per token,
 * quantised at KV-head granularity; "07 · MHA/MQA/GQA/MLA quick learn", the
 * question on changing the KV head count by a flag).
 *   k_cache, v_cache  [num_blocks, block_size, h_kv, d_head] e4m3 codes, one
 *                     byte each (1 sign, 4 exponent bits with bias 7, 3
 *                     fraction bits; finite-only, largest magnitude 448)
 *   k_scale, v_scale  [h_kv] fp32 device arrays: the cached value of KV head
 *                     j is e4m3(code) * k_scale[j] (resp. v_scale[j])
 *   q, out            [batch, h_q, d_head] in launch->dtype (fp16 / bf16)
 * Every other argument, status and layout rule as gqa_decode (workspace
 * sized by gqa_decode_workspace_size).  Scores and P.V run on tensor cores
 * with fp32 accumulation; K's scale multiplies the scores, V's the output.
 * Up to 16 query heads per KV head both take fp16 operands (the codes
 * convert exactly; q is rounded to fp16).  From 17 on, the scores take the
 * e4m3 codes as they are against q written as a sum of e4m3 terms (two for
 * bf16, three for fp16, each row scaled by a power of two; exact except for
 * parts below 2^-18 of the row's largest element), and P.V takes fp16
 * operands.
 */
int gqa_decode_fp8kv(const void* q, const void* k_cache, const void* v_cache,
                     const float* k_scale, const float* v_scale, const int32_t* block_table,
                     const int32_t* seq_lens, void* out, int h_q, int h_kv, int d_head,
                     float scale, const decattn_launch* launch);

/*
 * gqa_decode_window, gqa_decode_fp8kv_window -- the same decode restricted to
 * a sliding window: each sequence's query attends only to its last `window`
 * tokens ("07 · MHA/MQA/GQA/MLA quick learn", the question on what sliding-
 * window attention does differently).  For a sequence of length L the
 * attended tokens are positions [max(0, L - window), L), the newest (the
 * query's own, already in the cache) included; window >= L is full attention.
 *   window       >= 1 (else DECATTN_ERR_INVALID_ARG)
 * Every other argument, layout, status and the workspace rule as gqa_decode
 * (resp. gqa_decode_fp8kv).  Cache blocks wholly before the window are never
 * read and their block_table entries are neither read nor checked, so an
 * engine may have recycled them; the block holding the window's first token
 * is read whole, but its tokens before the window are not used (their values
 * may be anything).  Work and the planner's split count scale with
 * min(max_seq_len, window + min(block_size, 64) - 1), not max_seq_len.
 */
int gqa_decode_window(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* seq_lens, void* out, int h_q,
                      int h_kv, int d_head, float scale, int window,
                      const decattn_launch* launch);
int gqa_decode_fp8kv_window(const void* q, const void* k_cache, const void* v_cache,
                            const float* k_scale, const float* v_scale,
                            const int32_t* block_table, const int32_t* seq_lens, void* out,
                            int h_q, int h_kv, int d_head, float scale, int window,
                            const decattn_launch* launch);

/*
 * mla_decode -- absorbed multi-head latent attention decode ("MQA, GQA, and
 * MLA", section 5; "Why GQA's KV Cache Savings Don't Fully Reduce TPOT",
 * "What Makes MLA Different").  128 heads, d_c = 512, d_rope = 64.
 *   q_absorbed   [batch, 128, 512]   query times W_uk^(i), per head  fp16/bf16
 *   q_rope       [batch, 128, 64]    decoupled-RoPE query (rotated)   fp16/bf16
 *   latent_cache [num_blocks, block_size, 576]: elements [0,512) are the
 *                latent c_t, [512,576) the RoPE key shared by all heads
 *   block_table  [batch, max_blocks_per_seq] int32, seq_lens [batch] int32
 *   out          [batch, 128, 512]   sum_t p_t c_t (latent-space output;
 *                W_uv is applied by the caller)                      fp16/bf16
 *   scale        softmax scale (typically 1/sqrt(128 + 64))
 * s_t = scale * (q_absorbed . c_t + q_rope . k_rope_t).
 *
 * Work split: the 64-token tiles of all sequences, laid end to end, are cut
 * into launch->num_splits equal shares (the planner's choice for 0), each
 * streamed by one pair of CTAs; a share may cover the end of one sequence
 * and the start of the next, so ragged batches stay balanced.  A sequence
 * cut across shares is merged by a log-sum-exp combine; the workspace
 * (mla_decode_workspace_size) holds a per-sequence tile table and two fp32
 * partials per share.  num_splits = 1 needs no workspace.
 */
int mla_decode(const void* q_absorbed, const void* q_rope, const void* latent_cache,
               const int32_t* block_table, const int32_t* seq_lens, void* out, float scale,
               const decattn_launch* launch);

/*
 * gqa_kv_append, gqa_kv_append_fp8kv, mla_kv_append -- the decode step's
 * cache write: each sequence's new token joins the paged cache before its
 * query attends ("Compressing the KV Cache: DeepSeek's Latent Projections
 * (MLA) vs. Meta's Grouped Queries (GQA)": generation keeps the keys and
 * values of every past token in GPU memory, and "KV-Cache Management
 * Guardrails" keeps that cache in a paging engine; "MQA, GQA, and MLA",
 * section 5: MLA caches the latent with the decoupled RoPE key beside it).
 *   k_new, v_new   [batch, h_kv, d_head] in launch->dtype (fp16 / bf16)
 *   latent_new     [batch, 576] in launch->dtype: latent c_t then the RoPE key
 *   positions      [batch] int32: the slot the token takes in its sequence
 *                  (its position, normally the length before this step); a
 *                  negative position leaves the sequence untouched
 *   block_table    [batch, max_blocks_per_seq] int32
 *   k_cache, v_cache, latent_cache  the paged caches of gqa_decode,
 *                  gqa_decode_fp8kv and mla_decode; only the addressed slot
 *                  of each sequence is written
 *   k_scale, v_scale  [h_kv] fp32 (gqa_kv_append_fp8kv): value x of KV head
 *                  j is stored as the e4m3 code nearest to fp32(x) / scale[j]
 *                  (ties to even, magnitudes beyond 448 saturate to 448), so
 *                  gqa_decode_fp8kv reads back e4m3(code) * scale[j]
 * Of the launch block only batch, num_blocks, block_size, max_blocks_per_seq,
 * dtype, err_flag and stream are used (block_size as for the matching decode
 * call).  A position past the block table sets DECATTN_FLAG_BAD_SEQ_LEN, an
 * out-of-range block id DECATTN_FLAG_BAD_BLOCK; that sequence is skipped,
 * the others are written.  Sequences must name distinct slots.
 */
int gqa_kv_append(const void* k_new, const void* v_new, const int32_t* positions,
                  const int32_t* block_table, void* k_cache, void* v_cache, int h_kv, int d_head,
                  const decattn_launch* launch);
int gqa_kv_append_fp8kv(const void* k_new, const void* v_new, const float* k_scale,
                        const float* v_scale, const int32_t* positions,
                        const int32_t* block_table, void* k_cache, void* v_cache, int h_kv,
                        int d_head, const decattn_launch* launch);
int mla_kv_append(const void* latent_new, const int32_t* positions, const int32_t* block_table,
                  void* latent_cache, const decattn_launch* launch);

/*
 * mla_absorb_q, mla_unabsorb_out -- the two GEMMs either side of mla_decode
 * ("MQA, GQA, and MLA", section 5: q_i . k_i = x (W_q^(i) W_uk^(i)^T) c^T, so
 * the query is multiplied by W_uk^(i)^T once and the scores are taken
 * against the cached latent; "Why GQA's KV Cache Savings Don't Fully Reduce
 * TPOT", "What Makes MLA Different": matrix absorption needs no per-head
 * reconstruction at decode time).  With k_i = c W_uk^(i) and v_i = c W_uv^(i):
 *   mla_absorb_q      q_abs[b, i, :] = q_nope[b, i, :] W_uk^(i)^T
 *     q_nope  [batch, n_heads, d_h]      w_uk [n_heads, d_c, d_h] (w_uk[i] = W_uk^(i))
 *     q_abs   [batch, n_heads, d_c]      (written; mla_decode's q_absorbed)
 *   mla_unabsorb_out  out[b, i, :] = o_lat[b, i, :] W_uv^(i)
 *     o_lat   [batch, n_heads, d_c]      (mla_decode's out)
 *     w_uv_t  [n_heads, d_v, d_c]        (w_uv_t[i] = W_uv^(i) transposed)
 *     out     [batch, n_heads, d_v]      (written)
 * All tensors row-major in `dtype` (DECATTN_FP16 / DECATTN_BF16), 16-byte
 * aligned; products on tensor cores with fp32 accumulation,
 * results rounded to nearest-even.  Supported: the output width (d_c for
 * the query, d_v for the output) a multiple of 128, the contracted width (d_h,
 * resp. d_c) a multiple of 64; DeepSeek-V2/V3 use d_h = d_v = 128, d_c = 512.
 * err_flag (optional) gets DECATTN_FLAG_TIMEOUT if a pipeline wait gave up;
 * stream is a cudaStream_t (NULL: the default stream).
 */
int mla_absorb_q(const void* q_nope, const void* w_uk, void* q_abs, int batch, int n_heads,
                 int d_h, int d_c, int dtype, int* err_flag, void* stream);
int mla_unabsorb_out(const void* o_lat, const void* w_uv_t, void* out, int batch, int n_heads,
                     int d_c, int d_v, int dtype, int* err_flag, void* stream);

/* Split count the automatic planner picks (num_splits = 0).  num_sms <= 0
 * queries the current device.  Returns >= 1, or a negative status. */
int gqa_decode_plan_splits(int batch, int h_q, int h_kv, int d_head, int max_seq_len,
                           int num_sms);
int gqa_decode_fp8kv_plan_splits(int batch, int h_q, int h_kv, int d_head, int max_seq_len,
                                 int num_sms);
int mla_decode_plan_splits(int batch, int max_seq_len, int num_sms);
/* The windowed calls' planner: kv_bytes = 2 for gqa_decode_window, 1 for
 * gqa_decode_fp8kv_window; block_size a power of two. */
int gqa_decode_window_plan_splits(int batch, int h_q, int h_kv, int d_head, int max_seq_len,
                                  int window, int block_size, int kv_bytes, int num_sms);

/* Helpers of the interface with no defining passage on the pages (workspace
 * sizes, status text, version): conveniences of this C ABI.
 *
 * Workspace bytes needed for num_splits (>= 1): fp32 partial outputs and
 * log-sum-exps (GQA: one per split per row; MLA: two per share, plus a
 * per-sequence tile table).  0 when num_splits == 1.  Returns 0 for invalid
 * arguments as well; pure host arithmetic, no CUDA call. */
size_t gqa_decode_workspace_size(int batch, int h_q, int d_head, int num_splits);
size_t mla_decode_workspace_size(int batch, int num_splits);

/* KV-cache bytes per token: n_layers * n_kv * d_head * 2 (K and V) * bytes
 * ("Why GQA's KV Cache Savings Don't Fully Reduce TPOT", "KV Cache Size by
 * Attention Variant").  MLA: n_layers * (d_c + d_rope) * bytes ("MQA, GQA,
 * and MLA", section 5 "CACHE SIZE COMPARISON").  Negative on bad input. */
int64_t decattn_kv_bytes_per_token(int n_layers, int n_kv, int d_head, int bytes);
int64_t decattn_mla_bytes_per_token(int n_layers, int d_c, int d_rope, int bytes);

/* Static English text for a decattn_status value; never NULL. */
const char* decattn_status_string(int status);

/* decattn_selftest_wait_timeout -- runs the bounded mbarrier waits that
 * every kernel's pipeline uses on barriers that nothing completes, so that
 * they give up (a diagnostic for the failure path; the pages have no
 * counterpart).  One CTA: thread 0 waits with a limit of limit_us
 * microseconds (1..100000) and raises the CTA's abort word; thread 32 waits
 * with a 1000x longer limit but watches the abort word; thread 1 runs the
 * plain bounded wait.  Device writes: *err_flag |= DECATTN_FLAG_TIMEOUT;
 * result[0] = 1 if thread 0 gave up, result[1] = 1 if thread 32 left on the
 * abort word (well before its own limit), result[2], result[3] = the
 * microseconds each waited, result[4] = 1 if the plain wait gave up.
 * err_flag, result: device pointers (result holds 5 ints); stream: a
 * cudaStream_t or NULL. */
int decattn_selftest_wait_timeout(int* err_flag, int* result, int limit_us, void* stream);

/* Library version as major*10000 + minor*100 + patch. */
int decattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DECATTN_H */
