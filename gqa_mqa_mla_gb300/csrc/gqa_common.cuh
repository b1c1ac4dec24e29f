// gqa_common.cuh -- the per-CTA token range and bad-data handling shared by
// the GQA partial kernels (one CTA per split, KV head j and sequence b).
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace decattn {

// Token range [t_begin, t_end) of split `split` of sequence b, the window
// start w0 ("07 · MHA/MQA/GQA/MLA quick learn": each token attends only to
// the last W tokens), and this thread's share of the validity checks.
// Tiles start at the block (or 64-token) boundary holding w0; blocks wholly
// before the window are never read.  `bad` is this thread's verdict only: the
// caller ORs it over the CTA (block ids are checked strided by threadIdx.x).
struct GqaSpan {
  int w0, t_begin, t_end, bad;
};

DECATTN_DEV GqaSpan gqa_span(const GqaParams& p, int split, int j, int b) {
  GqaSpan r;
  const int seq_len = p.seq_lens[b];
  r.bad = 0;
  if (seq_len < 0 || seq_len > p.max_seq_len) {
    r.bad = 1;
    if (threadIdx.x == 0 && split == 0 && j == 0) flag_error(p.err_flag, kFlagBadSeqLen);
  }
  r.w0 = (p.window > 0 && seq_len > p.window) ? seq_len - p.window : 0;
  const int base = r.w0 & ~((p.block_size < kTile ? p.block_size : kTile) - 1);
  r.t_begin = base + split * p.tokens_per_split;
  r.t_end = r.bad ? r.t_begin : min(seq_len, r.t_begin + p.tokens_per_split);
  if (!r.bad && r.t_end > r.t_begin) {
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const int k1 = (r.t_end - 1) >> p.log2_block_size;
    for (int k = (r.t_begin >> p.log2_block_size) + threadIdx.x; k <= k1; k += blockDim.x) {
      const int id = bt[k];
      if (id < 0 || id >= p.num_blocks) {
        r.bad = 1;
        flag_error(p.err_flag, kFlagBadBlock);
      }
    }
  }
  return r;
}

// Rows row0 .. row0 + rows - 1 of a CTA that met bad data (zeros plus the
// poison marker for the combine) or an empty token range (zeros, lse = -inf).
DECATTN_DEV void gqa_write_empty(const GqaParams& p, size_t row0, int rows, int split, bool bad) {
  for (int e = threadIdx.x; e < rows * kHeadDim; e += blockDim.x) {
    const int r = e / kHeadDim, d = e % kHeadDim;
    if (p.n_split == 1) {
      static_cast<uint16_t*>(p.out)[(row0 + r) * kHeadDim + d] = 0;
    } else {
      p.part_o[((row0 + r) * p.n_split + split) * kHeadDim + d] = 0.f;
      if (d == 0)
        p.part_lse[(row0 + r) * p.n_split + split] = bad ? DECATTN_POISON_LSE : -__builtin_huge_valf();
    }
  }
}

}  // namespace decattn
