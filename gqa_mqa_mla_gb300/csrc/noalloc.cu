// noalloc.cu -- gqa_decode_noalloc: gqa_decode without a caller-provided
// workspace, for callers that are not allowed to allocate device memory.
//
// Some hosts of this library cannot call cudaMalloc (or any allocating
// routine) around a decode call: serving engines that reserve nearly all
// HBM for the paged KV cache up front and forbid later allocations, plugin
// interfaces of inference runtimes that hand the plugin only its inputs and
// outputs, and latency-critical loops where an allocation's implicit
// synchronisation is unacceptable.  For them the split-KV scratch lives in a
// fixed, file-scope device array that every GPU which loads this library
// holds until the process exits.
//
// Rules of use:
//   * the scratch holds at most kNoallocScratchBytes; a call whose split
//     plan needs more is rejected with DECATTN_ERR_WORKSPACE before any
//     launch;
//   * every call on a device shares the one array: calls that overlap on the
//     GPU (different streams, no ordering between them) race and corrupt
//     each other's results; serialise them;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first call
//     before any stream capture.  The address is kept for the life of the
//     process: a device reset (cudaDeviceReset, or a reset of the primary
//     context) is not supported afterwards;
//   * the array keeps the previous call's contents; nothing in it needs to
//     start at zero (each call overwrites every partial it later reads).
#include <mutex>

#include "decattn.h"
#include "internal.h"

namespace decattn {
namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;  // 8 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array for the current device (looked up once
// per device).  Returns nullptr on failure.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace decattn

extern "C" {

int gqa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* seq_lens, void* out, int h_q,
                       int h_kv, int d_head, float scale, const decattn_launch* launch) {
  // gqa_decode's own argument checks first, so that a bad argument gets the
  // status gqa_decode would return for it.
  const int st = decattn::gqa_check_args(q, k_cache, v_cache, nullptr, nullptr, false,
                                         block_table, seq_lens, out, h_q, h_kv, d_head, scale,
                                         0, launch);
  if (st != DECATTN_OK) return st;
  int n_split = launch->num_splits;
  if (n_split == 0) {
    n_split = gqa_decode_plan_splits(launch->batch, h_q, h_kv, d_head, launch->max_seq_len, 0);
    if (n_split < 0) return n_split;
  }
  // The scratch a plan needs depends on the split count gqa_decode will
  // actually run: a requested count is cut to the number of 64-token tiles
  // of the longest sequence (one split needs no scratch at all).
  int tokens_per_split = 0;
  const int eff = decattn::resolve_splits(launch->max_seq_len, n_split, &tokens_per_split);
  const size_t need = gqa_decode_workspace_size(launch->batch, h_q, d_head, eff);
  if (need > decattn::kNoallocScratchBytes) return DECATTN_ERR_WORKSPACE;
  void* scratch = decattn::scratch_for_current_device();
  if (!scratch) return DECATTN_ERR_CUDA;
  decattn_launch l = *launch;
  l.num_splits = n_split;
  l.workspace = scratch;
  l.workspace_bytes = decattn::kNoallocScratchBytes;
  return gqa_decode(q, k_cache, v_cache, block_table, seq_lens, out, h_q, h_kv, d_head, scale, &l);
}

}  // extern "C"
