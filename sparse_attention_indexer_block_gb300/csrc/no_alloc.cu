// indexer_decode_topk_noalloc: decode top-k with scratch that lives in this
// library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory where they run the indexer: code
// that runs while a stream is being captured into a CUDA graph (allocation
// calls are not recorded into the graph and may synchronise the device),
// serving loops that forbid allocator calls on their latency-critical path,
// and hosts whose device memory belongs to another allocator that this code
// path cannot reach. For them the scratch is a file-scope device array that
// exists once per GPU that loads the library and is held until the process
// exits.
#include <mutex>

#include "internal.h"

namespace {

// Scratch shared by every call on one GPU. 64 MiB holds the decode workspace
// of about 5700 requests at next_n = 1 (about 2050 at next_n = 2) with
// top-2048 on a 152-SM GPU.
constexpr size_t kNoAllocScratchBytes = 64u << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// In host code `g_noalloc_scratch` is only a host-side stand-in for the device
// array; its device address comes from cudaGetSymbolAddress, looked up once per
// device with that device current (the first lookup may load the library's
// device code).
std::mutex g_scratch_mutex;
void* g_scratch_ptr[saib::kMaxDevices] = {};

idx_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= saib::kMaxDevices) return IDX_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return IDX_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return IDX_OK;
}

}  // namespace

extern "C" idx_status indexer_decode_topk_noalloc(
    const void* q, const float* weights, const uint8_t* index_cache, int64_t num_pages,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width, const int32_t* row_seq_lens,
    int32_t num_reqs, int32_t next_n, int32_t num_heads, int32_t head_dim, int32_t topk,
    int32_t* out_idx, uint32_t* dev_error, void* stream) {
  size_t need = 0;
  idx_status st = indexer_decode_workspace_bytes(num_reqs, next_n, topk, &need);
  if (st != IDX_OK) return st;
  if (need > kNoAllocScratchBytes) return IDX_ERR_WORKSPACE;  // batch too large for the scratch
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != IDX_OK) return st;
  // The array keeps the previous call's contents; the decode path re-initialises
  // everything that must start at zero (segment counters, row histograms) on
  // every call before it is read.
  return indexer_decode_topk(q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                             row_seq_lens, num_reqs, next_n, num_heads, head_dim, topk, out_idx,
                             scratch, kNoAllocScratchBytes, dev_error, stream);
}
