// C ABI of the indexer: argument validation, workspace carve-up, the host
// prefill chunk planner and the launch sequences.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "internal.h"

namespace saib {

namespace {

thread_local cudaError_t g_last_cuda_error = cudaSuccess;
thread_local uint64_t* g_trace = nullptr;
thread_local size_t g_trace_bytes = 0;
thread_local cudaEvent_t g_prof_start = nullptr;
thread_local cudaEvent_t g_prof_stop = nullptr;

// Give-up time of the kernels' waits: 2 s, or the test setting of this thread;
// with g_stall_rows the split-row selection waits for a segment that never
// comes.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
thread_local uint64_t g_wait_ns = kDefaultWaitNs;
thread_local int32_t g_stall_rows = 0;

// The score/select launch and, in top-k mode, the split-row selection after
// it, bracketed by the profiling events when they are set.
idx_status timed_score(int G, bool logits, const ScoreParams& p, const CUtensorMap& map,
                       cudaStream_t s, bool mx = false) {
  if (g_prof_start) {
    const idx_status st = cuda_status(cudaEventRecord(g_prof_start, s));
    if (st != IDX_OK) return st;
  }
  const int streams = score_streams(G);
  idx_status st = launch_score(G, logits, mx, p, map, score_grid(), s);
  if (st == IDX_OK && !logits) {
    RowSelectParams r{};
    r.wr = p.wr;
    r.wr_tile_start = p.wr_tile_start;
    r.cta_row = p.cta_row;
    r.row_ctas = p.row_ctas;
    r.row_len = p.row_len;
    r.seg_counter = p.seg_counter;
    r.slot_key = p.slot_key;
    r.slot_idx = p.slot_idx;
    r.seg_cum = p.seg_cum;
    r.slot_cap = p.slot_cap;
    r.row_hist = p.row_hist;
    r.num_wr = p.num_wr;
    r.streams = streams;
    r.G = G;
    r.topk = p.topk;
    r.out_idx = p.out_idx;
    r.out_val = p.out_val;
    r.out_row_base = p.out_row_base;
    r.dev_error = p.dev_error;
    r.wait_ns = g_wait_ns;
    r.stall = g_stall_rows ? 1 : 0;
    const int64_t grid = max_split_rows(p.num_wr, streams) * G;
    // trace slots after the score kernel's (when the buffer holds both)
    size_t tb = 0;
    uint64_t* tbuf = trace_buffer(&tb);
    const size_t score_slots = static_cast<size_t>(kTrSlots) * streams;
    if (tbuf && tb >= 8 * (score_slots + static_cast<size_t>(kSelTrSlots) * grid))
      r.trace = tbuf + score_slots;
    st = launch_row_select(r, static_cast<int>(grid), s);
  }
  if (st == IDX_OK && g_prof_stop) return cuda_status(cudaEventRecord(g_prof_stop, s));
  return st;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

void record_cuda_error(cudaError_t e) { g_last_cuda_error = e; }

uint64_t* trace_buffer(size_t* bytes) {
  *bytes = g_trace_bytes;
  return g_trace;
}

WsLayout ws_layout(int64_t num_wr, int64_t rows, int G, int topk, int num_ctas) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = round_up(off, align);
    const size_t o = off;
    off += bytes;
    return o;
  };
  const int64_t nslots = 2 * static_cast<int64_t>(num_ctas);  // segment_slot
  const int64_t nsplit = max_split_rows(num_wr, num_ctas);
  L.wr = take(sizeof(WorkRow) * static_cast<size_t>(num_wr), 256);
  L.wr_tile_start = take(4 * static_cast<size_t>(num_wr + 1), 256);
  L.row_len = take(4 * static_cast<size_t>(rows), 256);
  // per work row its segment counter (zeroed by the prep kernel)
  L.seg_counter = take(4 * static_cast<size_t>(num_wr), 256);
  L.seg_cum = take(4 * static_cast<size_t>(nslots * G) * kRowHistBins, 256);
  L.q8 = take(static_cast<size_t>(rows) * kQRowBytes, 1024);
  L.wprime = take(4 * static_cast<size_t>(rows) * kHeads, 256);
  const size_t cap = static_cast<size_t>(candidate_capacity(G));
  L.slot_key = take(4 * static_cast<size_t>(nslots * G) * cap, 256);
  L.slot_idx = take(4 * static_cast<size_t>(nslots * G) * cap, 256);
  L.row_hist_words = static_cast<size_t>(nsplit) * G * kRowHistBins;
  L.row_hist = take(4 * L.row_hist_words, 256);
  L.cta_row = take(4 * static_cast<size_t>(num_ctas), 256);
  L.cta_tile = take(4 * static_cast<size_t>(num_ctas + 1), 256);
  L.row_vs = take(4 * static_cast<size_t>(num_wr + 1), 256);
  L.row_ctas = take(8 * static_cast<size_t>(num_wr), 256);
  L.total = round_up(off, 256);
  return L;
}

int device_sm_count() {
  static std::atomic<int> cached[kMaxDevices];  // 0 = not looked up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 1;
  if (dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

idx_status encode_cache_map(CUtensorMap* map, const uint8_t* cache, int64_t num_pages) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!encode) return IDX_ERR_CUDA;
  // [page][token][128 bytes]: one box is one page's 64 key rows (8 KB).
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(kPageTokens),
                              static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(kPageBytes)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kDim), static_cast<cuuint32_t>(kPageTokens), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(cache), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IDX_OK : IDX_ERR_CUDA;
}

namespace {

// Greedy chunking of prefill requests (split_indexer_prefill_chunks of the
// vLLM sparse-indexer backend): pack requests while the summed key count stays
// within the workspace and the M x N fp32 logits within the budget; a request
// that fits alone in neither goes by itself; cut each chunk's queries into
// pieces of max(1, budget_elems / N).
struct Chunk {
  int32_t r0, r1, q0, q1;
};

std::vector<Chunk> plan_chunks(const int32_t* sl, const int32_t* ql, int32_t n, int64_t ws_tokens,
                               int64_t budget_bytes) {
  std::vector<Chunk> out;
  const int64_t elems = budget_bytes / 4;
  int32_t end = 0;
  while (end < n) {
    const int32_t start = end;
    int64_t m = 0, keys = 0;
    for (; end < n; ++end) {
      const int64_t nm = m + ql[end], nk = keys + sl[end];
      if (nk > ws_tokens || nm * nk > elems) break;
      m = nm;
      keys = nk;
    }
    if (end == start) {
      m = ql[end];
      keys = sl[end];
      ++end;
    }
    const int64_t piece = keys > 0 ? std::max<int64_t>(1, elems / keys) : m;
    for (int64_t q = 0; q < m; q += piece)
      out.push_back(Chunk{start, end, static_cast<int32_t>(q),
                          static_cast<int32_t>(std::min(m, q + piece))});
  }
  return out;
}

// Prefill work rows: up to two consecutive queries of one request.
constexpr int kPrefillG = 2;

// Work rows of a chunk: groups of up to kPrefillG consecutive queries of one request.
int64_t chunk_work_rows(const std::vector<int64_t>& qsl, const Chunk& c, int64_t* row_lo,
                        int64_t* row_hi) {
  *row_lo = qsl[c.r0] + c.q0;
  *row_hi = qsl[c.r0] + c.q1;
  int64_t nw = 0;
  for (int32_t r = c.r0; r < c.r1; ++r) {
    const int64_t lo = std::max(qsl[r], *row_lo), hi = std::min(qsl[r + 1], *row_hi);
    if (hi > lo) nw += (hi - lo + kPrefillG - 1) / kPrefillG;
  }
  return nw;
}


idx_status check_common(const void* q, const float* w, const uint8_t* cache, int64_t num_pages,
                        const int32_t* bt, int64_t bt_stride, int32_t bt_width, int32_t num_heads,
                        int32_t head_dim, int32_t topk) {
  if (!q || !w || !cache || !bt) return IDX_ERR_INVALID_ARG;
  if (num_pages < 1 || num_pages > INT32_MAX || bt_width < 1 || bt_stride < bt_width)
    return IDX_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(w, 4) || !aligned(cache, 16) || !aligned(bt, 4))
    return IDX_ERR_INVALID_ARG;
  if (num_heads != kHeads || head_dim != kDim) return IDX_ERR_UNSUPPORTED;
  if (topk < 1 || topk > IDX_MAX_TOPK) return IDX_ERR_UNSUPPORTED;
  return IDX_OK;
}

// A work row that ends inside a stream's range costs that stream a segment
// finalisation (publication, and a fresh buffer for the next row that fills
// and is cut again) worth about `penalty` tiles of streaming; the split gives
// such streams correspondingly fewer tiles. When each stream streams >= 64
// tiles the penalty grows by the share / `div` (the fresh buffer's cuts grow
// with the row's length). One-token rows: fitted to per-stream end times on
// GB300 (end = a + b * tiles + c * row ends; c = 0.6 tiles on the decode
// batch, 23.5 on long context, share 431). Two-token rows: 12 + share / 24
// measured faster on MTP than the fit there (2 + share / 43).
void decode_row_penalty(bool logits, int next_n, int32_t* penalty, int32_t* div) {
  *penalty = logits ? 0 : (next_n == 1 ? 1 : 12);
  *div = logits ? 0 : (next_n == 1 ? 19 : 24);
}

// Token rows' key counts: given per row, or expanded from the requests'
// (seq_lens, decode_lens) by the prep kernel.
struct RowLens {
  const int32_t* row_seq_lens;
  const int32_t* seq_lens;
  const int32_t* decode_lens;
};

// Values mode: the selected keys' logits beside their indices, every row of
// > 0 keys selected; on one rank of a key-sharded cache (world > 1) the rows
// score the rank's share of their keys and the indices go out global.
struct ValuesOut {
  float* out_val;
  int32_t compress_ratio, rank, world, interleave;
};

bool valid_values(const ValuesOut* vo) {
  return vo->out_val && vo->compress_ratio >= 1 && vo->world >= 1 && vo->rank >= 0 &&
         vo->rank < vo->world && vo->interleave >= 1;
}

idx_status decode_common(bool logits, const void* q, const float* weights,
                         const uint8_t* index_cache, int64_t num_pages, const int32_t* block_table,
                         int64_t bt_stride, int32_t bt_width, const RowLens& lens,
                         int32_t num_reqs, int32_t next_n, int32_t num_heads, int32_t head_dim,
                         int32_t topk, int32_t* out_idx, float* out_logits, int64_t ld_logits,
                         void* workspace, size_t workspace_bytes, uint32_t* dev_error,
                         void* stream, const ValuesOut* vo = nullptr, bool mx = false) {
  if (num_reqs < 0) return IDX_ERR_INVALID_ARG;
  if (mx && next_n != 1) return IDX_ERR_UNSUPPORTED;
  const bool values = vo != nullptr;
  if (values && !valid_values(vo)) return IDX_ERR_INVALID_ARG;
  if (next_n != 1 && next_n != 2) return IDX_ERR_UNSUPPORTED;
  idx_status st = check_common(q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                               num_heads, head_dim, topk);
  if (st != IDX_OK) return st;
  if (!lens.row_seq_lens && (!lens.seq_lens || !lens.decode_lens)) return IDX_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return IDX_ERR_INVALID_ARG;
  if (logits) {
    if (!out_logits || ld_logits < static_cast<int64_t>(bt_width) * kPageTokens)
      return IDX_ERR_INVALID_ARG;
  } else if (!out_idx) {
    return IDX_ERR_INVALID_ARG;
  }
  if (num_reqs == 0) return IDX_OK;
  const int nC = score_streams(next_n);
  const int64_t rows = static_cast<int64_t>(num_reqs) * next_n;
  const WsLayout L = ws_layout(num_reqs, rows, next_n, topk, nC);
  if (workspace_bytes < L.total) return IDX_ERR_WORKSPACE;
  CUtensorMap map{};  // (MXFP4 pages are read with bulk copies)
  if (!mx && (st = encode_cache_map(&map, index_cache, num_pages)) != IDX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t row_penalty, row_penalty_div;
  decode_row_penalty(logits, next_n, &row_penalty, &row_penalty_div);
  DecodePrepArgs a{static_cast<const __nv_bfloat16*>(q), weights, lens.row_seq_lens, num_reqs,
                   next_n, topk, bt_width, (logits || values) ? 1 : 0, out_idx, dev_error, nC,
                   row_penalty, row_penalty_div, lens.seq_lens, lens.decode_lens};
  if (values) {
    a.out_val = vo->out_val;
    a.compress_ratio = vo->compress_ratio;
    a.dcp_rank = vo->rank;
    a.dcp_world = vo->world;
    a.dcp_interleave = vo->interleave;
  }
  if ((st = launch_decode_prep(a, ws, L, s)) != IDX_OK) return st;
  ScoreParams p{};
  p.cache = index_cache;
  p.num_pages = num_pages;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.wr = reinterpret_cast<const WorkRow*>(ws + L.wr);
  p.wr_tile_start = reinterpret_cast<const int32_t*>(ws + L.wr_tile_start);
  p.cta_row = reinterpret_cast<const int32_t*>(ws + L.cta_row);
  p.cta_tile = reinterpret_cast<const int32_t*>(ws + L.cta_tile);
  p.row_ctas = reinterpret_cast<const int2*>(ws + L.row_ctas);
  p.num_wr = num_reqs;
  p.row_len = reinterpret_cast<const int32_t*>(ws + L.row_len);
  p.q8 = ws + L.q8;
  p.wprime = reinterpret_cast<const float*>(ws + L.wprime);
  p.seg_counter = reinterpret_cast<int32_t*>(ws + L.seg_counter);
  p.slot_key = reinterpret_cast<uint32_t*>(ws + L.slot_key);
  p.slot_idx = reinterpret_cast<int32_t*>(ws + L.slot_idx);
  p.slot_cap = candidate_capacity(next_n);
  p.seg_cum = reinterpret_cast<uint32_t*>(ws + L.seg_cum);
  p.row_hist = reinterpret_cast<uint32_t*>(ws + L.row_hist);
  p.wait_ns = g_wait_ns;
  p.out_idx = out_idx;
  p.out_row_base = 0;
  p.topk = topk;
  p.short_len = values ? 0 : topk;
  p.out_val = values ? vo->out_val : nullptr;
  p.out_logits = out_logits;
  p.ld_logits = ld_logits;
  p.dev_error = dev_error;
  size_t tb = 0;
  p.trace = trace_buffer(&tb);
  if (tb < sizeof(uint64_t) * kTrSlots * static_cast<size_t>(nC)) p.trace = nullptr;
  st = timed_score(next_n, logits, p, map, s, mx);
  if (st == IDX_OK && values && vo->world > 1)
    st = launch_dcp_globalise(out_idx, rows * topk, vo->rank, vo->world, vo->interleave, s);
  return st;
}

}  // namespace
}  // namespace saib

using namespace saib;

extern "C" {

idx_status indexer_trace_buffer(void* buffer, size_t bytes) {
  g_trace = static_cast<uint64_t*>(buffer);
  g_trace_bytes = buffer ? bytes : 0;
  return IDX_OK;
}

idx_status indexer_debug_wait_limit(uint64_t limit_ns, int32_t stall_split_rows) {
  g_wait_ns = limit_ns ? limit_ns : kDefaultWaitNs;
  g_stall_rows = stall_split_rows;
  return IDX_OK;
}

idx_status indexer_debug_divide(const float* a, const float* b, int64_t n, float* quotient,
                                float* quotient_ieee, void* stream) {
  if (n < 0) return IDX_ERR_INVALID_ARG;
  if (n == 0) return IDX_OK;
  if (!a || !b || !quotient || !quotient_ieee) return IDX_ERR_INVALID_ARG;
  return launch_divide_check(a, b, n, quotient, quotient_ieee, static_cast<cudaStream_t>(stream));
}

idx_status indexer_profile_events(void* start_event, void* stop_event) {
  g_prof_start = static_cast<cudaEvent_t>(start_event);
  g_prof_stop = static_cast<cudaEvent_t>(stop_event);
  return IDX_OK;
}

const char* indexer_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}

const char* indexer_status_string(idx_status status) {
  switch (status) {
    case IDX_OK: return "ok";
    case IDX_ERR_INVALID_ARG: return "invalid argument";
    case IDX_ERR_UNSUPPORTED: return "unsupported configuration";
    case IDX_ERR_WORKSPACE: return "workspace too small";
    case IDX_ERR_CUDA: return "CUDA error";
    case IDX_ERR_CAPACITY: return "output capacity too small";
  }
  return "unknown status";
}

idx_status indexer_expand_decode_rows(const int32_t* seq_lens, const int32_t* decode_lens,
                                      int32_t num_reqs, int32_t next_n,
                                      const int32_t* block_table, int64_t bt_stride,
                                      int32_t bt_width, int32_t mode, int32_t* row_seq_lens,
                                      int32_t* row_block_table, int64_t out_stride,
                                      int64_t num_out_rows, uint32_t* dev_error, void* stream) {
  if (num_reqs < 0 || next_n < 1 || (mode != 0 && mode != 1) || num_out_rows < 0)
    return IDX_ERR_INVALID_ARG;
  if ((num_reqs > 0 && (!seq_lens || !decode_lens)) || (num_out_rows > 0 && !row_seq_lens))
    return IDX_ERR_INVALID_ARG;
  if (mode == 0 && num_out_rows < static_cast<int64_t>(num_reqs) * next_n)
    return IDX_ERR_CAPACITY;
  if (row_block_table && (!block_table || bt_width < 1 || bt_stride < bt_width ||
                          out_stride < bt_width))
    return IDX_ERR_INVALID_ARG;
  if (num_reqs == 0 && (mode == 0 || num_out_rows == 0)) return IDX_OK;
  return launch_expand(seq_lens, decode_lens, num_reqs, next_n, block_table, bt_stride, bt_width,
                       mode, row_seq_lens, row_block_table, out_stride, num_out_rows, dev_error,
                       static_cast<cudaStream_t>(stream));
}

idx_status indexer_quantize_q(const void* q, const float* weights, int64_t num_rows,
                              int32_t num_heads, int32_t head_dim, uint8_t* q_fp8,
                              float* weights_scaled, void* stream) {
  if (num_rows < 0) return IDX_ERR_INVALID_ARG;
  if (num_heads != kHeads || head_dim != kDim) return IDX_ERR_UNSUPPORTED;
  if (num_rows == 0) return IDX_OK;
  if (!q || !weights || !q_fp8 || !weights_scaled || !aligned(q, 16) || !aligned(q_fp8, 4))
    return IDX_ERR_INVALID_ARG;
  return launch_quantize_plain(static_cast<const __nv_bfloat16*>(q), weights, num_rows, q_fp8,
                               weights_scaled, static_cast<cudaStream_t>(stream));
}

idx_status indexer_insert_keys(const void* k, const int64_t* slot_mapping, int64_t num_tokens,
                               int32_t head_dim, uint8_t* index_cache, int64_t num_pages,
                               uint32_t* dev_error, void* stream) {
  if (num_tokens < 0 || num_pages < 0) return IDX_ERR_INVALID_ARG;
  if (head_dim != kDim) return IDX_ERR_UNSUPPORTED;
  if (num_tokens == 0) return IDX_OK;
  if (!k || !slot_mapping || !index_cache || !aligned(k, 8) || !aligned(slot_mapping, 8) ||
      !aligned(index_cache, 16))
    return IDX_ERR_INVALID_ARG;
  return launch_insert_keys(static_cast<const __nv_bfloat16*>(k), slot_mapping, num_tokens,
                            index_cache, num_pages, dev_error, static_cast<cudaStream_t>(stream));
}

idx_status indexer_decode_workspace_bytes(int32_t num_reqs, int32_t next_n, int32_t topk,
                                          size_t* bytes) {
  if (!bytes || num_reqs < 0) return IDX_ERR_INVALID_ARG;
  if ((next_n != 1 && next_n != 2) || topk < 1 || topk > IDX_MAX_TOPK) return IDX_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(num_reqs, static_cast<int64_t>(num_reqs) * next_n, next_n, topk,
                               score_streams(next_n));
  *bytes = L.total;
  return IDX_OK;
}

idx_status indexer_debug_decode_plan(int32_t num_reqs, int32_t next_n, int32_t topk,
                                     int64_t* offsets, int32_t* grid, int32_t* penalty) {
  if (!offsets || !grid || !penalty || num_reqs < 0) return IDX_ERR_INVALID_ARG;
  if ((next_n != 1 && next_n != 2) || topk < 1 || topk > IDX_MAX_TOPK) return IDX_ERR_UNSUPPORTED;
  const int nC = score_streams(next_n);
  const WsLayout L = ws_layout(num_reqs, static_cast<int64_t>(num_reqs) * next_n, next_n, topk, nC);
  offsets[0] = static_cast<int64_t>(L.wr_tile_start);
  offsets[1] = static_cast<int64_t>(L.cta_tile);
  offsets[2] = static_cast<int64_t>(L.row_ctas);
  offsets[3] = static_cast<int64_t>(L.cta_row);
  *grid = nC;
  decode_row_penalty(false, next_n, &penalty[0], &penalty[1]);
  return IDX_OK;
}

idx_status indexer_decode_topk(const void* q, const float* weights, const uint8_t* index_cache,
                               int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                               int32_t bt_width, const int32_t* row_seq_lens, int32_t num_reqs,
                               int32_t next_n, int32_t num_heads, int32_t head_dim, int32_t topk,
                               int32_t* out_idx, void* workspace, size_t workspace_bytes,
                               uint32_t* dev_error, void* stream) {
  return decode_common(false, q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                       RowLens{row_seq_lens, nullptr, nullptr}, num_reqs, next_n, num_heads,
                       head_dim, topk, out_idx, nullptr, 0, workspace, workspace_bytes, dev_error,
                       stream);
}

idx_status indexer_decode_topk_from_lens(const void* q, const float* weights,
                                         const uint8_t* index_cache, int64_t num_pages,
                                         const int32_t* block_table, int64_t bt_stride,
                                         int32_t bt_width, const int32_t* seq_lens,
                                         const int32_t* decode_lens, int32_t num_reqs,
                                         int32_t next_n, int32_t num_heads, int32_t head_dim,
                                         int32_t topk, int32_t* out_idx, void* workspace,
                                         size_t workspace_bytes, uint32_t* dev_error,
                                         void* stream) {
  if (!seq_lens || !decode_lens) return IDX_ERR_INVALID_ARG;
  return decode_common(false, q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                       RowLens{nullptr, seq_lens, decode_lens}, num_reqs, next_n, num_heads,
                       head_dim, topk, out_idx, nullptr, 0, workspace, workspace_bytes, dev_error,
                       stream);
}

idx_status indexer_decode_logits(const void* q, const float* weights, const uint8_t* index_cache,
                                 int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                                 int32_t bt_width, const int32_t* row_seq_lens, int32_t num_reqs,
                                 int32_t next_n, int32_t num_heads, int32_t head_dim,
                                 int32_t topk, float* out_logits, int64_t ld_logits,
                                 void* workspace, size_t workspace_bytes, uint32_t* dev_error,
                                 void* stream) {
  return decode_common(true, q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                       RowLens{row_seq_lens, nullptr, nullptr}, num_reqs, next_n, num_heads,
                       head_dim, topk, nullptr, out_logits, ld_logits, workspace, workspace_bytes,
                       dev_error, stream);
}

idx_status indexer_decode_topk_mxfp4(const void* q, const float* weights,
                                     const uint8_t* index_cache, int64_t num_pages,
                                     const int32_t* block_table, int64_t bt_stride,
                                     int32_t bt_width, const int32_t* row_seq_lens,
                                     int32_t num_reqs, int32_t next_n, int32_t num_heads,
                                     int32_t head_dim, int32_t topk, int32_t* out_idx,
                                     void* workspace, size_t workspace_bytes, uint32_t* dev_error,
                                     void* stream) {
  return decode_common(false, q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                       RowLens{row_seq_lens, nullptr, nullptr}, num_reqs, next_n, num_heads,
                       head_dim, topk, out_idx, nullptr, 0, workspace, workspace_bytes, dev_error,
                       stream, nullptr, true);
}

idx_status indexer_decode_logits_mxfp4(const void* q, const float* weights,
                                       const uint8_t* index_cache, int64_t num_pages,
                                       const int32_t* block_table, int64_t bt_stride,
                                       int32_t bt_width, const int32_t* row_seq_lens,
                                       int32_t num_reqs, int32_t next_n, int32_t num_heads,
                                       int32_t head_dim, int32_t topk, float* out_logits,
                                       int64_t ld_logits, void* workspace, size_t workspace_bytes,
                                       uint32_t* dev_error, void* stream) {
  return decode_common(true, q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                       RowLens{row_seq_lens, nullptr, nullptr}, num_reqs, next_n, num_heads,
                       head_dim, topk, nullptr, out_logits, ld_logits, workspace, workspace_bytes,
                       dev_error, stream, nullptr, true);
}

idx_status indexer_decode_topk_values(const void* q, const float* weights,
                                      const uint8_t* index_cache, int64_t num_pages,
                                      const int32_t* block_table, int64_t bt_stride,
                                      int32_t bt_width, const int32_t* row_seq_lens,
                                      int32_t num_reqs, int32_t next_n, int32_t num_heads,
                                      int32_t head_dim, int32_t topk, int32_t compress_ratio,
                                      int32_t dcp_rank, int32_t dcp_world, int32_t dcp_interleave,
                                      int32_t* out_idx, float* out_val, void* workspace,
                                      size_t workspace_bytes, uint32_t* dev_error, void* stream) {
  if (!out_val) return IDX_ERR_INVALID_ARG;
  const ValuesOut vo{out_val, compress_ratio, dcp_rank, dcp_world, dcp_interleave};
  return decode_common(false, q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                       RowLens{row_seq_lens, nullptr, nullptr}, num_reqs, next_n, num_heads,
                       head_dim, topk, out_idx, nullptr, 0, workspace, workspace_bytes, dev_error,
                       stream, &vo);
}

idx_status indexer_index_key_counts(const int32_t* row_seq_lens, int64_t num_rows,
                                   int32_t compress_ratio, int32_t dcp_rank, int32_t dcp_world,
                                   int32_t dcp_interleave, int32_t* key_counts, void* stream) {
  if (num_rows < 0 || compress_ratio < 1 || dcp_world < 1 || dcp_rank < 0 ||
      dcp_rank >= dcp_world || dcp_interleave < 1)
    return IDX_ERR_INVALID_ARG;
  if (num_rows == 0) return IDX_OK;
  if (!row_seq_lens || !key_counts) return IDX_ERR_INVALID_ARG;
  return launch_key_counts(row_seq_lens, num_rows, compress_ratio, dcp_rank, dcp_world,
                           dcp_interleave, key_counts, static_cast<cudaStream_t>(stream));
}

idx_status indexer_dcp_merge(const float* cand_val, const int32_t* cand_idx, int32_t dcp_world,
                             int64_t num_rows, int32_t topk, int32_t* out_idx, float* out_val,
                             void* stream) {
  if (num_rows < 0 || dcp_world < 1) return IDX_ERR_INVALID_ARG;
  if (topk < 1 || topk > IDX_MAX_TOPK) return IDX_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(dcp_world) * topk > IDX_DCP_MAX_CANDIDATES) return IDX_ERR_UNSUPPORTED;
  if (num_rows == 0) return IDX_OK;
  if (!cand_val || !cand_idx || !out_idx) return IDX_ERR_INVALID_ARG;
  return launch_dcp_merge(cand_val, cand_idx, dcp_world, num_rows, topk, out_idx, out_val,
                          static_cast<cudaStream_t>(stream));
}

idx_status indexer_plan_prefill_chunks(const int32_t* seq_lens_host,
                                       const int32_t* query_lens_host, int32_t num_reqs,
                                       int64_t workspace_tokens, int64_t logits_budget_bytes,
                                       int32_t* chunks, int32_t max_chunks, int32_t* num_chunks) {
  if (num_reqs < 0 || !num_chunks || max_chunks < 0 || (max_chunks > 0 && !chunks))
    return IDX_ERR_INVALID_ARG;
  if (num_reqs > 0 && (!seq_lens_host || !query_lens_host)) return IDX_ERR_INVALID_ARG;
  if (workspace_tokens < 0 || logits_budget_bytes < 0) return IDX_ERR_INVALID_ARG;
  const std::vector<Chunk> plan =
      plan_chunks(seq_lens_host, query_lens_host, num_reqs, workspace_tokens, logits_budget_bytes);
  *num_chunks = static_cast<int32_t>(plan.size());
  if (static_cast<int64_t>(plan.size()) > max_chunks) return IDX_ERR_CAPACITY;
  for (size_t i = 0; i < plan.size(); ++i) {
    chunks[4 * i + 0] = plan[i].r0;
    chunks[4 * i + 1] = plan[i].r1;
    chunks[4 * i + 2] = plan[i].q0;
    chunks[4 * i + 3] = plan[i].q1;
  }
  return IDX_OK;
}

namespace {

idx_status prefill_plan(const int32_t* sl, const int32_t* ql, int32_t num_reqs,
                        int64_t workspace_tokens, int64_t budget, std::vector<Chunk>* plan,
                        std::vector<int64_t>* qsl, int64_t* max_wr, int64_t* max_rows) {
  if (num_reqs < 0 || (num_reqs > 0 && (!sl || !ql)) || workspace_tokens < 0 || budget < 0)
    return IDX_ERR_INVALID_ARG;
  qsl->assign(num_reqs + 1, 0);
  for (int32_t r = 0; r < num_reqs; ++r) {
    if (ql[r] < 0 || sl[r] < 0 || ql[r] > sl[r]) return IDX_ERR_INVALID_ARG;
    (*qsl)[r + 1] = (*qsl)[r] + ql[r];
  }
  *plan = plan_chunks(sl, ql, num_reqs, workspace_tokens, budget);
  *max_wr = 0;
  *max_rows = 0;
  for (const Chunk& c : *plan) {
    int64_t lo, hi;
    const int64_t nw = chunk_work_rows(*qsl, c, &lo, &hi);
    *max_wr = std::max(*max_wr, nw);
    *max_rows = std::max(*max_rows, hi - lo);
  }
  return IDX_OK;
}

}  // namespace

idx_status indexer_prefill_workspace_bytes(const int32_t* seq_lens_host,
                                           const int32_t* query_lens_host, int32_t num_reqs,
                                           int32_t topk, int64_t workspace_tokens,
                                           int64_t logits_budget_bytes, size_t* bytes) {
  if (!bytes) return IDX_ERR_INVALID_ARG;
  if (topk < 1 || topk > IDX_MAX_TOPK) return IDX_ERR_UNSUPPORTED;
  std::vector<Chunk> plan;
  std::vector<int64_t> qsl;
  int64_t max_wr, max_rows;
  const idx_status st = prefill_plan(seq_lens_host, query_lens_host, num_reqs, workspace_tokens,
                                     logits_budget_bytes, &plan, &qsl, &max_wr, &max_rows);
  if (st != IDX_OK) return st;
  *bytes = ws_layout(max_wr, max_rows, kPrefillG, topk, score_streams(kPrefillG)).total;
  return IDX_OK;
}

}  // extern "C"

namespace {

idx_status prefill_common(const void* q, const float* weights, const uint8_t* index_cache,
                          int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                          int32_t bt_width, const int32_t* seq_lens,
                          const int32_t* query_start_loc, const int32_t* seq_lens_host,
                          const int32_t* query_lens_host, int32_t num_reqs, int32_t num_heads,
                          int32_t head_dim, int32_t topk, int64_t workspace_tokens,
                          int64_t logits_budget_bytes, int32_t* out_idx, void* workspace,
                          size_t workspace_bytes, uint32_t* dev_error, void* stream,
                          const ValuesOut* vo) {
  const bool values = vo != nullptr;
  if (values && !valid_values(vo)) return IDX_ERR_INVALID_ARG;
  idx_status st = check_common(q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                               num_heads, head_dim, topk);
  if (st != IDX_OK) return st;
  if (!seq_lens || !query_start_loc || !out_idx || !workspace || !aligned(workspace, 256))
    return IDX_ERR_INVALID_ARG;
  std::vector<Chunk> plan;
  std::vector<int64_t> qsl;
  int64_t max_wr, max_rows;
  if ((st = prefill_plan(seq_lens_host, query_lens_host, num_reqs, workspace_tokens,
                         logits_budget_bytes, &plan, &qsl, &max_wr, &max_rows)) != IDX_OK)
    return st;
  if (plan.empty()) return IDX_OK;
  const int nC = score_streams(kPrefillG);
  const WsLayout L = ws_layout(max_wr, max_rows, kPrefillG, topk, nC);
  if (workspace_bytes < L.total) return IDX_ERR_WORKSPACE;
  CUtensorMap map;
  if ((st = encode_cache_map(&map, index_cache, num_pages)) != IDX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  for (const Chunk& c : plan) {
    int64_t lo, hi;
    const int64_t nw = chunk_work_rows(qsl, c, &lo, &hi);
    if (nw == 0) continue;
    PrefillPrepArgs a{static_cast<const __nv_bfloat16*>(q), weights, seq_lens, query_start_loc,
                      c.r0, c.r1, lo, hi, static_cast<int32_t>(nw), topk, bt_width, out_idx,
                      dev_error, nC, 0};
    if (values) {
      a.out_val = vo->out_val;
      a.compress_ratio = vo->compress_ratio;
      a.dcp_rank = vo->rank;
      a.dcp_world = vo->world;
      a.dcp_interleave = vo->interleave;
    }
    if ((st = launch_prefill_prep(a, ws, L, s)) != IDX_OK) return st;
    ScoreParams p{};
    p.cache = index_cache;
    p.num_pages = num_pages;
    p.block_table = block_table;
    p.bt_stride = bt_stride;
    p.wr = reinterpret_cast<const WorkRow*>(ws + L.wr);
    p.wr_tile_start = reinterpret_cast<const int32_t*>(ws + L.wr_tile_start);
    p.cta_row = reinterpret_cast<const int32_t*>(ws + L.cta_row);
    p.cta_tile = reinterpret_cast<const int32_t*>(ws + L.cta_tile);
    p.row_ctas = reinterpret_cast<const int2*>(ws + L.row_ctas);
    p.num_wr = static_cast<int32_t>(nw);
    p.row_len = reinterpret_cast<const int32_t*>(ws + L.row_len);
    p.q8 = ws + L.q8;
    p.wprime = reinterpret_cast<const float*>(ws + L.wprime);
    p.seg_counter = reinterpret_cast<int32_t*>(ws + L.seg_counter);
    p.slot_key = reinterpret_cast<uint32_t*>(ws + L.slot_key);
    p.slot_idx = reinterpret_cast<int32_t*>(ws + L.slot_idx);
    p.slot_cap = candidate_capacity(kPrefillG);
    p.seg_cum = reinterpret_cast<uint32_t*>(ws + L.seg_cum);
    p.row_hist = reinterpret_cast<uint32_t*>(ws + L.row_hist);
    p.wait_ns = g_wait_ns;
    p.out_idx = out_idx;
    p.out_row_base = lo;
    p.topk = topk;
    p.short_len = values ? 0 : topk;
    p.out_val = values ? vo->out_val : nullptr;
    p.dev_error = dev_error;
    size_t tb = 0;
    p.trace = trace_buffer(&tb);
    if (tb < sizeof(uint64_t) * kTrSlots * static_cast<size_t>(nC)) p.trace = nullptr;
    if ((st = timed_score(kPrefillG, false, p, map, s)) != IDX_OK) return st;
    if (values && vo->world > 1 &&
        (st = launch_dcp_globalise(out_idx + lo * topk, (hi - lo) * topk, vo->rank, vo->world,
                                   vo->interleave, s)) != IDX_OK)
      return st;
  }
  return IDX_OK;
}

}  // namespace

extern "C" {

idx_status indexer_prefill_topk(const void* q, const float* weights, const uint8_t* index_cache,
                                int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                                int32_t bt_width, const int32_t* seq_lens,
                                const int32_t* query_start_loc, const int32_t* seq_lens_host,
                                const int32_t* query_lens_host, int32_t num_reqs,
                                int32_t num_heads, int32_t head_dim, int32_t topk,
                                int64_t workspace_tokens, int64_t logits_budget_bytes,
                                int32_t* out_idx, void* workspace, size_t workspace_bytes,
                                uint32_t* dev_error, void* stream) {
  return prefill_common(q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                        seq_lens, query_start_loc, seq_lens_host, query_lens_host, num_reqs,
                        num_heads, head_dim, topk, workspace_tokens, logits_budget_bytes, out_idx,
                        workspace, workspace_bytes, dev_error, stream, nullptr);
}

idx_status indexer_prefill_topk_values(
    const void* q, const float* weights, const uint8_t* index_cache, int64_t num_pages,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width, const int32_t* seq_lens,
    const int32_t* query_start_loc, const int32_t* seq_lens_host, const int32_t* query_lens_host,
    int32_t num_reqs, int32_t num_heads, int32_t head_dim, int32_t topk, int32_t compress_ratio,
    int32_t dcp_rank, int32_t dcp_world, int32_t dcp_interleave, int64_t workspace_tokens,
    int64_t logits_budget_bytes, int32_t* out_idx, float* out_val, void* workspace,
    size_t workspace_bytes, uint32_t* dev_error, void* stream) {
  if (!out_val) return IDX_ERR_INVALID_ARG;
  const ValuesOut vo{out_val, compress_ratio, dcp_rank, dcp_world, dcp_interleave};
  return prefill_common(q, weights, index_cache, num_pages, block_table, bt_stride, bt_width,
                        seq_lens, query_start_loc, seq_lens_host, query_lens_host, num_reqs,
                        num_heads, head_dim, topk, workspace_tokens, logits_budget_bytes, out_idx,
                        workspace, workspace_bytes, dev_error, stream, &vo);
}

}  // extern "C"
