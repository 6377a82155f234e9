// Internal launch interfaces shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

#include <utility>

namespace saib {

// Records a failed CUDA call's error for indexer_last_cuda_error (this host
// thread) and maps it to a status.
void record_cuda_error(cudaError_t e);
inline idx_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return IDX_OK;
  record_cuda_error(e);
  return IDX_ERR_CUDA;
}

// Launches `kernel` on `stream` with programmatic stream serialization (the
// kernel calls pdl_wait() before it reads anything earlier work wrote).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Row histogram of a split row: counts of its candidates' top 10 key bits.
constexpr int kRowHistBins = 1024;

// Slot of the segment that stream v holds of a split work row: only a
// stream's first and last work rows can be split, so two slots per stream
// (the first row's, and the last one's when it differs).
__host__ __device__ __forceinline__ int64_t segment_slot(int v, bool first_row) {
  return 2 * static_cast<int64_t>(v) + (first_row ? 0 : 1);
}

// Keys a rank of a key-sharded (decode context parallel) cache holds of a
// sequence of L keys, when the sequence is dealt to `world` ranks in runs of
// `interleave` tokens (token t on rank (t / interleave) % world): base +
// min(max(rem - rank * interleave, 0), interleave), base = L / interleave /
// world * interleave, rem = L - base * world (INDEXER page,
// _build_prefill_chunk_metadata_kernel, DCP branch). Negative L is returned
// as it is (the caller's validation reports it).
__host__ __device__ __forceinline__ int64_t dcp_local_len(int64_t L, int rank, int world,
                                                          int interleave) {
  if (world <= 1 || L < 0) return L;
  const int64_t base = L / interleave / world * interleave;
  const int64_t rem = L - base * world;
  const int64_t r = rem - static_cast<int64_t>(rank) * interleave;
  return base + (r < 0 ? 0 : (r > interleave ? interleave : r));
}

// Cache entries a row of L tokens sees when the cache holds one entry per
// `ratio` tokens (INDEXER page: DeepseekV4's compress_ratio divides the
// per-token seq_lens; _build_prefill_chunk_metadata_kernel divides each
// query's key count by COMPRESS_RATIO), then this rank's share of them.
__host__ __device__ __forceinline__ int64_t index_key_count(int64_t L, int ratio, int rank,
                                                            int world, int interleave) {
  if (L < 0) return L;
  return dcp_local_len(ratio > 1 ? L / ratio : L, rank, world, interleave);
}


// Everything the score/select kernel reads, for one launch.
struct ScoreParams {
  const uint8_t* cache;
  int64_t num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  const WorkRow* wr;
  const int32_t* wr_tile_start;  // [num_wr + 1], exclusive prefix of tiles per work row
  const int32_t* cta_row;        // [grid] work row holding each CTA's first tile
  const int32_t* cta_tile;       // [grid + 1] first tile of each CTA (cost-balanced split)
  const int2* row_ctas;          // [num_wr] first and last CTA holding each work row's tiles
  int32_t num_wr;
  const int32_t* row_len;        // [rows] validated key count per token row
  const uint8_t* q8;             // [rows, 8192] swizzled fp8 images of q
  const float* wprime;           // [rows, 64] w * sq
  int32_t* seg_counter;          // [num_wr] published segments per work row (zeroed by prep)
  uint32_t* slot_key;            // [nslots, G, slot_cap] candidate keys of split-row segments,
                                 // sorted by row bin, highest first
  int32_t* slot_idx;             // [nslots, G, slot_cap] their token indices
  uint32_t* seg_cum;             // [nslots, G, 1024] entries of each slot at or above every row bin
  int32_t slot_cap;              // entries per slot (the candidate buffer's capacity)
  uint32_t* row_hist;            // [nsplit, G, 1024] histograms of split work rows (zeroed by prep)
  uint64_t wait_ns;              // give-up time of every pipeline wait
  int32_t* out_idx;              // [*, topk] (row = out_row_base + token row)
  int64_t out_row_base;
  int32_t topk;
  // Top-k mode selects rows of more than short_len keys: topk (shorter rows
  // are written by the prep kernel), or 0 when out_val is set.
  int32_t short_len;
  float* out_val;                // nullable: [*, topk] logit of each output index, -inf if none
  float* out_logits;             // logits mode only
  int64_t ld_logits;
  uint32_t* dev_error;
  uint64_t* trace;               // optional per-CTA timestamps (kTraceSlots per CTA)
};

// Per-CTA trace slots (ns from %globaltimer, or counts).
enum TraceSlot {
  kTrStart = 0, kTrFirstTma, kTrLastTma, kTrFirstMma, kTrLastMma, kTrFirstEpi, kTrLastEpi,
  kTrFinal, kTrCompactNs, kTrCompactN, kTrMergeNs, kTrMergeN, kTrEnd, kTrTiles, kTrFinalizeNs,
  kTrEndEpi, kTrMergeFallback, kTrMergeUnion, kTrMergeCut, kTrMergeSegs, kTrSeen, kTrMergeCutNs, kTrMergeLoadNs, kTrMergeRadixNs, kTrCompactRadixNs,
  kTrRadixHistNs, kTrRadixBucketNs, kTrRadixPasses, kTrEpiWaitCyc, kTrEpiLdCyc,
  kTrEpiMathCyc, kTrEpiVoteCyc, kTrEpiSelCyc, kTrFinPackNs, kTrFinHistNs, kTrFinCutNs,
  kTrFinEmitNs, kTrFinPublishNs, kTrMergeTailNs, kTrSelWaitNs, kTrSelScanNs, kTrSelFinalNs,
  kTrSelRows, kTrSelLast, kTrSelList, kTrSelFallback, kTrRndLoadNs, kTrRndCutNs, kTrRndPassNs,
  kTrRndAtomicNs, kTrRndArriveNs, kTrRndListSize, kTrPassCountCyc, kTrPassScanCyc,
  kTrPassWriteCyc, kTrPassSyncCyc, kTrPickHistCyc, kTrPickScanCyc, kTrPickSplitCyc,
  kTrPickOutCyc, kTrSlots = 64
};

// Tile streams one CTA of the score/select kernel runs for work rows of G (1
// or 2) token rows: two for G = 1 (one epilogue group each), one for G = 2
// (one epilogue group per token row).
constexpr int score_streams_per_cta(int G) { return G == 1 ? 2 : 1; }

// Candidate-buffer capacity of one epilogue group (one token row); a published
// segment slot holds up to this many entries.
constexpr int candidate_capacity(int G) { return G == 1 ? 5120 : 6144; }

// Pipeline stages (128-key tiles in flight) of one CTA of the score/select
// kernel, over all its streams.
constexpr int score_stages(int G) { return G == 1 ? 6 : 4; }

// Split work rows (rows whose tiles several CTAs share) that one launch can
// have: each starts in a different CTA, and there is at most one per work row.
inline int64_t max_split_rows(int64_t num_wr, int num_ctas) {
  return num_wr < num_ctas ? num_wr : num_ctas;
}

// Workspace carve-up shared by decode and prefill.
struct WsLayout {
  size_t wr, wr_tile_start, row_len, seg_counter, seg_cum, q8, wprime, slot_key, slot_idx;
  size_t row_hist, row_hist_words, cta_row, cta_tile, row_vs, row_ctas;
  size_t total;
};
WsLayout ws_layout(int64_t num_wr, int64_t rows, int G, int topk, int num_ctas);

// Per-device facts and one-time setup (devices 0 .. kMaxDevices-1 are cached).
constexpr int kMaxDevices = 128;
int device_sm_count();
idx_status encode_cache_map(CUtensorMap* map, const uint8_t* cache, int64_t num_pages);

// Kernel launchers (return IDX_ERR_CUDA on a launch failure).
idx_status launch_expand(const int32_t* seq_lens, const int32_t* decode_lens, int32_t num_reqs,
                         int32_t next_n, const int32_t* bt, int64_t bt_stride, int32_t bt_width,
                         int32_t mode, int32_t* row_lens, int32_t* row_bt, int64_t out_stride,
                         int64_t num_out_rows, uint32_t* err, cudaStream_t s);

idx_status launch_insert_keys(const __nv_bfloat16* k, const int64_t* slots, int64_t n,
                              uint8_t* cache, int64_t num_pages, uint32_t* err, cudaStream_t s);

// Test hook: the insert's quotient and the IEEE quotient of n pairs.
idx_status launch_divide_check(const float* a, const float* b, int64_t n, float* fast, float* ieee,
                               cudaStream_t s);

idx_status launch_quantize_plain(const __nv_bfloat16* q, const float* w, int64_t rows,
                                 uint8_t* q8, float* wprime, cudaStream_t s);

struct DecodePrepArgs {
  const __nv_bfloat16* q;
  const float* w;
  const int32_t* row_seq_lens;  // per token row, or nullptr: from seq_lens / decode_lens below
  int32_t num_reqs;
  int32_t next_n;
  int32_t topk;
  int32_t bt_width;
  int32_t score_all;  // logits mode: every row with len > 0 is scored
  int32_t* out_idx;   // causal fill target (nullable in logits mode)
  uint32_t* err;
  int32_t num_ctas;     // grid of the score/select launch that follows
  int32_t row_penalty;  // tiles of streaming time one work row's end costs its CTA
  // When CTAs stream long segments (>= 64 tiles each), a row end also restarts
  // a segment's drop threshold (more buffer cuts): the penalty grows by the
  // per-CTA tile share divided by this (0: no growth).
  int32_t row_penalty_div;
  const int32_t* seq_lens = nullptr;     // [num_reqs] (when row_seq_lens is nullptr)
  const int32_t* decode_lens = nullptr;  // [num_reqs]
  // Values mode (score_all set, top-k output): rows of 0 keys get -1 / -inf.
  float* out_val = nullptr;
  // Compressed and / or key-sharded cache: every row scores
  // index_key_count(its length) keys.
  int32_t compress_ratio = 1, dcp_rank = 0, dcp_world = 1, dcp_interleave = 1;
};
idx_status launch_decode_prep(const DecodePrepArgs& a, uint8_t* ws, const WsLayout& L,
                              cudaStream_t s);

struct PrefillPrepArgs {
  const __nv_bfloat16* q;
  const float* w;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int32_t req_begin, req_end;  // requests of the chunk
  int64_t row_lo, row_hi;      // global query rows of the chunk
  int32_t num_wr;              // work rows of the chunk (host count)
  int32_t topk;
  int32_t bt_width;
  int32_t* out_idx;
  uint32_t* err;
  int32_t num_ctas;     // grid of the score/select launch that follows
  int32_t row_penalty;  // tiles of streaming time one work row's end costs its CTA
  // Values mode: every query with > 0 keys is scored, queries of 0 keys get
  // -1 / -inf; compressed and / or key-sharded cache as in DecodePrepArgs.
  float* out_val = nullptr;
  int32_t compress_ratio = 1, dcp_rank = 0, dcp_world = 1, dcp_interleave = 1;
};
idx_status launch_prefill_prep(const PrefillPrepArgs& a, uint8_t* ws, const WsLayout& L,
                               cudaStream_t s);

// G = token rows per work row (1 or 2); logits = write logits instead of selecting;
// mx = the cache holds MXFP4 keys (4352-byte pages; G = 1 only).
// Thread-local trace buffer set by indexer_trace_buffer (nullptr = off).
uint64_t* trace_buffer(size_t* bytes);

idx_status launch_score(int G, bool logits, bool mx, const ScoreParams& p, const CUtensorMap& map,
                        int num_ctas, cudaStream_t s);

// Everything the split-row selection kernel reads, for one launch (after the
// score/select launch, on the same workspace).
struct RowSelectParams {
  const WorkRow* wr;
  const int32_t* wr_tile_start;
  const int32_t* cta_row;        // [streams] work row holding each stream's first tile
  const int2* row_ctas;          // [num_wr] first and last stream of each work row
  const int32_t* row_len;
  const int32_t* seg_counter;
  const uint32_t* slot_key;
  const int32_t* slot_idx;
  const uint32_t* seg_cum;
  int32_t slot_cap;
  const uint32_t* row_hist;
  int32_t num_wr;
  int32_t streams;               // tile streams the score/select launch was planned over
  int32_t G;
  int32_t topk;
  int32_t* out_idx;
  float* out_val;                // nullable: the selected keys' logits; rows of <= k keys are
                                 // then selected here too (all their keys)
  int64_t out_row_base;
  uint32_t* dev_error;
  uint64_t wait_ns;
  int32_t stall;                 // test hook: wait for a segment that never comes (0)
  uint64_t* trace;               // optional: kSelTrSlots per CTA
};
// Trace slots of one split-row selection CTA (ns from %globaltimer, or counts).
enum SelTraceSlot {
  kSelTrEntry = 0, kSelTrWaited, kSelTrPrefix, kSelTrCut0, kSelTrEmit0, kSelTrEnd, kSelTrCand,
  kSelTrBin0, kSelTrBin1, kSelTrPath, kSelTrSegs, kSelTrSlots = 16
};
// One CTA per (possible split row, token row):
// max_split_rows(num_wr, streams) * G CTAs.
idx_status launch_row_select(const RowSelectParams& p, int grid, cudaStream_t s);

// Key-sharded decode: rank-local key counts, local-to-global output indices,
// and the merge of the ranks' (logit, index) candidates.
idx_status launch_key_counts(const int32_t* lens, int64_t n, int ratio, int rank, int world,
                             int interleave, int32_t* out, cudaStream_t s);
idx_status launch_dcp_globalise(int32_t* idx, int64_t n, int rank, int world, int interleave,
                                cudaStream_t s);
idx_status launch_dcp_merge(const float* val, const int32_t* idx, int world, int64_t rows,
                            int topk, int32_t* out_idx, float* out_val, cudaStream_t s);

// The score/select kernel runs one CTA per SM, each CTA
// score_streams_per_cta(G) tile streams: the work split is planned over
// score_streams(G) ranges and the launch has score_grid() CTAs.
inline int score_grid() { return device_sm_count(); }
inline int score_streams(int G) { return score_streams_per_cta(G) * device_sm_count(); }

}  // namespace saib
