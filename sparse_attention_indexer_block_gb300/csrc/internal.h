// Internal launch interfaces shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

#include <utility>

namespace saib {

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
  int32_t* seg_counter;          // [num_wr] finished segments per work row
  uint32_t* slot_key;            // [nslots, G, slot_cap] candidate keys of finished segments
  int32_t* slot_idx;             // [nslots, G, slot_cap] their token indices
  int32_t* slot_count;           // [nslots, G]
  int32_t* slot_thrbin;          // [nslots, G] row-histogram bin of the segment's final threshold
  int32_t slot_cap;              // entries per slot (the candidate buffer's capacity)
  uint32_t* row_hist;            // [nC, G, 1024] histograms of split work rows (zeroed by prep)
  int32_t* out_idx;              // [*, topk] (row = out_row_base + token row)
  int64_t out_row_base;
  int32_t topk;
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
  kTrFinEmitNs, kTrFinPublishNs, kTrMergeTailNs, kTrSlots = 40
};

// Candidate-buffer capacity per token row of the score/select kernel for work
// rows of G tokens; a published segment slot holds up to this many entries.
constexpr int candidate_capacity(int G) { return G == 1 ? 3072 : (G == 2 ? 4096 : 2560); }

// Workspace carve-up shared by decode and prefill.
struct WsLayout {
  size_t wr, wr_tile_start, row_len, seg_counter, slot_count, q8, wprime, slot_key, slot_idx;
  size_t row_hist, row_hist_words, cta_row, slot_thrbin, cta_tile, row_vs, row_ctas;
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

idx_status launch_quantize_plain(const __nv_bfloat16* q, const float* w, int64_t rows,
                                 uint8_t* q8, float* wprime, cudaStream_t s);

struct DecodePrepArgs {
  const __nv_bfloat16* q;
  const float* w;
  const int32_t* row_seq_lens;
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
};
idx_status launch_prefill_prep(const PrefillPrepArgs& a, uint8_t* ws, const WsLayout& L,
                               cudaStream_t s);

// G = token rows per work row (1, 2 or 4); logits = write logits instead of selecting.
// Thread-local trace buffer set by indexer_trace_buffer (nullptr = off).
uint64_t* trace_buffer(size_t* bytes);

idx_status launch_score(int G, bool logits, const ScoreParams& p, const CUtensorMap& map,
                        int num_ctas, cudaStream_t s);

// CTAs per SM the score/select kernel runs with for work rows of G tokens.
int score_ctas_per_sm(int G);

// CTAs of one score/select launch on the current device.
inline int score_ctas(int G) { return device_sm_count() * score_ctas_per_sm(G); }

}  // namespace saib
