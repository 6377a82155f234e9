/*
 * indexer.h — C ABI of the GB300 (sm_103a) sparse-attention indexer.
 *
 * The indexer picks, for every query token, the k (<= 2048) cached keys that a
 * sparse attention step will attend to:
 *
 *     logit[t, s] = sum_h w[t, h] * ReLU(scale_s * (q[t, h] . k_s)),   s < len_t
 *     out[t]      = indices of the k largest logit[t, s]      (len_t >  k)
 *     out[t]      = [0, 1, ..., len_t - 1, -1, ...]           (len_t <= k)
 *
 * over 64 index heads of dimension 128, reading the keys from a paged fp8 e4m3
 * cache through a block table.
 *
 * Sources (web pages, by title and section):
 *  [RUNNER]  "vllm.models.minimax_m3.amd.mono.runner" — token_rows: a request
 *            of q query tokens becomes q rows, token j seeing
 *            seq_len - (q - 1 - j) keys; StepTables: block table int32
 *            [rows, width], seq_lens int32 [rows]; the indexer's
 *            topk_blocks / init_blocks / local_blocks (names only).
 *  [INDEXER] "recipes/docker-images/glm52-nf3-hybrid/overlay/vllm/v1/attention/
 *            backends/mla/indexer.py" — DeepseekV32IndexerBackend
 *            (64-token blocks, cache shape (num_blocks, block_size, head_size),
 *            head sizes 32/64/128), get_max_prefill_buffer_size (128 fp8 bytes +
 *            4 scale bytes per entry), DeepSeekV32IndexerDecodeMetadata (2-D
 *            (B, next_n) per-token seq_lens [b, j] = L_b - next_n + j + 1),
 *            _prepare_decode_tensors (flatten path: worked example with
 *            seq_lens [10, 7, 12, 0], decode_lens [3, 1, 4, 0]),
 *            split_indexer_prefill_chunks (M*N logits-budget chunking),
 *            _build_prefill_chunk_metadata_kernel (query i of a request sees
 *            keys [0, seq_len - query_len + 1 + i); with COMPRESS_RATIO and
 *            its DCP branch, the compressed and key-sharded counts);
 *            use_fp4_indexer_cache (the MXFP4 index cache).
 *  [GLM5]    "vllm.models.glm5next.common.sparse_indexer" — _decode_topk_seq_lens
 *            (padded grid rows get seq_len 0), _fill_short_decode_causal_indices
 *            (exact causal rows when every key would be selected),
 *            _gather_workspace_shapes (fp8 values + 4-byte fp32 scale per token;
 *            its MXFP4 branch), kv_cache_as_quant_view (the MXFP4 token
 *            stride), pool_topk / expand_pools_and_append_tail (names only).
 *  The scoring formula and k = 2048 are the method's statement; the pages only
 *  name the kernels (fp8_fp4_paged_mqa_logits and "the topk kernels").
 *
 * Data layout (all device memory unless a name ends in _host):
 *  index cache  uint8 [num_pages, 8448]; page p holds 64 tokens as
 *               [64 x 128 fp8 e4m3 codes][64 x fp32 scale] (the pages fix 132
 *               bytes per token but not their order inside a page; values
 *               first keeps every 128-byte key row 16-byte aligned for TMA).
 *               Base address 16-byte aligned. Scales must be >= 0 and finite.
 *  block_table  int32 [num_reqs, bt_width] with row stride bt_stride (elements);
 *               entry c is the page holding tokens [64c, 64c + 64).
 *  q            bf16 [rows, 64, 128] contiguous; weights fp32 [rows, 64].
 *  out_idx      int32 [rows, topk] contiguous; request-relative token positions.
 *               Rows with len > topk hold the selected set in no particular
 *               order; rows with len <= topk hold the exact causal row.
 *
 * Conventions:
 *  - The caller owns every buffer; the library never allocates device memory,
 *    never synchronises the stream and never reads results back. Every call is
 *    enqueued on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *  - Host-detectable problems return a status before anything is enqueued.
 *  - Device-detectable problems (a block id outside [0, num_pages), a row
 *    length < 0 or > bt_width*64, a pipeline wait that gave up) OR a bit into
 *    *dev_error (nullable, a uint32 the caller zeroes) and never trap; the
 *    affected rows' outputs are then unspecified. Bad lengths are clamped.
 *  - Workspaces are caller-provided scratch of the size the *_workspace_bytes
 *    query returns for the current device; contents need no initialisation and
 *    are overwritten. Calls that share a workspace must not overlap.
 *  - Kernels are launched with programmatic dependent launch: a kernel may be
 *    scheduled while the previous work in the stream finishes, but it waits
 *    for that work to complete before it reads or writes any memory, so the
 *    stream's ordering is what the caller sees.
 *  - A top-k call is three launches: the prep kernel (row lengths, q
 *    quantisation, the work split), the score/select kernel (one CTA per SM)
 *    and the selection of rows whose keys several CTAs scored (one CTA per
 *    such row and token, after the score/select kernel has completed). No CTA
 *    waits on another; a CTA's own pipeline waits give up after 2 s and set
 *    IDX_DEV_TIMEOUT.
 *  - [INDEXER] _build_prefill_chunk_metadata_kernel (COMPRESS_RATIO, its DCP branch) also defines
 *    the compressed and key-sharded (decode context parallel) calls below.
 */
#ifndef SAIB_INDEXER_H
#define SAIB_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  IDX_OK = 0,
  IDX_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad alignment, bad mode */
  IDX_ERR_UNSUPPORTED = 2,   /* heads != 64, head_dim != 128, topk outside [1, 2048], ... */
  IDX_ERR_WORKSPACE = 3,     /* workspace smaller than the size query returned */
  IDX_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  IDX_ERR_CAPACITY = 5       /* an output array is too small (chunk list) */
} idx_status;

/* Bits of the device error word. */
#define IDX_DEV_BAD_BLOCK 1u /* a block-table entry outside [0, num_pages) was skipped */
#define IDX_DEV_BAD_LEN 2u   /* a row length < 0 or > bt_width * 64 was clamped */
#define IDX_DEV_TIMEOUT 4u   /* a pipeline wait gave up; the kernel returned early */
#define IDX_DEV_OVERFLOW 8u  /* more token rows than the output holds (flatten mode) */
#define IDX_DEV_INTERNAL 16u /* the split-row selection's counts disagreed (a library bug) */

#define IDX_NUM_HEADS 64
#define IDX_HEAD_DIM 128
#define IDX_PAGE_TOKENS 64
#define IDX_PAGE_BYTES 8448
#define IDX_MAX_TOPK 2048
#define IDX_DCP_MAX_CANDIDATES 16384 /* dcp_world * topk of indexer_dcp_merge */
#define IDX_MXFP4_PAGE_BYTES 4352    /* 64 entries x (64 B packed e2m1 + 4 ue8m0 scales) */

/* Human-readable name of a status code (static string). */
const char* indexer_status_string(idx_status status);

/* The CUDA error behind the last IDX_ERR_CUDA this host thread got from a
 * launch or CUDA call of the library (static string; "no error" if none). */
const char* indexer_last_cuda_error(void);

/*
 * Decode row expansion ([INDEXER] _prepare_uniform_decode_kernel and the
 * variable-length flatten branch of _prepare_decode_tensors; [RUNNER]
 * token_rows; [GLM5] _decode_topk_seq_lens).
 *
 * Inputs: seq_lens int32 [num_reqs] (keys of the request including its new
 * tokens), decode_lens int32 [num_reqs] (new tokens, 0 <= d <= next_n for
 * mode 0), block_table as above.
 * mode 0 (padded grid): row b*next_n + j gets len = L_b - d_b + j + 1 for
 *   j < d_b and 0 otherwise; num_out_rows must be >= num_reqs*next_n, and
 *   rows past num_reqs*next_n are left as they are.
 * mode 1 (flatten): the d_b tokens of request b take consecutive rows starting
 *   at sum_{b' < b} d_b' with the same len; rows from sum d_b up to
 *   num_out_rows get len 0; more tokens than num_out_rows sets
 *   IDX_DEV_OVERFLOW and drops the excess.
 * row_block_table (nullable) int32 [num_out_rows, >= bt_width], row stride
 *   out_stride: each token row gets its request's first bt_width entries;
 *   in mode 1 rows past the last token get column 0 set to 0 (the rest is
 *   left as it was).
 */
idx_status indexer_expand_decode_rows(const int32_t* seq_lens, const int32_t* decode_lens,
                                      int32_t num_reqs, int32_t next_n,
                                      const int32_t* block_table, int64_t bt_stride,
                                      int32_t bt_width, int32_t mode, int32_t* row_seq_lens,
                                      int32_t* row_block_table, int64_t out_stride,
                                      int64_t num_out_rows, uint32_t* dev_error, void* stream);

/*
 * Per (row, head) fp8 quantisation of q, the reading this library takes for
 * feeding bf16 q to an fp8 e4m3 MMA (the pages name an "fp8_fp4" paged MQA
 * logits kernel but not its q path): amax = max_d |q|, inv = 448 / amax
 * (fp32, correctly rounded), q8 = e4m3 round-to-nearest-even, saturating, of
 * the fp32 product q * inv; sq = amax / 448; weights_scaled = w * sq. A head
 * with amax == 0 gets q8 = 0 and weights_scaled = 0.
 * q bf16 [rows, 64, 128]; weights fp32 [rows, 64]; q_fp8 uint8 [rows, 64, 128];
 * weights_scaled fp32 [rows, 64]. The decode and prefill calls run this same
 * step internally; it is exposed for inspection and tests.
 */
idx_status indexer_quantize_q(const void* q, const float* weights, int64_t num_rows,
                              int32_t num_heads, int32_t head_dim, uint8_t* q_fp8,
                              float* weights_scaled, void* stream);

/*
 * Index-key cache insert: the step that fills the paged cache the decode and
 * prefill calls read ([INDEXER] DeepseekV32IndexerMetadata.slot_mapping gives
 * every new token its cache slot; get_max_prefill_buffer_size and [GLM5]
 * _gather_workspace_shapes fix 128 fp8 values + one fp32 scale per token; the
 * insert kernel itself is not shown on the pages). Token i's keys
 * k bf16 [num_tokens, 128] are quantised with the token's own scale
 * scale = amax / 448 (amax = max_d |k|, fp32, correctly rounded) into codes
 * e4m3_rne_satfinite(k / scale) (fp32, correctly rounded quotient) and written
 * to slot s = slot_mapping[i] (int64): page s / 64, token s % 64, in the page
 * layout above. A negative slot is padding and skipped; a slot >= num_pages*64
 * ORs IDX_DEV_BAD_BLOCK and is skipped; a token with amax == 0 gets zero codes
 * and scale 0. Two tokens with the same slot race. k 8-byte aligned,
 * slot_mapping 8-byte aligned, index_cache 16-byte aligned.
 */
idx_status indexer_insert_keys(const void* k, const int64_t* slot_mapping, int64_t num_tokens,
                               int32_t head_dim, uint8_t* index_cache, int64_t num_pages,
                               uint32_t* dev_error, void* stream);

/* Bytes of workspace indexer_decode_topk / indexer_decode_logits need for
 * num_reqs requests of next_n rows each, on the current CUDA device. */
idx_status indexer_decode_workspace_bytes(int32_t num_reqs, int32_t next_n, int32_t topk,
                                          size_t* bytes);

/*
 * Decode top-k ([INDEXER] DeepSeekV32IndexerDecodeMetadata: the logits and top-k
 * kernels see a (B, next_n) grid of per-token seq_lens; [GLM5]
 * _fill_short_decode_causal_indices for rows with len <= topk).
 *
 * Token rows form a [num_reqs, next_n] grid: row b*next_n + j is token j of
 * request b and reads block-table row b. row_seq_lens int32 [num_reqs*next_n]
 * is the per-token key count (from indexer_expand_decode_rows; 0 = padded row,
 * whose output is all -1). next_n is 1 or 2 (for longer speculative runs use
 * mode 1 of the expansion with next_n = 1 and its row block table).
 * num_heads must be 64, head_dim 128, 1 <= topk <= 2048.
 * Writes out_idx [num_reqs*next_n, topk]. No logits row is written to memory.
 */
idx_status indexer_decode_topk(const void* q, const float* weights, const uint8_t* index_cache,
                               int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                               int32_t bt_width, const int32_t* row_seq_lens, int32_t num_reqs,
                               int32_t next_n, int32_t num_heads, int32_t head_dim, int32_t topk,
                               int32_t* out_idx, void* workspace, size_t workspace_bytes,
                               uint32_t* dev_error, void* stream);

/*
 * indexer_decode_topk with the row expansion folded in ([RUNNER] token_rows,
 * [INDEXER] DeepSeekV32IndexerDecodeMetadata: token j of a request with
 * d = decode_lens[b] new tokens and L = seq_lens[b] keys sees L - d + j + 1
 * keys; rows j >= d of the [num_reqs, next_n] grid are padding, length 0).
 * The same lengths indexer_expand_decode_rows (mode 0) writes, computed by
 * the launch's first kernel instead of a separate one. seq_lens, decode_lens
 * int32 [num_reqs] on the device; other arguments, the workspace size and the
 * results as indexer_decode_topk.
 */
idx_status indexer_decode_topk_from_lens(const void* q, const float* weights,
                                         const uint8_t* index_cache, int64_t num_pages,
                                         const int32_t* block_table, int64_t bt_stride,
                                         int32_t bt_width, const int32_t* seq_lens,
                                         const int32_t* decode_lens, int32_t num_reqs,
                                         int32_t next_n, int32_t num_heads, int32_t head_dim,
                                         int32_t topk, int32_t* out_idx, void* workspace,
                                         size_t workspace_bytes, uint32_t* dev_error,
                                         void* stream);

/*
 * Introspection of the on-device work split (for tests): where, inside a
 * decode workspace for (num_reqs, next_n, topk) on the current device, the
 * prep kernel leaves the plan the score/select kernel follows, as byte
 * offsets into the workspace:
 *   offsets[0] wr_tile_start int32 [num_reqs + 1]: first 128-key tile of each
 *              request (the tile sequence is the requests' tiles in order);
 *              entry num_reqs is the total T
 *   offsets[1] cta_tile int32 [min(grid, T) + 1]: CTA c streams tiles
 *              [cta_tile[c], cta_tile[c + 1])
 *   offsets[2] row_ctas int32 pairs [num_reqs]: first and last CTA holding a
 *              request's tiles ((0, -1) for a request with none)
 *   offsets[3] cta_row int32 [grid]: the request holding CTA c's first tile
 * *grid gets the launch's CTA count; penalty[0..1] the row-end penalty in
 * tiles and its growth divisor (the split charges a CTA that finishes a
 * request inside its range penalty[0] + (T / min(grid, T)) / penalty[1] extra
 * tiles when that share is >= 64, else penalty[0]). Host only; no device
 * work. The arrays are valid after an indexer_decode_topk call on the
 * workspace until the next call.
 */
idx_status indexer_debug_decode_plan(int32_t num_reqs, int32_t next_n, int32_t topk,
                                     int64_t* offsets, int32_t* grid, int32_t* penalty);

/*
 * The decode logits themselves, from the same quantisation, page gather and
 * tensor-core scoring as indexer_decode_topk (for parity checks): for every
 * token row t and key s < len_t writes out_logits[t * ld_logits + s]; other
 * entries are left untouched. Same arguments as indexer_decode_topk (topk is
 * only validated).
 */
idx_status indexer_decode_logits(const void* q, const float* weights, const uint8_t* index_cache,
                                 int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                                 int32_t bt_width, const int32_t* row_seq_lens, int32_t num_reqs,
                                 int32_t next_n, int32_t num_heads, int32_t head_dim,
                                 int32_t topk, float* out_logits, int64_t ld_logits,
                                 void* workspace, size_t workspace_bytes, uint32_t* dev_error,
                                 void* stream);

/*
 * Decode top-k over an MXFP4 index cache ([GLM5] _gather_workspace_shapes, its
 * MXFP4 branch: head_dim / 2 bytes of packed mxfp4 values and head_dim /
 * MXFP4_BLOCK_SIZE ue8m0 scale bytes per token; kv_cache_as_quant_view: that
 * 68-byte token stride inside a page; [INDEXER] the use_fp4_indexer_cache
 * switch of the metadata builder).
 * index_cache uint8 [num_pages, 4352]: page p holds 64 token entries back to
 * back; an entry is 64 bytes of e2m1 codes (element 2i in the low nibble of
 * byte i, 2i + 1 in the high one) then 4 ue8m0 bytes (block b scales elements
 * 32b .. 32b + 31 by 2^(E_b - 127)); the key value of element d is
 * e2m1(code_d) * 2^(E_{d/32} - 127) (E = 255, NaN, must not occur). Base
 * address 16-byte aligned. Other arguments, the workspace size and the
 * results as indexer_decode_topk; next_n must be 1 (IDX_ERR_UNSUPPORTED
 * otherwise). The keys are re-encoded on chip for the fp8 tensor cores with
 * one power-of-two scale per key: exact for every block within 2^11 of the
 * key's largest block, smaller blocks rounded to e4m3.
 */
idx_status indexer_decode_topk_mxfp4(const void* q, const float* weights,
                                     const uint8_t* index_cache, int64_t num_pages,
                                     const int32_t* block_table, int64_t bt_stride,
                                     int32_t bt_width, const int32_t* row_seq_lens,
                                     int32_t num_reqs, int32_t next_n, int32_t num_heads,
                                     int32_t head_dim, int32_t topk, int32_t* out_idx,
                                     void* workspace, size_t workspace_bytes, uint32_t* dev_error,
                                     void* stream);

/* The logits of indexer_decode_topk_mxfp4 (for parity checks), written like
 * indexer_decode_logits's. */
idx_status indexer_decode_logits_mxfp4(const void* q, const float* weights,
                                       const uint8_t* index_cache, int64_t num_pages,
                                       const int32_t* block_table, int64_t bt_stride,
                                       int32_t bt_width, const int32_t* row_seq_lens,
                                       int32_t num_reqs, int32_t next_n, int32_t num_heads,
                                       int32_t head_dim, int32_t topk, float* out_logits,
                                       int64_t ld_logits, void* workspace, size_t workspace_bytes,
                                       uint32_t* dev_error, void* stream);

/*
 * Compressed and key-sharded caches ([INDEXER] _build_prefill_chunk_metadata_kernel
 * with COMPRESS_RATIO and its DCP_WORLD_SIZE > 1 branch; the DeepseekV4
 * decode metadata divides the per-token seq_lens by compress_ratio):
 *  - a compressed cache holds one entry per compress_ratio tokens C, so a
 *    row of L tokens sees L / C entries (integer division);
 *  - a key-sharded (decode context parallel) cache deals the entries of a
 *    sequence to dcp_world ranks in runs of dcp_interleave (entry e to rank
 *    (e / I) % W, as that rank's next local entry), so rank r holds, of n
 *    entries, base + min(max(rem - r * I, 0), I) with base = n / I / W * I
 *    and rem = n - base * W (I = dcp_interleave, W = dcp_world).
 * A rank's cache holds its local entries 0, 1, ... in its own pages. A row
 * then takes the top k over every rank's candidates: each rank runs
 * indexer_decode_topk_values (or indexer_prefill_topk_values) on its cache,
 * the ranks' outputs are gathered ([W, rows, topk] each, rank-major: what an
 * all-gather of them holds) and indexer_dcp_merge picks the k best.
 */

/*
 * Entry counts: key_counts[i] = rank dcp_rank's count of the entries a row of
 * row_seq_lens[i] tokens sees by the rules above (int32 [num_rows] each,
 * device; negative lengths are copied as they are). Rows of a plain
 * indexer_decode_topk over a compressed cache take these counts as their
 * row_seq_lens. compress_ratio >= 1, 1 <= dcp_world, 0 <= dcp_rank <
 * dcp_world, dcp_interleave >= 1, else IDX_ERR_INVALID_ARG.
 */
idx_status indexer_index_key_counts(const int32_t* row_seq_lens, int64_t num_rows,
                                   int32_t compress_ratio, int32_t dcp_rank, int32_t dcp_world,
                                   int32_t dcp_interleave, int32_t* key_counts, void* stream);

/*
 * Decode top-k with the selected logits, on one rank of a compressed and / or
 * key-sharded cache (compress_ratio = dcp_world = 1, dcp_rank 0: the plain
 * cache). Arguments as indexer_decode_topk (same workspace size), except:
 *  - row_seq_lens are the rows' token counts over the whole sequence; each row
 *    scores the rank's count of its entries (the rules above) from
 *    index_cache / block_table, the rank's own cache;
 *  - every row with at least one local key is scored and selected: a row of
 *    n <= topk local keys outputs all n (no causal shortcut: a merge needs
 *    their logits);
 *  - out_val float [num_reqs * next_n, topk] gets the logit of each output
 *    index (the indexer's score, as indexer_decode_logits computes it) and
 *    -inf where out_idx is -1;
 *  - out_idx holds global entry positions: local entry j of rank r is
 *    (j / I) * I * W + r * I + j % I. Entries are in no particular order.
 * IDX_ERR_INVALID_ARG for a null out_val or a ratio / rank / world /
 * interleave outside the ranges of indexer_index_key_counts.
 */
idx_status indexer_decode_topk_values(const void* q, const float* weights,
                                      const uint8_t* index_cache, int64_t num_pages,
                                      const int32_t* block_table, int64_t bt_stride,
                                      int32_t bt_width, const int32_t* row_seq_lens,
                                      int32_t num_reqs, int32_t next_n, int32_t num_heads,
                                      int32_t head_dim, int32_t topk, int32_t compress_ratio,
                                      int32_t dcp_rank, int32_t dcp_world, int32_t dcp_interleave,
                                      int32_t* out_idx, float* out_val, void* workspace,
                                      size_t workspace_bytes, uint32_t* dev_error, void* stream);

/*
 * Prefill top-k with the selected logits on one rank of a compressed and / or
 * key-sharded cache ([INDEXER] _build_prefill_chunk_metadata_kernel: query i
 * of a request of L tokens and Q queries sees (L - Q + 1 + i) / C entries,
 * then the rank's count of them). Arguments as indexer_prefill_topk (same
 * workspace size) plus compress_ratio / dcp_* (as indexer_decode_topk_values)
 * and out_val float [sum of query_lens, topk]; every query with at least one
 * entry is scored and selected (no causal shortcut), out_idx holds global
 * entry positions in no particular order, -1 / -inf in empty slots.
 */
idx_status indexer_prefill_topk_values(
    const void* q, const float* weights, const uint8_t* index_cache, int64_t num_pages,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width, const int32_t* seq_lens,
    const int32_t* query_start_loc, const int32_t* seq_lens_host, const int32_t* query_lens_host,
    int32_t num_reqs, int32_t num_heads, int32_t head_dim, int32_t topk, int32_t compress_ratio,
    int32_t dcp_rank, int32_t dcp_world, int32_t dcp_interleave, int64_t workspace_tokens,
    int64_t logits_budget_bytes, int32_t* out_idx, float* out_val, void* workspace,
    size_t workspace_bytes, uint32_t* dev_error, void* stream);

/*
 * Merge of the ranks' candidates: cand_val float / cand_idx int32
 * [dcp_world, num_rows, topk] (slab w = rank w's indexer_decode_topk_values
 * output; idx < 0 = empty). out_idx int32 [num_rows, topk] gets, per row, the
 * topk candidates with the largest values (any of several equal to the k-th),
 * in no particular order, -1 past the candidates when there are fewer;
 * out_val (nullable) float [num_rows, topk] their values (-inf past them).
 * dcp_world * topk <= IDX_DCP_MAX_CANDIDATES, else IDX_ERR_UNSUPPORTED. One
 * 1024-thread CTA per row; the candidates are read once.
 */
idx_status indexer_dcp_merge(const float* cand_val, const int32_t* cand_idx, int32_t dcp_world,
                             int64_t num_rows, int32_t topk, int32_t* out_idx, float* out_val,
                             void* stream);

/*
 * Block / pool selection over rows of logits ([RUNNER] the indexer's
 * topk_blocks, init_blocks, local_blocks; [GLM5] pool_topk and
 * expand_pools_and_append_tail: the pages give the names, the rules here are
 * this library's reading). Typically the logits are indexer_decode_logits's.
 *
 * indexer_block_topk: row r's len = row_lens[r] logits (logits[r * ld_logits
 * + s], s < len; len is clamped to [0, ld_logits]) are cut into
 * ceil(len / block_size) blocks (the last may be partial); a block's score is
 * its largest logit. The selection is the first init_blocks blocks, the last
 * local_blocks blocks and the topk_blocks highest-scoring others (any of
 * several equal to the last one taken); out_blocks [num_rows, out_cap] gets
 * them in ascending order (at most out_cap, -1 after them), out_counts
 * (nullable) [num_rows] how many. ceil(ld_logits / block_size) <= 16384,
 * else IDX_ERR_UNSUPPORTED. One 512-thread CTA per row.
 */
idx_status indexer_block_topk(const float* logits, int64_t ld_logits, const int32_t* row_lens,
                              int64_t num_rows, int32_t block_size, int32_t topk_blocks,
                              int32_t init_blocks, int32_t local_blocks, int32_t* out_blocks,
                              int32_t out_cap, int32_t* out_counts, void* stream);

/*
 * indexer_expand_pools: for row r, the token indices of the pools listed in
 * pools [num_rows, pools_cap] (the first pool_counts[r] entries, or all when
 * pool_counts is NULL), pool b being tokens [b * pool_size, (b + 1) *
 * pool_size), in list order, then the row's tail: tokens [floor(L / P) * P,
 * L) after its last complete pool (L = row_lens[r], P = pool_size). Entries
 * < 0 and pools that are not complete add nothing. out_idx [num_rows,
 * out_cap] (-1 after the tokens, which are cut at out_cap), out_counts
 * (nullable) their number.
 */
idx_status indexer_expand_pools(const int32_t* pools, int32_t pools_cap, const int32_t* pool_counts,
                                const int32_t* row_lens, int64_t num_rows, int32_t pool_size,
                                int32_t* out_idx, int32_t out_cap, int32_t* out_counts,
                                void* stream);

/*
 * Host-only prefill chunk plan ([INDEXER] split_indexer_prefill_chunks): pack
 * requests greedily while the summed key count N <= workspace_tokens and
 * (summed query count M) * N <= logits_budget_bytes / 4; a request that fits
 * alone in neither is taken by itself; cut each chunk's M queries into pieces
 * of max(1, (logits_budget_bytes / 4) / N) (all of them when N == 0; a chunk
 * with M == 0 yields no piece). Writes (req_begin, req_end, q_begin, q_end)
 * rows into chunks [max_chunks, 4] (q relative to the chunk's first query) and
 * the count into *num_chunks; IDX_ERR_CAPACITY if more are needed (then
 * *num_chunks holds the count required). Host pointers only.
 */
idx_status indexer_plan_prefill_chunks(const int32_t* seq_lens_host,
                                       const int32_t* query_lens_host, int32_t num_reqs,
                                       int64_t workspace_tokens, int64_t logits_budget_bytes,
                                       int32_t* chunks, int32_t max_chunks, int32_t* num_chunks);

/* Bytes of workspace indexer_prefill_topk needs (host arrays as there). */
idx_status indexer_prefill_workspace_bytes(const int32_t* seq_lens_host,
                                           const int32_t* query_lens_host, int32_t num_reqs,
                                           int32_t topk, int64_t workspace_tokens,
                                           int64_t logits_budget_bytes, size_t* bytes);

/*
 * Prefill top-k ([INDEXER] split_indexer_prefill_chunks,
 * build_prefill_chunk_metadata and _build_prefill_chunk_metadata_kernel).
 * Query token i of request r (global row query_start_loc[r] + i) sees keys
 * [0, seq_len_r - query_len_r + 1 + i) of request r (block-table row r).
 * The chunk plan above is computed from the host copies and the chunks are
 * enqueued in order; results do not depend on the plan (no logits are
 * materialised; the plan bounds each launch's rows the way the pages bound
 * their M x N logits buffer).
 * q bf16 [total_q, 64, 128], weights fp32 [total_q, 64], seq_lens int32 [R],
 * query_start_loc int32 [R + 1] (device), seq_lens_host / query_lens_host
 * int32 [R] (host, equal to the device data; 0 <= query_len <= seq_len);
 * out_idx int32 [total_q, topk].
 */
idx_status indexer_prefill_topk(const void* q, const float* weights, const uint8_t* index_cache,
                                int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                                int32_t bt_width, const int32_t* seq_lens,
                                const int32_t* query_start_loc, const int32_t* seq_lens_host,
                                const int32_t* query_lens_host, int32_t num_reqs,
                                int32_t num_heads, int32_t head_dim, int32_t topk,
                                int64_t workspace_tokens, int64_t logits_budget_bytes,
                                int32_t* out_idx, void* workspace, size_t workspace_bytes,
                                uint32_t* dev_error, void* stream);

/*
 * Profiling hook (the live per-kernel timing a benchmark needs): while set,
 * every decode/prefill call made from this host thread records start_event
 * immediately before and stop_event immediately after each launch of the
 * score/select kernel, on the call's stream (cudaEvent_t handles owned by the
 * caller; NULL, NULL turns it off). Meant for eager calls, not stream capture.
 */
idx_status indexer_profile_events(void* start_event, void* stop_event);

/*
 * Tracing hook: while set, score/select launches made from this host thread
 * write 64 uint64 per tile stream (two per CTA, one CTA per SM) into `buffer`
 * (device memory, zeroed by the caller, >= 64 * 8 * (2 x SM count) bytes;
 * smaller buffers disable it): %globaltimer
 * stamps of the start, the first/last TMA, MMA and epilogue tile and the end,
 * the ns and count of buffer compactions, segment publication, split-row
 * selection (waits, scans, final picks) and merges, and the CTA's tile count.
 * NULL turns it off.
 */
idx_status indexer_trace_buffer(void* buffer, size_t bytes);

/*
 * Failure-detection hook (for tests of the give-up path): score/select
 * launches made from this host thread give up every pipeline and split-row
 * wait after limit_ns nanoseconds instead of 2 s (0 restores 2 s). With
 * stall_split_rows != 0 their split-row waits also wait for one segment more
 * than the row has, a count nothing completes, so those waits run into the
 * limit. A wait that gives up ORs IDX_DEV_TIMEOUT into *dev_error; the kernel
 * then drains its own copies and tensor-core work, frees its tensor memory
 * and returns, leaving the call's outputs unspecified. Not for production
 * calls.
 */
idx_status indexer_debug_wait_limit(uint64_t limit_ns, int32_t stall_split_rows);

/*
 * Test hook for indexer_insert_keys's division: for n pairs (a[i], b[i])
 * (float, device) writes the quotient the insert computes (the correctly
 * rounded reciprocal of b and two correction steps when b >= 2^-100, else
 * the IEEE division) to quotient[i] and the IEEE round-to-nearest quotient
 * to quotient_ieee[i], so that tests can compare them.
 */
idx_status indexer_debug_divide(const float* a, const float* b, int64_t n, float* quotient,
                                float* quotient_ieee, void* stream);

/*
 * indexer_decode_topk without a caller workspace. The pages have no
 * counterpart: this is a convenience of this library.
 *
 * For callers that cannot allocate device memory where they run the indexer:
 * code running while a stream is captured into a CUDA graph, serving loops
 * that forbid allocator calls on their latency-critical path, or hosts whose
 * device memory is owned by an allocator this code cannot call. The scratch is
 * a 64 MiB device array inside the library (one per GPU that loads the
 * library, held until the process exits); the call allocates nothing. Same
 * arguments and results as indexer_decode_topk without the workspace.
 *  - Limit: the batch must fit the scratch, i.e. indexer_decode_workspace_bytes
 *    (num_reqs, next_n, topk) <= 64 MiB (about 5700 requests at next_n = 1,
 *    2050 at next_n = 2, top-2048, 152 SMs); a larger batch returns
 *    IDX_ERR_WORKSPACE before any work.
 *  - The first call on each device looks the scratch's device address up (this
 *    may load the library's device code); make that first call before any
 *    stream capture.
 *  - All calls on a device share the scratch, which keeps the last call's
 *    contents (each call re-initialises what it needs). Calls whose execution
 *    overlaps on the GPU (other streams, other host threads) race on it.
 */
idx_status indexer_decode_topk_noalloc(const void* q, const float* weights,
                                       const uint8_t* index_cache, int64_t num_pages,
                                       const int32_t* block_table, int64_t bt_stride,
                                       int32_t bt_width, const int32_t* row_seq_lens,
                                       int32_t num_reqs, int32_t next_n, int32_t num_heads,
                                       int32_t head_dim, int32_t topk, int32_t* out_idx,
                                       uint32_t* dev_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SAIB_INDEXER_H */
