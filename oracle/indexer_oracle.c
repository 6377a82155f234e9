/*
 * Plain CPU oracle for the decode/prefill sparse-attention indexer.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct restatement
 * of what the indexer computes; it is used by the tests, by the smoke check and
 * by the benchmark's CPU-baseline leg. The product path never links or calls it,
 * and it shares no code, header or table with the CUDA library.
 *
 * Sources (page titles, with the section each function follows):
 *  - "vllm.models.minimax_m3.amd.mono.runner", token_rows: a request of q query
 *    tokens becomes q rows, token j seeing seq_len - (q - 1 - j) keys.
 *  - "recipes/.../vllm/v1/attention/backends/mla/indexer.py":
 *      * _prepare_decode_tensors (flatten path, variable decode lengths, and the
 *        native 2-D path) for the per-token seq_len of decode rows;
 *      * split_indexer_prefill_chunks for the prefill chunk planner;
 *      * _build_prefill_chunk_metadata_kernel for the prefill key range
 *        [0, seq_len - query_len + 1 + i) of query i;
 *      * get_max_prefill_buffer_size for the 128 fp8 bytes + 4 scale bytes of
 *        one index-key entry; DeepseekV32IndexerBackend.get_kv_cache_shape for
 *        the (num_blocks, block_size, head_size) cache with 64-token blocks.
 *  - "vllm.models.glm5next.common.sparse_indexer": _decode_topk_seq_lens
 *    (padded rows get seq_len 0), _fill_short_decode_causal_indices (exact
 *    causal rows when every key would be selected), _gather_workspace_shapes
 *    (fp8 values + 4-byte fp32 scale per token; the MXFP4 path: head_dim / 2
 *    bytes of packed mxfp4 values + head_dim / MXFP4_BLOCK_SIZE ue8m0 scale
 *    bytes per token) and kv_cache_as_quant_view (the MXFP4 cache view: token
 *    stride head_dim / 2 + head_dim / MXFP4_BLOCK_SIZE bytes inside a page).
 *    _build_prefill_chunk_metadata_kernel's DCP branch also gives the key
 *    count of one rank of a key-sharded (decode context parallel) cache, and
 *    its COMPRESS_RATIO the key count of a compressed cache (DeepseekV4: one
 *    cache entry per compress_ratio tokens; the decode metadata divides the
 *    per-token seq_lens by the same ratio).
 *  - The scoring rule logit[t,s] = sum_h w[t,h] * ReLU(scale_s * (q[t,h] . k_s))
 *    and top-k = 2048 come from the statement of the method; the pages only name
 *    the kernels (fp8_fp4_paged_mqa_logits and "the topk kernels").
 *
 * Readings where the pages are silent or ambiguous (each one stated here):
 *  - Page byte layout: each 64-token page is [64 x 128 fp8 e4m3 values]
 *    followed by [64 x fp32 scales] = 8448 bytes (64 * 132).
 *  - q reaches an fp8 MMA, so q is quantised per (token, head): amax = max|q|,
 *    inv = 448 / amax (fp32), q8 = e4m3_rne_satfinite(q * inv) (fp32 product),
 *    sq = amax / 448; the head weight becomes w * sq. amax == 0 gives q8 = 0,
 *    sq = 0. The fp32 steps decide integer codes, so they are done in fp32 here
 *    exactly as the kernel does them; everything else is fp64.
 *  - Cache insert (not shown on the pages): slot s is page s / 64, token
 *    s % 64 (negative = padding); scale = amax / 448 and codes e4m3(x / scale),
 *    fp32 steps like the q quantisation; amax == 0 gives zero codes, scale 0.
 *  - Since scale_s >= 0, ReLU(scale_s * x) = scale_s * ReLU(x).
 *  - MXFP4 index keys (the cache format the INDEXER page gates behind
 *    use_fp4_indexer_cache): MXFP4_BLOCK_SIZE = 32 (so 4 scale bytes and a
 *    68-byte token entry); a page is 64 token entries back to back (4352
 *    bytes, the quant view's token stride with no padding); inside an entry
 *    the 64 value bytes come first (element 2i in the low nibble of byte i,
 *    2i + 1 in the high nibble), then the 4 scale bytes (block b covers
 *    elements 32b .. 32b + 31), in the order the gather workspace lists them.
 *    e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit, no infinities or NaN,
 *    largest magnitude 6; ue8m0: 2^(E - 127), E = 255 is NaN. A key's value
 *    d is e2m1(code_d) * 2^(E_{d/32} - 127); there is no per-token fp32 scale.
 *    The cache writer is not shown: the oracle quantises a block of 32 by the
 *    shared-exponent rule of the MX format: E = floor(log2(amax)) - 2 + 127
 *    (2 = the largest e2m1 exponent; clamped to [0, 254]; amax = 0 gives
 *    E = 0 and zero codes), codes = e2m1_rne_satfinite(x / 2^(E - 127)).
 *  - Key-sharded decode (the pages give only the local key count): each rank
 *    scores the keys it holds for a row (its local count of the row's
 *    length, dealt in runs of I tokens) and keeps its top k with their
 *    logits (a row of <= k local keys keeps them all); the ranks' candidates,
 *    in global token positions, are merged by the same rule as one row's
 *    top k. The merged set equals the unsharded row's top k, since every
 *    key of the global top k is in its own rank's top k.
 *  - Block / pool selection (the MiniMax runner's topk_blocks, init_blocks,
 *    local_blocks; GLM5's pool_topk and expand_pools_and_append_tail, named
 *    on the pages without their rules): blocks of B tokens scored by their
 *    largest logit; the first init and last local blocks always kept plus
 *    the k best of the others; pools expanded to their tokens and the row's
 *    incomplete last pool appended as its tail.
 *  - Rows with len <= k output [0, 1, ..., len-1, -1, ...]; rows with len > k
 *    output the k indices of the largest logits; ties are broken here by the
 *    smaller index (any k-subset that agrees within the tolerance is accepted
 *    by the tests).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread -ffp-contract=off
 * (no FMA contraction: the fp32 quantisation steps must round one by one).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORA_PAGE_TOKENS 64
#define ORA_DIM 128
#define ORA_PAGE_BYTES (ORA_PAGE_TOKENS * (ORA_DIM + 4))
#define ORA_SCALE_OFFSET (ORA_PAGE_TOKENS * ORA_DIM)

/* ------------------------------------------------------------------------ */
/* fp8 e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no     */
/* infinities; S.1111.111 is NaN; largest finite magnitude 448.              */
/* ------------------------------------------------------------------------ */

double ora_e4m3_decode(uint8_t code) {
  int s = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m * 2^-3 * 2^(1-7) */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Round-to-nearest-even onto the e4m3fn grid, saturating to +-448 (also for
 * infinities). Done by a plain search over the 127 non-negative finite codes,
 * which increase with the code. */
uint8_t ora_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  int lo = 0;
  for (int c = 0; c <= 0x7E; ++c) {
    if (ora_e4m3_decode((uint8_t)c) <= a) lo = c;
    else break;
  }
  double vlo = ora_e4m3_decode((uint8_t)lo);
  if (vlo == a) return sign | (uint8_t)lo;
  int hi = lo + 1; /* exists: a < 448 = decode(0x7E) */
  double vhi = ora_e4m3_decode((uint8_t)hi);
  double dlo = a - vlo, dhi = vhi - a; /* exact in double */
  int pick;
  if (dlo < dhi) pick = lo;
  else if (dhi < dlo) pick = hi;
  else pick = (lo & 1) ? hi : lo; /* tie: even mantissa */
  return sign | (uint8_t)pick;
}

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Per (row, head) quantisation of q and folding of the quantisation scale into
 * the head weight. q_bf16: [rows, heads, dim] raw bf16 bits; w: [rows, heads].
 * Outputs q8 [rows, heads, dim] e4m3 codes, sq [rows, heads] and
 * wprime = w * sq [rows, heads], both fp64. */
void ora_quantize_q(const uint16_t* q_bf16, const float* w, int64_t rows, int32_t heads,
                    int32_t dim, uint8_t* q8, double* sq, double* wprime) {
  for (int64_t r = 0; r < rows; ++r) {
    for (int32_t h = 0; h < heads; ++h) {
      const uint16_t* src = q_bf16 + (r * heads + h) * dim;
      uint8_t* dst = q8 + (r * heads + h) * dim;
      float amax = 0.0f;
      for (int32_t d = 0; d < dim; ++d) {
        float a = fabsf(bf16_to_float(src[d]));
        if (a > amax) amax = a;
      }
      double s;
      if (amax == 0.0f) {
        for (int32_t d = 0; d < dim; ++d) dst[d] = 0x00;
        s = 0.0;
      } else {
        float inv = 448.0f / amax; /* fp32 division */
        for (int32_t d = 0; d < dim; ++d) {
          float x = bf16_to_float(src[d]) * inv; /* fp32 product */
          dst[d] = ora_e4m3_encode(x);
        }
        s = (double)amax / 448.0;
      }
      sq[r * heads + h] = s;
      wprime[r * heads + h] = (double)w[r * heads + h] * s;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Index-key cache insert                                                    */
/* ------------------------------------------------------------------------ */

/* The step that fills the paged cache ("recipes/.../indexer.py",
 * DeepseekV32IndexerMetadata.slot_mapping: every new token has a cache slot;
 * get_max_prefill_buffer_size and the glm5next _gather_workspace_shapes: 128
 * fp8 values + one fp32 scale per token). Token i (k_bf16 [n, 128] raw bf16)
 * gets scale = amax / 448 (fp32 division) and codes e4m3(x / scale) (fp32
 * division, round to nearest even, saturating); slot s = slots[i] is page
 * s / 64, token s % 64. Negative or out-of-range slots are skipped; amax == 0
 * gives zero codes and scale 0. */
void ora_insert_keys(const uint16_t* k_bf16, const int64_t* slots, int64_t n, uint8_t* cache,
                     int64_t num_pages) {
  for (int64_t i = 0; i < n; ++i) {
    const int64_t s = slots[i];
    if (s < 0 || s >= num_pages * ORA_PAGE_TOKENS) continue;
    const uint16_t* src = k_bf16 + i * ORA_DIM;
    float amax = 0.0f;
    for (int d = 0; d < ORA_DIM; ++d) {
      const float a = fabsf(bf16_to_float(src[d]));
      if (a > amax) amax = a;
    }
    uint8_t* page = cache + (s / ORA_PAGE_TOKENS) * ORA_PAGE_BYTES;
    const int64_t tok = s % ORA_PAGE_TOKENS;
    const float scale = amax / 448.0f; /* fp32 division */
    for (int d = 0; d < ORA_DIM; ++d)
      page[tok * ORA_DIM + d] = amax == 0.0f ? 0x00 : ora_e4m3_encode(bf16_to_float(src[d]) / scale);
    memcpy(page + ORA_SCALE_OFFSET + tok * 4, &scale, 4);
  }
}

/* ------------------------------------------------------------------------ */
/* Decode row expansion                                                      */
/* ------------------------------------------------------------------------ */

/* mode 0 (padded [num_reqs, next_n] grid, as the native 2-D path and the
 * glm5next padded grid lay it out): row b*next_n + j has
 *     len = j < d_b ? L_b - d_b + j + 1 : 0.
 * mode 1 (flatten, as the variable-decode-length path): the d_b tokens of
 * request b occupy consecutive rows starting at sum_{b'<b} d_b'; token j has
 * the same len; the rows after the last token up to num_out_rows get len 0.
 * row_bt (nullable): the request's block-table row is copied to each of its
 * token rows (first bt_width entries); rows past the last token get column 0
 * set to 0 and the rest left untouched, as the flatten path does.
 * Returns the number of rows holding tokens, or -1 if they do not fit. */
int64_t ora_expand_rows(const int32_t* seq_lens, const int32_t* decode_lens, int32_t num_reqs,
                        int32_t next_n, int32_t mode, const int32_t* bt, int64_t bt_stride,
                        int32_t bt_width, int32_t* row_lens, int32_t* row_bt,
                        int64_t out_stride, int64_t num_out_rows) {
  if (mode == 0) {
    if ((int64_t)num_reqs * next_n > num_out_rows) return -1;
    for (int32_t b = 0; b < num_reqs; ++b) {
      for (int32_t j = 0; j < next_n; ++j) {
        int64_t row = (int64_t)b * next_n + j;
        int32_t d = decode_lens[b];
        row_lens[row] = (j < d) ? seq_lens[b] - d + j + 1 : 0;
        if (row_bt)
          for (int32_t c = 0; c < bt_width; ++c)
            row_bt[row * out_stride + c] = bt[(int64_t)b * bt_stride + c];
      }
    }
    return (int64_t)num_reqs * next_n;
  }
  int64_t total = 0;
  for (int32_t b = 0; b < num_reqs; ++b) total += decode_lens[b];
  if (total > num_out_rows) return -1;
  int64_t row = 0;
  for (int32_t b = 0; b < num_reqs; ++b) {
    int32_t d = decode_lens[b];
    for (int32_t j = 0; j < d; ++j, ++row) {
      row_lens[row] = seq_lens[b] - d + j + 1;
      if (row_bt)
        for (int32_t c = 0; c < bt_width; ++c)
          row_bt[row * out_stride + c] = bt[(int64_t)b * bt_stride + c];
    }
  }
  for (; row < num_out_rows; ++row) {
    row_lens[row] = 0;
    if (row_bt && bt_width > 0) row_bt[row * out_stride] = 0;
  }
  return total;
}

/* ------------------------------------------------------------------------ */
/* Scoring                                                                   */
/* ------------------------------------------------------------------------ */

static double g_dec[256];
static pthread_once_t g_dec_once = PTHREAD_ONCE_INIT;
static void init_dec(void) {
  for (int c = 0; c < 256; ++c) g_dec[c] = ora_e4m3_decode((uint8_t)c);
}

/* Logits of one token row over keys [0, len):
 *   logit[s] = scale_s * sum_h wprime[h] * max(dot_h(s), 0),
 *   dot_h(s) = sum_d q8[h][d] * k8_s[d]   (exact in fp64: 8-bit products, 128 terms).
 * The key s lives in page bt_row[s / 64], slot s % 64.
 * tol_a[s] = scale_s * sum_h |wprime[h]| * max(dot_h, 0) and
 * tol_b[s] = scale_s * sum_h |wprime[h]| * sum_d |q8[h][d] * k8_s[d]| are the
 * magnitudes the tests scale their tolerance by (either may be NULL).
 * Returns -1 when a page id is outside [0, num_pages), else 0. */
int ora_row_logits(const uint8_t* q8_row, const double* wprime_row, int32_t heads, int32_t dim,
                   const uint8_t* cache, int64_t num_pages, const int32_t* bt_row, int64_t len,
                   double* logits, double* tol_a, double* tol_b) {
  pthread_once(&g_dec_once, init_dec);
  double* qd = (double*)malloc(sizeof(double) * (size_t)heads * dim);
  double kd[ORA_DIM];
  if (!qd || dim != ORA_DIM) { free(qd); return -2; }
  for (int64_t i = 0; i < (int64_t)heads * dim; ++i) qd[i] = g_dec[q8_row[i]];
  for (int64_t s = 0; s < len; ++s) {
    int64_t page = bt_row[s / ORA_PAGE_TOKENS];
    if (page < 0 || page >= num_pages) { free(qd); return -1; }
    int64_t slot = s % ORA_PAGE_TOKENS;
    const uint8_t* pg = cache + page * ORA_PAGE_BYTES;
    const uint8_t* k8 = pg + slot * ORA_DIM;
    float scale_f;
    memcpy(&scale_f, pg + ORA_SCALE_OFFSET + 4 * slot, 4);
    double scale = (double)scale_f;
    for (int d = 0; d < ORA_DIM; ++d) kd[d] = g_dec[k8[d]];
    double acc = 0.0, acc_a = 0.0, acc_b = 0.0;
    for (int32_t h = 0; h < heads; ++h) {
      const double* qh = qd + (int64_t)h * dim;
      double dot = 0.0, adot = 0.0;
      for (int d = 0; d < ORA_DIM; ++d) {
        double p = qh[d] * kd[d];
        dot += p;
        adot += fabs(p);
      }
      double relu = dot > 0.0 ? dot : 0.0;
      acc += wprime_row[h] * relu;
      acc_a += fabs(wprime_row[h]) * relu;
      acc_b += fabs(wprime_row[h]) * adot;
    }
    logits[s] = scale * acc;
    if (tol_a) tol_a[s] = scale * acc_a;
    if (tol_b) tol_b[s] = scale * acc_b;
  }
  free(qd);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* MXFP4 index keys                                                           */
/* ------------------------------------------------------------------------ */

#define ORA_MX_BLOCK 32
#define ORA_MX_TOKEN_BYTES (ORA_DIM / 2 + ORA_DIM / ORA_MX_BLOCK) /* 68 */
#define ORA_MX_PAGE_BYTES (ORA_PAGE_TOKENS * ORA_MX_TOKEN_BYTES) /* 4352 */

/* e2m1 (the low 4 bits of code): e == 0 gives m * 0.5 (0 or 0.5), else
 * 2^(e - 1) * (1 + m / 2); the sign bit negates. */
double ora_e2m1_decode(uint8_t code) {
  int s = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* ue8m0: 2^(E - 127); E = 255 is NaN. */
double ora_ue8m0_decode(uint8_t e) {
  if (e == 255) return NAN;
  return ldexp(1.0, (int)e - 127);
}

/* Round-to-nearest-even onto the e2m1 grid, saturating to +-6: a search over
 * the 8 non-negative codes, which increase with the code. */
uint8_t ora_e2m1_encode(double x) {
  uint8_t sign = signbit(x) ? 0x8 : 0x0;
  double a = fabs(x);
  if (isnan(x)) return 0; /* never produced by the writer below */
  if (a >= 6.0) return sign | 0x7;
  int lo = 0;
  for (int c = 0; c <= 7; ++c) {
    if (ora_e2m1_decode((uint8_t)c) <= a) lo = c;
    else break;
  }
  double vlo = ora_e2m1_decode((uint8_t)lo);
  if (vlo == a) return sign | (uint8_t)lo;
  int hi = lo + 1;
  double vhi = ora_e2m1_decode((uint8_t)hi);
  double dlo = a - vlo, dhi = vhi - a;
  int pick;
  if (dlo < dhi) pick = lo;
  else if (dhi < dlo) pick = hi;
  else pick = (lo & 1) ? hi : lo; /* tie: even mantissa */
  return sign | (uint8_t)pick;
}

/* One token's MXFP4 entry (68 bytes) from its 128 values, by the MX
 * shared-exponent rule (see the readings above). */
void ora_mxfp4_quantize_token(const float* x, uint8_t* out) {
  memset(out, 0, ORA_MX_TOKEN_BYTES);
  for (int b = 0; b < ORA_DIM / ORA_MX_BLOCK; ++b) {
    double amax = 0.0;
    for (int i = 0; i < ORA_MX_BLOCK; ++i) {
      double a = fabs((double)x[b * ORA_MX_BLOCK + i]);
      if (a > amax) amax = a;
    }
    int E = 0;
    if (amax > 0.0) {
      int ex;
      frexp(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
      E = (ex - 1) - 2 + 127;
      if (E < 0) E = 0;
      if (E > 254) E = 254;
    }
    out[ORA_DIM / 2 + b] = (uint8_t)E;
    if (amax == 0.0) continue;
    double X = ldexp(1.0, E - 127);
    for (int i = 0; i < ORA_MX_BLOCK; ++i) {
      int d = b * ORA_MX_BLOCK + i;
      uint8_t c = ora_e2m1_encode((double)x[d] / X);
      out[d / 2] |= (uint8_t)((d & 1) ? (c << 4) : c);
    }
  }
}

/* Value d of an MXFP4 entry. */
static double mx_value(const uint8_t* entry, int d) {
  uint8_t byte = entry[d / 2];
  uint8_t code = (d & 1) ? (byte >> 4) : (byte & 0xF);
  return ora_e2m1_decode(code) * ora_ue8m0_decode(entry[ORA_DIM / 2 + d / ORA_MX_BLOCK]);
}

/* Logits of one token row over keys [0, len) with an MXFP4 cache:
 *   logit[s] = sum_h wprime[h] * max(dot_h(s), 0),
 *   dot_h(s) = sum_d q8[h][d] * k_s[d],  k_s[d] = e2m1(code) * 2^(E - 127)
 * (each block's 32 products are exact in fp64 and share one power of two).
 * tol_a / tol_b as ora_row_logits with scale 1 (either may be NULL).
 * Returns -1 when a page id is outside [0, num_pages), else 0. */
int ora_row_logits_mxfp4(const uint8_t* q8_row, const double* wprime_row, int32_t heads,
                         int32_t dim, const uint8_t* cache, int64_t num_pages,
                         const int32_t* bt_row, int64_t len, double* logits, double* tol_a,
                         double* tol_b) {
  pthread_once(&g_dec_once, init_dec);
  double* qd = (double*)malloc(sizeof(double) * (size_t)heads * dim);
  double kd[ORA_DIM];
  if (!qd || dim != ORA_DIM) { free(qd); return -2; }
  for (int64_t i = 0; i < (int64_t)heads * dim; ++i) qd[i] = g_dec[q8_row[i]];
  for (int64_t s = 0; s < len; ++s) {
    int64_t page = bt_row[s / ORA_PAGE_TOKENS];
    if (page < 0 || page >= num_pages) { free(qd); return -1; }
    const uint8_t* entry = cache + page * ORA_MX_PAGE_BYTES + (s % ORA_PAGE_TOKENS) * ORA_MX_TOKEN_BYTES;
    for (int d = 0; d < ORA_DIM; ++d) kd[d] = mx_value(entry, d);
    double acc = 0.0, acc_a = 0.0, acc_b = 0.0;
    for (int32_t h = 0; h < heads; ++h) {
      const double* qh = qd + (int64_t)h * dim;
      double dot = 0.0, adot = 0.0;
      for (int d = 0; d < ORA_DIM; ++d) {
        double p = qh[d] * kd[d];
        dot += p;
        adot += fabs(p);
      }
      double relu = dot > 0.0 ? dot : 0.0;
      acc += wprime_row[h] * relu;
      acc_a += fabs(wprime_row[h]) * relu;
      acc_b += fabs(wprime_row[h]) * adot;
    }
    logits[s] = acc;
    if (tol_a) tol_a[s] = acc_a;
    if (tol_b) tol_b[s] = acc_b;
  }
  free(qd);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Selection                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct { double v; int32_t i; } ora_pair;

static int cmp_pair(const void* a, const void* b) {
  const ora_pair* x = (const ora_pair*)a;
  const ora_pair* y = (const ora_pair*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i < y->i) ? -1 : (x->i > y->i);
}

/* len <= k: out = [0, 1, ..., len-1, -1, ...] (the exact causal row).
 * len > k: the k indices with the largest logits, by (logit desc, index asc),
 * written in that order. */
void ora_topk_row(const double* logits, int64_t len, int32_t k, int32_t* out) {
  if (len <= k) {
    for (int32_t i = 0; i < k; ++i) out[i] = (i < len) ? i : -1;
    return;
  }
  ora_pair* p = (ora_pair*)malloc(sizeof(ora_pair) * (size_t)len);
  for (int64_t s = 0; s < len; ++s) { p[s].v = logits[s]; p[s].i = (int32_t)s; }
  qsort(p, (size_t)len, sizeof(ora_pair), cmp_pair);
  for (int32_t i = 0; i < k; ++i) out[i] = p[i].i;
  free(p);
}

/* len <= k: every key, out = [0, ..., len-1, -1, ...] with its logit (-inf
 * past len); len > k: as ora_topk_row, with the logit of each index. The
 * form a key-sharded rank hands to the merge: its row of len <= k keys
 * still needs the logits. */
void ora_topk_row_values(const double* logits, int64_t len, int32_t k, int32_t* out,
                         double* out_val) {
  ora_topk_row(logits, len, k, out);
  for (int32_t i = 0; i < k; ++i) out_val[i] = out[i] >= 0 ? logits[out[i]] : -INFINITY;
}

/* ------------------------------------------------------------------------ */
/* Key-sharded decode (decode context parallelism)                           */
/* ------------------------------------------------------------------------ */
/* INDEXER page, _build_prefill_chunk_metadata_kernel, the DCP_WORLD_SIZE > 1
 * branch: a sequence's keys are dealt to the W ranks in runs of I tokens
 * (token t goes to rank (t / I) % W, after the rank's earlier tokens), so
 * rank r holds, of L keys,
 *   base + min(max(rem - r * I, 0), I),  base = L / I / W * I,  rem = L - base * W
 * (floor divisions, in the kernel's order). W <= 1: all L. */
int64_t ora_dcp_local_len(int64_t L, int32_t rank, int32_t world, int32_t interleave) {
  if (world <= 1) return L;
  const int64_t base = L / interleave / world * interleave;
  const int64_t rem = L - base * world;
  int64_t r = rem - (int64_t)rank * interleave;
  if (r < 0) r = 0;
  if (r > interleave) r = interleave;
  return base + r;
}

/* Index keys a row sees when the cache holds one entry per `ratio` tokens
 * (INDEXER page: DeepseekV4's compress_ratio; the decode path divides the
 * per-token seq_lens by it, _build_prefill_chunk_metadata_kernel computes
 * (start_pos + 1 + i) / COMPRESS_RATIO), then, on a key-sharded cache, the
 * rank's local count of those entries (the same kernel's DCP branch). */
int64_t ora_index_key_count(int64_t L, int32_t ratio, int32_t rank, int32_t world,
                            int32_t interleave) {
  return ora_dcp_local_len(L / ratio, rank, world, interleave);
}

/* Token of the whole sequence that rank `rank` holds as its local key j: its
 * (j / I)-th run, which comes after (j / I) full rounds of W runs and `rank`
 * runs of the current round; offset j % I inside the run. */
int64_t ora_dcp_global_index(int64_t j, int32_t rank, int32_t world, int32_t interleave) {
  if (world <= 1) return j;
  return (j / interleave) * (int64_t)interleave * world + (int64_t)rank * interleave +
         j % interleave;
}

/* One row's merge of the ranks' candidates: n (logit, global index) pairs,
 * index < 0 = an empty slot. out = the k best by (logit desc, index asc) in
 * that order, -1 (and -inf) past the candidates. */
void ora_merge_candidates(const double* val, const int32_t* idx, int64_t n, int32_t k,
                          int32_t* out, double* out_val) {
  ora_pair* p = (ora_pair*)malloc(sizeof(ora_pair) * (size_t)(n > 0 ? n : 1));
  int64_t m = 0;
  for (int64_t i = 0; i < n; ++i)
    if (idx[i] >= 0) { p[m].v = val[i]; p[m].i = idx[i]; ++m; }
  qsort(p, (size_t)m, sizeof(ora_pair), cmp_pair);
  for (int32_t i = 0; i < k; ++i) {
    out[i] = i < m ? p[i].i : -1;
    out_val[i] = i < m ? p[i].v : -INFINITY;
  }
  free(p);
}

/* ------------------------------------------------------------------------ */
/* Block / pool selection                                                    */
/* ------------------------------------------------------------------------ */
/* MiniMax runner (topk_blocks, init_blocks, local_blocks) and GLM5
 * (pool_topk, expand_pools_and_append_tail) select whole blocks of tokens;
 * the pages give the names only. Reading: a row of L tokens is cut into
 * nb = ceil(L / B) blocks of B tokens (the last may be partial); a block's
 * score is the largest logit of its tokens; the selection is the first
 * n_init blocks, the last n_local blocks and the k highest-scoring of the
 * others (ties: the smaller block index), out = the selected blocks in
 * ascending order, -1 after them; returns how many. */
int32_t ora_block_topk(const double* logits, int64_t L, int32_t B, int32_t k, int32_t n_init,
                       int32_t n_local, int32_t* out, int32_t out_cap) {
  const int64_t nb = (L + B - 1) / B;
  char* sel = (char*)calloc((size_t)(nb > 0 ? nb : 1), 1);
  ora_pair* p = (ora_pair*)malloc(sizeof(ora_pair) * (size_t)(nb > 0 ? nb : 1));
  int64_t m = 0;
  for (int64_t b = 0; b < nb; ++b) {
    if (b < n_init || b >= nb - n_local) {
      sel[b] = 1;
      continue;
    }
    double best = -INFINITY;
    for (int64_t t = b * B; t < L && t < (b + 1) * B; ++t)
      if (logits[t] > best) best = logits[t];
    p[m].v = best;
    p[m].i = (int32_t)b;
    ++m;
  }
  qsort(p, (size_t)m, sizeof(ora_pair), cmp_pair);
  for (int64_t i = 0; i < m && i < k; ++i) sel[p[i].i] = 1;
  int32_t n = 0;
  for (int64_t b = 0; b < nb; ++b)
    if (sel[b] && n < out_cap) out[n++] = (int32_t)b;
  for (int32_t i = n; i < out_cap; ++i) out[i] = -1;
  free(sel);
  free(p);
  return n;
}

/* GLM5 expand_pools_and_append_tail (reading): the tokens of the selected
 * complete pools (pool b covers [b P, b P + P)), in the order given, then the
 * row's tail [floor(L / P) P, L) (the tokens after its last complete pool);
 * a selected pool that is not complete contributes nothing (its tokens are
 * the tail). -1 after them; returns how many. */
int32_t ora_expand_pools(const int32_t* pools, int32_t npools, int64_t L, int32_t P,
                         int32_t* out, int32_t out_cap) {
  int32_t n = 0;
  const int64_t full = L / P;
  for (int32_t i = 0; i < npools; ++i) {
    const int64_t b = pools[i];
    if (b < 0 || b >= full) continue;
    for (int64_t t = b * P; t < (b + 1) * P && n < out_cap; ++t) out[n++] = (int32_t)t;
  }
  for (int64_t t = full * P; t < L && n < out_cap; ++t) out[n++] = (int32_t)t;
  for (int32_t i = n; i < out_cap; ++i) out[i] = -1;
  return n;
}

/* ------------------------------------------------------------------------ */
/* Batched rows over a thread pool                                           */
/* ------------------------------------------------------------------------ */

/* One scored token row: q8/wprime row `qrow`, block-table row `bt_row_idx`,
 * length `len`. Logits (and tolerance magnitudes) are written at
 * logit_off[i] .. logit_off[i] + len in the output arrays (nullable), the
 * top-k at out_idx[i * k]. */
typedef struct {
  const uint8_t* q8; const double* wprime; int32_t heads; int32_t dim;
  const uint8_t* cache; int64_t num_pages;
  const int32_t* bt; int64_t bt_stride;
  const int64_t* qrow; const int64_t* bt_row_idx; const int64_t* lens; int64_t n;
  int32_t k; int32_t* out_idx;
  const int64_t* logit_off; double* logits; double* tol_a; double* tol_b;
  int64_t next; int err;
} ora_job;

static void* worker(void* arg) {
  ora_job* J = (ora_job*)arg;
  for (;;) {
    int64_t i = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (i >= J->n) break;
    int64_t len = J->lens[i];
    double *lg, *ta = NULL, *tb = NULL, *own = NULL;
    if (J->logits) {
      lg = J->logits + J->logit_off[i];
      if (J->tol_a) ta = J->tol_a + J->logit_off[i];
      if (J->tol_b) tb = J->tol_b + J->logit_off[i];
    } else {
      own = (double*)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
      lg = own;
    }
    int rc = 0;
    if (len > 0 && (J->out_idx == NULL || len > J->k || J->logits != NULL))
      rc = ora_row_logits(J->q8 + J->qrow[i] * J->heads * J->dim,
                          J->wprime + J->qrow[i] * J->heads, J->heads, J->dim, J->cache,
                          J->num_pages, J->bt + J->bt_row_idx[i] * J->bt_stride, len, lg, ta, tb);
    if (rc) __atomic_store_n(&J->err, rc, __ATOMIC_RELAXED);
    else if (J->out_idx) ora_topk_row(lg, len, J->k, J->out_idx + i * J->k);
    free(own);
  }
  return NULL;
}

int ora_num_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/* Scores (and, when out_idx != NULL, selects) n token rows with `threads`
 * worker threads (<= 0: one per online core). Returns 0, or a negative code if
 * a row referenced a page outside the cache. */
int ora_score_select_rows(const uint8_t* q8, const double* wprime, int32_t heads, int32_t dim,
                          const uint8_t* cache, int64_t num_pages, const int32_t* bt,
                          int64_t bt_stride, const int64_t* qrow, const int64_t* bt_row_idx,
                          const int64_t* lens, int64_t n, int32_t k, int32_t* out_idx,
                          const int64_t* logit_off, double* logits, double* tol_a, double* tol_b,
                          int32_t threads) {
  ora_job J = {q8, wprime, heads, dim, cache, num_pages, bt, bt_stride, qrow, bt_row_idx,
               lens, n, k, out_idx, logit_off, logits, tol_a, tol_b, 0, 0};
  if (threads <= 0) threads = ora_num_threads();
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  int started = 0;
  for (int t = 1; t < threads; ++t)
    if (pthread_create(&tid[started], NULL, worker, &J) == 0) ++started;
  worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  return J.err;
}

/* ------------------------------------------------------------------------ */
/* Prefill                                                                   */
/* ------------------------------------------------------------------------ */

/* Greedy chunking of prefill requests, following split_indexer_prefill_chunks:
 * requests are packed while the summed key count N stays <= workspace_tokens and
 * (summed queries M) * N <= logits_budget_bytes / 4; a request that fits alone
 * in neither is taken by itself; each chunk is then cut on the query axis into
 * pieces of at most max(1, (budget/4) // N) queries (all of them when N == 0).
 * Output rows: (req_begin, req_end, q_begin, q_end), q relative to the chunk's
 * first query. A chunk with no queries produces no piece (the reference would
 * call range() with a zero step there). Returns the number of pieces, or -1 if
 * more than max_chunks would be needed. */
int64_t ora_plan_prefill_chunks(const int32_t* seq_lens, const int32_t* query_lens,
                                int32_t num_reqs, int64_t workspace_tokens,
                                int64_t logits_budget_bytes, int32_t* chunks,
                                int64_t max_chunks) {
  int64_t elems = logits_budget_bytes / 4;
  int64_t count = 0;
  int32_t end = 0;
  while (end < num_reqs) {
    int32_t start = end;
    int64_t m = 0, nn = 0;
    while (end < num_reqs) {
      int64_t q = query_lens[end], s = seq_lens[end];
      int64_t new_m = m + q, new_n = nn + s;
      if (new_n <= workspace_tokens && new_m * new_n <= elems) {
        m = new_m; nn = new_n; ++end;
      } else {
        break;
      }
    }
    if (end == start) {
      m = query_lens[end]; nn = seq_lens[end]; ++end;
    }
    int64_t max_q;
    if (nn > 0) { max_q = elems / nn; if (max_q < 1) max_q = 1; }
    else max_q = m;
    if (m <= 0) continue;
    for (int64_t off = 0; off < m; off += max_q) {
      int64_t sub = (max_q < m - off) ? max_q : m - off;
      if (count >= max_chunks) return -1;
      chunks[count * 4 + 0] = start;
      chunks[count * 4 + 1] = end;
      chunks[count * 4 + 2] = (int32_t)off;
      chunks[count * 4 + 3] = (int32_t)(off + sub);
      ++count;
    }
  }
  return count;
}

/* Per query token of a prefill batch: request id and the number of keys it
 * sees, len = seq_len - query_len + 1 + i for the request's i-th query
 * (_build_prefill_chunk_metadata_kernel, cu_seqlen_ke - cu_seqlen_ks with
 * compress ratio 1 and no decode-context parallelism). */
void ora_prefill_rows(const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_reqs,
                      int64_t* row_req, int64_t* row_len) {
  for (int32_t r = 0; r < num_reqs; ++r) {
    int32_t qs = query_start_loc[r], qe = query_start_loc[r + 1];
    int32_t ql = qe - qs;
    for (int32_t i = 0; i < ql; ++i) {
      row_req[qs + i] = r;
      row_len[qs + i] = (int64_t)seq_lens[r] - ql + 1 + i;
    }
  }
}
