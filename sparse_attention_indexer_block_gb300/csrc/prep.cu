// Row expansion, q quantisation, and the per-launch schedule + causal fill that
// precede the score/select kernel.
#include <climits>

#include "internal.h"

namespace saib {

namespace {

constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;

// Exclusive scan of one int per thread over a block of kPrepThreads threads.
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_tot[kPrepWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kPrepWarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    if (lane < kPrepWarps) warp_tot[lane] = t;
  }
  __syncthreads();
  const int before = warp > 0 ? warp_tot[warp - 1] : 0;
  *total = warp_tot[kPrepWarps - 1];
  __syncthreads();
  return before + x - v;
}

__device__ __forceinline__ int64_t clamp_len(int64_t v, int64_t bt_width, uint32_t* err,
                                             bool report) {
  const int64_t cap = bt_width * kPageTokens;
  if (v < 0) {
    if (report) set_error(err, IDX_DEV_BAD_LEN);
    return 0;
  }
  if (v > cap) {
    if (report) set_error(err, IDX_DEV_BAD_LEN);
    return cap;
  }
  return v;
}

// One warp quantises one head of 128 bf16 values (raw: the lane's 8 bytes of
// it): lane l owns elements [4l, 4l + 4). Returns the four e4m3 codes of the lane (element 4l in the
// low byte) and, in *wp, w * amax / 448 (all lanes).
__device__ __forceinline__ uint32_t quantize_head(uint2 raw, float w, int lane, float* wp) {
  const float x0 = __uint_as_float(raw.x << 16);
  const float x1 = __uint_as_float(raw.x & 0xffff0000u);
  const float x2 = __uint_as_float(raw.y << 16);
  const float x3 = __uint_as_float(raw.y & 0xffff0000u);
  float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (amax == 0.0f) {
    *wp = 0.0f;
    return 0u;
  }
  const float inv = __fdiv_rn(448.0f, amax);
  const uint32_t lo = cvt_e4m3x2(__fmul_rn(x0, inv), __fmul_rn(x1, inv));
  const uint32_t hi = cvt_e4m3x2(__fmul_rn(x2, inv), __fmul_rn(x3, inv));
  *wp = __fmul_rn(w, __fdiv_rn(amax, 448.0f));
  return lo | (hi << 16);
}

// Byte offset, inside a token row's 8 KB fp8 image, of the 4 codes lane `lane`
// holds for head h, in the layout the MMA reads: 128-byte rows (one per head)
// whose 16-byte chunks are XOR-swizzled by (head & 7) — the 128-byte swizzle
// a TMA copy would produce for a 1024-byte aligned tile.
__device__ __forceinline__ uint32_t swizzled_offset(int h, int lane) {
  return static_cast<uint32_t>(h) * 128u + ((static_cast<uint32_t>(lane >> 2) ^ (h & 7)) << 4) +
         (static_cast<uint32_t>(lane & 3) << 2);
}

// Quantises tasks [0, ntasks) (task = one head of one token row, source head
// src0 + task) with warp gw of nw: four tasks per round, all four loads issued
// before any is used. Codes go to the swizzled per-row image (kSwizzled) or
// to a plain [task, 128] array; w * amax / 448 to wprime[task].
template <bool kSwizzled>
__device__ __forceinline__ void quantize_tasks(const __nv_bfloat16* __restrict__ q,
                                               const float* __restrict__ w, int64_t src0,
                                               int64_t ntasks, uint8_t* __restrict__ q8,
                                               float* __restrict__ wprime, int64_t gw, int64_t nw) {
  const int lane = threadIdx.x & 31;
  for (int64_t base = gw * 4; base < ntasks; base += nw * 4) {
    uint2 raw[4];
    float wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      raw[u] = make_uint2(0u, 0u);
      wv[u] = 0.0f;
      if (base + u < ntasks) {
        const int64_t src = src0 + base + u;
        raw[u] = *reinterpret_cast<const uint2*>(q + src * kDim + 4 * lane);
        wv[u] = w[src];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t idx = base + u;
      if (idx >= ntasks) break;
      float wp;
      const uint32_t c = quantize_head(raw[u], wv[u], lane, &wp);
      if (kSwizzled)
        *reinterpret_cast<uint32_t*>(q8 + (idx / kHeads) * kQRowBytes +
                                     swizzled_offset(static_cast<int>(idx % kHeads), lane)) = c;
      else
        *reinterpret_cast<uint32_t*>(q8 + idx * kDim + 4 * lane) = c;
      if (lane == 0) wprime[idx] = wp;
    }
  }
}

// -------------------------------------------------------------------------

__global__ void __launch_bounds__(kPrepThreads) quantize_plain_kernel(
    const __nv_bfloat16* __restrict__ q, const float* __restrict__ w, int64_t rows,
    uint8_t* __restrict__ q8, float* __restrict__ wprime) {
  pdl_trigger();
  pdl_wait();
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * kPrepThreads + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * kPrepThreads) >> 5;
  quantize_tasks<false>(q, w, 0, rows * kHeads, q8, wprime, gw, nw);
}

// Inclusive prefix max of one int per thread over a block of kPrepThreads
// threads; *total = the block's max.
__device__ int block_inclusive_max(int v, int* total) {
  __shared__ int warp_max[kPrepWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v = max(v, y);
  }
  if (lane == 31) warp_max[warp] = v;
  __syncthreads();
  int before = INT_MIN, all = INT_MIN;
  for (int i = 0; i < kPrepWarps; ++i) {
    if (i < warp) before = max(before, warp_max[i]);
    all = max(all, warp_max[i]);
  }
  __syncthreads();
  *total = all;
  return max(before, v);
}

// Virtual start of every work row: its first tile plus `penalty` for every
// earlier work row that has tiles (each such row's end costs a finalisation).
// Block 0 only, after wts is complete.
__device__ void row_virtual_starts(const int32_t* wts, int num_wr, int penalty, int32_t* vs) {
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < num_wr; base += kPrepThreads) {
    const int w = base + threadIdx.x;
    const int nz = w < num_wr && wts[w + 1] > wts[w] ? 1 : 0;
    int total;
    const int excl = block_exclusive_scan(nz, &total);
    if (w < num_wr) vs[w] = wts[w] + penalty * (carry + excl);
    carry += total;
  }
  if (threadIdx.x == 0) vs[num_wr] = wts[num_wr] + penalty * carry;
}

constexpr int kMaxPlanCtas = 1024;
// Work rows whose tile starts block 0 keeps in shared memory while planning.
constexpr int kPlanRows = 1024;

// The score/select kernel's work split. CTA c of nC = min(grid, T) takes the
// tiles [cta_tile[c], cta_tile[c+1]): the virtual sequence (tiles plus a
// penalty after each work row's end) is cut evenly and mapped back to tiles,
// then every CTA is given at least one tile. Also the work row of each CTA's
// first tile and each work row's first and last CTA. Block 0 only.
__device__ void plan_ctas(const int32_t* wts, const int32_t* vs, int num_wr, int grid,
                          int32_t* cta_tile, int32_t* cta_row, int2* row_ctas) {
  __shared__ int32_t s_ct[kMaxPlanCtas + 1];
  __syncthreads();
  const int T = wts[num_wr];
  const int nC = min(grid, T);
  const int64_t V = vs[num_wr];
  const bool even = nC > kMaxPlanCtas;  // too many CTAs to plan here: plain even split
  if (!even) {
    int carry = INT_MIN;  // max of t - c over the earlier chunks
    for (int base = 0; base <= nC; base += kPrepThreads) {
      const int c = base + threadIdx.x;
      int u = INT_MIN;
      if (c <= nC) {
        int t = T;
        if (c < nC) {
          const int64_t v = static_cast<int64_t>(c) * V / nC;
          int lo = 0, hi = num_wr - 1;  // work row holding virtual position v
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (vs[mid] <= v) lo = mid;
            else hi = mid - 1;
          }
          t = wts[lo] + static_cast<int>(min(v - vs[lo], static_cast<int64_t>(wts[lo + 1] - wts[lo])));
        }
        // CTA c starts in [c, T - nC + c]; a prefix max of t - c then makes
        // the starts strictly increasing
        u = max(min(t, T - nC + c), c) - c;
      }
      int chunk;
      const int incl = block_inclusive_max(u, &chunk);
      if (c <= nC) s_ct[c] = max(carry, incl) + c;
      carry = max(carry, chunk);
    }
  }
  __syncthreads();
  auto start = [&](int c) -> int {
    return even ? static_cast<int>(static_cast<int64_t>(c) * T / nC) : s_ct[c];
  };
  for (int c = threadIdx.x; c <= nC; c += kPrepThreads) cta_tile[c] = start(c);
  for (int c = threadIdx.x; c < grid; c += kPrepThreads) {
    int w = 0;
    if (c < nC) {
      const int t = start(c);
      int lo = 0, hi = num_wr - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (wts[mid] <= t) lo = mid;
        else hi = mid - 1;
      }
      w = lo;
    }
    cta_row[c] = w;
  }
  auto cta_of = [&](int t) {  // the CTA whose range holds tile t
    int lo = 0, hi = nC - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (start(mid) <= t) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };
  for (int w = threadIdx.x; w < num_wr; w += kPrepThreads) {
    const int rs = wts[w], re = wts[w + 1];
    row_ctas[w] = re > rs ? make_int2(cta_of(rs), cta_of(re - 1)) : make_int2(0, -1);
  }
}

// Zeroes n 32-bit words (16-byte aligned) with the blocks after block 0.
__device__ __forceinline__ void zero_words(uint32_t* p, size_t n) {
  const size_t tid = static_cast<size_t>(blockIdx.x - 1) * kPrepThreads + threadIdx.x;
  const size_t nt = static_cast<size_t>(gridDim.x - 1) * kPrepThreads;
  uint4* p4 = reinterpret_cast<uint4*>(p);
  for (size_t i = tid; i < n / 4; i += nt) p4[i] = make_uint4(0, 0, 0, 0);
  for (size_t i = (n / 4) * 4 + tid; i < n; i += nt) p[i] = 0;
}

// Key count of token row r = b * next_n + j before validation: the given
// per-row length, or the row expansion's (token j of a request of d tokens
// and L keys sees L - d + j + 1 keys; rows j >= d are padding, 0); on a
// key-sharded cache, this rank's share of it.
__device__ __forceinline__ int64_t raw_row_len(const DecodePrepArgs& a, int64_t r) {
  int64_t len;
  if (a.row_seq_lens) {
    len = a.row_seq_lens[r];
  } else {
    const int64_t b = r / a.next_n, j = r % a.next_n;
    const int64_t L = a.seq_lens[b], d = a.decode_lens[b];
    len = j < d ? L - d + j + 1 : 0;
  }
  return index_key_count(len, a.compress_ratio, a.dcp_rank, a.dcp_world, a.dcp_interleave);
}

// Block 0: work-row schedule (tile counts and their exclusive prefix), validated
// row lengths and zeroed segment counters. Other blocks: zeroed row histograms,
// q quantisation into the swizzled images and the exact causal rows of short
// rows.
__global__ void __launch_bounds__(kPrepThreads) decode_prep_kernel(
    DecodePrepArgs a, WorkRow* __restrict__ wr, int32_t* __restrict__ wts,
    int32_t* __restrict__ row_len, int32_t* __restrict__ seg_counter, uint8_t* __restrict__ q8img,
    float* __restrict__ wprime, uint32_t* __restrict__ row_hist, size_t row_hist_words,
    int32_t* __restrict__ cta_row, int32_t* __restrict__ cta_tile, int32_t* __restrict__ row_vs,
    int2* __restrict__ row_ctas) {
  pdl_trigger();
  pdl_wait();
  const int G = a.next_n;
  const int64_t rows = static_cast<int64_t>(a.num_reqs) * G;
  if (blockIdx.x == 0) {
    // tile starts and virtual starts, in shared memory when they fit (the
    // planner's searches then stay on chip)
    __shared__ int32_t s_wts[kPlanRows + 1], s_vs[kPlanRows + 1];
    const bool cached = a.num_reqs <= kPlanRows;
    int carry = 0;
    for (int base = 0; base < a.num_reqs; base += kPrepThreads) {
      const int b = base + threadIdx.x;
      int tiles = 0;
      if (b < a.num_reqs) {
        int maxlen = 0;
        for (int g = 0; g < G; ++g) {
          const int64_t r = static_cast<int64_t>(b) * G + g;
          const int len = static_cast<int>(clamp_len(raw_row_len(a, r), a.bt_width, a.err, true));
          row_len[r] = len;
          const bool active = a.score_all ? len > 0 : len > a.topk;
          if (active) maxlen = max(maxlen, len);
        }
        tiles = (maxlen + kTileKeys - 1) / kTileKeys;
        wr[b] = WorkRow{b, b * G, G, maxlen};
        seg_counter[b] = 0;
      }
      int total;
      const int excl = block_exclusive_scan(tiles, &total);
      if (b < a.num_reqs) {
        wts[b] = carry + excl;
        if (cached) s_wts[b] = carry + excl;
      }
      carry += total;
    }
    if (threadIdx.x == 0) {
      wts[a.num_reqs] = carry;
      if (cached) s_wts[a.num_reqs] = carry;
    }
    const int32_t* pw = cached ? s_wts : wts;
    int32_t* pv = cached ? s_vs : row_vs;
    int penalty = a.row_penalty;
    const int share = carry / max(1, min(a.num_ctas, carry));  // tiles per CTA
    if (a.row_penalty_div > 0 && share >= 64) penalty += share / a.row_penalty_div;
    row_virtual_starts(pw, a.num_reqs, penalty, pv);
    plan_ctas(pw, pv, a.num_reqs, a.num_ctas, cta_tile, cta_row, row_ctas);
    return;
  }
  zero_words(row_hist, row_hist_words);
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x - 1) * kPrepThreads + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x - 1) * kPrepThreads) >> 5;
  quantize_tasks<true>(a.q, a.w, 0, rows * kHeads, q8img, wprime, gw, nw);
  if (!a.score_all || a.out_val) {
    // top k: rows of <= k keys are the causal row; values: rows of no keys
    // are empty (the others are all scored)
    const int64_t short_len = a.score_all ? 0 : a.topk;
    for (int64_t r = gw; r < rows; r += nw) {
      const int64_t len = clamp_len(raw_row_len(a, r), a.bt_width, a.err, false);
      if (len > short_len) continue;
      int32_t* o = a.out_idx + r * a.topk;
      for (int i = lane; i < a.topk; i += 32) o[i] = i < len ? i : -1;
      if (a.out_val)
        for (int i = lane; i < a.topk; i += 32) a.out_val[r * a.topk + i] = -INFINITY;
    }
  }
}

// Request owning global query row `row` among requests [r0, r1).
__device__ __forceinline__ int find_request(const int32_t* qsl, int r0, int r1, int64_t row) {
  int lo = r0, hi = r1 - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qsl[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int64_t prefill_len(const PrefillPrepArgs& a, int r, int64_t row,
                                               bool report) {
  const int64_t qs = a.qsl[r], qe = a.qsl[r + 1];
  const int64_t v = static_cast<int64_t>(a.seq_lens[r]) - (qe - qs) + 1 + (row - qs);
  return clamp_len(index_key_count(v, a.compress_ratio, a.dcp_rank, a.dcp_world, a.dcp_interleave),
                   a.bt_width, a.err, report);
}

// Block 0: work rows of the chunk (up to two consecutive queries of one
// request each), their tile prefix and zeroed segment counters. Other blocks:
// row lengths, q quantisation and the causal rows of short queries.
__global__ void __launch_bounds__(kPrepThreads) prefill_prep_kernel(
    PrefillPrepArgs a, WorkRow* __restrict__ wr, int32_t* __restrict__ wts,
    int32_t* __restrict__ row_len, int32_t* __restrict__ seg_counter, uint8_t* __restrict__ q8img,
    float* __restrict__ wprime, uint32_t* __restrict__ row_hist, size_t row_hist_words,
    int32_t* __restrict__ cta_row, int32_t* __restrict__ cta_tile, int32_t* __restrict__ row_vs,
    int2* __restrict__ row_ctas) {
  pdl_trigger();
  pdl_wait();
  constexpr int G = 2;
  const int64_t rows = a.row_hi - a.row_lo;
  if (blockIdx.x == 0) {
    // requests in batches of kPrepThreads: a scan of their work-row counts,
    // then every thread fills work rows of the batch
    __shared__ int s_off[kPrepThreads + 1];
    __shared__ int64_t s_lo[kPrepThreads], s_hi[kPrepThreads];
    int carry = 0;
    for (int base = a.req_begin; base < a.req_end; base += kPrepThreads) {
      const int r = base + threadIdx.x;
      int nw = 0;
      int64_t lo = 0, hi = 0;
      if (r < a.req_end) {
        lo = max(static_cast<int64_t>(a.qsl[r]), a.row_lo);
        hi = min(static_cast<int64_t>(a.qsl[r + 1]), a.row_hi);
        nw = hi > lo ? static_cast<int>((hi - lo + G - 1) / G) : 0;
      }
      int total;
      const int excl = block_exclusive_scan(nw, &total);
      s_off[threadIdx.x] = excl;
      s_lo[threadIdx.x] = lo;
      s_hi[threadIdx.x] = hi;
      __syncthreads();
      const int nreq = min(kPrepThreads, a.req_end - base);
      for (int i = threadIdx.x; i < total; i += kPrepThreads) {
        const int idx = carry + i;
        if (idx >= a.num_wr) {
          set_error(a.err, IDX_DEV_OVERFLOW);
          break;
        }
        int k0 = 0, k1 = nreq - 1;  // the request of batch work row i
        while (k0 < k1) {
          const int mid = (k0 + k1 + 1) >> 1;
          if (s_off[mid] <= i) k0 = mid;
          else k1 = mid - 1;
        }
        const int rq = base + k0;
        const int64_t first = s_lo[k0] + static_cast<int64_t>(i - s_off[k0]) * G;
        const int ntok = static_cast<int>(min(static_cast<int64_t>(G), s_hi[k0] - first));
        int maxlen = 0;
        for (int g = 0; g < ntok; ++g) {
          const int len = static_cast<int>(prefill_len(a, rq, first + g, true));
          if (len > (a.out_val ? 0 : a.topk)) maxlen = max(maxlen, len);
        }
        wr[idx] = WorkRow{rq, static_cast<int32_t>(first - a.row_lo), ntok, maxlen};
        wts[idx] = (maxlen + kTileKeys - 1) / kTileKeys;  // tile count, scanned below
        seg_counter[idx] = 0;
      }
      carry += total;
      __syncthreads();
    }
    if (carry != a.num_wr && threadIdx.x == 0) set_error(a.err, IDX_DEV_OVERFLOW);
    for (int idx = carry + threadIdx.x; idx < a.num_wr; idx += kPrepThreads) {
      wr[idx] = WorkRow{a.req_begin, 0, 0, 0};
      wts[idx] = 0;
      seg_counter[idx] = 0;
    }
    __syncthreads();
    int run = 0;
    for (int base = 0; base < a.num_wr; base += kPrepThreads) {
      const int idx = base + threadIdx.x;
      const int t = idx < a.num_wr ? wts[idx] : 0;
      int total;
      const int excl = block_exclusive_scan(t, &total);
      if (idx < a.num_wr) wts[idx] = run + excl;
      run += total;
    }
    if (threadIdx.x == 0) wts[a.num_wr] = run;
    row_virtual_starts(wts, a.num_wr, a.row_penalty, row_vs);
    plan_ctas(wts, row_vs, a.num_wr, a.num_ctas, cta_tile, cta_row, row_ctas);
    return;
  }
  zero_words(row_hist, row_hist_words);
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x - 1) * kPrepThreads + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x - 1) * kPrepThreads) >> 5;
  for (int64_t lr = gw; lr < rows; lr += nw) {
    const int64_t row = a.row_lo + lr;
    const int r = find_request(a.qsl, a.req_begin, a.req_end, row);
    const int64_t len = prefill_len(a, r, row, false);
    if (lane == 0) row_len[lr] = static_cast<int32_t>(len);
    // top k: queries of <= k keys are the causal row; values: queries of no
    // keys are empty (the others are all scored)
    if (len <= (a.out_val ? 0 : a.topk)) {
      int32_t* o = a.out_idx + row * a.topk;
      for (int i = lane; i < a.topk; i += 32) o[i] = i < len ? i : -1;
      if (a.out_val)
        for (int i = lane; i < a.topk; i += 32) a.out_val[row * a.topk + i] = -INFINITY;
    }
  }
  quantize_tasks<true>(a.q, a.w, a.row_lo * kHeads, rows * kHeads, q8img, wprime, gw, nw);
}

// Row expansion. One warp per request: it writes the request's token rows and
// copies its block-table row to each of them.
__global__ void __launch_bounds__(kPrepThreads) expand_kernel(
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ decode_lens,
    int32_t num_reqs, int32_t next_n, const int32_t* __restrict__ bt, int64_t bt_stride,
    int32_t bt_width, int32_t mode, int32_t* __restrict__ row_lens, int32_t* __restrict__ row_bt,
    int64_t out_stride, int64_t num_out_rows, uint32_t* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ int64_t s_carry, s_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b0 = blockIdx.x * kPrepWarps;
  const int b = b0 + warp;
  int64_t start = 0;
  if (mode == 1) {
    // tokens before this block's first request, and in all requests
    int64_t before = 0, all = 0;
    for (int i = threadIdx.x; i < num_reqs; i += kPrepThreads) {
      const int64_t d = decode_lens[i];
      all += d;
      if (i < b0) before += d;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, off);
      all += __shfl_xor_sync(0xffffffffu, all, off);
    }
    __shared__ int64_t s_before[kPrepWarps], s_all[kPrepWarps];
    if (lane == 0) {
      s_before[warp] = before;
      s_all[warp] = all;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int64_t x = 0, y = 0;
      for (int i = 0; i < kPrepWarps; ++i) {
        x += s_before[i];
        y += s_all[i];
      }
      s_carry = x;
      s_total = y;
    }
    __syncthreads();
    int64_t mine = 0;
    if (lane < warp && b0 + lane < num_reqs) mine = decode_lens[b0 + lane];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
    start = s_carry + mine;
  }
  if (b < num_reqs) {
    const int32_t L = seq_lens[b];
    const int32_t d = decode_lens[b];
    const int32_t nrows = mode == 0 ? next_n : d;
    for (int j = 0; j < nrows; ++j) {
      const int64_t row = mode == 0 ? static_cast<int64_t>(b) * next_n + j : start + j;
      if (row >= num_out_rows) {
        if (lane == 0) set_error(err, IDX_DEV_OVERFLOW);
        break;
      }
      if (lane == 0) row_lens[row] = (j < d) ? L - d + j + 1 : 0;
      if (row_bt) {
        const int32_t* src = bt + static_cast<int64_t>(b) * bt_stride;
        int32_t* dst = row_bt + row * out_stride;
        for (int c = lane; c < bt_width; c += 32) dst[c] = src[c];
      }
    }
  }
  if (mode == 1) {
    // rows after the last token: len 0 and block-table column 0 zeroed
    const int64_t first = s_total;
    for (int64_t row = first + static_cast<int64_t>(blockIdx.x) * kPrepThreads + threadIdx.x;
         row < num_out_rows; row += static_cast<int64_t>(gridDim.x) * kPrepThreads) {
      row_lens[row] = 0;
      if (row_bt && bt_width > 0) row_bt[row * out_stride] = 0;
    }
  }
}

// Correctly rounded a / b from the correctly rounded reciprocal y = RN(1 / b)
// by Markstein's correction (IBM J. Res. Dev. 34(1), 1990): when q is within
// one ulp of a / b, r = a - b q is exact as one fused multiply-add and
// RN(q + r y) is the correctly rounded quotient. q0 = RN(a y) can be up to
// about 1.5 ulp off (a / b just below a power of two), so one correction
// first brings it within one ulp (its residual is still exact: |q0 - a / b|
// stays within 2 ulp) and a second one rounds it correctly. The residuals
// are exact only without underflow. In the cache insert |a| <= 448 b, so
// nothing overflows; with b >= 2^-100 every quotient of magnitude >= 2^-10
// (the ones an e4m3 code depends on: smaller ones are code 0) has a normal
// a and exact residuals; a smaller b takes the IEEE division.
__device__ __forceinline__ float div_rn_recip(float a, float b, float y) {
  const float q0 = __fmul_rn(a, y);
  const float q1 = __fmaf_rn(__fmaf_rn(-b, q0, a), y, q0);
  return __fmaf_rn(__fmaf_rn(-b, q1, a), y, q1);
}
constexpr float kRecipDivMin = 0x1p-100f;  // smallest divisor of the reciprocal path

// Index-key cache insert: token i's 128 bf16 values are quantised with their
// own fp32 scale amax / 448 (correctly rounded) into e4m3 codes of x / scale
// (correctly rounded quotient, round-to-nearest-even, saturating) and written
// to slot slot_mapping[i] of the paged cache (page slot / 64, token slot % 64;
// values then scales in the page). A negative slot is padding and skipped; a
// slot past the cache sets IDX_DEV_BAD_BLOCK and is skipped; amax == 0 writes
// zero codes and scale 0. One warp per token, four tokens' loads per round.
__global__ void __launch_bounds__(kPrepThreads) insert_keys_kernel(
    const __nv_bfloat16* __restrict__ k, const int64_t* __restrict__ slots, int64_t n,
    uint8_t* __restrict__ cache, int64_t num_pages, uint32_t* err) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * kPrepThreads + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * kPrepThreads) >> 5;
  const int64_t nslot = num_pages * kPageTokens;
  for (int64_t base = gw * 4; base < n; base += nw * 4) {
    uint2 raw[4];
    int64_t sl[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      raw[u] = make_uint2(0u, 0u);
      sl[u] = -1;
      if (base + u < n) {
        raw[u] = *reinterpret_cast<const uint2*>(k + (base + u) * kDim + 4 * lane);
        sl[u] = slots[base + u];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (base + u >= n) break;
      if (sl[u] < 0) continue;  // same slot in every lane: warp-uniform
      if (sl[u] >= nslot) {
        if (lane == 0) set_error(err, IDX_DEV_BAD_BLOCK);
        continue;
      }
      const float x0 = __uint_as_float(raw[u].x << 16);
      const float x1 = __uint_as_float(raw[u].x & 0xffff0000u);
      const float x2 = __uint_as_float(raw[u].y << 16);
      const float x3 = __uint_as_float(raw[u].y & 0xffff0000u);
      float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      float scale = 0.0f;
      uint32_t codes = 0u;
      if (amax > 0.0f) {
        scale = __fdiv_rn(amax, 448.0f);
        float q0, q1, q2, q3;
        if (scale >= kRecipDivMin) {  // warp-uniform (one scale per token)
          const float y = __frcp_rn(scale);
          q0 = div_rn_recip(x0, scale, y);
          q1 = div_rn_recip(x1, scale, y);
          q2 = div_rn_recip(x2, scale, y);
          q3 = div_rn_recip(x3, scale, y);
        } else {
          q0 = __fdiv_rn(x0, scale);
          q1 = __fdiv_rn(x1, scale);
          q2 = __fdiv_rn(x2, scale);
          q3 = __fdiv_rn(x3, scale);
        }
        codes = static_cast<uint32_t>(cvt_e4m3x2(q0, q1)) |
                (static_cast<uint32_t>(cvt_e4m3x2(q2, q3)) << 16);
      }
      uint8_t* page = cache + (sl[u] / kPageTokens) * kPageBytes;
      const int tok = static_cast<int>(sl[u] % kPageTokens);
      *reinterpret_cast<uint32_t*>(page + tok * kDim + 4 * lane) = codes;
      if (lane == 0) *reinterpret_cast<float*>(page + kPageValueBytes + tok * 4) = scale;
    }
  }
}

// Test hook: both quotients of each pair (the insert's and the IEEE one).
__global__ void __launch_bounds__(kPrepThreads) divide_check_kernel(const float* a, const float* b,
                                                                    int64_t n, float* fast,
                                                                    float* ieee) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kPrepThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kPrepThreads + threadIdx.x; i < n;
       i += stride) {
    fast[i] = b[i] >= kRecipDivMin ? div_rn_recip(a[i], b[i], __frcp_rn(b[i]))
                                   : __fdiv_rn(a[i], b[i]);
    ieee[i] = __fdiv_rn(a[i], b[i]);
  }
}

int prep_grid(int64_t work_warps) {
  const int64_t blocks = (work_warps + kPrepWarps - 1) / kPrepWarps;
  const int64_t cap = 8 * static_cast<int64_t>(device_sm_count());
  return static_cast<int>(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

}  // namespace

idx_status launch_expand(const int32_t* seq_lens, const int32_t* decode_lens, int32_t num_reqs,
                         int32_t next_n, const int32_t* bt, int64_t bt_stride, int32_t bt_width,
                         int32_t mode, int32_t* row_lens, int32_t* row_bt, int64_t out_stride,
                         int64_t num_out_rows, uint32_t* err, cudaStream_t s) {
  int grid = (num_reqs + kPrepWarps - 1) / kPrepWarps;
  if (grid < 1) grid = 1;
  return cuda_status(launch_pdl(expand_kernel, grid, kPrepThreads, 0, s, seq_lens, decode_lens, num_reqs,
                    next_n, bt, bt_stride, bt_width, mode, row_lens, row_bt, out_stride,
                    num_out_rows, err));
}

idx_status launch_insert_keys(const __nv_bfloat16* k, const int64_t* slots, int64_t n,
                              uint8_t* cache, int64_t num_pages, uint32_t* err, cudaStream_t s) {
  return cuda_status(launch_pdl(insert_keys_kernel, prep_grid((n + 3) / 4), kPrepThreads, 0, s, k, slots, n,
                    cache, num_pages, err));
}

idx_status launch_divide_check(const float* a, const float* b, int64_t n, float* fast, float* ieee,
                               cudaStream_t s) {
  if (n <= 0) return IDX_OK;
  divide_check_kernel<<<prep_grid((n + 31) / 32), kPrepThreads, 0, s>>>(a, b, n, fast, ieee);
  return cuda_status(cudaGetLastError());
}

idx_status launch_quantize_plain(const __nv_bfloat16* q, const float* w, int64_t rows, uint8_t* q8,
                                 float* wprime, cudaStream_t s) {
  return cuda_status(launch_pdl(quantize_plain_kernel, prep_grid(rows * kHeads), kPrepThreads, 0, s, q, w, rows,
                    q8, wprime));
}

idx_status launch_decode_prep(const DecodePrepArgs& args, uint8_t* ws, const WsLayout& L,
                              cudaStream_t s) {
  DecodePrepArgs a = args;
  const int64_t rows = static_cast<int64_t>(a.num_reqs) * a.next_n;
  const int grid = 1 + prep_grid(rows * kHeads);
  const cudaError_t e = launch_pdl(
      decode_prep_kernel, grid, kPrepThreads, 0, s, a, reinterpret_cast<WorkRow*>(ws + L.wr),
      reinterpret_cast<int32_t*>(ws + L.wr_tile_start),
      reinterpret_cast<int32_t*>(ws + L.row_len), reinterpret_cast<int32_t*>(ws + L.seg_counter),
      ws + L.q8, reinterpret_cast<float*>(ws + L.wprime),
      reinterpret_cast<uint32_t*>(ws + L.row_hist), L.row_hist_words,
      reinterpret_cast<int32_t*>(ws + L.cta_row), reinterpret_cast<int32_t*>(ws + L.cta_tile),
      reinterpret_cast<int32_t*>(ws + L.row_vs), reinterpret_cast<int2*>(ws + L.row_ctas));
  return cuda_status(e);
}

idx_status launch_prefill_prep(const PrefillPrepArgs& args, uint8_t* ws, const WsLayout& L,
                               cudaStream_t s) {
  PrefillPrepArgs a = args;
  const int64_t rows = a.row_hi - a.row_lo;
  const int grid = 1 + prep_grid(rows * kHeads);
  const cudaError_t e = launch_pdl(
      prefill_prep_kernel, grid, kPrepThreads, 0, s, a, reinterpret_cast<WorkRow*>(ws + L.wr),
      reinterpret_cast<int32_t*>(ws + L.wr_tile_start),
      reinterpret_cast<int32_t*>(ws + L.row_len), reinterpret_cast<int32_t*>(ws + L.seg_counter),
      ws + L.q8, reinterpret_cast<float*>(ws + L.wprime),
      reinterpret_cast<uint32_t*>(ws + L.row_hist), L.row_hist_words,
      reinterpret_cast<int32_t*>(ws + L.cta_row), reinterpret_cast<int32_t*>(ws + L.cta_tile),
      reinterpret_cast<int32_t*>(ws + L.row_vs), reinterpret_cast<int2*>(ws + L.row_ctas));
  return cuda_status(e);
}

}  // namespace saib
