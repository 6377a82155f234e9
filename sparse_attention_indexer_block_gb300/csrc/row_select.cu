// Split-row selection: the top k of every work row whose tiles several tile
// streams of the score/select kernel scored.
//
// Each stream that held part of such a row ("segment") published the row's
// candidates it kept (a superset of its part's top k) in its slot, sorted by
// row bin (the top 10 bits of the order-preserving key: sign, exponent, one
// mantissa bit), highest bin first, together with the number of its entries
// at or above every bin, and added its bin counts to the row histogram. This
// kernel runs after the score/select kernel has completed (programmatic
// dependent launch, griddepcontrol.wait), one CTA per (split row, token row),
// so no CTA waits on another:
//   1. the row histogram gives the bin b0 that holds the k-th largest key and
//      the number of keys above it;
//   2. every segment's entries above b0 are a prefix of its slot: they are
//      copied to the output as they are; its entries in b0 follow and are
//      copied to shared memory (a list);
//   3. the list's keys are histogrammed over bits 21..10 (4096 bins): keys
//      above the bin b1 of the still missing ones go out, b1's keys are
//      ranked exactly (key, then list position) and the best of them
//      complete k.
// A cutoff bin too large for the list (many equal logits, for instance) is
// resolved the same way over the slots' b0 ranges, and a b1 bin too large to
// rank over bits 9..0 with tie tickets for keys equal in all 32 bits. Which of
// several equal keys at the k-th value are taken is arbitrary (the method
// leaves it open). The output row holds its k indices in no particular order.
// With values asked for, each index's logit goes out beside it, and rows of
// <= k keys (not causal-filled then) take all their keys, padded with -1.
#include <atomic>

#include "internal.h"

namespace saib {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kListCap = 16384;  // keys of the cutoff bin kept in shared memory
constexpr int kTieCap = 512;     // keys of the second-level bin ranked pairwise
constexpr int kMaxSegs = 1024;   // segments one row may have (tile streams of a launch)
static_assert(kMaxSegs % kSelThreads == 0 && kRowHistBins % kSelThreads == 0, "thread split");

struct Cut {
  int bin, above, count;
};

struct SelShared {
  int scan[kSelWarps][3];
  int64_t seg_base[kMaxSegs];  // first slot entry of each segment
  int seg_gt[kMaxSegs];        // its entries above b0
  int seg_gpre[kMaxSegs];      // entries above b0 in earlier segments
  int seg_epre[kMaxSegs];      // entries in b0 in earlier segments
  Cut cut;
  int nout;     // keys written so far
  int nlist;    // keys copied to a list
  int nticket;  // equal keys taken at the last digit
  int bad;
  int abort_flag;
  int bin1_count;  // keys in the second-level cutoff bin
  int path;        // 1: list, 2: slots; +4: ranked, +8: third level
};

struct SelSmem {
  uint32_t* lkey;  // [kListCap]
  int32_t* lidx;   // [kListCap]
  uint32_t* tkey;  // [kTieCap]
  int32_t* tidx;   // [kTieCap]
  uint32_t* hist;  // [4096]
  SelShared* sh;
};

constexpr size_t kSelSmemBytes =
    static_cast<size_t>(kListCap) * 8 + static_cast<size_t>(kTieCap) * 8 + 4096 * 4 +
    sizeof(SelShared);

__device__ __forceinline__ SelSmem sel_carve(uint8_t* base) {
  SelSmem s;
  s.lkey = reinterpret_cast<uint32_t*>(base);
  s.lidx = reinterpret_cast<int32_t*>(base + kListCap * 4);
  s.tkey = reinterpret_cast<uint32_t*>(base + kListCap * 8);
  s.tidx = reinterpret_cast<int32_t*>(base + kListCap * 8 + kTieCap * 4);
  s.hist = reinterpret_cast<uint32_t*>(base + kListCap * 8 + kTieCap * 8);
  s.sh = reinterpret_cast<SelShared*>(base + kListCap * 8 + kTieCap * 8 + 4096 * 4);
  return s;
}

// Inclusive scan of three ints over the warp's lanes.
__device__ __forceinline__ void warp_scan3(int (&x)[3]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int y = __shfl_up_sync(0xffffffffu, x[i], off);
      if (lane >= off) x[i] += y;
    }
  }
}

// Exclusive scans of three ints per thread in thread order (ex) and their sums
// (tot), for every thread. Three barriers.
__device__ void block_scan3(const int (&v)[3], int (&ex)[3], int (&tot)[3], int (*scratch)[3]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x[3] = {v[0], v[1], v[2]};
  warp_scan3(x);
  if (lane == 31)
#pragma unroll
    for (int i = 0; i < 3; ++i) scratch[warp][i] = x[i];
  __syncthreads();
  if (warp == 0) {
    int y[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) y[i] = lane < kSelWarps ? scratch[lane][i] : 0;
    warp_scan3(y);
    if (lane < kSelWarps)
#pragma unroll
      for (int i = 0; i < 3; ++i) scratch[lane][i] = y[i];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    ex[i] = (warp > 0 ? scratch[warp - 1][i] : 0) + x[i] - v[i];
    tot[i] = scratch[kSelWarps - 1][i];
  }
  __syncthreads();
}

// Bins are counted top-down in thread order: thread t holds c[j] = bin hi - j
// and `ex` keys lie in higher bins. The thread holding the need-th largest key
// records its bin, the count above it and the bin's count in sh->cut.
template <int PER>
__device__ __forceinline__ void claim_cut(const int (&c)[PER], int hi, int ex, int need,
                                          SelShared* sh) {
  int local = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) local += c[j];
  if (ex < need && need <= ex + local) {
    int acc = ex;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      if (acc + c[j] >= need) {
        sh->cut = Cut{hi - j, acc, c[j]};
        break;
      }
      acc += c[j];
    }
  }
}

// Highest bin of thread t when the threads hold PER bins each, top-down.
template <int PER>
__device__ __forceinline__ int top_bin() {
  return kSelThreads * PER - 1 - PER * static_cast<int>(threadIdx.x);
}

// The bin holding the need-th largest key of a kSelThreads * PER-bin
// histogram whose counts thread t holds as c[j] = bin top_bin<PER>() - j, the
// count in higher bins and the bin's own count, in sh->cut for every thread
// (bin -1 and the total count when fewer than `need` keys are counted).
template <int PER>
__device__ void find_cut(const int (&c)[PER], int need, SelShared* sh) {
  int local = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) local += c[j];
  if (threadIdx.x == 0) sh->cut = Cut{-1, 0, 0};
  const int v[3] = {local, 0, 0};
  int ex[3], tot[3];
  block_scan3(v, ex, tot, sh->scan);  // its barriers order the write above
  claim_cut<PER>(c, top_bin<PER>(), ex[0], need, sh);
  if (threadIdx.x == 0 && tot[0] < need) sh->cut = Cut{-1, tot[0], 0};  // no claim then
  __syncthreads();
}

// Calls write(j, pos) for every entry j of the lane flagged in `mask` (bit j),
// pos counted from one shared counter: one atomic per warp for all eight
// entries of its 32 lanes (the ballots are taken twice rather than held).
// All lanes of the warp.
template <class W>
__device__ __forceinline__ void emit8(int* counter, uint32_t mask, W&& write) {
  const int lane = threadIdx.x & 31;
  int total = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) total += __popc(__ballot_sync(0xffffffffu, (mask >> j) & 1u));
  if (total == 0) return;
  int base = 0;
  if (lane == 0) base = atomicAdd(counter, total);
  base = __shfl_sync(0xffffffffu, base, 0);
  const unsigned below = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const unsigned m = __ballot_sync(0xffffffffu, (mask >> j) & 1u);
    if ((mask >> j) & 1u) write(j, base + __popc(m & below));
    base += __popc(m);
  }
}

// Eight entries of one lane: keys, token indices and which of them exist.
struct Batch {
  uint32_t k[8];
  int32_t x[8];
  uint32_t valid;
};

// Largest i < n with pre[i] <= e (pre non-decreasing, pre[0] = 0 <= e): the
// segment of flattened position e.
__device__ __forceinline__ int segment_of(const int* pre, int n, int e) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= e) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Calls f(batch) for entries [0, n) of a shared-memory list, warp-uniformly
// (warp units of 256 entries, lane l holding entries l, l + 32, ...).
template <class F>
__device__ __forceinline__ void for_each_list_batch(const uint32_t* lk, const int32_t* lx, int n,
                                                    F&& f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e0 = warp * 256; e0 < n; e0 += kSelThreads * 8) {
    Batch b;
    b.valid = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + lane + 32 * j;
      const bool in = e < n;
      b.k[j] = in ? lk[e] : 0u;
      b.x[j] = in ? lx[e] : 0;
      b.valid |= in ? 1u << j : 0u;
    }
    f(b);
  }
}

// The row's b0 entries in the slots, flattened in segment order (n of them).
struct BinRanges {
  const uint32_t* key;
  const int32_t* idx;
  const SelShared* sh;
  int nseg, n;
};

// Calls f(batch) for every b0 entry of the row's slots, warp-uniformly (the
// path for cutoff bins larger than the list).
template <class F>
__device__ __forceinline__ void for_each_bin_batch(const BinRanges& r, F&& f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e0 = warp * 256; e0 < r.n; e0 += kSelThreads * 8) {
    Batch b;
    b.valid = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + lane + 32 * j;
      b.k[j] = 0u;
      b.x[j] = 0;
      if (e < r.n) {
        const int i = segment_of(r.sh->seg_epre, r.nseg, e);
        const int64_t src = r.sh->seg_base[i] + r.sh->seg_gt[i] + (e - r.sh->seg_epre[i]);
        b.k[j] = __ldcg(r.key + src);
        b.x[j] = __ldcg(r.idx + src);
        b.valid |= 1u << j;
      }
    }
    f(b);
  }
}

// Selects `need` keys of the bin b0 from the source `visit` hands out (the
// list, or the slots' b0 ranges) into out[0, need): bits 21..10 (4096 bins;
// s.hist is zero on entry), then either an exact rank of the last bin's keys
// or bits 9..0 and tie tickets; with kVals each key's logit goes to ov at
// its index's position. Returns false when the counts disagree.
template <bool kVals, class Visit>
__device__ bool select_in_bin(const SelSmem& s, Visit&& visit, int need, int32_t* out,
                              float* ov) {
  constexpr int P1 = 4096 / kSelThreads, P2 = 1024 / kSelThreads;
  SelShared* sh = s.sh;
  const int t = threadIdx.x;
  visit([&](const Batch& b) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((b.valid >> j) & 1u) atomicAdd(&s.hist[(b.k[j] >> 10) & 4095u], 1u);
  });
  __syncthreads();
  int c1[P1];
#pragma unroll
  for (int j = 0; j < P1; ++j) c1[j] = static_cast<int>(s.hist[top_bin<P1>() - j]);
  if (t == 0) {
    sh->nout = 0;
    sh->nlist = 0;
  }
  find_cut<P1>(c1, need, sh);
  const Cut cut1 = sh->cut;
  if (t == 0) {
    sh->bin1_count = cut1.count;
    sh->path |= cut1.count <= kTieCap ? 4 : 8;
  }
  if (cut1.bin < 0) return false;
  const int need1 = need - cut1.above;  // keys of bin b1 still to take
  const uint32_t b1 = static_cast<uint32_t>(cut1.bin);
  const bool rank = cut1.count <= kTieCap;
  visit([&](const Batch& b) {
    uint32_t gt = 0u, eq = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool in = (b.valid >> j) & 1u;
      const uint32_t d1 = (b.k[j] >> 10) & 4095u;
      gt |= (in && d1 > b1) ? 1u << j : 0u;
      eq |= (rank && in && d1 == b1) ? 1u << j : 0u;
    }
    emit8(&sh->nout, gt, [&](int j, int pos) {
      if (pos < cut1.above) {
        out[pos] = b.x[j];
        if (kVals) ov[pos] = key_float(b.k[j]);
      }
    });
    emit8(&sh->nlist, eq, [&](int j, int pos) {
      if (pos < kTieCap) {
        s.tkey[pos] = b.k[j];
        s.tidx[pos] = b.x[j];
      }
    });
  });
  __syncthreads();
  if (sh->nout != cut1.above || (rank && sh->nlist != cut1.count)) return false;
  int32_t* out1 = out + cut1.above;
  float* ov1 = kVals ? ov + cut1.above : nullptr;
  if (rank) {
    // rank by key, then list position: the first need1 are in
    const int m = cut1.count;
    for (int i = t; i < m; i += kSelThreads) {
      const uint32_t ki = s.tkey[i];
      int r = 0;
      for (int j = 0; j < m; ++j) {
        const uint32_t kj = s.tkey[j];
        r += (kj > ki || (kj == ki && j < i)) ? 1 : 0;
      }
      if (r < need1) {
        out1[r] = s.tidx[i];
        if (kVals) ov1[r] = key_float(ki);
      }
    }
    return true;
  }
  // a large second-level bin: bits 9..0, keys above the bin b2 go out, keys
  // equal in all 32 bits take tickets
  for (int b = t; b < 1024; b += kSelThreads) s.hist[b] = 0u;
  __syncthreads();
  visit([&](const Batch& b) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (((b.valid >> j) & 1u) && ((b.k[j] >> 10) & 4095u) == b1)
        atomicAdd(&s.hist[b.k[j] & 1023u], 1u);
  });
  __syncthreads();
  int c2[P2];
#pragma unroll
  for (int j = 0; j < P2; ++j) c2[j] = static_cast<int>(s.hist[top_bin<P2>() - j]);
  if (t == 0) {
    sh->nout = 0;
    sh->nticket = 0;
  }
  find_cut<P2>(c2, need1, sh);
  const Cut cut2 = sh->cut;
  if (cut2.bin < 0) return false;
  const int need2 = need1 - cut2.above;
  const uint32_t b2 = static_cast<uint32_t>(cut2.bin);
  visit([&](const Batch& b) {
    uint32_t gt = 0u, eq = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool in = ((b.valid >> j) & 1u) && ((b.k[j] >> 10) & 4095u) == b1;
      gt |= (in && (b.k[j] & 1023u) > b2) ? 1u << j : 0u;
      eq |= (in && (b.k[j] & 1023u) == b2) ? 1u << j : 0u;
    }
    emit8(&sh->nout, gt, [&](int j, int pos) {
      if (pos < cut2.above) {
        out1[pos] = b.x[j];
        if (kVals) ov1[pos] = key_float(b.k[j]);
      }
    });
    emit8(&sh->nticket, eq, [&](int j, int pos) {
      if (pos < need2) {
        out1[cut2.above + pos] = b.x[j];
        if (kVals) ov1[cut2.above + pos] = key_float(b.k[j]);
      }
    });
  });
  __syncthreads();
  return sh->nout == cut2.above && sh->nticket >= need2;
}

template <bool kVals>
__global__ void __launch_bounds__(kSelThreads, 1) row_select_kernel(const RowSelectParams p) {
  constexpr int P0 = kRowHistBins / kSelThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~static_cast<uintptr_t>(15));
  const SelSmem s = sel_carve(base);
  SelShared* sh = s.sh;
  const int t = threadIdx.x;
  uint64_t* tr = (p.trace && t == 0) ? p.trace + static_cast<int64_t>(blockIdx.x) * kSelTrSlots
                                     : nullptr;
  if (tr) tr[kSelTrEntry] = globaltimer_ns();
  for (int b = t; b < 4096; b += kSelThreads) s.hist[b] = 0u;
  pdl_trigger();
  pdl_wait();  // the score/select kernel has completed; its slots are visible
  if (tr) tr[kSelTrWaited] = globaltimer_ns();

  // this CTA's split row and token row
  const int g = static_cast<int>(blockIdx.x) % p.G;
  const int slot_i = static_cast<int>(blockIdx.x) / p.G;
  int w;
  if (p.num_wr <= p.streams) {
    w = slot_i;
    if (w >= p.num_wr) return;
  } else {
    // split rows start in different streams: the one starting in stream v
    // (if any) also holds stream v + 1's first tile
    const int v = slot_i;
    const int nV = static_cast<int>(min(static_cast<int64_t>(p.streams),
                                        static_cast<int64_t>(p.wr_tile_start[p.num_wr])));
    if (v + 1 >= nV) return;
    w = p.cta_row[v + 1];
    if (p.row_ctas[w].x != v) return;
  }
  const int2 rc = p.row_ctas[w];
  if (rc.y <= rc.x) return;  // no tiles, or scored whole by one stream
  const WorkRow wr = p.wr[w];
  if (g >= wr.ntok) return;
  const int K = p.topk;
  // a row of <= k keys: causal-filled by the prep kernel, or (values) all
  // its keys taken here
  const bool take_all = p.row_len[wr.row0 + g] <= K;
  if (!kVals && take_all) return;
  const int nseg = rc.y - rc.x + 1;
  if (nseg > kMaxSegs) {
    if (t == 0) set_error(p.dev_error, IDX_DEV_INTERNAL);
    return;
  }
  int32_t* out = p.out_idx + (p.out_row_base + wr.row0 + g) * static_cast<int64_t>(K);
  float* ov = kVals ? p.out_val + (p.out_row_base + wr.row0 + g) * static_cast<int64_t>(K)
                    : nullptr;
  // the first segment is the first stream's first row's only when the row
  // starts at that stream's first tile; later segments always are
  const bool first_is_first_row = p.cta_row[rc.x] == w;

  // level 0: the row histogram (thread t holds bins top_bin<P0>() - j)
  const int64_t hrow = p.num_wr <= p.streams ? w : rc.x;
  const uint32_t* rh = p.row_hist + (hrow * p.G + g) * kRowHistBins;
  int c0[P0];
#pragma unroll
  for (int j = 0; j < P0; ++j) c0[j] = static_cast<int>(__ldcg(&rh[top_bin<P0>() - j]));
  // every segment has published: each of a segment's G epilogue groups (one
  // per token row) counts in once (the wait is the test hook's: it asks for
  // one more than there are and must give up)
  if (t == 0) {
    sh->abort_flag = 0;
    int ok = 1;
    const int expected = nseg * p.G;
    if (p.stall) {
      ok = wait_count(&p.seg_counter[w], expected + 1, &sh->abort_flag, p.dev_error, p.wait_ns) ? 1
                                                                                               : 0;
    } else if (__ldcg(&p.seg_counter[w]) != expected) {
      // a segment missing: the score/select kernel gave up (timeout), else a bug
      const uint32_t e = p.dev_error ? *reinterpret_cast<volatile uint32_t*>(p.dev_error) : 0u;
      if (!(e & IDX_DEV_TIMEOUT)) set_error(p.dev_error, IDX_DEV_INTERNAL);
      ok = 0;
    }
    sh->bad = ok ? 0 : 1;
    sh->nout = 0;
    sh->nlist = 0;
    sh->bin1_count = -1;
  }
  find_cut<P0>(c0, K, sh);
  if (tr) tr[kSelTrPrefix] = globaltimer_ns();
  if (sh->bad) return;
  const Cut cut0 = sh->cut;
  if (cut0.bin < 0 && !(kVals && take_all)) {
    if (t == 0) set_error(p.dev_error, IDX_DEV_INTERNAL);
    return;
  }
  const int b0 = cut0.bin;  // -1: fewer than k keys (values mode), all of them go out
  // each segment's entries above b0 and in b0 (prefixes of its sorted slot),
  // and their prefixes over the segments
  int ngt = 0, neq = 0;
  for (int i0 = 0; i0 < nseg; i0 += kSelThreads) {
    const int i = i0 + t;
    int gt = 0, eq = 0;
    if (i < nseg) {
      const int64_t slot = segment_slot(rc.x + i, i > 0 || first_is_first_row);
      const uint32_t* cum = p.seg_cum + (slot * p.G + g) * kRowHistBins;
      const int at = min(static_cast<int>(__ldcg(&cum[kVals ? max(b0, 0) : b0])), p.slot_cap);
      gt = b0 + 1 < kRowHistBins ? min(static_cast<int>(__ldcg(&cum[b0 + 1])), at) : 0;
      eq = at - gt;
      sh->seg_base[i] = (slot * p.G + g) * p.slot_cap;
      sh->seg_gt[i] = gt;
    }
    const int v[3] = {gt, eq, 0};
    int ex[3], tot[3];
    block_scan3(v, ex, tot, sh->scan);
    if (i < nseg) {
      sh->seg_gpre[i] = ngt + ex[0];
      sh->seg_epre[i] = neq + ex[1];
    }
    ngt += tot[0];
    neq += tot[1];
  }
  __syncthreads();
  if (ngt != cut0.above || neq != cut0.count) {
    if (t == 0) set_error(p.dev_error, IDX_DEV_INTERNAL);
    return;
  }
  const bool list = cut0.count <= kListCap;
  if (t == 0) sh->path = list ? 1 : 2;
  if (tr) {
    tr[kSelTrCut0] = globaltimer_ns();
    tr[kSelTrCand] = static_cast<uint64_t>(cut0.above);
    tr[kSelTrBin0] = static_cast<uint64_t>(cut0.count);
    tr[kSelTrSegs] = static_cast<uint64_t>(nseg);
  }
  // keys above b0 straight to the output, b0's keys to the list: flattened
  // positions [0, ngt) and [ngt, ngt + nl), four per thread in flight
  const int nl = list ? neq : 0;
  for (int e0 = t; e0 < ngt + nl; e0 += 4 * kSelThreads) {
    int64_t src[4];
    int dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * kSelThreads;
      dst[u] = -1;
      src[u] = 0;
      if (e < ngt) {
        const int i = segment_of(sh->seg_gpre, nseg, e);
        src[u] = sh->seg_base[i] + (e - sh->seg_gpre[i]);
        dst[u] = e;
      } else if (e < ngt + nl) {
        const int el = e - ngt;
        const int i = segment_of(sh->seg_epre, nseg, el);
        src[u] = sh->seg_base[i] + sh->seg_gt[i] + (el - sh->seg_epre[i]);
        dst[u] = e;
      }
    }
    int32_t x[4];
    uint32_t k[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      x[u] = dst[u] >= 0 ? __ldcg(p.slot_idx + src[u]) : 0;
      k[u] = (kVals ? dst[u] >= 0 : dst[u] >= ngt) ? __ldcg(p.slot_key + src[u]) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (dst[u] < 0) continue;
      if (dst[u] < ngt) {
        out[dst[u]] = x[u];
        if (kVals) ov[dst[u]] = key_float(k[u]);
      } else {
        s.lkey[dst[u] - ngt] = k[u];
        s.lidx[dst[u] - ngt] = x[u];
      }
    }
  }
  __syncthreads();
  if (tr) tr[kSelTrEmit0] = globaltimer_ns();
  const int need0 = K - ngt;
  if (kVals && b0 < 0) {  // every key is out: pad
    for (int e = ngt + t; e < K; e += kSelThreads) {
      out[e] = -1;
      ov[e] = -INFINITY;
    }
    return;
  }
  bool ok;
  if (list) {
    ok = select_in_bin<kVals>(
        s, [&](auto&& f) { for_each_list_batch(s.lkey, s.lidx, neq, f); }, need0, out + ngt,
        kVals ? ov + ngt : nullptr);
  } else {
    const BinRanges r{p.slot_key, p.slot_idx, sh, nseg, neq};
    ok = select_in_bin<kVals>(s, [&](auto&& f) { for_each_bin_batch(r, f); }, need0, out + ngt,
                              kVals ? ov + ngt : nullptr);
  }
  if (!ok && t == 0) set_error(p.dev_error, IDX_DEV_INTERNAL);
  if (tr) {
    tr[kSelTrEnd] = globaltimer_ns();
    tr[kSelTrBin1] = static_cast<uint64_t>(static_cast<int64_t>(sh->bin1_count));
    tr[kSelTrPath] = static_cast<uint64_t>(sh->path);
  }
}

}  // namespace

idx_status launch_row_select(const RowSelectParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) return IDX_OK;
  static std::atomic<bool> configured[2][kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidDevice);
  const size_t smem = kSelSmemBytes + 16;
  const int vals = p.out_val ? 1 : 0;
  auto kernel = vals ? row_select_kernel<true> : row_select_kernel<false>;
  if (dev >= kMaxDevices || !configured[vals][dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < kMaxDevices) configured[vals][dev].store(true, std::memory_order_release);
  }
  return cuda_status(launch_pdl(kernel, grid, kSelThreads, smem, s, p));
}

}  // namespace saib
