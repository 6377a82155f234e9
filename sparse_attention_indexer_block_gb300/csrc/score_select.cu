// Score + select: the persistent kernel of the indexer.
//
// Every CTA (one per SM) owns a contiguous range of 128-key tiles of the
// global tile sequence (work rows in order, each work row cut into
// ceil(maxlen / 128) tiles). Per CTA, warp-specialised:
//   warp 0  TMA producer: two 64-token pages per tile (8 KB of fp8 keys via a
//           3-D tensor map with the 128-byte swizzle, 256 B of fp32 scales via
//           a bulk copy each) into a ring of shared-memory stages; the work
//           row's fp8 q image (G x 8 KB) into one of two q slots.
//   warp 1  MMA issuer: D[128 keys x 64G] = K_tile[128 x 128] . Q[64G x 128]^T
//           as four tcgen05 kind::f8f6f4 MMAs (K = 32 each) into one of two
//           tensor-memory accumulators.
//   warps 2-5  epilogue: each thread owns one key (one TMEM lane), loads its
//           64 head dots per token, applies ReLU, the folded head weights
//           w * sq and the key's scale, and feeds the logit to a streaming
//           top-k: a shared-memory candidate buffer per token, a threshold
//           below which keys are dropped, and a radix select that shrinks the
//           buffer back to k when it fills. No logits row leaves the SM.
// A work row covered by several CTAs is a set of segments: each segment's
// (<= k) candidates go to a workspace slot and the CTA that finishes the last
// segment merges the slots through the same buffer (an atomic counter per work
// row decides which CTA that is).
//
// Scoring (the method's statement; the pages name the kernel only):
//   logit[t, s] = sum_h w[t, h] ReLU(scale_s (q[t, h] . k_s))
//               = scale_s * sum_h (w[t, h] sq[t, h]) ReLU(q8[t, h] . k8_s),
// since scale_s >= 0 and q = q8 * sq per (token, head).
#include <atomic>

#include "internal.h"

namespace saib {

namespace {

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kEpiBarrier = 1;       // named barrier id of the epilogue warps
constexpr int kTeardownBarrier = 2;  // used once, by all warps, before TMEM is freed
constexpr int kSetupBarrier = 3;     // used once, by all warps, after barrier init and TMEM alloc

template <int G>
struct Cfg {
  static constexpr int N = 64 * G;
  // next_n = 1 runs two CTAs per SM (one's selection work overlaps the other's
  // streaming); wider work rows need the shared memory of a whole SM.
  static constexpr int kCtasPerSm = G == 1 ? 2 : 1;
  static constexpr int kStages = G == 1 ? 4 : (G == 2 ? 6 : 4);
  static constexpr int kCap = candidate_capacity(G);  // candidates per token row
  static constexpr int kRegion = kCap / 4;          // per-warp append region
  static constexpr int kPer = kRegion / 32;         // region entries per lane
  // a full buffer is cut to at most k + kSlack entries (whichever bucket
  // boundary the radix search reaches first)
  static constexpr int kSlack = kCap / 24;
  static constexpr int kHistBins = 1024;
  static constexpr uint32_t kTmemCols = 2 * N <= 128 ? 128u : (2 * N <= 256 ? 256u : 512u);
  static constexpr uint32_t kIdesc = f8_idesc(128, N);
  static constexpr int kKvOff = 0;
  static constexpr int kQOff = kKvOff + kStages * 16384;
  static constexpr int kScaleOff = kQOff + 2 * G * kQRowBytes;
  static constexpr int kCandKeyOff = kScaleOff + kStages * 512;
  static constexpr int kCandIdxOff = kCandKeyOff + G * kCap * 4;
  static constexpr int kWpOff = kCandIdxOff + G * kCap * 4;
  static constexpr int kHistOff = kWpOff + G * 256;
  static constexpr int kBarOff = kHistOff + kHistBins * 4;
  static constexpr int kNumBars = 2 * kStages + 10;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kTraceOff = kMiscOff + 256;  // trace slots (kept in shared memory)
  static constexpr int kSmemBytes = kTraceOff + kTrSlots * 8 + 1024;  // + alignment slack
  static_assert(kCap % kEpiThreads == 0, "capacity");
  static_assert(kCap >= IDX_MAX_TOPK, "a slot must hold any k");
  static_assert(kSmemBytes * kCtasPerSm + 1024 * kCtasPerSm <= 233472, "shared memory");
};

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  int cnt[4];
  uint32_t thr[4];
  int sel_out, sel_tie;
  int bucket, above, bcount;
  int is_last;
  int vote[2][4];
  int scan[4];
  uint32_t rmin[4], rmax[4];
  int cut_n, fallback;
  int epi_done;
  int wcnt[4][4];  // [token][epilogue warp] entries in the warp's region
  int staged_uses;  // phases of `staged` used so far
  int pending_row;  // work row this CTA must merge once its own tiles are done, or -1
};
static_assert(sizeof(Misc) <= 256, "misc block");

struct Smem {
  uint8_t* kv;
  uint8_t* q;
  float* scales;
  uint32_t* ckey;
  int32_t* cidx;
  float* wp;
  uint32_t* hist;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;   // [2]
  uint64_t* tempty;  // [2]
  uint64_t* qfull;   // [2]
  uint64_t* qempty;  // [2]
  uint64_t* done;
  uint64_t* staged;  // completion of the bulk copies that stage a merge's candidates
  Misc* misc;
  uint64_t* trace;   // this CTA's trace slots (shared memory, copied out at exit), or nullptr
};

template <int G>
__device__ __forceinline__ Smem carve(uint8_t* base) {
  using C = Cfg<G>;
  Smem s;
  s.kv = base + C::kKvOff;
  s.q = base + C::kQOff;
  s.scales = reinterpret_cast<float*>(base + C::kScaleOff);
  s.ckey = reinterpret_cast<uint32_t*>(base + C::kCandKeyOff);
  s.cidx = reinterpret_cast<int32_t*>(base + C::kCandIdxOff);
  s.wp = reinterpret_cast<float*>(base + C::kWpOff);
  s.hist = reinterpret_cast<uint32_t*>(base + C::kHistOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  s.full = bars;
  s.empty = bars + C::kStages;
  s.tfull = bars + 2 * C::kStages;
  s.tempty = s.tfull + 2;
  s.qfull = s.tempty + 2;
  s.qempty = s.qfull + 2;
  s.done = s.qempty + 2;
  s.staged = s.done + 1;
  s.misc = reinterpret_cast<Misc*>(base + C::kMiscOff);
  return s;
}

// Row histogram over the top 10 bits of the order-preserving key: sign, the
// 8 exponent bits and the leading mantissa bit (bins of half a binade).
constexpr int kRowHistBins = 1024;
__device__ __forceinline__ int row_bin(uint32_t key) { return static_cast<int>(key >> 22); }


__device__ __forceinline__ void trace_set(const Smem& s, int slot, uint64_t v) {
  if (s.trace) s.trace[slot] = v;
}

// ---------------------------------------------------------------------------
// producer (one thread)
// ---------------------------------------------------------------------------
template <int G>
__device__ void producer(const ScoreParams& p, const CUtensorMap* map, const Smem& s, int64_t t0,
                         int64_t t1) {
  using C = Cfg<G>;
  volatile int* abort_flag = &s.misc->abort_flag;
  int stage = 0;
  uint32_t phase = 0;
  int last_par[C::kStages];
#pragma unroll
  for (int i = 0; i < C::kStages; ++i) last_par[i] = -1;
  uint32_t qn[2] = {0, 0};
  int qslot = 0;

  int w = p.cta_row[blockIdx.x];
  int64_t rs = p.wr_tile_start[w], re = p.wr_tile_start[w + 1];
  WorkRow wr = p.wr[w];
  bool ok = true;

  auto load_q = [&]() -> bool {
    if (qn[qslot] > 0 && !mbar_wait(&s.qempty[qslot], (qn[qslot] - 1) & 1, abort_flag, p.dev_error))
      return false;
    const uint32_t bytes = static_cast<uint32_t>(wr.ntok) * kQRowBytes;
    mbar_arrive_expect_tx(&s.qfull[qslot], bytes);
    if (bytes)
      bulk_load(s.q + qslot * G * kQRowBytes, p.q8 + static_cast<int64_t>(wr.row0) * kQRowBytes,
                bytes, &s.qfull[qslot]);
    ++qn[qslot];
    return true;
  };

  ok = load_q();
  const int32_t* bt_row = p.block_table + static_cast<int64_t>(wr.req) * p.bt_stride;
  int npages = (wr.maxlen + kPageTokens - 1) / kPageTokens;

  for (int64_t t = t0; ok && t < t1; ++t) {
    if (*abort_flag) break;
    if (t >= re) {
      do {
        ++w;
        re = p.wr_tile_start[w + 1];
      } while (t >= re);
      rs = p.wr_tile_start[w];
      wr = p.wr[w];
      qslot ^= 1;
      if (!load_q()) break;
      bt_row = p.block_table + static_cast<int64_t>(wr.req) * p.bt_stride;
      npages = (wr.maxlen + kPageTokens - 1) / kPageTokens;
    }
    const int i = static_cast<int>(t - rs);
    if (!mbar_wait(&s.empty[stage], phase ^ 1, abort_flag, p.dev_error)) break;
    int pid[2];
    uint32_t bytes = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      pid[j] = -1;
      const int pg = 2 * i + j;
      if (pg < npages) {
        const int32_t v = bt_row[pg];
        if (v >= 0 && static_cast<int64_t>(v) < p.num_pages) {
          pid[j] = v;
          bytes += kPageValueBytes + 256;
        } else {
          set_error(p.dev_error, IDX_DEV_BAD_BLOCK);
        }
      }
    }
    if (t == t0) trace_set(s, kTrFirstTma, globaltimer_ns());
    mbar_arrive_expect_tx(&s.full[stage], bytes);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (pid[j] < 0) continue;
      tma_load_3d(s.kv + stage * 16384 + j * kPageValueBytes, map, 0, 0, pid[j], &s.full[stage]);
      bulk_load(s.scales + stage * 128 + j * 64,
                p.cache + static_cast<int64_t>(pid[j]) * kPageBytes + kPageValueBytes, 256,
                &s.full[stage]);
    }
    last_par[stage] = static_cast<int>(phase);
    if (++stage == C::kStages) {
      stage = 0;
      phase ^= 1;
    }
  }
  trace_set(s, kTrLastTma, globaltimer_ns());
  // Every copy this thread issued lands before the CTA may exit.
  int dummy = 0;
#pragma unroll
  for (int i = 0; i < C::kStages; ++i)
    if (last_par[i] >= 0) mbar_wait(&s.full[i], static_cast<uint32_t>(last_par[i]), &dummy, p.dev_error);
  for (int j = 0; j < 2; ++j)
    if (qn[j] > 0) mbar_wait(&s.qfull[j], (qn[j] - 1) & 1, &dummy, p.dev_error);
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread)
// ---------------------------------------------------------------------------
template <int G>
__device__ void mma_issuer(const ScoreParams& p, const Smem& s, uint32_t tmem, int64_t t0,
                           int64_t t1) {
  using C = Cfg<G>;
  volatile int* abort_flag = &s.misc->abort_flag;
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  uint32_t qn[2] = {0, 0};
  int qslot = 0;
  int w = p.cta_row[blockIdx.x];
  int64_t re = p.wr_tile_start[w + 1];
  bool issued = false;
  bool ok = mbar_wait(&s.qfull[qslot], qn[qslot] & 1, abort_flag, p.dev_error);
  for (int64_t t = t0; ok && t < t1; ++t) {
    if (*abort_flag) break;
    if (t >= re) {
      mma_commit(&s.qempty[qslot]);  // q slot free once this row's MMAs finish
      ++qn[qslot];
      do {
        ++w;
        re = p.wr_tile_start[w + 1];
      } while (t >= re);
      qslot ^= 1;
      if (!mbar_wait(&s.qfull[qslot], qn[qslot] & 1, abort_flag, p.dev_error)) break;
    }
    if (!mbar_wait(&s.full[stage], phase, abort_flag, p.dev_error)) break;
    if (!mbar_wait(&s.tempty[acc], acc_phase ^ 1, abort_flag, p.dev_error)) break;
    tc_fence_after();
    if (t == t0) trace_set(s, kTrFirstMma, globaltimer_ns());
    const uint32_t a_base = smem_u32(s.kv + stage * 16384);
    const uint32_t b_base = smem_u32(s.q + qslot * G * kQRowBytes);
    const uint32_t d = tmem + static_cast<uint32_t>(acc * C::N);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f8(d, sw128_kmajor_desc(a_base + kk * 32), sw128_kmajor_desc(b_base + kk * 32),
             C::kIdesc, kk > 0 ? 1u : 0u);
    mma_commit(&s.empty[stage]);
    mma_commit(&s.tfull[acc]);
    issued = true;
    if (++stage == C::kStages) {
      stage = 0;
      phase ^= 1;
    }
    if (++acc == 2) {
      acc = 0;
      acc_phase ^= 1;
    }
  }
  trace_set(s, kTrLastMma, globaltimer_ns());
  if (issued) {
    // all MMAs of this CTA complete before tensor memory is released
    mma_commit(s.done);
    int dummy = 0;
    mbar_wait(s.done, 0, &dummy, p.dev_error);
  }
}

// ---------------------------------------------------------------------------
// epilogue: streaming top-k over a shared-memory candidate buffer
// ---------------------------------------------------------------------------

// Exclusive scan of one int per epilogue thread (in thread order); *total gets
// the sum. Contains one epilogue barrier.
__device__ __forceinline__ int epi_exclusive_scan(Misc* m, int v, int* total) {
  const int lane = threadIdx.x & 31, ew = (threadIdx.x - 64) >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) m->scan[ew] = x;
  named_sync(kEpiBarrier, kEpiThreads);
  int before = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = m->scan[i];
    before += i < ew ? t : 0;
    tot += t;
  }
  *total = tot;
  return before + x - v;
}

// With hist[0, nb) complete (after an epilogue barrier; nb <= 1024): the bin
// holding the `remaining`-th largest key, the number of keys in higher bins and
// the bin's count, for every epilogue thread. Thread et reads (and zeroes)
// bins [nb - (et+1)*per, nb - et*per); a scan in thread order orders the bins
// from the top. The histogram is zero again after.
__device__ __forceinline__ void take_bucket(uint32_t* hist, Misc* m, int nb, int remaining,
                                            int* bucket, int* above, int* bcount) {
  const int et = threadIdx.x - 64;
  const int per = (nb + kEpiThreads - 1) / kEpiThreads;
  const int hi = nb - 1 - et * per;  // thread et: bins [hi - per + 1, hi], from the top
  const int lo = max(hi - per + 1, 0);
  int c[8];
  int local = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = (j < per && hi - j >= lo) ? static_cast<int>(hist[hi - j]) : 0;
    local += c[j];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < per && hi - j >= lo) hist[hi - j] = 0;
  int total;
  const int excl = epi_exclusive_scan(m, local, &total);  // keys in higher bins
  if (excl < remaining && remaining <= excl + local) {
    int acc = excl;
    bool found = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!found && acc + c[j] >= remaining) {
        m->bucket = hi - j;
        m->above = acc;
        m->bcount = c[j];
        found = true;
      }
      acc += c[j];
    }
  }
  named_sync(kEpiBarrier, kEpiThreads);
  *bucket = m->bucket;
  *above = m->above;
  *bcount = m->bcount;
}

// Digit layout of the fixed MSB-first radix select over 32-bit keys: 10, 10,
// 10 and 2 bits.
constexpr int kFixedPasses = 4;
__device__ __forceinline__ int digit_shift(int pass) {
  return pass == 0 ? 22 : (pass == 1 ? 12 : (pass == 2 ? 2 : 0));
}
__device__ __forceinline__ int digit_bins(int pass) { return pass == 3 ? 4 : 1024; }

// Warp-aggregated reservation of one slot per lane with `take` set; returns
// the lane's position (counter base + rank among the taking lanes).
__device__ __forceinline__ int warp_reserve(int* counter, bool take) {
  const int lane = threadIdx.x & 31;
  const unsigned tm = __ballot_sync(0xffffffffu, take);
  if (!tm) return 0;
  const int leader = __ffs(tm) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(tm));
  base = __shfl_sync(0xffffffffu, base, leader);
  return base + __popc(tm & ((1u << lane) - 1u));
}

// The K-th largest among the member keys of all epilogue threads (member j of
// this thread: key u[j] with bit j of `mem` set; K <= member count): an
// MSB-first radix select over v = key - min (10-bit digits below the top bit
// of max - min, so the bins spread over the keys present) with one shared
// histogram (zero on entry and on exit). Result: *mn (min member key), *hi and *pre (the member keys with
// (key - mn) >> hi > pre are in, those equal to pre are tied) and *rem (how
// many tied keys complete K). With slack > 0 the search may stop early at a
// bucket that holds at most `slack` keys beyond K: the whole bucket is then
// taken (*rem = its count), so up to K + slack keys are in. Contains epilogue
// barriers; all epilogue threads.
template <int N>
__device__ void radix_kth(const Smem& s, const uint32_t (&u)[N], uint64_t mem, int K,
                          uint32_t* mn_out, int* hi_out, uint64_t* pre_out, int* rem_out,
                          int slack = 0) {
  const int et = threadIdx.x - 64;
  const int lane = threadIdx.x & 31, ew = et >> 5;
  Misc* m = s.misc;
  uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
  for (int j = 0; j < N; ++j)
    if ((mem >> j) & 1) {
      mn = min(mn, u[j]);
      mx = max(mx, u[j]);
    }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    m->rmin[ew] = mn;
    m->rmax[ew] = mx;
  }
  named_sync(kEpiBarrier, kEpiThreads);
  mn = min(min(m->rmin[0], m->rmin[1]), min(m->rmin[2], m->rmin[3]));
  mx = max(max(m->rmax[0], m->rmax[1]), max(m->rmax[2], m->rmax[3]));
  int hi = mx >= mn ? 32 - __clz(mx - mn) : 0;  // bits of v still to resolve
  uint64_t pre = 0;                              // resolved high part: v >> hi
  int remaining = K;
#pragma unroll 1
  while (hi > 0) {
    const int lo = max(hi - 10, 0);
    const int nb = 1 << (hi - lo);
    const uint64_t ta = (et == 0 && s.trace) ? globaltimer_ns() : 0;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const uint64_t v = u[j] - mn;
      if (((mem >> j) & 1) && (v >> hi) == pre)
        atomicAdd(&s.hist[(v >> lo) & static_cast<uint64_t>(nb - 1)], 1u);
    }
    named_sync(kEpiBarrier, kEpiThreads);
    const uint64_t tb = (et == 0 && s.trace) ? globaltimer_ns() : 0;
    int bucket, above, bcount;
    take_bucket(s.hist, m, nb, remaining, &bucket, &above, &bcount);
    if (et == 0 && s.trace) {
      s.trace[kTrRadixHistNs] += tb - ta;
      s.trace[kTrRadixBucketNs] += globaltimer_ns() - tb;
      s.trace[kTrRadixPasses] += 1;
    }
    pre = (pre << (hi - lo)) | static_cast<uint64_t>(bucket);
    remaining -= above;
    hi = lo;
    if (bcount - remaining <= slack) {  // the whole bin is taken
      remaining = bcount;
      break;
    }
  }
  *mn_out = mn;
  *hi_out = hi;
  *pre_out = pre;
  *rem_out = remaining;
}

// Position p of a packed candidate buffer: buffers are split into four
// per-warp regions (appends need no shared counter); packed entries are dealt
// round-robin over the regions so every region has the same room afterwards.
template <int G>
__device__ __forceinline__ int buf_at(int g, int p) {
  return g * Cfg<G>::kCap + (p & 3) * Cfg<G>::kRegion + (p >> 2);
}

// Packs candidate buffer g (the four regions, counts in wcnt[g][*]) into its
// K largest keys (all of them when there are <= K; ties at the K-th value
// broken arbitrarily): the entries go to registers, radix_kth finds the K-th
// key, one scan gives every kept entry its packed position. The drop
// threshold becomes min + (resolved prefix of the K-th key): keys at or below
// it cannot displace the K kept ones. Sets cnt[g] to the entries kept and
// returns it; all epilogue threads.
template <int G>
__device__ int compact(const Smem& s, int g, int K, int slack = 0) {
  using C = Cfg<G>;
  static_assert(C::kPer <= 64, "member mask");
  const int et = threadIdx.x - 64;
  const int lane = threadIdx.x & 31, ew = et >> 5;
  uint32_t* ck = s.ckey;
  int32_t* ci = s.cidx;
  Misc* m = s.misc;
  const uint64_t tc0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  const int n_w = m->wcnt[g][ew];
  const int n = m->wcnt[g][0] + m->wcnt[g][1] + m->wcnt[g][2] + m->wcnt[g][3];
  uint32_t ku[C::kPer];
  int32_t ki[C::kPer];
  uint64_t mem = 0;
  const int rbase = g * C::kCap + ew * C::kRegion;
#pragma unroll
  for (int j = 0; j < C::kPer; ++j) {
    const int r = j * 32 + lane;
    ku[j] = r < n_w ? ck[rbase + r] : 0u;
    ki[j] = r < n_w ? ci[rbase + r] : 0;
    if (r < n_w) mem |= 1ull << j;
  }
  uint32_t mn = 0;
  int hi = 0, remaining = 0;
  uint64_t pre = 0;
  const bool select = n > K;
  if (select) {
    const uint64_t tr0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
    radix_kth(s, ku, mem, K, &mn, &hi, &pre, &remaining, slack);
    if (et == 0 && s.trace) s.trace[kTrCompactRadixNs] += globaltimer_ns() - tr0;
  }
  // One scan of (tied << 16 | greater) gives every thread the counts before it;
  // tied keys are taken in thread order until `remaining` of them are in.
  int n_gt = 0, n_eq = 0;
#pragma unroll
  for (int j = 0; j < C::kPer; ++j) {
    const bool in = (mem >> j) & 1;
    const uint64_t top = static_cast<uint64_t>(ku[j] - mn) >> hi;
    n_gt += (in && (!select || top > pre)) ? 1 : 0;
    n_eq += (in && select && top == pre) ? 1 : 0;
  }
  int tot;
  const int before = epi_exclusive_scan(m, (n_eq << 16) | n_gt, &tot);
  const int eq_before = before >> 16;
  int take_eq = min(max(remaining - eq_before, 0), n_eq);
  int pos = (before & 0xffff) + min(eq_before, remaining);
  const int kept = (tot & 0xffff) + min(tot >> 16, remaining);
#pragma unroll
  for (int j = 0; j < C::kPer; ++j) {
    const bool in = (mem >> j) & 1;
    const uint64_t top = static_cast<uint64_t>(ku[j] - mn) >> hi;
    bool take = in && (!select || top > pre);
    if (in && select && top == pre && take_eq > 0) {
      take = true;
      --take_eq;
    }
    if (take) {
      ck[buf_at<G>(g, pos)] = ku[j];
      ci[buf_at<G>(g, pos)] = ki[j];
      ++pos;
    }
  }
  named_sync(kEpiBarrier, kEpiThreads);
  if (et == 0) {
    m->cnt[g] = kept;
    if (select) m->thr[g] = max(m->thr[g], mn + static_cast<uint32_t>(pre << hi));
    if (s.trace) {
      s.trace[kTrCompactNs] += globaltimer_ns() - tc0;
      s.trace[kTrCompactN] += 1;
    }
  }
  if (lane == 0) m->wcnt[g][ew] = (kept - ew + 3) >> 2;
  named_sync(kEpiBarrier, kEpiThreads);
  return kept;
}

template <int G>
__device__ void merge_slots(const ScoreParams& p, const Smem& s, int w, int g, int64_t c_first,
                            int64_t c_last, int32_t* out) {
  const int et = threadIdx.x - 64;
  const int K = p.topk;
  Misc* m = s.misc;
  uint32_t prefix = 0, mask = 0;
  int remaining = K;
  int total = 0;
  for (int64_t c = c_first; c <= c_last; ++c) total += __ldcg(&p.slot_count[(c + w) * G + g]);
  if (total > K) {
#pragma unroll 1
    for (int pass = 0; pass < kFixedPasses; ++pass) {
      const int shift = digit_shift(pass), nb = digit_bins(pass);
      for (int64_t c = c_first; c <= c_last; ++c) {
        const int64_t slot = (c + w) * G + g;
        const int n = __ldcg(&p.slot_count[slot]);
        const uint32_t* keys = p.slot_key + slot * p.slot_cap;
#pragma unroll 4
        for (int e = et; e < n; e += kEpiThreads) {
          const uint32_t u = __ldcg(&keys[e]);
          if ((u & mask) == prefix)
            atomicAdd(&s.hist[(u >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
        }
      }
      named_sync(kEpiBarrier, kEpiThreads);
      int bucket, above, bcount;
      take_bucket(s.hist, s.misc, nb, remaining, &bucket, &above, &bcount);
      prefix |= static_cast<uint32_t>(bucket) << shift;
      mask |= static_cast<uint32_t>(nb - 1) << shift;
      remaining -= above;
      if (bcount == remaining) break;
    }
  }
  if (et == 0) {
    m->sel_out = 0;
    m->sel_tie = 0;
  }
  named_sync(kEpiBarrier, kEpiThreads);
  for (int64_t c = c_first; c <= c_last; ++c) {
    const int64_t slot = (c + w) * G + g;
    const int n = __ldcg(&p.slot_count[slot]);
    const uint32_t* keys = p.slot_key + slot * p.slot_cap;
    const int32_t* idxs = p.slot_idx + slot * p.slot_cap;
    for (int e0 = 0; e0 < n; e0 += kEpiThreads) {
      const int e = e0 + et;
      const uint32_t u = e < n ? __ldcg(&keys[e]) : 0u;
      const uint32_t top = u & mask;
      const bool gt = e < n && top > prefix;
      const bool eq = e < n && top == prefix;
      const int tie_rank = warp_reserve(&m->sel_tie, eq);
      const bool take = gt || (eq && tie_rank < remaining);
      const int pos = warp_reserve(&m->sel_out, take);
      if (take && pos < K) out[pos] = __ldcg(&idxs[e]);
    }
  }
  named_sync(kEpiBarrier, kEpiThreads);
  for (int e = m->sel_out + et; e < K; e += kEpiThreads) out[e] = -1;
}

// Entries of token g's buffer sit in four per-warp regions (counts in
// wcnt[g][*]); warp w's lane l visits its region's entries l, l + 32, ...
template <int G>
__device__ __forceinline__ int region_entries(const Smem& s, int g) {
  const int lane = threadIdx.x & 31, ew = (threadIdx.x - 64) >> 5;
  const int nw = s.misc->wcnt[g][ew];
  return lane < nw ? (nw - lane + 31) / 32 : 0;
}

// Output of a row held entirely by this CTA (its buffer holds <= k entries).
template <int G>
__device__ void write_rows(const ScoreParams& p, const Smem& s, const WorkRow& wr,
                           const bool (&active)[G]) {
  using C = Cfg<G>;
  const int et = threadIdx.x - 64;
  const int lane = threadIdx.x & 31, ew = et >> 5;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (!active[g]) continue;
    const int mine = region_entries<G>(s, g);
    int total;
    int pos = epi_exclusive_scan(s.misc, mine, &total);
    int32_t* o = p.out_idx + (p.out_row_base + wr.row0 + g) * p.topk;
    const int32_t* rx = s.cidx + g * C::kCap + ew * C::kRegion;
    for (int j = 0; j < mine; ++j)
      if (pos < p.topk) o[pos++] = rx[lane + 32 * j];
    for (int e = total + et; e < p.topk; e += kEpiThreads) o[e] = -1;
    named_sync(kEpiBarrier, kEpiThreads);
  }
}

// From a row histogram: cut = max(floor, the highest bin whose suffix count
// (keys in bins >= it) reaches K) and above = the count in bins > cut; cut is
// -1 when the histogram holds fewer than K keys and floor < 0.
// Row-histogram bins held by epilogue thread et in the cutoff scans:
// [hi - kCutPer + 1, hi] with hi = kRowHistBins - 1 - et * kCutPer, c[j] = bin hi - j.
constexpr int kCutPer = kRowHistBins / kEpiThreads;
__device__ __forceinline__ int cut_hi() { return kRowHistBins - 1 - (threadIdx.x - 64) * kCutPer; }

__device__ __forceinline__ void load_row_bins(const uint32_t* gh, int (&c)[kCutPer]) {
  const int hi = cut_hi();
#pragma unroll
  for (int j = 0; j < kCutPer; ++j) c[j] = static_cast<int>(__ldcg(&gh[hi - j]));
}

// row_cutoff over counts already held by the threads (c as in load_row_bins).
__device__ __forceinline__ void row_cutoff_vals(const int (&c)[kCutPer], Misc* m, int K, int floor,
                                                int* cut, int* above) {
  const int et = threadIdx.x - 64;
  if (et == 0) {
    m->bucket = -1;
    m->above = 0;
  }
  const int hi = cut_hi();
  int local = 0, local_above_floor = 0;
#pragma unroll
  for (int j = 0; j < kCutPer; ++j) {
    local += c[j];
    local_above_floor += hi - j > floor ? c[j] : 0;
  }
  int total;
  const int excl = epi_exclusive_scan(m, local, &total);  // contains a barrier
  if (excl < K && K <= excl + local) {
    int acc = excl;
#pragma unroll
    for (int j = 0; j < kCutPer; ++j) {
      if (acc + c[j] >= K) {
        m->bucket = hi - j;
        m->above = acc;
        break;
      }
      acc += c[j];
    }
  }
  named_sync(kEpiBarrier, kEpiThreads);
  int cb = m->bucket, ab = m->above;
  named_sync(kEpiBarrier, kEpiThreads);
  if (cb < floor) {
    int tot_above;
    epi_exclusive_scan(m, local_above_floor, &tot_above);
    named_sync(kEpiBarrier, kEpiThreads);
    cb = floor;
    ab = tot_above;
  }
  *cut = cb;
  *above = ab;
}

__device__ __forceinline__ void row_cutoff(const uint32_t* gh, Misc* m, int K, int floor,
                                           int* cut, int* above) {
  int c[kCutPer];
  load_row_bins(gh, c);
  row_cutoff_vals(c, m, K, floor, cut, above);
}

// Merges work row w's segment slots for token g into `out` (K indices).
// The row histogram is complete here (every segment added its keys before it
// counted itself finished), so its cutoff bin is exact. The union of the
// slots' keys is loaded into registers in one batch of independent loads;
// entries in bins above the cutoff are selected outright, radix_kth picks the
// missing ones among the cutoff bin's entries, and the selected entries'
// indices are gathered in a second batch. Unions larger than the register
// batch, or a histogram that disagrees with the slots, go to merge_slots.
template <int G>
__device__ void merge_row(const ScoreParams& p, const Smem& s, int w, int g, int64_t c_first,
                          int64_t c_last, const uint32_t* gh, int32_t* out) {
  constexpr int kMB = 48;  // union entries per thread (6144 per CTA)
  const int et = threadIdx.x - 64;
  const int K = p.topk;
  Misc* m = s.misc;
  const int nseg = static_cast<int>(c_last - c_first + 1);
  // The histogram holds every segment's final buffer, which is exact for all
  // bins above each segment's threshold bin; the row's cutoff is at or above
  // the highest of those bins.
  int floor = et < nseg ? __ldcg(&p.slot_thrbin[(c_first + et + w) * G + g]) : -1;
  floor = __reduce_max_sync(0xffffffffu, floor);
  if ((et & 31) == 0) m->scan[et >> 5] = floor;
  named_sync(kEpiBarrier, kEpiThreads);
  floor = max(max(m->scan[0], m->scan[1]), max(m->scan[2], m->scan[3]));
  named_sync(kEpiBarrier, kEpiThreads);
  const uint64_t tq0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  int cut, above;
  row_cutoff(gh, m, K, floor, &cut, &above);
  const uint64_t tq1 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  if (et == 0 && s.trace) s.trace[kTrMergeCutNs] += tq1 - tq0;
  if (cut < 0 || nseg > kEpiThreads) {
    if (et == 0 && s.trace) s.trace[kTrMergeFallback] += 1;
    merge_slots<G>(p, s, w, g, c_first, c_last, out);
    return;
  }
  // start offsets of the segments' entries in one flat index space, kept in
  // the token's candidate buffer (idle here; the histogram is radix_kth's)
  int* seg_start = reinterpret_cast<int*>(s.ckey + g * Cfg<G>::kCap);
  const int my_n = et < nseg ? __ldcg(&p.slot_count[(c_first + et + w) * G + g]) : 0;
  int total;
  const int my_start = epi_exclusive_scan(m, my_n, &total);
  if (et <= nseg) seg_start[et] = et < nseg ? my_start : total;
  named_sync(kEpiBarrier, kEpiThreads);
  if (total > kMB * kEpiThreads) {
    if (et == 0 && s.trace) s.trace[kTrMergeFallback] += 1000000;
    merge_slots<G>(p, s, w, g, c_first, c_last, out);
    return;
  }
  uint32_t u[kMB];
  uint64_t gt_mask = 0, eq_mask = 0;
  {
    int seg = 0;
#pragma unroll
    for (int j = 0; j < kMB; ++j) {
      const int i = j * kEpiThreads + et;
      u[j] = 0u;
      if (i < total) {
        while (seg_start[seg + 1] <= i) ++seg;
        const int64_t slot = (c_first + seg + w) * G + g;
        u[j] = __ldcg(&p.slot_key[slot * p.slot_cap + (i - seg_start[seg])]);
      }
    }
#pragma unroll
    for (int j = 0; j < kMB; ++j) {
      const bool valid = j * kEpiThreads + et < total;
      const int b = row_bin(u[j]);
      if (valid && b > cut) gt_mask |= 1ull << j;
      if (valid && b == cut) eq_mask |= 1ull << j;
    }
  }
  int tge;
  epi_exclusive_scan(m, (__popcll(eq_mask) << 16) | __popcll(gt_mask), &tge);
  const int t_gt = tge & 0xffff, t_eq = tge >> 16;
  named_sync(kEpiBarrier, kEpiThreads);
  const int need = K - above;
  const uint64_t tq2 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  if (et == 0 && s.trace) {
    s.trace[kTrMergeLoadNs] += tq2 - tq1;
    s.trace[kTrMergeUnion] += static_cast<uint64_t>(total);
    s.trace[kTrMergeCut] += static_cast<uint64_t>(t_eq);
    s.trace[kTrMergeSegs] += static_cast<uint64_t>(nseg);
  }
  if (t_gt != above || t_eq < need) {
    if (et == 0 && s.trace) s.trace[kTrMergeFallback] += 1000;
    merge_slots<G>(p, s, w, g, c_first, c_last, out);
    return;
  }
  // among the cutoff bin's entries: the `need` largest
  uint32_t mn = 0;
  int hi = 0, remaining = need;
  uint64_t pre = 0;
  if (t_eq > need) radix_kth(s, u, eq_mask, need, &mn, &hi, &pre, &remaining);
  const uint64_t tq3 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  if (et == 0 && s.trace) s.trace[kTrMergeRadixNs] += tq3 - tq2;
  uint64_t take_mask = gt_mask;
  int n_tie = 0;
#pragma unroll
  for (int j = 0; j < kMB; ++j) {
    if (!((eq_mask >> j) & 1)) continue;
    const uint64_t top = t_eq > need ? static_cast<uint64_t>(u[j] - mn) >> hi : 0;
    if (top > pre) take_mask |= 1ull << j;
    else if (top == pre) ++n_tie;
  }
  int tt;
  const int tie_before = epi_exclusive_scan(m, n_tie, &tt);
  named_sync(kEpiBarrier, kEpiThreads);
  int take_tie = min(max(remaining - tie_before, 0), n_tie);
#pragma unroll
  for (int j = 0; j < kMB; ++j) {
    if (!((eq_mask >> j) & 1) || ((take_mask >> j) & 1)) continue;
    const uint64_t top = t_eq > need ? static_cast<uint64_t>(u[j] - mn) >> hi : 0;
    if (top == pre && take_tie > 0) {
      take_mask |= 1ull << j;
      --take_tie;
    }
  }
  int t_take;
  int pos = epi_exclusive_scan(m, __popcll(take_mask), &t_take);
  {
    // gather the selected entries' indices in one batch (into the key
    // registers, which are no longer needed), then store them
    int seg = 0;
#pragma unroll
    for (int j = 0; j < kMB; ++j) {
      if ((take_mask >> j) & 1) {
        const int i = j * kEpiThreads + et;
        while (seg_start[seg + 1] <= i) ++seg;
        const int64_t slot = (c_first + seg + w) * G + g;
        u[j] = static_cast<uint32_t>(__ldcg(&p.slot_idx[slot * p.slot_cap + (i - seg_start[seg])]));
      }
    }
#pragma unroll
    for (int j = 0; j < kMB; ++j) {
      if ((take_mask >> j) & 1) {
        if (pos < K) out[pos] = static_cast<int32_t>(u[j]);
        ++pos;
      }
    }
  }
  named_sync(kEpiBarrier, kEpiThreads);
  for (int e = t_take + et; e < K; e += kEpiThreads) out[e] = -1;
  named_sync(kEpiBarrier, kEpiThreads);
  if (et == 0 && s.trace) s.trace[kTrMergeTailNs] += globaltimer_ns() - tq3;
}

// Where the selection finds each staged key's token index.
enum StagedIdx {
  kIdxStaged = 0,     // aux[e]: the indices were staged beside the keys
  kIdxSlotByPos = 1,  // slot entry at staged position e (segment offsets in cidx)
  kIdxSlotBySrc = 2,  // slot entry at union position aux[e] (segment offsets in cidx)
};

// Selection of work row w's k (token g) from keys staged in shared memory:
// keys[0, total_r) (total_r a multiple of 4 and keys 16-byte aligned; key 0
// is padding), cut = the row's exact cutoff bin and above = the count in the
// bins above it. Returns false (having written nothing final) when the staged
// keys disagree with the histogram.
template <int G>
__device__ bool select_staged(const ScoreParams& p, const Smem& s, int w, int g, int64_t c_first,
                              int nseg, const uint32_t* keys, const int32_t* aux, int total_r,
                              int cut, int above, int32_t* out, int mode, uint64_t tq0) {
  const int et = threadIdx.x - 64;
  const int lane = threadIdx.x & 31;
  const int K = p.topk;
  Misc* m = s.misc;
  const int32_t* seg_off = s.cidx;
  const uint64_t tq1 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  // One pass classifies every key against the cutoff bin (keys carry the row
  // bin in their top 10 bits) and histograms the next 10 bits of the keys in
  // it; further passes resolve 10 and then 2 more bits only while the bucket
  // holding the K-th key is not taken whole. Four keys per 16-byte load.
  const uint4* k4 = reinterpret_cast<const uint4*>(keys);
  const int n4 = total_r >> 2;
  const uint32_t ucut = static_cast<uint32_t>(cut);
  int n_gt = 0, n_eq = 0;
  for (int e = et; e < n4; e += kEpiThreads) {
    const uint4 q = k4[e];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (u[c] == 0u) continue;
      const uint32_t b = u[c] >> 22;
      n_gt += b > ucut ? 1 : 0;
      if (b == ucut) {
        ++n_eq;
        atomicAdd(&s.hist[(u[c] >> 12) & 1023u], 1u);
      }
    }
  }
  int tge;
  epi_exclusive_scan(m, (n_eq << 16) | n_gt, &tge);
  const int t_gt = tge & 0xffff, t_eq = tge >> 16;
  named_sync(kEpiBarrier, kEpiThreads);
  const int need = K - above;
  if (et == 0 && s.trace) {
    s.trace[kTrMergeLoadNs] += tq1 - tq0;
    s.trace[kTrMergeUnion] += static_cast<uint64_t>(total_r);
    s.trace[kTrMergeCut] += static_cast<uint64_t>(t_eq);
    s.trace[kTrMergeSegs] += static_cast<uint64_t>(nseg);
  }
  const bool fail = t_gt != above || t_eq < need;
  if (fail || t_eq == need) {
    for (int b = et; b < 1024; b += kEpiThreads) s.hist[b] = 0u;
    named_sync(kEpiBarrier, kEpiThreads);
    if (fail) return false;
  }
  // a key is in when key >> sh > pre; keys with key >> sh == pre are tied and
  // `remaining` of them complete K (all of them when all_tied)
  int sh = 22, remaining = need;
  uint32_t pre = ucut;
  bool all_tied = true;
  if (t_eq > need) {
    int bucket, ab, bc;
    take_bucket(s.hist, m, 1024, remaining, &bucket, &ab, &bc);
    pre = (pre << 10) | static_cast<uint32_t>(bucket);
    sh = 12;
    remaining -= ab;
    if (bc != remaining) {
      for (int e = et; e < n4; e += kEpiThreads) {
        const uint4 q = k4[e];
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (u[c] != 0u && (u[c] >> 12) == pre) atomicAdd(&s.hist[(u[c] >> 2) & 1023u], 1u);
      }
      named_sync(kEpiBarrier, kEpiThreads);
      take_bucket(s.hist, m, 1024, remaining, &bucket, &ab, &bc);
      pre = (pre << 10) | static_cast<uint32_t>(bucket);
      sh = 2;
      remaining -= ab;
      if (bc != remaining) {
        for (int e = et; e < n4; e += kEpiThreads) {
          const uint4 q = k4[e];
          const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (u[c] != 0u && (u[c] >> 2) == pre) atomicAdd(&s.hist[u[c] & 3u], 1u);
        }
        named_sync(kEpiBarrier, kEpiThreads);
        take_bucket(s.hist, m, 4, remaining, &bucket, &ab, &bc);
        pre = (pre << 2) | static_cast<uint32_t>(bucket);
        sh = 0;
        remaining -= ab;
        all_tied = bc == remaining;
      }
    }
  }
  const uint64_t tq2 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  // output: per key 1 = in, 2 = tied (`remaining` of the tied keys complete
  // K, in warp-major order). A counting pass gives each warp its output and
  // tie offsets; the writing pass places keys by ballot ranks (coalesced).
  auto klass = [&](uint32_t u) -> uint32_t {
    const uint32_t top = u >> sh;
    return u == 0u ? 0u : (top > pre ? 1u : (top == pre ? (all_tied ? 1u : 2u) : 0u));
  };
  const int ew = et >> 5;
  int n_in = 0, n_tie = 0;
  for (int e = et; e < n4; e += kEpiThreads) {
    const uint4 q = k4[e];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t k = klass(u[c]);
      n_in += k == 1u ? 1 : 0;
      n_tie += k == 2u ? 1 : 0;
    }
  }
  n_in = __reduce_add_sync(0xffffffffu, n_in);
  n_tie = __reduce_add_sync(0xffffffffu, n_tie);
  if (lane == 0) {
    m->scan[ew] = n_in;
    m->rmax[ew] = static_cast<uint32_t>(n_tie);
  }
  named_sync(kEpiBarrier, kEpiThreads);
  int tie_base = 0, ties_before_all = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    tie_base += i < ew ? static_cast<int>(m->rmax[i]) : 0;
  }
  int out_base = 0, t_take = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tb = ties_before_all;
    const int wt = static_cast<int>(m->rmax[i]);
    const int taken_ties = min(max(remaining - tb, 0), wt);
    ties_before_all += wt;
    const int w_take = m->scan[i] + taken_ties;
    out_base += i < ew ? w_take : 0;
    t_take += w_take;
  }
  named_sync(kEpiBarrier, kEpiThreads);
  const int4* x4 = reinterpret_cast<const int4*>(aux);
  int32_t* src = reinterpret_cast<int32_t*>(s.ckey);  // staged position of output p
  const uint32_t lt = (1u << lane) - 1u;
  for (int e0 = ew * 32; e0 < n4; e0 += kEpiThreads) {
    const int e = e0 + lane;
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    int4 xi = make_int4(0, 0, 0, 0);
    if (e < n4) {
      q = k4[e];
      if (mode == kIdxStaged) xi = x4[e];
    }
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
    const int32_t x[4] = {xi.x, xi.y, xi.z, xi.w};
    uint32_t kc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) kc[c] = klass(u[c]);
    if (!all_tied) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t tm = __ballot_sync(0xffffffffu, kc[c] == 2u);
        if (kc[c] == 2u) kc[c] = tie_base + __popc(tm & lt) < remaining ? 1u : 0u;
        tie_base += __popc(tm);
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t im = __ballot_sync(0xffffffffu, kc[c] == 1u);
      const int pos = out_base + __popc(im & lt);
      if (kc[c] == 1u && pos < K) {
        if (mode == kIdxStaged) out[pos] = x[c];
        else src[pos] = 4 * e + c;
      }
      out_base += __popc(im);
    }
  }
  if (mode != kIdxStaged) {
    named_sync(kEpiBarrier, kEpiThreads);
    for (int q = et; q < min(t_take, K); q += kEpiThreads) {
      int e = src[q];
      if (mode == kIdxSlotBySrc) e = aux[e];  // staged position -> position in the slots' union
      int lo = 0, hi = nseg - 1;  // the segment holding staged position e
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg_off[mid] <= e) lo = mid;
        else hi = mid - 1;
      }
      const int64_t seg_slot = (c_first + lo + w) * G + g;
      out[q] = __ldcg(&p.slot_idx[seg_slot * p.slot_cap + (e - seg_off[lo])]);
    }
  }
  for (int e = t_take + et; e < K; e += kEpiThreads) out[e] = -1;
  named_sync(kEpiBarrier, kEpiThreads);
  if (et == 0 && s.trace) {
    s.trace[kTrMergeRadixNs] += tq2 - tq1;
    s.trace[kTrMergeTailNs] += globaltimer_ns() - tq2;
  }
  return true;
}


// Merge for rows with more segments than epilogue threads, or a union of slot
// entries larger than the ring: every thread walks the slots' union (four
// coalesced loads in flight per round) and appends the entries in bins at or
// above the exact cutoff, with their union position, to the ring; the
// selection then runs on that filtered set and gathers the chosen indices
// from the slots. Returns false when the filtered set does not fit either.
template <int G>
__device__ bool merge_row_gathered(const ScoreParams& p, const Smem& s, int w, int g,
                                   int64_t c_first, int64_t c_last, const uint32_t* gh,
                                   int32_t* out) {
  using C = Cfg<G>;
  constexpr int kStageCap = C::kStages * 16384 / 8;
  const int et = threadIdx.x - 64;
  const int lane = threadIdx.x & 31, ew = et >> 5;
  const int K = p.topk;
  Misc* m = s.misc;
  const int nseg = static_cast<int>(c_last - c_first + 1);
  int32_t* seg_off = s.cidx;  // [nseg + 1] union offsets of the segments
  if (nseg + 1 > G * C::kCap) return false;
  const uint64_t tq0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  named_sync(kEpiBarrier, kEpiThreads);
  int floor = -1, carry = 0;
  for (int base = 0; base < nseg; base += kEpiThreads) {
    const int i = base + et;
    int n = 0;
    if (i < nseg) {
      const int64_t sl = (c_first + i + w) * G + g;
      n = __ldcg(&p.slot_count[sl]);
      floor = max(floor, __ldcg(&p.slot_thrbin[sl]));
    }
    int tot;
    const int excl = epi_exclusive_scan(m, n, &tot);
    if (i < nseg) seg_off[i] = carry + excl;
    carry += tot;
    named_sync(kEpiBarrier, kEpiThreads);
  }
  const int total = carry;
  if (et == 0) {
    seg_off[nseg] = total;
    m->sel_out = 0;
  }
  floor = __reduce_max_sync(0xffffffffu, floor);
  if (lane == 0) m->rmin[ew] = static_cast<uint32_t>(floor);
  named_sync(kEpiBarrier, kEpiThreads);
  floor = max(max(static_cast<int>(m->rmin[0]), static_cast<int>(m->rmin[1])),
              max(static_cast<int>(m->rmin[2]), static_cast<int>(m->rmin[3])));
  int cut, above;
  row_cutoff(gh, m, K, floor, &cut, &above);
  if (cut < 0) return false;
  uint32_t* keys = reinterpret_cast<uint32_t*>(s.kv);
  int32_t* src = reinterpret_cast<int32_t*>(s.kv) + kStageCap;
  const uint32_t lt = (1u << lane) - 1u;
  int seg = 0;  // this thread's segment; its union positions only grow
  for (int i0 = ew * 128; i0 < total; i0 += 4 * kEpiThreads) {
    uint32_t u4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * 32 + lane;
      u4[u] = 0u;
      if (i < total) {
        while (seg_off[seg + 1] <= i) ++seg;
        const int64_t sl = (c_first + seg + w) * G + g;
        u4[u] = __ldcg(&p.slot_key[sl * p.slot_cap + (i - seg_off[seg])]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * 32 + lane;
      const bool kp = i < total && row_bin(u4[u]) >= cut;
      const uint32_t km = __ballot_sync(0xffffffffu, kp);
      int b = 0;
      if (lane == 0 && km) b = atomicAdd(&m->sel_out, __popc(km));
      b = __shfl_sync(0xffffffffu, b, 0);
      const int pos = b + __popc(km & lt);
      if (kp && pos < kStageCap) {
        keys[pos] = u4[u];
        src[pos] = i;
      }
    }
  }
  named_sync(kEpiBarrier, kEpiThreads);
  const int kept = m->sel_out;
  const int kept_r = (kept + 3) & ~3;
  if (kept_r > kStageCap) return false;
  for (int e = kept + et; e < kept_r; e += kEpiThreads) keys[e] = 0u;  // padding
  named_sync(kEpiBarrier, kEpiThreads);
  return select_staged<G>(p, s, w, g, c_first, nseg, keys, src, kept_r, cut, above, out,
                          kIdxSlotBySrc, tq0);
}

// merge_row for a CTA whose own pipeline has finished (its shared-memory ring
// is idle): the slots' keys and indices are staged into the ring by one bulk
// copy per slot and segment (all completing on one mbarrier), then the cutoff
// classification, the radix select among the cutoff bin's keys and the output
// all run from shared memory. Returns false (having written nothing) when the
// union does not fit the ring or the slots disagree with the histogram.
template <int G>
__device__ bool merge_row_staged(const ScoreParams& p, const Smem& s, int w, int g,
                                 int64_t c_first, int64_t c_last, const uint32_t* gh,
                                 int32_t* out) {
  using C = Cfg<G>;
  constexpr int kStageCap = C::kStages * 16384 / 8;  // entries (key + index) in the ring
  const int et = threadIdx.x - 64;
  const int lane = threadIdx.x & 31;
  const int K = p.topk;
  Misc* m = s.misc;
  const int nseg = static_cast<int>(c_last - c_first + 1);
  if (nseg > kEpiThreads) return merge_row_gathered<G>(p, s, w, g, c_first, c_last, gh, out);
  const uint64_t tq0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  // the segments' counts and threshold bins and this thread's bins of the row
  // histogram, loaded together
  const int64_t sl = (c_first + et + w) * G + g;
  int floor = et < nseg ? __ldcg(&p.slot_thrbin[sl]) : -1;
  const int my_n = et < nseg ? __ldcg(&p.slot_count[sl]) : 0;
  int hc[kCutPer];
  load_row_bins(gh, hc);
  // staging offsets: each segment's entries start on a 16-byte boundary
  const int my_r = (my_n + 3) & ~3;
  int total_r;
  const int my_off = epi_exclusive_scan(m, my_r, &total_r);
  if (total_r > 2 * kStageCap) return merge_row_gathered<G>(p, s, w, g, c_first, c_last, gh, out);
  // Keys and indices are staged when both fit; otherwise only the keys, and
  // the selected entries' indices are gathered from the slots at the end
  // (segment staging offsets kept in the idle candidate-index buffer).
  const bool with_idx = total_r <= kStageCap;
  uint32_t* keys = reinterpret_cast<uint32_t*>(s.kv);
  int32_t* idxs = reinterpret_cast<int32_t*>(s.kv) + kStageCap;
  int32_t* seg_off = s.cidx;
  if (!with_idx && et <= nseg) seg_off[et] = et < nseg ? my_off : total_r;
  fence_proxy_async_shared();  // earlier generic accesses of the ring precede the copies
  named_sync(kEpiBarrier, kEpiThreads);
  const int use = m->staged_uses;
  if (et < nseg && my_n > 0) {
    const uint32_t bytes = static_cast<uint32_t>(my_r) * 4u;
    bulk_load(keys + my_off, p.slot_key + sl * p.slot_cap, bytes, s.staged);
    if (with_idx) bulk_load(idxs + my_off, p.slot_idx + sl * p.slot_cap, bytes, s.staged);
  }
  if (et == 0)
    mbar_arrive_expect_tx(s.staged, static_cast<uint32_t>(total_r) * (with_idx ? 8u : 4u));
  // while the copies are in flight: the row's cutoff, floored by the
  // segments' threshold bins (see merge_row)
  floor = __reduce_max_sync(0xffffffffu, floor);
  if (lane == 0) m->rmin[et >> 5] = static_cast<uint32_t>(floor);
  named_sync(kEpiBarrier, kEpiThreads);
  floor = max(max(static_cast<int>(m->rmin[0]), static_cast<int>(m->rmin[1])),
              max(static_cast<int>(m->rmin[2]), static_cast<int>(m->rmin[3])));
  int cut, above;
  row_cutoff_vals(hc, m, K, floor, &cut, &above);
  bool ok = true;
  if (lane == 0) ok = mbar_wait(s.staged, use & 1, &m->abort_flag, p.dev_error);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  // the padding after a segment's entries becomes key 0, which no logit maps to
  if (ok && et < nseg)
    for (int e = my_off + my_n; e < my_off + my_r; ++e) keys[e] = 0u;
  if (lane == 0) m->vote[0][et >> 5] = ok ? 1 : 0;
  named_sync(kEpiBarrier, kEpiThreads);
  const bool all_ok = m->vote[0][0] & m->vote[0][1] & m->vote[0][2] & m->vote[0][3];
  if (et == 0) m->staged_uses = use + 1;
  if (!all_ok || cut < 0) return false;
  return select_staged<G>(p, s, w, g, c_first, nseg, keys, with_idx ? idxs : nullptr, total_r, cut,
                          above, out, with_idx ? kIdxStaged : kIdxSlotByPos, tq0);
}

// Merge of work row w (every segment published) into its output rows, by a
// CTA whose own tiles are all done: staged in the idle ring, else from the
// slots directly.
template <int G>
__device__ void merge_work_row(const ScoreParams& p, const Smem& s, int w, const WorkRow& wr,
                               const bool (&active)[G], int64_t c_first, int64_t c_last) {
  const int et = threadIdx.x - 64;
  const uint64_t tm0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  __threadfence();
  const uint32_t* gh_base = p.row_hist + c_first * G * kRowHistBins;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (!active[g]) continue;
    int32_t* out = p.out_idx + (p.out_row_base + wr.row0 + g) * p.topk;
    const uint32_t* gh = gh_base + g * kRowHistBins;
    if (merge_row_staged<G>(p, s, w, g, c_first, c_last, gh, out)) continue;
    if (et == 0 && s.trace) s.trace[kTrMergeFallback] += 1;
    merge_row<G>(p, s, w, g, c_first, c_last, gh, out);
  }
  if (et == 0 && s.trace) {
    s.trace[kTrMergeNs] += globaltimer_ns() - tm0;
    s.trace[kTrMergeN] += 1;
  }
}

// End of this CTA's part of work row w: if the CTA holds the whole row, cut
// each buffer to k and write the output; else publish the candidates that can
// still make the row's top-k (bins at or above the row histogram's current
// cutoff; a slot holds a whole buffer) to the segment's slot; the CTA that
// publishes last merges (now, or at its end if it still has tiles to stream).
template <int G>
__device__ void finalize_segment(const ScoreParams& p, const Smem& s, int w, const WorkRow& wr,
                                 const bool (&active)[G], int64_t rs, int64_t re, int64_t t0,
                                 int64_t t1, int64_t T, int64_t nC) {
  using C = Cfg<G>;
  const int et = threadIdx.x - 64;
  const int K = p.topk;
  Misc* m = s.misc;
  const uint64_t tf0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  const int lane = threadIdx.x & 31, ew = et >> 5;
  named_sync(kEpiBarrier, kEpiThreads);
  // A row held whole by this CTA is written from the buffer, cut to exactly
  // k; a segment publishes its whole buffer (up to kCap entries, the slot's
  // capacity), filtered by the row histogram's cutoff below.
  const bool whole = rs >= t0 && re <= t1;
#pragma unroll
  for (int g = 0; g < G; ++g)
    if (whole && active[g] && m->wcnt[g][0] + m->wcnt[g][1] + m->wcnt[g][2] + m->wcnt[g][3] > K)
      compact<G>(s, g, K);  // cut to k (the regions stay the layout)
  uint64_t tf1 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  if (et == 0 && s.trace) s.trace[kTrFinPackNs] += tf1 - tf0;
  if (whole) {
    write_rows<G>(p, s, wr, active);
    if (et == 0 && s.trace) s.trace[kTrFinalizeNs] += globaltimer_ns() - tf0;
    return;
  }
  const int2 rc = p.row_ctas[w];
  const int64_t c_first = rc.x, c_last = rc.y;
  uint32_t* gh_base = p.row_hist + c_first * G * kRowHistBins;
  const int64_t slot = static_cast<int64_t>(blockIdx.x) + w;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    uint32_t* gh = gh_base + g * kRowHistBins;
    const uint32_t* rk = s.ckey + g * C::kCap + ew * C::kRegion;
    const int32_t* rx = s.cidx + g * C::kCap + ew * C::kRegion;
    // the segment's final buffer joins the row histogram: counted in shared
    // memory, then the non-zero bins are added to the global one (and the
    // shared bins zeroed again)
    const int nw = active[g] ? m->wcnt[g][ew] : 0;
    for (int j = lane; j < nw; j += 32) atomicAdd(&s.hist[row_bin(rk[j])], 1u);
    named_sync(kEpiBarrier, kEpiThreads);
    for (int b = et; b < kRowHistBins; b += kEpiThreads) {
      const uint32_t c = s.hist[b];
      if (c) {
        atomicAdd(&gh[b], c);
        s.hist[b] = 0u;
      }
    }
    if (et == 0 && s.trace) {
      const uint64_t now = globaltimer_ns();
      s.trace[kTrFinHistNs] += now - tf1;
      tf1 = now;
    }
    // publish the candidates that can still make the row's top-k (bins at or
    // above the histogram's current cutoff) and the threshold's bin
    int cut = -1, above = 0;
    if (active[g]) row_cutoff(gh, m, K, -1, &cut, &above);
    if (et == 0 && s.trace) {
      const uint64_t now = globaltimer_ns();
      s.trace[kTrFinCutNs] += now - tf1;
      tf1 = now;
    }
    const int64_t base = (slot * G + g) * p.slot_cap;
    int keep = 0;
    for (int j = lane; j < nw; j += 32) keep += row_bin(rk[j]) >= cut ? 1 : 0;
    keep = __reduce_add_sync(0xffffffffu, keep);
    if (lane == 0) m->scan[ew] = keep;
    named_sync(kEpiBarrier, kEpiThreads);
    int pos = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pos += i < ew ? m->scan[i] : 0;
      tot += m->scan[i];
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (int j0 = 0; j0 < nw; j0 += 32) {
      const int j = j0 + lane;
      const uint32_t u = j < nw ? rk[j] : 0u;
      const bool kp = j < nw && row_bin(u) >= cut;
      const uint32_t km = __ballot_sync(0xffffffffu, kp);
      if (kp) {
        p.slot_key[base + pos + __popc(km & lt)] = u;
        p.slot_idx[base + pos + __popc(km & lt)] = rx[j];
      }
      pos += __popc(km);
    }
    named_sync(kEpiBarrier, kEpiThreads);
    if (et == 0) {
      p.slot_count[slot * G + g] = tot;
      // a buffer that never filled dropped nothing: its histogram is exact
      p.slot_thrbin[slot * G + g] = m->thr[g] ? row_bin(m->thr[g]) : -1;
    }
    named_sync(kEpiBarrier, kEpiThreads);
    if (et == 0 && s.trace) {
      const uint64_t now = globaltimer_ns();
      s.trace[kTrFinEmitNs] += now - tf1;
      tf1 = now;
    }
  }
  __threadfence();
  named_sync(kEpiBarrier, kEpiThreads);
  if (et == 0) {
    const int old = atomicAdd(&p.seg_counter[w], 1);
    m->is_last = (old == static_cast<int>(c_last - c_first));
  }
  named_sync(kEpiBarrier, kEpiThreads);
  if (et == 0 && s.trace) s.trace[kTrFinPublishNs] += globaltimer_ns() - tf1;
  // The last segment to publish merges the row. A CTA with tiles still to
  // stream defers the merge to its end, when its ring is idle for staging.
  if (m->is_last && re < t1 && et == 0) m->pending_row = w;
  if (m->is_last && re >= t1) merge_work_row<G>(p, s, w, wr, active, c_first, c_last);
  if (et == 0 && s.trace) s.trace[kTrFinalizeNs] += globaltimer_ns() - tf0;
}

template <int G, bool kLogits>
__device__ void epilogue(const ScoreParams& p, const Smem& s, uint32_t tmem, int64_t t0, int64_t t1,
                         int64_t T, int64_t nC) {
  using C = Cfg<G>;
  volatile int* abort_flag = &s.misc->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int et = threadIdx.x - 64;
  const int sub = warp & 3;                 // tensor-memory lanes [32*sub, 32*sub + 32)
  const int mrow = sub * 32 + lane;         // key of the tile this thread scores
  const uint32_t lane_addr = static_cast<uint32_t>(sub * 32) << 16;
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;

  int w = p.cta_row[blockIdx.x];
  int64_t rs = p.wr_tile_start[w], re = p.wr_tile_start[w + 1];
  WorkRow wr;
  int len[G];
  bool active[G];
  int wcnt[G];        // entries in this warp's region of each token's buffer
  uint32_t thr[G];    // each buffer's drop threshold
  const int ew = et >> 5;

  for (int b = et; b < C::kHistBins; b += kEpiThreads) s.hist[b] = 0u;  // zero between uses

  auto begin_row = [&]() {
    wr = p.wr[w];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      len[g] = g < wr.ntok ? p.row_len[wr.row0 + g] : 0;
      active[g] = g < wr.ntok && (kLogits ? len[g] > 0 : len[g] > p.topk);
    }
    for (int i = et; i < G * kHeads; i += kEpiThreads) {
      const int g = i / kHeads;
      s.wp[i] = g < wr.ntok ? p.wprime[static_cast<int64_t>(wr.row0 + g) * kHeads + i % kHeads] : 0.f;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      wcnt[g] = 0;
      thr[g] = 0u;
    }
    if (et == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s.misc->cnt[g] = 0;
        s.misc->thr[g] = 0u;
      }
    }
    named_sync(kEpiBarrier, kEpiThreads);
  };
  auto publish_counts = [&]() {
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < G; ++g) s.misc->wcnt[g][ew] = wcnt[g];
  };
  begin_row();

  bool ok = true;
  long long cyc[5] = {0, 0, 0, 0, 0};  // per-phase clock totals (trace only)
  for (int64_t t = t0; t < t1; ++t) {
    if (t >= re) {
      publish_counts();
      if (!kLogits) finalize_segment<G>(p, s, w, wr, active, rs, re, t0, t1, T, nC);
      do {
        ++w;
        re = p.wr_tile_start[w + 1];
      } while (t >= re);
      rs = p.wr_tile_start[w];
      named_sync(kEpiBarrier, kEpiThreads);
      begin_row();
    }
    const int i = static_cast<int>(t - rs);
    const bool tr = s.trace != nullptr;  // per-phase clocks only when tracing
    const long long c0 = tr ? clock64() : 0;
    // lane 0 of each warp waits for the stage (scales) and the accumulator
    bool wok = true;
    if (lane == 0)
      wok = mbar_wait(&s.full[stage], phase, abort_flag, p.dev_error) &&
            mbar_wait(&s.tfull[acc], acc_phase, abort_flag, p.dev_error);
    wok = __shfl_sync(0xffffffffu, wok ? 1 : 0, 0) != 0;
    __syncwarp();
    const long long c1 = tr ? clock64() : 0;
    long long c2 = c1;
    float logit[G];
    if (t == t0 && et == 0 && s.trace) s.trace[kTrFirstEpi] = globaltimer_ns();
    if (wok) {
      tc_fence_after();
      const float scale = s.scales[stage * 128 + mrow];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint32_t col = lane_addr + tmem + static_cast<uint32_t>(acc * C::N + g * 64);
        float v0[32], v1[32];
        tmem_ld32(col, v0);
        tmem_ld32(col + 32, v1);
        tmem_ld_wait();
        if (g == 0 && tr) c2 = clock64();
        const float4* w4 = reinterpret_cast<const float4*>(s.wp + g * kHeads);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 x = w4[q];
          a0 = fmaf(x.x, fmaxf(v0[4 * q + 0], 0.f), a0);
          a1 = fmaf(x.y, fmaxf(v0[4 * q + 1], 0.f), a1);
          a2 = fmaf(x.z, fmaxf(v0[4 * q + 2], 0.f), a2);
          a3 = fmaf(x.w, fmaxf(v0[4 * q + 3], 0.f), a3);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 x = w4[8 + q];
          a0 = fmaf(x.x, fmaxf(v1[4 * q + 0], 0.f), a0);
          a1 = fmaf(x.y, fmaxf(v1[4 * q + 1], 0.f), a1);
          a2 = fmaf(x.z, fmaxf(v1[4 * q + 2], 0.f), a2);
          a3 = fmaf(x.w, fmaxf(v1[4 * q + 3], 0.f), a3);
        }
        logit[g] = ((a0 + a1) + (a2 + a3)) * scale;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s.tempty[acc]);
        mbar_arrive(&s.empty[stage]);
      }
    }
    const long long c3 = tr ? clock64() : 0;
    // Uniform decision across the four epilogue warps (double-buffered vote):
    // bit 0 = this warp's waits succeeded, bit 1 + g = its region of token g's
    // buffer has no room for another tile (then all warps compact it).
    const int par = static_cast<int>(t & 1);
    int need = 0;
#pragma unroll
    for (int g = 0; g < G; ++g)
      need |= (!kLogits && active[g] && wcnt[g] + 32 > C::kRegion) ? 2 << g : 0;
    publish_counts();
    if (lane == 0) s.misc->vote[par][ew] = (wok ? 1 : 0) | need;
    named_sync(kEpiBarrier, kEpiThreads);
    const long long c4 = tr ? clock64() : 0;
    const int v0 = s.misc->vote[par][0], v1 = s.misc->vote[par][1];
    const int v2 = s.misc->vote[par][2], v3 = s.misc->vote[par][3];
    if (!(v0 & v1 & v2 & v3 & 1)) {
      ok = false;
      break;
    }
    const int needs = (v0 | v1 | v2 | v3) >> 1;
    const int key = i * kTileKeys + mrow;
    if (kLogits) {
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (active[g] && key < len[g])
          p.out_logits[static_cast<int64_t>(wr.row0 + g) * p.ld_logits + key] = logit[g];
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g)
        if ((needs >> g) & 1) {
          const int kept = compact<G>(s, g, p.topk, C::kSlack);
          wcnt[g] = (kept - ew + 3) >> 2;
          thr[g] = s.misc->thr[g];
        }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        // append to this warp's region: ballot + popc, no shared counter
        const uint32_t k = float_key(logit[g]);
        const bool pass = active[g] && key < len[g] && k > thr[g];
        const unsigned pm = __ballot_sync(0xffffffffu, pass);
        if (pass) {
          const int at = g * C::kCap + ew * C::kRegion + wcnt[g] + __popc(pm & ((1u << lane) - 1u));
          s.ckey[at] = k;
          s.cidx[at] = key;
        }
        wcnt[g] += __popc(pm);
      }
    }
    if (tr) {
      const long long c5 = clock64();
      cyc[0] += c1 - c0;
      cyc[1] += c2 - c1;
      cyc[2] += c3 - c2;
      cyc[3] += c4 - c3;
      cyc[4] += c5 - c4;
    }
    if (++stage == C::kStages) {
      stage = 0;
      phase ^= 1;
    }
    if (++acc == 2) {
      acc = 0;
      acc_phase ^= 1;
    }
  }
  if (et == 0 && s.trace) {
    s.trace[kTrLastEpi] = globaltimer_ns();
    s.trace[kTrEpiWaitCyc] = cyc[0];
    s.trace[kTrEpiLdCyc] = cyc[1];
    s.trace[kTrEpiMathCyc] = cyc[2];
    s.trace[kTrEpiVoteCyc] = cyc[3];
    s.trace[kTrEpiSelCyc] = cyc[4];
  }
  publish_counts();
  if (!kLogits && ok) {
    finalize_segment<G>(p, s, w, wr, active, rs, re, t0, t1, T, nC);
    const int pw = s.misc->pending_row;  // set (by thread 0) before barriers all passed since
    if (pw >= 0) {
      const WorkRow pwr = p.wr[pw];
      bool pact[G];
#pragma unroll
      for (int g = 0; g < G; ++g)
        pact[g] = g < pwr.ntok && p.row_len[pwr.row0 + g] > p.topk;
      const int2 rc = p.row_ctas[pw];
      merge_work_row<G>(p, s, pw, pwr, pact, rc.x, rc.y);
    }
  }
  if (et == 0 && s.trace) s.trace[kTrFinal] = globaltimer_ns();
}

template <int G, bool kLogits>
__global__ void __launch_bounds__(kThreads, Cfg<G>::kCtasPerSm)
    score_select_kernel(const __grid_constant__ ScoreParams p,
                        const __grid_constant__ CUtensorMap map) {
  using C = Cfg<G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Smem s = carve<G>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Shared-memory setup needs nothing from earlier kernels; everything after
  // pdl_wait() may read what they wrote.
  if (warp == 0 && lane == 0) prefetch_tensormap(&map);
  pdl_wait();

  // With fewer tiles than CTAs only the first T CTAs take part, so that every
  // participating CTA owns at least one tile (segment counts rely on it).
  const int64_t T = p.wr_tile_start[p.num_wr];
  const int64_t nC = min(static_cast<int64_t>(gridDim.x), T);
  const bool part = static_cast<int64_t>(blockIdx.x) < nC;
  s.trace = (p.trace && part) ? reinterpret_cast<uint64_t*>(base + C::kTraceOff) : nullptr;
  const int64_t t0 = part ? p.cta_tile[blockIdx.x] : 0;
  const int64_t t1 = part ? p.cta_tile[blockIdx.x + 1] : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1 + 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 4);
      mbar_init(&s.qfull[i], 1);
      mbar_init(&s.qempty[i], 1);
    }
    mbar_init(s.done, 1);
    mbar_init(s.staged, 1);
    s.misc->abort_flag = 0;
    s.misc->epi_done = 0;
    s.misc->staged_uses = 0;
    s.misc->pending_row = -1;
    if (s.trace)
      for (int i = 0; i < kTrSlots; ++i) s.trace[i] = 0;
    fence_barrier_init();
  }
  __syncwarp();  // warp 0 reconverges before the block barrier (which counts whole warps)
  if (warp == 1) tmem_alloc(&s.misc->tmem_base, C::kTmemCols);
  tc_fence_before();
  named_sync(kSetupBarrier, kThreads);
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem = s.misc->tmem_base;
  if (threadIdx.x == 0 && s.trace) {
    s.trace[kTrStart] = globaltimer_ns();
    s.trace[kTrTiles] = static_cast<uint64_t>(t1 - t0);
  }

  if (t0 < t1) {
    // One lane of each of warps 0 and 1 runs its role; the warp reconverges
    // before the block barrier below (which counts whole warps).
    if (warp == 0) {
      if (lane == 0) producer<G>(p, &map, s, t0, t1);
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) mma_issuer<G>(p, s, tmem, t0, t1);
      __syncwarp();
    } else {
      epilogue<G, kLogits>(p, s, tmem, t0, t1, T, nC);
    }
  }
  if (threadIdx.x == 64) *reinterpret_cast<volatile int*>(&s.misc->epi_done) = 1;
  tc_fence_before();
  named_sync(kTeardownBarrier, kThreads);
  if (threadIdx.x == 0 && s.trace) {
    s.trace[kTrEnd] = globaltimer_ns();
    s.trace[kTrSeen] = static_cast<uint64_t>(*reinterpret_cast<volatile int*>(&s.misc->epi_done));
  }
  if (threadIdx.x == 64 && s.trace) s.trace[kTrEndEpi] = globaltimer_ns();
  if (s.trace) {
    named_sync(kTeardownBarrier, kThreads);
    if (threadIdx.x < kTrSlots)
      p.trace[static_cast<int64_t>(blockIdx.x) * kTrSlots + threadIdx.x] = s.trace[threadIdx.x];
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int G, bool kLogits>
idx_status launch_impl(const ScoreParams& p, const CUtensorMap& map, int num_ctas, cudaStream_t s) {
  using C = Cfg<G>;
  // the dynamic shared-memory limit is a per-device attribute of the kernel:
  // set once per device (any host thread; setting it twice is harmless)
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return IDX_ERR_CUDA;
  if (dev >= kMaxDevices || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(score_select_kernel<G, kLogits>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return IDX_ERR_CUDA;
    if (dev < kMaxDevices) configured[dev].store(true, std::memory_order_release);
  }
  return launch_pdl(score_select_kernel<G, kLogits>, num_ctas, kThreads, C::kSmemBytes, s, p, map) ==
                 cudaSuccess
             ? IDX_OK
             : IDX_ERR_CUDA;
}

}  // namespace

int score_ctas_per_sm(int G) {
  switch (G) {
    case 1: return Cfg<1>::kCtasPerSm;
    case 2: return Cfg<2>::kCtasPerSm;
    case 4: return Cfg<4>::kCtasPerSm;
    default: return 1;
  }
}

idx_status launch_score(int G, bool logits, const ScoreParams& p, const CUtensorMap& map,
                        int num_ctas, cudaStream_t s) {
  switch (G) {
    case 1: return logits ? launch_impl<1, true>(p, map, num_ctas, s)
                          : launch_impl<1, false>(p, map, num_ctas, s);
    case 2: return logits ? launch_impl<2, true>(p, map, num_ctas, s)
                          : launch_impl<2, false>(p, map, num_ctas, s);
    case 4: return logits ? launch_impl<4, true>(p, map, num_ctas, s)
                          : launch_impl<4, false>(p, map, num_ctas, s);
    default: return IDX_ERR_UNSUPPORTED;
  }
}

}  // namespace saib
