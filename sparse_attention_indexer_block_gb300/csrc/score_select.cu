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
#include "internal.h"

namespace saib {

namespace {

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kEpiBarrier = 1;  // named barrier id of the epilogue warps

template <int G>
struct Cfg {
  static constexpr int N = 64 * G;
  static constexpr int kStages = G == 1 ? 8 : (G == 2 ? 6 : 4);
  static constexpr int kCap = G <= 2 ? 4096 : 2560;  // candidate slots per token row
  static constexpr int kPer = kCap / kEpiThreads;
  static constexpr uint32_t kTmemCols = 2 * N <= 128 ? 128u : (2 * N <= 256 ? 256u : 512u);
  static constexpr uint32_t kIdesc = f8_idesc(128, N);
  static constexpr int kKvOff = 0;
  static constexpr int kQOff = kKvOff + kStages * 16384;
  static constexpr int kScaleOff = kQOff + 2 * G * kQRowBytes;
  static constexpr int kCandKeyOff = kScaleOff + kStages * 512;
  static constexpr int kCandIdxOff = kCandKeyOff + G * kCap * 4;
  static constexpr int kWpOff = kCandIdxOff + G * kCap * 4;
  static constexpr int kHistOff = kWpOff + G * 256;
  static constexpr int kBarOff = kHistOff + 1024;
  static constexpr int kNumBars = 2 * kStages + 9;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 256 + 1024;  // + alignment slack
  static_assert(kCap % kEpiThreads == 0, "capacity");
  static_assert(kSmemBytes <= 232448, "shared memory");
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
  Misc* misc;
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
  s.misc = reinterpret_cast<Misc*>(base + C::kMiscOff);
  return s;
}

// Largest work row w with wts[w] <= t (zero-tile rows share their start).
__device__ __forceinline__ int find_row(const int32_t* wts, int num_wr, int64_t t) {
  int lo = 0, hi = num_wr - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (wts[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// CTA whose tile range [c*T/nC, (c+1)*T/nC) contains tile t.
__device__ __forceinline__ int64_t cta_of(int64_t t, int64_t T, int64_t nC) {
  return ((t + 1) * nC - 1) / T;
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

  int w = find_row(p.wr_tile_start, p.num_wr, t0);
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
  int w = find_row(p.wr_tile_start, p.num_wr, t0);
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

// Shrinks candidate buffer g to exactly K entries (its K largest keys, ties at
// the K-th value broken arbitrarily) by an MSB-first 8-bit radix select over
// the order-preserving keys, and raises the buffer's drop threshold to the
// resolved prefix of the K-th key. Precondition: cnt[g] > K. Called by all
// epilogue threads.
template <int G>
__device__ void compact(const Smem& s, int g, int K) {
  using C = Cfg<G>;
  const int et = threadIdx.x - 64;
  const int lane = threadIdx.x & 31;
  uint32_t* ck = s.ckey + g * C::kCap;
  int32_t* ci = s.cidx + g * C::kCap;
  Misc* m = s.misc;
  const int n = m->cnt[g];
  uint32_t prefix = 0, mask = 0;
  int remaining = K;
  const int iters = (n + kEpiThreads - 1) / kEpiThreads;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = et; b < 256; b += kEpiThreads) s.hist[b] = 0;
    named_sync(kEpiBarrier, kEpiThreads);
#pragma unroll 1
    for (int j = 0; j < iters; ++j) {
      const int e = j * kEpiThreads + et;
      const uint32_t u = e < n ? ck[e] : 0u;
      const bool act = e < n && (u & mask) == prefix;
      const uint32_t digit = (u >> shift) & 0xffu;
      const unsigned am = __ballot_sync(0xffffffffu, act);
      if (act) {
        const unsigned peers = __match_any_sync(am, digit);
        if (lane == __ffs(peers) - 1) atomicAdd(&s.hist[digit], static_cast<uint32_t>(__popc(peers)));
      }
    }
    named_sync(kEpiBarrier, kEpiThreads);
    if (et < 32) {
      uint32_t c[8];
      int local = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = s.hist[8 * lane + j];
        local += static_cast<int>(c[j]);
      }
      int suf = local;  // keys in bins of this lane and above
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += v;
      }
      int above = suf - local;
      if (above < remaining && remaining <= suf) {
#pragma unroll
        for (int j = 7; j >= 0; --j) {
          if (above + static_cast<int>(c[j]) >= remaining) {
            m->bucket = 8 * lane + j;
            m->above = above;
            m->bcount = static_cast<int>(c[j]);
            break;
          }
          above += static_cast<int>(c[j]);
        }
      }
    }
    named_sync(kEpiBarrier, kEpiThreads);
    const int b = m->bucket;
    prefix |= static_cast<uint32_t>(b) << shift;
    mask |= 0xffu << shift;
    remaining -= m->above;
    const int bcount = m->bcount;
    if (bcount == remaining) break;  // the whole bucket is selected
  }
  // gather into registers, then write the selected keys to the front
  uint32_t ku[C::kPer];
  int32_t ki[C::kPer];
#pragma unroll
  for (int j = 0; j < C::kPer; ++j) {
    const int e = j * kEpiThreads + et;
    ku[j] = e < n ? ck[e] : 0u;
    ki[j] = e < n ? ci[e] : 0;
  }
  if (et == 0) {
    m->sel_out = 0;
    m->sel_tie = 0;
  }
  named_sync(kEpiBarrier, kEpiThreads);
#pragma unroll
  for (int j = 0; j < C::kPer; ++j) {
    const int e = j * kEpiThreads + et;
    const bool valid = e < n;
    const uint32_t top = ku[j] & mask;
    const bool gt = valid && top > prefix;
    const bool eq = valid && top == prefix;
    const unsigned em = __ballot_sync(0xffffffffu, eq);
    int tie_rank = 0;
    if (em) {
      int base = 0;
      const int leader = __ffs(em) - 1;
      if (lane == leader) base = atomicAdd(&m->sel_tie, __popc(em));
      base = __shfl_sync(0xffffffffu, base, leader);
      tie_rank = base + __popc(em & ((1u << lane) - 1u));
    }
    const bool take = gt || (eq && tie_rank < remaining);
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (tm) {
      int base = 0;
      const int leader = __ffs(tm) - 1;
      if (lane == leader) base = atomicAdd(&m->sel_out, __popc(tm));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (take) {
        const int pos = base + __popc(tm & ((1u << lane) - 1u));
        ck[pos] = ku[j];
        ci[pos] = ki[j];
      }
    }
  }
  named_sync(kEpiBarrier, kEpiThreads);
  if (et == 0) {
    m->cnt[g] = m->sel_out;
    m->thr[g] = max(m->thr[g], prefix);
  }
  named_sync(kEpiBarrier, kEpiThreads);
}

// Appends (key, idx) to buffer g when it passes the buffer's threshold. The
// caller guarantees room for one append per epilogue thread.
__device__ __forceinline__ void append(const Smem& s, int g, int cap, bool pass, uint32_t key,
                                       int32_t idx) {
  const int lane = threadIdx.x & 31;
  const unsigned am = __ballot_sync(0xffffffffu, pass);
  if (!am) return;
  int base = 0;
  const int leader = __ffs(am) - 1;
  if (lane == leader) base = atomicAdd(&s.misc->cnt[g], __popc(am));
  base = __shfl_sync(0xffffffffu, base, leader);
  if (pass) {
    const int pos = base + __popc(am & ((1u << lane) - 1u));
    s.ckey[g * cap + pos] = key;
    s.cidx[g * cap + pos] = idx;
  }
}

template <int G>
__device__ void write_rows(const ScoreParams& p, const Smem& s, const WorkRow& wr,
                           const bool (&active)[G]) {
  using C = Cfg<G>;
  const int et = threadIdx.x - 64;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (!active[g]) continue;
    const int n = s.misc->cnt[g];
    int32_t* o = p.out_idx + (p.out_row_base + wr.row0 + g) * p.topk;
    for (int e = et; e < p.topk; e += kEpiThreads) o[e] = e < n ? s.cidx[g * C::kCap + e] : -1;
  }
}

// End of this CTA's part of work row w: reduce each buffer to <= k, then write
// the output (sole segment) or publish a slot and merge if this is the last.
template <int G>
__device__ void finalize_segment(const ScoreParams& p, const Smem& s, int w, const WorkRow& wr,
                                 const bool (&active)[G], int64_t rs, int64_t re, int64_t t0,
                                 int64_t t1, int64_t T, int64_t nC) {
  using C = Cfg<G>;
  const int et = threadIdx.x - 64;
  const int K = p.topk;
  named_sync(kEpiBarrier, kEpiThreads);
#pragma unroll
  for (int g = 0; g < G; ++g)
    if (active[g] && s.misc->cnt[g] > K) compact<G>(s, g, K);
  if (rs >= t0 && re <= t1) {
    write_rows<G>(p, s, wr, active);
    return;
  }
  const int64_t c_first = cta_of(rs, T, nC), c_last = cta_of(re - 1, T, nC);
  const int64_t slot = static_cast<int64_t>(blockIdx.x) + w;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int n = active[g] ? s.misc->cnt[g] : 0;
    const int64_t base = (slot * G + g) * K;
    for (int e = et; e < n; e += kEpiThreads) {
      p.slot_key[base + e] = s.ckey[g * C::kCap + e];
      p.slot_idx[base + e] = s.cidx[g * C::kCap + e];
    }
    if (et == 0) p.slot_count[slot * G + g] = n;
  }
  __threadfence();
  named_sync(kEpiBarrier, kEpiThreads);
  if (et == 0) {
    const int old = atomicAdd(&p.seg_counter[w], 1);
    s.misc->is_last = (old == static_cast<int>(c_last - c_first));
  }
  named_sync(kEpiBarrier, kEpiThreads);
  if (!s.misc->is_last) return;
  __threadfence();
  for (int64_t c = c_first; c <= c_last; ++c) {
    if (c == blockIdx.x) continue;
    const int64_t os = c + w;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (!active[g]) continue;
      const int n = __ldcg(&p.slot_count[os * G + g]);
      const int64_t base = (os * G + g) * K;
      for (int e0 = 0; e0 < n; e0 += kEpiThreads) {
        named_sync(kEpiBarrier, kEpiThreads);
        if (s.misc->cnt[g] + kEpiThreads > C::kCap) compact<G>(s, g, K);
        const int e = e0 + et;
        uint32_t key = 0;
        int32_t idx = 0;
        if (e < n) {
          key = __ldcg(&p.slot_key[base + e]);
          idx = __ldcg(&p.slot_idx[base + e]);
        }
        append(s, g, C::kCap, e < n && key > s.misc->thr[g], key, idx);
      }
    }
  }
  named_sync(kEpiBarrier, kEpiThreads);
#pragma unroll
  for (int g = 0; g < G; ++g)
    if (active[g] && s.misc->cnt[g] > K) compact<G>(s, g, K);
  write_rows<G>(p, s, wr, active);
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

  int w = find_row(p.wr_tile_start, p.num_wr, t0);
  int64_t rs = p.wr_tile_start[w], re = p.wr_tile_start[w + 1];
  WorkRow wr;
  int len[G];
  bool active[G];

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
    if (et == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s.misc->cnt[g] = 0;
        s.misc->thr[g] = 0u;
      }
    }
    named_sync(kEpiBarrier, kEpiThreads);
  };
  begin_row();

  bool ok = true;
  for (int64_t t = t0; t < t1; ++t) {
    if (t >= re) {
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
    // lane 0 of each warp waits for the stage (scales) and the accumulator
    bool wok = true;
    if (lane == 0)
      wok = mbar_wait(&s.full[stage], phase, abort_flag, p.dev_error) &&
            mbar_wait(&s.tfull[acc], acc_phase, abort_flag, p.dev_error);
    wok = __shfl_sync(0xffffffffu, wok ? 1 : 0, 0) != 0;
    __syncwarp();
    float logit[G];
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
        const float* wg = s.wp + g * kHeads;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          a0 = fmaf(wg[j], fmaxf(v0[j], 0.f), a0);
          a1 = fmaf(wg[32 + j], fmaxf(v1[j], 0.f), a1);
        }
        logit[g] = (a0 + a1) * scale;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s.tempty[acc]);
        mbar_arrive(&s.empty[stage]);
      }
    }
    // uniform decision across the four epilogue warps (double-buffered vote)
    const int par = static_cast<int>(t & 1);
    if (lane == 0) s.misc->vote[par][warp - 2] = wok ? 1 : 0;
    named_sync(kEpiBarrier, kEpiThreads);
    if (!(s.misc->vote[par][0] & s.misc->vote[par][1] & s.misc->vote[par][2] &
          s.misc->vote[par][3])) {
      ok = false;
      break;
    }
    const int key = i * kTileKeys + mrow;
    if (kLogits) {
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (active[g] && key < len[g])
          p.out_logits[static_cast<int64_t>(wr.row0 + g) * p.ld_logits + key] = logit[g];
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (active[g] && s.misc->cnt[g] + kEpiThreads > C::kCap) compact<G>(s, g, p.topk);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint32_t k = float_key(logit[g]);
        append(s, g, C::kCap, active[g] && key < len[g] && k > s.misc->thr[g], k, key);
      }
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
  if (!kLogits && ok) finalize_segment<G>(p, s, w, wr, active, rs, re, t0, t1, T, nC);
}

template <int G, bool kLogits>
__global__ void __launch_bounds__(kThreads, 1)
    score_select_kernel(const __grid_constant__ ScoreParams p,
                        const __grid_constant__ CUtensorMap map) {
  using C = Cfg<G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Smem s = carve<G>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // With fewer tiles than CTAs only the first T CTAs take part, so that every
  // participating CTA owns at least one tile (segment counts rely on it).
  const int64_t T = p.wr_tile_start[p.num_wr];
  const int64_t nC = min(static_cast<int64_t>(gridDim.x), T);
  const bool part = static_cast<int64_t>(blockIdx.x) < nC;
  const int64_t t0 = part ? static_cast<int64_t>(blockIdx.x) * T / nC : 0;
  const int64_t t1 = part ? static_cast<int64_t>(blockIdx.x + 1) * T / nC : 0;

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
    s.misc->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&map);
  if (warp == 1) tmem_alloc(&s.misc->tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.misc->tmem_base;

  if (t0 < t1) {
    if (warp == 0) {
      if (lane == 0) producer<G>(p, &map, s, t0, t1);
    } else if (warp == 1) {
      if (lane == 0) mma_issuer<G>(p, s, tmem, t0, t1);
    } else {
      epilogue<G, kLogits>(p, s, tmem, t0, t1, T, nC);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int G, bool kLogits>
idx_status launch_impl(const ScoreParams& p, const CUtensorMap& map, int num_ctas, cudaStream_t s) {
  using C = Cfg<G>;
  static int configured_device = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
  if (configured_device != dev) {
    if (cudaFuncSetAttribute(score_select_kernel<G, kLogits>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return IDX_ERR_CUDA;
    configured_device = dev;
  }
  score_select_kernel<G, kLogits><<<num_ctas, kThreads, C::kSmemBytes, s>>>(p, map);
  return cudaPeekAtLastError() == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

}  // namespace

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
