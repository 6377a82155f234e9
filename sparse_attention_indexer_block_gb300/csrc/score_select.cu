// Score + select: the persistent kernel of the indexer.
//
// One CTA per SM (the occupancy of tensor-core kernels is one CTA per SM). The
// global sequence of 128-key tiles (work rows in order, each work row cut into
// ceil(maxlen / 128) tiles) is split into contiguous ranges ("streams"): for
// work rows of one token row (G = 1) a CTA runs two independent streams side
// by side, for work rows of two (G = 2) one stream whose two token rows are
// scored by separate epilogue groups. Warp-specialised, per stream j:
//   warp 2j      TMA producer: two 64-token pages per tile (8 KB of fp8 keys
//                via a 3-D tensor map with the 128-byte swizzle, 256 B of fp32
//                scales via a bulk copy each) into the stream's part of the
//                ring of shared-memory stages; the work row's fp8 q image
//                (G x 8 KB) into one of the stream's two q slots.
//   warp 2j + 1  MMA issuer: D[128 keys x 64G] = K_tile[128 x 128] .
//                Q[64G x 128]^T as four tcgen05 kind::f8f6f4 MMAs (K = 32 each)
//                into one of the stream's two tensor-memory accumulators.
//   warps 4-7 and 8-11: two epilogue groups (G = 1: one per stream; G = 2:
//           one per token row of the single stream). Each thread owns one key
//           (one TMEM lane), loads its group's 64 head dots, applies ReLU,
//           the folded head weights w * sq and the key's scale, and feeds the
//           logit to a streaming top-k: a shared-memory candidate buffer, a
//           threshold below which keys are dropped, and a radix select that
//           shrinks the buffer back to k when it fills. No logits row leaves
//           the SM.
// A work row covered by several streams is a set of segments. Each segment
// publishes the candidates it kept and adds their row-bin histogram to the
// row's; the row's top k is selected from them by the split-row selection
// kernel that runs after this one.
//
// MXFP4 keys (kMx): the stage area holds one 16 KB tile per stream for the
// MMA and, behind them, a ring of raw slots (a tile's two 4352-byte pages,
// three per stream). The producer copies raw pages into the ring; one tile
// ahead of its scoring, the epilogue group re-encodes a raw slot into its
// stream's tile as 128 e4m3 codes per key in the swizzled layout the MMA
// reads, with one power-of-two scale per key, and frees the raw slot; the
// MMA waits for that and frees the tile when it completes. An e2m1 value v of a block
// with exponent E_b becomes the e4m3 code of v * 2^(6 + E_b - E_max), E_max
// the key's largest block exponent, and the key's scale is 2^(E_max - 133):
// exact for every block within 2^11 of the key's largest (e4m3 normals;
// blocks further below are rounded to e4m3).
//
// Scoring (the method's statement; the pages name the kernel only):
//   logit[t, s] = sum_h w[t, h] ReLU(scale_s (q[t, h] . k_s))
//               = scale_s * sum_h (w[t, h] sq[t, h]) ReLU(q8[t, h] . k8_s),
// since scale_s >= 0 and q = q8 * sq per (token, head).
#include <atomic>

#include "internal.h"

namespace saib {

namespace {

constexpr int kThreads = 384;        // warps 0-3 TMA / MMA per stream, warps 4-11 two epilogue groups
constexpr int kEpiBase = 128;        // first epilogue thread
constexpr int kEpiThreads = 128;     // threads of one epilogue group
constexpr int kTeardownBarrier = 2;  // used once, by all warps, before TMEM is freed
constexpr int kSetupBarrier = 3;     // used once, by all warps, after barrier init and TMEM alloc
// (named barrier 1 belongs to epilogue group 0, 4 to group 1)

// Epilogue group of this thread (0: warps 4-7, 1: warps 8-11), its thread
// index in the group and the group's named barrier.
__device__ __forceinline__ int epi_group() { return (static_cast<int>(threadIdx.x) - kEpiBase) >> 7; }
__device__ __forceinline__ int epi_tid() { return (static_cast<int>(threadIdx.x) - kEpiBase) & 127; }
__device__ __forceinline__ void epi_sync() { named_sync(1 + 3 * epi_group(), kEpiThreads); }

template <int G>
struct Cfg {
  static constexpr int N = 64 * G;
  static constexpr int kStreams = score_streams_per_cta(G);  // tile streams per CTA
  static constexpr int kGroupsPerStream = 2 / kStreams;      // epilogue groups per stream
  static constexpr int kTokens = G / kGroupsPerStream;       // token rows per group
  static constexpr int kStages = score_stages(G);            // all streams
  static constexpr int kStreamStages = kStages / kStreams;
  static constexpr int kCap = candidate_capacity(G);  // candidates per token row
  static constexpr int kRegion = kCap / 4;            // per-warp append region
  // a full buffer is cut to at most k + kSlack entries (whichever bucket
  // boundary the radix search reaches first)
  static constexpr int kSlack = kCap / 24;
  static constexpr int kHistBins = 1024;
  static constexpr uint32_t kTmemCols = 2 * kStreams * N;  // two accumulators per stream
  static constexpr uint32_t kIdesc = f8_idesc(128, N);
  // Shared memory: the stage ring, the q slots (2 streams x 2), the scales,
  // then one block per epilogue group, the mbarriers and the CTA-wide words.
  static constexpr int kKvOff = 0;
  static constexpr int kQOff = kKvOff + kStages * 16384;
  static constexpr int kScaleOff = kQOff + 2 * kStreams * G * kQRowBytes;
  static constexpr int kGroupOff = kScaleOff + kStages * 512;
  static constexpr int kGCandKey = 0;
  static constexpr int kGCandIdx = kGCandKey + kTokens * kCap * 4;
  static constexpr int kGWp = kGCandIdx + kTokens * kCap * 4;
  static constexpr int kGHist = kGWp + kTokens * 256;
  static constexpr int kGMisc = kGHist + kHistBins * 4;
  static constexpr int kGTrace = kGMisc + 256;
  static constexpr int kGroupBytes = kGTrace + kTrSlots * 8;
  static constexpr int kBarOff = kGroupOff + 2 * kGroupBytes;
  static constexpr int kNumBars = 2 * kStages + 4 * 4 + 2 + 4;
  static constexpr int kSharedOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kSharedOff + 64 + 1024;  // + alignment slack
  static_assert(kCap % kEpiThreads == 0, "capacity");
  static_assert(kCap >= IDX_MAX_TOPK, "a slot must hold any k");
  static_assert(kTmemCols == 256, "tensor memory: a power of two the allocator takes");
  static_assert(kStreams * kGroupsPerStream == 2 && kTokens == 1, "one token row per group");
  static_assert(kGroupBytes % 16 == 0 && kGTrace % 8 == 0, "alignment");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

// Words shared by all roles of the CTA.
struct CtaShared {
  uint32_t tmem_base;
  int abort_flag;
  int epi_done;
};

// Scratch of one epilogue group.
struct Misc {
  int cnt[2];
  uint32_t thr[2];
  int bucket, above, bcount;
  int is_last;
  int vote[2][4];
  int scan[4];
  uint32_t rmin[4], rmax[4];
  int wcnt[2][4];   // [token][epilogue warp] entries in the warp's region
  int mx_ok;        // the raw pages of the stage being re-encoded arrived
};
static_assert(sizeof(Misc) <= 256, "misc block");

// The shared memory the roles of stream j (its producer, MMA issuer and
// epilogue group j) see: the common ring, q slots, scales and barriers, and
// the group's own candidate buffers, weights, histogram, scratch and trace
// slots.
struct Smem {
  uint8_t* kv;
  uint8_t* q;
  float* scales;
  uint32_t* ckey;
  int32_t* cidx;
  float* wp;
  uint32_t* hist;
  uint64_t* full;    // [kStages]: stream j owns stages [j, j + 1) * kStreamStages
  uint64_t* empty;   // [kStages]
  uint64_t* tfull;   // [4] accumulator 2j + b of stream j
  uint64_t* tempty;  // [4]
  uint64_t* qfull;   // [4] q slot 2j + b of stream j
  uint64_t* qempty;  // [4]
  uint64_t* done;    // [2] each stream's MMAs complete
  uint64_t* conv;    // [4] (MXFP4 keys) stream j's tile written (j), consumed (2 + j)
  Misc* misc;
  CtaShared* cs;
  uint64_t* trace;   // this stream's trace slots (shared memory, copied out at exit), or nullptr
  int group;
};

template <int G>
__device__ __forceinline__ Smem carve(uint8_t* base, int group) {
  using C = Cfg<G>;
  Smem s;
  s.kv = base + C::kKvOff;
  s.q = base + C::kQOff;
  s.scales = reinterpret_cast<float*>(base + C::kScaleOff);
  uint8_t* gb = base + C::kGroupOff + group * C::kGroupBytes;
  s.ckey = reinterpret_cast<uint32_t*>(gb + C::kGCandKey);
  s.cidx = reinterpret_cast<int32_t*>(gb + C::kGCandIdx);
  s.wp = reinterpret_cast<float*>(gb + C::kGWp);
  s.hist = reinterpret_cast<uint32_t*>(gb + C::kGHist);
  s.misc = reinterpret_cast<Misc*>(gb + C::kGMisc);
  s.trace = reinterpret_cast<uint64_t*>(gb + C::kGTrace);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  s.full = bars;
  s.empty = bars + C::kStages;
  s.tfull = bars + 2 * C::kStages;
  s.tempty = s.tfull + 4;
  s.qfull = s.tempty + 4;
  s.qempty = s.qfull + 4;
  s.done = s.qempty + 4;
  s.conv = s.done + 2;
  s.cs = reinterpret_cast<CtaShared*>(base + C::kSharedOff);
  s.group = group;
  return s;
}

// The stream of the CTA a role serves and the first token row of the work
// rows an epilogue group scores.
template <int G>
__device__ __forceinline__ int stream_of(const Smem& s) {
  return Cfg<G>::kStreams == 2 ? s.group : 0;
}
template <int G>
__device__ __forceinline__ int token_of(const Smem& s) {
  return Cfg<G>::kStreams == 2 ? 0 : s.group * Cfg<G>::kTokens;
}

// One of the CTA's tile streams: stream v = kStreams * blockIdx.x + j owns
// tiles [t0, t1) of the launch's tile sequence.
struct Stream {
  int64_t t0, t1;
  int v;
};

// Row histogram over the top 10 bits of the order-preserving key: sign, the
// 8 exponent bits and the leading mantissa bit (bins of half a binade).
__device__ __forceinline__ int row_bin(uint32_t key) { return static_cast<int>(key >> 22); }

// Index of split work row w (first virtual CTA v_first) among the launch's
// row histograms and cutoff-bin lists: the work row itself when the launch
// has no more work rows than virtual CTAs, else its first virtual CTA (split
// rows start in different virtual CTAs). Either way below
// max_split_rows(num_wr, 2 * gridDim.x).
template <int G>
__device__ __forceinline__ int64_t split_slot(const ScoreParams& p, int w, int v_first) {
  return p.num_wr <= Cfg<G>::kStreams * static_cast<int>(gridDim.x) ? w : v_first;
}

__device__ __forceinline__ void trace_set(const Smem& s, int slot, uint64_t v) {
  if (s.trace) s.trace[slot] = v;
}

// ---------------------------------------------------------------------------
// producer (one thread per stream)
// ---------------------------------------------------------------------------

// The block-table entries of a tile's two pages as read (kNoPage past the
// work row's pages), and the pages they name once checked (-1: none, or
// outside the cache, which is reported). Reading and checking are apart so
// that the producer can read one tile ahead without waiting for the load.
constexpr int32_t kNoPage = INT32_MIN;
struct TileRaw {
  int32_t v[2];
};
struct TilePages {
  int pid[2];
};

__device__ __forceinline__ TileRaw tile_raw(const int32_t* bt_row, int npages, int tile) {
  TileRaw r;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int pg = 2 * tile + h;
    r.v[h] = pg < npages ? bt_row[pg] : kNoPage;
  }
  return r;
}

__device__ __forceinline__ TilePages tile_check(const ScoreParams& p, const TileRaw& r) {
  TilePages tp;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    tp.pid[h] = -1;
    const int32_t pv = r.v[h];
    if (pv != kNoPage) {
      if (pv >= 0 && static_cast<int64_t>(pv) < p.num_pages) tp.pid[h] = pv;
      else set_error(p.dev_error, IDX_DEV_BAD_BLOCK);
    }
  }
  return tp;
}

// MXFP4 keys: stream j's MMA tile at kv + 16384 j, its raw slots (stage
// index of the ring, as for fp8 stages) from kv + kMxRawOff on.
constexpr int kMxRawOff = 2 * 16384;
constexpr int kMxRawSlot = 2 * kMxPageBytes;  // 8704
__device__ __forceinline__ uint8_t* mx_raw_slot(const Smem& s, int stage) {
  return s.kv + kMxRawOff + stage * kMxRawSlot;
}

template <int G, bool kMx>
__device__ void producer(const ScoreParams& p, const CUtensorMap* map, const Smem& s,
                         const Stream& st) {
  using C = Cfg<G>;
  static_assert(!kMx || (G == 1 && kMxRawOff + C::kStages * kMxRawSlot <= C::kStages * 16384),
                "MXFP4 tiles and raw slots fit the stage area");
  constexpr int S = C::kStreamStages;
  volatile int* abort_flag = &s.cs->abort_flag;
  const int j = stream_of<G>(s);
  uint64_t* full = s.full + j * S;
  uint64_t* empty = s.empty + j * S;
  uint8_t* kv = s.kv + j * S * 16384;
  float* scales = s.scales + j * S * 128;
  int last_par[S];
#pragma unroll
  for (int i = 0; i < S; ++i) last_par[i] = -1;
  uint32_t qn[2] = {0, 0};
  int qslot = 0;

  int w = p.cta_row[st.v];
  int64_t rs = p.wr_tile_start[w], re = p.wr_tile_start[w + 1];
  WorkRow wr = p.wr[w];
  bool ok = true;

  auto load_q = [&]() -> bool {
    const int q = 2 * j + qslot;
    if (qn[qslot] > 0 &&
        !mbar_wait(&s.qempty[q], (qn[qslot] - 1) & 1, abort_flag, p.dev_error, p.wait_ns))
      return false;
    const uint32_t bytes = static_cast<uint32_t>(wr.ntok) * kQRowBytes;
    mbar_arrive_expect_tx(&s.qfull[q], bytes);
    if (bytes)
      bulk_load(s.q + q * G * kQRowBytes, p.q8 + static_cast<int64_t>(wr.row0) * kQRowBytes,
                bytes, &s.qfull[q]);
    ++qn[qslot];
    return true;
  };

  ok = load_q();
  const int32_t* bt_row = p.block_table + static_cast<int64_t>(wr.req) * p.bt_stride;
  int npages = (wr.maxlen + kPageTokens - 1) / kPageTokens;
  // the page ids of the next tile are read one tile ahead (their load latency
  // overlaps the wait for a free stage)
  TileRaw next = tile_raw(bt_row, npages, static_cast<int>(st.t0 - rs));
  // the index pages are read once: first out of L2
  const uint64_t stream_policy = l2_evict_first_policy();

  int stage = 0;
  uint32_t phase = 0;
  for (int64_t t = st.t0; ok && t < st.t1; ++t) {
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
      next = tile_raw(bt_row, npages, static_cast<int>(t - rs));
    }
    const TilePages cur = tile_check(p, next);
    // (a stage's first use needs no wait: nothing has used it yet)
    if (t - st.t0 >= S && !mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.dev_error, p.wait_ns))
      break;
    uint32_t bytes = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      bytes += cur.pid[h] >= 0 ? (kMx ? kMxPageBytes : kPageValueBytes + 256) : 0;
    if (t == st.t0) trace_set(s, kTrFirstTma, globaltimer_ns());
    mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (cur.pid[h] < 0) continue;
      if constexpr (kMx) {
        bulk_load_hint(mx_raw_slot(s, j * S + stage) + h * kMxPageBytes,
                       p.cache + static_cast<int64_t>(cur.pid[h]) * kMxPageBytes, kMxPageBytes,
                       &full[stage], stream_policy);
      } else {
        tma_load_3d_hint(kv + stage * 16384 + h * kPageValueBytes, map, 0, 0, cur.pid[h],
                         &full[stage], stream_policy);
        bulk_load_hint(scales + stage * 128 + h * 64,
                       p.cache + static_cast<int64_t>(cur.pid[h]) * kPageBytes + kPageValueBytes,
                       256, &full[stage], stream_policy);
      }
    }
    // the next tile's block-table entries, read after this tile's copies are
    // issued (checked when that tile is issued)
    if (t + 1 < st.t1 && t + 1 < re) next = tile_raw(bt_row, npages, static_cast<int>(t + 1 - rs));
    last_par[stage] = static_cast<int>(phase);
    if (++stage == S) {
      stage = 0;
      phase ^= 1;
    }
  }
  trace_set(s, kTrLastTma, globaltimer_ns());
  // Every copy this thread issued lands before the CTA may exit.
  int dummy = 0;
#pragma unroll
  for (int i = 0; i < S; ++i)
    if (last_par[i] >= 0)
      mbar_wait(&full[i], static_cast<uint32_t>(last_par[i]), &dummy, p.dev_error);
  for (int q = 0; q < 2; ++q)
    if (qn[q] > 0) mbar_wait(&s.qfull[2 * j + q], (qn[q] - 1) & 1, &dummy, p.dev_error);
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread per stream)
// ---------------------------------------------------------------------------
template <int G, bool kMx>
__device__ void mma_issuer(const ScoreParams& p, const Smem& s, uint32_t tmem, const Stream& st) {
  using C = Cfg<G>;
  constexpr int S = C::kStreamStages;
  volatile int* abort_flag = &s.cs->abort_flag;
  const int j = stream_of<G>(s);
  uint64_t* full = s.full + j * S;
  uint64_t* empty = s.empty + j * S;
  const uint8_t* kv = s.kv + j * S * 16384;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t qn[2] = {0, 0};
  int qslot = 0;
  int w = p.cta_row[st.v];
  int64_t re = p.wr_tile_start[w + 1];
  bool issued = false;
  bool ok = mbar_wait(&s.qfull[2 * j], 0, abort_flag, p.dev_error, p.wait_ns);
  for (int64_t t = st.t0, k = 0; ok && t < st.t1; ++t, ++k) {
    if (*abort_flag) break;
    if (t >= re) {
      mma_commit(&s.qempty[2 * j + qslot]);  // q slot free once this row's MMAs finish
      ++qn[qslot];
      do {
        ++w;
        re = p.wr_tile_start[w + 1];
      } while (t >= re);
      qslot ^= 1;
      if (!mbar_wait(&s.qfull[2 * j + qslot], qn[qslot] & 1, abort_flag, p.dev_error, p.wait_ns))
        break;
    }
    const int acc = 2 * j + static_cast<int>(k & 1);
    const uint32_t acc_par = static_cast<uint32_t>((k >> 1) & 1);
    // the keys are in shared memory: copied (fp8), or re-encoded into the
    // stream's tile (MXFP4)
    if (!mbar_wait(kMx ? &s.conv[j] : &full[stage], kMx ? static_cast<uint32_t>(k & 1) : phase,
                   abort_flag, p.dev_error, p.wait_ns))
      break;
    // (an accumulator's first use needs no wait)
    if (k >= 2 && !mbar_wait(&s.tempty[acc], acc_par ^ 1, abort_flag, p.dev_error, p.wait_ns)) break;
    tc_fence_after();
    if (k == 0) trace_set(s, kTrFirstMma, globaltimer_ns());
    const uint32_t a_base = smem_u32(kMx ? s.kv + j * 16384 : kv + stage * 16384);
    const uint32_t b_base = smem_u32(s.q + (2 * j + qslot) * G * kQRowBytes);
    const uint32_t d = tmem + static_cast<uint32_t>(acc * C::N);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f8(d, sw128_kmajor_desc(a_base + kk * 32), sw128_kmajor_desc(b_base + kk * 32),
             C::kIdesc, kk > 0 ? 1u : 0u);
    mma_commit(kMx ? &s.conv[2 + j] : &empty[stage]);  // (MXFP4: the stream's tile is free)
    mma_commit(&s.tfull[acc]);
    issued = true;
    if (++stage == S) {
      stage = 0;
      phase ^= 1;
    }
  }
  trace_set(s, kTrLastMma, globaltimer_ns());
  if (issued) {
    // all of this stream's MMAs complete before tensor memory is released
    mma_commit(&s.done[j]);
    int dummy = 0;
    mbar_wait(&s.done[j], 0, &dummy, p.dev_error);
  }
}
// ---------------------------------------------------------------------------
// epilogue: streaming top-k over a shared-memory candidate buffer
// ---------------------------------------------------------------------------

// Exclusive scan of one int per epilogue thread (in thread order); *total gets
// the sum. Contains one epilogue barrier.
__device__ __forceinline__ int epi_exclusive_scan(Misc* m, int v, int* total) {
  const int lane = threadIdx.x & 31, ew = epi_tid() >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) m->scan[ew] = x;
  epi_sync();
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
  const int et = epi_tid();
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
  epi_sync();
  *bucket = m->bucket;
  *above = m->above;
  *bcount = m->bcount;
}

// The K-th largest key of token g's buffer (the group's four per-warp
// regions in shared memory, counts in wcnt[g][*]; K <= their total): an
// MSB-first radix select over v = key - min (10-bit digits below the top bit
// of max - min, so the bins spread over the keys present) with one shared
// histogram (zero on entry and on exit), reading the keys where they lie.
// Result: *mn (min key), *hi and *pre (keys with (key - mn) >> hi > pre are
// in, those equal to pre are tied) and *rem (how many tied keys complete K).
// With slack > 0 the search may stop early at a bucket that holds at most
// `slack` keys beyond K: the whole bucket is then taken (*rem = its count),
// so up to K + slack keys are in. Contains epilogue barriers; all epilogue
// threads.
template <int G>
__device__ void radix_kth(const Smem& s, int g, int K, uint32_t* mn_out, int* hi_out,
                          uint64_t* pre_out, int* rem_out, int slack = 0) {
  using C = Cfg<G>;
  const int et = epi_tid();
  const int lane = threadIdx.x & 31, ew = et >> 5;
  Misc* m = s.misc;
  const uint32_t* rk = s.ckey + g * C::kCap + ew * C::kRegion;
  const int n_w = m->wcnt[g][ew];
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int r = lane; r < n_w; r += 32) {
    const uint32_t u = rk[r];
    mn = min(mn, u);
    mx = max(mx, u);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    m->rmin[ew] = mn;
    m->rmax[ew] = mx;
  }
  epi_sync();
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
    for (int r = lane; r < n_w; r += 32) {
      const uint64_t v = rk[r] - mn;
      if ((v >> hi) == pre) atomicAdd(&s.hist[(v >> lo) & static_cast<uint64_t>(nb - 1)], 1u);
    }
    epi_sync();
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

// Cuts token g's buffer to its K largest keys (all of them when there are
// <= K; up to K + slack when the radix search stops early; ties at the K-th
// value broken arbitrarily): radix_kth finds the cut, then every warp packs
// the kept entries of its own region to the region's front, in place (a
// kept entry never moves past one not yet read). The drop threshold becomes
// min + (resolved prefix of the K-th key): keys at or below it cannot
// displace the kept ones. Leaves each warp's count in wcnt[g][*], sets
// cnt[g] to the entries kept and returns it; all epilogue threads.
template <int G>
__device__ int compact(const Smem& s, int g, int K, int slack = 0) {
  using C = Cfg<G>;
  const int et = epi_tid();
  const int lane = threadIdx.x & 31, ew = et >> 5;
  Misc* m = s.misc;
  uint32_t* rk = s.ckey + g * C::kCap + ew * C::kRegion;
  int32_t* rx = s.cidx + g * C::kCap + ew * C::kRegion;
  const uint64_t tc0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  const int n_w = m->wcnt[g][ew];
  const int n = m->wcnt[g][0] + m->wcnt[g][1] + m->wcnt[g][2] + m->wcnt[g][3];
  if (n <= K) return n;  // uniform: nothing to cut
  uint32_t mn = 0;
  int hi = 0, remaining = 0;
  uint64_t pre = 0;
  {
    const uint64_t tr0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
    radix_kth<G>(s, g, K, &mn, &hi, &pre, &remaining, slack);
    if (et == 0 && s.trace) s.trace[kTrCompactRadixNs] += globaltimer_ns() - tr0;
  }
  // tied keys are taken in warp order, then region order, until `remaining`
  int n_eq = 0;
  for (int r = lane; r < n_w; r += 32) n_eq += ((rk[r] - mn) >> hi) == pre ? 1 : 0;
  n_eq = __reduce_add_sync(0xffffffffu, n_eq);
  if (lane == 0) m->scan[ew] = n_eq;
  epi_sync();
  int eq_seen = 0;  // tied keys of the warps before this one, then of this warp so far
  for (int i = 0; i < ew; ++i) eq_seen += m->scan[i];
  const unsigned below = (1u << lane) - 1u;
  int kept_w = 0;
  for (int c0 = 0; c0 < n_w; c0 += 32) {
    const int r = c0 + lane;
    const bool in = r < n_w;
    const uint32_t key = in ? rk[r] : 0u;
    const int32_t idx = in ? rx[r] : 0;
    const uint64_t top = static_cast<uint64_t>(key - mn) >> hi;
    const bool eq = in && top == pre;
    const unsigned em = __ballot_sync(0xffffffffu, eq);
    const bool keep = (in && top > pre) || (eq && eq_seen + __popc(em & below) < remaining);
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    __syncwarp();  // every lane has read its entry before any is overwritten
    if (keep) {
      const int d = kept_w + __popc(km & below);
      rk[d] = key;
      rx[d] = idx;
    }
    __syncwarp();
    kept_w += __popc(km);
    eq_seen += __popc(em);
  }
  if (lane == 0) m->wcnt[g][ew] = kept_w;
  epi_sync();
  const int kept = m->wcnt[g][0] + m->wcnt[g][1] + m->wcnt[g][2] + m->wcnt[g][3];
  if (et == 0) {
    m->cnt[g] = kept;
    m->thr[g] = max(m->thr[g], mn + static_cast<uint32_t>(pre << hi));
    if (s.trace) {
      s.trace[kTrCompactNs] += globaltimer_ns() - tc0;
      s.trace[kTrCompactN] += 1;
    }
  }
  epi_sync();
  return kept;
}

// Entries of token g's buffer sit in four per-warp regions (counts in
// wcnt[g][*]); warp w's lane l visits its region's entries l, l + 32, ...
template <int G>
__device__ __forceinline__ int region_entries(const Smem& s, int g) {
  const int lane = threadIdx.x & 31, ew = epi_tid() >> 5;
  const int nw = s.misc->wcnt[g][ew];
  return lane < nw ? (nw - lane + 31) / 32 : 0;
}

// Output of a row held entirely by this CTA (its buffer holds <= k entries),
// with each index's logit when values are asked for.
template <int G>
__device__ void write_rows(const ScoreParams& p, const Smem& s, const WorkRow& wr,
                           const bool (&active)[Cfg<G>::kTokens]) {
  using C = Cfg<G>;
  const int et = epi_tid();
  const int lane = threadIdx.x & 31, ew = et >> 5;
#pragma unroll
  for (int g = 0; g < C::kTokens; ++g) {
    if (!active[g]) continue;
    const int mine = region_entries<G>(s, g);
    int total;
    int pos = epi_exclusive_scan(s.misc, mine, &total);
    const int64_t row = p.out_row_base + wr.row0 + token_of<G>(s) + g;
    int32_t* o = p.out_idx + row * p.topk;
    float* ov = p.out_val ? p.out_val + row * p.topk : nullptr;
    const int32_t* rx = s.cidx + g * C::kCap + ew * C::kRegion;
    const uint32_t* rk = s.ckey + g * C::kCap + ew * C::kRegion;
    for (int j = 0; j < mine; ++j)
      if (pos < p.topk) {
        if (ov) ov[pos] = key_float(rk[lane + 32 * j]);
        o[pos++] = rx[lane + 32 * j];
      }
    for (int e = total + et; e < p.topk; e += kEpiThreads) {
      o[e] = -1;
      if (ov) ov[e] = -INFINITY;
    }
    epi_sync();
  }
}

// ---------------------------------------------------------------------------
// segments of split rows
// ---------------------------------------------------------------------------

// Row-histogram bins one epilogue thread holds in the segment's bin sort:
// [hi - 7, hi] with hi = 1023 - 8 * et (highest bins first in thread order).
constexpr int kBinsPerThread = kRowHistBins / kEpiThreads;
static_assert(kBinsPerThread == 8, "bin split");

// End of this stream's part of work row w. A row held whole by this stream
// is cut to k and written out. A split row's segment publishes, per token
// row: its final buffer sorted by row bin, highest first, into the segment's
// slot (keys and token indices), the number of its entries at or above every
// row bin, and its counts added to the row histogram; then the segment
// counts itself in on the row's counter (which the selection kernel checks).
template <int G>
__device__ void finalize_segment(const ScoreParams& p, const Smem& s, int v, int w,
                                 const WorkRow& wr, const bool (&active)[Cfg<G>::kTokens], int64_t rs,
                                 int64_t re, int64_t t0, int64_t t1) {
  using C = Cfg<G>;
  const int et = epi_tid();
  const int K = p.topk;
  Misc* m = s.misc;
  const uint64_t tf0 = (et == 0 && s.trace) ? globaltimer_ns() : 0;
  const int lane = threadIdx.x & 31, ew = et >> 5;
  epi_sync();
  const bool whole = rs >= t0 && re <= t1;
  if (whole) {
#pragma unroll
    for (int g = 0; g < C::kTokens; ++g)
      if (active[g] && m->wcnt[g][0] + m->wcnt[g][1] + m->wcnt[g][2] + m->wcnt[g][3] > K)
        compact<G>(s, g, K);  // cut to k (the regions stay the layout)
    write_rows<G>(p, s, wr, active);
    if (et == 0 && s.trace) s.trace[kTrFinalizeNs] += globaltimer_ns() - tf0;
    return;
  }
  const int2 rc = p.row_ctas[w];
  uint32_t* gh_base = p.row_hist + split_slot<G>(p, w, rc.x) * G * kRowHistBins;
  const int64_t slot = segment_slot(v, w == p.cta_row[v]);
  uint64_t tf1 = tf0;
  const int hi = kRowHistBins - 1 - kBinsPerThread * et;
  const int g0 = token_of<G>(s);
#pragma unroll
  for (int g = 0; g < C::kTokens; ++g) {
    uint32_t* gh = gh_base + (g0 + g) * kRowHistBins;
    const uint32_t* rk = s.ckey + g * C::kCap + ew * C::kRegion;
    const int32_t* rx = s.cidx + g * C::kCap + ew * C::kRegion;
    const int nw = active[g] ? m->wcnt[g][ew] : 0;
    // the buffer's row-bin histogram in shared memory
    for (int j = lane; j < nw; j += 32) atomicAdd(&s.hist[row_bin(rk[j])], 1u);
    epi_sync();
    int c[kBinsPerThread];
    int local = 0;
#pragma unroll
    for (int i = 0; i < kBinsPerThread; ++i) {
      c[i] = static_cast<int>(s.hist[hi - i]);
      local += c[i];
    }
    int tot;
    int run = epi_exclusive_scan(m, local, &tot);  // entries in higher bins
    // per bin: the row histogram, the entries at or above it, and (in the
    // shared histogram) the first slot position of its entries
    uint32_t* cum = p.seg_cum + (slot * G + g0 + g) * kRowHistBins;
#pragma unroll
    for (int i = 0; i < kBinsPerThread; ++i) {
      if (c[i]) atomicAdd(&gh[hi - i], static_cast<uint32_t>(c[i]));
      s.hist[hi - i] = static_cast<uint32_t>(run);
      run += c[i];
      cum[hi - i] = static_cast<uint32_t>(run);
    }
    epi_sync();
    if (et == 0 && s.trace) {
      const uint64_t now = globaltimer_ns();
      s.trace[kTrFinHistNs] += now - tf1;
      tf1 = now;
    }
    // the entries to their bins' positions
    const int64_t base = (slot * G + g0 + g) * p.slot_cap;
    for (int j = lane; j < nw; j += 32) {
      const uint32_t key = rk[j];
      const int64_t pos = base + atomicAdd(&s.hist[row_bin(key)], 1u);
      p.slot_key[pos] = key;
      p.slot_idx[pos] = rx[j];
    }
    epi_sync();
#pragma unroll
    for (int i = 0; i < kBinsPerThread; ++i) s.hist[hi - i] = 0u;
    epi_sync();  // the shared histogram is zero again (reused for token g + 1)
    if (et == 0 && s.trace) {
      const uint64_t now = globaltimer_ns();
      s.trace[kTrFinEmitNs] += now - tf1;
      tf1 = now;
    }
  }
  // the selection kernel reads all this after this kernel has completed; the
  // counter only lets it check that every segment published
  if (et == 0) {
    atomicAdd(&p.seg_counter[w], 1);
    if (s.trace) {
      s.trace[kTrFinPublishNs] += globaltimer_ns() - tf1;
      s.trace[kTrFinalizeNs] += globaltimer_ns() - tf0;
    }
  }
}

// ---------------------------------------------------------------------------
// MXFP4 keys: re-encoding a stage for the fp8 MMA
// ---------------------------------------------------------------------------

// 2^e as fp32 (0 below the subnormal range), built from its bits.
__device__ __forceinline__ float pow2f(int e) {
  if (e >= -126) return __int_as_float((e + 127) << 23);
  if (e >= -149) return __int_as_float(1 << (e + 149));
  return 0.f;
}

// e4m3 codes of the e2m1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 scaled by
// 2^t, as two words (codes of magnitudes 0-3, 4-7) for byte permutes. For
// t >= -5 every scaled magnitude is an e4m3 normal (or 0) and its code is the
// unscaled code with t added to the exponent field (mx_lut); below, the
// scaled values are rounded to e4m3 (mx_lut_small, out of line: rare).
__device__ __forceinline__ uint2 mx_lut(int t) {
  constexpr uint32_t kLo = 0x3C383000u;  // 1.5, 1, 0.5, 0
  constexpr uint32_t kHi = 0x4C484440u;  // 6, 4, 3, 2
  const uint32_t d = static_cast<uint32_t>(t * 8);  // per-byte exponent step, no carries
  return make_uint2(kLo + d * 0x01010100u, kHi + d * 0x01010101u);
}

__device__ __noinline__ uint2 mx_lut_small(int t) {
  const float u = pow2f(t);
  const uint32_t lo = static_cast<uint32_t>(cvt_e4m3x2(0.f, 0.5f * u)) |
                      (static_cast<uint32_t>(cvt_e4m3x2(u, 1.5f * u)) << 16);
  const uint32_t hi = static_cast<uint32_t>(cvt_e4m3x2(2.f * u, 3.f * u)) |
                      (static_cast<uint32_t>(cvt_e4m3x2(4.f * u, 6.f * u)) << 16);
  return make_uint2(lo, hi);
}

// The epilogue group re-encodes tile c of stream j (raw slot `stage`, whose
// pages landed with phase `phase`) into the stream's MMA tile once the MMA
// of tile c - 1 has released it: thread et writes key et's 128 e4m3 codes
// as row et of the swizzled tile (16-byte chunk c at c ^ (et mod 8)) and the
// key's scale, makes them visible to the tensor cores, and its warp counts
// in on the tile and on the raw slot. Returns false (in every thread of the
// group alike) when a wait gave up.
template <int G>
__device__ bool mx_convert(const ScoreParams& p, const Smem& s, int j, int64_t c, int stage,
                           uint32_t phase, volatile int* abort_flag) {
  const int et = epi_tid();
  const int lane = threadIdx.x & 31;
  if (et == 0)
    s.misc->mx_ok =
        mbar_wait(&s.full[stage], phase, abort_flag, p.dev_error, p.wait_ns) &&
                (c == 0 || mbar_wait(&s.conv[2 + j], static_cast<uint32_t>((c - 1) & 1),
                                     abort_flag, p.dev_error, p.wait_ns))
            ? 1
            : 0;
  epi_sync();
  const bool wok = s.misc->mx_ok != 0;
  uint8_t* tile = s.kv + j * 16384;
  const uint32_t* raw = reinterpret_cast<const uint32_t*>(
      mx_raw_slot(s, stage) + (et >> 6) * kMxPageBytes + (et & 63) * kMxTokenBytes);
  uint32_t w[17];
#pragma unroll
  for (int i = 0; i < 17; ++i) w[i] = wok ? raw[i] : 0u;
  if (wok) {
    const uint32_t e = w[16];
    const int eb[4] = {static_cast<int>(e & 255u), static_cast<int>((e >> 8) & 255u),
                       static_cast<int>((e >> 16) & 255u), static_cast<int>(e >> 24)};
    const int emax = max(max(eb[0], eb[1]), max(eb[2], eb[3]));
    s.scales[stage * 128 + et] = pow2f(emax - 133);
    uint2 lut[4];
    const int emin = min(min(eb[0], eb[1]), min(eb[2], eb[3]));
    if (6 + emin - emax >= -5) {
#pragma unroll
      for (int b = 0; b < 4; ++b) lut[b] = mx_lut(6 + eb[b] - emax);
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b)
        lut[b] = 6 + eb[b] - emax >= -5 ? mx_lut(6 + eb[b] - emax)
                                        : mx_lut_small(6 + eb[b] - emax);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t x = w[2 * c + h];
        const uint2 l = lut[c >> 1];
        // magnitudes (bits 0-2 of each nibble) through the table, signs
        // (bit 3) to bit 7 of each byte (a permute reads the low 16 bits of
        // its selector)
        const uint32_t mag = x & 0x77777777u, sgn = (x >> 3) & 0x11111111u;
        o[2 * h] = __byte_perm(l.x, l.y, mag) | __byte_perm(0x8000u, 0u, sgn);
        o[2 * h + 1] = __byte_perm(l.x, l.y, mag >> 16) | __byte_perm(0x8000u, 0u, sgn >> 16);
      }
      *reinterpret_cast<uint4*>(tile + et * 128 + ((c ^ (et & 7)) << 4)) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
    fence_proxy_async_shared();
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(&s.conv[j]);       // the tile is ready for the MMA
    mbar_arrive(&s.empty[stage]);  // the raw slot is free
  }
  return wok;
}

// ---------------------------------------------------------------------------
// epilogue group: one stream's tiles
// ---------------------------------------------------------------------------

// Streams epilogue group j's tiles (stream j of the CTA) through the score
// and the streaming top-k, finalising each work row's segment as it ends.
// Returns false when a pipeline wait gave up. All threads of the group.
template <int G, bool kLogits, bool kMx>
__device__ bool epilogue(const ScoreParams& p, const Smem& s, uint32_t tmem, const Stream (&st)[2],
                         int j) {
  using C = Cfg<G>;
  volatile int* abort_flag = &s.cs->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int et = epi_tid();
  const int ew = et >> 5;
  const int sub = warp & 3;          // tensor-memory lanes [32*sub, 32*sub + 32)
  const int mrow = sub * 32 + lane;  // key of the tile this thread scores
  const uint32_t lane_addr = static_cast<uint32_t>(sub * 32) << 16;
  constexpr int S = C::kStreamStages;
  const int64_t t0 = st[j].t0, t1 = st[j].t1;
  const int v = st[j].v;

  for (int b = et; b < C::kHistBins; b += kEpiThreads) s.hist[b] = 0u;  // zero between uses
  if (t0 >= t1) return true;

  int w = p.cta_row[v];
  int64_t rs = p.wr_tile_start[w], re = p.wr_tile_start[w + 1];
  WorkRow wr;
  constexpr int GT = C::kTokens;  // token rows g0, g0 + 1, ... of the group
  const int g0 = token_of<G>(s);
  int len[GT];
  bool active[GT];
  int wcnt[GT];      // entries in this warp's region of each token's buffer
  uint32_t thr[GT];  // each buffer's drop threshold

  auto begin_row = [&]() {
    wr = p.wr[w];
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      len[g] = g0 + g < wr.ntok ? p.row_len[wr.row0 + g0 + g] : 0;
      active[g] = g0 + g < wr.ntok && (kLogits ? len[g] > 0 : len[g] > p.short_len);
    }
    for (int i = et; i < GT * kHeads; i += kEpiThreads) {
      const int g = g0 + i / kHeads;
      s.wp[i] =
          g < wr.ntok ? p.wprime[static_cast<int64_t>(wr.row0 + g) * kHeads + i % kHeads] : 0.f;
    }
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      wcnt[g] = 0;
      thr[g] = 0u;
    }
    if (et == 0) {
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        s.misc->cnt[g] = 0;
        s.misc->thr[g] = 0u;
      }
    }
    epi_sync();
  };
  auto publish_counts = [&]() {
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < GT; ++g) s.misc->wcnt[g][ew] = wcnt[g];
  };
  begin_row();

  bool ok = true;
  // MXFP4 keys: tile k + 1 is re-encoded before tile k is scored (the MMA
  // of tile k, which it waits for, was enabled one iteration earlier)
  if constexpr (kMx) {
    if (t0 < t1)
      ok = mx_convert<G>(p, s, j, 0, j * S, 0u, abort_flag);
  }
  long long cyc[5] = {0, 0, 0, 0, 0};  // per-phase clock totals (trace only)
  for (int64_t k = 0; (kMx ? ok : true) && t0 + k < t1; ++k) {
    const int64_t t = t0 + k;
    if constexpr (kMx) {
      const int64_t c = k + 1;
      if (t0 + c < t1 && !mx_convert<G>(p, s, j, c, j * S + static_cast<int>(c % S),
                                        static_cast<uint32_t>((c / S) & 1), abort_flag)) {
        ok = false;
        break;
      }
    }
    if (t >= re) {
      publish_counts();
      if (!kLogits) finalize_segment<G>(p, s, v, w, wr, active, rs, re, t0, t1);
      do {
        ++w;
        re = p.wr_tile_start[w + 1];
      } while (t >= re);
      rs = p.wr_tile_start[w];
      epi_sync();
      begin_row();
    }
    const int i = static_cast<int>(t - rs);
    const int stage = j * S + static_cast<int>(k % S);
    const uint32_t phase = static_cast<uint32_t>((k / S) & 1);
    const int acc = 2 * j + static_cast<int>(k & 1);
    const uint32_t acc_par = static_cast<uint32_t>((k >> 1) & 1);
    const bool tr = s.trace != nullptr;  // per-phase clocks only when tracing
    const long long c0 = tr ? clock64() : 0;
    // lane 0 of each warp waits for the stage (scales) and the accumulator
    bool wok = true;
    if (lane == 0)
      // (MXFP4: the group wrote the scales itself; the raw slot may be
      // holding a later tile already)
      wok = (kMx || mbar_wait(&s.full[stage], phase, abort_flag, p.dev_error, p.wait_ns)) &&
            mbar_wait(&s.tfull[acc], acc_par, abort_flag, p.dev_error, p.wait_ns);
    wok = __shfl_sync(0xffffffffu, wok ? 1 : 0, 0) != 0;
    __syncwarp();
    const long long c1 = tr ? clock64() : 0;
    long long c2 = c1;
    float logit[GT];
    if (k == 0 && et == 0 && s.trace) s.trace[kTrFirstEpi] = globaltimer_ns();
    if (wok) {
      tc_fence_after();
      const float scale = s.scales[stage * 128 + mrow];
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        const uint32_t col = lane_addr + tmem + static_cast<uint32_t>(acc * C::N + (g0 + g) * 64);
        float v0[32], v1[32];
        tmem_ld32(col, v0);
        tmem_ld32(col + 32, v1);
        tmem_ld_wait();
        if (g == 0 && tr) c2 = clock64();
        const float4* w4 = reinterpret_cast<const float4*>(s.wp + g * kHeads);
        // four chains (heads h = c mod 4) as two packed pairs (c = 0, 1 and
        // c = 2, 3): the same fp32 FMAs in the same order
        uint64_t a01 = 0ull, a23 = 0ull;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 x = w4[q];
          a01 = fma_f32x2(pack_f32x2(x.x, x.y),
                          pack_f32x2(fmaxf(v0[4 * q + 0], 0.f), fmaxf(v0[4 * q + 1], 0.f)), a01);
          a23 = fma_f32x2(pack_f32x2(x.z, x.w),
                          pack_f32x2(fmaxf(v0[4 * q + 2], 0.f), fmaxf(v0[4 * q + 3], 0.f)), a23);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 x = w4[8 + q];
          a01 = fma_f32x2(pack_f32x2(x.x, x.y),
                          pack_f32x2(fmaxf(v1[4 * q + 0], 0.f), fmaxf(v1[4 * q + 1], 0.f)), a01);
          a23 = fma_f32x2(pack_f32x2(x.z, x.w),
                          pack_f32x2(fmaxf(v1[4 * q + 2], 0.f), fmaxf(v1[4 * q + 3], 0.f)), a23);
        }
        const float2 s01 = unpack_f32x2(a01), s23 = unpack_f32x2(a23);
        logit[g] = ((s01.x + s01.y) + (s23.x + s23.y)) * scale;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s.tempty[acc]);
        if (!kMx) mbar_arrive(&s.empty[stage]);
      }
    }
    const long long c3 = tr ? clock64() : 0;
    // Uniform decision across the group's four warps (double-buffered vote):
    // bit 0 = this warp's waits succeeded, bit 1 + g = its region of token g's
    // buffer has no room for another tile (then all warps compact it).
    const int par = static_cast<int>(k & 1);
    int need = 0;
#pragma unroll
    for (int g = 0; g < GT; ++g)
      need |= (!kLogits && active[g] && wcnt[g] + 32 > C::kRegion) ? 2 << g : 0;
    publish_counts();
    if (lane == 0) s.misc->vote[par][ew] = (wok ? 1 : 0) | need;
    epi_sync();
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
      for (int g = 0; g < GT; ++g)
        if (active[g] && key < len[g])
          p.out_logits[static_cast<int64_t>(wr.row0 + g0 + g) * p.ld_logits + key] = logit[g];
    } else {
#pragma unroll
      for (int g = 0; g < GT; ++g)
        if ((needs >> g) & 1) {
          compact<G>(s, g, p.topk, C::kSlack);
          wcnt[g] = s.misc->wcnt[g][ew];
          thr[g] = s.misc->thr[g];
        }
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        // append to this warp's region: ballot + popc, no shared counter
        const uint32_t kk = float_key(logit[g]);
        const bool pass = active[g] && key < len[g] && kk > thr[g];
        const unsigned pm = __ballot_sync(0xffffffffu, pass);
        if (pass) {
          const int at =
              g * C::kCap + ew * C::kRegion + wcnt[g] + __popc(pm & ((1u << lane) - 1u));
          s.ckey[at] = kk;
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
  if (!kLogits && ok) finalize_segment<G>(p, s, v, w, wr, active, rs, re, t0, t1);
  return ok;
}

template <int G, bool kLogits, bool kMx>
__global__ void __launch_bounds__(kThreads, 1)
    score_select_kernel(const __grid_constant__ ScoreParams p,
                        const __grid_constant__ CUtensorMap map) {
  using C = Cfg<G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the stream this thread serves: warps 2j, 2j + 1 and epilogue group j
  const int group = warp < 4 ? (warp >> 1) : epi_group();
  Smem s = carve<G>(base, group);

  // The shared-memory setup (barriers, tensor memory) needs nothing from
  // earlier kernels and overlaps their tail; everything after pdl_wait() may
  // read what they wrote.
  if (!kMx && warp == 0 && lane == 0) prefetch_tensormap(&map);  // (MXFP4 pages: bulk copies)
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&s.full[i], 1);
      // the MMA's commit + the warps of the groups consuming the stage (MXFP4
      // raw slots: the converting group's warps)
      mbar_init(&s.empty[i], kMx ? 4 : 1 + 4 * C::kGroupsPerStream);
    }
    for (int a = 0; a < 4; ++a) {
      mbar_init(&s.tfull[a], 1);
      mbar_init(&s.tempty[a], 4 * C::kGroupsPerStream);
      mbar_init(&s.qfull[a], 1);
      mbar_init(&s.qempty[a], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(s.done + i, 1);
    if constexpr (kMx) {
      for (int i = 0; i < 2; ++i) mbar_init(&s.conv[i], 4);      // stream i's tile written
      for (int i = 2; i < 4; ++i) mbar_init(&s.conv[i], 1);      // ... and consumed (MMA)
    }
    s.cs->abort_flag = 0;
    s.cs->epi_done = 0;
    for (int gi = 0; gi < 2; ++gi) {
      const Smem sg = carve<G>(base, gi);
      for (int i = 0; i < kTrSlots; ++i) sg.trace[i] = 0;
    }
    fence_barrier_init();
  }
  __syncwarp();  // warp 0 reconverges before the block barrier (which counts whole warps)
  if (warp == 1) tmem_alloc(&s.cs->tmem_base, C::kTmemCols);
  tc_fence_before();
  named_sync(kSetupBarrier, kThreads);
  tc_fence_after();
  pdl_wait();

  // With fewer tiles than virtual CTAs only the first T take part, so that
  // every participating stream owns at least one tile (segment counts rely
  // on it).
  const int64_t T = p.wr_tile_start[p.num_wr];
  const int64_t nV = min(static_cast<int64_t>(C::kStreams * gridDim.x), T);
  Stream st[2];
  bool part[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int v = C::kStreams * static_cast<int>(blockIdx.x) + j;
    part[j] = j < C::kStreams && v < nV;
    st[j].v = v;
    st[j].t0 = part[j] ? p.cta_tile[v] : 0;
    st[j].t1 = part[j] ? p.cta_tile[v + 1] : 0;
  }
  // stream of this thread's role (warps 2 and 3 have none when kStreams == 1)
  const int js = warp < 4 ? (warp >> 1) : stream_of<G>(s);
  if (!(p.trace && part[js] && token_of<G>(s) == 0)) s.trace = nullptr;

  pdl_trigger();
  const uint32_t tmem = s.cs->tmem_base;
  if (warp >= 4 && epi_tid() == 0 && s.trace) {
    s.trace[kTrStart] = globaltimer_ns();
    s.trace[kTrTiles] = static_cast<uint64_t>(st[js].t1 - st[js].t0);
  }

  if (warp < 4) {
    // one lane runs the role; the warp reconverges before the block barrier
    const bool has_tiles = part[js] && st[js].t1 > st[js].t0;
    if (lane == 0 && has_tiles) {
      if (warp & 1) mma_issuer<G, kMx>(p, s, tmem, st[js]);
      else producer<G, kMx>(p, &map, s, st[js]);
    }
    __syncwarp();
  } else {
    epilogue<G, kLogits, kMx>(p, s, tmem, st, js);
    if (s.trace && epi_tid() == 0) s.trace[kTrFinal] = globaltimer_ns();
  }
  if (threadIdx.x == kEpiBase) *reinterpret_cast<volatile int*>(&s.cs->epi_done) = 1;
  tc_fence_before();
  named_sync(kTeardownBarrier, kThreads);
  if (warp >= 4 && s.trace) {
    if (epi_tid() == 0) s.trace[kTrEnd] = globaltimer_ns();
    __syncwarp();
    if (epi_tid() < kTrSlots)
      p.trace[static_cast<int64_t>(st[js].v) * kTrSlots + epi_tid()] = s.trace[epi_tid()];
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int G, bool kLogits, bool kMx>
idx_status launch_impl(const ScoreParams& p, const CUtensorMap& map, int num_ctas, cudaStream_t s) {
  using C = Cfg<G>;
  // the dynamic shared-memory limit is a per-device attribute of the kernel:
  // set once per device (any host thread; setting it twice is harmless)
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidDevice);
  if (dev >= kMaxDevices || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(score_select_kernel<G, kLogits, kMx>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < kMaxDevices) configured[dev].store(true, std::memory_order_release);
  }
  return cuda_status(launch_pdl(score_select_kernel<G, kLogits, kMx>, num_ctas, kThreads, C::kSmemBytes,
                                s, p, map));
}

}  // namespace

idx_status launch_score(int G, bool logits, bool mx, const ScoreParams& p, const CUtensorMap& map,
                        int num_ctas, cudaStream_t s) {
  if (mx) {  // MXFP4 keys: one-token work rows
    if (G != 1) return IDX_ERR_UNSUPPORTED;
    return logits ? launch_impl<1, true, true>(p, map, num_ctas, s)
                  : launch_impl<1, false, true>(p, map, num_ctas, s);
  }
  switch (G) {
    case 1: return logits ? launch_impl<1, true, false>(p, map, num_ctas, s)
                          : launch_impl<1, false, false>(p, map, num_ctas, s);
    case 2: return logits ? launch_impl<2, true, false>(p, map, num_ctas, s)
                          : launch_impl<2, false, false>(p, map, num_ctas, s);
    default: return IDX_ERR_UNSUPPORTED;
  }
}

}  // namespace saib
