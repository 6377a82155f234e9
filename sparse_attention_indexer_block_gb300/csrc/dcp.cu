// Key-sharded (decode context parallel) decode: a sequence's keys are dealt
// to W ranks in runs of I tokens (INDEXER page,
// _build_prefill_chunk_metadata_kernel, DCP branch). Each rank scores and
// selects over the keys it holds (the decode path in values mode, on its
// local cache and local key counts); its candidates, in global token
// positions, are merged here into the row's top k.
#include <atomic>

#include "internal.h"

namespace saib {

namespace {

constexpr int kMapThreads = 256;
constexpr int kMergeThreads = 1024;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeCap = IDX_DCP_MAX_CANDIDATES;  // candidates of a row in shared memory

__global__ void __launch_bounds__(kMapThreads) key_counts_kernel(const int32_t* lens, int64_t n,
                                                                 int ratio, int rank, int world,
                                                                 int interleave, int32_t* out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kMapThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kMapThreads + threadIdx.x; i < n;
       i += stride)
    out[i] = static_cast<int32_t>(index_key_count(lens[i], ratio, rank, world, interleave));
}

// Rank-local key j is global token (j / I) * I * W + rank * I + j % I: its
// (j / I)-th run comes after that many full rounds of W runs and `rank` runs
// of the current round. Negative (empty) entries stay as they are.
__global__ void __launch_bounds__(kMapThreads) dcp_globalise_kernel(int32_t* idx, int64_t n,
                                                                    int rank, int world,
                                                                    int interleave) {
  pdl_trigger();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kMapThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kMapThreads + threadIdx.x; i < n;
       i += stride) {
    const int32_t j = idx[i];
    if (j < 0) continue;
    const int64_t run = j / interleave;
    idx[i] = static_cast<int32_t>(run * interleave * world +
                                  static_cast<int64_t>(rank) * interleave + (j - run * interleave));
  }
}

struct MergeShared {
  uint32_t hist[256];
  int warp_sum[kMergeWarps];
  int valid;
  int nout;
  int ntie;
  int bin;
  int above;
};

// Adds 1 to hist[d] for every lane with `in` set, one atomic per distinct
// digit of the warp. All lanes of the warp.
__device__ __forceinline__ void warp_hist_add(uint32_t* hist, bool in, uint32_t d) {
  const unsigned act = __ballot_sync(0xffffffffu, in);
  if (!in) return;
  const unsigned same = __match_any_sync(act, d);
  if ((threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[d], __popc(same));
}

// One CTA per row: the top k of the row's world * k candidates (slab w of
// val / idx is rank w's [rows, k] output; idx < 0 = empty). Radix select
// over the order-preserving keys, 8 bits per pass from the top; keys equal
// in all 32 bits at the cut take tickets (which of them is arbitrary).
__global__ void __launch_bounds__(kMergeThreads, 1)
    dcp_merge_kernel(const float* __restrict__ val, const int32_t* __restrict__ idx, int world,
                     int64_t rows, int K, int32_t* __restrict__ out_idx,
                     float* __restrict__ out_val) {
  extern __shared__ uint32_t merge_smem[];
  __shared__ MergeShared sh;
  pdl_trigger();
  pdl_wait();
  const int n = world * K;
  uint32_t* skey = merge_smem;
  int32_t* sidx = reinterpret_cast<int32_t*>(merge_smem + n);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t row = blockIdx.x;
  int32_t* out = out_idx + row * K;
  float* ov = out_val ? out_val + row * K : nullptr;
  if (t == 0) {
    sh.nout = 0;
    sh.ntie = 0;
  }
  int mine = 0;
  for (int c = t; c < n; c += kMergeThreads) {
    const int w = c / K, i = c - w * K;
    const int64_t off = (static_cast<int64_t>(w) * rows + row) * K + i;
    const int32_t x = idx[off];
    sidx[c] = x;
    skey[c] = x >= 0 ? float_key(val[off]) : 0u;
    mine += x >= 0 ? 1 : 0;
  }
  for (int o = 16; o; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) sh.warp_sum[warp] = mine;
  __syncthreads();
  if (t == 0) {
    int v = 0;
    for (int w = 0; w < kMergeWarps; ++w) v += sh.warp_sum[w];
    sh.valid = v;
  }
  __syncthreads();
  const int valid = sh.valid;
  if (valid <= K) {  // every candidate is in
    for (int c = t; c < n; c += kMergeThreads) {
      if (sidx[c] < 0) continue;
      const int pos = atomicAdd(&sh.nout, 1);
      out[pos] = sidx[c];
      if (ov) ov[pos] = key_float(skey[c]);
    }
    for (int e = valid + t; e < K; e += kMergeThreads) {
      out[e] = -1;
      if (ov) ov[e] = -INFINITY;
    }
    return;
  }
  uint32_t prefix = 0u, pmask = 0u;
  int need = K;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = t; b < 256; b += kMergeThreads) sh.hist[b] = 0u;
    __syncthreads();
    for (int c0 = 0; c0 < n; c0 += kMergeThreads) {
      const int c = c0 + t;
      const bool in = c < n && sidx[c] >= 0 && (skey[c] & pmask) == prefix;
      warp_hist_add(sh.hist, in, in ? (skey[c] >> shift) & 255u : 0u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255 - 8l - j, j = 0..7 (top down)
      int cnt[8], local = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = static_cast<int>(sh.hist[255 - 8 * lane - j]);
        local += cnt[j];
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int ex = incl - local;
      if (ex < need && need <= incl) {
        int acc = ex;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + cnt[j] >= need) {
            sh.bin = 255 - 8 * lane - j;
            sh.above = acc;
            break;
          }
          acc += cnt[j];
        }
      }
    }
    __syncthreads();
    const uint32_t b = static_cast<uint32_t>(sh.bin);
    const int above = sh.above;
    for (int c = t; c < n; c += kMergeThreads) {
      if (sidx[c] < 0 || (skey[c] & pmask) != prefix || ((skey[c] >> shift) & 255u) <= b)
        continue;
      const int pos = atomicAdd(&sh.nout, 1);
      out[pos] = sidx[c];
      if (ov) ov[pos] = key_float(skey[c]);
    }
    need -= above;
    prefix |= b << shift;
    pmask |= 255u << shift;
    __syncthreads();
  }
  // keys equal to the k-th in all 32 bits: `need` of them complete the row
  const int base = sh.nout;
  for (int c = t; c < n; c += kMergeThreads) {
    if (sidx[c] < 0 || skey[c] != prefix) continue;
    const int tk = atomicAdd(&sh.ntie, 1);
    if (tk < need) {
      out[base + tk] = sidx[c];
      if (ov) ov[base + tk] = key_float(skey[c]);
    }
  }
}

unsigned map_grid(int64_t n) {
  const int64_t g = (n + kMapThreads - 1) / kMapThreads;
  const int64_t cap = 8 * static_cast<int64_t>(device_sm_count());
  return static_cast<unsigned>(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

idx_status launch_key_counts(const int32_t* lens, int64_t n, int ratio, int rank, int world,
                             int interleave, int32_t* out, cudaStream_t s) {
  if (n <= 0) return IDX_OK;
  key_counts_kernel<<<map_grid(n), kMapThreads, 0, s>>>(lens, n, ratio, rank, world, interleave,
                                                        out);
  return cuda_status(cudaGetLastError());
}

idx_status launch_dcp_globalise(int32_t* idx, int64_t n, int rank, int world, int interleave,
                                cudaStream_t s) {
  if (n <= 0) return IDX_OK;
  return cuda_status(launch_pdl(dcp_globalise_kernel, map_grid(n), kMapThreads, 0, s, idx, n,
                                rank, world, interleave));
}

idx_status launch_dcp_merge(const float* val, const int32_t* idx, int world, int64_t rows,
                            int topk, int32_t* out_idx, float* out_val, cudaStream_t s) {
  if (rows <= 0) return IDX_OK;
  if (static_cast<int64_t>(world) * topk > kMergeCap) return IDX_ERR_UNSUPPORTED;
  const size_t smem = static_cast<size_t>(world) * topk * 8;
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidDevice);
  if (dev >= kMaxDevices || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(dcp_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMergeCap * 8);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < kMaxDevices) configured[dev].store(true, std::memory_order_release);
  }
  return cuda_status(launch_pdl(dcp_merge_kernel, static_cast<unsigned>(rows), kMergeThreads, smem,
                                s, val, idx, world, rows, topk, out_idx, out_val));
}

}  // namespace saib
