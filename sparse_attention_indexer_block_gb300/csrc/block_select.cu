// Block and pool selection over rows of indexer logits: the MiniMax runner's
// topk_blocks / init_blocks / local_blocks and GLM5's pool_topk followed by
// expand_pools_and_append_tail (the pages name them; the rules are the
// readings stated in include/indexer.h). The logits come from the decode
// logits call (one pass over the keys); these kernels read 4 bytes per key.
#include <atomic>

#include "internal.h"

namespace saib {

namespace {

constexpr int kBlkThreads = 512;
constexpr int kBlkWarps = kBlkThreads / 32;
constexpr int kBlkCap = 16384;  // blocks of one row held in shared memory
constexpr int kBlkPerThread = kBlkCap / kBlkThreads;

struct BlkShared {
  uint32_t hist[256];
  int warp_sum[kBlkWarps];
  int bin, above, ntie, forced;
};

// Adds 1 to hist[d] for every lane with `in` set, one atomic per distinct
// digit of the warp. All lanes of the warp.
__device__ __forceinline__ void blk_hist_add(uint32_t* hist, bool in, uint32_t d) {
  const unsigned act = __ballot_sync(0xffffffffu, in);
  if (!in) return;
  const unsigned same = __match_any_sync(act, d);
  if ((threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[d], __popc(same));
}

// Sum of one int per thread over the CTA (two barriers).
__device__ __forceinline__ int blk_sum(int v, BlkShared* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) sh->warp_sum[warp] = v;
  __syncthreads();
  int total = 0;
  for (int w = 0; w < kBlkWarps; ++w) total += sh->warp_sum[w];
  return total;
}

// Exclusive scan of one int per thread in thread order, and the total.
__device__ __forceinline__ int blk_scan(int v, int* total, BlkShared* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sh->warp_sum[warp] = x;
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < kBlkWarps; ++w) {
    if (w < warp) before += sh->warp_sum[w];
    all += sh->warp_sum[w];
  }
  *total = all;
  return before + x - v;
}

// One CTA per row: block maxima (coalesced float4 reads folded into block
// keys when blocks are whole float4s, else a warp per block), the forced
// first n_init and last n_local blocks, the k best of the others by an 8-bit
// radix select over order-preserving keys (equal keys at the cut: any of
// them), then the selected blocks in ascending order.
__global__ void __launch_bounds__(kBlkThreads) block_topk_kernel(
    const float* __restrict__ logits, int64_t ld, const int32_t* __restrict__ row_lens, int B,
    int k, int n_init, int n_local, int32_t* __restrict__ out, int cap,
    int32_t* __restrict__ counts, int nb_max) {
  extern __shared__ uint32_t blk_smem[];
  uint32_t* key = blk_smem;                                   // [nb_max]
  uint8_t* sel = reinterpret_cast<uint8_t*>(blk_smem + nb_max);  // 0 ranked, 1 selected, 2 forced
  __shared__ BlkShared sh;
  pdl_trigger();
  pdl_wait();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t row = blockIdx.x;
  const int64_t L = min(max(static_cast<int64_t>(row_lens[row]), int64_t{0}), ld);
  const int nb = static_cast<int>((L + B - 1) / B);  // <= nb_max <= kBlkCap (L <= ld)
  const float* lg = logits + row * ld;
  if ((B & 3) == 0 && (ld & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
    // blocks of whole float4s: coalesced 16-byte reads, four per thread in
    // flight, each folded into its block's key (keys start at the minimum)
    for (int b = t; b < nb; b += kBlkThreads) key[b] = 0u;
    __syncthreads();
    const float4* lg4 = reinterpret_cast<const float4*>(lg);
    const int64_t n4 = (L + 3) / 4;
    for (int64_t i0 = t; i0 < n4; i0 += 4 * kBlkThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + u * kBlkThreads;
        if (i < n4) v[u] = lg4[i];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + u * kBlkThreads;
        if (i >= n4) continue;
        const int64_t x = 4 * i;  // tokens x .. x + 3 (those < L count)
        float m = v[u].x;
        if (x + 1 < L) m = fmaxf(m, v[u].y);
        if (x + 2 < L) m = fmaxf(m, v[u].z);
        if (x + 3 < L) m = fmaxf(m, v[u].w);
        atomicMax(&key[x / B], float_key(m));
      }
    }
    __syncthreads();
    for (int b = t; b < nb; b += kBlkThreads) sel[b] = (b < n_init || b >= nb - n_local) ? 2 : 0;
  } else {
    for (int b = warp; b < nb; b += kBlkWarps) {
      float m = -INFINITY;
      const int64_t end = min(L, static_cast<int64_t>(b) * B + B);
      for (int64_t i = static_cast<int64_t>(b) * B + lane; i < end; i += 32) m = fmaxf(m, lg[i]);
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) {
        key[b] = float_key(m);
        sel[b] = (b < n_init || b >= nb - n_local) ? 2 : 0;
      }
    }
  }
  __syncthreads();
  int mine = 0;
  for (int b = t; b < nb; b += kBlkThreads) mine += sel[b] == 2 ? 1 : 0;
  const int forced = blk_sum(mine, &sh);
  const int ranked = nb - forced;
  int need = min(k, ranked);
  if (need >= ranked) {
    for (int b = t; b < nb; b += kBlkThreads)
      if (sel[b] == 0) sel[b] = 1;
  } else if (need > 0) {
    uint32_t prefix = 0u, pmask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = t; b < 256; b += kBlkThreads) sh.hist[b] = 0u;
      __syncthreads();
      for (int b0 = 0; b0 < nb; b0 += kBlkThreads) {
        const int b = b0 + t;
        const bool in = b < nb && sel[b] == 0 && (key[b] & pmask) == prefix;
        blk_hist_add(sh.hist, in, in ? (key[b] >> shift) & 255u : 0u);
      }
      __syncthreads();
      if (warp == 0) {
        int cnt[8], local = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          cnt[i] = static_cast<int>(sh.hist[255 - 8 * lane - i]);
          local += cnt[i];
        }
        int incl = local;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int ex = incl - local;
        if (ex < need && need <= incl) {
          int acc = ex;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (acc + cnt[i] >= need) {
              sh.bin = 255 - 8 * lane - i;
              sh.above = acc;
              break;
            }
            acc += cnt[i];
          }
        }
        if (lane == 0) sh.ntie = 0;
      }
      __syncthreads();
      const uint32_t bin = static_cast<uint32_t>(sh.bin);
      for (int b = t; b < nb; b += kBlkThreads)
        if (sel[b] == 0 && (key[b] & pmask) == prefix && ((key[b] >> shift) & 255u) > bin)
          sel[b] = 1;
      need -= sh.above;
      prefix |= bin << shift;
      pmask |= 255u << shift;
      __syncthreads();
    }
    // keys equal to the k-th in all 32 bits: `need` of them
    for (int b = t; b < nb; b += kBlkThreads)
      if (sel[b] == 0 && key[b] == prefix && atomicAdd(&sh.ntie, 1) < need) sel[b] = 1;
  }
  __syncthreads();
  // the selected blocks in ascending order: thread t scans blocks
  // [t * kBlkPerThread, (t + 1) * kBlkPerThread)
  const int lo = t * kBlkPerThread, hi = min(nb, lo + kBlkPerThread);
  int cnt = 0;
  for (int b = lo; b < hi; ++b) cnt += sel[b] ? 1 : 0;
  int total;
  int pos = blk_scan(cnt, &total, &sh);
  int32_t* o = out + row * cap;
  for (int b = lo; b < hi; ++b)
    if (sel[b] && pos < cap) o[pos++] = b;
  for (int i = total + t; i < cap; i += kBlkThreads) o[i] = -1;
  if (t == 0 && counts) counts[row] = min(total, cap);
}

// One CTA per row: the tokens of the listed complete pools (pool b covers
// [b P, b P + P); -1 entries and pools past the row's last complete pool add
// nothing), in list order, then the row's tail [floor(L / P) P, L).
__global__ void __launch_bounds__(kBlkThreads) expand_pools_kernel(
    const int32_t* __restrict__ pools, int pcap, const int32_t* __restrict__ pcounts,
    const int32_t* __restrict__ row_lens, int P, int32_t* __restrict__ out, int cap,
    int32_t* __restrict__ counts) {
  __shared__ BlkShared sh;
  pdl_trigger();
  pdl_wait();
  const int t = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int64_t L = max(static_cast<int64_t>(row_lens[row]), int64_t{0});
  const int64_t full = L / P;
  const int np = pcounts ? min(max(pcounts[row], 0), pcap) : pcap;
  const int32_t* pl = pools + row * pcap;
  int32_t* o = out + row * cap;
  int written = 0;  // tokens before this chunk of the list
  for (int base = 0; base < np; base += kBlkThreads) {
    const int i = base + t;
    const int32_t b = i < np ? pl[i] : -1;
    const bool ok = b >= 0 && b < full;
    int total;
    const int pos = written + blk_scan(ok ? P : 0, &total, &sh);
    if (ok)
      for (int j = 0; j < P && pos + j < cap; ++j) o[pos + j] = static_cast<int32_t>(b * P + j);
    written += total;
  }
  const int64_t tail = L - full * P;
  for (int64_t j = t; j < tail; j += kBlkThreads)
    if (written + j < cap) o[written + j] = static_cast<int32_t>(full * P + j);
  const int n = static_cast<int>(min(static_cast<int64_t>(written) + tail, static_cast<int64_t>(cap)));
  for (int i = n + t; i < cap; i += kBlkThreads) o[i] = -1;
  if (t == 0 && counts) counts[row] = n;
}

}  // namespace

}  // namespace saib

using namespace saib;

extern "C" {

idx_status indexer_block_topk(const float* logits, int64_t ld_logits, const int32_t* row_lens,
                              int64_t num_rows, int32_t block_size, int32_t topk_blocks,
                              int32_t init_blocks, int32_t local_blocks, int32_t* out_blocks,
                              int32_t out_cap, int32_t* out_counts, void* stream) {
  if (num_rows < 0 || block_size < 1 || topk_blocks < 0 || init_blocks < 0 || local_blocks < 0 ||
      out_cap < 1 || ld_logits < 0)
    return IDX_ERR_INVALID_ARG;
  const int64_t nb_max = (ld_logits + block_size - 1) / block_size;
  if (nb_max > kBlkCap) return IDX_ERR_UNSUPPORTED;
  if (num_rows == 0) return IDX_OK;
  if (!logits || !row_lens || !out_blocks) return IDX_ERR_INVALID_ARG;
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidDevice);
  if (dev >= kMaxDevices || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(block_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBlkCap * 5);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < kMaxDevices) configured[dev].store(true, std::memory_order_release);
  }
  const size_t smem = static_cast<size_t>(nb_max) * 5;
  return cuda_status(launch_pdl(block_topk_kernel, static_cast<unsigned>(num_rows), kBlkThreads,
                                smem, static_cast<cudaStream_t>(stream), logits, ld_logits,
                                row_lens, block_size, topk_blocks, init_blocks, local_blocks,
                                out_blocks, out_cap, out_counts, static_cast<int>(nb_max)));
}

idx_status indexer_expand_pools(const int32_t* pools, int32_t pools_cap, const int32_t* pool_counts,
                                const int32_t* row_lens, int64_t num_rows, int32_t pool_size,
                                int32_t* out_idx, int32_t out_cap, int32_t* out_counts,
                                void* stream) {
  if (num_rows < 0 || pools_cap < 0 || pool_size < 1 || out_cap < 1) return IDX_ERR_INVALID_ARG;
  if (num_rows == 0) return IDX_OK;
  if ((pools_cap > 0 && !pools) || !row_lens || !out_idx) return IDX_ERR_INVALID_ARG;
  return cuda_status(launch_pdl(expand_pools_kernel, static_cast<unsigned>(num_rows), kBlkThreads,
                                0, static_cast<cudaStream_t>(stream), pools, pools_cap,
                                pool_counts, row_lens, pool_size, out_idx, out_cap, out_counts));
}

}  // extern "C"
