// Top-k consumer of the indexer logits for sm_103a.
//
// The indexer's logits feed a per-row top-k selection (index_topk = 2048 or
// 512 on the pages: aiter PR 5047, "GLM-5.2-MXFP4 E2E" and aiter issue 5477,
// Measurement); the caller's -inf outside the windows exists so that stale
// values cannot enter that selection (PR 5047, "GLM-5.2-MXFP4 E2E").  The
// pages do not define the selection itself; this library takes the plainest
// reading: row r's result is the positions of its k largest logits inside the
// row's window, ordered by value (descending) and then by position
// (ascending) -- the tie rule makes the result unique -- with -1 in the slots
// past the window length.  -0.0 and +0.0 compare equal.
//
// Design: one CTA (512 threads) per row.
//  * Keys: the f32 bit pattern mapped to an unsigned integer with the same
//    order (negative values bit-inverted, positive ones with the sign bit set).
//  * Radix select: a 4096-bin histogram of the key's top 12 bits over the
//    window (warp-aggregated shared atomics) finds the bin of the k-th
//    largest key.  If that bin and the bins above hold at most `cap` values,
//    one more pass copies them, in position order, into shared memory and the
//    remaining two levels (12 and 8 bits) and the selection run there;
//    otherwise (heavy ties) every level and the selection re-read the window.
//  * Selection: an ordered pass keeps every key above the k-th key T and the
//    first (k - #above) keys equal to T in position order (block-wide
//    prefix sums), so ties resolve to the lowest positions.
//  * The k survivors are sorted by (key desc, position asc) with a bitonic
//    sort of 64-bit composites in shared memory and written out.
// The kernel uses no global scratch memory and no atomics outside shared
// memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace fp8idx {

namespace {

constexpr int kT = kTopkThreads;
constexpr int kWarps = kT / 32;
constexpr int kPer = 8;  // consecutive elements per thread in ordered passes

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);  // -0.0 + 0.0 = +0.0: both zeros share one key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkShared {
  uint32_t* hist;      // [kTopkBins]
  uint32_t* cand_key;  // [cap]
  int32_t* cand_pos;   // [cap]
  uint64_t* sel;       // [kTopkMaxK]
  uint32_t* scan;      // [kWarps] warp totals + scratch
  uint32_t* misc;      // [8]
};

// Exclusive prefix sum over the block of one value per thread (in thread
// order); returns this thread's prefix and writes the total to *total.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < kWarps ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kWarps) warp_tot[lane] = t;  // inclusive
  }
  __syncthreads();
  const uint32_t base = warp ? warp_tot[warp - 1] : 0u;
  *total = warp_tot[kWarps - 1];
  __syncthreads();  // warp_tot is reused by the next call
  return base + x - v;
}

// Histogram with warp-aggregated shared atomics: lanes with the same bin add
// once.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool active, uint32_t bin) {
  const uint32_t mask = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const uint32_t peers = __match_any_sync(mask, bin);
  if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(hist + bin, static_cast<uint32_t>(__popc(peers)));
}

// Finds the bin b of the `need`-th largest key: above = #keys in bins > b,
// above < need <= above + hist[b].  nbins is 4096 or 256.  Result in
// misc[0] (bin), misc[1] (above).
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nbins, uint32_t need, uint32_t* warp_tot,
                                         uint32_t* misc) {
  const int per = (nbins + kT - 1) / kT;  // bins per thread, counted from the top
  const int b_hi = nbins - 1 - static_cast<int>(threadIdx.x) * per;
  uint32_t s = 0;
  for (int j = 0; j < per; ++j)
    if (b_hi - j >= 0) s += hist[b_hi - j];
  uint32_t total;
  uint32_t above = block_scan(s, warp_tot, &total);  // keys in bins above this thread's
  for (int j = 0; j < per; ++j) {
    const int b = b_hi - j;
    if (b < 0) break;
    const uint32_t h = hist[b];
    if (above < need && above + h >= need) {
      misc[0] = static_cast<uint32_t>(b);
      misc[1] = above;
    }
    above += h;
  }
  __syncthreads();
}

// Bitonic sort of n (a power of two, <= kTopkMaxK) 64-bit composites,
// descending.
__device__ __forceinline__ void bitonic_desc(uint64_t* a, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (n >> 1); i += kT) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = a[lo], y = a[hi];
        if ((x < y) == desc) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int32_t pos) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~pos);
}

}  // namespace

__global__ void __launch_bounds__(kTopkThreads, 1) topk_rows_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const TopkLayout Lo = topk_smem_layout(p.cap);
  TopkShared sh;
  sh.hist = reinterpret_cast<uint32_t*>(smem_raw + Lo.hist);
  sh.cand_key = reinterpret_cast<uint32_t*>(smem_raw + Lo.cand_key);
  sh.cand_pos = reinterpret_cast<int32_t*>(smem_raw + Lo.cand_pos);
  sh.sel = reinterpret_cast<uint64_t*>(smem_raw + Lo.sel);
  sh.scan = reinterpret_cast<uint32_t*>(smem_raw + Lo.scan);
  sh.misc = reinterpret_cast<uint32_t*>(smem_raw + Lo.misc);

  const int64_t r = blockIdx.x;
  // The row's window [lo, hi).
  int64_t lo = 0, hi = 0;
  if (p.mode == 0) {
    const int32_t ks = __ldg(p.ks + r), ke = __ldg(p.ke + r);
    lo = ks < 0 ? 0 : ks;
    hi = ke > p.cols ? p.cols : ke;
  } else {
    const int64_t b = r / p.next_n, n = r - b * p.next_n;
    int64_t ctx = __ldg(p.context_lens + b);
    if (ctx < 0) ctx = 0;
    hi = ctx - p.next_n + n + 1;
    if (hi > p.cols) hi = p.cols;
  }
  if (hi < lo) hi = lo;
  const int64_t L = hi - lo;
  const float* row = p.logits + r * p.stride + lo;
  int32_t* out_row = p.out + r * p.out_stride;
  const int k = p.k;
  const int tid = threadIdx.x;

  // Windows of at most k values: all of them, sorted.
  if (L <= k) {
    int n = 1;
    while (n < L) n <<= 1;
    for (int i = tid; i < n; i += kT)
      sh.sel[i] = i < L ? composite(order_key(__ldg(row + i)), static_cast<int32_t>(lo + i)) : 0ull;
    __syncthreads();
    bitonic_desc(sh.sel, n);
    for (int j = tid; j < k; j += kT)
      out_row[j] = j < L ? static_cast<int32_t>(~static_cast<uint32_t>(sh.sel[j])) : -1;
    return;
  }

  // Level 0: top 12 bits over the window.
  for (int i = tid; i < kTopkBins; i += kT) sh.hist[i] = 0u;
  __syncthreads();
  for (int64_t i0 = 0; i0 < L; i0 += kT) {
    const int64_t i = i0 + tid;
    const bool act = i < L;
    const uint32_t key = act ? order_key(__ldg(row + i)) : 0u;
    hist_add(sh.hist, act, key >> 20);
  }
  __syncthreads();
  find_bin(sh.hist, kTopkBins, static_cast<uint32_t>(k), sh.scan, sh.misc);
  const uint32_t b0 = sh.misc[0];
  const uint32_t above0 = sh.misc[1];
  const uint32_t n_cand = above0 + sh.hist[b0];
  const bool in_smem = n_cand <= static_cast<uint32_t>(p.cap);
  __syncthreads();

  // Fast path: the candidates (top-12-bit bin >= b0), in position order.
  if (in_smem) {
    uint32_t written = 0;
    for (int64_t c0 = 0; c0 < L; c0 += static_cast<int64_t>(kT) * kPer) {
      const int64_t i0 = c0 + static_cast<int64_t>(tid) * kPer;
      uint32_t keys[kPer];
      uint32_t cnt = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        keys[j] = (i0 + j < L) ? order_key(__ldg(row + i0 + j)) : 0u;
        cnt += (i0 + j < L && (keys[j] >> 20) >= b0) ? 1u : 0u;
      }
      uint32_t total;
      uint32_t slot = written + block_scan(cnt, sh.scan, &total);
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (i0 + j < L && (keys[j] >> 20) >= b0) {
          sh.cand_key[slot] = keys[j];
          sh.cand_pos[slot] = static_cast<int32_t>(lo + i0 + j);
          ++slot;
        }
      written += total;
    }
    __syncthreads();
  }

  // Source of levels 1-2 and of the selection: the candidates or the window.
  const int64_t n_src = in_smem ? static_cast<int64_t>(n_cand) : L;
  const auto key_at = [&](int64_t i) -> uint32_t { return in_smem ? sh.cand_key[i] : order_key(__ldg(row + i)); };
  const auto pos_at = [&](int64_t i) -> int32_t {
    return in_smem ? sh.cand_pos[i] : static_cast<int32_t>(lo + i);
  };

  // Level 1: bits 19..8 among keys in bin b0.
  for (int i = tid; i < kTopkBins; i += kT) sh.hist[i] = 0u;
  __syncthreads();
  for (int64_t i0 = 0; i0 < n_src; i0 += kT) {
    const int64_t i = i0 + tid;
    const uint32_t key = i < n_src ? key_at(i) : 0u;
    hist_add(sh.hist, i < n_src && (key >> 20) == b0, (key >> 8) & 0xFFFu);
  }
  __syncthreads();
  find_bin(sh.hist, kTopkBins, static_cast<uint32_t>(k) - above0, sh.scan, sh.misc);
  const uint32_t b1 = sh.misc[0];
  const uint32_t above1 = above0 + sh.misc[1];
  const uint32_t pre24 = (b0 << 12) | b1;
  __syncthreads();

  // Level 2: bits 7..0 among keys with the 24-bit prefix.
  for (int i = tid; i < 256; i += kT) sh.hist[i] = 0u;
  __syncthreads();
  for (int64_t i0 = 0; i0 < n_src; i0 += kT) {
    const int64_t i = i0 + tid;
    const uint32_t key = i < n_src ? key_at(i) : 0u;
    hist_add(sh.hist, i < n_src && (key >> 8) == pre24, key & 0xFFu);
  }
  __syncthreads();
  find_bin(sh.hist, 256, static_cast<uint32_t>(k) - above1, sh.scan, sh.misc);
  const uint32_t T = (pre24 << 8) | sh.misc[0];
  const uint32_t above = above1 + sh.misc[1];  // keys > T
  const uint32_t need_eq = static_cast<uint32_t>(k) - above;
  __syncthreads();

  // Selection in position order: every key > T, the first need_eq keys == T.
  uint32_t gt_done = 0, eq_done = 0;
  for (int64_t c0 = 0; c0 < n_src; c0 += static_cast<int64_t>(kT) * kPer) {
    const int64_t i0 = c0 + static_cast<int64_t>(tid) * kPer;
    uint32_t keys[kPer];
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      keys[j] = (i0 + j < n_src) ? key_at(i0 + j) : 0u;
      n_gt += (i0 + j < n_src && keys[j] > T) ? 1u : 0u;
      n_eq += (i0 + j < n_src && keys[j] == T) ? 1u : 0u;
    }
    uint32_t tot;
    const uint32_t packed = block_scan((n_gt << 16) | n_eq, sh.scan, &tot);  // chunk counts < 2^16
    uint32_t gt_before = gt_done + (packed >> 16), eq_before = eq_done + (packed & 0xFFFFu);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (i0 + j >= n_src) break;
      if (keys[j] > T) {
        sh.sel[gt_before + (eq_before < need_eq ? eq_before : need_eq)] = composite(keys[j], pos_at(i0 + j));
        ++gt_before;
      } else if (keys[j] == T) {
        if (eq_before < need_eq) sh.sel[gt_before + eq_before] = composite(keys[j], pos_at(i0 + j));
        ++eq_before;
      }
    }
    gt_done += tot >> 16;
    eq_done += tot & 0xFFFFu;
  }
  __syncthreads();

  int n = 1;
  while (n < k) n <<= 1;
  for (int i = k + tid; i < n; i += kT) sh.sel[i] = 0ull;
  __syncthreads();
  bitonic_desc(sh.sel, n);
  for (int j = tid; j < k; j += kT) out_row[j] = static_cast<int32_t>(~static_cast<uint32_t>(sh.sel[j]));
}

cudaError_t launch_topk(const TopkParams& p, int smem_bytes, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<p.rows, kTopkThreads, smem_bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fp8idx
