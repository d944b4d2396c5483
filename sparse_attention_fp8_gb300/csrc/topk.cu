// Top-k consumer of the indexer logits for sm_103a.
//
// The indexer's logits feed a per-row top-k selection (index_topk = 2048 or
// 512 on the pages: aiter PR 5047, "GLM-5.2-MXFP4 E2E" and aiter issue 5477,
// Measurement); the caller's -inf outside the windows exists so that stale
// values cannot enter that selection (PR 5047, "GLM-5.2-MXFP4 E2E").  The
// pages do not define the selection itself; this library takes the plainest
// reading: row r's result is the positions of its k largest logits inside the
// row's window, equal logits taken from the lowest positions first (which
// makes the set unique; -0.0 and +0.0 compare equal), listed in ascending
// position order, with -1 in the slots past the window length.
//
// Design: one CTA (512 threads) per row, two CTAs per SM.
//  * Keys: the f32 bit pattern mapped to an unsigned integer with the same
//    order (negative values bit-inverted, positive ones with the sign bit set).
//  * The window is read as aligned float4 groups (scalar loads for the
//    partial groups at its ends), several groups in flight per thread.
//  * Radix select of the k-th largest key T: three levels of histograms
//    (12, 12, 8 bits of the key; plain shared atomics).  A window of at most
//    `cap` values is copied into shared memory once and selected there.  A
//    longer one is sampled with a stride S (at most cap samples); the
//    sample's (2k/S + 32)-th largest key is a lower threshold, and one
//    ordered pass over the window keeps the values above it (about 2k + 32S
//    of them) in shared memory for the exact select.  If that count falls
//    outside [k, cap] (adversarial or heavily tied rows), the levels and the
//    selection re-read the window instead.
//  * Selection: an ordered pass keeps every key above the k-th key T and the
//    first (k - #above) keys equal to T in position order (block-wide
//    prefix sums), so ties resolve to the lowest positions, and writes the
//    kept positions straight to the output in position order.
// The kernel uses no global scratch memory and no atomics outside shared
// memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace fp8idx {

namespace {

constexpr int kT = kTopkThreads;
constexpr int kWarps = kT / 32;
constexpr int kPer = 8;  // elements per thread per chunk of an ordered pass

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);  // -0.0 + 0.0 = +0.0: both zeros share one key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkShared {
  uint32_t* hist;      // [kTopkBins]
  uint32_t* cand_key;  // [cap]
  int32_t* cand_pos;   // [cap]
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

// One histogram count (a plain shared atomic: measured twice as fast here as
// aggregating equal bins within the warp first).
__device__ __forceinline__ void hist_add(uint32_t* hist, bool active, uint32_t bin) {
  if (active) atomicAdd(hist + bin, 1u);
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

}  // namespace

__global__ void __launch_bounds__(kTopkThreads, 2) topk_rows_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const TopkLayout Lo = topk_smem_layout(p.cap);
  TopkShared sh;
  sh.hist = reinterpret_cast<uint32_t*>(smem_raw + Lo.hist);
  sh.cand_key = reinterpret_cast<uint32_t*>(smem_raw + Lo.cand_key);
  sh.cand_pos = reinterpret_cast<int32_t*>(smem_raw + Lo.cand_pos);
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
  int32_t* out_row = p.out + r * p.out_stride;
  const int k = p.k;
  const int tid = threadIdx.x;

  // Windows of at most k values: all of their positions.
  if (L <= k) {
    for (int j = tid; j < k; j += kT) out_row[j] = j < L ? static_cast<int32_t>(lo + j) : -1;
    return;
  }

  // The window is read in groups of 4 positions: one float4 load for a
  // group inside the window when the rows are 16-byte aligned, scalar loads
  // for the (at most two) partial groups at its ends -- nothing outside
  // [lo, hi) is read.
  const float* row_base = p.logits + r * p.stride;
  const bool vec = p.vec_ok != 0;
  const int64_t gstart = vec ? (lo & ~static_cast<int64_t>(3)) : lo;
  const int64_t ngroups = (hi - gstart + 3) / 4;
  const auto load_group = [&](int64_t gi, uint32_t (&key)[4]) -> uint32_t {  // returns the valid-lane mask
    const int64_t g = gstart + 4 * gi;
    if (gi >= ngroups) return 0u;
    if (vec && g >= lo && g + 4 <= hi) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row_base + g));
      key[0] = order_key(f.x);
      key[1] = order_key(f.y);
      key[2] = order_key(f.z);
      key[3] = order_key(f.w);
      return 0xFu;
    }
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool in = g + e >= lo && g + e < hi;
      key[e] = in ? order_key(__ldg(row_base + g + e)) : 0u;
      m |= in ? (1u << e) : 0u;
    }
    return m;
  };
  constexpr int kU = 4;  // groups in flight per thread in the histogram passes
  // Histogram over the window of `bin(key)` for keys with `sel(key)`.
  const auto window_hist = [&](auto sel, auto bin) {
    for (int64_t q0 = 0; q0 < ngroups; q0 += static_cast<int64_t>(kT) * kU) {
      uint32_t key[kU][4], m[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) m[u] = load_group(q0 + u * kT + tid, key[u]);
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) hist_add(sh.hist, ((m[u] >> e) & 1u) && sel(key[u][e]), bin(key[u][e]));
    }
  };
  // Ordered pass over the window with vector loads: `f(keys, pos0, valid)`
  // gets this thread's kPer consecutive positions of each chunk (chunks in
  // position order, threads in position order within a chunk).
  const auto window_ordered = [&](auto f) {
    for (int64_t q0 = 0; q0 < ngroups; q0 += static_cast<int64_t>(kT) * (kPer / 4)) {
      uint32_t keys[kPer], valid = 0;
      const int64_t pos0 = gstart + 4 * (q0 + static_cast<int64_t>(tid) * (kPer / 4));
#pragma unroll
      for (int h = 0; h < kPer / 4; ++h) {
        uint32_t k4[4];
        const uint32_t m = load_group(q0 + static_cast<int64_t>(tid) * (kPer / 4) + h, k4);
#pragma unroll
        for (int e = 0; e < 4; ++e) keys[4 * h + e] = k4[e];
        valid |= m << (4 * h);
      }
      f(keys, pos0, valid);
    }
  };

  // ---- sources: the window in global memory, or candidates in shared memory
  const auto smem_hist = [&](int64_t n_c, auto sel, auto bin) {
    for (int64_t i0 = 0; i0 < n_c; i0 += kT) {
      const int64_t i = i0 + tid;
      const uint32_t key = i < n_c ? sh.cand_key[i] : 0u;
      hist_add(sh.hist, i < n_c && sel(key), bin(key));
    }
  };
  // Ordered passes: element e of a source is (key, position); a chunk is
  // kT*kPer elements, warp w takes the chunk's w-th run of 32*kPer, step j
  // of the run one element per lane (consecutive lanes, consecutive
  // elements: coalesced in global memory, conflict-free in shared memory).
  // `keep(key)` returns 0 (drop) or the predicate bits; `place` gets the
  // element's key, position and its rank among the kept elements before it
  // in position order.  Counts per chunk go through one 16-entry scan of
  // warp totals (double-buffered, one barrier per chunk).
  const auto smem_get = [&](int64_t e, uint32_t& key, int32_t& pos) {
    key = sh.cand_key[e];
    pos = sh.cand_pos[e];
  };
  const auto global_get = [&](int64_t e, uint32_t& key, int32_t& pos) {
    key = order_key(__ldg(row_base + lo + e));
    pos = static_cast<int32_t>(lo + e);
  };
  // Two independent counts per element (packed 16:16 per chunk: a chunk has
  // kT*kPer < 2^16 elements): a = #(pred A) before it, b = #(pred B) before
  // it.  Returns the total of pred A.
  const auto ordered2 = [&](int64_t n, auto get, auto pred_a, auto pred_b, auto place) {
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t done_a = 0, done_b = 0;
    int parity = 0;
    for (int64_t c0 = 0; c0 < n; c0 += static_cast<int64_t>(kT) * kPer) {
      const int64_t wbase = c0 + static_cast<int64_t>(warp) * 32 * kPer;
      uint32_t keys[kPer], ba[kPer], bb[kPer];
      int32_t pos[kPer];
      uint32_t wa = 0, wb = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int64_t e = wbase + j * 32 + lane;
        const bool in = e < n;
        keys[j] = 0u;
        pos[j] = 0;
        if (in) get(e, keys[j], pos[j]);
        ba[j] = __ballot_sync(0xffffffffu, in && pred_a(keys[j]));
        bb[j] = __ballot_sync(0xffffffffu, in && pred_b(keys[j]));
        wa += __popc(ba[j]);
        wb += __popc(bb[j]);
      }
      uint32_t* tot = sh.scan + parity * kWarps;
      if (lane == 0) tot[warp] = (wa << 16) | wb;
      __syncthreads();
      uint32_t before = 0, all = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = tot[w];
        before += w < warp ? t : 0u;
        all += t;
      }
      uint32_t ra = done_a + (before >> 16), rb = done_b + (before & 0xFFFFu);
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const uint32_t a = ra + __popc(ba[j] & lt), b = rb + __popc(bb[j] & lt);
        const bool in_a = (ba[j] >> lane) & 1u, in_b = (bb[j] >> lane) & 1u;
        if (in_a || in_b) place(keys[j], pos[j], in_a, in_b, a, b);
        ra += __popc(ba[j]);
        rb += __popc(bb[j]);
      }
      done_a += all >> 16;
      done_b += all & 0xFFFFu;
      parity ^= 1;
    }
    __syncthreads();
    return done_a;
  };

  // ---- the `need`-th largest key T of a source and #keys > T, three radix
  // levels (12, 12 and 8 bits of the key)
  const auto radix_select = [&](auto hist_pass, uint32_t need, uint32_t* T_out, uint32_t* above_out) {
    for (int i = tid; i < kTopkBins; i += kT) sh.hist[i] = 0u;
    __syncthreads();
    hist_pass([](uint32_t) { return true; }, [](uint32_t key) { return key >> 20; });
    __syncthreads();
    find_bin(sh.hist, kTopkBins, need, sh.scan, sh.misc);
    const uint32_t b0 = sh.misc[0], a0 = sh.misc[1];
    __syncthreads();
    for (int i = tid; i < kTopkBins; i += kT) sh.hist[i] = 0u;
    __syncthreads();
    hist_pass([&](uint32_t key) { return (key >> 20) == b0; }, [](uint32_t key) { return (key >> 8) & 0xFFFu; });
    __syncthreads();
    find_bin(sh.hist, kTopkBins, need - a0, sh.scan, sh.misc);
    const uint32_t pre24 = (b0 << 12) | sh.misc[0], a1 = a0 + sh.misc[1];
    __syncthreads();
    for (int i = tid; i < 256; i += kT) sh.hist[i] = 0u;
    __syncthreads();
    hist_pass([&](uint32_t key) { return (key >> 8) == pre24; }, [](uint32_t key) { return key & 0xFFu; });
    __syncthreads();
    find_bin(sh.hist, 256, need - a1, sh.scan, sh.misc);
    *T_out = (pre24 << 8) | sh.misc[0];
    *above_out = a1 + sh.misc[1];
    __syncthreads();
  };

  // ---- selection in position order: every key > T and the first
  // (k - above) keys == T, written to the output as they come
  const auto select = [&](int64_t n, auto get, uint32_t T, uint32_t above) {
    const uint32_t need_eq = static_cast<uint32_t>(k) - above;
    ordered2(
        n, get, [&](uint32_t key) { return key > T; }, [&](uint32_t key) { return key == T; },
        [&](uint32_t, int32_t pos, bool gt, bool eq, uint32_t n_gt, uint32_t n_eq) {
          if (gt) out_row[n_gt + (n_eq < need_eq ? n_eq : need_eq)] = pos;
          else if (eq && n_eq < need_eq) out_row[n_gt + n_eq] = pos;
        });
  };

  uint32_t T = 0, above = 0;
  if (L <= p.cap) {
    // Short windows: the whole window into shared memory (positions in
    // order), then everything runs there.
    for (int64_t i0 = 0; i0 < L; i0 += static_cast<int64_t>(kT) * 4) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + u * kT + tid;
        v[u] = i < L ? __ldg(row_base + lo + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + u * kT + tid;
        if (i < L) {
          sh.cand_key[i] = order_key(v[u]);
          sh.cand_pos[i] = static_cast<int32_t>(lo + i);
        }
      }
    }
    __syncthreads();
    radix_select([&](auto sel, auto bin) { smem_hist(L, sel, bin); }, static_cast<uint32_t>(k), &T, &above);
    select(L, smem_get, T, above);
    return;
  }

  // Long windows.  A stride sample of at most cap values estimates a lower
  // threshold t_low: the (2k/S + 32)-th largest sample key, S the stride, so
  // about 2k + 32S window values lie above it (many standard deviations
  // from both k and cap for the strides used).  One ordered pass keeps the
  // values >= t_low in shared memory; if fewer than k or more than cap pass,
  // the exact radix select runs over the window instead.
  const int64_t S = (L + p.cap - 1) / p.cap;
  const int64_t ns = (L + S - 1) / S;
  for (int64_t j = tid; j < ns; j += kT) sh.cand_key[j] = order_key(__ldg(row_base + lo + j * S));
  __syncthreads();
  {
    const int64_t want = 2 * static_cast<int64_t>(k) / S + 32;
    const uint32_t rank = static_cast<uint32_t>(want < ns ? want : ns);
    radix_select([&](auto sel, auto bin) { smem_hist(ns, sel, bin); }, rank, &T, &above);
  }
  const uint32_t t_low = T;
  // candidates >= t_low in position order, from vector loads (few values
  // pass, so the strided shared stores cost little); slots past cap are
  // dropped, the count says whether any were
  uint32_t n_c = 0;
  window_ordered([&](const uint32_t (&keys)[kPer], int64_t pos0, uint32_t valid) {
    uint32_t cnt = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) cnt += (((valid >> j) & 1u) && keys[j] >= t_low) ? 1u : 0u;
    uint32_t total;
    uint32_t slot = n_c + block_scan(cnt, sh.scan, &total);
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (((valid >> j) & 1u) && keys[j] >= t_low) {
        if (slot < static_cast<uint32_t>(p.cap)) {
          sh.cand_key[slot] = keys[j];
          sh.cand_pos[slot] = static_cast<int32_t>(pos0 + j);
        }
        ++slot;
      }
    n_c += total;
  });
  __syncthreads();
  if (n_c >= static_cast<uint32_t>(k) && n_c <= static_cast<uint32_t>(p.cap)) {
    // Every key >= the k-th largest is a candidate, in position order.
    radix_select([&](auto sel, auto bin) { smem_hist(n_c, sel, bin); }, static_cast<uint32_t>(k), &T, &above);
    select(n_c, smem_get, T, above);
  } else {
    radix_select(window_hist, static_cast<uint32_t>(k), &T, &above);
    select(L, global_get, T, above);
  }
}

cudaError_t launch_topk(const TopkParams& p, int smem_bytes, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<p.rows, kTopkThreads, smem_bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fp8idx
