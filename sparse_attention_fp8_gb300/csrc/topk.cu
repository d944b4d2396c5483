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
//  * Radix select of the k-th largest key T: three levels of histograms
//    (12, 12, 8 bits of the key; plain shared atomics).
//  * A window of at most `cap` values is brought into shared memory by one
//    bulk copy straight into the key array, converted to keys in place while
//    the first radix level is counted, and selected there (positions
//    implicit).  A longer one is sampled with a stride S
//    (at most cap samples); the sample's (k/S + 5 sqrt(k/S) + 16)-th
//    largest key is a lower threshold (about six standard deviations of the
//    sampled rank above k/S), and the values above it (about that rank
//    times S: 3.2K for k = 2048 at S = 16) are
//    compacted into shared memory, in position order, for the exact select:
//    in one pass every warp appends the candidates of its own segment of the
//    window, in order, to its own share of the candidate arrays (no block
//    barrier per chunk); a staged copy then puts the shares in position
//    order (a share that overflows falls back to a second pass that writes
//    every candidate at its final slot).  If the kept count falls outside
//    [k, cap] (adversarial or heavily tied rows), the levels and the
//    selection re-read the window from global memory instead.
//  * Selection: every key above the k-th key T and the first (k - #above)
//    keys equal to T in position order are kept, so ties resolve to the
//    lowest positions, and written straight to the output in position
//    order: with one CTA per row each thread takes a run of consecutive
//    keys, marks the run's keys above the first level's bin while counting
//    the second level over it (only the bin's keys are visited by the third
//    level and compared with T afterwards), and one packed block scan places
//    the runs; in a cluster an ordered pass with warp ballots and block-wide
//    prefix sums.
// Rows far too few to fill the GPU (the host's rule: at most a quarter of
// the SM count) with long windows are each split over a thread-block cluster
// of C CTAs instead (or as many as the caller asks for): every step
// above runs per slice of the window, each CTA adding its histogram counts
// into every cluster member's sum histogram (remote shared-memory
// reductions) before each bin search, the candidate counts agreed
// cluster-wide, and each CTA's output offsets taken from the counts of the
// lower-ranked slices.
// The kernel uses no global scratch memory and no atomics outside shared
// memory.  The wait on the bulk copy is bounded: a wait that runs out sets a
// watchdog bit (read by the host) and the row finishes on whatever data it
// has, so no CTA leaves a cluster barrier unmatched.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace fp8idx {

static __device__ unsigned int g_topk_watchdog;

namespace {

constexpr int kT = kTopkThreads;
constexpr int kWarps = kT / 32;
constexpr int kPer = 8;     // elements per thread per chunk of an ordered pass

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);  // -0.0 + 0.0 = +0.0: both zeros share one key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkShared {
  uint32_t* hist;      // [kTopkBins] this CTA's counts
  uint32_t* hsum;      // [kTopkBins] the cluster's counts (== hist with one CTA per row)
  float* ring;         // a short window's values as copied (overlaps hist, hsum)
  uint32_t* cand_key;  // [cap]
  int32_t* cand_pos;   // [cap]
  uint32_t* scan;      // [2 * kWarps] warp totals
  uint32_t* misc;      // [8]: 0,1 bin search result; 4,5 cluster exchange; 7 abort flag
  uint32_t bar;        // the copy's mbarrier (shared address)
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
// above < need <= above + hist[b].  NBINS is 4096 (8 bins per thread, read
// as two 16-byte vectors: consecutive threads, consecutive addresses) or
// 256 (one bin per thread).  Result in misc[0] (bin), misc[1] (above).
template <int NBINS>
__device__ __forceinline__ void find_bin(const uint32_t* hist, uint32_t need, uint32_t* warp_tot, uint32_t* misc) {
  constexpr int kPerT = NBINS >= kT ? NBINS / kT : 1;
  static_assert(kPerT == 8 || kPerT == 1, "bins per thread");
  const int t = threadIdx.x;
  uint32_t h[kPerT];  // h[j]: bin b_hi - j, counted from the top
  const int b_hi = NBINS - 1 - t * kPerT;
  if constexpr (kPerT == 8) {
    const uint4* v = reinterpret_cast<const uint4*>(hist + (NBINS - 8 * (t + 1)));
    const uint4 lo4 = v[0], hi4 = v[1];
    h[0] = hi4.w, h[1] = hi4.z, h[2] = hi4.y, h[3] = hi4.x;
    h[4] = lo4.w, h[5] = lo4.z, h[6] = lo4.y, h[7] = lo4.x;
  } else {
    h[0] = b_hi >= 0 ? hist[b_hi] : 0u;
  }
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < kPerT; ++j) s += h[j];
  uint32_t total;
  uint32_t above = block_scan(s, warp_tot, &total);  // keys in bins above this thread's
#pragma unroll
  for (int j = 0; j < kPerT; ++j) {
    if (above < need && above + h[j] >= need) {
      misc[0] = static_cast<uint32_t>(b_hi - j);
      misc[1] = above;
    }
    above += h[j];
  }
  __syncthreads();
}

// Writes the positions of every key > T and of the first need_eq keys == T
// among kb[0, n) (keys in position order, key i at position pos_of(i)) to
// out_row in position order.  Thread t takes the run [t*m, t*m + m) (m
// odd, so the lanes of a warp read different banks), marks its keys > T and
// == T in two bit masks in one pass, one packed block scan gives every run
// its counts before it, and the run's kept positions are written in order.
// n <= 31 * kT.  Every thread of the block calls it.
// The writing half of write_kept_runs: this thread's run starts at key e0,
// bit j of mgt / meq marks its key e0 + j as > T / == T.
template <class PosOf>
__device__ __forceinline__ void write_kept_masks(uint32_t mgt, uint32_t meq, int e0, PosOf pos_of, uint32_t need_eq,
                                                 int32_t* out_row, uint32_t* scan) {
  uint32_t tot;  // both counts in one scan (16:16; fewer than 2^16 keys)
  const uint32_t ex = block_scan((static_cast<uint32_t>(__popc(mgt)) << 16) | static_cast<uint32_t>(__popc(meq)),
                                 scan, &tot);
  uint32_t n_gt = ex >> 16, n_eq = ex & 0xFFFFu;
  for (uint32_t keep = mgt | meq; keep != 0u; keep &= keep - 1u) {
    const int j = __ffs(keep) - 1;
    if ((mgt >> j) & 1u) {
      out_row[n_gt + (n_eq < need_eq ? n_eq : need_eq)] = pos_of(e0 + j);
      ++n_gt;
    } else {
      if (n_eq < need_eq) out_row[n_gt + n_eq] = pos_of(e0 + j);
      ++n_eq;
    }
  }
}

template <class PosOf>
__device__ __forceinline__ void write_kept_runs(const uint32_t* kb, int n, PosOf pos_of, uint32_t T,
                                                uint32_t need_eq, int32_t* out_row, uint32_t* scan) {
  const int m = ((n + kT - 1) / kT) | 1;
  const int e0 = threadIdx.x * m, e1 = min(n, e0 + m);
  uint32_t mgt = 0u, meq = 0u;
  for (int e = e0; e < e1; ++e) {
    const uint32_t key = kb[e];
    mgt |= (key > T ? 1u : 0u) << (e - e0);
    meq |= (key == T ? 1u : 0u) << (e - e0);
  }
  write_kept_masks(mgt, meq, e0, pos_of, need_eq, out_row, scan);
}

}  // namespace

// One row's selection by C CTAs: one CTA, or (kCluster) the C CTAs of a
// thread-block cluster, CTA c taking the c-th of C equal slices of the
// window.
template <bool kCluster>
__device__ __forceinline__ void topk_row(const TopkParams& p, uint8_t* smem_raw) {
  namespace cg = cooperative_groups;
  const TopkLayout Lo = topk_smem_layout(p.cap);
  TopkShared sh;
  sh.hist = reinterpret_cast<uint32_t*>(smem_raw + Lo.hist);
  sh.hsum = kCluster ? reinterpret_cast<uint32_t*>(smem_raw + Lo.hsum) : sh.hist;
  sh.ring = reinterpret_cast<float*>(smem_raw + Lo.ring);
  sh.cand_key = reinterpret_cast<uint32_t*>(smem_raw + Lo.cand_key);
  sh.cand_pos = reinterpret_cast<int32_t*>(smem_raw + Lo.cand_pos);
  sh.scan = reinterpret_cast<uint32_t*>(smem_raw + Lo.scan);
  sh.misc = reinterpret_cast<uint32_t*>(smem_raw + Lo.misc);
  sh.bar = ptx::smem_u32(smem_raw + Lo.bar);

  const int C = kCluster ? static_cast<int>(cg::this_cluster().num_blocks()) : 1;
  const int crank = kCluster ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
  const int64_t r = blockIdx.x / C;
  // (every CTA of a row's cluster takes the same branch)
  if (p.run_flag != nullptr && __ldg(p.run_flag) == 0u) return;
  if (p.row_mask != nullptr && __ldg(p.row_mask + r) == 0u) return;
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
    if (crank == 0)
      for (int j = tid; j < k; j += kT) out_row[j] = j < L ? static_cast<int32_t>(lo + j) : -1;
    return;
  }
  // This CTA's slice [slo, shi) of the window.
  const int64_t slo = lo + L * crank / C, shi = lo + L * (crank + 1) / C;
  const int64_t Ls = shi - slo;
  const float* row_base = p.logits + r * p.stride;
  const bool vec = p.vec_ok != 0;

  volatile uint32_t* abort_flag = sh.misc + 7;
  if (tid == 0) {
    *abort_flag = 0u;
    ptx::mbar_init(sh.bar, 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();

  // Cluster steps.  sync_all: every CTA's shared writes so far are done and
  // visible.  exchange2(a, b): this CTA's two values in; per value the sum
  // over lower ranks, the sum over all and the maximum out.
  const auto sync_all = [&]() {
    if constexpr (kCluster) cg::this_cluster().sync();
    else __syncthreads();
  };
  struct Sums {
    uint32_t before, all, max;
  };
  const auto exchange2 = [&](uint32_t a, uint32_t b, Sums& sa, Sums& sb) {
    if constexpr (!kCluster) {
      sa = Sums{0u, a, a};
      sb = Sums{0u, b, b};
    } else {
      if (tid == 0) sh.misc[4] = a, sh.misc[5] = b;
      sync_all();
      sa = Sums{0u, 0u, 0u};
      sb = Sums{0u, 0u, 0u};
      for (int c = 0; c < C; ++c) {
        const uint32_t* m = cg::this_cluster().map_shared_rank(sh.misc, c);
        const uint32_t x = m[4], y = m[5];
        sa.before += c < crank ? x : 0u;
        sb.before += c < crank ? y : 0u;
        sa.all += x;
        sb.all += y;
        sa.max = x > sa.max ? x : sa.max;
        sb.max = y > sb.max ? y : sb.max;
      }
      sync_all();  // before the slots are reused
    }
  };
  // After a local histogram pass (its counts complete in sh.hist): every
  // nonzero count added into each cluster member's hsum, then the cluster
  // barrier that makes the sums complete.
  const auto combine = [&](int nbins) {
    if constexpr (kCluster) {
      for (int i = tid; i < nbins; i += kT) {
        const uint32_t v = sh.hist[i];
        if (v)
          for (int c = 0; c < C; ++c) atomicAdd(cg::this_cluster().map_shared_rank(sh.hsum, c) + i, v);
      }
      sync_all();
    }
  };
  // Zeroes this CTA's counts (and sums) for a level of `nbins` bins; in a
  // cluster, no member adds into this CTA's sums before they are zeroed.
  const auto zero_level = [&](int nbins) {
    for (int i = tid; i < nbins; i += kT) {
      sh.hist[i] = 0u;
      if constexpr (kCluster) sh.hsum[i] = 0u;
    }
    sync_all();
  };

  // ---- global-memory window passes (the fallback): groups of 4 positions,
  // one float4 load for a group inside the slice when the rows are 16-byte
  // aligned, scalar loads for the partial groups at its ends -- nothing
  // outside [slo, shi) is read.
  const int64_t gstart = vec ? (slo & ~static_cast<int64_t>(3)) : slo;
  const int64_t ngroups = (shi - gstart + 3) / 4;
  const auto load_group = [&](int64_t gi, uint32_t (&key)[4]) -> uint32_t {  // returns the valid-lane mask
    const int64_t g = gstart + 4 * gi;
    if (gi >= ngroups) return 0u;
    if (vec && g >= slo && g + 4 <= shi) {
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
      const bool in = g + e >= slo && g + e < shi;
      key[e] = in ? order_key(__ldg(row_base + g + e)) : 0u;
      m |= in ? (1u << e) : 0u;
    }
    return m;
  };
  constexpr int kU = 4;  // groups in flight per thread in the histogram passes
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

  // ---- sources: the slice in global memory, or candidates in shared memory
  const auto smem_hist_at = [&](const uint32_t* src, int64_t n_c64, auto sel, auto bin) {
    const int n_c = static_cast<int>(n_c64);  // at most cap
    for (int i0 = 0; i0 < n_c; i0 += kT) {
      const int i = i0 + tid;
      const uint32_t key = i < n_c ? src[i] : 0u;
      hist_add(sh.hist, i < n_c && sel(key), bin(key));
    }
  };
  const auto smem_hist = [&](int64_t n_c64, auto sel, auto bin) { smem_hist_at(sh.cand_key, n_c64, sel, bin); };
  // Ordered passes: element e of a source is (key, position); a chunk is
  // kT*kPer elements, warp w takes the chunk's w-th run of 32*kPer, step j
  // of the run one element per lane (consecutive lanes, consecutive
  // elements: coalesced in global memory, conflict-free in shared memory).
  // `place` gets the element's key, position and its rank among the
  // elements of each predicate before it in position order.  Counts per
  // chunk go through one 16-entry scan of warp totals (double-buffered, one
  // barrier per chunk).
  const auto smem_get = [&](int e, uint32_t& key, int32_t& pos) {
    key = sh.cand_key[e];
    pos = sh.cand_pos[e];
  };
  const auto global_get = [&](int e, uint32_t& key, int32_t& pos) {
    key = order_key(__ldg(row_base + slo + e));
    pos = static_cast<int32_t>(slo + e);
  };
  // Two independent counts per element (packed 16:16 per chunk: a chunk has
  // kT*kPer < 2^16 elements), starting from done_a / done_b.
  const auto ordered2 = [&](int64_t n64, auto get, auto pred_a, auto pred_b, auto place, uint32_t done_a,
                            uint32_t done_b) {
    const int n = static_cast<int>(n64);  // a window or slice: fewer than 2^31 columns
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    int parity = 0;
    for (int c0 = 0; c0 < n; c0 += kT * kPer) {
      const int wbase = c0 + warp * 32 * kPer;
      uint32_t keys[kPer], ba[kPer], bb[kPer];
      int32_t pos[kPer];
      uint32_t wa = 0, wb = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int e = wbase + j * 32 + lane;
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
  };

  // ---- the `need`-th largest key T of the cluster's source and #keys > T,
  // three radix levels (12, 12 and 8 bits of the key)
  // (levels = 2: T is the lower edge of the 24-bit bin holding that key)
  // (level1_done: the caller has already counted every key's top 12 bits
  // into the zeroed histogram)
  const auto radix_select = [&](auto hist_pass, uint32_t need, uint32_t* T_out, uint32_t* above_out,
                                int levels = 3, bool level1_done = false) {
    if (!level1_done) {
      zero_level(kTopkBins);
      hist_pass([](uint32_t) { return true; }, [](uint32_t key) { return key >> 20; });
    }
    __syncthreads();
    combine(kTopkBins);
    find_bin<kTopkBins>(sh.hsum, need, sh.scan, sh.misc);
    const uint32_t b0 = sh.misc[0], a0 = sh.misc[1];
    zero_level(kTopkBins);
    hist_pass([&](uint32_t key) { return (key >> 20) == b0; }, [](uint32_t key) { return (key >> 8) & 0xFFFu; });
    __syncthreads();
    combine(kTopkBins);
    find_bin<kTopkBins>(sh.hsum, need - a0, sh.scan, sh.misc);
    const uint32_t pre24 = (b0 << 12) | sh.misc[0], a1 = a0 + sh.misc[1];
    if (levels == 2) {
      *T_out = pre24 << 8;
      *above_out = a1;
      __syncthreads();
      return;
    }
    zero_level(256);
    hist_pass([&](uint32_t key) { return (key >> 8) == pre24; }, [](uint32_t key) { return key & 0xFFu; });
    __syncthreads();
    combine(256);
    find_bin<256>(sh.hsum, need - a1, sh.scan, sh.misc);
    *T_out = (pre24 << 8) | sh.misc[0];
    *above_out = a1 + sh.misc[1];
    __syncthreads();
  };

  // ---- selection in position order: every key > T and the first
  // (k - above) keys == T, written to the output as they come
  const auto select = [&](int64_t n, auto get, uint32_t T, uint32_t above) {
    const uint32_t need_eq = static_cast<uint32_t>(k) - above;
    uint32_t gt0 = 0, eq0 = 0;  // keys > T and == T in the slices of lower-ranked CTAs
    if constexpr (kCluster) {
      uint32_t n_gt = 0, n_eq = 0;
      for (int64_t i = tid; i < n; i += kT) {
        uint32_t key;
        int32_t pos;
        get(i, key, pos);
        n_gt += key > T ? 1u : 0u;
        n_eq += key == T ? 1u : 0u;
      }
      uint32_t t_gt, t_eq;
      block_scan(n_gt, sh.scan, &t_gt);
      block_scan(n_eq, sh.scan, &t_eq);
      Sums s_gt, s_eq;
      exchange2(t_gt, t_eq, s_gt, s_eq);
      gt0 = s_gt.before;
      eq0 = s_eq.before;
    }
    ordered2(
        n, get, [&](uint32_t key) { return key > T; }, [&](uint32_t key) { return key == T; },
        [&](uint32_t, int32_t pos, bool gt, bool eq, uint32_t n_gt, uint32_t n_eq) {
          const bool w = gt || (eq && n_eq < need_eq);
          const uint32_t idx = n_gt + (n_eq < need_eq ? n_eq : need_eq);  // == n_gt + n_eq for a kept tie
          if (w) out_row[idx] = pos;
        },
        gt0, eq0);
  };

  // One CTA per row, keys kb[0, n) in shared memory in position order:
  // the exact selection written to the output.  The first radix level as in
  // radix_select (already counted when level1_done); the second is counted
  // over each thread's run of keys while the run's keys above the first
  // level's bin are marked as kept and the bin's keys as open; the third
  // level and the final comparison with T visit only the open keys, and the
  // runs are written (write_kept_masks) without a further pass.
  const auto exact_runs = [&](const uint32_t* kb, int n, auto pos_of, bool level1_done) {
    if (!level1_done) {
      zero_level(kTopkBins);
      smem_hist_at(kb, n, [](uint32_t) { return true; }, [](uint32_t key) { return key >> 20; });
    }
    __syncthreads();
    find_bin<kTopkBins>(sh.hist, static_cast<uint32_t>(k), sh.scan, sh.misc);
    const uint32_t b0 = sh.misc[0], a0 = sh.misc[1];
    const int m = ((n + kT - 1) / kT) | 1;  // odd: the lanes of a warp read different banks
    const int e0 = tid * m, e1 = min(n, e0 + m);
    // second level over the run: keys above the first level's bin are kept
    // whatever T is; the bin's own keys are marked for the later levels
    zero_level(kTopkBins);
    uint32_t mgt = 0u, mbin = 0u;
    for (int e = e0; e < e1; ++e) {
      const uint32_t key = kb[e], pre = key >> 20;
      mgt |= (pre > b0 ? 1u : 0u) << (e - e0);
      if (pre == b0) {
        mbin |= 1u << (e - e0);
        atomicAdd(sh.hist + ((key >> 8) & 0xFFFu), 1u);
      }
    }
    __syncthreads();
    find_bin<kTopkBins>(sh.hist, static_cast<uint32_t>(k) - a0, sh.scan, sh.misc);
    const uint32_t pre24 = (b0 << 12) | sh.misc[0], a1c = a0 + sh.misc[1];
    // third level over the marked keys only
    zero_level(256);
    uint32_t mcand = 0u;
    for (uint32_t c = mbin; c != 0u; c &= c - 1u) {
      const int j = __ffs(c) - 1;
      const uint32_t key = kb[e0 + j], pre = key >> 8;
      mgt |= (pre > pre24 ? 1u : 0u) << j;
      if (pre == pre24) {
        mcand |= 1u << j;
        atomicAdd(sh.hist + (key & 0xFFu), 1u);
      }
    }
    __syncthreads();
    find_bin<256>(sh.hist, static_cast<uint32_t>(k) - a1c, sh.scan, sh.misc);
    const uint32_t Tk = (pre24 << 8) | sh.misc[0];
    const uint32_t above_k = a1c + sh.misc[1];
    uint32_t meq = 0u;
    for (uint32_t c = mcand; c != 0u; c &= c - 1u) {
      const int j = __ffs(c) - 1;
      const uint32_t key = kb[e0 + j];
      mgt |= (key > Tk ? 1u : 0u) << j;
      meq |= (key == Tk ? 1u : 0u) << j;
    }
    write_kept_masks(mgt, meq, e0, pos_of, static_cast<uint32_t>(k) - above_k, out_row, sh.scan);
  };

  uint32_t T = 0, above = 0;
  if ((L + C - 1) / C + 4 <= p.cap) {
    // Short windows: each slice into its CTA's shared memory, then
    // everything runs there.  Aligned rows: one bulk copy of [slo rounded
    // down to 4, shi rounded down to 4) straight into the key array, the
    // last (at most 3) values by plain loads; the keys are converted in
    // place while the first radix level is counted, and the positions are
    // implicit (key i of the slice is position slo + i).
    const int64_t b0 = slo & ~static_cast<int64_t>(3), a1 = shi & ~static_cast<int64_t>(3);
    const bool staged = vec && a1 > b0;
    // (32-bit offsets: a slice here holds at most cap - 4 values, positions are below 2^31)
    const int Ls32 = static_cast<int>(Ls), slo32 = static_cast<int>(slo);
    const int a1r = static_cast<int>(a1 - slo);  // the staged part is [0, a1r) of the slice
    uint32_t* const kbase = sh.cand_key + (staged ? static_cast<int>(slo - b0) : 0);
    zero_level(kTopkBins);
    if (staged) {
      if (tid == 0) {
        ptx::fence_proxy_async_smem();
        const uint32_t bytes = static_cast<uint32_t>((a1 - b0) * 4);
        ptx::mbar_arrive_expect_tx(sh.bar, bytes);
        ptx::bulk_g2s(ptx::smem_u32(sh.cand_key), row_base + b0, bytes, sh.bar);
      }
      // bounded: a wait that runs out flags the watchdog; in-flight bytes
      // land before the array is reused
      wait_bounded(sh.bar, 0u, abort_flag, &g_topk_watchdog, kSiteStageFull);
      if (*abort_flag && tid == 0) wait_drain(sh.bar, 0u, &g_topk_watchdog);
    }
    for (int i0 = 0; i0 < Ls32; i0 += kT * 4) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kT + tid;
        v[u] = i >= Ls32 ? 0.f : (staged && i < a1r) ? __uint_as_float(kbase[i]) : __ldg(row_base + slo32 + i);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kT + tid;
        if (i < Ls32) {
          const uint32_t key = order_key(v[u]);
          kbase[i] = key;
          hist_add(sh.hist, true, key >> 20);
        }
      }
    }
    if constexpr (!kCluster) {
      exact_runs(kbase, Ls32, [&](int e) { return slo32 + e; }, true);
    } else {
      radix_select([&](auto sel, auto bin) { smem_hist_at(kbase, Ls, sel, bin); }, static_cast<uint32_t>(k), &T,
                   &above, 3, true);
      select(Ls, [&](int e, uint32_t& key, int32_t& pos) {
        key = kbase[e];
        pos = slo32 + e;
      }, T, above);
    }
    return;
  }

  // Long windows.  A stride sample of at most cap values (stride S over
  // the whole window, each CTA loading the samples in its slice) estimates a
  // lower threshold t_low: the (k/S + 5 sqrt(k/S) + 16)-th largest sample
  // key (rounded down to its 24-bit bin).  About k/S samples lie above the
  // true k-th value, give or take sqrt(k/S), so the rank sits about six of
  // those deviations above it, and about rank * S window values lie above
  // t_low (3.2K for k = 2048 at S = 16, 2.6K at S = 4: well inside cap).
  // The values >= t_low are then compacted into shared memory; if fewer than
  // k pass in the cluster, or more than cap in one CTA, the exact radix
  // select runs over the window instead.
  const int64_t S = (L + p.cap - 1) / p.cap;
  const int64_t ns = (L + S - 1) / S;  // samples lo + jS of the whole window: <= cap
  const int64_t j_lo = (slo - lo + S - 1) / S, j_hi = (shi - lo + S - 1) / S;  // this slice's samples
  const int64_t ns_c = j_hi - j_lo;
  {
    // (32-bit offsets: positions are below 2^31)
    const int ns32 = static_cast<int>(ns_c), S32 = static_cast<int>(S);
    const float* samp = row_base + lo + j_lo * S;
    for (int j0 = 0; j0 < ns32; j0 += kT * 16) {  // all of a cap-8192 sample in flight
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int j = j0 + u * kT + tid;
        v[u] = j < ns32 ? __ldg(samp + j * S32) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int j = j0 + u * kT + tid;
        if (j < ns32) sh.cand_key[j] = order_key(v[u]);
      }
    }
  }
  __syncthreads();
  {
    // the sample's count above the true k-th value is about k/S with a
    // standard deviation of about sqrt(k/S): keep about six of them as margin
    const float kS = static_cast<float>(k) / static_cast<float>(S);
    const int64_t want = static_cast<int64_t>(kS + 5.0f * sqrtf(kS)) + 16;
    const uint32_t rank = static_cast<uint32_t>(want < ns ? want : ns);
    radix_select([&](auto sel, auto bin) { smem_hist(ns_c, sel, bin); }, rank, &T, &above, 2);
  }
  // the lower edge of the 24-bit bin of the rank-th sample key, never below
  // the key of -inf (the edge of the bin holding -inf is a NaN pattern)
  const uint32_t t_low = T > order_key(-INFINITY) ? T : order_key(-INFINITY);

  // Candidates >= t_low in position order, tested as floats against the
  // value whose key is t_low (the key order is the float order, -0.0 ==
  // +0.0; no NaN in a window).  Each warp owns one contiguous segment of
  // the slice (groups of 4 positions from slo rounded down to 4; positions
  // before slo masked) and walks it without block barriers, lane l of a
  // step taking groups 2l and 2l+1 (8 consecutive positions).  The last (at
  // most 3) positions of an aligned slice are appended by thread 0.  Slots
  // past cap are dropped; the count says whether any were.
  const float f_low = __uint_as_float((t_low & 0x80000000u) ? (t_low & 0x7FFFFFFFu) : ~t_low);
  uint32_t n_c = 0;
  {
    const int lane = tid & 31, warp = tid >> 5;
    // positions are below 2^31: 32-bit offsets from here on
    const int32_t slo32 = static_cast<int32_t>(slo), shi32 = static_cast<int32_t>(shi);
    const int32_t b0 = slo32 & ~3;
    const int32_t a1 = vec ? (shi32 & ~3) : shi32;  // grouped part [b0, a1)
    const int32_t G = a1 > b0 ? (a1 - b0 + 3) / 4 : 0;
    const int32_t g_lo = static_cast<int32_t>(static_cast<int64_t>(G) * warp / kWarps);
    const int32_t g_hi = static_cast<int32_t>(static_cast<int64_t>(G) * (warp + 1) / kWarps);
    const int nsteps = (g_hi - g_lo + 63) / 64;  // warp-uniform
    const uint32_t cap = static_cast<uint32_t>(p.cap);
    // the 8 values of this lane in step st and their candidate mask
    const auto load8 = [&](int st, float (&f)[8]) -> uint32_t {
      uint32_t valid = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int32_t g = g_lo + st * 64 + 2 * lane + h, base = b0 + 4 * g;
        if (g < g_hi && vec) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(row_base + base));
          f[4 * h] = x.x, f[4 * h + 1] = x.y, f[4 * h + 2] = x.z, f[4 * h + 3] = x.w;
#pragma unroll
          for (int e = 0; e < 4; ++e) valid |= (base + e >= slo32) ? (1u << (4 * h + e)) : 0u;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const bool in = g < g_hi && base + e >= slo32 && base + e < a1;
            f[4 * h + e] = in ? __ldg(row_base + base + e) : 0.f;
            valid |= in ? (1u << (4 * h + e)) : 0u;
          }
        }
      }
      return valid;
    };
    const auto mask8 = [&](const float (&f)[8], uint32_t valid) -> uint32_t {
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) m |= f[e] >= f_low ? (1u << e) : 0u;
      return m & valid;
    };
    // One pass: each warp appends its candidates, in order, to its own
    // share of the candidate arrays (Q = cap / kWarps entries), counting
    // past the share if it overflows.  Two steps per iteration with one
    // packed (16:16) warp scan; the next two steps' loads are issued before
    // the current ones are placed.
    const uint32_t Q = cap / kWarps;
    // Candidates are sparse (a few per 256 values), so a lane spends work
    // only on its set bits: each iteration every lane with a bit left places
    // its lowest one; the warp iterates max-over-lanes times.
    const auto place8 = [&](const float (&f)[8], uint32_t m, uint32_t s0, int st, uint32_t limit, uint32_t off) {
      const int32_t p0 = b0 + 4 * (g_lo + st * 64 + 2 * lane);
      while (__any_sync(0xffffffffu, m != 0u)) {
        if (m) {
          const int e = __ffs(m) - 1;
          m &= m - 1u;
          float v = f[0];
#pragma unroll
          for (int q = 1; q < 8; ++q) v = e == q ? f[q] : v;
          if (s0 < limit) {
            sh.cand_key[off + s0] = order_key(v);
            sh.cand_pos[off + s0] = p0 + e;
          }
          ++s0;
        }
      }
    };
    // places steps st, st+1 (masks m0, m1) at run + their warp prefix; returns the pair's total
    const auto place2 = [&](const float (&f0)[8], uint32_t m0, const float (&f1)[8], uint32_t m1, int st,
                            uint32_t run, uint32_t limit, uint32_t off) -> uint32_t {
      const uint32_t c = (static_cast<uint32_t>(__popc(m0)) << 16) | static_cast<uint32_t>(__popc(m1));
      uint32_t x = c;  // inclusive warp scan of the packed lane counts
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const uint32_t tot = __shfl_sync(0xffffffffu, x, 31), ex = x - c;
      place8(f0, m0, run + (ex >> 16), st, limit, off);
      place8(f1, m1, run + (tot >> 16) + (ex & 0xFFFFu), st + 1, limit, off);
      return (tot >> 16) + (tot & 0xFFFFu);
    };
    uint32_t run = 0;
    {
      float fa[8], fb[8];
      uint32_t va = load8(0, fa), vb = load8(1, fb);
      for (int st = 0; st < nsteps; st += 2) {
        const uint32_t ma = mask8(fa, va), mb = mask8(fb, vb);
        float fc[8], fd[8];
        const uint32_t vc = load8(st + 2, fc), vd = load8(st + 3, fd);  // past the segment: nothing loaded
        run += place2(fa, ma, fb, mb, st, run, Q, static_cast<uint32_t>(warp) * Q);
#pragma unroll
        for (int e = 0; e < 8; ++e) fa[e] = fc[e], fb[e] = fd[e];
        va = vc, vb = vd;
      }
    }
    if (lane == 0) sh.scan[warp] = run;
    __syncthreads();
    uint32_t before = 0, n_main = 0, over = 0;  // this warp's first slot, the total, any share overflowed
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t t = sh.scan[w];
      before += w < warp ? t : 0u;
      n_main += t;
      over |= t > Q ? 1u : 0u;
    }
    if (!over) {
      // Compaction into position order through the idle histogram area
      // (>= cap words): keys first, then positions; warp w copies its own
      // share to offset `before` (coalesced, no search), a barrier, then
      // the block copies the staged array back to the front.
      uint32_t* const stage = sh.hist;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        uint32_t* const arr = part == 0 ? sh.cand_key : reinterpret_cast<uint32_t*>(sh.cand_pos);
        for (uint32_t o = lane; o < run; o += 32) stage[before + o] = arr[static_cast<uint32_t>(warp) * Q + o];
        __syncthreads();
        for (uint32_t i = tid; i < n_main; i += kT) arr[i] = stage[i];
        __syncthreads();
      }
    } else {
      // A share overflowed (candidates concentrated in one segment): a
      // second pass over the segments writes every candidate at its final
      // slot (the counts above give each warp's first slot).
      __syncthreads();
      uint32_t r2 = before;
      for (int st = 0; st < nsteps; st += 2) {
        float f0[8], f1[8];
        const uint32_t v0 = load8(st, f0), v1 = load8(st + 1, f1);
        r2 += place2(f0, mask8(f0, v0), f1, mask8(f1, v1), st, r2, cap, 0u);
      }
      __syncthreads();
    }
    n_c = n_main;
    if (a1 < shi32) {  // the last (at most 3) positions of an aligned slice
      uint32_t tail = 0;
      for (int32_t q = a1; q < shi32; ++q) {
        const float v = __ldg(row_base + q);
        if (v >= f_low) {
          if (tid == 0 && n_main + tail < cap) {
            sh.cand_key[n_main + tail] = order_key(v);
            sh.cand_pos[n_main + tail] = q;
          }
          ++tail;
        }
      }
      n_c += tail;
    }
  }
  __syncthreads();
  Sums cnt, unused;
  exchange2(n_c, 0u, cnt, unused);
  if (cnt.all >= static_cast<uint32_t>(k) && cnt.max <= static_cast<uint32_t>(p.cap)) {
    // Every key >= the k-th largest is a candidate, in position order.
    if constexpr (!kCluster) {
      exact_runs(sh.cand_key, static_cast<int>(n_c), [&](int e) { return sh.cand_pos[e]; }, false);
    } else {
      radix_select([&](auto sel, auto bin) { smem_hist(n_c, sel, bin); }, static_cast<uint32_t>(k), &T, &above);
      select(n_c, smem_get, T, above);
    }
  } else {
    radix_select(window_hist, static_cast<uint32_t>(k), &T, &above);
    select(Ls, global_get, T, above);
  }
}

__global__ void __launch_bounds__(kTopkThreads, 2) topk_rows_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  topk_row<false>(p, smem_raw);
}

// Launched with clusters of `ctas` CTAs along x, one cluster per row.
__global__ void __launch_bounds__(kTopkThreads, 2) topk_rows_cluster_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  topk_row<true>(p, smem_raw);
}

cudaError_t launch_topk(const TopkParams& p, int ctas, int smem_bytes, cudaStream_t stream) {
  if (ctas < 1 || ctas > kTopkMaxCluster) return cudaErrorInvalidValue;
  void (*kern)(TopkParams) = ctas > 1 ? topk_rows_cluster_kernel : topk_rows_kernel;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem_bytes);
  if (e != cudaSuccess) return e;
  if (ctas == 1) {
    kern<<<p.rows, kTopkThreads, smem_bytes, stream>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.rows) * static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ctas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// ------------------------------------------------ fused decode top-k passes
//
// fp8_paged_mqa_topk runs the decode kernel twice: once on every 32nd item
// of each request (the sample, written to the workspace's logits rows), once
// in its filter form, which keeps only the logits at or above each row's
// threshold (stored at their positions, marked in a bitmap) instead of
// writing every logit.  The two per-row kernels below sit before and after
// the filter pass.
namespace {

// Row r = b*next_n + n: window [0, W) of the decode logits, W = min(ctx_b -
// next_n + n + 1, max_model_len) (0 if negative).
__device__ __forceinline__ int64_t fused_window(const FusedTopkParams& p, int64_t r) {
  const int64_t b = r / p.next_n, n = r - b * p.next_n;
  int64_t ctx = __ldg(p.context_lens + b);
  if (ctx < 0) ctx = 0;
  int64_t hi = ctx - p.next_n + n + 1;
  if (hi > p.cols) hi = p.cols;
  return hi > 0 ? hi : 0;
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// The need-th largest of n keys get(i) (1 <= need <= n) and the number of
// keys above it: three radix levels (12, 12, 8 bits) over block-wide
// shared-memory histograms.  Every thread of the block calls it.
template <class Get>
__device__ uint32_t block_kth_key(Get get, int n, uint32_t need, uint32_t* hist, uint32_t* scan, uint32_t* misc,
                                  uint32_t* above_out, bool lower_edge_24 = false) {
  const int tid = threadIdx.x;
  const auto level = [&](int nbins, auto sel, auto bin) {
    for (int i = tid; i < nbins; i += kT) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kT) {
      const uint32_t key = get(i);
      hist_add(hist, sel(key), bin(key));
    }
    __syncthreads();
  };
  level(kTopkBins, [](uint32_t) { return true; }, [](uint32_t key) { return key >> 20; });
  find_bin<kTopkBins>(hist, need, scan, misc);
  const uint32_t b0 = misc[0], a0 = misc[1];
  __syncthreads();
  level(kTopkBins, [&](uint32_t key) { return (key >> 20) == b0; }, [](uint32_t key) { return (key >> 8) & 0xFFFu; });
  find_bin<kTopkBins>(hist, need - a0, scan, misc);
  const uint32_t pre24 = (b0 << 12) | misc[0], a1 = a0 + misc[1];
  __syncthreads();
  if (lower_edge_24) {  // the lower edge of the 24-bit bin holding that key (a lower bound of it)
    *above_out = a1;
    return pre24 << 8;
  }
  level(256, [&](uint32_t key) { return (key >> 8) == pre24; }, [](uint32_t key) { return key & 0xFFu; });
  find_bin<256>(hist, need - a1, scan, misc);
  const uint32_t T = (pre24 << 8) | misc[0];
  *above_out = a1 + misc[1];
  __syncthreads();
  return T;
}

}  // namespace

// Per row: reset of the row's per-call state, then the threshold.  The
// sampled logits of row r are its window positions in items 0, 32, 64, ...
// of its request (every q-th of those items when there are more than
// kFusedMaxSample values, q the smallest that fits).  About mu = k * f of
// them (f: the sampled fraction of the window) are expected among the row's
// k largest; the threshold is the m-th largest sample with m = mu + 4 sd + 1
// (binomial sd), so that the logits above it number about m / f >= k (a
// shortfall sends the row to the exact fallback) and stay far below the
// candidate capacity.  A sample that is the whole window gives m = k: the
// exact k-th largest.
__global__ void __launch_bounds__(kTopkThreads, 1) fused_threshold_kernel(const FusedTopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw);  // [kTopkBins]
  uint32_t* keys = hist + kTopkBins;                      // [kFusedMaxSample]
  __shared__ uint32_t scan[2 * kWarps];
  __shared__ uint32_t misc[8];
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t W = fused_window(p, r);
  if (tid == 0) {
    p.row_flag[r] = 0u;
    if (r % p.next_n == 0) p.req_flag[r / p.next_n] = 0u;
    if (r == 0) p.any[0] = 0u;
  }
  if (W <= p.k) {
    if (tid == 0) p.thr[r] = -INFINITY;
    return;
  }
  {
    // The row's candidate bitmap, cleared for the filter pass, which then
    // stores only the words that hold a candidate (the row's words start
    // 16-byte aligned; positions are below 2^31).
    const int nv = static_cast<int>((W + 127) / 128);
    uint4* b4 = reinterpret_cast<uint4*>(p.cand + r * p.tw);
    for (int v = tid; v < nv; v += kT) b4[v] = make_uint4(0u, 0u, 0u, 0u);
  }
  const int64_t I = p.item_tokens, SI = static_cast<int64_t>(kFusedSampleStride) * I;
  const int lgI = I == 256 ? 8 : 7;  // items are 128 or 256 tokens
  int64_t J = (W + SI - 1) / SI;  // sampled items starting inside the window
  int64_t q = 1;                  // every q-th of them
  while (((J + q - 1) / q) * I > kFusedMaxSample) ++q;
  const int64_t Jq = (J + q - 1) / q, last = (Jq - 1) * q;  // items used; the last one may be partial
  const int64_t n_s = (Jq - 1) * I + min(I, W - last * SI);
  const float* row = p.logits + r * p.ls;
  // the sample's keys into shared memory: eight loads in flight per thread
  {
    // (32-bit offsets: the sample holds at most kFusedMaxSample values, the
    // row's positions are below 2^31)
    const int n32 = static_cast<int>(n_s), qSI = static_cast<int>(q * SI);
    for (int e0 = 0; e0 < n32; e0 += 8 * kT) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * kT + tid, j = e >> lgI;
        v[u] = e < n32 ? row[j * qSI + (e - (j << lgI))] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * kT + tid;
        if (e < n32) keys[e] = order_key(v[u]);
      }
    }
  }
  __syncthreads();
  int64_t m;
  if (n_s >= W) {
    m = p.k;
  } else {
    const double f = static_cast<double>(n_s) / static_cast<double>(W);
    const double mu = p.k * f, sd = sqrt(mu * (1.0 - f));
    m = static_cast<int64_t>(ceil(mu + 4.0 * sd)) + 1;
  }
  float t = -INFINITY;
  if (m <= n_s) {
    uint32_t above;
    // (a threshold from a part of the window need only be a lower bound of
    // the m-th largest sample: two radix levels, the lower edge of its
    // 24-bit bin; a whole-window sample gives the exact k-th largest)
    uint32_t tk = block_kth_key([&](int i) { return keys[i]; }, static_cast<int>(n_s), static_cast<uint32_t>(m), hist,
                                scan, misc, &above, n_s < W);
    const uint32_t k_ninf = order_key(-INFINITY);  // (the edge of the bin holding -inf is a NaN pattern)
    t = key_value(tk > k_ninf ? tk : k_ninf);
  }
  if (tid == 0) p.thr[r] = t;
}

// Per row, after the filter pass: the row's candidates are the positions in
// its bitmap (their logits, at or above the threshold, stored at those
// positions of the row).  If they cannot hold the row's k largest -- more
// than the shared-memory capacity, or fewer than k -- the row (and its
// request) is flagged for the exact fallback and left to it.  Otherwise the
// candidates are compacted in position order; the k-th largest key T among
// them, every candidate above T and the first (k - #above T) equal to T are
// written in position order.
__global__ void __launch_bounds__(kTopkThreads, 1) fused_select_kernel(const FusedTopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw);        // [kTopkBins]
  uint32_t* keys = hist + kTopkBins;                              // [kTopkMaxCap]
  int32_t* pos = reinterpret_cast<int32_t*>(keys + kTopkMaxCap);  // [kTopkMaxCap]
  __shared__ uint32_t scan[2 * kWarps];
  __shared__ uint32_t misc[8];
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x;
  const int k = p.k;
  const int64_t W = fused_window(p, r);
  int32_t* out_row = p.out + r * p.out_stride;
  if (W <= k) {
    for (int j = tid; j < k; j += kT) out_row[j] = j < W ? j : -1;
    return;
  }
  // the bitmap's count; each thread owns a contiguous run of words, read as
  // 16-byte vectors (the row's words start 16-byte aligned)
  // (32-bit offsets: positions are below 2^31)
  const int nw = static_cast<int>((W + 31) / 32);
  const int nv = (nw + 3) / 4;
  const int vpt = (nv + kT - 1) / kT;
  const int v0 = min(nv, tid * vpt), v1 = min(nv, v0 + vpt);
  const uint4* bits4 = reinterpret_cast<const uint4*>(p.cand + r * p.tw);
  // (the filter pass writes every word whose first position is in the
  // window; the words of the last vector past the window are not read)
  const auto word = [&](int v, int q, const uint4& x) -> uint32_t {
    const uint32_t w = q == 0 ? x.x : q == 1 ? x.y : q == 2 ? x.z : x.w;
    return v * 4 + q < nw ? w : 0u;
  };
  uint32_t mine = 0;
  for (int v = v0; v < v1; ++v) {
    const uint4 x = bits4[v];
#pragma unroll
    for (int q = 0; q < 4; ++q) mine += __popc(word(v, q, x));
  }
  uint32_t cA;
  const uint32_t before = block_scan(mine, scan, &cA);
  if (cA > static_cast<uint32_t>(kTopkMaxCap) || cA < static_cast<uint32_t>(k)) {
    if (tid == 0) {
      p.row_flag[r] = 1u;
      atomicOr(p.req_flag + r / p.next_n, 1u);
      atomicOr(p.any, 1u);
    }
    return;
  }
  {
    uint32_t j = before;
    for (int v = v0; v < v1; ++v) {
      const uint4 x = bits4[v];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t bits = word(v, q, x);
        while (bits != 0u) {
          pos[j++] = static_cast<int32_t>((v * 4 + q) * 32 + __ffs(bits) - 1);
          bits &= bits - 1u;
        }
      }
    }
  }
  __syncthreads();
  const float* row = p.logits + r * p.ls;
  for (uint32_t i0 = 0; i0 < cA; i0 += 8 * kT) {  // their logits: eight loads in flight per thread
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t i = i0 + u * kT + tid;
      v[u] = i < cA ? row[pos[i]] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t i = i0 + u * kT + tid;
      if (i < cA) keys[i] = order_key(v[u]);
    }
  }
  __syncthreads();
  uint32_t above;
  const uint32_t T = block_kth_key([&](int i) { return keys[i]; }, static_cast<int>(cA), static_cast<uint32_t>(k), hist,
                                   scan, misc, &above);
  write_kept_runs(keys, static_cast<int>(cA), [&](int e) { return pos[e]; }, T, static_cast<uint32_t>(k) - above,
                  out_row, scan);
}

cudaError_t launch_fused_threshold(const FusedTopkParams& p, int smem_bytes, cudaStream_t stream) {
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fused_threshold_kernel), smem_bytes);
  if (e != cudaSuccess) return e;
  fused_threshold_kernel<<<p.rows, kTopkThreads, smem_bytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fused_select(const FusedTopkParams& p, int smem_bytes, cudaStream_t stream) {
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fused_select_kernel), smem_bytes);
  if (e != cudaSuccess) return e;
  fused_select_kernel<<<p.rows, kTopkThreads, smem_bytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t read_topk_watchdog(unsigned int* value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_topk_watchdog, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_topk_watchdog, &zero, sizeof(unsigned int));
}

}  // namespace fp8idx
