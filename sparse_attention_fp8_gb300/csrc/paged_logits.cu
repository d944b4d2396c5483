// Decode indexer logits (fp8_paged_mqa_logits) for sm_103a.
//
// Defined by aiter PR 5047 "[HIP] [JIT] fp8_paged_mqa_logits: hand-written
// gfx950 decode indexer kernel" (Motivation; Technical Details) and aiter
// issue 5477 "gfx950 paged MQA logits: next_n spends the tile on program
// count ..." (The ask):
//   out[b*next_n + n, p] = sum_h relu(<Q[b,n,h,:], K_b[p,:]>) * w[b*next_n+n, h]
//                          * kv_scale_b[p]       for p <= ctx_b - next_n + n,
// with K_b[p] and its scale read from the paged cache through block_tables.
//
// Design (one persistent CTA per SM, warp-specialised, 10 warps; 11 for
// block size 1):
//  * Work items are (request b, T consecutive 128-token tiles): T = 2 when
//    next_n*heads <= 128 (one barrier round trip per 256 tokens), else 1.
//    Each CTA takes one contiguous range of the flattened item list, found on
//    the device from context_lens (a prefix sum in shared memory), so no host
//    synchronisation is needed and every CTA gets the same number of items
//    (+-1).
//  * Producer warp 0: per item one 3-D TMA per cache block for the K rows
//    (view [block][row][128 B], 128-byte swizzle) and one 2-D TMA (or, for
//    16-token blocks, a bulk copy) per block for its scales, into a ring of
//    shared-memory stages; block-table entries are prefetched 32 blocks
//    ahead.  (One warp: a second one walking the same items only took issue
//    slots from the epilogue warps on its sub-partition.)  For block size 1
//    (co-packed 132-byte tokens, only 4-byte aligned) producer warps 0-1 each
//    gather 64 tokens of a tile with 4-byte cp.async into the same swizzled
//    layout instead.  Warp 0 also loads each request's Q block and weights
//    into one of two buffers.
//  * MMA warp (after the producers): the K tile is the A operand (M = 128 tokens) and the
//    request's whole Q block [next_n*heads, 128] is the B operand, so
//    N = next_n*heads: one K tile feeds every speculative row in one
//    tcgen05.mma chain (the fold of next_n into the MMA asked for in aiter
//    issue 5477, The ask).  Four K=32 e4m3 MMAs accumulate in f32 in tensor
//    memory, which holds 2..16 accumulators (as many as 512 columns allow).
//  * Epilogue warpgroups (the last 8 warps): with two tiles per item group g reads
//    tile g of every item; with one, the groups take alternate items.  Thread
//    = token (TMEM lane): read the token's scale and free the stage, then
//    reduce the accumulator's 32-column chunks (common.cuh reduce_rows: loads
//    rotate through register buffers, ReLU as packed x+|x|, packed FMA with
//    the weights, head sum in the thread), multiply once by the token's
//    kv_scale (the hoist of aiter PR 5047, Technical Details: scale >= 0 and
//    ReLU is positive-homogeneous) and store if inside the causal window.  A
//    warp stores 32 consecutive floats per row: coalesced 128 B.  The loop is
//    instantiated per chunk count (next_n*heads/32).
//  * Control loops keep ring indices and phases as counters (no division per
//    tile); every wait is bounded (common.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8idx {

static __device__ unsigned int g_paged_watchdog;

namespace {

// Cursor over a CTA's contiguous range of (request, tile) items.
struct ItemCursor {
  const int32_t* tp;  // tile prefix in smem, tp[b] = first item of request b
  int batch;
  int b, t, tiles_b;

  __device__ void start(int begin) {
    int lo = 0, hi = batch;  // largest b with tp[b] <= begin
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tp[mid] <= begin) lo = mid; else hi = mid;
    }
    b = lo;
    t = begin - tp[lo];
    tiles_b = tp[lo + 1] - tp[lo];
  }
  // Moves to the next item; returns true if it belongs to a new request.
  __device__ bool advance() {
    if (++t < tiles_b) return false;
    do { ++b; } while (b < batch && tp[b + 1] == tp[b]);
    t = 0;
    tiles_b = (b < batch) ? tp[b + 1] - tp[b] : 0;
    return true;
  }
};

__device__ __forceinline__ int64_t clamp_ctx(int32_t ctx, const PagedParams& p) {
  int64_t c = ctx < 0 ? 0 : ctx;
  const int64_t cap_table = static_cast<int64_t>(p.max_blocks) * p.block_size;
  if (c > p.max_model_len) c = p.max_model_len;
  if (c > cap_table) c = cap_table;
  return c;
}

__device__ __forceinline__ int32_t load_table(const PagedParams& p, int b, int64_t idx, int64_t limit) {
  if (idx < 0 || idx >= limit) return 0;
  return __ldg(p.block_tables + static_cast<int64_t>(b) * p.bt_stride + idx);
}

__device__ __forceinline__ int32_t clamp_block(int32_t v, int64_t num_blocks) {
  const int32_t hi = static_cast<int32_t>(num_blocks - 1);
  return v < 0 ? 0 : (v > hi ? hi : v);
}

}  // namespace

// MODE: kPlain (the logits), kFilter (the fused top-k's candidates instead
// of the logits) or kSample (the logits of every kFusedSampleStride-th item
// of each request).  The item stride is a compile-time constant: a runtime
// stride slowed the block-size-1 gather by a third.
enum PagedMode : int { kPlain = 0, kFilter = 1, kSample = 2 };

template <int HEADS, bool GATHER, int MODE>
__global__ void __launch_bounds__(paged_threads(GATHER), 1)
    paged_logits_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                        const __grid_constant__ CUtensorMap tm_sc, const PagedParams p) {
  constexpr bool FILTER = MODE == kFilter;
  // a launch that is only needed when an earlier one raised the flag
  if (p.run_flag != nullptr && __ldg(p.run_flag) == 0u) return;
  constexpr int kProdWarps = paged_producer_warps(GATHER);
  constexpr int kMmaWarp = kProdWarps;
  constexpr int kEpiWarp0 = kMmaWarp + 1;
  constexpr uint32_t kTmemCols = 512;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_up_1024(smem_raw);
  const int N = p.n_cols;
  const int S = p.stages;
  const int B = p.batch;
  const int AB = p.acc_bufs;
  const int T = p.sub_tiles;                         // 128-token tiles per item
  const int ITEM = kTileTokens * T;                  // tokens per item
  const uint32_t acc_cols = kTmemCols / AB;          // TMEM columns per item
  const uint32_t sub_cols = acc_cols / T;            // ... per 128-token tile
  const uint32_t stage_k = static_cast<uint32_t>(T) * kKTileBytes;
  const uint32_t stage_sc = static_cast<uint32_t>(T) * kTileTokens;  // scales (floats) per stage
  const PagedSmem L = paged_smem_layout(N, S, B, T);
  uint8_t* q_s = smem + L.q;
  uint8_t* k_s = smem + L.k;
  float* sc_s = reinterpret_cast<float*>(smem + L.scale);
  float* w_s = reinterpret_cast<float*>(smem + L.w);
  int32_t* tp = reinterpret_cast<int32_t*>(smem + L.tp);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile uint32_t* abort_flag = misc + 1;

  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * S;
  const uint32_t accf0 = empty0 + 8u * S;           // [kMaxAccBufs]
  const uint32_t acce0 = accf0 + 8u * kMaxAccBufs;  // [kMaxAccBufs]
  const uint32_t qf0 = acce0 + 8u * kMaxAccBufs;    // [2]
  const uint32_t qe0 = qf0 + 16u;                   // [2]
  const uint32_t drain_bar = qe0 + 16u;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- prologue: per-request tile counts, barriers, tensor memory --------
  constexpr int IS = MODE == kSample ? kFusedSampleStride : 1;  // items 0, IS, 2*IS, ... of every request
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const bool on = p.req_mask == nullptr || __ldg(p.req_mask + b) != 0u;
    const int64_t c = on ? clamp_ctx(__ldg(p.context_lens + b), p) : 0;
    const int64_t items = (c + ITEM - 1) / ITEM;
    tp[b + 1] = static_cast<int32_t>((items + IS - 1) / IS);
  }
  if (threadIdx.x == 0) {
    tp[0] = 0;
    misc[1] = 0u;
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full0 + 8u * s, GATHER ? 32u * kProdWarps : 1u);
      // MMA commit + the epilogue warps that read the stage's scales
      ptx::mbar_init(empty0 + 8u * s, 1u + 4u * (T > 1 ? kEpiGroups : 1));
    }
    for (int g = 0; g < AB; ++g) {
      ptx::mbar_init(accf0 + 8u * g, 1u);
      ptx::mbar_init(acce0 + 8u * g, 4u * (T > 1 ? kEpiGroups : 1));  // the epilogue warps that read it
    }
    for (int g = 0; g < 2; ++g) {
      ptx::mbar_init(qf0 + 8u * g, 1u);
      ptx::mbar_init(qe0 + 8u * g, 1u + 4u * kEpiGroups);  // MMA commit + every epilogue warp
    }
    ptx::mbar_init(drain_bar, 1u);
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    if (!GATHER) {
      ptx::prefetch_tmap(&tm_kv);
      ptx::prefetch_tmap(&tm_sc);
    }
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(misc), kTmemCols);
    ptx::tmem_relinquish();
  }
  __syncthreads();
  if (warp == 0) {  // inclusive scan of the tile counts
    int running = 0;
    for (int base = 0; base < B; base += 32) {
      const int idx = base + lane;
      int v = idx < B ? tp[idx + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (idx < B) tp[idx + 1] = running + v;
      running += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];

  const int total = tp[B];
  const int begin = static_cast<int>(static_cast<int64_t>(total) * blockIdx.x / gridDim.x);
  const int end = static_cast<int>(static_cast<int64_t>(total) * (blockIdx.x + 1) / gridDim.x);
  const int n_items = end - begin;
  ItemCursor cur{tp, B, 0, 0, 0};
  if (n_items > 0) cur.start(begin);

  if (warp < kProdWarps) {
    // =========================== producer ===============================
    Ring st{0u, 0u, static_cast<uint32_t>(S)};  // K ring
    Ring qr{0u, 0u, 2u};                          // Q/weight double buffer
    int issued = 0, q_issued = 0;
    int64_t ctx_eff = 0;
    if constexpr (!GATHER) {
      // With several producer warps each would take every kProdWarps-th item
      // and all walk every item to keep the ring and the block-table prefetch
      // in step; one warp is used (it also loads Q).
      const int pw = warp;              // 0 .. kProdWarps-1
      const int blk = p.block_size;     // 16, 32, 64 or 128
      const int P = ITEM / blk;         // cache blocks per item (divides 32)
      const uint32_t blk_bytes = static_cast<uint32_t>(blk) * (kHeadDim + 4);
      const uint32_t blk_k_bytes = static_cast<uint32_t>(blk) * kHeadDim;
      int chunk = 0, need_blocks = 0;
      int32_t tbl_cur = 0, tbl_nxt = 0;
      for (int it = 0; it < n_items; ++it) {
        if (it == 0 || cur.t == 0) {
          if (pw == 0) {
            if (!warp_wait_bounded(qe0 + 8u * qr.idx, qr.phase ^ 1u, abort_flag, &g_paged_watchdog, kSiteQEmpty))
              break;
            if (lane == 0) {
              const uint32_t qf = qf0 + 8u * qr.idx;
              ptx::mbar_arrive_expect_tx(qf, N * (kHeadDim + 4));
              ptx::tma_load_2d(ptx::smem_u32(q_s + qr.idx * N * kHeadDim), &tm_q, qf, 0, cur.b * N);
              ptx::bulk_g2s(ptx::smem_u32(w_s + qr.idx * N), p.weights + static_cast<int64_t>(cur.b) * N, N * 4, qf);
            }
            qr.next();
            ++q_issued;
          }
          ctx_eff = clamp_ctx(__ldg(p.context_lens + cur.b), p);
          need_blocks = static_cast<int>((ctx_eff + blk - 1) / blk);
        }
        const int rt = cur.t * IS;  // the item's index in its request
        const int first_blk = rt * P;
        if (it == 0 || cur.t == 0 || IS > 1) {  // (a sample jumps: reload the item's 32-block chunk)
          chunk = first_blk & ~31;
          tbl_cur = load_table(p, cur.b, chunk + lane, need_blocks);
          tbl_nxt = load_table(p, cur.b, chunk + 32 + lane, need_blocks);
        }
        const int32_t id = __shfl_sync(0xffffffffu, tbl_cur, (first_blk - chunk + lane) & 31);
        if (it % kProdWarps == pw) {
        if (!warp_wait_bounded(empty0 + 8u * st.idx, st.phase ^ 1u, abort_flag, &g_paged_watchdog, kSiteStageEmpty))
          break;
        const int valid = min(ITEM, static_cast<int>(ctx_eff - static_cast<int64_t>(rt) * ITEM));
        const int nblk = (valid + blk - 1) / blk;
        const uint32_t full = full0 + 8u * st.idx;
        if (lane == 0) ptx::mbar_arrive_expect_tx(full, nblk * blk_bytes);
        __syncwarp();
        if (lane < nblk) {
          const int32_t page = clamp_block(id, p.num_blocks);
          ptx::tma_load_3d(ptx::smem_u32(k_s + st.idx * stage_k + lane * blk_k_bytes), &tm_kv, full, 0, 0, page);
          // A tensor TMA needs a 128-byte-aligned destination: block sizes
          // >= 32 give one per block; block size 16 (64-byte scale runs)
          // uses the plain bulk copy, which needs only 16 bytes.
          if (blk >= 32)
            ptx::tma_load_2d(ptx::smem_u32(sc_s + st.idx * stage_sc + lane * blk), &tm_sc, full, 0, page);
          else
            ptx::bulk_g2s(ptx::smem_u32(sc_s + st.idx * stage_sc + lane * blk),
                          p.kv_cache + static_cast<int64_t>(page) * blk_bytes + blk_k_bytes, blk * 4, full);
        }
        issued = it + 1;
        }
        st.next();
        if (first_blk + P >= chunk + 32) {  // next tile starts a new 32-block chunk
          chunk += 32;
          tbl_cur = tbl_nxt;
          tbl_nxt = load_table(p, cur.b, chunk + 32 + lane, need_blocks);
        }
        cur.advance();
      }
      if (*abort_flag && lane == 0) {  // let issued copies land before the CTA exits
        for (int it = max(0, issued - S); it < issued; ++it)
          if (it % kProdWarps == pw) wait_drain(full0 + 8u * (it % S), (it / S) & 1, &g_paged_watchdog);
        for (int sg = max(0, q_issued - 2); sg < q_issued; ++sg)
          wait_drain(qf0 + 8u * (sg & 1), (sg >> 1) & 1, &g_paged_watchdog);
      }
    } else {
      // Block size 1: token p of request b is the 132-byte cache row
      // block_tables[b][p].  Producer warp w gathers tokens [64w, 64w+64) of
      // a tile, one token per instruction: lane l copies bytes [4l, 4l+4)
      // into the 128-byte-swizzled row; lane l also copies the scales of
      // tokens 64w+l and 64w+32+l.  Each lane turns its two table entries
      // into row addresses once (tokens past the window read row 0: in
      // bounds, and their logits are never stored), so a token costs a
      // shuffle of that address and one copy -- no per-token branch.
      // Copies are tracked per thread with cp.async groups; a tile is
      // published kLag tiles after it was issued.
      constexpr int kLag = 4;
      const int pw = warp;  // 0..1
      const auto row_addr = [&](int32_t slot) -> const uint8_t* {
        return p.kv_cache + static_cast<int64_t>(clamp_block(slot, p.num_blocks)) * (kHeadDim + 4);
      };
      const uint8_t *src_a = p.kv_cache, *src_b = p.kv_cache;
      // raw table entries of the next two tiles of the request: loaded two
      // tiles ahead and turned into addresses one tile ahead, so the load's
      // latency never stalls the copy issue
      int32_t raw1_a = 0, raw1_b = 0, raw2_a = 0, raw2_b = 0;
      // swizzled position of this lane's 4 bytes in a row whose (row & 7) is e
      uint32_t swz[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        swz[e] = ((static_cast<uint32_t>(lane >> 2) ^ static_cast<uint32_t>(e)) << 4) | (static_cast<uint32_t>(lane & 3) * 4u);
      int pending = 0;
      Ring pub{0u, 0u, static_cast<uint32_t>(S)};  // next stage to publish
      for (int it = 0; it < n_items; ++it) {
        if (it == 0 || cur.t == 0) {
          if (q_issued >= 2 && pending > 0) {
            // The Q buffer is freed only once the consumers finish request
            // q_issued-2, whose last tiles may still be among the deferred
            // arrivals: publish every tile in flight before waiting on it.
            ptx::cp_async_wait<0>();
            ptx::fence_proxy_async_smem();
            for (; pending > 0; --pending) {
              ptx::mbar_arrive(full0 + 8u * pub.idx);
              pub.next();
            }
          }
          if (!warp_wait_bounded(qe0 + 8u * qr.idx, qr.phase ^ 1u, abort_flag, &g_paged_watchdog, kSiteQEmpty))
            break;
          if (pw == 0 && lane == 0) {
            const uint32_t qf = qf0 + 8u * qr.idx;
            ptx::mbar_arrive_expect_tx(qf, N * (kHeadDim + 4));
            ptx::tma_load_2d(ptx::smem_u32(q_s + qr.idx * N * kHeadDim), &tm_q, qf, 0, cur.b * N);
            ptx::bulk_g2s(ptx::smem_u32(w_s + qr.idx * N), p.weights + static_cast<int64_t>(cur.b) * N, N * 4, qf);
          }
          qr.next();
          ++q_issued;
          ctx_eff = clamp_ctx(__ldg(p.context_lens + cur.b), p);
          const int64_t t0 = static_cast<int64_t>(cur.t) * IS * kTileTokens + pw * 64 + lane;
          src_a = row_addr(load_table(p, cur.b, t0, ctx_eff));
          src_b = row_addr(load_table(p, cur.b, t0 + 32, ctx_eff));
          if (cur.t + 1 < cur.tiles_b) {
            const int64_t t1 = t0 + static_cast<int64_t>(IS) * kTileTokens;
            raw1_a = load_table(p, cur.b, t1, ctx_eff);
            raw1_b = load_table(p, cur.b, t1 + 32, ctx_eff);
          }
        }
        if (cur.t + 2 < cur.tiles_b) {  // the rows two tiles ahead (same request only)
          const int64_t t2 = static_cast<int64_t>(cur.t + 2) * IS * kTileTokens + pw * 64 + lane;
          raw2_a = load_table(p, cur.b, t2, ctx_eff);
          raw2_b = load_table(p, cur.b, t2 + 32, ctx_eff);
        }
        if (!warp_wait_bounded(empty0 + 8u * st.idx, st.phase ^ 1u, abort_flag, &g_paged_watchdog, kSiteStageEmpty))
          break;
        const uint32_t tile_s = ptx::smem_u32(k_s + st.idx * kKTileBytes) + static_cast<uint32_t>(pw * 64 * kHeadDim);
#pragma unroll
        for (int j = 0; j < 64; ++j) {  // row (pw*64 + j) & 7 == j & 7
          const uint8_t* row = reinterpret_cast<const uint8_t*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(j < 32 ? src_a : src_b), j & 31));
          ptx::cp_async_4(tile_s + j * kHeadDim + swz[j & 7], row + lane * 4);
        }
        ptx::cp_async_4(ptx::smem_u32(sc_s + st.idx * kTileTokens + pw * 64 + lane), src_a + kHeadDim);
        ptx::cp_async_4(ptx::smem_u32(sc_s + st.idx * kTileTokens + pw * 64 + 32 + lane), src_b + kHeadDim);
        ptx::cp_async_commit();
        ++pending;
        st.next();
        issued = it + 1;
        if (pending > kLag) {  // the tile issued kLag tiles ago has landed
          ptx::cp_async_wait<kLag>();
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive(full0 + 8u * pub.idx);
          pub.next();
          --pending;
        }
        src_a = row_addr(raw1_a);  // (past the request's last tile: replaced at the next request)
        src_b = row_addr(raw1_b);
        raw1_a = raw2_a;
        raw1_b = raw2_b;
        cur.advance();
      }
      ptx::cp_async_wait<0>();
      ptx::fence_proxy_async_smem();
      for (; pending > 0; --pending) {
        ptx::mbar_arrive(full0 + 8u * pub.idx);
        pub.next();
      }
      if (*abort_flag && pw == 0 && lane == 0)
        for (int sg = max(0, q_issued - 2); sg < q_issued; ++sg)
          wait_drain(qf0 + 8u * (sg & 1), (sg >> 1) & 1, &g_paged_watchdog);
    }
  } else if (warp == kMmaWarp) {
    // ============================= MMA ==================================
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_e4m3_f32(kTileTokens, N);
      const uint64_t a_desc0 = ptx::smem_desc_sw128(ptx::smem_u32(k_s));
      const uint64_t b_desc0 = ptx::smem_desc_sw128(ptx::smem_u32(q_s));
      const uint64_t q_step = static_cast<uint64_t>((N * kHeadDim) >> 4);  // Q buffer stride, descriptor units
      Ring st{0u, 0u, static_cast<uint32_t>(S)};
      Ring ac{0u, 0u, static_cast<uint32_t>(AB)};
      Ring qr{0u, 0u, 2u};
      uint64_t b_desc = b_desc0;
      for (int it = 0; it < n_items; ++it) {
        if (it == 0 || cur.t == 0) {
          if (!wait_bounded(qf0 + 8u * qr.idx, qr.phase, abort_flag, &g_paged_watchdog, kSiteQFull)) break;
          b_desc = b_desc0 + qr.idx * q_step;
        }
        if (!wait_bounded(full0 + 8u * st.idx, st.phase, abort_flag, &g_paged_watchdog, kSiteStageFull)) break;
        if (!wait_bounded(acce0 + 8u * ac.idx, ac.phase ^ 1u, abort_flag, &g_paged_watchdog, kSiteAccEmpty)) break;
        ptx::tc_fence_after();
        for (int k = 0; k < T; ++k) {  // one 128-token tile per sub-tile, into its own TMEM columns
          const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(st.idx * T + k) * (kKTileBytes >> 4);
          const uint32_t d_tmem = tmem + ac.idx * acc_cols + k * sub_cols;
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 32; ++kk)  // K = 32 e4m3 per MMA: advance 32 bytes in the swizzled row
            ptx::mma_f8f6f4(d_tmem, a_desc + 2ull * kk, b_desc + 2ull * kk, idesc, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(empty0 + 8u * st.idx);
        ptx::mma_commit(accf0 + 8u * ac.idx);
        st.next();
        ac.next();
        if (cur.advance() || it + 1 == n_items) {
          ptx::mma_commit(qe0 + 8u * qr.idx);
          qr.next();
        }
      }
      if (*abort_flag) {
        ptx::mma_commit(drain_bar);
        wait_drain(drain_bar, 0, &g_paged_watchdog);
      }
    }
  } else {
    // =========================== epilogue ===============================
    // With two 128-token tiles per item both warpgroups work on every item,
    // group g on tile g, so an accumulator goes back to the MMA warp after
    // half the time.  With one tile per item the groups take alternate items
    // (all next_n rows each), which keeps the per-tile barrier traffic of a
    // wide accumulator at one round per group and tile.  The loop is
    // instantiated per chunk count (next_n * heads / 32).
    const int ew = warp - kEpiWarp0;   // 0 .. 4*kEpiGroups-1
    const int grp = ew >> 2;
    const int quad = warp & 3;         // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;  // token within the tile
    const int next_n = p.next_n;
    const auto run = [&](auto nchunks, auto shared) {
      constexpr int NCH = decltype(nchunks)::value;
      constexpr bool kShared = decltype(shared)::value != 0;
      const int k_tile = kShared ? grp : 0;
      const uint32_t col_off = static_cast<uint32_t>(k_tile) * sub_cols + (static_cast<uint32_t>(quad * 32) << 16);
      Ring st{0u, 0u, static_cast<uint32_t>(S)};
      Ring ac{0u, 0u, static_cast<uint32_t>(AB)};
      Ring qr{0u, 0u, 2u};
      int32_t ctx = 0;
      const float* w = w_s;
      // (FILTER) the thresholds of the current request's rows, in registers:
      // the emit below indexes them with compile-time row numbers
      constexpr int kRows = NCH / (HEADS / 32);
      float thr_r[kRows > 0 ? kRows : 1];
#pragma unroll
      for (int n = 0; n < kRows; ++n) thr_r[n] = 0.f;
      for (int it = 0; it < n_items; ++it) {
        if (it == 0 || cur.t == 0) {
          if (!warp_wait_bounded(qf0 + 8u * qr.idx, qr.phase, abort_flag, &g_paged_watchdog, kSiteQFull)) break;
          w = w_s + qr.idx * N;
          // the producers' clamped context: positions past what they loaded
          // are never stored, even for inputs that break the precondition
          ctx = static_cast<int32_t>(clamp_ctx(__ldg(p.context_lens + cur.b), p));
          if constexpr (FILTER) {
#pragma unroll
            for (int n = 0; n < kRows; ++n) thr_r[n] = __ldg(p.thr + static_cast<int64_t>(cur.b) * next_n + n);
          }
        }
        if (kShared || (it & 1) == grp) {
          if (!warp_wait_bounded(full0 + 8u * st.idx, st.phase, abort_flag, &g_paged_watchdog, kSiteStageFull))
            break;
          const float scale = sc_s[st.idx * stage_sc + k_tile * kTileTokens + row];
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(empty0 + 8u * st.idx);
          if (!warp_wait_bounded(accf0 + 8u * ac.idx, ac.phase, abort_flag, &g_paged_watchdog, kSiteAccFull)) break;
          ptx::tc_fence_after();
          // (32-bit: positions and context lengths are below 2^31)
          const int pos = cur.t * IS * ITEM + k_tile * kTileTokens + row;
          const int room = ctx - next_n - pos;  // row n is written iff n + room >= 0
          const bool in_model = pos < p.max_model_len;
          float* out_col = p.out + static_cast<int64_t>(cur.b) * next_n * p.out_stride + pos;
          const uint32_t acce = acce0 + 8u * ac.idx;
          reduce_rows<HEADS, NCH>(
              tmem + ac.idx * acc_cols + col_off, w,
              [&]() {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acce);
              },
              [&](int n, float v) {
                const bool in = n + room >= 0 && in_model;
                if constexpr (!FILTER) {
                  if (in) __stcs(out_col + static_cast<int64_t>(n) * p.out_stride, v * scale);
                } else {
                  // Candidates of row r: a logit at or above the row's
                  // threshold sets its bit in the row's bitmap, and a warp
                  // with any candidate stores all 32 of its logits (one whole
                  // 128-byte line: no partial-line writes).  A warp's 32
                  // tokens are one aligned 32-bit word of positions that no
                  // other warp covers, so lane 0 stores the warp's ballot as
                  // that word when it is not zero (the threshold pass
                  // cleared the bitmap over the window of every row it
                  // reads).
                  const float val = v * scale;
                  const bool cand = in && val >= thr_r[n];
                  const uint32_t m = __ballot_sync(0xffffffffu, cand);
                  if (m != 0u && in) __stcs(out_col + static_cast<int64_t>(n) * p.out_stride, val);
                  if (lane == 0 && m != 0u)
                    p.cand_bits[(static_cast<int64_t>(cur.b) * next_n + n) * p.bits_stride + (pos >> 5)] = m;
                }
              });
        }
        st.next();
        ac.next();
        if (cur.advance() || it + 1 == n_items) {
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(qe0 + 8u * qr.idx);
          qr.next();
        }
      }
    };
    const int nch = next_n * (HEADS / 32);
    if (T > 1)
      with_chunk_count<HEADS / 32, 4>(nch, [&](auto nc) { run(nc, IntC<1>{}); });
    else
      with_chunk_count<HEADS / 32, 8>(nch, [&](auto nc) { run(nc, IntC<0>{}); });
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

namespace {
using PagedKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, PagedParams);
template <int HEADS, int MODE>
PagedKernel paged_instance(bool gather) {
  return gather ? paged_logits_kernel<HEADS, true, MODE> : paged_logits_kernel<HEADS, false, MODE>;
}
template <int HEADS>
PagedKernel paged_instance(bool gather, int mode) {
  return mode == kFilter ? paged_instance<HEADS, kFilter>(gather)
         : mode == kSample ? paged_instance<HEADS, kSample>(gather)
                           : paged_instance<HEADS, kPlain>(gather);
}
}  // namespace

cudaError_t launch_paged(const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const CUtensorMap& tm_sc,
                         const PagedParams& p, int heads, bool gather, int grid, int smem_bytes, cudaStream_t stream,
                         int mode) {
  PagedKernel kern = nullptr;
  if (heads == 32)
    kern = paged_instance<32>(gather, mode);
  else if (heads == 64)
    kern = paged_instance<64>(gather, mode);
  else
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem_bytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, paged_threads(gather), smem_bytes, stream>>>(tm_q, tm_kv, tm_sc, p);
  return cudaGetLastError();
}

// Watchdog self-test: one warp initialises an mbarrier that nothing will
// ever arrive on and waits for it through the same bounded wait as the
// pipelines, with a short limit.  The wait runs out, sets the CTA's abort
// flag and the self-test bit of this translation unit's watchdog word, and
// the kernel returns.  No copy, MMA or tensor memory is involved.
__global__ void __launch_bounds__(32, 1) watchdog_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0u;
    ptx::mbar_init(ptx::smem_u32(&bar), 1u);
    ptx::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0)
    (void)wait_bounded(ptx::smem_u32(&bar), 0u, &abort_flag, &g_paged_watchdog, kSiteSelfTest, limit_ns);
  __syncwarp();
}

cudaError_t launch_watchdog_selftest(uint64_t limit_ns, cudaStream_t stream) {
  watchdog_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_paged_watchdog(unsigned int* value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_paged_watchdog, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_paged_watchdog, &zero, sizeof(unsigned int));
}

}  // namespace fp8idx
