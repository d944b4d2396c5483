// Prefill indexer logits (fp8_mqa_logits) for sm_103a.
//
// Defined by aiter PR 5046 "[HIP] [JIT] fp8_mqa_logits: hand-written gfx950
// prefill indexer kernel" (Motivation; Technical Details):
//   out[m, n] = sum_h relu(<Q[m,h,:], K[n,:]>) * kv_scale[n] * w[m,h]
//               for n in [ks[m], ke[m]) (clamped to [0, N)), -inf elsewhere,
// with every element written (the fused -inf fill of that PR).
//
// Design: persistent, one CTA per SM, warp-specialised like the decode kernel
// (producer warp, MMA warp, two epilogue warpgroups, -inf filler warp).
//  * A work unit is (row block, column split): block_m query rows whose Q
//    block [block_m*heads, 128] is the MMA B operand (N = block_m*heads, 256
//    at 32 heads), and the column tiles j = split_idx, split_idx + split, ...
//    (strided, so every unit has the same mix of computed and -inf tiles).
//    Units are ordered longest-first when `reverse` is set (row blocks from
//    the last one: under causal masking later rows have longer windows, same
//    PR, Technical Details) and dealt to CTAs round-robin.
//  * Per unit every role derives the union of the block's windows from
//    ks/ke; tiles meeting it are computed (TMA of K and its scales, four K=32
//    e4m3 tcgen05.mma into one of the TMEM accumulators), the others are
//    written with -inf.  Q and the weights (both by TMA) are double-buffered
//    across units.
//  * A filler warp writes the -inf tiles: TMA stores of a constant -inf tile
//    in shared memory (plain streaming stores when the output rows are not
//    16-byte aligned).  It waits on nothing, so the fill runs alongside the
//    MMA and the epilogue, and the producer warp only issues loads.
//  * The two epilogue warpgroups take alternate computed tiles.  A thread
//    owns one token: it reduces the accumulator's
//    32-column chunks (common.cuh reduce_rows, instantiated per chunk count
//    block_m*heads/32), scales by the token's kv_scale and stores the value
//    or -inf per element of the rows' windows.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8idx {

static __device__ unsigned int g_prefill_watchdog;

namespace {

struct Unit {
  int m0;      // first query row
  int sidx;    // column split index
  int n_j;     // column tiles of this unit
  int t_lo;    // union tile range [t_lo, t_hi) of computed tiles
  int t_hi;
  int j0;      // first computed tile of this unit
  int n_comp;  // computed tiles of this unit (j0, j0 + split, ...)
  int row_lo;  // this lane's row window (lanes < block_m), clamped; empty: 0,0
  int row_hi;
  int g_lo;    // paged K: output columns [g_lo, g_hi) covered by the computed tiles
  int g_hi;
};

// Paged K runs in a padded column space where every request starts on a
// tile boundary: request r owns padded tiles [tp[r], tp[r+1]), tile
// tp[r] + t holding its tokens [128t, 128t + 128), i.e. whole cache blocks.
// Largest r < n with a[r] <= v (a non-decreasing, a[0] <= v).
__device__ __forceinline__ int upper_index(const int32_t* a, int n, int64_t v) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= v) lo = mid; else hi = mid;
  }
  return lo;
}

// Warp-collective: unit u's geometry and window union.  Every lane gets the
// union; lane r < block_m also gets row r's window.
__device__ __forceinline__ Unit load_unit(const PrefillParams& p, int u, int num_rb, int n_tiles,
                                          const int32_t* cu = nullptr, const int32_t* tp = nullptr) {
  Unit U;
  const int lane = threadIdx.x & 31;
  const int rb_index = u / p.split;
  U.sidx = u - rb_index * p.split;
  const int rb = p.reverse ? (num_rb - 1 - rb_index) : rb_index;
  U.m0 = rb * p.block_m;
  U.n_j = (U.sidx < n_tiles) ? (n_tiles - U.sidx + p.split - 1) / p.split : 0;
  int rlo = 0, rhi = 0;
  const int m = U.m0 + lane;
  if (lane < p.block_m && m < p.rows) {
    const int ks = __ldg(p.ks + m), ke = __ldg(p.ke + m);
    rlo = ks < 0 ? 0 : ks;
    rhi = ke > p.cols ? p.cols : ke;
    if (rhi <= rlo) rlo = rhi = 0;
  }
  U.row_lo = rlo;
  U.row_hi = rhi;
  int lo = rhi > rlo ? rlo : p.cols;
  int hi = rhi > rlo ? rhi : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  U.t_lo = hi > lo ? lo / kTileTokens : 0;
  U.t_hi = hi > lo ? (hi + kTileTokens - 1) / kTileTokens : 0;
  U.g_lo = U.g_hi = 0;
  if (cu != nullptr && hi > lo) {  // paged: padded tiles of the first and last union columns
    const int ra = upper_index(cu, p.n_req, lo), rb2 = upper_index(cu, p.n_req, hi - 1);
    const int ta = (lo - cu[ra]) / kTileTokens, tb = (hi - 1 - cu[rb2]) / kTileTokens;
    U.t_lo = tp[ra] + ta;
    U.t_hi = tp[rb2] + tb + 1;
    U.g_lo = cu[ra] + ta * kTileTokens;
    U.g_hi = min(cu[rb2] + (tb + 1) * kTileTokens, cu[rb2 + 1]);
  }
  U.j0 = (U.t_lo <= U.sidx) ? U.sidx : U.sidx + ((U.t_lo - U.sidx + p.split - 1) / p.split) * p.split;
  U.n_comp = (U.t_hi > U.j0) ? (U.t_hi - U.j0 + p.split - 1) / p.split : 0;
  return U;
}

}  // namespace

// GATHER (paged K of block size 1 only): the producer gathers token rows
// with 4-byte copies instead of issuing one TMA per cache block; a separate
// instance, so that neither producer loop shapes the other's code.
template <int HEADS, bool PAGED, int DIM, bool GATHER>
__global__ void __launch_bounds__(prefill_threads(), 1)
    mqa_logits_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_out, const PrefillParams p) {
  constexpr int kEpiWarp0 = 2;
  constexpr int kFillWarp = kEpiWarp0 + 4 * kEpiGroups;
  constexpr uint32_t kTmemCols = 512;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_up_1024(smem_raw);
  const int N = p.n_cols;
  const int S = p.stages;
  const int BM = p.block_m;
  const int AB = p.acc_bufs;
  const uint32_t acc_cols = kTmemCols / AB;
  static_assert(DIM == 128 || DIM == 64, "head_dim 128 or 64");
  static_assert(PAGED || !GATHER, "the gather reads a paged cache");
  constexpr int kRow = DIM;                        // bytes per Q/K row
  constexpr int kTileB = kTileTokens * DIM;        // bytes per K tile
  const PrefillSmem L = prefill_smem_layout(N, S, PAGED ? 2 * (p.n_req + 1) : 0, DIM);
  uint8_t* q_s = smem + L.q;
  uint8_t* k_s = smem + L.k;
  float4* ninf_s = reinterpret_cast<float4*>(smem + L.ninf);
  float* sc_s = reinterpret_cast<float*>(smem + L.scale);
  float* w_s = reinterpret_cast<float*>(smem + L.w);
  int32_t* cu_s = reinterpret_cast<int32_t*>(smem + L.cu);  // paged: [n_req + 1] request offsets
  int32_t* tp_s = cu_s + (PAGED ? p.n_req + 1 : 0);          // paged: [n_req + 1] padded tile prefix
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
  const int num_rb = (p.rows + BM - 1) / BM;
  const int n_units = num_rb * p.split;

  if (threadIdx.x == 0) {
    misc[1] = 0u;
    for (int s = 0; s < S; ++s) {
      // TMA: one arrive with the byte count; token gather: every producer lane
      ptx::mbar_init(full0 + 8u * s, GATHER ? 32u : 1u);
      ptx::mbar_init(empty0 + 8u * s, 1u + 4u);  // MMA commit + the 4 warps that read the tile's scales
    }
    for (int g = 0; g < AB; ++g) {
      ptx::mbar_init(accf0 + 8u * g, 1u);
      ptx::mbar_init(acce0 + 8u * g, 4u);
    }
    for (int g = 0; g < 2; ++g) {
      ptx::mbar_init(qf0 + 8u * g, 1u);
      ptx::mbar_init(qe0 + 8u * g, 1u + 4u * kEpiGroups);  // MMA commit + every epilogue warp
    }
    ptx::mbar_init(drain_bar, 1u);
    ptx::fence_barrier_init();
    ptx::prefetch_tmap(&tm_q);
    if (!PAGED) {
      ptx::prefetch_tmap(&tm_k);
      ptx::prefetch_tmap(&tm_s);
    }
    ptx::prefetch_tmap(&tm_w);
    if (p.tma_fill) ptx::prefetch_tmap(&tm_out);
  }
  if (p.tma_fill) {  // the constant -inf tile read by the TMA stores
    for (int i = threadIdx.x; i < kNinfTileBytes / 16; i += blockDim.x)
      ninf_s[i] = make_float4(__int_as_float(0xff800000), __int_as_float(0xff800000), __int_as_float(0xff800000),
                              __int_as_float(0xff800000));
    ptx::fence_proxy_async_smem();
  }
  if (PAGED) {
    // Request offsets clamped into [0, N] and made non-decreasing (a running
    // maximum), so offsets that break the precondition cannot move a store
    // outside the output.
    for (int i = threadIdx.x; i <= p.n_req; i += blockDim.x)
      cu_s[i] = min(max(__ldg(p.cu_seq_lens + i), 0), p.cols);
    __syncthreads();
    if (warp == 0) {
      int carry = 0;
      for (int base = 0; base <= p.n_req; base += 32) {
        const int i = base + lane;
        int v = i <= p.n_req ? cu_s[i] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) v = max(v, __shfl_up_sync(0xffffffffu, v, o));
        v = max(v, carry);
        if (i <= p.n_req) cu_s[i] = v;
        carry = __shfl_sync(0xffffffffu, v, 31);
      }
      __syncwarp();
    }
    if (warp == 0) {  // padded tiles per request, inclusive scan
      if (lane == 0) tp_s[0] = 0;
      int running = 0;
      for (int base = 0; base < p.n_req; base += 32) {
        const int r = base + lane;
        int v = r < p.n_req ? (max(cu_s[r + 1] - cu_s[r], 0) + kTileTokens - 1) / kTileTokens : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += t;
        }
        if (r < p.n_req) tp_s[r + 1] = running + v;
        running += __shfl_sync(0xffffffffu, v, 31);
      }
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(misc), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const int n_tiles = PAGED ? tp_s[p.n_req] : (p.cols + kTileTokens - 1) / kTileTokens;
  const int32_t* const ucu = PAGED ? cu_s : nullptr;  // load_unit's paged mapping
  const int32_t* const utp = PAGED ? tp_s : nullptr;

  if (warp == 0) {
    // ============================ producer ==============================
    Ring st{0u, 0u, static_cast<uint32_t>(S)};
    Ring qr{0u, 0u, 2u};
    int issued = 0, q_issued = 0;
    bool ok = true;
    // Block size 1 (paged K as co-packed DIM+4-byte token rows, only 4-byte
    // aligned, so no TMA or 16-byte copy fits): the warp gathers each tile's
    // tokens with 4-byte cp.async into the swizzled layout the MMA reads
    // (128-byte swizzle: 16-byte chunk c of row j at chunk c ^ (j & 7);
    // 64-byte swizzle: c ^ ((j >> 1) & 3)), and publishes a tile kLag tiles
    // after issuing it (every lane arrives once its copies have landed).
    constexpr int kLag = 4;
    constexpr bool gather = GATHER;
    int pending = 0;
    Ring pub{0u, 0u, static_cast<uint32_t>(S)};
    const auto publish_all = [&]() {
      ptx::cp_async_wait<0>();
      ptx::fence_proxy_async_smem();
      for (; pending > 0; --pending) {
        ptx::mbar_arrive(full0 + 8u * pub.idx);
        pub.next();
      }
    };
    // Block size 1: this lane's block-table entries of a padded tile (its
    // tokens 32q + lane; raw, not yet clamped), loaded two computed tiles
    // ahead of their use so that the loads' latency never stalls the copy
    // issue.  (For larger blocks the same prefetch measured slower: their
    // producer issues one TMA per block and is not the bottleneck.)
    [[maybe_unused]] const auto tile_ids = [&](int j, int32_t (&e)[4]) {
      const int r = upper_index(tp_s, p.n_req, j);
      const int t = j - tp_s[r];
      const int len = cu_s[r + 1] - cu_s[r];
      const int32_t* bt_row = p.block_tables + static_cast<int64_t>(r) * p.bt_stride;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int tok = t * kTileTokens + 32 * q + lane;
        e[q] = tok < len ? __ldg(bt_row + min(tok, p.max_blocks - 1)) : 0;
      }
    };
    int32_t ids0[4] = {0, 0, 0, 0}, ids1[4] = {0, 0, 0, 0}, ids2[4] = {0, 0, 0, 0};
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit U = load_unit(p, u, num_rb, n_tiles, ucu, utp);
      if constexpr (gather) {
        if (U.n_comp > 0) tile_ids(U.j0, ids0);
        if (U.n_comp > 1) tile_ids(U.j0 + p.split, ids1);
      }
      // The Q buffer is freed once the MMA has consumed the unit before the
      // previous one, whose last tiles may still be unpublished.
      if (gather && pending > 0 && !__all_sync(0xffffffffu, ptx::mbar_test_wait(qe0 + 8u * qr.idx, qr.phase ^ 1u)))
        publish_all();
      if (!(ok = warp_wait_bounded(qe0 + 8u * qr.idx, qr.phase ^ 1u, abort_flag, &g_prefill_watchdog,
                                   kSiteQEmpty)))
        break;
      if (lane == 0) {
        const uint32_t qf = qf0 + 8u * qr.idx;
        ptx::mbar_arrive_expect_tx(qf, N * (kRow + 4));
        ptx::tma_load_2d(ptx::smem_u32(q_s + qr.idx * N * kRow), &tm_q, qf, 0, U.m0 * HEADS);
        ptx::tma_load_1d(ptx::smem_u32(w_s + qr.idx * N), &tm_w, qf, U.m0 * HEADS);
      }
      qr.next();
      ++q_issued;
      for (int c = 0, j = U.j0; c < U.n_comp; ++c, j += p.split) {
        if constexpr (gather) {
          if (c + 2 < U.n_comp) tile_ids(j + 2 * p.split, ids2);
        }
        if (!(ok = warp_wait_bounded(empty0 + 8u * st.idx, st.phase ^ 1u, abort_flag, &g_prefill_watchdog,
                                     kSiteStageEmpty)))
          break;
        if constexpr (!PAGED) {
          if (lane == 0) {
            const uint32_t full = full0 + 8u * st.idx;
            ptx::mbar_arrive_expect_tx(full, kTileB + kTileTokens * 4);
            ptx::tma_load_2d(ptx::smem_u32(k_s + st.idx * kTileB), &tm_k, full, 0, j * kTileTokens);
            ptx::tma_load_1d(ptx::smem_u32(sc_s + st.idx * kTileTokens), &tm_s, full, j * kTileTokens);
          }
        } else if constexpr (gather) {
          // Padded tile j: request r's tokens [128t, 128t + 128); token i's
          // row is block_tables[r][i] (tokens past the request read row 0,
          // in bounds, and are never stored); the entries were loaded two
          // tiles ago (tile_ids).
          const uint8_t* src[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            int32_t slot = ids0[q];
            slot = slot < 0 ? 0 : (slot >= p.num_blocks ? static_cast<int32_t>(p.num_blocks - 1) : slot);
            src[q] = p.kv_cache + static_cast<int64_t>(slot) * (DIM + 4);
          }
          const uint32_t tile_s = ptx::smem_u32(k_s + st.idx * kTileB);
          if constexpr (DIM == 128) {
            const uint32_t chunk = static_cast<uint32_t>(lane >> 2), inner = static_cast<uint32_t>(lane & 3) * 4u;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll 8
              for (int i = 0; i < 32; ++i) {
                const int row = 32 * q + i;
                const uint8_t* rp = reinterpret_cast<const uint8_t*>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(src[q]), i));
                ptx::cp_async_4(tile_s + row * DIM + (((chunk ^ static_cast<uint32_t>(row & 7)) << 4) | inner),
                                rp + lane * 4);
              }
            }
          } else {
            // 64-byte rows: lanes 0-15 copy token `row`, lanes 16-31 token row + 1
            const int hi = lane >> 4, l16 = lane & 15;
            const uint32_t chunk = static_cast<uint32_t>(l16 >> 2), inner = static_cast<uint32_t>(l16 & 3) * 4u;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll 8
              for (int i = 0; i < 32; i += 2) {
                const int row = 32 * q + i + hi;
                const uint8_t* rp = reinterpret_cast<const uint8_t*>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(src[q]), i + hi));
                ptx::cp_async_4(tile_s + row * DIM + (((chunk ^ static_cast<uint32_t>((row >> 1) & 3)) << 4) | inner),
                                rp + l16 * 4);
              }
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ptx::cp_async_4(ptx::smem_u32(sc_s + st.idx * kTileTokens + 32 * q + lane), src[q] + DIM);
          ptx::cp_async_commit();
          if (++pending > kLag) {  // the tile issued kLag tiles ago has landed
            ptx::cp_async_wait<kLag>();
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(full0 + 8u * pub.idx);
            pub.next();
            --pending;
          }
        } else {
          // Padded tile j: request r's tokens [128t, 128t + 128), whole cache
          // blocks: one 3-D TMA per block for its K rows and one copy of its
          // scales (2-D TMA, or a bulk copy for 16-token blocks whose 64-byte
          // scale runs are not 128-byte aligned in the stage).
          const int r = upper_index(tp_s, p.n_req, j);
          const int t = j - tp_s[r];
          const int len = cu_s[r + 1] - cu_s[r];
          const int valid = min(kTileTokens, len - t * kTileTokens);
          const int blk = p.block_size;
          const int nblk = (valid + blk - 1) / blk;
          const int fb = t * kTileTokens / blk;
          const uint32_t full = full0 + 8u * st.idx;
          if (lane == 0) ptx::mbar_arrive_expect_tx(full, nblk * blk * (DIM + 4));
          __syncwarp();
          if (lane < nblk) {
            int64_t b_id = __ldg(p.block_tables + static_cast<int64_t>(r) * p.bt_stride + min(fb + lane, p.max_blocks - 1));
            b_id = b_id < 0 ? 0 : (b_id >= p.num_blocks ? p.num_blocks - 1 : b_id);
            ptx::tma_load_3d(ptx::smem_u32(k_s + st.idx * kTileB + lane * blk * DIM), &tm_k, full, 0, 0,
                             static_cast<int32_t>(b_id));
            if (blk >= 32)
              ptx::tma_load_2d(ptx::smem_u32(sc_s + st.idx * kTileTokens + lane * blk), &tm_s, full, 0,
                               static_cast<int32_t>(b_id));
            else
              ptx::bulk_g2s(ptx::smem_u32(sc_s + st.idx * kTileTokens + lane * blk),
                            p.kv_cache + b_id * blk * (DIM + 4) + blk * DIM, blk * 4, full);
          }
        }
        st.next();
        ++issued;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          ids0[q] = ids1[q];
          ids1[q] = ids2[q];
        }
      }
    }
    if constexpr (gather) publish_all();  // (copies land before the CTA exits, abort or not)
    if (*abort_flag && lane == 0) {
      for (int c = max(0, issued - S); c < issued && !gather; ++c)
        wait_drain(full0 + 8u * (c % S), (c / S) & 1, &g_prefill_watchdog);
      for (int sg = max(0, q_issued - 2); sg < q_issued; ++sg)
        wait_drain(qf0 + 8u * (sg & 1), (sg >> 1) & 1, &g_prefill_watchdog);
    }
  } else if (warp == 1) {
    // ============================== MMA =================================
    const uint32_t idesc = ptx::idesc_e4m3_f32(kTileTokens, N);
    // 128-byte rows in the 128-byte swizzle, 64-byte rows in the 64-byte one
    const uint64_t a_desc0 = DIM == 128 ? ptx::smem_desc_sw128(ptx::smem_u32(k_s)) : ptx::smem_desc_sw64(ptx::smem_u32(k_s));
    const uint64_t b_desc0 = DIM == 128 ? ptx::smem_desc_sw128(ptx::smem_u32(q_s)) : ptx::smem_desc_sw64(ptx::smem_u32(q_s));
    const uint64_t q_step = static_cast<uint64_t>((N * kRow) >> 4);
    Ring st{0u, 0u, static_cast<uint32_t>(S)};
    Ring ac{0u, 0u, static_cast<uint32_t>(AB)};
    Ring qr{0u, 0u, 2u};
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit U = load_unit(p, u, num_rb, n_tiles, ucu, utp);
      if (lane == 0) {
        ok = wait_bounded(qf0 + 8u * qr.idx, qr.phase, abort_flag, &g_prefill_watchdog, kSiteQFull);
        const uint64_t b_desc = b_desc0 + qr.idx * q_step;
        for (int c = 0; c < U.n_comp && ok; ++c) {
          if (!(ok = wait_bounded(full0 + 8u * st.idx, st.phase, abort_flag, &g_prefill_watchdog, kSiteStageFull)))
            break;
          if (!(ok = wait_bounded(acce0 + 8u * ac.idx, ac.phase ^ 1u, abort_flag, &g_prefill_watchdog,
                                  kSiteAccEmpty)))
            break;
          ptx::tc_fence_after();
          const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(st.idx) * (kTileB >> 4);
          const uint32_t d_tmem = tmem + ac.idx * acc_cols;
#pragma unroll
          for (int kk = 0; kk < DIM / 32; ++kk)  // K = 32 e4m3 per MMA: 32 bytes into the swizzled row
            ptx::mma_f8f6f4(d_tmem, a_desc + 2ull * kk, b_desc + 2ull * kk, idesc, kk > 0 ? 1u : 0u);
          ptx::mma_commit(empty0 + 8u * st.idx);
          ptx::mma_commit(accf0 + 8u * ac.idx);
          st.next();
          ac.next();
        }
        if (ok) ptx::mma_commit(qe0 + 8u * qr.idx);
      }
      qr.next();
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0 && *abort_flag) {
      ptx::mma_commit(drain_bar);
      wait_drain(drain_bar, 0, &g_prefill_watchdog);
    }
  } else if (warp < kFillWarp) {
    // =========================== epilogue ===============================
    // Computed tile number ci (counted over the CTA) goes to accumulator
    // ci % AB and to warpgroup ci % 2.
    const int ew = warp - kEpiWarp0;      // 0 .. 4*kEpiGroups-1
    const int grp = ew >> 2;
    const int quad = warp & 3;            // TMEM lane quadrant
    const int row = quad * 32 + lane;     // token within the tile
    const float ninf = __int_as_float(0xff800000);
    // The loop is instantiated per chunk count (block_m * heads / 32).
    const auto run = [&](auto nchunks) {
      constexpr int NCH = decltype(nchunks)::value;
      Ring st{0u, 0u, static_cast<uint32_t>(S)};
      Ring ac{0u, 0u, static_cast<uint32_t>(AB)};
      Ring qr{0u, 0u, 2u};
      int ci = 0;
      bool ok = true;
      constexpr int kRows = NCH / (HEADS / 32);  // block_m
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit U = load_unit(p, u, num_rb, n_tiles, ucu, utp);
        // Every row's clamped window in registers for the whole unit (the
        // emit below indexes them with compile-time row numbers).
        int lo_r[kRows], hi_r[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          lo_r[r] = __shfl_sync(0xffffffffu, U.row_lo, r);
          hi_r[r] = __shfl_sync(0xffffffffu, U.row_hi, r);
        }
        const int rows_valid = p.rows - U.m0;  // rows r >= rows_valid lie past M
        float* const out_block = p.out + static_cast<int64_t>(U.m0) * p.out_stride;
        if (!(ok = warp_wait_bounded(qf0 + 8u * qr.idx, qr.phase, abort_flag, &g_prefill_watchdog, kSiteQFull)))
          break;
        const float* w = w_s + qr.idx * N;
        // Computed tiles j0, j0 + split, ...: alternate between the groups.
        for (int c = 0; c < U.n_comp; ++c) {
          const int col0 = (U.j0 + c * p.split) * kTileTokens;
          const bool mine = (ci & 1) == grp;
          ++ci;
          if (mine) {
            // the tile's output columns first: this work then overlaps the
            // waits instead of delaying the accumulator's release
            int n = col0 + row;
            bool col_ok = n < p.cols;
            if constexpr (PAGED) {  // padded tile -> the request's output columns; padding is not written
              const int j = U.j0 + c * p.split;
              const int r = upper_index(tp_s, p.n_req, j);
              const int local = (j - tp_s[r]) * kTileTokens + row;
              n = cu_s[r] + local;
              col_ok = local < cu_s[r + 1] - cu_s[r] && n < p.cols;
            }
            float* const out_col = out_block + n;
            if (!(ok = warp_wait_bounded(full0 + 8u * st.idx, st.phase, abort_flag, &g_prefill_watchdog,
                                         kSiteStageFull)))
              break;
            const float scale = sc_s[st.idx * kTileTokens + row];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty0 + 8u * st.idx);
            if (!(ok = warp_wait_bounded(accf0 + 8u * ac.idx, ac.phase, abort_flag, &g_prefill_watchdog,
                                         kSiteAccFull)))
              break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + ac.idx * acc_cols + (static_cast<uint32_t>(quad * 32) << 16);
            const uint32_t acce = acce0 + 8u * ac.idx;
            reduce_rows<HEADS, NCH>(
                taddr, w,
                [&]() {
                  ptx::tc_fence_before();
                  __syncwarp();
                  if (lane == 0) ptx::mbar_arrive(acce);
                },
                [&](int r, float v) {
                  const bool inside = n >= lo_r[r] && n < hi_r[r];
                  if (r < rows_valid && col_ok && (inside || p.clean))
                    __stcs(out_col + static_cast<int64_t>(r) * p.out_stride, inside ? v * scale : ninf);
                });
          }
          st.next();
          ac.next();
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(qe0 + 8u * qr.idx);
        qr.next();
      }
    };
    with_chunk_count<HEADS / 32, 8>(BM * (HEADS / 32), run);
  } else {
    // ============================ -inf filler ===========================
    // Every unit's column tiles that meet no row's window (k < k_lo or
    // k >= k_lo + n_comp) get -inf.  The filler shares no data with the
    // other roles (disjoint output elements) and waits on nothing, so it
    // runs ahead freely.  With tma_fill lane 0 issues one TMA store of the
    // constant -inf tile per column tile (the tensor map covers N rounded
    // down to whole 16-byte units, since a TMA store writes whole 16-byte
    // units; the lanes write the last tile's remaining columns directly);
    // otherwise the lanes write streaming stores (float4 where aligned).
    const float ninf = __int_as_float(0xff800000);
    const float4 f4 = make_float4(ninf, ninf, ninf, ninf);
    const int tail = p.cols - p.fill_cols;
    for (int u = blockIdx.x; PAGED && u < n_units && p.clean; u += gridDim.x) {
      // paged: -inf on [0, g_lo) and [g_hi, N), the columns outside the
      // computed tiles, per 128-column output tile: a TMA store when the
      // whole tile is outside, lane stores for the outside part otherwise
      const Unit U = load_unit(p, u, num_rb, n_tiles, ucu, utp);
      const int rv = min(BM, p.rows - U.m0);
      float* const out_block = p.out + static_cast<int64_t>(U.m0) * p.out_stride;
      const int n_out_tiles = (p.cols + kTileTokens - 1) / kTileTokens;
      // The union range [g_lo, g_hi) is the same for every split of a row
      // block and is exactly covered by the computed tiles of all its
      // splits; the splits share the rest by output tile index.
      for (int k = U.sidx; k < n_out_tiles; k += p.split) {
        const int c0 = k * kTileTokens, c1 = min(c0 + kTileTokens, p.cols);
        const bool outside = c1 <= U.g_lo || c0 >= U.g_hi;
        if (outside && p.tma_fill) {
          if (lane == 0) ptx::tma_store_2d(&tm_out, ptx::smem_u32(ninf_s), c0, U.m0);
          if (tail > 0 && c0 + kTileTokens > p.fill_cols && lane < rv * tail) {
            const int r = lane / tail;
            out_block[static_cast<int64_t>(r) * p.out_stride + p.fill_cols + (lane - r * tail)] = ninf;
          }
        } else if (c0 < U.g_lo || c1 > U.g_hi) {
          for (int e = lane; e < rv * kTileTokens; e += 32) {
            const int r = e / kTileTokens, col = c0 + (e - r * kTileTokens);
            if (col < c1 && (col < U.g_lo || col >= U.g_hi))
              __stcs(out_block + static_cast<int64_t>(r) * p.out_stride + col, ninf);
          }
        }
      }
      if (p.tma_fill && lane == 0) ptx::bulk_commit_group();
    }
    for (int u = blockIdx.x; !PAGED && u < n_units && p.clean; u += gridDim.x) {
      const Unit U = load_unit(p, u, num_rb, n_tiles, ucu, utp);
      const int k_lo = (U.j0 - U.sidx) / p.split;
      const int n_inf = U.n_j - U.n_comp;
      const int rv = min(BM, p.rows - U.m0);
      float* const out_block = p.out + static_cast<int64_t>(U.m0) * p.out_stride;
      for (int f = 0; f < n_inf; ++f) {
        const int k = f < k_lo ? f : f + U.n_comp;
        const int col0 = (U.sidx + k * p.split) * kTileTokens;
        if (p.tma_fill) {
          if (lane == 0) ptx::tma_store_2d(&tm_out, ptx::smem_u32(ninf_s), col0, U.m0);
          if (tail > 0 && col0 + kTileTokens > p.fill_cols && lane < rv * tail) {
            const int r = lane / tail;
            out_block[static_cast<int64_t>(r) * p.out_stride + p.fill_cols + (lane - r * tail)] = ninf;
          }
        } else {
          const int c4 = col0 + lane * 4;
          for (int r = 0; r < rv; ++r) {
            float* const dst = out_block + static_cast<int64_t>(r) * p.out_stride + c4;
            if (p.vec_ok && c4 + 4 <= p.cols) {
              __stcs(reinterpret_cast<float4*>(dst), f4);
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (c4 + i < p.cols) __stcs(dst + i, ninf);
            }
          }
        }
      }
      if (p.tma_fill && lane == 0) ptx::bulk_commit_group();
    }
    // The TMA stores read the constant tile until they complete: wait for
    // them before the CTA (and its shared memory) goes away.
    if (p.tma_fill && lane == 0) ptx::bulk_wait_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t launch_prefill(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_s,
                           const CUtensorMap& tm_w, const CUtensorMap& tm_out, const PrefillParams& p, int heads,
                           int head_dim, bool paged, int grid, int smem_bytes, cudaStream_t stream) {
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, PrefillParams) = nullptr;
  const bool gather = paged && p.block_size == 1;
  const auto pick = [&](auto heads_c, auto dim_c) {
    constexpr int H = decltype(heads_c)::value, D = decltype(dim_c)::value;
    kern = !paged ? mqa_logits_kernel<H, false, D, false>
                  : (gather ? mqa_logits_kernel<H, true, D, true> : mqa_logits_kernel<H, true, D, false>);
  };
  const auto pick_heads = [&](auto dim_c) {
    if (heads == 32) pick(IntC<32>{}, dim_c);
    else if (heads == 64) pick(IntC<64>{}, dim_c);
    else if (heads == 128) pick(IntC<128>{}, dim_c);
  };
  if (head_dim == 128) pick_heads(IntC<128>{});
  else if (head_dim == 64) pick_heads(IntC<64>{});
  if (kern == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem_bytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, prefill_threads(), smem_bytes, stream>>>(tm_q, tm_k, tm_s, tm_w, tm_out, p);
  return cudaGetLastError();
}

cudaError_t read_prefill_watchdog(unsigned int* value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_prefill_watchdog, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_prefill_watchdog, &zero, sizeof(unsigned int));
}

}  // namespace fp8idx
