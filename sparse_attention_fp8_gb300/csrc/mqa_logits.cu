// Prefill indexer logits (fp8_mqa_logits) for sm_103a.
//
// Defined by aiter PR 5046 "[HIP] [JIT] fp8_mqa_logits: hand-written gfx950
// prefill indexer kernel" (Motivation; Technical Details):
//   out[m, n] = sum_h relu(<Q[m,h,:], K[n,:]>) * kv_scale[n] * w[m,h]
//               for n in [ks[m], ke[m]) (clamped to [0, N)), -inf elsewhere,
// every element written (the fused -inf fill of that PR).
//
// Design: one CTA per (row block, column split); two CTAs share an SM so one
// CTA's epilogue overlaps the other's MMA and loads.
//  * A row block is block_m query rows; its Q block [block_m*heads, 128]
//    stays resident in shared memory as the MMA B operand (N = block_m*heads,
//    256 at 32 heads), so one K tile feeds every row of the block.
//  * Column tiles of 128 tokens are split across `split` CTAs in a strided
//    way (CTA s takes tiles s, s+split, ...), which gives every CTA the same
//    mix of computed and pure -inf tiles.
//  * Tiles that meet the union of the block's windows are computed: TMA of
//    the K tile (128-byte swizzle) and its 128 scales, four K=32 e4m3
//    tcgen05.mma into a TMEM accumulator, then the epilogue (thread = token)
//    applies ReLU * weight, sums the heads, multiplies by the token's scale
//    and stores each row's value or -inf (outside that row's own window).
//  * Tiles outside the union are written with -inf directly (float4 stores).
//  * Row blocks are dispatched from the last one when `reverse` is set: under
//    causal masking later rows have longer windows, so the long CTAs start
//    first and short ones fill in behind (same PR, Technical Details).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8idx {

static __device__ unsigned int g_prefill_watchdog;

template <int HEADS>
__global__ void __launch_bounds__(prefill_threads(), 2)
    mqa_logits_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_s, const PrefillParams p) {
  constexpr int kEpiWarp0 = 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_up_1024(smem_raw);
  const int N = p.n_cols;
  const int S = p.stages;
  const int BM = p.block_m;
  const PrefillSmem L = prefill_smem_layout(N, S, BM);
  uint8_t* q_s = smem + L.q;
  uint8_t* k_s = smem + L.k;
  float* sc_s = reinterpret_cast<float*>(smem + L.scale);
  float* w_s = reinterpret_cast<float*>(smem + L.w);
  int32_t* row_lo = reinterpret_cast<int32_t*>(smem + L.rows);
  int32_t* row_hi = row_lo + BM;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile uint32_t* abort_flag = misc + 1;

  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * S;
  const uint32_t accf = empty0 + 8u * S;
  const uint32_t acce = accf + 8u;
  const uint32_t drain_bar = acce + 8u;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_rb = (p.rows + BM - 1) / BM;
  const int rb_index = blockIdx.x / p.split;
  const int sidx = blockIdx.x % p.split;
  const int rb = p.reverse ? (num_rb - 1 - rb_index) : rb_index;
  const int m0 = rb * BM;
  const int n_tiles = (p.cols + kTileTokens - 1) / kTileTokens;
  const uint32_t tmem_cols = static_cast<uint32_t>(p.acc_cols);

  // ---- prologue ----------------------------------------------------------
  if (warp == 0) {
    // per-row clamped windows [lo, hi); empty rows get lo = hi = 0
    int lo = p.cols, hi = 0;
    if (lane < BM) {
      const int m = m0 + lane;
      int rlo = 0, rhi = 0;
      if (m < p.rows) {
        const int ks = __ldg(p.ks + m), ke = __ldg(p.ke + m);
        rlo = ks < 0 ? 0 : ks;
        rhi = ke > p.cols ? p.cols : ke;
        if (rhi <= rlo) rlo = rhi = 0;
      }
      row_lo[lane] = rlo;
      row_hi[lane] = rhi;
      if (rhi > rlo) { lo = rlo; hi = rhi; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      // union tile range [t_lo, t_hi) of computed tiles
      misc[2] = hi > lo ? static_cast<uint32_t>(lo / kTileTokens) : 0u;
      misc[3] = hi > lo ? static_cast<uint32_t>((hi + kTileTokens - 1) / kTileTokens) : 0u;
      misc[1] = 0u;
      for (int s = 0; s < S; ++s) {
        ptx::mbar_init(full0 + 8u * s, 1u);
        ptx::mbar_init(empty0 + 8u * s, 1u + 4u);
      }
      ptx::mbar_init(accf, 1u);
      ptx::mbar_init(acce, 4u);
      ptx::mbar_init(drain_bar, 1u);
      ptx::fence_barrier_init();
      ptx::prefetch_tmap(&tm_q);
      ptx::prefetch_tmap(&tm_k);
      ptx::prefetch_tmap(&tm_s);
    }
  } else if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(misc), tmem_cols);
    ptx::tmem_relinquish();
  } else {
    // weights of the block's rows (zero for rows past M)
    for (int i = threadIdx.x - 32 * kEpiWarp0; i < N; i += 128) {
      const int m = m0 + i / HEADS;
      w_s[i] = (m < p.rows) ? __ldg(p.weights + static_cast<int64_t>(m0) * HEADS + i) : 0.f;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  const int t_lo = static_cast<int>(misc[2]);
  const int t_hi = static_cast<int>(misc[3]);
  // computed tiles of this CTA: j = sidx + k*split with t_lo <= j < t_hi
  const int c_first = (t_lo <= sidx) ? sidx : sidx + ((t_lo - sidx + p.split - 1) / p.split) * p.split;
  const int n_comp = (t_hi > c_first) ? (t_hi - c_first + p.split - 1) / p.split : 0;

  if (warp == 0) {
    // ============================ producer ==============================
    if (lane == 0 && n_comp > 0) {
      // Q block: rows [m0*HEADS, m0*HEADS + N) of the [M*heads, 128] view; counted on stage 0's barrier
      int issued = 0;
      for (int c = 0; c < n_comp; ++c) {
        const int s = c % S;
        if (!wait_bounded(empty0 + 8u * s, ((c / S) & 1) ^ 1, abort_flag, &g_prefill_watchdog, kSiteStageEmpty))
          break;
        const uint32_t full = full0 + 8u * s;
        const int j = c_first + c * p.split;
        const uint32_t bytes = kKTileBytes + kTileTokens * 4 + (c == 0 ? N * kHeadDim : 0);
        ptx::mbar_arrive_expect_tx(full, bytes);
        if (c == 0) ptx::tma_load_2d(ptx::smem_u32(q_s), &tm_q, full, 0, m0 * HEADS);
        ptx::tma_load_2d(ptx::smem_u32(k_s + s * kKTileBytes), &tm_k, full, 0, j * kTileTokens);
        ptx::tma_load_1d(ptx::smem_u32(sc_s + s * kTileTokens), &tm_s, full, j * kTileTokens);
        issued = c + 1;
      }
      if (*abort_flag)
        for (int c = max(0, issued - S); c < issued; ++c)
          wait_drain(full0 + 8u * (c % S), (c / S) & 1, &g_prefill_watchdog);
    }
  } else if (warp == 1) {
    // ============================== MMA =================================
    if (lane == 0 && n_comp > 0) {
      const uint32_t idesc = ptx::idesc_e4m3_f32(kTileTokens, N);
      const uint64_t b_desc = ptx::smem_desc_sw128(ptx::smem_u32(q_s));
      for (int c = 0; c < n_comp; ++c) {
        const int s = c % S;
        if (!wait_bounded(full0 + 8u * s, (c / S) & 1, abort_flag, &g_prefill_watchdog, kSiteStageFull)) break;
        if (!wait_bounded(acce, (c & 1) ^ 1, abort_flag, &g_prefill_watchdog, kSiteAccEmpty)) break;
        ptx::tc_fence_after();
        const uint64_t a_desc = ptx::smem_desc_sw128(ptx::smem_u32(k_s + s * kKTileBytes));
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 32; ++kk)
          ptx::mma_f8f6f4(tmem, a_desc + 2ull * kk, b_desc + 2ull * kk, idesc, kk > 0 ? 1u : 0u);
        ptx::mma_commit(empty0 + 8u * s);
        ptx::mma_commit(accf);
      }
      if (*abort_flag) {
        ptx::mma_commit(drain_bar);
        wait_drain(drain_bar, 0, &g_prefill_watchdog);
      }
    }
  } else {
    // =========================== epilogue ===============================
    const int et = threadIdx.x - 32 * kEpiWarp0;  // 0..127
    const int quad = warp & 3;
    const int row = quad * 32 + lane;             // token within the tile
    const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float ninf = __int_as_float(0xff800000);
    int c = 0;  // computed-tile counter
    for (int j = sidx; j < n_tiles; j += p.split) {
      const int col0 = j * kTileTokens;
      if (j >= t_lo && j < t_hi) {
        const int s = c % S;
        if (!warp_wait_bounded(accf, c & 1, abort_flag, &g_prefill_watchdog, kSiteAccFull)) break;
        ptx::tc_fence_after();
        if (!warp_wait_bounded(full0 + 8u * s, (c / S) & 1, abort_flag, &g_prefill_watchdog, kSiteStageFull)) break;
        const float scale = sc_s[s * kTileTokens + row];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty0 + 8u * s);
        const int n = col0 + row;
        for (int r = 0; r < BM; ++r) {
          float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int hc = 0; hc < HEADS / 32; ++hc) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tbase + r * HEADS + hc * 32, v);
            ptx::tmem_wait_ld();
            relu_dot32(v, w_s + r * HEADS + hc * 32, a0, a1);
          }
          const int m = m0 + r;
          if (m < p.rows && n < p.cols) {
            const float logit = ((a0.x + a0.y) + (a1.x + a1.y)) * scale;
            const bool inside = n >= row_lo[r] && n < row_hi[r];
            __stcs(p.out + static_cast<int64_t>(m) * p.out_stride + n, inside ? logit : ninf);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(acce);
        ++c;
      } else {
        // pure -inf tile: rows of this block x 128 columns
        const int ncols = min(kTileTokens, p.cols - col0);
        if (p.vec_ok && ncols == kTileTokens) {
          const float4 f4 = make_float4(ninf, ninf, ninf, ninf);
          for (int e = et; e < BM * 32; e += 128) {
            const int r = e >> 5, c4 = e & 31;
            if (m0 + r < p.rows)
              __stcs(reinterpret_cast<float4*>(p.out + static_cast<int64_t>(m0 + r) * p.out_stride + col0) + c4, f4);
          }
        } else {
          for (int r = 0; r < BM; ++r)
            if (m0 + r < p.rows && row < ncols)
              __stcs(p.out + static_cast<int64_t>(m0 + r) * p.out_stride + col0 + row, ninf);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, tmem_cols);
  }
}

cudaError_t launch_prefill(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_s,
                           const PrefillParams& p, int heads, int grid, int smem_bytes, cudaStream_t stream) {
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, PrefillParams) = nullptr;
  if (heads == 32) kern = mqa_logits_kernel<32>;
  else if (heads == 64) kern = mqa_logits_kernel<64>;
  else return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, prefill_threads(), smem_bytes, stream>>>(tm_q, tm_k, tm_s, p);
  return cudaGetLastError();
}

cudaError_t read_prefill_watchdog(unsigned int* value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_prefill_watchdog, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_prefill_watchdog, &zero, sizeof(unsigned int));
}

}  // namespace fp8idx
