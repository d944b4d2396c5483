// Device-side pieces shared by the decode and prefill kernels: bounded
// mbarrier waits (every pipeline wait gives up after kWaitTimeoutNs, sets the
// CTA's abort flag and a bit in the translation unit's watchdog word, so a
// broken pipeline ends the kernel instead of hanging the GPU), and the
// ReLU * weight head-reduction over one 32-column TMEM chunk.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace fp8idx {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s: no legitimate wait comes close
constexpr uint64_t kDrainTimeoutNs = 200000000ull;  // 0.2 s: waiting out in-flight copies after an abort

// Watchdog bit per wait site (reported through fp8idx_device_status).
enum WaitSite : uint32_t {
  kSiteQEmpty = 1u << 0,
  kSiteStageEmpty = 1u << 1,
  kSiteQFull = 1u << 2,
  kSiteStageFull = 1u << 3,
  kSiteAccEmpty = 1u << 4,
  kSiteAccFull = 1u << 5,
  kSiteDrain = 1u << 6,
  kSiteSelfTest = 1u << 7,  // the watchdog self-test's deliberately unsatisfied wait
};

// Polls `bar` for the phase with parity `parity`.  Returns false if the CTA
// has aborted or the wait ran out after `limit_ns` (then it aborts the CTA
// and flags `wd`).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             unsigned int* wd, uint32_t site,
                                             uint64_t limit_ns = kWaitTimeoutNs) {
  if (ptx::mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1u;
      atomicOr(wd, site);
      return false;
    }
  }
}

// Waits out a phase after an abort (copies already issued must land before
// the CTA's shared memory is released).  Ignores the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned int* wd) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity, 100000u)) {
    if (ptx::globaltimer_ns() - t0 > kDrainTimeoutNs) {
      atomicOr(wd, static_cast<uint32_t>(kSiteDrain));
      return;
    }
  }
}

// One warp-collective bounded wait.  Fast path: every lane tests the phase
// and the warp votes (a completed phase cannot be overtaken before this
// warp's own later arrivals, so the lanes agree).  Slow path: lane 0 polls,
// the verdict is broadcast.
__device__ __forceinline__ bool warp_wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                  unsigned int* wd, uint32_t site) {
  if (__all_sync(0xffffffffu, ptx::mbar_test_wait(bar, parity))) return true;
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_bounded(bar, parity, abort_flag, wd, site) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Index and phase of a ring of `n` mbarrier-guarded slots, advanced by one
// slot per use (no division on the per-tile path).
struct Ring {
  uint32_t idx, phase, n;
  __device__ __forceinline__ void next() {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// One 32-column TMEM chunk in registers, with its 32 weights in registers,
// reduced into two float2 accumulators.  x + |x| = 2 * relu(x) exactly, and
// doubling commutes with rounding, so every form below yields the same bits
// once relu_dot_total applies its factor of 1/2.
//  * PACKED: every ReLU as a packed x + |x| (one f32x2 add per pair), then a
//    packed FMA with the weights: acc0/acc1 hold 2 * sum relu(x) * w.
//  * otherwise: half of the ReLUs as max(x, 0) on the ALU pipe (acc0 holds
//    sum relu(x) * w) and half as x + |x| on the FMA pipe (acc1 holds twice
//    its sum), which balances the two pipes.
// Which one is faster depends on the head count (measured: packed for 32
// heads, mixed for 64).
template <bool PACKED>
__device__ __forceinline__ void relu_dot32(const uint32_t (&r)[32], const float4 (&wv)[8], float2& acc0,
                                           float2& acc1) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float x0 = __uint_as_float(r[4 * j + 0]), x1 = __uint_as_float(r[4 * j + 1]);
    const float x2 = __uint_as_float(r[4 * j + 2]), x3 = __uint_as_float(r[4 * j + 3]);
    if constexpr (PACKED) {
      const float2 r01 = __fadd2_rn(make_float2(x0, x1), make_float2(fabsf(x0), fabsf(x1)));
      const float2 r23 = __fadd2_rn(make_float2(x2, x3), make_float2(fabsf(x2), fabsf(x3)));
      acc0 = __ffma2_rn(r01, make_float2(wv[j].x, wv[j].y), acc0);
      acc1 = __ffma2_rn(r23, make_float2(wv[j].z, wv[j].w), acc1);
    } else {
      acc0 = __ffma2_rn(make_float2(fmaxf(x0, 0.f), fmaxf(x1, 0.f)), make_float2(wv[j].x, wv[j].y), acc0);
      acc1 = __ffma2_rn(make_float2(x2 + fabsf(x2), x3 + fabsf(x3)), make_float2(wv[j].z, wv[j].w), acc1);
    }
  }
}

template <bool PACKED>
__device__ __forceinline__ float relu_dot_total(float2 acc0, float2 acc1) {
  if constexpr (PACKED)
    return 0.5f * ((acc0.x + acc0.y) + (acc1.x + acc1.y));
  else
    return (acc0.x + acc0.y) + 0.5f * (acc1.x + acc1.y);
}

// First chunk of round k when NB chunk buffers rotate: one chunk per round
// with 2 buffers, rounds of 2 and 1 chunks alternating with 3, two with 4.
template <int NB>
__host__ __device__ constexpr int round_start(int k) {
  return NB == 2 ? k : NB == 3 ? (3 * k + 1) / 2 : 2 * k;
}

// The epilogue's TMEM-to-register reduction for one tile and one thread's
// token: output row k (k < NCH * 32 / HEADS) is
//   sum_h relu(acc[k*HEADS + h]) * w[k*HEADS + h]
// over the NCH 32-column chunks starting at TMEM address `taddr`.  The chunk
// count is a template parameter so the loop is straight-line code.  Chunks
// rotate through NB register buffers (chunk c in buffer c % NB).  Because
// tcgen05.wait::ld waits for every outstanding load, the work is cut into
// rounds: wait for the round's chunks, issue the next round's loads into the
// free buffers, then reduce the round's chunks (weights read from shared
// memory, a broadcast) while those loads are in flight.  Once the last load
// has landed `release()` hands the accumulator back to the MMA warp;
// `emit(k, sum)` receives each row.  NB (measured): 4 for six or more chunks
// of 32 heads, else 3 (2 for a single chunk).
template <int HEADS, int NCH, class Release, class Emit>
__device__ __forceinline__ void reduce_rows(uint32_t taddr, const float* w, Release release, Emit emit) {
  constexpr int kChunksPerRow = HEADS / 32;
  constexpr bool kPacked = HEADS == 32;
  constexpr int NB = (HEADS == 32 && NCH >= 6) ? 4 : NCH >= 2 ? 3 : 2;
  static_assert(NCH >= 0 && NCH % kChunksPerRow == 0, "whole rows");
  if constexpr (NCH == 0) {
    release();
  } else {
    uint32_t r[NB][32];
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < round_start<NB>(1) && c < NCH; ++c) ptx::tmem_ld_32x32b_x32(taddr + c * 32, r[c % NB]);
#pragma unroll
    for (int k = 0; round_start<NB>(k) < NCH; ++k) {
      const int s0 = round_start<NB>(k);
      const int e0 = round_start<NB>(k + 1) < NCH ? round_start<NB>(k + 1) : NCH;
      const int e1 = round_start<NB>(k + 2) < NCH ? round_start<NB>(k + 2) : NCH;
      ptx::tmem_wait_ld_regs(r[s0 % NB]);
      if (e0 - s0 > 1) ptx::reg_fence(r[(s0 + 1) % NB]);
      if (e0 < NCH) {
#pragma unroll
        for (int c = e0; c < e1; ++c) ptx::tmem_ld_32x32b_x32(taddr + c * 32, r[c % NB]);
      } else {
        release();
      }
#pragma unroll
      for (int c = s0; c < e0; ++c) {
        float4 wv[8];
        const float4* w4 = reinterpret_cast<const float4*>(w + c * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j) wv[j] = w4[j];
        relu_dot32<kPacked>(r[c % NB], wv, a0, a1);
        if ((c + 1) % kChunksPerRow == 0) {
          emit(c / kChunksPerRow, relu_dot_total<kPacked>(a0, a1));
          a0 = make_float2(0.f, 0.f);
          a1 = make_float2(0.f, 0.f);
        }
      }
    }
  }
}

template <int N>
struct IntC {
  static constexpr int value = N;
};

// Calls f(IntC<n>{}) for the runtime chunk count n, 1 <= n <= MAX (n a
// multiple of STEP); the per-count code is instantiated once per kernel.
template <int STEP, int MAX, class F>
__device__ __forceinline__ void with_chunk_count(int n, F f) {
  static_assert(MAX <= 8, "at most 8 chunks (256 columns)");
  switch (n) {
    case 1: if constexpr (1 % STEP == 0 && MAX >= 1) f(IntC<1>{}); break;
    case 2: if constexpr (2 % STEP == 0 && MAX >= 2) f(IntC<2>{}); break;
    case 3: if constexpr (3 % STEP == 0 && MAX >= 3) f(IntC<3>{}); break;
    case 4: if constexpr (4 % STEP == 0 && MAX >= 4) f(IntC<4>{}); break;
    case 5: if constexpr (5 % STEP == 0 && MAX >= 5) f(IntC<5>{}); break;
    case 6: if constexpr (6 % STEP == 0 && MAX >= 6) f(IntC<6>{}); break;
    case 7: if constexpr (7 % STEP == 0 && MAX >= 7) f(IntC<7>{}); break;
    case 8: if constexpr (8 % STEP == 0 && MAX >= 8) f(IntC<8>{}); break;
    default: break;
  }
}

__device__ __forceinline__ uint8_t* align_up_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

}  // namespace fp8idx
