// Kernel parameter blocks, shared-memory layouts and launchers shared by the
// host API (api.cpp) and the kernel translation units.  Host and device both
// size shared memory with the functions below, so they cannot disagree.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8idx {

constexpr int kHeadDim = 128;     // bytes per e4m3 K/Q row
constexpr int kTileTokens = 128;  // KV tokens per MMA tile (MMA M)
constexpr int kKTileBytes = kTileTokens * kHeadDim;  // 16 KB
constexpr int kMaxBatch = 4096;   // decode requests per call (tile prefix lives in smem)
constexpr int kMaxSmem = 232448;  // 227 KB opt-in per CTA on sm_100-family parts

// ---------------------------------------------------------------- decode
struct PagedParams {
  const uint8_t* kv_cache;
  const float* weights;
  const int32_t* context_lens;
  const int32_t* block_tables;
  float* out;
  int64_t out_stride;  // elements between output rows
  int64_t bt_stride;   // elements between block-table rows
  int64_t num_blocks;
  int32_t batch;
  int32_t next_n;
  int32_t max_blocks;
  int32_t max_model_len;
  int32_t block_size;
  int32_t n_cols;    // next_n * heads = MMA N
  int32_t stages;
  int32_t acc_bufs;   // TMEM accumulator buffers: paged_acc_buffers(n_cols, sub_tiles)
  int32_t sub_tiles;  // 128-token MMA tiles per pipeline item (1 or 2)
  // Fused top-k passes (all zero / null for a plain logits call):
  const uint32_t* req_mask;     // requests with req_mask[b] == 0 get no items (null: every request)
  const uint32_t* run_flag;     // if non-null and *run_flag == 0 the launch does nothing
  // filter epilogue (the FILTER instance): a logit of row r at or above
  // thr[r] is stored (at its position in out) and sets its bit in the row's
  // candidate bitmap
  const float* thr;             // [rows]
  uint32_t* cand_bits;          // [rows][bits_stride] bitmaps over window positions
  int64_t bits_stride;          // 32-bit words per row
};

// Two epilogue warpgroups take alternate tiles; tensor memory holds 2..16
// accumulators (512 columns in buffers of the smallest power of two >=
// n_cols), so the MMA warp can run that many tiles ahead of the epilogue.
constexpr int kEpiGroups = 2;
// Decode positions (and a tile past them) stay below 2^31: the epilogue keeps
// them in 32-bit registers.
constexpr int32_t kMaxModelLen = 0x7FFFFE00;
constexpr int kMaxAccBufs = 16;
__host__ __device__ constexpr int pow2_cols(int n_cols) {
  return n_cols <= 32 ? 32 : n_cols <= 64 ? 64 : n_cols <= 128 ? 128 : 256;
}
// Decode pipeline items: two 128-token tiles per item (one barrier round
// trip for 256 tokens) when two accumulators of an item still leave room for
// double buffering, else one.  The per-block gather path keeps one.
__host__ __device__ constexpr int paged_sub_tiles(int n_cols, bool gather) {
  return (!gather && n_cols <= 128) ? 2 : 1;
}
__host__ __device__ constexpr int paged_acc_buffers(int n_cols, int sub_tiles = 1) {
  return 512 / (pow2_cols(n_cols) * sub_tiles) > kMaxAccBufs ? kMaxAccBufs : 512 / (pow2_cols(n_cols) * sub_tiles);
}

// Roles: producer warp(s), one MMA warp, kEpiGroups epilogue warpgroups.
__host__ __device__ constexpr int paged_producer_warps(bool gather) { return gather ? 2 : 1; }
__host__ __device__ constexpr int paged_threads(bool gather) {
  return 32 * (paged_producer_warps(gather) + 1 + 4 * kEpiGroups);
}

struct PagedSmem {
  uint32_t q, k, scale, w, tp, bars, misc, total;
};
__host__ __device__ inline PagedSmem paged_smem_layout(int n_cols, int stages, int batch, int sub_tiles) {
  PagedSmem L;
  uint32_t off = 0;
  L.q = off;     off += 2u * n_cols * kHeadDim;          // two Q buffers (1024-aligned: n_cols % 8 == 0)
  L.k = off;     off += (uint32_t)(stages * sub_tiles) * kKTileBytes;   // K ring: sub_tiles tiles per stage
  L.scale = off; off += (uint32_t)(stages * sub_tiles) * kTileTokens * 4;
  L.w = off;     off += 2u * n_cols * 4;                  // two weight rows
  L.tp = off;    off += (uint32_t)(batch + 1) * 4;        // per-request tile prefix
  off = (off + 7u) & ~7u;
  L.bars = off;  off += 8u * (2u * stages + 2u * kMaxAccBufs + 5u);  // full/empty per stage, accf/acce, qf/qe x2, drain
  L.misc = off;  off += 32u;
  L.total = off + 1024u;                                  // slack for 1024-byte alignment
  return L;
}

// --------------------------------------------------------------- prefill
struct PrefillParams {
  const int32_t* ks;
  const int32_t* ke;
  float* out;
  int64_t out_stride;
  int32_t rows;     // M
  int32_t cols;     // N
  int32_t block_m;  // query rows per work unit
  int32_t n_cols;   // block_m * heads = MMA N
  int32_t stages;
  int32_t split;    // column-tile splits per row block (strided)
  int32_t reverse;  // 1: row blocks dealt from the last one
  int32_t vec_ok;   // out rows are 16-byte aligned: float4 -inf fill
  int32_t acc_bufs; // TMEM accumulator buffers: paged_acc_buffers(n_cols)
  int32_t tma_fill; // 1: -inf tiles are TMA stores of a constant shared tile (needs vec_ok)
  int32_t fill_cols; // columns covered by the -inf tensor map: N rounded down to a multiple of 4
  int32_t clean;     // 1: -inf outside the windows; 0: only the windows are written
  // paged K (the gather fused into the producer): column n of request r
  // (cu_seq_lens[r] <= n < cu_seq_lens[r+1]) is token n - cu_seq_lens[r] of
  // that request, read through its block-table row from the split-page cache
  const uint8_t* kv_cache;
  const int32_t* block_tables;
  const int32_t* cu_seq_lens;  // [n_req + 1]
  int64_t bt_stride;
  int64_t num_blocks;
  int32_t max_blocks;
  int32_t block_size;          // 16, 32, 64 or 128
  int32_t n_req;
};

// Roles: producer warp, MMA warp, kEpiGroups epilogue warpgroups, -inf filler warp.
__host__ __device__ constexpr int prefill_threads() { return 32 * (1 + 1 + 4 * kEpiGroups + 1); }

struct PrefillSmem {
  uint32_t q, k, ninf, scale, w, cu, bars, misc, total;
};
// The -inf tile (block_m rows x 128 floats, the source of the TMA -inf
// stores) is at most 8 x 512 B: block_m * heads <= 256 with heads >= 32.
constexpr int kNinfTileBytes = 8 * kTileTokens * 4;
// cu_entries: request offsets kept in shared memory by the paged variant (0
// for contiguous K).
// head_dim: bytes per Q/K row (128, or 64 with the 64-byte swizzle).
__host__ __device__ inline PrefillSmem prefill_smem_layout(int n_cols, int stages, int cu_entries = 0,
                                                           int head_dim = kHeadDim) {
  PrefillSmem L;
  uint32_t off = 0;
  L.q = off;     off += 2u * n_cols * head_dim;            // two Q blocks
  L.k = off;     off += (uint32_t)stages * kTileTokens * head_dim;
  L.ninf = off;  off += kNinfTileBytes;                     // 1024-aligned (follows whole K tiles)
  L.scale = off; off += (uint32_t)stages * kTileTokens * 4;
  L.w = off;     off += 2u * n_cols * 4;                    // two weight blocks
  L.cu = off;    off += 4u * (uint32_t)cu_entries;
  off = (off + 7u) & ~7u;
  L.bars = off;  off += 8u * (2u * stages + 2u * kMaxAccBufs + 5u);  // full/empty per stage, accf/acce, qf/qe x2, drain
  L.misc = off;  off += 32u;
  L.total = off + 1024u;
  return L;
}

// ----------------------------------------------------------------- top-k
struct TopkParams {
  const float* logits;
  int64_t stride;               // elements between logits rows
  const int32_t* ks;            // mode 0: row windows [max(ks,0), min(ke,cols))
  const int32_t* ke;
  const int32_t* context_lens;  // mode 1: row b*next_n+n has window [0, ctx_b - next_n + n + 1) within cols
  int32_t* out;
  int64_t out_stride;
  int32_t rows;
  int32_t k;
  int32_t cols;    // row width the windows are clamped to (N, or max_model_len)
  int32_t next_n;
  int32_t mode;    // 0 prefill windows, 1 decode windows
  int32_t cap;     // candidates held in shared memory
  int32_t vec_ok;  // every row starts 16-byte aligned: float4 loads inside the windows
  const uint32_t* row_mask;  // rows with row_mask[r] == 0 are skipped (null: every row)
  const uint32_t* run_flag;  // if non-null and *run_flag == 0 the launch does nothing
};

constexpr int kTopkThreads = 512;
constexpr int kTopkBins = 4096;  // 12-bit radix levels (the last level has 8 bits)
constexpr int kTopkMaxK = 2048;
constexpr int kTopkMaxCap = 8192;  // 97 KB of shared memory per CTA: two CTAs per SM
constexpr int kTopkMaxCluster = 8;      // CTAs per row at most (portable cluster size)
constexpr int kTopkMinSlice = 8192;     // window values per CTA below which a row keeps one CTA
// Shared memory of one top-k CTA: the copy buffer for a short window, which
// also holds the histogram and (in a cluster) the cluster's summed
// histogram once the window is in the candidate arrays; the candidates; scan
// slots; flags; the copy's mbarrier.
struct TopkLayout {
  uint32_t ring, hist, hsum, cand_key, cand_pos, scan, misc, bar, total;
};
__host__ __device__ inline TopkLayout topk_smem_layout(int cap) {
  TopkLayout L;
  // (the histogram area also stages a compaction of up to cap words)
  constexpr uint32_t kHists = 8u * kTopkBins, kWindow = (4u * (kTopkMaxCap + 4) + 15u) & ~15u;
  constexpr uint32_t kRing = kHists > kWindow ? kHists : kWindow;
  L.ring = 0;
  L.hist = 0;
  L.hsum = 4u * kTopkBins;
  uint32_t off = kRing;
  L.cand_key = off; off += 4u * (uint32_t)cap;
  L.cand_pos = off; off += 4u * (uint32_t)cap;
  L.scan = off;     off += 4u * 32u;
  L.misc = off;     off += 4u * 8u;
  L.bar = off;      off += 8u;
  L.total = off;
  return L;
}

// ------------------------------------------------- fused decode top-k
// Scratch of fp8_paged_mqa_topk (caller-provided workspace), per call:
//   logits   [rows][ls] f32   the sampled items, the candidates at their positions,
//                             and whole rows of the requests that need the exact fallback
//   thr      [rows] f32       each row's candidate threshold
//   cand     [rows][tw] u32   bitmap of window positions whose logit is at or above it
//   req_flag [batch] u32, row_flag [rows] u32, any [4] u32   rows left to the fallback
struct FusedTopkLayout {
  uint64_t logits, thr, cand, req_flag, row_flag, any, total;
  int64_t ls, tw;
};
constexpr int kFusedSampleStride = 32;  // the threshold sample: every 32nd item of each request
constexpr int kFusedMaxSample = 16384;  // sampled logits a row's threshold is taken from, at most
__host__ __device__ inline FusedTopkLayout fused_topk_layout(int64_t batch, int64_t next_n, int64_t max_model_len,
                                                             int32_t k) {
  (void)k;
  FusedTopkLayout L;
  const int64_t rows = batch * next_n;
  L.ls = (max_model_len + 3) & ~static_cast<int64_t>(3);
  L.tw = (((max_model_len + 31) / 32) + 3) & ~static_cast<int64_t>(3);
  uint64_t off = 0;
  const auto take = [&](uint64_t bytes) {
    const uint64_t at = off;
    off = (off + bytes + 255u) & ~static_cast<uint64_t>(255u);
    return at;
  };
  L.logits = take(static_cast<uint64_t>(rows) * L.ls * 4u);
  L.thr = take(static_cast<uint64_t>(rows) * 4u);
  L.cand = take(static_cast<uint64_t>(rows) * L.tw * 4u);
  L.req_flag = take(static_cast<uint64_t>(batch) * 4u);
  L.row_flag = take(static_cast<uint64_t>(rows) * 4u);
  L.any = take(16u);
  L.total = off;
  return L;
}
// The per-row passes of the fused top-k around the decode kernel's sample and
// filter passes: windows of the decode rows (as fp8_paged_topk), k, and the
// workspace pointers.
struct FusedTopkParams {
  const int32_t* context_lens;
  int32_t rows, next_n, cols, k;  // cols: max_model_len
  int32_t item_tokens;            // tokens per item of the decode kernel (128 or 256)
  float* logits;                  // workspace rows (stride ls)
  int64_t ls, tw;
  float* thr;
  uint32_t* cand;
  uint32_t* req_flag;
  uint32_t* row_flag;
  uint32_t* any;
  int32_t* out;                   // indices [rows][out_stride]
  int64_t out_stride;
};

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute is set once per (kernel, device) and size
// (cached on the host), not on every launch.
cudaError_t ensure_dynamic_smem(const void* kernel, int bytes);

// ------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.  The tensor maps are encoded
// by the caller; `heads` selects the template instance.
// mode 0: the logits; 1: the fused top-k's filter pass (candidates instead of
// the logits); 2: the logits of every kFusedSampleStride-th item (its sample)
cudaError_t launch_paged(const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const CUtensorMap& tm_sc,
                         const PagedParams& p, int heads, bool gather, int grid, int smem_bytes, cudaStream_t stream,
                         int mode = 0);
cudaError_t launch_prefill(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_s,
                           const CUtensorMap& tm_w, const CUtensorMap& tm_out, const PrefillParams& p, int heads,
                           int head_dim, bool paged, int grid, int smem_bytes, cudaStream_t stream);

// ctas: CTAs per row (1: one CTA per row; 2..kTopkMaxCluster: one cluster per row)
cudaError_t launch_topk(const TopkParams& p, int ctas, int smem_bytes, cudaStream_t stream);
// Fused decode top-k, per row: the threshold from the sampled logits (and
// the workspace reset), then the exact selection from the candidates (or
// the row handed to the fallback).  One CTA of kTopkThreads per row.
cudaError_t launch_fused_threshold(const FusedTopkParams& p, int smem_bytes, cudaStream_t stream);
// dynamic shared memory of the threshold kernel (histogram, sample keys) and
// of the select kernel (histogram, candidate keys and positions)
__host__ __device__ constexpr int fused_threshold_smem_bytes() { return 4 * kTopkBins + 4 * kFusedMaxSample; }
__host__ __device__ constexpr int fused_select_smem_bytes() { return 4 * kTopkBins + 8 * kTopkMaxCap; }
cudaError_t launch_fused_select(const FusedTopkParams& p, int smem_bytes, cudaStream_t stream);

// Launches the watchdog self-test kernel: a bounded wait that nothing
// satisfies, given up after limit_ns (sets the decode word's self-test bit).
cudaError_t launch_watchdog_selftest(uint64_t limit_ns, cudaStream_t stream);

// Watchdog words of the two translation units (synchronous read, optional clear).
cudaError_t read_paged_watchdog(unsigned int* value, bool clear);
cudaError_t read_prefill_watchdog(unsigned int* value, bool clear);
cudaError_t read_topk_watchdog(unsigned int* value, bool clear);

}  // namespace fp8idx
