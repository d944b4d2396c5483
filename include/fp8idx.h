/*
 * fp8idx -- FP8 "lightning indexer" logits on NVIDIA GB300 (sm_103a).
 *
 * The operation (aiter PR 5047 "[HIP] [JIT] fp8_paged_mqa_logits:
 * hand-written gfx950 decode indexer kernel", section Motivation; aiter PR
 * 5046 "[HIP] [JIT] fp8_mqa_logits: hand-written gfx950 prefill indexer
 * kernel", section Motivation):
 *
 *     logits[m, n] = sum_h relu(<Q[m,h,:], K[n,:]>) * kv_scale[n] * weights[m,h]
 *
 * Q and K are e4m3 (OCP FP8, "e4m3fn": bias 7, no infinities, S.1111.111 =
 * NaN); kv_scale, weights and logits are IEEE f32.  Products are formed on
 * the tensor cores with f32 accumulation; the ReLU, weight, head sum and scale
 * run in f32 on the CUDA cores.
 *
 * Conventions for every entry point:
 *  - All tensor data pointers are DEVICE pointers on the current device,
 *    owned by the caller; the library keeps no reference after the call
 *    returns and allocates no memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously; no call synchronises the
 *    host, so the compute calls can be captured in a CUDA graph.
 *  - Shapes, dtypes, strides and alignment are checked on the host before
 *    anything is launched.  A non-OK status launches nothing (except
 *    FP8IDX_ERR_CUDA, returned when the launch itself failed); the message
 *    for the last non-OK status on the calling thread is available from
 *    fp8idx_last_error().
 *  - Values are not checked (they live on the device).  Preconditions:
 *    kv_scale >= 0 (the hoist of the scale out of the ReLU relies on it);
 *    no NaN in owned Q/K/scales/weights; block ids in range.  Indices read
 *    from the device are clamped so that bad values cannot fault, but the
 *    results for inputs that break a precondition are unspecified.
 *  - Every in-kernel pipeline wait is bounded (about 2 s).  A wait that runs
 *    out abandons the call's remaining work, records the failure on the
 *    device, and the kernel exits normally; fp8idx_device_status() reports
 *    it.
 */
#ifndef FP8IDX_H_
#define FP8IDX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8IDX_OK = 0,
  FP8IDX_ERR_INVALID = 1,     /* null pointer, bad shape/dtype/stride/alignment */
  FP8IDX_ERR_UNSUPPORTED = 2, /* legal input this build does not implement    */
  FP8IDX_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed          */
  FP8IDX_ERR_TIMEOUT = 4      /* a device pipeline wait ran out (watchdog)     */
} fp8idx_status;

typedef enum {
  FP8IDX_U8 = 0,  /* e4m3 codes or raw bytes */
  FP8IDX_F32 = 1,
  FP8IDX_I32 = 2
} fp8idx_dtype;

/* A strided view of caller-owned device memory.  Strides are in elements.
 * Only dimensions 0..ndim-1 are read. */
typedef struct {
  void* data;
  int32_t dtype; /* fp8idx_dtype */
  int32_t ndim;  /* 1..4 */
  int64_t shape[4];
  int64_t stride[4];
} fp8idx_tensor;

/* Tunables; 0 (or -1 for reverse_rows) means "let the host planner decide",
 * after the pages' "zero means use the host heuristic" (aiter PR 5047,
 * Technical Details; aiter PR 5046, Technical Details). */
typedef struct {
  int32_t num_ctas;     /* decode: persistent CTAs (<= SMs); top-k: CTAs per  */
                        /* row, 1 .. 8 (more than one: a thread-block      */
                        /* cluster per row)                                */
  int32_t stages;       /* K-tile pipeline depth in shared memory             */
  int32_t split_n;      /* prefill: column-tile splits per row block          */
  int32_t reverse_rows; /* prefill: -1 planner, 0 natural, 1 longest-first    */
  int32_t block_m;      /* prefill: query rows per CTA (block_m*heads <= 256) */
  int32_t clean_logits; /* prefill: 0 or 1 write -inf outside each row's     */
                        /* window (the default); -1 leaves those elements    */
                        /* untouched (the pages' clean_logits=False)         */
} fp8idx_options;

/* The launch the planner chose (filled by the fp8idx_plan_* queries). */
typedef struct {
  int32_t grid;        /* CTAs launched                                  */
  int32_t threads;     /* threads per CTA                                */
  int32_t smem_bytes;  /* dynamic shared memory per CTA                  */
  int32_t stages;      /* K-tile pipeline depth                          */
  int32_t tile_n;      /* MMA N: next_n*heads (decode), block_m*heads    */
  int32_t block_m;     /* prefill query rows per CTA; decode: next_n     */
  int32_t split_n;     /* prefill column splits; decode: 1               */
  int32_t reverse_rows;/* prefill dispatch order; decode: 0              */
  int32_t tmem_cols;   /* tensor-memory columns allocated per CTA        */
  int32_t gather;      /* decode: 1 = per-token gather (block size 1)    */
} fp8idx_plan;

/*
 * Decode: fp8_paged_mqa_logits.
 * Defined by aiter PR 5047, sections Motivation and Technical Details: K and
 * its per-token f32 dequant scale are read from a paged cache through a block
 * table; row r = b*next_n + n of the output receives, at column p, the logit
 * of query row (b, n) against token p of request b, for
 *     0 <= p <= context_lens[b] - next_n + n   (and p < max_model_len);
 * positions outside that causal window are NOT written -- pre-filling them
 * (with -inf) is the caller's job (same PR, section "GLM-5.2-MXFP4 E2E":
 * the caller pre-fills -inf; aiter issue 5477, section "The ask": the causal
 * bound context_length - next_n + pid_next_n, one output row per token).
 *
 *  q_fp8        [batch, next_n, heads, head_dim] U8 (e4m3), contiguous,
 *               16-byte aligned.
 *  kv_cache     [num_blocks, block_size*(head_dim+4)] U8, contiguous,
 *               16-byte aligned.  Block i holds block_size K rows of head_dim
 *               e4m3 bytes followed by block_size f32 scales (little endian).
 *               block_size is shape[1]/(head_dim+4).  block_size 1 is the
 *               plain co-packed cache (128 K bytes then a 4-byte scale per
 *               token).
 *  weights      [batch*next_n, heads] F32, contiguous, 16-byte aligned.
 *  context_lens [batch] I32 (device).  Must satisfy context_lens[b] <=
 *               min(max_model_len, max_blocks*block_size).
 *  block_tables [batch, max_blocks] I32, contiguous rows (stride[0] >=
 *               max_blocks, stride[1] == 1); entry j of row b is the physical
 *               block holding tokens [j*block_size, (j+1)*block_size).
 *  max_model_len  output width, at most 2^31 - 512 (UNSUPPORTED above: the
 *               kernel keeps positions in 32-bit registers).
 *  out          [batch*next_n, >= max_model_len] F32, stride[1] == 1,
 *               stride[0] >= max_model_len.
 * Supported (fp8idx_paged_is_supported): head_dim 128; heads 32 or 64;
 * next_n*heads in {32, 64, ..., 256} (a multiple of 32); block_size in
 * {1, 16, 32, 64, 128}; batch <= 4096.
 * Returns FP8IDX_OK, FP8IDX_ERR_INVALID, FP8IDX_ERR_UNSUPPORTED or
 * FP8IDX_ERR_CUDA.
 */
fp8idx_status fp8_paged_mqa_logits(const fp8idx_tensor* q_fp8,
                                   const fp8idx_tensor* kv_cache,
                                   const fp8idx_tensor* weights,
                                   const fp8idx_tensor* context_lens,
                                   const fp8idx_tensor* block_tables,
                                   int32_t max_model_len,
                                   const fp8idx_tensor* out, void* stream);

/* As fp8_paged_mqa_logits, with tunables (NULL = all heuristic). */
fp8idx_status fp8_paged_mqa_logits_ex(const fp8idx_tensor* q_fp8,
                                      const fp8idx_tensor* kv_cache,
                                      const fp8idx_tensor* weights,
                                      const fp8idx_tensor* context_lens,
                                      const fp8idx_tensor* block_tables,
                                      int32_t max_model_len,
                                      const fp8idx_tensor* out,
                                      const fp8idx_options* opts, void* stream);

/*
 * Prefill: fp8_mqa_logits.
 * Defined by aiter PR 5046, section Motivation: K is a contiguous [N, 128]
 * e4m3 buffer with a separate [N] f32 scale; row m is defined for n in
 * [cu_seqlen_ks[m], cu_seqlen_ke[m]) and is -inf elsewhere.  Every element of
 * out is written (the "clean_logits" semantics, same PR, Technical Details:
 * the -inf fill is fused into the kernel); with opts->clean_logits = -1 only
 * the windows are written (clean_logits=False, same PR, Test Plan: both
 * settings are graded).  Windows are clamped to [0, N);
 * ke <= ks, or ke <= 0, gives an all -inf row (same PR, Test Plan: empty and
 * past_end windows are legal input).
 *
 *  q_fp8        [M, heads, head_dim] U8 (e4m3), contiguous, 16-byte aligned.
 *  k_fp8        [N, head_dim] U8 (e4m3), contiguous, 16-byte aligned.
 *  kv_scale     [N] F32, contiguous, 16-byte aligned, values >= 0.
 *  weights      [M, heads] F32, contiguous, 16-byte aligned (loaded by TMA).
 *  cu_seqlen_ks, cu_seqlen_ke  [M] I32, contiguous.
 *  out          [M, >= N] F32, stride[1] == 1, stride[0] >= N.
 * Supported (fp8idx_prefill_is_supported): head_dim 128 or 64 (64-byte
 * rows: Q [M, heads, 64] and K [N, 64]); heads 32, 64 or 128 (the pages'
 * prefill sweep, same PR, Test Plan); M, N >= 0 with M*heads and N below
 * 2^31.
 */
fp8idx_status fp8_mqa_logits(const fp8idx_tensor* q_fp8,
                             const fp8idx_tensor* k_fp8,
                             const fp8idx_tensor* kv_scale,
                             const fp8idx_tensor* weights,
                             const fp8idx_tensor* cu_seqlen_ks,
                             const fp8idx_tensor* cu_seqlen_ke,
                             const fp8idx_tensor* out, void* stream);

fp8idx_status fp8_mqa_logits_ex(const fp8idx_tensor* q_fp8,
                                const fp8idx_tensor* k_fp8,
                                const fp8idx_tensor* kv_scale,
                                const fp8idx_tensor* weights,
                                const fp8idx_tensor* cu_seqlen_ks,
                                const fp8idx_tensor* cu_seqlen_ke,
                                const fp8idx_tensor* out,
                                const fp8idx_options* opts, void* stream);

/*
 * Prefill with the K gather fused in: fp8_mqa_logits_paged.
 * On the pages the prefill caller first gathers each request's K (and its
 * scale) out of the paged cache into the contiguous [N, 128] buffer that
 * fp8_mqa_logits reads (aiter PR 5046, section Motivation: "the caller has
 * already gathered K out of the paged cache").  This entry point reads K
 * through the block tables instead: column n, with cu_seq_lens[r] <= n <
 * cu_seq_lens[r+1], is token n - cu_seq_lens[r] of request r, i.e. slot
 * (t % block_size) of physical block block_tables[r][t / block_size] of the
 * split-page cache described under fp8_paged_mqa_logits.  The result equals
 * fp8_mqa_logits on the gathered buffer.
 *
 *  q_fp8, weights, cu_seqlen_ks, cu_seqlen_ke, out  as for fp8_mqa_logits;
 *               N = out->shape[1] is the gathered length.
 *  kv_cache     [num_blocks, block_size*(head_dim+4)] U8, contiguous,
 *               16-byte aligned; block_size in {16, 32, 64, 128}.
 *  block_tables [requests, max_blocks] I32, rows contiguous.
 *  cu_seq_lens  [requests + 1] I32 (device), contiguous: 0 = cu[0] <= cu[1]
 *               <= ... <= cu[requests] = N, and each request's length at
 *               most max_blocks*block_size (preconditions; requests <= 4096).
 * opts may be NULL (heuristic); stages, split_n, reverse_rows, block_m and
 * clean_logits as for fp8_mqa_logits_ex (split_n counts tiles of a padded
 * column space in which every request starts on a 128-column boundary).
 */
fp8idx_status fp8_mqa_logits_paged(const fp8idx_tensor* q_fp8,
                                   const fp8idx_tensor* kv_cache,
                                   const fp8idx_tensor* block_tables,
                                   const fp8idx_tensor* cu_seq_lens,
                                   const fp8idx_tensor* weights,
                                   const fp8idx_tensor* cu_seqlen_ks,
                                   const fp8idx_tensor* cu_seqlen_ke,
                                   const fp8idx_tensor* out,
                                   const fp8idx_options* opts, void* stream);

/*
 * Top-k consumers of the logits: the positions of each row's k largest
 * logits inside the row's window.  The step after the logits on the pages is
 * a per-row top-k selection with index_topk 2048 or 512 (aiter PR 5047,
 * section "GLM-5.2-MXFP4 E2E": stale finite logits outside the window would
 * corrupt it, hence the -inf contract; aiter issue 5477, section Measurement:
 * index_topk 512).  The pages do not define the selection further; this
 * library's definition: row r selects the min(k, L_r) positions (columns of
 * the logits row) of its window with the largest logits, equal logits taken
 * from the lowest positions first (so the set is unique; -0.0 == +0.0);
 * indices[r, 0 .. min(k, L_r)) lists them in ascending position order and
 * indices[r, j] = -1 for j >= L_r, the window length.
 *
 *  logits   [rows, width] F32, stride[1] == 1, stride[0] >= width.  Only the
 *           windows are read, so values outside them do not matter.
 *  indices  [rows, k] I32 output, stride[1] == 1, stride[0] >= k.
 *  k        1 .. 2048.
 * No NaN inside a window (precondition).  One CTA per row, or, when the
 * rows number at most a quarter of the SMs and the width allows at least
 * 8192 values per CTA, a thread-block cluster of up to 8 CTAs per row
 * sharing its window; no scratch memory.  Returns FP8IDX_OK, FP8IDX_ERR_INVALID,
 * FP8IDX_ERR_UNSUPPORTED (k or num_ctas out of range) or FP8IDX_ERR_CUDA.
 *
 * fp8_paged_topk: decode windows.  rows = batch*next_n; row r = b*next_n+n
 * has window [0, min(context_lens[b] - next_n + n + 1, max_model_len)) -- the
 * columns fp8_paged_mqa_logits writes.  context_lens [batch] I32 contiguous;
 * max_model_len <= width.
 */
fp8idx_status fp8_paged_topk(const fp8idx_tensor* logits,
                             const fp8idx_tensor* context_lens,
                             int32_t next_n, int32_t max_model_len, int32_t k,
                             const fp8idx_tensor* indices, void* stream);

/* fp8_mqa_topk: prefill windows.  Row m has window
 * [max(cu_seqlen_ks[m], 0), min(cu_seqlen_ke[m], width)) -- the columns
 * fp8_mqa_logits computes.  cu_seqlen_ks/ke [rows] I32 contiguous. */
fp8idx_status fp8_mqa_topk(const fp8idx_tensor* logits,
                           const fp8idx_tensor* cu_seqlen_ks,
                           const fp8idx_tensor* cu_seqlen_ke, int32_t k,
                           const fp8idx_tensor* indices, void* stream);

/* As above, with tunables (NULL = heuristic): opts->num_ctas fixes the CTAs
 * per row (0 = heuristic, 1 .. 8); the other fields are ignored.  The result
 * does not depend on it. */
fp8idx_status fp8_paged_topk_ex(const fp8idx_tensor* logits,
                                const fp8idx_tensor* context_lens,
                                int32_t next_n, int32_t max_model_len,
                                int32_t k, const fp8idx_tensor* indices,
                                const fp8idx_options* opts, void* stream);
fp8idx_status fp8_mqa_topk_ex(const fp8idx_tensor* logits,
                              const fp8idx_tensor* cu_seqlen_ks,
                              const fp8idx_tensor* cu_seqlen_ke, int32_t k,
                              const fp8idx_tensor* indices,
                              const fp8idx_options* opts, void* stream);

/*
 * Fused decode logits + top-k: fp8_paged_mqa_topk.
 * The decode logits of fp8_paged_mqa_logits followed by the selection of
 * fp8_paged_topk on them (the index_topk step that follows the indexer on the
 * pages: aiter PR 5047, section "GLM-5.2-MXFP4 E2E"; aiter issue 5477,
 * section Measurement), computed without writing the logits of every row:
 * indices[r] is exactly what fp8_paged_topk returns on the logits
 * fp8_paged_mqa_logits writes (same window, tie rule, order and -1 padding).
 *
 * How: the decode kernel first runs on every 32nd item (128 or 256 tokens)
 * of each request, and each row's threshold is taken from that sample so
 * that more than k of the row's logits lie at or above it (about 1.5k for
 * long windows); a second pass of the decode kernel keeps, per row, only the
 * logits at or above the threshold (stored at their positions) and a bitmap
 * of those positions; a per-row kernel then selects the k largest of them
 * exactly.  A row whose candidates cannot be shown to contain its k largest
 * (fewer than k, or more than 8192) is recomputed exactly instead: its
 * request's logits are written to the workspace and the top-k kernel
 * selects from them.  The result never depends on which path a row took.
 *
 *  q_fp8, kv_cache, weights, context_lens, block_tables, max_model_len
 *               as for fp8_paged_mqa_logits (same support gate).
 *  k            1 .. 2048.
 *  indices      [batch*next_n, k] I32 output, stride[1] == 1.
 *  workspace    device scratch of at least
 *               fp8idx_paged_mqa_topk_workspace(batch, next_n,
 *               max_model_len, k) bytes, 256-byte aligned, owned by the
 *               caller; its contents on entry do not matter and are
 *               overwritten.  Two calls in flight at once need two
 *               workspaces.  (It holds one f32 row per output row for the
 *               sample and the fallback, so it is about the size of the
 *               logits fp8_paged_mqa_logits would write.)
 *  opts         as for fp8_paged_mqa_logits_ex (NULL = heuristic).
 * Six kernels are enqueued on `stream`; no host synchronisation.  Returns
 * FP8IDX_OK, FP8IDX_ERR_INVALID (bad arguments, workspace too small or
 * misaligned), FP8IDX_ERR_UNSUPPORTED or FP8IDX_ERR_CUDA.
 */
fp8idx_status fp8_paged_mqa_topk(const fp8idx_tensor* q_fp8,
                                 const fp8idx_tensor* kv_cache,
                                 const fp8idx_tensor* weights,
                                 const fp8idx_tensor* context_lens,
                                 const fp8idx_tensor* block_tables,
                                 int32_t max_model_len, int32_t k,
                                 const fp8idx_tensor* indices, void* workspace,
                                 size_t workspace_bytes,
                                 const fp8idx_options* opts, void* stream);

/* Bytes of workspace fp8_paged_mqa_topk needs (0 for invalid arguments).
 * Pure host function. */
size_t fp8idx_paged_mqa_topk_workspace(int64_t batch, int32_t next_n,
                                       int32_t max_model_len, int32_t k);

/*
 * fp8_paged_mqa_topk without a workspace argument: the same computation and
 * result, with its scratch taken from a fixed area inside the library.  The
 * paper has no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory -- a serving engine that gives all free
 * device memory to its KV-cache pool at start-up and allows no allocation
 * afterwards, a plugin that runs inside a host framework without access to
 * its allocator, or a latency-critical path on which a cudaMalloc, which can
 * synchronise the device, is not acceptable.  This call allocates nothing.
 *
 *  - The scratch is one static device array of 16 MiB (16777216 bytes) that
 *    every GPU which loads the library holds until the process exits.  A
 *    shape whose workspace (fp8idx_paged_mqa_topk_workspace) is larger is
 *    rejected with FP8IDX_ERR_UNSUPPORTED and a message naming both sizes,
 *    before anything is launched; such shapes need fp8_paged_mqa_topk.
 *  - The first call on a device looks up the array's device address on that
 *    device (cudaGetSymbolAddress) and keeps it; make that first call before
 *    any stream capture.
 *  - Every call on a device uses the same array, and it keeps whatever the
 *    last call left in it; each call resets what it needs.  Calls whose
 *    kernels overlap on the GPU (other streams, other host threads) race on
 *    the array and give wrong results: order them on one stream or wait for
 *    one before starting the next.
 * Arguments, outputs and statuses as for fp8_paged_mqa_topk.
 */
fp8idx_status fp8_paged_mqa_topk_noalloc(const fp8idx_tensor* q_fp8,
                                         const fp8idx_tensor* kv_cache,
                                         const fp8idx_tensor* weights,
                                         const fp8idx_tensor* context_lens,
                                         const fp8idx_tensor* block_tables,
                                         int32_t max_model_len, int32_t k,
                                         const fp8idx_tensor* indices,
                                         const fp8idx_options* opts,
                                         void* stream);

/* Support gates, after the pages' is_supported(num_heads, head_dim,
 * kv_block_size) (aiter PR 5047, Technical Details) and is_supported(
 * num_heads, head_dim) (aiter PR 5046, Technical Details): 1 if the shape is
 * implemented, else 0.  Pure host functions; no device needed. */
int fp8idx_paged_is_supported(int32_t heads, int32_t head_dim,
                              int32_t block_size, int32_t next_n);
int fp8idx_prefill_is_supported(int32_t heads, int32_t head_dim);
/* The decode gate under its short name, with the arguments of the decode
 * page's is_supported(num_heads, head_dim, kv_block_size) plus next_n (which
 * the fold of next_n into the MMA N dimension bounds: next_n*heads <= 256).
 * Identical to fp8idx_paged_is_supported; prefill shapes have their own
 * gate because the prefill kernel supports other head dims and head counts. */
int fp8idx_is_supported(int32_t heads, int32_t head_dim,
                        int32_t kv_block_size, int32_t next_n);

/* The launch the planner would choose for a shape, for `num_sms` SMs (pass 0
 * to query the current device).  After the pages' host heuristics that pick
 * the split and tile from the problem size (aiter PR 5047, Technical
 * Details: from batch * max_model_len; aiter PR 5046, Technical Details:
 * BlockM, SplitN, reverse_rows).  Pure host functions when num_sms > 0. */
fp8idx_status fp8idx_plan_paged(int32_t batch, int32_t next_n, int32_t heads,
                                int32_t head_dim, int32_t block_size,
                                int32_t max_model_len, int32_t num_sms,
                                const fp8idx_options* opts, fp8idx_plan* plan);
fp8idx_status fp8idx_plan_prefill(int64_t rows, int64_t cols, int32_t heads,
                                  int32_t head_dim, int32_t num_sms,
                                  const fp8idx_options* opts, fp8idx_plan* plan);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* fp8idx_last_error(void);

/* Reads and optionally clears the device watchdog word of the current
 * device.  FP8IDX_OK if no in-kernel wait has run out since the last clear,
 * FP8IDX_ERR_TIMEOUT if one has.  This call synchronises with the device
 * (it copies the word back), so it does not belong inside a captured graph. */
fp8idx_status fp8idx_device_status(int32_t clear);

/* The device address of page-locked host memory, so that a host buffer can
 * be the output of fp8_paged_mqa_logits or of the top-k calls (whose kernels
 * write their results with plain stores): the results then go straight into
 * host memory while the kernel runs (on Grace-Blackwell over NVLink-C2C),
 * with no separate device-to-host copy.  Inputs, and the prefill output
 * (written partly by TMA stores), stay in device memory.
 * host_ptr: an address inside an allocation made by cudaHostAlloc /
 * cudaMallocHost or registered with cudaHostRegister.  FP8IDX_OK with
 * *device_ptr set; FP8IDX_ERR_INVALID if an argument is null or host_ptr is
 * not page-locked host memory; FP8IDX_ERR_UNSUPPORTED if the memory is not
 * mapped into the current device's address space.  Neither synchronises nor
 * allocates. */
fp8idx_status fp8idx_host_mapped_pointer(const void* host_ptr, void** device_ptr);

/* Test hook for the watchdog above.  Enqueues one small kernel that waits,
 * through the same bounded wait as every pipeline stage, on a shared-memory
 * barrier that nothing ever arrives on, and gives up after limit_us
 * microseconds (1 .. 100000) instead of the pipelines' 2 s.  The kernel then
 * returns normally: afterwards fp8idx_device_status() reports
 * FP8IDX_ERR_TIMEOUT with the self-test site (bit 0x80 of the decode word)
 * until it is cleared, and the device stays usable.  No copy, tensor-core
 * operation or tensor memory is involved.  Returns FP8IDX_OK,
 * FP8IDX_ERR_INVALID (limit out of range) or FP8IDX_ERR_CUDA. */
fp8idx_status fp8idx_watchdog_selftest(int32_t limit_us, void* stream);

/* Library version: major*10000 + minor*100 + patch. */
int32_t fp8idx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8IDX_H_ */
