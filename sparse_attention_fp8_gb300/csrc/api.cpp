// C-ABI entry points of libfp8idx: argument validation, the host planner,
// TMA tensor-map encoding and kernel launch.  No allocation, no host
// synchronisation on the compute paths (both are graph-capturable).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "fp8idx.h"
#include "kernels.h"

namespace {

using namespace fp8idx;

thread_local std::string g_last_error;

fp8idx_status fail(fp8idx_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

fp8idx_status ok() { return FP8IDX_OK; }

// ---------------------------------------------------------- device facts
struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
  bool valid = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

fp8idx_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return fail(FP8IDX_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.valid) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return fail(FP8IDX_ERR_CUDA, "cudaDeviceGetAttribute failed");
    if (major != 10 || minor != 3)
      return fail(FP8IDX_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", major, minor);
    d.valid = true;
  }
  *out = d;
  return FP8IDX_OK;
}

// ------------------------------------------ per-kernel shared-memory limit
struct SmemAttr {
  const void* kernel;
  int device;
  int bytes;
};
constexpr int kMaxSmemAttrs = 256;
SmemAttr g_smem_attr[kMaxSmemAttrs];
int g_smem_attr_n = 0;
std::mutex g_smem_attr_mu;

}  // namespace

namespace fp8idx {

// Sets the message fp8idx_last_error() returns on this thread (for entry
// points defined in other translation units).
void set_last_error_message(const char* msg) { g_last_error = msg; }

cudaError_t ensure_dynamic_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_smem_attr_mu);
  SmemAttr* hit = nullptr;
  for (int i = 0; i < g_smem_attr_n; ++i)
    if (g_smem_attr[i].kernel == kernel && g_smem_attr[i].device == dev) hit = &g_smem_attr[i];
  if (hit != nullptr && hit->bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (hit != nullptr) {
    hit->bytes = bytes;
  } else if (g_smem_attr_n < kMaxSmemAttrs) {
    g_smem_attr[g_smem_attr_n++] = SmemAttr{kernel, dev, bytes};
  }
  return cudaSuccess;
}

}  // namespace fp8idx

namespace {

using namespace fp8idx;

// ---------------------------------------------------- tensor-map encoding
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

fp8idx_status encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(FP8IDX_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t gd[5], gs[5];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i < rank - 1) gs[i] = strides_bytes[i];
  }
  CUresult r = fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FP8IDX_ERR_CUDA, "tensor map for %s: cuTensorMapEncodeTiled error %d", what, (int)r);
  return FP8IDX_OK;
}

// ------------------------------------------------------------ validation
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fp8idx_status check_tensor(const fp8idx_tensor* t, const char* name, int dtype, int ndim) {
  if (!t) return fail(FP8IDX_ERR_INVALID, "%s: null descriptor", name);
  if (t->ndim != ndim) return fail(FP8IDX_ERR_INVALID, "%s: ndim %d, expected %d", name, t->ndim, ndim);
  if (t->dtype != dtype) return fail(FP8IDX_ERR_INVALID, "%s: wrong dtype %d", name, t->dtype);
  int64_t numel = 1;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return fail(FP8IDX_ERR_INVALID, "%s: negative extent", name);
    numel *= t->shape[i];
  }
  if (numel > 0 && !t->data) return fail(FP8IDX_ERR_INVALID, "%s: null data pointer", name);
  return FP8IDX_OK;
}

bool contiguous(const fp8idx_tensor* t) {
  int64_t expect = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->stride[i] != expect) return false;
    expect *= t->shape[i];
  }
  return true;
}

#define TRY(expr)                          \
  do {                                     \
    fp8idx_status _st = (expr);            \
    if (_st != FP8IDX_OK) return _st;      \
  } while (0)

// ---------------------------------------------------------------- planner

bool paged_supported(int heads, int head_dim, int block_size, int next_n) {
  if (head_dim != kHeadDim) return false;
  if (heads != 32 && heads != 64) return false;
  if (next_n < 1 || next_n * heads > 256) return false;
  return block_size == 1 || block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128;
}

bool prefill_supported(int heads, int head_dim) {
  return (head_dim == kHeadDim || head_dim == 64) && (heads == 32 || heads == 64 || heads == 128);
}

fp8idx_status plan_paged(int32_t batch, int32_t next_n, int32_t heads, int32_t head_dim, int32_t block_size,
                         int32_t max_model_len, int32_t num_sms, int32_t smem_limit, const fp8idx_options* o,
                         fp8idx_plan* plan) {
  if (!paged_supported(heads, head_dim, block_size, next_n))
    return fail(FP8IDX_ERR_UNSUPPORTED, "decode: heads=%d head_dim=%d block_size=%d next_n=%d not supported", heads,
                head_dim, block_size, next_n);
  if (batch < 0 || batch > kMaxBatch) return fail(FP8IDX_ERR_UNSUPPORTED, "decode: batch %d > %d", batch, kMaxBatch);
  if (num_sms <= 0) return fail(FP8IDX_ERR_INVALID, "num_sms must be positive");
  const bool gather = block_size == 1;
  const int n_cols = next_n * heads;
  const int sub = paged_sub_tiles(n_cols, gather);
  int stages = (o && o->stages > 0) ? o->stages : 12 / sub;  // stages hold `sub` 128-token tiles each
  const int min_stages = gather ? 6 : 2;
  while (stages > min_stages && (int)paged_smem_layout(n_cols, stages, batch, sub).total > smem_limit) --stages;
  if (stages < min_stages || (int)paged_smem_layout(n_cols, stages, batch, sub).total > smem_limit)
    return fail(FP8IDX_ERR_UNSUPPORTED, "decode: shared memory too small for %d stages", stages);
  // Upper bound on work items without reading context_lens: every request
  // full to max_model_len.  The persistent grid never exceeds the SM count.
  const int64_t item_tokens = static_cast<int64_t>(kTileTokens) * sub;
  const int64_t tiles_per_req = (static_cast<int64_t>(std::max(max_model_len, 0)) + item_tokens - 1) / item_tokens;
  const int64_t items_ub = static_cast<int64_t>(batch) * tiles_per_req;
  int grid = static_cast<int>(std::min<int64_t>(num_sms, std::max<int64_t>(items_ub, 1)));
  if (o && o->num_ctas > 0) grid = std::min(o->num_ctas, num_sms);
  std::memset(plan, 0, sizeof(*plan));
  plan->grid = grid;
  plan->threads = paged_threads(gather);
  plan->smem_bytes = (int)paged_smem_layout(n_cols, stages, batch, sub).total;
  plan->stages = stages;
  plan->tile_n = n_cols;
  plan->block_m = next_n;
  plan->split_n = 1;
  plan->reverse_rows = 0;
  plan->tmem_cols = 512;
  plan->gather = gather ? 1 : 0;
  return FP8IDX_OK;
}

fp8idx_status plan_prefill(int64_t rows, int64_t cols, int32_t heads, int32_t head_dim, int32_t num_sms,
                           int32_t smem_limit, const fp8idx_options* o, fp8idx_plan* plan, int cu_entries = 0,
                           int min_stages = 2) {
  if (!prefill_supported(heads, head_dim))
    return fail(FP8IDX_ERR_UNSUPPORTED, "prefill: heads=%d head_dim=%d not supported", heads, head_dim);
  if (rows < 0 || cols < 0 || rows * heads >= (1ll << 31) || cols >= (1ll << 31))
    return fail(FP8IDX_ERR_UNSUPPORTED, "prefill: M=%lld N=%lld out of range", (long long)rows, (long long)cols);
  if (num_sms <= 0) return fail(FP8IDX_ERR_INVALID, "num_sms must be positive");
  int block_m = (o && o->block_m > 0) ? o->block_m : 256 / heads;
  if (block_m * heads > 256 || block_m > 32)
    return fail(FP8IDX_ERR_UNSUPPORTED, "prefill: block_m %d too large for %d heads", block_m, heads);
  const int n_cols = block_m * heads;
  int stages = (o && o->stages > 0) ? o->stages : 12;
  while (stages > min_stages && (int)prefill_smem_layout(n_cols, stages, cu_entries, head_dim).total > smem_limit)
    --stages;
  if (stages < min_stages)
    return fail(FP8IDX_ERR_UNSUPPORTED, "prefill: %d stages (this K source needs at least %d)", stages, min_stages);
  if ((int)prefill_smem_layout(n_cols, stages, cu_entries, head_dim).total > smem_limit)
    return fail(FP8IDX_ERR_UNSUPPORTED, "prefill: shared memory too small");
  const int64_t num_rb = (rows + block_m - 1) / block_m;
  const int64_t n_tiles = (cols + kTileTokens - 1) / kTileTokens;
  int64_t split = 1;
  if (o && o->split_n > 0) {
    split = o->split_n;
  } else if (num_rb > 0) {
    // about 16 work units per persistent CTA keeps the round-robin deal
    // within a few percent of even
    split = (16ll * num_sms + num_rb - 1) / num_rb;
  }
  split = std::max<int64_t>(1, std::min<int64_t>(split, std::max<int64_t>(n_tiles, 1)));
  int reverse = (cols > 2048) ? 1 : 0;  // longest-first pays off only for long rows
  if (o && o->reverse_rows >= 0 && o->reverse_rows <= 1) reverse = o->reverse_rows;
  const int64_t units = num_rb * split;
  if (units > 0x7fffffffll) return fail(FP8IDX_ERR_UNSUPPORTED, "prefill: too many work units");
  int grid = (int)std::min<int64_t>(num_sms, std::max<int64_t>(units, 1));
  if (o && o->num_ctas > 0) grid = std::min(o->num_ctas, num_sms);
  std::memset(plan, 0, sizeof(*plan));
  plan->grid = grid;
  plan->threads = prefill_threads();
  plan->smem_bytes = (int)prefill_smem_layout(n_cols, stages, cu_entries, head_dim).total;
  plan->stages = stages;
  plan->tile_n = n_cols;
  plan->block_m = block_m;
  plan->split_n = static_cast<int32_t>(split);
  plan->reverse_rows = reverse;
  plan->tmem_cols = 512;
  plan->gather = 0;
  return FP8IDX_OK;
}

// ----------------------------------------------------------------- decode
// Everything a decode launch needs except its output: the inputs checked,
// the plan, the tensor maps and the parameter block.
struct PagedSetup {
  CUtensorMap tm_q, tm_kv, tm_sc;
  PagedParams p;
  fp8idx_plan plan;
  int heads = 0;
  bool empty = false;  // nothing to compute (no requests or max_model_len 0)
};

fp8idx_status paged_setup(const fp8idx_tensor* q, const fp8idx_tensor* kv, const fp8idx_tensor* w,
                          const fp8idx_tensor* cl, const fp8idx_tensor* bt, int32_t max_model_len,
                          const fp8idx_options* opts, PagedSetup* S) {
  TRY(check_tensor(q, "q_fp8", FP8IDX_U8, 4));
  TRY(check_tensor(kv, "kv_cache", FP8IDX_U8, 2));
  TRY(check_tensor(w, "weights", FP8IDX_F32, 2));
  TRY(check_tensor(cl, "context_lens", FP8IDX_I32, 1));
  TRY(check_tensor(bt, "block_tables", FP8IDX_I32, 2));
  const int64_t B = q->shape[0], next_n = q->shape[1], H = q->shape[2], D = q->shape[3];
  if (max_model_len < 0) return fail(FP8IDX_ERR_INVALID, "max_model_len < 0");
  if (max_model_len > kMaxModelLen)
    return fail(FP8IDX_ERR_UNSUPPORTED, "max_model_len %d > %d (positions are kept in 32 bits)", max_model_len,
                kMaxModelLen);
  if (!contiguous(q)) return fail(FP8IDX_ERR_INVALID, "q_fp8 must be contiguous");
  if (!contiguous(kv)) return fail(FP8IDX_ERR_INVALID, "kv_cache must be contiguous");
  if (!contiguous(w)) return fail(FP8IDX_ERR_INVALID, "weights must be contiguous");
  if (cl->shape[0] != B || (B > 1 && cl->stride[0] != 1)) return fail(FP8IDX_ERR_INVALID, "context_lens must be [batch] contiguous");
  if (w->shape[0] != B * next_n || w->shape[1] != H) return fail(FP8IDX_ERR_INVALID, "weights must be [batch*next_n, heads]");
  if (bt->shape[0] != B || (bt->shape[1] > 1 && bt->stride[1] != 1) || (B > 1 && bt->stride[0] < bt->shape[1]))
    return fail(FP8IDX_ERR_INVALID, "block_tables must be [batch, max_blocks] with unit inner stride");
  if (D <= 0 || kv->shape[1] % (D + 4) != 0) return fail(FP8IDX_ERR_INVALID, "kv_cache row is not block_size*(head_dim+4) bytes");
  const int64_t blk = kv->shape[1] / (D + 4);
  if (next_n <= 0 || H <= 0 || blk <= 0) return fail(FP8IDX_ERR_INVALID, "empty next_n/heads/block_size");
  if (!paged_supported((int)H, (int)D, (int)blk, (int)next_n))
    return fail(FP8IDX_ERR_UNSUPPORTED, "decode: heads=%lld head_dim=%lld block_size=%lld next_n=%lld not supported",
                (long long)H, (long long)D, (long long)blk, (long long)next_n);
  S->empty = B == 0 || max_model_len == 0;
  if (S->empty) return ok();
  if (kv->shape[0] < 1) return fail(FP8IDX_ERR_INVALID, "kv_cache has no blocks");
  if (bt->shape[1] < 1) return fail(FP8IDX_ERR_INVALID, "block_tables has no columns");
  if (!aligned16(q->data) || !aligned16(kv->data) || !aligned16(w->data))
    return fail(FP8IDX_ERR_INVALID, "q_fp8, kv_cache and weights must be 16-byte aligned");
  if (B * next_n * H >= (1ll << 31) || kv->shape[0] >= (1ll << 31) || bt->shape[1] >= (1ll << 31))
    return fail(FP8IDX_ERR_UNSUPPORTED, "decode: extents too large");

  DeviceInfo dev;
  TRY(device_info(&dev));
  fp8idx_plan& plan = S->plan;
  TRY(plan_paged((int)B, (int)next_n, (int)H, (int)D, (int)blk, max_model_len, dev.sms, dev.smem_optin, opts, &plan));

  const int n_cols = (int)(next_n * H);
  {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)(B * n_cols)};
    const uint64_t strides[1] = {(uint64_t)D};
    const uint32_t box[2] = {(uint32_t)D, (uint32_t)n_cols};
    TRY(encode(&S->tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q->data, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
               "q"));
  }
  if (!plan.gather) {
    // K rows: [block][row][128 B]; scales: [block][blk f32], starting after the block's K rows
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)blk, (uint64_t)kv->shape[0]};
    const uint64_t strides[2] = {(uint64_t)D, (uint64_t)kv->shape[1]};
    const uint32_t box[3] = {(uint32_t)D, (uint32_t)blk, 1u};
    TRY(encode(&S->tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, kv->data, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
               "kv_cache"));
    const uint64_t sdims[2] = {(uint64_t)blk, (uint64_t)kv->shape[0]};
    const uint64_t sstrides[1] = {(uint64_t)kv->shape[1]};
    const uint32_t sbox[2] = {(uint32_t)blk, 1u};
    TRY(encode(&S->tm_sc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, static_cast<const uint8_t*>(kv->data) + blk * D, sdims,
               sstrides, sbox, CU_TENSOR_MAP_SWIZZLE_NONE, "kv_cache scales"));
  } else {
    S->tm_kv = S->tm_q;  // unused by the gather kernel
    S->tm_sc = S->tm_q;
  }
  PagedParams& p = S->p;
  std::memset(&p, 0, sizeof(p));
  p.kv_cache = static_cast<const uint8_t*>(kv->data);
  p.weights = static_cast<const float*>(w->data);
  p.context_lens = static_cast<const int32_t*>(cl->data);
  p.block_tables = static_cast<const int32_t*>(bt->data);
  p.bt_stride = B > 1 ? bt->stride[0] : bt->shape[1];
  p.num_blocks = kv->shape[0];
  p.batch = (int32_t)B;
  p.next_n = (int32_t)next_n;
  p.max_blocks = (int32_t)bt->shape[1];
  p.max_model_len = max_model_len;
  p.block_size = (int32_t)blk;
  p.n_cols = n_cols;
  p.stages = plan.stages;
  p.sub_tiles = paged_sub_tiles(n_cols, plan.gather != 0);
  p.acc_bufs = paged_acc_buffers(n_cols, p.sub_tiles);
  S->heads = (int)H;
  return ok();
}

// mode: 0 the logits, 1 the fused top-k's filter pass, 2 its sample pass
fp8idx_status paged_launch(const PagedSetup& S, const PagedParams& p, int mode, void* stream) {
  cudaError_t e = launch_paged(S.tm_q, S.tm_kv, S.tm_sc, p, S.heads, S.plan.gather != 0, S.plan.grid,
                               S.plan.smem_bytes, static_cast<cudaStream_t>(stream), mode);
  if (e != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return ok();
}

fp8idx_status paged_impl(const fp8idx_tensor* q, const fp8idx_tensor* kv, const fp8idx_tensor* w,
                         const fp8idx_tensor* cl, const fp8idx_tensor* bt, int32_t max_model_len,
                         const fp8idx_tensor* out, const fp8idx_options* opts, void* stream) {
  g_last_error.clear();
  TRY(check_tensor(q, "q_fp8", FP8IDX_U8, 4));
  TRY(check_tensor(kv, "kv_cache", FP8IDX_U8, 2));
  TRY(check_tensor(w, "weights", FP8IDX_F32, 2));
  TRY(check_tensor(cl, "context_lens", FP8IDX_I32, 1));
  TRY(check_tensor(bt, "block_tables", FP8IDX_I32, 2));
  TRY(check_tensor(out, "out", FP8IDX_F32, 2));
  const int64_t B = q->shape[0], next_n = q->shape[1];
  if (max_model_len < 0) return fail(FP8IDX_ERR_INVALID, "max_model_len < 0");
  if (out->shape[0] != B * next_n || out->shape[1] < max_model_len ||
      (out->shape[1] > 1 && out->stride[1] != 1) || (out->shape[0] > 1 && out->stride[0] < out->shape[1]))
    return fail(FP8IDX_ERR_INVALID, "out must be [batch*next_n, >=max_model_len] with unit inner stride");
  PagedSetup S;
  TRY(paged_setup(q, kv, w, cl, bt, max_model_len, opts, &S));
  if (S.empty) return ok();
  PagedParams p = S.p;
  p.out = static_cast<float*>(out->data);
  p.out_stride = out->shape[0] > 1 ? out->stride[0] : out->shape[1];
  return paged_launch(S, p, 0, stream);
}

// ----------------------------------------------------- fused decode top-k
// fp8_paged_mqa_topk: six launches on the caller's stream, none of which
// writes the logits of every row:
//   1. the decode kernel on every 32nd item of each request, its logits into
//      the workspace (the threshold sample);
//   2. per row: reset of the row's state, the threshold;
//   3. the decode kernel in its filter form: per row only the logits at or
//      above the threshold, with a bitmap of their positions, instead of
//      every logit;
//   4. per row: the exact top-k from the candidates, or the row flagged;
//   5. the decode kernel over the flagged requests only, all their logits
//      into the workspace, and 6. the top-k kernel over the flagged rows --
//      both return at once when no row was flagged.
size_t paged_topk_workspace(int64_t batch, int64_t next_n, int64_t max_model_len, int32_t k) {
  return static_cast<size_t>(fused_topk_layout(batch, next_n, max_model_len, k).total);
}

fp8idx_status paged_topk_impl(const fp8idx_tensor* q, const fp8idx_tensor* kv, const fp8idx_tensor* w,
                              const fp8idx_tensor* cl, const fp8idx_tensor* bt, int32_t max_model_len, int32_t k,
                              const fp8idx_tensor* indices, void* workspace, size_t workspace_bytes,
                              const fp8idx_options* opts, void* stream) {
  g_last_error.clear();
  TRY(check_tensor(q, "q_fp8", FP8IDX_U8, 4));
  TRY(check_tensor(indices, "indices", FP8IDX_I32, 2));
  const int64_t B = q->shape[0], next_n = q->shape[1], R = B * next_n;
  if (k < 1 || k > kTopkMaxK) return fail(FP8IDX_ERR_UNSUPPORTED, "top-k: k=%d not in [1, %d]", k, kTopkMaxK);
  if (max_model_len < 0) return fail(FP8IDX_ERR_INVALID, "max_model_len < 0");
  if (indices->shape[0] != R || indices->shape[1] != k || (k > 1 && indices->stride[1] != 1) ||
      (R > 1 && indices->stride[0] < k))
    return fail(FP8IDX_ERR_INVALID, "indices must be [batch*next_n, k] with unit inner stride");
  PagedSetup S;
  TRY(paged_setup(q, kv, w, cl, bt, max_model_len, opts, &S));
  if (R == 0) return ok();
  const FusedTopkLayout L = fused_topk_layout(B, next_n, max_model_len, k);
  if (workspace == nullptr || workspace_bytes < L.total)
    return fail(FP8IDX_ERR_INVALID, "workspace of %zu bytes, %llu needed (fp8idx_paged_mqa_topk_workspace)",
                workspace_bytes, (unsigned long long)L.total);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(FP8IDX_ERR_INVALID, "workspace must be 256-byte aligned");
  if (R >= (1ll << 31) / kTopkMaxCluster) return fail(FP8IDX_ERR_UNSUPPORTED, "top-k: too many rows");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  FusedTopkParams f;
  std::memset(&f, 0, sizeof(f));
  f.context_lens = static_cast<const int32_t*>(cl->data);
  f.rows = (int32_t)R;
  f.next_n = (int32_t)next_n;
  f.cols = max_model_len;
  f.k = k;
  f.logits = reinterpret_cast<float*>(ws + L.logits);
  f.ls = L.ls;
  f.tw = L.tw;
  f.thr = reinterpret_cast<float*>(ws + L.thr);
  f.cand = reinterpret_cast<uint32_t*>(ws + L.cand);
  f.req_flag = reinterpret_cast<uint32_t*>(ws + L.req_flag);
  f.row_flag = reinterpret_cast<uint32_t*>(ws + L.row_flag);
  f.any = reinterpret_cast<uint32_t*>(ws + L.any);
  f.out = static_cast<int32_t*>(indices->data);
  f.out_stride = R > 1 ? indices->stride[0] : k;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (S.empty) {  // max_model_len 0: every window is empty
    f.item_tokens = kTileTokens;
    cudaError_t e = launch_fused_threshold(f, fused_threshold_smem_bytes(), st);
    if (e == cudaSuccess) e = launch_fused_select(f, fused_select_smem_bytes(), st);
    if (e != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "top-k launch: %s", cudaGetErrorString(e));
    return ok();
  }
  f.item_tokens = kTileTokens * S.p.sub_tiles;

  // 1. the sample
  PagedParams p = S.p;
  p.out = f.logits;
  p.out_stride = L.ls;
  TRY(paged_launch(S, p, 2, stream));
  // 2. thresholds
  cudaError_t e = launch_fused_threshold(f, fused_threshold_smem_bytes(), st);
  if (e != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "top-k threshold launch: %s", cudaGetErrorString(e));
  // 3. the filter pass
  p = S.p;
  p.out = f.logits;
  p.out_stride = L.ls;
  p.thr = f.thr;
  p.cand_bits = f.cand;
  p.bits_stride = L.tw;
  TRY(paged_launch(S, p, 1, stream));
  // 4. the exact selection, or the row flagged
  e = launch_fused_select(f, fused_select_smem_bytes(), st);
  if (e != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "top-k select launch: %s", cudaGetErrorString(e));
  // 5. and 6. the exact fallback for flagged rows
  p = S.p;
  p.out = f.logits;
  p.out_stride = L.ls;
  p.req_mask = f.req_flag;
  p.run_flag = f.any;
  TRY(paged_launch(S, p, 0, stream));
  TopkParams tp;
  std::memset(&tp, 0, sizeof(tp));
  tp.mode = 1;
  tp.k = k;
  tp.rows = (int32_t)R;
  tp.context_lens = f.context_lens;
  tp.cols = max_model_len;
  tp.next_n = (int32_t)next_n;
  tp.logits = f.logits;
  tp.stride = L.ls;
  tp.out = f.out;
  tp.out_stride = f.out_stride;
  tp.vec_ok = 1;  // workspace rows are 16-byte aligned
  tp.row_mask = f.row_flag;
  tp.run_flag = f.any;
  DeviceInfo dev;
  TRY(device_info(&dev));
  int cap = kTopkMaxCap;
  while (cap > 1024 && (int)topk_smem_layout(cap).total > dev.smem_optin) cap >>= 1;
  tp.cap = cap;
  e = launch_topk(tp, 1, (int)topk_smem_layout(cap).total, st);
  if (e != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "top-k fallback launch: %s", cudaGetErrorString(e));
  return ok();
}

// ---------------------------------------------------------------- prefill
// The K source of a prefill call: contiguous (k, s) or paged (kv, bt, cu).
struct PrefillK {
  const fp8idx_tensor* k = nullptr;
  const fp8idx_tensor* s = nullptr;
  const fp8idx_tensor* kv = nullptr;
  const fp8idx_tensor* bt = nullptr;
  const fp8idx_tensor* cu = nullptr;
};

fp8idx_status prefill_impl(const fp8idx_tensor* q, const PrefillK& src, const fp8idx_tensor* w,
                           const fp8idx_tensor* ks, const fp8idx_tensor* ke, const fp8idx_tensor* out,
                           const fp8idx_options* opts, void* stream) {
  g_last_error.clear();
  const bool paged = src.kv != nullptr;
  TRY(check_tensor(q, "q_fp8", FP8IDX_U8, 3));
  TRY(check_tensor(w, "weights", FP8IDX_F32, 2));
  TRY(check_tensor(ks, "cu_seqlen_ks", FP8IDX_I32, 1));
  TRY(check_tensor(ke, "cu_seqlen_ke", FP8IDX_I32, 1));
  TRY(check_tensor(out, "out", FP8IDX_F32, 2));
  const int64_t M = q->shape[0], H = q->shape[1], D = q->shape[2];
  int64_t N = 0, blk = 0, R = 0;
  if (!paged) {
    TRY(check_tensor(src.k, "k_fp8", FP8IDX_U8, 2));
    TRY(check_tensor(src.s, "kv_scale", FP8IDX_F32, 1));
    N = src.k->shape[0];
    if (!contiguous(src.k) || !contiguous(src.s)) return fail(FP8IDX_ERR_INVALID, "prefill inputs must be contiguous");
    if (src.k->shape[1] != D || src.s->shape[0] != N)
      return fail(FP8IDX_ERR_INVALID, "k_fp8 must be [N, head_dim], kv_scale [N]");
  } else {
    TRY(check_tensor(src.kv, "kv_cache", FP8IDX_U8, 2));
    TRY(check_tensor(src.bt, "block_tables", FP8IDX_I32, 2));
    TRY(check_tensor(src.cu, "cu_seq_lens", FP8IDX_I32, 1));
    N = out->shape[1];
    R = src.bt->shape[0];
    if (!contiguous(src.kv) || !contiguous(src.cu)) return fail(FP8IDX_ERR_INVALID, "kv_cache and cu_seq_lens must be contiguous");
    if (src.bt->shape[1] > 1 && src.bt->stride[1] != 1) return fail(FP8IDX_ERR_INVALID, "block_tables rows must be contiguous");
    if (src.cu->shape[0] != R + 1) return fail(FP8IDX_ERR_INVALID, "cu_seq_lens must be [requests + 1]");
    if (D != kHeadDim && D != 64)
      return fail(FP8IDX_ERR_UNSUPPORTED, "paged prefill: head_dim %lld (128 or 64)", (long long)D);
    if (src.kv->shape[1] % (D + 4) != 0) return fail(FP8IDX_ERR_INVALID, "kv_cache rows must be block_size*(head_dim+4) bytes");
    blk = src.kv->shape[1] / (D + 4);
    if (blk != 1 && blk != 16 && blk != 32 && blk != 64 && blk != 128)
      return fail(FP8IDX_ERR_UNSUPPORTED, "paged prefill: block_size %lld not in {1, 16, 32, 64, 128}", (long long)blk);
    if (R < 1 || R > kMaxBatch) return fail(FP8IDX_ERR_UNSUPPORTED, "paged prefill: %lld requests (1..%d)", (long long)R, kMaxBatch);
    if (src.bt->shape[1] < 1 || src.kv->shape[0] < 1) return fail(FP8IDX_ERR_INVALID, "empty block table or cache");
    if (!aligned16(src.kv->data)) return fail(FP8IDX_ERR_INVALID, "kv_cache must be 16-byte aligned");
  }
  if (!contiguous(q) || !contiguous(w) || !contiguous(ks) || !contiguous(ke))
    return fail(FP8IDX_ERR_INVALID, "prefill inputs must be contiguous");
  if (w->shape[0] != M || w->shape[1] != H) return fail(FP8IDX_ERR_INVALID, "weights must be [M, heads]");
  if (ks->shape[0] != M || ke->shape[0] != M) return fail(FP8IDX_ERR_INVALID, "cu_seqlen_ks/ke must be [M]");
  if (out->shape[0] != M || out->shape[1] != N || (N > 1 && out->stride[1] != 1) || (M > 1 && out->stride[0] < N))
    return fail(FP8IDX_ERR_INVALID, "out must be [M, N] with unit inner stride");
  if (!prefill_supported((int)H, (int)D))
    return fail(FP8IDX_ERR_UNSUPPORTED, "prefill: heads=%lld head_dim=%lld not supported", (long long)H, (long long)D);
  if (M == 0 || N == 0) return ok();
  if (!aligned16(q->data) || !aligned16(w->data) || (!paged && (!aligned16(src.k->data) || !aligned16(src.s->data))))
    return fail(FP8IDX_ERR_INVALID, "q_fp8, k_fp8, kv_scale and weights must be 16-byte aligned");
  DeviceInfo dev;
  TRY(device_info(&dev));
  fp8idx_plan plan;
  // the block-size-1 token gather publishes tiles 4 behind: at least 6 stages
  TRY(plan_prefill(M, N, (int)H, (int)D, dev.sms, dev.smem_optin, opts, &plan, paged ? 2 * ((int)R + 1) : 0,
                   (paged && blk == 1) ? 6 : 2));
  CUtensorMap tm_q, tm_k, tm_s;
  {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)(M * H)};
    const uint64_t strides[1] = {(uint64_t)D};
    const uint32_t box[2] = {(uint32_t)D, (uint32_t)plan.tile_n};
    TRY(encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q->data, dims, strides, box,
               D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, "q"));
  }
  std::memset(&tm_k, 0, sizeof(tm_k));
  std::memset(&tm_s, 0, sizeof(tm_s));
  if (paged && blk > 1) {  // (block size 1 is gathered per token with cp.async: no tensor maps)
    // K rows of the cache: [block][row][D bytes]; scales: [block][blk f32] after the block's K rows
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)blk, (uint64_t)src.kv->shape[0]};
    const uint64_t strides[2] = {(uint64_t)D, (uint64_t)src.kv->shape[1]};
    const uint32_t box[3] = {(uint32_t)D, (uint32_t)blk, 1u};
    TRY(encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, src.kv->data, dims, strides, box,
               D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, "kv_cache"));
    if (blk >= 32) {
      const uint64_t sdims[2] = {(uint64_t)blk, (uint64_t)src.kv->shape[0]};
      const uint64_t sstrides[1] = {(uint64_t)src.kv->shape[1]};
      const uint32_t sbox[2] = {(uint32_t)blk, 1u};
      TRY(encode(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, static_cast<const uint8_t*>(src.kv->data) + blk * D,
                 sdims, sstrides, sbox, CU_TENSOR_MAP_SWIZZLE_NONE, "kv_cache scales"));
    }
  } else if (!paged) {
    {
      const uint64_t dims[2] = {(uint64_t)D, (uint64_t)N};
      const uint64_t strides[1] = {(uint64_t)D};
      const uint32_t box[2] = {(uint32_t)D, (uint32_t)kTileTokens};
      TRY(encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, src.k->data, dims, strides, box,
                 D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, "k"));
    }
    {
      const uint64_t dims[1] = {(uint64_t)N};
      const uint32_t box[1] = {(uint32_t)kTileTokens};
      TRY(encode(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, src.s->data, dims, nullptr, box,
                 CU_TENSOR_MAP_SWIZZLE_NONE, "kv_scale"));
    }
  }
  CUtensorMap tm_w;
  {
    const uint64_t dims[1] = {(uint64_t)(M * H)};
    const uint32_t box[1] = {(uint32_t)plan.tile_n};
    TRY(encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, w->data, dims, nullptr, box, CU_TENSOR_MAP_SWIZZLE_NONE,
               "weights"));
  }
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  if (paged) {
    p.kv_cache = static_cast<const uint8_t*>(src.kv->data);
    p.block_tables = static_cast<const int32_t*>(src.bt->data);
    p.cu_seq_lens = static_cast<const int32_t*>(src.cu->data);
    p.bt_stride = R > 1 ? src.bt->stride[0] : src.bt->shape[1];
    p.num_blocks = src.kv->shape[0];
    p.max_blocks = (int32_t)src.bt->shape[1];
    p.block_size = (int32_t)blk;
    p.n_req = (int32_t)R;
  }
  p.ks = static_cast<const int32_t*>(ks->data);
  p.ke = static_cast<const int32_t*>(ke->data);
  p.out = static_cast<float*>(out->data);
  p.out_stride = M > 1 ? out->stride[0] : N;
  p.rows = (int32_t)M;
  p.cols = (int32_t)N;
  p.block_m = plan.block_m;
  p.n_cols = plan.tile_n;
  p.stages = plan.stages;
  p.split = plan.split_n;
  p.reverse = plan.reverse_rows;
  p.vec_ok = (aligned16(out->data) && (p.out_stride % 4) == 0) ? 1 : 0;
  p.clean = (opts && opts->clean_logits < 0) ? 0 : 1;
  p.acc_bufs = paged_acc_buffers(plan.tile_n);
  // -inf tiles as TMA stores need 16-byte aligned rows (the tensor map's
  // stride rule); otherwise the epilogue warps write them.  A TMA store
  // writes whole 16-byte units, so the map is N rounded down to a multiple
  // of 4 columns wide and the kernel writes the rest of the row directly.
  CUtensorMap tm_out;
  std::memset(&tm_out, 0, sizeof(tm_out));
  p.tma_fill = 0;
  p.fill_cols = (int32_t)(N & ~3ll);
  if (p.clean && p.vec_ok && p.fill_cols > 0) {
    const uint64_t dims[2] = {(uint64_t)p.fill_cols, (uint64_t)M};
    const uint64_t strides[1] = {(uint64_t)p.out_stride * 4u};
    const uint32_t box[2] = {(uint32_t)kTileTokens, (uint32_t)plan.block_m};
    TRY(encode(&tm_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, out->data, dims, strides, box,
               CU_TENSOR_MAP_SWIZZLE_NONE, "out"));
    p.tma_fill = 1;
  }
  cudaError_t e = launch_prefill(tm_q, tm_k, tm_s, tm_w, tm_out, p, (int)H, (int)D, paged, plan.grid, plan.smem_bytes,
                                 static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  return ok();
}

// ------------------------------------------------------------------ top-k
// mode 0: prefill windows from ks/ke over the row width; mode 1: decode
// windows from context_lens/next_n within max_model_len columns.
fp8idx_status topk_impl(int mode, const fp8idx_tensor* logits, const fp8idx_tensor* ks, const fp8idx_tensor* ke,
                        const fp8idx_tensor* cl, int32_t next_n, int32_t max_model_len, int32_t k,
                        const fp8idx_tensor* indices, const fp8idx_options* opts, void* stream) {
  g_last_error.clear();
  TRY(check_tensor(logits, "logits", FP8IDX_F32, 2));
  TRY(check_tensor(indices, "indices", FP8IDX_I32, 2));
  const int64_t R = logits->shape[0], W = logits->shape[1];
  if (k < 1 || k > kTopkMaxK) return fail(FP8IDX_ERR_UNSUPPORTED, "top-k: k=%d not in [1, %d]", k, kTopkMaxK);
  if (W > 1 && logits->stride[1] != 1) return fail(FP8IDX_ERR_INVALID, "logits must have unit inner stride");
  if (R > 1 && logits->stride[0] < W) return fail(FP8IDX_ERR_INVALID, "logits rows overlap");
  if (indices->shape[0] != R || indices->shape[1] != k || (k > 1 && indices->stride[1] != 1) ||
      (R > 1 && indices->stride[0] < k))
    return fail(FP8IDX_ERR_INVALID, "indices must be [rows, k] with unit inner stride");
  if (W >= (1ll << 31) || R * kTopkMaxCluster >= (1ll << 31))
    return fail(FP8IDX_ERR_UNSUPPORTED, "top-k: logits too large");
  const int32_t ctas_req = opts ? opts->num_ctas : 0;
  if (ctas_req < 0 || ctas_req > kTopkMaxCluster)
    return fail(FP8IDX_ERR_UNSUPPORTED, "top-k: num_ctas=%d not in [0, %d]", ctas_req, kTopkMaxCluster);
  TopkParams p;
  std::memset(&p, 0, sizeof(p));
  p.mode = mode;
  p.k = k;
  p.rows = (int32_t)R;
  if (mode == 0) {
    TRY(check_tensor(ks, "cu_seqlen_ks", FP8IDX_I32, 1));
    TRY(check_tensor(ke, "cu_seqlen_ke", FP8IDX_I32, 1));
    if (ks->shape[0] != R || ke->shape[0] != R || !contiguous(ks) || !contiguous(ke))
      return fail(FP8IDX_ERR_INVALID, "cu_seqlen_ks/ke must be contiguous [rows]");
    p.ks = static_cast<const int32_t*>(ks->data);
    p.ke = static_cast<const int32_t*>(ke->data);
    p.cols = (int32_t)W;
    p.next_n = 1;
  } else {
    TRY(check_tensor(cl, "context_lens", FP8IDX_I32, 1));
    if (next_n < 1) return fail(FP8IDX_ERR_INVALID, "next_n must be positive");
    if (!contiguous(cl) || cl->shape[0] * next_n != R)
      return fail(FP8IDX_ERR_INVALID, "context_lens must be contiguous [rows / next_n]");
    if (max_model_len < 0 || max_model_len > W)
      return fail(FP8IDX_ERR_INVALID, "max_model_len must be in [0, logits width]");
    p.context_lens = static_cast<const int32_t*>(cl->data);
    p.cols = max_model_len;
    p.next_n = next_n;
  }
  if (R == 0) return ok();
  p.logits = static_cast<const float*>(logits->data);
  p.stride = R > 1 ? logits->stride[0] : W;
  p.out = static_cast<int32_t*>(indices->data);
  p.out_stride = R > 1 ? indices->stride[0] : k;
  p.vec_ok = (aligned16(logits->data) && (p.stride % 4) == 0) ? 1 : 0;
  DeviceInfo dev;
  TRY(device_info(&dev));
  // CTAs per row: a cluster per row only when the rows leave most SMs idle
  // (at most a quarter of the SM count) and the longest possible window
  // gives each CTA at least kTopkMinSlice values; with more rows the
  // cluster's barriers cost more than the extra SMs return (measured).
  int ctas = 1;
  if (p.cols >= 2 * kTopkMinSlice && 4 * R <= dev.sms) {
    const int64_t by_rows = dev.sms / R, by_len = p.cols / kTopkMinSlice;
    ctas = (int)std::min<int64_t>(kTopkMaxCluster, std::min(by_rows, by_len));
    if (ctas < 2) ctas = 1;
  }
  if (ctas_req > 0) ctas = ctas_req;
  int cap = kTopkMaxCap;
  while (cap > 1024 && (int)topk_smem_layout(cap).total > dev.smem_optin) cap >>= 1;
  p.cap = cap;
  cudaError_t e = launch_topk(p, ctas, (int)topk_smem_layout(cap).total, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "top-k launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

fp8idx_status fp8_paged_mqa_logits(const fp8idx_tensor* q_fp8, const fp8idx_tensor* kv_cache,
                                   const fp8idx_tensor* weights, const fp8idx_tensor* context_lens,
                                   const fp8idx_tensor* block_tables, int32_t max_model_len,
                                   const fp8idx_tensor* out, void* stream) {
  return paged_impl(q_fp8, kv_cache, weights, context_lens, block_tables, max_model_len, out, nullptr, stream);
}

fp8idx_status fp8_paged_mqa_logits_ex(const fp8idx_tensor* q_fp8, const fp8idx_tensor* kv_cache,
                                      const fp8idx_tensor* weights, const fp8idx_tensor* context_lens,
                                      const fp8idx_tensor* block_tables, int32_t max_model_len,
                                      const fp8idx_tensor* out, const fp8idx_options* opts, void* stream) {
  return paged_impl(q_fp8, kv_cache, weights, context_lens, block_tables, max_model_len, out, opts, stream);
}

fp8idx_status fp8_mqa_logits(const fp8idx_tensor* q_fp8, const fp8idx_tensor* k_fp8, const fp8idx_tensor* kv_scale,
                             const fp8idx_tensor* weights, const fp8idx_tensor* cu_seqlen_ks,
                             const fp8idx_tensor* cu_seqlen_ke, const fp8idx_tensor* out, void* stream) {
  PrefillK src;
  src.k = k_fp8;
  src.s = kv_scale;
  return prefill_impl(q_fp8, src, weights, cu_seqlen_ks, cu_seqlen_ke, out, nullptr, stream);
}

fp8idx_status fp8_mqa_logits_ex(const fp8idx_tensor* q_fp8, const fp8idx_tensor* k_fp8,
                                const fp8idx_tensor* kv_scale, const fp8idx_tensor* weights,
                                const fp8idx_tensor* cu_seqlen_ks, const fp8idx_tensor* cu_seqlen_ke,
                                const fp8idx_tensor* out, const fp8idx_options* opts, void* stream) {
  PrefillK src;
  src.k = k_fp8;
  src.s = kv_scale;
  return prefill_impl(q_fp8, src, weights, cu_seqlen_ks, cu_seqlen_ke, out, opts, stream);
}

fp8idx_status fp8_mqa_logits_paged(const fp8idx_tensor* q_fp8, const fp8idx_tensor* kv_cache,
                                   const fp8idx_tensor* block_tables, const fp8idx_tensor* cu_seq_lens,
                                   const fp8idx_tensor* weights, const fp8idx_tensor* cu_seqlen_ks,
                                   const fp8idx_tensor* cu_seqlen_ke, const fp8idx_tensor* out,
                                   const fp8idx_options* opts, void* stream) {
  PrefillK src;
  src.kv = kv_cache;
  src.bt = block_tables;
  src.cu = cu_seq_lens;
  return prefill_impl(q_fp8, src, weights, cu_seqlen_ks, cu_seqlen_ke, out, opts, stream);
}

fp8idx_status fp8_paged_mqa_topk(const fp8idx_tensor* q_fp8, const fp8idx_tensor* kv_cache,
                                 const fp8idx_tensor* weights, const fp8idx_tensor* context_lens,
                                 const fp8idx_tensor* block_tables, int32_t max_model_len, int32_t k,
                                 const fp8idx_tensor* indices, void* workspace, size_t workspace_bytes,
                                 const fp8idx_options* opts, void* stream) {
  return paged_topk_impl(q_fp8, kv_cache, weights, context_lens, block_tables, max_model_len, k, indices, workspace,
                         workspace_bytes, opts, stream);
}

size_t fp8idx_paged_mqa_topk_workspace(int64_t batch, int32_t next_n, int32_t max_model_len, int32_t k) {
  if (batch < 0 || next_n < 1 || max_model_len < 0 || k < 1 || k > kTopkMaxK) return 0;
  return paged_topk_workspace(batch, next_n, max_model_len, k);
}

fp8idx_status fp8_paged_topk(const fp8idx_tensor* logits, const fp8idx_tensor* context_lens, int32_t next_n,
                             int32_t max_model_len, int32_t k, const fp8idx_tensor* indices, void* stream) {
  return topk_impl(1, logits, nullptr, nullptr, context_lens, next_n, max_model_len, k, indices, nullptr, stream);
}

fp8idx_status fp8_mqa_topk(const fp8idx_tensor* logits, const fp8idx_tensor* cu_seqlen_ks,
                           const fp8idx_tensor* cu_seqlen_ke, int32_t k, const fp8idx_tensor* indices, void* stream) {
  return topk_impl(0, logits, cu_seqlen_ks, cu_seqlen_ke, nullptr, 1, 0, k, indices, nullptr, stream);
}
fp8idx_status fp8_paged_topk_ex(const fp8idx_tensor* logits, const fp8idx_tensor* context_lens, int32_t next_n,
                                int32_t max_model_len, int32_t k, const fp8idx_tensor* indices,
                                const fp8idx_options* opts, void* stream) {
  return topk_impl(1, logits, nullptr, nullptr, context_lens, next_n, max_model_len, k, indices, opts, stream);
}
fp8idx_status fp8_mqa_topk_ex(const fp8idx_tensor* logits, const fp8idx_tensor* cu_seqlen_ks,
                              const fp8idx_tensor* cu_seqlen_ke, int32_t k, const fp8idx_tensor* indices,
                              const fp8idx_options* opts, void* stream) {
  return topk_impl(0, logits, cu_seqlen_ks, cu_seqlen_ke, nullptr, 1, 0, k, indices, opts, stream);
}

int fp8idx_paged_is_supported(int32_t heads, int32_t head_dim, int32_t block_size, int32_t next_n) {
  return paged_supported(heads, head_dim, block_size, next_n) ? 1 : 0;
}

int fp8idx_prefill_is_supported(int32_t heads, int32_t head_dim) { return prefill_supported(heads, head_dim) ? 1 : 0; }

int fp8idx_is_supported(int32_t heads, int32_t head_dim, int32_t kv_block_size, int32_t next_n) {
  return paged_supported(heads, head_dim, kv_block_size, next_n) ? 1 : 0;
}

fp8idx_status fp8idx_plan_paged(int32_t batch, int32_t next_n, int32_t heads, int32_t head_dim, int32_t block_size,
                                int32_t max_model_len, int32_t num_sms, const fp8idx_options* opts,
                                fp8idx_plan* plan) {
  g_last_error.clear();
  if (!plan) return fail(FP8IDX_ERR_INVALID, "plan: null output");
  int smem = kMaxSmem;
  if (num_sms <= 0) {
    DeviceInfo dev;
    TRY(device_info(&dev));
    num_sms = dev.sms;
    smem = dev.smem_optin;
  }
  return plan_paged(batch, next_n, heads, head_dim, block_size, max_model_len, num_sms, smem, opts, plan);
}

fp8idx_status fp8idx_plan_prefill(int64_t rows, int64_t cols, int32_t heads, int32_t head_dim, int32_t num_sms,
                                  const fp8idx_options* opts, fp8idx_plan* plan) {
  g_last_error.clear();
  if (!plan) return fail(FP8IDX_ERR_INVALID, "plan: null output");
  int smem = kMaxSmem;
  if (num_sms <= 0) {
    DeviceInfo dev;
    TRY(device_info(&dev));
    num_sms = dev.sms;
    smem = dev.smem_optin;
  }
  return plan_prefill(rows, cols, heads, head_dim, num_sms, smem, opts, plan);
}

const char* fp8idx_last_error(void) { return g_last_error.c_str(); }

fp8idx_status fp8idx_host_mapped_pointer(const void* host_ptr, void** device_ptr) {
  g_last_error.clear();
  if (host_ptr == nullptr || device_ptr == nullptr) return fail(FP8IDX_ERR_INVALID, "host_mapped_pointer: null argument");
  cudaPointerAttributes a;
  std::memset(&a, 0, sizeof(a));
  const cudaError_t e = cudaPointerGetAttributes(&a, host_ptr);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(FP8IDX_ERR_INVALID, "host_mapped_pointer: %s", cudaGetErrorString(e));
  }
  if (a.type != cudaMemoryTypeHost) return fail(FP8IDX_ERR_INVALID, "host_mapped_pointer: not page-locked host memory");
  if (a.devicePointer == nullptr)
    return fail(FP8IDX_ERR_UNSUPPORTED, "host_mapped_pointer: the memory is not mapped into the device");
  *device_ptr = a.devicePointer;
  return ok();
}

fp8idx_status fp8idx_device_status(int32_t clear) {
  g_last_error.clear();
  unsigned int a = 0, b = 0, c = 0;
  if (read_paged_watchdog(&a, clear != 0) != cudaSuccess || read_prefill_watchdog(&b, clear != 0) != cudaSuccess ||
      read_topk_watchdog(&c, clear != 0) != cudaSuccess)
    return fail(FP8IDX_ERR_CUDA, "reading the device watchdog failed");
  if (a | b | c)
    return fail(FP8IDX_ERR_TIMEOUT, "device wait timed out (decode sites 0x%x, prefill sites 0x%x, top-k sites 0x%x)",
                a, b, c);
  return FP8IDX_OK;
}

fp8idx_status fp8idx_watchdog_selftest(int32_t limit_us, void* stream) {
  g_last_error.clear();
  if (limit_us < 1 || limit_us > 100000) return fail(FP8IDX_ERR_INVALID, "limit_us %d not in [1, 100000]", limit_us);
  DeviceInfo dev;
  TRY(device_info(&dev));
  cudaError_t e = launch_watchdog_selftest(static_cast<uint64_t>(limit_us) * 1000ull, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FP8IDX_ERR_CUDA, "watchdog self-test launch: %s", cudaGetErrorString(e));
  return ok();
}

int32_t fp8idx_version(void) { return 102; }

}  // extern "C"
