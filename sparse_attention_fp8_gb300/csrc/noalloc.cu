// fp8_paged_mqa_topk for callers that cannot allocate device memory.
//
// The fused decode top-k needs scratch memory between its kernels.  Most
// callers pass it in, but some cannot obtain any: a serving engine that
// hands all free device memory to its KV-cache pool at start-up and forbids
// later allocation, a plugin inside a host framework that exposes no
// allocator to it, or code on a latency-critical path where a cudaMalloc
// (which can synchronise the device) is not acceptable.  For them this file
// keeps one fixed scratch area in the library itself, a static device array
// that every GPU loading the library holds until the process exits, and an
// entry point that uses it in place of a caller's workspace.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "fp8idx.h"
#include "kernels.h"

namespace fp8idx {
void set_last_error_message(const char* msg);
}

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB

// The scratch itself.  In host code this name is only a stand-in for the
// device object: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mu;

// The array's device address on the current device, looked up once per
// device (the first call of the entry point on that device does it).
fp8idx_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    fp8idx::set_last_error_message("cudaGetDevice failed");
    return FP8IDX_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    fp8idx::set_last_error_message("device index out of range");
    return FP8IDX_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ready[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char buf[160];
      std::snprintf(buf, sizeof(buf), "cudaGetSymbolAddress of the static scratch failed: %s",
                    cudaGetErrorString(e));
      fp8idx::set_last_error_message(buf);
      return FP8IDX_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
    g_scratch_ready[dev] = true;
  }
  *out = g_scratch_addr[dev];
  return FP8IDX_OK;
}

}  // namespace

extern "C" fp8idx_status fp8_paged_mqa_topk_noalloc(const fp8idx_tensor* q_fp8, const fp8idx_tensor* kv_cache,
                                                    const fp8idx_tensor* weights,
                                                    const fp8idx_tensor* context_lens,
                                                    const fp8idx_tensor* block_tables, int32_t max_model_len,
                                                    int32_t k, const fp8idx_tensor* indices,
                                                    const fp8idx_options* opts, void* stream) {
  if (q_fp8 == nullptr || q_fp8->ndim != 4) {
    fp8idx::set_last_error_message("q_fp8: expected [batch, next_n, heads, head_dim]");
    return FP8IDX_ERR_INVALID;
  }
  const size_t need = fp8idx_paged_mqa_topk_workspace(q_fp8->shape[0], static_cast<int32_t>(q_fp8->shape[1]),
                                                      max_model_len, k);
  if (need > kStaticScratchBytes) {
    char buf[200];
    std::snprintf(buf, sizeof(buf),
                  "this shape needs %zu bytes of scratch; the library's static scratch holds %zu "
                  "(use fp8_paged_mqa_topk with a workspace)",
                  need, kStaticScratchBytes);
    fp8idx::set_last_error_message(buf);
    return FP8IDX_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  const fp8idx_status st = scratch_address(&scratch);
  if (st != FP8IDX_OK) return st;
  return fp8_paged_mqa_topk(q_fp8, kv_cache, weights, context_lens, block_tables, max_model_len, k, indices, scratch,
                            kStaticScratchBytes, opts, stream);
}
