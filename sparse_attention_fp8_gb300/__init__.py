"""GB300-native FP8 lightning-indexer logits.

Thin Python binding over the C-ABI library ``libfp8idx.so`` (see
``include/fp8idx.h``): it only marshals torch CUDA tensors into descriptors
and calls the library; every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is missing the
import of the binding raises.

    logits[m, n] = sum_h relu(<Q[m,h,:], K[n,:]>) * kv_scale[n] * weights[m,h]

Entry points (same names as the C ABI):
  fp8_paged_mqa_logits(q_fp8, kv_cache, weights, context_lens, block_tables,
                       max_model_len, out, stream=None, options=None)
  fp8_mqa_logits(q_fp8, k_fp8, kv_scale, weights, cu_seqlen_ks, cu_seqlen_ke,
                 out, stream=None, options=None, clean_logits=True)
  fp8_mqa_logits_paged(q_fp8, kv_cache, block_tables, cu_seq_lens, weights,
                       cu_seqlen_ks, cu_seqlen_ke, out, stream=None,
                       options=None, clean_logits=True)
  fp8_paged_topk(logits, context_lens, next_n, max_model_len, k, indices,
                 stream=None)
  fp8_mqa_topk(logits, cu_seqlen_ks, cu_seqlen_ke, k, indices, stream=None)
  fp8_paged_mqa_topk(q_fp8, kv_cache, weights, context_lens, block_tables,
                     max_model_len, k, indices, workspace=None, stream=None)
"""
from ._native import (  # noqa: F401
    FP8IDX_ERR_CUDA,
    FP8IDX_ERR_INVALID,
    FP8IDX_ERR_TIMEOUT,
    FP8IDX_ERR_UNSUPPORTED,
    FP8IDX_OK,
    Fp8IdxError,
    Options,
    Plan,
    device_status,
    device_status_message,
    fp8_mqa_logits,
    fp8_mqa_logits_paged,
    fp8_mqa_topk,
    fp8_paged_mqa_logits,
    fp8_paged_mqa_topk,
    fp8_paged_topk,
    is_supported,
    library,
    library_path,
    paged_mqa_topk_workspace,
    paged_is_supported,
    plan_paged,
    plan_prefill,
    prefill_is_supported,
    version,
    watchdog_selftest,
)
