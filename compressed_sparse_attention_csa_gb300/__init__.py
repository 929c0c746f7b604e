"""Compressed Sparse Attention (CSA) hot path for one NVIDIA GB300 (sm_103a).

The computation lives in libcsa (hand-written CUDA, C ABI in include/csa.h); this package is
its thin Python binding.  See :mod:`compressed_sparse_attention_csa_gb300.ops`.
"""
from .ops import (Config, CsaError, DecodeStepCall, HcaDecodeStepCall, NormRope, block_pool, compress_kv, compress_kv_norm_rope,  # noqa: F401
                  compress_kv_single, decode_step, decode_step_reset, dense_attn, get_last_error, hca_decode_step, indexer_scores,
                  indexer_topk, inverse_rope_quant, kv_pack_fp8, kv_pack_mxfp4, compress_kv_norm_rope_fp8kv,
                  launch_count, norm_rope, StepInputs, sparse_attn, sparse_attn_fp8kv, sparse_attn_mxfp4kv, topk, version,
                  workspace_size)
