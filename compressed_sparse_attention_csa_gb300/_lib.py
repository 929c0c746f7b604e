"""ctypes view of libcsa's C ABI (include/csa.h).  Loads the in-tree library and fails
loudly when it is missing: there is no fallback implementation."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcsa.so")

c_i32, c_i64, c_f32, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

CSA_F32, CSA_BF16, CSA_E4M3, CSA_MXFP4 = 0, 1, 2, 3
(CSA_OP_COMPRESS, CSA_OP_INDEXER, CSA_OP_TOPK, CSA_OP_ATTN, CSA_OP_DECODE, CSA_OP_POOL, CSA_OP_INDEXER_TOPK,
 CSA_OP_DENSE_ATTN, CSA_OP_HCA_DECODE, CSA_OP_TOPK_BF16, CSA_OP_INDEXER_TOPK_BF16) = range(11)
STATUS = {0: "CSA_OK", 1: "CSA_ERR_NULL", 2: "CSA_ERR_SHAPE", 3: "CSA_ERR_DTYPE", 4: "CSA_ERR_ALIGN",
          5: "CSA_ERR_WORKSPACE", 6: "CSA_ERR_CUDA", 7: "CSA_ERR_TIMEOUT", 8: "CSA_ERR_INDEX"}


class csa_config(ctypes.Structure):
    _fields_ = [("B", c_i32), ("H", c_i32), ("d", c_i32), ("HI", c_i32), ("dI", c_i32), ("m", c_i32),
                ("k", c_i32), ("W", c_i32), ("act", ctypes.c_int), ("kidx", ctypes.c_int),
                ("softmax_scale", c_f32)]


class csa_decode_args(ctypes.Structure):
    _fields_ = [("E_cap", c_i64), ("q_pos", c_vp), ("q", c_vp), ("qI", c_vp), ("w", c_vp), ("sink", c_vp),
                ("kv_comp", c_vp), ("kI", c_vp), ("kscale", c_vp), ("kv_tail", c_vp), ("z_tail", c_vp),
                ("kvI_tail", c_vp), ("zI_tail", c_vp), ("bias", c_vp), ("biasI", c_vp), ("kv_local", c_vp),
                ("L", c_i64), ("local_base", c_vp), ("out", c_vp), ("lse", c_vp), ("idx_out", c_vp),
                ("scores_out", c_vp), ("bf16_scores", ctypes.c_int32)]


class csa_hca_decode_args(ctypes.Structure):
    _fields_ = [("E_cap", c_i64), ("q_pos", c_vp), ("q", c_vp), ("sink", c_vp), ("kv_comp", c_vp),
                ("kv_tail", c_vp), ("z_tail", c_vp), ("bias", c_vp), ("kv_local", c_vp), ("L", c_i64),
                ("local_base", c_vp), ("out", c_vp), ("lse", c_vp)]


class csa_norm_rope(ctypes.Structure):
    _fields_ = [("norm_weight", c_vp), ("eps", c_f32), ("rope_dims", c_i32), ("rope_theta", c_f32)]


# name -> (restype, argtypes); the exported symbols of include/csa.h
SIGNATURES = {
    "csa_version": (c_i32, []),
    "csa_launch_count": (c_i64, []),
    "csa_debug_set": (ctypes.c_int, [ctypes.c_int, c_i64]),
    "csa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "csa_get_last_error": (ctypes.c_int, [c_vp]),
    "csa_workspace_size": (c_sz, [ctypes.c_int, ctypes.POINTER(csa_config), c_i64, c_i64]),
    "csa_block_pool_workspace_size": (c_sz, [c_i64, c_i64, c_i32, c_i32]),
    "csa_compress_kv": (ctypes.c_int, [ctypes.POINTER(csa_config), c_i32, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64,
                                       c_i64, c_vp, ctypes.c_int, c_vp, c_i64, c_vp]),
    "csa_compress_kv_single": (ctypes.c_int, [ctypes.POINTER(csa_config), c_i32, c_vp, c_vp, c_vp, c_i64, c_i64,
                                              c_i64, c_i64, c_vp, c_i64, c_vp]),
    "csa_indexer_scores": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_vp, c_i32, c_vp, c_vp, c_vp, c_i64,
                                          c_vp, c_i32, c_vp, c_i64, c_vp, c_sz, c_vp]),
    "csa_indexer_scores_bf16": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_vp, c_i32, c_vp, c_vp, c_vp,
                                               c_i64, c_vp, c_i32, c_vp, c_i64, c_vp, c_sz, c_vp]),
    "csa_indexer_topk": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_vp, c_i32, c_vp, c_vp, c_vp, c_i64,
                                        c_vp, c_vp, c_sz, c_vp]),
    "csa_indexer_topk_bf16": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_vp, c_i32, c_vp, c_vp, c_vp,
                                             c_i64, c_vp, c_vp, c_sz, c_vp]),
    "csa_topk": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp, c_vp,
                                c_sz, c_vp]),
    "csa_topk_bf16": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp,
                                     c_vp, c_sz, c_vp]),
    "csa_topk_noalloc": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_vp,
                                        c_vp]),
    "csa_block_pool": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i64, c_i64, c_i64, c_vp, c_i32, c_i32,
                                      c_vp, c_vp, c_vp, c_sz, c_vp]),
    "csa_sparse_attn": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i32, c_vp, c_i64, c_vp, c_vp, c_i64,
                                       c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "csa_dense_attn": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i32, c_vp, c_i64, c_vp, c_i64, c_vp, c_vp,
                                      c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "csa_hca_decode_step": (ctypes.c_int, [ctypes.POINTER(csa_config), ctypes.POINTER(csa_hca_decode_args), c_vp,
                                           c_sz, c_vp]),
    "csa_norm_rope_apply": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_vp, c_i64, c_i32, c_i32, c_vp,
                                           ctypes.POINTER(csa_norm_rope), c_vp]),
    "csa_compress_kv_norm_rope": (ctypes.c_int, [ctypes.POINTER(csa_config), c_i32, c_i32, c_vp, c_vp, c_vp, c_i64,
                                                 c_i64, c_i64, c_i64, c_vp, c_i64, ctypes.POINTER(csa_norm_rope), c_vp]),
    "csa_inverse_rope_quant": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i64, c_vp, c_i32, c_f32, c_vp,
                                              ctypes.c_int, c_vp, c_vp]),
    "csa_kv_pack_fp8": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i64, c_i32, c_vp, c_vp]),
    "csa_compress_kv_norm_rope_fp8kv": (ctypes.c_int, [ctypes.POINTER(csa_config), c_i32, c_i32, c_vp, c_vp, c_vp,
                                                       c_i64, c_i64, c_i64, c_i64, c_vp, c_i64,
                                                       ctypes.POINTER(csa_norm_rope), c_vp]),
    "csa_sparse_attn_fp8kv": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i32, c_vp, c_i64, c_vp, c_vp, c_i64,
                                             c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "csa_kv_pack_mxfp4": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i64, c_i32, c_vp, c_vp]),
    "csa_sparse_attn_mxfp4kv": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_i32, c_vp, c_i64, c_vp, c_vp,
                                               c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "csa_decode_step": (ctypes.c_int, [ctypes.POINTER(csa_config), ctypes.POINTER(csa_decode_args), c_vp, c_sz,
                                       c_vp]),
    "csa_decode_step_fp8kv": (ctypes.c_int, [ctypes.POINTER(csa_config), ctypes.POINTER(csa_decode_args), c_vp, c_sz,
                                             c_vp]),
    "csa_decode_step_mxfp4kv": (ctypes.c_int, [ctypes.POINTER(csa_config), ctypes.POINTER(csa_decode_args), c_vp, c_sz,
                                             c_vp]),
    "csa_decode_step_reset": (ctypes.c_int, [ctypes.POINTER(csa_config), c_vp, c_sz, c_vp]),
}

_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libcsa (building it first if the toolkit is present and the file is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            from . import build as _build
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libcsa not found at {path}; run compressed_sparse_attention_csa_gb300.build")
        import torch  # noqa: F401  (loads the CUDA runtime libcsa links against)
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
