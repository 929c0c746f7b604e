"""Python binding of libcsa: the same calls as include/csa.h, taking torch tensors.

Argument marshalling only: shapes and dtypes are checked, device pointers and the current
CUDA stream are passed to the C ABI, and the scratch workspace the library asks for is
allocated here (torch owns device memory; the library allocates nothing).  Every step of
the computation runs in libcsa's kernels.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib as L


class CsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {L.STATUS.get(status, status)}")
        self.status = status


@dataclass
class Config:
    B: int
    H: int
    d: int
    HI: int
    dI: int
    m: int
    k: int
    W: int
    act: torch.dtype = torch.bfloat16          # torch.float32 or torch.bfloat16
    fp8_keys: bool = False                     # indexer keys stored as e4m3 + fp32 scale
    softmax_scale: Optional[float] = None      # default 1/sqrt(d)
    mx_keys: bool = False                      # indexer keys stored as MXFP4 (payload + scale words)

    def c(self) -> L.csa_config:
        act = L.CSA_F32 if self.act == torch.float32 else L.CSA_BF16
        scale = self.softmax_scale if self.softmax_scale is not None else self.d ** -0.5
        kidx = L.CSA_MXFP4 if self.mx_keys else L.CSA_E4M3 if self.fp8_keys else act
        return L.csa_config(self.B, self.H, self.d, self.HI, self.dI, self.m, self.k, self.W, act, kidx, scale)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libcsa takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libcsa takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn: str, st: int):
    if st != 0:
        raise CsaError(fn, st)


_ws_cache = {}


def _workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    if nbytes == ctypes.c_size_t(-1).value:
        raise CsaError("csa_workspace_size", 2)
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


_decode_ws = {}


def _decode_workspace(nbytes: int, device, batch: int) -> torch.Tensor:
    """The decode step's own workspace, zero-filled when allocated: its first bytes carry the
    top-k histograms from step to step, laid out by the batch size (one per device and batch
    size; steps on it must be stream-ordered)."""
    key = (str(device), batch)
    buf = _decode_ws.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        _decode_ws[key] = buf
    return buf


def _ws_args(buf):
    return (None, 0) if buf is None else (ctypes.c_void_p(buf.data_ptr()), buf.numel())


def version() -> int:
    return L.load().csa_version()


def launch_count() -> int:
    """Kernels enqueued through libcsa by this process so far."""
    return L.load().csa_launch_count()


def get_last_error() -> int:
    """Synchronise the current stream and return (and clear) the device error word."""
    return L.load().csa_get_last_error(_stream())


def workspace_size(op: int, cfg: Config, rows: int, n_cols: int) -> int:
    c = cfg.c()
    return L.load().csa_workspace_size(op, ctypes.byref(c), rows, n_cols)


def compress_kv(cfg: Config, kv: torch.Tensor, z: torch.Tensor, bias: torch.Tensor, tok0: int, ent_begin: int,
                ent_end: int, out: torch.Tensor, out_scale: Optional[torch.Tensor] = None) -> None:
    """csa_compress_kv: kv, z [B, n_tok, 2, dim]; bias [2, m, dim] fp32; out [B, E_cap, dim] (fp32,
    bf16, or e4m3 codes with out_scale [B, E_cap] fp32), or MXFP4 keys: out [B, E_cap, dim/2]
    uint8 payload with out_scale [B, E_cap] int32 scale words."""
    lib = L.load()
    c = cfg.c()
    dim = kv.shape[-1]
    if out.dtype == torch.float32:
        od = L.CSA_F32
    elif out.dtype == torch.bfloat16:
        od = L.CSA_BF16
    elif out.dtype == torch.uint8:
        od = L.CSA_MXFP4 if out.shape[-1] * 2 == dim else L.CSA_E4M3
    else:
        raise ValueError("out dtype")
    _check("csa_compress_kv", lib.csa_compress_kv(ctypes.byref(c), dim, _p(kv), _p(z), _p(bias), kv.shape[1], tok0,
                                                  ent_begin, ent_end, _p(out), od, _p(out_scale), out.shape[1],
                                                  _stream()))


def compress_kv_single(cfg: Config, kv: torch.Tensor, z: torch.Tensor, bias: Optional[torch.Tensor], tok0: int,
                       ent_begin: int, ent_end: int, out: torch.Tensor) -> None:
    """csa_compress_kv_single (one stream, no overlap; ratio cfg.m): kv, z [B, n_tok, dim];
    bias [m, dim] fp32 or None; out [B, E_cap, dim] in cfg.act."""
    lib = L.load()
    c = cfg.c()
    _check("csa_compress_kv_single",
           lib.csa_compress_kv_single(ctypes.byref(c), kv.shape[-1], _p(kv), _p(z), _p(bias), kv.shape[1], tok0,
                                      ent_begin, ent_end, _p(out), out.shape[1], _stream()))


def indexer_scores(cfg: Config, qI: torch.Tensor, w: torch.Tensor, q_pos: torch.Tensor, kI: torch.Tensor,
                   scores: torch.Tensor, kscale: Optional[torch.Tensor] = None,
                   cand: Optional[torch.Tensor] = None) -> None:
    """csa_indexer_scores: qI [B, T, HI, dI], w [B, T, HI], kI [B, E_cap, dI] (+ kscale); scores
    fp32, or bfloat16 (csa_indexer_scores_bf16: each score rounded to BF16)."""
    lib = L.load()
    c = cfg.c()
    T = qI.shape[1]
    n_cand = cand.shape[-1] if cand is not None else 0
    ws = _workspace(lib.csa_workspace_size(L.CSA_OP_INDEXER, ctypes.byref(c), cfg.B * T, T), qI.device)
    wp, wb = _ws_args(ws)
    bf16 = scores.dtype == torch.bfloat16
    fn = lib.csa_indexer_scores_bf16 if bf16 else lib.csa_indexer_scores
    _check("csa_indexer_scores_bf16" if bf16 else "csa_indexer_scores",
           fn(ctypes.byref(c), _p(qI), _p(w), T, _p(q_pos), _p(kI), _p(kscale), kI.shape[1],
              _p(cand), n_cand, _p(scores), scores.shape[-1], wp, wb, _stream()))


def indexer_topk(cfg: Config, qI: torch.Tensor, w: torch.Tensor, q_pos: torch.Tensor, kI: torch.Tensor,
                 idx: torch.Tensor, kscale: Optional[torch.Tensor] = None, bf16_scores: bool = False) -> None:
    """csa_indexer_topk (csa_indexer_topk_bf16 with bf16_scores): the k best visible entries of
    every query row (ascending, -1 padded), the scores kept in the call's workspace.
    qI [B, T, HI, dI], w [B, T, HI], kI [B, E_cap, dI]."""
    lib = L.load()
    c = cfg.c()
    T = qI.shape[1]
    E_cap = kI.shape[1]
    op = L.CSA_OP_INDEXER_TOPK_BF16 if bf16_scores else L.CSA_OP_INDEXER_TOPK
    ws = _workspace(lib.csa_workspace_size(op, ctypes.byref(c), cfg.B * T, E_cap), qI.device)
    wp, wb = _ws_args(ws)
    fn = lib.csa_indexer_topk_bf16 if bf16_scores else lib.csa_indexer_topk
    _check("csa_indexer_topk_bf16" if bf16_scores else "csa_indexer_topk",
           fn(ctypes.byref(c), _p(qI), _p(w), T, _p(q_pos), _p(kI), _p(kscale), E_cap, _p(idx), wp, wb, _stream()))


def topk(cfg: Config, scores: torch.Tensor, idx: torch.Tensor, n_valid: Optional[torch.Tensor] = None,
         cand: Optional[torch.Tensor] = None, n_cols: Optional[int] = None) -> None:
    """csa_topk: scores [rows, ld] fp32 (csa_topk_bf16: bfloat16) -> idx [rows, k] int32
    (ascending, -1 padded)."""
    lib = L.load()
    c = cfg.c()
    rows, ld = scores.shape
    n_cols = ld if n_cols is None else n_cols
    bf16 = scores.dtype == torch.bfloat16
    op = L.CSA_OP_TOPK_BF16 if bf16 else L.CSA_OP_TOPK
    ws = _workspace(lib.csa_workspace_size(op, ctypes.byref(c), rows, n_cols), scores.device)
    wp, wb = _ws_args(ws)
    fn = lib.csa_topk_bf16 if bf16 else lib.csa_topk
    _check("csa_topk_bf16" if bf16 else "csa_topk",
           fn(ctypes.byref(c), _p(scores), ld, rows, n_cols, _p(n_valid), _p(cand), _p(idx), wp, wb, _stream()))


def topk_noalloc(cfg: Config, scores: torch.Tensor, idx: torch.Tensor, n_valid: Optional[torch.Tensor] = None,
                 cand: Optional[torch.Tensor] = None, n_cols: Optional[int] = None) -> None:
    """csa_topk_noalloc: csa_topk using the library's fixed device scratch (no workspace)."""
    lib = L.load()
    c = cfg.c()
    rows, ld = scores.shape
    n_cols = ld if n_cols is None else n_cols
    _check("csa_topk_noalloc", lib.csa_topk_noalloc(ctypes.byref(c), _p(scores), ld, rows, n_cols, _p(n_valid),
                                                    _p(cand), _p(idx), _stream()))


def block_pool(cfg: Config, scores: torch.Tensor, pool: torch.Tensor, pool_count: Optional[torch.Tensor] = None,
               n_valid: Optional[torch.Tensor] = None, block: int = 8, n_blocks: int = 2048,
               n_cols: Optional[int] = None) -> None:
    """csa_block_pool: scores [rows, ld] -> pool [rows, n_blocks*block] int32 positions."""
    lib = L.load()
    c = cfg.c()
    rows, ld = scores.shape
    n_cols = ld if n_cols is None else n_cols
    ws = _workspace(lib.csa_block_pool_workspace_size(rows, n_cols, block, n_blocks), scores.device)
    wp, wb = _ws_args(ws)
    _check("csa_block_pool", lib.csa_block_pool(ctypes.byref(c), _p(scores), ld, rows, n_cols, _p(n_valid), block,
                                                n_blocks, _p(pool), _p(pool_count), wp, wb, _stream()))


def sparse_attn(cfg: Config, q: torch.Tensor, kv_comp: torch.Tensor, idx: torch.Tensor, kv_local: torch.Tensor,
                local_base: torch.Tensor, q_pos: torch.Tensor, sink: torch.Tensor, out: torch.Tensor,
                lse: Optional[torch.Tensor] = None) -> None:
    """csa_sparse_attn: q [B, T, H, d]; kv_comp [B, E_cap, d]; idx [B*T, k]; kv_local [B, L, d]."""
    lib = L.load()
    c = cfg.c()
    B, T = q.shape[0], q.shape[1]
    ws = _workspace(lib.csa_workspace_size(L.CSA_OP_ATTN, ctypes.byref(c), B * T, T), q.device)
    wp, wb = _ws_args(ws)
    _check("csa_sparse_attn",
           lib.csa_sparse_attn(ctypes.byref(c), _p(q), T, _p(kv_comp), kv_comp.shape[1], _p(idx), _p(kv_local),
                               kv_local.shape[1], _p(local_base), _p(q_pos), _p(sink), _p(out), _p(lse), wp, wb,
                               _stream()))


def decode_step(cfg: Config, *, q_pos, q, qI, w, sink, kv_comp, kI, kv_tail, z_tail, kvI_tail, zI_tail, bias,
                biasI, kv_local, local_base, out, kscale=None, lse=None, idx_out=None, scores_out=None,
                fp8kv: bool = False, bf16_scores: bool = False, mxfp4kv: bool = False) -> None:
    """csa_decode_step (csa_decode_step_fp8kv with fp8kv: kv_comp [B, E_cap, 576] uint8 FP8
    entries; csa_decode_step_mxfp4kv with mxfp4kv: [B, E_cap, 288] uint8 MXFP4 entries): one
    token per sequence (T = 1); caches are updated in place.  scores_out
    [B, E_cap] fp32 (optional; bfloat16 with bf16_scores) receives the indexer scores the step
    selected from.  bf16_scores: the scores are rounded to BF16 before the selection."""
    lib = L.load()
    c = cfg.c()
    a = L.csa_decode_args(kv_comp.shape[1], _p(q_pos), _p(q), _p(qI), _p(w), _p(sink), _p(kv_comp), _p(kI),
                          _p(kscale), _p(kv_tail), _p(z_tail), _p(kvI_tail), _p(zI_tail), _p(bias), _p(biasI),
                          _p(kv_local), kv_local.shape[1], _p(local_base), _p(out), _p(lse), _p(idx_out),
                          _p(scores_out), int(bf16_scores))
    nbytes = lib.csa_workspace_size(L.CSA_OP_DECODE, ctypes.byref(c), cfg.B, kv_comp.shape[1])
    if nbytes == ctypes.c_size_t(-1).value:
        raise CsaError("csa_workspace_size", 2)
    wp, wb = _ws_args(_decode_workspace(nbytes, q.device, cfg.B))
    fn = lib.csa_decode_step_mxfp4kv if mxfp4kv else lib.csa_decode_step_fp8kv if fp8kv else lib.csa_decode_step
    _check("csa_decode_step", fn(ctypes.byref(c), ctypes.byref(a), wp, wb, _stream()))


def decode_step_reset(cfg: Config, device=None) -> None:
    """csa_decode_step_reset on the decode workspace this binding keeps for (device, cfg.B):
    clears the state one step hands to the next, e.g. after a step that reported an error.
    Enqueued on the current stream; a no-op when no step has run on that workspace yet."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    buf = _decode_ws.get((str(device), cfg.B))
    if buf is None:
        return
    lib = L.load()
    c = cfg.c()
    wp, wb = _ws_args(buf)
    _check("csa_decode_step_reset", lib.csa_decode_step_reset(ctypes.byref(c), wp, wb, _stream()))


def dense_attn(cfg: Config, q: torch.Tensor, kv_comp: torch.Tensor, kv_local: torch.Tensor, local_base: torch.Tensor,
               q_pos: torch.Tensor, sink: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor] = None) -> None:
    """csa_dense_attn (HCA): every entry s < floor((q_pos+1)/cfg.m) of kv_comp [B, E_cap, d] plus
    the window rows of kv_local [B, L, d]; q [B, T, H, d]."""
    lib = L.load()
    c = cfg.c()
    B, T = q.shape[0], q.shape[1]
    E_cap = kv_comp.shape[1]
    ws = _workspace(lib.csa_workspace_size(L.CSA_OP_DENSE_ATTN, ctypes.byref(c), B * T, E_cap), q.device)
    wp, wb = _ws_args(ws)
    _check("csa_dense_attn",
           lib.csa_dense_attn(ctypes.byref(c), _p(q), T, _p(kv_comp), E_cap, _p(kv_local), kv_local.shape[1],
                              _p(local_base), _p(q_pos), _p(sink), _p(out), _p(lse), wp, wb, _stream()))


def hca_decode_step(cfg: Config, *, q_pos, q, sink, kv_comp, kv_tail, z_tail, bias, kv_local, local_base, out,
                    lse=None) -> None:
    """csa_hca_decode_step: one token per sequence (T = 1); kv_tail / z_tail [B, m, d] hold
    tokens t-m+1 .. t; kv_comp is updated in place when the token completes a block."""
    lib = L.load()
    c = cfg.c()
    a = L.csa_hca_decode_args(kv_comp.shape[1], _p(q_pos), _p(q), _p(sink), _p(kv_comp), _p(kv_tail), _p(z_tail),
                              _p(bias), _p(kv_local), kv_local.shape[1], _p(local_base), _p(out), _p(lse))
    ws = _workspace(lib.csa_workspace_size(L.CSA_OP_HCA_DECODE, ctypes.byref(c), cfg.B, kv_comp.shape[1]), q.device)
    wp, wb = _ws_args(ws)
    _check("csa_hca_decode_step", lib.csa_hca_decode_step(ctypes.byref(c), ctypes.byref(a), wp, wb, _stream()))


@dataclass
class NormRope:
    """RMSNorm weight [dim] fp32 (None: no RMSNorm), epsilon, rotated dims at the end of each
    head (0: no RoPE) and rotary base."""
    weight: Optional[torch.Tensor] = None
    eps: float = 1e-6
    rope_dims: int = 64
    theta: float = 10000.0

    def c(self) -> L.csa_norm_rope:
        return L.csa_norm_rope(_p(self.weight), self.eps, self.rope_dims, self.theta)


def norm_rope(cfg: Config, x: torch.Tensor, pos: torch.Tensor, nr: NormRope, out: Optional[torch.Tensor] = None) -> None:
    """csa_norm_rope_apply: x [rows, heads, dim] (or [B, T, heads, dim]), pos [rows] int64;
    writes out (default: in place)."""
    lib = L.load()
    c = cfg.c()
    y = x if out is None else out
    heads, dim = x.shape[-2], x.shape[-1]
    rows = x.numel() // (heads * dim)
    n = nr.c()
    _check("csa_norm_rope_apply",
           lib.csa_norm_rope_apply(ctypes.byref(c), _p(x), _p(y), rows, heads, dim, _p(pos), ctypes.byref(n), _stream()))


def compress_kv_norm_rope(cfg: Config, streams: int, kv: torch.Tensor, z: torch.Tensor, bias: Optional[torch.Tensor],
                          tok0: int, ent_begin: int, ent_end: int, out: torch.Tensor, nr: NormRope) -> None:
    """csa_compress_kv_norm_rope: streams 2 (kv, z [B, n_tok, 2, dim]) or 1 ([B, n_tok, dim]);
    out [B, E_cap, dim] in cfg.act."""
    lib = L.load()
    c = cfg.c()
    n = nr.c()
    _check("csa_compress_kv_norm_rope",
           lib.csa_compress_kv_norm_rope(ctypes.byref(c), streams, kv.shape[-1], _p(kv), _p(z), _p(bias), kv.shape[1],
                                         tok0, ent_begin, ent_end, _p(out), out.shape[1], ctypes.byref(n), _stream()))


def inverse_rope_quant(cfg: Config, o: torch.Tensor, pos: torch.Tensor, out: torch.Tensor,
                       out_scale: Optional[torch.Tensor] = None, rope_dims: int = 64, theta: float = 10000.0) -> None:
    """csa_inverse_rope_quant: o [rows, H, d] (or [B, T, H, d]) in cfg.act; out the same shape in
    cfg.act, or uint8 e4m3 codes with out_scale [rows, H] fp32."""
    lib = L.load()
    c = cfg.c()
    rows = o.numel() // (cfg.H * cfg.d)
    od = L.CSA_E4M3 if out.dtype == torch.uint8 else (L.CSA_BF16 if out.dtype == torch.bfloat16 else L.CSA_F32)
    _check("csa_inverse_rope_quant",
           lib.csa_inverse_rope_quant(ctypes.byref(c), _p(o), rows, _p(pos), rope_dims, theta, _p(out), od,
                                      _p(out_scale), _stream()))


def kv_pack_fp8(cfg: Config, x: torch.Tensor, out: torch.Tensor) -> None:
    """csa_kv_pack_fp8: rows x [..., dim] in cfg.act -> FP8 main-KV entries out [..., dim + 64] uint8."""
    lib = L.load()
    c = cfg.c()
    dim = x.shape[-1]
    _check("csa_kv_pack_fp8", lib.csa_kv_pack_fp8(ctypes.byref(c), _p(x), x.numel() // dim, dim, _p(out), _stream()))


def compress_kv_norm_rope_fp8kv(cfg: Config, streams: int, kv: torch.Tensor, z: torch.Tensor,
                                bias: Optional[torch.Tensor], tok0: int, ent_begin: int, ent_end: int, out: torch.Tensor,
                                nr: NormRope) -> None:
    """csa_compress_kv_norm_rope_fp8kv: as compress_kv_norm_rope, out [B, E_cap, dim + 64] uint8."""
    lib = L.load()
    c = cfg.c()
    n = nr.c()
    _check("csa_compress_kv_norm_rope_fp8kv",
           lib.csa_compress_kv_norm_rope_fp8kv(ctypes.byref(c), streams, kv.shape[-1], _p(kv), _p(z), _p(bias),
                                               kv.shape[1], tok0, ent_begin, ent_end, _p(out), out.shape[1],
                                               ctypes.byref(n), _stream()))


def sparse_attn_fp8kv(cfg: Config, q: torch.Tensor, kv_fp8: torch.Tensor, idx: torch.Tensor, kv_local: torch.Tensor,
                      local_base: torch.Tensor, q_pos: torch.Tensor, sink: torch.Tensor, out: torch.Tensor,
                      lse: Optional[torch.Tensor] = None) -> None:
    """csa_sparse_attn_fp8kv: kv_fp8 [B, E_cap, 576] uint8 FP8 entries; the rest as sparse_attn."""
    lib = L.load()
    c = cfg.c()
    B, T = q.shape[0], q.shape[1]
    ws = _workspace(lib.csa_workspace_size(L.CSA_OP_ATTN, ctypes.byref(c), B * T, T), q.device)
    wp, wb = _ws_args(ws)
    _check("csa_sparse_attn_fp8kv",
           lib.csa_sparse_attn_fp8kv(ctypes.byref(c), _p(q), T, _p(kv_fp8), kv_fp8.shape[1], _p(idx), _p(kv_local),
                                     kv_local.shape[1], _p(local_base), _p(q_pos), _p(sink), _p(out), _p(lse), wp, wb,
                                     _stream()))


def kv_pack_mxfp4(cfg: Config, x: torch.Tensor, out: torch.Tensor) -> None:
    """csa_kv_pack_mxfp4: rows x [..., dim] in cfg.act -> MXFP4 entries out [..., dim/2 + dim/16] uint8."""
    lib = L.load()
    c = cfg.c()
    dim = x.shape[-1]
    _check("csa_kv_pack_mxfp4", lib.csa_kv_pack_mxfp4(ctypes.byref(c), _p(x), x.numel() // dim, dim, _p(out),
                                                      _stream()))


def sparse_attn_mxfp4kv(cfg: Config, q: torch.Tensor, kv_mx: torch.Tensor, idx: torch.Tensor, kv_local: torch.Tensor,
                        local_base: torch.Tensor, q_pos: torch.Tensor, sink: torch.Tensor, out: torch.Tensor,
                        lse: Optional[torch.Tensor] = None) -> None:
    """csa_sparse_attn_mxfp4kv: kv_mx [B, E_cap, 288] uint8 MXFP4 entries; the rest as sparse_attn."""
    lib = L.load()
    c = cfg.c()
    B, T = q.shape[0], q.shape[1]
    ws = _workspace(lib.csa_workspace_size(L.CSA_OP_ATTN, ctypes.byref(c), B * T, T), q.device)
    wp, wb = _ws_args(ws)
    _check("csa_sparse_attn_mxfp4kv",
           lib.csa_sparse_attn_mxfp4kv(ctypes.byref(c), _p(q), T, _p(kv_mx), kv_mx.shape[1], _p(idx), _p(kv_local),
                                       kv_local.shape[1], _p(local_base), _p(q_pos), _p(sink), _p(out), _p(lse), wp,
                                       wb, _stream()))


class DecodeStepCall:
    """csa_decode_step with its arguments marshalled once: for a decode loop that keeps its
    buffers (caches, tails, window rows, outputs) fixed and rewrites their contents each step.
    Calling the object enqueues one step on the current stream."""

    def __init__(self, cfg: Config, *, q_pos, q, qI, w, sink, kv_comp, kI, kv_tail, z_tail, kvI_tail, zI_tail, bias,
                 biasI, kv_local, local_base, out, kscale=None, lse=None, idx_out=None, scores_out=None,
                 fp8kv: bool = False, bf16_scores: bool = False, mxfp4kv: bool = False):
        self._lib = L.load()
        self._fn = (self._lib.csa_decode_step_mxfp4kv if mxfp4kv else
                    self._lib.csa_decode_step_fp8kv if fp8kv else self._lib.csa_decode_step)
        self._c = cfg.c()
        self._a = L.csa_decode_args(kv_comp.shape[1], _p(q_pos), _p(q), _p(qI), _p(w), _p(sink), _p(kv_comp), _p(kI),
                                    _p(kscale), _p(kv_tail), _p(z_tail), _p(kvI_tail), _p(zI_tail), _p(bias),
                                    _p(biasI), _p(kv_local), kv_local.shape[1], _p(local_base), _p(out), _p(lse),
                                    _p(idx_out), _p(scores_out), int(bf16_scores))
        nbytes = self._lib.csa_workspace_size(L.CSA_OP_DECODE, ctypes.byref(self._c), cfg.B, kv_comp.shape[1])
        if nbytes == ctypes.c_size_t(-1).value:
            raise CsaError("csa_workspace_size", 2)
        self._ws = _decode_workspace(nbytes, q.device, cfg.B)
        self._wp, self._wb = _ws_args(self._ws)
        self._refs = (q_pos, q, qI, w, sink, kv_comp, kI, kv_tail, z_tail, kvI_tail, zI_tail, bias, biasI, kv_local,
                      local_base, out, kscale, lse, idx_out, scores_out)   # keep the buffers alive
        self._cref, self._aref = ctypes.byref(self._c), ctypes.byref(self._a)

    def __call__(self) -> None:
        _check("csa_decode_step", self._fn(self._cref, self._aref, self._wp, self._wb, _stream()))


class HcaDecodeStepCall:
    """csa_hca_decode_step with its arguments marshalled once (see DecodeStepCall)."""

    def __init__(self, cfg: Config, *, q_pos, q, sink, kv_comp, kv_tail, z_tail, bias, kv_local, local_base, out,
                 lse=None):
        self._lib = L.load()
        self._c = cfg.c()
        self._a = L.csa_hca_decode_args(kv_comp.shape[1], _p(q_pos), _p(q), _p(sink), _p(kv_comp), _p(kv_tail),
                                        _p(z_tail), _p(bias), _p(kv_local), kv_local.shape[1], _p(local_base), _p(out),
                                        _p(lse))
        self._ws = _workspace(self._lib.csa_workspace_size(L.CSA_OP_HCA_DECODE, ctypes.byref(self._c), cfg.B,
                                                           kv_comp.shape[1]), q.device)
        self._wp, self._wb = _ws_args(self._ws)
        self._refs = (q_pos, q, sink, kv_comp, kv_tail, z_tail, bias, kv_local, local_base, out, lse)
        self._cref, self._aref = ctypes.byref(self._c), ctypes.byref(self._a)

    def __call__(self) -> None:
        _check("csa_hca_decode_step",
               self._lib.csa_hca_decode_step(self._cref, self._aref, self._wp, self._wb, _stream()))


class StepInputs:
    """A step's per-step input tensors packed back to back in one device buffer, with a host
    mirror of the same layout (pinned when the buffer is on a GPU).

    The caller writes a step's inputs into ``host[name]`` and ``upload()`` moves all of them
    with one host-to-device copy on the current stream; the step reads ``dev[name]``.  Each
    tensor starts on a 256-byte boundary of the buffer, so the views keep the alignment the
    library's kernels ask of their inputs.  The views are contiguous and have the shapes and
    dtypes of the tensors given; their initial contents are those tensors' values."""

    ALIGN = 256

    def __init__(self, tensors: dict, device=None):
        if not tensors:
            raise ValueError("StepInputs needs at least one tensor")
        device = torch.device(device) if device is not None else next(iter(tensors.values())).device
        spans, off = {}, 0
        for name, t in tensors.items():
            nb = t.numel() * t.element_size()
            spans[name] = (off, nb, t.shape, t.dtype)
            off += (nb + self.ALIGN - 1) // self.ALIGN * self.ALIGN
        self.nbytes = off
        self._dbuf = torch.empty(off, dtype=torch.uint8, device=device)
        self._hbuf = torch.empty(off, dtype=torch.uint8, pin_memory=device.type == "cuda")
        self.dev, self.host = {}, {}
        for name, (o, nb, shape, dt) in spans.items():
            self.dev[name] = self._dbuf[o:o + nb].view(dt).view(shape)
            self.host[name] = self._hbuf[o:o + nb].view(dt).view(shape)
            self.host[name].copy_(tensors[name])
            self.dev[name].copy_(tensors[name])

    def upload(self) -> None:
        """Enqueue the one host-to-device copy of every input on the current stream."""
        if self._dbuf.is_cuda:
            self._dbuf.copy_(self._hbuf, non_blocking=True)
        else:
            self._dbuf.copy_(self._hbuf)
