"""Algorithmic work of one CSA step: the bytes the method itself must move and the
flops it must do, independent of any kernel design.  Used for roofline fractions.

Indexer cost: one multiply-add per (indexer head, dim, scored position), as in the
cost bound printed by "DeepSeek-V4.1-Flash's KV-Cache Compression, Checked Down to the
Byte", section 3 (Cell 4).
"""
from __future__ import annotations

from typing import Dict


def indexer_macs(heads: int, dim: int, positions: int) -> int:
    """Multiply-adds of the lightning-indexer dot products over `positions` keys."""
    return heads * dim * positions


def _act_bytes(act: str) -> int:
    return 4 if act == "f32" else 2


def indexer_key_bytes(cfg) -> int:
    """Bytes of one stored indexer key (FP8 keys carry one fp32 scale; MXFP4 keys are dI/2 payload
    bytes and one UE8M0 byte per 32 channels: 64 + 4 for dI = 128)."""
    if cfg.kidx == "fp8":
        return cfg.dI + 4
    if cfg.kidx == "mxfp4":
        return cfg.dI // 2 + cfg.dI // 32
    return cfg.dI * _act_bytes(cfg.act)


def decode_step_work(cfg, kv_entry_bytes=None) -> Dict[str, float]:
    """Per-step algorithmic bytes/flops of a decode workload (T queries per sequence).

    indexer: every visible key once, qI and w once per query.
    attention: q and out once; each of the k selected entries (kv_entry_bytes each: a stored
    format's size, default d activations) and W window rows once.
    compression: for a decode step, the 2m stream tokens (kv and gate, both streams, main
    and indexer dims) of the completed block and the two entries written.
    """
    ab = _act_bytes(cfg.act)
    B, T = cfg.B, cfg.T
    nv = (cfg.N) // cfg.m            # last query t = N-1 sees floor(N/m) entries
    key_b = indexer_key_bytes(cfg)
    idx_bytes = B * nv * key_b + B * T * cfg.HI * (cfg.dI * ab + 4)
    rows = min(cfg.k, nv) + cfg.W
    entry_b = kv_entry_bytes if kv_entry_bytes is not None else cfg.d * ab
    sel = min(cfg.k, nv)
    attn_bytes = B * T * (sel * entry_b + cfg.W * cfg.d * ab + 2 * cfg.H * cfg.d * ab + cfg.k * 4)
    comp_bytes = 0
    if cfg.mode == "decode":
        comp_bytes = B * (2 * cfg.m * 2 * 2 * (cfg.d + cfg.dI) * ab
                          + entry_b + key_b)
    idx_flops = 2 * indexer_macs(cfg.HI, cfg.dI, nv) * B * T
    attn_flops = 4 * cfg.H * cfg.d * rows * B * T
    return {
        "indexer_bytes": idx_bytes,
        "attention_bytes": attn_bytes,
        "compress_bytes": comp_bytes,
        "bytes": idx_bytes + attn_bytes + comp_bytes,
        "indexer_flops": idx_flops,
        "attention_flops": attn_flops,
        "flops": idx_flops + attn_flops,
    }


def prefill_work(cfg) -> Dict[str, float]:
    """Algorithmic work of one prefill chunk: T new queries at t = N-T .. N-1 per sequence.

    indexer: one multiply-add per (head, dim, visible key) for each query (causal pairs only);
    attention: QK^T and PV over the k selected entries plus min(W, t+1) window rows per query;
    compression: the T/m new entries of both caches from T+m stream tokens.
    """
    ab = _act_bytes(cfg.act)
    B, T, m = cfg.B, cfg.T, cfg.m
    t0 = cfg.N - T
    pairs = 0
    rows = 0
    for t in range(t0, cfg.N):
        nv = min((t + 1) // m, cfg.E)
        pairs += nv
        rows += min(cfg.k, nv) + min(cfg.W, t + 1)
    pairs *= B
    rows *= B
    idx_flops = 2 * indexer_macs(cfg.HI, cfg.dI, pairs)
    attn_flops = 4 * cfg.H * cfg.d * rows
    n_new = T // m
    comp_bytes = B * ((T + m) * 2 * 2 * (cfg.d + cfg.dI) * ab + n_new * (cfg.d + cfg.dI) * ab)
    idx_bytes = B * cfg.E * indexer_key_bytes(cfg) + B * T * cfg.HI * (cfg.dI * ab + 4)
    attn_bytes = B * (cfg.E * cfg.d * ab + T * 2 * cfg.H * cfg.d * ab)   # every entry once, q/out once
    return {"pairs": pairs, "attention_rows": rows, "indexer_flops": idx_flops, "attention_flops": attn_flops,
            "flops": idx_flops + attn_flops, "indexer_bytes": idx_bytes, "attention_bytes": attn_bytes,
            "compress_bytes": comp_bytes, "bytes": idx_bytes + attn_bytes + comp_bytes}


def csa2_group_work(cfg, pool_blocks: int = 2048, block: int = 8, layers: int = 4) -> Dict[str, float]:
    """Algorithmic bytes of one CSA2 decoder-group token per sequence (m = 1).

    scan: the Full layer reads every visible indexer key once; rescoring: the Reindex layer
    reads the pooled keys once; each of the `layers` attentions gathers k + W rows and reads
    q / writes out once.
    """
    ab = _act_bytes(cfg.act)
    B = cfg.B
    nv = min(cfg.N, cfg.E)
    pool = min(pool_blocks * block, nv)
    key_b = indexer_key_bytes(cfg)
    q_b = cfg.HI * (cfg.dI * ab + 4)
    scan = B * (nv * key_b + q_b)
    rescore = B * (pool * key_b + q_b)
    rows = min(cfg.k, pool) + cfg.W
    attn = layers * B * (rows * cfg.d * ab + 2 * cfg.H * cfg.d * ab)
    return {"scan_bytes": scan, "rescore_bytes": rescore, "attention_bytes": attn,
            "bytes": scan + rescore + attn, "bytes_without_scan": rescore + attn,
            "scan_flops": 2 * indexer_macs(cfg.HI, cfg.dI, nv) * B}


def hca_decode_work(cfg) -> Dict[str, float]:
    """Algorithmic bytes of one HCA decode token per sequence ("Heavily Compressed Attention":
    no indexer; dense over every entry).

    attention: each visible entry and window row once, q read and out written once;
    compression (the token completes a block): the m stream tokens (C and Z), the positional
    bias and the entry written.
    """
    ab = _act_bytes(cfg.act)
    B = cfg.B
    nv = cfg.N // cfg.m
    rows = nv + cfg.W
    attn = B * (rows * cfg.d * ab + 2 * cfg.H * cfg.d * ab)
    comp = B * (2 * cfg.m * cfg.d * ab + cfg.d * ab) + cfg.m * cfg.d * 4
    return {"attention_bytes": attn, "compress_bytes": comp, "bytes": attn + comp,
            "attention_flops": 4 * cfg.H * cfg.d * rows * B}


def hca_prefill_work(cfg) -> Dict[str, float]:
    """Algorithmic work of one HCA prefill chunk: T new queries at t = N-T .. N-1 per sequence,
    each attending to its floor((t+1)/m) visible entries plus min(W, t+1) window rows;
    compression of the chunk's T/m new entries from its T stream tokens."""
    ab = _act_bytes(cfg.act)
    B, T, m = cfg.B, cfg.T, cfg.m
    rows = 0
    for t in range(cfg.N - T, cfg.N):
        rows += min((t + 1) // m, cfg.E) + min(cfg.W, t + 1)
    rows *= B
    flops = 4 * cfg.H * cfg.d * rows
    comp = B * (2 * T * cfg.d * ab + (T // m) * cfg.d * ab) + m * cfg.d * 4
    attn = B * (cfg.E * cfg.d * ab + T * 2 * cfg.H * cfg.d * ab)     # every entry once, q/out once
    return {"attention_rows": rows, "attention_flops": flops, "flops": flops, "attention_bytes": attn,
            "compress_bytes": comp, "bytes": attn + comp}


def epilogue_work(cfg) -> Dict[str, float]:
    """Algorithmic bytes of the attention prologue / epilogue of a prefill chunk: the queries
    read and written once (RMSNorm + RoPE), the chunk's compression streams read and its
    entries written once (fused RMSNorm + RoPE), the attention output read once and written
    as e4m3 codes with one fp32 scale per (token, head)."""
    ab = _act_bytes(cfg.act)
    B, T, H, d, m = cfg.B, cfg.T, cfg.H, cfg.d, cfg.m
    q = 2 * B * T * H * d * ab + B * T * 8
    comp = B * ((T + m) * 2 * 2 * d * ab + (T // m) * d * ab) + 2 * m * d * 4 + d * 4
    o = B * T * H * d * (ab + 1) + B * T * H * 4
    return {"q_bytes": q, "compress_bytes": comp, "out_bytes": o, "bytes": q + comp + o}
