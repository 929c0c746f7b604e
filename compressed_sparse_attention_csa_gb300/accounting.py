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
    """Bytes of one stored indexer key (FP8 keys carry one fp32 scale)."""
    if cfg.kidx == "fp8":
        return cfg.dI + 4
    return cfg.dI * _act_bytes(cfg.act)


def decode_step_work(cfg) -> Dict[str, float]:
    """Per-step algorithmic bytes/flops of a decode workload (T queries per sequence).

    indexer: every visible key once, qI and w once per query.
    attention: q and out once; each of the k selected entries and W window rows once.
    compression: for a decode step, the 2m stream tokens (kv and gate, both streams, main
    and indexer dims) of the completed block and the two entries written.
    """
    ab = _act_bytes(cfg.act)
    B, T = cfg.B, cfg.T
    nv = (cfg.N) // cfg.m            # last query t = N-1 sees floor(N/m) entries
    key_b = indexer_key_bytes(cfg)
    idx_bytes = B * nv * key_b + B * T * cfg.HI * (cfg.dI * ab + 4)
    rows = min(cfg.k, nv) + cfg.W
    attn_bytes = B * T * (rows * cfg.d * ab + 2 * cfg.H * cfg.d * ab + cfg.k * 4)
    comp_bytes = 0
    if cfg.mode == "decode":
        comp_bytes = B * (2 * cfg.m * 2 * 2 * (cfg.d + cfg.dI) * ab
                          + cfg.d * ab + key_b)
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
