"""CPU oracle for the Compressed Sparse Attention (CSA) hot path.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU-baseline leg of
the benchmark may import this module.  The CUDA library never calls it and shares no
code with it: it is a plain, slow restatement of what each step computes, in float64
numpy, stage by stage, so that it can be checked against the source pages by eye.

Sources (cited by page title and section):
  [V4]   "DeepSeek V4-Flash: The Cost of Deciding What to Read"
         (thesoftwarefrontier.com): sections "The compressor has two streams and they
         overlap", "The Lightning Indexer", "Attention sink, and heads that abstain",
         "The sliding window is not an optimisation", "Key and value are the same vector".
  [V41]  "DeepSeek-V4.1-Flash's KV-Cache Compression, Checked Down to the Byte"
         (flozi-tech-stuff.pages.dev): section 3 "CSA2: three multiplicative
         dimensions, three modes, one cadence" (Hierarchical Sparse Indexer, Cell 4);
         section 5 "SWA Bounded Replay" (window bounds [max(s, i-W+1), i]).
  [V41d] "deepseek-v4-1-flash" (shuhuayu.github.io): "CSA2: separate producing,
         selecting, and reading" and "Hierarchical indexing bounds the deeper searches".

Readings taken where the pages are open (each is a documented reading, not a fact of
the pages):
  * compressor intervals are half-open: entry i mixes stream a over tokens
    [m*i, m*(i+1)) and stream b over [m*(i-1), m*i) (8 tokens at stride 4 for m = 4);
  * entry 0 has no b-stream: those logits are absent from its softmax;
  * the positional bias B^a, B^b is added to the gate logits before the softmax,
    indexed by the token's position inside its block;
  * the indexer score has no extra scale and w is not normalised;
  * a query at t sees compressed entry s iff s < floor((t + 1) / m);
  * the window is positions [max(0, t - W + 1), t] (t included) that the caller's
    local rows hold; window rows and selected entries are not de-duplicated;
  * top-k order is (score descending, index ascending) with -0 == +0; output indices
    ascending, padded with -1 when fewer than k entries are visible;
  * attention logits are softmax_scale * q . r with softmax_scale = 1/sqrt(d) by default;
  * the one-stream compressor (HCA at m' = 128, the CSA2 encoder at m = 2) mixes the m
    tokens of its own block only; HCA's positional bias is added to the gate logits by
    position inside the block, and the CSA2 compressor has none;
  * an HCA query at t attends to every entry s < floor((t + 1) / m') plus the same window
    and sink as the CSA core attention;
  * RMSNorm: y = x / sqrt(mean(x^2) + eps) * weight over the head's d dims, eps = 1e-6 by
    default, one weight vector [d] shared by the heads; it is applied before RoPE;
  * RoPE on the last rope_dims (64) dims of a head: interleaved pairs (2j, 2j+1) of that
    slice rotate by angle pos * theta^(-2j / rope_dims), theta = 10000 by default; a
    compressed entry i sits at position m * i (the first token of its block); a window row
    and a query at their token positions; inverse RoPE on an output uses position -t;
  * FP8 output of the attention: one fp32 scale per (row, head), the key recipe;
  * FP8 main-KV entries (576 B): e4m3 codes of dims 0 .. d-65 (round to nearest even,
    saturating, no scale: RMSNorm bounds the entries well inside e4m3's range), then the last
    64 (RoPE) dims in bf16;
  * MXFP4 main-KV entries (288 B for 512 channels): per block of 16 channels one e4m3 scale
    = e4m3(amax / 6) (amax / 6 in binary32), codes = nearest E2M1 value of x / scale in binary32
    (ties to the even code, saturating at +-6, sign kept); element 2i in the low nibble of byte
    i; the d/2 payload bytes, then the d/16 scale bytes;
  * MXFP4 indexer keys (68 B for 128 channels): per block of 32 channels one UE8M0 scale
    X = 2^(floor(log2(amax)) - 2), the OCP MX rule with E2M1's largest exponent 2, its
    exponent clamped to [-127, 127] (an all-zero or subnormal block gets 2^-127); codes = the
    nearest E2M1 value of x / X (ties to the even code, saturating at +-6, sign kept), decided
    on the binary32 key; element 2i in the low nibble of byte i; the 64 payload bytes, and the
    4 scale bytes (byte j for channels 32j .. 32j+31) kept beside them as one 32-bit word.

Parity status: every function here is pinned by tests (closed forms, hand-computed
examples, brute force against library routines, invariants); see tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# ----------------------------------------------------------------------------------
# storage formats, from their public definitions
# ----------------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 is the upper half of an IEEE binary32: widen by 16 zero bits."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 value (8 significant bits, ties to even) of float64 values in bf16's
    normal range, taken in one rounding from float64; returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def round_to_store(x: np.ndarray, store: str) -> np.ndarray:
    """A value as a cache of the given dtype holds it: "bf16", "f32" (IEEE binary32) or "f64"."""
    if store == "bf16":
        return round_to_bf16(x)
    if store == "f32":
        return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)
    return np.asarray(x, np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 to bfloat16 bits, round-to-nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = u + np.uint64(0x7FFF) + lsb
    return ((u >> np.uint64(16)) & np.uint64(0xFFFF)).astype(np.uint16)


def _e4m3_value(c: int) -> float:
    """OCP 8-bit floating point, E4M3 (no infinities): bias 7, 3 mantissa bits.

    exponent field 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; max 448.
    """
    sign = -1.0 if c & 0x80 else 1.0
    e = (c >> 3) & 0xF
    mant = c & 0x7
    if e == 15 and mant == 7:
        return math.nan
    if e == 0:
        return sign * (mant / 8.0) * 2.0 ** -6
    return sign * (1.0 + mant / 8.0) * 2.0 ** (e - 7)


_E4M3_ALL = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Values of E4M3 codes (a lookup in the 256-entry table of _e4m3_value)."""
    return _E4M3_ALL[np.asarray(codes, dtype=np.uint8)]


_E4M3_POS = _E4M3_ALL[:0x7F]  # codes 0x00..0x7E, ascending


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code, ties to the even code, saturating to +-448 (finite inputs); the sign
    bit is kept, so -0 and negative values that round to zero encode as -0 (0x80)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.searchsorted(_E4M3_POS, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_E4M3_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def quantize_rows_e4m3(x_f32: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """One fp32 scale per row: scale = amax/448 and codes = e4m3(x / scale), in binary32.

    The scale and the division are taken in binary32 so that the code decision is made in
    the same precision as a binary32 kernel would make it.
    """
    x = np.asarray(x_f32, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    y = (x / scale[..., None]).astype(np.float32)
    return e4m3_encode(y), scale


# ----------------------------------------------------------------------------------
# a1: gated two-stream compressor  [V4] "The compressor has two streams and they overlap"
# ----------------------------------------------------------------------------------


def compress_entry(kv: np.ndarray, z: np.ndarray, bias: np.ndarray, m: int, i: int,
                   tok0: int = 0, return_weights: bool = False):
    """Compressed entry i.

    kv, z: [n_tok, 2, dim] rows of tokens tok0 .. tok0 + n_tok - 1; [:, 0] is stream a
    (C^a, Z^a), [:, 1] stream b.  bias: [2, m, dim] (B^a, B^b).
    Stream a contributes tokens m*i .. m*i + m - 1, stream b tokens m*(i-1) .. m*i - 1;
    the softmax runs over those 2m logits (m for entry 0) separately for every channel,
    and the entry is the weighted sum of the matching C values.
    """
    logits: List[np.ndarray] = []
    values: List[np.ndarray] = []
    for j in range(m):                                   # stream a, current block
        r = m * i + j - tok0
        logits.append(z[r, 0].astype(np.float64) + bias[0, j])
        values.append(kv[r, 0].astype(np.float64))
    if i >= 1:
        for j in range(m):                               # stream b, previous block
            r = m * (i - 1) + j - tok0
            if r < 0:
                raise ValueError("stream rows for the previous block are missing")
            logits.append(z[r, 1].astype(np.float64) + bias[1, j])
            values.append(kv[r, 1].astype(np.float64))
    lg = np.stack(logits)                                # [2m or m, dim]
    lg = lg - lg.max(axis=0, keepdims=True)
    wts = np.exp(lg)
    wts = wts / wts.sum(axis=0, keepdims=True)
    entry = (wts * np.stack(values)).sum(axis=0)
    return (entry, wts) if return_weights else entry


def compress_range(kv, z, bias, m: int, i_begin: int, i_end: int, tok0: int = 0) -> np.ndarray:
    """Entries i_begin .. i_end - 1, stacked [i_end - i_begin, dim]."""
    dim = kv.shape[-1]
    out = np.empty((max(0, i_end - i_begin), dim), dtype=np.float64)
    for n, i in enumerate(range(i_begin, i_end)):
        out[n] = compress_entry(kv, z, bias, m, i, tok0)
    return out


# ----------------------------------------------------------------------------------
# one-stream compressor without overlap
#   [V4] "Heavily Compressed Attention": the same compressor at m' = 128 with a single KV
#   stream, so no overlap between blocks; its positional bias runs over the m' positions of
#   a block.  [V41d] "Encoder groups compress pairs": ratio 2, a learned channel-wise softmax
#   pools each pair and the groups do not overlap; [V41d] also notes that the CSA2
#   compressor drops the learned absolute position embedding (bias=None).
# ----------------------------------------------------------------------------------


def compress_single_entry(kv: np.ndarray, z: np.ndarray, bias: Optional[np.ndarray], m: int, i: int,
                          tok0: int = 0, return_weights: bool = False):
    """Entry i of the one-stream compressor.

    kv, z: [n_tok, dim] rows (C and Z) of tokens tok0 .. tok0 + n_tok - 1; bias: [m, dim]
    positional bias by position inside the block, or None.  For every channel the softmax
    runs over the m logits Z[m*i + j] (+ bias[j]), j = 0 .. m-1, and the entry is the
    weighted sum of C over the same m tokens.
    """
    r0 = m * i - tok0
    if r0 < 0 or r0 + m > kv.shape[0]:
        raise ValueError("stream rows of the block are missing")
    lg = z[r0:r0 + m].astype(np.float64)
    if bias is not None:
        lg = lg + np.asarray(bias, np.float64)
    lg = lg - lg.max(axis=0, keepdims=True)
    wts = np.exp(lg)
    wts = wts / wts.sum(axis=0, keepdims=True)
    entry = (wts * kv[r0:r0 + m].astype(np.float64)).sum(axis=0)
    return (entry, wts) if return_weights else entry


def compress_single_range(kv, z, bias, m: int, i_begin: int, i_end: int, tok0: int = 0) -> np.ndarray:
    """One-stream entries i_begin .. i_end - 1, stacked [i_end - i_begin, dim]."""
    out = np.empty((max(0, i_end - i_begin), kv.shape[-1]), dtype=np.float64)
    for n, i in enumerate(range(i_begin, i_end)):
        out[n] = compress_single_entry(kv, z, bias, m, i, tok0)
    return out


# ----------------------------------------------------------------------------------
# a2: lightning indexer  [V4] "The Lightning Indexer";  causality: "The sliding window is
# not an optimisation" (entry i may be read from t only if m(i+1) - 1 <= t)
# ----------------------------------------------------------------------------------


def visible_entries(t: int, m: int) -> int:
    """Number of compressed entries a query at position t may read: floor((t+1)/m)."""
    return (t + 1) // m


def indexer_scores(qI: np.ndarray, w: np.ndarray, kI: np.ndarray, nv: int) -> np.ndarray:
    """I(t, s) = sum_h w[h] * ReLU(qI[h] . kI[s]) for s < nv, -inf for s >= nv.

    qI: [HI, dI], w: [HI], kI: [E, dI] (already dequantised).  float64 result.
    """
    E = kI.shape[0]
    out = np.full(E, -np.inf, dtype=np.float64)
    if nv > 0:
        dots = kI[:nv].astype(np.float64) @ qI.astype(np.float64).T      # [nv, HI]
        out[:nv] = np.maximum(dots, 0.0) @ w.astype(np.float64)
    return out


def indexer_scores_subset(qI, w, kI, positions: np.ndarray) -> np.ndarray:
    """Scores of the listed positions only (CSA2 Reindex rescoring of a candidate pool)."""
    dots = kI[positions].astype(np.float64) @ qI.astype(np.float64).T
    return np.maximum(dots, 0.0) @ w.astype(np.float64)


# ----------------------------------------------------------------------------------
# a3: top-k  [V4] "The Lightning Indexer" ("a cheap scoring pass picks the top 512")
# ----------------------------------------------------------------------------------


def topk(scores_f32: np.ndarray, nv: int, k: int) -> np.ndarray:
    """The k best of scores[0:nv] under (score desc, index asc); ascending, -1 padded."""
    vals = np.asarray(scores_f32[:nv], dtype=np.float64)
    pos = np.arange(nv)
    order = np.lexsort((pos, -vals))            # primary -score, secondary index
    chosen = np.sort(order[:min(k, nv)])
    out = np.full(k, -1, dtype=np.int64)
    out[:chosen.size] = chosen
    return out


def topk_bf16(scores_f32: np.ndarray, nv: int, k: int) -> np.ndarray:
    """The selector on BF16 index scores ([V4] "FP4, down to the index scores": the scores are
    quantised from FP32 to BF16 before the top-k): each binary32 score rounded to the nearest
    BF16 value (ties to even), then the same (score desc, index asc) top-k.  Scores that BF16
    makes equal are ties, won by the lowest index."""
    s = np.asarray(scores_f32, np.float32).astype(np.float64)
    fin = np.isfinite(s)
    r = s.copy()
    r[fin] = round_to_bf16(s[fin])
    return topk(r, nv, k)


# ----------------------------------------------------------------------------------
# a3': CSA2 hierarchical candidate pool  [V41] section 3, [V41d] "Hierarchical indexing"
# ----------------------------------------------------------------------------------


def hier_pool(scores_f32: np.ndarray, nv: int, block: int = 8, n_blocks: int = 2048) -> np.ndarray:
    """Candidate positions: the n_blocks best `block`-position blocks by their max score.

    Block j covers visible positions [block*j, min(block*(j+1), nv)); its score is the max
    over them.  Blocks are ranked (max desc, block asc); the kept blocks expand to their
    visible positions, returned ascending.
    """
    if nv <= 0:
        return np.zeros(0, dtype=np.int64)
    nb = -(-nv // block)
    vals = np.asarray(scores_f32[:nv], dtype=np.float64)
    bmax = np.array([vals[j * block:min((j + 1) * block, nv)].max() for j in range(nb)])
    order = np.lexsort((np.arange(nb), -bmax))
    kept = np.sort(order[:min(n_blocks, nb)])
    pos = [p for j in kept for p in range(j * block, min((j + 1) * block, nv))]
    return np.asarray(pos, dtype=np.int64)


# ----------------------------------------------------------------------------------
# a4: sparse MQA attention with window and sink
#     [V4] "Key and value are the same vector", "Attention sink, and heads that abstain",
#     "The sliding window is not an optimisation"; window bounds as in [V41] section 5.
# ----------------------------------------------------------------------------------


def window_positions(t: int, W: int, local_base: int, n_local: int) -> List[int]:
    """Positions max(0, t-W+1) .. t that the local rows [local_base, local_base+n_local) hold."""
    lo = max(0, t - W + 1, local_base)
    hi = min(t, local_base + n_local - 1)
    return list(range(lo, hi + 1))


def gather_rows(kv_comp: np.ndarray, idx: np.ndarray, kv_local: np.ndarray,
                local_base: int, t: int, W: int) -> np.ndarray:
    """The rows one query attends to: selected compressed entries, then window rows."""
    sel = [kv_comp[i] for i in idx if i >= 0]
    win = [kv_local[p - local_base] for p in window_positions(t, W, local_base, kv_local.shape[0])]
    rows = sel + win
    d = kv_comp.shape[-1]
    return np.stack(rows).astype(np.float64) if rows else np.zeros((0, d))


def sparse_attention(q: np.ndarray, rows: np.ndarray, sink: np.ndarray, scale: float):
    """Per head h: o = sum_j e^{l_j} r_j / (sum_j e^{l_j} + e^{sink_h}), l_j = scale q_h . r_j.

    Every row is both key and value.  Returns (out [H, d], lse [H]) where
    lse = log(sum_j e^{l_j} + e^{sink_h}).
    """
    q = q.astype(np.float64)
    sink = np.asarray(sink, dtype=np.float64)
    logits = scale * (q @ rows.T) if rows.shape[0] else np.zeros((q.shape[0], 0))
    mx = np.maximum(logits.max(axis=1) if rows.shape[0] else -np.inf, sink)
    e = np.exp(logits - mx[:, None])
    den = e.sum(axis=1) + np.exp(sink - mx)
    out = (e @ rows) / den[:, None] if rows.shape[0] else np.zeros_like(q)
    return out, mx + np.log(den)


# ----------------------------------------------------------------------------------
# HCA core attention  [V4] "Heavily Compressed Attention": no indexer and no top-k; the
# layer attends densely over every entry it holds, with the window and per-head sink of
# the CSA core attention ("Attention sink, and heads that abstain": both CSA and HCA carry
# one sink logit per head).
# ----------------------------------------------------------------------------------


def dense_rows(kv_comp: np.ndarray, nv: int, kv_local: np.ndarray, local_base: int, t: int, W: int) -> np.ndarray:
    """HCA's rows for a query at t: compressed entries 0 .. nv-1, then the window rows."""
    return gather_rows(kv_comp, np.arange(nv), kv_local, local_base, t, W)


# ----------------------------------------------------------------------------------
# compositions
# ----------------------------------------------------------------------------------


def decode_token(cfg, inp: Dict[str, np.ndarray], b: int, tq: int,
                 kv_comp: np.ndarray, kI_deq: np.ndarray) -> Dict[str, np.ndarray]:
    """Indexer -> top-k -> attention for one query (sequence b, query slot tq).

    kv_comp [E, d] and kI_deq [E, dI] are sequence b's caches after compression.
    `inp` holds float64 numpy views of the inputs of `synth.make_inputs`.
    """
    t = int(inp["q_pos"][b * cfg.T + tq])
    nv = min(visible_entries(t, cfg.m), kv_comp.shape[0])
    s64 = indexer_scores(inp["qI"][b, tq], inp["w"][b, tq], kI_deq, nv)
    s32 = s64.astype(np.float32)
    idx = topk(s32, nv, cfg.k)
    rows = gather_rows(kv_comp, idx, inp["kv_local"][b], int(inp["local_base"][b]), t, cfg.W)
    out, lse = sparse_attention(inp["q"][b, tq], rows, inp["sink"], cfg.softmax_scale)
    return {"scores": s64, "scores_f32": s32, "idx": idx, "out": out, "lse": lse, "nv": nv}


def decode_step_sequence(cfg, inp: Dict[str, np.ndarray], b: int, kv_comp: np.ndarray,
                         kI_deq: np.ndarray, fp8_keys: bool = False, fp8_kv: bool = False,
                         mx_keys: bool = False, mxfp4_kv: bool = False) -> Dict[str, np.ndarray]:
    """One decode token of sequence b (T = 1).

    When the token at t completes a block ((t + 1) % m == 0), entry e = (t + 1)/m - 1 is
    compressed from the tail streams (rows = tokens t-2m+1 .. t, so the previous block's
    b-stream tokens m(e-1) .. me-1 sit in rows 0 .. m-1) and stored into the caches kv_comp
    [E, d] and kI_deq [E, dI] (updated in place) before anything is scored: each value is
    computed in float64 and stored in the cache's dtype (cfg.act: "bf16" or "f32"; FP8 keys as
    e4m3 codes with one binary32 scale amax/448, read back dequantised; MXFP4 keys (mx_keys) as
    E2M1 codes with a UE8M0 scale per 32 channels, read back decoded; with fp8_kv the main-KV
    entry as an FP8 entry, with mxfp4_kv as an MXFP4 entry, read back decoded); then indexer ->
    top-k -> attention over the
    caches as stored.  r["entry"] = (e, stored main-KV entry, stored key, exact main-KV entry,
    exact key) or None.
    """
    t = int(inp["q_pos"][b])
    store = getattr(cfg, "act", "f64")
    entry = None
    if (t + 1) % cfg.m == 0:
        e = (t + 1) // cfg.m - 1
        tok0 = t - 2 * cfg.m + 1
        kv_exact = compress_entry(inp["kv_str"][b], inp["z_str"][b], inp["bias"], cfg.m, e, tok0)
        if fp8_kv:   # kv_comp holds the cache as stored: FP8 entries, read back decoded
            kv_comp[e] = kv_fp8_decode(kv_fp8_encode(kv_exact))
        elif mxfp4_kv:
            kv_comp[e] = mxfp4_decode(mxfp4_encode(kv_exact))
        else:
            kv_comp[e] = round_to_store(kv_exact, store)
        ki = compress_entry(inp["kvI_str"][b], inp["zI_str"][b], inp["biasI"], cfg.m, e, tok0)
        if fp8_keys:
            codes, sc = quantize_rows_e4m3(ki.astype(np.float32)[None, :])
            kI_deq[e] = e4m3_decode(codes[0]) * float(sc[0])
        elif mx_keys:
            kI_deq[e] = mxfp4_key_decode(*mxfp4_key_encode(ki))
        else:
            kI_deq[e] = round_to_store(ki, store)
        entry = (e, kv_comp[e].copy(), kI_deq[e].copy(), kv_exact, ki)
    r = decode_token(cfg, inp, b, 0, kv_comp, kI_deq)
    r["entry"] = entry
    return r


def hca_token(cfg, inp: Dict[str, np.ndarray], b: int, tq: int, kv_comp: np.ndarray) -> Dict[str, np.ndarray]:
    """HCA attention for one query (sequence b, query slot tq) over sequence b's cache
    kv_comp [E, d] (entries 0 .. nv-1 with nv = min(floor((t+1)/m), E)) plus the window."""
    t = int(inp["q_pos"][b * cfg.T + tq])
    nv = min(visible_entries(t, cfg.m), kv_comp.shape[0])
    rows = dense_rows(kv_comp, nv, inp["kv_local"][b], int(inp["local_base"][b]), t, cfg.W)
    out, lse = sparse_attention(inp["q"][b, tq], rows, inp["sink"], cfg.softmax_scale)
    return {"out": out, "lse": lse, "nv": nv}


def hca_decode_step_sequence(cfg, inp: Dict[str, np.ndarray], b: int, kv_comp: np.ndarray) -> Dict[str, np.ndarray]:
    """One HCA decode token of sequence b (T = 1).

    When the token at t completes a block ((t + 1) % m == 0), entry (t + 1)/m - 1 is
    compressed from the one-stream tail (rows = tokens t-m+1 .. t of kv_str / z_str, bias
    [m, d] or None) into kv_comp [E, d] (updated in place); then dense attention.
    """
    t = int(inp["q_pos"][b])
    entry = None
    if (t + 1) % cfg.m == 0:
        e = (t + 1) // cfg.m - 1
        if e < kv_comp.shape[0]:
            kv_comp[e] = compress_single_entry(inp["kv_str"][b], inp["z_str"][b], inp.get("bias"), cfg.m, e,
                                               tok0=t - cfg.m + 1)
            entry = (e, kv_comp[e].copy())
    r = hca_token(cfg, inp, b, 0, kv_comp)
    r["entry"] = entry
    return r


# ----------------------------------------------------------------------------------
# attention prologue / epilogue
#   [V4] "Key and value are the same vector": RoPE on exactly the last 64 dims, and the fix
#   for a shared key/value, RoPE at position minus the query's position on the last 64 dims
#   of each head's output; vLLM fuses that inverse RoPE with the FP8 quantisation ahead of
#   the output projection.  [V4] "Grouped output projection": RMSNorm per head on the queries
#   and on the single head of the compressed KV entry, just before core attention.
# ----------------------------------------------------------------------------------


def rms_norm(x: np.ndarray, weight: Optional[np.ndarray], eps: float = 1e-6) -> np.ndarray:
    """x / sqrt(mean(x^2 over the last axis) + eps), times weight (None: no weight)."""
    x = np.asarray(x, np.float64)
    y = x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    return y * np.asarray(weight, np.float64) if weight is not None else y


def rope_angles(pos, rope_dims: int, theta: float = 10000.0) -> np.ndarray:
    """Angle of pair j at each position: pos * theta^(-2j / rope_dims); shape [..., rope_dims/2]."""
    j = np.arange(rope_dims // 2, dtype=np.float64)
    freq = theta ** (-2.0 * j / rope_dims)
    return np.asarray(pos, np.float64)[..., None] * freq


def rope(x: np.ndarray, pos, rope_dims: int = 64, theta: float = 10000.0) -> np.ndarray:
    """Rotate the last rope_dims dims of x (last axis) at position pos (broadcast over the
    leading axes; a scalar or an array of x.shape[:-1] or a prefix of it): pair (2j, 2j+1)
    of that slice rotates by its angle; the other dims are unchanged."""
    x = np.asarray(x, np.float64).copy()
    if rope_dims == 0:
        return x
    d = x.shape[-1]
    p = np.asarray(pos, np.float64)
    p = p.reshape(p.shape + (1,) * (x.ndim - 1 - p.ndim))
    a = rope_angles(p, rope_dims, theta)
    c, s_ = np.cos(a), np.sin(a)
    x0 = x[..., d - rope_dims::2].copy()
    x1 = x[..., d - rope_dims + 1::2].copy()
    x[..., d - rope_dims::2] = x0 * c - x1 * s_
    x[..., d - rope_dims + 1::2] = x0 * s_ + x1 * c
    return x


def norm_rope(x: np.ndarray, pos, weight, eps: float = 1e-6, rope_dims: int = 64, theta: float = 10000.0):
    """RMSNorm over each head's dims (last axis; skipped when weight is None), then RoPE on
    its last rope_dims dims."""
    y = rms_norm(x, weight, eps) if weight is not None else np.asarray(x, np.float64)
    return rope(y, pos, rope_dims, theta)


def compressed_entry_position(m: int, i: int) -> int:
    """RoPE position of compressed entry i: the first token of its block."""
    return m * i


def inverse_rope(o: np.ndarray, t, rope_dims: int = 64, theta: float = 10000.0) -> np.ndarray:
    """The output fix of a shared key/value: RoPE at position -t on the last rope_dims dims."""
    return rope(o, -np.asarray(t, np.float64), rope_dims, theta)


# ----------------------------------------------------------------------------------
# production storage of the main KV  [V4] "What the cache costs, checked four ways": the
# 64 RoPE dims in bf16 and the other 448 in FP8, 64 * 2 + 448 = 576 bytes an entry.
# ----------------------------------------------------------------------------------

KV_ROPE_DIMS = 64


def kv_fp8_encode(x: np.ndarray) -> np.ndarray:
    """Entries [..., d] -> bytes [..., d - 64 + 128]: e4m3 codes of dims 0 .. d-65, then the
    bf16 bits (little endian) of the last 64 dims."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    nf = d - KV_ROPE_DIMS
    codes = e4m3_encode(x[..., :nf])
    rope = f32_to_bf16_bits(x[..., nf:].astype(np.float32))
    out = np.empty(x.shape[:-1] + (nf + 2 * KV_ROPE_DIMS,), np.uint8)
    out[..., :nf] = codes
    out[..., nf:] = rope.astype("<u2").view(np.uint8).reshape(x.shape[:-1] + (2 * KV_ROPE_DIMS,))
    return out


def kv_fp8_decode(b: np.ndarray) -> np.ndarray:
    """Bytes [..., d - 64 + 128] -> entries [..., d] in float64."""
    b = np.asarray(b, np.uint8)
    nf = b.shape[-1] - 2 * KV_ROPE_DIMS
    head = e4m3_decode(b[..., :nf])
    tail = bf16_bits_to_f64(np.ascontiguousarray(b[..., nf:]).view("<u2"))
    return np.concatenate([head, tail], axis=-1)


# ----------------------------------------------------------------------------------
# V4.1 main-KV storage  [V41] section 4 "FP4: the norm argument, and hunting the 890-byte
# ledger": MXFP4 with E2M1 payloads and one E4M3 scale per 16 channels, no second-level global
# scale, quantised after RoPE: 512 * 0.5 + 512 / 16 = 288 bytes a token side.
# ----------------------------------------------------------------------------------

# OCP Microscaling Formats: E2M1 (bias 1), magnitudes of codes 0..7; bit 3 is the sign
_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
MX_BLOCK = 16


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, np.uint8)
    v = _E2M1_POS[c & 7]
    return np.where(c & 8, -v, v)


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code, ties to the even code, saturating to +-6; the sign bit is kept."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), 6.0)
    hi = np.minimum(np.searchsorted(_E2M1_POS, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _E2M1_POS[lo], _E2M1_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | 8, code).astype(np.uint8)


def mxfp4_encode(x: np.ndarray) -> np.ndarray:
    """Entries [..., d] (d % 16 == 0) -> bytes [..., d/2 + d/16]."""
    x32 = np.asarray(x, np.float64).astype(np.float32)
    d = x32.shape[-1]
    blk = x32.reshape(x32.shape[:-1] + (d // MX_BLOCK, MX_BLOCK))
    amax = np.abs(blk).max(axis=-1)
    sc_code = e4m3_encode((amax / np.float32(6.0)).astype(np.float32))
    sc = e4m3_decode(sc_code).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sc[..., None] > 0, blk / np.where(sc[..., None] > 0, sc[..., None], np.float32(1)), np.float32(0))
    codes = e2m1_encode(q.astype(np.float32)).reshape(x32.shape[:-1] + (d,))
    payload = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return np.concatenate([payload, sc_code], axis=-1)


def mxfp4_decode(b: np.ndarray) -> np.ndarray:
    """Bytes [..., d/2 + d/16] -> entries [..., d] in float64."""
    b = np.asarray(b, np.uint8)
    d = b.shape[-1] * 16 // 9
    payload, sc_code = b[..., :d // 2], b[..., d // 2:]
    codes = np.empty(b.shape[:-1] + (d,), np.uint8)
    codes[..., 0::2] = payload & 15
    codes[..., 1::2] = payload >> 4
    vals = e2m1_decode(codes).reshape(b.shape[:-1] + (d // MX_BLOCK, MX_BLOCK))
    return (vals * e4m3_decode(sc_code)[..., None]).reshape(b.shape[:-1] + (d,))


# ----------------------------------------------------------------------------------
# V4.1 indexer keys  [V41d] byte ledger "Single request / logical serving KV storage" (Indexer
# K: 128 channels in MXFP4, 64 packed bytes + 4 UE8M0 scales); [V4] "FP4, down to the index
# scores" (the indexer's keys cached and multiplied in FP4).  The block format is the OCP
# Microscaling (MX) one: 32 E2M1 elements sharing one power-of-two scale.
# ----------------------------------------------------------------------------------

MXK_BLOCK = 32
E2M1_EMAX = 2          # exponent of E2M1's largest normal value, 6 = 1.5 * 2^2


def ue8m0_decode(codes: np.ndarray) -> np.ndarray:
    """UE8M0 (8 exponent bits, bias 127, no sign, no mantissa): 2^(c - 127); 0xFF is NaN."""
    c = np.asarray(codes, np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))


def mxfp4_key_encode(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Keys [..., dI] (dI % 32 == 0) -> (payload [..., dI/2] uint8, scales [..., dI/32] uint8).

    Per block of 32 channels: X = 2^(floor(log2(amax)) - 2) (exponent clamped to [-127, 127];
    amax 0 or subnormal gives 2^-127), codes = e2m1_encode(x / X), all on the binary32 key.
    """
    x32 = np.asarray(x, np.float64).astype(np.float32).astype(np.float64)
    dI = x32.shape[-1]
    blk = x32.reshape(x32.shape[:-1] + (dI // MXK_BLOCK, MXK_BLOCK))
    amax = np.abs(blk).max(axis=-1)
    _, ex = np.frexp(amax)                       # amax = f * 2^ex, 0.5 <= f < 1: floor(log2) = ex - 1
    e_x = np.where(amax >= np.ldexp(1.0, -126), ex - 1 - E2M1_EMAX, -127)
    e_x = np.clip(e_x, -127, 127)
    codes = e2m1_encode(blk / np.ldexp(1.0, e_x)[..., None]).reshape(x32.shape)
    payload = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return payload, (e_x + 127).astype(np.uint8)


def mxfp4_key_decode(payload: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """(payload [..., dI/2], scales [..., dI/32]) -> keys [..., dI] in float64."""
    p = np.asarray(payload, np.uint8)
    dI = p.shape[-1] * 2
    codes = np.empty(p.shape[:-1] + (dI,), np.uint8)
    codes[..., 0::2] = p & 15
    codes[..., 1::2] = p >> 4
    vals = e2m1_decode(codes).reshape(p.shape[:-1] + (dI // MXK_BLOCK, MXK_BLOCK))
    return (vals * ue8m0_decode(scales)[..., None]).reshape(p.shape[:-1] + (dI,))


def mxfp4_key_words(scales: np.ndarray) -> np.ndarray:
    """The 4 scale bytes of a 128-channel key as one little-endian 32-bit word (byte j = block j)."""
    s = np.asarray(scales, np.uint32)
    return (s[..., 0] | (s[..., 1] << 8) | (s[..., 2] << 16) | (s[..., 3] << 24)).astype(np.uint32)


def mxfp4_key_unwords(words: np.ndarray) -> np.ndarray:
    """Inverse of mxfp4_key_words: [...] uint32 -> [..., 4] uint8."""
    w = np.asarray(words, np.uint32)
    return np.stack([(w >> np.uint32(8 * j)) & np.uint32(0xFF) for j in range(4)], axis=-1).astype(np.uint8)

