"""Counter-based seeded generator and the workload presets.

Every element of every tensor is a pure function of (seed, tensor id, flat element
index), so any slice of a tensor can be regenerated on its own, on the CPU or on a
CUDA device, with identical bits:

* splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014): state_c = seed + (c + 1) * 0x9E3779B97F4A7C15 mod 2**64, followed by the
  published xor-shift-multiply finaliser.
* uniform u in (0, 1): ((x >> 11) + 0.5) * 2**-53 from the top 53 bits.
* standard normal by Box-Muller (cosine branch) from counters 2e and 2e + 1 of element e.

Values are drawn in float64 and then rounded once to the storage dtype by torch's own
round-to-nearest-even conversion.  Indexer keys stored as FP8 e4m3 get one fp32 scale
per entry, scale = amax / 448, codes = e4m3(x / scale); that is the input recipe, not a
step of the method.  Indexer keys stored as MXFP4 are drawn as codes: uniform random
payload bytes (every E2M1 code equally likely) and per 32 channels a scale byte uniform in
121 .. 124 (2^-6 .. 2^-3, the range the N(0, 1/128) keys' blocks take).

The tensors and their distributions follow the workload descriptions of the CSA
pages: q, qI, the a/b KV and gate streams, compressed caches and window rows are
N(0, 1) / sqrt(last dim); the indexer gate w ~ N(0, 1); the positional bias
~ N(0, 0.1^2); one sink logit per head ~ N(0, 1).  Seed = 0xC5A0 + preset number.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

_MASK64 = (1 << 64) - 1


def _s64(v: int) -> int:
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_MIX1 = _s64(0xBF58476D1CE4E5B9)
_MIX2 = _s64(0x94D049BB133111EB)


def _lsr(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor viewed as uint64."""
    return torch.bitwise_and(torch.bitwise_right_shift(x, s), (1 << (64 - s)) - 1)


def splitmix64(seed: int, counter: torch.Tensor) -> torch.Tensor:
    """splitmix64 output for each int64 counter (bits returned as int64)."""
    z = counter.add(1).mul_(_GOLDEN).add_(_s64(seed))
    z = torch.bitwise_xor(z, _lsr(z, 30)).mul_(_MIX1)
    z = torch.bitwise_xor(z, _lsr(z, 27)).mul_(_MIX2)
    return torch.bitwise_xor(z, _lsr(z, 31))


def uniform01(seed: int, counter: torch.Tensor) -> torch.Tensor:
    """Uniform float64 in the open interval (0, 1)."""
    top53 = _lsr(splitmix64(seed, counter), 11).to(torch.float64)
    return (top53 + 0.5) * (2.0 ** -53)


def random_bytes(seed: int, numel: int, *, device="cpu", offset: int = 0, chunk: int = 1 << 23) -> torch.Tensor:
    """Flat uint8 tensor: the low byte of splitmix64 for elements offset .. offset+numel-1."""
    out = torch.empty(numel, dtype=torch.uint8, device=device)
    for lo in range(0, numel, chunk):
        hi = min(numel, lo + chunk)
        e = torch.arange(offset + lo, offset + hi, dtype=torch.int64, device=device)
        out[lo:hi] = torch.bitwise_and(splitmix64(seed, e), 0xFF).to(torch.uint8)
    return out


def _tensor_seed(base: int, tensor_id: int) -> int:
    # one splitmix64 step decorrelates the per-tensor streams
    c = torch.tensor([tensor_id], dtype=torch.int64)
    return int(splitmix64(base, c)[0].item())


def normal(seed: int, numel: int, *, device="cpu", std: float = 1.0,
           dtype=torch.float64, offset: int = 0, chunk: int = 1 << 23) -> torch.Tensor:
    """Flat tensor of `numel` N(0, std^2) draws for elements offset .. offset+numel-1."""
    out = torch.empty(numel, dtype=dtype, device=device)
    two_pi = 2.0 * math.pi
    for lo in range(0, numel, chunk):
        hi = min(numel, lo + chunk)
        e = torch.arange(offset + lo, offset + hi, dtype=torch.int64, device=device)
        u1 = uniform01(seed, e * 2)
        u2 = uniform01(seed, e * 2 + 1)
        x = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(two_pi * u2)
        out[lo:hi] = (x * std).to(dtype)
    return out


def normal_rows(seed: int, row_len: int, rows: torch.Tensor, *, std: float,
                dtype=torch.float64) -> torch.Tensor:
    """Rows `rows` (int64, any device) of a [*, row_len] tensor drawn by `normal`."""
    rows = rows.to(torch.int64)
    e = (rows[:, None] * row_len + torch.arange(row_len, device=rows.device)[None, :]).reshape(-1)
    u1 = uniform01(seed, e * 2)
    u2 = uniform01(seed, e * 2 + 1)
    x = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)
    return (x * std).to(dtype).reshape(rows.numel(), row_len)


# ----------------------------------------------------------------------------------
# workload presets
# ----------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class CsaConfig:
    cid: int
    name: str
    B: int            # sequences
    N: int            # tokens of context including the query tokens (last query t = N-1)
    m: int            # compression ratio (1 = CSA2 1:1 store)
    d: int            # main KV / query head dim
    H: int            # query heads
    HI: int           # indexer heads
    dI: int           # indexer dim
    k: int            # top-k
    W: int            # sliding window
    T: int            # query tokens per sequence, at t = N-T .. N-1
    act: str          # "f32" | "bf16": dtype of q, qI, KV streams, caches, window rows
    kidx: str         # "act" | "fp8" | "mxfp4": storage of the indexer keys
    mode: str         # "full" | "decode" | "prefill" | "csa2" | "hca_full" | "hca_decode" | "hca_prefill"
    pool_block: int = 8
    pool_blocks: int = 2048
    n_reuse: int = 3

    @property
    def seed(self) -> int:
        return 0xC5A0 + self.cid

    @property
    def E(self) -> int:
        return self.N // self.m

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_act(self):
        return torch.float32 if self.act == "f32" else torch.bfloat16

    def replace(self, **kw) -> "CsaConfig":
        return dataclasses.replace(self, **kw)


CONFIGS: Dict[int, CsaConfig] = {
    1: CsaConfig(1, "tiny CSA layer fp32 (N 2048, m 4, 8x64 heads, indexer 4x32, k 64, W 32, 16 queries)",
                 B=1, N=2048, m=4, d=64, H=8, HI=4, dI=32, k=64, W=32, T=16,
                 act="f32", kidx="act", mode="full"),
    2: CsaConfig(2, "V4-Flash CSA decode bf16 (B 16 @ 65,536 ctx)",
                 B=16, N=65536, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=1,
                 act="bf16", kidx="act", mode="decode"),
    3: CsaConfig(3, "V4-Flash CSA prefill bf16 (4,096 tokens after 131,072)",
                 B=1, N=131072 + 4096, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=4096,
                 act="bf16", kidx="act", mode="prefill"),
    4: CsaConfig(4, "V4-Flash CSA decode @1M ctx (B 4, FP8 e4m3 indexer keys)",
                 B=4, N=1 << 20, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=1,
                 act="bf16", kidx="fp8", mode="decode"),
    5: CsaConfig(5, "V4.1-Flash CSA2 decoder group bf16 (B 8 @ 262,144, 1 Reindex + 3 Reuse)",
                 B=8, N=262144, m=1, d=512, H=64, HI=32, dI=128, k=512, W=128, T=1,
                 act="bf16", kidx="act", mode="csa2"),
    # Heavily Compressed Attention: one-stream compression at m' = 128, dense attention over
    # every visible entry plus the window (the indexer fields are not used)
    6: CsaConfig(6, "V4-Flash HCA decode @1M ctx (B 4, m' 128: 8,192 entries, dense attention)",
                 B=4, N=1 << 20, m=128, d=512, H=64, HI=64, dI=128, k=512, W=128, T=1,
                 act="bf16", kidx="act", mode="hca_decode"),
    7: CsaConfig(7, "V4-Flash HCA prefill bf16 (4,096 tokens after 131,072; m' 128)",
                 B=1, N=131072 + 4096, m=128, d=512, H=64, HI=64, dI=128, k=512, W=128, T=4096,
                 act="bf16", kidx="act", mode="hca_prefill"),
    8: CsaConfig(8, "tiny HCA layer fp32 (N 4096, m' 128, 8x64 heads, W 128, 16 queries)",
                 B=1, N=4096, m=128, d=64, H=8, HI=4, dI=32, k=64, W=128, T=16,
                 act="f32", kidx="act", mode="hca_full"),
    # attention prologue / epilogue on the prefill chunk: query RMSNorm + RoPE, the chunk's
    # compression fused with RMSNorm + RoPE, inverse RoPE + FP8 of the attention output
    9: CsaConfig(9, "V4-Flash attention prologue/epilogue, prefill chunk (4,096 tokens after 131,072)",
                 B=1, N=131072 + 4096, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=4096,
                 act="bf16", kidx="act", mode="epilogue"),
    # the decode attention at 1M over FP8 main-KV entries (448 e4m3 + 64 bf16 dims, 576 B)
    10: CsaConfig(10, "V4-Flash CSA decode attention @1M over FP8 main-KV entries (B 4, k 512, W 128)",
                  B=4, N=1 << 20, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=1,
                  act="bf16", kidx="act", mode="fp8kv_attn"),
    # the same over V4.1's MXFP4 main-KV entries (E2M1 + one e4m3 scale per 16 channels, 288 B)
    11: CsaConfig(11, "CSA decode attention @1M over MXFP4 main-KV entries (B 4, k 512, W 128)",
                  B=4, N=1 << 20, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=1,
                  act="bf16", kidx="act", mode="fp8kv_attn"),
    # the 1M decode step at V4's production precision: FP8 indexer keys and FP8 main-KV entries
    12: CsaConfig(12, "V4-Flash CSA decode @1M ctx, FP8 indexer keys + FP8 main-KV entries (576 B)",
                  B=4, N=1 << 20, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=1,
                  act="bf16", kidx="fp8", mode="decode"),
    # the 1M decode step with FP4 indexer keys: MXFP4, 64 payload bytes + 4 UE8M0 scales a key
    13: CsaConfig(13, "CSA decode @1M ctx (B 4, MXFP4 indexer keys: 64 B + 4 UE8M0 scales)",
                  B=4, N=1 << 20, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=1,
                  act="bf16", kidx="mxfp4", mode="decode"),
    # V4.1's storage throughout: MXFP4 indexer keys and MXFP4 main-KV entries (288 B)
    14: CsaConfig(14, "CSA decode @1M ctx (B 4, MXFP4 indexer keys + MXFP4 main-KV entries)",
                  B=4, N=1 << 20, m=4, d=512, H=64, HI=64, dI=128, k=512, W=128, T=1,
                  act="bf16", kidx="mxfp4", mode="decode"),
}

# tensor ids of the per-tensor streams (stable: changing one changes the inputs)
_IDS = {
    "q": 1, "qI": 2, "w": 3, "sink": 4, "kv_local": 5, "kv_comp": 6, "kI": 7,
    "kv_str": 8, "z_str": 9, "kvI_str": 10, "zI_str": 11, "bias": 12, "biasI": 13,
    "qI_full": 14, "w_full": 15, "kI_mx": 16, "kscale_mx": 17,
}


def _gen(cfg: CsaConfig, name: str, shape, std, dtype, device, layer: int = 0, row0: int = 0):
    """Draws of one tensor; with row0 > 0 the leading axis holds rows row0.. of a larger batch."""
    seed = _tensor_seed(cfg.seed, _IDS[name] + 64 * layer)
    n = 1
    for s in shape:
        n *= s
    per_row = n // shape[0] if shape[0] else 0
    return normal(seed, n, device=device, std=std, dtype=dtype, offset=row0 * per_row).reshape(shape)


def quantize_keys_e4m3(x: torch.Tensor):
    """Input recipe for FP8 indexer keys: per row scale = amax/448, codes = e4m3(x/scale)."""
    x32 = x.to(torch.float32)
    amax = x32.abs().amax(dim=-1).clamp_min(1e-30)
    scale = amax / 448.0
    y = (x32 / scale[..., None]).clamp(-448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def mxfp4_keys(cfg: CsaConfig, B: int, E: int, dI: int, device, row0: int = 0):
    """Drawn MXFP4 keys: payload [B, E, dI/2] uint8 and the scale bytes of every key as one
    little-endian word (byte j for channels 32j .. 32j+31), [B, E] int32 (dI = 128)."""
    payload = random_bytes(_tensor_seed(cfg.seed, _IDS["kI_mx"]), B * E * dI // 2, device=device,
                           offset=row0 * E * dI // 2).reshape(B, E, dI // 2)
    sb = random_bytes(_tensor_seed(cfg.seed, _IDS["kscale_mx"]), B * E * 4, device=device,
                      offset=row0 * E * 4).reshape(B, E, 4)
    sb = (121 + torch.bitwise_and(sb, 3)).to(torch.int32)
    words = sb[..., 0] | (sb[..., 1] << 8) | (sb[..., 2] << 16) | (sb[..., 3] << 24)
    return payload, words


def make_inputs(cfg: CsaConfig, device="cpu", *, skip=(), row0: int = 0) -> Dict[str, torch.Tensor]:
    """All input tensors of one preset, generated on `device`.

    With row0 > 0 the cfg.B sequences are sequences row0 .. row0+B-1 of a larger batch: every
    per-sequence tensor holds exactly the values the larger batch has in those rows, so a
    batch can be split across processes that each generate only their own rows.

    Keys (shapes use B, T, H, d, HI, dI, E = N // m, L = window rows held):
      q [B,T,H,d], qI [B,T,HI,dI], w [B,T,HI] f32, sink [H] f32, q_pos [B*T] i64,
      kv_local [B,L,d], local_base [B] i64,
      kv_comp [B,E,d], kI [B,E,dI] (or kI codes u8 + kscale [B,E] f32 for FP8, or
      kI payload u8 [B,E,dI/2] + kscale [B,E] i32 scale words for MXFP4),
      compression streams kv_str/z_str [B,n_str,2,d], kvI_str/zI_str [B,n_str,2,dI],
      bias [2,m,d] f32, biasI [2,m,dI] f32, str_base [B] i64 (token of stream row 0).
    CSA2 presets add per-layer q/kv_local/sink stacks and the Full-layer indexer query.
    HCA presets (mode hca_*) have no indexer tensors and one compression stream:
      kv_str/z_str [B,n_str,d], bias [m,d] f32, str_base [B] i64.
    """
    act = cfg.torch_act
    B, T, H, d, HI, dI, m, E, W = cfg.B, cfg.T, cfg.H, cfg.d, cfg.HI, cfg.dI, cfg.m, cfg.E, cfg.W
    f32 = torch.float32
    out: Dict[str, torch.Tensor] = {}
    t0 = cfg.N - T
    out["q_pos"] = (torch.arange(t0, cfg.N, dtype=torch.int64, device=device)
                    .repeat(B))
    local_base = max(0, t0 - W + 1)
    L = cfg.N - local_base
    out["local_base"] = torch.full((B,), local_base, dtype=torch.int64, device=device)

    if cfg.mode == "csa2":
        nl = 1 + cfg.n_reuse
        out["q"] = torch.stack([_gen(cfg, "q", (B, T, H, d), 1 / math.sqrt(d), act, device, l, row0=row0)
                                for l in range(nl)])
        out["kv_local"] = torch.stack([_gen(cfg, "kv_local", (B, L, d), 1 / math.sqrt(d), act, device, l, row0=row0)
                                       for l in range(nl)])
        out["sink"] = torch.stack([_gen(cfg, "sink", (H,), 1.0, f32, device, l) for l in range(nl)])
        out["qI_full"] = _gen(cfg, "qI_full", (B, T, HI, dI), 1 / math.sqrt(dI), act, device, row0=row0)
        out["w_full"] = _gen(cfg, "w_full", (B, T, HI), 1.0, f32, device, row0=row0)
    else:
        out["q"] = _gen(cfg, "q", (B, T, H, d), 1 / math.sqrt(d), act, device, row0=row0)
        out["kv_local"] = _gen(cfg, "kv_local", (B, L, d), 1 / math.sqrt(d), act, device, row0=row0)
        out["sink"] = _gen(cfg, "sink", (H,), 1.0, f32, device)
    if cfg.mode.startswith("hca"):
        return _hca_inputs(cfg, out, device, row0, skip)
    if cfg.mode == "epilogue":
        return _epilogue_inputs(cfg, out, device, row0)
    if cfg.mode == "fp8kv_attn":
        return _fp8kv_inputs(cfg, out, device, row0)
    out["qI"] = _gen(cfg, "qI", (B, T, HI, dI), 1 / math.sqrt(dI), act, device, row0=row0)
    out["w"] = _gen(cfg, "w", (B, T, HI), 1.0, f32, device, row0=row0)

    # compressed caches: entries not produced by compression in this workload are drawn
    if "kv_comp" not in skip:
        if cfg.mode == "full":
            out["kv_comp"] = torch.zeros((B, E, d), dtype=act, device=device)
        else:
            out["kv_comp"] = _gen(cfg, "kv_comp", (B, E, d), 1 / math.sqrt(d), act, device, row0=row0)
    if "kI" not in skip and cfg.kidx == "mxfp4":
        if cfg.mode == "full":
            out["kI"] = torch.zeros((B, E, dI // 2), dtype=torch.uint8, device=device)
            out["kscale"] = torch.zeros((B, E), dtype=torch.int32, device=device)
        else:
            out["kI"], out["kscale"] = mxfp4_keys(cfg, B, E, dI, device, row0)
    elif "kI" not in skip:
        if cfg.mode == "full":
            kI = torch.zeros((B, E, dI), dtype=f32, device=device)
        else:
            kI = _gen(cfg, "kI", (B, E, dI), 1 / math.sqrt(dI), f32, device, row0=row0)
        if cfg.kidx == "fp8":
            out["kI"], out["kscale"] = quantize_keys_e4m3(kI)
        else:
            out["kI"] = kI.to(act)
        del kI

    if cfg.mode in ("full", "decode", "prefill"):
        if cfg.mode == "full":
            base, n_str = 0, cfg.N
        elif cfg.mode == "decode":
            base, n_str = cfg.N - 2 * m, 2 * m
        else:
            base, n_str = t0 - m, T + m
        out["str_base"] = torch.full((B,), base, dtype=torch.int64, device=device)
        out["kv_str"] = _gen(cfg, "kv_str", (B, n_str, 2, d), 1 / math.sqrt(d), act, device, row0=row0)
        out["z_str"] = _gen(cfg, "z_str", (B, n_str, 2, d), 1 / math.sqrt(d), act, device, row0=row0)
        out["kvI_str"] = _gen(cfg, "kvI_str", (B, n_str, 2, dI), 1 / math.sqrt(dI), act, device, row0=row0)
        out["zI_str"] = _gen(cfg, "zI_str", (B, n_str, 2, dI), 1 / math.sqrt(dI), act, device, row0=row0)
        out["bias"] = _gen(cfg, "bias", (2, m, d), 0.1, f32, device)
        out["biasI"] = _gen(cfg, "biasI", (2, m, dI), 0.1, f32, device)
    return out


def _hca_inputs(cfg: CsaConfig, out: Dict[str, torch.Tensor], device, row0: int, skip) -> Dict[str, torch.Tensor]:
    """The compressed cache and the one-stream compression inputs of an HCA preset."""
    act = cfg.torch_act
    B, T, d, m, E = cfg.B, cfg.T, cfg.d, cfg.m, cfg.E
    t0 = cfg.N - T
    if "kv_comp" not in skip:
        if cfg.mode == "hca_full":
            out["kv_comp"] = torch.zeros((B, E, d), dtype=act, device=device)
        else:
            out["kv_comp"] = _gen(cfg, "kv_comp", (B, E, d), 1 / math.sqrt(d), act, device, row0=row0)
    if cfg.mode == "hca_full":
        base, n_str = 0, cfg.N
    elif cfg.mode == "hca_decode":
        base, n_str = cfg.N - m, m
    else:
        if t0 % m:
            raise ValueError("an HCA prefill chunk starts on a block boundary")
        base, n_str = t0, T
    out["str_base"] = torch.full((B,), base, dtype=torch.int64, device=device)
    out["kv_str"] = _gen(cfg, "kv_str", (B, n_str, d), 1 / math.sqrt(d), act, device, row0=row0)
    out["z_str"] = _gen(cfg, "z_str", (B, n_str, d), 1 / math.sqrt(d), act, device, row0=row0)
    out["bias"] = _gen(cfg, "bias", (m, d), 0.1, torch.float32, device)
    return out


_IDS.update({"o": 16, "q_norm": 17, "kv_norm": 18})


def _epilogue_inputs(cfg: CsaConfig, out: Dict[str, torch.Tensor], device, row0: int) -> Dict[str, torch.Tensor]:
    """Attention prologue / epilogue inputs: the attention output o [B,T,H,d] ~ N(0,1)/sqrt(d),
    RMSNorm weights q_norm / kv_norm [d] ~ 1 + N(0, 0.1^2), the chunk's two-stream compression
    streams and bias, and the cache it writes into."""
    act = cfg.torch_act
    B, T, H, d, m, E = cfg.B, cfg.T, cfg.H, cfg.d, cfg.m, cfg.E
    t0 = cfg.N - T
    out["o"] = _gen(cfg, "o", (B, T, H, d), 1 / math.sqrt(d), act, device, row0=row0)
    out["q_norm"] = 1.0 + _gen(cfg, "q_norm", (d,), 0.1, torch.float32, device)
    out["kv_norm"] = 1.0 + _gen(cfg, "kv_norm", (d,), 0.1, torch.float32, device)
    out["kv_comp"] = _gen(cfg, "kv_comp", (B, E, d), 1 / math.sqrt(d), act, device, row0=row0)
    base, n_str = t0 - m, T + m
    out["str_base"] = torch.full((B,), base, dtype=torch.int64, device=device)
    out["kv_str"] = _gen(cfg, "kv_str", (B, n_str, 2, d), 1 / math.sqrt(d), act, device, row0=row0)
    out["z_str"] = _gen(cfg, "z_str", (B, n_str, 2, d), 1 / math.sqrt(d), act, device, row0=row0)
    out["bias"] = _gen(cfg, "bias", (2, m, d), 0.1, torch.float32, device)
    return out


_IDS.update({"sel": 19})


def fp8kv_selection(cfg: CsaConfig, device, row0: int = 0, draw: int = 0) -> torch.Tensor:
    """Selection `draw` of k distinct visible entries a query: the k smallest of uniform draws
    over the entries, ascending ([B, k] int32)."""
    B, E, k = cfg.B, cfg.E, cfg.k
    seed = _tensor_seed(cfg.seed, _IDS["sel"] + 64 * draw)
    rows = []
    for b in range(B):
        u = uniform01(seed, torch.arange((row0 + b) * E, (row0 + b + 1) * E, dtype=torch.int64, device=device))
        rows.append(torch.sort(torch.topk(u, k, largest=False).indices).values.to(torch.int32))
    return torch.stack(rows)


def _fp8kv_inputs(cfg: CsaConfig, out: Dict[str, torch.Tensor], device, row0: int) -> Dict[str, torch.Tensor]:
    """Cache entries at the scale RMSNorm leaves them (N(0, 1)) and selection 0."""
    B, E, d = cfg.B, cfg.E, cfg.d
    out["kv_comp"] = _gen(cfg, "kv_comp", (B, E, d), 1.0, cfg.torch_act, device, row0=row0)
    out["idx"] = fp8kv_selection(cfg, device, row0, 0)
    return out


def small_variant(cfg: CsaConfig, **kw) -> CsaConfig:
    """A reduced copy of a preset (same structure, fewer tokens/rows) for fast tests."""
    return cfg.replace(**kw)
