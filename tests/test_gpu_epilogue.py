"""Parity of the attention prologue / epilogue kernels (RMSNorm, partial RoPE, the fused
compressor + RMSNorm + RoPE, inverse RoPE and FP8 output quantisation) with the CPU oracle.

Agreement: the output rounding (bf16: 2^-8 relative; fp32: 2^-22) plus 4e-6 of the vector's
largest magnitude (fp32 arithmetic, single-precision sine/cosine of the reduced angle); FP8
codes: the dequantised value within half an e4m3 step of the oracle's value (plus 1 % of a
step), the scale within 2^-20 relative.
"""
import numpy as np
import pytest
import torch

import compressed_sparse_attention_csa_gb300 as csa
from _helpers import np64
from oracle import csa_oracle as O
from synth import gen

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


def rnd(seed, shape, std=1.0, dtype=torch.float32):
    n = int(np.prod(shape))
    return gen.normal(seed, n, device=DEV, std=std).reshape(shape).to(dtype)


def cfg_obj(**kw):
    base = dict(B=2, H=64, d=512, HI=64, dI=128, m=4, k=512, W=128, act=BF16, fp8_keys=False, softmax_scale=None)
    base.update(kw)
    return csa.Config(**base)


def check_dev_error():
    assert csa.get_last_error() == 0


def positions(seed, n):
    g = torch.Generator().manual_seed(seed)
    p = torch.randint(0, 1 << 20, (n,), generator=g).to(torch.int64)
    p[:3] = torch.tensor([0, (1 << 20) - 1, 7])
    return p


def assert_vectors_close(got, ref, act, what):
    got = np.asarray(got, np.float64)
    rel = 2.0 ** -8 if act == BF16 else 2.0 ** -22
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    tol = rel * np.abs(ref) + 4e-6 * scale + 1e-30
    worst = float((np.abs(got - ref) / tol).max())
    assert worst <= 1.0, f"{what}: worst error is {worst:.3f} x tolerance"
    return worst


@pytest.mark.parametrize("act,H,d,rd,with_w", [(BF16, 64, 512, 64, True), (BF16, 64, 512, 64, False),
                                              (BF16, 1, 512, 0, True), (torch.float32, 8, 64, 16, True),
                                              (torch.float32, 3, 1024, 64, True)])
def test_norm_rope_matches_oracle(act, H, d, rd, with_w):
    rows = 2 * 37
    x = rnd(500 + d + H, (rows, H, d), 2.0, act)
    w = rnd(501, (d,), 1.0) if with_w else None
    pos = positions(rows + d, rows)
    nr = csa.NormRope(weight=w, eps=1e-6, rope_dims=rd, theta=10000.0)
    y = torch.empty_like(x)
    csa.norm_rope(cfg_obj(act=act), x, pos.to(DEV), nr, out=y)
    check_dev_error()
    ref = O.norm_rope(np64(x), pos.numpy(), np64(w) if with_w else None, 1e-6, rd, 10000.0)
    assert_vectors_close(np64(y), ref, act, "norm_rope")
    csa.norm_rope(cfg_obj(act=act), x, pos.to(DEV), nr)          # in place
    check_dev_error()
    assert torch.equal(x, y)


@pytest.mark.parametrize("streams,m,dim,act,with_bias,with_w,ent_begin,n_ent", [
    (2, 4, 512, BF16, True, True, 0, 37),      # CSA main KV entries, from entry 0
    (2, 4, 128, BF16, True, True, 9, 20),      # indexer-key width, a range past entry 0
    (1, 128, 512, BF16, True, True, 0, 5),     # HCA entries
    (1, 2, 128, torch.float32, False, True, 3, 40),   # CSA2 encoder pairs, no positional bias
    (1, 128, 64, torch.float32, True, False, 0, 3),   # RoPE only
])
def test_compress_norm_rope_matches_oracle(streams, m, dim, act, with_bias, with_w, ent_begin, n_ent):
    B = 2
    tok0 = m * max(ent_begin - 1, 0) if streams == 2 else m * ent_begin
    n_tok = m * (ent_begin + n_ent) - tok0 + 3
    shape = (B, n_tok, 2, dim) if streams == 2 else (B, n_tok, dim)
    kv = rnd(600 + dim + m, shape, dim ** -0.5, act)
    z = rnd(601 + dim + m, shape, 1.0, act)
    bias = rnd(602, (2, m, dim) if streams == 2 else (m, dim), 0.1) if with_bias else None
    w = rnd(603, (dim,), 1.0) if with_w else None
    E_cap = ent_begin + n_ent + 1
    out = torch.full((B, E_cap, dim), 3.0, device=DEV, dtype=act)
    nr = csa.NormRope(weight=w, eps=1e-6, rope_dims=64 if dim >= 64 else 16, theta=10000.0)
    csa.compress_kv_norm_rope(cfg_obj(m=m, act=act, d=dim), streams, kv, z, bias, tok0, ent_begin, ent_begin + n_ent,
                              out, nr)
    check_dev_error()
    bn = np64(bias) if with_bias else None
    for b in range(B):
        ents = []
        for i in range(ent_begin, ent_begin + n_ent):
            if streams == 2:
                e = O.compress_entry(np64(kv[b]), np64(z[b]), bn, m, i, tok0=tok0)
            else:
                e = O.compress_single_entry(np64(kv[b]), np64(z[b]), bn, m, i, tok0=tok0)
            ents.append(O.norm_rope(e, O.compressed_entry_position(m, i), np64(w) if with_w else None, 1e-6,
                                    nr.rope_dims, 10000.0))
        assert_vectors_close(np64(out[b, ent_begin:ent_begin + n_ent]), np.stack(ents), act, f"entries b={b}")
        assert torch.all(out[b, :ent_begin] == 3.0) and torch.all(out[b, ent_begin + n_ent:] == 3.0)


def e4m3_half_step(v):
    """Half the spacing of e4m3 values at magnitude v (normal: 2^(floor(log2 v) - 3); below
    2^-6: the subnormal step 2^-9)."""
    v = np.maximum(np.abs(v), 2.0 ** -6)
    return 0.5 * 2.0 ** (np.floor(np.log2(v)) - 3)


@pytest.mark.parametrize("act,H,d,rd", [(BF16, 64, 512, 64), (torch.float32, 8, 64, 16)])
def test_inverse_rope_and_fp8_output(act, H, d, rd):
    rows = 3 * 29
    o = rnd(700 + d, (rows, H, d), 0.5, act)
    o[5] = 0                                  # an all-zero row
    pos = positions(rows, rows)
    c = cfg_obj(H=H, d=d, act=act)
    ref = O.inverse_rope(np64(o), pos.numpy(), rd, 10000.0)
    y = torch.empty_like(o)
    csa.inverse_rope_quant(c, o, pos.to(DEV), y, rope_dims=rd)
    check_dev_error()
    assert_vectors_close(np64(y), ref, act, "inverse rope")
    codes = torch.empty(rows, H, d, dtype=torch.uint8, device=DEV)
    scale = torch.empty(rows, H, device=DEV)
    csa.inverse_rope_quant(c, o, pos.to(DEV), codes, out_scale=scale, rope_dims=rd)
    check_dev_error()
    sc = scale.cpu().numpy().astype(np.float64)
    amax = np.abs(ref).max(axis=-1)
    exp_sc = np.where(amax > 0, amax / 448.0, 1.0)
    np.testing.assert_allclose(sc, exp_sc, rtol=2.0 ** -20)
    deq = O.e4m3_decode(codes.cpu().numpy()) * sc[..., None]
    tol = 1.01 * e4m3_half_step(ref / sc[..., None]) * sc[..., None] + 1e-6 * amax[..., None]
    worst = float((np.abs(deq - ref) / tol).max())
    assert worst <= 1.0, f"fp8 output: worst error is {worst:.3f} x tolerance"
    # the all-zero row: scale 1 and every code a zero (rotating zeros can give -0, code 0x80)
    assert np.all(O.e4m3_decode(codes[5].cpu().numpy()) == 0) and sc[5].min() == 1.0
