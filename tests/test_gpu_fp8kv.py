"""Parity of the quantised main-KV entries with the CPU oracle: FP8 (448 e4m3 dims + 64 bf16
RoPE dims, 576 B) and MXFP4 (E2M1 + one e4m3 scale per 16 channels, 288 B).  The packers are
bit-exact, the fused compressor within the e4m3 / bf16 rounding of its output, and the decode
attention over quantised entries agrees with the oracle's attention over the decoded entries
(and is bit-identical to the bf16 path over the same decoded values)."""
import numpy as np
import pytest
import torch

import compressed_sparse_attention_csa_gb300 as csa
from _helpers import assert_rows_close, np64
from oracle import csa_oracle as O
from synth import gen
from test_gpu_epilogue import assert_vectors_close, e4m3_half_step
from test_gpu_parity import _attn_inputs, _attn_ref

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


@pytest.mark.parametrize("act,dim", [(BF16, 512), (torch.float32, 512), (BF16, 128)])
def test_kv_pack_fp8_bit_exact(act, dim):
    rows = 333
    x = rnd(800 + dim, (rows, dim), 30.0, act)          # wide range: saturation and subnormals
    x[0, :8] = torch.tensor([0.0, -0.0, 448.0, -449.0, 1e-4, 2.0 ** -9, 3.0 * 2.0 ** -10, 1000.0])
    out = torch.empty(rows, dim + 64, dtype=torch.uint8, device=DEV)
    csa.kv_pack_fp8(cfg_obj(act=act), x, out)
    assert csa.get_last_error() == 0
    ref = O.kv_fp8_encode(np64(x))
    got = out.cpu().numpy()
    assert np.array_equal(got, ref)


def test_compress_norm_rope_fp8kv_matches_oracle():
    B, m, dim, ent_begin, n_ent = 2, 4, 512, 5, 30
    tok0 = m * (ent_begin - 1)
    n_tok = m * (ent_begin + n_ent) - tok0
    kv = rnd(810, (B, n_tok, 2, dim), dim ** -0.5, BF16)
    z = rnd(811, (B, n_tok, 2, dim), 1.0, BF16)
    bias = rnd(812, (2, m, dim), 0.1)
    w = 1.0 + rnd(813, (dim,), 0.1)
    E_cap = ent_begin + n_ent
    out = torch.zeros(B, E_cap, dim + 64, dtype=torch.uint8, device=DEV)
    nr = csa.NormRope(weight=w, eps=1e-6, rope_dims=64, theta=10000.0)
    csa.compress_kv_norm_rope_fp8kv(cfg_obj(m=m, B=B), 2, kv, z, bias, tok0, ent_begin, E_cap, out, nr)
    assert csa.get_last_error() == 0
    for b in range(B):
        ref = np.stack([O.norm_rope(O.compress_entry(np64(kv[b]), np64(z[b]), np64(bias), m, i, tok0=tok0),
                                    O.compressed_entry_position(m, i), np64(w), 1e-6, 64, 10000.0)
                        for i in range(ent_begin, E_cap)])
        dec = O.kv_fp8_decode(out[b, ent_begin:].cpu().numpy())
        tol = 1.01 * e4m3_half_step(ref[:, :448]) + 4e-6 * np.abs(ref).max(axis=-1, keepdims=True)
        assert float((np.abs(dec[:, :448] - ref[:, :448]) / tol).max()) <= 1.0, f"FP8 dims b={b}"
        assert_vectors_close(dec[:, 448:], ref[:, 448:], BF16, f"RoPE dims b={b}")
        assert np.all(out[b, :ent_begin].cpu().numpy() == 0)


@pytest.mark.parametrize("B,nsel", [(3, [512, 40, 0]), (4, [512]), (1, [300])])
def test_sparse_attn_fp8kv_decode(B, nsel):
    H, d, E, k, W, L, T = 64, 512, 1500, 512, 128, 200, 1
    q, kv, kl, sink, idx = _attn_inputs(820 + B, B, T, H, d, E, k, L, BF16, nsel)
    kv = kv * 8.0                                      # RMSNorm-scale entries (|x| ~ 0.35)
    local_base = torch.tensor([[1000, 1040, 0][b % 3] for b in range(B)], dtype=torch.int64, device=DEV)
    q_pos = torch.tensor([[1150, 1100, 50][b % 3] for b in range(B)], dtype=torch.int64, device=DEV)
    c = cfg_obj(B=B)
    packed = torch.empty(B, E, d + 64, dtype=torch.uint8, device=DEV)
    csa.kv_pack_fp8(c, kv, packed)
    assert np.array_equal(packed.cpu().numpy(), O.kv_fp8_encode(np64(kv)))   # the oracle's own encoding
    out = torch.empty(B, T, H, d, device=DEV, dtype=BF16)
    lse = torch.empty(B, T, H, device=DEV)
    csa.sparse_attn_fp8kv(c, q, packed, idx, kl, local_base, q_pos, sink, out, lse)
    assert csa.get_last_error() == 0
    dec = torch.from_numpy(O.kv_fp8_decode(packed.cpu().numpy())).to(DEV).to(BF16)   # exact in bf16
    ro, rl = _attn_ref(q, dec, idx, kl, local_base, q_pos, sink, W, d ** -0.5)
    assert_rows_close(np64(out), ro, 2e-2)
    np.testing.assert_allclose(np64(lse), rl, atol=5e-3, rtol=0)
    # the same products as the bf16 path over the decoded entries
    out_b = torch.empty_like(out)
    lse_b = torch.empty_like(lse)
    csa.sparse_attn(c, q, dec, idx, kl, local_base, q_pos, sink, out_b, lse_b)
    assert torch.equal(out, out_b) and torch.equal(lse, lse_b)


@pytest.mark.parametrize("fmt", ["fp8", "mxfp4"])
@pytest.mark.parametrize("B,T", [(1, 300), (2, 170)])
def test_sparse_attn_quantkv_many_queries(fmt, B, T):
    """Many queries (a prefill chunk: one CTA a query on the pipelined kernel) over FP8 / MXFP4
    entries: the rows widened to bf16 in the gather, exactly, so the result is bit-identical to
    csa_sparse_attn over the decoded cache, and it matches the oracle; ragged selections (fewer
    than k rows, an empty one) and windows clipped at the cache start."""
    H, d, E, k, W, L = 64, 512, 1500, 512, 128, 400
    nsel = [512, 300, 0, 511] if T > 1 else None
    q, kv, kl, sink, idx = _attn_inputs(830 + T, B, T, H, d, E, k, L, BF16, nsel)
    kv = kv * 8.0
    c = cfg_obj(B=B)
    if fmt == "fp8":
        packed = torch.empty(B, E, d + 64, dtype=torch.uint8, device=DEV)
        csa.kv_pack_fp8(c, kv, packed)
        dec = torch.from_numpy(O.kv_fp8_decode(packed.cpu().numpy())).to(DEV).to(BF16)
        fn = csa.sparse_attn_fp8kv
    else:
        packed = torch.empty(B, E, d // 2 + d // 16, dtype=torch.uint8, device=DEV)
        csa.kv_pack_mxfp4(c, kv, packed)
        dec = torch.from_numpy(O.mxfp4_decode(packed.cpu().numpy())).to(DEV).to(BF16)
        fn = csa.sparse_attn_mxfp4kv
    local_base = torch.tensor([0, 60][:B], dtype=torch.int64, device=DEV)
    q_pos = (torch.arange(T, dtype=torch.int64, device=DEV)[None, :] + torch.tensor([20, 200][:B], device=DEV)[:, None])
    q_pos = q_pos.reshape(-1).contiguous()
    out = torch.empty(B, T, H, d, device=DEV, dtype=BF16)
    lse = torch.empty(B, T, H, device=DEV)
    fn(c, q, packed, idx, kl, local_base, q_pos, sink, out, lse)
    assert csa.get_last_error() == 0
    out_b = torch.empty_like(out)
    lse_b = torch.empty_like(lse)
    csa.sparse_attn(c, q, dec, idx, kl, local_base, q_pos, sink, out_b, lse_b)
    assert torch.equal(out, out_b) and torch.equal(lse, lse_b)
    ro, rl = _attn_ref(q, dec, idx, kl, local_base, q_pos, sink, W, d ** -0.5)
    assert_rows_close(np64(out), ro, 2e-2)
    np.testing.assert_allclose(np64(lse), rl, atol=5e-3, rtol=0)


@pytest.mark.parametrize("act,dim", [(BF16, 512), (torch.float32, 512), (BF16, 128)])
def test_kv_pack_mxfp4_bit_exact(act, dim):
    rows = 257
    x = rnd(840 + dim, (rows, dim), 1.0, act) * rnd(841 + dim, (rows, 1), 3.0).abs().to(act)
    x[0, :16] = torch.tensor([6.0, -0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.0, -0.0, 4.0, 3.0, 2.0, 1.0, 0.5, -6.0])
    x[1, :16] = 0                                       # an all-zero block: scale code 0, zero codes
    x[2, :16] = 1e-12                                   # a scale that underflows e4m3
    out = torch.empty(rows, dim // 2 + dim // 16, dtype=torch.uint8, device=DEV)
    csa.kv_pack_mxfp4(cfg_obj(act=act), x, out)
    assert csa.get_last_error() == 0
    assert np.array_equal(out.cpu().numpy(), O.mxfp4_encode(np64(x)))


@pytest.mark.parametrize("B,nsel", [(3, [512, 40, 0]), (4, [512])])
def test_sparse_attn_mxfp4kv_decode(B, nsel):
    H, d, E, k, W, L, T = 64, 512, 1500, 512, 128, 200, 1
    q, kv, kl, sink, idx = _attn_inputs(850 + B, B, T, H, d, E, k, L, BF16, nsel)
    kv = kv * 8.0
    local_base = torch.tensor([[1000, 1040, 0][b % 3] for b in range(B)], dtype=torch.int64, device=DEV)
    q_pos = torch.tensor([[1150, 1100, 50][b % 3] for b in range(B)], dtype=torch.int64, device=DEV)
    c = cfg_obj(B=B)
    packed = torch.empty(B, E, d // 2 + d // 16, dtype=torch.uint8, device=DEV)
    csa.kv_pack_mxfp4(c, kv, packed)
    assert np.array_equal(packed.cpu().numpy(), O.mxfp4_encode(np64(kv)))   # the oracle's own encoding
    out = torch.empty(B, T, H, d, device=DEV, dtype=BF16)
    lse = torch.empty(B, T, H, device=DEV)
    csa.sparse_attn_mxfp4kv(c, q, packed, idx, kl, local_base, q_pos, sink, out, lse)
    assert csa.get_last_error() == 0
    dec = torch.from_numpy(O.mxfp4_decode(packed.cpu().numpy())).to(DEV).to(BF16)   # exact in bf16
    ro, rl = _attn_ref(q, dec, idx, kl, local_base, q_pos, sink, W, d ** -0.5)
    assert_rows_close(np64(out), ro, 2e-2)
    np.testing.assert_allclose(np64(lse), rl, atol=5e-3, rtol=0)
    out_b = torch.empty_like(out)
    lse_b = torch.empty_like(lse)
    csa.sparse_attn(c, q, dec, idx, kl, local_base, q_pos, sink, out_b, lse_b)
    assert torch.equal(out, out_b) and torch.equal(lse, lse_b)


@pytest.mark.parametrize("cid,N", [(4, 4 * 2500), (2, 4 * 1500)])
def test_decode_step_fp8kv_matches_oracle(cid, N):
    """The full decode step over an FP8-entry main-KV cache: the entry the token completes is
    stored as an FP8 entry, the attention reads FP8 entries (oracle: the same on the decoded
    cache)."""
    from _helpers import (assert_out_close_with_swaps, assert_selection_ok, keys_f64, lib_config, np_inputs,
                          swap_bound)
    cfg = gen.CONFIGS[cid].replace(B=3, N=N)
    inp = gen.make_inputs(cfg, DEV)
    inp["q_pos"][1] = N - 3                          # this token completes no block
    c = lib_config(cfg)
    kv8 = torch.empty(cfg.B, cfg.E, cfg.d + 64, dtype=torch.uint8, device=DEV)
    csa.kv_pack_fp8(c, inp["kv_comp"], kv8)
    assert np.array_equal(kv8.cpu().numpy(), O.kv_fp8_encode(np64(inp["kv_comp"])))
    dec_cache = O.kv_fp8_decode(kv8.cpu().numpy())
    nb = np_inputs(inp)
    fp8k = cfg.kidx == "fp8"
    refs = []
    for b in range(cfg.B):
        kdeq = keys_f64(inp["kI"][b], inp["kscale"][b] if fp8k else None)
        kvc = dec_cache[b].copy()
        r = O.decode_step_sequence(cfg, nb, b, kvc, kdeq, fp8_keys=fp8k, fp8_kv=True)
        r["kv_comp"] = kvc
        refs.append(r)
    before = kv8.clone()
    out = torch.empty(cfg.B, cfg.H, cfg.d, device=DEV, dtype=BF16)
    lse = torch.empty(cfg.B, cfg.H, device=DEV)
    idx = torch.empty(cfg.B, cfg.k, dtype=torch.int32, device=DEV)
    csa.decode_step(c, q_pos=inp["q_pos"], q=inp["q"], qI=inp["qI"], w=inp["w"], sink=inp["sink"], kv_comp=kv8,
                    kI=inp["kI"], kscale=inp.get("kscale"), kv_tail=inp["kv_str"], z_tail=inp["z_str"],
                    kvI_tail=inp["kvI_str"], zI_tail=inp["zI_str"], bias=inp["bias"], biasI=inp["biasI"],
                    kv_local=inp["kv_local"], local_base=inp["local_base"], out=out, lse=lse, idx_out=idx, fp8kv=True)
    assert csa.get_last_error() == 0
    rtol_s = 5e-2 if fp8k else 1e-2
    for b in range(cfg.B):
        r = refs[b]
        if r["entry"] is None:
            assert torch.equal(kv8[b], before[b])
        else:
            e = r["entry"][0]
            got = O.kv_fp8_decode(kv8[b, e].cpu().numpy())
            exact = O.compress_entry(nb["kv_str"][b], nb["z_str"][b], nb["bias"], cfg.m, e, int(nb["q_pos"][b]) - 2 * cfg.m + 1)
            tol = 1.01 * e4m3_half_step(exact[:448]) + 1e-6 * np.abs(exact).max()
            assert np.all(np.abs(got[:448] - exact[:448]) <= tol), f"FP8 part of the new entry b={b}"
            assert_vectors_close(got[448:][None], exact[448:][None], BF16, f"bf16 part of the new entry b={b}")
        fin = r["scores"][np.isfinite(r["scores"])]
        tol_s = rtol_s * max(np.sqrt((fin ** 2).mean()), 1e-30)
        gi = idx[b].cpu().numpy()
        swaps = assert_selection_ok(gi, r["idx"], r["scores"], cfg.k, tol_s)
        g_set, r_set = set(gi[gi >= 0].tolist()), set(r["idx"][r["idx"] >= 0].tolist())
        bound = swap_bound(r["q"] if "q" in r else nb["q"][b, 0], r["lse"], cfg.softmax_scale,
                           [r["kv_comp"][x] for x in g_set - r_set], [r["kv_comp"][y] for y in r_set - g_set])
        assert_out_close_with_swaps(np64(out[b]), r["out"], 2e-2, bound, what=f"out b={b} swaps={swaps}")
        np.testing.assert_allclose(np64(lse[b]), r["lse"], atol=5e-3)


@pytest.mark.parametrize("cid,N", [(13, 4 * 2500), (4, 4 * 2500), (2, 4 * 1500)])
def test_decode_step_mxfp4kv_matches_oracle(cid, N):
    """The fused decode step over an MXFP4-entry main-KV cache (V4.1's 288-byte entries): the
    entry the token completes is written as an MXFP4 entry by the indexer CTAs (16-channel
    blocks inside one CTA), the attention reads MXFP4 entries (oracle: the same on the decoded
    cache); with MXFP4, FP8 and bf16 indexer keys."""
    from _helpers import (assert_out_close_with_swaps, assert_selection_ok, keys_f64, lib_config, np_inputs,
                          swap_bound)
    cfg = gen.CONFIGS[cid].replace(B=3, N=N)
    inp = gen.make_inputs(cfg, DEV)
    inp["q_pos"][1] = N - 3                          # this token completes no block
    c = lib_config(cfg)
    kv4 = torch.empty(cfg.B, cfg.E, cfg.d // 2 + cfg.d // 16, dtype=torch.uint8, device=DEV)
    csa.kv_pack_mxfp4(c, inp["kv_comp"], kv4)
    dec_cache = O.mxfp4_decode(kv4.cpu().numpy())
    nb = np_inputs(inp)
    qk = cfg.kidx in ("fp8", "mxfp4")
    refs = []
    for b in range(cfg.B):
        kdeq = keys_f64(inp["kI"][b], inp["kscale"][b] if qk else None)
        kvc = dec_cache[b].copy()
        r = O.decode_step_sequence(cfg, nb, b, kvc, kdeq, fp8_keys=cfg.kidx == "fp8", mx_keys=cfg.kidx == "mxfp4",
                                   mxfp4_kv=True)
        r["kv_comp"] = kvc
        refs.append(r)
    before = kv4.clone()
    out = torch.empty(cfg.B, cfg.H, cfg.d, device=DEV, dtype=BF16)
    lse = torch.empty(cfg.B, cfg.H, device=DEV)
    idx = torch.empty(cfg.B, cfg.k, dtype=torch.int32, device=DEV)
    csa.decode_step(c, q_pos=inp["q_pos"], q=inp["q"], qI=inp["qI"], w=inp["w"], sink=inp["sink"], kv_comp=kv4,
                    kI=inp["kI"], kscale=inp.get("kscale"), kv_tail=inp["kv_str"], z_tail=inp["z_str"],
                    kvI_tail=inp["kvI_str"], zI_tail=inp["zI_str"], bias=inp["bias"], biasI=inp["biasI"],
                    kv_local=inp["kv_local"], local_base=inp["local_base"], out=out, lse=lse, idx_out=idx,
                    mxfp4kv=True)
    assert csa.get_last_error() == 0
    rtol_s = 5e-2 if qk else 1e-2
    for b in range(cfg.B):
        r = refs[b]
        if r["entry"] is None:
            assert torch.equal(kv4[b], before[b])
        else:
            e = r["entry"][0]
            raw = kv4[b, e].cpu().numpy()
            exact = r["entry"][3]
            ref_raw = O.mxfp4_encode(exact)
            assert int((raw != ref_raw).sum()) <= 4, f"new MXFP4 entry b={b}: {int((raw != ref_raw).sum())} bytes differ"
            got = O.mxfp4_decode(raw)
            sc = O.e4m3_decode(raw[cfg.d // 2:]).repeat(16)
            amax = np.abs(exact).reshape(-1, 16).max(-1).repeat(16)
            bound = 1.01 * sc + np.maximum(0.0, amax - 6 * sc) + 1e-6 * np.abs(exact).max()
            assert np.all(np.abs(got - exact) <= bound), f"new MXFP4 entry b={b}"
        fin = r["scores"][np.isfinite(r["scores"])]
        tol_s = rtol_s * max(np.sqrt((fin ** 2).mean()), 1e-30)
        gi = idx[b].cpu().numpy()
        swaps = assert_selection_ok(gi, r["idx"], r["scores"], cfg.k, tol_s)
        g_set, r_set = set(gi[gi >= 0].tolist()), set(r["idx"][r["idx"] >= 0].tolist())
        bound = swap_bound(nb["q"][b, 0], r["lse"], cfg.softmax_scale,
                           [r["kv_comp"][x] for x in g_set - r_set], [r["kv_comp"][y] for y in r_set - g_set])
        assert_out_close_with_swaps(np64(out[b]), r["out"], 2e-2, bound, what=f"out b={b} swaps={swaps}")
        np.testing.assert_allclose(np64(lse[b]), r["lse"], atol=5e-3)
