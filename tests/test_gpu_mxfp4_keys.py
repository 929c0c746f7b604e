"""MXFP4 indexer keys (V4.1 diagram, byte ledger "Single request / logical serving KV storage":
128 channels as 64 packed E2M1 bytes + 4 UE8M0 scales; V4 page, "FP4, down to the index
scores") against the oracle (GPU required).

The tensor-core path multiplies the E2M1 keys by the query's two E4M3 terms with the keys'
scales applied by the block-scaled MMA, so the keys enter exactly and the only rounding is
the query's split (the FP8-key path's, about 2^-8 relative per product) and fp32 accumulation:
scores agree within the FP8 tolerance, |g - r| <= 5e-2 * max(|r|, row rms).  The selection is
bit-exact on the scores the step wrote.  Keys written by the compressor and by the decode step
are MX encodings of the compressed value: every code and scale byte equals the oracle's
encoding of the fp32 key, except where the exact value sits within fp32 rounding of a
decision boundary (then the code may be either neighbour).
"""
import numpy as np
import pytest
import torch

import compressed_sparse_attention_csa_gb300 as csa
from _helpers import (assert_decode_matches, assert_scores_close, assert_step_selection_exact, keys_f64, lib_config,
                      np64, oracle_decode, run_gpu_decode)
from oracle import csa_oracle as O
from synth import gen

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


def rnd(seed, shape, std=1.0, dtype=torch.float32):
    n = int(np.prod(shape))
    return gen.normal(seed, n, device=DEV, std=std).reshape(shape).to(dtype)


def cfg_obj(**kw):
    base = dict(B=2, H=64, d=512, HI=64, dI=128, m=4, k=512, W=128, act=BF16, fp8_keys=False, softmax_scale=None,
                mx_keys=True)
    base.update(kw)
    return csa.Config(**base)


def mx_keys(seed, B, E):
    """Drawn MXFP4 keys (the input recipe of the MXFP4 presets) for B sequences of E keys."""
    cfg = gen.CONFIGS[13].replace(cid=13 + seed, B=B, N=4 * E)
    return gen.mxfp4_keys(cfg, B, E, 128, DEV)


def indexer_ref(qI, w, q_pos, kdeq, m, T):
    B, E = kdeq.shape[0], kdeq.shape[1]
    q, ww, pos = np64(qI), np64(w), q_pos.cpu().numpy()
    out = np.empty((B * T, E))
    for r in range(B * T):
        b, t = divmod(r, T)
        out[r] = O.indexer_scores(q[b, t], ww[b, t], kdeq[b], min(O.visible_entries(int(pos[r]), m), E))
    return out


@pytest.mark.parametrize("HI,T", [(64, 1), (32, 1), (64, 9), (32, 21), (64, 700), (128, 1)])
def test_indexer_mx_keys(HI, T):
    """Scores over MXFP4 keys: one query per sequence (key range split over CTAs), several
    (query groups), many (one CTA per SM), and HI = 128 (the CUDA-core path)."""
    B, dI, m, E = 3, 128, 4, 128 * 9 + 36          # a ragged last tile
    qI = rnd(51 + HI + T, (B, T, HI, dI), dI ** -0.5, BF16)
    w = rnd(52 + T, (B, T, HI))
    kI, ks = mx_keys(1, B, E)
    if T == 1:
        q_pos = torch.tensor([m * E - 1, m * 700 + 2, m * 128 - 1], dtype=torch.int64, device=DEV)
    else:
        g = torch.Generator().manual_seed(T)
        q_pos = torch.randint(0, m * E + 40, (B * T,), generator=g).to(torch.int64).to(DEV)
    c = cfg_obj(B=B, HI=HI, m=m)
    scores = torch.full((B * T, E + 5), 3.0, device=DEV)
    csa.indexer_scores(c, qI, w, q_pos, kI, scores, kscale=ks)
    assert csa.get_last_error() == 0
    got = np64(scores)
    assert np.all(got[:, E:] == 3.0)
    ref = indexer_ref(qI, w, q_pos, keys_f64(kI, ks), m, T)
    worst = assert_scores_close(got[:, :E], ref, 5e-2)
    print(f"MXFP4 indexer HI={HI} T={T}: worst/tol = {worst:.3f}")


def test_indexer_mx_keys_extreme_scales():
    """Scale bytes across the UE8M0 range the keys can take (2^-40 .. 2^+20 per block, blocks of
    one key far apart) still enter exactly: the products stay within fp32's range."""
    B, dI, m, E, HI = 2, 128, 4, 128 * 3 + 8, 64
    kI, ks = mx_keys(2, B, E)
    g = torch.Generator().manual_seed(5)
    sb = torch.randint(127 - 40, 127 + 21, (B, E, 4), generator=g).to(torch.int32)
    ks = (sb[..., 0] | (sb[..., 1] << 8) | (sb[..., 2] << 16) | (sb[..., 3] << 24)).to(DEV)
    qI = rnd(61, (B, 1, HI, dI), dI ** -0.5, BF16)
    w = rnd(62, (B, 1, HI))
    q_pos = torch.tensor([m * E - 1, m * 200 + 1], dtype=torch.int64, device=DEV)
    scores = torch.empty(B, E, device=DEV)
    csa.indexer_scores(cfg_obj(B=B, HI=HI, m=m), qI, w, q_pos, kI, scores, kscale=ks)
    assert csa.get_last_error() == 0
    assert_scores_close(np64(scores), indexer_ref(qI, w, q_pos, keys_f64(kI, ks), m, 1), 5e-2)


@pytest.mark.parametrize("T", [700, 5])
def test_indexer_topk_mx_keys(T):
    """csa_indexer_topk over MXFP4 keys equals csa_topk on the scores csa_indexer_scores writes."""
    B, HI, m, E, k = 2, 64, 4, 128 * 60 + 36, 512
    qI = rnd(71, (B, T, HI, 128), 128 ** -0.5, BF16)
    w = rnd(72, (B, T, HI))
    kI, ks = mx_keys(3, B, E)
    g = torch.Generator().manual_seed(T)
    q_pos = torch.randint(0, m * E + 40, (B * T,), generator=g).to(torch.int64)
    q_pos[:3] = torch.tensor([3, m * 100, m * E - 1])
    q_pos = q_pos.to(DEV)
    c = cfg_obj(B=B, HI=HI, m=m, k=k)
    idx = torch.full((B * T, k), -7, dtype=torch.int32, device=DEV)
    csa.indexer_topk(c, qI, w, q_pos, kI, idx, kscale=ks)
    scores = torch.empty(B * T, E, device=DEV)
    csa.indexer_scores(c, qI, w, q_pos, kI, scores, kscale=ks)
    nv = ((q_pos + 1) // m).clamp(max=E).to(torch.int32)
    ref_idx = torch.empty(B * T, k, dtype=torch.int32, device=DEV)
    csa.topk(c, scores, ref_idx, n_valid=nv)
    assert csa.get_last_error() == 0
    assert torch.equal(idx, ref_idx)
    s32, nvn = scores.cpu().numpy(), nv.cpu().numpy()
    for r in [0, 1, 2, B * T - 1]:
        np.testing.assert_array_equal(idx[r].cpu().numpy(), O.topk(s32[r], int(nvn[r]), k))


def assert_mx_key_valid(payload, words, exact):
    """GPU-written MXFP4 keys against the oracle's encoding of the same compressed values
    (float64 `exact`, [n, 128]): scale bytes and codes equal, except that a code (or a block's
    scale) may take the neighbouring choice where the exact value lies within 1e-5 relative
    of that decision boundary (the GPU decided on its own fp32 value)."""
    p_ref, s_ref = O.mxfp4_key_encode(exact)
    s_got = O.mxfp4_key_unwords(words)
    x32 = exact.astype(np.float32).astype(np.float64)
    blk = np.abs(x32).reshape(-1, 4, 32).max(-1)
    for i, j in zip(*np.nonzero(s_got != s_ref)):
        # a different scale only where amax sits next to a power of two
        l2 = np.log2(blk[i, j])
        assert abs(l2 - np.round(l2)) < 1e-5, ("scale byte", i, j, s_got[i, j], s_ref[i, j], blk[i, j])
    dec_got = O.mxfp4_key_decode(payload, s_got)
    dec_ref = O.mxfp4_key_decode(p_ref, s_ref)
    bad = np.nonzero(dec_got != dec_ref)
    for i, c in zip(*bad):
        X = O.ue8m0_decode(s_got[i, c // 32])
        y = x32[i, c] / X
        # the boundaries of E2M1 rounding (midpoints of the grid) and the saturation edge
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
        near = np.min(np.abs(np.abs(y) - mids)) <= 1e-5 * max(abs(y), 1.0) or s_got[i, c // 32] != s_ref[i, c // 32]
        assert near, ("code", i, c, x32[i, c], dec_got[i, c], dec_ref[i, c])
    return len(bad[0])


def test_compress_mx_keys():
    """csa_compress_kv with MXFP4 output: each key an MX encoding of its compressed value."""
    B, m, dim, n_tok, tok0 = 3, 4, 128, 160, 16
    kv = rnd(81, (B, n_tok, 2, dim), dim ** -0.5, BF16)
    z = rnd(82, (B, n_tok, 2, dim), 1.0, BF16)
    bias = rnd(83, (2, m, dim), 0.1)
    E_cap, e0, e1 = 48, 5, 44
    out = torch.full((B, E_cap, dim // 2), 0xEE, dtype=torch.uint8, device=DEV)
    sc = torch.full((B, E_cap), 0x11111111, dtype=torch.int32, device=DEV)
    csa.compress_kv(cfg_obj(B=B, m=m), kv, z, bias, tok0, e0, e1, out, out_scale=sc)
    assert csa.get_last_error() == 0
    o, s = out.cpu().numpy(), sc.cpu().numpy().view(np.uint32)
    assert np.all(o[:, :e0] == 0xEE) and np.all(o[:, e1:] == 0xEE)            # rows outside untouched
    assert np.all(s[:, :e0] == 0x11111111) and np.all(s[:, e1:] == 0x11111111)
    for b in range(B):
        exact = O.compress_range(np64(kv[b]), np64(z[b]), np64(bias), m, e0, e1, tok0)
        n = assert_mx_key_valid(o[b, e0:e1], s[b, e0:e1], exact)
        assert n <= 3, n


@pytest.mark.parametrize("B,N", [(3, 4 * 2400), (2, 4 * 5000 + 1), (4, 4 * 784)])
def test_decode_step_mx_keys(B, N):
    """The fused decode step over MXFP4 keys: when the token completes a block its new key is
    written as MXFP4 and scored in the same step; outputs match the oracle, and the selection is
    exactly the top-k of the scores the step wrote."""
    cfg = gen.CONFIGS[13].replace(B=B, N=N)
    inp = gen.make_inputs(cfg, DEV)
    ref = oracle_decode(cfg, inp)
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    out, lse, idx = run_gpu_decode(cfg, inp, scores_out=scores)
    assert_decode_matches(cfg, inp, ref, out, lse, idx)
    assert_step_selection_exact(cfg, ref, idx, scores)
    for b in range(cfg.B):
        if ref[b]["entry"] is not None:
            e, _, _, _, ki_exact = ref[b]["entry"]
            assert_mx_key_valid(inp["kI"][b, e:e + 1].cpu().numpy(),
                                inp["kscale"][b, e:e + 1].cpu().numpy().view(np.uint32), ki_exact[None, :])
