"""Parity of every CUDA stage with the CPU oracle on seeded inputs (GPU required).

Sizes span several tiles with ragged tails; agreement per stage:
  top-k / pool: bit-exact given the same fp32 scores;
  indexer: |g - r| <= rtol * max(|r|, row rms), rtol 1e-2 (bf16), 5e-2 (FP8 keys), 1e-5 (fp32);
  attention: |g - r| <= 2e-2 * max|r_row| for bf16 outputs, 1e-4 absolute for fp32;
  compressor: bf16 rounding (2^-8 relative) or fp32 (1e-5 relative).
"""
import math

import numpy as np
import pytest
import torch

import compressed_sparse_attention_csa_gb300 as csa
from _helpers import (assert_out_close_with_swaps, assert_step_selection_exact, assert_rows_close, assert_scores_close, assert_selection_ok,
                      keys_f64, lib_config, np64, np_inputs, oracle_decode, run_gpu_decode, swap_bound,
                      assert_decode_matches, assert_entries_close, assert_pool_valid)
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


# ------------------------------------------------------------------ compressor

def test_compress_tiny_fp32_all_entries():
    cfg = gen.CONFIGS[1]
    inp = gen.make_inputs(cfg, DEV)
    c = lib_config(cfg)
    for kv, z, bias, dim in [(inp["kv_str"], inp["z_str"], inp["bias"], cfg.d),
                             (inp["kvI_str"], inp["zI_str"], inp["biasI"], cfg.dI)]:
        out = torch.zeros(cfg.B, cfg.E, dim, device=DEV)
        csa.compress_kv(c, kv, z, bias, 0, 0, cfg.E, out)
        check_dev_error()
        ref = O.compress_range(np64(kv[0]), np64(z[0]), np64(bias), cfg.m, 0, cfg.E)
        np.testing.assert_allclose(np64(out[0]), ref, rtol=1e-5, atol=1e-7)


def test_compress_bf16_range_and_e4m3():
    B, m, dim, n_tok, tok0 = 3, 4, 512, 160, 16
    kv = rnd(11, (B, n_tok, 2, dim), dim ** -0.5, BF16)
    z = rnd(12, (B, n_tok, 2, dim), 1.0, BF16)
    bias = rnd(13, (2, m, dim), 0.1)
    c = cfg_obj(B=B, m=m)
    e0, e1, cap = 5, 44, 50
    out = torch.full((B, cap, dim), 7.0, device=DEV, dtype=BF16)
    csa.compress_kv(c, kv, z, bias, tok0, e0, e1, out)
    codes = torch.zeros(B, cap, dim, device=DEV, dtype=torch.uint8)
    scale = torch.zeros(B, cap, device=DEV)
    csa.compress_kv(c, kv, z, bias, tok0, e0, e1, codes, out_scale=scale)
    check_dev_error()
    o = np64(out)
    assert np.all(o[:, :e0] == 7.0) and np.all(o[:, e1:] == 7.0)
    for b in range(B):
        ref = O.compress_range(np64(kv[b]), np64(z[b]), np64(bias), m, e0, e1, tok0=tok0)
        assert_entries_close(o[b, e0:e1], ref, np64(kv[b]))
        ref32 = ref.astype(np.float32)
        rc, rs = O.quantize_rows_e4m3(ref32)
        gs = scale[b, e0:e1].cpu().numpy()
        np.testing.assert_allclose(gs, rs, rtol=2e-6)
        gc = codes[b, e0:e1].cpu().numpy()
        deq = O.e4m3_decode(gc) * gs[:, None]
        bound = 2.0 ** -4 * np.abs(ref) + 2.0 ** -9 * gs[:, None] + 1e-12
        assert np.all(np.abs(deq - ref) <= bound)
        assert (gc == rc).mean() > 0.999


# ------------------------------------------------------------------ indexer

def _indexer_ref(qI, w, q_pos, kdeq, m, T):
    B = kdeq.shape[0]
    E = kdeq.shape[1]
    q = np64(qI)
    ww = np64(w)
    pos = q_pos.cpu().numpy()
    out = np.empty((B * T, E))
    for r in range(B * T):
        b, t = divmod(r, T)
        nv = min(O.visible_entries(int(pos[r]), m), E)
        out[r] = O.indexer_scores(q[b, t], ww[b, t], kdeq[b], nv)
    return out


@pytest.mark.parametrize("HI,T,fp8", [(64, 1, False), (64, 37, False), (32, 21, False), (64, 1, True),
                                      (64, 9, True),
                                      # one query per sequence: the CTAs build the query image
                                      (32, 1, True), (128, 1, False), (128, 1, True),
                                      # enough query groups for one CTA per SM over the whole key range
                                      (64, 700, False), (32, 700, False), (64, 700, True)])
def test_indexer_tensor_cores(HI, T, fp8):
    B, dI, m, E = 3, 128, 4, 128 * 9 + 37
    qI = rnd(21 + HI + T, (B, T, HI, dI), dI ** -0.5, BF16)
    w = rnd(22 + T, (B, T, HI))
    kf = rnd(23, (B, E, dI), dI ** -0.5)
    if fp8:
        kI, ks = gen.quantize_keys_e4m3(kf)
    else:
        kI, ks = kf.to(BF16), None
    if T == 1:
        q_pos = torch.tensor([m * E - 1, m * 700 + 2, m * 128 - 1], dtype=torch.int64, device=DEV)
    else:
        g = torch.Generator().manual_seed(T)
        q_pos = torch.randint(0, m * E + 40, (B * T,), generator=g).to(torch.int64).to(DEV)
    c = cfg_obj(B=B, HI=HI, dI=dI, m=m, fp8_keys=fp8)
    scores = torch.full((B * T, E + 5), 3.0, device=DEV)
    csa.indexer_scores(c, qI, w, q_pos, kI, scores, kscale=ks)
    check_dev_error()
    got = np64(scores)
    assert np.all(got[:, E:] == 3.0)           # columns past E_cap untouched
    ref = _indexer_ref(qI, w, q_pos, keys_f64(kI, ks), m, T)
    worst = assert_scores_close(got[:, :E], ref, 5e-2 if fp8 else 1e-2)
    print(f"indexer HI={HI} T={T} fp8={fp8}: worst/tol = {worst:.3f}")


@pytest.mark.parametrize("HI,fp8,B,n_cand", [(64, False, 3, 128 * 5 + 19), (64, True, 3, 128 * 5 + 19),
                                             (32, False, 2, 40), (64, True, 160, 300)])
def test_indexer_tensor_cores_candidates(HI, fp8, B, n_cand):
    """Candidate lists (one query per sequence) scored on the tensor cores: each slot holds the
    score of its position, -inf for -1 and for positions not yet visible; duplicates allowed."""
    dI, m, E = 128, 4, 128 * 7 + 45
    qI = rnd(31 + HI, (B, 1, HI, dI), dI ** -0.5, BF16)
    w = rnd(32, (B, 1, HI))
    kf = rnd(33, (B, E, dI), dI ** -0.5)
    kI, ks = gen.quantize_keys_e4m3(kf) if fp8 else (kf.to(BF16), None)
    g = torch.Generator().manual_seed(n_cand + B)
    q_pos = torch.randint(m * 300, m * E + 40, (B,), generator=g).to(torch.int64)
    q_pos[0] = m * E - 1
    cand = torch.randint(0, E, (B, n_cand), generator=g).to(torch.int32)
    cand[:, n_cand - 7:] = -1                    # padded tail
    cand[:, 3] = -1                              # a hole
    cand[:, 5] = cand[:, 4]                      # a duplicate
    c = cfg_obj(B=B, HI=HI, dI=dI, m=m, fp8_keys=fp8)
    scores = torch.full((B, n_cand + 3), 3.0, device=DEV)
    csa.indexer_scores(c, qI, w, q_pos.to(DEV), kI, scores, kscale=ks, cand=cand.to(DEV).contiguous())
    check_dev_error()
    got = np64(scores)
    assert np.all(got[:, n_cand:] == 3.0)
    ref = _indexer_ref(qI, w, q_pos, keys_f64(kI, ks), m, 1)
    cn = cand.numpy()
    ref_c = np.where(cn >= 0, np.take_along_axis(ref, np.maximum(cn, 0), axis=1), -np.inf)
    assert_scores_close(got[:, :n_cand], ref_c, 5e-2 if fp8 else 1e-2)


@pytest.mark.parametrize("HI,T,fp8,mode", [(64, 700, False, "random"), (64, 700, True, "random"),
                                           (64, 640, False, "rising"), (64, 640, False, "ties"),
                                           (32, 300, False, "random"), (64, 5, False, "random")])
def test_indexer_topk_matches_scores_then_topk(HI, T, fp8, mode):
    """csa_indexer_topk returns exactly what csa_topk returns on the scores csa_indexer_scores
    writes, and agrees with the oracle up to score-tolerance swaps; rising scores and long runs
    of tied scores are the selection's hard cases."""
    B, dI, m, E, k = 2, 128, 4, 128 * 60 + 37, 512
    qI = rnd(41 + HI, (B, T, HI, dI), dI ** -0.5, BF16)
    w = rnd(42, (B, T, HI))
    kf = rnd(43, (B, E, dI), dI ** -0.5)
    if mode == "rising":        # every query scores a key higher than all keys before it
        qI = qI.abs()
        w = w.abs()
        kf = kf.abs() * 0.05 + (torch.arange(E, device=DEV, dtype=torch.float32) / E)[None, :, None]
    elif mode == "ties":        # 37 distinct keys: long runs of equal scores
        kf = kf[:, torch.arange(E, device=DEV) % 37]
    kI, ks = gen.quantize_keys_e4m3(kf) if fp8 else (kf.to(BF16), None)
    g = torch.Generator().manual_seed(T + HI)
    q_pos = torch.randint(0, m * E + 40, (B * T,), generator=g).to(torch.int64)
    q_pos[:3] = torch.tensor([3, m * 100, m * E - 1])   # no entries, fewer than k, every entry
    q_pos = q_pos.to(DEV)
    c = cfg_obj(B=B, HI=HI, dI=dI, m=m, k=k, fp8_keys=fp8)
    idx = torch.full((B * T, k), -7, dtype=torch.int32, device=DEV)
    csa.indexer_topk(c, qI, w, q_pos, kI, idx, kscale=ks)
    scores = torch.empty(B * T, E, device=DEV)
    csa.indexer_scores(c, qI, w, q_pos, kI, scores, kscale=ks)
    nv = ((q_pos + 1) // m).clamp(max=E).to(torch.int32)
    ref_idx = torch.empty(B * T, k, dtype=torch.int32, device=DEV)
    csa.topk(c, scores, ref_idx, n_valid=nv)
    check_dev_error()
    assert torch.equal(idx, ref_idx)
    # and against the oracle on a few rows (score tolerance for swaps at near-ties)
    kdeq, qn, wn, nvn = keys_f64(kI, ks), np64(qI), np64(w), nv.cpu().numpy()
    for r in [0, 1, 2, 3, B * T // 2, B * T - 1]:
        b, t = divmod(r, T)
        ref = O.indexer_scores(qn[b, t], wn[b, t], kdeq[b], int(nvn[r]))
        fin = ref[np.isfinite(ref)]
        tol = (5e-2 if fp8 else 1e-2) * max(np.sqrt((fin ** 2).mean()) if fin.size else 0.0, 1e-30)
        assert_selection_ok(idx[r].cpu().numpy(), O.topk(ref.astype(np.float32), int(nvn[r]), k), ref, k, tol)


def test_indexer_cuda_core_fp32_and_candidates():
    cfg = gen.CONFIGS[1].replace(mode="decode")
    inp = gen.make_inputs(cfg, DEV)
    c = lib_config(cfg)
    rows = cfg.B * cfg.T
    scores = torch.empty(rows, cfg.E, device=DEV)
    csa.indexer_scores(c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"], scores)
    check_dev_error()
    ref = _indexer_ref(inp["qI"], inp["w"], inp["q_pos"], np64(inp["kI"]), cfg.m, cfg.T)
    assert_scores_close(np64(scores), ref, 1e-5)
    # candidate mode: positions with -1 tail and some beyond the visible range
    g = torch.Generator().manual_seed(5)
    cand = torch.sort(torch.randperm(cfg.E, generator=g)[:100]).values.to(torch.int32)
    cand = torch.cat([cand, torch.full((28,), -1, dtype=torch.int32)]).repeat(rows, 1).to(DEV).contiguous()
    sc = torch.empty(rows, 128, device=DEV)
    csa.indexer_scores(c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"], sc, cand=cand)
    check_dev_error()
    cn = cand.cpu().numpy()
    ref_c = np.where(cn >= 0, np.take_along_axis(ref, np.maximum(cn, 0), axis=1), -np.inf)
    assert_scores_close(np64(sc), ref_c, 1e-5)


# ------------------------------------------------------------------ top-k

def _topk_check(scores, k, n_valid=None, cand=None):
    rows, n = scores.shape
    c = cfg_obj(k=k)
    idx = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    nvt = None if n_valid is None else torch.tensor(n_valid, dtype=torch.int32, device=DEV)
    csa.topk(c, scores, idx, n_valid=nvt, cand=cand)
    check_dev_error()
    s = scores.cpu().numpy()
    got = idx.cpu().numpy()
    for r in range(rows):
        nv = n if n_valid is None else n_valid[r]
        if cand is not None:
            cn = cand[r].cpu().numpy()
            nv = min(nv, int((cn >= 0).sum()))
            slots = O.topk(s[r], nv, k)
            ref = np.where(slots >= 0, cn[np.maximum(slots, 0)], -1)
        else:
            ref = O.topk(s[r], nv, k)
        assert np.array_equal(got[r], ref), f"row {r}"


def test_topk_long_rows_multilevel_with_ties():
    n = 300007
    s = rnd(31, (5, n))
    s = torch.round(s * 64) / 64          # coarse grid: many exact ties
    _topk_check(s.contiguous(), 512, n_valid=[n, 200000, 300, 511, 0])


def test_topk_small_rows_and_adversarial():
    s = rnd(32, (16, 512))
    _topk_check(s, 64)
    rows = torch.stack([torch.zeros(5000), torch.where(torch.arange(5000) % 2 == 0, 0.0, -0.0),
                        torch.full((5000,), -math.inf), torch.arange(5000, dtype=torch.float32),
                        -torch.arange(5000, dtype=torch.float32)]).to(DEV)
    _topk_check(rows.contiguous(), 512)
    _topk_check(rows.contiguous(), 4096)


def test_topk_long_rows_histogram_path_adversarial():
    """Few long rows take the histogram-guided path; ties that overflow its candidate list
    fall back to selecting over the whole row."""
    n = 40000
    coarse = (torch.round(rnd(35, (n,)) * 4) / 4).cpu()
    rows = torch.stack([torch.zeros(n), torch.where(torch.arange(n) % 2 == 0, 0.0, -0.0),
                        torch.arange(n, dtype=torch.float32), coarse, -torch.arange(n, dtype=torch.float32)])
    rows = rows.to(DEV).contiguous()
    _topk_check(rows, 512)
    _topk_check(rows, 512, n_valid=[n, 100, 30000, 1, 513])
    _topk_check(rows, 2048, n_valid=[n, 5000, 0, 39999, 2048])


def test_topk_many_prefill_rows():
    """More than 64 rows of prefill length take the one-CTA-per-row kernel (2,048 candidate
    slots for k <= 512): ragged and tiny valid counts, ties that overflow the candidate list,
    a candidate map, and a longer row."""
    n = 33792 + 5
    s = rnd(36, (80, n))
    s[40:] = torch.round(s[40:] * 8) / 8          # coarse values: many exact ties
    nv = [n, n - 3, 0, 1, 511, 512, 513, 20000, 36, 37]
    _topk_check(s.contiguous(), 512, n_valid=nv * 8)
    cand = torch.sort(torch.randperm(262144, generator=torch.Generator().manual_seed(9))[:n]).values.to(torch.int32)
    cand = cand.repeat(80, 1)
    cand[3, 30000:] = -1
    _topk_check(s.contiguous(), 512, cand=cand.to(DEV).contiguous())
    s2 = rnd(37, (70, 50000))
    _topk_check(s2.contiguous(), 512, n_valid=[50000, 40000, 7, 600, 36865] * 14)


def test_topk_many_rows_structured_against_the_sample():
    """Long rows of the one-CTA-per-row kernel whose large scores sit at positions the
    threshold estimate samples (the first 8 of every 64) or never samples: the estimate then
    finds all of them, none of them, or fewer than k at or above its digit (the whole-row
    histogram decides), and the selection stays exact."""
    rows, n = 80, 33792
    s = rnd(38, (rows, n)).cpu()
    pos = torch.arange(n)
    spikes = 100.0 + rnd(39, (rows, n)).cpu()
    s[20:40] = torch.where(pos % 64 == 3, spikes[20:40], s[20:40])      # all sampled
    s[40:60] = torch.where(pos % 64 == 40, spikes[40:60], s[40:60])     # never sampled
    s[60:80] = torch.where(pos % 64 < 8, spikes[60:80], s[60:80])       # the whole sample
    s = s.to(DEV).contiguous()
    for k in (512, 600, 64):
        _topk_check(s, k)
    _topk_check(s, 512, n_valid=[n, 16384, 16383, 8192] * 20)


def test_topk_candidate_map():
    rows, n = 4, 16384
    s = rnd(33, (rows, n))
    cand = torch.stack([torch.sort(torch.randperm(262144, generator=torch.Generator().manual_seed(r))[:n]).values
                        for r in range(rows)]).to(torch.int32)
    cand[1, 9000:] = -1
    cand = cand.to(DEV).contiguous()
    _topk_check(s, 512, cand=cand)


@pytest.mark.parametrize("n,nv,ties", [(20005, [20005, 12345, 100], True),
                                        (131072 + 37, [131072 + 37, 100003, 5000, 1], False),
                                        (131072 + 37, [131072 + 37, 70001], True)])
def test_block_pool_matches_oracle(n, nv, ties):
    """Sizes on both sides of the histogram-guided selection (>= 16,384 blocks a row), rows with
    fewer blocks than kept, and tied block maxima (the whole-row fallback)."""
    rows = len(nv)
    s = rnd(34, (rows, n))
    if ties:
        s = torch.round(s * 16) / 16
    c = cfg_obj()
    for n_blocks in (256, 2048):
        pool = torch.full((rows, n_blocks * 8), -7, dtype=torch.int32, device=DEV)
        cnt = torch.zeros(rows, dtype=torch.int32, device=DEV)
        csa.block_pool(c, s, pool, cnt, n_valid=torch.tensor(nv, dtype=torch.int32, device=DEV),
                       n_blocks=n_blocks)
        check_dev_error()
        sn = s.cpu().numpy()
        for r in range(rows):
            ref = O.hier_pool(sn[r], nv[r], 8, n_blocks)
            got = pool[r].cpu().numpy()
            assert int(cnt[r]) == ref.size
            assert np.array_equal(got[:ref.size], ref)
            assert np.all(got[ref.size:] == -1)


# ------------------------------------------------------------------ attention

def _attn_inputs(seed, B, T, H, d, E, k, L, dtype, n_sel_rows=None):
    q = rnd(seed, (B, T, H, d), d ** -0.5, dtype)
    kv = rnd(seed + 1, (B, E, d), d ** -0.5, dtype)
    kl = rnd(seed + 2, (B, L, d), d ** -0.5, dtype)
    sink = rnd(seed + 3, (H,))
    g = torch.Generator().manual_seed(seed)
    idx = torch.full((B * T, k), -1, dtype=torch.int32)
    for r in range(B * T):
        nsel = k if n_sel_rows is None else n_sel_rows[r % len(n_sel_rows)]
        idx[r, :nsel] = torch.sort(torch.randperm(E, generator=g)[:nsel]).values.to(torch.int32)
    return q, kv, kl, sink, idx.to(DEV)


def _attn_ref(q, kv, idx, kl, local_base, q_pos, sink, W, scale):
    B, T = q.shape[:2]
    qn, kvn, kln = np64(q), np64(kv), np64(kl)
    idn, lb, qp, sk = idx.cpu().numpy(), local_base.cpu().numpy(), q_pos.cpu().numpy(), np64(sink)
    outs, lses = [], []
    for r in range(B * T):
        b, t = divmod(r, T)
        rows = O.gather_rows(kvn[b], idn[r], kln[b], int(lb[b]), int(qp[r]), W)
        o, l = O.sparse_attention(qn[b, t], rows, sk, scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs).reshape(q.shape), np.stack(lses).reshape(B, T, -1)


# B = 3, 2: four head groups per decode CTA; B = 10: two; B = 16: one (64 heads).
# >= 152 query rows take the one-CTA-per-query pipelined kernel (64-row tiles): ragged tiles,
# empty selections and clipped windows
@pytest.mark.parametrize("B,T,nsel", [(3, 1, [512, 300, 512]), (1, 160, [512, 77]), (2, 2, [0, 512]),
                                      (10, 1, [512, 300, 17, 0, 512]), (16, 1, [512, 1, 400]),
                                      (3, 60, [0, 512, 1, 63, 64, 65, 300])])
def test_attention_tensor_cores(B, T, nsel):
    H, d, E, k, W, L = 64, 512, 1500, 512, 128, 200
    q, kv, kl, sink, idx = _attn_inputs(40 + T + B, B, T, H, d, E, k, L, BF16, nsel)
    local_base = torch.tensor([[1000, 1040, 0][b % 3] for b in range(B)], dtype=torch.int64, device=DEV)
    # windows: fully held, clipped by the local rows' start, and t < W - 1 (starts at 0)
    base_t = [1000 + 150, 1040 + 60, 50]
    q_pos = torch.tensor([base_t[b % 3] + (t % 3) for b in range(B) for t in range(T)], dtype=torch.int64, device=DEV)
    c = cfg_obj(B=B)
    out = torch.empty(B, T, H, d, device=DEV, dtype=BF16)
    lse = torch.empty(B, T, H, device=DEV)
    csa.sparse_attn(c, q, kv, idx, kl, local_base, q_pos, sink, out, lse)
    check_dev_error()
    ro, rl = _attn_ref(q, kv, idx, kl, local_base, q_pos, sink, W, d ** -0.5)
    w1 = assert_rows_close(np64(out), ro, 2e-2)
    np.testing.assert_allclose(np64(lse), rl, atol=2e-3, rtol=0)
    print(f"attention B={B} T={T}: worst/tol = {w1:.3f}")


def test_attention_cuda_core_fp32():
    cfg = gen.CONFIGS[1]
    H, d, k, W = cfg.H, cfg.d, cfg.k, cfg.W
    B, T, E, L = 2, 16, 512, 60
    q, kv, kl, sink, idx = _attn_inputs(50, B, T, H, d, E, k, L, torch.float32, [64, 10, 0, 64])
    local_base = torch.tensor([100, 0], dtype=torch.int64, device=DEV)
    q_pos = torch.tensor([130 + t for t in range(T)] + [5 + t for t in range(T)], dtype=torch.int64, device=DEV)
    c = lib_config(cfg, B=B)
    out = torch.empty(B, T, H, d, device=DEV)
    lse = torch.empty(B, T, H, device=DEV)
    csa.sparse_attn(c, q, kv, idx, kl, local_base, q_pos, sink, out, lse)
    check_dev_error()
    ro, rl = _attn_ref(q, kv, idx, kl, local_base, q_pos, sink, W, cfg.softmax_scale)
    np.testing.assert_allclose(np64(out), ro, atol=1e-5, rtol=1e-4)
    np.testing.assert_allclose(np64(lse), rl, atol=1e-5, rtol=1e-5)


# ------------------------------------------------------------------ compositions

@pytest.mark.parametrize("cid,N,HI", [(2, 4 * 1500, 64), (4, 4 * 2500, 64),
                                      # fewer visible entries than k (padded selection), windows
                                      # reaching back to position 0, and the 32-head indexer
                                      (2, 4 * 30, 64), (4, 4 * 130, 64), (2, 4 * 700, 32)])
def test_decode_step_matches_oracle(cid, N, HI):
    cfg = gen.CONFIGS[cid].replace(B=3, N=N, HI=HI)
    inp = gen.make_inputs(cfg, DEV)
    inp["q_pos"][1] = N - 3          # this token completes no block: no compression
    kv_before = inp["kv_comp"].clone()
    ref = oracle_decode(cfg, inp)   # oracle reads the inputs before the step mutates the caches
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    out, lse, idx = run_gpu_decode(cfg, inp, scores_out=scores)
    assert_decode_matches(cfg, inp, ref, out, lse, idx)
    assert_step_selection_exact(cfg, ref, idx, scores)
    for b in range(cfg.B):
        if ref[b]["entry"] is None:
            assert torch.equal(inp["kv_comp"][b], kv_before[b])


@pytest.mark.parametrize("cid", [2, 4])
@pytest.mark.parametrize("kind", ["duplicate_keys", "zero_gates", "skewed"])
def test_decode_step_selection_exact_on_ties(cid, kind):
    """The in-step selection on rows full of exact ties or skewed toward the end: 3,000 copies
    of one key row (equal scores straddling the threshold), all gates zero (every score 0:
    positions 0 .. k-1), and key magnitudes growing with the position (the best scores crowd
    the end of the row)."""
    cfg = gen.CONFIGS[cid].replace(B=2, N=4 * 5000)
    inp = gen.make_inputs(cfg, DEV)
    if kind == "duplicate_keys":
        inp["kI"][:, 1000:4000] = inp["kI"][:, 7:8]
        if "kscale" in inp:
            inp["kscale"][:, 1000:4000] = inp["kscale"][:, 7:8]
    elif kind == "zero_gates":
        inp["w"].zero_()
    else:
        inp["qI"].abs_()
        inp["w"].abs_()
        if "kscale" in inp:
            inp["kI"].copy_(inp["kI"] & 0x7F)      # positive e4m3 codes
            inp["kscale"].copy_(torch.arange(1, cfg.E + 1, device=DEV, dtype=torch.float32)[None] * 1e-3)
        else:
            inp["kI"].copy_((inp["kI"].float().abs() * torch.arange(1, cfg.E + 1, device=DEV)[None, :, None] * 1e-3)
                            .to(inp["kI"].dtype))
    ref = oracle_decode(cfg, inp)
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    out, lse, idx = run_gpu_decode(cfg, inp, scores_out=scores)
    assert_step_selection_exact(cfg, ref, idx, scores)
    if kind == "zero_gates":
        np.testing.assert_array_equal(idx.cpu().numpy(), np.tile(np.arange(cfg.k), (cfg.B, 1)))
    assert_decode_matches(cfg, inp, ref, out, lse, idx)


def _candidates(s32, nv, k):
    """Candidates of the histogram selection over s32[:nv]: scores whose 12-bit digit (of the
    order-preserving key) is at least the digit of the k-th largest."""
    bits = s32[:nv].astype(np.float32).view(np.uint32)
    key = np.where(bits >> 31, ~bits, bits | np.uint32(0x80000000)).astype(np.uint32)
    dig = key >> 20
    b1 = np.sort(dig)[::-1][min(k, nv) - 1]
    return int((dig >= b1).sum())


@pytest.mark.parametrize("cid", [2, 4])
def test_decode_step_cut_tie_among_few_candidates(cid):
    """Sixty keys given one score ranked just above the k-th largest, in a row of few
    candidates: the step's attention starts on the candidates before the list is written and
    masks them with the published threshold and tie cut; the selection (lowest positions among
    the tied keys) and the outputs stay exact."""
    cfg = gen.CONFIGS[cid].replace(B=2, N=4 * 20000)
    inp = gen.make_inputs(cfg, DEV)
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    run_gpu_decode(cfg, {kk: v.clone() for kk, v in inp.items()}, scores_out=scores)
    nv = [min(int(inp["q_pos"][b]) + 1, cfg.m * cfg.E) // cfg.m for b in range(cfg.B)]
    for b in range(cfg.B):
        order = torch.argsort(scores[b, :nv[b] - 1], descending=True).cpu()
        src = int(order[cfg.k - 25])
        dst = order[cfg.k + 100:cfg.k + 160].to(DEV)      # sixty keys ranked below it
        inp["kI"][b, dst] = inp["kI"][b, src].clone()
        if "kscale" in inp:
            inp["kscale"][b, dst] = inp["kscale"][b, src].clone()
    ref = oracle_decode(cfg, inp)
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    out, lse, idx = run_gpu_decode(cfg, inp, scores_out=scores)
    for b in range(cfg.B):
        s32 = scores[b].cpu().numpy()
        assert _candidates(s32, nv[b], cfg.k) <= 1024, "the row must stay in the candidate mode"
        top = O.topk(s32, nv[b], cfg.k)
        t = np.sort(s32[:nv[b]])[::-1][cfg.k - 1]
        assert int((s32[:nv[b]] == t).sum()) > int((s32[top] == t).sum()), "a tie must be cut"
    assert_step_selection_exact(cfg, ref, idx, scores)
    assert_decode_matches(cfg, inp, ref, out, lse, idx)


def test_decode_step_counters_across_modes():
    """Consecutive steps on one workspace alternate between a row of few candidates (the
    attention starts on them before the selection writes its list) and a row whose threshold
    bin holds thousands of equal scores (the attention waits for the written list): the step
    counters stay in step and every selection is exact."""
    cfg = gen.CONFIGS[4].replace(B=2, N=4 * 20000)
    plain = gen.make_inputs(cfg, DEV)
    tied = {kk: v.clone() for kk, v in plain.items()}
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    run_gpu_decode(cfg, {kk: v.clone() for kk, v in plain.items()}, scores_out=scores)
    nv = [min(int(plain["q_pos"][b]) + 1, cfg.m * cfg.E) // cfg.m for b in range(cfg.B)]
    for b in range(cfg.B):
        order = torch.argsort(scores[b, :nv[b] - 1], descending=True).cpu()
        src = int(order[cfg.k - 25])
        dst = order[cfg.k + 100:cfg.k + 3100].to(DEV)     # 3,000 keys ranked below it
        tied["kI"][b, dst] = tied["kI"][b, src].clone()
        tied["kscale"][b, dst] = tied["kscale"][b, src].clone()
    for inp, list_mode in ((plain, False), (tied, True), (plain, False), (tied, True), (plain, False)):
        run = {kk: v.clone() for kk, v in inp.items()}
        ref = oracle_decode(cfg, run)
        scores = torch.empty(cfg.B, cfg.E, device=DEV)
        out, lse, idx = run_gpu_decode(cfg, run, scores_out=scores)
        for b in range(cfg.B):
            n_cand = _candidates(scores[b].cpu().numpy(), nv[b], cfg.k)
            assert (n_cand > 1024) == list_mode, (b, n_cand, list_mode)
        assert_step_selection_exact(cfg, ref, idx, scores)
        assert_decode_matches(cfg, run, ref, out, lse, idx)


def test_decode_step_through_step_inputs():
    """The decode step reading its per-step inputs (queries, gates, stream tails, window rows)
    from one StepInputs buffer: another sequence pair's inputs written into the host mirror and
    moved with one upload give the outputs the oracle computes for them."""
    cfg = gen.CONFIGS[2].replace(B=2, N=4 * 5000)
    keys = ["q", "qI", "w", "q_pos", "kv_str", "z_str", "kvI_str", "zI_str", "kv_local"]
    inp = gen.make_inputs(cfg, DEV)
    other = gen.make_inputs(cfg, DEV, row0=2)
    st = csa.StepInputs({k: inp[k] for k in keys})
    run = dict(inp)
    run.update(st.dev)
    for k in keys:
        if k != "q_pos":            # the caches and window base stay those of the first pair
            st.host[k].copy_(other[k])
    st.upload()
    want = {k: v.clone() for k, v in run.items()}
    ref = oracle_decode(cfg, want)
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    out, lse, idx = run_gpu_decode(cfg, run, scores_out=scores)
    assert torch.equal(run["q"], other["q"])
    assert_step_selection_exact(cfg, ref, idx, scores)
    assert_decode_matches(cfg, run, ref, out, lse, idx)


def test_tiny_end_to_end_fp32():
    """Preset 1: compress every entry from the streams, index, select, attend (16 queries)."""
    cfg = gen.CONFIGS[1]
    inp = gen.make_inputs(cfg, DEV)
    c = lib_config(cfg)
    kvc = torch.zeros(cfg.B, cfg.E, cfg.d, device=DEV)
    kI = torch.zeros(cfg.B, cfg.E, cfg.dI, device=DEV)
    csa.compress_kv(c, inp["kv_str"], inp["z_str"], inp["bias"], 0, 0, cfg.E, kvc)
    csa.compress_kv(c, inp["kvI_str"], inp["zI_str"], inp["biasI"], 0, 0, cfg.E, kI)
    rows = cfg.B * cfg.T
    scores = torch.empty(rows, cfg.E, device=DEV)
    csa.indexer_scores(c, inp["qI"], inp["w"], inp["q_pos"], kI, scores)
    idx = torch.empty(rows, cfg.k, dtype=torch.int32, device=DEV)
    nv = ((inp["q_pos"] + 1) // cfg.m).clamp(max=cfg.E).to(torch.int32)
    csa.topk(c, scores, idx, n_valid=nv)
    out = torch.empty(cfg.B, cfg.T, cfg.H, cfg.d, device=DEV)
    lse = torch.empty(cfg.B, cfg.T, cfg.H, device=DEV)
    csa.sparse_attn(c, inp["q"], kvc, idx, inp["kv_local"], inp["local_base"], inp["q_pos"], inp["sink"], out, lse)
    check_dev_error()
    nb = np_inputs(inp)
    kv_ref = O.compress_range(nb["kv_str"][0], nb["z_str"][0], nb["bias"], cfg.m, 0, cfg.E)
    ki_ref = O.compress_range(nb["kvI_str"][0], nb["zI_str"][0], nb["biasI"], cfg.m, 0, cfg.E)
    for tq in range(cfg.T):
        r = O.decode_token(cfg, nb, 0, tq, kv_ref, ki_ref)
        fin = r["scores"][np.isfinite(r["scores"])]
        tol = 1e-5 * np.sqrt((fin ** 2).mean())
        swaps = assert_selection_ok(idx[tq].cpu().numpy(), r["idx"], r["scores"], cfg.k, tol)
        assert swaps == 0
        np.testing.assert_allclose(np64(out[0, tq]), r["out"], atol=1e-4, rtol=0)
        np.testing.assert_allclose(np64(lse[0, tq]), r["lse"], atol=1e-4, rtol=0)


def test_csa2_group_matches_oracle():
    """CSA2 decoder group: Full-layer scan -> block pool -> Reindex rescoring -> top-k -> 4 attentions."""
    base = gen.CONFIGS[5]
    cfg = base.replace(B=2, N=6000)
    n_blocks = 128
    inp = gen.make_inputs(cfg, DEV)
    c = lib_config(cfg)
    B, E = cfg.B, cfg.E
    s_full = torch.empty(B, E, device=DEV)
    csa.indexer_scores(c, inp["qI_full"], inp["w_full"], inp["q_pos"], inp["kI"], s_full)
    pool = torch.empty(B, n_blocks * 8, dtype=torch.int32, device=DEV)
    cnt = torch.empty(B, dtype=torch.int32, device=DEV)
    csa.block_pool(c, s_full, pool, cnt, n_blocks=n_blocks)
    s_pool = torch.empty(B, n_blocks * 8, device=DEV)
    csa.indexer_scores(c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"], s_pool, cand=pool)
    idx = torch.empty(B, cfg.k, dtype=torch.int32, device=DEV)
    csa.topk(c, s_pool, idx, n_valid=cnt, cand=pool)
    outs = []
    for layer in range(1 + cfg.n_reuse):
        o = torch.empty(B, 1, cfg.H, cfg.d, device=DEV, dtype=BF16)
        csa.sparse_attn(c, inp["q"][layer], inp["kv_comp"], idx, inp["kv_local"][layer], inp["local_base"],
                        inp["q_pos"], inp["sink"][layer], o)
        outs.append(o)
    check_dev_error()
    nb = np_inputs(inp)
    for b in range(B):
        t = int(nb["q_pos"][b])
        nv = min(t + 1, E)
        sf64 = O.indexer_scores(nb["qI_full"][b, 0], nb["w_full"][b, 0], nb["kI"][b], nv)
        gpool = pool[b, :int(cnt[b])].cpu().numpy().astype(np.int64)
        tol_scan = 1e-2 * np.sqrt((sf64[:nv] ** 2).mean())
        assert_pool_valid(gpool, sf64.astype(np.float32), nv, 8, n_blocks, tol_scan)
        srei = O.indexer_scores_subset(nb["qI"][b, 0], nb["w"][b, 0], nb["kI"][b], gpool)
        slots = O.topk(srei.astype(np.float32), gpool.size, cfg.k)
        ridx = np.where(slots >= 0, gpool[np.maximum(slots, 0)], -1)
        all_rei = O.indexer_scores(nb["qI"][b, 0], nb["w"][b, 0], nb["kI"][b], nv)
        tol = 1e-2 * np.sqrt((all_rei[:nv] ** 2).mean())
        gi = idx[b].cpu().numpy()
        assert_selection_ok(gi, ridx, all_rei, cfg.k, tol)
        g_set, r_set = set(gi[gi >= 0].tolist()), set(ridx[ridx >= 0].tolist())
        for layer in range(1 + cfg.n_reuse):
            rows = O.gather_rows(nb["kv_comp"][b], ridx, nb["kv_local"][layer][b], int(nb["local_base"][b]), t,
                                 cfg.W)
            ro, rl = O.sparse_attention(nb["q"][layer][b, 0], rows, nb["sink"][layer], cfg.softmax_scale)
            bound = swap_bound(nb["q"][layer][b, 0], rl, cfg.softmax_scale,
                               [nb["kv_comp"][b][x] for x in g_set - r_set], [nb["kv_comp"][b][y] for y in r_set - g_set])
            assert_out_close_with_swaps(np64(outs[layer][b, 0]), ro, 2e-2, bound, what=f"layer {layer} b={b}")


def test_decode_step_call_matches_decode_step():
    """The prepared decode-step call enqueues exactly what decode_step does."""
    cfg = gen.CONFIGS[2].replace(B=2, N=4 * 900)
    inp = gen.make_inputs(cfg, DEV)
    c = lib_config(cfg)
    kwargs = dict(q_pos=inp["q_pos"], q=inp["q"], qI=inp["qI"], w=inp["w"], sink=inp["sink"], kv_comp=inp["kv_comp"],
                  kI=inp["kI"], kv_tail=inp["kv_str"], z_tail=inp["z_str"], kvI_tail=inp["kvI_str"],
                  zI_tail=inp["zI_str"], bias=inp["bias"], biasI=inp["biasI"], kv_local=inp["kv_local"],
                  local_base=inp["local_base"])
    outs = []
    for prepared in (False, True):
        out = torch.empty(cfg.B, cfg.H, cfg.d, device=DEV, dtype=BF16)
        lse = torch.empty(cfg.B, cfg.H, device=DEV)
        idx = torch.empty(cfg.B, cfg.k, dtype=torch.int32, device=DEV)
        if prepared:
            call = csa.DecodeStepCall(c, out=out, lse=lse, idx_out=idx, **kwargs)
            call()
            call()
        else:
            csa.decode_step(c, out=out, lse=lse, idx_out=idx, **kwargs)
        check_dev_error()
        outs.append((out, lse, idx))
    assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1]))
