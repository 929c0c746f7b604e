"""Parity at the benchmark's full sizes, through the benchmark's own step functions.

The workloads are built by bench.py's workload classes and run as a CUDA-graph replay of
their step, exactly as the benchmark times them, then checked against the oracle:
  decode @64K (batch 16, bf16 keys) and @1M (batch 4, FP8 keys; and MXFP4 keys): every sequence;
  prefill chunk (4,096 queries after 131,072 tokens): all 1,024 new entries of both caches,
  and indexer scores / top-k / attention on sampled query rows (first and last included);
  CSA2 decoder group at 262,144 tokens (batch 8): every sequence through all four layers;
  HCA decode @1M (batch 4, 8,192 entries a sequence): every sequence; HCA prefill chunk: the 32
  new entries and sampled query rows; the attention prologue / epilogue of the prefill chunk:
  every new cache entry and sampled tokens of the query and output passes; the decode
  attention @1M over FP8 and over MXFP4 main-KV entries: the packed rows bit-exact, every
  sequence's output.
Agreement criteria are those of the small-size parity tests.
"""
import numpy as np
import pytest
import torch

import compressed_sparse_attention_csa_gb300 as csa
from _helpers import (assert_decode_matches, assert_step_selection_exact, assert_entries_close, assert_out_close_with_swaps, assert_pool_valid,
                      assert_rows_close, assert_scores_close, assert_selection_ok, np64, np_inputs, oracle_decode,
                      swap_bound)
from test_gpu_epilogue import assert_vectors_close, e4m3_half_step
from test_gpu_hca import assert_single_entries_close
from bench import Csa2Group, Decode, Epilogue, Fp8KvAttn, HcaDecode, HcaPrefill, Mxfp4KvAttn, Prefill
from oracle import csa_oracle as O
from synth import gen

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0)


def replay_once(fn):
    fn()                       # first call allocates the workspace outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    assert csa.get_last_error() == 0


def host(x):
    return np64(x) if x.is_floating_point() else x.cpu().numpy()


@pytest.mark.parametrize("cid", [2, 4, 13])
def test_decode_full_size(cid):
    cfg = gen.CONFIGS[cid]
    wl = Decode(cfg, csa, torch, DEV, 0)
    wl.args["scores_out"] = wl.scores          # the step's scores, for the exact selection check
    ref = oracle_decode(cfg, wl.inp)          # reads the caches before the step writes entry E-1
    replay_once(wl.step)
    assert_decode_matches(cfg, wl.inp, ref, wl.out, wl.lse, wl.idx)
    assert_step_selection_exact(cfg, ref, wl.idx, wl.scores)


def test_prefill_full_size_sampled_rows():
    cfg = gen.CONFIGS[3]
    wl = Prefill(cfg, csa, torch, DEV, 0)
    inp = wl.inp
    h = {k: host(v if k in ("bias", "biasI", "sink", "q_pos") else v[0:1]) for k, v in inp.items()}
    kv_o, kI_o = h["kv_comp"][0].copy(), h["kI"][0].copy()
    replay_once(wl.step)

    # the chunk's compression: every new entry of both caches
    new_kv = O.compress_range(h["kv_str"][0], h["z_str"][0], h["bias"], cfg.m, wl.e0, wl.e1, tok0=wl.tok0)
    new_kI = O.compress_range(h["kvI_str"][0], h["zI_str"][0], h["biasI"], cfg.m, wl.e0, wl.e1, tok0=wl.tok0)
    assert_entries_close(np64(inp["kv_comp"][0, wl.e0:wl.e1]), new_kv, h["kv_str"])
    assert_entries_close(np64(inp["kI"][0, wl.e0:wl.e1]), new_kI, h["kvI_str"])
    kv_o[wl.e0:wl.e1] = new_kv
    kI_o[wl.e0:wl.e1] = new_kI

    rng = np.random.default_rng(3)
    rows = sorted(set([0, 1, 2, 3, 4, 1023, 2048, 3071, 4092, 4093, 4094, 4095] +
                      rng.integers(0, cfg.T, 12).tolist()))
    sub = cfg.replace(B=1)
    scores = wl.scores
    for tq in rows:
        r = O.decode_token(sub, h, 0, tq, kv_o, kI_o)
        nv = r["nv"]
        got_s = np64(scores[tq])
        assert_scores_close(got_s[:nv], r["scores"][:nv], 1e-2, what=f"scores row {tq}")
        assert np.all(np.isneginf(got_s[nv:])), f"row {tq}: invisible entries must be -inf"
        fin = r["scores"][:nv]
        tol = 1e-2 * np.sqrt((fin ** 2).mean())
        gi = wl.idx[tq].cpu().numpy()
        swaps = assert_selection_ok(gi, r["idx"], r["scores"], cfg.k, tol)
        g_set, r_set = set(gi[gi >= 0].tolist()), set(r["idx"][r["idx"] >= 0].tolist())
        bound = swap_bound(h["q"][0, tq], r["lse"], cfg.softmax_scale, [kv_o[x] for x in g_set - r_set],
                           [kv_o[y] for y in r_set - g_set])
        assert_out_close_with_swaps(np64(wl.out[0, tq]), r["out"], 2e-2, bound, what=f"out row {tq} swaps={swaps}")
        np.testing.assert_allclose(np64(wl.lse[0, tq]), r["lse"], atol=5e-3)


def test_csa2_group_full_size():
    cfg = gen.CONFIGS[5]
    wl = Csa2Group(cfg, csa, torch, DEV, 0)
    inp = wl.inp
    replay_once(wl.step)
    for b in range(cfg.B):
        h = {}
        for k, v in inp.items():
            if k in ("q", "kv_local"):
                h[k] = host(v[:, b])
            elif k == "sink":
                h[k] = host(v)
            else:
                h[k] = host(v[b])
        t = int(h["q_pos"])
        nv = min(t + 1, cfg.E)
        sf64 = O.indexer_scores(h["qI_full"][0], h["w_full"][0], h["kI"], nv)
        assert_scores_close(np64(wl.s_full[b])[:nv], sf64[:nv], 1e-2, what=f"full scan b={b}")
        # The GPU pool comes from the GPU's scan scores: it must be one of the pools that
        # scores within tolerance of the oracle's give (membership differs only at near-tied
        # block maxima).  The Reindex step is then checked on that validated pool.
        gpool = wl.pool[b, :int(wl.cnt[b])].cpu().numpy().astype(np.int64)
        tol_scan = 1e-2 * np.sqrt((sf64[:nv] ** 2).mean())
        assert_pool_valid(gpool, sf64.astype(np.float32), nv, 8, wl.N_BLOCKS, tol_scan)
        all_rei = O.indexer_scores(h["qI"][0], h["w"][0], h["kI"], nv)
        slots = O.topk(all_rei[gpool].astype(np.float32), gpool.size, cfg.k)
        ridx = np.where(slots >= 0, gpool[np.maximum(slots, 0)], -1)
        tol = 1e-2 * np.sqrt((all_rei[:nv] ** 2).mean())
        gi = wl.idx[b].cpu().numpy()
        assert_selection_ok(gi, ridx, all_rei, cfg.k, tol)
        assert np.all(np.isin(gi[gi >= 0], gpool))
        g_set, r_set = set(gi[gi >= 0].tolist()), set(ridx[ridx >= 0].tolist())
        for layer in range(wl.layers):
            rows = O.gather_rows(h["kv_comp"], ridx, h["kv_local"][layer], int(h["local_base"]), t, cfg.W)
            ro, rl = O.sparse_attention(h["q"][layer][0], rows, h["sink"][layer], cfg.softmax_scale)
            bound = swap_bound(h["q"][layer][0], rl, cfg.softmax_scale, [h["kv_comp"][x] for x in g_set - r_set],
                               [h["kv_comp"][y] for y in r_set - g_set])
            assert_out_close_with_swaps(np64(wl.outs[layer, b, 0]), ro, 2e-2, bound, what=f"layer {layer} b={b}")


def test_hca_decode_full_size():
    cfg = gen.CONFIGS[6]
    wl = HcaDecode(cfg, csa, torch, DEV, 0)
    h = np_inputs(wl.inp)
    kv_before = [h["kv_comp"][b].copy() for b in range(cfg.B)]
    replay_once(wl.step)
    for b in range(cfg.B):
        kvc = kv_before[b]
        r = O.hca_decode_step_sequence(cfg, h, b, kvc)
        e, ent = r["entry"]
        assert_single_entries_close(np64(wl.inp["kv_comp"][b, e]), ent, h["kv_str"][b], cfg.m, torch.bfloat16)
        assert_rows_close(np64(wl.out[b]), r["out"], 2e-2, what=f"out b={b}")
        np.testing.assert_allclose(np64(wl.lse[b]), r["lse"], atol=5e-3)


def test_hca_prefill_full_size_sampled_rows():
    cfg = gen.CONFIGS[7]
    wl = HcaPrefill(cfg, csa, torch, DEV, 0)
    inp = wl.inp
    h = {k: host(v if k in ("bias", "sink", "q_pos") else v[0:1]) for k, v in inp.items()}
    kv_o = h["kv_comp"][0].copy()
    replay_once(wl.step)
    new = O.compress_single_range(h["kv_str"][0], h["z_str"][0], h["bias"], cfg.m, wl.e0, wl.e1, tok0=wl.tok0)
    assert_single_entries_close(np64(inp["kv_comp"][0, wl.e0:wl.e1]), new, h["kv_str"], cfg.m, torch.bfloat16)
    kv_o[wl.e0:wl.e1] = new
    sub = cfg.replace(B=1)
    for tq in [0, 1, 127, 128, 2047, 4094, 4095]:
        r = O.hca_token(sub, h, 0, tq, kv_o)
        assert_rows_close(np64(wl.out[0, tq]), r["out"], 2e-2, what=f"out row {tq}")
        np.testing.assert_allclose(np64(wl.lse[0, tq]), r["lse"], atol=5e-3)


def test_epilogue_full_size_sampled_tokens():
    cfg = gen.CONFIGS[9]
    wl = Epilogue(cfg, csa, torch, DEV, 0)
    inp = wl.inp
    h = {k: host(inp[k] if k in ("bias", "q_norm", "kv_norm", "q_pos") else inp[k][0:1])
         for k in ["q", "o", "q_pos", "kv_str", "z_str", "bias", "q_norm", "kv_norm"]}
    replay_once(wl.step)
    ents = np.stack([O.norm_rope(O.compress_entry(h["kv_str"][0], h["z_str"][0], h["bias"], cfg.m, i, tok0=wl.tok0),
                                 O.compressed_entry_position(cfg.m, i), h["kv_norm"], 1e-6, 64, 10000.0)
                     for i in range(wl.e0, wl.e1)])
    assert_vectors_close(np64(inp["kv_comp"][0, wl.e0:wl.e1]), ents, torch.bfloat16, "new cache entries")
    codes = wl.codes.cpu().numpy()
    sc = wl.scales.cpu().numpy().astype(np.float64)
    for tq in [0, 1, 1000, 4095]:
        t = int(h["q_pos"][tq])
        ref_q = O.norm_rope(h["q"][0, tq], t, h["q_norm"], 1e-6, 64, 10000.0)
        assert_vectors_close(np64(wl.q_out[0, tq]), ref_q, torch.bfloat16, f"query {tq}")
        ref_o = O.inverse_rope(h["o"][0, tq], t, 64, 10000.0)
        amax = np.abs(ref_o).max(axis=-1)
        np.testing.assert_allclose(sc[tq], amax / 448.0, rtol=2.0 ** -20)
        deq = O.e4m3_decode(codes[0, tq]) * sc[tq][:, None]
        tol = 1.01 * e4m3_half_step(ref_o / sc[tq][:, None]) * sc[tq][:, None] + 1e-6 * amax[:, None]
        assert float((np.abs(deq - ref_o) / tol).max()) <= 1.0, f"fp8 output of token {tq}"


@pytest.mark.parametrize("cid,Wl,enc,dec_fn", [(10, Fp8KvAttn, O.kv_fp8_encode, O.kv_fp8_decode),
                                               (11, Mxfp4KvAttn, O.mxfp4_encode, O.mxfp4_decode)])
def test_quantised_kv_attention_full_size(cid, Wl, enc, dec_fn):
    cfg = gen.CONFIGS[cid]
    wl = Wl(cfg, csa, torch, DEV, 0)
    inp = wl.inp
    replay_once(wl.step)
    for b in range(cfg.B):
        sel = inp["idx"][b].long()
        ent = np64(inp["kv_comp"][b][sel])
        code = enc(ent)
        assert np.array_equal(wl.kv8[b][sel].cpu().numpy(), code)
        dec = dec_fn(code)
        lb, t = int(inp["local_base"][b]), int(inp["q_pos"][b])
        kl = np64(inp["kv_local"][b])
        rows = np.concatenate([dec, np.stack([kl[p - lb] for p in O.window_positions(t, cfg.W, lb, kl.shape[0])])])
        ro, rl = O.sparse_attention(np64(inp["q"][b, 0]), rows, np64(inp["sink"]), cfg.softmax_scale)
        assert_rows_close(np64(wl.out[b, 0]), ro, 2e-2, what=f"out b={b}")
        np.testing.assert_allclose(np64(wl.lse[b, 0]), rl, atol=5e-3)
