"""Parity of the HCA path (one-stream compressor, dense attention, HCA decode step) with the
CPU oracle on seeded inputs (GPU required).

Agreement:
  compressor: the output rounding (bf16: 2^-8 relative; fp32: 2^-23) plus the fp32 error of
    the m-term softmax-weighted sum, bounded by 4 m 2^-24 of the largest stream value;
  attention: |g - r| <= 2e-2 * max|r_row| for bf16 outputs (lse within 5e-3), 1e-4 for fp32.
"""
import numpy as np
import pytest
import torch

import compressed_sparse_attention_csa_gb300 as csa
from _helpers import assert_rows_close, lib_config, np64, np_inputs
from oracle import csa_oracle as O
from synth import gen

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


def rnd(seed, shape, std=1.0, dtype=torch.float32):
    n = int(np.prod(shape))
    return gen.normal(seed, n, device=DEV, std=std).reshape(shape).to(dtype)


def check_dev_error():
    assert csa.get_last_error() == 0


def hca_cfg(**kw):
    base = dict(B=2, H=64, d=512, HI=64, dI=128, m=128, k=512, W=128, act=BF16, fp8_keys=False,
                softmax_scale=None)
    base.update(kw)
    return csa.Config(**base)


def assert_single_entries_close(got, ref, streams, m, act):
    """Output rounding plus 4 m 2^-24 of the largest stream value (fp32 weighted sum of m terms)."""
    atol = 4.0 * m * 2.0 ** -24 * float(np.abs(streams).max())
    rel = 2.0 ** -8 if act == BF16 else 2.0 ** -23
    err = np.abs(np.asarray(got, np.float64) - ref)
    worst = float((err / (rel * np.abs(ref) + atol)).max())
    assert worst <= 1.0, f"one-stream entries: worst error is {worst:.3f} x tolerance"
    return worst


# ------------------------------------------------------------------ one-stream compressor

@pytest.mark.parametrize("m,dim,act,with_bias,ent_begin,n_ent", [
    (128, 512, BF16, True, 0, 9),      # HCA main KV
    (128, 512, BF16, True, 5, 3),      # a range that starts past entry 0
    (2, 128, BF16, False, 0, 301),     # CSA2 encoder pairs, no positional bias
    (2, 512, BF16, False, 7, 64),
    (128, 64, torch.float32, True, 0, 4),
    (16, 96, torch.float32, False, 1, 11),
    (1, 32, torch.float32, True, 0, 40),
])
def test_compress_single_matches_oracle(m, dim, act, with_bias, ent_begin, n_ent):
    B = 3
    tok0 = m * ent_begin - (m if ent_begin else 0)   # the buffer starts one block early when it can
    n_tok = m * (ent_begin + n_ent) - tok0 + 5          # and runs 5 tokens past the last block
    kv = rnd(300 + m + dim, (B, n_tok, dim), dim ** -0.5, act)
    z = rnd(301 + m + dim, (B, n_tok, dim), 1.0, act)
    bias = rnd(302 + m, (m, dim), 0.1) if with_bias else None
    E_cap = ent_begin + n_ent + 2
    c = hca_cfg(B=B, m=m, act=act, d=dim)
    out = torch.full((B, E_cap, dim), 7.0, device=DEV, dtype=act)
    csa.compress_kv_single(c, kv, z, bias, tok0, ent_begin, ent_begin + n_ent, out)
    check_dev_error()
    bn = np64(bias) if with_bias else None
    for b in range(B):
        ref = O.compress_single_range(np64(kv[b]), np64(z[b]), bn, m, ent_begin, ent_begin + n_ent, tok0=tok0)
        assert_single_entries_close(np64(out[b, ent_begin:ent_begin + n_ent]), ref, np64(kv), m, act)
        # rows outside the range are untouched
        assert torch.all(out[b, :ent_begin] == 7.0) and torch.all(out[b, ent_begin + n_ent:] == 7.0)


# ------------------------------------------------------------------ dense attention

def _dense_ref(q, kv, kl, local_base, q_pos, sink, m, W, scale):
    qn, kvn, kln, sn = np64(q), np64(kv), np64(kl), np64(sink)
    B, T = q.shape[0], q.shape[1]
    outs = np.zeros(qn.shape)
    lses = np.zeros(qn.shape[:3])
    for b in range(B):
        for t in range(T):
            p = int(q_pos[b * T + t])
            nv = min(O.visible_entries(p, m), kvn.shape[1])
            rows = O.dense_rows(kvn[b], nv, kln[b], int(local_base[b]), p, W)
            outs[b, t], lses[b, t] = O.sparse_attention(qn[b, t], rows, sn, scale)
    return outs, lses


@pytest.mark.parametrize("B,T,E,m", [
    (1, 300, 600, 128),    # many queries: one CTA per query, long dense row lists
    (2, 90, 1100, 128),    # 180 queries
    (3, 1, 2000, 128),     # decode: TMA-streamed splits of the rows, merged with the sink
    (4, 1, 8192 + 37, 128),
    (2, 1, 100, 128),      # few rows: two splits
    (5, 1, 3000, 4),       # dense over a CSA-rate cache
    (2, 20, 700, 128),     # few queries per sequence, each split over CTAs
    (1, 1, 40000, 128),    # more entries than the streaming kernel's splits hold: pipelined splits
])
def test_dense_attn_tensor_cores(B, T, E, m):
    H, d, W, L = 64, 512, 128, 300
    q = rnd(400 + B + T, (B, T, H, d), d ** -0.5, BF16)
    kv = rnd(401 + E, (B, E, d), d ** -0.5, BF16)
    kl = rnd(402 + B, (B, L, d), d ** -0.5, BF16)
    sink = rnd(403, (H,))
    g = torch.Generator().manual_seed(B * 1000 + T + E)
    top = m * E + 60
    q_pos = torch.randint(0, top, (B * T,), generator=g).to(torch.int64)
    # every entry visible, entries past E_cap, a token inside the first block (no entry, window
    # only), the last token of a block, and one short of it
    special = [m * E - 1, top - 1, 3, m * 7 - 1, m * 7 - 2]
    q_pos[:min(len(special), B * T)] = torch.tensor(special[:B * T])
    local_base = (q_pos.view(B, T)[:, 0] - 150).clamp(min=0).to(DEV)
    local_base[0] = max(int(q_pos[0]) - 40, 0)          # window clipped by the held rows
    q_pos = q_pos.to(DEV)   # (queries past local_base + L see only the held part of their window)
    c = hca_cfg(B=B, m=m)
    out = torch.empty(B, T, H, d, device=DEV, dtype=BF16)
    lse = torch.empty(B, T, H, device=DEV)
    csa.dense_attn(c, q, kv, kl, local_base, q_pos, sink, out, lse)
    check_dev_error()
    ro, rl = _dense_ref(q, kv, kl, local_base.cpu(), q_pos.cpu(), sink, m, W, d ** -0.5)
    w1 = assert_rows_close(np64(out), ro, 2e-2)
    np.testing.assert_allclose(np64(lse), rl, atol=5e-3, rtol=0)
    print(f"dense attention B={B} T={T} E={E}: worst/tol = {w1:.3f}")


def test_dense_attn_cuda_core_fp32():
    cfg = gen.CONFIGS[8]
    inp = gen.make_inputs(cfg, DEV)
    c = lib_config(cfg)
    csa.compress_kv_single(c, inp["kv_str"], inp["z_str"], inp["bias"], 0, 0, cfg.E, inp["kv_comp"])
    out = torch.empty(cfg.B, cfg.T, cfg.H, cfg.d, device=DEV)
    lse = torch.empty(cfg.B, cfg.T, cfg.H, device=DEV)
    csa.dense_attn(c, inp["q"], inp["kv_comp"], inp["kv_local"], inp["local_base"], inp["q_pos"], inp["sink"],
                   out, lse)
    check_dev_error()
    h = np_inputs(inp)
    kv = O.compress_single_range(h["kv_str"][0], h["z_str"][0], h["bias"], cfg.m, 0, cfg.E)
    assert_single_entries_close(np64(inp["kv_comp"][0]), kv, h["kv_str"], cfg.m, torch.float32)
    for tq in range(cfg.T):
        r = O.hca_token(cfg, h, 0, tq, kv)
        np.testing.assert_allclose(np64(out[0, tq]), r["out"], atol=1e-4, rtol=1e-4)
        np.testing.assert_allclose(np64(lse[0, tq]), r["lse"], atol=1e-5, rtol=1e-5)


# ------------------------------------------------------------------ HCA decode step

def oracle_hca_decode(cfg, inp):
    h = np_inputs(inp)
    res = []
    for b in range(cfg.B):
        kvc = h["kv_comp"][b].copy()
        r = O.hca_decode_step_sequence(cfg, h, b, kvc)
        r["kv_comp"] = kvc
        res.append(r)
    return res


def run_hca_decode(cfg, inp):
    c = lib_config(cfg)
    out = torch.empty(cfg.B, cfg.H, cfg.d, device=DEV, dtype=cfg.torch_act)
    lse = torch.empty(cfg.B, cfg.H, device=DEV)
    csa.hca_decode_step(c, q_pos=inp["q_pos"], q=inp["q"], sink=inp["sink"], kv_comp=inp["kv_comp"],
                        kv_tail=inp["kv_str"], z_tail=inp["z_str"], bias=inp["bias"], kv_local=inp["kv_local"],
                        local_base=inp["local_base"], out=out, lse=lse)
    check_dev_error()
    return out, lse


def assert_hca_decode_matches(cfg, inp, ref, out, lse, kv_before):
    for b in range(cfg.B):
        r = ref[b]
        assert_rows_close(np64(out[b]), r["out"], 2e-2, what=f"out b={b}")
        np.testing.assert_allclose(np64(lse[b]), r["lse"], atol=5e-3)
        if r["entry"] is None:
            assert torch.equal(inp["kv_comp"][b], kv_before[b])
        else:
            e, ent = r["entry"]
            assert_single_entries_close(np64(inp["kv_comp"][b, e]), ent, np64(inp["kv_str"][b]), cfg.m, cfg.torch_act)


@pytest.mark.parametrize("N", [128 * 300, 128 * 2, 128 * 5000])
def test_hca_decode_step_matches_oracle(N):
    cfg = gen.CONFIGS[6].replace(B=3, N=N)
    inp = gen.make_inputs(cfg, DEV)
    inp["q_pos"][1] = N - 2          # this token completes no block: no compression
    kv_before = inp["kv_comp"].clone()
    ref = oracle_hca_decode(cfg, inp)
    out, lse = run_hca_decode(cfg, inp)
    assert_hca_decode_matches(cfg, inp, ref, out, lse, kv_before)
