"""BF16 index scores before the top-k (V4 page, "FP4, down to the index scores": FP32 -> BF16
scores give the selector a two-times speedup at 99.7 % recall).  GPU required.

The indexer's BF16 scores are the round-to-nearest-even of the fp32 scores it computes
(bit-exact against the fp32 call); the selection over BF16 scores is bit-exact against the
oracle's top-k on the same BF16 values (many of them equal: ties go to the lowest position);
the decode step with BF16 scores selects exactly the top-k of the BF16 scores it wrote and
matches the oracle's outputs up to near-tie swaps.  The recall of the BF16 selection against
the fp32 one is printed.
"""
import numpy as np
import pytest
import torch

import compressed_sparse_attention_csa_gb300 as csa
from _helpers import (assert_decode_matches, assert_step_selection_exact, oracle_decode, run_gpu_decode)
from oracle import csa_oracle as O
from synth import gen

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


def cfg_obj(**kw):
    base = dict(B=2, H=64, d=512, HI=64, dI=128, m=4, k=512, W=128, act=BF16, fp8_keys=False, softmax_scale=None)
    base.update(kw)
    return csa.Config(**base)


def rnd(seed, shape, std=1.0, dtype=torch.float32):
    n = int(np.prod(shape))
    return gen.normal(seed, n, device=DEV, std=std).reshape(shape).to(dtype)


@pytest.mark.parametrize("rows,n,k,mode", [(8, 262144, 512, "normal"), (6, 200000, 512, "coarse"),
                                          (300, 5000, 512, "normal"), (64, 33792, 512, "coarse"),
                                          (50, 1000, 64, "normal"), (3, 100, 64, "normal"),
                                          (40, 9000, 2048, "coarse")])
def test_topk_bf16_exact(rows, n, k, mode):
    """csa_topk_bf16 (the histogram path for few long rows, the row kernel otherwise) against the
    oracle's top-k of the same BF16 values; -inf tails, -0, rows shorter than k."""
    x = rnd(100 + rows, (rows, n))
    if mode == "coarse":
        x = torch.round(x * 4) / 4                   # long runs of equal scores
    x[0, : n // 3] = float("-inf")
    x[1, 5::7] = -0.0
    s = x.to(BF16).contiguous()
    nv = torch.tensor([max(0, n - 977 * r) for r in range(rows)], dtype=torch.int32, device=DEV)
    idx = torch.full((rows, k), -7, dtype=torch.int32, device=DEV)
    csa.topk(cfg_obj(k=k), s, idx, n_valid=nv)
    assert csa.get_last_error() == 0
    sf, nvn, got = s.float().cpu().numpy(), nv.cpu().numpy(), idx.cpu().numpy()
    for r in list(range(min(rows, 6))) + [rows - 1]:
        np.testing.assert_array_equal(got[r], O.topk(sf[r], int(nvn[r]), k), err_msg=f"row {r}")


def test_topk_bf16_candidate_map():
    """A candidate map (ascending positions, -1 padded): idx holds the winners' positions."""
    rows, n, k = 70, 6000, 256
    x = rnd(7, (rows, n)).to(BF16).contiguous()
    g = torch.Generator().manual_seed(3)
    cand = torch.sort(torch.randint(0, 1 << 20, (rows, n), generator=g), dim=1).values.to(torch.int32)
    cand[:, n - 500:] = -1
    idx = torch.empty(rows, k, dtype=torch.int32, device=DEV)
    csa.topk(cfg_obj(k=k), x, idx, cand=cand.to(DEV))
    assert csa.get_last_error() == 0
    xf, cn, got = x.float().cpu().numpy(), cand.numpy(), idx.cpu().numpy()
    for r in [0, 1, rows - 1]:
        sel = O.topk(xf[r], n - 500, k)
        np.testing.assert_array_equal(got[r], np.where(sel >= 0, cn[r][np.maximum(sel, 0)], -1))


@pytest.mark.parametrize("HI,T,fp8", [(64, 1, False), (64, 700, False), (64, 1, True), (32, 9, False)])
def test_indexer_scores_bf16_is_rounded_fp32(HI, T, fp8):
    B, dI, m, E = 3, 128, 4, 128 * 9 + 37
    qI = rnd(21 + HI + T, (B, T, HI, dI), dI ** -0.5, BF16)
    w = rnd(22 + T, (B, T, HI))
    kf = rnd(23, (B, E, dI), dI ** -0.5)
    kI, ks = gen.quantize_keys_e4m3(kf) if fp8 else (kf.to(BF16), None)
    g = torch.Generator().manual_seed(T)
    q_pos = torch.randint(0, m * E + 40, (B * T,), generator=g).to(torch.int64).to(DEV)
    c = cfg_obj(B=B, HI=HI, m=m, fp8_keys=fp8)
    s32 = torch.empty(B * T, E, device=DEV)
    s16 = torch.empty(B * T, E, device=DEV, dtype=BF16)
    csa.indexer_scores(c, qI, w, q_pos, kI, s32, kscale=ks)
    csa.indexer_scores(c, qI, w, q_pos, kI, s16, kscale=ks)
    assert csa.get_last_error() == 0
    assert torch.equal(s16.view(torch.int16), s32.to(BF16).view(torch.int16))


@pytest.mark.parametrize("T", [700, 5])
def test_indexer_topk_bf16(T):
    """csa_indexer_topk_bf16 equals csa_topk_bf16 on the scores csa_indexer_scores_bf16 writes;
    the recall of the BF16 selection against the fp32 one is printed."""
    B, HI, m, E, k = 2, 64, 4, 128 * 60 + 37, 512
    qI = rnd(41, (B, T, HI, 128), 128 ** -0.5, BF16)
    w = rnd(42, (B, T, HI))
    kI = rnd(43, (B, E, 128), 128 ** -0.5).to(BF16)
    g = torch.Generator().manual_seed(T)
    q_pos = torch.randint(m * 1000, m * E + 40, (B * T,), generator=g).to(torch.int64)
    q_pos[:2] = torch.tensor([3, m * E - 1])
    q_pos = q_pos.to(DEV)
    c = cfg_obj(B=B, HI=HI, m=m, k=k)
    idx16 = torch.full((B * T, k), -7, dtype=torch.int32, device=DEV)
    csa.indexer_topk(c, qI, w, q_pos, kI, idx16, bf16_scores=True)
    s16 = torch.empty(B * T, E, device=DEV, dtype=BF16)
    csa.indexer_scores(c, qI, w, q_pos, kI, s16)
    nv = ((q_pos + 1) // m).clamp(max=E).to(torch.int32)
    ref = torch.empty(B * T, k, dtype=torch.int32, device=DEV)
    csa.topk(c, s16, ref, n_valid=nv)
    idx32 = torch.empty(B * T, k, dtype=torch.int32, device=DEV)
    csa.indexer_topk(c, qI, w, q_pos, kI, idx32)
    assert csa.get_last_error() == 0
    assert torch.equal(idx16, ref)
    sf, nvn = s16.float().cpu().numpy(), nv.cpu().numpy()
    for r in [0, 1, 2, B * T - 1]:
        np.testing.assert_array_equal(idx16[r].cpu().numpy(), O.topk(sf[r], int(nvn[r]), k))
    a16, a32 = idx16.cpu().numpy(), idx32.cpu().numpy()
    hits = sum(len(set(a16[r][a16[r] >= 0]) & set(a32[r][a32[r] >= 0])) for r in range(B * T))
    total = sum(int((a32[r] >= 0).sum()) for r in range(B * T))
    print(f"BF16 selection recall vs fp32: {hits / max(total, 1):.4f} over {B * T} rows")
    assert hits / max(total, 1) > 0.9


@pytest.mark.parametrize("cid,B,N", [(2, 4, 4 * 3000), (4, 2, 4 * 5000 + 1), (13, 3, 4 * 2400)])
def test_decode_step_bf16_scores(cid, B, N):
    cfg = gen.CONFIGS[cid].replace(B=B, N=N)
    inp = gen.make_inputs(cfg, DEV)
    ref = oracle_decode(cfg, inp)
    scores = torch.empty(cfg.B, cfg.E, device=DEV, dtype=BF16)
    out, lse, idx = run_gpu_decode(cfg, inp, scores_out=scores, bf16_scores=True)
    assert_decode_matches(cfg, inp, ref, out, lse, idx)
    assert_step_selection_exact(cfg, ref, idx, scores)
