"""Shared pieces of the GPU parity tests: preset -> library config, tensor -> float64 numpy,
the oracle's dequantisation of stored keys, and the per-stage agreement checks."""
import numpy as np
import torch

import compressed_sparse_attention_csa_gb300 as csa
from compressed_sparse_attention_csa_gb300 import Config
from oracle import csa_oracle as O


def lib_config(cfg, **kw) -> Config:
    c = Config(B=cfg.B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
               act=cfg.torch_act, fp8_keys=(cfg.kidx == "fp8"), softmax_scale=cfg.softmax_scale,
               mx_keys=(cfg.kidx == "mxfp4"))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def np64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of an fp32 / bf16 tensor to float64 numpy on the host."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def keys_f64(kI: torch.Tensor, kscale=None) -> np.ndarray:
    """Dequantised indexer keys as the oracle reads them (MXFP4: uint8 payload [.., dI/2] with
    int32 scale words)."""
    if kI.dtype == torch.uint8 and kscale is not None and kscale.dtype == torch.int32:
        words = kscale.cpu().numpy().view(np.uint32)
        return O.mxfp4_key_decode(kI.cpu().numpy(), O.mxfp4_key_unwords(words))
    if kI.dtype == torch.uint8:
        return O.e4m3_decode(kI.cpu().numpy()) * kscale.cpu().numpy().astype(np.float64)[..., None]
    return np64(kI)


def assert_scores_close(got: np.ndarray, ref: np.ndarray, rtol: float, what: str = "scores"):
    """|g - r| <= rtol * max(|r|, rms of the row's finite reference values); -inf must match."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    inf_r = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_r), f"{what}: -inf pattern differs"
    fin = ~inf_r
    rr = np.where(fin, ref, 0.0)
    rms = np.sqrt((rr ** 2).sum(-1, keepdims=True) / np.maximum(fin.sum(-1, keepdims=True), 1))
    tol = rtol * np.maximum(np.abs(rr), rms) + 1e-30
    err = np.where(fin, np.abs(np.where(fin, got, 0.0) - rr), 0.0)
    worst = float((err / tol).max()) if err.size else 0.0
    assert worst <= 1.0, f"{what}: worst error is {worst:.3f} x tolerance"
    return worst


def assert_rows_close(got: np.ndarray, ref: np.ndarray, rtol: float, atol: float = 0.0, what: str = "out"):
    """Per output row (last axis): |g - r| <= rtol * max|r_row| + atol."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    tol = rtol * scale + atol
    worst = float((np.abs(got - ref) / np.maximum(tol, 1e-300)).max())
    assert worst <= 1.0, f"{what}: worst error is {worst:.3f} x tolerance"
    return worst


def swap_bound(q, lse, scale, rows_in, rows_out):
    """First-order change of the attention output when rows_out leave the selection and rows_in
    join it: sum over those rows of weight_h(row) * |row|, with weight_h = exp(scale q_h.r - lse_h)."""
    q = np.asarray(q, np.float64)
    bound = np.zeros_like(q)
    for r in list(rows_in) + list(rows_out):
        r = np.asarray(r, np.float64)
        w = np.exp(scale * (q @ r) - lse)            # [H]
        bound += w[:, None] * np.abs(r)[None, :]
    return bound


def assert_out_close_with_swaps(got, ref, rtol, bound, what="out"):
    """|g - r| <= rtol * max|r_row| + 1.5 * (swap bound); the bound is 0 without swaps."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = rtol * np.abs(ref).max(axis=-1, keepdims=True) + 1.5 * bound
    worst = float((np.abs(got - ref) / np.maximum(tol, 1e-300)).max())
    assert worst <= 1.0, f"{what}: worst error is {worst:.3f} x tolerance"
    return worst


def assert_selection_ok(got_idx, ref_idx, ref_scores: np.ndarray, k: int, score_tol: float):
    """The selections agree except for swaps at near-ties: every entry only one side kept has an
    oracle score within score_tol of the oracle's k-th score."""
    g = set(int(x) for x in got_idx if x >= 0)
    r = set(int(x) for x in ref_idx if x >= 0)
    assert len(g) == len(r), (len(g), len(r))
    assert sorted(int(x) for x in got_idx if x >= 0) == [int(x) for x in got_idx if x >= 0], "not ascending"
    if g == r:
        return 0
    vals = np.array([ref_scores[i] for i in r])
    kth = vals.min()
    for x in g - r:
        assert ref_scores[x] >= kth - score_tol, ("swap far from the threshold", x, ref_scores[x], kth)
    for y in r - g:
        assert ref_scores[y] <= kth + score_tol, ("swap far from the threshold", y, ref_scores[y], kth)
    return len(g - r)


def np_inputs(inp):
    out = {}
    for k_, v in inp.items():
        if v.dtype in (torch.float32, torch.bfloat16):
            out[k_] = np64(v)
        else:
            out[k_] = v.cpu().numpy()
    return out


def oracle_decode(cfg, inp):
    """The oracle's decode step for every sequence of the batch."""
    nb = np_inputs(inp)
    fp8 = cfg.kidx == "fp8"
    mx = cfg.kidx == "mxfp4"
    res = []
    for b in range(cfg.B):
        kdeq = keys_f64(inp["kI"][b], inp["kscale"][b] if (fp8 or mx) else None)
        kvc = nb["kv_comp"][b].copy()
        r = O.decode_step_sequence(cfg, nb, b, kvc, kdeq, fp8_keys=fp8, mx_keys=mx)
        r["kv_comp"] = kvc
        r["q"] = nb["q"][b, 0]
        res.append(r)
    return res


def run_gpu_decode(cfg, inp, scores_out=None, bf16_scores=False):
    c = lib_config(cfg)
    out = torch.empty(cfg.B, cfg.H, cfg.d, device=inp["q"].device, dtype=cfg.torch_act)
    lse = torch.empty(cfg.B, cfg.H, device=inp["q"].device)
    idx = torch.empty(cfg.B, cfg.k, dtype=torch.int32, device=inp["q"].device)
    csa.decode_step(c, q_pos=inp["q_pos"], q=inp["q"], qI=inp["qI"], w=inp["w"], sink=inp["sink"],
                    kv_comp=inp["kv_comp"], kI=inp["kI"], kscale=inp.get("kscale"), kv_tail=inp["kv_str"],
                    z_tail=inp["z_str"], kvI_tail=inp["kvI_str"], zI_tail=inp["zI_str"], bias=inp["bias"],
                    biasI=inp["biasI"], kv_local=inp["kv_local"], local_base=inp["local_base"], out=out, lse=lse,
                    idx_out=idx, scores_out=scores_out, bf16_scores=bf16_scores)
    assert csa.get_last_error() == 0
    return out, lse, idx


def assert_step_selection_exact(cfg, ref, idx, scores_out):
    """The decode step's selection is exactly the top-k (score desc, position asc; ascending,
    -1 padded) of the fp32 scores it wrote, and those scores match the oracle's within the
    indexer tolerance, -inf past the visible entries."""
    rtol_s = 5e-2 if cfg.kidx in ("fp8", "mxfp4") else 1e-2
    for b in range(cfg.B):
        nv = ref[b]["nv"]
        s32 = scores_out[b].float().cpu().numpy()
        assert np.all(np.isneginf(s32[nv:])), f"b={b}: invisible entries must be -inf"
        assert_scores_close(s32[:nv], ref[b]["scores"][:nv], rtol_s, what=f"step scores b={b}")
        gi = idx[b].cpu().numpy().astype(np.int64)
        np.testing.assert_array_equal(gi, O.topk(s32, nv, cfg.k), err_msg=f"b={b}: selection differs from the top-k")


def assert_decode_matches(cfg, inp, ref, out, lse, idx):
    """Decode-step agreement per sequence: selection valid up to score-tolerance swaps, output
    within 2e-2 of the row maximum plus the swaps' first-order effect, LSE within 5e-3, and
    the compressed entry (when the token completed a block) within bf16 rounding."""
    rtol_s = 5e-2 if cfg.kidx in ("fp8", "mxfp4") else 1e-2
    for b in range(cfg.B):
        r = ref[b]
        fin = r["scores"][np.isfinite(r["scores"])]
        tol = rtol_s * max(np.sqrt((fin ** 2).mean()), 1e-30)
        gi = idx[b].cpu().numpy()
        swaps = assert_selection_ok(gi, r["idx"], r["scores"], cfg.k, tol)
        g_set, r_set = set(gi[gi >= 0].tolist()), set(r["idx"][r["idx"] >= 0].tolist())
        bound = swap_bound(r["q"], r["lse"], cfg.softmax_scale, [r["kv_comp"][x] for x in g_set - r_set],
                           [r["kv_comp"][y] for y in r_set - g_set])
        assert_out_close_with_swaps(np64(out[b]), r["out"], 2e-2, bound, what=f"out b={b} swaps={swaps}")
        np.testing.assert_allclose(np64(lse[b]), r["lse"], atol=5e-3)
        if r["entry"] is not None:
            e, _, _, ent_exact, _ = r["entry"]
            assert_entries_close(np64(inp["kv_comp"][b, e]), ent_exact, np64(inp["kv_str"][b]))


def assert_pool_valid(gpool, ref_scores_f32, nv: int, block: int, n_blocks: int, score_tol: float):
    """A block pool computed from scores that differ from the oracle's within score_tol is one
    of the correct pools: it keeps as many blocks as the oracle's pool; a block only one side
    kept has an oracle block maximum within score_tol of the oracle's last kept block maximum;
    the kept blocks expand to their visible positions in ascending order."""
    gpool = np.asarray(gpool, np.int64)
    nb = -(-nv // block)
    vals = np.asarray(ref_scores_f32[:nv], np.float64)
    pad = np.full(nb * block, -np.inf)
    pad[:nv] = vals
    bmax = pad.reshape(nb, block).max(axis=1)
    ref_pool = O.hier_pool(ref_scores_f32, nv, block, n_blocks)
    r_blocks = set((ref_pool // block).tolist())
    g_blocks = sorted(set((gpool // block).tolist()))
    assert len(g_blocks) == len(r_blocks), (len(g_blocks), len(r_blocks))
    expect = np.asarray([p for j in g_blocks for p in range(j * block, min((j + 1) * block, nv))], np.int64)
    assert np.array_equal(gpool, expect), "pool is not the ascending expansion of its blocks"
    thr = bmax[sorted(r_blocks)].min()
    for j in set(g_blocks) - r_blocks:
        assert bmax[j] >= thr - score_tol, ("pool block far from the threshold", j, bmax[j], thr)
    for j in r_blocks - set(g_blocks):
        assert bmax[j] <= thr + score_tol, ("pool block far from the threshold", j, bmax[j], thr)
    return len(set(g_blocks) - r_blocks)


def assert_entries_close(got, ref, streams):
    """Compressed entries stored in bf16 after fp32 arithmetic: the bf16 rounding (at most half
    an ulp, 2^-8 relative) plus the fp32 error of the 2m-term weighted sum, bounded by
    2^-18 of the largest stream value (a 4x margin over 2m * 2^-23)."""
    atol = 2.0 ** -18 * float(np.abs(streams).max())
    err = np.abs(np.asarray(got, np.float64) - ref)
    tol = 2.0 ** -8 * np.abs(ref) + atol
    worst = float((err / tol).max())
    assert worst <= 1.0, f"compressed entries: worst error is {worst:.3f} x tolerance"
    return worst
