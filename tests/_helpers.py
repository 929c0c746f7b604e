"""Shared pieces of the GPU parity tests: preset -> library config, tensor -> float64 numpy,
the oracle's dequantisation of stored keys, and the per-stage agreement checks."""
import numpy as np
import torch

from compressed_sparse_attention_csa_gb300 import Config
from oracle import csa_oracle as O


def lib_config(cfg, **kw) -> Config:
    c = Config(B=cfg.B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
               act=cfg.torch_act, fp8_keys=(cfg.kidx == "fp8"), softmax_scale=cfg.softmax_scale)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def np64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of an fp32 / bf16 tensor to float64 numpy on the host."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def keys_f64(kI: torch.Tensor, kscale=None) -> np.ndarray:
    """Dequantised indexer keys as the oracle reads them."""
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
