"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one oracle function to a hand-computed example, a closed form, a
library routine on a special case, or an invariant stated by the CSA pages, chosen so
that a dropped term, a swapped stream, a wrong index or a transposed operand fails.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ------------------------------------------------------------------ formats

def test_bf16_roundtrip_matches_torch():
    x = rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 20000)
    ours = O.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = O.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy())


def test_e4m3_decode_spec_points():
    # OCP FP8 E4M3: bias 7, max normal S.1111.110 = 448, min subnormal 2^-9, 0x7F NaN
    assert O.e4m3_decode(np.array([0x7E], np.uint8))[0] == 448.0
    assert O.e4m3_decode(np.array([0x01], np.uint8))[0] == 2.0 ** -9
    assert O.e4m3_decode(np.array([0x08], np.uint8))[0] == 2.0 ** -6
    assert O.e4m3_decode(np.array([0x38], np.uint8))[0] == 1.0
    assert O.e4m3_decode(np.array([0xB8], np.uint8))[0] == -1.0
    assert np.isnan(O.e4m3_decode(np.array([0x7F], np.uint8))[0])


def test_e4m3_tables_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.e4m3_decode(codes)
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), ~fin)
    assert np.array_equal(ours[fin], ref[fin])
    x = (rng.standard_normal(50000) * 60).astype(np.float32)
    x = np.clip(x, -448, 448)
    enc = O.e4m3_encode(x)
    ref_enc = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # -0 and +0 are the same value; compare decoded values
    assert np.array_equal(O.e4m3_decode(enc), O.e4m3_decode(ref_enc))


def test_quantize_rows_e4m3_roundtrip_bound():
    x = rng.standard_normal((64, 128)).astype(np.float32)
    codes, scale = O.quantize_rows_e4m3(x)
    back = O.e4m3_decode(codes) * scale[:, None]
    # relative error of a normal e4m3 value is at most 2^-4; subnormals: 2^-10 * scale
    err = np.abs(back - x)
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale[:, None]) + 1e-12)
    assert np.all(np.max(np.abs(back), axis=1) == pytest.approx(np.max(np.abs(x), axis=1), rel=1e-6))



def test_quantize_rows_e4m3_divisor_is_448():
    # a row whose amax is 56 = 448 / 8: the scale is exactly 1/8 and the amax lands on e4m3's
    # largest normal code 0x7E (= 448); -1.5 -> -12 and 0.7 -> 5.6 -> nearest 5.5 (step 0.5)
    x = np.array([[56.0, -1.5, 3.0, 0.7]], np.float32)
    codes, scale = O.quantize_rows_e4m3(x)
    assert scale[0] == np.float32(0.125)
    assert codes[0, 0] == 0x7E
    np.testing.assert_array_equal(O.e4m3_decode(codes[0]) * float(scale[0]), [56.0, -1.5, 3.0, 0.6875])


def test_round_to_bf16_single_rounding():
    # binary32 inputs: the same as the (torch-pinned) binary32 -> bf16 conversion
    x = (rng.standard_normal(5000) * 10.0 ** rng.integers(-3, 3, 5000)).astype(np.float32)
    np.testing.assert_array_equal(O.round_to_bf16(x.astype(np.float64)), O.bf16_bits_to_f64(O.f32_to_bf16_bits(x)))
    # exact halfway points go to the even neighbour; a float64 value just above a halfway point
    # rounds up (rounding through binary32 first would land on the halfway point and go down)
    assert O.round_to_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert O.round_to_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6
    assert O.round_to_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -30]))[0] == 1.0 + 2.0 ** -7
    assert O.round_to_bf16(np.array([-3.0]))[0] == -3.0 and O.round_to_bf16(np.array([0.0]))[0] == 0.0
    assert O.round_to_store(np.array([0.1]), "f32")[0] == float(np.float32(0.1))


# ------------------------------------------------------------------ compressor

def _load_compress_golden():
    rows = {}
    with open(os.path.join(GOLDEN, "compress_m4_two_entries.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            if key.startswith("expect"):
                rows[key] = [Fraction(v) for v in rest.split()]
            else:
                rows[key] = np.array([[float(v) for v in g.split()] for g in rest.split("|")])
    return rows


def test_compress_hand_example():
    g = _load_compress_golden()
    n = g["Ca"].shape[0]
    kv = np.stack([g["Ca"], g["Cb"]], axis=1)                   # [8, 2, 2]
    z = np.log(np.stack([g["expZa"], g["expZb"]], axis=1))
    bias = np.log(np.stack([g["expBa"], g["expBb"]], axis=0))   # [2, 4, 2]
    e0 = O.compress_entry(kv, z, bias, 4, 0)
    e1 = O.compress_entry(kv, z, bias, 4, 1)
    assert n == 8
    np.testing.assert_allclose(e0, [float(v) for v in g["expect_entry0"]], rtol=1e-13)
    np.testing.assert_allclose(e1, [float(v) for v in g["expect_entry1"]], rtol=1e-13)


def _rand_streams(n_tok, dim, m, scale=1.0):
    kv = rng.standard_normal((n_tok, 2, dim))
    z = rng.standard_normal((n_tok, 2, dim)) * scale
    bias = rng.standard_normal((2, m, dim)) * 0.1
    return kv, z, bias


def test_compress_constant_gate_is_mean():
    m, dim = 4, 5
    kv, _, _ = _rand_streams(16, dim, m)
    z = np.full((16, 2, dim), 0.7)
    bias = np.zeros((2, m, dim))
    e0 = O.compress_entry(kv, z, bias, m, 0)
    np.testing.assert_allclose(e0, kv[0:4, 0].mean(axis=0), rtol=1e-12)
    e2 = O.compress_entry(kv, z, bias, m, 2)
    np.testing.assert_allclose(e2, (kv[8:12, 0].sum(0) + kv[4:8, 1].sum(0)) / 8, rtol=1e-12)


def test_compress_dominant_logit_copies_token():
    m, dim = 4, 3
    kv, z, bias = _rand_streams(12, dim, m)
    z[5, 1, :] = 800.0          # token 5 in stream b; it belongs to block 1 -> entry 2
    e2 = O.compress_entry(kv, z, bias, m, 2)
    np.testing.assert_allclose(e2, kv[5, 1], rtol=1e-12)
    e1 = O.compress_entry(kv, z, bias, m, 1)
    assert not np.allclose(e1, kv[5, 1])


def test_compress_weights_positive_sum_to_one():
    m, dim = 4, 7
    kv, z, bias = _rand_streams(20, dim, m, scale=3.0)
    for i in range(5):
        _, w = O.compress_entry(kv, z, bias, m, i, return_weights=True)
        assert w.shape[0] == (m if i == 0 else 2 * m)
        assert np.all(w > 0)
        np.testing.assert_allclose(w.sum(axis=0), 1.0, rtol=1e-13)


def test_compress_each_token_in_two_entries_and_causal():
    m, dim, n = 4, 3, 24
    kv, z, bias = _rand_streams(n, dim, m)
    base = O.compress_range(kv, z, bias, m, 0, n // m)
    for t in range(n):
        kv2 = kv.copy()
        kv2[t, :, :] += 1.0
        changed = np.where(np.any(O.compress_range(kv2, z, bias, m, 0, n // m) != base, axis=1))[0]
        expect = [i for i in (t // m, t // m + 1) if i < n // m]
        assert list(changed) == expect, (t, changed)
        # causality: entry i uses no token >= m*(i+1)
        assert all(t < m * (i + 1) for i in changed)
    # every token t >= m (with a following block) appears in exactly two entries
    for t in range(m, n - m):
        assert len([i for i in (t // m, t // m + 1)]) == 2


def test_compress_tok0_offset_equivalent():
    m, dim = 4, 4
    kv, z, bias = _rand_streams(32, dim, m)
    full = O.compress_range(kv, z, bias, m, 3, 8)
    part = O.compress_range(kv[8:], z[8:], bias, m, 3, 8, tok0=8)
    np.testing.assert_array_equal(full, part)
    with pytest.raises(ValueError):
        O.compress_entry(kv[8:], z[8:], bias, m, 2, tok0=8)


# ------------------------------------------------------------------ indexer

def test_indexer_one_hot_closed_form():
    # q_h = a_h e_{c_h}, k_s = e_{c}: score_s = sum_h w_h relu(a_h) [c_h == c_s]
    HI, dI, E = 5, 6, 6
    a = np.array([1.5, -2.0, 0.5, 3.0, -1.0])
    ch = np.array([0, 0, 3, 5, 5])
    qI = np.zeros((HI, dI))
    qI[np.arange(HI), ch] = a
    w = np.array([2.0, 7.0, -1.0, 0.25, 4.0])
    kI = np.eye(dI)[:E]
    s = O.indexer_scores(qI, w, kI, nv=E)
    expect = np.zeros(E)
    expect[0] = 2.0 * 1.5          # head 1 (a=-2) vetoed by ReLU
    expect[3] = -1.0 * 0.5
    expect[5] = 0.25 * 3.0          # head 4 (a=-1) vetoed
    np.testing.assert_array_equal(s, expect)


def test_indexer_single_head_is_matvec_and_causal_mask():
    dI, E = 16, 40
    q = np.abs(rng.standard_normal((1, dI)))
    kI = np.abs(rng.standard_normal((E, dI)))       # all dots positive: ReLU inactive
    s = O.indexer_scores(q, np.array([1.0]), kI, nv=25)
    np.testing.assert_allclose(s[:25], np.dot(kI[:25], q[0]), rtol=1e-14)
    assert np.all(np.isneginf(s[25:]))


def test_indexer_relu_veto_and_w_linearity():
    HI, dI, E = 4, 8, 30
    qI = rng.standard_normal((HI, dI))
    kI = rng.standard_normal((E, dI))
    w = rng.standard_normal(HI)
    s = O.indexer_scores(qI, w, kI, E)
    np.testing.assert_allclose(O.indexer_scores(qI, 3.5 * w, kI, E), 3.5 * s, rtol=1e-13)
    # a key anti-aligned with every head scores exactly 0
    kneg = -np.abs(rng.standard_normal(dI))
    qpos = np.abs(rng.standard_normal((HI, dI)))
    s2 = O.indexer_scores(qpos, w, kneg[None, :], 1)
    assert s2[0] == 0.0
    # brute force over heads with explicit loops
    brute = np.array([sum(w[h] * max(0.0, sum(qI[h, c] * kI[s_, c] for c in range(dI)))
                          for h in range(HI)) for s_ in range(E)])
    np.testing.assert_allclose(s, brute, rtol=1e-12, atol=1e-15)


def test_indexer_fp8_scale_one_equals_exact_path():
    HI, dI, E = 4, 16, 20
    codes = rng.integers(0, 0x7E, (E, dI)).astype(np.uint8) | (rng.integers(0, 2, (E, dI)) * 0x80).astype(np.uint8)
    kdeq = O.e4m3_decode(codes) * 1.0
    qI = rng.standard_normal((HI, dI))
    w = rng.standard_normal(HI)
    s_fp8 = O.indexer_scores(qI, w, kdeq, E)
    s_f64 = O.indexer_scores(qI, w, O.e4m3_decode(codes), E)
    np.testing.assert_array_equal(s_fp8, s_f64)


def test_indexer_mac_count_matches_pages():
    vals = {}
    with open(os.path.join(GOLDEN, "indexer_mac_counts.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    from compressed_sparse_attention_csa_gb300.accounting import indexer_macs
    assert indexer_macs(vals["heads"], vals["dim"], vals["positions_full"]) == vals["macs_full"]
    assert indexer_macs(vals["heads"], vals["dim"], vals["pool_blocks"] * vals["pool_block"]) == vals["macs_pool"]



def test_indexer_scores_subset_brute_force():
    HI, dI, E = 3, 5, 40
    qI = rng.standard_normal((HI, dI))
    kI = rng.standard_normal((E, dI))
    w = rng.standard_normal(HI)
    pos = np.array([0, 7, 8, 31, 39, 7])             # any order, repeats allowed
    got = O.indexer_scores_subset(qI, w, kI, pos)
    brute = [sum(w[h] * max(0.0, math.fsum(qI[h, c] * kI[p, c] for c in range(dI))) for h in range(HI)) for p in pos]
    np.testing.assert_allclose(got, brute, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(got, O.indexer_scores(qI, w, kI, E)[pos], rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------------ top-k

def test_topk_brute_force_sort():
    for trial in range(50):
        n = int(rng.integers(1, 300))
        k = int(rng.integers(1, 80))
        nv = int(rng.integers(0, n + 1))
        s = rng.standard_normal(n).astype(np.float32)
        s[rng.random(n) < 0.2] = 0.0
        got = O.topk(s, nv, k)
        # brute force: python sort of (score, index) pairs
        pairs = sorted(((-float(s[i]), i) for i in range(nv)))
        expect = sorted(i for _, i in pairs[:min(k, nv)])
        assert list(got[:len(expect)]) == expect
        assert np.all(got[len(expect):] == -1)
        assert (got >= 0).sum() == min(k, nv)


def test_topk_adversarial_ties():
    k = 16
    assert list(O.topk(np.zeros(100, np.float32), 100, k)) == list(range(k))
    assert list(O.topk(np.full(100, 2.5, np.float32), 100, k)) == list(range(k))
    mix = np.where(np.arange(100) % 2 == 0, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
    assert list(O.topk(mix, 100, k)) == list(range(k))        # -0 == +0
    inc = np.arange(100, dtype=np.float32)
    assert list(O.topk(inc, 100, k)) == list(range(100 - k, 100))
    assert list(O.topk(inc, 5, k)) == list(range(5)) + [-1] * (k - 5)


def test_topk_bf16_ties_and_brute_force():
    # 1 + 2^-10 is above 1 in binary32 but rounds to 1 in BF16: the two tie, the lower index wins
    s = np.array([1.0, 1.0 + 2.0 ** -10, 0.5, -0.0], np.float32)
    assert list(O.topk(s, 4, 1)) == [1]
    assert list(O.topk_bf16(s, 4, 1)) == [0]
    # 1 + 2^-8 + 2^-9 and 1 + 3 * 2^-9 both round to 1 + 2^-7; 1 + 2^-8 (half an ulp) ties to even, 1
    t = np.array([1.0 + 2.0 ** -8 + 2.0 ** -9, 1.0 + 3 * 2.0 ** -9, 1.0 + 2.0 ** -8], np.float32)
    assert list(O.topk_bf16(t, 3, 1)) == [0]          # both round to 1 + 2^-7: index 0 first
    assert list(O.topk_bf16(np.array([0.0, -0.0, 0.0], np.float32), 3, 2)) == [0, 1]
    inf = np.array([-np.inf, 1.0, -np.inf], np.float32)
    assert list(O.topk_bf16(inf, 3, 3)) == [0, 1, 2]
    # brute force: sort (bf16 value via torch, index) pairs
    for trial in range(30):
        n = int(rng.integers(1, 400))
        k = int(rng.integers(1, 90))
        nv = int(rng.integers(0, n + 1))
        x = (rng.standard_normal(n) * 3).astype(np.float32)
        b = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
        pairs = sorted(((-float(b[i]), i) for i in range(nv)))
        expect = sorted(i for _, i in pairs[:min(k, nv)])
        got = O.topk_bf16(x, nv, k)
        assert list(got[:len(expect)]) == expect and np.all(got[len(expect):] == -1)


# ------------------------------------------------------------------ hierarchical pool

def test_hier_pool_superset_of_topk_and_size():
    for trial in range(20):
        nv = int(rng.integers(1, 5000))
        s = rng.standard_normal(nv + 37).astype(np.float32)
        block, nblk, k = 8, int(rng.integers(1, 200)), int(rng.integers(1, 64))
        k = min(k, nblk)   # a block holding a top-k position has max >= k-th score
        pool = O.hier_pool(s, nv, block, nblk)
        nb = -(-nv // block)
        kept = min(nblk, nb)
        # size: kept blocks x 8, minus the invisible tail of the last block if it is kept
        last_kept = (nb - 1) in set(pool // block)
        assert pool.size == kept * block - (nb * block - nv if last_kept else 0)
        assert np.all(np.diff(pool) > 0) and pool.max() < nv
        full = O.topk(s, nv, k)
        sub_slots = O.topk(s[pool], pool.size, k)
        sub = np.where(sub_slots >= 0, pool[np.maximum(sub_slots, 0)], -1)
        assert np.array_equal(full, sub)


def test_hier_pool_block_max_ranking():
    s = np.zeros(64, np.float32)
    s[13] = 5.0     # block 1
    s[40] = 4.0     # block 5
    s[63] = 3.0     # block 7
    pool = O.hier_pool(s, 64, 8, 2)
    assert list(pool) == list(range(8, 16)) + list(range(40, 48))
    pool = O.hier_pool(s, 60, 8, 3)   # position 63 invisible; block 7 covers 56..59
    assert list(pool) == list(range(0, 16)) + list(range(40, 48))


# ------------------------------------------------------------------ attention

def _sdpa_with_sink(q, rows, sink, scale):
    """torch's scaled_dot_product_attention, sink as an extra key of value zero."""
    H, d = q.shape
    n = rows.shape[0]
    K = torch.from_numpy(np.concatenate([rows, np.zeros((1, d))]))[None, None]
    V = K.clone()
    Q = torch.from_numpy(q)[None, :, None, :].transpose(0, 1)    # [H,1,1,d]
    mask = torch.zeros(H, 1, 1, n + 1, dtype=torch.float64)
    mask[:, 0, 0, n] = torch.from_numpy(np.asarray(sink, np.float64))
    out = torch.nn.functional.scaled_dot_product_attention(
        Q, K.expand(H, 1, n + 1, d), V.expand(H, 1, n + 1, d), attn_mask=mask, scale=scale)
    return out[:, 0, 0, :].numpy()


def test_attention_matches_sdpa_with_sink_column():
    H, d, n = 6, 16, 37
    q = rng.standard_normal((H, d))
    rows = rng.standard_normal((n, d))
    sink = rng.standard_normal(H)
    out, lse = O.sparse_attention(q, rows, sink, 1 / math.sqrt(d))
    np.testing.assert_allclose(out, _sdpa_with_sink(q, rows, sink, 1 / math.sqrt(d)), rtol=1e-12, atol=1e-14)
    lg = q @ rows.T / math.sqrt(d)
    np.testing.assert_allclose(lse, np.log(np.exp(lg).sum(1) + np.exp(sink)), rtol=1e-13)


def test_attention_sink_limits():
    H, d, n = 4, 8, 20
    q = rng.standard_normal((H, d))
    rows = rng.standard_normal((n, d))
    # sink -> -inf: plain softmax attention (SDPA without the extra column)
    out, _ = O.sparse_attention(q, rows, np.full(H, -np.inf), 0.3)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, None, :], torch.from_numpy(rows)[None, None].expand(H, 1, n, d),
        torch.from_numpy(rows)[None, None].expand(H, 1, n, d), scale=0.3)[:, 0, 0]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12)
    # a large sink drives the output to 0 (the head abstains)
    out, _ = O.sparse_attention(q, rows, np.full(H, 60.0), 0.3)
    assert np.max(np.abs(out)) < 1e-20
    # equal rows r: out = r * (1 - sink mass)
    r = rng.standard_normal(d)
    eq = np.tile(r, (n, 1))
    sink = rng.standard_normal(H)
    out, _ = O.sparse_attention(q, eq, sink, 0.3)
    lg = 0.3 * q @ r
    mass = np.exp(sink) / (n * np.exp(lg) + np.exp(sink))
    np.testing.assert_allclose(out, (1 - mass)[:, None] * r[None, :], rtol=1e-12)


def test_attention_dense_reduction():
    # k = all entries, window empty: dense MQA attention over the compressed cache
    H, d, E = 4, 8, 24
    q = rng.standard_normal((H, d))
    kv = rng.standard_normal((E, d))
    idx = O.topk(rng.standard_normal(E).astype(np.float32), E, E)
    rows = O.gather_rows(kv, idx, np.zeros((1, d)), local_base=10 ** 9, t=100, W=0)
    np.testing.assert_array_equal(rows, kv)
    sink = rng.standard_normal(H)
    out, _ = O.sparse_attention(q, rows, sink, 0.25)
    np.testing.assert_allclose(out, _sdpa_with_sink(q, kv, sink, 0.25), rtol=1e-12)


def test_window_positions():
    assert O.window_positions(t=10, W=4, local_base=0, n_local=100) == [7, 8, 9, 10]
    assert O.window_positions(t=2, W=4, local_base=0, n_local=100) == [0, 1, 2]
    assert O.window_positions(t=10, W=4, local_base=9, n_local=100) == [9, 10]     # replay start
    assert O.window_positions(t=10, W=4, local_base=0, n_local=9) == [7, 8]
    assert O.window_positions(t=10, W=0, local_base=0, n_local=100) == []


def test_gather_rows_order_and_padding():
    d = 3
    kv = np.arange(30, dtype=np.float64).reshape(10, d)
    loc = -np.arange(12, dtype=np.float64).reshape(4, d)
    rows = O.gather_rows(kv, np.array([2, 7, -1, -1]), loc, local_base=20, t=22, W=2)
    np.testing.assert_array_equal(rows, np.stack([kv[2], kv[7], loc[1], loc[2]]))


# ------------------------------------------------------------------ one-stream compressor (HCA, CSA2 encoder)

def test_compress_single_hand_example():
    # m = 2, two channels.  Channel 0: logits 0 and ln 3 give weights 1/4, 3/4 -> 1 + 6 = 7;
    # channel 1: equal logits -> the mean 2.  With bias (ln 3, 0) / (0, ln 2): channel 0
    # logits ln 3, ln 3 -> mean 6; channel 1 logits 0, ln 2 -> 1/3 * 1 + 2/3 * 3 = 7/3.
    kv = np.array([[4.0, 1.0], [8.0, 3.0]])
    z = np.array([[0.0, 0.0], [math.log(3.0), 0.0]])
    np.testing.assert_allclose(O.compress_single_entry(kv, z, None, 2, 0), [7.0, 2.0], rtol=1e-15)
    bias = np.array([[math.log(3.0), 0.0], [0.0, math.log(2.0)]])
    np.testing.assert_allclose(O.compress_single_entry(kv, z, bias, 2, 0), [6.0, 7.0 / 3.0], rtol=1e-15)
    # entry 1 reads tokens 2, 3 only (no overlap with entry 0)
    kv2 = np.concatenate([kv, [[10.0, -2.0], [20.0, 4.0]]])
    z2 = np.concatenate([z, [[0.0, math.log(3.0)], [0.0, 0.0]]])
    np.testing.assert_allclose(O.compress_single_entry(kv2, z2, None, 2, 1), [15.0, 0.75 * -2.0 + 0.25 * 4.0],
                               rtol=1e-15)


def test_compress_single_closed_forms():
    m, dim = 128, 7
    kv = rng.standard_normal((3 * m, dim))
    # constant gate, no bias: the arithmetic mean of the block's m tokens
    z = np.full((3 * m, dim), 0.37)
    for i in range(3):
        np.testing.assert_allclose(O.compress_single_entry(kv, z, None, m, i), kv[m * i:m * (i + 1)].mean(0),
                                   rtol=1e-12, atol=1e-15)
    # a bias that cancels the gate's variation also gives the mean
    z = rng.standard_normal((m, dim))
    np.testing.assert_allclose(O.compress_single_entry(kv[:m], z, -z, m, 0), kv[:m].mean(0), rtol=1e-12, atol=1e-15)
    # one dominant logit per channel copies that token's value
    z = rng.standard_normal((m, dim))
    pick = rng.integers(0, m, dim)
    z[pick, np.arange(dim)] += 1e4
    np.testing.assert_allclose(O.compress_single_entry(kv[:m], z, None, m, 0), kv[pick, np.arange(dim)], rtol=1e-12)
    # m = 1: the softmax over one logit is 1, the entry is the token
    z = rng.standard_normal((5, dim))
    np.testing.assert_allclose(O.compress_single_range(kv[:5], z, None, 1, 0, 5), kv[:5], rtol=0, atol=0)
    # weights are positive and sum to 1 per channel
    _, w = O.compress_single_entry(kv, rng.standard_normal((3 * m, dim)) * 4, rng.standard_normal((m, dim)), m, 2,
                                   return_weights=True)
    assert w.shape == (m, dim) and np.all(w > 0)
    np.testing.assert_allclose(w.sum(0), 1.0, rtol=1e-14)


def test_compress_single_each_token_in_one_entry_and_causal():
    m, dim, n_ent = 4, 3, 6
    kv = rng.standard_normal((m * n_ent, dim))
    z = rng.standard_normal((m * n_ent, dim))
    bias = rng.standard_normal((m, dim)) * 0.1
    base = O.compress_single_range(kv, z, bias, m, 0, n_ent)
    for p in range(m * n_ent):
        kv2 = kv.copy()
        kv2[p] += 1.0
        changed = np.any(O.compress_single_range(kv2, z, bias, m, 0, n_ent) != base, axis=1)
        assert changed.tolist() == [i == p // m for i in range(n_ent)], p
    # the bias is indexed by the position inside the block, not by the token
    b2 = bias.copy()
    b2[1] += 0.5
    moved = np.any(O.compress_single_range(kv, z, b2, m, 0, n_ent) != base, axis=1)
    assert moved.all()
    # tok0 offset: the same entries from a buffer that starts at token m*2
    np.testing.assert_array_equal(O.compress_single_range(kv[2 * m:], z[2 * m:], bias, m, 2, n_ent, tok0=2 * m),
                                  base[2:])


def test_compress_single_is_two_stream_entry_zero():
    # the two-stream compressor's entry 0 has no stream b: it is the one-stream entry of
    # stream a with bias B^a
    m, dim = 4, 5
    kv = rng.standard_normal((m, 2, dim))
    z = rng.standard_normal((m, 2, dim))
    bias = rng.standard_normal((2, m, dim))
    np.testing.assert_allclose(O.compress_single_entry(kv[:, 0], z[:, 0], bias[0], m, 0),
                               O.compress_entry(kv, z, bias, m, 0), rtol=1e-15)


# ------------------------------------------------------------------ HCA attention

def test_hca_dense_rows_and_sdpa_reduction():
    H, d, E, W = 4, 16, 40, 6
    q = rng.standard_normal((H, d))
    kv = rng.standard_normal((E, d))
    loc = rng.standard_normal((W + 3, d))
    m, t, base = 128, 128 * 23 + 5, 128 * 23 + 5 - W - 2
    nv = O.visible_entries(t, m)
    assert nv == 23
    rows = O.dense_rows(kv, nv, loc, base, t, W)
    np.testing.assert_array_equal(rows, np.concatenate([kv[:nv], loc[t - W + 1 - base:t + 1 - base]]))
    # no window, sink -> -inf: dense MQA attention over the visible entries (torch SDPA)
    rows0 = O.dense_rows(kv, nv, loc, base, t, 0)
    out, _ = O.sparse_attention(q, rows0, np.full(H, -np.inf), 1 / math.sqrt(d))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, None, :], torch.from_numpy(kv[:nv])[None, None].expand(H, 1, nv, d),
        torch.from_numpy(kv[:nv])[None, None].expand(H, 1, nv, d), scale=1 / math.sqrt(d))[:, 0, 0]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12)
    # with window and sink: SDPA over the same rows with the sink as a zero-value column
    sink = rng.standard_normal(H)
    out, _ = O.sparse_attention(q, rows, sink, 1 / math.sqrt(d))
    np.testing.assert_allclose(out, _sdpa_with_sink(q, rows, sink, 1 / math.sqrt(d)), rtol=1e-12, atol=1e-14)


def test_hca_decode_step_writes_the_block_entry_first():
    class C:
        m, W, T, softmax_scale = 8, 4, 1, 0.25
    H, d, E = 2, 6, 10
    t = 8 * 7 - 1                                   # completes block 6
    inp = {"q_pos": np.array([t]), "q": rng.standard_normal((1, 1, H, d)), "sink": rng.standard_normal(H),
           "kv_local": rng.standard_normal((1, 8, d)), "local_base": np.array([t - 7]),
           "kv_str": rng.standard_normal((1, 8, d)), "z_str": rng.standard_normal((1, 8, d)),
           "bias": rng.standard_normal((8, d))}
    kv = rng.standard_normal((E, d))
    kv_before = kv.copy()
    r = O.hca_decode_step_sequence(C, inp, 0, kv)
    assert r["nv"] == 7 and r["entry"][0] == 6
    ent = O.compress_single_entry(inp["kv_str"][0], inp["z_str"][0], inp["bias"], 8, 6, tok0=t - 7)
    np.testing.assert_array_equal(kv[6], ent)
    np.testing.assert_array_equal(np.delete(kv, 6, 0), np.delete(kv_before, 6, 0))
    rows = np.concatenate([kv[:7], inp["kv_local"][0][4:8]])
    out, lse = O.sparse_attention(inp["q"][0, 0], rows, inp["sink"], 0.25)
    np.testing.assert_allclose(r["out"], out, rtol=1e-15)
    # a token inside a block writes nothing and sees only the completed entries
    inp["q_pos"] = np.array([t + 3])
    inp["local_base"] = np.array([t - 4])
    kv2 = kv.copy()
    r2 = O.hca_decode_step_sequence(C, inp, 0, kv2)
    assert r2["entry"] is None and r2["nv"] == 7
    np.testing.assert_array_equal(kv2, kv)



def test_decode_token_composition_against_torch():
    """Indexer -> top-k -> attention for one query, recomputed with torch routines: scores by a
    torch matmul + ReLU, selection by torch.topk (continuous scores, no ties), attention by SDPA
    over the selected entries then the window rows, the sink as a zero-value key."""
    class C:
        m, k, W, T, softmax_scale = 4, 5, 3, 2, 0.3
    H, d, HI, dI, E = 3, 8, 2, 6, 30
    t = 4 * 20 + 1                                   # nv = 20
    inp = {"q_pos": np.array([t - 5, t]), "q": rng.standard_normal((1, 2, H, d)),
           "qI": rng.standard_normal((1, 2, HI, dI)), "w": rng.standard_normal((1, 2, HI)),
           "sink": rng.standard_normal(H), "kv_local": rng.standard_normal((1, 10, d)),
           "local_base": np.array([t - 8])}
    kv = rng.standard_normal((E, d))
    kI = rng.standard_normal((E, dI))
    r = O.decode_token(C, inp, 0, 1, kv, kI)
    nv = 20
    assert r["nv"] == nv
    qI_t, w_t = torch.from_numpy(inp["qI"][0, 1]), torch.from_numpy(inp["w"][0, 1])
    ref_s = torch.relu(torch.from_numpy(kI[:nv]) @ qI_t.T) @ w_t
    np.testing.assert_allclose(r["scores"][:nv], ref_s.numpy(), rtol=1e-12)
    assert np.all(np.isneginf(r["scores"][nv:]))
    sel = np.sort(torch.topk(torch.from_numpy(r["scores_f32"][:nv].copy()), C.k).indices.numpy())
    np.testing.assert_array_equal(r["idx"], sel)
    rows = np.concatenate([kv[sel], inp["kv_local"][0][t - 2 - (t - 8):t + 1 - (t - 8)]])
    ref_out = _sdpa_with_sink(inp["q"][0, 1], rows, inp["sink"], C.softmax_scale)
    np.testing.assert_allclose(r["out"], ref_out, rtol=1e-12, atol=1e-14)


def _decode_case(store, d=6, dI=4):
    class C:
        m, W, T, k, softmax_scale = 4, 3, 1, 4, 0.25
    C.act = store
    m, H, HI, E = 4, 2, 2, 12
    t = 4 * 9 - 1                                   # completes block 8
    tok0 = t - 2 * m + 1                            # rows 0..3: block 7, rows 4..7: block 8
    kv_str = rng.standard_normal((1, 2 * m, 2, d))
    z_str = rng.standard_normal((1, 2 * m, 2, d))
    kvI_str = rng.standard_normal((1, 2 * m, 2, dI))
    zI_str = rng.standard_normal((1, 2 * m, 2, dI))
    # main KV: token 33 of stream a (the current block) dominates every channel's softmax
    u = np.resize(np.array([0.1, -0.3, 1.0 / 3.0, 2.0, -7.77, 1e-3]), d)
    z_str[0, 33 - tok0, 0, :] = 800.0
    kv_str[0, 33 - tok0, 0] = u
    # indexer key: token 30 of stream b (the previous block) dominates
    v = np.zeros(dI)
    v[:4] = [56.0, -1.5, 3.0, 0.7]
    zI_str[0, 30 - tok0, 1, :] = 800.0
    kvI_str[0, 30 - tok0, 1] = v
    inp = {"q_pos": np.array([t]), "q": rng.standard_normal((1, 1, H, d)), "sink": rng.standard_normal(H),
           "qI": np.eye(dI)[[0, 2]][None, None], "w": np.array([[[1.0, 2.0]]]),
           "kv_local": rng.standard_normal((1, 8, d)), "local_base": np.array([t - 7]),
           "kv_str": kv_str, "z_str": z_str, "kvI_str": kvI_str, "zI_str": zI_str,
           "bias": rng.standard_normal((2, m, d)) * 0.1, "biasI": rng.standard_normal((2, m, dI)) * 0.1}
    kv = rng.standard_normal((E, d))
    kI = rng.standard_normal((E, dI)) * 0.1
    kI[8] = 0.0                                     # stale row: indexing before the write scores 0
    return C, inp, kv, kI, t, u, v


@pytest.mark.parametrize("store", ["bf16", "f32"])
def test_decode_step_stores_the_entry_before_indexing(store):
    C, inp, kv, kI, t, u, v = _decode_case(store)
    kv0, kI0 = kv.copy(), kI.copy()
    r = O.decode_step_sequence(C, inp, 0, kv, kI)
    e = r["entry"][0]
    assert e == 8 and r["nv"] == 9
    want_u = O.round_to_bf16(u) if store == "bf16" else u.astype(np.float32).astype(np.float64)
    want_v = O.round_to_bf16(v) if store == "bf16" else v.astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(kv[8], want_u)            # the stream-a token, as the cache stores it
    np.testing.assert_array_equal(kI[8], want_v)            # the stream-b token of the previous block
    assert not np.array_equal(kv[8], u)
    np.testing.assert_array_equal(r["entry"][3], u)         # exact entry before storage
    np.testing.assert_array_equal(np.delete(kv, 8, 0), np.delete(kv0, 8, 0))
    np.testing.assert_array_equal(np.delete(kI, 8, 0), np.delete(kI0, 8, 0))
    # the new key is scored in this step: 1 * relu(56) + 2 * relu(3) = 62 is the best score
    assert r["scores"][8] == 62.0
    assert 8 in r["idx"] and (r["idx"] >= 0).sum() == 4
    rows = np.concatenate([kv[r["idx"]], inp["kv_local"][0][5:8]])
    out, lse = O.sparse_attention(inp["q"][0, 0], rows, inp["sink"], 0.25)
    np.testing.assert_allclose(r["out"], out, rtol=1e-15)
    # a token inside a block stores nothing and sees the same 9 entries
    inp["q_pos"] = np.array([t + 2])
    inp["local_base"] = np.array([t - 5])
    kv2, kI2 = kv.copy(), kI.copy()
    r2 = O.decode_step_sequence(C, inp, 0, kv2, kI2)
    assert r2["entry"] is None and r2["nv"] == 9
    np.testing.assert_array_equal(kv2, kv)
    np.testing.assert_array_equal(kI2, kI)


def test_decode_step_fp8_key_and_entry_storage():
    C, inp, kv, kI, t, u, v = _decode_case("bf16", d=72)   # an FP8 entry: 8 e4m3 dims + 64 bf16 dims
    r = O.decode_step_sequence(C, inp, 0, kv, kI, fp8_keys=True, fp8_kv=True)
    # the key re-quantised with scale amax / 448 = 56 / 448 = 1/8: 0.7 / (1/8) = 5.6 -> 5.5
    np.testing.assert_array_equal(kI[8], [56.0, -1.5, 3.0, 0.6875])
    assert r["scores"][8] == 62.0
    np.testing.assert_array_equal(kv[8], O.kv_fp8_decode(O.kv_fp8_encode(u)))


def test_decode_step_mxfp4_entry_storage():
    C, inp, kv, kI, t, u, v = _decode_case("bf16", d=32)   # two MXFP4 blocks of 16 channels
    r = O.decode_step_sequence(C, inp, 0, kv, kI, mxfp4_kv=True)
    np.testing.assert_array_equal(kv[8], O.mxfp4_decode(O.mxfp4_encode(r["entry"][3])))
    assert not np.array_equal(kv[8], r["entry"][3])
    # block 0 of u = [0.1, -0.3, 1/3, 2, -7.77, 1e-3, ...]: amax 7.77, scale e4m3(7.77/6 = 1.295) = 1.25;
    # -7.77 / 1.25 = -6.216 saturates to -6 (-7.5); 2 / 1.25 = 1.6 -> 1.5 (1.875)
    assert kv[8][4] == -7.5 and kv[8][3] == 1.875


def test_decode_step_mxfp4_key_storage():
    C, inp, kv, kI, t, u, v = _decode_case("bf16", dI=32)
    r = O.decode_step_sequence(C, inp, 0, kv, kI, mx_keys=True)
    # one block of 32 channels, amax 56: X = 2^(floor(log2 56) - 2) = 2^3; 56/8 = 7 saturates to
    # 6 (48), -1.5/8 = -0.1875 -> -0, 3/8 = 0.375 -> 0.5 (4), 0.7/8 = 0.0875 -> 0
    want = np.zeros(32)
    want[:4] = [48.0, -0.0, 4.0, 0.0]
    np.testing.assert_array_equal(kI[8], want)
    assert np.signbit(kI[8][1])
    assert r["scores"][8] == 1.0 * 48.0 + 2.0 * 4.0


# ------------------------------------------------------------------ MXFP4 indexer keys (OCP MX)

def test_mxfp4_key_ledger_and_scale_rule():
    # [V41d]: 128 channels = 64 packed bytes + 4 UE8M0 scales = 68 B a key
    p, sc = O.mxfp4_key_encode(np.ones((3, 128)))
    assert p.shape == (3, 64) and sc.shape == (3, 4) and p.itemsize * 64 + sc.itemsize * 4 == 68
    # UE8M0: 2^(c - 127), 0xFF is NaN
    np.testing.assert_array_equal(O.ue8m0_decode([127, 0, 254, 128]), [1.0, 2.0 ** -127, 2.0 ** 127, 2.0])
    assert np.isnan(O.ue8m0_decode([255])[0])
    # the shared exponent is floor(log2 amax) - 2 (E2M1's emax), as a biased byte: hand values
    cases = {6.0: 127, 4.0: 127, 3.99: 126, 8.0: 128, 7.99: 127, 0.088: 121, 1.0: 125, 2.0 ** 100: 225,
             0.0: 0, 1e-40: 0, 2.0 ** -125: 0, 2.0 ** -120: 5}
    for amax, byte in cases.items():
        blk = np.zeros(32)
        blk[5] = -amax
        assert O.mxfp4_key_encode(blk)[1][0] == byte, amax


def test_mxfp4_key_worked_example_and_nibble_order():
    x = np.zeros(128)
    x[:4] = [6.0, -0.5, 0.25, 3.3]        # block 0: X = 1; codes 7, 0x9, 0 (tie to even), 5 (3.3 -> 3)
    x[32] = 7.9                            # block 1: X = 1, 7.9 saturates to 6
    x[64] = 8.0                            # block 2: X = 2, 8/2 = 4 -> code 6
    p, sc = O.mxfp4_key_encode(x)
    assert p[0] == 0x97 and p[1] == 0x50 and p[16] == 0x07 and p[32] == 0x06
    np.testing.assert_array_equal(sc, [127, 127, 128, 0])
    d = O.mxfp4_key_decode(p, sc)
    np.testing.assert_array_equal(d[[0, 1, 2, 3, 32, 64]], [6.0, -0.5, 0.0, 3.0, 6.0, 8.0])
    # element 2i in the low nibble of byte i
    y = np.zeros(32)
    y[:2] = [1.0, 0.5]                     # X = 2^(0 - 2): codes of 4 and 2 -> 6 and 4
    assert O.mxfp4_key_encode(y)[0][0] == 0x46
    # the scale word keeps block j in byte j
    assert O.mxfp4_key_words(np.array([1, 2, 3, 4], np.uint8)) == 0x04030201
    np.testing.assert_array_equal(O.mxfp4_key_unwords(np.uint32(0x04030201)), [1, 2, 3, 4])


def test_mxfp4_key_round_trip_and_error_bound():
    # blocks whose largest magnitude is 4X or 6X re-encode to the same bytes
    codes = rng.integers(0, 16, (40, 128)).astype(np.uint8)
    codes[codes == 8] = 0                              # -0 decodes to 0 and re-encodes as +0
    for j in range(4):
        codes[:, 32 * j + rng.integers(0, 32)] = rng.choice([6, 7, 14, 15], 40)
    sc = rng.integers(100, 150, (40, 4)).astype(np.uint8)
    payload = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    p2, s2 = O.mxfp4_key_encode(O.mxfp4_key_decode(payload, sc))
    np.testing.assert_array_equal(p2, payload)
    np.testing.assert_array_equal(s2, sc)
    # error: at most half a grid step of the E2M1 value, times X (within the unsaturated range)
    x = rng.standard_normal((64, 128)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    p, sc = O.mxfp4_key_encode(x)
    x32 = x.astype(np.float32).astype(np.float64)
    err = np.abs(O.mxfp4_key_decode(p, sc) - x32).reshape(64, 4, 32)
    X = O.ue8m0_decode(sc)[..., None]
    a = np.abs(x32).reshape(64, 4, 32) / X
    half = np.where(a < 2, 0.25, np.where(a < 4, 0.5, np.where(a <= 6, 1.0, 2.0)))
    assert np.all(err <= half * X * (1 + 1e-12))
    assert np.all(a < 8)                   # floor(log2 amax) - 2 keeps every x / X below 8


# ------------------------------------------------------------------ RMSNorm, partial RoPE, inverse RoPE

def test_rms_norm_matches_torch():
    x = rng.standard_normal((5, 3, 64)) * 3.0
    w = rng.standard_normal(64)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, w, 1e-6), ref, rtol=1e-13, atol=1e-13)
    # unit weight: every row has mean square 1 / (1 + eps / ms)
    y = O.rms_norm(x, None, 0.0)
    np.testing.assert_allclose((y * y).mean(-1), 1.0, rtol=1e-13)


def test_rope_is_complex_rotation_of_the_last_dims():
    d, rd, theta = 48, 16, 500.0
    x = rng.standard_normal((7, d))
    pos = rng.integers(0, 10 ** 6, 7)
    y = O.rope(x, pos, rd, theta)
    np.testing.assert_array_equal(y[:, :d - rd], x[:, :d - rd])          # the other dims untouched
    z = x[:, d - rd::2] + 1j * x[:, d - rd + 1::2]
    freq = np.array([theta ** (-2.0 * j / rd) for j in range(rd // 2)])
    zr = z * np.exp(1j * pos[:, None] * freq[None, :])
    np.testing.assert_allclose(y[:, d - rd::2], zr.real, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(y[:, d - rd + 1::2], zr.imag, rtol=1e-9, atol=1e-12)
    # a rotation: norms kept, and RoPE(-p) undoes RoPE(p); rope_dims = 0 is the identity
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_allclose(O.rope(y, -pos, rd, theta), x, rtol=1e-9, atol=1e-9)
    np.testing.assert_array_equal(O.rope(x, pos, 0), x)
    # pair 0 turns by exactly pos radians
    p1 = O.rope(np.concatenate([np.zeros(d - rd), [1.0, 0.0], np.zeros(rd - 2)]), 2, rd, theta)
    np.testing.assert_allclose(p1[d - rd:d - rd + 2], [math.cos(2.0), math.sin(2.0)], rtol=1e-15)


def test_rope_scores_depend_on_relative_position():
    d, rd = 32, 16
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    s1 = O.rope(q, 1000, rd) @ O.rope(k, 937, rd)
    s2 = O.rope(q, 1000 + 4321, rd) @ O.rope(k, 937 + 4321, rd)
    assert abs(s1 - s2) < 1e-9 * (1 + abs(s1))
    assert abs(s1 - O.rope(q, 1000, rd) @ O.rope(k, 938, rd)) > 1e-6


def test_inverse_rope_restores_translation_invariance_of_shared_kv():
    # Key = value = RoPE'd row: the raw attention output depends on absolute positions; RoPE at
    # minus the query position on the output makes it depend on distances only.
    H, d, rd, n = 4, 32, 16, 9
    q = rng.standard_normal((H, d))
    rows = rng.standard_normal((n, d))
    sink = rng.standard_normal(H)
    t, pos = 5000, 5000 - rng.integers(0, 3000, n)

    def attend(shift):
        r = O.rope(rows, pos + shift, rd)
        out, _ = O.sparse_attention(O.rope(q, t + shift, rd), r, sink, 0.2)
        return out, O.inverse_rope(out, t + shift, rd)
    raw0, fix0 = attend(0)
    raw1, fix1 = attend(12345)
    np.testing.assert_allclose(fix1, fix0, rtol=1e-9, atol=1e-12)
    assert np.max(np.abs(raw1 - raw0)) > 1e-3


def test_norm_rope_composition_and_entry_position():
    x = rng.standard_normal((3, 2, 64))
    w = rng.standard_normal(64)
    pos = np.array([0, 17, 99])
    np.testing.assert_allclose(O.norm_rope(x, pos, w, 1e-6, 16), O.rope(O.rms_norm(x, w, 1e-6), pos, 16), rtol=0)
    assert O.compressed_entry_position(4, 10) == 40 and O.compressed_entry_position(128, 3) == 384


# ------------------------------------------------------------------ FP8 main-KV entries

def test_kv_fp8_entry_layout_and_roundtrip():
    # the pages' byte model: 64 RoPE dims in bf16 + 448 in FP8 = 576 bytes an entry
    x = rng.standard_normal((5, 512)) * 3.0
    b = O.kv_fp8_encode(x)
    assert b.shape == (5, 576) and b.dtype == np.uint8 and 64 * 2 + 448 == 576
    y = O.kv_fp8_decode(b)
    # FP8 part: the nearest e4m3 value (torch's conversion); RoPE part: the nearest bf16
    ref_head = torch.from_numpy(x[:, :448].astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref_tail = torch.from_numpy(x[:, 448:].astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(y[:, :448], ref_head)
    np.testing.assert_array_equal(y[:, 448:], ref_tail)
    # values already on the grids survive exactly; beyond 448 the FP8 part saturates
    np.testing.assert_array_equal(O.kv_fp8_decode(O.kv_fp8_encode(y)), y)
    big = np.zeros(512)
    big[0], big[1], big[500] = 1000.0, -1000.0, 1000.0
    yb = O.kv_fp8_decode(O.kv_fp8_encode(big))
    assert yb[0] == 448.0 and yb[1] == -448.0 and yb[500] == 1000.0
    # little-endian bf16 bits of the RoPE dims, right after the 448 codes
    one = np.zeros(512)
    one[448] = 1.0
    assert list(O.kv_fp8_encode(one)[448:450]) == [0x80, 0x3F]


def test_e4m3_encode_signed_zero_matches_torch():
    # OCP E4M3 has a signed zero: -0 and negatives that round to zero keep the sign bit
    v = np.array([0.0, -0.0, -1e-4, 1e-4, -2.0 ** -11, 2.0 ** -11, -3.0 * 2.0 ** -11, 448.0, -448.0])
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_encode(v), ref)


# ------------------------------------------------------------------ MXFP4 main-KV entries

def test_e2m1_grid_and_rounding():
    # OCP MX E2M1: codes 0..7 = 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 the sign
    np.testing.assert_array_equal(O.e2m1_decode(np.arange(8)), [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    np.testing.assert_array_equal(O.e2m1_decode(np.arange(8, 16)), -np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6]))
    np.testing.assert_array_equal(O.e2m1_encode(O.e2m1_decode(np.arange(16))), [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11,
                                                                                   12, 13, 14, 15])
    # midpoints tie to the even code; beyond 6 saturates; small negatives keep the sign
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.1, -5.0])
    np.testing.assert_array_equal(O.e2m1_decode(O.e2m1_encode(mids)), [0, 1, 1, 2, 2, 4, 4, 6, 6, -0.0, -4])
    assert O.e2m1_encode(np.array([-0.1]))[0] == 8


def test_mxfp4_entry_layout_range_and_roundtrip():
    # the pages' ledger: 512 channels at 0.5 B + one scale byte per 16 = 288 B
    x = rng.standard_normal((3, 512))
    b = O.mxfp4_encode(x)
    assert b.shape == (3, 288) and 512 // 2 + 512 // 16 == 288
    # values on the grid of their block's scale survive exactly (amax = 6 * scale)
    sc = np.array([0.5, 2.0 ** -6, 448.0, 0.0078125])
    grid = np.tile(np.array([6, -4, 3, 0.5, 0, 1, -1.5, 2, 6, -6, 4, 3, 2, 1, 0.5, 0]), 4) * np.repeat(sc, 16)
    y = np.concatenate([grid, rng.standard_normal(448)])
    np.testing.assert_array_equal(O.mxfp4_decode(O.mxfp4_encode(y))[:64], grid)
    # the largest magnitude: E2M1's 6 times E4M3's 448 = 2688
    big = np.zeros(16)
    big[3] = 2688.0
    assert O.mxfp4_decode(O.mxfp4_encode(big))[3] == 2688.0
    # element 2i in the low nibble, the scales after the payload
    one = np.zeros(16)
    one[0], one[1] = 6.0, -3.0          # scale 1, codes 7 and 8 | 5
    e = O.mxfp4_encode(one)
    assert e[0] == (7 | (13 << 4)) and O.e4m3_decode(e[8:9])[0] == 1.0
    # per element, the error is at most half a step of the block's grid (plus the scale's rounding)
    dec = O.mxfp4_decode(b).reshape(3, 32, 16)
    xb = x.reshape(3, 32, 16)
    s_ = O.e4m3_decode(b[:, 256:]).reshape(3, 32, 1)
    step = np.where(np.abs(xb) / s_ < 2, 0.5, np.where(np.abs(xb) / s_ < 4, 1.0, 2.0)) * s_
    assert np.all(np.abs(dec - xb) <= 0.5 * step + 1e-12 + np.maximum(np.abs(xb) - 6 * s_, 0))
