"""The C ABI without a GPU: the library loads, exports every declared symbol, and its host-side
validation rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

from compressed_sparse_attention_csa_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")

A = ctypes.c_void_p(0x10000)      # 16-byte aligned fake device pointer (never dereferenced)
MIS = ctypes.c_void_p(0x10004)    # misaligned


def _declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z_0-9]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def lib():
    return L.load()


def _cfg(**kw):
    c = dict(B=2, H=64, d=512, HI=64, dI=128, m=4, k=512, W=128, act=L.CSA_BF16, kidx=L.CSA_BF16,
             softmax_scale=512 ** -0.5)
    c.update(kw)
    return L.csa_config(**c)


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "csa_decode_step" in names and "csa_topk" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(L.SIGNATURES), set(names) ^ set(L.SIGNATURES)


def test_version_and_strings(lib):
    assert lib.csa_version() >= 100
    assert lib.csa_status_string(0) == b"ok"
    assert lib.csa_status_string(7) == b"device wait timed out"


def test_config_validation(lib):
    bad = [_cfg(B=0), _cfg(dI=48), _cfg(k=0), _cfg(k=5000), _cfg(W=-1), _cfg(m=0)]
    for c in bad:
        st = lib.csa_topk(ctypes.byref(c), A, 10, 1, 10, None, None, A, A, 1 << 20, None)
        assert st == 2, (c.B, c.dI, c.k)
    c = _cfg(act=L.CSA_E4M3)
    assert lib.csa_topk(ctypes.byref(c), A, 10, 1, 10, None, None, A, A, 1 << 20, None) == 3
    assert lib.csa_topk(None, A, 10, 1, 10, None, None, A, A, 1 << 20, None) == 1


def test_topk_argument_errors(lib):
    c = _cfg()
    assert lib.csa_topk(ctypes.byref(c), None, 10, 1, 10, None, None, A, A, 1 << 20, None) == 1
    assert lib.csa_topk(ctypes.byref(c), MIS, 10, 1, 10, None, None, A, A, 1 << 20, None) == 4
    assert lib.csa_topk(ctypes.byref(c), A, 5, 1, 10, None, None, A, A, 1 << 20, None) == 2   # ld < n_cols
    # a long row needs workspace
    need = lib.csa_workspace_size(L.CSA_OP_TOPK, ctypes.byref(c), 4, 262144)
    assert 0 < need < (1 << 40)
    assert lib.csa_topk(ctypes.byref(c), A, 262144, 4, 262144, None, None, A, A, need - 1, None) == 5
    assert lib.csa_topk(ctypes.byref(c), A, 262144, 4, 262144, None, None, A, None, 0, None) == 5


def test_compress_argument_errors(lib):
    c = _cfg()
    f = lib.csa_compress_kv
    # entries 2..3 need tokens from m*(2-1) = 4 up to m*4 = 16: tok0 = 4, n_tok = 12 is the minimum
    assert f(ctypes.byref(c), 512, A, A, A, 12, 5, 2, 4, A, L.CSA_BF16, None, 8, None) == 2   # tok0 too late
    assert f(ctypes.byref(c), 512, A, A, A, 11, 4, 2, 4, A, L.CSA_BF16, None, 8, None) == 2   # too few tokens
    assert f(ctypes.byref(c), 512, A, A, A, 12, 4, 2, 9, A, L.CSA_BF16, None, 8, None) == 2   # beyond E_cap
    assert f(ctypes.byref(c), 512, A, A, A, 12, 4, 2, 4, A, L.CSA_E4M3, None, 8, None) == 1   # e4m3 needs scale
    assert f(ctypes.byref(c), 512, None, A, A, 12, 4, 2, 4, A, L.CSA_BF16, None, 8, None) == 1
    assert f(ctypes.byref(c), 512, A, MIS, A, 12, 4, 2, 4, A, L.CSA_BF16, None, 8, None) == 4
    assert f(ctypes.byref(c), 2048, A, A, A, 12, 4, 2, 4, A, L.CSA_BF16, None, 8, None) == 2  # dim too large


def test_indexer_and_attention_argument_errors(lib):
    c = _cfg()
    f = lib.csa_indexer_scores
    assert f(ctypes.byref(c), A, A, 1, A, A, None, 100, None, 0, A, 50, None, 0, None) == 2   # ld < E_cap
    ce = _cfg(kidx=L.CSA_E4M3)
    assert f(ctypes.byref(ce), A, A, 1, A, A, None, 100, None, 0, A, 100, None, 0, None) == 1  # no kscale
    g = lib.csa_sparse_attn
    assert g(ctypes.byref(c), A, 1, A, 10, A, A, 4, A, A, None, A, None, None, 0, None) == 1    # sink NULL
    odd = _cfg(d=256, H=64)     # neither the tensor-core shape nor a CUDA-core shape
    assert g(ctypes.byref(odd), A, 1, A, 10, A, A, 4, A, A, A, A, None, None, 0, None) == 2


def test_decode_step_argument_errors(lib):
    c = _cfg()
    args = L.csa_decode_args()
    assert lib.csa_decode_step(ctypes.byref(c), ctypes.byref(args), A, 1 << 30, None) == 1
    for name, _ in L.csa_decode_args._fields_:
        if name not in ("E_cap", "L", "kscale", "lse", "idx_out", "scores_out"):
            setattr(args, name, 0x10000)
    args.E_cap, args.L = 1 << 16, 128
    assert lib.csa_decode_step(ctypes.byref(c), ctypes.byref(args), A, 16, None) == 5        # workspace
    args.q = 0x10008
    assert lib.csa_decode_step(ctypes.byref(c), ctypes.byref(args), A, 1 << 30, None) == 4
    args.q = 0x10000
    ce = _cfg(kidx=L.CSA_E4M3)
    assert lib.csa_decode_step(ctypes.byref(ce), ctypes.byref(args), A, 1 << 30, None) == 1  # kscale


def test_workspace_queries(lib):
    c = _cfg(B=4)
    assert lib.csa_workspace_size(L.CSA_OP_COMPRESS, ctypes.byref(c), 4, 1) == 0
    dec = lib.csa_workspace_size(L.CSA_OP_DECODE, ctypes.byref(c), 4, 262144)
    assert dec > 4 * 262144 * 4
    assert lib.csa_block_pool_workspace_size(8, 262144, 8, 2048) > 0
    assert lib.csa_block_pool_workspace_size(8, 262144, 8, 5000) == ctypes.c_size_t(-1).value
    bad = _cfg(dI=7)
    assert lib.csa_workspace_size(L.CSA_OP_TOPK, ctypes.byref(bad), 1, 10) == ctypes.c_size_t(-1).value


def test_decode_step_reset_argument_errors(lib):
    c = _cfg(B=3)
    need = 4 * 4166 * 3
    f = lib.csa_decode_step_reset
    assert f(None, A, need, None) == 1
    assert f(ctypes.byref(c), None, need, None) == 1
    assert f(ctypes.byref(_cfg(B=0)), A, need, None) == 2
    assert f(ctypes.byref(c), MIS, need, None) == 4
    assert f(ctypes.byref(c), A, need - 1, None) == 5
    # the state region is at the front of the step's own workspace
    assert lib.csa_workspace_size(L.CSA_OP_DECODE, ctypes.byref(c), 3, 262144) >= need


def test_mxfp4_key_argument_errors(lib):
    f = lib.csa_indexer_scores
    mx = _cfg(kidx=L.CSA_MXFP4)
    A32 = ctypes.c_void_p(0x10020)                 # 32-byte aligned
    A16 = ctypes.c_void_p(0x10010)                 # 16-byte but not 32-byte aligned
    assert f(ctypes.byref(mx), A, A, 1, A, A32, None, 100, None, 0, A, 100, None, 0, None) == 1   # scale words
    assert f(ctypes.byref(mx), A, A, 1, A, A16, A, 100, None, 0, A, 100, None, 0, None) == 4      # payload alignment
    assert f(ctypes.byref(mx), A, A, 1, A, A32, A, 102, None, 0, A, 102, None, 0, None) == 2      # E_cap % 4
    assert f(ctypes.byref(_cfg(kidx=L.CSA_MXFP4, act=L.CSA_F32)), A, A, 1, A, A32, A, 100, None, 0, A, 100,
             None, 0, None) == 3                                                                  # bf16 queries only
    assert f(ctypes.byref(_cfg(kidx=L.CSA_MXFP4, dI=64)), A, A, 1, A, A32, A, 100, None, 0, A, 100,
             None, 0, None) == 2                                                                  # 128 channels
    g = lib.csa_compress_kv
    assert g(ctypes.byref(mx), 128, A, A, A, 12, 4, 2, 4, A, L.CSA_MXFP4, None, 8, None) == 1    # scale words
    assert g(ctypes.byref(mx), 64, A, A, A, 12, 4, 2, 4, A, L.CSA_MXFP4, A, 8, None) == 2        # dim 128 only
    args = L.csa_decode_args()
    for name, _ in L.csa_decode_args._fields_:
        if name not in ("E_cap", "L", "kscale", "lse", "idx_out", "scores_out"):
            setattr(args, name, 0x10020)
    args.E_cap, args.L = 1 << 16, 128
    assert lib.csa_decode_step(ctypes.byref(mx), ctypes.byref(args), A, 1 << 30, None) == 1        # scale words
    args.kscale = 0x10020
    args.E_cap = (1 << 16) + 2
    assert lib.csa_decode_step(ctypes.byref(mx), ctypes.byref(args), A, 1 << 30, None) == 2        # E_cap % 4


def test_step_inputs_layout_on_cpu():
    """StepInputs packs the tensors 256-byte aligned, keeps shapes, dtypes and values, and its
    upload moves the host mirror's contents into the device views in one copy."""
    import torch
    from compressed_sparse_attention_csa_gb300.ops import StepInputs
    g = torch.Generator().manual_seed(5)
    ts = {"q": torch.randn(3, 5, 7, generator=g).to(torch.bfloat16),
          "pos": torch.tensor([1, 2, 3], dtype=torch.int64),
          "x": torch.randn(33, generator=g)}
    st = StepInputs(ts, "cpu")
    assert st.nbytes == 256 * (1 + 1 + 1)
    for k, t in ts.items():
        assert st.dev[k].shape == t.shape and st.dev[k].dtype == t.dtype and st.dev[k].is_contiguous()
        assert st.dev[k].data_ptr() % 256 == st.dev["q"].data_ptr() % 256
        assert torch.equal(st.dev[k], t) and torch.equal(st.host[k], t)
    st.host["pos"].copy_(torch.tensor([7, 8, 9]))
    st.host["x"].zero_()
    assert torch.equal(st.dev["pos"], ts["pos"])
    st.upload()
    assert torch.equal(st.dev["pos"], torch.tensor([7, 8, 9])) and not st.dev["x"].any()
    assert torch.equal(st.dev["q"], ts["q"])
