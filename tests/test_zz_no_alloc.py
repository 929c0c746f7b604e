"""csa_topk_noalloc: the top-k for callers that cannot allocate device memory.

Such callers (a plugin inside another runtime that owns every device allocation, or a
latency-critical path where an allocation could block or fail) have no workspace to give
csa_topk.  The no-allocation entry point uses a fixed scratch array inside the library; its
results must equal csa_topk's exactly (the selection is exact), and the oracle's top-k of the
same fp32 scores, on consecutive calls that reuse the same scratch.
"""
import ctypes

import numpy as np
import pytest
import torch

from compressed_sparse_attention_csa_gb300 import _lib as L
from oracle import csa_oracle as O
from synth import gen

pytestmark = pytest.mark.gpu


def _cfg(k):
    return L.csa_config(B=1, H=64, d=512, HI=64, dI=128, m=4, k=k, W=128, act=L.CSA_BF16, kidx=L.CSA_BF16,
                        softmax_scale=512 ** -0.5)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _topk_with_workspace(lib, scores, k, n_valid):
    rows, n = scores.shape
    cfg = _cfg(k)
    idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    need = lib.csa_workspace_size(L.CSA_OP_TOPK, ctypes.byref(cfg), rows, n)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    st = lib.csa_topk(ctypes.byref(cfg), _ptr(scores), n, rows, n, _ptr(n_valid), None, _ptr(idx), _ptr(ws),
                      ws.numel(), _stream())
    assert st == 0
    return idx


def _topk_noalloc(lib, scores, k, n_valid):
    rows, n = scores.shape
    cfg = _cfg(k)
    idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    st = lib.csa_topk_noalloc(ctypes.byref(cfg), _ptr(scores), n, rows, n, _ptr(n_valid), None, _ptr(idx), _stream())
    assert st == 0, L.STATUS.get(st, st)
    return idx


@pytest.mark.parametrize("rows,n,k", [(4, 262144, 512), (16, 5000, 64)])
def test_noalloc_equals_topk_on_two_calls(rows, n, k):
    lib = L.load()
    for call in range(2):  # the second call reuses the scratch the first one left behind
        x = gen.normal(900 + call, rows * n, device="cuda").reshape(rows, n).to(torch.float32)
        x = torch.round(x * 32) / 32  # many exact ties
        nv = torch.tensor([n - 3 * r for r in range(rows)], dtype=torch.int32, device="cuda")
        ref = _topk_with_workspace(lib, x, k, nv)
        got = _topk_noalloc(lib, x, k, nv)
        assert lib.csa_get_last_error(_stream()) == 0
        assert torch.equal(got, ref), f"call {call}"
        xs, nvs, gs = x.cpu().numpy(), nv.cpu().numpy(), got.cpu().numpy()
        for r in range(rows):
            np.testing.assert_array_equal(gs[r], O.topk(xs[r], int(nvs[r]), k), err_msg=f"call {call} row {r}")


def test_noalloc_rejects_sizes_beyond_the_scratch():
    lib = L.load()
    cfg = _cfg(512)
    rows, n = 16, 262144     # the histogram path's candidate slots for these need about 8.4 MB
    need = lib.csa_workspace_size(L.CSA_OP_TOPK, ctypes.byref(cfg), rows, n)
    assert need > (4 << 20)
    scores = torch.zeros(rows, n, dtype=torch.float32, device="cuda")
    out = torch.full((rows, 512), -7, dtype=torch.int32, device="cuda")
    st = lib.csa_topk_noalloc(ctypes.byref(cfg), _ptr(scores), n, rows, n, None, None, _ptr(out), _stream())
    assert st == 5  # CSA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert bool((out == -7).all())
