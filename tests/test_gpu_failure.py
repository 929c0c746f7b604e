"""Failure detection of the fused decode step, tested without a GPU fault.

Every wait of the decode step's indexer launch is bounded.  A fault-injection hook
(csa_debug_set) stops its producer from issuing any key-tile load and shortens the wait budget
to 1 ms, so its consumers' waits run out: the step must report CSA_ERR_TIMEOUT through
csa_get_last_error, every role of every CTA must still reach its exit (the process carries on
with a usable context), and the workspace state the step keeps for the next one (tickets and
list counters of the selection) must be left clean: the next step on the same workspace must
match the oracle exactly.  The pages have no counterpart; this is the failure path of the
library itself.
"""
import pytest
import torch

import compressed_sparse_attention_csa_gb300 as csa
from compressed_sparse_attention_csa_gb300 import _lib as L
from _helpers import assert_decode_matches, assert_step_selection_exact, lib_config, oracle_decode, run_gpu_decode
from synth import gen

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)

CSA_ERR_TIMEOUT = 7
WAIT_BUDGET_NS, SKIP_KEY_LOADS = 0, 1
DEFAULT_BUDGET_NS = 2_000_000_000


def _step(cfg, inp):
    c = lib_config(cfg)
    out = torch.empty(cfg.B, cfg.H, cfg.d, device=DEV, dtype=cfg.torch_act)
    idx = torch.empty(cfg.B, cfg.k, dtype=torch.int32, device=DEV)
    csa.decode_step(c, q_pos=inp["q_pos"], q=inp["q"], qI=inp["qI"], w=inp["w"], sink=inp["sink"],
                    kv_comp=inp["kv_comp"], kI=inp["kI"], kscale=inp.get("kscale"), kv_tail=inp["kv_str"],
                    z_tail=inp["z_str"], kvI_tail=inp["kvI_str"], zI_tail=inp["zI_str"], bias=inp["bias"],
                    biasI=inp["biasI"], kv_local=inp["kv_local"], local_base=inp["local_base"], out=out,
                    idx_out=idx)
    return idx


@pytest.mark.parametrize("cid", [2, 4])
def test_decode_step_timeout_is_reported_and_the_next_step_is_clean(cid):
    lib = L.load()
    cfg = gen.CONFIGS[cid].replace(B=2, N=4 * 3000)
    assert csa.get_last_error() == 0
    assert lib.csa_debug_set(WAIT_BUDGET_NS, 10) != 0          # out of range: refused
    assert lib.csa_debug_set(WAIT_BUDGET_NS, 1_000_000) == 0
    assert lib.csa_debug_set(SKIP_KEY_LOADS, 1) == 0
    try:
        idx = _step(cfg, gen.make_inputs(cfg, DEV))
        status = csa.get_last_error()
    finally:
        assert lib.csa_debug_set(SKIP_KEY_LOADS, 0) == 0
        assert lib.csa_debug_set(WAIT_BUDGET_NS, DEFAULT_BUDGET_NS) == 0
    assert status == CSA_ERR_TIMEOUT
    assert bool(((idx >= -1) & (idx < cfg.E)).all())            # whatever it selected is in range
    assert csa.get_last_error() == 0                            # read once, then cleared
    # the next step on the same workspace
    inp = gen.make_inputs(cfg, DEV)
    ref = oracle_decode(cfg, inp)
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    out, lse, idx = run_gpu_decode(cfg, inp, scores_out=scores)
    assert_decode_matches(cfg, inp, ref, out, lse, idx)
    assert_step_selection_exact(cfg, ref, idx, scores)


def test_decode_step_reset_clears_a_dirty_workspace():
    """A workspace whose carried state is dirty (as after a step whose launches never ran) is
    made usable again by csa_decode_step_reset: the next step matches the oracle exactly."""
    from compressed_sparse_attention_csa_gb300 import ops
    cfg = gen.CONFIGS[2].replace(B=3, N=4 * 2500)
    inp = gen.make_inputs(cfg, DEV)
    ref = oracle_decode(cfg, inp)
    run_gpu_decode(cfg, gen.make_inputs(cfg, DEV))          # the workspace exists and is clean
    ws = ops._decode_ws[(str(DEV), cfg.B)]
    state = 4 * 4166 * cfg.B
    ws[:state].fill_(0x5A)                                   # dirty every carried histogram, ticket, counter
    csa.decode_step_reset(lib_config(cfg))
    torch.cuda.synchronize()
    assert int(ws[:state].count_nonzero()) == 0
    scores = torch.empty(cfg.B, cfg.E, device=DEV)
    out, lse, idx = run_gpu_decode(cfg, inp, scores_out=scores)
    assert_decode_matches(cfg, inp, ref, out, lse, idx)
    assert_step_selection_exact(cfg, ref, idx, scores)
