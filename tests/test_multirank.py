"""Multi-process decode path on the CPU: two `gloo` ranks split a batch of sequences.

Each rank generates only its own sequences (the generator's row offset), runs the oracle's
decode step on them, and the gathered outputs must equal a single process running the whole
batch, value for value.  The host reductions used for timing (max over ranks, sum over ranks,
whole-job throughput) are checked on the same process group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from compressed_sparse_attention_csa_gb300.shard import (job_throughput, max_over_ranks, shard_rows,
                                                           sum_over_ranks)
from oracle import csa_oracle as O
from synth import gen

WORLD = 2


def _small_cfg():
    # decode preset with the 64K-context structure, shortened so the oracle runs in seconds
    return gen.small_variant(gen.CONFIGS[2], B=3, N=2048, k=128, W=32)


def _decode_rows(cfg, inp):
    """Oracle decode outputs [B, H, d] and selections [B, k] for the given inputs."""
    np_inp = {k: v.to(torch.float64).numpy() if v.is_floating_point() else v.numpy() for k, v in inp.items()}
    outs, sels = [], []
    for b in range(cfg.B):
        kv = np_inp["kv_comp"][b].copy()
        ki = np_inp["kI"][b].copy()
        r = O.decode_step_sequence(cfg, np_inp, b, kv, ki)
        outs.append(r["out"])
        sels.append(r["idx"])
    return np.stack(outs), np.stack(sels)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = _small_cfg()
        start, count = shard_rows(cfg.B, world, rank)
        local = cfg.replace(B=count)
        inp = gen.make_inputs(local, "cpu", row0=start)
        out, sel = _decode_rows(local, inp)
        # pad to the largest shard so the gather has equal shapes
        cmax = shard_rows(cfg.B, world, 0)[1]
        pad_o = np.zeros((cmax,) + out.shape[1:])
        pad_s = np.full((cmax,) + sel.shape[1:], -7, dtype=np.int64)
        pad_o[:count] = out
        pad_s[:count] = sel
        go = [torch.zeros(pad_o.shape, dtype=torch.float64) for _ in range(world)]
        gs = [torch.zeros(pad_s.shape, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(go, torch.from_numpy(pad_o))
        dist.all_gather(gs, torch.from_numpy(pad_s))
        mx = max_over_ranks(1.5 + rank)
        sm = sum_over_ranks(10.0 * (rank + 1))
        tp = job_throughput(4.0, 2.0 + rank)
        if rank == 0:
            rows_o, rows_s = [], []
            for r in range(world):
                n = shard_rows(cfg.B, world, r)[1]
                rows_o.append(go[r].numpy()[:n])
                rows_s.append(gs[r].numpy()[:n])
            np.savez(os.path.join(result_dir, "gathered.npz"), out=np.concatenate(rows_o),
                     idx=np.concatenate(rows_s), mx=mx, sm=sm, tp=tp)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("B,world", [(4, 2), (3, 2), (1, 2), (0, 3), (7, 4), (8, 8), (5, 1)])
def test_shard_rows_cover_batch_once(B, world):
    seen = []
    prev_end = 0
    for r in range(world):
        s, c = shard_rows(B, world, r)
        assert s == prev_end and c >= 0
        prev_end = s + c
        seen.extend(range(s, s + c))
    assert seen == list(range(B))
    counts = [shard_rows(B, world, r)[1] for r in range(world)]
    assert max(counts) - min(counts) <= 1


def test_shard_rows_rejects_bad_requests():
    for args in [(4, 0, 0), (4, 2, 2), (4, 2, -1), (-1, 2, 0)]:
        with pytest.raises(ValueError):
            shard_rows(*args)


def test_row_offset_generation_matches_full_batch():
    cfg = _small_cfg()
    full = gen.make_inputs(cfg, "cpu")
    part = gen.make_inputs(cfg.replace(B=2), "cpu", row0=1)
    for k, v in part.items():
        if k in ("sink", "bias", "biasI"):
            assert torch.equal(v, full[k]), k
        else:
            assert torch.equal(v, full[k][1:3]), k


def test_two_gloo_ranks_match_single_process(tmp_path):
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, WORLD, port, str(tmp_path))) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = np.load(tmp_path / "gathered.npz")
    cfg = _small_cfg()
    ref_out, ref_idx = _decode_rows(cfg, gen.make_inputs(cfg, "cpu"))
    np.testing.assert_array_equal(res["idx"], ref_idx)
    np.testing.assert_array_equal(res["out"], ref_out)
    assert float(res["mx"]) == 1.5 + (WORLD - 1)
    assert float(res["sm"]) == sum(10.0 * (r + 1) for r in range(WORLD))
    assert float(res["tp"]) == pytest.approx(4.0 * WORLD / (2.0 + WORLD - 1))
