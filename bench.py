#!/usr/bin/env python
"""CSA hot-path benchmark: decode tokens/s of the fused decode step at 1M-token context.

Workload (default): V4-Flash CSA decode at 1,048,576 tokens of context, batch 4, m = 4
(262,144 compressed entries per sequence), FP8 e4m3 indexer keys with one fp32 scale per
entry, bf16 KV, 64 query heads x 512, indexer 64 heads x 128, top-k 512, window 128.
One step = one decode token for each of the 4 sequences through csa_decode_step: compress
the completed block, score every visible entry, top-512, sparse attention with sink.

Timing: W warm-up steps, then K timed steps; L2 is flushed (512 MiB written) before every
step, outside the timed events; each step is bracketed by CUDA events on the launching
stream.  `value` uses inputs resident in HBM; `e2e` adds, every step, the pinned-host ->
device copy of the step's inputs and the device -> host copy of its output.  The dominant
kernel (the indexer) is timed the same way on its own for the roofline entry.

`--impl reference` times the CPU oracle (oracle/csa_oracle.py, float64 numpy) on a bounded
sample of the same workload on the host cores.  Multi-GPU (torchrun): every rank runs its
own batch (sequences are independent; no collective on the data path), `value` is the sum
over ranks, time is the max over ranks.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, choices=[2, 4])
    ap.add_argument("--cpu-seqs", type=int, default=12, help="decode tokens in the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["step", "indexer"], default=None,
                    help="run only this stage on the workload (for profiler captures); prints its time")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


STAGE_PROFILES = {4: "indexer_tc_e4m3_1M_decode.md", 2: "indexer_tc_bf16_64K_decode.md"}
STAGE_KERNELS = ("indexer_qprep_kernel", "indexer_tc_kernel")
STAGE_SOURCES = ("k_indexer.cu", "csa_ptx.cuh", "csa_internal.h")


def stage_traffic(config):
    """DRAM bytes per indexer-stage launch from the committed ncu summary, or None.

    The summary carries `traffic-bytes-per-launch <kernel> <bytes>` lines and the sha256 of
    the kernel sources it was taken with; the figure is used only while every stage kernel
    has a line and the sources are unchanged."""
    import hashlib
    path = os.path.join(ROOT, "profiles", STAGE_PROFILES.get(config, ""))
    if not os.path.isfile(path):
        return None
    per, sha = {}, None
    with open(path) as f:
        for line in f:
            w = line.split()
            if len(w) == 3 and w[0] == "traffic-bytes-per-launch":
                per[w[1]] = int(w[2])
            elif len(w) == 2 and w[0] == "sources-sha256":
                sha = w[1]
    src = os.path.join(ROOT, "compressed_sparse_attention_csa_gb300", "csrc")
    h = hashlib.sha256()
    for name in STAGE_SOURCES:
        with open(os.path.join(src, name), "rb") as f:
            h.update(f.read())
    if sha != h.hexdigest() or any(k not in per for k in STAGE_KERNELS):
        return None
    return sum(per[k] for k in STAGE_KERNELS)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed loop runs."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-i", gpu_id, "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l for (ts, l) in self.lines if t0 - 0.05 <= ts <= t1 + 0.1] or [l for (_, l) in self.lines[-3:]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in rows:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle sample

def oracle_sample(cfg, inp, n_seqs):
    """Time the oracle on n_seqs sequences of the workload (float64 numpy on the host cores)."""
    import numpy as np
    import torch
    from oracle import csa_oracle as O

    n_seqs = max(1, n_seqs)
    elapsed = 0.0
    cache = {}
    sub = cfg.replace(B=1)
    for i in range(n_seqs):
        b = (i * cfg.B) // n_seqs
        if b not in cache:
            # host copies of sequence b's inputs (not timed: the oracle reads host arrays)
            host = {}
            for k, v in inp.items():
                x = v if k in ("bias", "biasI", "sink") else v[b:b + 1]
                host[k] = x.cpu().to(torch.float64).numpy() if x.is_floating_point() else x.cpu().numpy()
            cache = {b: host}
        host = dict(cache[b])
        codes = host.pop("kI")
        kscale = host.pop("kscale", None)
        kv_comp = host["kv_comp"][0].copy()
        t0 = time.perf_counter()
        kdeq = O.e4m3_decode(codes[0]) * kscale[0][:, None] if kscale is not None else codes[0].astype(np.float64)
        O.decode_step_sequence(sub, host, 0, kv_comp, kdeq, fp8_keys=kscale is not None)
        elapsed += time.perf_counter() - t0
    return n_seqs, elapsed


def cpu_threads():
    try:
        import numpy as np  # noqa: F401
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return max(int(i.get("num_threads", 1)) for i in info)
    except Exception:
        pass
    return os.cpu_count() or 1


# ------------------------------------------------------------------ main

def main():
    args = parse_args()
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from synth import gen
    cfg = gen.CONFIGS[args.config]
    workload = ("V4-Flash CSA decode step, batch 4 @ 1,048,576-token context (262,144 entries/seq), "
                "FP8 e4m3 indexer keys + fp32 scale, bf16 KV, 64x512 heads, indexer 64x128, k 512, W 128"
                if args.config == 4 else
                "V4-Flash CSA decode step, batch 16 @ 65,536-token context (16,384 entries/seq), bf16, "
                "64x512 heads, indexer 64x128, k 512, W 128")
    metric = "CSA decode tok/s @1M ctx" if args.config == 4 else "CSA decode tok/s @64K ctx"
    config_obj = {"workload": workload, "batch": cfg.B, "context": cfg.N, "m": cfg.m, "entries_per_seq": cfg.E,
                  "heads": cfg.H, "head_dim": cfg.d, "indexer": f"{cfg.HI}x{cfg.dI}", "top_k": cfg.k,
                  "window": cfg.W, "indexer_keys": "e4m3+fp32 scale" if cfg.kidx == "fp8" else "bf16",
                  "l2": "flushed (512 MiB write) before every timed step",
                  "timing": "device time per step: CUDA events around a CUDA-graph replay of csa_decode_step"}

    if args.impl == "reference":
        if rank != 0:
            return
        torch.manual_seed(0)
        inp = gen.make_inputs(cfg.replace(B=1), "cpu")
        for _ in range(max(0, args.warmup and 1)):
            pass
        n_total, t_total = 0, 0.0
        for _ in range(args.steps):
            n, t = oracle_sample(cfg.replace(B=1), inp, 1)
            n_total += n
            t_total += t
        v = n_total / t_total
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config_obj,
                "cpu_baseline": {"value": v, "unit": "tok/s", "cores": cpu_threads(), "kind": "oracle",
                                 "sample": "each step: one sequence of the workload (compress, 262,144-key indexer, "
                                           "top-512, attention) in float64 numpy"},
                "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import compressed_sparse_attention_csa_gb300 as csa
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    # weak scaling: every rank decodes its own cfg.B sequences of a batch of cfg.B * world
    from compressed_sparse_attention_csa_gb300.shard import max_over_ranks, shard_rows
    row0, n_rows = shard_rows(cfg.B * world, world, rank)
    assert n_rows == cfg.B
    inp = gen.make_inputs(cfg, dev, row0=row0)
    c = csa.Config(B=cfg.B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
                   act=torch.bfloat16, fp8_keys=cfg.kidx == "fp8", softmax_scale=cfg.softmax_scale)
    out = torch.empty(cfg.B, cfg.H, cfg.d, device=dev, dtype=torch.bfloat16)
    lse = torch.empty(cfg.B, cfg.H, device=dev)
    idx = torch.empty(cfg.B, cfg.k, device=dev, dtype=torch.int32)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    args_d = dict(q_pos=inp["q_pos"], q=inp["q"], qI=inp["qI"], w=inp["w"], sink=inp["sink"],
                  kv_comp=inp["kv_comp"], kI=inp["kI"], kscale=inp.get("kscale"), kv_tail=inp["kv_str"],
                  z_tail=inp["z_str"], kvI_tail=inp["kvI_str"], zI_tail=inp["zI_str"], bias=inp["bias"],
                  biasI=inp["biasI"], kv_local=inp["kv_local"], local_base=inp["local_base"], out=out, lse=lse,
                  idx_out=idx)

    def step():
        csa.decode_step(c, **args_d)

    stream = torch.cuda.current_stream(dev)
    if args.only:
        scores_only = torch.empty(cfg.B, cfg.E, device=dev)

        def only_fn():
            if args.only == "step":
                step()
            else:
                csa.indexer_scores(c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"], scores_only,
                                   kscale=inp.get("kscale"))
        for _ in range(args.warmup):
            only_fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            only_fn()
        torch.cuda.synchronize(dev)
        assert csa.get_last_error() == 0
        print(json.dumps({"only": args.only, "config": args.config, "calls": args.steps,
                          "ms_per_call_back_to_back": 1e3 * (time.perf_counter() - t0) / max(args.steps, 1)}))
        return
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    assert csa.get_last_error() == 0

    # The decode step is captured once into a CUDA graph (the library's launches are
    # stream-ordered and allocate nothing) and replayed: the device time of a step then does
    # not depend on how fast the host enqueues it.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize(dev)
        return g

    n_cap = csa.launch_count()
    g_step = capture(step)
    launches_per_step = csa.launch_count() - n_cap
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        g_step.replay()
    torch.cuda.synchronize(dev)
    assert csa.get_last_error() == 0

    gpu_id = "0"
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(dev.index or 0)
    sampler = ClockSampler(gpu_id) if rank == 0 else None

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        g_step.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    launches = launches_per_step * K
    total_ms = sum(a.elapsed_time(b) for a, b in ev)
    assert csa.get_last_error() == 0
    total_ms = max_over_ranks(total_ms)
    clocks = sampler.stop(t_wall0, t_wall1) if sampler else None

    tokens = cfg.B * K * world
    value = tokens / (total_ms / 1e3)
    ms_per_step = total_ms / K

    # ---- dominant kernel alone: the indexer over the same inputs (same launch configuration)
    from compressed_sparse_attention_csa_gb300.accounting import decode_step_work
    work = decode_step_work(cfg)
    scores = torch.empty(cfg.B, cfg.E, device=dev)
    Ki = max(3, min(K, 200))
    evi = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ki)]

    def indexer_call():
        csa.indexer_scores(c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"], scores, kscale=inp.get("kscale"))

    indexer_call()
    g_idx = capture(indexer_call)  # the query-operand prep kernel plus the indexer kernel
    for _ in range(3):
        g_idx.replay()
    for i in range(Ki):
        flush.zero_()
        evi[i][0].record(stream)
        g_idx.replay()
        evi[i][1].record(stream)
    torch.cuda.synchronize(dev)
    idx_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evi) / Ki)
    idx_bytes = work["indexer_bytes"] + cfg.B * cfg.E * 4        # + the fp32 scores the kernel writes
    hbm, bf16, peak_kind = peaks()
    achieved = idx_bytes / (idx_ms / 1e3) / 1e9
    traffic = stage_traffic(args.config)
    roofline = {"bound": "hbm",
                "kernel": "indexer stage: indexer_qprep_kernel + indexer_tc_kernel<%s>" % (
                    "e4m3" if cfg.kidx == "fp8" else "bf16"),
                "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": traffic, "peak_kind": f"{peak_kind} HBM copy bandwidth (burst)",
                "bytes_per_launch": idx_bytes, "launch_us": round(idx_ms * 1e3, 2),
                "step_frac_of_hbm": round(work["bytes"] / (ms_per_step / 1e3) / 1e9 / hbm, 4)}

    # ---- end to end: host buffers, copies inside the timed region
    per_step_in = ["q", "qI", "w", "q_pos", "kv_str", "z_str", "kvI_str", "zI_str", "kv_local"]
    host_in = {k: inp[k].cpu().pin_memory() for k in per_step_in}
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = host_out.numel() * host_out.element_size()
    Ke = max(3, min(K, 500))
    eve = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke)]
    for i in range(Ke):
        flush.zero_()
        eve[i][0].record(stream)
        for k, v in host_in.items():
            inp[k].copy_(v, non_blocking=True)
        step()
        host_out.copy_(out, non_blocking=True)
        eve[i][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in eve) / Ke)
    e2e_val = cfg.B * world / (e2e_ms / 1e3)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, t = oracle_sample(cfg, inp, args.cpu_seqs)
        cpu = {"value": n / t, "unit": "tok/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{n} sequence(s) of this workload, one decode token each (compress, "
                         f"{cfg.E:,}-key indexer, top-{cfg.k}, attention over {cfg.k}+{cfg.W} rows), "
                         f"float64 numpy, {t:.1f} s"}

    if rank == 0:
        line = {"metric": metric, "value": round(value, 1), "unit": "tok/s", "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config_obj, "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": round(e2e_val, 1), "unit": "tok/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": launches, "clocks": clocks}
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
