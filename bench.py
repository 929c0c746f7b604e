#!/usr/bin/env python
"""CSA hot-path benchmark.

Default workload: the fused decode step at 1M-token context: V4-Flash CSA, batch 4,
1,048,576 tokens of context, m = 4 (262,144 compressed entries per sequence), FP8 e4m3
indexer keys with one fp32 scale per entry, bf16 KV, 64 query heads x 512, indexer 64 heads
x 128, top-k 512, window 128.  One step = one decode token for each sequence through
csa_decode_step: compress the completed block, score every visible entry, top-512, sparse
attention with sink.

Other workloads (`--config`): 2 = decode at 64K context (batch 16, bf16 keys); 3 = prefill
chunk (4,096 new queries after 131,072 tokens: compression of the chunk, indexer, top-k and
attention for every query); 5 = CSA2 decoder group at 262,144 tokens (Full-layer indexer
scan, block pool, Reindex rescoring, top-k, four attentions), also timed without the scan.

Timing: the workload is built R times (independent copies, like the caches of R layers) so
that stepping the copies in rotation keeps every step's inputs out of L2.  W warm-up steps,
then K timed steps: CUDA-graph replays of the step's library calls, back to back between one
pair of CUDA events on the launching stream.  `value` uses inputs resident in HBM;
`flushed_step` times one copy's step alone after a 512 MiB L2 flush, one event pair per step;
`e2e` calls the public API eagerly and adds, every step, the pinned-host -> device copy of
the step's inputs (one copy: they sit in one StepInputs buffer) and the device -> host copy
of its output, pipelined on two copy streams beside the previous step's compute (one event
pair around all the steps); `e2e_serial` does the same with the copies and the step in order
on one stream, one event pair a step.  The dominant kernel stage is
timed in the same rotation on its own for the roofline entry.

`--impl reference` times the CPU oracle (oracle/csa_oracle.py, float64 numpy) on a bounded
sample of the same workload on the host cores.  Multi-GPU (torchrun): every rank runs its
own slice of a batch of B x world sequences (sequences are independent; no collective on the
data path), `value` is the units of all ranks over the slowest rank's time.
"""
import argparse
import hashlib
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
L2_BYTES = 129 << 20


def copies_for(touched_bytes):
    """Copies to rotate so that more than twice the L2 of other data passes between two
    steps on the same copy."""
    import math
    return max(2, math.ceil(2 * L2_BYTES / max(touched_bytes, 1)) + 1)
REFERENCE_BUDGET_S = 120.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, choices=[2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14])
    ap.add_argument("--cpu-sample", type=int, default=None,
                    help="oracle sample size (sequences for decode / CSA2, query rows for prefill)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill-chunk leg that the default (1M decode) run adds to its line")
    ap.add_argument("--only", choices=["step", "stage", "indexer"], default=None,
                    help="run only the step or the workload's dominant stage (\"indexer\": the stage of the CSA "
                         "workloads), eagerly (for profiler captures)")
    return ap.parse_args()


def peaks():
    """(HBM GB/s, bf16 TF/s burst, bf16 TF/s sustained, kind) from the measured peaks file."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


_INDEXER_STAGE = (("indexer_qprep_kernel", "indexer_tc_kernel"), ("k_indexer.cu", "csa_ptx.cuh", "csa_internal.h"))
# one query per sequence: the indexer CTAs build the query image themselves (no query-prep launch)
_INDEXER_STAGE_1Q = (("indexer_tc_kernel",), _INDEXER_STAGE[1])
_DENSE_STAGE = (("attn_hca_dec_kernel", "attn_merge_wide_kernel"), ("k_attn.cu", "csa_ptx.cuh", "csa_internal.h"))
# config -> (summary file, kernels of the stage, sources the summary's counters were taken with)
STAGE_PROFILES = {4: ("indexer_tc_e4m3_1M_decode.md",) + _INDEXER_STAGE_1Q,
                  12: ("indexer_tc_e4m3_1M_decode.md",) + _INDEXER_STAGE_1Q,
                  13: ("indexer_tc_mxfp4_1M_decode.md",) + _INDEXER_STAGE_1Q,
                  14: ("indexer_tc_mxfp4_1M_decode.md",) + _INDEXER_STAGE_1Q,
                  2: ("indexer_tc_bf16_64K_decode.md",) + _INDEXER_STAGE_1Q,
                  3: ("indexer_tc_bf16_prefill_4K.md",) + _INDEXER_STAGE,
                  5: ("indexer_tc_bf16_csa2_scan_256K.md",) + _INDEXER_STAGE_1Q,
                  6: ("hca_dense_attn_1M_decode.md",) + _DENSE_STAGE,
                  7: ("hca_dense_attn_prefill_4K.md", ("attn_pf_kernel",), _DENSE_STAGE[1]),
                  9: ("epilogue_norm_rope_prefill_4K.md", ("norm_rope_kernel",),
                      ("k_epilogue.cu", "csa_ptx.cuh", "csa_epi.h")),
                  10: ("fp8kv_attn_1M_decode.md", ("attn_dec_kernel", "attn_merge_wide_kernel"),
                       ("k_attn.cu", "csa_ptx.cuh", "csa_epi.h", "csa_internal.h")),
                  11: ("mxfp4kv_attn_1M_decode.md", ("attn_dec_kernel", "attn_merge_wide_kernel"),
                       ("k_attn.cu", "csa_ptx.cuh", "csa_epi.h", "csa_internal.h"))}


def stage_traffic(config):
    """DRAM bytes per indexer-stage launch from the committed ncu summary, or None.

    The summary carries `traffic-bytes-per-launch <kernel> <bytes>` lines and the sha256 of
    the kernel sources it was taken with; the figure is used only while every stage kernel
    has a line and the sources are unchanged."""
    if config not in STAGE_PROFILES:
        return None
    fname, kernels, sources = STAGE_PROFILES[config]
    path = os.path.join(ROOT, "profiles", fname)
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
    for name in sources:
        with open(os.path.join(src, name), "rb") as f:
            h.update(f.read())
    if sha != h.hexdigest() or any(k not in per for k in kernels):
        return None
    return sum(per[k] for k in kernels)


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


def _host64(x):
    import torch
    return x.cpu().to(torch.float64).numpy() if x.is_floating_point() else x.cpu().numpy()


# ------------------------------------------------------------------ workloads
#
# A workload builds its inputs and buffers and exposes:
#   step()             one pass of the whole hot path over the batch (inputs resident)
#   units              tokens per step (the metric's unit)
#   stage_fn()         the dominant kernel stage alone, with stage_bound / stage_amount
#   staging / e2e_out  the per-step inputs a user copies in (StepInputs) and the output read back
#   oracle(n)          (units, seconds, description) of the CPU oracle on a bounded sample


def staged(csa, inp, keys):
    """Pack a workload's per-step inputs into one StepInputs buffer (one host-to-device copy a
    step) and point the workload's input dict at its views."""
    st = csa.StepInputs({k: inp[k] for k in keys})
    inp.update(st.dev)
    return st


class Decode:
    FP8KV = False   # main-KV entries stored as FP8 entries (576 B)
    MXKV = False    # main-KV entries stored as MXFP4 entries (288 B)

    # the per-step inputs: one StepInputs buffer, copied in every end-to-end step
    E2E_KEYS = ["q", "qI", "w", "q_pos", "kv_str", "z_str", "kvI_str", "zI_str", "kv_local"]

    def __init__(self, cfg, csa, torch, dev, row0, host_only=False):
        from synth import gen
        self.cfg = cfg
        self.units = cfg.B
        self.metric = "CSA decode tok/s @1M ctx" if cfg.N == 1 << 20 else "CSA decode tok/s @64K ctx"
        if self.FP8KV:
            self.metric += ", FP8 main-KV entries"
        if self.MXKV:
            self.metric += ", MXFP4 main-KV entries"
        if cfg.kidx == "mxfp4":
            self.metric += ", MXFP4 indexer keys"
        keys = {"fp8": "FP8 e4m3 indexer keys + fp32 scale",
                "mxfp4": "MXFP4 indexer keys (64 B E2M1 + 4 UE8M0 scales)"}.get(cfg.kidx, "bf16 indexer keys")
        self.workload = (f"V4-Flash CSA decode step, batch {cfg.B} @ {cfg.N:,}-token context "
                         f"({cfg.E:,} entries/seq), " +
                         keys +
                         (", FP8 main-KV entries (448 e4m3 + 64 bf16 dims, 576 B)" if self.FP8KV else
                          ", MXFP4 main-KV entries (E2M1 + e4m3 scale per 16 dims, 288 B)" if self.MXKV else ", bf16 KV") +
                         f", {cfg.H}x{cfg.d} heads, indexer {cfg.HI}x{cfg.dI}, k {cfg.k}, W {cfg.W}")
        self.config_extra = {"batch": cfg.B, "context": cfg.N, "m": cfg.m, "entries_per_seq": cfg.E,
                             "heads": cfg.H, "head_dim": cfg.d, "indexer": f"{cfg.HI}x{cfg.dI}", "top_k": cfg.k,
                             "window": cfg.W,
                             "indexer_keys": {"fp8": "e4m3+fp32 scale", "mxfp4": "MXFP4 E2M1+UE8M0/32"}.get(cfg.kidx, "bf16"),
                             "kv_entries": "FP8 (576 B)" if self.FP8KV else "MXFP4 (288 B)" if self.MXKV else "bf16 (1 KiB)"}
        if host_only:
            return
        self.csa = csa
        inp = gen.make_inputs(cfg, dev, row0=row0)
        self.inp = inp
        self.staging = staged(csa, inp, self.E2E_KEYS)
        self.c = csa.Config(B=cfg.B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
                            act=torch.bfloat16, fp8_keys=cfg.kidx == "fp8", softmax_scale=cfg.softmax_scale,
                            mx_keys=cfg.kidx == "mxfp4")
        self.out = torch.empty(cfg.B, cfg.H, cfg.d, device=dev, dtype=torch.bfloat16)
        self.lse = torch.empty(cfg.B, cfg.H, device=dev)
        self.idx = torch.empty(cfg.B, cfg.k, device=dev, dtype=torch.int32)
        self.scores = torch.empty(cfg.B, cfg.E, device=dev)
        if self.FP8KV:
            self.kv8 = torch.empty(cfg.B, cfg.E, cfg.d + 64, dtype=torch.uint8, device=dev)
            csa.kv_pack_fp8(self.c, inp["kv_comp"], self.kv8)
        if self.MXKV:
            self.kv8 = torch.empty(cfg.B, cfg.E, cfg.d // 2 + cfg.d // 16, dtype=torch.uint8, device=dev)
            csa.kv_pack_mxfp4(self.c, inp["kv_comp"], self.kv8)
        self.args = dict(q_pos=inp["q_pos"], q=inp["q"], qI=inp["qI"], w=inp["w"], sink=inp["sink"],
                         kv_comp=self.kv8 if (self.FP8KV or self.MXKV) else inp["kv_comp"], kI=inp["kI"],
                         kscale=inp.get("kscale"),
                         kv_tail=inp["kv_str"],
                         z_tail=inp["z_str"], kvI_tail=inp["kvI_str"], zI_tail=inp["zI_str"], bias=inp["bias"],
                         biasI=inp["biasI"], kv_local=inp["kv_local"], local_base=inp["local_base"],
                         out=self.out, lse=self.lse, idx_out=self.idx)
        self.call = None   # the step's arguments, marshalled at the first call
        from compressed_sparse_attention_csa_gb300.accounting import decode_step_work
        work = decode_step_work(cfg, kv_entry_bytes=cfg.d - 64 + 128 if self.FP8KV else
                                cfg.d // 2 + cfg.d // 16 if self.MXKV else None)
        self.stage_label = "indexer stage: indexer_tc_kernel<%s> (query image built in each CTA)" % (
            {"fp8": "e4m3", "mxfp4": "mxfp4"}.get(cfg.kidx, "bf16"))
        self.stage_bound = "hbm"
        self.stage_amount = work["indexer_bytes"] + cfg.B * cfg.E * 4   # + the fp32 scores written
        self.step_bytes = work["bytes"]
        self.touched_bytes = work["bytes"] + cfg.B * cfg.E * 4
        self.e2e_out = self.out

    def step(self):
        if self.call is None:
            self.call = self.csa.DecodeStepCall(self.c, fp8kv=self.FP8KV, mxfp4kv=self.MXKV, **self.args)
        self.call()

    def step_bf16(self):
        """The same step with the index scores rounded to BF16 before the selection."""
        if getattr(self, "call16", None) is None:
            self.call16 = self.csa.DecodeStepCall(self.c, fp8kv=self.FP8KV, mxfp4kv=self.MXKV, bf16_scores=True,
                                                  **self.args)
        self.call16()

    def stage_fn(self):
        inp = self.inp
        self.csa.indexer_scores(self.c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"], self.scores,
                                kscale=inp.get("kscale"))

    def oracle(self, n, inp_cpu=None):
        """n sequences of the workload, one decode token each."""
        import numpy as np
        from oracle import csa_oracle as O
        cfg = self.cfg
        n = max(1, n)
        src = inp_cpu if inp_cpu is not None else self.inp
        nb = src["q_pos"].shape[0]
        elapsed = 0.0
        sub = cfg.replace(B=1)
        cache = {}
        for i in range(n):
            b = (i * nb) // n
            if b not in cache:
                # host copies of sequence b's inputs (not timed: the oracle reads host arrays)
                cache = {b: {k: _host64(v if k in ("bias", "biasI", "sink") else v[b:b + 1])
                             for k, v in src.items()}}
            host = dict(cache[b])
            codes = host.pop("kI")
            kscale = host.pop("kscale", None)
            kv_comp = host["kv_comp"][0].copy()
            t0 = time.perf_counter()
            mx = cfg.kidx == "mxfp4"
            if mx:
                kdeq = O.mxfp4_key_decode(codes[0], O.mxfp4_key_unwords(kscale[0].astype(np.uint32)))
            elif kscale is not None:
                kdeq = O.e4m3_decode(codes[0]) * kscale[0][:, None]
            else:
                kdeq = codes[0].astype(np.float64)
            O.decode_step_sequence(sub, host, 0, kv_comp, kdeq, fp8_keys=kscale is not None and not mx, mx_keys=mx,
                                   fp8_kv=self.FP8KV, mxfp4_kv=self.MXKV)
            elapsed += time.perf_counter() - t0
        desc = (f"{n} sequence(s) of this workload, one decode token each (compress, {cfg.E:,}-key indexer, "
                f"top-{cfg.k}, attention over {cfg.k}+{cfg.W} rows), float64 numpy, {elapsed:.1f} s")
        return n, elapsed, desc


class Prefill:
    # the per-step inputs: one StepInputs buffer, copied in every end-to-end step
    E2E_KEYS = ["q", "qI", "w", "q_pos", "kv_str", "z_str", "kvI_str", "zI_str", "kv_local"]

    def __init__(self, cfg, csa, torch, dev, row0, host_only=False):
        from synth import gen
        self.cfg = cfg
        B, T, E = cfg.B, cfg.T, cfg.E
        self.units = B * T
        self.metric = "CSA prefill tok/s (4,096-token chunk @128K ctx)"
        self.workload = (f"V4-Flash CSA prefill chunk: {T:,} new tokens after {cfg.N - T:,} (entries "
                         f"{(cfg.N - T) // cfg.m:,} -> {E:,}), batch {B}, bf16, {cfg.H}x{cfg.d} heads, indexer "
                         f"{cfg.HI}x{cfg.dI}, k {cfg.k}, W {cfg.W}; compression of the chunk, indexer, top-k, "
                         f"attention")
        self.config_extra = {"batch": B, "chunk": T, "context_before": cfg.N - T, "m": cfg.m,
                             "entries_after": E, "heads": cfg.H, "head_dim": cfg.d,
                             "indexer": f"{cfg.HI}x{cfg.dI}", "top_k": cfg.k, "window": cfg.W}
        self.tok0 = cfg.N - T - cfg.m
        self.e0, self.e1 = (cfg.N - T) // cfg.m, cfg.N // cfg.m
        if host_only:
            return
        self.csa = csa
        inp = gen.make_inputs(cfg, dev, row0=row0)
        self.inp = inp
        self.staging = staged(csa, inp, self.E2E_KEYS)
        self.c = csa.Config(B=B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
                            act=torch.bfloat16, fp8_keys=False, softmax_scale=cfg.softmax_scale)
        self.scores = torch.empty(B * T, E, device=dev)
        self.idx = torch.empty(B * T, cfg.k, device=dev, dtype=torch.int32)
        self.out = torch.empty(B, T, cfg.H, cfg.d, device=dev, dtype=torch.bfloat16)
        self.lse = torch.empty(B, T, cfg.H, device=dev)
        from compressed_sparse_attention_csa_gb300.accounting import prefill_work
        work = prefill_work(cfg)
        self.stage_label = "indexer stage: indexer_qprep_kernel + indexer_tc_kernel<bf16>"
        self.stage_bound = "tensor"
        self.stage_amount = work["indexer_flops"]
        self.step_flops = work["flops"]
        self.touched_bytes = work["bytes"] + B * T * E * 4
        self.e2e_out = self.out

    def step(self):
        csa, c, inp = self.csa, self.c, self.inp
        csa.compress_kv(c, inp["kv_str"], inp["z_str"], inp["bias"], self.tok0, self.e0, self.e1, inp["kv_comp"])
        csa.compress_kv(c, inp["kvI_str"], inp["zI_str"], inp["biasI"], self.tok0, self.e0, self.e1, inp["kI"])
        self.stage_fn()
        csa.topk(c, self.scores, self.idx)
        csa.sparse_attn(c, inp["q"], inp["kv_comp"], self.idx, inp["kv_local"], inp["local_base"], inp["q_pos"],
                        inp["sink"], self.out, self.lse)

    def _bf16_buffers(self):
        if getattr(self, "scores16", None) is None:
            import torch
            cfg = self.cfg
            self.scores16 = torch.empty(cfg.B * cfg.T, cfg.E, device=self.scores.device, dtype=torch.bfloat16)
            self.idx16 = torch.empty_like(self.idx)

    def step_bf16(self):
        """The step with the index scores written in BF16 and the selector run on them."""
        csa, c, inp = self.csa, self.c, self.inp
        self._bf16_buffers()
        csa.compress_kv(c, inp["kv_str"], inp["z_str"], inp["bias"], self.tok0, self.e0, self.e1, inp["kv_comp"])
        csa.compress_kv(c, inp["kvI_str"], inp["zI_str"], inp["biasI"], self.tok0, self.e0, self.e1, inp["kI"])
        csa.indexer_scores(c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"],
                           self.scores16.view(self.cfg.B, self.cfg.T, self.cfg.E))
        csa.topk(c, self.scores16, self.idx16)
        csa.sparse_attn(c, inp["q"], inp["kv_comp"], self.idx16, inp["kv_local"], inp["local_base"], inp["q_pos"],
                        inp["sink"], self.out, self.lse)

    def topk_fp32(self):
        self.csa.topk(self.c, self.scores, self.idx)

    def _packed(self):
        if getattr(self, "kv8", None) is None:
            import torch
            cfg, inp = self.cfg, self.inp
            dev = inp["kv_comp"].device
            self.kv8 = torch.empty(cfg.B, cfg.E, cfg.d + 64, dtype=torch.uint8, device=dev)
            self.kv4 = torch.empty(cfg.B, cfg.E, cfg.d // 2 + cfg.d // 16, dtype=torch.uint8, device=dev)
            self.csa.kv_pack_fp8(self.c, inp["kv_comp"], self.kv8)
            self.csa.kv_pack_mxfp4(self.c, inp["kv_comp"], self.kv4)

    def attn_bf16(self):
        inp = self.inp
        self.csa.sparse_attn(self.c, inp["q"], inp["kv_comp"], self.idx, inp["kv_local"], inp["local_base"],
                             inp["q_pos"], inp["sink"], self.out, self.lse)

    def attn_fp8(self):
        inp = self.inp
        self._packed()
        self.csa.sparse_attn_fp8kv(self.c, inp["q"], self.kv8, self.idx, inp["kv_local"], inp["local_base"],
                                   inp["q_pos"], inp["sink"], self.out, self.lse)

    def attn_mxfp4(self):
        inp = self.inp
        self._packed()
        self.csa.sparse_attn_mxfp4kv(self.c, inp["q"], self.kv4, self.idx, inp["kv_local"], inp["local_base"],
                                     inp["q_pos"], inp["sink"], self.out, self.lse)

    def topk_bf16(self):
        self._bf16_buffers()
        self.csa.topk(self.c, self.scores16, self.idx16)

    def stage_fn(self):
        inp = self.inp
        self.csa.indexer_scores(self.c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"],
                                self.scores.view(self.cfg.B, self.cfg.T, self.cfg.E))

    def oracle(self, n, inp_cpu=None):
        """The chunk's compression (charged pro rata) plus n query rows spread over the chunk."""
        from oracle import csa_oracle as O
        cfg = self.cfg
        n = max(1, n)
        src = inp_cpu if inp_cpu is not None else self.inp
        h = {k: _host64(v if k in ("bias", "biasI", "sink", "q_pos") else v[0:1]) for k, v in src.items()}
        kv_comp, kI = h["kv_comp"][0].copy(), h["kI"][0].copy()
        t0 = time.perf_counter()
        kv_comp[self.e0:self.e1] = O.compress_range(h["kv_str"][0], h["z_str"][0], h["bias"], cfg.m, self.e0,
                                                    self.e1, tok0=self.tok0)
        kI[self.e0:self.e1] = O.compress_range(h["kvI_str"][0], h["zI_str"][0], h["biasI"], cfg.m, self.e0,
                                               self.e1, tok0=self.tok0)
        t_comp = time.perf_counter() - t0
        sub = cfg.replace(B=1)
        t_rows = 0.0
        for i in range(n):
            tq = (i * (cfg.T - 1)) // max(n - 1, 1)
            t0 = time.perf_counter()
            O.decode_token(sub, h, 0, tq, kv_comp, kI)
            t_rows += time.perf_counter() - t0
        elapsed = t_rows + t_comp * n / cfg.T
        desc = (f"{n} query row(s) of the chunk (indexer over ~{cfg.E:,} entries, top-{cfg.k}, attention) plus "
                f"{n}/{cfg.T} of the chunk's compression ({t_comp:.1f} s whole), float64 numpy, "
                f"{t_rows:.1f} s of rows")
        return n, elapsed, desc


class Csa2Group:
    N_BLOCKS = 2048

    # the per-step inputs: one StepInputs buffer, copied in every end-to-end step
    E2E_KEYS = ["q", "qI", "w", "qI_full", "w_full", "q_pos", "kv_local"]

    def __init__(self, cfg, csa, torch, dev, row0, host_only=False):
        from synth import gen
        self.cfg = cfg
        B, E = cfg.B, cfg.E
        self.units = B
        self.layers = 1 + cfg.n_reuse
        self.metric = "CSA2 decoder-group tok/s @256K ctx"
        self.workload = (f"V4.1-Flash CSA2 decoder group, batch {B} @ {cfg.N:,} tokens at 1:1 (indexer "
                         f"{cfg.HI}x{cfg.dI} bf16), Full-layer scan -> {self.N_BLOCKS} blocks of 8 -> Reindex "
                         f"rescoring -> top-{cfg.k} -> {self.layers} attentions ({cfg.H}x{cfg.d}, W {cfg.W})")
        self.config_extra = {"batch": B, "context": cfg.N, "m": cfg.m, "indexer": f"{cfg.HI}x{cfg.dI}",
                             "pool_blocks": self.N_BLOCKS, "block": 8, "top_k": cfg.k, "window": cfg.W,
                             "layers": self.layers}
        if host_only:
            return
        self.csa = csa
        inp = gen.make_inputs(cfg, dev, row0=row0)
        self.inp = inp
        self.staging = staged(csa, inp, self.E2E_KEYS)
        self.c = csa.Config(B=B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
                            act=torch.bfloat16, fp8_keys=False, softmax_scale=cfg.softmax_scale)
        P = self.N_BLOCKS * 8
        self.s_full = torch.empty(B, E, device=dev)
        self.pool = torch.empty(B, P, dtype=torch.int32, device=dev)
        self.cnt = torch.empty(B, dtype=torch.int32, device=dev)
        self.s_pool = torch.empty(B, P, device=dev)
        self.idx = torch.empty(B, cfg.k, dtype=torch.int32, device=dev)
        self.outs = torch.empty(self.layers, B, 1, cfg.H, cfg.d, device=dev, dtype=torch.bfloat16)
        from compressed_sparse_attention_csa_gb300.accounting import csa2_group_work
        work = csa2_group_work(cfg, self.N_BLOCKS, 8, self.layers)
        self.work = work
        self.stage_label = "Full-layer scan, indexer stage: indexer_tc_kernel<bf16> (query image built in each CTA)"
        self.stage_bound = "hbm"
        self.stage_amount = work["scan_bytes"] + B * E * 4
        self.step_bytes = work["bytes"]
        self.touched_bytes = work["bytes"] + B * E * 4
        self.e2e_out = self.outs

    def stage_fn(self):
        inp = self.inp
        self.csa.indexer_scores(self.c, inp["qI_full"], inp["w_full"], inp["q_pos"], inp["kI"], self.s_full)

    def step_without_scan(self):
        csa, c, inp = self.csa, self.c, self.inp
        csa.indexer_scores(c, inp["qI"], inp["w"], inp["q_pos"], inp["kI"], self.s_pool, cand=self.pool)
        csa.topk(c, self.s_pool, self.idx, n_valid=self.cnt, cand=self.pool)
        for layer in range(self.layers):
            csa.sparse_attn(c, inp["q"][layer], inp["kv_comp"], self.idx, inp["kv_local"][layer],
                            inp["local_base"], inp["q_pos"], inp["sink"][layer], self.outs[layer])

    def step(self):
        self.stage_fn()
        self.csa.block_pool(self.c, self.s_full, self.pool, self.cnt, n_blocks=self.N_BLOCKS)
        self.step_without_scan()

    def oracle(self, n, inp_cpu=None):
        """n sequences of the group, one token each, all four layers."""
        import numpy as np
        from oracle import csa_oracle as O
        cfg = self.cfg
        n = max(1, n)
        src = inp_cpu if inp_cpu is not None else self.inp
        nb = src["q_pos"].shape[0]
        elapsed = 0.0
        for i in range(n):
            b = (i * nb) // n
            h = {}
            for k, v in src.items():
                if k in ("q", "kv_local"):
                    h[k] = _host64(v[:, b])
                elif k == "sink":
                    h[k] = _host64(v)
                else:
                    h[k] = _host64(v[b])
            t = int(h["q_pos"])
            t0 = time.perf_counter()
            nv = min(t + 1, cfg.E)
            sf = O.indexer_scores(h["qI_full"][0], h["w_full"][0], h["kI"], nv).astype(np.float32)
            pool = O.hier_pool(sf, nv, 8, self.N_BLOCKS)
            sr = O.indexer_scores_subset(h["qI"][0], h["w"][0], h["kI"], pool)
            slots = O.topk(sr.astype(np.float32), pool.size, cfg.k)
            sel = np.where(slots >= 0, pool[np.maximum(slots, 0)], -1)
            for layer in range(self.layers):
                rows = O.gather_rows(h["kv_comp"], sel, h["kv_local"][layer], int(h["local_base"]), t, cfg.W)
                O.sparse_attention(h["q"][layer][0], rows, h["sink"][layer], cfg.softmax_scale)
            elapsed += time.perf_counter() - t0
        desc = (f"{n} sequence(s) of the group, one token each (Full scan over {cfg.E:,} positions, block pool, "
                f"Reindex rescoring, top-{cfg.k}, {self.layers} attentions), float64 numpy, {elapsed:.1f} s")
        return n, elapsed, desc


class HcaDecode:
    """HCA ("Heavily Compressed Attention") decode: one-stream compression of the block the
    token completes, then dense attention over every visible entry plus the window."""

    # the per-step inputs: one StepInputs buffer, copied in every end-to-end step
    E2E_KEYS = ["q", "q_pos", "kv_str", "z_str", "kv_local"]

    def __init__(self, cfg, csa, torch, dev, row0, host_only=False):
        from synth import gen
        self.cfg = cfg
        self.units = cfg.B
        self.metric = "HCA decode tok/s @1M ctx"
        self.workload = (f"V4-Flash HCA decode step, batch {cfg.B} @ {cfg.N:,}-token context (m' {cfg.m}: "
                         f"{cfg.E:,} entries/seq, dense attention), bf16 KV, {cfg.H}x{cfg.d} heads, W {cfg.W}; "
                         f"one-stream compression of the completed block")
        self.config_extra = {"batch": cfg.B, "context": cfg.N, "m": cfg.m, "entries_per_seq": cfg.E,
                             "heads": cfg.H, "head_dim": cfg.d, "window": cfg.W}
        if host_only:
            return
        self.csa = csa
        inp = gen.make_inputs(cfg, dev, row0=row0)
        self.inp = inp
        self.staging = staged(csa, inp, self.E2E_KEYS)
        self.c = csa.Config(B=cfg.B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
                            act=torch.bfloat16, softmax_scale=cfg.softmax_scale)
        self.out = torch.empty(cfg.B, cfg.H, cfg.d, device=dev, dtype=torch.bfloat16)
        self.lse = torch.empty(cfg.B, cfg.H, device=dev)
        self.args = dict(q_pos=inp["q_pos"], q=inp["q"], sink=inp["sink"], kv_comp=inp["kv_comp"],
                         kv_tail=inp["kv_str"], z_tail=inp["z_str"], bias=inp["bias"], kv_local=inp["kv_local"],
                         local_base=inp["local_base"], out=self.out, lse=self.lse)
        self.call = None
        from compressed_sparse_attention_csa_gb300.accounting import hca_decode_work
        work = hca_decode_work(cfg)
        self.stage_label = ("dense attention: attn_hca_dec_kernel (rows split over CTAs, two TMA passes) + "
                            "attn_merge_wide_kernel")
        self.stage_bound = "hbm"
        self.stage_amount = work["attention_bytes"]
        self.step_bytes = work["bytes"]
        self.touched_bytes = work["bytes"]
        self.e2e_out = self.out

    def step(self):
        if self.call is None:
            self.call = self.csa.HcaDecodeStepCall(self.c, **self.args)
        self.call()

    def stage_fn(self):
        inp = self.inp
        self.csa.dense_attn(self.c, inp["q"], inp["kv_comp"], inp["kv_local"], inp["local_base"], inp["q_pos"],
                            inp["sink"], self.out, self.lse)

    def oracle(self, n, inp_cpu=None):
        """n sequences of the workload, one decode token each."""
        from oracle import csa_oracle as O
        cfg = self.cfg
        n = max(1, n)
        src = inp_cpu if inp_cpu is not None else self.inp
        nb = src["q_pos"].shape[0]
        sub = cfg.replace(B=1)
        elapsed, cache = 0.0, {}
        for i in range(n):
            b = (i * nb) // n
            if b not in cache:
                cache = {b: {k: _host64(v if k in ("bias", "sink") else v[b:b + 1]) for k, v in src.items()}}
            host = cache[b]
            kv_comp = host["kv_comp"][0].copy()
            t0 = time.perf_counter()
            O.hca_decode_step_sequence(sub, host, 0, kv_comp)
            elapsed += time.perf_counter() - t0
        desc = (f"{n} sequence(s) of this workload, one decode token each (one-stream compression, dense "
                f"attention over {cfg.E:,}+{cfg.W} rows), float64 numpy, {elapsed:.1f} s")
        return n, elapsed, desc


class HcaPrefill:
    """HCA prefill chunk: one-stream compression of the chunk's new entries, then dense
    attention for every query of the chunk."""

    # the per-step inputs: one StepInputs buffer, copied in every end-to-end step
    E2E_KEYS = ["q", "q_pos", "kv_str", "z_str", "kv_local"]

    def __init__(self, cfg, csa, torch, dev, row0, host_only=False):
        from synth import gen
        self.cfg = cfg
        B, T, E = cfg.B, cfg.T, cfg.E
        self.units = B * T
        self.metric = "HCA prefill tok/s (4,096-token chunk @128K ctx)"
        self.workload = (f"V4-Flash HCA prefill chunk: {T:,} new tokens after {cfg.N - T:,} (m' {cfg.m}: entries "
                         f"{(cfg.N - T) // cfg.m:,} -> {E:,}), batch {B}, bf16, {cfg.H}x{cfg.d} heads, W {cfg.W}; "
                         f"one-stream compression of the chunk, dense attention")
        self.config_extra = {"batch": B, "chunk": T, "context_before": cfg.N - T, "m": cfg.m,
                             "entries_after": E, "heads": cfg.H, "head_dim": cfg.d, "window": cfg.W}
        self.tok0 = cfg.N - T
        self.e0, self.e1 = (cfg.N - T) // cfg.m, cfg.N // cfg.m
        if host_only:
            return
        self.csa = csa
        inp = gen.make_inputs(cfg, dev, row0=row0)
        self.inp = inp
        self.staging = staged(csa, inp, self.E2E_KEYS)
        self.c = csa.Config(B=B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
                            act=torch.bfloat16, softmax_scale=cfg.softmax_scale)
        self.out = torch.empty(B, T, cfg.H, cfg.d, device=dev, dtype=torch.bfloat16)
        self.lse = torch.empty(B, T, cfg.H, device=dev)
        from compressed_sparse_attention_csa_gb300.accounting import hca_prefill_work
        work = hca_prefill_work(cfg)
        self.stage_label = "dense attention: attn_pf_kernel (one CTA per query)"
        self.stage_bound = "tensor"
        self.stage_amount = work["attention_flops"]
        self.step_flops = work["flops"]
        self.touched_bytes = work["bytes"]
        self.e2e_out = self.out

    def step(self):
        csa, c, inp = self.csa, self.c, self.inp
        csa.compress_kv_single(c, inp["kv_str"], inp["z_str"], inp["bias"], self.tok0, self.e0, self.e1,
                               inp["kv_comp"])
        self.stage_fn()

    def stage_fn(self):
        inp = self.inp
        self.csa.dense_attn(self.c, inp["q"], inp["kv_comp"], inp["kv_local"], inp["local_base"], inp["q_pos"],
                            inp["sink"], self.out, self.lse)

    def oracle(self, n, inp_cpu=None):
        """The chunk's compression (charged pro rata) plus n query rows spread over the chunk."""
        from oracle import csa_oracle as O
        cfg = self.cfg
        n = max(1, n)
        src = inp_cpu if inp_cpu is not None else self.inp
        h = {k: _host64(v if k in ("bias", "sink", "q_pos") else v[0:1]) for k, v in src.items()}
        kv_comp = h["kv_comp"][0].copy()
        t0 = time.perf_counter()
        kv_comp[self.e0:self.e1] = O.compress_single_range(h["kv_str"][0], h["z_str"][0], h["bias"], cfg.m,
                                                           self.e0, self.e1, tok0=self.tok0)
        t_comp = time.perf_counter() - t0
        sub = cfg.replace(B=1)
        t_rows = 0.0
        for i in range(n):
            tq = (i * (cfg.T - 1)) // max(n - 1, 1)
            t0 = time.perf_counter()
            O.hca_token(sub, h, 0, tq, kv_comp)
            t_rows += time.perf_counter() - t0
        elapsed = t_rows + t_comp * n / cfg.T
        desc = (f"{n} query row(s) of the chunk (dense attention over ~{cfg.E:,}+{cfg.W} rows) plus {n}/{cfg.T} "
                f"of the chunk's compression ({t_comp:.1f} s whole), float64 numpy, {t_rows:.1f} s of rows")
        return n, elapsed, desc


class Epilogue:
    """Attention prologue / epilogue of the prefill chunk: query RMSNorm + RoPE, the chunk's
    compression fused with RMSNorm + RoPE + cache insert, inverse RoPE + FP8 of the output."""

    # the per-step inputs: one StepInputs buffer, copied in every end-to-end step
    E2E_KEYS = ["q", "o", "q_pos", "kv_str", "z_str"]

    def __init__(self, cfg, csa, torch, dev, row0, host_only=False):
        from synth import gen
        self.cfg = cfg
        B, T = cfg.B, cfg.T
        self.units = B * T
        self.metric = "CSA attention prologue/epilogue tok/s (4,096-token chunk)"
        self.workload = (f"V4-Flash attention prologue/epilogue on a prefill chunk of {T:,} tokens after {cfg.N - T:,}: "
                         f"query RMSNorm + RoPE ({cfg.H}x{cfg.d}, last 64 dims), compression of {T // cfg.m:,} entries "
                         f"fused with RMSNorm + RoPE + cache insert, inverse RoPE + e4m3 of the attention output")
        self.config_extra = {"batch": B, "chunk": T, "heads": cfg.H, "head_dim": cfg.d, "rope_dims": 64,
                             "rope_theta": 10000.0, "m": cfg.m}
        self.tok0 = cfg.N - T - cfg.m
        self.e0, self.e1 = (cfg.N - T) // cfg.m, cfg.N // cfg.m
        if host_only:
            return
        self.csa = csa
        inp = gen.make_inputs(cfg, dev, row0=row0)
        self.inp = inp
        self.staging = staged(csa, inp, self.E2E_KEYS)
        self.c = csa.Config(B=B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
                            act=torch.bfloat16, softmax_scale=cfg.softmax_scale)
        self.nr_q = csa.NormRope(weight=inp["q_norm"], eps=1e-6, rope_dims=64, theta=10000.0)
        self.nr_kv = csa.NormRope(weight=inp["kv_norm"], eps=1e-6, rope_dims=64, theta=10000.0)
        self.q_out = torch.empty_like(inp["q"])
        self.codes = torch.empty(inp["o"].shape, dtype=torch.uint8, device=dev)
        self.scales = torch.empty(B * T, cfg.H, device=dev)
        from compressed_sparse_attention_csa_gb300.accounting import epilogue_work
        work = epilogue_work(cfg)
        self.stage_label = "query RMSNorm + RoPE: norm_rope_kernel<bf16> (one warp per (token, head))"
        self.stage_bound = "hbm"
        self.stage_amount = work["q_bytes"]
        self.step_bytes = work["bytes"]
        self.touched_bytes = work["bytes"]
        self.e2e_out = self.codes

    def step(self):
        csa, c, inp = self.csa, self.c, self.inp
        self.stage_fn()
        csa.compress_kv_norm_rope(c, 2, inp["kv_str"], inp["z_str"], inp["bias"], self.tok0, self.e0, self.e1,
                                  inp["kv_comp"], self.nr_kv)
        csa.inverse_rope_quant(c, inp["o"], inp["q_pos"], self.codes, out_scale=self.scales)

    def stage_fn(self):
        inp = self.inp
        self.csa.norm_rope(self.c, inp["q"], inp["q_pos"], self.nr_q, out=self.q_out)

    def oracle(self, n, inp_cpu=None):
        """n tokens of the chunk (query RMSNorm + RoPE, inverse RoPE + e4m3 of the output) plus
        n/T of the chunk's compression."""
        import numpy as np
        from oracle import csa_oracle as O
        cfg = self.cfg
        n = max(1, n)
        src = inp_cpu if inp_cpu is not None else self.inp
        h = {k: _host64(src[k] if k in ("bias", "q_norm", "kv_norm", "q_pos") else src[k][0:1])
             for k in ["q", "o", "q_pos", "kv_str", "z_str", "bias", "q_norm", "kv_norm"]}
        t0 = time.perf_counter()
        for i in range(self.e0, self.e1):
            e = O.compress_entry(h["kv_str"][0], h["z_str"][0], h["bias"], cfg.m, i, tok0=self.tok0)
            O.norm_rope(e, O.compressed_entry_position(cfg.m, i), h["kv_norm"], 1e-6, 64, 10000.0)
        t_comp = time.perf_counter() - t0
        t_rows = 0.0
        for i in range(n):
            tq = (i * (cfg.T - 1)) // max(n - 1, 1)
            t = int(h["q_pos"][tq])
            t0 = time.perf_counter()
            O.norm_rope(h["q"][0, tq], t, h["q_norm"], 1e-6, 64, 10000.0)
            r = O.inverse_rope(h["o"][0, tq], t, 64, 10000.0)
            O.quantize_rows_e4m3(r.astype(np.float32))
            t_rows += time.perf_counter() - t0
        elapsed = t_rows + t_comp * n / cfg.T
        desc = (f"{n} token(s) of the chunk (query RMSNorm + RoPE over {cfg.H} heads, inverse RoPE + e4m3 of the "
                f"output) plus {n}/{cfg.T} of the chunk's fused compression ({t_comp:.1f} s whole), float64 numpy")
        return n, elapsed, desc


class Fp8KvAttn:
    """The decode attention at 1M over FP8 main-KV entries (576 B: 448 e4m3 + 64 bf16 dims) for a
    fixed selection; the same selection over the bf16 cache is timed beside it."""
    _shared = {}
    FMT = "fp8"

    # the per-step inputs: one StepInputs buffer, copied in every end-to-end step
    E2E_KEYS = ["q", "q_pos", "kv_local", "idx"]

    def __init__(self, cfg, csa, torch, dev, row0, host_only=False):
        from synth import gen
        self.cfg = cfg
        B = cfg.B
        self.units = B
        fp8 = self.FMT == "fp8"
        self.entry_bytes = cfg.d - 64 + 128 if fp8 else cfg.d // 2 + cfg.d // 16
        self.metric = "CSA decode attention tok/s @1M, " + ("FP8" if fp8 else "MXFP4") + " main-KV entries"
        self.workload = (f"CSA sparse attention, batch {B} @ {cfg.N:,} tokens ({cfg.E:,} entries/seq) over "
                         + ("FP8 main-KV entries (448 e4m3 + 64 bf16 dims, 576 B)" if fp8 else
                            "MXFP4 main-KV entries (E2M1 + one e4m3 scale per 16 channels, 288 B)")
                         + f", k {cfg.k} selected + W {cfg.W} window rows, {cfg.H}x{cfg.d} heads, sink")
        self.config_extra = {"batch": B, "context": cfg.N, "entries_per_seq": cfg.E, "top_k": cfg.k, "window": cfg.W,
                             "kv_entry_bytes": self.entry_bytes,
                             "l2": ("the copies stepped in rotation share the cache and differ in their selections: "
                                    "more than twice the L2 of distinct rows between two reads of a row")}
        if host_only:
            return
        self.csa = csa
        # The copies the benchmark rotates through share one cache (1.6 GB at 1M) and differ in
        # their selections, so a step reads rows no recent step read.
        key = (str(dev), row0, self.FMT)
        shared = Fp8KvAttn._shared.get(key)
        self.c = csa.Config(B=B, H=cfg.H, d=cfg.d, HI=cfg.HI, dI=cfg.dI, m=cfg.m, k=cfg.k, W=cfg.W,
                            act=torch.bfloat16, softmax_scale=cfg.softmax_scale)
        if shared is None:
            inp = gen.make_inputs(cfg, dev, row0=row0)
            kv8 = torch.empty(B, cfg.E, self.entry_bytes, dtype=torch.uint8, device=dev)
            (csa.kv_pack_fp8 if fp8 else csa.kv_pack_mxfp4)(self.c, inp["kv_comp"], kv8)
            shared = Fp8KvAttn._shared[key] = {"inp": inp, "kv8": kv8, "draws": 0}
        self.kv8 = shared["kv8"]
        inp = dict(shared["inp"])
        if shared["draws"] > 0:
            inp["idx"] = gen.fp8kv_selection(cfg, dev, row0, shared["draws"])
        shared["draws"] += 1
        self.inp = inp
        self.staging = staged(csa, inp, self.E2E_KEYS)
        self.out = torch.empty(B, 1, cfg.H, cfg.d, device=dev, dtype=torch.bfloat16)
        self.lse = torch.empty(B, 1, cfg.H, device=dev)
        ab = 2
        self.stage_label = ("attn_dec_kernel<16, " + ("FP8" if fp8 else "MXFP4") + " entries> + "
                            "attn_merge_wide_kernel")
        self.stage_bound = "hbm"
        self.stage_amount = B * (cfg.k * self.entry_bytes + cfg.W * cfg.d * ab + 2 * cfg.H * cfg.d * ab + cfg.k * 4)
        self.step_bytes = self.stage_amount
        self.touched_bytes = self.stage_amount
        self.e2e_out = self.out

    def step(self):
        inp = self.inp
        fn = self.csa.sparse_attn_fp8kv if self.FMT == "fp8" else self.csa.sparse_attn_mxfp4kv
        fn(self.c, inp["q"], self.kv8, inp["idx"], inp["kv_local"], inp["local_base"], inp["q_pos"], inp["sink"],
           self.out, self.lse)

    def stage_fn(self):
        self.step()

    def bf16_step(self):
        inp = self.inp
        self.csa.sparse_attn(self.c, inp["q"], inp["kv_comp"], inp["idx"], inp["kv_local"], inp["local_base"],
                             inp["q_pos"], inp["sink"], self.out, self.lse)

    def oracle(self, n, inp_cpu=None):
        """n sequences: the oracle's FP8 encoding of the selected entries, then attention."""
        import numpy as np
        from oracle import csa_oracle as O
        cfg = self.cfg
        n = max(1, n)
        src = inp_cpu if inp_cpu is not None else self.inp
        nb = src["q_pos"].shape[0]
        elapsed = 0.0
        for i in range(n):
            b = (i * nb) // n
            h = {k: _host64(src[k] if k == "sink" else src[k][b:b + 1]) for k in
                 ["q", "kv_local", "local_base", "q_pos", "sink", "idx"]}
            sel = h["idx"][0]
            ent = _host64(src["kv_comp"][b][src["idx"][b].long()])
            t0 = time.perf_counter()
            dec = (O.kv_fp8_decode(O.kv_fp8_encode(ent)) if self.FMT == "fp8"
                   else O.mxfp4_decode(O.mxfp4_encode(ent)))
            cache = {int(x): dec[j] for j, x in enumerate(sel)}
            rows = np.stack([cache[int(x)] for x in sel] + [h["kv_local"][0][p - int(h["local_base"][0])]
                            for p in O.window_positions(int(h["q_pos"][0]), cfg.W, int(h["local_base"][0]),
                                                        h["kv_local"].shape[1])])
            O.sparse_attention(h["q"][0, 0], rows, h["sink"], cfg.softmax_scale)
            elapsed += time.perf_counter() - t0
        desc = (f"{n} sequence(s), one decode token each ({self.FMT} encode/decode of the {cfg.k} selected entries, attention "
                f"over {cfg.k}+{cfg.W} rows), float64 numpy, {elapsed:.2f} s")
        return n, elapsed, desc


class Mxfp4KvAttn(Fp8KvAttn):
    """The decode attention at 1M over MXFP4 main-KV entries (288 B)."""
    _shared = {}
    FMT = "mxfp4"


class Fp8KvDecode(Decode):
    """The decode step over FP8 main-KV entries (V4's production precision with FP8 keys)."""
    FP8KV = True


class Mxfp4KvDecode(Decode):
    """The decode step over MXFP4 main-KV entries with MXFP4 indexer keys (V4.1's storage)."""
    MXKV = True


WORKLOADS = {2: Decode, 4: Decode, 12: Fp8KvDecode, 13: Decode, 14: Mxfp4KvDecode, 3: Prefill, 5: Csa2Group, 6: HcaDecode, 7: HcaPrefill, 9: Epilogue, 10: Fp8KvAttn,
             11: Mxfp4KvAttn}


def config_of(wl):
    """The JSON line's `config` (identical for both arms)."""
    c = dict(workload=wl.workload, l2="inputs larger than L2: independent copies of the workload stepped in rotation",
             timing=("K steps back to back between one pair of CUDA events: every full rotation of the copies "
                     "replayed as one CUDA graph (a step of each copy), the remaining steps one graph each"))
    c.update(wl.config_extra)
    return c
DEFAULT_SAMPLE = {2: 12, 4: 12, 3: 16, 5: 6, 6: 64, 7: 2048, 9: 4096, 10: 400, 11: 400, 12: 12, 13: 12, 14: 12}


def prefill_leg(csa, torch, dev, row0, K, max_over_ranks, world):
    """The other half of the headline metric, measured in the same run: the V4-Flash prefill
    chunk (4,096 new tokens after 131,072) stepped in rotation over independent copies, every
    full rotation one CUDA graph, between one event pair; then its indexer stage (the
    tensor-core GEMM that dominates it) timed alone the same way, against the measured dense
    bf16 peaks."""
    from synth import gen
    cfg = gen.CONFIGS[3]
    w0 = Prefill(cfg, csa, torch, dev, row0)
    R = copies_for(w0.touched_bytes)
    wls = [w0] + [Prefill(cfg, csa, torch, dev, row0) for _ in range(R - 1)]
    for w in wls:
        w.step()
    torch.cuda.synchronize(dev)
    assert csa.get_last_error() == 0
    stream = torch.cuda.current_stream(dev)

    def graphs(fn_name):
        gs = []
        for w in wls:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                getattr(w, fn_name)()
            gs.append(g)
        g_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_all):
            for w in wls:
                getattr(w, fn_name)()
        torch.cuda.synchronize(dev)
        return gs, g_all

    def timed(gs, g_all, n):
        full, rem = divmod(n, len(gs))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(full):
            g_all.replay()
        for i in range(rem):
            gs[i].replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    Kp = max(3 * R, min(K, 200))
    gs, g_all = graphs("step")
    timed(gs, g_all, 3 * R)
    step_ms = max_over_ranks(timed(gs, g_all, Kp) / Kp)
    gs_s, g_all_s = graphs("stage_fn")
    timed(gs_s, g_all_s, 3 * R)
    stage_ms = max_over_ranks(timed(gs_s, g_all_s, Kp) / Kp)
    assert csa.get_last_error() == 0
    # BF16 index scores ("FP4, down to the index scores"): the whole step with the indexer writing
    # BF16 and the selector run on them, the selector alone on fp32 vs BF16 scores of the same
    # rows, and the recall of the BF16 selection against the fp32 one
    for w in wls:
        w.step_bf16()
    gs16, g_all16 = graphs("step_bf16")
    timed(gs16, g_all16, 3 * R)
    step16_ms = max_over_ranks(timed(gs16, g_all16, Kp) / Kp)
    sel = {}
    for name in ("topk_fp32", "topk_bf16"):
        gx, gx_all = graphs(name)
        timed(gx, gx_all, 3 * R)
        sel[name] = max_over_ranks(timed(gx, gx_all, Kp) / Kp)
        del gx, gx_all
    # the chunk's attention over the selected entries stored as bf16 rows, FP8 entries (576 B) and
    # MXFP4 entries (288 B): the same selections, the quantised rows widened in the gather
    for w in wls:
        w.step()
        w.attn_fp8()
        w.attn_mxfp4()
    for name in ("attn_bf16", "attn_fp8", "attn_mxfp4"):
        gx, gx_all = graphs(name)
        timed(gx, gx_all, 3 * R)
        sel[name] = max_over_ranks(timed(gx, gx_all, Kp) / Kp)
        del gx, gx_all
    w0.step()
    w0.step_bf16()
    torch.cuda.synchronize(dev)
    a32, a16 = w0.idx, w0.idx16
    m32 = torch.zeros(a32.shape[0], cfg.E, dtype=torch.bool, device=dev)
    m32.scatter_(1, a32.clamp(min=0).long(), a32 >= 0)
    hits = int(torch.gather(m32, 1, a16.clamp(min=0).long()).logical_and(a16 >= 0).sum())
    recall = hits / max(int((a32 >= 0).sum()), 1)
    assert csa.get_last_error() == 0
    hbm, bf16, bf16_sus, peak_kind = peaks()
    tflops = w0.stage_amount / (stage_ms / 1e3) / 1e12
    out = {"metric": w0.metric, "value": round(w0.units * world / (step_ms / 1e3), 1), "unit": "tok/s",
           "ms_per_step": round(step_ms, 5), "steps": Kp, "step_tflops": round(w0.step_flops / (step_ms / 1e3) / 1e12, 1),
           "config": config_of(w0),
           "roofline": {"bound": "tensor", "kernel": w0.stage_label, "achieved": round(tflops, 1), "peak": bf16,
                        "unit": "TFLOP/s", "frac": round(tflops / bf16, 4), "peak_sustained": bf16_sus,
                        "frac_of_sustained": round(tflops / bf16_sus, 4),
                        "peak_kind": f"{peak_kind} dense bf16 GEMM throughput (burst; sustained beside it)",
                        "amount_per_launch": w0.stage_amount, "launch_us": round(stage_ms * 1e3, 2),
                        "traffic": stage_traffic(3)},
           "bf16_scores": {"value": round(w0.units * world / (step16_ms / 1e3), 1), "ms_per_step": round(step16_ms, 5),
                           "selector_us_fp32": round(sel["topk_fp32"] * 1e3, 2),
                           "selector_us_bf16": round(sel["topk_bf16"] * 1e3, 2),
                           "selector_speedup": round(sel["topk_fp32"] / sel["topk_bf16"], 3),
                           "recall_vs_fp32": round(recall, 5)},
           "entry_formats": {"attention_us_bf16_entries": round(sel["attn_bf16"] * 1e3, 2),
                             "attention_us_fp8_entries": round(sel["attn_fp8"] * 1e3, 2),
                             "attention_us_mxfp4_entries": round(sel["attn_mxfp4"] * 1e3, 2)}}
    del gs, g_all, gs_s, g_all_s, gs16, g_all16, wls, w0
    torch.cuda.empty_cache()
    return out


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
    Wl = WORKLOADS[args.config]
    sample_n = args.cpu_sample if args.cpu_sample is not None else DEFAULT_SAMPLE[args.config]

    if args.impl == "reference":
        # The CPU oracle on the host cores, on this workload's config and metric.
        if rank != 0:
            return
        # One step = the oracle on one sequence (decode, CSA2) or on 4 query rows (prefill).  A
        # float64 numpy step takes seconds, so the run stops after REFERENCE_BUDGET_S of oracle
        # time even if fewer than --steps steps ran; `steps` reports the steps actually timed.
        wl = Wl(cfg, None, torch, "cpu", 0, host_only=True)
        n1 = 4 if args.config in (3, 7) else (256 if args.config == 9 else 1)
        inp = gen.make_inputs(cfg.replace(B=1), "cpu")
        n_total, t_total, desc, done = 0, 0.0, "", 0
        while done < max(args.steps, 1) and (done == 0 or t_total < REFERENCE_BUDGET_S):
            n, t, desc = wl.oracle(n1, inp_cpu=inp)
            n_total += n
            t_total += t
            done += 1
        v = n_total / t_total
        line = {"impl": "reference", "metric": wl.metric, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
                "steps": done, "steps_requested": args.steps, "warmup": 0,
                "ms_per_step": 1e3 * t_total / done,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config_of(wl),
                "cpu_baseline": {"value": v, "unit": "tok/s", "cores": cpu_threads(), "kind": "oracle",
                                 "sample": f"{done} step(s) of {REFERENCE_BUDGET_S:.0f} s oracle budget; "
                                           f"last step: " + desc},
                "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import compressed_sparse_attention_csa_gb300 as csa
    from compressed_sparse_attention_csa_gb300.shard import max_over_ranks, shard_rows
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    # weak scaling: every rank runs its own cfg.B sequences of a batch of cfg.B * world
    row0, n_rows = shard_rows(cfg.B * world, world, rank)
    assert n_rows == cfg.B
    wl = Wl(cfg, csa, torch, dev, row0)
    stream = torch.cuda.current_stream(dev)

    if args.only:
        fn = wl.step if args.only == "step" else wl.stage_fn
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            fn()
        torch.cuda.synchronize(dev)
        assert csa.get_last_error() == 0
        print(json.dumps({"only": args.only, "config": args.config, "calls": args.steps,
                          "ms_per_call_back_to_back": 1e3 * (time.perf_counter() - t0) / max(args.steps, 1)}))
        return

    # Inputs larger than L2: R independent copies of the workload (like the caches of R
    # layers) are stepped in rotation, so the data a step reads was last touched R - 1 steps
    # earlier, with more than twice the L2 of other traffic in between.
    R = copies_for(wl.touched_bytes)
    wls = [wl] + [Wl(cfg, csa, torch, dev, row0) for _ in range(R - 1)]
    for w in wls:
        for _ in range(max(1, args.warmup // R)):
            w.step()
    torch.cuda.synchronize(dev)
    assert csa.get_last_error() == 0

    # Each timed function is captured once per copy into a CUDA graph (the library's launches
    # are stream-ordered and allocate nothing once the workspace exists); the graphs are
    # replayed back to back between one pair of CUDA events, so the host stays ahead of the
    # device and the time is the device's.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize(dev)
        return g

    def time_rotation(gs, n, whole=None):
        """Exactly n steps in rotation over the copies; with `whole` (one graph holding a step of
        every copy, in order) the full rotations replay as one graph each, so the host's graph
        launches keep ahead of a short step the way a serving loop's multi-layer graph does."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        full, rem = divmod(n, len(gs)) if whole is not None else (0, n)
        e0.record(stream)
        for _ in range(full):
            whole.replay()
        for i in range(rem):
            gs[i % len(gs)].replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    def capture_all(fns):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for f in fns:
                f()
        torch.cuda.synchronize(dev)
        return g

    n_cap = csa.launch_count()
    g_steps = [capture(w.step) for w in wls]
    g_all = capture_all([w.step for w in wls])
    launches_per_step = (csa.launch_count() - n_cap) // (2 * R)
    time_rotation(g_steps, max(3, args.warmup))
    g_all.replay()
    assert csa.get_last_error() == 0

    gpu_id = "0"
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(dev.index or 0)
    sampler = ClockSampler(gpu_id) if rank == 0 else None

    K = args.steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    total_ms = time_rotation(g_steps, K, g_all)
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    launches = launches_per_step * K
    assert csa.get_last_error() == 0
    total_ms = max_over_ranks(total_ms)
    clocks = sampler.stop(t_wall0, t_wall1) if sampler else None

    value = wl.units * K * world / (total_ms / 1e3)
    ms_per_step = total_ms / K

    # ---- the same step timed alone: L2 flushed (512 MiB written) before each step, one event
    #      pair per step (includes the device-side cost of starting a graph from idle)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    Kf = max(3, min(K, 500))
    evf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kf)]
    for i in range(Kf):
        flush.zero_()
        evf[i][0].record(stream)
        g_steps[0].replay()
        evf[i][1].record(stream)
    torch.cuda.synchronize(dev)
    flushed_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evf) / Kf)
    del flush

    # ---- dominant kernel stage alone, same inputs and launch configuration, same rotation
    g_stages = [capture(w.stage_fn) for w in wls]
    g_stages_all = capture_all([w.stage_fn for w in wls])
    time_rotation(g_stages, 3 * R, g_stages_all)
    Ki = max(3 * R, min(K, 500))
    stage_ms = max_over_ranks(time_rotation(g_stages, Ki, g_stages_all) / Ki)
    hbm, bf16, bf16_sus, peak_kind = peaks()
    if wl.stage_bound == "hbm":
        achieved = wl.stage_amount / (stage_ms / 1e3) / 1e9
        peak, unit, pk = hbm, "GB/s", f"{peak_kind} HBM copy bandwidth (burst)"
        step_frac = {"step_frac_of_hbm": round(wl.step_bytes / (ms_per_step / 1e3) / 1e9 / hbm, 4)}
    else:
        achieved = wl.stage_amount / (stage_ms / 1e3) / 1e12
        peak, unit, pk = bf16, "TFLOP/s", f"{peak_kind} dense bf16 GEMM throughput (burst)"
        step_frac = {"step_tflops": round(wl.step_flops / (ms_per_step / 1e3) / 1e12, 1),
                     "stage_frac_of_sustained": round(achieved / bf16_sus, 4)}
    roofline = {"bound": wl.stage_bound, "kernel": wl.stage_label, "achieved": round(achieved, 1), "peak": peak,
                "unit": unit, "frac": round(achieved / peak, 4), "traffic": stage_traffic(args.config),
                "peak_kind": pk, "amount_per_launch": wl.stage_amount, "launch_us": round(stage_ms * 1e3, 2)}
    roofline.update(step_frac)

    extra = {"flushed_step": {"ms_per_step": round(flushed_ms, 5),
                              "value": round(wl.units * world / (flushed_ms / 1e3), 1)}}
    if isinstance(wl, Fp8KvAttn):
        g_b = [capture(w.bf16_step) for w in wls]
        g_b_all = capture_all([w.bf16_step for w in wls])
        time_rotation(g_b, 3 * R, g_b_all)
        b_ms = max_over_ranks(time_rotation(g_b, K, g_b_all) / K)
        extra["bf16_entries"] = {"value": round(wl.units * world / (b_ms / 1e3), 1), "ms_per_step": round(b_ms, 5)}
    if isinstance(wl, Decode):
        # the same step with the index scores rounded to BF16 before the selection
        for w in wls:
            w.step_bf16()
        g_16 = [capture(w.step_bf16) for w in wls]
        g_16_all = capture_all([w.step_bf16 for w in wls])
        time_rotation(g_16, 3 * R, g_16_all)
        s16_ms = max_over_ranks(time_rotation(g_16, K, g_16_all) / K)
        extra["bf16_scores"] = {"value": round(wl.units * world / (s16_ms / 1e3), 1), "ms_per_step": round(s16_ms, 5)}
        assert csa.get_last_error() == 0
    if isinstance(wl, Csa2Group):
        g_ns = [capture(w.step_without_scan) for w in wls]
        g_ns_all = capture_all([w.step_without_scan for w in wls])
        time_rotation(g_ns, 3 * R, g_ns_all)
        ns_ms = max_over_ranks(time_rotation(g_ns, K, g_ns_all) / K)
        extra["without_scan"] = {"value": round(wl.units * world / (ns_ms / 1e3), 1), "ms_per_step": round(ns_ms, 5),
                                 "frac_of_hbm": round(wl.work["bytes_without_scan"] / (ns_ms / 1e3) / 1e9 / hbm, 4)}

    # ---- end to end: the public API called eagerly with host buffers.  Every step copies its
    #      inputs in from pinned host memory (the workload's StepInputs mirror: one copy) and its
    #      output back.  Pipelined (`e2e`): the upload of a step runs on a copy stream while the
    #      previous step computes, the read-back on a third stream, each waiting only for what it
    #      overwrites (a copy's inputs once its last step consumed them, its output once read
    #      back); one event pair around all the steps.  Serial (`e2e_serial`): upload, step and
    #      read-back in order on one stream, one event pair per step.
    host_out = torch.empty(wl.e2e_out.shape, dtype=wl.e2e_out.dtype).pin_memory()
    h2d = wl.staging.nbytes
    d2h = host_out.numel() * host_out.element_size()
    Ke = max(3, min(K, 500))
    up_s, dn_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_up = [torch.cuda.Event() for _ in range(R)]
    ev_done = [torch.cuda.Event() for _ in range(R)]
    ev_read = [torch.cuda.Event() for _ in range(R)]

    def pipelined(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up_s.wait_stream(stream)
        dn_s.wait_stream(stream)
        for i in range(n):
            j = i % R
            w = wls[j]
            with torch.cuda.stream(up_s):
                if i >= R:
                    up_s.wait_event(ev_done[j])     # copy j's last step has read its inputs
                w.staging.upload()
                ev_up[j].record(up_s)
            stream.wait_event(ev_up[j])
            if i >= R:
                stream.wait_event(ev_read[j])        # copy j's last output has been read back
            w.step()
            ev_done[j].record(stream)
            with torch.cuda.stream(dn_s):
                dn_s.wait_event(ev_done[j])
                host_out.copy_(w.e2e_out, non_blocking=True)
                ev_read[j].record(dn_s)
        stream.wait_stream(up_s)
        stream.wait_stream(dn_s)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    pipelined(R + 3)
    e2e_ms = max_over_ranks(pipelined(Ke) / Ke)
    assert csa.get_last_error() == 0
    e2e_val = wl.units * world / (e2e_ms / 1e3)
    eve = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke)]
    for i in range(Ke):
        w = wls[i % R]
        eve[i][0].record(stream)
        w.staging.upload()
        w.step()
        host_out.copy_(w.e2e_out, non_blocking=True)
        eve[i][1].record(stream)
    torch.cuda.synchronize(dev)
    assert csa.get_last_error() == 0
    e2es_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in eve) / Ke)
    extra["e2e_serial"] = {"value": round(wl.units * world / (e2es_ms / 1e3), 1), "unit": "tok/s",
                           "ms_per_step": round(e2es_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # ---- the prefill half of the headline metric (the default decode run only)
    prefill = None
    if args.config == 4 and not args.no_prefill:
        prefill = prefill_leg(csa, torch, dev, row0, K, max_over_ranks, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, t, desc = wl.oracle(sample_n)
        cpu = {"value": n / t, "unit": "tok/s", "cores": cpu_threads(), "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {"metric": wl.metric, "value": round(value, 1), "unit": "tok/s", "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config_of(wl),
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": round(e2e_val, 1), "unit": "tok/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                        "copies": "pipelined: a step's upload overlaps the previous step's compute"},
                "gpu_launches": launches, "clocks": clocks}
        line.update(extra)
        if prefill is not None:
            line["prefill"] = prefill
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
