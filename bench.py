#!/usr/bin/env python
"""Benchmark of the PaTH attention library on one GB300 (or N, one process each).

Step = one forward + backward pass of PaTH attention over batch 32, 32 heads, head dim 64,
L = 4096, bf16 inputs (q, k, v, w, dO; beta fp32, 5 % of beta in [1.95, 2)), i.e. every step
of the fwd/bwd hot path.  The decode workload (batch 32, 32 heads, cache 32768 -> 33023 bf16,
256 steps) is measured in the same run and reported under "decode".

Metric: fwd+bwd TFLOP/s with FLOPs counted per head as
  fwd 2 L^2 d + L^2 d^2 / B_fwd,  bwd 5 L^2 d + 2 L^2 d^2 / B_bwd
at the chunk sizes the kernels use (the FlashAttention-convention count, fwd 2 L^2 d + bwd
5 L^2 d, is reported beside it).  Decode: HBM GB/s counting 3 x t x d x 2 bytes per head per step
(read K, write K, read V).

Usage: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from softmax_attention_chunk_gb300.inputs import (BETA_MAX_BELOW_2, CONFIGS, gen_decode_inputs,  # noqa: E402
                                                  gen_path_inputs)

METRIC = "PaTH fwd+bwd TFLOP/s (B32 H32 d64 L4K) vs bf16 peak; decode HBM GB/s"
FWD_CFG = "fig1_fwd_l4096"
DEC_CFG = "decode_b32h32_t32768"
L2_BYTES = 129 * 2**20
WORKLOAD = ("PaTH fwd+bwd, batch 32, 32 heads, d=64, L=4096, bf16 (beta fp32, 5% near-reflection beta), "
            "per rank")
D = 64


# Algorithmic multiply-adds of the per-chunk UT kernels of the bf16 tensor-core path (2 flops
# each): every product is a 64 x 64 x 64 tcgen05 MMA.
UT_PREP64_MMAS = 12  # G, M1, N2, QK^T; M1 U, U N2, U^T W; A W, X^T W, M1 X, W^T Y; P V
UT_BWD64_MMAS = 31   # the diagonal-chunk attention backward and the chain rule through U, X, M1, N2, G
# DRAM bytes per head of one bwd_scan_tc_kernel launch at L = 4096: ncu (dram__bytes_read.sum +
# dram__bytes_write.sum) of a 64-head launch (batch 4 x 16 heads: four head groups, a working set
# above L2) divided by 64 — the kernel takes heads 16 at a time, so a launch over more heads repeats
# that traffic per group.  To be retaken whenever the kernel changes.
BWD_SCAN_DRAM_BYTES_PER_HEAD_L4096 = (1713337088 + 439145472) / 64
# DRAM bytes per head of one decode step at t = 32768 (split + combine kernels): ncu
# (dram__bytes_read.sum + dram__bytes_write.sum) of a batch-4 x 32-head step divided by 128 heads
# (the step's traffic grows in proportion to the heads it processes).  To be retaken whenever the
# kernel changes.
DECODE_DRAM_BYTES_PER_HEAD_T32768 = (1074203392 + 494862592 + 1309440) / 128


def tiles_steps(L):
    """(number of 128-row query tiles, sum over tiles of scan steps) for one head."""
    nt = (L + 127) // 128
    steps = sum(2 * t + (1 if (2 * t + 1) * 64 < L else 0) for t in range(nt))
    return nt, steps


def phase_roofline(L, BH, pk):
    """Per phase of the fwd+bwd step: (algorithmic work per launch, bound, peak, unit); work is
    flops for the tensor-core phases and HBM bytes for the bandwidth-bound one."""
    nc64 = (L + 127) // 128 * 2
    Lp = nc64 * 64
    npairs = nc64 * (nc64 - 1) // 2
    return {
        "fwd_prepare": (2 * BH * nc64 * UT_PREP64_MMAS * 64 ** 3, "tensor", pk["bf16"], "TFLOP/s"),
        "fwd_scan": (BH * npairs * (4 * 64 * 64 * D + 2 * 64 * D * D), "tensor", pk["bf16"], "TFLOP/s"),
        # the forward's preparation and transported queries are reused: the backward prepare phase
        # reads o and dO for D_i (bf16), writes D_i and zeroes the fp32 accumulators dK->, dV, dF
        "bwd_prepare": (BH * (2 * L * D * 2 + Lp * 4 + 2 * Lp * D * 4 + nc64 * D * D * 4), "hbm", pk["hbm"], "GB/s"),
        "bwd_scan": (BH * npairs * (10 * 64 * 64 * D + 4 * 64 * D * D), "tensor", pk["bf16"], "TFLOP/s"),
        "bwd_finish": (2 * BH * nc64 * UT_BWD64_MMAS * 64 ** 3, "tensor", pk["bf16"], "TFLOP/s"),
    }


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-d128", action="store_true", help="skip the head-dim-128 measurements")
    ap.add_argument("--clocks-dir", default=None, help="where to keep the raw nvidia-smi clock samples "
                                                        "(default: the system temporary directory)")
    ap.add_argument("--e2e-steps", type=int, default=30,
                    help="pipelined steps of the end-to-end leg (the first input copy and the last output "
                         "copy are not overlapped: they add about 27 ms / steps to the per-step time)")
    ap.add_argument("--batch", type=int, default=None, help="override the batch (profiling on a smaller case)")
    ap.add_argument("--heads", type=int, default=None, help="override the heads (profiling on a smaller case)")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="override the decode workload's batch (profiling on a smaller case)")
    ap.add_argument("--only", default=None, choices=["train", "decode", "configs", "handoff", "d128",
                                                     "d128_train_small"],
                    help="run one leg alone (profiling): the training step, the decode step, the "
                         "per-workload forward/training legs, the prefill -> decode hand-off, the "
                         "head-dim-128 legs, or a small head-dim-128 training step (batch 1 x 8 heads x "
                         "2048 unless --batch / --heads say otherwise) for profiler captures")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload legs")
    return ap.parse_args()


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def fwd_flops_per_head(L, d, B):
    return 2 * L * L * d + L * L * d * d / B


def bwd_flops_per_head(L, d, B):
    return 5 * L * L * d + 2 * L * L * d * d / B


class Clocks:
    """Samples nvidia-smi clocks and throttle reasons in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, directory=None):
        self.index = index
        self.proc = None
        self.path = os.path.join(directory or tempfile.gettempdir(), f"clocks_{os.getpid()}_{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            # the timed region starts once the sampler has written its first line (its start-up
            # takes about as long as a short timed region)
            t0 = time.time()
            while time.time() - t0 < 3.0 and self.proc.poll() is None and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline_sample(cfg, B_f, B_b, budget_s=15.0, max_heads=16):
    """The fp64 oracle, as it stands, on whole heads of the same workload (fwd + bwd)."""
    from oracle import oracle as orc

    L, d = cfg["seqlen"], cfg["head_dim"]
    flops = 0.0
    t0 = time.perf_counter()
    n = 0
    while n < max_heads and (time.perf_counter() - t0) < budget_s:
        x = gen_path_inputs(**cfg, with_dO=True, heads_subset=[n])
        orc.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, cfg["scale"])
        orc.bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, cfg["scale"], x["dO"])
        flops += fwd_flops_per_head(L, d, B_f) + bwd_flops_per_head(L, d, B_b)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{n} of {cfg['batch'] * cfg['heads']} heads (L={L}, fwd+bwd, fp64, input generation "
                      f"included), {dt:.1f} s"}


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    from oracle import oracle as orc

    cfg = dict(CONFIGS[FWD_CFG])
    B_f, B_b = TC_CHUNK, TC_CHUNK  # the flop count of the tensor-core path (this arm loads only the oracle)
    L, d = cfg["seqlen"], cfg["head_dim"]
    per_step = fwd_flops_per_head(L, d, B_f) + bwd_flops_per_head(L, d, B_b)

    def step(h):
        x = gen_path_inputs(**cfg, with_dO=True, heads_subset=[h])
        orc.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, cfg["scale"])
        orc.bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, cfg["scale"], x["dO"])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps * per_step / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "chunk_fwd": B_f, "chunk_bwd": B_b},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
                             "sample": "one (batch, head) of the B32 H32 L4096 workload per step, fwd+bwd fp64"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# Key chunk of the bf16 tensor-core path at head dim 64 (what path_attn_chunk reports for the
# workloads below); the reference arm counts flops with it without loading the library.
TC_CHUNK = 64


def chunk_sizes():
    from softmax_attention_chunk_gb300 import path_attn as pa

    cfg = CONFIGS[FWD_CFG]
    desc = pa.path_attn_desc_t(cfg["batch"], cfg["heads"], cfg["seqlen"], cfg["head_dim"], pa.PATH_BF16,
                               cfg["scale"], 0)
    return pa.path_attn_chunk(desc, 0), pa.path_attn_chunk(desc, 1)


def ev():
    e = torch.cuda.Event(enable_timing=True)
    e.record()
    return e


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(x, ws):
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if ws == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_config(rank):
    """The training workload of one rank: the same shape on every rank, its own (batch, head)
    problems (weak scaling: the seed moves with the rank)."""
    cfg = dict(CONFIGS[FWD_CFG])
    cfg["seed"] = cfg["seed"] + 7919 * rank
    return cfg


def job_value(flops_per_rank, ms_max, ws):
    """Whole-job TFLOP/s: the work of all ranks over the slowest rank's time."""
    return ws * flops_per_rank / (ms_max * 1e-3) / 1e12


def run_ours(args):
    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    if ws > 1:
        torch.distributed.init_process_group("nccl")
    from softmax_attention_chunk_gb300 import path_attn as pa

    pk = peaks()
    dev = torch.device("cuda", local)
    if args.only == "decode":
        print(json.dumps({"decode": run_decode(args, pa, dev, rank, ws, pk)}), flush=True)
        return
    if args.only == "configs":
        print(json.dumps({"configs": run_configs(args, pa, dev, pk, False)}), flush=True)
        return
    if args.only == "handoff":
        print(json.dumps({"prefill_handoff": run_prefill_handoff(args, pa, dev, pk)}), flush=True)
        return
    if args.only == "d128":
        print(json.dumps({"head_dim_128": run_head_dim_128(args, pa, dev, pk)}), flush=True)
        return
    if args.only == "d128_train_small":
        print(json.dumps({"d128_train_small": run_d128_train_small(args, pa, dev)}), flush=True)
        return
    if args.only == "train":
        args.no_decode = args.no_configs = args.no_cpu_baseline = True
    cfg = rank_config(rank)  # each rank owns its own (batch, head) problems
    if args.batch:
        cfg["batch"] = args.batch
    if args.heads:
        cfg["heads"] = args.heads
    Bt, H, L, d = cfg["batch"], cfg["heads"], cfg["seqlen"], cfg["head_dim"]
    BH = Bt * H
    B_f, B_b = chunk_sizes()

    host = gen_path_inputs(**cfg, with_dO=True)
    host = {k: v.pin_memory() for k, v in host.items() if v is not None}
    x = {k: v.to(dev, non_blocking=True) for k, v in host.items()}
    torch.cuda.synchronize()
    q, k, v, w, beta, dO = (x[n] for n in ("q", "k", "v", "w", "beta", "dO"))
    desc = pa.make_desc(q, cfg["scale"])
    ws_b = pa.workspace(desc, 1, dev)
    o = torch.empty_like(q)
    lse = torch.empty(Bt, H, L, dtype=torch.float32, device=dev)
    grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q), dw=torch.empty_like(q),
                 dbeta=torch.empty_like(beta))

    # Training step: the forward runs in the backward's workspace and stores its transported
    # query tiles (PATH_FWD_STORE_Z); the backward reuses them and the per-chunk preparation
    # (PATH_BWD_Z_FROM_FWD, PATH_BWD_REUSE_FWD), as a training framework keeps forward state.
    bwd_phases = (pa.PATH_BWD_PREPARE | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD, pa.PATH_BWD_SCAN,
                  pa.PATH_BWD_FINISH)

    def step(evs=None):
        marks = [ev()] if evs is not None else None
        pa.fwd(q, k, v, w, beta, None, cfg["scale"], ws=ws_b, out=(o, lse), phases=pa.PATH_FWD_PREPARE)
        if marks is not None: marks.append(ev())
        pa.fwd(q, k, v, w, beta, None, cfg["scale"], ws=ws_b, out=(o, lse),
               phases=pa.PATH_FWD_SCAN | pa.PATH_FWD_STORE_Z)
        if marks is not None: marks.append(ev())
        for ph in bwd_phases:
            pa.bwd(q, k, v, w, beta, o, lse, dO, cfg["scale"], ws=ws_b, out=grads, phases=ph)
            if marks is not None: marks.append(ev())
        if evs is not None:
            evs.append(marks)

    for _ in range(args.warmup):
        step()
    clocks = Clocks(local, args.clocks_dir)
    barrier(ws)
    clocks.start()
    evs = []
    for _ in range(args.steps):
        step(evs)
    barrier(ws)
    clocks_rec = clocks.stop()
    phase_names = ["fwd_prepare", "fwd_scan", "bwd_prepare", "bwd_scan", "bwd_finish"]
    phase_ms = {n: statistics.mean(m[i].elapsed_time(m[i + 1]) for m in evs) for i, n in enumerate(phase_names)}
    total_ms = evs[0][0].elapsed_time(evs[-1][-1])
    total_ms = max_over_ranks(total_ms, ws)
    ms_step = total_ms / args.steps
    flops_step = BH * (fwd_flops_per_head(L, d, B_f) + bwd_flops_per_head(L, d, B_b))
    fa_flops_step = BH * 7 * L * L * d
    value = job_value(flops_step, ms_step, ws)

    # roofline per phase; the dominant phase is reported as "roofline"
    pr = phase_roofline(L, BH, pk)
    phases = {}
    for n, ms in phase_ms.items():
        work, bound, peak, unit = pr[n]
        ach = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
        phases[n] = {"ms": ms, "share": ms / sum(phase_ms.values()), ("flops" if unit == "TFLOP/s" else "bytes"): work,
                     "achieved": ach, "unit": unit, "bound": bound, "peak": peak, "frac": ach / peak}
    dom = max(phase_ms, key=lambda n: phase_ms[n])
    kernels = {"fwd_prepare": "ut_prep64_kernel (tcgen05 UT preparation)",
               "fwd_scan": "fwd_scan_tc_kernel (tcgen05)",
               "bwd_prepare": "bwd_dot_kernel + accumulator memsets (forward preparation and Z tiles reused)",
               "bwd_scan": "bwd_scan_tc_kernel (tcgen05)",
               "bwd_finish": "ut_bwd64_kernel (tcgen05 UT backward)"}
    d = phases[dom]
    traffic = BWD_SCAN_DRAM_BYTES_PER_HEAD_L4096 * BH if (dom == "bwd_scan" and L == 4096) else None
    roofline = {"kernel": f"{dom}: {kernels[dom]}", "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac"], "traffic": traffic,
                "peak_source": (f"bf16 dense ({pk['src']})" if d["bound"] == "tensor" else f"HBM copy ({pk['src']})")}

    # PaTH-FoX training step on the same inputs plus a forget gate (log f = log sigmoid(N(2, 1)),
    # drawn on the device): forward with the forget bias, backward with dlog f
    gf = torch.Generator(device=dev).manual_seed(cfg["seed"] + 17)
    log_f = torch.nn.functional.logsigmoid(torch.randn(beta.shape, device=dev, generator=gf) + 2.0)
    dlog_f = torch.empty_like(log_f)
    fox_out = dict(grads, dlog_f=dlog_f)
    fx = []
    for i in range(args.warmup + args.steps):
        a = ev()
        pa.fwd(q, k, v, w, beta, log_f, cfg["scale"], ws=ws_b, out=(o, lse), phases=pa.PATH_FWD_ALL | pa.PATH_FWD_STORE_Z)
        pa.bwd(q, k, v, w, beta, o, lse, dO, cfg["scale"], ws=ws_b, log_f=log_f, out=fox_out,
               phases=pa.PATH_BWD_ALL | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD)
        b = ev()
        if i >= args.warmup:
            fx.append((a, b))
    torch.cuda.synchronize()
    fox_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in fx), ws)
    ff = []  # the forget-gate forward alone (inference: no transported-query store)
    for i in range(args.warmup + args.steps):
        a = ev()
        pa.fwd(q, k, v, w, beta, log_f, cfg["scale"], ws=ws_b, out=(o, lse))
        b = ev()
        if i >= args.warmup:
            ff.append((a, b))
    torch.cuda.synchronize()
    fox_fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in ff)
    fox_fwd_tf = BH * fwd_flops_per_head(L, cfg["head_dim"], B_f) / (fox_fwd_ms * 1e-3) / 1e12
    fox_train = {"ms_per_step": fox_ms, "tflops": ws * flops_step / (fox_ms * 1e-3) / 1e12,
                 "frac_of_bf16_peak": flops_step / (fox_ms * 1e-3) / 1e12 / pk["bf16"],
                 "forward_ms": fox_fwd_ms, "forward_frac_of_bf16_peak": fox_fwd_tf / pk["bf16"],
                 "note": "PaTH-FoX training step (forget gate; dlog f included), same workload, same flop count; "
                         "forward_ms: the forget-gate inference forward alone"}
    del log_f, dlog_f, fox_out

    # the forward on its own (inference: no transported-query store), against the bf16 peak
    fw = []
    for i in range(args.warmup + args.steps):
        a = ev()
        pa.fwd(q, k, v, w, beta, None, cfg["scale"], ws=ws_b, out=(o, lse))
        b = ev()
        if i >= args.warmup:
            fw.append((a, b))
    torch.cuda.synchronize()
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in fw)
    fwd_tf = BH * fwd_flops_per_head(L, cfg["head_dim"], B_f) / (fwd_ms * 1e-3) / 1e12
    forward = {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_bf16_peak": fwd_tf / pk["bf16"],
               "note": "inference forward (prepare + scan, no Z store), same inputs, after the timed steps"}
    scan_roofline = {n: {"achieved": phases[n]["achieved"], "peak": phases[n]["peak"], "frac": phases[n]["frac"],
                         "unit": "TFLOP/s", "of": "measured bf16 dense"} for n in ("fwd_scan", "bwd_scan")}

    # end-to-end through the public API: every step copies its inputs in from pinned host memory and
    # its outputs and gradients back out.  As in a training loop with a prefetching loader, the next
    # step's input copy and the previous step's output copy run on two copy streams beside the
    # current step (two device buffer sets; events order each copy against the step that uses it).
    outs_h = {"o": torch.empty_like(o, device="cpu").pin_memory(),
              "lse": torch.empty_like(lse, device="cpu").pin_memory()}
    for n, t in grads.items():
        outs_h[n] = torch.empty_like(t, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_h.values())
    xin = [x, {n: torch.empty_like(t) for n, t in x.items()}]
    xout = [dict(o=o, lse=lse, **grads), {n: torch.empty_like(t) for n, t in dict(o=o, lse=lse, **grads).items()}]
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(nsteps):
        """nsteps pipelined steps; returns (start, end) events on the main stream."""
        in_ready = [torch.cuda.Event() for _ in range(nsteps)]
        used = [torch.cuda.Event() for _ in range(nsteps)]     # step done with its buffers
        drained = [torch.cuda.Event() for _ in range(nsteps)]  # outputs of the step copied out
        start = ev()
        s_in.wait_event(start)

        def copy_in(i):
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(used[i - 2])
                for n, t in host.items():
                    xin[i % 2][n].copy_(t, non_blocking=True)
                in_ready[i].record(s_in)

        copy_in(0)
        for i in range(nsteps):
            if i + 1 < nsteps:
                copy_in(i + 1)
            b, X, Y = i % 2, xin[i % 2], xout[i % 2]
            main.wait_event(in_ready[i])
            if i >= 2:
                main.wait_event(drained[i - 2])
            g = {n: Y[n] for n in grads}
            pa.fwd(X["q"], X["k"], X["v"], X["w"], X["beta"], None, cfg["scale"], ws=ws_b, out=(Y["o"], Y["lse"]),
                   phases=pa.PATH_FWD_ALL | pa.PATH_FWD_STORE_Z)
            pa.bwd(X["q"], X["k"], X["v"], X["w"], X["beta"], Y["o"], Y["lse"], X["dO"], cfg["scale"], ws=ws_b,
                   out=g, phases=pa.PATH_BWD_ALL | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD)
            used[i].record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(used[i])
                for n, t in outs_h.items():
                    t.copy_(Y[n], non_blocking=True)
                drained[i].record(s_out)
        main.wait_stream(s_out)
        return start, ev()

    e2e_run(max(2, args.e2e_steps))  # warm-up at the timed depth (the first pass of the pipeline is slower)
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = e2e_run(args.e2e_steps)
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, ws)
    e2e = {"value": ws * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": args.e2e_steps,
           "note": "pipelined: step i+1's input copy and step i-1's output copy run beside step i on two copy "
                   "streams; the first input copy and the last output copy are not overlapped"}
    del ws_b, grads, x, host, outs_h
    torch.cuda.empty_cache()

    confs = None if args.no_configs else run_configs(args, pa, dev, pk, rank == 0 and ws == 1 and
                                                     not args.no_cpu_baseline)
    torch.cuda.empty_cache()
    dec = None if args.no_decode else run_decode(args, pa, dev, rank, ws, pk)
    torch.cuda.empty_cache()
    handoff = None if args.no_decode else run_prefill_handoff(args, pa, dev, pk)
    torch.cuda.empty_cache()
    d128 = None if (args.no_decode or args.no_d128) else run_head_dim_128(args, pa, dev, pk)
    torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(dict(CONFIGS[FWD_CFG]), B_f, B_b)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD if (Bt, H) == (32, 32) else f"{WORKLOAD}; batch {Bt}, {H} heads",
                           "chunk_fwd": B_f, "chunk_bwd": B_b, "flops_per_step": flops_step,
                           "l2": "inputs larger than L2 (6 x 512 MiB per step)"},
                "frac_of_bf16_peak": value / ws / pk["bf16"],
                "fa_convention_tflops": ws * fa_flops_step / (ms_step * 1e-3) / 1e12,
                "phases": phases, "roofline": roofline, "scan_roofline": scan_roofline, "forward": forward,
                "fox_train": fox_train, "e2e": e2e,
                "clocks": clocks_rec, "gpu_launches": 5 * args.steps, "memset_ops": 4 * args.steps,
                "peaks": pk, "decode": dec, "prefill_handoff": handoff, "head_dim_128": d128,
                "configs": confs, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def device_inputs(Bt, H, L, d, gen, near2_frac=0.0, fox=False, with_dO=False):
    """One workload's inputs drawn on the device with the distributions of inputs.py: q, k, v ~
    N(0, 1)/sqrt(d) and w unit (bf16), beta = 2 sigmoid(N(0, 1)) with a fraction near2_frac in
    [1.95, 2) (fp32), log f = log sigmoid(N(2, 1)) (fp32), dO ~ N(0, 1) (bf16)."""
    sd = 1.0 / math.sqrt(d)
    dev = gen.device
    x = {n: (torch.randn(Bt, H, L, d, device=dev, generator=gen) * sd).to(torch.bfloat16) for n in ("q", "k", "v")}
    w = torch.randn(Bt, H, L, d, device=dev, generator=gen)
    x["w"] = (w / w.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    beta = 2.0 * torch.sigmoid(torch.randn(Bt, H, L, device=dev, generator=gen))
    if near2_frac > 0:
        m = torch.rand(Bt, H, L, device=dev, generator=gen) < near2_frac
        beta = torch.where(m, 1.95 + 0.05 * torch.rand(Bt, H, L, device=dev, generator=gen), beta)
    x["beta"] = beta.clamp(max=BETA_MAX_BELOW_2).contiguous()
    x["log_f"] = (torch.nn.functional.logsigmoid(torch.randn(Bt, H, L, device=dev, generator=gen) + 2.0)
                  if fox else None)
    x["dO"] = torch.randn(Bt, H, L, d, device=dev, generator=gen).to(torch.bfloat16) if with_dO else None
    return x


def time_events(fn, warmup, reps):
    """Mean ms of fn over reps calls after warmup calls (CUDA events on the current stream)."""
    for _ in range(warmup):
        fn()
    marks = [ev()]
    for _ in range(reps):
        fn()
        marks.append(ev())
    torch.cuda.synchronize()
    return statistics.mean(marks[i].elapsed_time(marks[i + 1]) for i in range(reps))


def oracle_rate(fn, work_per_call, budget_s, max_calls):
    """(work per second, calls, seconds) of fn run on the host cores until budget_s or max_calls."""
    t0 = time.perf_counter()
    n = 0
    while n < max_calls and (n == 0 or time.perf_counter() - t0 < budget_s):
        fn(n)
        n += 1
    dt = time.perf_counter() - t0
    return work_per_call * n / dt, n, dt


def run_configs(args, pa, dev, pk, with_cpu):
    """The other workloads, one leg each, with inputs drawn on the device (same distributions as
    the parity tests' CPU generator): the inference forward at batch 32 x 32 heads, L 2048 and
    4096; the training step at batch 8 x 16 heads, L 4096; the PaTH-FoX inference forward at
    batch 1 x 32 heads, L 16384; the fp32 tiny forward (batch 1 x 2 heads, L 128).  Each reports
    ms, TFLOP/s (per-head flops of the metric, chunk 64) against the bf16 peak and tokens/s; with
    with_cpu also the oracle timed on whole heads of the same shape on the host cores, in the same
    unit."""
    from oracle import oracle as orc

    g = torch.Generator(device=dev).manual_seed(9001)
    reps = max(3, args.steps)
    out = {}
    ffl = lambda L: fwd_flops_per_head(L, D, TC_CHUNK)
    bfl = lambda L: bwd_flops_per_head(L, D, TC_CHUNK)

    def cpu_fwd(Bt, H, L, fox, near2, flops_head, bwd=False):
        if not with_cpu:
            return None
        seeds = dict(seed=4242, batch=Bt, heads=H, seqlen=L, head_dim=D, dtype="bf16", near2_frac=near2, fox=fox)

        def one(n):
            x = gen_path_inputs(**seeds, with_dO=bwd, heads_subset=[n])
            orc.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], 1.0)
            if bwd:
                orc.bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], 1.0, x["dO"])
        rate, n, dt = oracle_rate(one, flops_head, 4.0, 8)
        return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
                "sample": f"{n} whole head(s) of this shape, {'fwd+bwd' if bwd else 'fwd'} fp64 (input generation "
                          f"included), {dt:.1f} s"}

    for name, (Bt, H, L, near2) in {"fig1_fwd_l2048": (32, 32, 2048, 0.05),
                                     "fig1_fwd_l4096": (32, 32, 4096, 0.05)}.items():
        x = device_inputs(Bt, H, L, D, g, near2_frac=near2)
        desc = pa.make_desc(x["q"], 1.0)
        wsf = pa.workspace(desc, 0, dev)
        o, lse = torch.empty_like(x["q"]), torch.empty(Bt, H, L, device=dev)
        ms = time_events(lambda: pa.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, 1.0, ws=wsf,
                                        out=(o, lse)), args.warmup, reps)
        tf = Bt * H * ffl(L) / (ms * 1e-3) / 1e12
        out[name] = {"workload": f"inference forward, batch {Bt}, {H} heads, d=64, L={L}, bf16, 5% near-reflection "
                                 "beta", "ms": ms, "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16"],
                     "tokens_per_s": Bt * L / (ms * 1e-3),
                     "fa_convention_tflops": Bt * H * 2 * L * L * D / (ms * 1e-3) / 1e12,
                     "cpu_oracle": cpu_fwd(Bt, H, L, False, near2, ffl(L))}
        del x, wsf, o, lse
        torch.cuda.empty_cache()

    # training step, batch 8 x 16 heads, L 4096 (the bench's reuse path)
    Bt, H, L = 8, 16, 4096
    x = device_inputs(Bt, H, L, D, g, with_dO=True)
    desc = pa.make_desc(x["q"], 1.0)
    wsb = pa.workspace(desc, 1, dev)
    o, lse = torch.empty_like(x["q"]), torch.empty(Bt, H, L, device=dev)
    gr = dict(dq=torch.empty_like(o), dk=torch.empty_like(o), dv=torch.empty_like(o), dw=torch.empty_like(o),
              dbeta=torch.empty_like(x["beta"]))

    def train():
        a = (x["q"], x["k"], x["v"], x["w"], x["beta"])
        pa.fwd(*a, None, 1.0, ws=wsb, out=(o, lse), phases=pa.PATH_FWD_ALL | pa.PATH_FWD_STORE_Z)
        pa.bwd(*a, o, lse, x["dO"], 1.0, ws=wsb, out=gr,
               phases=pa.PATH_BWD_ALL | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD)
    ms = time_events(train, args.warmup, reps)
    fl = Bt * H * (ffl(L) + bfl(L))
    out["train_b8h16_l4096"] = {"workload": "training step (fwd storing Z + bwd reusing it), batch 8, 16 heads, d=64, "
                                            "L=4096, bf16", "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                                "frac_of_bf16_peak": fl / (ms * 1e-3) / 1e12 / pk["bf16"],
                                "tokens_per_s": Bt * L / (ms * 1e-3),
                                "cpu_oracle": cpu_fwd(Bt, H, L, False, 0.0, ffl(L) + bfl(L), bwd=True)}
    del x, wsb, o, lse, gr
    torch.cuda.empty_cache()

    # PaTH-FoX inference forward, batch 1 x 32 heads, L 16384
    Bt, H, L = 1, 32, 16384
    x = device_inputs(Bt, H, L, D, g, fox=True)
    desc = pa.make_desc(x["q"], 1.0)
    wsf = pa.workspace(desc, 0, dev)
    o, lse = torch.empty_like(x["q"]), torch.empty(Bt, H, L, device=dev)
    ms = time_events(lambda: pa.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], 1.0, ws=wsf,
                                    out=(o, lse)), args.warmup, reps)
    tf = Bt * H * ffl(L) / (ms * 1e-3) / 1e12
    out["fox_long_l16384"] = {"workload": "PaTH-FoX inference forward, batch 1, 32 heads, d=64, L=16384, bf16",
                              "ms": ms, "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16"],
                              "tokens_per_s": Bt * L / (ms * 1e-3),
                              "cpu_oracle": cpu_fwd(Bt, H, L, True, 0.0, ffl(L))}
    del x, wsf, o, lse
    torch.cuda.empty_cache()

    # fp32 tiny forward (the 1e-4 mode), batch 1 x 2 heads, L 128: launch bound
    Bt, H, L = 1, 2, 128
    x = {n: (t.float() if t is not None and t.dtype == torch.bfloat16 else t)
         for n, t in device_inputs(Bt, H, L, D, g).items()}
    desc = pa.make_desc(x["q"], 1.0)
    wsf = pa.workspace(desc, 0, dev)
    o, lse = torch.empty_like(x["q"]), torch.empty(Bt, H, L, device=dev)
    ms = time_events(lambda: pa.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, 1.0, ws=wsf, out=(o, lse)),
                     args.warmup, 20)
    out["pr1_tiny_fwd"] = {"workload": "forward, batch 1, 2 heads, d=64, L=128, fp32 CUDA-core kernels", "ms": ms,
                           "tokens_per_s": Bt * L / (ms * 1e-3), "bound": "launch latency (two small launches)"}
    del x, wsf, o, lse
    torch.cuda.empty_cache()
    out["cp_fox_l16384_4shards"] = run_cp(args, pa, g, pk)
    return out


def run_cp(args, pa, g, pk):
    """Context-parallel forward of the PaTH-FoX long sequence (batch 1 x 32 heads, L 16384, bf16) cut
    into 4 shards of 4096, the ranks emulated on this one GPU (the chain's schedule and C-ABI
    calls, messages as device copies, no collective): the whole chain (every shard's preparation,
    the 6 block merges and 3 block passes, every shard's scan) against the single-device forward
    of the same sequence, and the time of each kind of shard operation (one instrumented run)."""
    from softmax_attention_chunk_gb300.context_parallel import ShardOps, emulate_ring

    Bt, H, L, world = 1, 32, 16384, 4
    Ls = L // world
    x = device_inputs(Bt, H, L, D, g, fox=True)
    sh = [{n: (None if t is None else t[:, :, r * Ls:(r + 1) * Ls].contiguous()) for n, t in x.items() if n != "dO"}
          for r in range(world)]

    def chain():
        ops = [ShardOps(s["q"], s["k"], s["v"], s["w"], s["beta"], s["log_f"], 1.0) for s in sh]
        return emulate_ring(ops)

    reps = max(3, args.steps)
    ms = time_events(chain, args.warmup, reps)
    desc = pa.make_desc(x["q"], 1.0)
    wsf = pa.workspace(desc, 0, g.device)
    o, lse = torch.empty_like(x["q"]), torch.empty(Bt, H, L, device=g.device)
    ms1 = time_events(lambda: pa.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], 1.0, ws=wsf,
                                     out=(o, lse)), args.warmup, reps)
    # one instrumented chain: events around each kind of operation
    parts = {"prepare": 0.0, "merge_block": 0.0, "pass_block": 0.0, "scan": 0.0}

    def timed(kind, fn):
        a = ev()
        r = fn()
        b = ev()
        torch.cuda.synchronize()
        parts[kind] += a.elapsed_time(b)
        return r

    ops = [timed("prepare", lambda s=s: ShardOps(s["q"], s["k"], s["v"], s["w"], s["beta"], s["log_f"], 1.0))
           for s in sh]
    held = [op.own_block() for op in ops]
    from softmax_attention_chunk_gb300.context_parallel import step_roles
    for st in range(1, world):
        sent = [held[r] if step_roles(r, world, st)[0] else None for r in range(world)]
        for r in range(world):
            if step_roles(r, world, st)[1]:
                got = {k: (None if t is None else t.clone()) for k, t in sent[r - 1].items()}
                timed("merge_block", lambda: ops[r].attend(got))
                held[r] = timed("pass_block", lambda: ops[r].pass_block(got)) if r <= world - 2 else None
    res = [timed("scan", op.finish) for op in ops]
    err = max((torch.cat([q[0] for q in res], dim=2).float() - o.float()).abs().max().item(),
              (torch.cat([q[1] for q in res], dim=2) - lse).abs().max().item())
    fl = Bt * H * fwd_flops_per_head(L, D, TC_CHUNK)
    return {"workload": f"context-parallel PaTH-FoX forward, batch {Bt}, {H} heads, d=64, L={L} bf16, {world} shards "
                        f"of {Ls} emulated on one GPU (no collectives)",
            "ms": ms, "single_device_fwd_ms": ms1, "work_ratio": ms / ms1,
            "tflops_at_the_forward_flop_count": fl / (ms * 1e-3) / 1e12, "parts_ms": parts,
            "max_abs_diff_vs_single_device": err}


def run_decode(args, pa, dev, rank, ws, pk):
    cfg = dict(CONFIGS[DEC_CFG])
    cfg["seed"] += 7919 * rank
    if args.decode_batch:
        cfg["batch"] = args.decode_batch
    Bt, H, d, t0 = cfg["batch"], cfg["heads"], cfg["head_dim"], cfg["t0"]
    steps = args.decode_steps
    di = gen_decode_inputs(**{**cfg, "steps": steps})
    kc0 = di["k_cache"].to(dev)
    vc0 = di["v_cache"].to(dev)
    kc, vc = kc0.clone(), vc0.clone()
    sx = {n: di[n].to(dev) for n in ("q", "k", "v", "w", "beta")}
    del di
    desc = pa.make_decode_desc(kc, cfg["scale"])
    wsd = pa.decode_workspace(desc, dev)
    o = torch.empty(Bt, H, d, dtype=kc.dtype, device=dev)
    for s in range(3):  # warm-up on the copy, then restore the pristine cache
        pa.decode_step(kc, vc, t0 + s, *(sx[n][s] for n in ("q", "k", "v", "w", "beta")), scale=cfg["scale"],
                       ws=wsd, out=o)
    kc.copy_(kc0)
    vc.copy_(vc0)
    clocks = Clocks(dev.index, args.clocks_dir)
    barrier(ws)
    clocks.start()
    marks = [ev()]
    for s in range(steps):
        pa.decode_step(kc, vc, t0 + s, *(sx[n][s] for n in ("q", "k", "v", "w", "beta")), scale=cfg["scale"],
                       ws=wsd, out=o)
        marks.append(ev())
    barrier(ws)
    crec = clocks.stop()
    per = [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
    total_ms = max_over_ranks(sum(per), ws)
    nbytes = sum(Bt * H * 3 * (t0 + s) * d * 2 for s in range(steps))
    gbs = ws * nbytes / (total_ms * 1e-3) / 1e9

    # PaTH-FoX decode on the same cache: forget-gate prefix sums of the cached rows and a log f per
    # step (drawn on the device: log sigmoid(N(2, 1))), restored cache, same steps
    kc.copy_(kc0)
    vc.copy_(vc0)
    g = torch.Generator(device=dev).manual_seed(cfg["seed"] + 13)
    logf = lambda *shape: torch.nn.functional.logsigmoid(torch.randn(*shape, device=dev, generator=g) + 2.0)
    ac = torch.zeros(Bt, H, kc.shape[2], device=dev)
    ac[:, :, :t0] = torch.cumsum(logf(Bt, H, t0).double(), dim=2).float()
    lf = logf(steps, Bt, H)
    torch.cuda.synchronize()
    fmarks = [ev()]
    for s in range(steps):
        pa.decode_step_fox(kc, vc, ac, t0 + s, *(sx[n][s] for n in ("q", "k", "v", "w", "beta")), lf[s],
                           scale=cfg["scale"], ws=wsd, out=o)
        fmarks.append(ev())
    torch.cuda.synchronize()
    fox_ms = max_over_ranks(sum(fmarks[i].elapsed_time(fmarks[i + 1]) for i in range(steps)), ws)
    fox_bytes = nbytes + sum(Bt * H * (t0 + s) * 4 for s in range(steps))  # + the prefix cache
    fox_gbs = ws * fox_bytes / (fox_ms * 1e-3) / 1e9
    traffic = (DECODE_DRAM_BYTES_PER_HEAD_T32768 * Bt * H
               if DECODE_DRAM_BYTES_PER_HEAD_T32768 is not None and t0 == 32768 else None)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        from oracle import oracle as orc

        sub = gen_decode_inputs(**{**cfg, "steps": 8}, heads_subset=[0, 1])
        kref = sub["k_cache"].double().numpy().copy()
        vref = sub["v_cache"].double().numpy().copy()

        def one(s):
            orc.decode_step(kref, vref, t0 + s, *(sub[n][s] for n in ("q", "k", "v", "w", "beta")), cfg["scale"])
        rate, n, dt = oracle_rate(one, 2 * 3 * t0 * d * 2, 4.0, 8)
        cpu = {"value": rate / 1e9, "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
               "sample": f"{n} decode steps of 2 heads at t = {t0}..{t0 + n - 1} (fp64 caches; bytes counted as the "
                         f"GPU's 3 t d 2 per head), {dt:.1f} s"}
    return {"value": gbs, "unit": "GB/s", "tokens_per_s": ws * Bt * steps / (total_ms * 1e-3),
            "ms_per_step": total_ms / steps, "steps": steps, "frac_of_hbm": gbs / ws / pk["hbm"],
            "roofline": {"kernel": "decode step (split + combine)", "bound": "hbm", "achieved": gbs / ws,
                         "peak": pk["hbm"], "unit": "GB/s", "frac": gbs / ws / pk["hbm"], "traffic": traffic,
                         "traffic_note": "DRAM bytes of one step at t = 32768 (decode_split_kernel + "
                                         "decode_combine_kernel), scaled by heads from an ncu capture of a "
                                         "4-batch step"},
            "cpu_oracle": cpu,
            "clocks": crec, "gpu_launches": 2 * steps,
            "workload": f"decode, batch {Bt}, {H} heads, d=64, cache {t0} -> {t0 + steps - 1} bf16, {steps} steps",
            "fox": {"value": fox_gbs, "unit": "GB/s", "ms_per_step": fox_ms / steps,
                    "frac_of_hbm": fox_gbs / ws / pk["hbm"], "gpu_launches": 2 * steps,
                    "workload": "PaTH-FoX decode, same cache and steps, forget-gate prefix sums beside the cache"}}


def run_prefill_handoff(args, pa, dev, pk):
    """Prefill -> decode hand-off of a prompt as long as the decode workload's cache (batch 32,
    32 heads, 32768 tokens, bf16), inputs drawn on the device; CUDA events around the call."""
    cfg = dict(CONFIGS[DEC_CFG])
    if args.decode_batch:
        cfg["batch"] = args.decode_batch
    Bt, H, d, L = cfg["batch"], cfg["heads"], cfg["head_dim"], cfg["t0"]
    g = torch.Generator(device=dev).manual_seed(cfg["seed"] + 11)
    sd = 1.0 / math.sqrt(d)
    k = (torch.randn(Bt, H, L, d, device=dev, generator=g) * sd).to(torch.bfloat16)
    v = (torch.randn(Bt, H, L, d, device=dev, generator=g) * sd).to(torch.bfloat16)
    w = torch.randn(Bt, H, L, d, device=dev, generator=g)
    w = (w / w.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    beta = 2.0 * torch.sigmoid(torch.randn(Bt, H, L, device=dev, generator=g))
    kc = torch.empty(Bt, H, L + 256, d, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    desc = pa.make_decode_desc(kc, cfg["scale"])
    wsp = torch.empty(pa.path_decode_prefill_workspace_size(desc, L), dtype=torch.uint8, device=dev)
    for _ in range(2):
        pa.decode_prefill(kc, vc, k, v, w, beta, ws=wsp)
    reps = 3
    marks = [ev()]
    for _ in range(reps):
        pa.decode_prefill(kc, vc, k, v, w, beta, ws=wsp)
        marks.append(ev())
    torch.cuda.synchronize()
    ms = statistics.mean(marks[i].elapsed_time(marks[i + 1]) for i in range(reps))
    # compulsory HBM bytes: read k, v, w (bf16) and beta, write both cache slabs
    nbytes = Bt * H * L * (3 * d * 2 + 4 + 2 * d * 2)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "tokens_per_s": Bt * L / (ms * 1e-3), "compulsory_bytes": nbytes, "achieved_gbs": gbs,
            "frac_of_hbm": gbs / pk["hbm"],
            "bound": "latency: the per-chunk tcgen05 UT preparation (split F from split bf16 products) and the "
                     "per-head tcgen05 suffix walk (one CTA per head, chunks right to left)",
            "gpu_launches": 2,
            "workload": f"prefill -> decode hand-off, batch {Bt}, {H} heads, d={d}, prompt {L} bf16"}


def run_head_dim_128(args, pa, dev, pk):
    """Head dim 128: the decode step (batch 32, 32 heads, bf16 cache of 32768 entries, 32 steps;
    HBM bound, against the copy peak); the bf16 forward on the head-dim-128 tensor-core kernels
    (batch 4 x 16 heads x 2048 and batch 16 x 32 heads x 4096; TFLOP/s at chunk 64 against the bf16
    peak); a training step (batch 4, 16 heads, L 2048, bf16 inputs): that forward plus the backward
    on the fp32 CUDA-core kernels (32-row chunks), the backward also timed alone against the FP32
    FMA peak 152 SMs x 128 lanes x 2 flop x the maximum SM clock.  Inputs drawn on the device."""
    g = torch.Generator(device=dev).manual_seed(4242)
    sd = 1.0 / math.sqrt(128)
    # ---- decode ----
    Bt, H, d, t0, steps = 32, 32, 128, 32768, 32
    kc = (torch.randn(Bt, H, t0 + steps, d, device=dev, generator=g) * sd).to(torch.bfloat16)
    vc = (torch.randn(Bt, H, t0 + steps, d, device=dev, generator=g) * sd).to(torch.bfloat16)

    def unit(*shape):
        x = torch.randn(*shape, device=dev, generator=g)
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    sx = {"q": (torch.randn(steps, Bt, H, d, device=dev, generator=g) * sd).to(torch.bfloat16),
          "k": (torch.randn(steps, Bt, H, d, device=dev, generator=g) * sd).to(torch.bfloat16),
          "v": (torch.randn(steps, Bt, H, d, device=dev, generator=g) * sd).to(torch.bfloat16),
          "w": unit(steps, Bt, H, d),
          "beta": 2.0 * torch.sigmoid(torch.randn(steps, Bt, H, device=dev, generator=g))}
    desc = pa.make_decode_desc(kc, 1.0)
    wsd = pa.decode_workspace(desc, dev)
    o = torch.empty(Bt, H, d, dtype=torch.bfloat16, device=dev)
    for s in range(3):  # warm-up on scratch positions, then the timed steps from t0
        pa.decode_step(kc, vc, t0 - 3 + s, *(sx[n][s] for n in ("q", "k", "v", "w", "beta")), ws=wsd, out=o)
    torch.cuda.synchronize()
    marks = [ev()]
    for s in range(steps):
        pa.decode_step(kc, vc, t0 + s, *(sx[n][s] for n in ("q", "k", "v", "w", "beta")), ws=wsd, out=o)
        marks.append(ev())
    torch.cuda.synchronize()
    dms = sum(marks[i].elapsed_time(marks[i + 1]) for i in range(steps))
    nbytes = sum(Bt * H * 3 * (t0 + s) * d * 2 for s in range(steps))
    dgbs = nbytes / (dms * 1e-3) / 1e9
    decode = {"value": dgbs, "unit": "GB/s", "ms_per_step": dms / steps, "frac_of_hbm": dgbs / pk["hbm"],
              "tokens_per_s": Bt * steps / (dms * 1e-3), "gpu_launches": 2 * steps,
              "workload": "decode, batch 32, 32 heads, d=128, cache 32768 -> 32799 bf16, 32 steps"}
    del kc, vc, sx
    torch.cuda.empty_cache()
    # ---- forward on the tensor cores ----
    fwd = {}
    for Bt, H, L in ((4, 16, 2048), (16, 32, 4096)):
        x = {n: (torch.randn(Bt, H, L, d, device=dev, generator=g) * sd).to(torch.bfloat16) for n in ("q", "k", "v")}
        x["w"] = unit(Bt, H, L, d)
        x["beta"] = 2.0 * torch.sigmoid(torch.randn(Bt, H, L, device=dev, generator=g))
        dsc = pa.make_desc(x["q"], 1.0)
        wsf = pa.workspace(dsc, 0, dev)
        o2, lse = torch.empty_like(x["q"]), torch.empty(Bt, H, L, device=dev)
        ms = time_events(lambda: pa.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, 1.0, ws=wsf, out=(o2, lse)),
                         args.warmup, max(3, args.steps))
        tf = Bt * H * fwd_flops_per_head(L, d, TC_CHUNK) / (ms * 1e-3) / 1e12
        fwd[f"b{Bt}h{H}_l{L}"] = {"ms": ms, "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16"],
                                  "tokens_per_s": Bt * L / (ms * 1e-3), "gpu_launches": 2,
                                  "workload": f"inference forward, batch {Bt}, {H} heads, d=128, L={L}, bf16, "
                                              "tcgen05 (chunk 64)"}
        del x, wsf, o2, lse
        torch.cuda.empty_cache()
    # ---- training step (tcgen05 forward; backward on TF32 warp MMAs with fp32 accumulation) ----
    Bt, H, L, B = 4, 16, 2048, 32
    x = {n: (torch.randn(Bt, H, L, d, device=dev, generator=g) * sd).to(torch.bfloat16) for n in ("q", "k", "v")}
    x["w"] = unit(Bt, H, L, d)
    x["beta"] = 2.0 * torch.sigmoid(torch.randn(Bt, H, L, device=dev, generator=g))
    x["dO"] = torch.randn(Bt, H, L, d, device=dev, generator=g).to(torch.bfloat16)
    dsc = pa.make_desc(x["q"], 1.0)
    wsf, wsb = pa.workspace(dsc, 0, dev), pa.workspace(dsc, 1, dev)
    o2, lse = torch.empty_like(x["q"]), torch.empty(Bt, H, L, device=dev)
    grads = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["q"]), dv=torch.empty_like(x["q"]),
                 dw=torch.empty_like(x["q"]), dbeta=torch.empty_like(x["beta"]))

    def tstep():
        pa.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, 1.0, ws=wsf, out=(o2, lse))
        pa.bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], o2, lse, x["dO"], 1.0, ws=wsb, out=grads)
    for _ in range(2):
        tstep()
    torch.cuda.synchronize()
    reps = 3
    a = ev()
    for _ in range(reps):
        tstep()
    b = ev()
    torch.cuda.synchronize()
    tms = a.elapsed_time(b) / reps
    bms = time_events(lambda: pa.bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], o2, lse, x["dO"], 1.0, ws=wsb,
                                     out=grads), 1, reps)
    ffl, bfl = Bt * H * fwd_flops_per_head(L, d, TC_CHUNK), Bt * H * bwd_flops_per_head(L, d, B)
    clk = pk.get("sm_max_mhz", 2070.0)
    fp32_peak = 152 * 128 * 2 * clk * 1e6 / 1e12
    tf32_peak = pk["bf16"] * 1.1 / 2.25
    btf = bfl / (bms * 1e-3) / 1e12
    train = {"ms_per_step": tms, "tflops": (ffl + bfl) / (tms * 1e-3) / 1e12, "flops_per_step": ffl + bfl,
             "backward": {"ms": bms, "tflops": btf, "bound": "tensor", "peak": tf32_peak, "unit": "TFLOP/s",
                          "frac": btf / tf32_peak, "chunk": B,
                          "peak_source": f"tf32 dense: measured bf16 {pk['bf16']:.1f} x nominal tf32/bf16 (1.1/2.25)",
                          "fp32_fma_peak": fp32_peak, "frac_of_fp32_fma_peak": btf / fp32_peak},
             "workload": "fwd+bwd, batch 4, 16 heads, d=128, L=2048, bf16 inputs: tcgen05 forward (chunk 64), "
                         "backward (chunk 32) on TF32 warp MMAs (mma.sync, fp32 accumulation)"}
    return {"decode": decode, "forward": fwd, "train": train}


def run_d128_train_small(args, pa, dev):
    """A small head-dim-128 training step (tcgen05 forward + the backward's three phases) for
    profiler captures: batch 1 x 8 heads x 2048 unless --batch / --heads override; each backward
    phase also timed alone with CUDA events."""
    Bt, H, L, d = args.batch or 1, args.heads or 8, 2048, 128
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    x = {n: (torch.randn(Bt, H, L, d, device=dev, generator=g) / math.sqrt(d)).to(torch.bfloat16)
         for n in ("q", "k", "v")}
    wr = torch.randn(Bt, H, L, d, device=dev, generator=g)
    x["w"] = (wr / wr.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    x["beta"] = 2.0 * torch.sigmoid(torch.randn(Bt, H, L, device=dev, generator=g))
    x["dO"] = torch.randn(Bt, H, L, d, device=dev, generator=g).to(torch.bfloat16)
    o, lse = pa.fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, 1.0)
    wsb = pa.workspace(pa.make_desc(x["q"], 1.0), 1, dev)
    grads = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["q"]), dv=torch.empty_like(x["q"]),
                 dw=torch.empty_like(x["q"]), dbeta=torch.empty_like(x["beta"]))

    def bwd(phases):
        pa.bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], o, lse, x["dO"], 1.0, ws=wsb, out=grads, phases=phases)
    out = {"workload": f"fwd+bwd, batch {Bt}, {H} heads, d=128, L={L}, bf16"}
    for name, ph in (("prepare", 1), ("scan", 2), ("finish", 4)):
        ms = []
        for _ in range(max(1, args.steps)):
            if ph > 1:
                bwd(ph - 1)  # the phases before this one, untimed
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            bwd(ph)
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        out[f"{name}_ms"] = min(ms)
    return out


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
