#!/usr/bin/env python
"""Throughput of the nanochat pretraining step (forward + mean next-token
cross-entropy + full backward) on B300 GPUs, one process per GPU.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload d20] [--no-cpu-baseline]
  python bench.py --kernel CASE [--reps N]     (one op of the path, for ncu)

Under torchrun (N > 1) each rank runs an independent replica of the step on
its own batch (the pages' data-parallel recipe without the gradient
all-reduce, which is out of scope here), so per-GPU work is fixed and the
scaling is weak. Rank 0 prints one JSON line.

Our arm: one call of nc_forward_loss_async + nc_backward on device-resident
inputs is captured into a CUDA graph; W warm-up replays, then K timed
replays with CUDA events between them on the library's stream, between a
barrier and a synchronise (mean, median, p10 and p90 per step; and, when
K < 50, a further 50 replays after 10 warm-up replays for the distribution).
The per-kernel-family times come from K more eager steps in which the
library brackets every launch with CUDA events.
The end-to-end figure times nc_train_step_host_u16: each step copies the
batch's packed uint16 token rows [B, T+1] (the token-shard format) from
pinned host memory, widens them on the device into inputs and next-token
targets, runs forward and backward and reads the loss back (vocabularies
above 65,536 ids use nc_train_step_host with int32 token and target
buffers). The CPU baseline is the oracle on one 2048-token sequence of the
same workload, timed after the GPU work in this process.

Reference arm (--impl reference): the oracle as it stands, on rank 0's host
cores, W + K steps each over one 512-token sample of one sequence of the
same workload (causality makes those positions' work exactly that of the
first 512 positions of a full sequence).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workload as W  # noqa: E402

METRIC = "training tokens/sec (fwd+bwd) at depth 20 on 1 B300; MFU vs bf16 dense peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="d20", choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-optimizer", action="store_true",
                    help="skip timing the optimizer step (Muon + AdamW) after the fwd+bwd step")
    ap.add_argument("--no-infer", action="store_true",
                    help="skip timing generation (prefill + KV-cache decode steps)")
    ap.add_argument("--protocol-steps", type=int, default=50,
                    help="replayed steps of the timing-distribution block run when --steps is smaller (0: none)")
    ap.add_argument("--kernel", default=None, choices=sorted(KERNEL_CASES),
                    help="time one op of the path at the d20 shapes through the C ABI (for ncu captures)")
    ap.add_argument("--reps", type=int, default=3, help="launches of the --kernel case after one warm-up launch")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(w: W.Workload) -> str:
    return (f"{w.name}: depth {w.depth}, d_model {w.d_model}, {w.n_head} heads x 128, MLP {w.ffn} ReLU^2, "
            f"vocab {w.vocab} untied, seq {w.seq_len}, batch {w.batch} per GPU; Zipf(1.1) tokens, "
            f"N(0,0.02) weights, seeded")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


# ------------------------------------------------------------------ oracle timing

def oracle_tokens_per_s(w: W.Workload, params: np.ndarray, tokens: int, steps: int, warmup: int):
    """Time the CPU oracle (fp32) on `tokens` positions of one sequence."""
    import oracle

    s = oracle.Shape(w.depth, w.d_model, w.n_head, w.vocab)
    tok, tgt = W.make_tokens(w.with_batch(1))
    tok, tgt = tok[:, :tokens], tgt[:, :tokens]
    for _ in range(warmup):
        oracle.step(params, tok, tgt, s, np.float32)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.step(params, tok, tgt, s, np.float32)
        times.append(time.perf_counter() - t0)
    return tokens * len(times) / sum(times), sum(times)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ------------------------------------------------------------------ arms

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_over_ranks(ms: float, launches: int, device) -> tuple:
    """(max of ms, sum of launches) over all ranks of the default process
    group (NCCL on GPUs, gloo works as well); identity without one."""
    import torch
    import torch.distributed as dist

    t_ms = torch.tensor([ms], dtype=torch.float64, device=device)
    t_n = torch.tensor([float(launches)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t_ms, op=dist.ReduceOp.MAX)
        dist.all_reduce(t_n, op=dist.ReduceOp.SUM)
    return float(t_ms.item()), int(t_n.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms_max: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms_max / 1000.0)


def reference_arm(args):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    w = W.WORKLOADS[args.workload]
    params = W.make_params(w)
    sample = 512
    tps, total_s = oracle_tokens_per_s(w, params, sample, args.steps, args.warmup)
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total_s / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": w.batch * args.gpus, "seq_len": w.seq_len,
                   "parallelism": "oracle on host cores (rank 0 only)"},
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: the first {sample} positions of one sequence of the {w.name} "
                                   f"workload, forward + loss + backward in numpy float32"},
        "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def our_arm(args):
    import torch
    import torch.distributed as dist

    import decoder_transformer_step_nanochat_b300 as nc

    ws, rank, local = dist_setup()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    w = W.WORKLOADS[args.workload]
    M = w.tokens
    pk, pk_kind = peaks()

    params_np = W.make_params(w)
    tok_np, tgt_np = W.make_tokens(w, seed=rank)
    stream = torch.cuda.Stream()
    prec = nc.NC_FP32_DEBUG if w.dtype == "fp32" else nc.NC_BF16
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, w.batch, prec, stream=stream)
    params = torch.from_numpy(params_np)
    params = (params if prec == nc.NC_FP32_DEBUG else params.to(torch.bfloat16)).cuda()
    tok = torch.from_numpy(tok_np).cuda()
    tgt = torch.from_numpy(tgt_np).cuda()
    grads = torch.empty(st.n_params, dtype=torch.float32, device="cuda")
    d_loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()  # uploads ran on the default stream

    def step():
        st.forward_loss_async(params, tok, tgt, d_loss)
        st.backward(grads)

    # one eager step sets the kernels' attributes up; the step is then
    # captured once into a CUDA graph (no host decision depends on device
    # data) and replayed: W warm-up replays, then exactly K timed replays
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    n0 = nc.nc_launch_count(st.ctx)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        step()
    launches_per_step = nc.nc_launch_count(st.ctx) - n0
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    loss0 = float(d_loss.item())

    # ---- timed region: device-resident inputs, per-step CUDA events on the library's stream
    sampler = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(args.steps):
            graph.replay()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    ms = ev[0].elapsed_time(ev[-1]) / args.steps
    launches = launches_per_step * args.steps
    ms_max, launches_all = reduce_over_ranks(ms, launches, "cuda")
    value = job_tokens_per_s(ws, M, ms_max)
    dist_ms = step_distribution(per_step)

    # the timing protocol of at least 50 replayed steps after 10 warm-up
    # replays, reported beside the K-step headline when K < 50
    protocol = None
    npro = args.protocol_steps
    if 0 < args.steps < npro:
        for _ in range(10):
            graph.replay()
        torch.cuda.synchronize()
        ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(npro + 1)]
        with torch.cuda.stream(stream):
            ev2[0].record(stream)
            for i in range(npro):
                graph.replay()
                ev2[i + 1].record(stream)
        torch.cuda.synchronize()
        protocol = step_distribution([ev2[i].elapsed_time(ev2[i + 1]) for i in range(npro)])
    elif npro > 0:
        protocol = dict(dist_ms)
    if protocol is not None:
        protocol["tokens_per_s_median"] = job_tokens_per_s(ws, M, protocol["median_ms"])
    del graph

    # ---- per-kernel-family device time: K eager steps, every launch
    # bracketed by CUDA events on the library's stream
    nc.nc_profile_enable(st.ctx, True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    ms_eager = e0.elapsed_time(e1) / args.steps
    fam = {}
    for name, f in (("gemm", nc.NC_FAM_GEMM), ("attn_fwd", nc.NC_FAM_ATTN_FWD),
                    ("attn_bwd", nc.NC_FAM_ATTN_BWD), ("rows", nc.NC_FAM_ROWS)):
        fam[name] = nc.nc_profile_read(st.ctx, f)
    nc.nc_profile_enable(st.ctx, False)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        if w.vocab <= 65536:
            # the same ids as tok_np / tgt_np, as packed rows
            h_rows = torch.from_numpy(W.make_packed_tokens(w, seed=rank).view(np.int16)).pin_memory()
            h2d = h_rows.numel() * 2

            def host_step():
                nc.nc_train_step_host_u16(st.ctx, params.data_ptr(), h_rows.data_ptr(), grads.data_ptr())
        else:
            h_tok = torch.from_numpy(tok_np).pin_memory()
            h_tgt = torch.from_numpy(tgt_np).pin_memory()
            h2d = 2 * M * 4

            def host_step():
                nc.nc_train_step_host(st.ctx, params.data_ptr(), h_tok.data_ptr(), h_tgt.data_ptr(), grads.data_ptr())
        host_step()
        if ws > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            host_step()
        dt_max, _ = reduce_over_ranks(1000.0 * (time.perf_counter() - t0) / args.steps, 0, "cuda")
        e2e = {"value": job_tokens_per_s(ws, M, dt_max), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4}

    # ---- roofline: every family against its bound; the dominant one is the headline
    steps = args.steps
    alg = algorithmic_work(w)
    families = {}
    for k, (fms, fn, fwork) in fam.items():
        if fms <= 0:
            continue
        per = fms / steps
        if k == "rows":
            ach = fwork / (fms / 1000.0) / 1e9
            families[k] = {"ms_per_step": per, "launches_per_step": fn / steps, "gbs": ach,
                           "bound": "hbm", "peak": pk["hbm_gbs"], "frac": ach / pk["hbm_gbs"]}
        else:
            work = alg[k] * steps  # algorithmic FLOPs (no recompute)
            ach = work / (fms / 1000.0) / 1e12
            hw = fwork / (fms / 1000.0) / 1e12
            families[k] = {"ms_per_step": per, "launches_per_step": fn / steps, "tflops": ach, "tflops_hw": hw,
                           "bound": "tensor", "peak": pk["bf16_tflops_sustained"],
                           "frac": ach / pk["bf16_tflops_sustained"]}
    dom = max(fam, key=lambda k: fam[k][0])
    dms, dn, _ = fam[dom]
    fd = families[dom]
    roofline = {"bound": fd["bound"], "kernel": dom,
                "achieved": fd["gbs"] if dom == "rows" else fd["tflops"], "peak": fd["peak"],
                "unit": "GB/s" if dom == "rows" else "TFLOP/s", "frac": fd["frac"],
                "peak_kind": f"{pk_kind} ({'HBM copy' if dom == 'rows' else 'sustained bf16'})",
                "traffic": read_traffic(dom, w.name), "launches": dn, "avg_launch_ms": dms / max(1, dn),
                "share_of_step": dms / (ms_eager * steps),
                "work": "algorithmic: 6*M*(12*L*d^2 + d*V) FLOPs per step for the GEMMs (the lm_head "
                        "backward's logit recompute excluded; it is in achieved_hw)"}
    if dom != "rows":
        roofline["achieved_hw"] = fd["tflops_hw"]
        roofline["frac_hw"] = fd["tflops_hw"] / fd["peak"]

    fpt = W.model_flops_per_token(w)
    mfu = value * fpt / (ws * pk["bf16_tflops"] * 1e12)

    # ---- the optimizer step (clip, AdamW, Muon) on the same buffers, timed on its own
    opt = None
    if not args.no_optimizer:
        lr_a, lr_m, wd, clip = 3e-3, 2e-2, 0.1, 1.0
        state = torch.empty(nc.nc_optim_state_bytes(st.ctx) // 4, dtype=torch.float32, device="cuda")
        stats = torch.zeros(2, dtype=torch.float32, device="cuda")
        nc.nc_optim_init(st.ctx, params.data_ptr(), state.data_ptr())

        def opt_step(t):
            nc.nc_optim_step(st.ctx, params.data_ptr(), grads.data_ptr(), state.data_ptr(), t, lr_a, lr_m, wd, clip,
                             stats.data_ptr())

        for t in range(1, args.warmup + 1):
            opt_step(t)
        torch.cuda.synchronize()
        nc.nc_profile_enable(st.ctx, True)
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            o0.record(stream)
            for t in range(args.steps):
                opt_step(args.warmup + 1 + t)
            o1.record(stream)
        torch.cuda.synchronize()
        ms_opt = o0.elapsed_time(o1) / args.steps
        ns = nc.nc_profile_read(st.ctx, nc.NC_FAM_OPT_NS)
        el = nc.nc_profile_read(st.ctx, nc.NC_FAM_OPT_ELEM)
        nc.nc_profile_enable(st.ctx, False)
        ms_opt_max, _ = reduce_over_ranks(ms_opt, 0, "cuda")
        opt = {
            "ms_per_step": ms_opt_max,
            "newton_schulz": {"ms_per_step": ns[0] / args.steps, "launches_per_step": ns[1] / args.steps,
                              "tflops": ns[2] / (ns[0] / 1000.0) / 1e12 if ns[0] > 0 else None},
            "elementwise": {"ms_per_step": el[0] / args.steps, "launches_per_step": el[1] / args.steps,
                            "gbs": el[2] / (el[0] / 1000.0) / 1e9 if el[0] > 0 else None},
            "tokens_per_s_with_optimizer": job_tokens_per_s(ws, M, ms_max + ms_opt_max),
            "hyper": {"lr_adamw": lr_a, "lr_muon": lr_m, "weight_decay": wd, "max_grad_norm": clip,
                      "muon_momentum": 0.95, "ns_steps": 5},
            "grad_norm": float(stats[0].item()),
        }
        del state

    # ---- generation: prefill of the batch's prompts, then greedy decode steps
    inf = None
    if not args.no_infer:
        inf = infer_timing(nc, st, w, params, tok, stream, args, ws, pk)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tps, _ = oracle_tokens_per_s(w, params_np, w.seq_len, 1, 0)
        cpu = {"value": tps, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"one {w.seq_len}-token sequence of the {w.name} workload (same weights), forward + "
                         f"loss + backward in numpy float32, BLAS on all host cores"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if prec == nc.NC_FP32_DEBUG else "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(w), "global_batch": w.batch * ws, "seq_len": w.seq_len,
                       "tokens_per_step": M * ws,
                       "parallelism": f"{ws} independent data-parallel replicas (no collective)",
                       "l2": "inputs larger than L2: the step streams a ~17 GB activation stash",
                       "timing": "one CUDA graph of nc_forward_loss_async + nc_backward, replayed; CUDA events "
                                 "between replays on the library's stream"},
            "mfu": mfu, "mfu_peak_tflops": pk["bf16_tflops"],
            "mfu_vs_sustained": value * fpt / (ws * pk["bf16_tflops_sustained"] * 1e12),
            "model_flops_per_token": fpt,
            "loss": loss0,
            "clocks": clocks, "e2e": e2e, "gpu_launches": launches_all,
            "step_ms": dist_ms, "timing_protocol": protocol, "eager_ms_per_step": ms_eager,
            "launches_per_step": launches_per_step,
            "roofline": roofline, "families": families, "optimizer": opt, "inference": inf,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    st.close()
    if ws > 1:
        dist.destroy_process_group()
    return 0


def step_distribution(per_step_ms):
    """Median, 10th and 90th percentile and mean of per-step times (ms)."""
    a = np.asarray(per_step_ms, dtype=np.float64)
    return {"steps": int(a.size), "median_ms": float(np.median(a)), "p10_ms": float(np.percentile(a, 10)),
            "p90_ms": float(np.percentile(a, 90)), "mean_ms": float(a.mean())}


def algorithmic_work(w: W.Workload) -> dict:
    """Algorithmic FLOPs of one step per tensor-core family: every linear
    layer and the lm_head once forward (2 FLOPs per weight and token) and
    twice backward (input and weight gradients); causal attention over the
    lower triangle, 2*128*T*(T+1) FLOPs per (sequence, head) for QK^T and PV
    forward and twice that backward. No recompute is counted."""
    L, d, V, T, B, H = w.depth, w.d_model, w.vocab, w.seq_len, w.batch, w.n_head
    M = B * T
    fwd_attn = 2.0 * 128 * T * (T + 1) * B * H * L
    return {"gemm": 6.0 * M * (12.0 * L * d * d + d * V), "attn_fwd": fwd_attn, "attn_bwd": 2.0 * fwd_attn}


def infer_timing(nc, st, w, params, tok, stream, args, ws, pk):
    """Prefill time and decode-step time through the generation ABI
    (include/nc_infer.h), with the decode step's HBM roofline: the weights
    the step streams plus the cached keys/values it reads."""
    import torch

    B, T, d, L = w.batch, w.seq_len, w.d_model, w.depth
    steps = max(8, args.steps)
    max_len = T + args.warmup + 2 * steps + 4
    kv = torch.empty(nc.nc_kv_cache_bytes(st.ctx, max_len) + 256, dtype=torch.uint8, device="cuda")
    kvp = (kv.data_ptr() + 255) // 256 * 256
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    cur = torch.empty(B, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nc.nc_prefill(st.ctx, params.data_ptr(), tok.data_ptr(), kvp, max_len, nxt.data_ptr())  # warm-up
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        nc.nc_prefill(st.ctx, params.data_ptr(), tok.data_ptr(), kvp, max_len, nxt.data_ptr())
        e1.record(stream)
    torch.cuda.synchronize()
    ms_prefill = e0.elapsed_time(e1)
    pos = T
    for _ in range(args.warmup):
        cur.copy_(nxt)
        nc.nc_decode_step(st.ctx, params.data_ptr(), cur.data_ptr(), pos, kvp, max_len, nxt.data_ptr())
        pos += 1
    torch.cuda.synchronize()
    nc.nc_profile_enable(st.ctx, True)
    pos0 = pos
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            cur.copy_(nxt)
            nc.nc_decode_step(st.ctx, params.data_ptr(), cur.data_ptr(), pos, kvp, max_len, nxt.data_ptr())
            pos += 1
        e1.record(stream)
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / steps
    fam = {k: nc.nc_profile_read(st.ctx, f) for k, f in (("gemm", nc.NC_FAM_DEC_GEMM), ("attn", nc.NC_FAM_DEC_ATTN),
                                                         ("rows", nc.NC_FAM_DEC_ROWS))}
    nc.nc_profile_enable(st.ctx, False)
    # the same steps replayed from one captured CUDA graph (device position)
    d_pos = torch.full((1,), pos, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        cur.copy_(nxt)
        nc.nc_decode_step_dev(st.ctx, params.data_ptr(), cur.data_ptr(), d_pos.data_ptr(), kvp, max_len,
                              nxt.data_ptr())
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        cur.copy_(nxt)
        nc.nc_decode_step_dev(st.ctx, params.data_ptr(), cur.data_ptr(), d_pos.data_ptr(), kvp, max_len,
                              nxt.data_ptr())
    gsteps = min(steps, max_len - pos - 2)
    graph.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(gsteps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms_graph = e0.elapsed_time(e1) / max(1, gsteps)
    nc.nc_sync(st.ctx)
    esz = 2 if w.dtype == "bf16" else 4
    weights = (12 * L * d * d + w.vocab * d) * esz       # every block matrix and lm_head, once
    kv_read = 2 * L * B * d * esz * ((pos0 + pos - 1) / 2 + 1)  # mean cached length over the timed steps
    step_bytes = weights + kv_read
    ms_prefill_max, _ = reduce_over_ranks(ms_prefill, 0, "cuda")
    ms_step_max, _ = reduce_over_ranks(ms_step, 0, "cuda")
    ms_graph_max, _ = reduce_over_ranks(ms_graph, 0, "cuda")
    gbs = step_bytes / (ms_graph_max / 1000.0) / 1e9
    del kv, graph
    return {
        "prefill": {"ms": ms_prefill_max, "tokens_per_s": ws * B * T / (ms_prefill_max / 1000.0)},
        "decode": {"ms_per_step": ms_step_max, "tokens_per_s": ws * B / (ms_step_max / 1000.0),
                   "graph_ms_per_step": ms_graph_max, "graph_tokens_per_s": ws * B / (ms_graph_max / 1000.0),
                   "batch": B, "context": f"{pos0}..{pos - 1}", "launches_per_step": sum(v[1] for v in fam.values()) / steps,
                   "families_ms_per_step": {k: v[0] / steps for k, v in fam.items()}},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                     "bytes_per_step": step_bytes,
                     "note": "graph-replayed decode step: weights streamed once + cached keys/values read"},
    }


def read_traffic(family: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary of this kernel
    family, or None when absent, taken on a different kernel source, or taken
    on another workload."""
    path = os.path.join(ROOT, "profiles", f"traffic_{family}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("workload", workload) != workload:
        return None
    src = kv.get("source_sha256")
    files = kv.get("source_files", "").split()
    if not src or not files:
        return None
    h = hashlib.sha256()
    for fn in files:
        p = os.path.join(ROOT, fn)
        if not os.path.exists(p):
            return None
        with open(p, "rb") as f:
            h.update(f.read())
    if h.hexdigest() != src:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ single ops (for ncu captures)

# Ops of the path at the d20 shapes (batch 16 x seq 2048, d_model 1280, 10
# heads, vocab 65,536) unless stated: name -> (bound, what one launch moves or
# computes, description).
KERNEL_CASES = {
    "gemm_qkv": ("tensor", "2*M*N*K FLOPs", "32768 x 3840 x 1280 forward GEMM, QK-norm + RoPE epilogue"),
    "gemm_fc": ("tensor", "2*M*N*K FLOPs", "32768 x 5120 x 1280 forward GEMM, ReLU^2 epilogue (a only)"),
    "gemm_relu2_bwd": ("tensor", "2*M*N*K FLOPs", "32768 x 5120 x 1280 GEMM with the ReLU^2 backward epilogue"),
    "gemm_dw": ("tensor", "2*M*N*K FLOPs", "1280 x 5120 x 32768 weight gradient (k-splits summed in the kernel)"),
    "attn_fwd": ("tensor", "2*128*T*(T+1)*B*H FLOPs", "causal attention forward"),
    "attn_bwd": ("tensor", "4*128*T*(T+1)*B*H FLOPs", "attn_rowdot_k + causal attention backward"),
    "lmhead_ce": ("tensor", "2*M*V*d FLOPs", "lm_head + CE forward, 4096 rows (GEMM partials + ce_reduce_k)"),
    "rmsnorm_fwd": ("hbm", "M*d*(4+2) + 4*M bytes", "rmsnorm_fwd_k: fp32 x -> bf16 y, fp32 r"),
    "rmsnorm_bwd": ("hbm", "M*d*(4+4+2+2+2) + 4*M bytes", "rmsnorm_bwd_k, accumulating into fp32 dx, bf16 copy"),
    "qk_norm_rope_bwd": ("hbm", "2*M*d*(4+2+2) + 8*M*H bytes", "qk_norm_rope_bwd_k over q and k heads"),
    "embed_fwd": ("hbm", "M*d*(2+4) + 4*M bytes", "embed_fwd_k: gather of Zipf(1.1) ids into fp32 x"),
    "embed_bwd": ("hbm", "M*d*(4+4) + 4*M bytes",
                  "deterministic embedding gradient: key sort, run sums, per-id merge (after a memset of dW_te)"),
}


def kernel_arm(args):
    """One op of the path through the C ABI at the d20 shapes on random
    device-resident inputs: one warm-up launch, then --reps launches timed
    with CUDA events on the library's stream. Prints one JSON line with the
    mean time per launch and the algorithmic work per launch."""
    import torch

    import decoder_transformer_step_nanochat_b300 as nc

    torch.cuda.set_device(0)
    pk, pk_kind = peaks()
    case = args.kernel
    B, T, H, V = 16, 2048, 10, 65536
    d = H * 128
    if case == "lmhead_ce":
        B = 2
    M = B * T
    stream = torch.cuda.Stream()
    # the norm cases need no vocabulary: a small one keeps the context's
    # workspace (its cross-entropy buffer grows with the vocabulary) small
    v_ctx = 1024 if case in ("rmsnorm_fwd", "rmsnorm_bwd", "qk_norm_rope_bwd") else V
    st = nc.Step(1, d, H, T, v_ctx, B, nc.NC_BF16, stream=stream)
    ctx = st.ctx
    bf = torch.bfloat16
    g = torch.Generator(device="cuda").manual_seed(0)

    def randn(*shape, scale=1.0, dtype=bf):
        return (torch.randn(shape, device="cuda", generator=g) * scale).to(dtype)

    def gemm(Mg, N, K, ak, bk, epi, c_dtype, c2=None):
        A = randn(*((Mg, K) if ak else (K, Mg)))
        Bm = randn(*((N, K) if bk else (K, N)), scale=0.05)
        C = torch.empty((Mg, N), device="cuda", dtype=c_dtype)
        args_ = (ctx, Mg, N, K, A.data_ptr(), K if ak else Mg, ak, Bm.data_ptr(), K if bk else N, bk, epi, 1.0, 0.0,
                 C.data_ptr(), N, c2.data_ptr() if c2 is not None else None, c2.shape[1] if c2 is not None else 0)
        return (lambda: nc.nc_op_gemm(*args_)), (A, Bm, C, c2), 2.0 * Mg * N * K

    if case == "gemm_qkv":
        rqk = torch.empty((M, 2 * H), device="cuda", dtype=torch.float32)
        run, keep, work = gemm(M, 3 * d, d, 1, 1, nc.NC_EPI_QKNORM_ROPE, bf, rqk)
    elif case == "gemm_fc":
        run, keep, work = gemm(M, 4 * d, d, 1, 1, nc.NC_EPI_RELU2A, bf)
    elif case == "gemm_relu2_bwd":
        a = torch.rand((M, 4 * d), device="cuda", generator=g).to(bf)
        run, keep, work = gemm(M, 4 * d, d, 1, 0, nc.NC_EPI_RELU2_BWD, bf, a)
    elif case == "gemm_dw":
        run, keep, work = gemm(d, 4 * d, M, 0, 0, nc.NC_EPI_STORE_F32, torch.float32)
    elif case in ("attn_fwd", "attn_bwd"):
        qkv = randn(M, 3 * d)
        o = torch.empty((M, d), device="cuda", dtype=bf)
        lse = torch.empty((B, H, T), device="cuda", dtype=torch.float32)
        dout = randn(M, d)
        dqk = torch.empty((2, M, d), device="cuda", dtype=torch.float32)
        dqkv = torch.empty((M, 3 * d), device="cuda", dtype=bf)
        nc.nc_op_attention_fwd(ctx, qkv.data_ptr(), o.data_ptr(), lse.data_ptr())
        fwd = 2.0 * 128 * T * (T + 1) * B * H
        if case == "attn_fwd":
            def run():
                nc.nc_op_attention_fwd(ctx, qkv.data_ptr(), o.data_ptr(), lse.data_ptr())
            work = fwd
        else:
            def run():
                nc.nc_op_attention_bwd(ctx, qkv.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                                       dqk.data_ptr(), dqkv.data_ptr())
            work = 2.0 * fwd
        keep = (qkv, o, lse, dout, dqk, dqkv)
    elif case == "lmhead_ce":
        hf = randn(M, d)
        wl = randn(V, d, scale=0.02)
        tgt = torch.randint(0, V, (M,), device="cuda", dtype=torch.int32, generator=g)
        lse, nll = torch.empty(M, device="cuda"), torch.empty(M, device="cuda")
        am = torch.empty(M, device="cuda", dtype=torch.int32)

        def run():
            nc.nc_op_lmhead_ce_fwd(ctx, hf.data_ptr(), wl.data_ptr(), tgt.data_ptr(), lse.data_ptr(), nll.data_ptr(),
                                   am.data_ptr())
        keep, work = (hf, wl, tgt, lse, nll, am), 2.0 * M * V * d
    else:
        x = torch.randn((M, d), device="cuda", generator=g)
        r = torch.rand(M, device="cuda", generator=g) + 0.5
        if case == "rmsnorm_fwd":
            y = torch.empty((M, d), device="cuda", dtype=bf)

            def run():
                nc.nc_op_rmsnorm_fwd(ctx, x.data_ptr(), y.data_ptr(), r.data_ptr())
            keep, work = (x, y, r), M * d * 6.0 + 4.0 * M
        elif case == "rmsnorm_bwd":
            dy, y = randn(M, d), randn(M, d)
            dxe = torch.empty((M, d), device="cuda", dtype=bf)

            def run():
                nc.nc_op_rmsnorm_bwd(ctx, dy.data_ptr(), y.data_ptr(), r.data_ptr(), x.data_ptr(), dxe.data_ptr(), 1)
            keep, work = (x, r, dy, y, dxe), M * d * 14.0 + 4.0 * M
        elif case == "qk_norm_rope_bwd":
            dqk = torch.randn((2, M, d), device="cuda", generator=g)
            qkv = randn(M, 3 * d)
            rqk = torch.rand((M, 2 * H), device="cuda", generator=g) + 0.5
            dqkv = torch.empty((M, 3 * d), device="cuda", dtype=bf)

            def run():
                nc.nc_op_qk_norm_rope_bwd(ctx, dqk.data_ptr(), qkv.data_ptr(), rqk.data_ptr(), dqkv.data_ptr())
            keep, work = (dqk, qkv, rqk, dqkv), 2.0 * M * d * 8 + 8.0 * M * H
        else:
            ids = torch.from_numpy(W.make_tokens(W.WORKLOADS["d20"])[0].reshape(-1).copy()).cuda()
            if case == "embed_fwd":
                wte = randn(V, d, scale=0.02)

                def run():
                    nc.nc_op_embed_fwd(ctx, ids.data_ptr(), wte.data_ptr(), x.data_ptr())
                keep, work = (x, wte, ids), M * d * 6.0 + 4.0 * M
            else:
                dwte = torch.empty((V, d), device="cuda", dtype=torch.float32)

                def run():
                    nc.nc_op_embed_bwd(ctx, ids.data_ptr(), x.data_ptr(), dwte.data_ptr())
                keep, work = (x, dwte, ids), M * d * 8.0 + 4.0 * M
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        run()
    nc.nc_sync(ctx)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.reps):
            run()
        e1.record(stream)
    nc.nc_sync(ctx)
    ms = e0.elapsed_time(e1) / max(1, args.reps)
    bound, unit_of_work, desc = KERNEL_CASES[case]
    if bound == "hbm":
        ach, peak, unit = work / (ms / 1000.0) / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        ach, peak, unit = work / (ms / 1000.0) / 1e12, pk["bf16_tflops"], "TFLOP/s"
    print(json.dumps({"kernel": case, "desc": desc, "bound": bound, "work_per_launch": work,
                      "work_unit": unit_of_work, "ms_per_launch": ms, "launches": args.reps, "achieved": ach,
                      "peak": peak, "peak_kind": f"{pk_kind} ({'HBM copy' if bound == 'hbm' else 'bf16 burst'})",
                      "unit": unit, "frac": ach / peak}), flush=True)
    del keep
    st.close()
    return 0


def main():
    args = parse_args()
    if args.kernel:
        return kernel_arm(args)
    if args.impl == "reference":
        return reference_arm(args)
    return our_arm(args)


if __name__ == "__main__":
    sys.exit(main())
