#!/usr/bin/env python3
"""Benchmark of the contextually sparse (DejaVu) layer decode at the OPT-175B shape.

One step = one sparse decode of one OPT-175B-shaped layer (d=12288, 96 heads
x 128, N=49152, predictor rank 1000, fp16 storage, fp32 arithmetic, batch 1,
KV length 2048, keep 2458 neurons / 20 heads): predictor + top-k, head-sparse
QKV + KV append, decode attention over the selected heads, head-sparse
out-projection, fc1 gather + ReLU, fc2 gather, both residuals: seven
kernels chained by programmatic dependent launch (dv_layer_decode).  The
persistent streaming kernel (one launch) is timed beside it for comparison.

Inputs are synthetic (seeded torch RNG on the device) and resident in HBM
before timing.  Each step decodes the next of `--copies` distinct layer
copies (4 x 3.9 GB by default), so no step's 519 MB of required bytes can be
served from the 129 MB L2 left over by the previous step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle (the
plain binary64 C implementation) on the same workload.  Under torchrun (N > 1)
each rank runs an independent replica (the path has no cross-GPU exchange).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

KERNELS = ["pred_stage1_head_topk", "pred_stage2_neuron_topk", "qkv_ln1_kv_append",
           "attn_decode", "oproj_residual", "fc1_ln2_relu", "fc2_residual"]
KERNEL_BYTES_KEY = ["pred_stage1", "pred_stage2", "qkv", "attn", "oproj", "fc1", "fc2"]
GRAPH_STEPS = 64
METRIC = "µs per sparse layer-decode and achieved HBM GB/s (% roofline) at OPT-175B shape"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    p.add_argument("--config", default="opt175b")
    p.add_argument("--batch", type=int, default=None)
    p.add_argument("--copies", type=int, default=4)
    p.add_argument("--cpu-budget-s", type=float, default=15.0)
    p.add_argument("--row-kernel", choices=["mma", "tc"], default="mma",
                   help="fc1 rows on mma.sync (default) or on the opt-in tcgen05 kernel "
                        "(binary16, from 9 batch rows)")
    p.add_argument("--no-extras", action="store_true",
                   help="skip dense baseline, e2e, copy peak, CPU baseline and stack legs")
    p.add_argument("--stack-layers", type=int, default=24,
                   help="layers of the stack leg (0 skips it)")
    p.add_argument("--stack-batches", default="1,2,4,8,16,32",
                   help="batch sizes of the stack leg")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: a barrier and a max over ranks, nothing else)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist

    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (the whole job ends when the slowest rank does)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_decode(max_ms: float, steps: int, world: int) -> float:
    """Aggregate time per layer decode over all replicas: the slowest rank's
    wall time divided by every decode the job completed."""
    return max_ms * 1000.0 / (steps * world)


# ---------------------------------------------------------------------------
# clocks sampled while the timed loop runs


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid=None, interval_ms=50):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(interval_ms)]
        if gpu_uuid:
            cmd += ["-i", gpu_uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [ln.split(",") for ln in out.strip().splitlines() if ln.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "of fallback (6.8 TB/s)"


def profile_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    from attention_dv_predict_gb300 import build as dv_build

    if d.get("source_hash") != dv_build.source_hash():
        return None
    v = d.get("kernels", {}).get(kernel, {}).get("dram_bytes_per_launch")
    return float(v) if v is not None else None


# ---------------------------------------------------------------------------
# the CUDA arm


def workload_config(cfg, B):
    return {"workload": f"{cfg.name}-sparse-layer-decode", "d_model": cfg.d_model,
            "n_heads": cfg.n_heads, "head_dim": cfg.head_dim, "d_ffn": cfg.d_ffn,
            "pred_rank": cfg.pred_rank, "batch": B, "kv_len": cfg.kv_len,
            "k_neurons": cfg.k_neurons, "k_heads": cfg.k_heads, "storage": cfg.dtype}


def run_cuda(args):
    import torch

    rank, world = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        from attention_dv_predict_gb300 import build as dv_build

        dv_build.build()
    barrier()
    from attention_dv_predict_gb300 import dv
    from attention_dv_predict_gb300 import traffic
    import dv_inputs

    dv.dv_set_row_kernel(1 if args.row_kernel == "tc" else 0)
    cfg = dv_inputs.CONFIGS[args.config]
    B = args.batch or cfg.batch
    cfg = cfg.with_(batch=B)
    k_h, k_n = cfg.k_heads, cfg.k_neurons
    desc = dv.desc_from_config(cfg)
    copies = max(1, args.copies)

    layers, caches = [], []
    for i in range(copies):
        w = dv_inputs.make_weights(cfg, seed=1000 * rank + i, device=dev)
        layers.append(dv.Layer(desc, w))
        caches.append(dv_inputs.make_kv(cfg, B, seed=1000 * rank + i, device=dev))
    x = dv_inputs.make_x(cfg, B, seed=rank, device=dev)
    y = torch.empty_like(x)
    sel = dv.SelectionBuffers(desc, B, k_h, k_n)
    ws = dv.Workspace(desc, B)
    stream = torch.cuda.Stream(device=dev)
    n_launch = dv.dv_layer_decode_launches(desc, B)

    def step(i, s):
        kc, vc = caches[i % copies]
        dv.dv_layer_decode(layers[i % copies], x, k_h, k_n, kc, vc, cfg.kv_len, sel, y, ws,
                           stream=s)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(copies):
            step(i, stream)
    stream.synchronize()
    if dv.dv_check(ws, stream) != dv.DV_OK:
        raise RuntimeError("device status set after the first steps")
    u_h, u_n = sel.unions()
    n_u_h, n_u_n = int(u_h.numel()), int(u_n.numel())

    # the steps run from CUDA graphs of up to GRAPH_STEPS consecutive decodes
    # (step i decodes layer copy i % copies), as a serving loop replays one
    # graph per token over all layers: no host launch gaps between steps
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    step(i, stream)
        return g

    def plan(n):
        full, rem = divmod(n, GRAPH_STEPS)
        return ([capture(GRAPH_STEPS)] * full if full else []) + ([capture(rem)] if rem else [])

    warm_graphs = plan(args.warmup)
    timed_graphs = plan(args.steps)
    stream.synchronize()

    with torch.cuda.stream(stream):
        for g in warm_graphs:
            g.replay()
    stream.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    time.sleep(0.3)  # let the sampler start before the timed region
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for g in timed_graphs:
            g.replay()
        t1.record(stream)
    t1.synchronize()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1)
    ms_max = max_over_ranks(ms, dev)
    if dv.dv_check(ws, stream) != dv.DV_OK:
        raise RuntimeError("device status set during the timed steps")

    us_per_decode = whole_job_us_per_decode(ms_max, args.steps, world)
    step_bytes = traffic.sparse_step_bytes(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn,
                                           cfg.pred_rank, 2 if cfg.dtype == "f16" else 4, B,
                                           n_u_h, n_u_n, cfg.kv_len)
    peak, peak_src = measured_peaks()
    rank_us = ms_max * 1000.0 / args.steps
    achieved = step_bytes.total / (rank_us * 1e-6) / 1e9

    kb = traffic.kernel_bytes(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn, cfg.pred_rank,
                              2 if cfg.dtype == "f16" else 4, B, n_u_h, n_u_n, cfg.kv_len,
                              n_parts=torch.cuda.get_device_properties(dev).multi_processor_count)
    kt = min(args.steps, 200)

    # the same steps with an event before every kernel: each kernel's
    # duration (the events serialise the kernels)
    n_chain = dv.dv_layer_decode_launches(desc, B)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_chain + 1)] for _ in range(kt)]
    with torch.cuda.stream(stream):
        for i in range(kt):
            kc, vc = caches[i % copies]
            dv.dv_layer_decode_traced(layers[i % copies], x, k_h, k_n, kc, vc, cfg.kv_len, sel,
                                      y, ws, evs[i], stream=stream)
    stream.synchronize()
    per_kernel = [statistics.mean(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(kt))
                  for k in range(n_chain)]
    traced_step_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][n_chain]) for i in range(kt))
    names, keys = list(KERNELS), list(KERNEL_BYTES_KEY)
    if dv.dv_mlp_one_pass(desc, B, min(B * k_n, cfg.d_ffn)):
        names[5:7] = ["mlp_fc1_fc2_partials", "mlp_partials_sum"]
        keys[5:7] = ["mlp", "mlp_reduce"]
    kernels = {names[k]: {"us": round(per_kernel[k] * 1e3, 2),
                          "share": round(per_kernel[k] / sum(per_kernel), 4),
                          "alg_bytes": kb[keys[k]],
                          "gbs": round(kb[keys[k]] / (per_kernel[k] * 1e-3) / 1e9, 1)}
               for k in range(n_chain)}

    dom = max(range(n_chain), key=lambda k: per_kernel[k])
    kern_ms, dom_name, dom_bytes = per_kernel[dom], names[dom], kb[keys[dom]]
    dom_gbs = dom_bytes / (kern_ms * 1e-3) / 1e9

    # the same decode as one persistent streaming kernel, where it serves,
    # timed like the step (graph replays), for comparison
    persistent = None
    if dv.dv_layer_decode_persistent_ok(desc, B):
        p_graphs = []
        with torch.cuda.stream(stream):
            for i in range(copies):
                g = torch.cuda.CUDAGraph()
                kc, vc = caches[i]
                with torch.cuda.graph(g, stream=stream):
                    dv.dv_layer_decode_persistent(layers[i], x, k_h, k_n, kc, vc, cfg.kv_len,
                                                  sel, y, ws, stream=stream)
                p_graphs.append(g)
            for i in range(3):
                p_graphs[i % copies].replay()
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for i in range(kt):
                p_graphs[i % copies].replay()
            c1.record(stream)
        c1.synchronize()
        p_us = c0.elapsed_time(c1) * 1e3 / kt
        del p_graphs
        if dv.dv_check(ws, stream) != dv.DV_OK:
            raise RuntimeError("device status set by the persistent decode")
        persistent = {"us_per_decode": round(p_us, 2),
                      "achieved_gbs": round(step_bytes.total / (p_us * 1e-6) / 1e9, 1),
                      "note": "the same decode as one persistent streaming kernel "
                              "(dv_layer_decode_persistent), graph replays"}

    line = {
        "metric": METRIC, "value": round(us_per_decode, 3), "unit": "µs per layer-decode",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(cfg, B), copies=copies,
                       l2="each step reads a different layer copy; 519 MB/step > 129 MB L2",
                       parallelism="replicas" if world > 1 else "single GPU",
                       fc1_rows="tcgen05" if args.row_kernel == "tc" else "mma.sync"),
        "achieved_gbs": round(achieved, 1),
        "roofline_frac_step": round(achieved / peak, 4),
        "required_bytes_per_step": step_bytes.total,
        "union": {"heads": n_u_h, "neurons": n_u_n},
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": round(dom_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(dom_gbs / peak, 4),
                     "traffic": profile_traffic(dom_name), "peak_source": peak_src,
                     "alg_bytes_per_launch": dom_bytes,
                     "launch_us": round(kern_ms * 1e3, 2)},
        "kernels_per_step": n_launch,
        "kernels": kernels,
        "traced_step_us": round(traced_step_ms * 1e3, 2),
        "persistent": persistent,
        "gpu_launches": args.steps * n_launch,
        "clocks": clocks,
    }

    if not args.no_extras:
        line.update(extras(args, dv, traffic, cfg, desc, layers, caches, x, sel, ws, stream,
                           rank, us_per_decode, k_h, k_n, B))
        del layers, caches
        torch.cuda.empty_cache()
        line["variants"] = variant_bench(dv, traffic, x.device, peak)
        if args.stack_layers > 0:
            torch.cuda.empty_cache()
            line["stack"] = stack_bench(args, dv, traffic, cfg, x.device)
    if rank == 0:
        print(json.dumps(line), flush=True)


def extras(args, dv, traffic, cfg, desc, layers, caches, x, sel, ws, stream, rank,
           us_per_decode, k_h, k_n, B):
    import numpy as np
    import torch

    out = {}
    copies = len(layers)
    # end to end through the C ABI with host activations (pinned), copies inside
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    ke = min(args.steps, 500)
    for i in range(min(5, ke)):
        kc, vc = caches[i % copies]
        dv.dv_layer_decode_host(layers[i % copies], xh, k_h, k_n, kc, vc, cfg.kv_len, yh, ws,
                                stream=stream)
    t = time.perf_counter()
    for i in range(ke):
        kc, vc = caches[i % copies]
        dv.dv_layer_decode_host(layers[i % copies], xh, k_h, k_n, kc, vc, cfg.kv_len, yh, ws,
                                stream=stream)
    e2e_us = (time.perf_counter() - t) * 1e6 / ke
    out["e2e"] = {"value": round(e2e_us, 3), "unit": "µs per layer-decode",
                  "h2d_bytes_per_step": int(xh.numel() * 4), "d2h_bytes_per_step": int(yh.numel() * 4),
                  "steps": ke, "api": "dv_layer_decode_host"}

    # dense-decode baseline: the same library with every head and neuron selected
    dsel = dv.SelectionBuffers(desc, B, cfg.n_heads, cfg.d_ffn)
    yd = torch.empty_like(x)
    kd = min(args.steps, 30)
    with torch.cuda.stream(stream):
        for i in range(3):
            kc, vc = caches[i % copies]
            dv.dv_layer_decode(layers[i % copies], x, cfg.n_heads, cfg.d_ffn, kc, vc, cfg.kv_len,
                               dsel, yd, ws, stream=stream)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(kd):
            kc, vc = caches[i % copies]
            dv.dv_layer_decode(layers[i % copies], x, cfg.n_heads, cfg.d_ffn, kc, vc, cfg.kv_len,
                               dsel, yd, ws, stream=stream)
        b.record(stream)
    b.synchronize()
    dense_us = a.elapsed_time(b) * 1e3 / kd
    dense_bytes = traffic.dense_step_bytes(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn,
                                           2 if cfg.dtype == "f16" else 4, B, cfg.kv_len)
    out["dense_baseline"] = {"us_per_decode": round(dense_us, 2),
                             "speedup_sparse": round(dense_us / us_per_decode, 3),
                             "bytes_per_step": dense_bytes,
                             "achieved_gbs": round(dense_bytes / (dense_us * 1e-6) / 1e9, 1),
                             "note": "same library, every head and neuron selected"}

    # blocked neuron selection (64-channel blocks, k rounded up to whole
    # blocks) on the same weights, timed like the step (graph replays)
    if cfg.d_ffn % 64 == 0 and B <= 2:
        blk = 64
        k_nb = -(-k_n // blk) * blk
        bdesc = dv.make_desc(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn, cfg.pred_rank,
                             desc.dtype, desc.kv_cap, desc.norm, desc.ln_eps, neuron_block=blk)
        blayers = [dv.Layer(bdesc, l.weights) for l in layers]
        bsel = dv.SelectionBuffers(bdesc, B, k_h, k_nb)
        yb = torch.empty_like(x)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(copies):  # warm, outside the capture
                kc, vc = caches[i]
                dv.dv_layer_decode(blayers[i], x, k_h, k_nb, kc, vc, cfg.kv_len, bsel, yb, ws,
                                   stream=stream)
            with torch.cuda.graph(g, stream=stream):
                for i in range(copies):
                    kc, vc = caches[i]
                    dv.dv_layer_decode(blayers[i], x, k_h, k_nb, kc, vc, cfg.kv_len, bsel, yb, ws,
                                       stream=stream)
            g.replay()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            reps = 10
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        b.synchronize()
        if dv.dv_check(ws, stream) != dv.DV_OK:
            raise RuntimeError("device status set by the blocked decode")
        blk_us = a.elapsed_time(b) * 1e3 / (reps * copies)
        bu_h, bu_n = bsel.unions()
        bbytes = traffic.sparse_step_bytes(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn,
                                           cfg.pred_rank, 2 if cfg.dtype == "f16" else 4, B,
                                           int(bu_h.numel()), int(bu_n.numel()), cfg.kv_len).total
        out["blocked_selection"] = {
            "block": blk, "k_neurons": k_nb, "union_neurons": int(bu_n.numel()),
            "us_per_decode": round(blk_us, 2),
            "achieved_gbs": round(bbytes / (blk_us * 1e-6) / 1e9, 1),
            "required_bytes_per_step": bbytes,
            "note": "neurons kept in 64-channel blocks (each scored by its largest member "
                    "score), same weights, graph replays of consecutive decodes"}
        del g, blayers

    # copy bandwidth of the library's own copy kernel (read + write bytes)
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, device=x.device)
    dst = torch.empty_like(src)
    with torch.cuda.stream(stream):
        for _ in range(3):
            dv.dv_hbm_copy(dst, src, stream=stream)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(10):
            dv.dv_hbm_copy(dst, src, stream=stream)
        b.record(stream)
    b.synchronize()
    out["copy_peak_gbs"] = round(2 * n * 10 / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
    del src, dst

    if rank == 0:
        out["cpu_baseline"] = cpu_baseline(cfg, layers[0], caches[0], x, k_h, k_n,
                                           args.cpu_budget_s)
    return out


def variant_bench(dv, traffic, device, peak):
    """The LLaMA-style layer (RMSNorm, SwiGLU MLP) at the LLaMA-3-70B shape of
    the guide's traffic arithmetic, batch 1, timed like the main step (graph
    replays of consecutive decodes over 4 layer copies)."""
    import torch

    import dv_inputs

    out = {}
    cfg = dv_inputs.CONFIGS["llama3_70b"]
    desc = dv.desc_from_config(cfg)
    k_h, k_n, copies, B = cfg.k_heads, cfg.k_neurons, 4, 1
    layers, caches = [], []
    for i in range(copies):
        layers.append(dv.Layer(desc, dv_inputs.make_weights(cfg, seed=200 + i, device=device)))
        caches.append(dv_inputs.make_kv(cfg, B, seed=200 + i, device=device))
    x = dv_inputs.make_x(cfg, B, seed=7, device=device)
    y = torch.empty_like(x)
    sel = dv.SelectionBuffers(desc, B, k_h, k_n)
    ws = dv.Workspace(desc, B)
    stream = torch.cuda.Stream(device=device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(copies):
            kc, vc = caches[i]
            dv.dv_layer_decode(layers[i], x, k_h, k_n, kc, vc, cfg.kv_len, sel, y, ws,
                               stream=stream)
        with torch.cuda.graph(g, stream=stream):
            for i in range(copies):
                kc, vc = caches[i]
                dv.dv_layer_decode(layers[i], x, k_h, k_n, kc, vc, cfg.kv_len, sel, y, ws,
                                   stream=stream)
        for _ in range(3):
            g.replay()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        reps = 10
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
    b.synchronize()
    if dv.dv_check(ws, stream) != dv.DV_OK:
        raise RuntimeError("device status set by the LLaMA-style decode")
    us = a.elapsed_time(b) * 1e3 / (reps * copies)
    u_h, u_n = sel.unions()
    req = traffic.sparse_step_bytes(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn,
                                    cfg.pred_rank, 2, B, int(u_h.numel()), int(u_n.numel()),
                                    cfg.kv_len, swiglu=True).total
    out["llama3_70b"] = {
        "us_per_decode": round(us, 2), "required_bytes_per_step": req,
        "achieved_gbs": round(req / (us * 1e-6) / 1e9, 1),
        "roofline_frac_step": round(req / (us * 1e-6) / 1e9 / peak, 4),
        "union": {"heads": int(u_h.numel()), "neurons": int(u_n.numel())},
        "config": {"d_model": cfg.d_model, "n_heads": cfg.n_heads, "head_dim": cfg.head_dim,
                   "d_ffn": cfg.d_ffn, "pred_rank": cfg.pred_rank, "kv_len": cfg.kv_len,
                   "batch": B, "norm": cfg.norm, "mlp": cfg.mlp, "k_heads": k_h,
                   "k_neurons": k_n},
        "note": "LLaMA-style layer (RMSNorm, SwiGLU with gate and up rows side by side), "
                "MHA with all 64 heads; graph replays of consecutive decodes, 4 layer copies"}
    del g, layers, caches
    torch.cuda.empty_cache()
    return out


def stack_bench(args, dv, traffic, cfg, device):
    """Tokens/s of an L-layer stack of this layer shape with the lookahead
    predictor (attention_dv_predict_gb300/stack.py), one CUDA graph per token
    step; at batch 1 also the chained modes for comparison."""
    import torch

    import dv_inputs
    from attention_dv_predict_gb300 import stack

    n = args.stack_layers
    desc = dv.desc_from_config(cfg)
    weights = stack.make_stack_weights(cfg, n, device=device, seed0=100)
    layers = stack.layers_from_weights(desc, weights)
    P = 2 if cfg.dtype == "f16" else 4
    out = {"layers": n, "shape": cfg.name, "kv_len": cfg.kv_len,
           "note": "layer l+1's selection predicted from layer l's input (overlap: on a side "
                   "stream beside the decode; fused: inside each layer's dv_layer_decode "
                   "call); one CUDA graph per token step; GB/s on the stack's required bytes",
           "batches": []}
    for B in [int(b) for b in args.stack_batches.split(",") if b]:
        caches = stack.stack_caches(cfg, n, B, device=device, seed0=100)
        x0 = dv_inputs.make_x(cfg, B, seed=5, device=device)
        st = stack.LayerStack(desc, layers, B, cfg.k_heads, cfg.k_neurons, device=device)
        st.keep_selection = True
        st.run(x0, caches, cfg.kv_len)
        req = sum(traffic.sparse_step_bytes(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn,
                                            cfg.pred_rank, P, B, int(k["n_u_h"].item()),
                                            int(k["n_u_n"].item()), cfg.kv_len).total
                  for k in st.kept)
        st.keep_selection = False
        entry = {"batch": B, "required_bytes": req}
        # the default mode (predictor on a side stream), plus the other two
        # at batch 1 for comparison
        modes = [("overlap", False)]
        if B == 1:
            modes += [("fused", True), ("serial", False)]
        entry["mode"] = modes[0][0]
        for mode, fused in modes:
            serial = mode == "serial"
            st.run(x0, caches, cfg.kv_len, serial=serial, fused=fused)
            cs = torch.cuda.Stream(device=device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs):
                st.enqueue(x0, caches, cfg.kv_len, serial=serial, fused=fused)
            reps = max(3, 40 // B)
            for _ in range(2):
                g.replay()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
            b.synchronize()
            ms = a.elapsed_time(b) / reps
            key = "" if mode == entry["mode"] else mode + "_"
            entry[key + "ms_per_token_step"] = round(ms, 4)
            entry[key + "tokens_per_s"] = round(B / (ms * 1e-3), 1)
            entry[key + "us_per_layer"] = round(ms * 1e3 / n, 2)
            if not key:
                entry["achieved_gbs"] = round(req / (ms * 1e-3) / 1e9, 1)
            del g
        out["batches"].append(entry)
        del caches, st
        torch.cuda.empty_cache()
    return out


def _oracle_inputs(cfg, layer, cache, x):
    import oracle

    w = {k: v.detach().cpu().numpy() for k, v in layer.weights.items()}
    D = oracle.desc_from_config(cfg)
    kc, vc = cache
    return D, w, kc.cpu().numpy(), vc.cpu().numpy(), x.cpu().numpy()


def _time_oracle(fn, budget_s, min_runs=3, max_runs=50):
    times = []
    t_end = time.perf_counter() + budget_s
    while True:
        t = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t)
        if len(times) >= max_runs or (time.perf_counter() >= t_end and len(times) >= min_runs):
            break
    return statistics.median(times) * 1e6, len(times)


def cpu_baseline(cfg, layer, cache, x, k_h, k_n, budget_s):
    """The CPU oracle (C, binary64) on the same workload: on every host core
    (the OpenMP build, same bits) and on one thread."""
    import oracle

    D, w, kc, vc, xh = _oracle_inputs(cfg, layer, cache, x)
    host = os.cpu_count() or 1

    def run(threads):
        return _time_oracle(lambda: oracle.layer_decode(D, w, xh, k_h, k_n, kc, vc, cfg.kv_len,
                                                        inplace=True, threads=threads),
                            budget_s / 2)

    us1, n1 = run(0)
    single = {"value": round(us1, 1), "cores": 1, "runs": n1}
    try:
        cores = oracle.threads_used(-1)
        usn, nn = run(-1)
    except RuntimeError:  # no OpenMP build on this host: the single-thread figure only
        return {"value": round(us1, 1), "unit": "µs per layer-decode", "cores": 1,
                "host_cores": host, "kind": "oracle", "single_thread": single,
                "sample": f"{n1} full layer decodes of the same {cfg.name} workload (median), "
                          "single-threaded C oracle (no OpenMP on this host)"}
    return {"value": round(usn, 1), "unit": "µs per layer-decode", "cores": cores,
            "host_cores": host, "kind": "oracle", "single_thread": single,
            "sample": f"{nn} full layer decodes of the same {cfg.name} workload (median) on "
                      f"{cores} threads (OpenMP build of the C oracle, same bits); "
                      f"single_thread: {n1} decodes on one thread"}


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch

    import dv_inputs
    import oracle
    from oracle import build as oracle_build

    oracle_build.build()
    cfg = dv_inputs.CONFIGS[args.config]
    B = args.batch or cfg.batch
    cfg = cfg.with_(batch=B)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = dv_inputs.make_weights(cfg, seed=0, device=gen_dev)
    kc, vc = dv_inputs.make_kv(cfg, B, seed=0, device=gen_dev)
    x = dv_inputs.make_x(cfg, B, seed=0, device=gen_dev)
    wn = {k: v.cpu().numpy() for k, v in w.items()}
    del w
    kch, vch, xh = kc.cpu().numpy(), vc.cpu().numpy(), x.cpu().numpy()
    D = oracle.desc_from_config(cfg)

    try:
        threads = -1
        cores = oracle.threads_used(threads)
    except RuntimeError:  # no OpenMP build on this host
        threads, cores = 0, 1

    def one():
        oracle.layer_decode(D, wn, xh, cfg.k_heads, cfg.k_neurons, kch, vch, cfg.kv_len,
                            inplace=True, threads=threads)

    budget = 150.0
    t = time.perf_counter()
    one()
    first = time.perf_counter() - t
    warm = min(args.warmup, max(0, int(20.0 / max(first, 1e-3))))
    for _ in range(max(0, warm - 1)):
        one()
    steps_run = max(1, min(args.steps, int(budget / max(first, 1e-3))))
    t = time.perf_counter()
    for _ in range(steps_run):
        one()
    sec = time.perf_counter() - t
    us = sec * 1e6 / steps_run
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1),
        "unit": "µs per layer-decode", "n_gpus": world, "steps": args.steps,
        "steps_run": steps_run, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(cfg, B),
        "cpu_baseline": {"value": round(us, 1), "unit": "µs per layer-decode", "cores": cores,
                         "host_cores": os.cpu_count() or 1, "kind": "oracle",
                         "sample": f"{steps_run} of the {args.steps} requested steps (bounded to "
                                   f"~{int(budget)} s), each one full layer decode on {cores} "
                                   f"thread(s)"},
        "e2e": {"value": round(us, 1), "unit": "µs per layer-decode", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "note": "the reference arm is the CPU oracle (no upstream code exists to install)",
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
