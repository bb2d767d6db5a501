#!/usr/bin/env python
"""Throughput of the window-attention KV selection path on GB300.

One step = the whole path over one batch of the workload: kvsel_score,
[kvsel_combine_layers], kvsel_topk, kvsel_compact (and kvsel_pagetable when
the workload has a block mask).  Default workload: LLaMA-3.1-8B shape, 32
layers, 32 / 8 heads, d = 128, 128K-token prefix, W = 32, max over the group,
page max P = 16, top 128 pages + 4 recent pages, compacted K/V.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the same metric instead (a bounded sample of the workload per step).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefix tokens scored+selected/s (per layer, 128K ctx); % of HBM/TC roofline"
DEFAULT_WORKLOAD = "llama8b_32l_h32x8_d128_L131072_W32_paged16"
HBM_FALLBACK_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="kvsel", choices=["kvsel", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--layers", type=int, default=0,
                   help="run only this many layers of the workload (small cases for profiler captures)")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--cpu-units", type=int, default=0,
                   help="(layer, KV head) units in the CPU-baseline sample (default: one per host core)")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--attend", action="store_true",
                   help="time attention over the selected pages in place (page table) against compact + dense")
    p.add_argument("--n-q", type=int, default=1, help="query rows per head for --attend")
    p.add_argument("--prefill", action="store_true",
                   help="time causal prefill attention and the selection scored from its lse (one pass) "
                        "against the selection scored with two passes")
    return p.parse_args()


# ----------------------------------------------------------------------------- oracle (CPU) leg

def _oracle_unit(args):
    """The oracle's whole path for one unit; returns seconds spent.

    A unit is one (layer, KV head) — or, for selections shared by every KV head,
    one layer with all its KV heads (q_group [h_kv, G, W, d], k_unit / v_unit
    [h_kv, L + W, d]).
    """
    wd, q_group, k_unit, v_unit = args
    import numpy as np
    from oracle import kvsel_oracle as O
    t0 = time.perf_counter()
    L, W, P = wd["L"], wd["W"], wd["P"]
    Wapp = W if wd["append"] else 0
    if wd["all_heads"]:
        raw = [O.group_scores(O._f64(q_group[g]), O._f64(k_unit[g]), L, wd["reduce"], wd["softmax"])
               for g in range(len(q_group))]
        u = O.pool(O.head_sum(np.stack(raw)), wd["pool_k"], wd["pool_type"])
        sel = O.select_tokens(u, wd["k"], L, Wapp)
        for g in range(len(q_group)):
            O.gather_rows(O._f64(k_unit[g]), sel, P)
            O.gather_rows(O._f64(v_unit[g]), sel, P)
        return time.perf_counter() - t0
    s = O.group_scores(O._f64(q_group), O._f64(k_unit), L, wd["reduce"], wd["softmax"])
    u = O.pool(s, wd["pool_k"], wd["pool_type"])
    if P > 1:
        U = O.page_reduce(u, P, wd["page_reduce"])
        sel = O.select_pages(U, wd["k"], wd["n_recent"], L, Wapp, P)
    else:
        sel = O.select_tokens(u, wd["k"], L, Wapp)
    O.gather_rows(O._f64(k_unit), sel, P)
    O.gather_rows(O._f64(v_unit), sel, P)
    return time.perf_counter() - t0


def _pool_init():
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"


def _all_heads(w):
    return w.head_reduce == "all" or w.claa is not None


def _k_keep(w):
    return keep_count(w.claa[3], w.prefix_lens[0]) if w.claa is not None else w.k_keep


def keep_count(rate, L):
    from oracle.kvsel_oracle import keep_count as kc      # the CPU leg takes k from the oracle
    return kc(rate, L)


def oracle_rate(w, units, pool, cores):
    """Prefix tokens per second per layer of the oracle over ``units`` = [(q_group, k_unit, v_unit)]."""
    wd = dict(L=w.prefix_lens[0], W=w.window, P=w.page_size, G=w.group, h_kv=w.h_kv, reduce=w.group_reduce,
              pool_k=w.pool_k, page_reduce=w.page_reduce, k=_k_keep(w), n_recent=w.n_recent,
              softmax=w.score_mode == "softmax", pool_type=w.pool_type, append=w.append_window,
              all_heads=_all_heads(w))
    t0 = time.perf_counter()
    pool.map(_oracle_unit, [(wd, q, k, v) for (q, k, v) in units], chunksize=1)
    wall = time.perf_counter() - t0
    per_unit_layers = 1.0 if _all_heads(w) else 1.0 / w.h_kv
    tokens_layers = len(units) * per_unit_layers * w.prefix_lens[0]
    return tokens_layers / wall, wall


def oracle_units(w, q, kk, vv, layers, count):
    """``count`` oracle units cycled over ``layers`` (per-sequence q [n_layers, ...], kk / vv per layer)."""
    G = w.group
    units = []
    for i in range(count):
        if _all_heads(w):
            layer = layers[i % len(layers)]
            qg = q[layer].reshape(w.h_kv, G, w.window, w.head_dim)
            units.append((qg.cpu(), kk(layer).cpu(), vv(layer).cpu()))
        else:
            layer, g = divmod(i, w.h_kv)
            layer = layers[layer % len(layers)]
            units.append((q[layer, g * G:(g + 1) * G].cpu(), kk(layer)[g].cpu(), vv(layer)[g].cpu()))
    return units


def make_pool(cores):
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(cores, initializer=_pool_init)
    pool.map(time.sleep, [0.0] * cores)       # start the workers before timing
    return pool


# ----------------------------------------------------------------------------- measurement helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return HBM_FALLBACK_GBS, "fallback"


CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(REASONS, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_bytes(w, n_sel_rows, n_layers=None):
    """Algorithmic HBM bytes of one launch of each kernel (the whole workload per launch); n_layers = the
    layers one launch covers (default: all of the workload's)."""
    d, W = w.head_dim, w.window
    nl = w.n_layers if n_layers is None else n_layers
    units = [(nl * w.h_kv, L) for L in w.prefix_lens]
    q_bytes = w.batch * nl * w.h_q * W * d * 2
    k_all = sum(u * (L + W) * d * 2 for u, L in units)
    k_prefix = sum(u * L * d * 2 for u, L in units)
    score_w = sum(u * L * 4 for u, L in units)
    P = w.page_size
    page_w = sum(u * (-(-L // P)) * 4 for u, L in units) if P > 1 else 0
    sel_read = page_w if P > 1 else score_w
    idx_w = w.batch * nl * w.h_kv * w.n_sel() * 4
    gather = 2 * 2 * w.batch * nl * w.h_kv * n_sel_rows * d * 2
    pass1 = k_all + q_bytes
    pass2 = k_prefix + q_bytes + score_w + page_w
    return {
        "score_pass1_simt": pass1, "score_pass1_tc": pass1,
        "score_pass2_simt": pass2, "score_pass2_tc": pass2,
        "topk_radix": sel_read + idx_w,
        "kv_compact": gather + idx_w,
    }


def kernel_flops(w, n_layers=None):
    """Algorithmic tensor flops of one launch of the scoring kernels: Q K^T of the window rows against
    every key of the pass (2 flops per multiply-add)."""
    d, W = w.head_dim, w.window
    nl = w.n_layers if n_layers is None else n_layers
    rows = nl * w.h_q * W
    pass1 = sum(2 * rows * (L + W) * d for L in w.prefix_lens)
    pass2 = sum(2 * rows * L * d for L in w.prefix_lens)
    return {"score_pass1_tc": pass1, "score_pass2_tc": pass2}


def alu_peak_tflops():
    """fp32 FMA peak of the CUDA-core scoring kernels: 152 SMs x 128 FMA lanes x 2 flops x the maximum SM
    clock in MEASURED_PEAKS.json (2070 MHz when absent): 80.5 TFLOP/s on a GB300."""
    mhz = 2070.0
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def traffic_record(kernel):
    """dram bytes per launch from the committed ncu summary, if taken on the kernel's current source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and parts[0] == kernel and not line.startswith("#"):
                src, digest = parts[2].split(":")
                with open(os.path.join(ROOT, "attention_kv_cache_gb300", "csrc", src), "rb") as g:
                    if hashlib.sha256(g.read()).hexdigest()[:12] != digest:
                        return None
                return float(parts[1])
    return None


# ----------------------------------------------------------------------------- distributed plumbing

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- the CUDA path

def run_kvsel(args):
    import torch
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300 import synth as S
    from attention_kv_cache_gb300.pipeline import ClaaPipeline, Pipeline, pack

    rank, world, local = dist_setup()
    w = S.by_name(args.workload)
    if args.layers:
        w = S.scaled(w, n_layers=args.layers)
        if w.claa is not None:
            m, lp, nbuf, rate = w.claa
            w = w.with_(claa=(min(m, args.layers - 1), args.layers - 1, nbuf, rate))
    n_cpu_units = args.cpu_units or (os.cpu_count() or 1)
    cores = min(os.cpu_count() or 1, n_cpu_units)
    pool = make_pool(cores) if (rank == 0 and world == 1 and not args.no_cpu) else None  # before any GPU call

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = S.make_inputs(w, str(dev))
    q, k, v = pack(inp, dev)
    mask = inp.mask
    nkv = inp.n_kvblk
    claa = w.claa is not None
    pipe = ClaaPipeline(w, dev) if claa else Pipeline(w, dev)
    stream = torch.cuda.current_stream(dev)
    scored_layers = pipe.n_sc if claa else w.n_layers

    def run_step(v_src=None):
        vs = v if v_src is None else v_src
        if claa:
            pipe.run(q, k, vs)
        else:
            pipe.run(q, k, vs, mask, nkv)

    for _ in range(args.warmup):
        run_step()
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(pipe.ws) == K.OK

    # ---- timed region: inputs (K/V) are far larger than L2, so every step streams them from HBM
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    K.kvsel_trace_enable(True)
    K.kvsel_trace_read()
    n0 = K.kvsel_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        run_step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = K.kvsel_launch_count() - n0
    trace = K.kvsel_trace_read()
    K.kvsel_trace_enable(False)
    clocks = sampler.stop()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    assert K.kvsel_read_device_error(pipe.ws) == K.OK

    tokens_per_step = sum(L for L in w.prefix_lens) * scored_layers
    value = world * tokens_per_step * args.steps / (ms / 1e3)

    # ---- roofline of the dominant kernel (largest share of the timed region)
    name, (n_launch, k_ms) = max(trace.items(), key=lambda kv: kv[1][1])
    bytes_per_launch = kernel_bytes(w, pipe.n_sel * w.page_size, scored_layers).get(name)
    flops_per_launch = kernel_flops(w, scored_layers).get(name)
    peak, peak_src = measured_peaks()
    tc_peak, tc_src = measured_tensor_peak()
    roof = None
    t_launch = k_ms / n_launch / 1e3
    # the roofline is the larger of the HBM time and the tensor time at the measured peaks (with 256
    # window rows per unit, as in the 70B-shaped workload, the two are about equal)
    alu_flops = kernel_flops(w, scored_layers).get(name.replace("_simt", "_tc")) if name.endswith("_simt") else None
    if alu_flops is not None and bytes_per_launch is not None and \
            alu_flops / (alu_peak_tflops() * 1e12) > bytes_per_launch / (peak * 1e9):
        # the CUDA-core kernels make the logits with fp32 FMA: bound by that rate, not by HBM
        achieved = alu_flops / t_launch / 1e12
        roof = {"bound": "alu", "kernel": name, "achieved": round(achieved, 1), "peak": round(alu_peak_tflops(), 1),
                "unit": "TFLOP/s", "frac": round(achieved / alu_peak_tflops(), 4),
                "peak_source": "fp32 FMA lanes x SM clock", "traffic": None, "algorithmic_flops": alu_flops,
                "algorithmic_bytes": bytes_per_launch, "hbm_frac": round(bytes_per_launch / t_launch / 1e9 / peak, 4),
                "share": round(k_ms / sum(x[1] for x in trace.values()), 4)}
    elif (bytes_per_launch is not None and flops_per_launch is not None
            and flops_per_launch / (tc_peak * 1e12) > bytes_per_launch / (peak * 1e9)):
        achieved = flops_per_launch / t_launch / 1e12
        roof = {"bound": "tensor", "kernel": name, "achieved": round(achieved, 1), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(achieved / tc_peak, 4), "peak_source": tc_src, "traffic": None,
                "algorithmic_flops": flops_per_launch, "algorithmic_bytes": bytes_per_launch,
                "hbm_frac": round(bytes_per_launch / t_launch / 1e9 / peak, 4),
                "share": round(k_ms / sum(x[1] for x in trace.values()), 4)}
    elif bytes_per_launch is not None:
        achieved = bytes_per_launch / t_launch / 1e9
        roof = {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_src,
                # the committed traffic record is per launch of the full 128K paged workload
                "traffic": traffic_record(name) if (w.name == DEFAULT_WORKLOAD and not args.layers) else None,
                "algorithmic_bytes": bytes_per_launch,
                "share": round(k_ms / sum(x[1] for x in trace.values()), 4)}

    # ---- end to end through the C ABI with host buffers (copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        qh = q.cpu().pin_memory()
        kh = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
        kh.copy_(k)
        vh = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
        vh.copy_(v)
        outs = [pipe.idx, pipe.k_out, pipe.v_out] + ([pipe.kv_indptr, pipe.kv_indices] if mask is not None else [])
        if claa:
            outs.append(pipe.prune_idx)
        outs_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        mask_h = mask.cpu().pin_memory() if mask is not None else None

        # Q and K cross the host link whole (every key is scored, K is read twice); V stays in
        # pinned host memory and the compaction kernel reads only its kept rows over the link
        def e2e_step():
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            if mask is not None:
                mask.copy_(mask_h, non_blocking=True)
            run_step(vh)
            for o, oh in zip(outs, outs_h):
                oh.copy_(o, non_blocking=True)

        # the first passes over a freshly pinned multi-GB buffer run slower (69 and 56 ms instead of
        # 41 ms for 8.6 GB): warm up as many steps as the kernel-only leg does
        for _ in range(max(args.warmup, 3)):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), world, dev)
        # V's share: every row of the compacted V (an upper bound: page-mode rows past the cache are not read)
        v_read = pipe.v_out.numel() * pipe.v_out.element_size()
        h2d = q.numel() * 2 + k.numel() * 2 + v_read + (mask.numel() if mask is not None else 0)
        d2h = sum(o.numel() * o.element_size() for o in outs)
        e2e = {"value": world * tokens_per_step * args.e2e_steps / (ems / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "v_source": "pinned host memory, kept rows read by the compaction kernel"}

    # ---- CPU baseline: the oracle on a bounded sample of the same workload (rank 0, N = 1)
    cpu = None
    if pool is not None:
        layers = list(range(pipe.m, pipe.lp + 1)) if claa else list(range(w.n_layers))
        units = oracle_units(w, inp.q[0], lambda l: inp.k[0][l], lambda l: inp.v[0][l], layers, n_cpu_units)
        rate, wall = oracle_rate(w, units, pool, cores)
        what = "layers (all KV heads)" if _all_heads(w) else "(layer, KV head) units"
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{len(units)} {what} of the same workload, full path per unit, "
                         f"{wall:.1f} s wall on {cores} worker processes (1 BLAS thread each)"}
        pool.close()

    if rank == 0:
        line = {
            "metric": metric_for(w), "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 inputs, f32 arithmetic", "data": "synthetic",
            "config": {"workload": w.name, "layers": w.n_layers, "h_q": w.h_q, "h_kv": w.h_kv, "d": w.head_dim,
                       "prefix_len": list(w.prefix_lens), "window": w.window, "group_reduce": w.group_reduce,
                       "pool_k": w.pool_k, "pool_type": w.pool_type, "score_mode": w.score_mode,
                       "head_reduce": w.head_reduce, "claa": w.claa, "scored_layers": scored_layers,
                       "page_size": w.page_size, "k_keep": _k_keep(w), "n_recent": w.n_recent,
                       "l2": "inputs exceed L2 (K+V %.1f GB per step)" % ((k.numel() + v.numel()) * 2 / 1e9),
                       "parallelism": f"replicas x{world}"},
            "clocks": clocks, "gpu_launches": launches, "kernels": {n: {"launches": c, "ms": round(t, 3)}
                                                                   for n, (c, t) in trace.items()},
            "roofline": roof, "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _ctx(w):
    """Prefix length(s) of a workload for its metric name: '64K', '512', or a range for a ragged batch."""
    def f(L):
        return f"{L // 1024}K" if L >= 1024 else str(L)
    lo, hi = min(w.prefix_lens), max(w.prefix_lens)
    return f(lo) if lo == hi else f"{f(lo)}-{f(hi)}"


def metric_for(w):
    if w.name == DEFAULT_WORKLOAD:
        return METRIC
    return f"prefix tokens scored+selected/s (per layer, {_ctx(w)} ctx, {w.name})"


# ----------------------------------------------------------------------------- attention over the selection

def run_attend(args):
    """Decode-style attention over the selected pages: read in place through the page table
    (CompactAttention's zero-copy execution, DELTA's sparse layers) against the copy path (compact,
    then dense attention over the compacted cache)."""
    import torch
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300 import synth as S
    from attention_kv_cache_gb300.pipeline import Pipeline, pack

    w = S.by_name(args.workload)
    if args.layers:
        w = S.scaled(w, n_layers=args.layers)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = S.make_inputs(w, str(dev))
    q, k, v = pack(inp, dev)
    pipe = Pipeline(w, dev)
    pipe.run(q, k, v, inp.mask, inp.n_kvblk)
    n_q = args.n_q
    qd = S.make_decode_queries(w, n_q, str(dev))
    P, n_sel = w.page_size, pipe.n_sel
    o = torch.empty((w.batch, w.n_layers, w.h_q, n_q, w.head_dim), dtype=torch.float32, device=dev)

    def ws_for(desc, max_blocks):
        n = K.kvsel_attend_workspace_size(desc, n_q, P, max_blocks)
        buf = torch.zeros(n + K.WS_ALIGN, dtype=torch.uint8, device=dev)
        off = (-buf.data_ptr()) % K.WS_ALIGN
        return buf[off:off + n]

    ws_a = ws_for(pipe.desc, n_sel)
    rows = n_sel * P
    dc = K.make_desc(n_layers=w.n_layers, h_q=w.h_q, h_kv=w.h_kv, head_dim=w.head_dim, window=w.window,
                     prefix_lens=[rows - w.window])
    ws_c = ws_for(dc, n_sel)
    oc = torch.empty_like(o)
    kc, vc = pipe.k_out.reshape(-1), pipe.v_out.reshape(-1)

    def in_place():
        K.kvsel_attend(pipe.desc, qd, n_q, k, v, None, pipe.idx, n_sel, P, n_sel, o, ws_a)

    def copy_path():
        pipe.compact(k, v)
        K.kvsel_attend(dc, qd, n_q, kc, vc, None, None, 0, P, n_sel, oc, ws_c)

    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, fn in (("in_place", in_place), ("copy", copy_path)):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        sampler = ClockSampler(0)
        K.kvsel_trace_enable(True)
        K.kvsel_trace_read()
        n0 = K.kvsel_launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        trace = K.kvsel_trace_read()
        K.kvsel_trace_enable(False)
        res[name] = {"ms": e0.elapsed_time(e1) / args.steps, "launches": K.kvsel_launch_count() - n0,
                     "clocks": sampler.stop(),
                     "kernels": {n: {"launches": c, "ms": round(t, 4)} for n, (c, t) in trace.items()}}
    assert K.kvsel_read_device_error(ws_a) == K.OK
    units = w.batch * w.n_layers * w.h_kv
    kv_rows = units * rows                                  # selected cache rows attended per step
    att_bytes = kv_rows * 2 * w.head_dim * 2 + qd.numel() * 2
    c_att = res["in_place"]["kernels"]["attend_split"]
    att_ms = c_att["ms"] / c_att["launches"]
    peak, peak_src = measured_peaks()
    achieved = att_bytes / (att_ms / 1e3) / 1e9
    line = {
        "metric": f"selected KV rows attended/s (decode, n_q={n_q}, in place through the page table)",
        "value": kv_rows / (res["in_place"]["ms"] / 1e3), "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["in_place"]["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 inputs, f32 arithmetic", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.n_layers, "pages_per_row": n_sel, "page_size": P,
                   "rows_per_step": kv_rows, "l2": "selected K+V %.0f MB per step" % (kv_rows * 512 / 1e6)},
        "clocks": res["in_place"]["clocks"], "gpu_launches": res["in_place"]["launches"],
        "kernels": res["in_place"]["kernels"],
        "roofline": {"bound": "hbm", "kernel": "attend_split", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_src, "traffic": None,
                     "algorithmic_bytes": att_bytes},
        "copy_path": {"ms_per_step": res["copy"]["ms"], "kernels": res["copy"]["kernels"],
                      "in_place_speedup": res["copy"]["ms"] / res["in_place"]["ms"]},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- prefill with the window scores

def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["bf16_tflops_sustained"]), "measured (sustained)"
    return 1700.0, "fallback (sustained)"


def run_prefill(args):
    """Causal prefill attention of every prompt row (tensor cores), then the selection path scored from
    the prefill's lse (one pass over the prefix keys), against the same selection scored with its own
    two passes."""
    import torch
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300 import synth as S
    from attention_kv_cache_gb300.pipeline import Pipeline, pack

    w = S.by_name(args.workload if args.workload != DEFAULT_WORKLOAD else "llama8b_32l_h32x8_d128_L32768_W32")
    w = w.with_(n_layers=args.layers or 4)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = S.make_inputs(w, str(dev))
    _, k, v = pack(inp, dev)
    q = torch.cat([S.make_prompt_queries(w, b, str(dev)).reshape(-1) for b in range(w.batch)])
    o = torch.empty_like(q)
    G, W = w.group, w.window
    lse_win = torch.empty((w.batch, w.n_layers, w.h_kv, G * W), dtype=torch.float32, device=dev)
    q_win = torch.empty((w.batch, w.n_layers, w.h_q, W, w.head_dim), dtype=torch.bfloat16, device=dev)
    pipe = Pipeline(w, dev)

    def prefill():
        K.kvsel_prefill_attention(pipe.desc, q, k, v, o, None, lse_win, q_win, pipe.ws)

    def fused():
        prefill()
        K.kvsel_score_from_lse(pipe.desc_score, q_win, k, lse_win, pipe.scores, pipe.page_scores, pipe.ws,
                               pipe.ws_bytes)
        pipe.select()
        pipe.compact(k, v)

    def unfused():
        prefill()
        pipe.run(q_win, k, v)

    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, fn in (("prefill", prefill), ("fused", fused), ("unfused", unfused)):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        sampler = ClockSampler(0)
        K.kvsel_trace_enable(True)
        K.kvsel_trace_read()
        n0 = K.kvsel_launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        trace = K.kvsel_trace_read()
        K.kvsel_trace_enable(False)
        res[name] = {"ms": e0.elapsed_time(e1) / args.steps, "launches": K.kvsel_launch_count() - n0,
                     "clocks": sampler.stop(),
                     "kernels": {n: {"launches": c, "ms": round(t, 4)} for n, (c, t) in trace.items()}}
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    # causal flops: Q K^T and P V over keys t <= i, 2 flops per multiply-add
    flops = sum(4.0 * w.n_layers * w.h_q * (L + W) * (L + W + 1) / 2 * w.head_dim for L in w.prefix_lens)
    # the committed traffic record is per launch of 4 layers of the 32K LLaMA-8B prompt
    rec = traffic_record("prefill_tc") if w.name == "llama8b_32l_h32x8_d128_L32768_W32" else None
    prefill_traffic = rec * w.n_layers / 4 if rec is not None else None
    pf = res["prefill"]["kernels"]["prefill_tc"]
    pf_ms = pf["ms"] / pf["launches"]
    peak, peak_src = measured_tensor_peak()
    achieved = flops / (pf_ms / 1e3) / 1e12
    tokens = sum(L for L in w.prefix_lens) * w.n_layers

    def sel_ms(name):   # selection kernels per step (their event times; the prefill's dwarfs the difference)
        return sum(v["ms"] for n, v in res[name]["kernels"].items() if n != "prefill_tc") / args.steps

    line = {
        "metric": "causal prefill attention TFLOP/s (bf16 in, fp32 accumulate), with the window scores' lse",
        "value": achieved, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res["prefill"]["ms"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 inputs, f32 accumulate", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.n_layers, "h_q": w.h_q, "h_kv": w.h_kv, "d": w.head_dim,
                   "prompt_len": [L + W for L in w.prefix_lens], "causal_flops_per_step": flops},
        "clocks": res["prefill"]["clocks"], "gpu_launches": res["prefill"]["launches"],
        "kernels": res["prefill"]["kernels"],
        "roofline": {"bound": "tensor", "kernel": "prefill_tc", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "traffic": prefill_traffic, "algorithmic_flops": flops},
        "selection_after_prefill": {
            "fused_ms_per_step": res["fused"]["ms"], "unfused_ms_per_step": res["unfused"]["ms"],
            "fused_kernels": res["fused"]["kernels"], "unfused_kernels": res["unfused"]["kernels"],
            "selection_ms_fused": sel_ms("fused"), "selection_ms_unfused": sel_ms("unfused"),
            "prefix_tokens_per_s_fused": tokens / (sel_ms("fused") / 1e3)},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- the oracle arm

def run_reference(args):
    """The fp64 oracle on the host cores: each step is one (layer, KV head) unit of the workload (the
    path's smallest independent piece), and the steps run concurrently on one worker process per core."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from attention_kv_cache_gb300 import synth as S
    w = S.by_name(args.workload)
    cores = min(os.cpu_count() or 1, max(1, args.steps))
    pool = make_pool(cores)
    q = S.make_queries(w, 0, "cpu")
    layer0 = w.claa[0] if w.claa is not None else 0
    kk, vv, _ = S.make_layer(w, 0, layer0, q, "cpu")
    units = oracle_units(w, q, lambda l: kk, lambda l: vv, [layer0], max(args.steps, args.warmup, 1))
    if args.warmup > 0:
        oracle_rate(w, units[:min(args.warmup, cores)], pool, cores)
    value, wall = oracle_rate(w, units[:args.steps], pool, cores)
    line = {
        "impl": "reference", "metric": metric_for(w), "value": value, "unit": "tokens/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name,
                   "sample_per_step": "one (layer, KV head) unit: scores, pooling, page scores, selection, gather"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} units of layer {layer0} (cycled over its {w.h_kv} KV heads, or the "
                                   f"whole layer for all-head selection), {wall:.1f} s wall on {cores} worker processes"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    pool.close()
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.attend:
        run_attend(a)
    elif a.prefill:
        run_prefill(a)
    else:
        run_kvsel(a)
