"""Benchmark: mixed-batch paged attention on GB300 through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pps|reference]

One step = the whole hot path over one batch: kv_append of the step's new
rows, attn_plan on the host, attn_run (bandwidth tasks, tensor-core tasks,
partial merge).  Default workload: 256 decode requests, 32/8 heads, head_dim
128, page_size 16, cached length uniform in [512, 4096], seed 1 (2.4 GB of KV,
larger than the 129 MB L2, so no flush is needed between steps).

Prints one JSON line.  ``value`` is tokens/s with inputs resident in HBM;
``e2e`` is the same metric with every step's inputs copied from pinned host
memory and the output copied back inside the timed region.  Under torchrun
each rank runs its own batch (weak scaling, no data-path collective).
``--impl reference`` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

DESCRIPTIONS = {
    "decode_heavy": "256 decode requests (q_len 1), Hq/Hkv 32/8, head_dim 128, page_size 16, "
                    "cached kv uniform [512,4096], no sharing, scattered pages, seed 1",
    "radix_sharing": "64 decode requests in 8 radix subtrees (2048-token root x8 members, "
                     "512-token branch per pair, private tails U[64,1024]), 32/8, d 128, P 16, seed 2",
    "mixed_budget": "8192-token budget: prefill 2048 on 1024 cached + 24 verify rows q U[4,8] + "
                    "~6000 decode rows, cached lognormal(7,1) clipped [16,16384], 32/8, d 128, P 16, seed 3",
    "long_prefill": "4 requests x 32768 tokens as 4 causal chunks of 8192, 32/8, d 128, P 64, seed 4",
    "tiny_mixed": "4 requests 8/2 heads d 64 P 16, cached {37,64,100,129} sharing a 32-token prefix, "
                  "q {1,1,4,16}, seed 0",
    "tree_verify": "128 requests each verifying a 64-token random draft tree (parent of token j "
                   "uniform in [0, j)), cached kv uniform [512,4096], 32/8, d 128, P 16, seed 5",
}
METRIC = "attention tokens/s and achieved HBM GB/s / tensor TFLOPS vs GB300 roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(x: float, world: int, device) -> float:
    """Max of a per-rank float across ranks (identity when world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while a region runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index, self.period_ms = index, period_ms
        self.lines, self.proc, self.t0, self.t1 = [], None, None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._th = threading.Thread(target=self._read, daemon=True)
            self._th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(self.period_ms / 1000 * 2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [(t, l.split(", ")) for t, l in self.lines]
        inside = [r for t, r in rows if self.t0 and self.t1 and self.t0 <= t <= self.t1 + 0.1]
        sample = inside if len(inside) >= 3 else [r for _, r in rows]
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in sample:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names[1:], r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons),
                "samples": len(sample),
                "samples_in_timed_region": len(inside)}


def traffic_record(kernel_file: str, workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, valid only while the
    kernel's source is unchanged (sha256 recorded beside the figure)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(f"{kernel_file}:{workload}")
    if not rec:
        return None
    src = os.path.join(ROOT, "paged_prefix_shared_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return rec["dram_bytes_per_launch"] if rec.get("source_sha256") == sha else None


# ---------------------------------------------------------------------------


def run_pps(args):
    import numpy as np
    import torch

    import paged_prefix_shared_gb300 as pps
    import workloads

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pps.build()
    pps.lib()

    if args.workload == "decode_heavy":
        wl = workloads.decode_heavy(seed=1 + 1000 * rank, device=dev,
                                    num_requests=args.requests or 256)
    elif args.workload == "long_prefill" and args.requests:
        wl = workloads.long_prefill(device=dev, num_requests=args.requests)
    elif args.workload == "tree_verify" and args.requests:
        wl = workloads.tree_verify(device=dev, num_requests=args.requests)
    else:
        wl = workloads.make(args.workload, device=dev)
    # device-resident inputs
    # The library appends into a copy; the drawn pool stays as the generator
    # made it (the CPU baseline starts from it).  Re-appending the same rows
    # every step is idempotent.
    pk, pv = wl.pool_k.clone(), wl.pool_v.clone()
    steps = []
    for st in wl.steps:
        L = st.layout
        tabs = {n: torch.as_tensor(getattr(L, n), dtype=torch.int32, device=dev)
                for n in ("q_indptr", "cached_len", "page_indptr", "page_indices")}
        out = torch.empty_like(st.q)
        plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                             L.num_kv_heads, L.head_dim, L.page_size, L.num_pages,
                             tree_parent=L.tree_parent)
        info = plan.info()
        ws = torch.empty(info["workspace_bytes"], dtype=torch.uint8, device=dev)
        steps.append(dict(L=L, st=st, tabs=tabs, out=out, ws=ws, info=info))
    stream = torch.cuda.current_stream()
    nk = pps.NUM_KERNEL_CLASSES

    def one_step(ev=None):
        for i, s in enumerate(steps):
            L, st, t = s["L"], s["st"], s["tabs"]
            pps.kv_append(pk, pv, st.k_new, st.v_new, t["q_indptr"], t["cached_len"],
                          t["page_indptr"], t["page_indices"])
            plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                                 L.num_q_heads, L.num_kv_heads, L.head_dim, L.page_size,
                                 L.num_pages, tree_parent=L.tree_parent)
            pps.attn_run(plan, st.q, pk, pv, s["out"], s["ws"],
                         events=None if ev is None else ev[i])

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()

    # per-kernel events (one set per step per chunk) -> average launch duration
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)] for _ in steps]
          for _ in range(args.steps)]
    for per_step in ev:                 # torch creates events on first record: do it now,
        for per_chunk in per_step:      # outside the timed region
            for e in per_chunk:
                e.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    n_launch0 = pps.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark("t0")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(args.steps):
        one_step(ev[k])
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    barrier(world)
    launches = pps.launch_count() - n_launch0
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    kern_ms = [0.0] * nk
    for k in range(args.steps):
        for i in range(len(steps)):
            for c in range(nk):
                kern_ms[c] += ev[k][i][2 * c].elapsed_time(ev[k][i][2 * c + 1])
    kern_ms = [x / args.steps for x in kern_ms]        # per step (summed over chunks)

    # ---- kernel times with a cold L2 (KV that L2 could partly hold) -----------------------
    # Each step is preceded by a write of a buffer four times the L2 size; only the
    # per-kernel events count, so the flush itself is never timed.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129e6)
    kv_unique0 = sum(s["info"]["kv_bytes_unique"] for s in steps)
    flush = args.flush_l2 == "on" or (args.flush_l2 == "auto" and kv_unique0 < 4 * l2_bytes)
    cold_ms = None
    if flush:
        fbuf = torch.empty(4 * l2_bytes // 4, dtype=torch.int32, device=dev)
        cold = [0.0] * nk
        for k in range(args.steps):
            fbuf.fill_(k)
            one_step(ev[k])
        torch.cuda.synchronize()
        for k in range(args.steps):
            for i in range(len(steps)):
                for c in range(nk):
                    cold[c] += ev[k][i][2 * c].elapsed_time(ev[k][i][2 * c + 1])
        cold_ms = [x / args.steps for x in cold]
        del fbuf
    roof_ms = cold_ms if cold_ms is not None else kern_ms

    tokens = sum(s["L"].num_tokens for s in steps)
    total_tokens = sum_over_ranks(tokens, world, dev)
    value = total_tokens / (ms_max / 1e3)

    # ---- e2e: host buffers in, host result out, through the public API -------------------
    h = []
    for s in steps:
        st = s["st"]
        host = {n: st.__dict__[n].cpu().pin_memory() for n in ("q", "k_new", "v_new")}
        host.update({n: v.cpu().pin_memory() for n, v in s["tabs"].items()})
        dv = {n: torch.empty_like(v, device=dev) for n, v in host.items()}
        h.append(dict(host=host, dev=dv, out_h=torch.empty_like(s["out"], device="cpu").pin_memory()))
    bi = sum(v.numel() * v.element_size() for x in h for v in x["host"].values())
    bo = sum(x["out_h"].numel() * x["out_h"].element_size() for x in h)

    def e2e_step():
        for s, x in zip(steps, h):
            L = s["L"]
            for n, v in x["host"].items():
                x["dev"][n].copy_(v, non_blocking=True)
            d = x["dev"]
            pps.kv_append(pk, pv, d["k_new"], d["v_new"], d["q_indptr"], d["cached_len"],
                          d["page_indptr"], d["page_indices"])
            plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                                 L.num_q_heads, L.num_kv_heads, L.head_dim, L.page_size,
                                 L.num_pages, tree_parent=L.tree_parent)
            pps.attn_run(plan, d["q"], pk, pv, s["out"], s["ws"])
            x["out_h"].copy_(s["out"], non_blocking=True)

    for _ in range(max(3, args.warmup // 4)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    k_e2e = max(3, args.steps // 2)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(k_e2e):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_e2e = max_over_ranks(f0.elapsed_time(f1) / k_e2e, world, dev)
    e2e_value = total_tokens / (ms_e2e / 1e3)

    # ---- roofline of the dominant kernel ------------------------------------------------
    peaks, peak_src = load_peaks()
    infos = [s["info"] for s in steps]
    dom = int(np.argmax(roof_ms))
    L0 = steps[0]["L"]
    qo_bytes = sum(2 * s["L"].num_tokens * L0.num_q_heads * L0.head_dim * 2 for s in steps)
    kv_unique = sum(i["kv_bytes_unique"] for i in infos)
    kv_bw = sum(i["kv_bytes_bw"] for i in infos)            # K/V read by bandwidth tasks
    flops_mma = sum(i["flops_mma"] for i in infos)
    # K/V the tensor-core tasks read, each byte once (a page several tiles
    # re-read counts once): at most the unique bytes of the batch
    kv_mma = min(sum(i["kv_bytes_read"] - i["kv_bytes_bw"] for i in infos), kv_unique)
    mma_hbm = (kv_mma + qo_bytes) / (roof_ms[pps.KERNEL_TENSOR] / 1e3) / 1e9 \
        if roof_ms[pps.KERNEL_TENSOR] > 0 else 0.0
    mma_tf = flops_mma / (roof_ms[pps.KERNEL_TENSOR] / 1e3) / 1e12 \
        if roof_ms[pps.KERNEL_TENSOR] > 0 else 0.0
    tpeak = peaks.get("bf16_tflops_sustained" if len(steps) > 1 else "bf16_tflops", 1900.0)
    hpeak = peaks.get("hbm_gbs", 6800.0)
    if dom == pps.KERNEL_TENSOR and mma_tf / tpeak >= mma_hbm / hpeak:
        roof = {"bound": "tensor", "achieved": mma_tf, "peak": tpeak, "unit": "TFLOP/s",
                "frac": mma_tf / tpeak, "traffic": traffic_record("attn_mma.cu", args.workload),
                "kernel": "tcgen05 attention tiles",
                "algorithmic": f"{flops_mma:.4g} FLOP per step (4*d per visible (row,key) pair)"}
    elif dom == pps.KERNEL_TENSOR:
        # few query rows per K/V byte (verify trees): the tile kernel is bound by HBM
        roof = {"bound": "hbm", "achieved": mma_hbm, "peak": hpeak, "unit": "GB/s",
                "frac": mma_hbm / hpeak, "traffic": traffic_record("attn_mma.cu", args.workload),
                "kernel": "tcgen05 attention tiles",
                "algorithmic": f"{kv_mma + qo_bytes} B per step (K+V each tensor-core task "
                               f"reads: {kv_mma}; Q and O rows: {qo_bytes}); "
                               f"{mma_tf:.1f} TFLOP/s = {mma_tf / tpeak:.3f} of the tensor peak"}
    else:
        alg = kv_bw + qo_bytes
        ach = alg / (roof_ms[dom] / 1e3) / 1e9
        peak = peaks.get("hbm_gbs", 6800.0)
        roof = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak,
                "traffic": traffic_record("attn_bw.cu" if dom == 0 else "merge.cu", args.workload),
                "kernel": ["split-KV bandwidth attention", "", "partial merge"][dom],
                "algorithmic": f"{alg} B per step (K+V read by the bandwidth tasks, each "
                               f"once: {kv_bw}; Q and O rows: {qo_bytes})"}
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else \
        "fallback"

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, seeded layouts; no dataset)",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}" +
                   (f" [{args.requests} requests]" if args.requests else ""),
                   "tokens_per_step": tokens, "kv_bytes_unique_per_step": kv_unique,
                   "l2": (f"step time warm (KV only {kv_unique / l2_bytes:.1f}x L2); kernel "
                          f"times for the roofline re-measured with a {4 * l2_bytes} B L2 flush "
                          f"before every step") if flush else
                   "inputs larger than L2 (KV > 4x the 129 MB L2), no flush",
                   "parallelism": f"dp{world} (independent batch per GPU, no collective)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": ms_e2e},
        "gpu_launches": launches,
        "kernel_ms_per_step": {"bandwidth": kern_ms[0], "tensor": kern_ms[1], "merge": kern_ms[2]},
        "roofline": roof,
        **({"cold_l2": {"kernel_ms_per_step": dict(zip(("bandwidth", "tensor", "merge"), cold_ms)),
                        "attention_unique_gbs": kv_unique / (max(cold_ms[0], cold_ms[1])
                                                             + cold_ms[2]) * 1e3 / 1e9,
                        "flush_bytes": 4 * l2_bytes}} if cold_ms is not None else {}),
        "clocks": clocks,
        "achieved": {"kv_unique_gbs": kv_unique / (ms_max / 1e3) / 1e9,
                     "attention_unique_gbs": kv_unique / (max(kern_ms[0], kern_ms[1]) + kern_ms[2])
                     * 1e3 / 1e9,
                     "tflops_total": sum(i["flops_total"] for i in infos) / (ms_max / 1e3) / 1e12},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _oracle_sample_time(wl, reqs, step):
    """Oracle wall time (s) and tokens for a subset of requests of one step."""
    from oracle_run import oracle_steps
    import workloads
    sub = workloads.sub_workload(wl, step, reqs)
    t0 = time.perf_counter()
    oracle_steps(sub)
    dt = time.perf_counter() - t0
    return dt, sub.steps[step].layout.num_tokens


def cpu_baseline(wl, budget_s=15.0, step=None):
    """The fp64 oracle, as it stands, timed on this host on a bounded sample
    of the same workload (whole requests, in order, until ~budget_s)."""
    L = wl.steps[-1].layout
    step = len(wl.steps) - 1 if step is None else step
    cores = len(os.sched_getaffinity(0))
    used, tok, secs = [], 0, 0.0
    for r in range(L.num_requests):
        if L.q_len[r] == 0:
            continue
        dt, n = _oracle_sample_time(wl, [r], step)
        used.append(r)
        tok += n
        secs += dt
        if secs >= budget_s:
            break
    return {"value": tok / secs if secs else None, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{len(used)} of {L.num_requests} requests ({tok} new tokens, all their "
                      f"rows, step {step}) in {secs:.1f} s; numpy fp64 with BLAS threads = "
                      f"{os.environ.get('OPENBLAS_NUM_THREADS', 'all')} of {cores} cores"}


def run_reference(args):
    """The oracle as the reference arm (rank 0 only)."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import torch
    import workloads
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = workloads.make(args.workload, device=dev)
    L = wl.steps[-1].layout
    step = len(wl.steps) - 1
    reqs = [r for r in range(L.num_requests) if L.q_len[r] > 0]
    # calibrate: time per request, then size each step's sample to fit the budget
    dt0, n0 = _oracle_sample_time(wl, reqs[:1], step)
    per_step = max(0.05, args.cpu_seconds * 8 / max(1, args.steps + args.warmup))
    m = max(1, min(len(reqs), int(per_step / max(dt0, 1e-6))))
    for w in range(args.warmup):
        _oracle_sample_time(wl, reqs[(w * m) % len(reqs):][:m] or reqs[:m], step)
    tot_t, tot_tok = 0.0, 0
    for k in range(args.steps):
        sel = reqs[(k * m) % len(reqs):][:m] or reqs[:m]
        dt, n = _oracle_sample_time(wl, sel, step)
        tot_t += dt
        tot_tok += n
    value = tot_tok / tot_t
    cores = len(os.sched_getaffinity(0))
    sample = (f"{m} of {L.num_requests} requests per step (consecutive, wrapping), fp64 numpy "
              f"oracle on {cores} host cores")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, seeded layouts; no dataset)",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                   "parallelism": "host cores, rank 0 only"},
        "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample, "value": value,
                         "unit": "tokens/s"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="decode_heavy", choices=sorted(DESCRIPTIONS))
    ap.add_argument("--impl", default="pps", choices=["pps", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--flush-l2", default="auto", choices=["auto", "on", "off"],
                    help="re-time the kernels with an L2 flush before each step "
                         "(auto: when the unique KV is under 4x the L2 size)")
    ap.add_argument("--requests", type=int, default=0,
                    help="decode_heavy / long_prefill: number of requests (default 256 / 4); "
                         "for small profiling captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_pps(args)


if __name__ == "__main__":
    main()
