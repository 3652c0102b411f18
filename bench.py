"""Benchmark: mixed-batch paged attention on GB300 through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pps|reference]

One step = the whole hot path over one batch: kv_append of the step's new
rows, attn_plan on the host, attn_run (bandwidth tasks, tensor-core tasks,
partial merge), issued as one pps_attn_step call per batch (a long-prefill
step is its four causal chunks).

Without --workload the run measures every configuration of the attention path
one after the other: tiny_mixed, decode_heavy, radix_sharing, mixed_budget and
long_prefill.  The JSON line's own fields (value, e2e, roofline, clocks) are
the headline configuration's, mixed_budget (8192 new tokens over ~44 GB of KV,
the largest that fits one GPU); ``configs`` holds every configuration's full
record, each with its own roofline, e2e and CPU baseline.  --workload NAME
measures one workload alone (also the serving loops, the draft-tree batch and
the projection GEMMs).

``value`` is tokens/s with inputs resident in HBM; ``e2e`` is the same metric
with every step's inputs copied from pinned host memory and the output copied
back inside the timed region: one ``pps_attn_step_host`` call per batch (host
rows and tables in, host rows out; the serving loops make the same call after
each step's cache or engine calls; the projection GEMMs copy their activations
in and outputs out around the GEMM calls).  Under torchrun each rank runs its
own batch (weak scaling, no data-path collective).  ``--impl reference`` times
the fp64 CPU oracle on a bounded sample instead.
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
    "cache_serving": "prefix cache + attention serving loop: 256 active requests over 32 shared "
                     "system prompts (U[1024,4096] tokens) + private suffixes U[32,256], outputs "
                     "U[16,128]; per step 8 admitted (cache begin, copy-on-write), the rest decode; "
                     "32/8 heads, d 128, P 16, 131072-page pool, LRU, seed 6",
    "engine_serving": "token-wise scheduler + prefix cache + attention: 8192-token budget (512 "
                      "reserved for generation), up to 256 requests in the system, 32 shared "
                      "system prompts U[1024,4096], 25% with a private document U[2048,8192], "
                      "suffix U[32,256], outputs U[16,128]; 25% verify 4-token drafts, the rest "
                      "decode; chunked prefill; 32/8 heads, d 128, P 16, 262144-page pool, LRU, "
                      "seed 7",
    "projections": "QKV (N 6144) and O (N 4096) projection GEMMs of a mixed batch of 8229 tokens, "
                   "hidden 4096, bf16, virtual padding of the ragged last tile, seed 8",
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


def roofline(pps, roof_ms, infos, qo_bytes, workload, sustained):
    """Roofline object of the dominant kernel class.  ``roof_ms`` (per kernel
    class), ``infos`` (plan info dicts) and ``qo_bytes`` cover the same work."""
    import numpy as np
    peaks, peak_src = load_peaks()
    dom = int(np.argmax(roof_ms))
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
    tpeak = peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops", 1900.0)
    hpeak = peaks.get("hbm_gbs", 6800.0)
    if dom == pps.KERNEL_TENSOR and mma_tf / tpeak >= mma_hbm / hpeak:
        roof = {"bound": "tensor", "achieved": mma_tf, "peak": tpeak, "unit": "TFLOP/s",
                "frac": mma_tf / tpeak, "traffic": traffic_record("attn_mma.cu", workload),
                "kernel": "tcgen05 attention tiles",
                "algorithmic": f"{flops_mma:.4g} FLOP per step (4*d per visible (row,key) pair)"}
    elif dom == pps.KERNEL_TENSOR:
        # few query rows per K/V byte (verify trees): the tile kernel is bound by HBM
        roof = {"bound": "hbm", "achieved": mma_hbm, "peak": hpeak, "unit": "GB/s",
                "frac": mma_hbm / hpeak, "traffic": traffic_record("attn_mma.cu", workload),
                "kernel": "tcgen05 attention tiles",
                "algorithmic": f"{kv_mma + qo_bytes:.0f} B per step (K+V each tensor-core task "
                               f"reads: {kv_mma:.0f}; Q and O rows: {qo_bytes:.0f}); "
                               f"{mma_tf:.1f} TFLOP/s = {mma_tf / tpeak:.3f} of the tensor peak"}
    else:
        alg = kv_bw + qo_bytes
        ach = alg / (roof_ms[dom] / 1e3) / 1e9
        # small-row tasks run on the key-tile tcgen05 kernel (attn_tt.cu) when
        # the plan says so, else on the CUDA-core split-KV kernel (attn_bw.cu)
        tt = any(i.get("small_rows_on_tensor") for i in infos)
        src = ("attn_tt.cu" if tt else "attn_bw.cu") if dom == 0 else "merge.cu"
        name = ("key-tile tcgen05 attention (small-row tasks)" if tt else
                "split-KV bandwidth attention (CUDA cores)") if dom == 0 else "partial merge"
        roof = {"bound": "hbm", "achieved": ach, "peak": hpeak, "unit": "GB/s",
                "frac": ach / hpeak,
                "traffic": traffic_record(src, workload),
                "kernel": name,
                "algorithmic": f"{alg:.0f} B per step (K+V read by the bandwidth tasks, each "
                               f"once: {kv_bw:.0f}; Q and O rows: {qo_bytes:.0f})"}
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else \
        "fallback"
    return roof


# ---------------------------------------------------------------------------


# The five configurations of the attention path, in the order the default run
# measures them; the headline line is the largest one that fits one GPU.
SUITE = ["tiny_mixed", "decode_heavy", "radix_sharing", "mixed_budget", "long_prefill"]
HEADLINE = "mixed_budget"


def init_device():
    import torch
    import paged_prefix_shared_gb300 as pps
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    pps.build()
    pps.lib()
    return torch.device("cuda", local_rank)


def make_attention_workload(name, args, dev, rank):
    import workloads
    if name == "decode_heavy":
        return workloads.decode_heavy(seed=1 + 1000 * rank, device=dev,
                                      num_requests=args.requests or 256)
    if name == "long_prefill" and args.requests:
        return workloads.long_prefill(device=dev, num_requests=args.requests)
    if name == "tree_verify" and args.requests:
        return workloads.tree_verify(device=dev, num_requests=args.requests)
    kw = {} if rank == 0 else {"seed": {"tiny_mixed": 0, "radix_sharing": 2, "mixed_budget": 3,
                                        "long_prefill": 4, "tree_verify": 5}[name] + 1000 * rank}
    return workloads.make(name, device=dev, **kw)


def measure_attention(name, args, dev, cpu_seconds):
    """One configuration of the attention path: the record of its bench line.

    Device-resident loop: one pps_attn_step call per step and chunk (tables
    uploaded, new rows appended, batch planned on the host, attention), with
    CUDA events around every kernel class.  e2e: one pps_attn_step_host call
    per step and chunk (rows from page-locked host memory, output back)."""
    import torch

    import paged_prefix_shared_gb300 as pps

    rank, local_rank, world = dist_env()
    wl = make_attention_workload(name, args, dev, rank)
    # The library appends into a copy; the drawn pool stays as the generator
    # made it (the CPU baseline starts from it).  Re-appending the same rows
    # every step is idempotent.
    pk, pv = wl.pool_k.clone(), wl.pool_v.clone()
    flags = (pps.PLAN_FUSED_APPEND if args.fused_append else 0) | \
        (pps.PLAN_SMALL_ROWS_CUDA_CORES if args.small_rows_cuda_cores else 0)
    steps = []
    for st in wl.steps:
        L = st.layout
        out = torch.empty_like(st.q)
        call = pps.StepCall(pk, pv, st.q, st.k_new, st.v_new, L.q_indptr, L.kv_len,
                            L.page_indptr, L.page_indices, out, tree_parent=L.tree_parent,
                            flags=flags)
        plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                             L.num_kv_heads, L.head_dim, L.page_size, L.num_pages,
                             tree_parent=L.tree_parent, flags=flags & ~pps.PLAN_FUSED_APPEND)
        steps.append(dict(L=L, st=st, out=out, call=call, info=plan.info()))
        plan.destroy()
    stream = torch.cuda.current_stream()
    nk = pps.NUM_KERNEL_CLASSES

    def one_step(evs=None):
        for i, s in enumerate(steps):
            s["call"](None if evs is None else evs[i])

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()

    # per-kernel events (one set per step per chunk) -> average launch duration;
    # created, recorded once and converted to C arrays outside the timed region
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)] for _ in steps]
          for _ in range(args.steps)]
    evh = [[pps.event_array(per_chunk) for per_chunk in per_step] for per_step in ev]
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    n_launch0 = pps.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark("t0")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    e0.record(stream)
    for k in range(args.steps):
        one_step()
    e1.record(stream)
    host_ms = (time.perf_counter() - h0) / args.steps * 1e3    # enqueue time per step
    torch.cuda.synchronize()
    sampler.mark("t1")
    barrier(world)
    launches = pps.launch_count() - n_launch0
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    # host cost of one step's calls with the GPU idle (plan, uploads, launches):
    # inside the loop above the host may also wait for a staging buffer
    hc = []
    for k in range(min(args.steps, 20)):
        torch.cuda.synchronize()
        c0 = time.perf_counter()
        one_step()
        hc.append(time.perf_counter() - c0)
    host_call_ms = statistics.median(hc) * 1e3
    torch.cuda.synchronize()
    # the same steps again with events around every kernel class (per-kernel
    # times; the events are kept out of the step-time loop above)
    for k in range(args.steps):
        one_step(evh[k])
    torch.cuda.synchronize()

    def kernel_ms():
        acc = [0.0] * nk
        for k in range(args.steps):
            for i in range(len(steps)):
                for c in range(nk):
                    acc[c] += ev[k][i][2 * c].elapsed_time(ev[k][i][2 * c + 1])
        return [x / args.steps for x in acc]        # per step (summed over chunks)

    kern_ms = kernel_ms()

    # ---- kernel times with a cold L2 (KV that L2 could partly hold) -----------------------
    # Each step is preceded by a write of a buffer four times the L2 size; only the
    # per-kernel events count, so the flush itself is never timed.  The write leaves
    # L2 full of dirty lines, whose write-back then lands inside the next kernel (up to
    # 129 MB of writes the kernel never made), so the roofline times are taken with the
    # buffer also read back after its write: L2 then holds clean lines of the flush
    # buffer and none of the step's data.  The dirty-L2 times are reported beside them.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129e6)
    kv_unique0 = sum(s["info"]["kv_bytes_unique"] for s in steps)
    flush = args.flush_l2 == "on" or (args.flush_l2 == "auto" and kv_unique0 < 4 * l2_bytes)
    cold_ms = dirty_ms = None
    if flush:
        fbuf = torch.empty(4 * l2_bytes // 4, dtype=torch.int32, device=dev)
        for k in range(args.steps):
            fbuf.fill_(k)
            one_step(evh[k])
        torch.cuda.synchronize()
        dirty_ms = kernel_ms()
        for k in range(args.steps):
            fbuf.fill_(k)
            fbuf.sum(dtype=torch.int64)
            one_step(evh[k])
        torch.cuda.synchronize()
        cold_ms = kernel_ms()
        del fbuf
    roof_ms = cold_ms if cold_ms is not None else kern_ms

    tokens = sum(s["L"].num_tokens for s in steps)
    total_tokens = sum_over_ranks(tokens, world, dev)
    value = total_tokens / (ms_max / 1e3)

    # ---- e2e: host buffers in, host result out, through the public API -------------------
    # One pps_attn_step_host call per step and chunk: the rows and tables go from
    # page-locked host memory to the device, through append, plan and
    # attention, and the output rows come back, all enqueued by the library.
    h = []
    for s in steps:
        st, L = s["st"], s["L"]
        host = {n: st.__dict__[n].cpu().pin_memory() for n in ("q", "k_new", "v_new")}
        out_h = torch.empty_like(s["out"], device="cpu").pin_memory()
        call = pps.StepCall(pk, pv, host["q"], host["k_new"], host["v_new"], L.q_indptr,
                            L.kv_len, L.page_indptr, L.page_indices, out_h,
                            tree_parent=L.tree_parent, host=True, flags=flags)
        h.append(dict(host=host, out_h=out_h, call=call))
    tab_bytes = sum(4 * (3 * s["L"].num_requests + 2 + len(s["L"].page_indices)) for s in steps)
    bi = sum(v.numel() * v.element_size() for x in h for v in x["host"].values()) + tab_bytes
    bo = sum(x["out_h"].numel() * x["out_h"].element_size() for x in h)

    def e2e_step():
        for x in h:
            x["call"]()

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
    infos = [s["info"] for s in steps]
    L0 = steps[0]["L"]
    qo_bytes = sum(2 * s["L"].num_tokens * L0.num_q_heads * L0.head_dim * 2 for s in steps)
    kv_unique = sum(i["kv_bytes_unique"] for i in infos)
    # the committed DRAM records are for the full-size launches: a resized batch
    # gets none (its key names the request count)
    key = name if not args.requests else f"{name}[{args.requests} requests]"
    roof = roofline(pps, roof_ms, infos, qo_bytes, key, sustained=len(steps) > 1)
    if kv_unique < 1 << 20:
        roof["note"] = ("launch-latency bound (under 1 MB of K/V per step): the fraction is "
                        "reported, not targeted")

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, seeded layouts; no dataset)",
        "config": {"workload": f"{name}: {DESCRIPTIONS[name]}" +
                   (f" [{args.requests} requests]" if args.requests else ""),
                   "tokens_per_step": tokens, "kv_bytes_unique_per_step": kv_unique,
                   "l2": (f"step time warm (KV only {kv_unique / l2_bytes:.1f}x L2); kernel "
                          f"times for the roofline re-measured with a {4 * l2_bytes} B L2 flush "
                          f"before every step (the buffer written, then read back so that L2 "
                          f"holds no dirty lines)") if flush else
                   "inputs larger than L2 (KV > 4x the 129 MB L2), no flush",
                   "parallelism": f"dp{world} (independent batch per GPU, no collective)",
                   "step_call": "pps_attn_step: one native call per step and chunk (tables "
                                "uploaded, rows appended, batch planned on the host, attention)" +
                                ("; append fused into the first attention kernel"
                                 if args.fused_append else "") +
                                ("; small-row tasks on the CUDA-core kernel"
                                 if args.small_rows_cuda_cores else "")},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": ms_e2e},
        "gpu_launches": launches,
        "host_ms_per_step": host_ms,
        "host_ms_per_call_idle_gpu": host_call_ms,
        "kernel_ms_per_step": {"bandwidth": kern_ms[0], "tensor": kern_ms[1], "merge": kern_ms[2]},
        "roofline": roof,
        **({"cold_l2": {"kernel_ms_per_step": dict(zip(("bandwidth", "tensor", "merge"), cold_ms)),
                        "attention_unique_gbs": kv_unique / (max(cold_ms[0], cold_ms[1])
                                                             + cold_ms[2]) * 1e3 / 1e9,
                        "flush_bytes": 4 * l2_bytes, "flush": "write, then read back",
                        "kernel_ms_per_step_dirty_l2": dict(zip(("bandwidth", "tensor", "merge"),
                                                                dirty_ms))}}
           if cold_ms is not None else {}),
        "clocks": clocks,
        "achieved": {"kv_unique_gbs": kv_unique / (ms_max / 1e3) / 1e9,
                     "attention_unique_gbs": kv_unique / (max(kern_ms[0], kern_ms[1]) + kern_ms[2])
                     * 1e3 / 1e9,
                     "tflops_total": sum(i["flops_total"] for i in infos) / (ms_max / 1e3) / 1e12},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, budget_s=cpu_seconds)
    del steps, h, pk, pv, wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return result


def run_pps(args):
    """One attention workload (--workload)."""
    rank, _, world = dist_env()
    dev = init_device()
    result = measure_attention(args.workload, args, dev, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_suite(args):
    """The default run: every configuration of the attention path, one after
    the other on the same GPU; the line's own fields are the headline
    configuration's (the largest that fits one GPU), ``configs`` holds every
    configuration's full record."""
    rank, _, world = dist_env()
    dev = init_device()
    recs = {}
    for name in SUITE:
        recs[name] = measure_attention(name, args, dev, args.cpu_seconds)
    result = dict(recs[HEADLINE])
    result["configs"] = {n: {k: v for k, v in r.items()
                             if k not in ("metric", "unit", "n_gpus", "steps", "warmup",
                                          "higher_is_better", "scaling", "vs_baseline", "dtype",
                                          "data")}
                         for n, r in recs.items()}
    result["config"] = dict(result["config"])
    result["config"]["suite"] = ("every configuration of the attention path measured in this "
                                 "run (configs); the line's value, e2e and roofline are "
                                 f"{HEADLINE}'s")
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


class CacheServer:
    """A serving loop over the prefix cache: every step retires finished
    requests (their pages go into the radix tree), decodes one token for each
    active request, admits new ones (pps_cache_begin: shared system-prompt
    pages reused, copy-on-write of a partly matched page), then runs the step's
    copy-on-write copies, kv_append, attn_plan and attn_run over the page lists
    the cache produced.  New K/V/Q rows are slices of seeded device buffers."""

    def __init__(self, pps, torch, dev, trace, num_pages=131072, page_size=16, num_q_heads=32,
                 num_kv_heads=8, head_dim=128, active=256, max_rows=65536, seed=6,
                 make_cache=True):
        self.pps, self.torch, self.dev = pps, torch, dev
        self.prompts, self.reqs = trace
        self.P, self.Hq, self.Hkv, self.D = page_size, num_q_heads, num_kv_heads, head_dim
        self.num_pages, self.target, self.max_rows = num_pages, active, max_rows
        self.cache = pps.Cache(num_pages, page_size) if make_cache else None
        bf = torch.bfloat16
        self.pk = torch.zeros((num_pages, num_kv_heads, page_size, head_dim), dtype=bf, device=dev)
        self.pv = torch.zeros_like(self.pk)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.rows_k = torch.randn((max_rows, num_kv_heads, head_dim), generator=g, device=dev).to(bf)
        self.rows_v = torch.randn((max_rows, num_kv_heads, head_dim), generator=g, device=dev).to(bf)
        self.q = torch.randn((max_rows, num_q_heads, head_dim), generator=g, device=dev).to(bf)
        self.out = torch.empty_like(self.q)
        self.ws = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        # two page-locked staging buffers for the step's tables, each reused
        # only after the upload that last read it has completed
        self.h_tab = [torch.empty(1 << 22, dtype=torch.int32).pin_memory() for _ in range(2)]
        self.h_ev = [None, None]
        self.d_tab = torch.empty(1 << 22, dtype=torch.int32, device=dev)
        self.nstep = 0
        self.next_req = 0
        # active requests: cache id, trace index, outputs produced so far
        import numpy as np
        self.a_rid = np.zeros(0, np.int32)
        self.a_idx = np.zeros(0, np.int32)
        self.a_k = np.zeros(0, np.int32)
        self.new_idx = []
        self.out_len = np.array([len(r[2]) for r in self.reqs], np.int32)
        self.out_tok = np.zeros((len(self.reqs), int(self.out_len.max()) + 1), np.int32)
        for i, r in enumerate(self.reqs):
            self.out_tok[i, :len(r[2])] = r[2]
        self.host_s = 0.0                     # host time inside cache calls
        self.cache_calls = 0
        self.io = None                        # (pinned q/k/v rows, pinned out) for the e2e run

    def warm_prefix(self, tokens):
        rid, _, _ = self.cache.begin(tokens)
        self.cache.finish(rid)

    def stats(self):
        return self.cache.stats()

    def step(self, admit, events=None):
        import numpy as np
        torch, pps = self.torch, self.pps
        t0 = time.perf_counter()
        # retire requests that produced all their tokens (pages go into the tree)
        if len(self.a_rid):
            done = self.a_k >= self.out_len[self.a_idx]
            for rid in self.a_rid[done]:
                self.cache.finish(int(rid))
            self.cache_calls += int(done.sum())
            keep = ~done
            self.a_rid, self.a_idx, self.a_k = self.a_rid[keep], self.a_idx[keep], self.a_k[keep]
        # one decode token for every active request, in one native call
        n_dec = len(self.a_rid)
        first = np.zeros(0, np.int32)
        if n_dec:
            toks = self.out_tok[self.a_idx, self.a_k]
            first = self.cache.extend_batch(self.a_rid, np.arange(n_dec + 1, dtype=np.int32), toks)
            self.a_k += 1
            self.cache_calls += n_dec
        # admissions
        new_rid, new_cached, copies = [], [], []
        while admit > 0 and len(self.a_rid) + len(new_rid) < self.target and \
                self.next_req < len(self.reqs):
            i = self.next_req
            self.next_req += 1
            rid, cached, copy = self.cache.begin(self.reqs[i][1])
            if copy is not None:
                copies.append(copy)
            new_rid.append(rid)
            new_cached.append(cached)
            self.new_idx.append(i)
            admit -= 1
            self.cache_calls += 1
        rids = np.concatenate([self.a_rid, np.array(new_rid, np.int32)]).astype(np.int32)
        kv_len, page_indptr, page_indices = self.cache.tables(rids)
        cached = np.concatenate([first, np.array(new_cached, np.int32)]).astype(np.int32)
        self.a_rid = rids
        self.a_idx = np.concatenate([self.a_idx, np.array(self.new_idx, np.int32)]).astype(np.int32)
        self.a_k = np.concatenate([self.a_k, np.zeros(len(new_rid), np.int32)]).astype(np.int32)
        self.new_idx = []
        self.host_s += time.perf_counter() - t0
        return self._run_batch(kv_len, cached, page_indptr, page_indices, copies, events)

    def _run_batch(self, kv_len, cached, page_indptr, page_indices, copies, events=None):
        """Device side of a step: copy-on-write copies, then one pps_attn_step
        call (append of positions [cached, kv_len) of every request, plan,
        attention), or in the end-to-end run one pps_attn_step_host call."""
        import numpy as np
        torch, pps = self.torch, self.pps
        R = len(kv_len)
        q_len = kv_len.astype(np.int64) - cached
        q_indptr = np.concatenate([[0], np.cumsum(q_len)]).astype(np.int32)
        T = int(q_indptr[-1])
        if T > self.max_rows:
            raise RuntimeError("step larger than the row buffers")
        # copy-on-write copies, split into calls whose copies do not touch each
        # other's pages (a later call may hand a source page out again)
        waves, cur, used = [], [], set()
        for c in copies:
            if c[0] in used or c[1] in used:
                waves.append(cur)
                cur, used = [], set()
            cur.append(c)
            used |= {c[0], c[1]}
        if cur:
            waves.append(cur)
        # the copy-on-write tables in one upload (the step call uploads its own)
        if waves:
            parts = [np.array(w, np.int32).T.reshape(-1) for w in waves]
            flat = np.concatenate(parts).astype(np.int32)
            hb = self.nstep & 1
            self.nstep += 1
            if self.h_ev[hb] is not None:
                self.h_ev[hb].synchronize()
            self.h_tab[hb][:len(flat)].copy_(torch.from_numpy(flat))
            self.d_tab[:len(flat)].copy_(self.h_tab[hb][:len(flat)], non_blocking=True)
            self.h_ev[hb] = torch.cuda.Event()
            self.h_ev[hb].record()
            off = 0
            for w, a in zip(waves, parts):
                n = len(w)
                v = self.d_tab[off:off + 3 * n]
                pps.copy_slots(self.pk, self.pv, v[:n], v[n:2 * n], v[2 * n:3 * n])
                off += len(a)
        if self.io is not None:
            # end to end: the step's rows from page-locked host memory and its
            # output rows back, through the one-call host-row step
            hq, hk, hv, ho = self.io
            t1 = time.perf_counter()
            pps.attn_step_host(self.pk, self.pv, hq[:T], hk[:T], hv[:T], q_indptr, kv_len,
                               page_indptr, page_indices, ho[:T])
            self.host_s += time.perf_counter() - t1
            return T, R, None, len(copies)
        # the step's append, plan and attention: one pps_attn_step call; the
        # tables are kept so the plan's figures for the roofline can be taken
        # after the timed loop
        t1 = time.perf_counter()
        pps.attn_step(self.pk, self.pv, self.q[:T], self.rows_k[:T], self.rows_v[:T], q_indptr,
                      kv_len, page_indptr, page_indices, self.out[:T], scratch=self.ws,
                      events=events)
        self.host_s += time.perf_counter() - t1
        return T, R, (q_indptr, kv_len.copy(), page_indptr.copy(), page_indices.copy()), \
            len(copies)

    def plan_info(self, tables):
        q_indptr, kv_len, page_indptr, page_indices = tables
        return self.pps.attn_plan(q_indptr, kv_len, page_indptr, page_indices, self.Hq, self.Hkv,
                                  self.D, self.P, self.num_pages).info()


class EngineServer(CacheServer):
    """Scheduler + prefix cache + attention through the native serving-step
    runtime (pps_engine_*): every step pps_engine_schedule picks the batch
    within a token budget (the generation requests, decode: 1 token,
    speculative verify: a draft of ``draft`` tokens, all accepted; then chunks
    of pending prompts, the part the prefix cache did not already hold), and
    pps_engine_commit appends the generated tokens and writes the batch's
    tables.  Requests are admitted (pps_engine_add) while fewer than
    ``active`` are in the system."""

    def __init__(self, pps, torch, dev, trace, budget=8192, reserved=512, draft=4,
                 verify_frac=0.25, admit_max=32, **kw):
        import numpy as np
        super().__init__(pps, torch, dev, trace, make_cache=False, **kw)
        self.eng = pps.Engine(self.num_pages, self.P, budget, reserved)
        self.draft, self.admit_max = draft, admit_max
        rng = np.random.default_rng(17)
        self.gen_k = np.where(rng.random(len(self.reqs)) < verify_frac, draft, 1).astype(np.int32)
        pad = np.zeros((len(self.reqs), draft), np.int32)
        self.out_tok = np.concatenate([self.out_tok, pad], axis=1)
        # per request id (ids are handed out in admission order): trace index,
        # generated tokens so far; ids of the requests in the system
        n = len(self.reqs) + len(self.prompts) + 1
        self.r_idx = np.zeros(n, np.int32)
        self.r_prod = np.zeros(n, np.int32)
        self.live = np.zeros(0, np.int32)

    def warm_prefix(self, tokens):
        rid, _, _ = self.eng.add(tokens)
        self.eng.finish(rid)

    def stats(self):
        return self.eng.stats()

    def step(self, admit=None, events=None):
        import numpy as np
        t0 = time.perf_counter()
        eng = self.eng
        # retire requests that produced all their outputs
        if len(self.live):
            done = self.r_prod[self.live] >= self.out_len[self.r_idx[self.live]]
            for rid in self.live[done].tolist():
                eng.finish(rid)
            self.cache_calls += int(done.sum())
            self.live = self.live[~done]
        copies, new = [], []
        while len(self.live) + len(new) < self.target and len(new) < self.admit_max and \
                self.next_req < len(self.reqs):
            i = self.next_req
            self.next_req += 1
            rid, cached, copy = eng.add(self.reqs[i][1], int(self.gen_k[i]))
            if copy is not None:
                copies.append(copy)
            self.r_idx[rid], self.r_prod[rid] = i, 0
            new.append(rid)
        if new:
            self.live = np.concatenate([self.live, np.array(new, np.int32)])
            self.cache_calls += len(new)
        req, tok, pre = eng.schedule()
        gen = pre == 0
        g_rid, k = req[gen], tok[gen]
        cols = self.r_prod[g_rid][:, None] + np.arange(self.draft)[None, :]
        mat = self.out_tok[self.r_idx[g_rid][:, None], np.minimum(cols, self.out_tok.shape[1] - 1)]
        toks = mat[np.arange(self.draft)[None, :] < k[:, None]].astype(np.int32)
        rq, qi, cl, kl, pi, px = eng.commit(toks)
        if len(rq) == len(req):
            self.r_prod[g_rid] += k
        else:                                  # some generation entries found no page
            kept = np.isin(g_rid, rq)
            self.r_prod[g_rid[kept]] += k[kept]
        self.cache_calls += len(g_rid)
        self.host_s += time.perf_counter() - t0
        return self._run_batch(kl, cl, pi, px, copies, events)


def run_cache_serving(args):
    """The cache_serving workload: prefix cache + attention, step by step."""
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
    engine = args.workload == "engine_serving"
    if engine:
        trace = workloads.cache_trace(seed=7 + 1000 * rank, doc_frac=0.25)
        srv = EngineServer(pps, torch, dev, trace, num_pages=262144)
    else:
        trace = workloads.cache_trace(seed=6 + 1000 * rank)
        srv = CacheServer(pps, torch, dev, trace)
    stream = torch.cuda.current_stream()
    # warm up: every system prompt once, then fill the system
    for k in range(len(trace[0])):
        srv.warm_prefix(trace[0][k])
    if engine:
        for _ in range(60):
            srv.step()
    else:
        while len(srv.a_rid) < srv.target:
            srv.step(admit=64)
    for _ in range(args.warmup):
        srv.step(admit=8)
    torch.cuda.synchronize()
    nk = pps.NUM_KERNEL_CLASSES
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)] for _ in range(args.steps)]
    for per in ev:
        for e in per:
            e.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    n0 = pps.launch_count()
    srv.host_s, srv.cache_calls = 0.0, 0
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark("t0")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    tokens, infos, reqs, ncopy = 0, [], 0, 0
    for k in range(args.steps):
        T, R, info, nc = srv.step(admit=8, events=ev[k])
        tokens += T
        reqs += R
        ncopy += nc
        infos.append(info)
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    barrier(world)
    launches = pps.launch_count() - n0
    clocks = sampler.stop()
    host_ms = srv.host_s / args.steps * 1e3
    calls = srv.cache_calls
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    total_tokens = sum_over_ranks(tokens, world, dev)
    value = total_tokens / (ms * args.steps / 1e3)
    kern_ms = [sum(ev[k][2 * c].elapsed_time(ev[k][2 * c + 1]) for k in range(args.steps))
               / args.steps for c in range(nk)]

    # e2e: the step's Q/K/V rows come from pinned host memory, outputs go back,
    # one pps_attn_step_host call per step (after the step's copy-on-write copies)
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype).pin_memory().copy_(t.cpu())
    srv.io = (pin(srv.q), pin(srv.rows_k), pin(srv.rows_v),
              torch.empty(srv.out.shape, dtype=srv.out.dtype).pin_memory())
    k_e2e = max(3, args.steps // 2)
    for _ in range(3):
        srv.step(admit=8)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    tok_e2e, h2d, d2h = 0, 0, 0
    row_b = srv.Hkv * srv.D * 2
    for _ in range(k_e2e):
        T, R, info, nc = srv.step(admit=8)
        tok_e2e += T
        h2d += T * (srv.Hq * srv.D * 2 + 2 * row_b)
        d2h += T * srv.Hq * srv.D * 2
    f1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(f0.elapsed_time(f1) / k_e2e, world, dev)
    e2e_value = sum_over_ranks(tok_e2e, world, dev) / (ms_e2e * k_e2e / 1e3)

    infos = [srv.plan_info(t) for t in infos]        # the timed steps' plans, planned again
    avg = lambda key: sum(i[key] for i in infos) / len(infos)
    avg_infos = [{k: avg(k) for k in ("kv_bytes_unique", "kv_bytes_bw", "flops_mma", "small_rows_on_tensor",
                                      "kv_bytes_read", "flops_total")}]
    qo = tokens / args.steps * 2 * srv.Hq * srv.D * 2
    roof = roofline(pps, kern_ms, avg_infos, qo, args.workload, sustained=False)
    st = srv.stats()
    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded token ids and N(0,1) bf16 Q/K/V rows; no dataset)",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                   "tokens_per_step": tokens / args.steps, "requests_per_step": reqs / args.steps,
                   "kv_bytes_unique_per_step": avg("kv_bytes_unique"),
                   "l2": "inputs larger than L2 (system-prompt KV ~0.3 GB plus private KV), "
                         "no flush",
                   "parallelism": f"dp{world} (independent server per GPU, no collective)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d / k_e2e,
                "d2h_bytes_per_step": d2h / k_e2e, "ms_per_step": ms_e2e},
        "gpu_launches": launches,
        "kernel_ms_per_step": {"bandwidth": kern_ms[0], "tensor": kern_ms[1], "merge": kern_ms[2]},
        "roofline": roof,
        "clocks": clocks,
        "host_cache": {"host_ms_per_step": host_ms, "cache_calls_per_step": calls / args.steps,
                       "us_per_cache_call_incl_plan": srv.host_s / max(calls, 1) * 1e6,
                       "copies_per_step": ncopy / args.steps,
                       "reused_token_fraction": st["reused_tokens"] / max(st["begun_tokens"], 1),
                       "tree_pages": st["tree_nodes"], "evictions": st["evictions"]},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cache_serving_cpu_baseline(trace, budget_s=args.cpu_seconds)
    if engine:
        result["host_cache"]["scheduler"] = "pps_engine_* (budget 8192, reserved 512)"
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def cache_serving_cpu_baseline(trace, budget_s=15.0, steps=None):
    """The oracles on the host: the reference radix cache replays the serving
    trace's cache calls and the fp64 attention oracle attends every decode
    token of a sample of requests (their K/V rows drawn on the host), until
    about ``budget_s`` seconds are spent.  tokens/s = attended tokens / time."""
    import math as _m
    import numpy as np
    import torch
    import oracle
    from oracle import radix_cache as rc
    P, Hq, Hkv, D = 16, 32, 8, 128
    prompts, reqs = trace
    cores = len(os.sched_getaffinity(0))
    o = rc.RadixCacheOracle(8192, P)          # the reference scans every page per call
    for k in range(len(prompts)):              # the system prompts, not timed
        rid, _, _ = o.begin(prompts[k].tolist())
        o.finish(rid)
    t0 = time.perf_counter()
    tok, i = 0, 0
    g = torch.Generator().manual_seed(6)
    while time.perf_counter() - t0 < budget_s and i < len(reqs):
        toks = reqs[i][1].tolist()
        rid, cached, copy = o.begin(toks)
        n = len(toks)
        k = torch.randn((n + 1, Hkv, D), generator=g).to(torch.bfloat16)
        v = torch.randn((n + 1, Hkv, D), generator=g).to(torch.bfloat16)
        q = torch.randn((1, Hq, D), generator=g).to(torch.bfloat16)
        o.extend(rid, reqs[i][2][:1].tolist())
        npg = -(-(n + 1) // P)
        pk = torch.zeros((npg * P, Hkv, D), dtype=torch.bfloat16)
        pv = torch.zeros_like(pk)
        pk[:n + 1] = k
        pv[:n + 1] = v
        pk = pk.view(npg, P, Hkv, D).permute(0, 2, 1, 3).contiguous()
        pv = pv.view(npg, P, Hkv, D).permute(0, 2, 1, 3).contiguous()
        oracle.paged_attention(q, pk, pv, np.array([0, 1]), np.array([n + 1]), np.array([0, npg]),
                               np.arange(npg), P, 1 / _m.sqrt(D), Hkv)
        o.finish(rid)
        tok += 1
        i += 1
    secs = time.perf_counter() - t0
    return {"value": tok / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{i} requests of the trace after the system prompts were cached "
                      f"(untimed): reference radix cache (8192-page pool) begin/extend/finish "
                      f"and the fp64 attention oracle for one decode token each (K/V drawn on "
                      f"the host), {secs:.1f} s; numpy fp64 with BLAS threads = "
                      f"{os.environ.get('OPENBLAS_NUM_THREADS', 'all')} of {cores} cores"}


def run_projections(args):
    """The projections workload: the QKV (6144 outputs) and O (4096 outputs)
    GEMMs of a mixed batch of 8192 + 37 tokens, hidden 4096, through
    pps_gemm_bf16.  One step = both GEMMs."""
    import numpy as np
    import torch

    import paged_prefix_shared_gb300 as pps

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pps.build()
    M, K, shapes = 8229, 4096, (6144, 4096)
    g = torch.Generator(device=dev)
    g.manual_seed(8 + 1000 * rank)
    a = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    ws = [(torch.randn((N, K), generator=g, device=dev) / K ** 0.5).to(torch.bfloat16)
          for N in shapes]
    cs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for N in shapes]
    stream = torch.cuda.current_stream()
    flops = sum(2.0 * M * N * K for N in shapes)

    def step():
        for w, c in zip(ws, cs):
            pps.gemm_bf16(a, w, c)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    n0 = pps.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark("t0")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    barrier(world)
    launches = pps.launch_count() - n0
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    value = sum_over_ranks(M, world, dev) / (ms / 1e3)
    tf = flops / (ms / 1e3) / 1e12
    # e2e: activations in from pinned host memory, outputs back
    ha = a.cpu().pin_memory()
    hc = [torch.empty(c.shape, dtype=c.dtype).pin_memory() for c in cs]
    k_e2e = max(3, args.steps // 2)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(k_e2e):
        a.copy_(ha, non_blocking=True)
        step()
        for c, h in zip(cs, hc):
            h.copy_(c, non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(f0.elapsed_time(f1) / k_e2e, world, dev)
    # library GEMM on the same shapes, for context only
    cub = []
    for w in ws:
        torch.matmul(a, w.t())
        torch.cuda.synchronize()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        for _ in range(10):
            torch.matmul(a, w.t())
        x1.record(stream)
        torch.cuda.synchronize()
        cub.append(x0.elapsed_time(x1) / 10)
    peaks, peak_src = load_peaks()
    peak = peaks.get("bf16_tflops", 1900.0)
    result = {
        "metric": "projection GEMM tokens/s and achieved tensor TFLOPS vs GB300 roofline",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, "
        "N(0,1/K) weights; no trained weights)",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                   "tokens_per_step": M, "flop_per_step": flops,
                   "l2": "inputs (67 MB activations + 88 MB weights) about L2-sized; no flush: "
                         "warm-L2 figure, as the projections of one step are",
                   "parallelism": f"dp{world} (independent batch per GPU, no collective)"},
        "e2e": {"value": sum_over_ranks(M, world, dev) / (ms_e2e / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": M * K * 2,
                "d2h_bytes_per_step": sum(M * N * 2 for N in shapes), "ms_per_step": ms_e2e},
        "gpu_launches": launches,
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                     "frac": tf / peak, "traffic": traffic_record("gemm.cu", "projections"),
                     "kernel": "tcgen05 projection GEMM",
                     "algorithmic": f"{flops:.4g} FLOP per step (2*M*N*K, QKV and O)",
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json, burst)"},
        "library_gemm_ms": {"qkv": cub[0], "o": cub[1],
                            "tflops": flops / (sum(cub) / 1e3) / 1e12},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = projections_cpu_baseline(a, ws, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def projections_cpu_baseline(a, ws, budget_s=15.0):
    """The fp64 oracle (oracle.gemm.linear) on row blocks of the same batch
    until about budget_s seconds; tokens/s = rows through both GEMMs / time."""
    from oracle import gemm as og
    cores = len(os.sched_getaffinity(0))
    wc = [w.cpu() for w in ws]
    rows, t0, blk = 0, time.perf_counter(), 64
    while time.perf_counter() - t0 < budget_s and rows < a.shape[0]:
        ab = a[rows:rows + blk].cpu()
        for w in wc:
            og.linear(ab, w)
        rows += ab.shape[0]
    secs = time.perf_counter() - t0
    return {"value": rows / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows} of {a.shape[0]} rows through both GEMMs in {secs:.1f} s; numpy "
                      f"fp64 matmul with BLAS threads = "
                      f"{os.environ.get('OPENBLAS_NUM_THREADS', 'all')} of {cores} cores"}


class OracleSampler:
    """Times the fp64 oracle, as it stands, on units of a workload: a unit is
    one request's new rows at one step, taken in a fixed random order.  Setting a request up (its pages and
    every step's new rows copied to the host, appended with the oracle's own
    scatter) is not timed; the oracle's attention over the unit is.  A unit
    of more than ``cap`` rows is timed on ``cap`` evenly spaced rows and its
    time scaled to all of its rows."""

    def __init__(self, wl, cap=64):
        import numpy as np
        self.wl, self.cap = wl, cap
        self.last = len(wl.steps) - 1
        L = wl.steps[self.last].layout
        self.reqs = [r for r in range(L.num_requests)
                     if any(int(st.layout.q_len[r]) > 0 for st in wl.steps)]
        units = [(r, s) for r in self.reqs for s in range(len(wl.steps))
                 if int(wl.steps[s].layout.q_len[r]) > 0]
        # a fixed random order, so that any prefix of it samples the batch's mix
        # (prefill chunks, verify drafts, decode rows) without favouring the first
        perm = np.random.default_rng(12345).permutation(len(units))
        self.units = [units[i] for i in perm]
        self.pos = 0
        self._req, self._sub, self._pools = None, None, None
        self._done = {}
        self.np = np

    def _setup(self, r):
        import oracle
        import workloads
        if self._req == r:
            return
        if r in self._done:
            self._req, (self._sub, self._pools) = r, self._done[r]
            return
        sub = workloads.sub_workload(self.wl, self.last, [r])
        pk, pv = sub.pool_k, sub.pool_v
        for st in sub.steps:
            L = st.layout
            pk, pv = oracle.reference_scatter(pk, pv, st.k_new, st.v_new, L.q_indptr,
                                              L.cached_len, L.page_indptr, L.page_indices,
                                              L.page_size)
        self._req, self._sub, self._pools = r, sub, (pk, pv)
        if len(self._done) < 16:                 # requests set up so far, kept for the wrap
            self._done[r] = (sub, (pk, pv))

    def next_unit(self):
        """(rows of the unit, rows timed, seconds timed) of the next unit (wrapping)."""
        import oracle
        np = self.np
        r, s = self.units[self.pos % len(self.units)]
        self.pos += 1
        self._setup(r)
        st = self._sub.steps[s]
        L = st.layout
        n = int(L.q_len[0])
        sel = np.unique(np.linspace(0, n - 1, min(n, self.cap)).round().astype(np.int64))
        pk, pv = self._pools
        t0 = time.perf_counter()
        oracle.paged_attention(st.q, pk, pv, L.q_indptr, L.kv_len, L.page_indptr,
                               L.page_indices, L.page_size, L.sm_scale, L.num_kv_heads,
                               tokens=sel, tree_parent=L.tree_parent)
        return n, len(sel), time.perf_counter() - t0

    def run(self, budget_s, min_units=1):
        """Units until ``budget_s`` of timed oracle work (or four times that of
        wall time, set-up included): (rows, estimated s, units, timed s)."""
        rows, est, units, timed = 0, 0.0, 0, 0.0
        w0 = time.perf_counter()
        while units < min_units or (timed < budget_s and
                                    time.perf_counter() - w0 < 4 * budget_s):
            n, m, dt = self.next_unit()
            rows += n
            est += dt * n / m
            timed += dt
            units += 1
            if units >= len(self.units) and timed >= 0.2 * budget_s:
                break
        return rows, est, units, timed


def cpu_baseline(wl, budget_s=15.0):
    """The fp64 oracle, as it stands, timed on this host on a bounded sample
    of the same workload (OracleSampler units, in request order)."""
    cores = len(os.sched_getaffinity(0))
    smp = OracleSampler(wl)
    rows, est, units, timed = smp.run(budget_s)
    L = wl.steps[-1].layout
    return {"value": rows / est if est else None, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{units} of {len(smp.units)} (request, step) units (fixed random order) of "
                      f"{L.num_requests} "
                      f"requests x {len(wl.steps)} step(s), {rows} new tokens; units of more than "
                      f"{smp.cap} rows timed on {smp.cap} evenly spaced rows and scaled "
                      f"({timed:.1f} s of oracle time); numpy fp64 with BLAS threads = "
                      f"{os.environ.get('OPENBLAS_NUM_THREADS', 'all')} of {cores} cores"}


def run_reference(args):
    """The oracle as the reference arm (rank 0 only)."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import torch
    import workloads
    if args.workload in ("cache_serving", "engine_serving"):
        cores = len(os.sched_getaffinity(0))
        trace = workloads.cache_trace(seed=6) if args.workload == "cache_serving" else \
            workloads.cache_trace(seed=7, doc_frac=0.25)
        cache_serving_cpu_baseline(trace, budget_s=min(2.0, args.cpu_seconds))   # warm-up
        t0 = time.perf_counter()
        base = cache_serving_cpu_baseline(trace, budget_s=args.cpu_seconds)
        wall = time.perf_counter() - t0
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": base["value"], "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded token ids and N(0,1) bf16 Q/K/V rows; no dataset)",
            "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                       "parallelism": "host cores, rank 0 only"},
            "cpu_baseline": base,
            "e2e": {"value": base["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    if args.workload == "projections":
        cores = len(os.sched_getaffinity(0))
        g = torch.Generator().manual_seed(8)
        M, K = 8229, 4096
        a = torch.randn((M, K), generator=g).to(torch.bfloat16)
        ws = [(torch.randn((N, K), generator=g) / K ** 0.5).to(torch.bfloat16) for N in (6144, 4096)]
        t0 = time.perf_counter()
        base = projections_cpu_baseline(a, ws, budget_s=args.cpu_seconds)
        wall = time.perf_counter() - t0
        print(json.dumps({
            "impl": "reference", "metric": "projection GEMM tokens/s and achieved tensor TFLOPS "
            "vs GB300 roofline", "value": base["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) activations, N(0,1/K) weights)",
            "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                       "parallelism": "host cores, rank 0 only"},
            "cpu_baseline": base,
            "e2e": {"value": base["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    # The attention configurations: the same seeded workload as the GPU arm
    # (drawn on the GPU when there is one, so the values are identical), the
    # oracle timed on a bounded sample per step.
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    name = args.workload or HEADLINE
    wl = make_attention_workload(name, args, dev, 0)
    smp = OracleSampler(wl)
    per_step = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        smp.run(per_step)
    rows, est, units, timed = 0, 0.0, 0, 0.0
    for _ in range(args.steps):
        n, e, u, t = smp.run(per_step)
        rows, est, units, timed = rows + n, est + e, units + u, timed + t
    value = rows / est
    cores = len(os.sched_getaffinity(0))
    sample = (f"per step about {per_step:.2f} s of oracle time: (request, step) units in a "
              f"fixed random order, wrapping; units of more than {smp.cap} rows timed on {smp.cap} evenly "
              f"spaced rows and scaled; {units} units, {rows} new tokens over {args.steps} timed "
              f"steps; fp64 numpy oracle on {cores} host cores")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": est / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, seeded layouts; no dataset)",
        "config": {"workload": f"{name}: {DESCRIPTIONS[name]}",
                   "parallelism": "host cores, rank 0 only"},
        "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample, "value": value,
                         "unit": "tokens/s"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None, choices=sorted(DESCRIPTIONS),
                    help="one workload; default: every configuration of the attention path "
                         f"({', '.join(SUITE)}), headline {HEADLINE}")
    ap.add_argument("--impl", default="pps", choices=["pps", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=6.0,
                    help="oracle time of the CPU baseline, per configuration")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: oracle time over all warm-up and timed steps")
    ap.add_argument("--flush-l2", default="auto", choices=["auto", "on", "off"],
                    help="re-time the kernels with an L2 flush before each step "
                         "(auto: when the unique KV is under 4x the L2 size)")
    ap.add_argument("--small-rows-cuda-cores", action="store_true",
                    help="small-row tasks on the CUDA-core split-KV kernel "
                         "(PPS_PLAN_SMALL_ROWS_CUDA_CORES) instead of the key-tile kernel")
    ap.add_argument("--fused-append", action="store_true",
                    help="device-resident steps with the append inside the first attention "
                         "kernel (PPS_PLAN_FUSED_APPEND) instead of its own launch")
    ap.add_argument("--requests", type=int, default=0,
                    help="decode_heavy / long_prefill: number of requests (default 256 / 4); "
                         "for small profiling captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in ("cache_serving", "engine_serving"):
        run_cache_serving(args)
    elif args.workload == "projections":
        run_projections(args)
    elif args.workload is None:
        run_suite(args)
    else:
        run_pps(args)


if __name__ == "__main__":
    main()
