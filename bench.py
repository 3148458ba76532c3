"""Benchmark: packed document-masked attention TFLOP/s on one GB300 (or N
independent replicas under torchrun).

A step is one pass of the hot path over one synthetic pack: the device
worklist build (slices, exact pair costs, LPT over persistent CTAs) and the
tcgen05 attention forward.  FLOPs count only allowed (unmasked) query-key
pairs: 4 * head_dim per pair and q head (QK^T and PV).  The zigzag context-
parallel path (shard maps, row gathers, per-pair partial attention, merges)
is timed beside it on the same pack.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 128k]
    python bench.py --impl reference     # the fp64 CPU oracle on a bounded sample
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
import tempfile
import time
from typing import Optional

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from packed_varlen_attention_cu_gb300 import workloads as W  # noqa: E402

METRIC = "packed doc-masked attn TFLOP/s (unmasked pairs) and % of GB300 BF16 peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
DISPATCH = {"dynamic": 0, "static": 1}  # pva_dispatch

WORKLOADS = {
    "128k": (W.zigzag_pack, "128K causal pack: lognormal lengths (median 2048, sigma 1.5, "
                            "clip [1, 65536], seed 0), 32 q / 8 kv heads, d=128, bf16 N(0,1)"),
    "libra": (W.libra_pair, "Libra pair: 1x40960 + 10x4096 tokens, 16/16 heads, d=128"),
    "longtail": (W.long_tail_gqa, "long-tail GQA: 8 packs x 32768 (median 644, sigma 1.6), "
                                  "14 q / 2 kv heads, d=64"),
    "sq": (W.shared_question, "shared question: 4096 + 8x2048, 16/4 heads, d=128"),
    "window": (W.sliding_window, "sliding window 4096: docs 131072/65536/49152/16384, "
                                 "16/4 heads, d=128"),
    "tiny": (W.tiny_pack, "tiny pack: 2048 tokens, lognormal(5,1) clip [16,1024], 4/4 heads, d=64"),
    "short": (W.short_docs, "short-document pack: 131072 tokens, lognormal(ln 64, 0.75) clip "
                            "[8, 512], 32 q / 8 kv heads, d=128"),
}


# ----------------------------------------------------------------- helpers
def make_workload(args):
    """The named workload; --pack-tokens shrinks the 128K pack to a smaller
    pack drawn with the same length recipe (used for profiling captures)."""
    mk, desc = WORKLOADS[args.workload]
    if args.pack_tokens and args.workload == "128k":
        w = W.Workload(f"{args.pack_tokens}-token causal pack H=32/8 d=128",
                       W.lognormal_doc_lengths(args.pack_tokens, math.log(2048.0), 1.5, 1,
                                               65536, 0), 32, 8, 128, cp=8)
        desc = desc.replace("128K", f"{args.pack_tokens}-token")
    elif args.workload == "longtail" and getattr(args, "longtail_packs", 8) != 8:
        w = W.long_tail_gqa(args.longtail_packs)
        desc = desc.replace("8 packs", f"{args.longtail_packs} pack(s)")
    else:
        w = mk()
    if args.c_tile is None:
        from packed_varlen_attention_cu_gb300 import api
        args.c_tile = api.default_c_tile(w.head_dim)
    return w, desc


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# device headers every kernel source includes: a change to them changes the kernel too
KERNEL_HEADERS = ("common.h", "ptx.cuh", "tma_map.h", "unit_feed.cuh", "wl_layout.cuh")


def kernel_source_sha(kernel_file: str):
    """sha256 over a kernel source and the device headers it includes (None if missing)."""
    csrc = os.path.join(ROOT, "packed_varlen_attention_cu_gb300", "csrc")
    h = hashlib.sha256()
    for name in (kernel_file,) + KERNEL_HEADERS:
        path = os.path.join(csrc, name)
        if not os.path.exists(path):
            return None
        h.update(open(path, "rb").read())
    return h.hexdigest()


def profile_traffic(kernel_file: str, profile_name: str):
    """Per-launch DRAM bytes from a committed ncu summary, if the kernel
    source and its headers are unchanged since it was taken (sha256 recorded
    in the summary, from kernel_source_sha)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    sha = kernel_source_sha(kernel_file)
    if not os.path.exists(path) or sha is None:
        return None
    vals = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_dir: Optional[str] = None):
        self.gpu = gpu_index
        self.proc = None
        out_dir = out_dir or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"pva_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples under load: drop the idle ramp at both ends
        load = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus: int):
    """(rank, world, local_rank) from the torchrun environment, NCCL group for N > 1."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def aggregate(seconds: float, flops: float, world: int):
    """Whole-job numbers: max time over ranks, sum of FLOPs (weak scaling, no
    data-path collective; the reduction only collects the timing)."""
    if world <= 1:
        return seconds, flops
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    f = torch.tensor([flops], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(f, op=dist.ReduceOp.SUM)
    return float(t.item()), float(f.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- device arm
def run_pva(args, rank, world, local):
    import torch

    from packed_varlen_attention_cu_gb300 import api
    from packed_varlen_attention_cu_gb300 import build as pva_build

    pva_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w, desc = make_workload(args)
    T, hq, hkv, d = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    stream = torch.cuda.current_stream()
    cu_np = w.cu_seqlens
    cu = torch.from_numpy(cu_np).to(dev)
    q, k, v = W.workload_qkv(w, device=str(dev))
    mask = api.mask_for_workload(w)
    out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((hq, T), dtype=torch.float32, device=dev)
    num_ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    busy = torch.zeros((num_ctas, 2), dtype=torch.int64, device=dev)
    fit = None
    if args.fit_cost:
        # warm-up calibration ("数据并行负载均衡" §4.2): two runs whose worklists are
        # balanced with different per-tile costs, per-CTA times pooled into the fit
        cal_wl, cal_busy = [], []
        for ct in (0, 4 * args.c_tile):
            cp_ = api.make_params(hq, hkv, num_ctas=0, c_tile=ct, dispatch=api.DISPATCH_STATIC)
            cw = api.alloc_worklist(w.num_docs, mask, cp_, dev)
            cb = torch.zeros((num_ctas, 2), dtype=torch.int64, device=dev)
            api.build_worklist(cu, mask, cp_, cw, stream)
            for _ in range(2):
                api.attn_fwd(q, k, v, cu, mask, cp_, cw, out, lse, 0.0, cb, stream)
            cal_wl.append(cw)
            cal_busy.append(cb)
        torch.cuda.synchronize()
        fitted, coef = api.fit_tile_cost(cal_wl, cal_busy)
        fit = {"default_c_tile": args.c_tile, "fitted_c_tile": fitted,
               "ns_per_pair": coef[0], "ns_per_tile": coef[1],
               "calibration": "warm-up: 2 runs with c_tile 0 and 4x default, per-CTA times "
                              "fitted t = a*pairs + c*(tiles + sub-tiles), a, c >= 0"}
        args.c_tile = fitted
        del cal_wl, cal_busy
    params = api.make_params(hq, hkv, num_ctas=0, c_tile=args.c_tile,
                             refine_iters=args.refine_iters, dispatch=DISPATCH[args.dispatch],
                             pack_docs=1 if args.pack_docs else 0)
    wl = api.alloc_worklist(w.num_docs, mask, params, dev)

    api.build_worklist(cu, mask, params, wl)
    counts = api.worklist_counts(wl)
    assert counts["status"] == 0, counts
    pairs = counts["pairs_per_head"]
    flops = 4.0 * d * hq * pairs
    n_wl_kernels = api.worklist_build_kernels(params)
    io_bytes = (q.numel() + k.numel() + v.numel() + out.numel()) * 2 + lse.numel() * 4

    def step(ev_a=None, ev_b=None):
        api.build_worklist(cu, mask, params, wl, stream)
        if ev_a is not None:
            ev_a.record(stream)
        api.attn_fwd(q, k, v, cu, mask, params, wl, out, lse, 0.0, None, stream)
        if ev_b is not None:
            ev_b.record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert api.worklist_error(wl) == 0

    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local, args.clocks_dir) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(K):
            step(*evs[i])
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    total_s = start.elapsed_time(end) / 1e3
    attn_ms = [a.elapsed_time(b) for a, b in evs]
    wall_s, job_flops = aggregate(total_s, flops * K, world)
    value = job_flops / wall_s / 1e12
    attn_avg_s = sum(attn_ms) / len(attn_ms) / 1e3
    achieved = flops / attn_avg_s / 1e12

    # per-CTA busy time of one more launch (same configuration)
    api.attn_fwd(q, k, v, cu, mask, params, wl, out, lse, 0.0, busy, stream)
    torch.cuda.synchronize()
    b = busy.cpu().numpy().astype(np.float64)
    dur = b[:, 1] - b[:, 0]
    worked = dur[dur > 0]
    imbalance = float(worked.max() / worked.min() - 1.0) if worked.size else None

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # a summary covers one workload at its full size; a shrunk pack has none
    shrunk = args.pack_tokens or args.longtail_packs != 8
    traffic = None if shrunk else profile_traffic("attn_fwd.cu", f"attn_fwd_{args.workload}.txt")

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(wall_s / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator; lengths and values described in config)",
        "config": {"workload": desc, "tokens": T, "docs": w.num_docs, "q_heads": hq,
                   "kv_heads": hkv, "head_dim": d, "mask": w.mask_kind,
                   "pairs_per_head": pairs, "flops_per_step": flops,
                   "step": f"device worklist build ({n_wl_kernels} kernels) + attention forward (1 kernel)",
                   "l2": f"inputs larger than L2: Q+K+V+O+LSE = {io_bytes / 1e9:.2f} GB "
                         f"> {L2_BYTES / 1e6:.0f} MB, no flush",
                   "num_ctas": num_ctas, "c_tile": args.c_tile, "c_tile_fit": fit,
                   "dispatch": args.dispatch, "pack_docs": bool(args.pack_docs),
                   "refine_iters": args.refine_iters,
                   "parallelism": f"{world} independent replica(s), one per GPU"},
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst); frac vs sustained "
                                    f"{peak_sus}: {achieved / peak_sus:.4f}",
                     "kernel": "attn_fwd_kernel<128, false>" if d == 128 else "attn_fwd_kernel<64, false>",
                     "algorithmic_flops_per_launch": flops,
                     "avg_launch_ms": round(attn_avg_s * 1e3, 4)},
        "imbalance": None if imbalance is None else round(imbalance, 4),
        "gpu_launches": K * (n_wl_kernels + 1),
        "clocks": clocks.summary(),
        "worklist_ms": round((wall_s - attn_avg_s * K) / K * 1e3, 4),
        "worklist": {"units": counts["units"], "lpt_steps": counts["lpt_steps"],
                     "tiles_per_head": counts["tiles_per_head"],
                     "refine_rounds": api.worklist_refine_rounds(wl)},
    }
    return result, (w, q, k, v, cu_np, flops, mask, params, hbm)


def run_e2e(args, ctx, world):
    """Same metric through the public C ABI with host buffers
    (pva_attn_fwd_host): per step, H2D of Q/K/V/cu_seqlens from pinned memory,
    worklist + attention, D2H of O/LSE, all enqueued by the one call.  Steps
    rotate over args.e2e_streams streams with their own device buffers, as a
    caller streaming packs would, so a step's copies in overlap the previous
    steps' attention and copies out (a stream's next copy in waits for its own
    copy out, so two streams leave the link idle while a step computes); every
    step still moves all of its bytes."""
    import torch

    from packed_varlen_attention_cu_gb300 import api
    w, q, k, v, cu_np, flops, mask, params, _ = ctx
    dev = q.device
    hq_, hk_, hv_ = (t.cpu().pin_memory() for t in (q, k, v))
    hcu = torch.from_numpy(cu_np).pin_memory()
    T, hq, d = q.shape
    o_h = torch.empty((T, hq, d), dtype=torch.bfloat16).pin_memory()
    l_h = torch.empty((hq, T), dtype=torch.float32).pin_memory()
    ns = max(1, args.e2e_streams)
    streams = [torch.cuda.Stream(device=dev) for _ in range(ns)]
    bufs = [api.alloc_host_path_buffers(hq_, hk_, w.num_docs, mask, params, dev)
            for _ in range(ns)]
    nsteps = [0]

    def step():
        i = nsteps[0] % ns
        nsteps[0] += 1
        api.attn_fwd_host(hq_, hk_, hv_, hcu, w.num_docs, mask, params, o_h, l_h, bufs[i],
                          0.0, streams[i])

    for _ in range(max(4, ns)):
        step()
    torch.cuda.synchronize()
    # at least twenty rounds of the rotation: each window starts with the link and
    # the SMs idle and ends with the last step's compute and copy out, which the
    # steps of a continuous stream of packs would overlap (about one step's
    # compute plus its copy out per window)
    K = max(20 * ns, (args.steps // 2) // ns * ns)
    cur = torch.cuda.current_stream()
    # The host link is shared with the rest of the machine and its rate moves between
    # runs, so three windows of K steps are timed and the median window is reported
    # (every window listed).
    windows = []
    for _ in range(3):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        s.record(cur)
        for st in streams:
            st.wait_event(s)
        for _ in range(K):
            step()
        for st in streams:
            cur.wait_stream(st)
        e.record(cur)
        torch.cuda.synchronize()
        barrier(world)
        windows.append(aggregate(s.elapsed_time(e) / 1e3, flops * K, world))
    for b in bufs:
        assert api.worklist_error(b["worklist"]) == 0
    t, f = sorted(windows)[1]
    h2d = (q.numel() + k.numel() + v.numel()) * 2 + cu_np.nbytes
    d2h = o_h.numel() * 2 + l_h.numel() * 4
    return {"value": round(f / t / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": K, "ms_per_step": round(t / K * 1e3, 4),
            "windows_ms_per_step": [round(w[0] / K * 1e3, 4) for w in windows],
            "path": f"pva_attn_fwd_host (pinned host buffers), {ns} streams in rotation"}


def run_zigzag(args, ctx, world, per_step=False, fused=False):
    """Zigzag CP emulation on one GPU (packed_varlen_attention_cu_gb300.ring):
    cp virtual ranks; rank r runs its Q shard against the KV shard of rank
    (r - t) mod cp at ring step t, merging into the running (O, LSE); outputs
    stay rank-local.  per_step: one worklist + attention launch per ring step
    over every rank (Q/K/V in ring order) instead of one per (rank, step) pair.
    fused: steps t > 0 merge in the attention epilogue (pva_attn_fwd_accumulate)
    instead of writing a partial and running pva_merge_partials."""
    import torch

    from packed_varlen_attention_cu_gb300.ring import ZigzagRing
    w, q, k, v, cu_np, flops, _, base_params, hbm = ctx
    cp = w.cp or 8
    dev = q.device
    stream = torch.cuda.current_stream()
    T, hq, d = q.shape
    ring = ZigzagRing(cu_np, cp, hq, k.shape[1], d, c_tile=base_params.c_tile,
                      dispatch=base_params.dispatch, per_step=per_step, fused=fused, device=dev)
    merge_ev = []
    ring.step(q, k, v, stream)
    torch.cuda.synchronize()
    K = max(2, args.steps // 20)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    s.record(stream)
    for i in range(K):
        ring.step(q, k, v, stream, merge_ev if i == K - 1 else None)
    e.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    import packed_varlen_attention_cu_gb300.api as api
    for wl in ring.worklists():
        assert api.worklist_error(wl) == 0
    t, f = aggregate(s.elapsed_time(e) / 1e3, flops * K, world)
    scheme = ("one worklist + attention launch per ring step over all ranks (Q/K/V in ring "
              "order)" if per_step else "one worklist + attention launch per (rank, step) pair")
    res = {"value": round(f / t / 1e12, 2), "unit": "TFLOP/s", "cp": cp, "steps": K,
           "ms_per_step": round(t / K * 1e3, 3),
           "gpu_launches_per_step": ring.launches_per_step(),
           "note": f"cp virtual ranks on one GPU: {scheme}; "
                   + ("ring steps t > 0 merge into the running (O, LSE) in the attention "
                      "epilogue (no partials, no merge launches)" if fused else
                      "fp32 partials merged in place by pva_merge_partials")}
    if merge_ev:
        mtimes = [a.elapsed_time(b) / 1e3 for a, b, _ in merge_ev]
        mbytes = [n * hq * (3 * 4 * d + 3 * 4) for _, _, n in merge_ev]
        gbs = sum(mbytes) / sum(mtimes) / 1e9
        res["merge"] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(gbs / hbm, 4), "bytes_per_row": 3 * 4 * d + 3 * 4,
                        "launches_per_step": len(merge_ev),
                        "avg_launch_ms": round(1e3 * sum(mtimes) / len(mtimes), 4)}
    return res


def run_dispatch(args, ctx):
    """Sharding solvers ("03 · 长文负载均衡" §4.2-§4.4) on this pack: device chunk
    areas + min-heap dispatch (timed), the balance they reach against contiguous,
    zigzag and striped chunk placement, and WLB-LLM's per-seq / per-doc choice."""
    import torch

    from packed_varlen_attention_cu_gb300 import api
    w, q, k, v, cu_np, flops, _, base_params, hbm = ctx
    if w.mask_kind not in (W.MASK_CAUSAL, W.MASK_SLIDING_WINDOW, W.MASK_SHARED_QUESTION):
        return None
    cp = w.cp or 8
    T = w.total_tokens
    cs = 1024
    while ((T + cs - 1) // cs) % cp and cs > 1:
        cs //= 2
    n = (T + cs - 1) // cs
    if n % cp or n > 8192:
        return None
    dev = q.device
    stream = torch.cuda.current_stream()
    cu = torch.from_numpy(cu_np).to(dev)
    mask = api.mask_for_workload(w)
    areas = torch.empty((n,), dtype=torch.int64, device=dev)
    bucket = torch.empty((n,), dtype=torch.int32, device=dev)
    loads = torch.empty((cp,), dtype=torch.int64, device=dev)
    reps = 20
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for i in range(reps + 3):
        if i == 3:
            ev[0].record(stream)
        api.chunk_areas(cu, mask, cs, areas, stream)
        if i == 3:
            ev[1].record(stream)
        api.dispatch_chunks(areas, cp, bucket, loads, stream)
        if i == 3:
            ev[2].record(stream)
    torch.cuda.synchronize()
    t_areas = ev[0].elapsed_time(ev[1]) * 1e3
    t_disp = ev[1].elapsed_time(ev[2]) * 1e3
    a = areas.cpu().numpy()
    mean = a.sum() / cp

    def ratio(assign):
        return round(float(np.bincount(assign, weights=a, minlength=cp).max() / mean), 4)

    idx = np.arange(n)
    zz_rank = np.where((idx * 2 * cp // n) < cp, idx * 2 * cp // n, 2 * cp - 1 - idx * 2 * cp // n)
    choice, costs = api.wlb_choose(cu_np, cp, 128, w.head_dim)
    return {"chunk_size": cs, "chunks": n, "cp": cp,
            "chunk_areas_us": round(t_areas, 1), "dispatch_us": round(t_disp, 1),
            "max_bucket_over_mean": {"minheap": ratio(bucket.cpu().numpy()),
                                     "contiguous": ratio(idx * cp // n),
                                     "zigzag_chunks": ratio(zz_rank),
                                     "striped_chunks": ratio(idx % cp)},
            "wlb": {"choice": ("per-sequence", "per-document")[choice],
                    "max_worker_tflop": {"per_sequence": round(costs[0].max() * w.num_q_heads / 1e12, 3),
                                         "per_document": round(costs[1].max() * w.num_q_heads / 1e12, 3)}},
            "note": "areas = allowed pairs per query chunk; buckets hold n/cp chunks each; "
                    "WLB costs are tile-rounded (128) FLOPs of the most loaded worker"}


def run_backward(args, ctx, world):
    """Attention backward on this pack (pva_attn_bwd): per step the backward
    plan build (2 kernels + sort) and the backward (D, dQ, dK/dV kernels), with
    a seeded dO.  FLOPs = 10 d per allowed pair per q head (S, dP, dV, dK, dQ;
    the dQ and dK/dV passes each recompute S and dP, not counted)."""
    import torch

    from packed_varlen_attention_cu_gb300 import api
    w, q, k, v, cu_np, flops_fwd, mask, params, hbm = ctx
    dev = q.device
    stream = torch.cuda.current_stream()
    T, hq, d = q.shape
    cu = torch.from_numpy(cu_np).to(dev)
    wl = api.alloc_worklist(w.num_docs, mask, params, dev)
    api.build_worklist(cu, mask, params, wl, stream)
    out = torch.empty_like(q)
    lse = torch.empty((hq, T), dtype=torch.float32, device=dev)
    api.attn_fwd(q, k, v, cu, mask, params, wl, out, lse, 0.0, None, stream)
    dout = W.make_qkv(T, T, hq, k.shape[1], d, w.seed + 1000, device=str(dev))[0]
    plan = api.alloc_bwd_plan(w.num_docs, mask, params, dev)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)

    def step():
        api.build_bwd_plan(wl, w.num_docs, mask, params, plan, stream)
        api.attn_bwd(q, k, v, out, lse, dout, cu, w.num_docs, mask, params, wl, plan, dq, dk,
                     dv, 0.0, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert api.worklist_error(wl) == 0
    K = max(3, args.steps // 2)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    s.record(stream)
    for _ in range(K):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    flops = flops_fwd * 2.5
    t, f = aggregate(s.elapsed_time(e) / 1e3, flops * K, world)
    return {"value": round(f / t / 1e12, 2), "unit": "TFLOP/s", "steps": K,
            "ms_per_step": round(t / K * 1e3, 4),
            "frac_of_peak": None,
            "flops_per_step": flops, "gpu_launches_per_step": 3 + 4,
            "note": "backward plan (plan kernel, chunk sort, merge rank) + D, dQ and dK/dV "
                    "kernels, bf16 gradients; 10 d FLOPs per allowed pair per q head"}


def run_libra_ratio(args, ctx):
    """Libra's example ("03 · 长文负载均衡" §1.1): the same token count as one
    40960-token document (pack A) or ten 4096-token documents (pack B); the
    attention work ratio is 10 in sum l^2.  Each pack is timed on its own."""
    import torch

    from packed_varlen_attention_cu_gb300 import api
    w, q, k, v = ctx[:4]
    dev = q.device
    stream = torch.cuda.current_stream()
    res = {}
    for name, lengths, rows in (("A", [40960], slice(0, 40960)),
                                ("B", [4096] * 10, slice(40960, 81920))):
        cu_np = W.cu_seqlens_of(lengths)
        cu = torch.from_numpy(cu_np).to(dev)
        qa, ka, va = q[rows].contiguous(), k[rows].contiguous(), v[rows].contiguous()
        T = qa.shape[0]
        mask = api.make_mask(W.MASK_CAUSAL, T, T)
        params = api.make_params(w.num_q_heads, w.num_kv_heads, num_ctas=0, c_tile=args.c_tile,
                                 dispatch=DISPATCH[args.dispatch])
        wl = api.alloc_worklist(len(lengths), mask, params, dev)
        out = torch.empty_like(qa)
        lse = torch.empty((qa.shape[1], T), dtype=torch.float32, device=dev)
        api.build_worklist(cu, mask, params, wl)
        for _ in range(3):
            api.attn_fwd(qa, ka, va, cu, mask, params, wl, out, lse)
        reps = 10
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s.record(stream)
        for _ in range(reps):
            api.attn_fwd(qa, ka, va, cu, mask, params, wl, out, lse)
        e.record(stream)
        torch.cuda.synchronize()
        pairs = api.worklist_counts(wl)["pairs_per_head"]
        t = s.elapsed_time(e) / reps
        res[name] = {"ms": round(t, 4), "pairs_per_head": pairs,
                     "tflops": round(4.0 * w.head_dim * w.num_q_heads * pairs / t / 1e9, 2)}
    res["time_ratio_A_over_B"] = round(res["A"]["ms"] / res["B"]["ms"], 4)
    res["sum_sq_ratio"] = 10.0
    res["pairs_ratio"] = round(40961 / 4097, 5)
    res["tile_ratio_b128"] = round(51360 / 5280, 5)
    return res


# ----------------------------------------------------------------- CPU oracle
def oracle_sample(w, q_bits, k_bits, v_bits, seconds: float, seed: int = 7):
    """Time the fp64 oracle on a bounded random sample of (row, head) jobs
    of the workload; returns (TFLOP/s, cores, description, elapsed)."""
    import oracle
    oracle.compile_oracle()
    T, hq, d = w.total_tokens, w.num_q_heads, w.head_dim
    cu = w.cu_seqlens
    docs = np.searchsorted(cu, np.arange(T), side="right") - 1
    keys_per_row = (np.arange(T) - cu[docs] + 1).astype(np.int64)  # causal per document
    if w.mask_kind == W.MASK_SLIDING_WINDOW:
        keys_per_row = np.minimum(keys_per_row, w.window)
    elif w.mask_kind == W.MASK_SHARED_QUESTION:
        keys_per_row = keys_per_row + np.where(docs >= w.num_prefix_docs,
                                               int(cu[w.num_prefix_docs]), 0)
    m = oracle.Mask(w.mask_kind, window=w.window, num_prefix=w.num_prefix_docs)

    def run(n, s):
        jobs = W.random_rows(T, hq, n, seed=s)
        t0 = time.perf_counter()
        oracle.attention(q_bits, k_bits, v_bits, cu, m, jobs=jobs)
        dt = time.perf_counter() - t0
        return dt, float(keys_per_row[jobs[:, 0]].sum()), n

    dt, _, n = run(256, seed)
    n_target = int(max(256, min(2_000_000, 256 * seconds / max(dt, 1e-3))))
    dt, pairs, n = run(n_target, seed + 1)
    flops = 4.0 * d * pairs
    cores = oracle.num_threads()
    desc = (f"{n} random (row, head) jobs of the workload, fp64, OpenMP over {cores} threads, "
            f"{pairs:.3e} allowed pairs, {dt:.1f} s")
    return flops / dt / 1e12, cores, desc, dt


def run_reference(args):
    """The oracle, as it stands, on the host cores: each step a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import torch
    w, desc = make_workload(args)
    import oracle
    q, k, v = W.workload_qkv(w, device="cpu")
    qb, kb, vb = oracle.bf16_bits(q), oracle.bf16_bits(k), oracle.bf16_bits(v)
    per_step = max(1.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    vals, times, cores, sample = [], [], 1, ""
    for i in range(args.warmup + args.steps):
        tf, cores, sample, dt = oracle_sample(w, qb, kb, vb, per_step, seed=100 + i)
        if i >= args.warmup:
            vals.append(tf)
            times.append(dt)
    value = float(np.mean(vals))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * float(np.mean(times)), 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": desc, "tokens": w.total_tokens,
                                            "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                                            "head_dim": w.head_dim},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("pva", "reference"), default="pva")
    ap.add_argument("--workload", choices=tuple(WORKLOADS), default="128k")
    ap.add_argument("--c-tile", type=int, default=None,
                    help="per-tile fixed cost in pair units (default: api.default_c_tile(d))")
    ap.add_argument("--pack-tokens", type=int, default=0)
    ap.add_argument("--longtail-packs", type=int, default=8,
                    help="packs of the long-tail workload (seeds 0..n-1)")
    ap.add_argument("--dispatch", choices=tuple(DISPATCH), default="dynamic",
                    help="forward units: claimed in LPT order at run time, or the builder's "
                         "static per-CTA LPT lists")
    ap.add_argument("--pack-docs", action="store_true",
                    help="short documents share tiles (pva_worklist_params.pack_docs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="streams (each with its own device buffers) the e2e steps rotate over")
    ap.add_argument("--no-zigzag", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--fit-cost", action="store_true",
                    help="fit the per-tile cost to per-CTA times of two warm-up runs")
    ap.add_argument("--refine-iters", type=int, default=20,
                    help="move/swap rounds after LPT (0: none)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--clocks-dir", default=None,
                    help="folder for the nvidia-smi clock samples of the timed region "
                         "(default: the system temp folder)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        res = run_reference(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0

    rank, world, local = dist_setup(args.gpus)
    res, ctx = run_pva(args, rank, world, local)
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, ctx, world)
    if not args.no_zigzag and ctx[0].cp:
        res["zigzag_cp"] = run_zigzag(args, ctx, world)
        res["zigzag_cp_fused"] = run_zigzag(args, ctx, world, fused=True)
        res["zigzag_cp_step"] = run_zigzag(args, ctx, world, per_step=True)
        res["zigzag_cp_step_fused"] = run_zigzag(args, ctx, world, per_step=True, fused=True)
    if not args.no_backward:
        bwd = run_backward(args, ctx, world)
        if bwd is not None:
            bwd["frac_of_peak"] = round(bwd["value"] / res["roofline"]["peak"], 4)
            res["backward"] = bwd
    if not args.no_zigzag:
        disp = run_dispatch(args, ctx)
        if disp is not None:
            res["dispatch"] = disp
    if args.workload == "libra":
        res["libra_ratio"] = run_libra_ratio(args, ctx)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # noqa: F401  (CPU baseline leg only)
        from oracle import bf16_bits
        w, q, k, v = ctx[:4]
        tf, cores, sample, _ = oracle_sample(w, bf16_bits(q), bf16_bits(k), bf16_bits(v),
                                             args.cpu_seconds)
        res["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores,
                               "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
