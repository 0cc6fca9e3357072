"""Benchmark: paged MLA decode on GB300, one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all] [--impl ours|reference]

A step is one mla_decode call (split-KV kernel + reduction) over one synthetic
decode batch resident in HBM.  The headline value is the uniform batch; the
default run also measures the varlen, fp8spec and window batches and reports
each under "workloads" with its own roofline record.  L2 is flushed (a 256 MB device write, outside
the timed events) before every timed step.  Under torchrun every rank decodes
its own batch of the same shape (requests are independent: weak scaling, no
collective on the data path); the step time is the maximum over ranks.

--impl reference times the fp64 CPU oracle (the correctness reference) on a
bounded sample of the same workload, on this host's cores.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_latent_attention_mla_gb300 import _native  # noqa: E402
from paged_latent_attention_mla_gb300 import build as nbuild  # noqa: E402
from paged_latent_attention_mla_gb300 import decoder_for  # noqa: E402
from paged_latent_attention_mla_gb300 import workloads as wl  # noqa: E402
from paged_latent_attention_mla_gb300.sharding import max_over_ranks, rank_seed  # noqa: E402

METRIC = "MLA decode µs/call, TFLOP/s and KV HBM GB/s vs GB300 roofline fraction"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLOP_PER_KEY_HEAD = 2 * (576 + 512)  # QK^T over 576 dims + P.V over 512 dims
HEADLINE = "uniform"  # the headline value; the other 128-head workloads get records beside it
ALL = ["uniform", "varlen", "fp8spec", "window"]

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one split-KV kernel launch,
# from an ncu capture of the same batch (profiles/split_kv_tc_<workload>.md; captured with
# --compact-pool, the same pages and tiles in a pool small enough to capture), valid only for
# the kernel sources it was taken on: reported when their hash still matches, else null.
KERNEL_SOURCES = ("mla_split_tc.cu", "mla_common.cuh", "schedule.cuh", "tma_pages.cuh", "ptx.cuh")
NCU_TRAFFIC = {
    "uniform": {"sources_sha256": "c1995718be5b00232ab7e8a732b698b787ec4bb01a2a2cb8fee52dd4cf344551", "bytes": 322160896 + 7964416},
    "varlen": {"sources_sha256": "c1995718be5b00232ab7e8a732b698b787ec4bb01a2a2cb8fee52dd4cf344551", "bytes": 558129152 + 15618560},
    "fp8spec": {"sources_sha256": "c1995718be5b00232ab7e8a732b698b787ec4bb01a2a2cb8fee52dd4cf344551", "bytes": 310328064 + 8987648},
    "window": {"sources_sha256": "c1995718be5b00232ab7e8a732b698b787ec4bb01a2a2cb8fee52dd4cf344551", "bytes": 44969984 + 766976},
}


def kernel_sources_sha256() -> str:
    """Hash of the kernel sources' code: comments and blank lines are left out, so a change
    to the comments alone keeps the captured traffic."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_latent_attention_mla_gb300", "csrc", name)) as f:
            for line in f:
                code = re.sub(r"//.*", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()


def measured_traffic(workload: str):
    rec = NCU_TRAFFIC.get(workload)
    if rec is None or rec["sources_sha256"] != kernel_sources_sha256():
        return None
    return rec["bytes"]


def describe(prob) -> str:
    w = prob.w
    lens = prob.seq_lens.tolist()
    klen = f"K={lens[0]}" if len(set(lens)) == 1 else f"K log-uniform [1,{w.max_len}] (sum {sum(lens)})"
    extra = (" causal" if w.causal else "") + (f" window_left={w.window_left}" if w.window_left >= 0 else "")
    return f"{w.name}: B={w.B} H={w.H} Sq={w.Sq} {klen}{extra} {w.dtype} page_size={w.page_size} pool={prob.pool_pages} pages"


def algorithmic_counts(prob):
    """FLOPs = 2*(576+512)*H*sum|vis(b,t)|; KV bytes = sum_b |union_t vis(b,t)| * 576 * elt."""
    w = prob.w
    elt = 1 if w.dtype == "e4m3" else 2
    flops, kv = 0, 0
    for K in prob.seq_lens.tolist():
        lo_u, hi_u, vis = None, None, 0
        for t in range(w.Sq):
            hi = K - (w.Sq - 1 - t) if w.causal else K
            lo = K - w.Sq - w.window_left + t if w.window_left >= 0 else 0
            hi, lo = min(max(hi, 0), K), min(max(lo, 0), K)
            lo = min(lo, hi)
            vis += hi - lo
            if hi > lo:
                lo_u = lo if lo_u is None else min(lo_u, lo)
                hi_u = hi if hi_u is None else max(hi_u, hi)
        flops += FLOP_PER_KEY_HEAD * w.H * vis
        if lo_u is not None:
            kv += (hi_u - lo_u) * 576 * elt
    return flops, kv


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(prob, budget_s: float = 12.0, threads: int = 0):
    """The oracle as it stands, on this host's cores, over a bounded sample of rows."""
    import oracle

    p = prob.host_inputs()
    total = prob.B * prob.Sq * prob.H
    cores = threads if threads > 0 else len(os.sched_getaffinity(0))
    rows = wl.sample_rows(prob, min(total, 4 * cores))
    t0 = time.perf_counter()
    oracle.decode(p, rows=rows, threads=cores)
    dt = time.perf_counter() - t0
    # the sample sized to a third of the budget, then timed three times (the median)
    n = min(total, max(len(rows), int(len(rows) * budget_s / 3 / max(dt, 1e-3))))
    if n > len(rows):
        rows = wl.sample_rows(prob, n, seed=11)
    times = []
    for _ in range(3):
        t0 = time.perf_counter()
        oracle.decode(p, rows=rows, threads=cores)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    flops = row_flops(prob, rows)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} of {total} (request, token, head) rows, every visible key, fp64 oracle, "
                      f"{cores} thread(s), median of 3 runs of {dt:.2f} s",
            "seconds": dt}


def row_flops(prob, rows):
    w = prob.w
    lens = prob.seq_lens.tolist()
    f = 0
    for r in rows:
        t = (r // w.H) % w.Sq
        b = r // (w.H * w.Sq)
        K = lens[b]
        hi = K - (w.Sq - 1 - t) if w.causal else K
        lo = K - w.Sq - w.window_left + t if w.window_left >= 0 else 0
        hi, lo = min(max(hi, 0), K), min(max(lo, 0), K)
        f += FLOP_PER_KEY_HEAD * max(0, hi - min(lo, hi))
    return f


def run_reference(args, world, rank):
    if rank != 0:
        return
    prob = wl.make_problem(HEADLINE if args.workload == "all" else args.workload)
    times = []
    cb = None
    per_step = min(args.ref_budget, 150.0 / max(1, args.warmup + args.steps))  # whole run within a few minutes
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(prob, budget_s=per_step)
        if i >= args.warmup:
            times.append(cb["seconds"])
    v = cb["value"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(prob), "sample": cb["sample"]},
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def decode_options(args, prob) -> dict:
    """Decoder options the run asks for: the wrapper's defaults (PDL reduction, fp16 partials
    for e4m3) unless told otherwise."""
    opts = {"use_pdl": not args.no_pdl, "combine_in_kernel": args.combine_in_kernel}
    if args.num_clusters:
        opts["num_clusters"] = args.num_clusters
    if args.reducer_d_tiles:
        opts["reducer_d_tiles"] = args.reducer_d_tiles
    if args.fp32_partials:
        opts["partial_fp16"] = False
    return opts


def ev_pair():
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def measure(name, args, world, rank, local_rank, peaks, peak_src):
    """One workload: the device-resident call (L2 flushed before each), the split-KV kernel
    alone, the call through host buffers, and the call without the flush."""
    # --compact-pool: only the pages the batch uses (profiling: the same tiles and traffic in a
    # pool small enough to capture); the default keeps the workload's own pool
    prob = wl.make_problem(name, seed=rank_seed(wl.WORKLOADS[name].seed, rank),
                           pool_pages=0 if args.compact_pool else None, page_size=args.page_size or None)
    d = prob.device_inputs("cuda")
    dec = decoder_for(prob, **decode_options(args, prob))
    flops, kv = algorithmic_counts(prob)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((prob.B, prob.Sq, prob.H, 512), dtype=dec.out_dtype, device="cuda")
    lse = torch.empty((prob.B, prob.Sq, prob.H), dtype=torch.float32, device="cuda")

    def step():
        dec(d["q_latent"], d["q_rope"], d["ckv"], d["kpe"], d["page_table"], d["seq_lens"], d["scale"], out=out,
            lse=lse, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    assert dec.status() == _native.MLA_OK, f"{name}: decode reported an error during warm-up"

    ev = [ev_pair() for _ in range(args.steps)]
    # the split-KV kernel alone: mla_decode records these around its launch (split_timing)
    kev = [ev_pair() for _ in range(args.steps)]
    for a, b in kev:  # create the handles
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        # a second pass of the same steps for the split-KV kernel alone
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            dec.cfg.split_timing[0] = kev[i][0].cuda_event
            dec.cfg.split_timing[1] = kev[i][1].cuda_event
            step()
        torch.cuda.synchronize()
    dec.cfg.split_timing[0] = None
    dec.cfg.split_timing[1] = None
    assert dec.status() == _native.MLA_OK, f"{name}: decode reported an error"
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev))
    kernel_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in kev))

    # end to end through the public API with host buffers: H2D of the step's queries,
    # page table and lengths from pinned memory, decode, D2H of out and lse
    keys = ("q_latent", "q_rope", "page_table", "seq_lens")
    hq = [d[k].cpu().pin_memory() for k in keys]
    dq = [torch.empty_like(d[k]) for k in keys]
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h_lse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in hq)
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

    def e2e_step():
        for h, dv in zip(hq, dq):
            dv.copy_(h, non_blocking=True)
        dec(dq[0], dq[1], d["ckv"], d["kpe"], dq[2], dq[3], d["scale"], out=out, lse=lse, stream=stream)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        a, b = ev_pair()
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    e2e_serial_ms = max_over_ranks(statistics.mean(e_ms))

    # The same steps pipelined as a serving loop runs them: step i's H2D on a copy-in stream,
    # its decode on the compute stream once they land, its D2H on a copy-out stream after
    # it, two sets of buffers, so step i + 1's H2D and step i - 1's D2H overlap step i's
    # decode.  Timed over all steps as a whole (events on the copy streams), with no L2 flush
    # between steps; reported where the batch's KV is larger than L2 (129 MB), so that no
    # step finds its KV left in L2 by the one before.
    e2e_mode = "serial: each step's H2D, decode and D2H in turn, L2 flushed before each step"
    e2e_ms = e2e_serial_ms
    if kv > 129e6:
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        sets = []
        for _ in range(2):
            sets.append(dict(dq=[torch.empty_like(t) for t in dq], out=torch.empty_like(out),
                             lse=torch.empty_like(lse), h_out=torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
                             h_lse=torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)))

        def pipelined(n):
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            done_in = [torch.cuda.Event() for _ in range(n)]
            done_dec = [torch.cuda.Event() for _ in range(n)]
            done_out = [torch.cuda.Event() for _ in range(n)]
            start.record(s_in)
            s_out.wait_event(start)
            stream.wait_event(start)
            for i in range(n):
                b = sets[i & 1]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(done_dec[i - 2])  # set i & 1 no longer read
                    for h, dv in zip(hq, b["dq"]):
                        dv.copy_(h, non_blocking=True)
                    done_in[i].record(s_in)
                stream.wait_event(done_in[i])
                if i >= 2:
                    stream.wait_event(done_out[i - 2])  # set i & 1's outputs read back
                dec(b["dq"][0], b["dq"][1], d["ckv"], d["kpe"], b["dq"][2], b["dq"][3], d["scale"], out=b["out"],
                    lse=b["lse"], stream=stream)
                done_dec[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done_dec[i])
                    b["h_out"].copy_(b["out"], non_blocking=True)
                    b["h_lse"].copy_(b["lse"], non_blocking=True)
                    done_out[i].record(s_out)
            s_out.wait_event(done_in[n - 1])
            end.record(s_out)
            end.synchronize()
            return start.elapsed_time(end) / n

        pipelined(max(2, args.warmup))
        e2e_ms = max_over_ranks(pipelined(args.steps))
        e2e_mode = ("pipelined: step i+1's H2D and step i-1's D2H on copy streams overlap step i's decode "
                    "(two buffer sets), timed over all steps, no L2 flush (the KV is larger than L2)")

    # the same device-resident call back to back with no L2 flush between calls (part of
    # the KV can then still be in L2 from the previous call): reported beside the number
    nf = [ev_pair() for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in nf:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    nf_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in nf))
    launches_per_call = dec.launches_per_call()

    t_hbm = kv / (peaks["hbm_gbs"] * 1e9)
    e4m3 = prob.w.dtype == "e4m3"
    tc_peak = peaks["bf16_tflops"] * (2.0 if e4m3 else 1.0)
    t_tc = flops / (tc_peak * 1e12)
    t_roof = max(t_hbm, t_tc)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    k_gbs = kv / (kernel_ms * 1e-3) / 1e9
    k_tflops = flops / (kernel_ms * 1e-3) / 1e12
    src = "MEASURED_PEAKS.json" if peak_src == "measured" else "the profiling recipe's fallback"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": k_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": k_gbs / peaks["hbm_gbs"], "peak_source": f"{peak_src}: hbm_gbs of {src}"}
    else:
        roof = {"bound": "tensor", "achieved": k_tflops, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": k_tflops / tc_peak,
                "peak_source": (f"{peak_src}: 2 x bf16_tflops of {src} (burst); e4m3 is not measured on its own, "
                                "2x is the nominal e4m3/bf16 dense ratio (4.5 / 2.25 PFLOP/s)") if e4m3 else
                               f"{peak_src}: bf16_tflops of {src} (burst)"}
    roof.update({"traffic": measured_traffic(name), "kernel": "split_kv_tc (the split-KV kernel of mla_decode)",
                 "kernel_us": kernel_ms * 1e3, "t_roofline_us": 1e6 * t_roof,
                 # the whole call (split-KV kernel and reduction) against the same roofline
                 "frac_call": (1e6 * t_roof) / (ms * 1e3)})
    rec = {"workload": describe(prob), "us_per_call": ms * 1e3, "kernel_us": kernel_ms * 1e3,
           "tflops": world * flops / (ms * 1e-3) / 1e12, "kv_gbs": world * kv / (ms * 1e-3) / 1e9,
           "flops_per_step": flops, "kv_bytes_per_step": kv, "dtype": prob.w.dtype, "roofline": roof,
           "clocks": clk.summary(),
           "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "mode": e2e_mode,
                   "serial": {"value": world * flops / (e2e_serial_ms * 1e-3) / 1e12, "ms_per_step": e2e_serial_ms}},
           "no_flush": {"us_per_call": nf_ms * 1e3, "l2": "not flushed between calls"},
           "gpu_launches": launches_per_call * args.steps, "ms": ms}
    del d, dec, flush, out, lse, hq, dq
    torch.cuda.empty_cache()
    return prob, rec


def run_ours(args, world, rank, local_rank):
    torch.cuda.set_device(local_rank)
    nbuild.build()
    _native.load()
    peaks, peak_src = load_peaks()
    names = ALL if args.workload == "all" else [args.workload]
    head = HEADLINE if HEADLINE in names else names[0]
    records, probs = {}, {}
    for name in names:
        probs[name], records[name] = measure(name, args, world, rank, local_rank, peaks, peak_src)
    if rank != 0:
        return
    h = records[head]
    cb = cb1 = None
    if args.cpu_budget > 0:
        cb = cpu_baseline(probs[head], budget_s=args.cpu_budget)
        cb1 = cpu_baseline(probs[head], budget_s=max(1.0, args.cpu_budget / 3), threads=1)
    line = {
        "metric": METRIC,
        "value": h["tflops"],
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": h["ms"],
        "us_per_call": h["us_per_call"],
        "kv_gbs": h["kv_gbs"],
        "tflops": h["tflops"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": h["dtype"],
        "data": "synthetic",
        "config": {"workload": h["workload"], "l2": "flushed before every timed step (256 MB device write)",
                   "parallelism": f"{world} independent batches (one per GPU)", "flops_per_step": h["flops_per_step"],
                   "kv_bytes_per_step": h["kv_bytes_per_step"]},
        "roofline": h["roofline"],
        "clocks": h["clocks"],
        "e2e": h["e2e"],
        "no_flush": h["no_flush"],
        "gpu_launches": h["gpu_launches"],
        "cpu_baseline": ({k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")} if cb else None),
        "cpu_baseline_1core": ({k: cb1[k] for k in ("value", "unit", "cores", "kind", "sample")} if cb1 else None),
        "workloads": {n: {k: v for k, v in r.items() if k != "ms"} for n, r in records.items()},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="all", choices=["all"] + list(wl.WORKLOADS),
                    help="all (default): the uniform headline plus records for varlen, fp8spec and window")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline (0: skip)")
    ap.add_argument("--fp32-partials", action="store_true", help="fp32 split partials (default: fp16, scaled)")
    ap.add_argument("--num-clusters", type=int, default=0, help="CTA pairs of the split-KV launch (0: the planner's)")
    ap.add_argument("--page-size", type=int, default=0, help="keys per KV page (0: the workload's, 64)")
    ap.add_argument("--reducer-d-tiles", type=int, default=0, help="reduction CTAs per work row across the dims (0: 8)")
    ap.add_argument("--no-pdl", action="store_true", help="launch the reduction without programmatic dependent launch")
    ap.add_argument("--combine-in-kernel", action="store_true",
                    help="combine split rows inside the split-KV kernel instead of in the reduction kernel")
    ap.add_argument("--compact-pool", action="store_true",
                    help="allocate only the pages the batch uses (for profiling captures; same tiles and traffic)")
    ap.add_argument("--ref-budget", type=float, default=6.0, help="seconds of oracle work per reference-arm step")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, world, rank, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
