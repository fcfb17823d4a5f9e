"""Benchmark: one mixed chunked-prefill + decode step (paged KV append + fused
attention forward + split combine) on synthetic inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints ONE JSON line (rank 0).  ``value`` is query tokens per second over the
timed steps (all ranks), ``ms_per_step`` the device time of one step.  The
default workload is the long-context step, the largest that fits one GPU: one
2048-token chunk after 126976 history tokens plus 64 decodes over contexts
U[65536, 131072], 32 q / 8 kv heads, head_dim 128, 16-token pages (~26 GB of
KV read per step).
``--impl reference`` times the CPU oracle on a bounded sample instead.
Under torchrun every rank runs an independent replica (the step does not
shard); timing is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "mixed prefill+decode paged-attn step µs, tokens/s, % of HBM/TC roofline"
UNIT = "query tokens/s"
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# algorithmic work of one step (what the method must move / compute)
# ---------------------------------------------------------------------------

def algorithmic(w, rows=None):
    """Bytes and tensor FLOPs of one step, per the roofline definition: every
    KV position read once per kv head (K and V), Q read and O written once;
    the append reads and writes the new rows; tensor FLOPs are the visible
    (query, key) pairs of the chunk segments x 2 matmuls x 2 flops x D x H_q.
    With ``rows`` (token indices) only those query rows are computed: the KV a
    listed token sees, read once per kv head, and its Q / O rows."""
    D, Hq, Hkv = w.head_dim, w.num_q_heads, w.num_kv_heads
    if rows is not None:
        cu = np.concatenate([[0], np.cumsum(w.q_lens)])
        seg = np.searchsorted(cu, rows, side="right") - 1
        vis = {}
        for t, s in zip(rows, seg):  # a segment's KV is read up to its last listed token
            vis[s] = max(vis.get(s, 0), w.k_lens[s] - w.q_lens[s] + int(t - cu[s]) + 1)
        kv_bytes = sum(vis.values()) * Hkv * D * 2 * 2
        qo = len(rows) * Hq * D * 2
        append_bytes = w.total_q * Hkv * D * 2 * 2 * 2
        return dict(kv_bytes=kv_bytes, q_bytes=qo, o_bytes=qo, append_bytes=append_bytes,
                    fwd_bytes=kv_bytes + 2 * qo, flops_tc=0, flops_dec=0)
    kv_bytes = sum(w.k_lens[s] for s in range(w.num_seqs) if w.q_lens[s] > 0) * Hkv * D * 2 * 2
    q_bytes = w.total_q * Hq * D * 2
    o_bytes = w.total_q * Hq * D * 2
    append_bytes = w.total_q * Hkv * D * 2 * 2 * 2
    G = Hq // Hkv
    flops_tc = 0
    flops_dec = 0
    for lq, lk in zip(w.q_lens, w.k_lens):
        pairs = lq * (lk - lq) + lq * (lq + 1) // 2
        if lq * G > 16:
            flops_tc += 4 * D * Hq * pairs
        else:
            flops_dec += 4 * D * Hq * pairs
    return dict(kv_bytes=kv_bytes, q_bytes=q_bytes, o_bytes=o_bytes, append_bytes=append_bytes,
                fwd_bytes=kv_bytes + q_bytes + o_bytes, flops_tc=flops_tc, flops_dec=flops_dec)


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of ``x`` over the ranks (the job is as slow as its
    slowest replica); ``device``: where the collective's tensor lives (the
    GPU under NCCL, the CPU under gloo)."""
    if world <= 1:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput of ``world`` replicas that each processed
    ``units_per_rank`` units, timed by the slowest one."""
    return world * units_per_rank / seconds


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return dict(hbm=float(m["hbm_gbs"]), bf16=float(m["bf16_tflops"]),
                    bf16_sustained=float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("attn_fwd.cu", "ptx.cuh", "mcp_internal.h"):
        with open(os.path.join(ROOT, "mixed_chunked_prefill_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch of the fused kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"mixed_attn_fwd_kernel.{workload}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_sha():
        return None
    return float(m.group(1))


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples every 20 ms from start() to stop(); the summary is
    taken over the samples whose timestamps fall between mark_begin() and
    mark_end() (the timed region), or over all samples, labelled, when the
    region was too short to catch one."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None
        self.t_begin = self.t_end = None

    def start(self):
        try:
            self.out = open("/tmp/_mcp_clocks_%d.csv" % os.getpid(), "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark_begin(self):
        self.t_begin = time.time()

    def mark_end(self):
        self.t_end = time.time()

    @staticmethod
    def parse(lines):
        """(epoch seconds or None, sm MHz, max MHz, [reason names]) per CSV line."""
        import datetime

        out = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            try:
                sm, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            reasons = [ClockSampler.REASONS[i] for i in range(4)
                       if parts[6 + i].lower() == "active"]
            out.append((ts, sm, mx, reasons))
        return out

    def summary(self, samples):
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [x for x in samples if x[0] is not None and self.t_begin is not None
                  and self.t_end is not None and self.t_begin <= x[0] <= self.t_end]
        use = inside or samples
        return {"sm_mhz": statistics.median(x[1] for x in use),
                "sm_max_mhz": max(x[2] for x in samples),
                "reasons": sorted({r for x in use for r in x[3]}),
                "samples": len(samples), "samples_in_region": len(inside),
                "window": "timed region" if inside else
                          "whole run (the timed region was shorter than the 20 ms sampling)"}

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        with open(self.out.name) as f:
            lines = f.readlines()
        os.unlink(self.out.name)
        return self.summary(self.parse(lines))


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, rank, world, local_rank):
    import torch

    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300 import build as mcp_build
    from mixed_chunked_prefill_gb300.step import HostStep, MixedStep, write_history

    if rank == 0 or not os.path.exists(mcp_build.LIB_PATH):
        mcp_build.build()
    if world > 1:
        torch.distributed.barrier()
    mcp.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    w = synth.make_workload(args.config, head_dim=args.head_dim, page_size=args.page_size)
    cu0 = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
    rows = mcp.build_logits_indices(cu0) if args.rows == "logits" else None
    alg = algorithmic(w, rows)
    peaks = load_peaks()

    with torch.cuda.stream(stream):
        t = w.tensors(dev)
        shape = (w.num_pages, w.page_size, w.num_kv_heads, w.head_dim)
        k_cache = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        v_cache = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        bt = w.block_tables()
        write_history(bt, w.hist_lens, t["k_hist"], t["v_hist"], k_cache, v_cache, w.page_size,
                      stream=stream)
        del t["k_hist"], t["v_hist"]
        cu = np.concatenate([[0], np.cumsum(w.q_lens)]).astype(np.int32)
        step = MixedStep(w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size, w.num_pages,
                         w.sm_scale, cu, w.k_lens, bt, device=dev, stream=stream, rows=rows)
        # host planning of one step (the work the host step repeats per step):
        # median of 20 plans from host metadata, no upload
        plan_times = []
        for _ in range(20):
            t0 = time.perf_counter()
            if rows is None:
                mcp.mixed_attn_plan(step.desc, cu, w.k_lens, step.options)
            else:
                mcp.mixed_attn_plan_rows(step.desc, cu, w.k_lens, rows, step.options)
            plan_times.append((time.perf_counter() - t0) * 1e6)
        plan_us = statistics.median(plan_times)
        q, k_new, v_new = t["q"], t["k_new"], t["v_new"]
        out = torch.empty_like(q)
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream.synchronize()

    def one_step():
        step.run(q, k_new, v_new, k_cache, v_cache, out)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            one_step()
    step.check()

    # timed region: K steps, L2 flushed (untimed) between steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    fwd_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    clocks.mark_begin()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.fill_(float(i))
            evs[i][0].record(stream)
            step.append(k_new, v_new, k_cache, v_cache)
            fwd_evs[i][0].record(stream)
            step.attention(q, k_cache, v_cache, out)
            fwd_evs[i][1].record(stream)
            evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark_end()
    clk = clocks.stop()
    step.check()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    fwd_ms = [a.elapsed_time(b) for a, b in fwd_evs]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    tokens_per_s = job_rate(w.total_q * args.steps, world, total_ms / 1e3)

    # end to end through the C ABI from pinned host buffers
    e2e = None
    if args.e2e_steps > 0 and rows is None:
        q_h = q.cpu().pin_memory()
        k_h = k_new.cpu().pin_memory()
        v_h = v_new.cpu().pin_memory()
        # two output buffers: consecutive steps are in flight together
        outs_h = [torch.empty_like(q_h).pin_memory() for _ in range(2)]
        # the arenas hold this step's plan: its split partials and work lists
        hs = HostStep(w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size, w.num_pages,
                      w.sm_scale, w.total_q, w.num_seqs, w.max_pages_per_seq, device=dev,
                      stream=stream, workspace_bytes=max(64 << 20, int(step.plan.workspace_bytes)),
                      list_bytes=max(4 << 20, int(step.plan.off_part_o)))
        for i in range(3):
            hs(q_h, k_h, v_h, cu, w.k_lens, bt, k_cache, v_cache, outs_h[i & 1])
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        ticket = -1
        for i in range(args.e2e_steps):
            ticket = hs.run(q_h, k_h, v_h, cu, w.k_lens, bt, k_cache, v_cache, outs_h[i & 1])
        hs.wait(ticket)  # the last step's output is in host memory (and every earlier one)
        e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
        hs.close()
        e2e = {"value": job_rate(w.total_q * args.e2e_steps, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": int(hs.h2d_bytes), "d2h_bytes_per_step": int(hs.d2h_bytes),
               "ms_per_step": 1e3 * e2e_s / args.e2e_steps, "steps": args.e2e_steps}

    # roofline of the dominant kernel (the fused forward; its call also runs
    # the split combine when the plan has splits)
    fwd_avg_s = statistics.mean(fwd_ms) / 1e3
    t_tc = alg["flops_tc"] / (peaks["bf16"] * 1e12)
    t_hbm = alg["fwd_bytes"] / (peaks["hbm"] * 1e9)
    if t_tc >= t_hbm:
        achieved = alg["flops_tc"] / fwd_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16"]}
    else:
        achieved = alg["fwd_bytes"] / fwd_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": achieved / peaks["hbm"]}
    # the committed captures are of the named workloads at their own shapes
    overridden = args.head_dim is not None or args.page_size is not None
    roof["traffic"] = None if overridden else profiled_traffic(args.config)
    roof["peak_source"] = f"{peaks['source']} ({'burst bf16' if roof['bound'] == 'tensor' else 'copy'})"
    roof["kernel_ms"] = statistics.mean(fwd_ms)
    step_roof_s = max(t_tc, (alg["fwd_bytes"] + alg["append_bytes"]) / (peaks["hbm"] * 1e9))
    launches_per_step = 2 + (1 if step.plan.num_combine > 0 else 0)
    res = {
        "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, random page permutation)",
        "config": {"workload": synth.describe(args.config, args.head_dim, args.page_size),
                   "name": args.config, "segments": w.num_seqs, "total_q": w.total_q,
                   "kv_tokens": int(sum(w.k_lens)), "l2": "flushed between steps (256 MB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "step": "paged_kv_append + mixed_attn_fwd (+ combine)",
                   "rows": ("all" if rows is None else
                            f"logits_indices only ({len(rows)} of {w.total_q} query rows)"),
                   "work_items": int(step.plan.num_items),
                   "decode_items": int(step.plan.num_decode_items),
                   "prefill_items": int(step.plan.num_prefill_items),
                   "combine_groups": int(step.plan.num_combine)},
        "step_us": ms_per_step * 1e3,
        "step_us_p10_p90": [float(np.percentile(step_ms, 10) * 1e3),
                            float(np.percentile(step_ms, 90) * 1e3)],
        "kv_gbps": alg["kv_bytes"] / (ms_per_step / 1e3) / 1e9,
        "step_roofline_frac": step_roof_s / (ms_per_step / 1e3),
        "step_roofline_us": step_roof_s * 1e6,
        "plan_host_us": plan_us,
        "roofline": roof,
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
    }
    if step_roof_s < 2e-6:
        # a step whose bytes and FLOPs take under 2 us at the peaks is bound by launch
        # latency and per-item set-up, not by HBM or the tensor cores
        res["launch_bound"] = (f"roofline time {step_roof_s * 1e6:.2f} us: the step is bound by "
                               "launch latency and per-item set-up; reported, no % target")
    return res


# ---------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def blas_threads():
    """Threads of the BLAS NumPy's matmul runs on (threadpoolctl), else the
    thread count the usual environment variables set, else None."""
    try:
        import threadpoolctl

        info = [i for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas"]
        if info:
            return int(max(i.get("num_threads", 1) for i in info))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return None


def oracle_cores():
    """Host threads the oracle uses: its BLAS thread count, else the affinity size."""
    n = blas_threads()
    if n:
        return n
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def host_details():
    """What the oracle's timing ran on: core counts, architecture, BLAS threads."""
    return {"os_cpu_count": os.cpu_count(),
            "affinity": (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                         else None),
            "machine": os.uname().machine,
            "blas_threads": blas_threads() or "not reported (no threadpoolctl; OpenBLAS "
                                              "defaults to every core of the affinity set)",
            "threading": "multi-thread: NumPy's BLAS on all its threads for the matmuls; "
                         "masking, exp and the page gather single-threaded; no "
                         "single-thread run was timed"}


def sample_segments(w):
    """The segments the CPU legs time on a big workload: the shortest and the
    longest decode plus every chunk segment."""
    dec = [s for s in range(w.num_seqs) if w.q_lens[s] == 1]
    chunk = [s for s in range(w.num_seqs) if w.q_lens[s] > 1]
    return [min(dec, key=lambda s: w.k_lens[s]), max(dec, key=lambda s: w.k_lens[s])] + chunk


class OracleSample:
    """The oracle on one workload's inputs, restricted to a row sample.

    The two big workloads (tens of GB of KV history) are sampled by segment:
    the shortest and the longest decode plus the chunk, as a workload of
    their own whose values are drawn for those segments alone (same lengths,
    heads, page size and value distribution), so the host never holds the
    whole history."""

    def __init__(self, name, head_dim=None, page_size=None):
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from harness import OracleStep

        w = synth.make_workload(name, head_dim=head_dim, page_size=page_size)
        self.w = w
        if name in ("decode-heavy", "long-context"):
            segs = sample_segments(w)
            w = synth.make_workload_from_lengths(
                w.name + "-sample", w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size,
                w.sm_scale, [w.q_lens[s] for s in segs], [w.k_lens[s] for s in segs], w.seed)
            self.w = w
            self.note = ("the shortest and the longest decode + the chunk segment of the "
                         "workload, values drawn for those segments alone")
        else:
            self.note = "all segments"
        self.step = OracleStep(w, w.tensors("cpu"))
        self.step.do_append()

    def rows(self, n):
        """n query tokens spread over the whole stream (decodes first)."""
        T = self.w.total_q
        n = max(1, min(n, T))
        return sorted(set(np.linspace(0, T - 1, n).round().astype(int).tolist()))

    def time_rows(self, rows):
        t0 = time.perf_counter()
        self.step.attention(tokens=rows)
        return time.perf_counter() - t0


def run_kv_swap(args):
    """Swap-out / swap-in rate of KV pages between the device pool and a
    page-locked host pool (mcp_kv_copy_pages), against a contiguous
    page-locked cudaMemcpyAsync of the same bytes (the host link's practical
    peak on this machine)."""
    import torch

    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300 import build as mcp_build

    mcp_build.build()
    mcp.load()
    dev = torch.device("cuda", 0)
    P, Hkv, D = 16, 8, 128
    pool, n = 16384, 8192                       # 1 GB device pool; 512 MB (K+V) moved
    page_bytes = 2 * P * Hkv * D * 2            # K and V of one page
    kc = torch.zeros((pool, P, Hkv, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    hk = torch.zeros((n, P, Hkv, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    rng = np.random.Generator(np.random.PCG64(11))
    dev_pages = torch.from_numpy(rng.permutation(pool)[:n].astype(np.int32)).to(dev)
    host_slots = torch.arange(n, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn, reps=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps / 1e3

    t_out = timed(lambda: mcp.kv_copy_pages(kc, vc, hk, hv, dev_pages, host_slots))
    t_in = timed(lambda: mcp.kv_copy_pages(hk, hv, kc, vc, host_slots, dev_pages))
    flat_d = kc[:n].view(-1)
    flat_h = hk.view(-1)
    t_d2h = timed(lambda: (flat_h.copy_(flat_d, non_blocking=True),
                           hv.view(-1).copy_(vc[:n].view(-1), non_blocking=True)))
    t_h2d = timed(lambda: (flat_d.copy_(flat_h, non_blocking=True),
                           vc[:n].view(-1).copy_(hv.view(-1), non_blocking=True)))
    moved = n * page_bytes
    gbs = lambda t: moved / t / 1e9
    return {"metric": "KV page swap-out / swap-in (mcp_kv_copy_pages)", "value": gbs(t_in),
            "unit": "GB/s", "n_gpus": 1, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic (zero-filled pools, random page permutation)",
            "config": {"workload": f"{n} random pages of {page_bytes // 1024} KB (K+V, 16 tokens "
                                   f"x {Hkv} kv heads x {D}) between a {pool}-page device pool "
                                   "and a page-locked host pool", "pages": n},
            "swap_out_gbs": gbs(t_out), "swap_in_gbs": gbs(t_in),
            "contiguous_memcpy_d2h_gbs": gbs(t_d2h), "contiguous_memcpy_h2d_gbs": gbs(t_h2d),
            "frac_of_memcpy": {"out": t_d2h / t_out, "in": t_h2d / t_in}}


def run_serve(args):
    """Step-time distribution of a serving loop with and without chunked
    prefill ([W] "Token 预算", [X] "Chunked Prefill 的核心算法思想"): 32 requests
    decoding over 4096-token contexts while 8192-token prompts arrive every 50
    steps; each step (schedule, copy-in, append + attention, copy-out) is
    timed by wall clock after its outputs reach host memory."""
    import torch

    import mixed_chunked_prefill_gb300 as mcp
    from mixed_chunked_prefill_gb300 import build as mcp_build
    from mixed_chunked_prefill_gb300.serve import ServeLoop

    mcp_build.build()
    mcp.load()
    Hq, Hkv, D = 32, 8, 128
    n_dec, ctx, long_prompt, every, steps = 32, 4096, 8192, 50, 200
    new_tokens = 1000  # outlasts the untimed warm-up (prompts of the decodes) + timed steps
    pages = (n_dec * (ctx + new_tokens + 16) + 8 * (long_prompt + 16)) // 16 + 64
    mp = (max(long_prompt, ctx + new_tokens) + 16) // 16 + 1
    gen = torch.Generator().manual_seed(5)
    cap = long_prompt + n_dec + 64
    qb = torch.randn((cap, Hq, D), generator=gen).to(torch.bfloat16).pin_memory()
    kb = torch.randn((cap, Hkv, D), generator=gen).to(torch.bfloat16).pin_memory()
    vb = torch.randn((cap, Hkv, D), generator=gen).to(torch.bfloat16).pin_memory()

    def token_fn(plan):
        T = plan.total_q
        return qb[:T], kb[:T], vb[:T]

    out = {}
    for label, budget in (("chunked_512", 512), ("unchunked", long_prompt + n_dec)):
        loop = ServeLoop(Hq, Hkv, D, pages, 1.0 / math.sqrt(D), max_num_batched_tokens=budget,
                         max_pages_per_seq=mp, max_num_seqs=64)
        for r in range(n_dec):
            loop.add_request(r, ctx, new_tokens)
        # bring every decode request past its prompt (untimed)
        for _ in range(10 ** 4):
            res = loop.step(token_fn)
            loop.wait(res)
            if (res.plan.q_lens == 1).sum() == n_dec:
                break
        times, tokens, arrivals = [], 0, 0
        t_all = time.perf_counter()
        for i in range(steps):
            if i % every == 0:
                loop.add_request(1000 + arrivals, long_prompt, 1)
                arrivals += 1
            t0 = time.perf_counter()
            res = loop.step(token_fn)
            loop.wait(res)
            times.append(time.perf_counter() - t0)
            tokens += res.plan.total_q
        t_all = time.perf_counter() - t_all
        ms = np.array(times) * 1e3
        out[label] = {"budget": budget, "step_ms_p50": float(np.percentile(ms, 50)),
                      "step_ms_p99": float(np.percentile(ms, 99)), "step_ms_max": float(ms.max()),
                      "step_ms_mean": float(ms.mean()), "tokens_per_s": tokens / t_all,
                      "prompts": arrivals}
        loop.close()
    c = out["chunked_512"]
    return {"metric": "serving step time seen by decoding requests (p99)", "value": c["step_ms_p99"],
            "unit": "ms", "n_gpus": 1, "higher_is_better": False, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": f"{n_dec} requests decoding over {ctx}-token contexts; an "
                                   f"{long_prompt}-token prompt arrives every {every} steps; "
                                   f"{steps} timed steps; 32 q / 8 kv heads, head_dim 128",
                       "step": "schedule + copy-in + append + attention + copy-out, waited"},
            "chunked": out["chunked_512"], "unchunked": out["unchunked"]}


def cpu_baseline(name, budget_s=15.0, head_dim=None, page_size=None):
    s = OracleSample(name, head_dim, page_size)
    rows = s.rows(4)
    dt = s.time_rows(rows)
    n = len(rows)
    # the per-segment K/V gather is a fixed cost, so grow the row sample until
    # the timed call reaches about half the budget (or covers every row)
    while dt < budget_s / 2 and n < s.w.total_q:
        n = min(s.w.total_q, n * 4)
        rows = s.rows(n)
        dt = s.time_rows(rows)
    return {"value": len(rows) / dt, "unit": UNIT, "cores": oracle_cores(), "kind": "oracle",
            "sample": f"{len(rows)} of {s.w.total_q} query tokens (all heads), {s.note}; "
                      f"{dt:.1f} s", "seconds": dt, "host": host_details()}


def run_reference(args):
    s = OracleSample(args.config, args.head_dim, args.page_size)
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    rows = s.rows(2)
    dt = s.time_rows(rows)
    n = len(rows)
    while dt < per_step / 4 and n < s.w.total_q:
        n = min(s.w.total_q, n * 2)
        rows = s.rows(n)
        dt = s.time_rows(rows)
    for _ in range(args.warmup):
        s.time_rows(rows)
    times = [s.time_rows(rows) for _ in range(args.steps)]
    total = sum(times)
    value = len(rows) * args.steps / total
    sample = (f"{len(rows)} of {s.w.total_q} query tokens (all heads) per step, {s.note}")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, random page permutation)",
            "config": {"workload": synth.describe(args.config, args.head_dim, args.page_size),
                       "name": args.config},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_cores(),
                             "kind": "oracle", "sample": sample, "host": host_details()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="long-context", choices=synth.CONFIG_NAMES + synth.PROFILE_NAMES)
    ap.add_argument("--head-dim", type=int, default=None, choices=[64, 96, 128, 256],
                    help="run the workload's segments at this head_dim")
    ap.add_argument("--page-size", type=int, default=None, choices=[1, 8, 16, 32, 64],
                    help="run the workload's segments with this page size")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--serve", action="store_true",
                    help="serving-loop step times with and without chunked prefill")
    ap.add_argument("--kv-swap", action="store_true",
                    help="time KV page swap-out / swap-in instead of the step")
    ap.add_argument("--rows", default="all", choices=["all", "logits"],
                    help="logits: attention only for logits_indices (the last layer's rows)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.kv_swap:
        if rank == 0:
            print(json.dumps(run_kv_swap(args)), flush=True)
        return
    if args.serve:
        if rank == 0:
            print(json.dumps(run_serve(args)), flush=True)
        return

    if world > 1:
        import torch

        torch.cuda.set_device(local_rank)
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1 and args.rows == "all":
            res["cpu_baseline"] = cpu_baseline(args.config, head_dim=args.head_dim,
                                               page_size=args.page_size)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch

        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
