"""Benchmark of batched row-wise TopK on B300: effective HBM GB/s and rows/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c4] [--impl ours|reference]

A step is one ds_topk call over one batch of the workload (the whole hot path:
load, NaN check, threshold, radix select, ordered output write). The timed
region holds exactly K steps replayed from CUDA graphs that were each replayed
once before it, bracketed by a barrier and a device synchronize. Every step
reads its input from HBM: the decode-shaped indexer batch (1.07 GB) is larger
than L2, and smaller workloads rotate over resident copies that together exceed
four times L2. Rank 0 prints one JSON line. Under torchrun every rank runs the
same workload on its own GPU (rows are independent: no collective on the data
path), and the value is the bytes of all ranks over the slowest rank's time.

The line's headline is the decode-shaped bf16 indexer call (16384 rows of 32768,
k=512), the largest single-GPU workload. The other workloads (fp32 sampler,
bf16 indexer prefill, adversarial rows, the small fp32 case) ride along in the
same line under "per_workload", each timed over at least --min-ms of device
work, with its own roofline fraction and CPU-oracle baseline. Each workload that
fits in L2 also gets an "l2_hot" figure (every step on one input copy; labelled,
never the headline), and each a "torch_topk" figure: torch.topk on the same
input, as context for the speed-ups the method's pages quote, not as a baseline.

The metric is the pages' own: effective memory bandwidth, (input bytes read +
output bytes written) / time, because TopK does no floating-point math
(github-research.aiutil.com, "deepseek-ai/DeepSelect", section 关键技术亮点).
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "effective HBM GB/s and rows/s for batched TopK (bf16 indexer, fp32 sampler)"
DEFAULT_WORKLOAD = "c4"
EXTRA_WORKLOADS = ("c2", "c5", "c3", "c1")
L2_BYTES_FALLBACK = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6400.0
TRAFFIC_FILE = os.path.join("profiles", "traffic.json")
CSRC = os.path.join("sampler_topk_selection_ds_b300", "csrc")
# The sources each selection kernel is built from: its own header, the shared
# device helpers, the host file that plans and launches it, and the C header.
_COMMON_SOURCES = [os.path.join(CSRC, "topk_kernel.cuh"), os.path.join(CSRC, "ds_topk.cu"),
                   os.path.join("include", "ds_topk.h")]
KERNEL_SOURCES = {
    "topk_rows_kernel": _COMMON_SOURCES,
    "topk_warp_rows_kernel": _COMMON_SOURCES + [os.path.join(CSRC, "warp_rows_kernel.cuh")],
}

SAMPLE_TEMPERATURE = 1.0
SAMPLE_TOP_P = 0.9


def kernel_name(w, plan) -> str:
    es = 2 if w.dtype == torch.bfloat16 else 4
    if plan.path == 2:
        return f"topk_warp_rows_kernel<{es}>"
    return f"topk_rows_kernel<{es},{plan.cluster_size}>"


def value_order_by_warp(w, sm_count) -> bool:
    """Whether the library sorts this workload's value order one row per warp (many
    bf16 rows of at most 65536 elements, k <= 1024, at least 8 rows per SM) rather
    than one CTA per row: the rule the library's launcher applies."""
    return (w.dtype == torch.bfloat16 and w.length <= 65536 and w.k <= 1024 and
            w.batch >= 8 * sm_count)


def shifted(x, shift):
    """x (contiguous) copied into a new device buffer `shift` elements past its
    16-byte aligned start: with shift * sizeof(dtype) not a multiple of 16, no row
    starts on a 16-byte boundary."""
    if not shift:
        return x
    buf = torch.empty(x.numel() + shift + 16, dtype=x.dtype, device=x.device)
    view = buf[shift:shift + x.numel()].view(x.shape)
    view.copy_(x)
    return view


def plan_for(dstk, w, sm_count, shift):
    """The launch plan ds_topk takes for the workload's rows at this shift (the
    plan call assumes a 16-byte aligned x, so a shift that breaks 16-byte
    alignment is stood for by a row stride that is not a multiple of 16 bytes:
    both put rows off 16-byte boundaries)."""
    stride = w.length
    if (shift * w.elem_size) % 16:
        stride = w.length + 1
        while (stride * w.elem_size) % 16 == 0:
            stride += 1
    return dstk.ds_topk_plan(dstk.dtype_code(w.dtype), w.batch, w.length, stride, w.k, sm_count)


def code_only(src: str) -> str:
    """C/C++/CUDA source without its comments and with whitespace runs collapsed,
    so that edits to comments or layout leave a kernel's hash unchanged. String
    and character literals are kept as written."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            out.append(" ")
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_hash(kernel: str) -> str:
    """Hash of the code (comments aside) of the sources the named kernel (e.g.
    "topk_warp_rows_kernel<2>") is built from."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel.split("<")[0]]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of the dominant kernel on this
    workload, from the ncu figures recorded in the traffic data file
    (profiles/traffic.json: workload -> kernel, kernel_hash,
    dram_bytes_per_launch, summary), if they were taken on the current kernel
    code; else None with the reason."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_FILE), encoding="utf-8") as fh:
            table = json.load(fh)
    except (OSError, ValueError):
        return None, "no traffic data file"
    entry = table.get(workload)
    if not entry:
        return None, f"no ncu traffic recorded for {workload}"
    if entry.get("kernel") != kernel:
        return None, f"recorded traffic is for {entry.get('kernel')}, not {kernel}"
    if entry.get("kernel_hash") != kernel_hash(kernel):
        return None, f"stale: recorded on kernel code {entry.get('kernel_hash')}"
    return int(entry["dram_bytes_per_launch"]), f"ncu capture summarised in {entry.get('summary')}"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.out or "")) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        busy = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def _dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def _barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(bytes_per_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job effective GB/s: bytes moved by all ranks over the slowest rank's time."""
    return bytes_per_step * steps * world / max_seconds / 1e9


def sample_rows(w: workloads.Workload, max_rows: int):
    """A bounded, evenly spread sample of the workload's rows (all of them if few)."""
    if w.batch <= max_rows:
        return list(range(w.batch))
    step = w.batch / max_rows
    return [int(i * step) for i in range(max_rows)]


def _oracle_gbs(w, x, nthreads, min_seconds, repeats):
    """`repeats` timings of the oracle on the sample x, each the median call time
    over calls that together take about min_seconds / repeats."""
    import oracle
    sub = w.scaled(x.shape[0])
    per = []
    for _ in range(repeats):
        t, _n = oracle.time_topk(x, w.k, return_value=w.return_value, nthreads=nthreads,
                                 min_seconds=min_seconds / repeats)
        per.append(t)
    gbs = sorted((sub.bytes_in + sub.bytes_out) / t / 1e9 for t in per)
    return {"value": round(statistics.median(gbs), 4), "spread": [round(gbs[0], 4), round(gbs[-1], 4)],
            "repeats": repeats, "ms_per_call": round(statistics.median(per) * 1e3, 3)}


def cpu_baseline(w: workloads.Workload, min_seconds: float, max_rows: int = 256, repeats: int = 3):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload (evenly spread whole rows): all cores (the reported value) and one
    thread, each timed `repeats` times with the spread of those repeats."""
    import oracle
    cores = oracle.cores()
    rows = sample_rows(w, max_rows)
    x = workloads.generate_rows(w, rows)
    oracle.topk(x, w.k, return_value=w.return_value)  # warm
    allc = _oracle_gbs(w, x, 0, min_seconds, repeats)
    # one thread on at most 32 of the sampled rows
    x1 = x[: min(32, x.shape[0])].contiguous()
    one = _oracle_gbs(w, x1, 1, min_seconds, repeats)
    return {"value": allc["value"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} of {w.batch} rows of {w.name} (evenly spread), all {cores} host "
                      f"threads, {repeats} timed repeats ({allc['ms_per_call']} ms per call); one "
                      f"thread on the first {x1.shape[0]} of them",
            "spread": allc["spread"], "repeats": repeats,
            "single_thread": {"value": one["value"], "unit": "GB/s", "cores": 1, "spread": one["spread"],
                              "repeats": repeats, "rows": x1.shape[0]},
            "rows_per_s": round(len(rows) / (allc["ms_per_call"] / 1e3), 2)}


def run_reference(args, w):
    """The reference arm: the CPU oracle on the host cores. Each step is one
    oracle call on a bounded sample of the workload's rows (all host threads);
    W untimed steps, then K timed ones. Only rank 0 runs it."""
    import oracle
    world, rank, _local = _dist_setup()
    if rank != 0:
        return 0
    rows = sample_rows(w, args.ref_rows)
    x = workloads.generate_rows(w, rows)
    sub = w.scaled(len(rows))
    for _ in range(max(1, args.warmup)):
        oracle.topk(x, w.k, return_value=w.return_value)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.topk(x, w.k, return_value=w.return_value)
    sec = time.perf_counter() - t0
    value = (sub.bytes_in + sub.bytes_out) * args.steps / sec / 1e9
    cores = oracle.cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w, None, args.shift),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {len(rows)} of {w.batch} rows of {w.name} (evenly "
                                   f"spread), all {cores} host threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "reference arm = the CPU oracle (plain sort per row), host cores only",
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(w, l2_note, shift=0):
    cfg = {"workload": f"{w.name}: {w.description}" + (f"; rows start {shift} element(s) past a 16-byte "
                                                        f"boundary" if shift else ""),
           "batch": w.batch, "len": w.length, "k": w.k,
           "input_dtype": "bf16" if w.dtype == torch.bfloat16 else "fp32",
           "sorted_index": w.sorted_index, "return_value": w.return_value,
           "seed": w.seed, "parallelism": "rows independent; one GPU per rank (weak scaling)"}
    if l2_note is not None:
        cfg["l2"] = l2_note
    return cfg


class Bench:
    """One workload resident on the device, its outputs, and the CUDA graphs that
    replay its steps. Steps rotate over `copies` resident inputs so that each
    reads a copy not touched for copies - 1 steps (copies = 1 when one input
    alone exceeds four times L2)."""

    def __init__(self, dstk, w, dev, stream, shift=0, order="workload"):
        self.dstk, self.w, self.dev, self.stream = dstk, w, dev, stream
        props = torch.cuda.get_device_properties(dev)
        l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK
        self.copies = 1 if w.bytes_in >= 4 * l2 else min(64, math.ceil(4 * l2 / w.bytes_in))
        x0 = shifted(workloads.generate(w, device=dev), shift)
        self.xs = [x0] + [shifted(x0.contiguous(), shift) for _ in range(self.copies - 1)]
        self.l2_note = (f"inputs larger than L2 ({w.bytes_in / 1e6:.0f} MB per step > {l2 / 1e6:.0f} MB)"
                        if self.copies == 1 else
                        f"rotating {self.copies} resident input copies ({self.copies * w.bytes_in / 1e6:.0f} MB "
                        f"> 4x L2 {l2 / 1e6:.0f} MB); each step reads a copy not touched for "
                        f"{self.copies - 1} steps")
        self.dt_code = dstk.dtype_code(w.dtype)
        self.sampling = order == "sample"
        self.idx = torch.empty((w.batch, w.k), dtype=torch.int32, device=dev)
        self.vals = (torch.empty((w.batch, w.k), dtype=w.dtype, device=dev)
                     if (w.return_value or self.sampling) else None)
        self.flag = torch.zeros(1, dtype=torch.int32, device=dev)
        if self.sampling:  # one fixed uniform number per row
            self.u = torch.rand(w.batch, generator=torch.Generator().manual_seed(w.seed)).to(dev)
            self.tokens = torch.empty(w.batch, dtype=torch.int32, device=dev)
        rc, self.plan = plan_for(dstk, w, props.multi_processor_count, shift)
        assert rc == dstk.OK, dstk.status_string(rc)
        self.kernel = kernel_name(w, self.plan)
        # kernel launches per step: value order adds a sort; the sampler tail adds a
        # draw only after the one-warp-per-row sort (the CTA sort draws itself)
        warp_sort = value_order_by_warp(w, props.multi_processor_count)
        self.launches = (self.plan.launches + (1 if int(w.sorted_index) == 2 else 0) +
                         (1 if self.sampling and warp_sort else 0))
        self.chunk = self.copies * max(1, math.ceil(64 / self.copies))
        self.graphs = {}

    def step(self, i, stream):
        d, w = self.dstk, self.w
        x = self.xs[i % self.copies]
        if self.sampling:
            r = d.ds_topk_sample(x.data_ptr(), self.dt_code, w.batch, w.length, w.length, w.k,
                                 SAMPLE_TEMPERATURE, SAMPLE_TOP_P, self.u.data_ptr(), self.vals.data_ptr(),
                                 self.idx.data_ptr(), self.tokens.data_ptr(), self.flag.data_ptr(),
                                 stream.cuda_stream)
        else:
            r = d.ds_topk(x.data_ptr(), self.dt_code, w.batch, w.length, w.length, w.k,
                          int(w.sorted_index), int(w.return_value),
                          self.vals.data_ptr() if (w.return_value and self.vals is not None) else None,
                          self.idx.data_ptr(), self.flag.data_ptr(), stream.cuda_stream)
        if r != d.OK:
            raise d.DsTopkError(r)

    def warm(self, n):
        with torch.cuda.stream(self.stream):
            for i in range(n):
                self.step(i, self.stream)
        self.stream.synchronize()

    def graph(self, n, hot=False):
        """A CUDA graph of n steps (starting at copy 0; every step on copy 0 if
        hot), replayed once before use so that no timed replay is a graph's first."""
        if (n, hot) not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    self.step(0 if hot else i, torch.cuda.current_stream())
            g.replay()
            self.stream.synchronize()
            self.graphs[(n, hot)] = g
        return self.graphs[(n, hot)]

    def _time_graph(self, g, replays):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        with torch.cuda.stream(self.stream):
            ev0.record(self.stream)
            for _ in range(replays):
                g.replay()
            ev1.record(self.stream)
        self.stream.synchronize()
        return ev0.elapsed_time(ev1) / 1e3

    def l2_hot(self, min_ms):
        """The same step with every call on one input copy, which stays in L2
        between calls: labelled L2-hot, beside the cold (rotating) figure. None
        when one input alone exceeds four times L2."""
        if self.copies == 1:
            return None
        n = self.chunk
        g = self.graph(n, hot=True)
        est = self._time_graph(g, 1) / n
        replays = max(3, math.ceil(min_ms / 1e3 / est / n))
        sec = self._time_graph(g, replays)
        steps = replays * n
        w = self.w
        return {"steps": steps, "ms_per_step": round(sec / steps * 1e3, 6),
                "value": round(aggregate_value(w.bytes_in + w.bytes_out, steps, 1, sec), 3), "unit": "GB/s",
                "note": "L2-hot: every step reads the same resident input copy (not the headline figure)"}

    def torch_topk_context(self, min_ms):
        """torch.topk(x, k, sorted=False) on the same resident input, warm, in the
        same units (this method's algorithmic bytes over its time): context for
        the speed-ups the method's pages quote, not a baseline of the method."""
        w, x = self.w, self.xs[0]
        if x.stride(1) != 1 or x.stride(0) != w.length:
            return None
        with torch.cuda.stream(self.stream):
            for _ in range(3):
                torch.topk(x, w.k, dim=1, largest=True, sorted=False)
            self.stream.synchronize()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(self.stream)
            torch.topk(x, w.k, dim=1, largest=True, sorted=False)
            ev1.record(self.stream)
            self.stream.synchronize()
            est = ev0.elapsed_time(ev1) / 1e3
            calls = max(3, min(2000, math.ceil(min_ms / 1e3 / est)))
            ev0.record(self.stream)
            for _ in range(calls):
                torch.topk(x, w.k, dim=1, largest=True, sorted=False)
            ev1.record(self.stream)
        self.stream.synchronize()
        sec = ev0.elapsed_time(ev1) / 1e3
        return {"calls": calls, "ms_per_call": round(sec / calls * 1e3, 6),
                "value": round(aggregate_value(w.bytes_in + w.bytes_out, calls, 1, sec), 3), "unit": "GB/s",
                "note": "context only: torch.topk(x, k, sorted=False), same input, warm (copy 0, "
                        "so L2-hot when it fits); a library kernel, not this method"}

    def replay(self, steps):
        """Enqueue exactly `steps` steps (whole chunks, then the remainder)."""
        full, rem = divmod(steps, self.chunk)
        g_full = self.graph(self.chunk) if full else None
        g_rem = self.graph(rem) if rem else None
        return lambda: ([g_full.replay() for _ in range(full)], g_rem.replay() if g_rem else None)

    def time_steps(self, steps, world=1, sampler=None):
        """Device seconds of exactly `steps` steps, bracketed by a barrier and a
        device synchronize on both sides (CUDA events on the launching stream)."""
        go = self.replay(steps)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        torch.cuda.synchronize(self.dev)
        with torch.cuda.stream(self.stream):
            ev0.record(self.stream)
            go()
            ev1.record(self.stream)
        self.stream.synchronize()
        torch.cuda.synchronize(self.dev)
        _barrier(world)
        return ev0.elapsed_time(ev1) / 1e3

    def per_step_estimate(self):
        return self.time_steps(self.chunk) / self.chunk

    def roofline(self, seconds, steps, name):
        w = self.w
        bytes_step = w.bytes_in + w.bytes_out
        # one step's bytes over one launch's share of the step time
        per_launch_s = seconds / (steps * self.plan.launches)
        achieved = bytes_step / self.plan.launches / per_launch_s / 1e9
        peak, peak_src = measured_peak()
        traffic, traffic_note = profiled_traffic(name, self.kernel)
        return {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "peak_source": peak_src + (" (of measured)" if peak_src != "fallback" else " (of fallback)"),
                "traffic": traffic, "traffic_note": traffic_note,
                "kernel": self.kernel, "kernel_hash": kernel_hash(self.kernel)}

    def free(self):
        self.graphs.clear()
        self.xs = None
        torch.cuda.synchronize(self.dev)
        torch.cuda.empty_cache()


def run_extra(dstk, w, dev, stream, args):
    """One more workload in the same line: timed over at least args.min_ms of
    device work (exact step count reported), with its roofline and oracle baseline."""
    b = Bench(dstk, w, dev, stream, 0, "workload")
    b.warm(max(3, args.warmup))
    est = b.per_step_estimate()
    steps = max(args.steps, min(200000, math.ceil(args.min_ms / 1e3 / est)))
    sec = b.time_steps(steps)
    out = {"workload": f"{w.name}: {w.description}", "steps": steps,
           "ms_per_step": round(sec / steps * 1e3, 6),
           "value": round(aggregate_value(w.bytes_in + w.bytes_out, steps, 1, sec), 3), "unit": "GB/s",
           "rows_per_s": round(w.batch * steps / sec, 1), "l2": b.l2_note,
           "roofline": b.roofline(sec, steps, w.name), "plan": b.plan.as_dict(),
           "gpu_launches": steps * b.launches}
    if not args.no_context:
        out["l2_hot"] = b.l2_hot(args.min_ms / 4)
        out["torch_topk"] = b.torch_topk_context(args.min_ms / 4)
    b.free()
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, min_seconds=args.cpu_seconds / 2)
    return out


def run_ours(args, w):
    import sampler_topk_selection_ds_b300 as dstk

    world, rank, local = _dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    stream = torch.cuda.Stream(dev)
    name = w.name + (f"+shift{args.shift}" if args.shift else "")

    b = Bench(dstk, w, dev, stream, args.shift, args.order)
    warmup = max(3, args.warmup)
    b.warm(warmup)
    b.replay(args.steps)  # capture and replay once every graph the timed region uses
    sampler = ClockSampler(local)
    with sampler:
        seconds = b.time_steps(args.steps, world)
    max_seconds = _max_over_ranks(seconds, world)
    clocks = sampler.summary()
    bytes_step = w.bytes_in + w.bytes_out
    value = aggregate_value(bytes_step, args.steps, world, max_seconds)
    roof = b.roofline(seconds, args.steps, name)
    # the same steps over at least --min-ms of device work: a check that the
    # K-step figure is not an artefact of a short timed region
    est = b.per_step_estimate()
    long_steps = max(args.steps, min(200000, math.ceil(args.min_ms / 1e3 / est)))
    long_sec = b.time_steps(long_steps)
    long_run = {"steps": long_steps, "ms_per_step": round(long_sec / long_steps * 1e3, 6),
                "value": round(aggregate_value(bytes_step, long_steps, 1, long_sec), 3)}
    l2_note, plan, launches = b.l2_note, b.plan, b.launches
    context = {}
    if rank == 0 and not args.no_context:
        context = {"l2_hot": b.l2_hot(args.min_ms / 4),
                   "torch_topk": b.torch_topk_context(args.min_ms / 4) if args.order == "workload" else None}
    b.free()

    # end to end through the public API with host buffers (pinned), copies inside
    e2e = e2e_measure(w, dstk, dev, stream, min(args.steps, args.e2e_steps), args.shift)
    per_workload = {}
    if world == 1 and not args.no_extra and args.shift == 0 and args.order == "workload":
        for extra in EXTRA_WORKLOADS:
            if extra != w.name:
                per_workload[extra] = run_extra(dstk, workloads.WORKLOADS[extra], dev, stream, args)
    cb = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(w, min_seconds=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": warmup,
            "ms_per_step": round(max_seconds / args.steps * 1e3, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u16" if w.dtype == torch.bfloat16 else "u32",
            "data": "synthetic (seeded SplitMix64 + Box-Muller, workloads.py)",
            "config": dict(_config(w, l2_note, args.shift),
                           **({"call": f"ds_topk_sample (temperature {SAMPLE_TEMPERATURE}, top_p {SAMPLE_TOP_P})"}
                              if args.order == "sample" else {})),
            "rows_per_s": round(w.batch * args.steps * world / max_seconds, 1),
            "roofline": roof,
            "long_run": long_run,
            **context,
            "e2e": e2e,
            "gpu_launches": args.steps * launches,
            "plan": plan.as_dict(),
            "clocks": clocks,
            "cpu_baseline": cb,
            "per_workload": per_workload or None,
            "gpu": props.name,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def e2e_measure(w, dstk, dev, stream, steps, shift=0):
    """Same metric through topk() with the input in pinned host memory: every step
    copies the batch host->device, selects, and copies the outputs back."""
    steps = max(1, steps)
    x_host = workloads.generate(w).pin_memory()
    x_dev = shifted(torch.empty_like(x_host, device=dev), shift)
    idx_dev = torch.empty((w.batch, w.k), dtype=torch.int32, device=dev)
    vals_dev = torch.empty((w.batch, w.k), dtype=w.dtype, device=dev) if w.return_value else None
    idx_host = torch.empty((w.batch, w.k), dtype=torch.int32).pin_memory()
    vals_host = torch.empty((w.batch, w.k), dtype=w.dtype).pin_memory() if w.return_value else None
    flag = torch.zeros(1, dtype=torch.int32, device=dev)

    def one():
        x_dev.copy_(x_host, non_blocking=True)
        dstk.topk(x_dev, w.k, sorted_index=w.sorted_index, return_value=w.return_value,
                  nan_flag=flag, out=(vals_dev, idx_dev), stream=stream)
        idx_host.copy_(idx_dev, non_blocking=True)
        if vals_host is not None:
            vals_host.copy_(vals_dev, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            one()
        e1.record(stream)
    stream.synchronize()
    sec = e0.elapsed_time(e1) / 1e3
    h2d = w.bytes_in
    d2h = w.batch * w.k * 4 + (w.batch * w.k * w.elem_size if w.return_value else 0)
    return {"value": round((w.bytes_in + w.bytes_out) * steps / sec / 1e9, 3), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(sec / steps * 1e3, 4)}


def run_case(args, w):
    """Profiling case (for ncu captures): generate the workload (first --rows rows)
    on the GPU and call topk() --calls times. No timing, no JSON line."""
    import sampler_topk_selection_ds_b300 as dstk
    if args.rows:
        w = w.scaled(args.rows)
    x = shifted(workloads.generate(w, device="cuda"), args.shift)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(args.calls):
        dstk.topk(x, w.k, sorted_index=w.sorted_index, return_value=w.return_value, nan_flag=flag)
    torch.cuda.synchronize()
    print(f"case {w.name}: {w.batch} rows x {w.length}, {args.calls} calls, nan_flag={int(flag.item())}")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--min-ms", type=float, default=100.0,
                    help="device time of the long check run and of each per-workload run")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=6.0)
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="--impl reference: rows of the workload per oracle step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-context", action="store_true",
                    help="skip the L2-hot figure and the torch.topk context figure")
    ap.add_argument("--order", default="workload", choices=["workload", "value", "sample"],
                    help="value: value-ordered output (sorted_index 2; one more launch per call); "
                         "sample: the sampler tail ds_topk_sample (temperature 1, top_p 0.9; "
                         "two or three launches per call)")
    ap.add_argument("--shift", type=int, default=0,
                    help="place the input this many elements past a 16-byte boundary (an odd "
                         "shift puts every row off a 16-byte boundary)")
    ap.add_argument("--case", action="store_true",
                    help="profiling case: run the workload --calls times, untimed (for ncu)")
    ap.add_argument("--rows", type=int, default=0, help="--case: use only the first ROWS rows")
    ap.add_argument("--calls", type=int, default=3, help="--case: number of calls")
    args = ap.parse_args(argv)
    w = workloads.WORKLOADS[args.workload]
    if args.order in ("value", "sample"):
        w = dataclasses.replace(w, sorted_index=2, return_value=True)
    if args.case:
        return run_case(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
