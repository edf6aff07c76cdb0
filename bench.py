#!/usr/bin/env python
"""Benchmark of the paged quantized-KV hot path on one GB300 (or N, weak scaling).

One step = one pass of the whole path over the long-context stress workload:
kv_append_quant of an 8192-token chunk into a fragmented E4M3 pool, then
paged_attention verify (q_len 5, causal among the draft) over 2 x 524288 +
6 x 32768 cached tokens, 32 query / 8 KV heads, head_dim 128, 16-token pages,
balanced split-KV merged by log-sum-exp.  Inputs are seeded synthetic data
resident in HBM (2.55 GB of KV, larger than L2, so no L2 flush is needed).

Prints one JSON line (rank 0).  Metric: effective KV GB/s of the step =
algorithmic bytes (KV codes read by attention + the append's fp16 read and
codes written + queries, outputs, block tables, slots) / device time per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pqkv|reference]
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged quantized-KV attention: effective KV GB/s (% of HBM peak), µs/step"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
REFERENCE_BUDGET_S = 90.0     # host time of the whole --impl reference run


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["pqkv", "reference"], default="pqkv")
    ap.add_argument("--workload", default="e4m3_verify_512k_stress")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--scale", type=float, default=1.0,
                    help="context-length scale of the workload (1.0 = the full workload; "
                         "smaller values are for profiling captures)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window of keys per query (0: none); the attention reads "
                         "only the pages some query's window holds, and its algorithmic bytes "
                         "count those")
    ap.add_argument("--append-tokens", type=int, default=0,
                    help="size of the step's append chunk for workloads that have one "
                         "(default: the workload's own; e.g. 8192 with --scale 0.25 profiles "
                         "the full-size append on a smaller pool)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay timing of the same step")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload figures (every workload at full size and the "
                         "8192-token append, about a minute)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed (one process per GPU; the path has no exchange step)
# ---------------------------------------------------------------------------
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest value of x over all ranks (the job's time is its slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples every 100 ms; only those taken inside the timed
    region (by their own timestamps) enter the summary."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    @classmethod
    def summarize(cls, path, t_start, t_end):
        import datetime as dt
        sm, smax, reasons, total = [], None, set(), 0
        with open(path) as f:
            lines = f.readlines()
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = dt.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                mhz, mx = float(f[2]), float(f[3])
            except ValueError:
                continue
            total += 1
            smax = mx
            if not (t_start <= ts <= t_end):
                continue
            sm.append(mhz)
            for n, v in zip(cls.REASONS, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples_in_timed_region": len(sm),
                "samples_total": total}

    def window(self, t_start, t_end):
        """Summary of the samples inside [t_start, t_end] (host wall time)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        r = self.summarize(self.path, t_start, t_end)
        r["window_s"] = round(t_end - t_start, 4)
        return r

    def close(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def remove(self):
        if self.path and os.path.exists(self.path):
            os.unlink(self.path)


# ---------------------------------------------------------------------------
# workload set-up (seeded synthetic inputs, resident in HBM)
# ---------------------------------------------------------------------------
def setup(wname: str, device: str, scale: float = 1.0, append_tokens: int = 0):
    import numpy as np
    import torch
    import paged_quantized_kv_append_gb300 as pq
    import workloads as W

    w = W.workload(wname, scale)
    if append_tokens and w.append_tokens:
        w.append_tokens = append_tokens      # a smaller pool with the full-size chunk
    plan = W.plan_pool(w)
    ks, vs = W.calibrated_scales(w, device)
    pages = pq.new_pages(plan.num_pages, w.num_kv_heads, w.kv_dtype, device, fill=0)
    for s, L in enumerate(w.seq_lens):
        for a in range(0, L, 1 << 16):
            b = min(L, a + (1 << 16))
            k, v = W.kv_tokens(w, s, a, b, device)
            slots = torch.from_numpy(W.slots_for(plan, s, a, b)).to(device)
            pq.kv_append_quant(k, v, slots, w.kv_dtype, ks, vs, pages)
    ctx = dict(w=w, plan=plan, ks=ks, vs=vs, pages=pages)
    ctx["q"] = W.query(w, device)
    ctx["out"] = torch.empty_like(ctx["q"])
    ctx["bt"] = torch.from_numpy(plan.block_table).to(device)
    ctx["seq_lens"] = torch.tensor(w.seq_lens, dtype=torch.int32, device=device)
    if w.append_tokens:
        ctx["ak"], ctx["av"] = W.append_chunk(w, device)
        ctx["aslots"] = torch.from_numpy(plan.append_slots).to(device)
    elif w.append_per_step:
        ctx["ak"], ctx["av"], sl = W.step_tokens(w, plan, device)
        ctx["aslots"] = torch.from_numpy(sl).to(device)
    ctx["ws"] = pq.Workspace(device)
    torch.cuda.synchronize()
    return ctx


def algorithmic_bytes(ctx):
    import workloads as W

    w = ctx["w"]
    B, H = w.num_seqs, w.num_kv_heads
    attn = (w.kv_bytes() + 2 * ctx["q"].numel() * 2
            + sum(w.pages_of(L) for L in w.seq_lens) * 4 + B * 4)
    n = W.step_append_tokens(w)
    app = w.append_bytes(n) if n else 0
    return attn, app


def kernel_source_hash(texts=None):
    """Hash of the attention kernel's code (comments and blank lines left out,
    so a comment edit does not orphan a capture taken on the same code)."""
    import re
    h = hashlib.sha256()
    if texts is None:
        texts = [open(os.path.join(ROOT, "paged_quantized_kv_append_gb300", "csrc", f)).read()
                 for f in ("attention_impl.cuh", "pqkv_common.cuh")]
    for text in texts:
        code = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(l.rstrip() for l in code.splitlines() if l.strip()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload, full_size):
    """DRAM bytes per attention launch from a committed ncu summary, if it was
    taken on the current kernel source and on this line's configuration (the
    workload at full size, balanced split, no window); otherwise None."""
    p = os.path.join(ROOT, "profiles", "attention_dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    if d.get("workload") != workload or not full_size:
        return None
    return d.get("dram_bytes_per_launch")


def hbm_peak():
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------
def cpu_cores():
    """Host cores this process may run on (its CPU affinity)."""
    return len(os.sched_getaffinity(0))


def blas_threads():
    """Threads of the BLAS pool numpy runs the oracle's products on, or None
    when it cannot be queried: threadpoolctl when installed, else the thread
    count the loaded OpenBLAS library reports about itself."""
    import ctypes
    import numpy  # noqa: F401  (loads numpy's BLAS before it is inspected)
    try:
        from threadpoolctl import threadpool_info
        pools = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if pools:
            return max(pools)
    except Exception:
        pass
    try:
        paths = {line.split()[-1] for line in open("/proc/self/maps")
                 if "openblas" in line.lower() and ".so" in line}
    except OSError:
        return None
    for path in sorted(paths):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("openblas_get_num_threads", "openblas_get_num_threads64_",
                    "scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return None


class OracleSample:
    """One (sequence, kv-head) segment of the workload -- its shortest
    sequence, up to 32768 tokens -- encoded once by the oracle; run(n) times
    the oracle's paged attention over the first n tokens of it."""

    def __init__(self, wname: str):
        import numpy as np
        import oracle
        import workloads as W
        self.oracle, self.np = oracle, np
        w = W.workload(wname)
        self.w = w
        s = int(np.argmin(w.seq_lens))
        self.L = L = w.seq_lens[s]
        n = w.pages_of(L)
        rng = np.random.default_rng(0)
        self.bt = rng.permutation(n).astype(np.int32)[None, :]
        k, v = W.kv_tokens(w, s, 0, L, "cpu")
        self.ks = W.scale_from_amax(k.float().abs().max().item(), 448.0)
        self.vs = W.scale_from_amax(v.float().abs().max().item(), 448.0)
        t = np.arange(L)
        pool = oracle.new_pool(n, w.num_kv_heads, w.head_dim, w.kv_dtype)
        self.pool = oracle.kv_append_quant(k.numpy(), v.numpy(),
                                           self.bt[0, t // 16].astype(np.int64) * 16 + t % 16,
                                           w.kv_dtype, [self.ks], [self.vs], pool)
        self.q = W.query(w, "cpu").numpy()[s * w.q_len:(s + 1) * w.q_len]
        self.h = 0

    def run(self, n_tokens: int):
        """(KV code bytes read, seconds) of one oracle call over n_tokens keys."""
        w = self.w
        n = max(w.q_len, min(int(n_tokens), self.L))
        t0 = time.perf_counter()
        self.oracle.paged_attention(self.q, self.pool, self.bt, [n], w.q_len, w.kv_dtype,
                                    [self.ks], [self.vs], heads=[self.h])
        dt = time.perf_counter() - t0
        self.h = (self.h + 1) % w.num_kv_heads
        return n * w.head_dim * 2 * w.elem_bytes, dt

    def describe(self, n):
        w = self.w
        return ("oracle paged_attention (float64 numpy) over (sequence, kv-head) segments of %d "
                "tokens (q_len %d, %d query rows each) of the workload's %d-token sequences; KV code "
                "bytes read / wall time" % (n, w.q_len, w.group * w.q_len, self.L))


def oracle_sample(wname: str, seconds: float, max_segments: int = 64):
    """Time the oracle on whole segments of the workload's shortest sequence
    until `seconds` have elapsed (at least one segment)."""
    smp = OracleSample(wname)
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds and done < max_segments:
        b, _ = smp.run(smp.L)
        nbytes += b
        done += 1
    dt = time.perf_counter() - t0
    return {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": cpu_cores(),
            "blas_threads": blas_threads(), "kind": "oracle",
            "sample": "%d segments: " % done + smp.describe(smp.L), "seconds": dt}


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------
LOAD_S = 0.6          # seconds of identical load before and after the headline's timed steps
CONFIG_MIN_S = 1.0    # each per-config figure is timed over at least this much wall time


def run_for(fn, seconds):
    """Run fn back to back for about `seconds` of wall time, keeping at most
    two batches queued so the GPU never idles for long."""
    import torch
    prev = None
    t_end = time.time() + seconds
    while time.time() < t_end:
        for _ in range(8):
            fn()
        ev = torch.cuda.Event()
        ev.record()
        if prev is not None:
            prev.synchronize()
        prev = ev
    torch.cuda.synchronize()


def graph_time(fns, reps, min_s):
    """Capture `reps` passes over fns in one CUDA graph, replay it back to
    back for at least min_s seconds, and return (us per pass, (t0, t1)) from
    CUDA events around the replays on the current stream."""
    import math
    import torch
    stream = torch.cuda.current_stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            for f in fns:
                f()
    g.replay()
    torch.cuda.synchronize()
    c0 = time.perf_counter()
    g.replay()
    torch.cuda.synchronize()
    one = time.perf_counter() - c0
    n = max(3, int(math.ceil(min_s / max(one, 1e-6))))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(n):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    del g
    return e0.elapsed_time(e1) * 1e3 / (n * reps), (t0, t1)


def reps_for(fn, target_s=2e-3, cap=200):
    """Passes per graph so that one replay lasts about target_s."""
    import torch
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        fn()
    e1.record()
    torch.cuda.synchronize()
    per = e0.elapsed_time(e1) * 1e-3 / 5
    return max(1, min(cap, int(target_s / max(per, 1e-7))))


class L2Flush:
    """Reads a buffer twice the size of L2 (a read leaves no dirty lines for
    the next kernel to write back)."""

    def __init__(self, device):
        import torch
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.buf = torch.ones(max(1, 2 * l2 // 4), dtype=torch.float32, device=device)
        self.l2 = l2

    def __call__(self):
        self.buf.sum()


def _span(windows):
    return min(a for a, _ in windows), max(b for _, b in windows)


def _rate(nbytes, us, peak):
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_step": us, "gbs": gbs, "frac_of_hbm": gbs / peak}


def window_bytes(w, window):
    """Algorithmic bytes of a sliding-window attention launch: K and V codes of
    the keys some query's window holds (keys L - q_len - window + 1 .. L - 1
    of each sequence), q, out, the block-table entries of the pages read, and
    seq_lens."""
    kv = toks = pages = 0
    for L in w.seq_lens:
        lo = max(0, L - w.q_len - window + 1)
        toks += L - lo
        pages += w.pages_of(L) - lo // w.page_size
    kv = toks * w.num_kv_heads * w.head_dim * 2 * w.elem_bytes
    q_bytes = w.num_seqs * w.q_len * w.num_q_heads * w.head_dim * 2
    return kv + 2 * q_bytes + pages * 4 + w.num_seqs * 4


def config_entry(pq, W, ctx, peak, flush=None, headline=None, window=0):
    """One workload's figures: the step (append if the workload appends every
    step, then attention) and the attention alone, each a CUDA graph of
    back-to-back launches replayed for at least CONFIG_MIN_S; with `flush`,
    also the same launches after an L2 flush (flush + launch minus flush).
    `window` > 0 times the sliding-window attention instead (no append)."""
    w = ctx["w"]
    attn_bytes, app_bytes = algorithmic_bytes(ctx)
    step_appends = (bool(w.append_per_step) or bool(w.append_tokens)) and not window
    if window:
        attn_bytes = window_bytes(w, window)

    def attention():
        pq.paged_attention(ctx["q"], ctx["pages"], ctx["bt"], ctx["seq_lens"], w.q_len,
                           w.kv_dtype, ctx["ks"], ctx["vs"], ctx["out"], workspace=ctx["ws"],
                           max_seq_len=max(w.seq_lens), window=window)

    def append():
        pq.kv_append_quant(ctx["ak"], ctx["av"], ctx["aslots"], w.kv_dtype, ctx["ks"], ctx["vs"],
                           ctx["pages"])

    step = [append, attention] if step_appends else [attention]
    windows = []
    reps = reps_for(lambda: [f() for f in step])
    step_us, win = graph_time(step, reps, CONFIG_MIN_S)
    windows.append(win)
    if step_appends:
        attn_us, win = graph_time([attention], reps, CONFIG_MIN_S / 2)
        windows.append(win)
    else:
        attn_us = step_us
    e = {"workload": w.name + ("_window%d" % window if window else ""),
         "shape": "%s x %s tokens, %d/%d heads, q_len %d, %s" % (
             w.num_seqs, (w.seq_lens[0] if len(set(w.seq_lens)) == 1 else
                          "%d..%d" % (min(w.seq_lens), max(w.seq_lens))),
             w.num_q_heads, w.num_kv_heads, w.q_len,
             {0: "fp16", 1: "e4m3", 2: "int8", 3: "int8 row scales"}[w.kv_dtype]),
         "step": ("append %d tokens + attention" % W.step_append_tokens(w)) if step_appends
         else "attention",
         "attention_bytes": attn_bytes, "append_bytes": app_bytes if step_appends else 0,
         "l2": "warm: back-to-back launches on the same inputs" if flush else
               "inputs larger than L2 (%.2f GB of KV)" % (w.kv_bytes() / 1e9)}
    if window:
        e["window"] = window
    e.update(_rate(attn_bytes + (app_bytes if step_appends else 0), step_us, peak))
    e["attention_us"] = attn_us
    e["attention_frac_of_hbm"] = attn_bytes / (attn_us * 1e-6) / 1e9 / peak
    if headline is not None:
        e["bench_line_attention_us"] = headline
    if flush is not None:
        f_reps = max(1, min(reps, 50))
        both_us, win = graph_time([flush] + step, f_reps, CONFIG_MIN_S / 2)
        windows.append(win)
        fl_us, win = graph_time([flush], f_reps, CONFIG_MIN_S / 2)
        windows.append(win)
        us = both_us - fl_us
        e["l2_flushed"] = dict(_rate(attn_bytes, us, peak),
                               how="each launch after a read of %d MB (2x L2): graph of "
                                   "(read, launch) minus graph of (read)" % (2 * flush.l2 >> 20))
    e["_win"] = _span(windows)
    e["timing"] = ("CUDA graph of %d back-to-back steps replayed for >= %.1f s, CUDA events "
                   "around the replays" % (reps, CONFIG_MIN_S))
    return e


def append_entry(pq, W, device, peak, ks, vs, n_sets=6):
    """The 8192-token append of the long-context stress workload on its own:
    n_sets copies of the chunk, each into its own fragmented set of free pages
    (offset 7 inside the first), cycled so the inputs and written pages
    (6 x 50 MB) exceed L2."""
    import numpy as np
    import torch
    w = W.workload("e4m3_verify_512k_stress")
    npg = w.pages_of(w.append_tokens + w.append_offset)
    rng = np.random.default_rng(np.random.SeedSequence([w.seed, 9]))
    num_pages = n_sets * npg + 64
    perm = rng.permutation(num_pages).astype(np.int64)
    pages = pq.new_pages(num_pages, w.num_kv_heads, w.kv_dtype, device, fill=0)
    ak, av = W.append_chunk(w, device)
    t = np.arange(w.append_tokens, dtype=np.int64) + w.append_offset
    sets = []
    for i in range(n_sets):
        chunk = perm[i * npg:(i + 1) * npg]
        sl = torch.from_numpy(chunk[t // 16] * 16 + t % 16).to(device)
        sets.append((ak.clone(), av.clone(), sl))

    def one(i):
        k, v, sl = sets[i]
        return lambda: pq.kv_append_quant(k, v, sl, w.kv_dtype, ks, vs, pages)

    fns = [one(i) for i in range(n_sets)]
    reps = reps_for(lambda: [f() for f in fns])
    us, win = graph_time(fns, reps, CONFIG_MIN_S)
    us /= n_sets
    nbytes = w.append_bytes(w.append_tokens)
    e = {"workload": "append_8192_fragmented",
         "shape": "8192 tokens x 8 kv-heads, E4M3, into a fragmented pool at page offset 7",
         "append_bytes": nbytes, "l2": "%d rotating input/page sets (%.0f MB) > L2" % (
             n_sets, n_sets * nbytes / 1e6)}
    e.update(_rate(nbytes, us, peak))
    e["_win"] = win
    e["timing"] = "CUDA graph of %d x %d appends replayed for >= %.1f s" % (reps, n_sets,
                                                                          CONFIG_MIN_S)
    del pages, sets
    return e


def per_config(pq, W, device, peak, headline_ctx, headline_us):
    """Every workload of the path at full size (with the row-scaled INT8 and
    32-row verify variants), plus the 8192-token append."""
    import gc
    import torch
    out = {}
    flush = L2Flush(device)
    out[headline_ctx["w"].name] = config_entry(pq, W, headline_ctx, peak, headline=headline_us)
    for name in ("tiny_fp16_decode", "e4m3_decode_b8", "e4m3_verify_131k",
                 "int8_decode_append_262k", "int8_row_decode_262k", "int8_row_verify_131k",
                 "e4m3_verify_q8_131k"):
        ctx = setup(name, device)
        small = ctx["w"].kv_bytes() < 2 * flush.l2
        out[name] = config_entry(pq, W, ctx, peak, flush=flush if small else None)
        if name == "e4m3_verify_131k":
            # the same verify restricted to a 2048-token sliding window
            e = config_entry(pq, W, ctx, peak, flush=flush, window=2048)
            out[e["workload"]] = e
        del ctx
        gc.collect()
        torch.cuda.empty_cache()
    out["append_8192_fragmented"] = append_entry(pq, W, device, peak, headline_ctx["ks"],
                                                 headline_ctx["vs"])
    del flush
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    workload: every step runs the oracle over the first n tokens of one
    (sequence, kv-head) segment, n chosen from a calibration so that all
    warm-up and timed steps fit about REFERENCE_BUDGET_S seconds."""
    if rank != 0:
        return
    smp = OracleSample(args.workload)
    b0, t0 = smp.run(min(smp.L, 2048))                      # calibration
    per_token = t0 / max(1, min(smp.L, 2048))
    per_step = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    n = int(max(256, min(smp.L, per_step / max(per_token, 1e-9))))
    for _ in range(args.warmup):
        smp.run(n)
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b, dt = smp.run(n)
        tot_b += b
        tot_s += dt
    value = tot_b / tot_s / 1e9
    cb = {"value": value, "unit": UNIT, "cores": cpu_cores(), "blas_threads": blas_threads(),
          "kind": "oracle",
          "sample": "%d steps, each: " % args.steps + smp.describe(n), "seconds": tot_s}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_s * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "sample": cb["sample"]},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_pqkv(args, rank, local, world):
    import torch
    import paged_quantized_kv_append_gb300 as pq
    import workloads as W
    from paged_quantized_kv_append_gb300 import build as pqbuild

    pqbuild.build()
    pq.load_library()
    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    ctx = setup(args.workload, dev, args.scale, args.append_tokens)
    w = ctx["w"]
    stream = torch.cuda.current_stream()
    attn_bytes, app_bytes = algorithmic_bytes(ctx)
    if args.window:
        attn_bytes = window_bytes(w, args.window)
    appends = "ak" in ctx
    launches_per_step = 1 + (1 if appends else 0)

    def step(ev=None):
        if appends:
            pq.kv_append_quant(ctx["ak"], ctx["av"], ctx["aslots"], w.kv_dtype, ctx["ks"],
                               ctx["vs"], ctx["pages"])
        if ev is not None:
            ev[0].record(stream)
        pq.paged_attention(ctx["q"], ctx["pages"], ctx["bt"], ctx["seq_lens"], w.q_len,
                           w.kv_dtype, ctx["ks"], ctx["vs"], ctx["out"],
                           num_splits=args.num_splits, workspace=ctx["ws"],
                           max_seq_len=max(w.seq_lens), window=args.window)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- device-timed region: exactly --steps steps between a barrier and a
    #      synchronize on each side.  The clock record covers a load window of
    #      identical back-to-back steps around it (LOAD_S before and after), so
    #      the 100 ms nvidia-smi samples fall under the same load even when the
    #      timed region itself is shorter than one sampling interval.
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    attn_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    load_start = time.time()
    run_for(step, LOAD_S)
    barrier(world)
    torch.cuda.synchronize()
    w_start = time.time()
    t0.record(stream)
    for i in range(args.steps):
        step(attn_ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    w_end = time.time()
    barrier(world)
    run_for(step, LOAD_S)
    torch.cuda.synchronize()
    load_end = time.time()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    ms_step = total_ms / args.steps
    attn_ms = [a.elapsed_time(b) for a, b in attn_ev]
    attn_avg = statistics.mean(attn_ms)
    step_bytes = attn_bytes + app_bytes
    value = world * step_bytes / (ms_step * 1e-3) / 1e9

    # ---- the same step captured once in a CUDA graph and replayed
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(max(3, args.warmup)):
            g.replay()
        torch.cuda.synchronize()
        barrier(world)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        g_ms = max_over_ranks(g0.elapsed_time(g1), world) / args.steps
        graph = {"value": world * (attn_bytes + app_bytes) / (g_ms * 1e-3) / 1e9, "unit": UNIT,
                 "us_per_step": g_ms * 1e3, "launches_per_step": launches_per_step}
        del g

    # ---- end to end through the public API with host buffers.  Every step
    #      copies its own inputs from pinned host memory and reads its output
    #      back on the host; step i+1's inputs travel on a second stream while
    #      step i computes (two buffer sets), the usual serving pipeline.
    e2e = None
    if not args.no_e2e:
        names = ["q", "bt", "seq_lens"] + (["ak", "av", "aslots"] if appends else [])
        host = {n: ctx[n].cpu().pin_memory() for n in names}
        dev_in = [{n: torch.empty_like(ctx[n]) for n in names} for _ in range(2)]
        outs = [torch.empty_like(ctx["out"]) for _ in range(2)]
        out_host = [torch.empty(ctx["out"].shape, dtype=ctx["out"].dtype, pin_memory=True)
                    for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host[0].numel() * out_host[0].element_size()
        copy_stream = torch.cuda.Stream()
        ev_copied = [torch.cuda.Event() for _ in range(2)]
        ev_freed = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        seen = []

        def enqueue(i):
            b = i % 2
            d = dev_in[b]
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(ev_freed[b])      # step i-2 is done with buffer b
                for n, t in host.items():
                    d[n].copy_(t, non_blocking=True)
                ev_copied[b].record(copy_stream)
            stream.wait_event(ev_copied[b])
            if appends:
                pq.kv_append_quant(d["ak"], d["av"], d["aslots"], w.kv_dtype, ctx["ks"],
                                   ctx["vs"], ctx["pages"])
            pq.paged_attention(d["q"], ctx["pages"], d["bt"], d["seq_lens"], w.q_len, w.kv_dtype,
                               ctx["ks"], ctx["vs"], outs[b], num_splits=args.num_splits,
                               workspace=ctx["ws"], max_seq_len=max(w.seq_lens),
                               window=args.window)
            ev_freed[b].record(stream)
            out_host[b].copy_(outs[b], non_blocking=True)
            ev_done[b].record(stream)

        def read(i):
            ev_done[i % 2].synchronize()
            seen.append(float(out_host[i % 2][0, 0, 0]))         # the host reads the result

        def run(n):
            for i in range(n):
                enqueue(i)
                if i >= 1:
                    read(i - 1)
            read(n - 1)

        run(max(3, args.warmup))
        torch.cuda.synchronize()
        barrier(world)
        s0 = time.perf_counter()
        run(args.steps)
        el = max_over_ranks(time.perf_counter() - s0, world)
        torch.cuda.synchronize()
        same = bool(torch.equal(outs[(args.steps - 1) % 2], ctx["out"]))
        e2e = {"value": world * step_bytes * args.steps / el / 1e9, "unit": UNIT,
               "output_matches_device_run": same,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": el * 1e3 / args.steps,
               "pipeline": "step i+1's inputs copied on a second stream while step i computes; "
                           "each step's output copied back and read on the host"}

    peak, peak_src = hbm_peak()
    configs = None
    if (not args.no_per_config and args.scale == 1.0 and not args.window and
            args.workload == "e4m3_verify_512k_stress"):
        configs = per_config(pq, W, dev, peak, ctx, attn_avg * 1e3)
    clocks.close()
    clk = clocks.window(load_start, load_end)
    clk["window"] = ("load window: the timed steps with %.1f s of the same back-to-back steps "
                     "before and after" % LOAD_S)
    clk["samples_in_timed_steps"] = clocks.window(w_start, w_end)["samples_in_timed_region"]
    clk["timed_steps_s"] = round(w_end - w_start, 4)
    if configs:
        for e in configs.values():
            e["clocks"] = clocks.window(*e.pop("_win"))
    clocks.remove()
    if rank != 0:
        return
    achieved = attn_bytes / (attn_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
        "pct_of_hbm_peak": 100.0 * (step_bytes / (ms_step * 1e-3) / 1e9) / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 codes, f16 products, f32 accumulation" if w.kv_dtype == 1 else
                 ("int8 codes, f16 products, f32 accumulation" if w.kv_dtype == 2 else "f16"),
        "data": "synthetic",
        "config": {"workload": w.name, "scale": args.scale,
                   "seq_lens": "2x524288+6x32768" if (w.name.endswith("stress") and args.scale == 1.0)
                   else w.seq_lens, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "page_size": w.page_size, "q_len": w.q_len,
                   "append_tokens": W.step_append_tokens(w), "num_splits": args.num_splits,
                   "window": args.window,
                   "attention_bytes": attn_bytes, "append_bytes": app_bytes,
                   "l2": "inputs larger than L2 (%.2f GB of KV per step)" % (w.kv_bytes() / 1e9)},
        "roofline": {"bound": "hbm", "kernel": "paged_attention_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_src
                     if peak_src == "measured" else "fallback",
                     "traffic": measured_traffic(w.name, args.scale == 1.0 and not args.window and
                                                 args.num_splits == 0),
                     "attention_us": attn_avg * 1e3},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "e2e": e2e,
        "graph": graph,
        "per_config": configs,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample(args.workload, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, local, world = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_pqkv(args, rank, local, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
