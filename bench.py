"""Benchmark: paged split-KV decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

One step = one fd_decode_paged call (split + merge) over one batch of the
synthetic workload, inputs resident in HBM.  Workloads larger than 2x L2 are
timed back to back between one CUDA-event pair on the launching stream; for
smaller ones every timed step is preceded by an L2 flush (a write, then read,
of 2x the L2 size) outside that step's event pair; in `per_config` their
us per call is the marginal time of a call in a stream of (flush, call) pairs
(an event pair around many pairs minus one around as many flushes), with the
per-call event-pair mean beside it.  Prints ONE JSON line (rank 0).

metric: achieved HBM GB/s of the decode call = algorithmic bytes (K+V of the
live tokens, q, out, lse, live block-table entries, seq_lens, FP8 scales) /
device time; us per call is reported beside it.  The headline workload is the
Llama-3-8B-shaped GQA batch; at one GPU the line also carries `per_config`:
all five workloads (tiny MHA, single-sequence MHA, GQA batch, 131k-token long
context, mixed FP8 batch) with us per call, GB/s, fraction of the measured
copy peak, the plan, and the fp64 oracle timed on the host cores beside each.

Under torchrun (N > 1) every rank runs its own replica of the workload (seed
offset by rank, no collective on the data path: weak scaling) and value =
bytes of all ranks / max over ranks of the elapsed time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

HEADLINE_CONFIG = 3
METRIC = "decode-attention achieved HBM GB/s"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the kernel sources plus fd_api.cu, which encodes the TMA maps (box shape,
# swizzle, L2 promotion) that shape the kernel's DRAM traffic
DECODE_KERNEL_FILES = ("decode_kernel.cuh", "decode_dispatch.cuh", "decode_f16.cu", "decode_bf16.cu",
                       "decode_e4m3.cu", "ptx.cuh", "fd_internal.h", "fd_api.cu")


def kernel_source_hash():
    """Hash of the code that defines the decode kernel, comments and blank
    lines left out (ties a committed ncu traffic figure to the kernel it was
    measured on)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "split_kv_decode_paged_gb300", "csrc")
    for f in DECODE_KERNEL_FILES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            code = [ln.split("//", 1)[0].rstrip() for ln in fh]
        h.update(f.encode() + "\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload_tag):
    """DRAM bytes per launch of the decode kernel for a workload, from the
    committed ncu summary profiles/decode_traffic.json, or None when absent
    or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)["workloads"][workload_tag]
    except Exception:
        return None
    if entry.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return int(entry["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []
        self.first = 0

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()  # start timing only once samples flow
            while not self.lines and time.time() - t0 < 3.0:
                time.sleep(0.01)
            self.first = len(self.lines)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(elapsed_s, bytes_done, group=None):
    """Whole-job aggregation across ranks: total bytes and the max elapsed
    time.  Works with any torch.distributed backend (gloo on CPU tensors in
    the tests, NCCL on the GPU)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return elapsed_s, bytes_done
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" else torch.device("cpu")
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    b = torch.tensor([float(bytes_done)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(b, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), int(b.item())


# ------------------------------------------------------------- GPU timing
_flush_sink = {}


def l2_flush(buf):
    """Make the L2 cold and clean: write a buffer larger than L2, then read
    it back (the read evicts the dirty lines the write left, so their
    write-back is not charged to the next timed call)."""
    buf.zero_()
    sink = _flush_sink.setdefault(buf.device, torch.empty((), dtype=buf.dtype, device=buf.device))
    torch.sum(buf, dim=0, out=sink)


def time_decode(wl, steps, warmup, flush, stream=None, **plan_opts):
    import split_kv_decode_paged_gb300 as fd
    dec = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens.cpu(), **plan_opts)
    out = torch.empty_like(wl.q)
    lse = torch.empty(wl.q.shape[:2], dtype=torch.float32, device=wl.q.device)
    args = (wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    kw = dict(k_scale=wl.k_scale, v_scale=wl.v_scale, out=out, lse=lse)
    for _ in range(warmup):
        if flush is not None:
            l2_flush(flush)
        dec(*args, **kw)
    torch.cuda.synchronize()
    dec.check()
    st = torch.cuda.current_stream()
    torch.cuda.nvtx.range_push("fd_timed")
    if flush is None:
        # Back to back, one event pair around all steps: consecutive calls
        # overlap one's prologue with the previous one's tail (programmatic
        # dependent launch), as in a serving loop.  Per-step times are the mean.
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(steps):
            dec(*args, **kw)
        b.record(st)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        dec.check()
        return [a.elapsed_time(b) / steps] * steps, dec
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        l2_flush(flush)
        ev[i][0].record(st)
        dec(*args, **kw)
        ev[i][1].record(st)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    dec.check()
    ms = [a.elapsed_time(b) for a, b in ev]
    return ms, dec


def flushed_marginal_us(wl, dec, flush, pairs=50, reps=5):
    """Marginal time of one call in a stream of (L2 flush, call) pairs: one
    event pair around `pairs` (flush, call) pairs minus one around `pairs`
    flushes alone, divided by `pairs`; the median over `reps`.  Like the
    back-to-back timing of the large workloads it leaves out the launch
    latency that queued work hides, while every call still starts with a
    cold L2 (an event pair around each call measures that latency too)."""
    out = torch.empty_like(wl.q)
    lse = torch.empty(wl.q.shape[:2], dtype=torch.float32, device=wl.q.device)
    args = (wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    kw = dict(k_scale=wl.k_scale, v_scale=wl.v_scale, out=out, lse=lse)
    st = torch.cuda.current_stream()
    res = []
    for _ in range(reps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(st)
        for _ in range(pairs):
            l2_flush(flush)
            dec(*args, **kw)
        e[1].record(st)
        for _ in range(pairs):
            l2_flush(flush)
        e[2].record(st)
        torch.cuda.synchronize()
        res.append((e[0].elapsed_time(e[1]) - e[1].elapsed_time(e[2])) * 1e3 / pairs)
    dec.check()
    return statistics.median(res)


def time_warm_and_graph(wl, dec, iters=50):
    """Warm-L2 and CUDA-graph-replay per-call times (labelled as such)."""
    out = torch.empty_like(wl.q)
    lse = torch.empty(wl.q.shape[:2], dtype=torch.float32, device=wl.q.device)
    args = (wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    kw = dict(k_scale=wl.k_scale, v_scale=wl.v_scale, out=out, lse=lse)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            dec(*args, **kw)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(iters):
            dec(*args, **kw)
        b.record(s)
    torch.cuda.synchronize()
    warm = a.elapsed_time(b) / iters
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(10):
            dec(*args, **kw)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters // 10):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    graph = a.elapsed_time(b) / (iters // 10 * 10)
    dec.check()
    return warm, graph


def time_e2e(wl, dec, steps):
    """End to end through the C ABI with host buffers: every step copies a
    packed pinned host block holding q, the block table and seq_lens to the
    device (one copy, fd_host_copy_in, on a copy stream where it overlaps the
    previous step's decode: two sets of blocks in turn, HostPipeline) and runs
    the decode (fd_decode_paged_staged), which stores out + lse into the packed
    pinned host output block (mapped for the device), all inside the timed
    region; the timer stops after a synchronise, with every step's results in
    host memory.  The paged K/V cache is state that lives in HBM across
    steps."""
    pipe = dec.host_pipeline(2)
    for io in pipe.ios:
        io.q.copy_(wl.q.cpu())
        io.block_table.copy_(wl.block_table.cpu())
        io.seq_lens.copy_(wl.seq_lens.cpu())

    def step():
        pipe.submit(wl.k_pages, wl.v_pages, wl.k_scale, wl.v_scale)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    dec.check()
    return dt, pipe.ios[0].layout.in_bytes, pipe.ios[0].layout.out_bytes


# ------------------------------------------------------------ CPU oracle
def cpu_baseline(wl_cpu, target_s=12.0, seed=0):
    import numpy as np
    from oracle import oracle as orc
    s = wl_cpu.spec
    code = {torch.float16: orc.F16, torch.bfloat16: orc.BF16, torch.float8_e4m3fn: orc.E4M3}
    p = orc.problem(s.B, s.Hq, s.Hkv, s.D, s.page_size, wl_cpu.max_blocks, wl_cpu.num_pages,
                    code[wl_cpu.q.dtype], code[wl_cpu.k_pages.dtype])
    lens = wl_cpu.seq_lens.numpy().astype(np.int64)
    total_work = int(lens.sum()) * s.Hq
    cores = len(os.sched_getaffinity(0))
    rng = np.random.default_rng(seed)
    order = [(int(b), int(h)) for b in rng.permutation(s.B) for h in rng.permutation(s.Hq)]
    # calibrate on a small batch, then size the sample to ~target_s
    done, work, elapsed = 0, 0, 0.0
    n = max(cores, 8)
    while done < len(order) and elapsed < target_s:
        batch = order[done:done + n]
        t0 = time.perf_counter()
        orc.decode_paged_pairs(p, wl_cpu.q, wl_cpu.k_pages, wl_cpu.v_pages, wl_cpu.k_scale, wl_cpu.v_scale,
                               wl_cpu.block_table, wl_cpu.seq_lens, batch, nthreads=cores)
        elapsed += time.perf_counter() - t0
        work += sum(int(lens[b]) for b, _ in batch)
        done += len(batch)
        rate = work / max(elapsed, 1e-9)
        n = max(cores, int(rate * min(target_s - elapsed, target_s / 3) / max(1, lens.mean())))
    us_per_call = elapsed / max(work, 1) * total_work * 1e6
    from split_kv_decode_paged_gb300 import workloads as W
    gbs = W.algorithmic_bytes(s, wl_cpu.seq_lens) / (us_per_call * 1e-6) / 1e9
    return {"value": gbs, "unit": "GB/s", "us_per_call": us_per_call, "cores": cores, "kind": "oracle",
            "sample": f"{done} of {s.B * s.Hq} (b, hq) pairs, {work} of {total_work} token-heads, "
                      f"{elapsed:.1f} s fp64 on {cores} host threads, scaled to one call by token-heads"}


# ------------------------------------------------------ shared-prefix batch
def bench_cascade(args):
    """Cascade decode (shared prefix read in one pass for all sequences) against
    a plain decode over the same concatenated tables, both from a cold L2."""
    from split_kv_decode_paged_gb300 import workloads as W
    from split_kv_decode_paged_gb300.cascade import CascadeDecoder
    import split_kv_decode_paged_gb300 as fd
    dev = torch.device("cuda", torch.cuda.current_device())
    from split_kv_decode_paged_gb300 import build as fd_build
    fd_build.build()
    B, prefix = 64, 4096
    g = torch.Generator().manual_seed(2024)
    suffix = torch.randint(16, 1025, (B,), generator=g, dtype=torch.int32)
    spec = W.Spec("shared-prefix batch", B=B, Hq=32, Hkv=8, D=128, page_size=16, kv="bf16", q="bf16",
                  lens=("const", 1))
    sp = W.make_shared_prefix(spec, 2024, prefix, suffix, dev)
    fl = sp.flat
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)
    cas = CascadeDecoder(B, spec.Hq, spec.Hkv, spec.D, 16, fl.num_pages, sp.prefix_table.shape[1],
                         sp.suffix_table.shape[1], prefix, sp.suffix_lens.cpu(), fl.q.dtype, fl.k_pages.dtype)
    plen = torch.tensor([prefix], dtype=torch.int32, device=dev)
    dec = fd.PagedDecoder.for_pools(fl.q, fl.k_pages, fl.v_pages, fl.block_table, fl.seq_lens.cpu())

    def run_cas():
        cas(fl.q, fl.k_pages, fl.v_pages, sp.prefix_table, plen, sp.suffix_table, sp.suffix_lens)

    def run_flat():
        dec(fl.q, fl.k_pages, fl.v_pages, fl.block_table, fl.seq_lens)

    def timeit(fn):
        for _ in range(args.warmup):
            l2_flush(flush)
            fn()
        ev = []
        for _ in range(args.steps):
            l2_flush(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            ev.append((a, b))
        torch.cuda.synchronize()
        return statistics.median([x.elapsed_time(y) for x, y in ev]) * 1e3

    us_cas, us_flat = timeit(run_cas), timeit(run_flat)
    cas.check()
    dec.check()
    kv_row = spec.Hkv * spec.D * 2 * 2
    unique = (prefix + int(suffix.sum())) * kv_row + 2 * B * spec.Hq * spec.D * 2
    flat_bytes = W.algorithmic_bytes(fl.spec, fl.seq_lens.cpu())
    peak, kind = measured_peak()
    print(json.dumps({
        "metric": "cascade decode achieved HBM GB/s (unique K/V bytes)", "value": unique / us_cas / 1e3,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "us_per_call": us_cas,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"shared-prefix batch: B={B}, Hq=32, Hkv=8, D=128, bf16, 16-token pages, "
                               f"shared prefix {prefix} tokens, own suffix U[16,1024] (seed 2024)",
                   "l2": "flushed before every timed call (write, then read, of 256 MB)"},
        "flat_decode_us_per_call": us_flat, "speedup_vs_flat": us_flat / us_cas,
        "unique_kv_bytes": unique, "flat_algorithmic_bytes": flat_bytes,
        "frac_of_peak": unique / us_cas / 1e3 / peak, "peak_source": kind,
        "gpu_launches_per_call": 3}))


# ------------------------------------------------------- append and merge
def _time_flushed(fn, steps, warmup, flush):
    for _ in range(warmup):
        l2_flush(flush)
        fn()
    ev = []
    torch.cuda.nvtx.range_push("fd_timed")
    for _ in range(steps):
        l2_flush(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ms = sorted(x.elapsed_time(y) for x, y in ev)
    return statistics.median(ms) * 1e3, ms[len(ms) // 10] * 1e3, ms[(len(ms) * 9) // 10] * 1e3


def bench_append(args):
    """fd_append_kv (one new K and V row per sequence and KV head written into
    the paged pools) on the GQA-batch pools (bf16) and the mixed FP8 pools
    (bf16 rows quantised to E4M3 with the page's scale), L2 flushed before
    every call."""
    from split_kv_decode_paged_gb300 import workloads as W
    import split_kv_decode_paged_gb300 as fd
    from split_kv_decode_paged_gb300 import _lib
    from split_kv_decode_paged_gb300 import build as fd_build
    fd_build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)
    peak, kind = measured_peak()
    cases = {}
    for c in (3, 5):
        wl = W.make_config(c, dev)
        spec = wl.spec
        B, Hkv, D = spec.B, spec.Hkv, spec.D
        in_dtype = wl.q.dtype if wl.k_pages.dtype == torch.float8_e4m3fn else wl.k_pages.dtype
        g = torch.Generator(device=dev).manual_seed(77 + c)
        k_new = torch.randn((B, Hkv, D), generator=g, device=dev).to(in_dtype)
        v_new = torch.randn((B, Hkv, D), generator=g, device=dev).to(in_dtype)
        pos = (wl.seq_lens - 1).clamp(min=0).to(torch.int32)  # rewrite each sequence's last token
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def run():
            fd.append_kv(wl.q.dtype, k_new, v_new, wl.k_pages, wl.v_pages, wl.block_table, pos,
                         wl.k_scale, wl.v_scale, status=status)

        med, p10, p90 = _time_flushed(run, args.steps, args.warmup, flush)
        if int(status.item()) != 0:
            raise RuntimeError(f"append flagged status {int(status.item())}")
        e_in, e_c = k_new.element_size(), wl.k_pages.element_size()
        nbytes = B * Hkv * D * 2 * (e_in + e_c) + 8 * B + (8 * B * Hkv if e_c == 1 else 0)
        cases[f"config {c}"] = {"workload": f"{spec.name}: B={B}, Hkv={Hkv}, D={D}, {spec.kv} pages of {spec.page_size}",
                                "us_median": med, "us_p10": p10, "us_p90": p90, "bytes": nbytes,
                                "gbs": nbytes / med / 1e3}
        # The same append with rotary embedding fused in: K rotated before the
        # cache write and q [B, Hq, D] rotated in place (GPT-NeoX pairs, the
        # full head dimension), cos/sin tables for every position of the pool.
        max_pos = wl.max_blocks * spec.page_size
        ang = (torch.arange(max_pos, dtype=torch.float64)[:, None] *
               (10000.0 ** (-torch.arange(D // 2, dtype=torch.float64) * 2 / D))[None, :])
        cos, sin = ang.cos().float().to(dev), ang.sin().float().to(dev)
        prob = _lib.make_problem(B, spec.Hq, Hkv, D, spec.page_size, wl.max_blocks, wl.num_pages, wl.q.dtype,
                                 wl.k_pages.dtype)

        def run_rot():
            _lib.fd_append_kv_rotary(prob, k_new, v_new, wl.k_pages, wl.v_pages, wl.k_scale, wl.v_scale,
                                     wl.block_table, pos, cos, sin, interleaved=False, q_inout=wl.q, status=status)

        med, p10, p90 = _time_flushed(run_rot, args.steps, args.warmup, flush)
        if int(status.item()) != 0:
            raise RuntimeError(f"rotary append flagged status {int(status.item())}")
        qb = 2 * B * spec.Hq * D * wl.q.element_size()
        nb_rot = nbytes + qb + 2 * B * (D // 2) * 4 * 2  # + q read and written, cos/sin rows read
        cases[f"config {c} rotary"] = {"workload": f"rotary append, q rotated in place (Hq={spec.Hq})",
                                       "us_median": med, "us_p10": p10, "us_p90": p90, "bytes": nb_rot,
                                       "gbs": nb_rot / med / 1e3}
        del wl
        torch.cuda.empty_cache()
    head = cases["config 3"]
    print(json.dumps({
        "metric": "fd_append_kv achieved GB/s", "value": head["gbs"], "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "us_per_call": head["us_median"], "higher_is_better": True,
        "dtype": "bf16 / e4m3", "data": "synthetic", "cases": cases, "peak": peak, "peak_source": kind,
        "config": {"workload": "append one token per sequence into the GQA-batch and FP8-batch pools",
                   "l2": "flushed before every timed call (write, then read, of 256 MB)"},
        "gpu_launches_per_call": 1}))


def bench_ex(args):
    """fd_decode_paged_ex on the GQA batch: q rows reach their cache rows
    through a permuted cache_batch_idx and attend [leftpad, seq_len) with a
    random left padding of up to a quarter of each length; against the plain
    call on the same pools (both back to back, one event pair)."""
    from split_kv_decode_paged_gb300 import workloads as W
    import split_kv_decode_paged_gb300 as fd
    from split_kv_decode_paged_gb300 import _lib
    from split_kv_decode_paged_gb300 import build as fd_build
    fd_build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = W.make_config(3, dev)
    spec = wl.spec
    B = spec.B
    g = torch.Generator().manual_seed(303)
    bidx = torch.randperm(B, generator=g).to(torch.int32)
    lens = wl.seq_lens.cpu()
    lpad = (torch.rand(B, generator=g) * (lens.float() / 4)).to(torch.int32)
    attended = (lens[bidx.long()] - lpad[bidx.long()]).clamp(min=0)
    dec = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, wl.block_table, lens)
    plan_ex = _lib.fd_plan(dec.problem, attended)
    ws = torch.zeros(max(256, plan_ex.workspace_bytes), dtype=torch.uint8, device=dev)
    out = torch.empty_like(wl.q)
    lse = torch.empty((B, spec.Hq), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bidx_d, lpad_d = bidx.to(dev), lpad.to(dev)

    def run_ex():
        _lib.fd_decode_paged_ex(plan_ex, wl.q, wl.k_pages, wl.v_pages, None, None, wl.block_table, wl.seq_lens,
                                out, lse, ws, cache_batch_idx=bidx_d, cache_leftpad=lpad_d, cache_rows=B,
                                status=status)

    def run_plain():
        dec(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens, out=out, lse=lse)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("fd_timed")
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        return a.elapsed_time(b) * 1e3 / args.steps

    us_ex, us_plain = timed(run_ex), timed(run_plain)
    if int(status.item()) != 0:
        raise RuntimeError(f"decode_paged_ex flagged status {int(status.item())}")
    dec.check()
    nbytes = W.algorithmic_bytes(spec, attended) + 8 * B  # + the index and padding arrays
    peak, kind = measured_peak()
    print(json.dumps({
        "metric": "fd_decode_paged_ex achieved HBM GB/s", "value": nbytes / us_ex / 1e3, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "us_per_call": us_ex,
        "plain_decode_us_per_call": us_plain, "plain_decode_gbs": W.algorithmic_bytes(spec, lens) / us_plain / 1e3,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic", "bytes": nbytes, "frac_of_peak":
        nbytes / us_ex / 1e3 / peak, "peak": peak, "peak_source": kind,
        "config": {"workload": "GQA batch (B=64, Hq=32, Hkv=8, D=128, bf16, 16-token pages) with a permuted "
                               "cache_batch_idx and left padding up to a quarter of each length (seed 303)",
                   "l2": "inputs > 2x L2: back to back, one event pair"},
        "gpu_launches_per_call": 1}))


def bench_multi(args):
    """Several query tokens per sequence (causal among them) on the GQA batch:
    q [64, 4, 32, 128], token i of 4 attending the cached tokens
    [0, L - 4 + i + 1), in one call that streams each sequence's K/V once,
    against four one-token decodes of the same tokens (each over its own
    prefix), both back to back."""
    from split_kv_decode_paged_gb300 import workloads as W
    import split_kv_decode_paged_gb300 as fd
    from split_kv_decode_paged_gb300 import build as fd_build
    fd_build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    q_len = 4
    wl = W.make_config(3, dev)
    spec = wl.spec
    B, Hq, D = spec.B, spec.Hq, spec.D
    g = torch.Generator(device=dev).manual_seed(404)
    qm = torch.randn((B, q_len, Hq, D), generator=g, device=dev).to(wl.q.dtype)
    dec = fd.PagedDecoder.for_pools(qm, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens.cpu())
    out = torch.empty_like(qm)
    lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=dev)
    singles = []
    for i in range(q_len):
        lens_i = (wl.seq_lens - (q_len - 1 - i)).to(torch.int32)
        d1 = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, wl.block_table, lens_i.cpu())
        singles.append((d1, qm[:, i].contiguous(), lens_i, torch.empty_like(wl.q),
                        torch.empty((B, Hq), dtype=torch.float32, device=dev)))

    def run_multi():
        dec(qm, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens, out=out, lse=lse)

    def run_singles():
        for d1, qi, li, oi, si in singles:
            d1(qi, wl.k_pages, wl.v_pages, wl.block_table, li, out=oi, lse=si)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("fd_timed")
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        return a.elapsed_time(b) * 1e3 / args.steps

    us_multi, us_singles = timed(run_multi), timed(run_singles)
    dec.check()
    for d1, *_ in singles:
        d1.check()
    lens = wl.seq_lens.cpu()
    nbytes = W.algorithmic_bytes(spec, lens) + (q_len - 1) * B * Hq * (D * 4 + 4)  # + 3 more q/out rows and lse
    peak, kind = measured_peak()
    plan = dec.plan
    print(json.dumps({
        "metric": "multi-token decode achieved HBM GB/s", "value": nbytes / us_multi / 1e3, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "us_per_call": us_multi,
        "four_single_token_decodes_us": us_singles, "speedup_vs_single_token_decodes": us_singles / us_multi,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic", "bytes": nbytes,
        "frac_of_peak": nbytes / us_multi / 1e3 / peak, "peak": peak, "peak_source": kind,
        "plan": {"q_len": plan.q_len, "num_splits": plan.num_splits, "head_subgroups": plan.head_subgroups,
                 "tile_tokens": plan.tile_tokens, "ctas_per_sm": plan.ctas_per_sm},
        "config": {"workload": "GQA batch (B=64, Hq=32, Hkv=8, D=128, bf16, 16-token pages, lengths U[512, 8192], "
                               "seed 1003) with 4 causal query tokens per sequence (q seed 404)",
                   "l2": "inputs > 2x L2: back to back, one event pair"},
        "gpu_launches_per_call": 1}))


def bench_large(args):
    """The plain decode on two large batches (1024 bf16 sequences of 256-1024
    tokens; 2048 FP8 sequences of 16-4096 tokens), timed back to back like the
    headline; the dispatch tables of such batches are built by every warp."""
    from split_kv_decode_paged_gb300 import workloads as W
    from split_kv_decode_paged_gb300 import build as fd_build
    fd_build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    peak, kind = measured_peak()
    cases = {}
    for name, spec in W.LARGE_BATCHES.items():
        wl = W.make(spec, W.LARGE_BATCH_SEED, dev)
        ms, dec = time_decode(wl, args.steps, args.warmup, None)
        us = statistics.mean(ms) * 1e3
        nbytes = W.algorithmic_bytes(spec, wl.seq_lens.cpu())
        cases[name] = {"workload": f"{spec.name}: B={spec.B}, Hq={spec.Hq}, Hkv={spec.Hkv}, D={spec.D}, {spec.kv}, "
                                   f"{spec.page_size}-token pages, lengths {spec.lens} (seed {W.LARGE_BATCH_SEED})",
                       "us_per_call": us, "bytes": nbytes, "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak,
                       "plan": {"num_splits": dec.plan.num_splits, "chunk_tokens": dec.plan.chunk_tokens,
                                "stages": dec.plan.stages, "tile_tokens": dec.plan.tile_tokens}}
        del wl, dec
        torch.cuda.empty_cache()
    head = cases["bf16 B=1024"]
    print(json.dumps({
        "metric": "decode-attention achieved HBM GB/s (large batches)", "value": head["gbs"], "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "us_per_call": head["us_per_call"],
        "higher_is_better": True, "dtype": "bf16 / e4m3", "data": "synthetic", "cases": cases, "peak": peak,
        "peak_source": kind, "config": {"workload": "large batches (value: the bf16 B=1024 case)",
                                        "l2": "inputs > 2x L2: back to back, one event pair"},
        "gpu_launches_per_call": 1}))


def bench_merge(args):
    """fd_merge_states on fp32 partial states [B=64, Hq=32, S=8, D=128] to a
    bf16 output, L2 flushed before every call."""
    import split_kv_decode_paged_gb300 as fd
    from split_kv_decode_paged_gb300 import build as fd_build
    fd_build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)
    B, Hq, S, D = 64, 32, 8, 128
    g = torch.Generator(device=dev).manual_seed(99)
    o = torch.randn((B, Hq, S, D), generator=g, device=dev)
    m = torch.randn((B, Hq, S), generator=g, device=dev) * 4
    d = torch.rand((B, Hq, S), generator=g, device=dev) * 10 + 0.5
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    from split_kv_decode_paged_gb300 import _lib

    def run():
        _lib.fd_merge_states(o, m, d, out, lse, None)

    med, p10, p90 = _time_flushed(run, args.steps, args.warmup, flush)
    nbytes = B * Hq * S * (D + 2) * 4 + B * Hq * D * 2 + 4 * B * Hq
    peak, kind = measured_peak()
    print(json.dumps({
        "metric": "fd_merge_states achieved GB/s", "value": nbytes / med / 1e3, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "us_per_call": med, "us_p10": p10, "us_p90": p90,
        "higher_is_better": True, "dtype": "f32 partials -> bf16", "data": "synthetic", "bytes": nbytes,
        "peak": peak, "peak_source": kind,
        "config": {"workload": f"merge of partial states B={B}, Hq={Hq}, S={S}, D={D}",
                   "l2": "flushed before every timed call (write, then read, of 256 MB)"},
        "gpu_launches_per_call": 1}))


# ------------------------------------------------------------ per config
CONFIG_TAGS = {1: "tiny_mha", 2: "single_seq_mha", 3: "gqa_batch", 4: "long_context", 5: "mixed_fp8"}


def spread(ms):
    """Median, p10 and p90 in microseconds of per-call times in ms."""
    srt = sorted(ms)
    return (statistics.median(srt) * 1e3, srt[len(srt) // 10] * 1e3, srt[(len(srt) * 9) // 10] * 1e3)


def per_call_spread(wl, dec, calls=50):
    """Per-call event pairs around each call, no flush in between (inputs
    larger than 2x L2: one call's K/V stream evicts the previous one's).  An
    event pair per call breaks the launch overlap of consecutive calls, so
    these times run a few microseconds above the back-to-back mean."""
    out = torch.empty_like(wl.q)
    lse = torch.empty(wl.q.shape[:2], dtype=torch.float32, device=wl.q.device)
    args = (wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    kw = dict(k_scale=wl.k_scale, v_scale=wl.v_scale, out=out, lse=lse)
    st = torch.cuda.current_stream()
    for _ in range(3):
        dec(*args, **kw)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
    for a, b in ev:
        a.record(st)
        dec(*args, **kw)
        b.record(st)
    torch.cuda.synchronize()
    dec.check()
    return [a.elapsed_time(b) for a, b in ev]


def config_entry(cfg, wl, ms, dec, peak, flushed, cpu=None, spread_ms=None, marginal_us=None):
    from split_kv_decode_paged_gb300 import workloads as W
    spec = W.CONFIGS[cfg]
    nbytes = W.algorithmic_bytes(spec, wl.seq_lens.cpu())
    us = marginal_us if (flushed and marginal_us is not None) else statistics.mean(ms) * 1e3
    gbs = nbytes / us / 1e3
    plan = dec.plan
    e = {"workload": f"{spec.name}: B={spec.B}, Hq={spec.Hq}, Hkv={spec.Hkv}, D={spec.D}, {spec.kv} K/V, "
                     f"{spec.page_size}-token pages, lengths {tuple(spec.lens)} (seed {W.config_seed(cfg)})",
         "us_per_call": us, "algorithmic_bytes": nbytes, "gbs": gbs, "frac_of_peak": gbs / peak,
         "timing": ("L2 flushed before every call; marginal time of a call in a stream of (flush, call) "
                    "pairs: an event pair around 50 pairs minus one around 50 flushes (median of 5)"
                    if flushed and marginal_us is not None else
                    "L2 flushed before every call, per-call event pairs (mean)" if flushed else
                    "back to back, one event pair (mean)"),
         "traffic": profiled_traffic(CONFIG_TAGS[cfg]),
         "plan": {"num_splits": plan.num_splits, "chunk_tokens": plan.chunk_tokens, "tile_tokens": plan.tile_tokens,
                  "stages": plan.stages, "grid_ctas": plan.grid_ctas, "work_items": plan.work_items_hint}}
    sp = spread(ms if flushed else (spread_ms or []) or ms)
    e["us_median"], e["us_p10"], e["us_p90"] = sp
    if not flushed:
        e["spread_timing"] = "per-call event pairs, no flush (inputs > 2x L2)"
    elif marginal_us is not None:
        e["us_per_call_event_pair"] = statistics.mean(ms) * 1e3
        e["spread_timing"] = ("per-call event pairs around each flushed call (they add the launch latency "
                              "that the marginal time leaves out)")
    if cpu is not None:
        e["oracle"] = {"us_per_call": cpu["us_per_call"], "gbs": cpu["value"], "cores": cpu["cores"],
                       "sample": cpu["sample"]}
    return e


def per_config_block(args, dev, peak, flush_buf, flush_bytes, headline):
    """Every workload at one GPU, with the fp64 oracle timed on the host cores
    beside it (a bounded sample of each, scaled to one call)."""
    from split_kv_decode_paged_gb300 import workloads as W
    per = {}
    for c in (1, 2, 3, 4, 5):
        if c == args.config:
            wl, ms, dec, sp = headline
        else:
            wl = W.make_config(c, dev)
            big = W.algorithmic_bytes(W.CONFIGS[c], wl.seq_lens.cpu()) > flush_bytes
            ms, dec = time_decode(wl, 100 if big else 200, args.warmup, None if big else flush_buf)
            sp = per_call_spread(wl, dec) if big else None
        big = W.algorithmic_bytes(W.CONFIGS[c], wl.seq_lens.cpu()) > flush_bytes
        marginal = None if big else flushed_marginal_us(wl, dec, flush_buf)
        cpu = None if args.no_cpu_baseline else cpu_baseline(wl.to("cpu"), target_s=args.per_config_cpu_seconds)
        per[str(c)] = config_entry(c, wl, ms, dec, peak, not big, cpu, sp, marginal)
        if c != args.config:
            del wl, dec
            torch.cuda.empty_cache()
    return per


# ------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=HEADLINE_CONFIG)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config block (every workload, with the oracle timed beside it)")
    ap.add_argument("--all-configs", action="store_true", help=argparse.SUPPRESS)  # the default now
    ap.add_argument("--per-config-cpu-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "cascade", "append", "merge", "ex", "large", "multi"],
                    help="cascade: shared-prefix batch, cascade vs plain decode; append: fd_append_kv (plain "
                         "and rotary); merge: fd_merge_states; ex: fd_decode_paged_ex with cache_batch_idx "
                         "and left padding; large: two large batches; multi: 4 causal query tokens per "
                         "sequence on the GQA batch")
    ap.add_argument("--quick", action="store_true",
                    help="only the timed decode calls (no warm-L2/graph/e2e extras, no CPU baseline)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    if args.workload != "decode":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference",
                              "unavailable": f"the {args.workload} workload is measured on the GPU path only"}))
            return
        {"cascade": bench_cascade, "append": bench_append, "merge": bench_merge, "ex": bench_ex,
         "large": bench_large, "multi": bench_multi}[args.workload](args)
        return
    from split_kv_decode_paged_gb300 import workloads as W
    ws, rank, local = dist_env()
    spec = W.CONFIGS[args.config]
    tag = CONFIG_TAGS[args.config]
    config = {"workload": f"{spec.name} (config {args.config})", "B": spec.B, "Hq": spec.Hq, "Hkv": spec.Hkv,
              "D": spec.D, "page_size": spec.page_size, "kv_dtype": spec.kv, "q_dtype": spec.q,
              "lengths": list(spec.lens), "l2": "flushed before every timed call (2x L2 write)"}

    if args.impl == "reference":
        if rank != 0:
            return
        config["l2"] = "not applicable (host cores)"
        wl = W.make_config(args.config, "cpu", seed=W.config_seed(args.config))
        per, cb = [], None
        per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
        for i in range(args.warmup + args.steps):
            cb = cpu_baseline(wl, target_s=per_step, seed=i)
            if i >= args.warmup:
                per.append(cb["us_per_call"])
        us = statistics.median(per)
        bytes_call = W.algorithmic_bytes(spec, wl.seq_lens)
        gbs = bytes_call / (us * 1e-6) / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "us_per_call": us,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cb["cores"], "kind": "oracle",
                                 "sample": f"each step: {cb['sample']}"},
                "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    from split_kv_decode_paged_gb300 import build as fd_build
    if rank == 0 or ws == 1:
        fd_build.build()
    if ws > 1:
        torch.distributed.barrier()
    wl = W.make_config(args.config, dev, seed=W.config_seed(args.config) + 7919 * rank)
    bytes_call = W.algorithmic_bytes(spec, wl.seq_lens.cpu())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # GB300 reports the L2 of one die; flush with at least 2x the whole chip's 126 MB.
    flush_bytes = max(2 * l2, 256 << 20)
    flush_buf = torch.empty(flush_bytes // 4, dtype=torch.float32, device=dev)
    # Inputs larger than 2x L2 are timed back to back between one event pair
    # (no flush: one call's K/V stream evicts the previous one's); smaller
    # inputs get an L2 flush (a write, then read, of 2x L2) before every timed
    # call, outside that call's event pair.
    big = bytes_call > flush_bytes
    flush = None if big else flush_buf
    config["l2"] = (f"inputs {bytes_call / 1e9:.2f} GB > {flush_bytes / 1e6:.0f} MB (2x L2): timed back to back, no flush, one event pair around all steps"
                    if big else f"L2 flushed before every timed call (write, then read, of {flush_bytes / 1e6:.0f} MB)")

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(index=dev.index) as clk:
        t0 = time.perf_counter()
        ms, dec = time_decode(wl, args.steps, args.warmup, flush)
        wall = time.perf_counter() - t0
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    total_ms = sum(ms)
    elapsed_s, bytes_all = aggregate(total_ms / 1e3, bytes_call * args.steps)
    value = bytes_all / elapsed_s / 1e9
    peak, peak_kind = measured_peak()
    achieved = bytes_call / (total_ms / args.steps * 1e-3) / 1e9
    ms_flushed = None
    if big and not args.quick:
        ms_f, _ = time_decode(wl, min(args.steps, 50), 3, flush_buf)
        ms_flushed = sum(ms_f) / len(ms_f)
    spread_ms = per_call_spread(wl, dec) if big and not args.quick else None
    if args.quick:
        warm_ms = graph_ms = float("nan")
        e2e_s, h2d, d2h = float("nan"), 0, 0
        args.no_cpu_baseline = True
        args.no_per_config = True
    else:
        warm_ms, graph_ms = time_warm_and_graph(wl, dec)
        e2e_s, h2d, d2h = time_e2e(wl, dec, max(10, args.steps // 2))
    plan = dec.plan
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "us_per_call": total_ms / args.steps * 1e3,
        # per-call spread: the flushed calls' own event pairs, or (inputs
        # larger than 2x L2) a second pass with an event pair around each call
        **dict(zip(("us_median", "us_p10", "us_p90"),
                   spread(ms) if not big else (spread(spread_ms) if spread_ms else (None, None, None)))),
        "us_spread_timing": ("per-call event pairs after an L2 flush" if not big else
                             "second pass: per-call event pairs, no flush (inputs > 2x L2); the event pair per "
                             "call breaks the launch overlap, so these run above the back-to-back mean"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "f16": "f16", "e4m3": "e4m3 (f16 MMA, fp32 accumulate)"}[spec.kv],
        "data": "synthetic (seeded generator: split_kv_decode_paged_gb300/workloads.py)", "config": config,
        "algorithmic_bytes_per_call": bytes_call,
        "plan": {"num_splits": plan.num_splits, "chunk_tokens": plan.chunk_tokens, "grid_ctas": plan.grid_ctas,
                 "stages": plan.stages, "work_items": plan.work_items_hint, "fuse_merge": plan.fuse_merge},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(tag),
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json burst copy)"},
        "us_per_call_after_l2_flush": None if ms_flushed is None else ms_flushed * 1e3,
        "warm_l2_us_per_call": None if args.quick else warm_ms * 1e3,
        "graph_replay_us_per_call": None if args.quick else graph_ms * 1e3,
        "e2e": None if args.quick else {"value": bytes_call / e2e_s / 1e9, "unit": "GB/s",
                                        "us_per_step": e2e_s * 1e6, "h2d_bytes_per_step": h2d,
                                        "d2h_bytes_per_step": d2h,
                                        "path": "HostPipeline: per step one pinned H2D copy of q + block table "
                                                "+ seq_lens (fd_host_copy_in, on a copy stream, overlapping the "
                                                "previous step's decode; two block sets in turn), then the decode "
                                                "(fd_decode_paged_staged), whose kernel stores out + lse straight "
                                                "into the mapped pinned host block (d2h bytes cross during the "
                                                "kernel, no separate copy)"},
        "gpu_launches": args.steps * (1 if plan.fuse_merge or plan.num_splits == 1 else 2),
        "clocks": clk.summary(), "wall_s_timed_region": wall,
    }
    if ws == 1 and not args.no_per_config:
        line["per_config"] = per_config_block(args, dev, peak, flush_buf, flush_bytes, (wl, ms, dec, spread_ms))
    if rank == 0 and not args.no_cpu_baseline:
        wl_cpu = wl.to("cpu")
        line["cpu_baseline"] = cpu_baseline(wl_cpu, target_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
