"""Benchmark of CSR-indexed sparse/paged attention on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--rows ...]

One JSON line on rank 0. The headline workload is the paged GQA batch decode (batch 64,
32 query / 8 kv heads, head_dim 128, bf16, page_size 16, kv lengths U[512, 4096], pages
randomly permuted in a shared pool): one step = bskv_run_decode over the whole batch, one
kernel launch that computes the attention and merges the split-KV partial states (the
plan is made once, as a serving engine does per decode step, and timed apart). The metric is the KV bytes the method must read per second.
The K timed steps run back to back between two CUDA events on the launching stream; a second
pass with an event pair around each step gives the per-launch distribution.
The same run measures the other rows of the hot path on their own workloads (BSR prefill,
tiny BSR, the MLA prologue and sparse FP8 decode, long-context split-KV decode) and
reports them under "rows". Inputs are synthetic (seeded) and resident in HBM before the
timed region; the headline's KV (about 0.6 GB) is larger than L2, the smaller rows flush
L2 between timed iterations (a 512 MiB write, then a 256 MiB read so that the write-back
of the flushed lines is not charged to the timed kernel).

--impl reference times the float64 CPU oracle (the only reference implementation of
this method here) on the host cores, on a bounded sample of the same workload.
With N > 1 (torchrun) every rank runs an independent replica (weak scaling, no
collective on the data path); value = bytes of all ranks / max-over-ranks time.
"""

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention KV GB/s (decode) and TFLOPS (BSR/MLA) as % of 1×GB300 roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
HEADLINE_WORKLOAD = ("paged_decode: batch 64, 32/8 heads, head_dim 128, bf16, page_size 16, "
                     "kv len U[512,4096], pages permuted in a shared pool")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    try:
        with open(PEAKS_FILE) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


# ---------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------------------

def dist_setup(n_gpus):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend)
        return dist, dist.get_rank(), ws
    return None, 0, 1


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x):
    if dist is None:
        return x
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x):
    if dist is None:
        return x
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
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
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        under = [x for x in sm if mx and x > 0.3 * mx] or sm
        return {"sm_mhz": statistics.median(under) if under else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------------------

_flush_buf = None
_clean_buf = None


def flush_l2():
    """Write 512 MiB (4x the 129 MB L2), then read 256 MiB of another buffer: the read
    evicts the written lines, so their write-back to HBM happens here and not inside the
    timed kernel that follows."""
    global _flush_buf, _clean_buf
    if _flush_buf is None:
        _flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        _clean_buf = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")
    _flush_buf.fill_(1)
    _clean_buf.sum()


def time_iters(fn, iters, warmup, flush=False):
    """Per-iteration CUDA-event times (ms) on the current stream; L2 flushed in between."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = []
    st = torch.cuda.current_stream()
    for _ in range(iters):
        if flush:
            flush_l2()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def summary(ms):
    return {"median_us": 1e3 * statistics.median(ms), "mean_us": 1e3 * statistics.mean(ms),
            "std_us": 1e3 * (statistics.pstdev(ms) if len(ms) > 1 else 0.0), "n": len(ms)}


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_sparse_kv_gb300", "csrc", n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(summary_name, kernel_sources):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel source; else None."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != source_sha(*kernel_sources):
        return None
    return float(t.group(1))


def measure_tensor_peaks(sizes=(8192, 16384), iters=10):
    """Dense tensor-core peaks of this GPU, measured in this run with library GEMMs
    (n x n x n, 2 n^3 flops, best of `iters` CUDA-event timings after warm-up, best over the
    sizes): bf16 and fp16 through torch.matmul, E4M3 x E4M3 -> bf16 through torch._scaled_mm
    (per-tensor scales). These are the denominators of the fp16 (BSR) and FP8 (MLA) fractions;
    the bf16 figure is reported beside MEASURED_PEAKS.json's."""
    res = {"how": "2 n^3 / best of %d CUDA-event times after 3 warm-up calls, best of n in %s"
                  % (iters, list(sizes))}
    for n in sizes:
        for k, v in _measure_tensor_peaks_n(n, iters).items():
            if v is None or isinstance(v, str):
                res.setdefault(k, v)
            else:
                res[k] = max(v, res.get(k) or 0.0)
    torch.cuda.empty_cache()
    return res


def _measure_tensor_peaks_n(n, iters):
    res = {}
    g = torch.Generator(device="cuda").manual_seed(5)

    def best(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(iters):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return 2.0 * n ** 3 / (min(ts) * 1e-3) / 1e12

    for name, dt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
        try:
            x = torch.randn((n, n), device="cuda", generator=g).to(dt)
            y = torch.randn((n, n), device="cuda", generator=g).to(dt)
            res[name + "_tflops"] = best(lambda: torch.matmul(x, y))
            del x, y
        except Exception as e:  # noqa: BLE001
            res[name + "_tflops"] = None
            res[name + "_error"] = str(e)[:200]
    try:
        x = torch.randn((n, n), device="cuda", generator=g).to(torch.float8_e4m3fn)
        yt = torch.randn((n, n), device="cuda", generator=g).to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device="cuda")
        res["fp8_e4m3_tflops"] = best(
            lambda: torch._scaled_mm(x, yt.t(), scale_a=one, scale_b=one,
                                     out_dtype=torch.bfloat16))
        del x, yt
    except Exception as e:  # noqa: BLE001
        res["fp8_e4m3_tflops"] = None
        res["fp8_e4m3_error"] = str(e)[:200]
    return res


def tensor_peak(peaks, tp, kind):
    """(denominator, source) of a tensor-core fraction: fp16 and fp8 from this run's
    measurement, bf16 from MEASURED_PEAKS.json (burst)."""
    if kind == "bf16":
        return peaks["bf16_tflops"], "bf16 dense burst (MEASURED_PEAKS.json)"
    if kind == "fp16" and tp and tp.get("fp16_tflops"):
        # fp16 and bf16 share one nominal rate: the larger measured figure is the denominator
        pk = max(tp["fp16_tflops"], tp.get("bf16_tflops") or 0.0, peaks["bf16_tflops"])
        return pk, ("max of the fp16 GEMM measured in this run (%.0f TF/s) and the bf16 burst "
                    "figures (same nominal rate)" % tp["fp16_tflops"])
    key = {"fp16": "fp16_tflops", "fp8": "fp8_e4m3_tflops"}[kind]
    if tp and tp.get(key):
        return tp[key], "%s dense, measured in this run (%s)" % (kind, tp["how"])
    ratio = 2.0 if kind == "fp8" else 1.0
    return ratio * peaks["bf16_tflops"], "%s = %g x bf16 burst (measurement failed: nominal ratio)" % (kind, ratio)


# ---------------------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------------------

TP = None  # tensor peaks measured in this run (rank 0), set by main()


def variant_name(plan):
    """Kernel that serves a BSR-family plan (metadata header word 15)."""
    return {0: "general (mma.sync)", 1: "tcgen05", 2: "general (mma.sync)",
            3: "general (mma.sync)", 4: "tcgen05", 5: "tcgen05"}.get(plan.metadata()[15], "?")


def decode_kv_bytes(d):
    return int(d["kv_lens"].to(torch.int64).sum()) * d["num_kv_heads"] * d["head_dim"] * 2 * 2


def decode_launches(meta):
    """Kernels one bskv_run_decode launches for a plan (metadata header: merges at word 6,
    grid at 13, merge-section offset at 10): the attention kernel, plus the merge kernel
    when no worker exists or some unit has more than 8 pieces."""
    nm, grid, off = meta[6], meta[13], meta[10]
    most = max([meta[off + 3 * i + 2] for i in range(nm)] or [0])
    return (1 if grid > 0 else 0) + (1 if nm > 0 and (grid == 0 or most > 8) else 0)


def bench_decode(bskv, synth, name, steps, warmup, dist, sampler=None, headline=False,
                 **over):
    """Paged decode (+ merge) on one of the decode workloads."""
    d = synth.make(name, device="cuda", **over)
    # host planning time: the median of 5 calls after a first one (which pays one-time costs)
    plan_times = []
    for _ in range(6):
        t0 = time.perf_counter()
        plan = bskv.bskv_plan_decode(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"],
                                     d["num_pages"], d["page_size"], d["num_qo_heads"],
                                     d["num_kv_heads"], d["head_dim"], torch.bfloat16)
        plan_times.append(1e6 * (time.perf_counter() - t0))
    plan_us = statistics.median(plan_times[1:])
    plan.upload("cuda")
    q, kv = d["q"], d["kv_cache"]
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    meta = plan.metadata()

    def step(ev=None):
        # the attention kernel, which merges split units itself unless they have many pieces
        if ev is not None:
            ev[0].record()
        bskv.bskv_run_decode(plan, q, kv, out=out, lse=lse)
        if ev is not None:
            ev[1].record()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(dist)
    # timed region: the steps back to back between two events (no event between steps)
    t_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    if sampler:
        sampler.start()
    torch.cuda.synchronize()
    barrier(dist)
    t_ev[0].record()
    for i in range(steps):
        step()
    t_ev[1].record()
    torch.cuda.synchronize()
    barrier(dist)
    clocks = sampler.stop() if sampler else None
    total_ms = t_ev[0].elapsed_time(t_ev[1])
    # per-launch distribution: the same steps again with an event pair around each one
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize()
    kern_ms = [e[0].elapsed_time(e[1]) for e in evs]
    nbytes = decode_kv_bytes(d)
    # the same step captured once in a CUDA graph and replayed back to back (how a serving
    # loop issues it); reported beside the eager numbers
    graph_ms = None
    if headline:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        graph_ms = a.elapsed_time(b) / steps
        del g
    res = dict(workload=name, kv_bytes=nbytes, plan_us=plan_us, total_ms=total_ms,
               ms_per_step=total_ms / steps, decode_kernel=summary(kern_ms),
               variant="page-major (all kv heads of a page per CTA)" if meta[15] == 1
               else "per kv head (one worker per warp)",
               split_units=meta[6], launches_per_step=decode_launches(meta), clocks=clocks,
               graph_ms_per_step=graph_ms)
    res["gbs_step"] = nbytes / (res["ms_per_step"] * 1e-3) / 1e9
    res["gbs_kernel"] = nbytes / (statistics.mean(kern_ms) * 1e-3) / 1e9
    del d, kv, q
    return res, plan


def bench_decode_e2e(bskv, synth, steps, warmup):
    """Same workload through the public API with host buffers: pinned H2D of q, the KV
    cache and the page table, plan + upload, decode + merge, D2H of the output."""
    d = synth.make("paged_decode", device="cpu")
    hq, hkv = d["q"].pin_memory(), d["kv_cache"].pin_memory()
    hidx = [d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"]]
    dq = torch.empty_like(hq, device="cuda")
    dkv = torch.empty_like(hkv, device="cuda")
    hout = torch.empty_like(hq).pin_memory()
    plan = bskv.bskv_plan_decode(*hidx, d["num_pages"], d["page_size"], d["num_qo_heads"],
                                 d["num_kv_heads"], d["head_dim"], torch.bfloat16)
    plan.upload("cuda")
    int_ws, float_ws = plan.int_ws, plan.float_ws

    def step():
        dq.copy_(hq, non_blocking=True)
        dkv.copy_(hkv, non_blocking=True)
        p = bskv.bskv_plan_decode(*hidx, d["num_pages"], d["page_size"], d["num_qo_heads"],
                                  d["num_kv_heads"], d["head_dim"], torch.bfloat16)
        p.upload("cuda", int_ws=int_ws, float_ws=float_ws)
        dout = bskv.bskv_run_decode(p, dq, dkv)
        hout.copy_(dout, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return p

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    ms = 1e3 * (time.perf_counter() - t0) / steps
    h2d = hq.numel() * 2 + hkv.numel() * 2 + sum(x.numel() * 4 for x in hidx) + \
        plan.workspace_sizes()[0]
    d2h = hout.numel() * 2
    nbytes = decode_kv_bytes(d)
    return {"value": nbytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def bench_split(bskv, synth, steps, warmup, peaks):
    res, _ = bench_decode(bskv, synth, "split_decode", steps, warmup, None)
    res["frac_step"] = res["gbs_step"] / peaks["hbm_gbs"]
    res["frac_kernel"] = res["gbs_kernel"] / peaks["hbm_gbs"]
    res.pop("clocks", None)
    return res


def bsr_flops(d):
    """4 * D * Hq * visible (query, key) pairs, causal-exact."""
    R, C, M, N = d["R"], d["C"], d["M"], d["N"]
    indptr, indices = d["indptr"].tolist(), d["indices"].tolist()
    pairs = 0
    for i in range(len(indptr) - 1):
        r0, r1 = i * R, min(M, (i + 1) * R)
        for j in indices[indptr[i]:indptr[i + 1]]:
            c0, c1 = j * C, (j + 1) * C
            if not d["causal"]:
                pairs += (r1 - r0) * (c1 - c0)
            else:
                for r in range(r0, r1):
                    lim = r + (N - M)
                    pairs += max(0, min(c1, lim + 1) - c0)
    return 4 * d["head_dim"] * d["num_qo_heads"] * pairs


def bench_bsr(bskv, synth, name, steps, warmup, peaks, flush):
    d = synth.make(name, device="cuda")
    plan = bskv.bskv_plan_bsr(d["indptr"], d["indices"], d["M"], d["N"], d["R"], d["C"],
                              d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                              causal=d["causal"], dtype=torch.float16)
    plan.upload("cuda")
    out = torch.empty_like(d["q"])
    fn = lambda: bskv.bskv_run_bsr(plan, d["q"], d["k"], d["v"], out=out)  # noqa: E731
    ms = time_iters(fn, steps, warmup, flush=flush)
    fl = bsr_flops(d)
    med = statistics.median(ms)
    tf = fl / (med * 1e-3) / 1e12
    variant = plan.metadata()[15]
    pk, src = tensor_peak(peaks, TP, "fp16")
    extra = {}
    if name == "bsr_tiny":
        # launch-bound: the eager time above includes the host's launch latency; 20 runs
        # captured in one CUDA graph give the device-side time per run
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(20):
                fn()
        g.replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            reps.append(a.elapsed_time(b) * 1e3 / 20)
        del g
        extra["graph_us_per_run"] = statistics.median(reps)
    return dict(workload=name, flops=fl, kernel="tcgen05" if variant == 1 else "general",
                **summary(ms), tflops=tf, frac=tf / pk, peak=src, peak_tflops=pk,
                frac_of_bf16_burst=tf / peaks["bf16_tflops"], **extra)


def bench_bsr_masked(bskv, synth, steps, warmup, peaks):
    """The BSR prefill workload expressed as a per-block token mask (diagonal blocks carry
    the causal pattern, the listed off-diagonal blocks are full): the same visible pairs as
    the causal run, through the masked entry point."""
    d = synth.make("bsr_prefill", device="cuda")
    R, C = d["R"], d["C"]
    ip, ix = d["indptr"].numpy(), d["indices"].numpy()
    nnz = int(ip[-1])
    tri = np.tril(np.ones((R, C), bool))
    bm = np.ones((nnz, R, C), bool)
    for a in range(len(ip) - 1):
        for e in range(int(ip[a]), int(ip[a + 1])):
            if int(ix[e]) == a:
                bm[e] = tri
    packed = torch.from_numpy(np.packbits(bm.reshape(-1), bitorder="little").copy()).cuda()
    plan = bskv.bskv_plan_bsr_masked(d["indptr"], d["indices"], d["M"], d["N"], R, C,
                                     d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                                     dtype=torch.float16)
    plan.upload("cuda")
    out = torch.empty_like(d["q"])
    fn = lambda: bskv.bskv_run_bsr_masked(plan, d["q"], d["k"], d["v"], packed, out=out)  # noqa
    ms = time_iters(fn, steps, warmup, flush=True)
    fl = bsr_flops(d)
    tf = fl / (statistics.median(ms) * 1e-3) / 1e12
    pk, src = tensor_peak(peaks, TP, "fp16")
    return dict(workload="bsr_prefill as a token mask (causal pattern in the diagonal blocks)",
                flops=fl, kernel="tcgen05" if plan.metadata()[15] == 1 else "general",
                **summary(ms), tflops=tf, frac=tf / pk, peak=src, peak_tflops=pk,
                mask_bytes=int(packed.numel()))


def variable_block_flops(d):
    """4 * head_dim * (query heads per kv head) * visible (query, key) pairs, over kv heads."""
    bm = np.asarray(d["block_mask_map"], bool)
    rs = np.asarray(d["block_row_sz"], np.int64)
    cs = np.asarray(d["block_col_sz"], np.int64)
    H, MB, NB = bm.shape
    shift = d["kv_len"] - d["qo_len"]
    pairs = 0
    for h in range(H):
        r0 = np.concatenate([[0], np.cumsum(rs[h])])
        c0 = np.concatenate([[0], np.cumsum(cs[h])])
        for a in range(MB):
            rows = np.arange(r0[a], r0[a + 1])
            for c in np.nonzero(bm[h, a])[0]:
                if d["causal"]:
                    pairs += int(np.clip(np.minimum(c0[c + 1], rows + shift + 1) - c0[c], 0,
                                         c0[c + 1] - c0[c]).sum())
                else:
                    pairs += len(rows) * int(c0[c + 1] - c0[c])
    g = d["num_qo_heads"] // d["num_kv_heads"]
    return 4.0 * d["head_dim"] * g * pairs


def bench_bsr_variable(bskv, synth, steps, warmup, peaks):
    """Variable-block sparse attention: 16384 query and key tokens, 32/8 heads, head_dim 128,
    fp16; every kv head cuts them into 128 x 128 blocks of its own random sizes and keeps
    10 % of them, causal."""
    d = synth.make("bsr_variable", device="cuda")
    plan = bskv.bskv_plan_bsr_variable(d["block_mask_map"], d["block_row_sz"], d["block_col_sz"],
                                       d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                                       causal=d["causal"], dtype=torch.float16)
    plan.upload("cuda")
    out = torch.empty_like(d["q"])
    fn = lambda: bskv.bskv_run_bsr_variable(plan, d["q"], d["k"], d["v"], out=out)  # noqa
    ms = time_iters(fn, steps, warmup, flush=True)
    fl = variable_block_flops(d)
    tf = fl / (statistics.median(ms) * 1e-3) / 1e12
    pk, src = tensor_peak(peaks, TP, "fp16")
    return dict(workload="bsr_variable: 16384 tokens, 32/8 heads, D 128, fp16, 128 x 128 "
                         "blocks of random sizes per kv head, 10 % kept, causal (L2 flushed)",
                flops=fl, kernel=variant_name(plan), **summary(ms), tflops=tf,
                frac=tf / pk, peak=src, peak_tflops=pk)


def bench_prefill_paged(bskv, synth, steps, warmup, peaks):
    """Batch prefill over the paged cache: 16 requests of 2048-8192 tokens whose last 1024
    tokens are the queries (causal, bottom-right), 32/8 heads, head_dim 128, bf16, page 16."""
    d = synth.make("prefill_paged", device="cuda")
    plan = bskv.bskv_plan_prefill_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                        d["kv_last_page_len"], d["num_pages"], d["page_size"],
                                        d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                                        causal=True, dtype=torch.bfloat16)
    plan.upload("cuda")
    out = torch.empty_like(d["q"])
    fn = lambda: bskv.bskv_run_prefill_paged(plan, d["q"], d["kv_cache"], out=out)  # noqa
    ms = time_iters(fn, steps, warmup, flush=True)
    pairs = 0
    for L, nq in zip(d["kv_lens"].tolist(), d["qo_lens"].tolist()):
        pairs += sum(min(L, t + L - nq + 1) for t in range(nq))
    fl = 4.0 * d["head_dim"] * d["num_qo_heads"] * pairs
    tf = fl / (statistics.median(ms) * 1e-3) / 1e12
    pk, src = tensor_peak(peaks, TP, "bf16")
    return dict(workload="prefill_paged: 16 requests, L ~ U[2048,8192], 1024 new tokens each, "
                         "32/8 heads, D 128, bf16, page 16, causal (L2 flushed)",
                flops=fl, kernel=variant_name(plan), **summary(ms), tflops=tf,
                frac=tf / pk, peak=src, peak_tflops=pk)


def bench_mla(bskv, synth, steps, warmup, peaks):
    m = synth.make("mla_decode", device="cuda")
    B, H, K = m["batch"], m["heads"], m["top_k"]
    query = torch.empty((B, 1, H, 576), dtype=torch.uint8, device="cuda")
    pool = torch.empty((m["pool_rows"], 576), dtype=torch.uint8, device="cuda")

    pos_k, pos_q = m["pos_k"].cuda(), m["pos_q"].cuda()

    def prologue_k():
        bskv.bskv_rope_quantize_fp8(None, m["k_rope"], None, m["k_nope"], m["cos_sin"],
                                    None, True, k_rope_out=pool[:, 512:],
                                    k_nope_out=pool[:, :512], pos_ids_k=pos_k)

    def prologue_q():
        bskv.bskv_rope_quantize_fp8(m["q_rope"], None, m["q_nope"], None, m["cos_sin"],
                                    pos_q, True, q_rope_out=query[:, 0, :, 512:],
                                    q_nope_out=query[:, 0, :, :512])

    def prologue_qk():
        # both groups in one call (one launch over the query and key rows)
        bskv.bskv_rope_quantize_fp8(m["q_rope"], m["k_rope"], m["q_nope"], m["k_nope"],
                                    m["cos_sin"], pos_q, True, q_rope_out=query[:, 0, :, 512:],
                                    q_nope_out=query[:, 0, :, :512], k_rope_out=pool[:, 512:],
                                    k_nope_out=pool[:, :512], pos_ids_k=pos_k)

    pk = time_iters(prologue_k, steps, warmup, flush=True)
    pq = time_iters(prologue_q, steps, warmup, flush=True)
    pqk = time_iters(prologue_qk, steps, warmup, flush=True)
    kbytes = m["pool_rows"] * (1152 + 576 + 256)
    qbytes = B * H * (1152 + 576) + B * 256
    res = dict(workload="mla_decode",
               prologue_k=dict(**summary(pk), bytes=kbytes,
                               gbs=kbytes / (statistics.median(pk) * 1e-3) / 1e9),
               prologue_q=dict(**summary(pq), bytes=qbytes,
                               gbs=qbytes / (statistics.median(pq) * 1e-3) / 1e9),
               prologue_qk=dict(**summary(pqk), bytes=kbytes + qbytes, launches=1,
                                gbs=(kbytes + qbytes) / (statistics.median(pqk) * 1e-3) / 1e9))
    for k in ("prologue_k", "prologue_q", "prologue_qk"):
        res[k]["frac"] = res[k]["gbs"] / peaks["hbm_gbs"]
    try:
        plan = bskv.bskv_plan_mla_sparse(m["seq_lens"], B, 1, H, K)
        plan.upload("cuda")
        idx = m["indices"].cuda()
        out = torch.empty((B, 1, H, 512), dtype=torch.bfloat16, device="cuda")
        scale = 1.0 / math.sqrt(576)
        fn = lambda: bskv.bskv_run_mla_sparse(plan, query, pool, idx, scale, 1.0, out=out)  # noqa
        for flush in (False, True):
            ms = time_iters(fn, steps, warmup, flush=flush)
            fl = 2.0 * H * int(m["seq_lens"].sum()) * (576 + 512)
            tf = fl / (statistics.median(ms) * 1e-3) / 1e12
            fp8_peak, src = tensor_peak(peaks, TP, "fp8")
            res["decode_l2_flushed" if flush else "decode_l2_warm"] = dict(
                **summary(ms), flops=fl, tflops=tf, frac=tf / fp8_peak, peak=src,
                peak_tflops=fp8_peak)
    except bskv.BskvError as e:
        res["decode"] = "not available: %s" % e.status
    return res


def bench_mla_paged(bskv, synth, steps, warmup, peaks):
    """Dense paged MLA decode: 128 requests x 128 heads over all of their 2048-8192 tokens
    (page_size 64, pages permuted in a pool). Each token row is read once per step, so the
    row reads (~0.4 GB, larger than L2) and the FP8 contraction are both reported."""
    d = synth.make("mla_paged", device="cuda")
    B, H = d["batch"], d["heads"]
    plan = bskv.bskv_plan_mla_paged(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"], B,
                                    d["num_pages"], d["page_size"], H)
    plan.upload("cuda")
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    scale = 1.0 / math.sqrt(576)
    fn = lambda: bskv.bskv_run_mla_paged(plan, d["query"], d["kv_pages"], scale, 1.0, out=out)  # noqa
    ms = time_iters(fn, steps, warmup, flush=True)
    tokens = int(d["lens"].sum())
    fl = 2.0 * H * tokens * (576 + 512)
    nbytes = tokens * 576 + B * H * (576 + 1024)
    med = statistics.median(ms) * 1e-3
    tf = fl / med / 1e12
    gbs = nbytes / med / 1e9
    fp8_peak, src = tensor_peak(peaks, TP, "fp8")
    return dict(workload="mla_paged: batch 128, 128 heads, E4M3 rows of 576, page_size 64, "
                         "kv len U[2048,8192], pages permuted in a pool (L2 flushed)",
                **summary(ms), flops=fl, tflops=tf, frac=tf / fp8_peak, peak=src,
                peak_tflops=fp8_peak,
                bytes=nbytes, gbs=gbs, hbm_frac=gbs / peaks["hbm_gbs"],
                launches_per_step=1 + (1 if plan.metadata()[6] > 0 else 0))


def bench_mla_append(bskv, synth, steps, warmup, peaks):
    """RoPE + FP8 of 128 requests x 512 new key rows appended into the page-64 latent cache
    (an HBM stream: 1152 bytes in, 576 out and 256 of cos/sin per row)."""
    d = synth.make("mla_append", device="cuda")
    cache = d["kv_pages"]
    args = [d["k_rope"], d["k_nope"], d["pos_k"].cuda(), d["cos_sin"], d["batch_indices"].cuda(),
            d["positions"].cuda(), d["kv_indptr"].cuda(), d["kv_indices"].cuda(), cache]
    fn = lambda: bskv.bskv_rope_quantize_fp8_append_paged(*args)  # noqa
    ms = time_iters(fn, steps, warmup, flush=True)
    rows = d["k_rope"].shape[0]
    nbytes = rows * (1152 + 576 + 256)
    gbs = nbytes / (statistics.median(ms) * 1e-3) / 1e9
    return dict(workload="mla_append: 128 requests x 512 new rows (65536) appended to the page-64 "
                         "latent cache (L2 flushed)",
                **summary(ms), bytes=nbytes, gbs=gbs, frac=gbs / peaks["hbm_gbs"],
                launches_per_step=1)


# ---------------------------------------------------------------------------------------
# CPU baseline: the float64 oracle on the host cores, on a bounded sample
# ---------------------------------------------------------------------------------------

def oracle_decode_sample(synth, budget_s=12.0):
    from oracle import attention as att
    d = synth.make("paged_decode", device="cpu")
    qb = d["q"].view(torch.int16).numpy().view(np.uint16)
    kvb = d["kv_cache"].view(torch.int16).numpy().view(np.uint16)
    ip, ix, lp = d["kv_indptr"].numpy(), d["kv_indices"].numpy(), d["kv_last_page_len"].numpy()
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    while done < d["batch"] and (time.perf_counter() - t0 < budget_s or done < 2):
        att.paged_decode(qb, kvb, "bf16", ip, ix, lp, d["page_size"], d["sm_scale"], [done])
        nbytes += int(d["kv_lens"][done]) * d["num_kv_heads"] * d["head_dim"] * 4
        done += 1
    el = time.perf_counter() - t0
    try:
        import threadpoolctl
        threads = max((i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()), default=1)
    except Exception:  # noqa: BLE001
        threads = os.cpu_count()
    return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": int(threads), "kind": "oracle",
            "sample": "%d of 64 requests of the paged decode workload (float64 numpy), %.1f s"
                      % (done, el), "seconds": el}


# ---------------------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------------------

def run_reference(args):
    """The oracle as the reference arm: host cores, bounded samples of the same workload."""
    dist, rank, ws = dist_setup(args.gpus)
    if rank != 0:
        return
    import synth
    vals = []
    for _ in range(args.warmup):
        oracle_decode_sample(synth, budget_s=2.0)
    for _ in range(args.steps):
        vals.append(oracle_decode_sample(synth, budget_s=10.0 / max(args.steps, 1)))
    v = statistics.mean(x["value"] for x in vals)
    cb = dict(vals[-1])
    cb["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(x["seconds"] for x in vals),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": HEADLINE_WORKLOAD,
                       "parallelism": "replicas" if args.gpus > 1 else "single"},
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rows", default="all",
                    help="comma list of extra rows: bsr_prefill,bsr_tiny,bsr_masked,bsr_variable,prefill_paged,"
                         "mla,mla_paged,"
                         "mla_append,"
                         "split,e2e,cpu "
                         "or all/none")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    args.warmup = max(args.warmup, 3)

    import block_sparse_kv_gb300 as bskv
    import synth
    bskv.build()
    dist, rank, ws = dist_setup(args.gpus)
    peaks, peak_src = load_peaks()
    rows = set(["bsr_prefill", "bsr_tiny", "bsr_masked", "bsr_variable", "prefill_paged", "mla",
                "mla_paged", "mla_append", "split", "e2e", "cpu"]
               if args.rows == "all" else [] if args.rows == "none" else args.rows.split(","))

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    head, _ = bench_decode(bskv, synth, "paged_decode", args.steps, args.warmup, dist,
                           headline=True)
    t_max = max_over_ranks(dist, head["total_ms"])
    total_bytes = sum_over_ranks(dist, head["kv_bytes"] * args.steps)
    value = total_bytes / (t_max * 1e-3) / 1e9
    status = bskv.bskv_get_device_status()

    extra = {}
    global TP
    if rank == 0 and rows & {"bsr_prefill", "bsr_tiny", "bsr_masked", "bsr_variable",
                             "prefill_paged", "mla", "mla_paged"}:
        TP = measure_tensor_peaks()
    if rank == 0:
        K = max(5, min(args.steps, 50))  # timed iterations per row (median and std reported)
        jobs = [("split", "split_decode", lambda: bench_split(bskv, synth, K, args.warmup, peaks)),
                ("bsr_prefill", "bsr_prefill",
                 lambda: bench_bsr(bskv, synth, "bsr_prefill", K, args.warmup, peaks, True)),
                ("bsr_tiny", "bsr_tiny",
                 lambda: bench_bsr(bskv, synth, "bsr_tiny", K, args.warmup, peaks, True)),
                ("mla", "mla_decode", lambda: bench_mla(bskv, synth, K, args.warmup, peaks)),
                ("mla_paged", "mla_paged",
                 lambda: bench_mla_paged(bskv, synth, K, args.warmup, peaks)),
                ("mla_append", "mla_append",
                 lambda: bench_mla_append(bskv, synth, K, args.warmup, peaks)),
                ("bsr_masked", "bsr_masked",
                 lambda: bench_bsr_masked(bskv, synth, K, args.warmup, peaks)),
                ("bsr_variable", "bsr_variable",
                 lambda: bench_bsr_variable(bskv, synth, K, args.warmup, peaks)),
                ("prefill_paged", "prefill_paged",
                 lambda: bench_prefill_paged(bskv, synth, K, args.warmup, peaks))]
        for key, name, job in jobs:
            if key in rows:
                try:
                    extra[name] = job()
                except bskv.BskvError as e:
                    extra[name] = "not available: %s" % e
                torch.cuda.empty_cache()
    clocks = sampler.stop() if sampler else None
    e2e = None
    if rank == 0 and "e2e" in rows:
        e2e = bench_decode_e2e(bskv, synth, max(3, min(args.steps, 10)), 2)
    cpu = oracle_decode_sample(synth) if (rank == 0 and "cpu" in rows and ws == 1) else None
    status = status or bskv.bskv_get_device_status()

    if rank != 0:
        return
    # the kernel's average duration over the timed region (one launch per step: the step
    # time, inter-launch gaps included); the event-bracketed per-launch mean is in the breakdown
    kern_us = (1e3 * head["ms_per_step"] if head["launches_per_step"] == 1
               else head["decode_kernel"]["mean_us"])
    achieved = head["kv_bytes"] / (kern_us * 1e-6) / 1e9
    peak = peaks["hbm_gbs"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, random page permutation, NaN canary pages)",
        "config": {"workload": HEADLINE_WORKLOAD,
                   "global_batch": 64 * args.gpus, "kv_bytes_per_step": head["kv_bytes"],
                   "l2": "inputs larger than L2 (0.6 GB KV per step)",
                   "parallelism": "replicas x%d" % args.gpus if args.gpus > 1 else "single"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src + " (hbm_gbs, burst)",
                     "kernel": "decode_group_kernel", "bytes_per_launch": head["kv_bytes"],
                     "traffic": profile_traffic("decode_group_kernel_paged_decode.txt",
                                                ["decode.cu", "common.cuh"])},
        "clocks": clocks,
        "gpu_launches": head["launches_per_step"] * args.steps,
        "plan_us": head["plan_us"],
        "step_breakdown_us": {"decode_kernel_with_fused_merge": head["decode_kernel"]["mean_us"],
                              "decode_kernel_median_event_bracketed": head["decode_kernel"]["median_us"],
                              "graph_replay_per_step": (1e3 * head["graph_ms_per_step"]
                                                        if head["graph_ms_per_step"] else None)},
        "decode_variant": head["variant"],
        "device_status": bskv.STATUS.get(status, status),
        "e2e": e2e,
        "cpu_baseline": cpu,
        "tensor_peaks": TP,
        "rows": extra,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
