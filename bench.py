"""Benchmark of gated GQA attention (head_dim 256) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: 27B-shape decode - 16 sequences, 24 query heads over 4 KV
heads, one row each, kv lengths 1987..32233 (sum 297,628) in a [16,4,32768,256]
bf16 cache.  Metric: decode KV GB/s (K and V bytes of the keys each sequence
holds, plus Q, G and out) as a fraction of the measured HBM bandwidth.  One step
is one decode call: the split kernel, then the LSE merge (with the gate).  The
same JSON line carries the prefill side of the metric, measured on the 27B-shape
prefill (24/4 heads, 8192 causal rows, 1% key outliers) in TFLOP/s against the
measured dense-bf16 peak.

Inputs are seeded synthetic bf16 tensors (synth/), generated on the host and
copied to the device once.  L2 is flushed before every timed step, outside the
timed events: a 256 MiB write, then a 256 MiB read, so that the write's dirty
lines are written back to HBM before the step rather than during it.  N > 1 ranks each run an independent replica of
the workload (no collective on the data path): "scaling": "weak".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import numpy as np  # noqa: E402
import torch  # noqa: E402

from synth import inputs as S  # noqa: E402

METRIC = "prefill attn TFLOP/s & decode KV GB/s (% of GB300 roofline), D256 GQA"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- traffic
def dram_traffic(kernel, units):
    """DRAM bytes per launch for `kernel` on a workload of `units`, scaled from the
    ncu capture recorded in profiles/dram_traffic.json; None when there is no record
    or the kernel's source changed since the capture (hash mismatch)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)[kernel]
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["sha256"]:
                return None
    except (OSError, KeyError, ValueError):
        return None
    return round((rec["dram_read"] + rec["dram_write"]) * units / rec["units"])


# ----------------------------------------------------------------------------- work counts
def decode_bytes(x):
    """Algorithmic bytes of one decode call: K and V of every key a sequence holds
    (read once per KV head), plus Q, G and out."""
    Hkv = x.k_cache.shape[1]
    kv = int(x.kv_lens.sum()) * Hkv * 256 * 2 * 2
    qgo = x.q.numel() * 2 * 3
    return kv, kv + qgo


def prefill_flops(x):
    """4 * 256 FLOP per causal-visible (query row, key) pair per query head."""
    B, Hq, Lq, _ = x.q.shape
    pairs = sum(x.kv_offset + i + 1 for i in range(Lq))
    return 4.0 * 256 * pairs * B * Hq


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of one GPU while the
    timed region runs.  Reads NVML (libnvidia-ml, read-only queries) from a thread
    every ~2 ms, so even a few-millisecond region gets samples; falls back to an
    `nvidia-smi -lms` subprocess when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index, period_s=0.002):
        self.dev = device_index
        self.period = period_s
        self.samples = []          # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._t = None
        self._nvml = None
        self._h = None
        self._proc = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        # The NVML index of the CUDA device: match by PCI bus id.
        # The NVML handle of the CUDA device: by UUID (robust to CUDA_VISIBLE_DEVICES),
        # else by index.
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.dev)
        uuid = getattr(props, "uuid", None)
        ok = False
        if uuid is not None:
            u = str(uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            ok = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.dev, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self._nvml, self._h = lib, h
        self._reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def _poll(self):
        import ctypes
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0:
                r = rs.value if self._reason_fn(self._h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), int(r)))
            time.sleep(self.period)

    def _smi(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown")
        self._proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "20",
                                       "-i", str(self.dev)],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        bits = [0x4, 0x8, 0x20, 0x40]
        for line in self._proc.stdout:
            f = [c.strip() for c in line.split(",")]
            try:
                self.max_mhz = float(f[1])
                r = sum(b for b, v in zip(bits, f[2:6]) if v.lower().startswith("active"))
                self.samples.append((float(f[0]), r))
            except (ValueError, IndexError):
                pass

    def __enter__(self):
        try:
            self._nvml_open()
            self.source = "nvml"
            self._t = threading.Thread(target=self._poll, daemon=True)
        except (OSError, AttributeError):
            self.source = "nvidia-smi"
            self._t = threading.Thread(target=self._smi, daemon=True)
        self._t.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5.0:   # sampler is live before timing
            time.sleep(0.001)
        self.samples.clear()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        if self._t is not None:
            self._t.join(timeout=5)
        if self._nvml is not None:
            self._nvml.nvmlShutdown()

    def summary(self):
        if not self.samples:
            return None
        mask = 0
        for _, r in self.samples:
            mask |= r
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if mask & b),
                "samples": len(self.samples), "source": self.source}


# ----------------------------------------------------------------------------- helpers
class L2Flush:
    """Evicts the step's inputs from L2: a 256 MiB write (twice L2), then a 256 MiB
    read.  The read evicts the write's dirty lines, so their write-back to HBM
    happens here and not inside the next timed step (a write alone cost the 27B
    decode and 35B verify steps ~12 us of write-back each); L2 is left holding clean
    lines of an unrelated buffer."""

    def __init__(self, dev):
        self.buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.rbuf = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.fill_(1)
        torch.sum(self.rbuf, 0, out=self.acc)


def elapsed_ms(pairs):
    return [a.elapsed_time(b) for a, b in pairs]


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle timing
def oracle_decode_sample(x, budget_s=10.0, min_seqs=1):
    """Times the float64 oracle on whole sequences of the decode workload (all heads
    of each) until about budget_s of CPU work; returns (GB/s, description)."""
    import oracle
    Hkv = x.k_cache.shape[1]
    done_bytes = 0
    n = 0
    t_total = 0.0
    cu = x.cu_rows.tolist()
    for b in range(x.k_cache.shape[0]):
        L = int(x.kv_lens[b])
        Kc = x.k_cache[b:b + 1, :, :L].double().numpy()
        Vc = x.v_cache[b:b + 1, :, :L].double().numpy()
        Q = x.q[cu[b]:cu[b + 1]].double().numpy()
        Gt = x.g[cu[b]:cu[b + 1]].double().numpy()
        t0 = time.perf_counter()
        oracle.decode(Q, Kc, Vc, Gt, [L], [0, cu[b + 1] - cu[b]])
        t_total += time.perf_counter() - t0
        done_bytes += L * Hkv * 256 * 4 + Q.size * 6
        n += 1
        if t_total >= budget_s and n >= min_seqs:
            break
    return done_bytes / t_total / 1e9, t_total, f"{n} of {x.k_cache.shape[0]} sequences, all heads"


# ----------------------------------------------------------------------------- our arm
DECODE_WORKLOAD = ("27B-shape decode: B=16, Hq=24, Hkv=4, head_dim=256, 1 row/seq, kv_lens "
                   "uniform [1024,32768] (sum 297,628), cache [16,4,32768,256] bf16, seed 1")
BAL_PARTS = 16     # part slots per row of the one-call decode's balanced shares
def last_launch(prefix):
    """The library's record (gqa_launch_log) of its newest launch of a kernel whose
    name starts with `prefix`: grid, block and dynamic shared memory as launched."""
    import gqa_head_gated_gb300 as G
    for r in G.launch_log():
        if r["kernel"].startswith(prefix):   # a string or a tuple of prefixes
            return {"kernel": r["kernel"], "grid": r["grid"], "block": r["block"],
                    "dynamic_smem_bytes": r["dynamic_smem"], "source": "gqa_launch_log"}
    return None


def decode_config(x):
    """The `config` both arms print (the workload and how it is timed)."""
    kv_bytes, step_bytes = decode_bytes(x)
    return {"workload": DECODE_WORKLOAD,
            "bytes_per_step": step_bytes,
            "kv_bytes_per_step": kv_bytes,
            "l2": "GPU arm: flushed before every timed step, outside the events (256 MiB "
                  "write, then 256 MiB read so the write's dirty lines are written back "
                  "before the step); reference arm: host cores",
            "parallelism": "one replica per GPU, no data-path collective; reference arm: "
                           "rank 0 on the host cores"}


def setup_decode(x, steps, dev, with_rows=False):
    """Device copies and the split plan of a decode (one row per sequence) or, with
    `with_rows`, a verify workload (cu_rows passed to the kernels)."""
    import gqa_head_gated_gb300 as G
    q, kc, vc, g = (t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.g))
    kv = x.kv_lens.to(dev)
    cu = x.cu_rows.to(dev) if with_rows else None
    max_rows = max(x.rows) if with_rows else 1
    B, Hkv = kc.shape[0], kc.shape[1]
    T, Hq = q.shape[0], q.shape[1]
    max_kv = int(x.kv_lens.max())
    S_, C_ = G.decode_plan(B, T, Hq, Hkv, max_rows, max_kv)
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(steps)]
    ws = torch.empty(G.decode_workspace_size(B, T, Hq, Hkv, max_rows, max_kv), dtype=torch.uint8,
                     device=dev)
    return dict(q=q, kc=kc, vc=vc, g=g, kv=kv, cu=cu, max_rows=max_rows, max_kv=max_kv,
                plan=(S_, C_), ev=ev, ws=ws, out=torch.empty_like(q), flush=L2Flush(dev))


def run_decode_timed(ctx, steps, tree_mask=None, noalloc=False):
    """One decode step = one gqa_attn_decode call (gqa_attn_verify_tree with a tree
    mask, gqa_attn_decode_noalloc with `noalloc`): the split kernel, then the merge
    launched as its programmatic dependent.  Bracketed by events on the launching
    (current) stream; L2 flushed before each step, outside the events."""
    import gqa_head_gated_gb300 as G
    q, kc, vc, kv, g = ctx["q"], ctx["kc"], ctx["vc"], ctx["kv"], ctx["g"]
    for i in range(steps):
        ctx["flush"]()
        a, b = ctx["ev"][i % len(ctx["ev"])]
        a.record()
        if noalloc:
            G.decode_noalloc(q, kc, vc, g, kv, ctx["cu"], max_rows=ctx["max_rows"],
                             max_kv_len=ctx["max_kv"], out=ctx["out"])
        elif tree_mask is None:
            G.decode(q, kc, vc, g, kv, ctx["cu"], max_rows=ctx["max_rows"],
                     max_kv_len=ctx["max_kv"], workspace=ctx["ws"], out=ctx["out"])
        else:
            G.verify_tree(q, kc, vc, g, kv, ctx["cu"], tree_mask, max_rows=ctx["max_rows"],
                          max_kv_len=ctx["max_kv"], workspace=ctx["ws"], out=ctx["out"])
        b.record()


def bench_e2e_decode(x, steps, warmup, dev):
    """Through the one-call public API with host buffers: per step, the pinned-host
    Q, G and kv lengths go to the device, gqa_attn_decode runs, out comes back."""
    import gqa_head_gated_gb300 as G
    kc, vc = x.k_cache.to(dev), x.v_cache.to(dev)          # resident cache
    # The step's host inputs (Q, G, kv lengths) sit back to back in one pinned buffer
    # and go to the device in one copy; out comes back in one copy.
    nq, ng, nkv = x.q.numel() * 2, x.g.numel() * 2, x.kv_lens.numel() * 4
    hin = torch.empty(nq + ng + nkv, dtype=torch.uint8).pin_memory()
    hin[:nq].copy_(x.q.reshape(-1).view(torch.uint8))
    hin[nq:nq + ng].copy_(x.g.reshape(-1).view(torch.uint8))
    hin[nq + ng:].copy_(x.kv_lens.view(torch.uint8))
    din = torch.empty_like(hin, device=dev)
    dq = din[:nq].view(torch.bfloat16).view(x.q.shape)
    dg = din[nq:nq + ng].view(torch.bfloat16).view(x.g.shape)
    dkv = din[nq + ng:].view(torch.int32)
    hout = torch.empty_like(x.q).pin_memory()
    max_kv = int(x.kv_lens.max())
    B, Hkv = kc.shape[0], kc.shape[1]
    T, Hq = x.q.shape[0], x.q.shape[1]
    ws = torch.empty(G.decode_workspace_size(B, T, Hq, Hkv, 1, max_kv), dtype=torch.uint8,
                     device=dev)
    dout = torch.empty_like(dq)
    flush = L2Flush(dev)

    def step():
        din.copy_(hin, non_blocking=True)
        G.decode(dq, kc, vc, dg, dkv, None, max_rows=1, max_kv_len=max_kv, workspace=ws, out=dout)
        hout.copy_(dout, non_blocking=True)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    h2d = hin.numel()
    d2h = hout.numel() * 2
    ok = torch.isfinite(hout.float()).all().item()
    return sum(times), h2d, d2h, ok


def bench_decode_graphs(x, steps, warmup, dev):
    """The headline decode step and its end-to-end form captured once in CUDA graphs
    (after eager warm-up calls) and replayed: the step's device time without host
    launch overhead between its operations."""
    import gqa_head_gated_gb300 as G
    kc, vc = x.k_cache.to(dev), x.v_cache.to(dev)
    nq, ng, nkv = x.q.numel() * 2, x.g.numel() * 2, x.kv_lens.numel() * 4
    hin = torch.empty(nq + ng + nkv, dtype=torch.uint8).pin_memory()
    hin[:nq].copy_(x.q.reshape(-1).view(torch.uint8))
    hin[nq:nq + ng].copy_(x.g.reshape(-1).view(torch.uint8))
    hin[nq + ng:].copy_(x.kv_lens.view(torch.uint8))
    din = torch.empty_like(hin, device=dev)
    din.copy_(hin)
    dq = din[:nq].view(torch.bfloat16).view(x.q.shape)
    dg = din[nq:nq + ng].view(torch.bfloat16).view(x.g.shape)
    dkv = din[nq + ng:].view(torch.int32)
    hout = torch.empty_like(x.q).pin_memory()
    max_kv = int(x.kv_lens.max())
    B, Hkv = kc.shape[0], kc.shape[1]
    T, Hq = x.q.shape[0], x.q.shape[1]
    ws = torch.empty(G.decode_workspace_size(B, T, Hq, Hkv, 1, max_kv), dtype=torch.uint8,
                     device=dev)
    dout = torch.empty_like(dq)
    flush = L2Flush(dev)

    def kernel_step():
        G.decode(dq, kc, vc, dg, dkv, None, max_rows=1, max_kv_len=max_kv, workspace=ws, out=dout)

    def e2e_step():
        din.copy_(hin, non_blocking=True)
        kernel_step()
        hout.copy_(dout, non_blocking=True)

    res = {}
    for name, fn in (("step", kernel_step), ("e2e", e2e_step)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        times = []
        for i in range(warmup + steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            b.synchronize()
            if i >= warmup:
                times.append(a.elapsed_time(b))
        res[name] = sum(times) / len(times)
        del graph
    res["finite"] = bool(torch.isfinite(hout.float()).all().item())
    return res


def bench_prefill_code_warm(x, steps, warmup, dev):
    """The prefill call with its inputs cold but its code warm: after each flush the
    same call runs once on a second, separate set of inputs of the same shape, then
    the timed call runs on the flushed inputs.  For a latency-bound launch this
    separates the instruction and parameter fetch from HBM (which the flush also
    evicts) from the kernel's own work."""
    import gqa_head_gated_gb300 as G
    q, k, v, g = (t.to(dev) for t in (x.q, x.k, x.v, x.g))
    out = torch.empty_like(q)
    q2, k2, v2, g2 = (t.clone() for t in (q, k, v, g))
    out2 = torch.empty_like(q)
    flush = L2Flush(dev)
    ms = []
    for i in range(warmup + steps):
        flush()
        G.prefill(q2, k2, v2, g2, kv_offset=x.kv_offset, out=out2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        G.prefill(q, k, v, g, kv_offset=x.kv_offset, out=out)
        b.record()
        if i >= warmup:
            ms.append((a, b))
    torch.cuda.synchronize()
    return elapsed_ms(ms)


def bench_prefill(x, steps, warmup, dev, e2e=True):
    import gqa_head_gated_gb300 as G
    q, k, v, g = (t.to(dev) for t in (x.q, x.k, x.v, x.g))
    out = torch.empty_like(q)
    flush = L2Flush(dev)
    for _ in range(warmup):
        flush()
        G.prefill(q, k, v, g, kv_offset=x.kv_offset, out=out)
    torch.cuda.synchronize()
    pairs = []
    with ClockSampler(dev.index) as clk:
        for _ in range(steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            G.prefill(q, k, v, g, kv_offset=x.kv_offset, out=out)
            b.record()
            pairs.append((a, b))
        torch.cuda.synchronize()
    status = G.last_device_status()
    ms = elapsed_ms(pairs)
    if not e2e:
        return ms, status, None, None, None, clk.summary()
    # e2e: host buffers in, out back
    hq, hk, hv, hg = (t.pin_memory() for t in (x.q, x.k, x.v, x.g))
    hout = torch.empty_like(x.q).pin_memory()
    e2e = []
    for _ in range(max(1, min(steps, 5))):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        g.copy_(hg, non_blocking=True)
        G.prefill(q, k, v, g, kv_offset=x.kv_offset, out=out)
        hout.copy_(out, non_blocking=True)
        b.record()
        b.synchronize()
        e2e.append(a.elapsed_time(b))
    h2d = sum(t.numel() * 2 for t in (hq, hk, hv, hg))
    return ms, status, e2e, h2d, hout.numel() * 2, clk.summary()


def ours(args):
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    import gqa_head_gated_gb300 as G
    G.load()
    peaks, peak_src = load_peaks()
    x = S.decode_27b()
    kv_bytes, step_bytes = decode_bytes(x)

    ctx = setup_decode(x, args.steps, dev)
    S_, C_ = ctx["plan"]
    run_decode_timed(ctx, args.warmup)
    torch.cuda.synchronize()

    barrier(world)
    torch.cuda.synchronize()
    seq0 = G.launch_log(1)[0]["seq"]
    with ClockSampler(local) as clk:
        run_decode_timed(ctx, args.steps)
        torch.cuda.synchronize()
    launches = G.launch_log(1)[0]["seq"] - seq0    # the library's launches in the timed region
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ctx["ev"]]
    total_ms = max_over_ranks(world, sum(step_ms))
    # The dominant kernel alone (for the roofline): the same split launch, K more steps,
    # events around gqa_attn_decode_split on the same stream, L2 flushed before each.
    T_, Hq_ = x.q.shape[:2]
    op = torch.empty((BAL_PARTS, T_ * Hq_, 256), dtype=torch.float32, device=dev)
    lp = torch.empty((BAL_PARTS, T_ * Hq_), dtype=torch.float32, device=dev)
    split_ms = []
    for i in range(args.warmup + args.steps):
        ctx["flush"]()
        a, b = ctx["ev"][i % len(ctx["ev"])]
        a.record()
        G.decode_split(ctx["q"], ctx["kc"], ctx["vc"], ctx["kv"], None, max_rows=1,
                       max_kv_len=ctx["max_kv"], num_splits=BAL_PARTS, split_keys=0,
                       o_parts=op, lse_parts=lp)
        b.record()
        b.synchronize()
        if i >= args.warmup:
            split_ms.append(a.elapsed_time(b))
    del op, lp
    split_launch = last_launch("decode_split_kernel")
    status = G.last_device_status()
    out_ok = bool(torch.isfinite(ctx["out"].float()).all().item())

    value = world * step_bytes * args.steps / (total_ms / 1e3) / 1e9
    split_bytes = kv_bytes + x.q.numel() * 2
    split_avg = sum(split_ms) / len(split_ms)
    achieved = split_bytes / (split_avg / 1e3) / 1e9
    hbm_peak = float(peaks["hbm_gbs"])

    e2e_ms, h2d, d2h, e2e_ok = bench_e2e_decode(x, args.steps, args.warmup, dev)
    e2e_ms = max_over_ranks(world, e2e_ms)
    e2e_val = world * step_bytes * args.steps / (e2e_ms / 1e3) / 1e9

    graphs = None
    if not args.no_extra:
        try:
            graphs = bench_decode_graphs(x, args.steps, args.warmup, dev)
        except Exception as exc:   # noqa: BLE001 - reported, not fatal
            graphs = {"error": f"{type(exc).__name__}: {exc}"[:200]}

    # prefill side of the metric (27B-shape prefill)
    pf = S.prefill_27b()
    flops = prefill_flops(pf)
    pf_steps = max(3, min(args.steps, 10))
    pf_ms, pf_status, pf_e2e, pf_h2d, pf_d2h, pf_clk = bench_prefill(pf, pf_steps,
                                                                     max(3, args.warmup), dev)
    pf_launch = last_launch(("attn_tc_kernel<prefill", "attn_pair_kernel<prefill"))
    pf_avg = sum(pf_ms) / len(pf_ms)
    pf_tflops = flops / (pf_avg / 1e3) / 1e12
    bf16_peak = float(peaks["bf16_tflops"])
    pf_e2e_avg = sum(pf_e2e) / len(pf_e2e)
    # DRAM bytes of the prefill launch: the capture of this very workload when its
    # record matches the kernel source, else the 4,096-row capture scaled by input bytes
    pf_in_bytes = (pf.q.numel() + pf.k.numel() + pf.v.numel() + pf.g.numel()) * 2
    pf_pair = bool(pf_launch and pf_launch["kernel"].startswith("attn_pair"))
    pf_traffic = args.prefill_traffic
    pf_traffic_note = "given on the command line"
    if pf_traffic is None and pf_pair:
        pf_traffic = dram_traffic("attn_pair_kernel_prefill_27b", pf_in_bytes)
        pf_traffic_note = ("ncu capture of this workload's launch (bench.py --case prefill_27b, "
                           "one pass, cold L2); output writes still in L2 when the kernel "
                           "ended are not counted")
    if pf_traffic is None and args.prefill_traffic is None:
        pf_traffic = dram_traffic("attn_pair_kernel_prefill" if pf_pair
                                  else "attn_tc_kernel_prefill", pf_in_bytes)
        pf_traffic_note = ("not measured on this launch: the DRAM bytes of the 4,096-row "
                           "capture, scaled by input bytes; output writes still in L2 when "
                           "that kernel ended are not counted")

    # the other throughput workloads of the metric, inside the same line
    more = {}
    if graphs is not None:
        if "error" in graphs:
            more["decode_27b_cuda_graph"] = graphs
        else:
            more["decode_27b_cuda_graph"] = {
                "workload": "the headline decode step and its end-to-end form (pinned inputs "
                            "in, out back) captured once in CUDA graphs and replayed",
                "value": round(step_bytes / (graphs["step"] / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(graphs["step"], 5),
                "e2e_value": round(step_bytes / (graphs["e2e"] / 1e3) / 1e9, 2),
                "e2e_ms_per_step": round(graphs["e2e"], 5),
                "outputs_finite": graphs["finite"]}
    if not args.no_extra:
        cp = S.chunked_prefill_35b()
        cp_flops = prefill_flops(cp)
        cp_ms = bench_prefill(cp, pf_steps, max(3, args.warmup), dev, e2e=False)[0]
        cp_avg = sum(cp_ms) / len(cp_ms)
        more["chunked_prefill_35b"] = {
            "workload": "35B-A3B chunked prefill: B=1, Hq=16, Hkv=2, 2048 rows at kv_offset "
                        "30720 (Lkv 32768) causal, seed 3",
            "value": round(cp_flops / (cp_avg / 1e3) / 1e12, 2), "unit": "TFLOP/s",
            "frac_of_bf16_peak": round(cp_flops / (cp_avg / 1e3) / 1e12 / float(peaks["bf16_tflops"]), 4),
            "avg_ms": round(cp_avg, 4)}
        del cp
        # The 128-row prompt (24/4 heads): 28 CTAs, one key tile each, so it measures
        # the kernel's latency, not its throughput.
        tp = S.tiny_prefill()
        tp_flops = prefill_flops(tp)
        tp_ms = bench_prefill(tp, max(pf_steps, 20), max(3, args.warmup), dev, e2e=False)[0]
        tp_avg = sum(tp_ms) / len(tp_ms)
        tw_ms = bench_prefill_code_warm(tp, max(pf_steps, 20), max(3, args.warmup), dev)
        tw_avg = sum(tw_ms) / len(tw_ms)
        more["tiny_prefill"] = {
            "workload": "tiny prefill: B=1, Hq=24, Hkv=4, Lq=Lkv=128 causal, seed 0 "
                        "(latency-bound: 28 CTAs of one key tile)",
            "value": round(tp_flops / (tp_avg / 1e3) / 1e12, 3), "unit": "TFLOP/s",
            "avg_us": round(tp_avg * 1e3, 2),
            "avg_us_code_warm": round(tw_avg * 1e3, 2),
            "code_warm_note": "inputs flushed as for avg_us, then the same call once on a "
                              "separate set of inputs before the timed call: the kernel's "
                              "code and parameters are in L2, its inputs are not"}
        del tp
        vx = S.verify_35b()
        v_kv, v_bytes = decode_bytes(vx)
        vctx = setup_decode(vx, args.steps, dev, with_rows=True)
        run_decode_timed(vctx, args.warmup)
        torch.cuda.synchronize()
        run_decode_timed(vctx, args.steps)
        torch.cuda.synchronize()
        v_step = sum(a.elapsed_time(b) for a, b in vctx["ev"]) / args.steps
        more["verify_35b"] = {
            "workload": "35B-A3B draft verify: B=8, Hq=16, Hkv=2, rows [1,3,4,8,16,32,1,3], "
                        "kv_lens 4271..45513 in a [8,2,65536,256] cache, seed 4",
            "value": round(v_bytes / (v_step / 1e3) / 1e9, 2), "unit": "GB/s",
            "frac_of_hbm": round(v_bytes / (v_step / 1e3) / 1e9 / hbm_peak, 4),
            "split_plan": {"num_splits": vctx["plan"][0], "split_keys": vctx["plan"][1]},
            "ms_per_step": round(v_step, 5)}
        # the same verify workload over seeded token trees (one 64-bit mask per row)
        tm = torch.tensor(S.random_tree_masks(vx.rows, 5), dtype=torch.int64, device=dev)
        run_decode_timed(vctx, args.warmup, tree_mask=tm)
        torch.cuda.synchronize()
        run_decode_timed(vctx, args.steps, tree_mask=tm)
        torch.cuda.synchronize()
        t_avg = sum(a.elapsed_time(b) for a, b in vctx["ev"]) / args.steps
        more["verify_tree_35b"] = {
            "workload": "the 35B draft-verify workload over seeded token trees "
                        "(synth.random_tree_masks(rows, 5)), gqa_attn_verify_tree",
            "value": round(v_bytes / (t_avg / 1e3) / 1e9, 2), "unit": "GB/s",
            "frac_of_hbm": round(v_bytes / (t_avg / 1e3) / 1e9 / hbm_peak, 4),
            "ms_per_step": round(t_avg, 5)}
        del vctx, vx
        torch.cuda.empty_cache()
        # KV-cache append of a whole 8192-row prompt's K/V (24/4 heads) into a cache
        kn = pf.k.to(dev)[0].transpose(0, 1).contiguous()      # [8192, 4, 256]
        vn = pf.v.to(dev)[0].transpose(0, 1).contiguous()
        kcache = torch.empty((1, 4, 16384, 256), dtype=torch.bfloat16, device=dev)
        vcache = torch.empty_like(kcache)
        zl = torch.zeros(1, dtype=torch.int32, device=dev)
        cu1 = torch.tensor([0, 8192], dtype=torch.int32, device=dev)
        for _ in range(args.warmup):
            G.kv_append(kn, vn, zl, kcache, vcache, cu1)
        torch.cuda.synchronize()
        aps = []
        for _ in range(args.steps):
            ctx["flush"]()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record()
            G.kv_append(kn, vn, zl, kcache, vcache, cu1)
            b_.record()
            aps.append((a_, b_))
        torch.cuda.synchronize()
        ap_ms = sum(a_.elapsed_time(b_) for a_, b_ in aps) / len(aps)
        ap_bytes = 2 * 2 * kn.numel() * 2                       # K and V, read and written
        more["kv_append_27b_prompt"] = {
            "workload": "gqa_kv_append of 8192 new rows x 4 KV heads (K and V, 33.5 MB) into "
                        "a [1,4,16384,256] cache",
            "value": round(ap_bytes / (ap_ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "frac_of_hbm": round(ap_bytes / (ap_ms / 1e3) / 1e9 / hbm_peak, 4),
            "ms_per_call": round(ap_ms, 5)}
        del kn, vn, kcache, vcache
        torch.cuda.empty_cache()
        # FP16 twins of the headline decode and of the 27B prefill (same draws rounded to
        # fp16, the _f16 entry points; same byte and FLOP counts as bf16)
        xf = S.decode_27b(dtype=torch.float16)
        fctx = setup_decode(xf, args.steps, dev)
        run_decode_timed(fctx, args.warmup)
        torch.cuda.synchronize()
        run_decode_timed(fctx, args.steps)
        torch.cuda.synchronize()
        f_step = sum(a.elapsed_time(b) for a, b in fctx["ev"]) / args.steps
        f_ok = bool(torch.isfinite(fctx["out"].float()).all().item())
        more["decode_27b_fp16"] = {
            "workload": "the 27B-shape decode workload in fp16 (gqa_attn_decode_f16)",
            "value": round(step_bytes / (f_step / 1e3) / 1e9, 2), "unit": "GB/s",
            "frac_of_hbm": round(step_bytes / (f_step / 1e3) / 1e9 / hbm_peak, 4),
            "ms_per_step": round(f_step, 5), "outputs_finite": f_ok}
        del fctx, xf
        torch.cuda.empty_cache()
        # the headline decode through gqa_attn_decode_noalloc (the library's fixed area
        # as workspace; same kernels and plan)
        nctx = setup_decode(x, args.steps, dev)
        run_decode_timed(nctx, args.warmup, noalloc=True)
        torch.cuda.synchronize()
        run_decode_timed(nctx, args.steps, noalloc=True)
        torch.cuda.synchronize()
        n_step = sum(a.elapsed_time(b) for a, b in nctx["ev"]) / args.steps
        n_same = bool(torch.equal(nctx["out"], ctx["out"]))
        more["decode_27b_noalloc"] = {
            "workload": "the headline decode step through gqa_attn_decode_noalloc (no "
                        "caller workspace)",
            "value": round(step_bytes / (n_step / 1e3) / 1e9, 2), "unit": "GB/s",
            "frac_of_hbm": round(step_bytes / (n_step / 1e3) / 1e9 / hbm_peak, 4),
            "ms_per_step": round(n_step, 5), "same_bits_as_decode": n_same,
            "launch": last_launch("decode_split_kernel")}
        del nctx
        torch.cuda.empty_cache()
        pff = S.prefill_27b(dtype=torch.float16)
        pff_ms = bench_prefill(pff, pf_steps, max(3, args.warmup), dev, e2e=False)[0]
        pff_avg = sum(pff_ms) / len(pff_ms)
        more["prefill_27b_fp16"] = {
            "workload": "the 27B-shape prefill in fp16 (gqa_attn_prefill_f16)",
            "value": round(flops / (pff_avg / 1e3) / 1e12, 2), "unit": "TFLOP/s",
            "frac_of_fp16_peak": round(flops / (pff_avg / 1e3) / 1e12 / bf16_peak, 4),
            "peak_note": "fp16 dense peak = measured bf16 burst peak x 1 (equal nominal rates)",
            "avg_ms": round(pff_avg, 4)}
        del pff
        # General masks on the 27B prefill (gqa_attn_masked, causal rule on): an additive
        # bf16 bias [8192, 8192] broadcast over batch and heads (every causal pair stays
        # visible, so the FLOPs equal the plain prefill's), and a bool block-diagonal
        # document mask (documents of 1024 rows)
        q_, k_, v_, g_ = (t.to(dev) for t in (pf.q, pf.k, pf.v, pf.g))
        Lp = q_.shape[2]
        gen = torch.Generator().manual_seed(7)
        bias = (torch.randn(Lp, Lp, generator=gen) * 2).to(torch.bfloat16).to(dev)
        doc = torch.arange(Lp, device=dev) // 1024
        docm = doc[:, None] == doc[None, :]
        mout = torch.empty_like(q_)
        for name, m in (("masked_prefill_27b_bias", bias), ("masked_prefill_27b_doc", docm)):
            for _ in range(max(3, args.warmup)):
                ctx["flush"]()
                G.masked(q_, k_, v_, g_, m, causal=True, kv_offset=0, out=mout)
            torch.cuda.synchronize()
            mp = []
            for _ in range(pf_steps):
                ctx["flush"]()
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record()
                G.masked(q_, k_, v_, g_, m, causal=True, kv_offset=0, out=mout)
                b_.record()
                mp.append((a_, b_))
            torch.cuda.synchronize()
            m_avg = sum(a_.elapsed_time(b_) for a_, b_ in mp) / len(mp)
            entry = {"value": round(flops / (m_avg / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                     "frac_of_bf16_peak": round(flops / (m_avg / 1e3) / 1e12 / bf16_peak, 4),
                     "avg_ms": round(m_avg, 4), "vs_unmasked_prefill": round(pf_avg / m_avg, 4),
                     "mask_bytes": m.numel() * m.element_size()}
            if name.endswith("bias"):
                entry["workload"] = ("the 27B prefill with an additive bf16 bias [8192, 8192] "
                                     "(N(0,2), seed 7) broadcast over heads, causal")
            else:
                vis = 8 * (1024 * 1025 // 2)
                entry["workload"] = ("the 27B prefill with a bool block-diagonal document mask "
                                     "(8 documents of 1024 rows), causal; value counts every "
                                     "causal pair the kernel computes")
                entry["visible_pair_tflops"] = round(4.0 * 256 * vis * 24 / (m_avg / 1e3) / 1e12, 2)
            more[name] = entry
        del q_, k_, v_, g_, bias, docm, mout
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0:
        gbs, secs, desc = oracle_decode_sample(x, budget_s=args.cpu_budget)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": _CORES, "kind": "oracle",
               "sample": f"float64 numpy oracle on {desc} of the 27B-shape decode workload "
                         f"({secs:.1f} s)"}

    if rank == 0:
        # DRAM bytes of the split launch: the capture of this very workload when its
        # record matches the kernel source, else the 8K-key capture scaled by keys held
        held = int(x.kv_lens.sum()) * x.k_cache.shape[1]
        dec_traffic, dec_traffic_note = args.traffic, "given on the command line"
        if dec_traffic is None:
            dec_traffic = dram_traffic("decode_split_kernel_27b", held)
            dec_traffic_note = ("ncu capture of this workload's split launch (bench.py --case "
                                "decode_27b, one pass, cold L2)")
        if dec_traffic is None:
            dec_traffic = dram_traffic("decode_split_kernel", held)
            dec_traffic_note = ("not measured on this launch: the DRAM bytes of the 8K-key "
                                "capture (bench.py --case decode_8k), scaled by keys held")
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 Q/K/V, G ~ N(0,2)); no dataset",
            "config": decode_config(x),
            "split_plan": {"mode": "balanced shares (one per resident CTA)",
                           "part_slots": BAL_PARTS},
            "roofline": {
                "kernel": "decode_split_kernel",
                "bound": "hbm",
                "achieved": round(achieved, 2),
                "peak": hbm_peak,
                "peak_source": f"{peak_src} hbm_gbs",
                "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4),
                "traffic": dec_traffic,
                "traffic_note": dec_traffic_note,
                "avg_launch_ms": round(split_avg, 5),
                "launch": split_launch,
                "timing": "events around gqa_attn_decode_split alone in the step's form "
                          "(balanced shares, 16 part slots), K steps right after the headline "
                          "steps, L2 flushed before each",
                "algorithmic_bytes_per_launch": split_bytes,
            },
            "step_note": "one gqa_attn_decode call per step: decode_split_kernel, then "
                         "lse_merge_kernel launched as its programmatic dependent (scheduled "
                         "while the split kernel drains; it waits for the split grid before "
                         "reading the parts)",
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "note": "gqa_attn_decode with pinned host Q/G/kv_lens in (one copy) and "
                            "out back (one copy); the KV cache is resident device state"},
            "gpu_launches": launches,
            "cpu_baseline": cpu,
            "prefill": {
                "workload": "27B-shape prefill: B=1, Hq=24, Hkv=4, Lq=Lkv=8192 causal, "
                            "1% of K rows x8, seed 2",
                "value": round(pf_tflops, 2),
                "unit": "TFLOP/s",
                "flops_per_call": flops,
                "avg_ms": round(pf_avg, 4),
                "steps": pf_steps,
                "launch": pf_launch,
                "roofline": {"kernel": pf_launch["kernel"] if pf_launch else None, "bound": "tensor",
                             "achieved": round(pf_tflops, 2), "peak": bf16_peak,
                             "peak_source": f"{peak_src} bf16_tflops (burst)",
                             "unit": "TFLOP/s", "frac": round(pf_tflops / bf16_peak, 4),
                             "traffic": pf_traffic,
                             "traffic_note": pf_traffic_note},
                "e2e": {"value": round(flops / (pf_e2e_avg / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                        "h2d_bytes_per_step": pf_h2d, "d2h_bytes_per_step": pf_d2h},
                "device_status": pf_status,
                "clocks": pf_clk,
            },
            "more_workloads": more,
            "clocks": clk.summary(),
            "device_status": status,
            "outputs_finite": out_ok and e2e_ok,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm
def reference(args):
    """The float64 oracle, as it stands, on the host cores: each step is a bounded
    sample (whole sequences of the decode workload)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x = S.decode_27b()
    budget = max(0.5, args.ref_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_decode_sample(x, budget_s=budget)
    vals, secs, desc = [], 0.0, ""
    for _ in range(args.steps):
        v, s, desc = oracle_decode_sample(x, budget_s=budget)
        vals.append(v)
        secs += s
    value = statistics.median(vals)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, G ~ N(0,2)); no dataset",
        "config": decode_config(x),
        "sample": "each step a bounded sample of whole sequences (see cpu_baseline)",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": _CORES,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- ncu cases
CASES = {
    # 24/4 heads, 4096 causal rows: 160 MB of Q/K/V/G/out (> L2), ~0.2 ms per launch
    "prefill_4k": lambda: S.make_prefill(1, 24, 4, 4096, seed=2, outlier_frac=0.01),
    # 16 sequences x 24/4 heads, kv lengths 2048..8192 in a [16,4,8192,256] cache (537 MB)
    "decode_8k": lambda: S.make_decode(16, 24, 4, [1] * 16,
                                       [2048 + (b * 389) % 6145 for b in range(16)],
                                       Lcap=8192, seed=1),
    # 8 sequences x 16/2 heads, verify rows 1..32, kv lengths a fifth of the 35B
    # draft-verify workload's in a [8,2,16384,256] cache (268 MB)
    "verify_16k": lambda: S.make_decode(8, 16, 2, [1, 3, 4, 8, 16, 32, 1, 3],
                                        [4325, 854, 4593, 4238, 7757, 3758, 4011, 9102],
                                        Lcap=16384, seed=4),
    # the prefill_4k inputs with an additive bf16 bias [4096, 4096] (N(0,2), seed 7,
    # 32 MB) broadcast over heads, causal: the general-mask kernel, staged mask rows
    "masked_4k": lambda: S.make_prefill(1, 24, 4, 4096, seed=2, outlier_frac=0.01),
    # the 128-row prompt of the bench's tiny-prefill line (28 CTAs of one key tile)
    "prefill_tiny": lambda: S.tiny_prefill(),
    # the 27B-shape prefill at full size (8192 causal rows, 24/4 heads, 320 MiB of
    # Q/K/V/G/out, ~0.53 ms per launch): for single-pass DRAM counters only
    "prefill_27b": lambda: S.WORKLOADS["prefill_27b"](),
    # the 27B-shape decode at full size (16 sequences, kv lengths 1024..32768 in a
    # [16,4,32768,256] cache, 2.1 GB; ~0.18 ms per split launch): single-pass counters only
    "decode_27b": lambda: S.WORKLOADS["decode_27b"](),
}


def run_case(name, launches, warmup):
    """Launches one small case `warmup + launches` times and prints nothing to stdout
    (for profiler captures: select the kernel with -k and skip the warm-up launches)."""
    import gqa_head_gated_gb300 as G
    dev = torch.device("cuda", 0)
    x = CASES[name]()
    if name.startswith("prefill"):
        q, k, v, g = (t.to(dev) for t in (x.q, x.k, x.v, x.g))
        out = torch.empty_like(q)
        for _ in range(warmup + launches):
            G.prefill(q, k, v, g, kv_offset=x.kv_offset, out=out)
    elif name.startswith("masked"):
        q, k, v, g = (t.to(dev) for t in (x.q, x.k, x.v, x.g))
        L = q.shape[2]
        bias = (torch.randn(L, L, generator=torch.Generator().manual_seed(7)) * 2).to(
            torch.bfloat16).to(dev)
        out = torch.empty_like(q)
        for _ in range(warmup + launches):
            G.masked(q, k, v, g, bias, causal=True, kv_offset=0, out=out)
    else:
        q, kc, vc, g = (t.to(dev) for t in (x.q, x.k_cache, x.v_cache, x.g))
        kv, cu = x.kv_lens.to(dev), x.cu_rows.to(dev)
        for _ in range(warmup + launches):
            G.decode(q, kc, vc, g, kv, cu, max_rows=max(x.rows), max_kv_len=int(x.kv_lens.max()))
    torch.cuda.synchronize()
    st = G.last_device_status()
    log(f"case {name}: {warmup + launches} launches, device status {st}")
    if st != 0:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of oracle work for the whole reference arm")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per split launch from an ncu capture of this kernel")
    ap.add_argument("--prefill-traffic", type=float, default=None)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 35B chunked-prefill and draft-verify measurements")
    ap.add_argument("--case", choices=sorted(CASES), default=None,
                    help="only launch this small case (for ncu captures); no JSON line")
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.steps, args.warmup)
        return
    args.warmup = max(3, args.warmup)     # at least three untimed warm-up steps
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
