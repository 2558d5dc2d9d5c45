"""Benchmark of the paged attention hot path on one GB300 (or N replicas).

A step is one decode round of the batched-decode workload (8 streams x 8,192
positions, 32 query / 8 KV heads, head_dim 128, bf16 KV; streams 0-3 on slabs,
4-7 on 256-position pages of a permuted 512-page pool): each stream's new
K/V row stored and decoded by one tfpa_decode_append call (split-K partials,
whose CTAs store the new rows they read, then the merge).  value =
algorithmic KV bytes (+ Q and O) per step / step time,
in GB/s.  The prompt-chunk workload (28,672-position paged prefix plus a
4,096-row causal chunk) is timed beside it and reported in TFLOP/s of its
unmasked (row, key) pairs.

Inputs are 268 MB of KV per step, above the 129 MB L2, so no flush is needed
between decode steps; the prompt-chunk timing flushes L2 between launches.

e2e is a decode loop through the public API with host buffers, one step at a
time and every stream one position longer each step: while the previous step
runs, the host writes the step's inputs into pinned memory and plans the
step anew (tfpa_plan_decode_append, plan in device mode), packing its
lengths into the same pinned buffer (tfpa_plan_dyn_pack); then one
CUDA-graph replay runs the planned launches, which read the inputs and
lengths from host memory and write the output there over NVLink-C2C, and
the host waits.  The same loop with copy-engine copies to and from device
buffers, with the plan in parameter mode (tfpa_plan_launch each step) and
with direct tfpa_decode_append calls is reported beside it, with host
times.

Launch: ``python bench.py [--gpus N --steps K --warmup W] [--impl reference]``;
for N > 1 under torchrun every rank runs its own replica (no collective on the
data path) and rank 0 prints one JSON line with the max time over ranks.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s (% HBM peak); prompt-chunk attn TFLOP/s (% TC peak)"


# DRAM traffic of one decode partial launch on the batched-decode workload
# (dram__bytes_read.sum + dram__bytes_write.sum from one ncu capture of this
# bench's partial launch), valid only while the kernel's sources hash to the
# value below: after any change to them the line reports null until the
# counters are taken again.
DECODE_TRAFFIC = {"bytes": 268_608_000 + 3_727_104, "sources_sha256_16": "97252c9c62ebf467"}
DECODE_SOURCES = ["paged_kv_cache_235_gb300/csrc/decode.cu",
                  "paged_kv_cache_235_gb300/csrc/common.cuh",
                  "paged_kv_cache_235_gb300/csrc/params.h",
                  "paged_kv_cache_235_gb300/csrc/tcgen05.cuh"]


def decode_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return DECODE_TRAFFIC["bytes"] if h.hexdigest()[:16] == DECODE_TRAFFIC["sources_sha256_16"] \
        else None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self._proc = None
        return self

    def _read(self):
        for line in self._proc.stdout:
            self.samples.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self._proc:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if len(s) > 3 + i and s[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


# --------------------------------------------------------------------- set-up
def device_case(w, torch, B):
    """A workload's cache on the GPU with device-generated N(0,1) values.

    The bench measures speed; parity is established by the tests.  Every
    stream's K/V goes through tfpa_write_kv, as in the tests."""
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    fp8 = w.kv_dtype == "fp8"

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)

    store = torch.uint8 if fp8 else torch.bfloat16
    kp = torch.empty(w.num_pages, w.hkv, 256, 128, dtype=store, device=dev)
    vp = torch.empty_like(kp)
    if fp8:
        kp.random_(0, 127, generator=g)
        vp.random_(0, 127, generator=g)
    else:
        kp.copy_(randn(*kp.shape))
        vp.copy_(randn(*vp.shape))
    ks = vs = None
    if fp8:   # amax/448 of N(0,1) draws at these sizes
        ks = torch.full((w.hkv,), 5.6 / 448, dtype=torch.float32, device=dev)
        vs = ks.clone()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    cache = B.Cache(w.kv_dtype, w.hq, w.hkv, kp, vp, ks, vs, err, w.num_pages)
    segs = []
    for st in w.streams:
        if st.paged:
            segs.append(B.Seg(st.seq_len, page_table=torch.from_numpy(st.page_table).to(dev),
                              page_table_host=st.page_table))
        else:
            cap = st.slab_cap
            segs.append(B.Seg(st.seq_len, k_slab=torch.empty(w.hkv, cap, 128, dtype=store, device=dev),
                              v_slab=torch.empty(w.hkv, cap, 128, dtype=store, device=dev),
                              slab_cap=cap))
    for s, st in enumerate(w.streams):
        L = st.seq_len
        for a in range(0, L, 65536):
            n = min(65536, L - a)
            B.tfpa_write_kv(cache, segs, randn(n, w.hkv, 128), randn(n, w.hkv, 128),
                            np.full(n, s, np.int32), np.arange(a, a + n, dtype=np.int32))
    torch.cuda.synchronize()
    q = randn(w.rows, w.hq, 128)
    return cache, segs, q


def kv_bytes(w):
    b = 1 if w.kv_dtype == "fp8" else 2
    kv = sum(st.seq_len for st in w.streams) * w.hkv * 128 * 2 * b
    return kv, w.rows * w.hq * 128 * 2 * 2   # KV, Q + O


def prefill_flops(w):
    return 4.0 * 128 * w.hq * float(np.sum(w.row_pos.astype(np.float64) + 1))


def barrier(dist, torch):
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()


def max_over_ranks(dist, torch, x):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------- oracle
def cpu_oracle_sample(seconds: float = 12.0):
    """The oracle on this host's cores, on stream 0 of the batched-decode
    workload (1 row x 32 heads over 8,192 keys), repeated for ~`seconds`."""
    from oracle import attention, kvcache
    from paged_kv_cache_235_gb300 import workloads as wl
    w = wl.batched_decode()
    k, v = w.stream_kv_bits(0)
    L = w.streams[0].seq_len
    cache = kvcache.Cache("bf16", w.hkv, w.d, None, None)
    seg = kvcache.Segment(L, k_slab=k, v_slab=v)
    q = w.q_bits()[:1]
    n, t0 = 0, time.perf_counter()
    while True:
        attention.attend(cache, [seg], q, [0], [L - 1], w.softmax_scale)
        n += 1
        if time.perf_counter() - t0 > seconds:
            break
    dt = (time.perf_counter() - t0) / n
    bytes_ = L * w.hkv * 128 * 2 * 2
    return {"value": bytes_ / dt / 1e9, "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle", "calls": n, "s_per_call": dt,
            "sample": "stream 0 of the batched-decode workload: 1 row x 32 heads over 8,192 "
                      "bf16 keys (1/8 of a step), float64 NumPy, "
                      + ("repeated for ~%ds" % seconds if seconds > 0 else "one call")}


# --------------------------------------------------------------------- timing
def time_decode(w, torch, B, steps, warmup, dist):
    """Device-timed decode steps plus the partial kernel timed on its own."""
    cache, segs, q = device_case(w, torch, B)
    sc = B.make_scratch(min(128, w.rows), w.hq)
    out = torch.empty(w.rows, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.rows, w.hq, dtype=torch.float32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    newk = torch.randn(len(w.streams), w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    newv = torch.randn(len(w.streams), w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    last = np.array([st.seq_len - 1 for st in w.streams], np.int32)
    sidx = np.arange(len(w.streams), dtype=np.int32)

    def step():
        B.tfpa_decode_append(cache, segs, newk, newv, q, sidx, last, w.softmax_scale, sc, out, lse)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # One step captured as a CUDA graph (the library enqueues only kernels,
    # with parameters by value, so a step replays without host work).
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            step()
    torch.cuda.current_stream().wait_stream(cap)
    for _ in range(warmup):
        graph.replay()
    barrier(dist, torch)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        graph.replay()
    e1.record(s)
    barrier(dist, torch)
    step_ms = e0.elapsed_time(e1) / steps

    # A/A: the same replays timed again right after
    e0.record(s)
    for _ in range(steps):
        graph.replay()
    e1.record(s)
    barrier(dist, torch)
    step_ms_again = e0.elapsed_time(e1) / steps

    # the dominant kernel alone: decode partial launches, back to back, for at
    # least about 0.2 s, enqueued while the GPU sleeps (the host runs ahead)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    n = max(steps, 4000)
    for _ in range(3):
        B.tfpa_decode_partial(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale, sc)
    host_cover(torch)
    ev[0].record(s)
    for _ in range(n):
        B.tfpa_decode_partial(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale, sc)
    ev[1].record(s)
    torch.cuda.synchronize()
    partial_ms = ev[0].elapsed_time(ev[1]) / n
    assert int(cache.err_flag.item()) == 0, "kernel error flag set"
    return step_ms, partial_ms, (cache, segs, q, sc, out), step_ms_again


def time_e2e_graph(w, torch, B, ctx, steps, warmup):
    """Upper bound: the whole step (copies in, kernels, copy out) captured once
    as a CUDA graph and replayed, the host waiting for each step's output.
    The replay repeats one step's kernel parameters (lengths frozen at
    capture), so a decode loop whose lengths advance cannot run this way; the
    inputs are written once, not every step."""
    cache, segs, _, sc, out = ctx
    nst = len(w.streams)
    feed = FreshInputs(w, torch, 1)
    feed.write(0)
    h_in = feed.rows(0)
    d_in = torch.empty(feed.nbytes, dtype=torch.uint8, device="cuda")
    dq, dk, dv = feed.split(d_in)
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    last = np.array([st.seq_len - 1 for st in w.streams], np.int32)
    sidx = np.arange(nst, dtype=np.int32)

    def enqueue():
        d_in.copy_(h_in, non_blocking=True)
        B.tfpa_decode_append(cache, segs, dk, dv, dq, sidx, last, w.softmax_scale, sc, out)
        hout.copy_(out, non_blocking=True)

    for _ in range(warmup):
        enqueue()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            enqueue()
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        graph.replay()
        s.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        graph.replay()
        s.synchronize()
    dt = (time.perf_counter() - t0) / steps
    return dt, graph_device_us(torch, graph.replay, steps)


class FreshInputs:
    """The host's inputs of a decode loop: each step's q rows and new K / V
    rows, written by the host into a pinned buffer while the GPU runs an
    earlier step.  `nbuf` pinned buffers rotate (step i uses buffer
    i % nbuf) and each step copies in one of four seeded sets, so that
    consecutive steps carry new values (a kernel that reads host memory
    cannot find a step's inputs in the GPU's L2).  `extra` bytes follow the
    rows in each buffer (a device-mode plan's packed data)."""

    def __init__(self, w, torch, nbuf, extra=0):
        self.torch, self.w, self.nbuf = torch, w, nbuf
        nst = len(w.streams)
        self.nq, self.nk = w.rows * w.hq * 128, nst * w.hkv * 128
        n = self.nq + 2 * self.nk
        self.nbytes = 2 * n
        g = torch.Generator()
        g.manual_seed(17)
        self.src = [torch.randn(n, generator=g).to(torch.bfloat16).view(torch.int16).numpy()
                    for _ in range(4)]
        self.buf = [torch.zeros(self.nbytes + extra, dtype=torch.uint8).pin_memory()
                    for _ in range(nbuf)]
        self._dst = [b[:self.nbytes].numpy().view(np.int16) for b in self.buf]

    def write(self, i):
        """Step i's inputs into its buffer (the host's part of the step)."""
        np.copyto(self._dst[i % self.nbuf], self.src[i % 4])

    def rows(self, i):
        return self.buf[i % self.nbuf][:self.nbytes]

    def split(self, t):
        """q, K, V views of a row buffer (host or device, uint8)."""
        w, nq, nk = self.w, self.nq, self.nk
        nst = len(w.streams)
        r = t[:self.nbytes].view(self.torch.bfloat16)
        return (r[:nq].view(w.rows, w.hq, 128), r[nq:nq + nk].view(nst, w.hkv, 128),
                r[nq + nk:].view(nst, w.hkv, 128))


def time_e2e_planned(w, torch, B, ctx, steps, warmup):
    """The decode loop of time_e2e_calls, one step at a time, with each step
    planned while the previous one runs: after enqueueing step i the host
    writes step i + 1's inputs and plans it (B.Plan:
    tfpa_plan_decode_append, lengths one position longer), then waits for
    step i's output, then enqueues the next input copy, launches the plan
    and enqueues the output copy.  Returns (s per step, KV + Q + O bytes per
    step, host us per plan launch, host us planning a step)."""
    cache, segs, _, sc, out = ctx
    nst = len(w.streams)
    tab = B.SegTable(segs)
    feed = FreshInputs(w, torch, 2)
    d_in = torch.empty(feed.nbytes, dtype=torch.uint8, device="cuda")
    dq, dk, dv = feed.split(d_in)
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    sidx = np.arange(nst, dtype=np.int32)
    s = torch.cuda.current_stream()
    sh = s.cuda_stream
    L = w.streams[0].seq_len
    total = warmup + steps
    plan = B.Plan()
    ev = torch.cuda.Event()
    b = 2 if w.kv_dtype == "bf16" else 1
    t_launch, t_plan = [], []
    kvb = 0

    def plan_step(i):
        n = L - total + 1 + i
        for j in range(nst):
            tab.set_seq_len(j, n)
        rp = np.full(nst, n - 1, np.int32)
        plan.clear()
        plan.decode_append(cache, tab, dk, dv, dq, sidx, rp, w.softmax_scale, sc, out)
        feed.write(i)
        return n

    n = plan_step(0)
    t0 = None
    for i in range(total):
        if i == warmup:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        d_in.copy_(feed.rows(i), non_blocking=True)
        a = time.perf_counter_ns()
        plan.launch(sh)
        t_launch.append((time.perf_counter_ns() - a) / 1e3)
        hout.copy_(out, non_blocking=True)
        ev.record(s)
        if i >= warmup:
            kvb += n * nst * w.hkv * 128 * 2 * b
        if i + 1 < total:
            a = time.perf_counter_ns()
            n = plan_step(i + 1)                 # while the GPU runs step i
            t_plan.append((time.perf_counter_ns() - a) / 1e3)
        ev.synchronize()
    dt = (time.perf_counter() - t0) / steps
    for j, st in enumerate(w.streams):
        tab.set_seq_len(j, st.seq_len)
    qo = w.rows * w.hq * 128 * 2 * 2
    return dt, kvb / steps + qo, statistics.median(t_launch[warmup:]), statistics.median(t_plan)


def time_e2e_device(w, torch, B, ctx, steps, warmup, zero_copy):
    """The decode loop of time_e2e_planned with plans in device mode
    (tfpa_plan_set_device): each step is still planned anew with lengths one
    position longer, but its launches read their lengths, splits and CTA
    ranges from the plan's buffer, so each plan is captured once as a CUDA
    graph (tfpa_plan_capture) and replayed (tfpa_plan_replay) step after
    step.  Two plans, each with its own pinned buffer (the step's q / K / V
    rows, then the plan's packed data), alternate: while the GPU runs step i
    the host plans step i + 1 on the other plan, packs it
    (tfpa_plan_dyn_pack) and writes that step's inputs into that plan's
    buffer, then waits for step i's output and replays.
    zero_copy: the plans read the rows and the packed data straight from the
    pinned buffer and write the output to pinned memory (the kernels load
    and store over the host link), so a graph holds only the launches.
    Else a graph is one copy of the pinned buffer (rows and packed data) to
    the device, the launches, and the output copy back.
    Returns (s per step, KV + Q + O bytes per step, host us per replay, host
    us planning, packing and writing a step, bytes brought from the host per
    step, bytes sent back, device us per replay)."""
    cache, segs, _, sc, out = ctx
    nst = len(w.streams)
    tab = B.SegTable(segs)
    dyn_cap = 1 << 15
    feed = FreshInputs(w, torch, 2, extra=dyn_cap)
    nin = feed.nbytes                              # a multiple of 16
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    if zero_copy:
        views = [feed.split(hb) for hb in feed.buf]
        dyn = [hb[nin:] for hb in feed.buf]
        dst = hout
    else:
        d = torch.empty(nin + dyn_cap, dtype=torch.uint8, device="cuda")
        views = [feed.split(d)] * 2
        dyn = [d[nin:]] * 2
        dst = out
    sidx = np.arange(nst, dtype=np.int32)
    s = torch.cuda.current_stream()
    sh = s.cuda_stream
    L = w.streams[0].seq_len
    total = warmup + steps
    plans = [B.Plan(), B.Plan()]
    for k in range(2):
        plans[k].set_device(dyn[k])
    ev = torch.cuda.Event()
    b = 2 if w.kv_dtype == "bf16" else 1
    t_launch, t_plan = [], []
    kvb = 0

    def plan_step(i):
        k = i % 2
        n = L - total + 1 + i
        for j in range(nst):
            tab.set_seq_len(j, n)
        rp = np.full(nst, n - 1, np.int32)
        pl = plans[k]
        pl.clear()
        q, kk, vv = views[k]
        pl.decode_append(cache, tab, kk, vv, q, sidx, rp, w.softmax_scale, sc, dst)
        pl.pack(feed.buf[k][nin:])
        feed.write(i)
        return n

    plan_step(1)
    n = plan_step(0)
    nb = plans[0].dyn_bytes()
    if not zero_copy:
        d[:nin + nb].copy_(feed.buf[0][:nin + nb], non_blocking=True)
    plans[0].launch()                              # sets the kernels up before capture
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    for k in range(2):
        if zero_copy:
            plans[k].capture(stream=cap)
        else:
            plans[k].capture(before=[(d, feed.buf[k], nin + nb)],
                             after=[(hout, out, hout.numel() * 2)], stream=cap)
    torch.cuda.synchronize()
    t0 = None
    for i in range(total):
        if i == warmup:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        a = time.perf_counter_ns()
        plans[i % 2].replay(sh)
        t_launch.append((time.perf_counter_ns() - a) / 1e3)
        ev.record(s)
        if i >= warmup:
            kvb += n * nst * w.hkv * 128 * 2 * b
        if i + 1 < total:
            a = time.perf_counter_ns()
            n = plan_step(i + 1)                 # while the GPU runs step i
            t_plan.append((time.perf_counter_ns() - a) / 1e3)
        ev.synchronize()
    dt = (time.perf_counter() - t0) / steps
    last = plans[(total - 1) % 2]
    dev_us = graph_device_us(torch, lambda: last.replay(sh), steps)
    for j, st in enumerate(w.streams):
        tab.set_seq_len(j, st.seq_len)
    qo = w.rows * w.hq * 128 * 2 * 2
    return (dt, kvb / steps + qo, statistics.median(t_launch[warmup:]), statistics.median(t_plan),
            nin + nb, hout.numel() * 2, dev_us)


def graph_device_us(torch, replay, n):
    """Device time of one call of `replay` (a graph replay, its copies
    included): n calls back to back between CUDA events, enqueued during a
    GPU sleep."""
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    replay()
    torch.cuda.synchronize()
    host_cover(torch)
    e0.record(s)
    for _ in range(n):
        replay()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / n


def time_e2e_calls(w, torch, B, ctx, steps, warmup, in_flight=1):
    """A decode loop through the public API with host buffers, one real call
    of each entry point per step.  Every stream's length grows by one each
    step, so every call is planned anew (lengths, splits, CTA ranges): step i
    of n has length L - n + 1 + i (L = the workload's 8,192), writes each
    stream's new K/V row at its last position and decodes that row.  Per step:
    one copy of the step's inputs (q and the new K/V rows, one pinned buffer,
    written by the host while the step before ran) to the device,
    tfpa_decode_append (the new rows stored and decoded), the output copied
    back to pinned host memory, and the host waits for it.  With in_flight =
    2 the host enqueues step i + 1 before it waits for step i's output
    (double-buffered outputs).  Returns (s per step, KV + Q + O bytes per
    step on average, host us per tfpa_decode_append call, 0.0, h2d bytes,
    d2h bytes)."""
    cache, segs, _, sc, out0 = ctx
    nst = len(w.streams)
    assert list(w.row_seg) == list(range(nst)), "one decode row per stream"
    tab = B.SegTable(segs)
    feed = FreshInputs(w, torch, in_flight + 1)
    d_in = [torch.empty(feed.nbytes, dtype=torch.uint8, device="cuda") for _ in range(in_flight)]
    dviews = [feed.split(d) for d in d_in]
    houts = [torch.empty(out0.shape, dtype=out0.dtype).pin_memory() for _ in range(in_flight)]
    outs = [out0] + [torch.empty_like(out0) for _ in range(in_flight - 1)]
    evs = [torch.cuda.Event() for _ in range(in_flight)]
    sidx = np.arange(nst, dtype=np.int32)
    pos = [np.zeros(nst, np.int32) for _ in range(in_flight)]
    s = torch.cuda.current_stream()
    sh = s.cuda_stream
    L = w.streams[0].seq_len
    assert all(st.seq_len == L for st in w.streams)
    total = warmup + steps
    t_w, t_d = [], []
    b, kvb = (2 if w.kv_dtype == "bf16" else 1), 0

    def enqueue(i, k):
        dq, dk, dv = dviews[k]
        n = L - total + 1 + i
        for j in range(nst):
            tab.set_seq_len(j, n)
        rp = pos[k]
        rp.fill(n - 1)
        d_in[k].copy_(feed.rows(i), non_blocking=True)
        t0 = time.perf_counter_ns()
        B.tfpa_decode_append(cache, tab, dk, dv, dq, sidx, rp, w.softmax_scale, sc, outs[k],
                             stream=sh)
        t1 = time.perf_counter_ns()
        houts[k].copy_(outs[k], non_blocking=True)
        evs[k].record(s)
        return n, (t1 - t0) / 1e3, 0.0

    def run(first, count, keep):
        nonlocal kvb
        for i in range(first, first + count):
            k = i % in_flight
            if i - first >= in_flight:
                evs[k].synchronize()            # the output of step i - in_flight is home
            n, a, d = enqueue(i, k)
            feed.write(i + 1)     # its buffer's last step, i - in_flight, is done
            if keep:
                t_w.append(a)
                t_d.append(d)
                kvb += n * nst * w.hkv * 128 * 2 * b
        for k in range(in_flight):
            evs[k].synchronize()

    feed.write(0)
    run(0, warmup, False)
    t0 = time.perf_counter()
    run(warmup, steps, True)
    dt = (time.perf_counter() - t0) / steps
    for j, st in enumerate(w.streams):          # back to the workload's lengths
        tab.set_seq_len(j, st.seq_len)
    qo = w.rows * w.hq * 128 * 2 * 2
    return (dt, kvb / steps + qo, statistics.median(t_w), statistics.median(t_d), feed.nbytes,
            houts[0].numel() * 2)


def host_cover(torch):
    """A GPU sleep of about 200 us before a per-call timing's first event:
    the host plans and enqueues the call while the GPU sleeps, so the events
    bracket the call's device work back to back (as a CUDA graph would),
    not the host's planning."""
    torch.cuda._sleep(400_000)


class L2Flush:
    """Leaves the 129 MB L2 holding nothing a timed call can use, and nothing
    dirty: a 256 MB write evicts every line, then a read of a second 256 MB
    buffer writes the dirty lines back, both before the timed region, so the
    timed call neither hits in L2 nor pays for the flush's write-back."""

    def __init__(self, torch):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")

    def __call__(self, i):
        self.w.fill_(i & 0xFF)
        self.r.max()


def time_prefill(w, torch, B, reps):
    """One launch per rep, L2 flushed between reps, CUDA events around each."""
    cache, segs, _ = device_case(w, torch, B)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    q = torch.randn(w.rows, w.hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    flush = L2Flush(torch)
    s = torch.cuda.current_stream()
    times = []
    for i in range(reps + 2):
        flush(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        host_cover(torch)
        e0.record(s)
        B.tfpa_prefill(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale, out)
        e1.record(s)
        torch.cuda.synchronize()
        if i >= 2:
            times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def time_store_and_keep(w, torch, B, reps):
    """tfpa_write_kv_rope of every chunk row and tfpa_keep_kv of 256 rows, one
    call at a time, L2 flushed before each, CUDA events; medians in ms."""
    cache, segs, _ = device_case(w, torch, B)
    g = torch.Generator(device="cuda")
    g.manual_seed(13)
    k = torch.randn(w.rows, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(w.rows, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    n_pos = int(w.row_pos.max()) + 1
    cos, sin = wl_rope(n_pos)
    cos, sin = torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda()
    base = int(w.row_pos.min())
    ks = np.zeros(256, np.int32)
    src = (base + 2 * np.arange(256) + 1).astype(np.int32)
    dst = (base + 1024 + np.arange(256)).astype(np.int32)
    flush = L2Flush(torch)
    s = torch.cuda.current_stream()
    t_store, t_keep = [], []
    for i in range(reps + 3):
        for fn, acc in ((lambda: B.tfpa_write_kv_rope(cache, segs, k, v, w.row_seg, w.row_pos,
                                                      cos, sin), t_store),
                        (lambda: B.tfpa_keep_kv(cache, segs, ks, src, dst), t_keep)):
            flush(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            host_cover(torch)
            e0.record(s)
            fn()
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 3:
                acc.append(e0.elapsed_time(e1))
    assert int(cache.err_flag.item()) == 0, "kernel error flag set"
    return statistics.median(t_store), statistics.median(t_keep)


def time_save_restore(w, torch, B, reps):
    """tfpa_save_kv / tfpa_restore_kv of a whole 32k-position stream to and
    from pinned host memory, next to plain runtime copies of the same byte
    count (device -> pinned host, and back) as the link's reference; medians
    in ms: (save, restore, d2h copy, h2d copy)."""
    cache, segs, _ = device_case(w, torch, B)
    seg = segs[0]
    L = w.streams[0].seq_len
    nbytes = 2 * w.hkv * L * 128 * 2
    img = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    out = {k: [] for k in ("save", "restore", "d2h", "h2d")}
    ops = (("save", lambda: B.tfpa_save_kv(cache, seg, 0, L, img)),
           ("restore", lambda: B.tfpa_restore_kv(cache, seg, 0, L, img)),
           ("d2h", lambda: img.copy_(dev, non_blocking=True)),
           ("h2d", lambda: dev.copy_(img, non_blocking=True)))
    for i in range(reps + 2):
        for name, fn in ops:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            host_cover(torch)
            e0.record(s)
            fn()
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 2:
                out[name].append(e0.elapsed_time(e1))
    assert int(cache.err_flag.item()) == 0, "kernel error flag set"
    return nbytes, {k: statistics.median(v) for k, v in out.items()}


def time_page_staging(w, torch, B, reps):
    """Two consecutive prompt chunks of the prompt-chunk workload (rows
    28,672..30,719, then 30,720..32,767; 8 new pages each).  Before each chunk
    its 8 page ids are written into the stream's device page table, then its
    K/V rows are stored (tfpa_write_kv) and its attention runs (tfpa_prefill).
    The ids are written three ways: tfpa_stage_pages (ids in the launch
    parameters), a copy from pinned host memory (cudaMemcpyAsync), and a copy
    from pageable host memory, which the runtime performs only after the
    stream's earlier work has finished, so the host stops between chunks.
    CUDA events around both chunks, host enqueue included (no GPU sleep
    first), L2 flushed before each pair; median ms per pair of chunks."""
    cache, segs, _ = device_case(w, torch, B)
    table = segs[0].page_table
    ids = np.ascontiguousarray(w.streams[0].page_table, np.int32)
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    q = torch.randn(w.rows, w.hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(w.rows, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(w.rows, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    half = w.rows // 2
    chunks = []
    for c in range(2):
        rp = np.ascontiguousarray(w.row_pos[c * half:(c + 1) * half])
        first = int(rp[0]) // 256
        n = half // 256
        host = ids[first:first + n].copy()
        chunks.append((c, rp, first, n, host, torch.from_numpy(host).pin_memory(),
                       torch.from_numpy(host.copy())))
    rs = np.zeros(half, np.int32)
    flush = L2Flush(torch)
    s = torch.cuda.current_stream()

    def pair(mode):
        for c, rp, first, n, host, pinned, pageable in chunks:
            if mode == "stage":
                B.tfpa_stage_pages(table, first, host)
            elif mode == "pinned_copy":
                table[first:first + n].copy_(pinned, non_blocking=True)
            else:
                table[first:first + n].copy_(pageable)
            sl = slice(c * half, (c + 1) * half)
            B.tfpa_write_kv(cache, segs, k[sl], v[sl], rs, rp)
            B.tfpa_prefill(cache, segs, q[sl], rs, rp, w.softmax_scale, out[sl])

    times = {m: [] for m in ("stage", "pinned_copy", "pageable_copy")}
    for i in range(reps + 2):
        for m in times:
            flush(i)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            pair(m)
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 2:
                times[m].append(e0.elapsed_time(e1))
    assert int(cache.err_flag.item()) == 0, "kernel error flag set"
    return {m: statistics.median(t) for m, t in times.items()}


def wl_rope(n_pos):
    from paged_kv_cache_235_gb300 import workloads as wl
    return wl.rope_table(1e6, n_pos)


def time_tree_calls(w, torch, B, reps):
    """tfpa_decode_tree one call at a time, CUDA events around each; median ms."""
    cache, segs, q = device_case(w, torch, B)
    anc = torch.from_numpy(np.ascontiguousarray(w.row_anc).view(np.int64)).cuda()
    sc = B.make_scratch(min(128, w.rows), w.hq)
    out = torch.empty(w.rows, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream()
    times = []
    for i in range(reps + 3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        host_cover(torch)
        e0.record(s)
        B.tfpa_decode_tree(cache, segs, q, w.row_seg, w.row_pos, anc, w.softmax_scale, sc, out)
        e1.record(s)
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1))
    assert int(cache.err_flag.item()) == 0, "kernel error flag set"
    return statistics.median(times)


def time_decode_calls(w, torch, B, reps, flush, fused_merge=True):
    """tfpa_decode (partial + merge) one call at a time, CUDA events around
    each, optionally with L2 flushed before each call; median in ms."""
    cache, segs, q = device_case(w, torch, B)
    sc = B.make_scratch(min(128, w.rows), w.hq, fused_merge=fused_merge)
    out = torch.empty(w.rows, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    buf = L2Flush(torch) if flush else None
    s = torch.cuda.current_stream()
    times = []
    for i in range(reps + 3):
        if buf is not None:
            buf(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        host_cover(torch)
        e0.record(s)
        B.tfpa_decode(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale, sc, out)
        e1.record(s)
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1))
    assert int(cache.err_flag.item()) == 0, "kernel error flag set"
    return statistics.median(times)


def time_tiny_layer_calls(torch, B, wl, layers=32, reps=20):
    """The tiny decode as one layer of a model's decode step: `layers` calls,
    each with its own pool, page table, queries and scratch (1 MB of KV
    each), captured after an L2 flush as one CUDA graph; per call = (graph -
    the same flush alone) / layers, medians over `reps` replays.  The first
    call meets a cold instruction cache, the others a warm one (no other
    kernels run between them), and every call's KV is cold."""
    cases = []
    for i in range(layers):
        w = wl.tiny_paged_decode(seed=500 + i)
        cache, segs, q = device_case(w, torch, B)
        sc = B.make_scratch(1, w.hq)
        out = torch.empty(w.rows, w.hq, 128, dtype=torch.bfloat16, device="cuda")
        cases.append((w, cache, segs, q, sc, out))
    flush = L2Flush(torch)

    def calls():
        for w, cache, segs, q, sc, out in cases:
            B.tfpa_decode(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale, sc, out)

    calls()                                    # per-device set-up before capture
    flush(0)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g_all, g_flush = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g_all, stream=cap):
            flush(1)
            calls()
        with torch.cuda.graph(g_flush, stream=cap):
            flush(1)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()

    def med(g):
        t = []
        for i in range(reps + 3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 3:
                t.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(t)

    t_all, t_flush = med(g_all), med(g_flush)
    for _, cache, _, _, _, _ in cases:
        assert int(cache.err_flag.item()) == 0, "kernel error flag set"
    return (t_all - t_flush) / layers, t_all, t_flush


def time_launch_floor(torch, reps=40):
    """The event-timing floor of a call: an empty event pair, and one and two
    one-element torch kernels between the events (same method as the
    per-call lines: a GPU sleep first, medians in us)."""
    s = torch.cuda.current_stream()
    x = torch.zeros(1, device="cuda")

    def med(fn):
        t = []
        for i in range(reps + 3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            host_cover(torch)
            e0.record(s)
            fn()
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 3:
                t.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(t)

    return {"event_pair_us": med(lambda: None), "one_kernel_us": med(lambda: x.add_(1)),
            "two_kernels_us": med(lambda: (x.add_(1), x.add_(1)))}


def profile_case(args, torch, B, wl):
    """One workload's kernels only, for profiler captures (a small launch list)."""
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    if args.case in ("prefill", "prefill_fp8"):
        w = wl.prompt_chunk(kv_dtype="fp8" if args.case == "prefill_fp8" else "bf16")
        ms = time_prefill(w, torch, B, args.steps)
        print(f"{args.case}: {ms:.4f} ms, {prefill_flops(w) / ms / 1e9:.1f} TFLOP/s")
        return
    if args.case in ("tree_verify", "tree_verify_bf16"):
        w = wl.tree_verify(kv_dtype="bf16" if args.case == "tree_verify_bf16" else "fp8")
    else:
        w = wl.batched_decode() if args.case == "decode" else wl.fp8_verify()
    cache, segs, q = device_case(w, torch, B)
    sc = B.make_scratch(min(128, w.rows), w.hq)
    out = torch.empty(w.rows, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    anc = None
    if w.row_anc is not None:
        anc = torch.from_numpy(np.ascontiguousarray(w.row_anc).view(np.int64)).cuda()
    for _ in range(args.warmup + args.steps):
        if anc is None:
            B.tfpa_decode(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale, sc, out)
        else:
            B.tfpa_decode_tree(cache, segs, q, w.row_seg, w.row_pos, anc, w.softmax_scale, sc,
                               out)
    torch.cuda.synchronize()
    assert int(cache.err_flag.item()) == 0, "kernel error flag set"
    print(f"{args.case}: {args.warmup + args.steps} decode calls done")


# --------------------------------------------------------------------- main
def reference_arm(args):
    """The CPU oracle as the reference arm: same metric, config and unit."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for _ in range(args.warmup):
        cpu_oracle_sample(seconds=0.0)
    secs = []
    base = None
    for _ in range(args.steps):
        base = cpu_oracle_sample(seconds=0.0)
        secs.append(base["s_per_call"] * 8)          # 8 streams make one step
    from paged_kv_cache_235_gb300 import workloads as wl
    w = wl.batched_decode()
    kv, qo = kv_bytes(w)
    ms = statistics.mean(secs) * 1e3
    value = (kv + qo) / (ms / 1e3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) rounded to bf16)",
        "config": {"workload": "batched_decode: 8 streams x 8,192 positions, 32/8 heads, "
                               "head_dim 128, bf16 KV, streams 0-3 slabs, 4-7 paged",
                   "sample": "each step runs stream 0 once and counts it 8 times"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": base["sample"]},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--case", default=None,
                    choices=["decode", "fp8_verify", "prefill", "prefill_fp8", "tree_verify",
                             "tree_verify_bf16"],
                    help="profiling mode: run only this workload's kernels --steps times "
                         "after --warmup, print its timing, no JSON line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        reference_arm(args)
        return

    import torch
    from paged_kv_cache_235_gb300 import binding as B
    from paged_kv_cache_235_gb300 import workloads as wl

    if args.case:
        profile_case(args, torch, B, wl)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    B.lib()
    pk = peaks()
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample()      # before any timed GPU work

    w = wl.batched_decode()
    kv, qo = kv_bytes(w)
    extra = {}
    w3 = wl.fp8_verify()
    kv3, qo3 = kv_bytes(w3)
    with ClockSampler(local) as clk:
        step_ms, partial_ms, ctx, step_ms_aa = time_decode(w, torch, B, args.steps, args.warmup,
                                                          dist)
        step_ms = max_over_ranks(dist, torch, step_ms)
        n_e2e = max(10, min(args.steps, 500))
        e2e = time_e2e_calls(w, torch, B, ctx, n_e2e, args.warmup)
        e2e_s = max_over_ranks(dist, torch, e2e[0])
        e2e_pipe = time_e2e_calls(w, torch, B, ctx, n_e2e, args.warmup, in_flight=2)
        e2e_plan = time_e2e_planned(w, torch, B, ctx, n_e2e, args.warmup)
        e2e_plan = (max_over_ranks(dist, torch, e2e_plan[0]),) + tuple(e2e_plan[1:])
        e2e_plan_aa = time_e2e_planned(w, torch, B, ctx, n_e2e, args.warmup)
        e2e_graph_s, e2e_graph_dev_us = time_e2e_graph(w, torch, B, ctx, n_e2e, args.warmup)
        # three runs of the loop; the line reports the median run and lists
        # all three (a transient on the shared host can slow one run)
        e2e_runs = [time_e2e_device(w, torch, B, ctx, n_e2e, args.warmup, zero_copy=True)
                    for _ in range(3)]
        e2e_runs = [(max_over_ranks(dist, torch, r[0]),) + tuple(r[1:]) for r in e2e_runs]
        e2e_dev = sorted(e2e_runs, key=lambda r: r[0])[1]
        ce_runs = [time_e2e_device(w, torch, B, ctx, n_e2e, args.warmup, zero_copy=False)
                   for _ in range(3)]
        ce_runs = [(max_over_ranks(dist, torch, r[0]),) + tuple(r[1:]) for r in ce_runs]
        e2e_ce = sorted(ce_runs, key=lambda r: r[0])[1]
        del ctx
        s3, p3, ctx3, _ = time_decode(w3, torch, B, max(10, args.steps // 4), args.warmup, None)
        del ctx3
        if not args.skip_prefill:
            w4 = wl.prompt_chunk()
            try:
                ms4 = time_prefill(w4, torch, B, 5)
                fl = prefill_flops(w4)
                extra["prefill"] = {
                    "workload": "28,672-position paged prefix + 4,096-row causal chunk, "
                                "32/8 heads, bf16, one launch, L2 flushed before each",
                    "ms_per_call": ms4, "tflops": fl / (ms4 / 1e3) / 1e12,
                    "frac_of_measured_bf16": fl / (ms4 / 1e3) / 1e12 / pk["bf16_tflops"],
                    "kernel": "prefill_kernel (tcgen05)"}
            except B.TfpaError as e:
                extra["prefill"] = {"unavailable": str(e)}
            w5 = wl.prompt_chunk(kv_dtype="fp8")
            ms5 = time_prefill(w5, torch, B, 5)
            fl5 = prefill_flops(w5)
            extra["prefill_fp8"] = {
                "workload": "the same prompt chunk over an e4m3 cache (f16 MMAs)",
                "ms_per_call": ms5, "tflops": fl5 / (ms5 / 1e3) / 1e12,
                "frac_of_measured_bf16": fl5 / (ms5 / 1e3) / 1e12 / pk["bf16_tflops"]}
        w1 = wl.tiny_paged_decode()
        ms1 = time_decode_calls(w1, torch, B, 50, flush=True)
        ms1s = time_decode_calls(w1, torch, B, 50, flush=True, fused_merge=False)
        kv1, qo1 = kv_bytes(w1)
        extra["tiny_decode"] = {
            "workload": "1 stream, 1 row at position 999, 8/2 heads, bf16, 4 of 16 pool pages; "
                        "tfpa_decode per call, L2 flushed before each",
            "us_per_call": ms1 * 1e3, "kv_gbs": (kv1 + qo1) / (ms1 / 1e3) / 1e9,
            "frac_of_measured_hbm": (kv1 + qo1) / (ms1 / 1e3) / 1e9 / pk["hbm_gbs"],
            "merge": "inside the partial kernel (scratch with arrival counters)",
            "us_per_call_separate_merge": ms1s * 1e3,
            "timing_floor": time_launch_floor(torch),
            "note": "1 MB of KV: launch and latency bound, the HBM roofline is out of reach; "
                    "timing_floor is the same event method around nothing and around one "
                    "and two one-element kernels"}
        lc, lc_all, lc_flush = time_tiny_layer_calls(torch, B, wl)
        extra["tiny_decode"]["layer_calls"] = {
            "workload": "32 calls of the same shape, each on its own 1 MB of KV (own pool, "
                        "page table, queries, scratch), one CUDA graph after an L2 flush, as "
                        "one attention call per layer of a decode step",
            "us_per_call": lc, "graph_us": lc_all, "flush_us": lc_flush,
            "note": "(graph - flush alone) / 32; every call's KV is cold, the instruction "
                    "cache is warm after the first call"}
        w6 = wl.overcommitted_pool()
        ms6 = time_decode_calls(w6, torch, B, 20, flush=False)
        kv6, qo6 = kv_bytes(w6)
        extra["overcommitted_pool"] = {
            "workload": "16 streams of U[1k,109k] positions + one of 262,144, fp8, 32/8 heads, "
                        "first-fit pool of 5,078 pages after seeded churn, 1 row each; "
                        "tfpa_decode per call",
            "seated_streams": len(w6.streams), "waiting_streams": len(w6.waiting),
            "us_per_call": ms6 * 1e3, "kv_gbs": (kv6 + qo6) / (ms6 / 1e3) / 1e9,
            "frac_of_measured_hbm": (kv6 + qo6) / (ms6 / 1e3) / 1e9 / pk["hbm_gbs"]}
        w8 = wl.prompt_chunk()
        ms_st, ms_kp = time_store_and_keep(w8, torch, B, 20)
        st_bytes = w8.rows * w8.hkv * 128 * 2 * (2 + 2) + w8.rows * 64 * 4 * 2
        kp_bytes = 256 * w8.hkv * 2 * 256 * 2
        extra["kv_store_rope"] = {
            "workload": "4,096 prompt-chunk rows into a paged bf16 cache, 8 kv heads, K rotated "
                        "by its position (float32 cos/sin table); L2 flushed before each call",
            "us_per_call": ms_st * 1e3, "gbs": st_bytes / (ms_st / 1e3) / 1e9,
            "frac_of_measured_hbm": st_bytes / (ms_st / 1e3) / 1e9 / pk["hbm_gbs"],
            "bytes": st_bytes}
        extra["keep"] = {
            "workload": "256 stored rows (8 kv heads, K and V, bf16) moved within one paged "
                        "stream in one call; L2 flushed before each call",
            "us_per_call": ms_kp * 1e3, "gbs": kp_bytes / (ms_kp / 1e3) / 1e9,
            "note": "2 MB moved: launch and latency bound"}
        w9 = wl.prompt_chunk(prefix=28672, chunk=4096)
        nb9, t9 = time_save_restore(w9, torch, B, 10)
        gbs = {k: nb9 / (v / 1e3) / 1e9 for k, v in t9.items()}
        extra["save_restore"] = {
            "workload": "one 32,768-position bf16 stream, 8 kv heads (134 MB of K and V), saved "
                        "to and restored from pinned host memory by one kernel each",
            "bytes": nb9, "save_ms": t9["save"], "restore_ms": t9["restore"],
            "save_gbs": gbs["save"], "restore_gbs": gbs["restore"],
            "runtime_copy_gbs": {"d2h": gbs["d2h"], "h2d": gbs["h2d"]},
            "frac_of_runtime_copy": {"save": gbs["save"] / gbs["d2h"],
                                     "restore": gbs["restore"] / gbs["h2d"]},
            "note": "the reference is a plain runtime copy of the same byte count between a "
                    "contiguous device buffer and the same pinned buffer"}
        w10 = wl.prompt_chunk()
        t10 = time_page_staging(w10, torch, B, 10)
        extra["page_staging"] = {
            "workload": "two consecutive 2,048-row prompt chunks (positions 28,672..32,767, bf16, "
                        "32/8 heads), each preceded by writing its 8 page ids into the device "
                        "page table, then tfpa_write_kv and tfpa_prefill; host enqueue included, "
                        "L2 flushed before each pair",
            "ms_per_two_chunks": t10,
            "gap_us_per_chunk_vs_stage": {m: (t - t10["stage"]) * 1e3 / 2
                                          for m, t in t10.items() if m != "stage"},
            "note": "stage = tfpa_stage_pages (ids in kernel parameters); pinned_copy = "
                    "cudaMemcpyAsync from pinned memory; pageable_copy = a copy from pageable "
                    "memory, which waits for the stream's earlier work (the host stops between "
                    "chunks)"}
        for kvd in ("fp8", "bf16"):
            w7 = wl.tree_verify(kv_dtype=kvd)
            ms7 = time_tree_calls(w7, torch, B, 20)
            kv7, qo7 = kv_bytes(w7)
            extra["tree_verify" + ("" if kvd == "fp8" else "_bf16")] = {
                "workload": f"8 streams x 65,536 positions, {kvd} KV, a seeded 16-node draft "
                            "tree per stream (one row per node, ancestor masks); "
                            "tfpa_decode_tree per call",
                "ms_per_call": ms7, "kv_gbs": (kv7 + qo7) / (ms7 / 1e3) / 1e9,
                "frac_of_measured_hbm": (kv7 + qo7) / (ms7 / 1e3) / 1e9 / pk["hbm_gbs"]}
    value = world * (kv + qo) / (step_ms / 1e3) / 1e9
    achieved = (kv + qo) / (partial_ms / 1e3) / 1e9
    extra["fp8_verify"] = {
        "workload": "8 streams x 65,536 positions, 4 causal verify rows each, fp8 e4m3 KV",
        "ms_per_call": s3, "kv_gbs": (kv3 + qo3) / (s3 / 1e3) / 1e9,
        "partial_ms": p3, "partial_gbs": (kv3 + qo3) / (p3 / 1e3) / 1e9,
        "frac_of_measured_hbm": (kv3 + qo3) / (p3 / 1e3) / 1e9 / pk["hbm_gbs"]}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) rounded to bf16; pages from a seeded permutation)",
        "config": {"workload": "batched_decode: 8 streams x 8,192 positions, 1 row each, "
                               "32/8 heads, head_dim 128, bf16 KV, streams 0-3 slabs, 4-7 "
                               "paged in a 512-page pool; step = tfpa_decode_append (the new rows' K/V "
                               "stored, then decoded)",
                   "l2": "no flush: 268 MB of KV per step exceeds the 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": decode_traffic(),
                     "kernel": "decode_partial_kernel<bf16>", "peak_source": pk["source"],
                     "partial_ms": partial_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": world * e2e_dev[1] / e2e_dev[0] / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": e2e_dev[4], "d2h_bytes_per_step": e2e_dev[5],
                "h2d_copies_per_step": 0,
                "transfer": "zero-copy: the kernels read the step's q, new K/V rows and packed "
                            "plan data from pinned host memory and the merge writes the output "
                            "to pinned host memory, over the host link (NVLink-C2C), inside "
                            "the timed step; the host writes each step's inputs anew",
                "ms_per_step": e2e_dev[0] * 1e3, "vs_device_step": e2e_dev[0] * 1e3 / step_ms,
                "host_us_per_call": {"tfpa_plan_replay": e2e_dev[2],
                                     "planning_packing_and_writing_a_step_overlapped":
                                         e2e_dev[3]},
                "steps": n_e2e,
                "how": "a decode loop through the public API with host buffers, one step at a "
                       "time: each stream one position longer every step (%d..%d), every step "
                       "planned anew (tfpa_plan_decode_append, two plans in device "
                       "mode, alternating) and packed (tfpa_plan_dyn_pack) into its plan's "
                       "pinned buffer, and its inputs written there by the host, while the "
                       "previous step runs; per step one tfpa_plan_replay of the plan's CUDA "
                       "graph (tfpa_plan_capture, once per plan: the planned launches); the "
                       "host waits for the output before the next step; host times are host "
                       "clock, median" % (w.streams[0].seq_len - n_e2e + 1, w.streams[0].seq_len),
                "packed_bytes_per_step": e2e_dev[4] - e2e[4],
                "graph_device_us_per_step": e2e_dev[6],
                "copy_engine": {
                    "value": world * e2e_ce[1] / e2e_ce[0] / 1e9, "unit": "GB/s",
                    "ms_per_step": e2e_ce[0] * 1e3, "vs_device_step": e2e_ce[0] * 1e3 / step_ms,
                    "h2d_bytes_per_step": e2e_ce[4], "d2h_bytes_per_step": e2e_ce[5],
                    "h2d_copies_per_step": 1,
                    "host_us_per_call": {"tfpa_plan_replay": e2e_ce[2]},
                    "graph_device_us_per_step": e2e_ce[6],
                    "how": "the same loop with the inputs, packed data and output in device "
                           "memory: each graph is one copy of the pinned buffer (rows and "
                           "packed data) to the device, the launches and the output copy"},
                "planned_calls": {
                    "value": world * e2e_plan[1] / e2e_plan[0] / 1e9, "unit": "GB/s",
                    "ms_per_step": e2e_plan[0] * 1e3,
                    "vs_device_step": e2e_plan[0] * 1e3 / step_ms,
                    "host_us_per_call": {"tfpa_plan_launch": e2e_plan[2],
                                         "planning_a_step_overlapped": e2e_plan[3]},
                    "how": "the same loop with the plan in parameter mode: tfpa_plan_launch "
                           "enqueues the planned launches each step (no graph)"},
                "direct_calls": {
                    "value": world * e2e[1] / e2e_s / 1e9, "unit": "GB/s",
                    "ms_per_step": e2e_s * 1e3, "vs_device_step": e2e_s * 1e3 / step_ms,
                    "host_us_per_call": {"tfpa_decode_append": e2e[2]},
                    "how": "the same loop calling tfpa_decode_append directly "
                           "(planning and launching inside each call)"}},
        "e2e_aa_repeat": {"ms_per_step": [r[0] * 1e3 for r in e2e_runs],
                          "spread_pct": 100 * (max(r[0] for r in e2e_runs) -
                                               min(r[0] for r in e2e_runs)) / e2e_dev[0],
                          "reported": "median of the three runs",
                          "copy_engine_ms_per_step": [r[0] * 1e3 for r in ce_runs],
                          "planned_calls_ms_per_step": [e2e_plan[0] * 1e3, e2e_plan_aa[0] * 1e3]},
        "e2e_two_in_flight": {
            "value": world * e2e_pipe[1] / e2e_pipe[0] / 1e9, "unit": "GB/s",
            "ms_per_step": e2e_pipe[0] * 1e3,
            "host_us_per_call": {"tfpa_decode_append": e2e_pipe[2]},
            "how": "the same loop with step i + 1 enqueued before the host waits for step "
                   "i's output (two input and output buffers)"},
        "e2e_graph_replay": {
            "value": world * (kv + qo) / e2e_graph_s / 1e9, "unit": "GB/s",
            "ms_per_step": e2e_graph_s * 1e3,
            "graph_device_us_per_step": e2e_graph_dev_us,
            "how": "upper bound: one step (copies, 2 kernels) captured once as a CUDA graph "
                   "and replayed with its lengths frozen; no host planning per step"},
        "aa_repeat": {"ms_per_step": [step_ms, step_ms_aa],
                      "spread_pct": 100 * abs(step_ms_aa - step_ms) / step_ms},
        "gpu_launches": 2 * args.steps,
        "timing": "decode step = one CUDA-graph replay of tfpa_decode_append "
                  "(2 kernels: partial with the rows' store, merge), CUDA events over --steps replays (device time); e2e = real "
                  "planned calls per step, host clock (see e2e.how); the per-call lines (prefill, "
                  "tiny_decode, overcommitted_pool, tree_verify, kv_store_rope, keep, "
                  "save_restore) are device time: CUDA events around one call, enqueued by "
                  "the host during a preceding GPU sleep",
        "clocks": clk.summary(),
        **extra,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
