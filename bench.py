"""Benchmark: paged decode HBM GB/s (and prefill TFLOP/s) on seeded inputs.

One step = the whole hot path over one batch: reshape_and_cache of the new
K/V rows, then paged attention (decode kernel, split-KV partials folded by
LSE).  The timed workload is the batched Llama-3-8B-shape decode: 64
requests, query_len 1, 32/8 heads, D 128, block_size 16, lengths U[512, 4096]
from a shuffled 20k-block pool, bf16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  ``value`` is the algorithmic bytes of a step
(admissible KV rows, Q, O, block-table rows, seqused/cu_seqlens, and the
new K/V rows read and written by the cache write) divided by the device time
per step, summed over ranks.  ``--impl reference`` times the float64 CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

# the CPU oracle legs run single-threaded numpy; say so by construction
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_318_gb300 import _build, api, workloads  # noqa: E402
from paged_kv_cache_318_gb300.batch import DeviceBatch  # noqa: E402

METRIC = ("paged decode HBM GB/s & prefill attn TFLOP/s "
          "(% of GB300 roofline)")
UNIT = "GB/s"
SEED_DECODE = 319
SEED_PREFILL = 320
CLOCK_SOAK_S = 0.5      # seconds of extra load for the clock samples


# --------------------------------------------------------------- accounting
def decode_bytes(wl) -> dict:
    """Algorithmic bytes of one decode step (what the method must move)."""
    e = 2  # bf16
    Hq, Hkv, D, BS = wl.num_heads, wl.num_kv_heads, wl.head_size, \
        wl.block_size
    L = wl.seq_lens.astype(np.int64)
    T = wl.num_tokens
    kv = int(L.sum()) * 2 * Hkv * D * e
    qo = 2 * T * Hq * D * e
    tables = int((-(-L // BS)).sum()) * 4 + wl.batch * 4 + (wl.batch + 1) * 4
    cache_write = T * Hkv * D * e * 2 * 2 + T * 8
    return dict(kv=kv, qo=qo, tables=tables, cache_write=cache_write,
                attention=kv + qo + tables,
                step=kv + qo + tables + cache_write)


def prefill_flops(wl, min_rows=0) -> float:
    """QK^T + PV flops over admissible (query, key) pairs (causal, with the
    workload's left window), of requests with at least ``min_rows`` packed
    query rows."""
    G = wl.num_heads // wl.num_kv_heads
    left = wl.window_size[0]
    total = 0
    for b in range(wl.batch):
        q, L = int(wl.q_lens[b]), int(wl.seq_lens[b])
        if q * G < min_rows:
            continue
        c = L - q
        for i in range(q):
            n = c + i + 1                            # causal keys
            total += n if left < 0 else min(n, left + 1)
    return 4.0 * wl.head_size * wl.num_heads * total


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), \
            "measured"
    return 6800.0, 1900.0, "fallback"


def ncu_traffic(kernel_tag):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source (null otherwise)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "%s_traffic.txt" % kernel_tag)
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    h = hashlib.sha256()
    for name in fields.get("source", "").split(","):
        src = os.path.join(ROOT, "paged_kv_cache_318_gb300", "csrc",
                           name.strip())
        if not name.strip() or not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    h = h.hexdigest()[:16]
    if fields.get("source_sha256_16") != h:
        return None
    try:
        return float(fields["dram_bytes_per_launch_full_workload"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background.

    A reader thread timestamps every sample, so the summary can be limited
    to the window between ``begin()`` and ``end()``."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        import threading
        self.proc = None
        self.lines = []                     # (time, line)
        self.window = [None, None]
        self.first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index),
                 "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        self.first.wait(timeout=10.0)       # sampling has started

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line))
            self.first.set()

    def begin(self):
        self.window[0] = time.time()

    def end(self):
        self.window[1] = time.time()

    def stop(self, label):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=5)
        t0, t1 = self.window
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for t, line in self.lines:
            if t0 is not None and (t < t0 or (t1 is not None and t > t1)):
                continue
            parts = [p.strip() for p in line.split(",")]
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
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "window": label}


# ------------------------------------------------------------ multi-rank
def max_over_ranks(values, device, world):
    """Element-wise max of per-rank timings (the slowest rank sets the pace
    of a weak-scaling step)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def aggregate_value(bytes_per_rank_step, step_ms, world):
    """Whole-job GB/s: every rank moves its own batch per step."""
    return world * bytes_per_rank_step / (step_ms * 1e-3) / 1e9


# ---------------------------------------------------------------- GPU arm
def time_steps(fn, steps, stream, attn_events=None):
    """Total device ms of ``steps`` calls of fn on ``stream``."""
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        fn(i)
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop)


def gpu_arm(args, rank, world, dev):
    hbm_peak, tf_peak, peak_src = measured_peaks()
    wl = workloads.batched_decode(seed=SEED_DECODE, device=dev)
    batch = DeviceBatch(wl, dev, poison=False)
    batch.write_context()
    stream = torch.cuda.current_stream(dev)
    acct = decode_bytes(wl)

    # per-step events around the attention call (decode + split combine)
    n_ev = args.steps
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    timing = {"on": False}

    def step(i):
        batch.write_new()
        if timing["on"]:
            ev_a[i].record(stream)
        batch.attend(return_lse=False)
        if timing["on"]:
            ev_b[i].record(stream)

    clocks = ClockSampler(dev.index or 0)
    clocks.begin()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    launches0 = api.launch_count()
    ms = time_steps(step, args.steps, stream)
    launches = api.launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    # the attention call's own time: the same steps again, with events
    # around each call (kept out of the step timing above)
    timing["on"] = True
    time_steps(step, args.steps, stream)
    timing["on"] = False
    attn_ms = float(np.mean([a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]))
    # the timed region is shorter than the sampling interval: keep the same
    # step running for CLOCK_SOAK_S more so the samples see this load
    t_soak = time.time()
    while time.time() - t_soak < CLOCK_SOAK_S:
        for i in range(20):
            step(0)
        torch.cuda.synchronize()
    clocks.end()
    clk = clocks.stop("warm-up, timed region and %.1f s of the same steps "
                      "right after it" % CLOCK_SOAK_S)
    api.check_device_errors(dev)

    # e2e: same step through the public API from pinned host memory.  The
    # step's inputs live in one pinned host buffer; each step copies them
    # into one of two device buffers (256-byte aligned segments; the
    # batch's tensors become views of it), runs the step, and copies the
    # output back into one of two pinned host buffers.  The copies run on a
    # second stream, one step ahead (inputs) and one step behind (output),
    # as a serving loop overlaps them; every copy of every timed step is
    # inside the timed region.
    names = ("q", "k_new", "v_new", "slots_new", "block_table", "seqused_k",
             "cu_seqlens_q")
    ref_out = batch.out.clone()        # the step's output, device-resident
    segs, total = [], 0
    for k in names:
        t = getattr(batch, k)
        nb = t.numel() * t.element_size()
        segs.append((k, total, nb))
        total = (total + nb + 255) // 256 * 256
    host_in = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for k, off, nb in segs:
        t = getattr(batch, k)
        host_in[off:off + nb].copy_(t.contiguous().view(-1).view(torch.uint8)
                                    .cpu())
    slots = []
    for _ in range(2):
        dev_in = torch.empty(total, dtype=torch.uint8, device=dev)
        views = {k: dev_in[off:off + nb].view(getattr(batch, k).dtype)
                 .view(getattr(batch, k).shape) for k, off, nb in segs}
        out_host = torch.empty(batch.out.shape, dtype=batch.out.dtype,
                               pin_memory=True)
        slots.append({"dev_in": dev_in, "views": views,
                      "out": torch.empty_like(batch.out), "out_host": out_host,
                      "h2d": torch.cuda.Event(), "done": torch.cuda.Event(),
                      "d2h": torch.cuda.Event()})
    copy_stream = torch.cuda.Stream(dev)
    h2d = sum(nb for _, _, nb in segs)
    d2h = slots[0]["out_host"].numel() * slots[0]["out_host"].element_size()

    def h2d_copy(sl):
        # the buffer's previous step must be done with it
        copy_stream.wait_event(sl["done"])
        with torch.cuda.stream(copy_stream):
            sl["dev_in"].copy_(host_in, non_blocking=True)
        sl["h2d"].record(copy_stream)

    def e2e_run(steps):
        """steps e2e steps; returns device ms from the first copy to the
        last output copy."""
        if steps <= 0:
            return 0.0
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(stream)
        copy_stream.wait_event(start)
        h2d_copy(slots[0])
        for i in range(steps):
            sl = slots[i % 2]
            if i + 1 < steps:
                h2d_copy(slots[(i + 1) % 2])        # next step's inputs
            stream.wait_event(sl["h2d"])
            for k, v in sl["views"].items():
                setattr(batch, k, v)
            batch.out = sl["out"]
            batch.step()
            sl["done"].record(stream)
            copy_stream.wait_event(sl["done"])
            with torch.cuda.stream(copy_stream):
                sl["out_host"].copy_(sl["out"], non_blocking=True)
            sl["d2h"].record(copy_stream)
        for sl in slots:
            stream.wait_event(sl["d2h"])        # the last output copies
        stop.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(stop)

    e2e_run(args.warmup)
    e2e_ms = e2e_run(args.steps)
    # the same inputs every step: the copied-back output must equal it
    if not torch.equal(slots[(args.steps - 1) % 2]["out_host"],
                       ref_out.cpu()):
        raise RuntimeError("e2e output differs from the device step's")

    # secondary: varlen causal prefill with prefix cache (TFLOP/s)
    pre = workloads.prefill_with_prefix(seed=SEED_PREFILL, device=dev)
    pb = DeviceBatch(pre, dev, poison=False)
    pb.write_context()
    pb.write_new()
    for _ in range(3):
        pb.attend(return_lse=False)
    # 40 calls: the first call's host launch time (the device idles in the
    # timed region until it arrives) is then about 1 us per call
    pre_ms = time_steps(lambda i: pb.attend(return_lse=False), 40, stream) / 40
    flops = prefill_flops(pre)
    del pb

    step_ms, e2e_step_ms, attn_ms, pre_ms = max_over_ranks(
        [ms / args.steps, e2e_ms / args.steps, attn_ms, pre_ms], dev, world)
    value = aggregate_value(acct["step"], step_ms, world)
    achieved = acct["attention"] / (attn_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "batched_paged_decode_llama3_8b",
            "requests": wl.batch, "query_len": 1, "num_heads": 32,
            "num_kv_heads": 8, "head_size": 128, "block_size": 16,
            "context_lens": "U[512,4096] seed %d" % SEED_DECODE,
            "sum_context": int(wl.seq_lens.sum()),
            "pool_blocks": wl.num_blocks,
            "num_splits": "auto",
            "l2": "inputs larger than L2: %.0f MB of KV per step vs 129 MB"
                  % (acct["kv"] / 1e6),
            "parallelism": "replicas" if world > 1 else "single",
        },
        "step_bytes": acct,
        "gpu_launches": int(launches),
        "launches_per_step": launches / args.steps,
        "e2e": {"value": round(aggregate_value(acct["step"], e2e_step_ms,
                                               world), 1),
                "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_step_ms, 5)},
        "roofline": {
            "kernel": "paged decode attention call (TMA decode kernel, "
                      "plus the split combine when the plan splits)",
            "bound": "hbm", "achieved": round(achieved, 1),
            "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4),
            "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_src,
            "traffic": ncu_traffic("decode_attention_batched_decode"),
            "avg_launch_ms": round(attn_ms, 5),
            "algorithmic_bytes_per_launch": acct["attention"],
        },
        "prefill": {
            "workload": "varlen_causal_prefill_with_prefix",
            "seqs": pre.batch, "tokens": pre.num_tokens,
            "flops": flops, "ms": round(pre_ms, 4),
            "tflops": round(flops / (pre_ms * 1e-3) / 1e12, 1),
            "peak_tflops": tf_peak,
            "frac": round(flops / (pre_ms * 1e-3) / 1e12 / tf_peak, 4),
        },
        "clocks": clk,
    }
    return res


# ------------------------------------------------- other workloads (rank 0)
def _time_ms(fn, iters=40, warm=3):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def _kv_bytes(wl, elem=2):
    """Admissible K/V bytes of the requests, each read once (window aware:
    a request's queries see at most its last window + query-count keys)."""
    L = wl.seq_lens.astype(np.int64)
    if wl.window_size[0] >= 0:
        L = np.minimum(L, wl.window_size[0] + wl.q_lens.astype(np.int64))
    return int(L.sum()) * 2 * wl.num_kv_heads * wl.head_size * elem


def cache_write_bytes(wl, elem=2):
    """Algorithmic bytes of writing the workload's new K/V rows: each row
    read and written once, plus its 8-byte slot."""
    T = len(wl.slot_mapping_new)
    return T * 2 * wl.num_kv_heads * wl.head_size * elem * 2 + 8 * T


def _time_flushed_ms(fn, flush, iters=10, warm=3):
    """Median device ms of fn, with the L2 flushed before each timed call
    and events around the call only.  The flush is a read pass over 1 GB:
    the L2 then holds clean lines, so no write-back of the flush competes
    with the call, and its 0.15 ms of device time keep the device busy
    while the host queues the events and the call, so host launch time does
    not enter the interval."""
    for _ in range(warm):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush.max()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return float(np.median([a.elapsed_time(b) for a, b in ev]))


def other_workloads(dev, hbm_peak, tf_peak):
    """Attention-call rates on the other configurations (CUDA events; each
    decode working set exceeds the L2)."""
    out = {}

    def rec(name, desc, ms, amount, unit, peak):
        rate = amount / (ms * 1e-3) / (1e9 if unit == "GB/s" else 1e12)
        out[name] = {"workload": desc, "ms": round(ms, 4),
                     "value": round(rate, 1), "unit": unit,
                     "frac": round(rate / peak, 4)}

    # the varlen prefill workload's cache write (11207 new tokens): its
    # 92 MB fit in the L2, so the L2 is flushed before each timed call
    wl = workloads.prefill_with_prefix(seed=SEED_PREFILL, device=dev)
    b = DeviceBatch(wl, dev, poison=False)
    flush = torch.zeros(1 << 30, dtype=torch.uint8, device=dev)
    rec("cache_write", "reshape_and_cache of the varlen prefill workload's "
        "%d new tokens (8 KV heads, D 128, bf16; L2 flushed before each "
        "call)" % len(wl.slot_mapping_new),
        _time_flushed_ms(b.write_new, flush), cache_write_bytes(wl), "GB/s",
        hbm_peak)
    del b, flush
    # the Gemma-like mixed batch as one call, against max(bytes / BW,
    # flops / F); and its prefill part (four 512-token chunks, D 256) alone
    wl = workloads.mixed_gemma(device=dev)
    b = DeviceBatch(wl, dev, poison=False)
    b.write_context()
    b.write_new()
    ms = _time_ms(lambda: b.attend(return_lse=False))
    nbytes = _kv_bytes(wl)
    flops = prefill_flops(wl, min_rows=17)
    t_roof = max(nbytes / (hbm_peak * 1e9), flops / (tf_peak * 1e12))
    out["mixed_batch"] = {
        "workload": "one call: 124 decodes (L ~ U[1024, 16384]) + 4 x "
                    "512-token chunks (context U[0, 8192]), 16/8 heads, "
                    "D 256, window (4095, 0), soft-cap 50",
        "ms": round(ms, 4), "bytes": nbytes, "flops": flops,
        "t_roof_ms": round(t_roof * 1e3, 4),
        "frac": round(t_roof * 1e3 / ms, 4),
        "bound": "hbm" if nbytes / (hbm_peak * 1e9) >= flops /
                 (tf_peak * 1e12) else "tensor"}
    del b
    wl = workloads.mixed_gemma(device=dev, n_decode=0)
    b = DeviceBatch(wl, dev, poison=False)
    b.write_context()
    b.write_new()
    rec("mixed_prefill_part", "the mixed batch's 4 x 512-token prefill "
        "chunks alone (D 256, window 4095, soft-cap 50)",
        _time_ms(lambda: b.attend(return_lse=False)),
        prefill_flops(wl, min_rows=17), "TFLOP/s", tf_peak)
    del b

    wl = workloads.long_decode(device=dev)
    b = DeviceBatch(wl, dev, poison=False)
    b.write_context()
    b.write_new()
    rec("long_decode", "8 x 131072-key decodes, 64/8 heads, D 128, BS 64, "
        "16 splits", _time_ms(lambda: b.attend(return_lse=False)),
        _kv_bytes(wl), "GB/s", hbm_peak)
    del b
    wl = workloads.mixed_gemma(device=dev, n_prefill=0)
    b = DeviceBatch(wl, dev, poison=False)
    b.write_context()
    b.write_new()
    rec("mixed_decode", "124 decodes, L ~ U[1024, 16384], 16/8 heads, D 256, "
        "window (4095, 0), soft-cap 50", _time_ms(
            lambda: b.attend(return_lse=False)), _kv_bytes(wl), "GB/s",
        hbm_peak)
    del b
    wl = workloads.cascade_decode(device=dev)
    b = DeviceBatch(wl, dev, poison=False, cascade=True)
    b.write_context()
    b.write_new()
    P = wl.common_prefix_len
    uniq = (P + int((wl.seq_lens - P).sum())) * 2 * wl.num_kv_heads * \
        wl.head_size * 2
    rec("cascade_decode", "256 decodes sharing an 8192-token prefix + 512 own "
        "keys each, 64/8 heads, D 128 (unique K/V bytes)", _time_ms(
            lambda: b.attend(return_lse=False)), uniq, "GB/s", hbm_peak)
    del b
    # fp8 (E4M3) cache: the batched decode workload's cache quantized
    wl = workloads.batched_decode(seed=SEED_DECODE, device=dev)
    b = DeviceBatch(wl, dev, poison=False)
    b.write_context()
    b.write_new()
    c8 = torch.zeros(wl.cache_shape(), dtype=torch.uint8, device=dev)
    k8, v8 = c8.unbind(0)
    ks = torch.tensor([0.02], device=dev)
    vs = torch.tensor([0.02], device=dev)
    for rk, rv, sl in ((b.k_ctx, b.v_ctx, b.slots_ctx),
                       (b.k_new, b.v_new, b.slots_new)):
        api.reshape_and_cache_flash(rk, rv, k8, v8, sl, "fp8", ks, vs)
    rec("fp8_decode", "batched decode workload over an E4M3 cache (fp8 "
        "bytes)", _time_ms(lambda: api.flash_attn_varlen_func(
            b.q, k8, v8, 1, b.cu_seqlens_q, wl.max_seqlen_k,
            seqused_k=b.seqused_k, softmax_scale=wl.softmax_scale,
            causal=True, block_table=b.block_table, out=b.out,
            k_descale=ks, v_descale=vs)), _kv_bytes(wl, 1), "GB/s",
        hbm_peak)
    # the same with E4M3 queries, as the vLLM FA backend runs an fp8 cache:
    # scaled_fp8_quant of the query, then the attention call
    qs = torch.tensor([0.02], device=dev)
    q8 = torch.empty(b.q.shape, dtype=torch.float8_e4m3fn, device=dev)

    def fp8q_call():
        api.scaled_fp8_quant(b.q, qs, out=q8)
        api.flash_attn_varlen_func(
            q8, k8, v8, 1, b.cu_seqlens_q, wl.max_seqlen_k,
            seqused_k=b.seqused_k, softmax_scale=wl.softmax_scale,
            causal=True, block_table=b.block_table, out=b.out,
            k_descale=ks, v_descale=vs, q_descale=qs)
    rec("fp8q_decode", "batched decode workload, E4M3 queries and cache "
        "(query quantization + attention call; fp8 bytes)",
        _time_ms(fp8q_call), _kv_bytes(wl, 1), "GB/s", hbm_peak)
    del b, c8, q8
    wl = workloads.build_workload("long_prefill", 324, [2048], [8192], 32, 8,
                                  128, 64, device=dev)
    b = DeviceBatch(wl, dev, poison=False)
    b.write_context()
    b.write_new()
    rec("long_prefill", "one request, 2048 queries over 8192 keys (causal), "
        "32/8 heads, D 128 (K/V fit in L2)", _time_ms(
            lambda: b.attend(return_lse=False)), prefill_flops(wl),
        "TFLOP/s", tf_peak)
    del b
    torch.cuda.empty_cache()
    return out


# -------------------------------------------------------------- CPU legs
_POOL_WL = None          # the workload the oracle pool's workers read


def _oracle_request(b):
    from oracle.harness import request_reference
    request_reference(_POOL_WL, b)
    return b


def make_oracle_pool(wl):
    """A process pool for the oracle on every host core, forked before this
    process touches the GPU (the workers inherit ``wl`` and never use
    CUDA)."""
    import multiprocessing as mp
    global _POOL_WL
    _POOL_WL = wl
    cores = os.cpu_count() or 1
    return mp.get_context("fork").Pool(cores), cores


def _request_bytes(wl, b):
    e = 2
    return int(wl.seq_lens[b]) * 2 * wl.num_kv_heads * wl.head_size * e + \
        2 * wl.num_heads * wl.head_size * e


def oracle_pool_sample(pool, cores, wl, budget_s):
    """Wall time of the oracle over passes of the whole batch, one request
    per worker at a time, until ``budget_s``.  Returns (bytes, seconds,
    requests)."""
    nbytes, done, t_total = 0, 0, 0.0
    while t_total < budget_s:
        t0 = time.perf_counter()
        pool.map(_oracle_request, range(wl.batch), chunksize=1)
        t_total += time.perf_counter() - t0
        nbytes += sum(_request_bytes(wl, b) for b in range(wl.batch))
        done += wl.batch
    return nbytes, t_total, done


def oracle_sample(wl, budget_s, max_requests=None, start=0):
    """Time the oracle on whole requests (from ``start``) until ``budget_s``
    is spent.  Returns (bytes processed, seconds, requests)."""
    from oracle.harness import request_reference
    done, nbytes, t_total = 0, 0, 0.0
    e = 2
    per_tok = 2 * wl.num_kv_heads * wl.head_size * e
    order = [(start + i) % wl.batch for i in range(wl.batch)]
    for b in order:
        t0 = time.perf_counter()
        request_reference(wl, b)
        t_total += time.perf_counter() - t0
        L = int(wl.seq_lens[b])
        nbytes += L * per_tok + 2 * wl.num_heads * wl.head_size * e
        done += 1
        if t_total >= budget_s or (max_requests and done >= max_requests):
            break
    return nbytes, t_total, done


def cpu_baseline(wl, pool, cores, budget_s=10.0):
    """The float64 oracle on every host core (a process per core, one
    request each at a time), and on one core."""
    nbytes, secs, n = oracle_pool_sample(pool, cores, wl, budget_s)
    b1, s1, n1 = oracle_sample(wl, budget_s / 3)
    return {"value": round(nbytes / secs / 1e9, 4), "unit": UNIT,
            "cores": cores, "kind": "oracle",
            "sample": "%d requests (%d passes over the 64 of the batched "
                      "decode workload) in %.1f s of wall time on %d "
                      "processes (float64 numpy oracle, one thread each)"
                      % (n, n // wl.batch, secs, cores),
            "one_core": {"value": round(b1 / s1 / 1e9, 4), "cores": 1,
                         "sample": "%d requests in %.1f s, one thread"
                                   % (n1, s1)}}


def reference_arm(args):
    wl = workloads.batched_decode(seed=SEED_DECODE, device="cpu")
    pool, cores = make_oracle_pool(wl)
    per_step = []
    try:
        for i in range(args.warmup + args.steps):
            # one step: `cores` requests of the batch, one per process
            reqs = [(i * cores + j) % wl.batch for j in range(cores)]
            t0 = time.perf_counter()
            pool.map(_oracle_request, reqs, chunksize=1)
            secs = time.perf_counter() - t0
            if i >= args.warmup:
                per_step.append((sum(_request_bytes(wl, b) for b in reqs),
                                 secs))
    finally:
        pool.close()
        pool.join()
    tot_b = sum(b for b, _ in per_step)
    tot_s = sum(s for _, s in per_step)
    value = tot_b / tot_s / 1e9
    sample = ("%d requests of the batched decode workload per step, one "
              "per process on %d host cores (float64 numpy oracle, one "
              "thread each)" % (cores, cores))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4),
        "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / len(per_step), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": "batched_paged_decode_llama3_8b",
                   "requests": wl.batch},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT,
                         "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------ profiling cases
def profile_case(name, dev):
    """Set up one workload and run its call a few times (warm-up included),
    for a profiler to select launches from: batched_decode (the step: cache
    write, then attention), batched_decode_persistent (the same step on the
    persistent decode kernel), fp8_decode (the batched decode over an E4M3
    cache), fp8q_decode (the same with E4M3 queries), cache_write (the varlen prefill workload's new rows), prefill
    (the varlen prefill attention), mixed_prefill (the Gemma-like batch's
    four D = 256 prefill chunks), cascade (shared-prefix decode)."""
    if name == "batched_decode":
        wl = workloads.batched_decode(seed=SEED_DECODE, device=dev)
        b = DeviceBatch(wl, dev, poison=False)
        b.write_context()
        run = b.step
    elif name == "batched_decode_persistent":
        # the persistent decode kernel on the same step, for a side-by-side
        # capture with the per-unit kernel the library picks here
        api.set_decode_kernel(api.DECODE_PERSISTENT)
        wl = workloads.batched_decode(seed=SEED_DECODE, device=dev)
        b = DeviceBatch(wl, dev, poison=False)
        b.write_context()
        run = b.step
    elif name == "fp8_decode":
        wl = workloads.batched_decode(seed=SEED_DECODE, device=dev)
        b = DeviceBatch(wl, dev, poison=False)
        b.write_context()
        b.write_new()
        c8 = torch.zeros(wl.cache_shape(), dtype=torch.uint8, device=dev)
        k8, v8 = c8.unbind(0)
        ks = torch.tensor([0.02], device=dev)
        vs = torch.tensor([0.02], device=dev)
        for rk, rv, sl in ((b.k_ctx, b.v_ctx, b.slots_ctx),
                           (b.k_new, b.v_new, b.slots_new)):
            api.reshape_and_cache_flash(rk, rv, k8, v8, sl, "fp8", ks, vs)

        def run():
            api.flash_attn_varlen_func(
                b.q, k8, v8, 1, b.cu_seqlens_q, wl.max_seqlen_k,
                seqused_k=b.seqused_k, softmax_scale=wl.softmax_scale,
                causal=True, block_table=b.block_table, out=b.out,
                k_descale=ks, v_descale=vs)
    elif name == "fp8q_decode":
        wl = workloads.batched_decode(seed=SEED_DECODE, device=dev)
        b = DeviceBatch(wl, dev, poison=False)
        b.write_context()
        b.write_new()
        c8 = torch.zeros(wl.cache_shape(), dtype=torch.uint8, device=dev)
        k8, v8 = c8.unbind(0)
        ks = torch.tensor([0.02], device=dev)
        vs = torch.tensor([0.02], device=dev)
        qs = torch.tensor([0.02], device=dev)
        for rk, rv, sl in ((b.k_ctx, b.v_ctx, b.slots_ctx),
                           (b.k_new, b.v_new, b.slots_new)):
            api.reshape_and_cache_flash(rk, rv, k8, v8, sl, "fp8", ks, vs)
        q8 = torch.empty(b.q.shape, dtype=torch.float8_e4m3fn, device=dev)

        def run():
            api.scaled_fp8_quant(b.q, qs, out=q8)
            api.flash_attn_varlen_func(
                q8, k8, v8, 1, b.cu_seqlens_q, wl.max_seqlen_k,
                seqused_k=b.seqused_k, softmax_scale=wl.softmax_scale,
                causal=True, block_table=b.block_table, out=b.out,
                k_descale=ks, v_descale=vs, q_descale=qs)
    elif name == "cache_write":
        wl = workloads.prefill_with_prefix(seed=SEED_PREFILL, device=dev)
        b = DeviceBatch(wl, dev, poison=False)
        run = b.write_new
    elif name in ("prefill", "mixed_prefill", "cascade"):
        if name == "prefill":
            wl = workloads.prefill_with_prefix(seed=SEED_PREFILL, device=dev)
        elif name == "mixed_prefill":
            wl = workloads.mixed_gemma(device=dev, n_decode=0)
        else:
            wl = workloads.cascade_decode(device=dev)
        b = DeviceBatch(wl, dev, poison=False, cascade=name == "cascade")
        b.write_context()
        b.write_new()

        def run():
            b.attend(return_lse=False)
    else:
        raise SystemExit("unknown case %r" % name)
    for _ in range(6):
        run()
    torch.cuda.synchronize()
    api.check_device_errors(dev)
    print(json.dumps({"case": name, "calls": 6, "ok": True}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native",
                    choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other-workload rates")
    ap.add_argument("--case", default=None,
                    help="run one workload's call 6 times and exit (for a "
                         "profiler): batched_decode, "
                         "batched_decode_persistent, fp8_decode, "
                         "fp8q_decode, cache_write, prefill, mixed_prefill, "
                         "cascade")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.case:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        if not os.path.exists(_build.LIB_PATH):
            _build.build()
        api.load_library()
        profile_case(args.case, dev)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return

    # the oracle's process pool is forked before this process uses CUDA
    cpu_wl = pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_wl = workloads.batched_decode(seed=SEED_DECODE, device="cpu")
        pool, cores = make_oracle_pool(cpu_wl)
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    if rank == 0 and not os.path.exists(_build.LIB_PATH):
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    api.load_library()
    res = gpu_arm(args, rank, world, dev)
    if rank == 0 and world == 1 and not args.no_extras:
        hbm_peak, tf_peak, _ = measured_peaks()
        res["other_workloads"] = other_workloads(dev, hbm_peak, tf_peak)
    if pool is not None:
        try:
            res["cpu_baseline"] = cpu_baseline(cpu_wl, pool, cores)
        finally:
            pool.close()
            pool.join()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
