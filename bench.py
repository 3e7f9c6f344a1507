#!/usr/bin/env python
"""Benchmark of the multi-head scaled dot-product attention forward.

One step = one ``mha_fwd`` call (the whole path: load, Q K^T, scale + mask,
softmax, P V, normalise + store) over one batch of the workload.  Default
(``--workload all``): the headline is the long-context causal configuration
(bf16, B=4, H=16, L=8192, d=128; TFLOP/s against the bf16 tensor peak), and
the line's ``configs`` object carries the other four configurations of the
metric, each timed the same way: the fp32 parity case, the Transformer-base
padded encoder (B=256, H=8, L=64, lengths uniform in [8, 64]), the causal
decoder (B=128, H=8, L=128) and the Transformer-big cross-attention (B=64,
H=16, Lq=96, Lk=128, source lengths uniform in [16, 128]) -- GB/s against
HBM.  ``--workload NAME`` times one workload of gen.WORKLOADS alone.  The ``sublayer_*`` workloads (gen.SUBLAYERS) time the whole
multi-head sublayer per step (projections with biases, attention, output
projection; TFLOP/s), with the projection kernel as the roofline kernel.  The
``bwd_*`` workloads time the backward pass (``mha_bwd``: dq, dk, dv of a
forward workload; TFLOP/s of the five products the chain rule needs).

value  device throughput, inputs resident in HBM; K launches captured in one
       CUDA graph whose first and last nodes record the two timing events;
       consecutive launches read different input sets whose total exceeds 3x
       the L2 size, so no launch finds its inputs in L2.
host_us_per_call  host time to enqueue one call, through the C entry point
       and through the Python binding, and the device time per call when the
       K calls are launched one by one (no graph).
e2e    the same metric through the public call with host buffers: pinned
       host -> device copies of Q, K, V (and lengths), mha_fwd, device -> host
       copy of the output, every step, inside the timed region; two device
       buffer slots and separate copy streams let step i+1's inputs arrive and
       step i-1's output leave while step i computes.
--impl reference   times the fp64 CPU oracle (the only other implementation
       of this path) on the host cores, on a bounded sample of the workload.

Multi-GPU (torchrun): every rank runs the same workload on its own GPU (the
(batch, head) pairs are independent; no collective on the data path), weak
scaling; value = all ranks' work / the slowest rank's time.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gen  # noqa: E402

# BASELINE's headline metric: TFLOP/s and fraction of the bf16 tensor peak for
# long sequences, GB/s and fraction of HBM bandwidth for short ones
BASELINE_METRIC = ("attention fwd TFLOP/s & % bf16 tensor peak (long n); GB/s & % HBM "
                   "(short n)")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_NAMES = {1: "attn_f32_simt_kernel", 2: "attn_short_tc_kernel", 3: "attn_long_tc_kernel",
                4: "zero_fill_kernel", 5: "attn_decode_tc_kernel"}
# backward workloads: the gradients of a forward workload (training shapes)
BWD_WORKLOADS = {"bwd_" + n: n for n in ("enc_pad_bf16_b256_h8_l64_d64",
                                         "dec_causal_bf16_b128_h8_l128_d64",
                                         "cross_pad_bf16_b64_h16_lq96_lk128_d64",
                                         "long_causal_bf16_b4_h16_l8192_d128")}


# ---------------------------------------------------------------------------
# algorithmic work of one launch
# ---------------------------------------------------------------------------
def algorithmic(spec, lens):
    """(bytes, flops) one launch must move / compute, from the realised lengths.

    bytes: Q rows that are not query padding, K and V rows that are not key
    padding, every output row (zeros included), and the lengths.
    flops: 2 * (d_k + d_v) per allowed (query, key) pair.
    """
    B, H, Lq, Lk, dk, dv = (spec[x] for x in ("B", "H", "Lq", "Lk", "dk", "dv"))
    Hkv = spec.get("Hkv", H)
    esz = 4 if spec["dtype"] == "f32" else 2
    m = spec["mask"]
    L = np.full(B, Lk, dtype=np.int64) if lens is None else np.clip(lens.astype(np.int64), 0, Lk)
    q_rows = (np.minimum(L, Lq) if m & gen.MASK_QUERY_PADDING else np.full(B, Lq)).sum() * H
    kv_rows = (L if m & gen.MASK_KEY_PADDING else np.full(B, Lk)).sum() * Hkv
    nbytes = esz * (q_rows * dk + kv_rows * (dk + dv) + B * H * Lq * dv)
    if lens is not None and m & (gen.MASK_KEY_PADDING | gen.MASK_QUERY_PADDING):
        nbytes += 4 * B
    pairs = 0
    for b in range(B):
        kmax = int(L[b]) if m & gen.MASK_KEY_PADDING else Lk
        nq = min(int(L[b]), Lq) if m & gen.MASK_QUERY_PADDING else Lq
        if m & gen.MASK_CAUSAL:
            i = np.arange(nq)
            pairs += int(np.minimum(i + 1, kmax).sum())
        elif m & gen.MASK_CAUSAL_TAIL:
            i = np.arange(nq)
            pairs += int(np.clip(kmax - Lq + i + 1, 0, kmax).sum())
        else:
            pairs += nq * kmax
    flops = 2 * (dk + dv) * pairs * H
    return int(nbytes), int(flops)


def bound_of(spec):
    """Tensor-bound when the work is long in both the query and the key
    direction (about 2 (d_k + d_v) min(Lq, Lk) / (2 d) flop per byte); HBM-bound
    for sentence-length attention and for generation steps (few queries)."""
    return "tensor" if min(spec["Lq"], spec["Lk"]) > 128 else "hbm"


def metric_of(spec):
    if bound_of(spec) == "tensor":
        return "attention fwd TFLOP/s (long n)", "TFLOP/s"
    return "attention fwd GB/s (short n)", "GB/s"


def throughput(spec, nbytes, flops, seconds):
    if bound_of(spec) == "tensor":
        return flops / seconds / 1e12
    return nbytes / seconds / 1e9


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# the source file of each profiled kernel (the digest also covers the shared
# headers and the dispatcher, which set its launch parameters)
KERNEL_FILES = {"attn_short_tc_kernel": "attn_short_tc.cu", "attn_long_tc_kernel": "attn_long_tc.cu",
                "attn_decode_tc_kernel": "attn_decode_tc.cu", "linear_tc_kernel": "linear_tc.cu",
                "attn_f32_simt_kernel": "attn_f32_simt.cu", "bwd_tc": "attn_bwd_tc.cu"}
SHARED_FILES = ("common.cuh", "ptx.cuh", "mha_api.cu")


def kernel_source_digest(kernel=None):
    """Digest of the sources a kernel is built from (all of csrc/ when
    `kernel` is None or unknown)."""
    csrc = os.path.join(ROOT, "transformer_head_scaled_mha_gb300", "csrc")
    names = sorted(os.listdir(csrc))
    if kernel in KERNEL_FILES:
        names = sorted(SHARED_FILES + (KERNEL_FILES[kernel],))
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def bwd_kernel_names(dk, Lq, Lk, mask):
    """(kernels, traffic kernel) of one backward call given the forward's row
    statistics: the fused single-tile kernel for d 64 and lengths <= 128 (its
    storing form <1> unless the mask is causal), else the D pass, dq and
    dk/dv kernels."""
    if dk == 64 and Lq <= 128 and Lk <= 128:
        form = "bwd_short_tc_kernel<%d>" % (0 if mask & gen.MASK_CAUSAL else 1)
        return form + " (one launch)", form
    return ("bwd_dsum_kernel + bwd_dq_tc_kernel + bwd_dkdv_tc_kernel (one mha_bwd_lse call, "
            "3 launches)", "bwd_dkdv_tc_kernel (the largest share of the call)")


def linear_kernel_name(K, N):
    """The projection kernel mha_linear_fwd runs for x [M, K] W [K, N]: 128 x 256
    tiles when K and N are multiples of 64 and N >= 256, else 128 x 128."""
    return "linear_wide_kernel" if K % 64 == 0 and N % 64 == 0 and N >= 256 else \
        "linear_tc_kernel"


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None
    if not rec or rec.get("source_digest") != kernel_source_digest(rec.get("kernel")):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks sampled with nvidia-smi while the GPU is loaded
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []  # (t, sm_mhz, max_mhz, power, reasons)
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = [n for n, v in zip(self.NAMES, parts[5:9]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, mx, parts[3], reasons))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        if not self.samples:
            return None
        t0, t1 = self.window if self.window else (0, float("inf"))
        inside = [s for s in self.samples if t0 - 0.05 <= s[0] <= t1 + 0.05] or self.samples[-3:]
        reasons = sorted({r for s in inside for r in s[4]})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside)}


# ---------------------------------------------------------------------------
# distributed plumbing (torchrun: one rank per GPU)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Slowest rank's time (all_reduce MAX); identity for one process."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(spec, nbytes, flops, slowest_seconds, world: int) -> float:
    """Whole-job throughput: every rank ran the same launch; all ranks' work
    divided by the slowest rank's time."""
    return throughput(spec, nbytes, flops, slowest_seconds) * world


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# end to end: host buffers in, result back, every step
# ---------------------------------------------------------------------------
E2E_PIPELINE = ("two device buffer slots, three streams: the host->device copies of step i+1 "
                "and the device->host copy of step i-1 run while step i computes")


def e2e_seconds_per_step(slots_in, launch, slots_out, steps, stream, world):
    """Seconds per step of a pipelined host -> call -> host loop.

    slots_in[s]  (device dst, pinned host src) pairs copied in for a step on slot s
    launch(s, stream)  enqueues the call that reads slot s's inputs and writes
                 its outputs
    slots_out[s] (pinned host dst, device src) pairs copied back after the call
    Step i uses slot i % 2.  Its input copies wait until the call of step i - 2
    (the slot's previous user) has read the slot; its call waits for its input
    copies and for the read-back of step i - 2 (which frees the slot's
    outputs); its read-back waits for its call.  Every step's copies and call
    lie between the two timing events."""
    import torch
    dev = stream.device
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        s = i % 2
        if i >= 2:
            s_in.wait_event(done[s])
        with torch.cuda.stream(s_in):
            for dst, src in slots_in[s]:
                dst.copy_(src, non_blocking=True)
        in_ready[s].record(s_in)
        stream.wait_event(in_ready[s])
        if i >= 2:
            stream.wait_event(out_read[s])
        launch(s, stream)
        done[s].record(stream)
        s_out.wait_event(done[s])
        with torch.cuda.stream(s_out):
            for dst, src in slots_out[s]:
                dst.copy_(src, non_blocking=True)
        out_read[s].record(s_out)

    for i in range(2):  # warm-up: both slots once
        step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        step(i)
    s_out.wait_stream(stream)
    s_out.wait_stream(s_in)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / 1e3 / steps


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_sample_rows(spec, lens, target_flops, seed=0):
    """A random sample of query rows whose oracle work is about target_flops."""
    B, H, Lq = spec["B"], spec["H"], spec["Lq"]
    total_rows = B * H * Lq
    _, total_flops = algorithmic(spec, lens)
    frac = min(1.0, target_flops / max(total_flops, 1))
    n = max(1, int(total_rows * frac))
    if n >= total_rows:
        return None, 1.0
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(total_rows, size=n, replace=False)).astype(np.int64)
    return rows, n / total_rows


def time_oracle(spec, q, k, v, lens, rows, threads=0, reps=1):
    import oracle
    scale = gen.default_scale(spec["dk"])
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.mha_fwd(q, k, v, mask_kind=spec["mask"], key_lengths=lens, scale=scale,
                       rows=rows, threads=threads, layout=spec.get("layout", "bhsd"))
    return time.perf_counter() - t0


def oracle_baseline(spec, q, k, v, lens, budget_s=12.0):
    """Oracle throughput on a bounded random row sample, scaled by the sample's
    share of the rows (rows are independent units of equal expected cost)."""
    import oracle
    cores = oracle.max_threads()
    _, total_flops = algorithmic(spec, lens)
    # calibrate on a small sample, then size the real sample for the budget
    probe_rows, probe_frac = oracle_sample_rows(spec, lens, 2e8)
    t_probe = time_oracle(spec, q, k, v, lens, probe_rows)
    rate = (total_flops * probe_frac) / max(t_probe, 1e-6)  # oracle flop/s
    rows, frac = oracle_sample_rows(spec, lens, rate * budget_s, seed=1)
    # a workload smaller than the budget is run whole, several times over
    reps = max(1, int(budget_s * rate / max(total_flops, 1))) if rows is None else 1
    t = time_oracle(spec, q, k, v, lens, rows, reps=reps)
    nbytes, flops = algorithmic(spec, lens)
    value = throughput(spec, nbytes * frac * reps, flops * frac * reps, t)
    n_rows = spec["B"] * spec["H"] * spec["Lq"] if rows is None else len(rows)
    sample = ("%d of %d query rows (%.4g%%), drawn uniformly at random, x%d, %.1f s on %d "
              "threads; work scaled by the sampled share" % (
                  n_rows, spec["B"] * spec["H"] * spec["Lq"], 100 * frac, reps, t, cores))
    return {"value": value, "unit": metric_of(spec)[1], "cores": cores, "kind": "oracle",
            "sample": sample}


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------
_EVENT_RECORD = None


def _event_record_fn():
    """cuEventRecordWithFlags from the CUDA driver (one per process), or None."""
    global _EVENT_RECORD
    if _EVENT_RECORD is None:
        import ctypes
        try:
            drv = ctypes.CDLL("libcuda.so.1")
            fn = drv.cuEventRecordWithFlags
            fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
            fn.restype = ctypes.c_int
            _EVENT_RECORD = fn
        except (OSError, AttributeError):
            _EVENT_RECORD = False
    return _EVENT_RECORD or None


def graph_timer(stream, fn, steps):
    """Captures fn(i, stream) for i < steps in one CUDA graph whose first and
    last nodes record two timing events (external event-record nodes), so the
    elapsed time covers the launches and not the graph launch before them.
    Returns (run, elapsed_seconds, how); run() replays the graph on `stream`."""
    import ctypes

    import torch
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)  # materialise the events
    ev1.record(stream)
    stream.synchronize()
    rec = _event_record_fn()
    inside = False
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        if rec is not None:
            inside = rec(ctypes.c_void_p(ev0.cuda_event), ctypes.c_void_p(stream.cuda_stream),
                         1) == 0
        for i in range(steps):
            fn(i, stream)
        if inside:
            inside = rec(ctypes.c_void_p(ev1.cuda_event), ctypes.c_void_p(stream.cuda_stream),
                         1) == 0

    def run():
        with torch.cuda.stream(stream):
            if not inside:
                ev0.record(stream)
            graph.replay()
            if not inside:
                ev1.record(stream)

    how = ("CUDA graph of %d launches, CUDA events recorded as the graph's first and last "
           "nodes" % steps) if inside else "CUDA graph of %d launches, CUDA events" % steps
    return run, (lambda: ev0.elapsed_time(ev1) / 1e3), how


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
# the configurations of the headline metric: the long causal one (TFLOP/s,
# bf16 tensor peak) heads the line; the sentence-length ones (GB/s, HBM) and
# the fp32 parity configuration follow under "configs"
HEADLINE_WORKLOAD = "long_causal_bf16_b4_h16_l8192_d128"
CONFIG_WORKLOADS = ("enc_f32_b2_h8_l32_d64", "enc_pad_bf16_b256_h8_l64_d64",
                    "dec_causal_bf16_b128_h8_l128_d64", "cross_pad_bf16_b64_h16_lq96_lk128_d64")
DEFAULT_WORKLOAD = "all"


def gpu_context():
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    return world, rank, local, dev


def measure_forward(name, args, world, rank, local, dev, cpu_budget):
    """Everything the JSON line reports for one forward workload: device
    throughput, end-to-end throughput, roofline, host and eager per-call
    times, clocks, the oracle's CPU baseline (rank 0, one process only)."""
    import ctypes

    import torch

    import transformer_head_scaled_mha_gb300 as mha

    spec = gen.WORKLOADS[name]
    dt = spec["dtype"]
    q, k, v, lens = gen.make_inputs(spec, seed=args.seed)
    nbytes, flops = algorithmic(spec, lens)
    metric, unit = metric_of(spec)
    scale = gen.default_scale(spec["dk"])
    mask = spec["mask"]
    B, H, Lq, Lk, dk, dv = (spec[x] for x in ("B", "H", "Lq", "Lk", "dk", "dv"))
    Hkv = spec.get("Hkv", H)
    layout = spec.get("layout", "bhsd")
    path = mha.mha_fwd_path_ex(B, H, Hkv, Lq, Lk, dk, dv, mask, 1 if dt == "bf16" else 0)
    kernel = KERNEL_NAMES.get(path, "?")

    def host_tensor(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.view(torch.bfloat16) if dt == "bf16" else t

    hq, hk, hv = host_tensor(q), host_tensor(k), host_tensor(v)
    out_shape = (B, Lq, H, dv) if layout == "bshd" else (B, H, Lq, dv)
    set_bytes = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    set_bytes += B * H * Lq * dv * hq.element_size()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(1, math.ceil(3 * l2 / set_bytes))
    sets = []
    for _ in range(n_sets):
        sets.append((hq.to(dev), hk.to(dev), hv.to(dev),
                     torch.empty(out_shape, dtype=hq.dtype, device=dev)))
    kl = torch.from_numpy(lens).to(dev) if lens is not None else None
    stream = torch.cuda.Stream(device=dev)
    plain = Hkv == H and layout == "bhsd"

    def call(qq, kk, vv, oo, lens_dev, s):
        if plain:
            mha.mha_fwd(qq, kk, vv, oo, mask_kind=mask, key_lengths=lens_dev, scale=scale,
                        stream=s)
        else:
            mha.mha_fwd_ex(qq, kk, vv, oo, layout=layout, mask_kind=mask,
                           key_lengths=lens_dev, scale=scale, stream=s)

    def step(i, s=None):
        qq, kk, vv, oo = sets[i % n_sets]
        call(qq, kk, vv, oo, kl, s)

    # warm-up (eager): W steps
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, stream)
    stream.synchronize()

    if args.no_graph:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def run_steps():
            with torch.cuda.stream(stream):
                ev0.record(stream)
                for i in range(args.steps):
                    step(i, stream)
                ev1.record(stream)
        elapsed_of = lambda: ev0.elapsed_time(ev1) / 1e3
        timing = "eager launches, CUDA events"
    else:
        run_steps, elapsed_of, timing = graph_timer(stream, step, args.steps)

    # Clocks are sampled from the start of an untimed soak (the same launches,
    # so the GPU is at its loaded clocks) to the end of the timed region.
    sampler = ClockSampler(local)
    sampler.start()
    t_soak = time.time()
    while time.time() - t_soak < args.soak:
        run_steps()
        stream.synchronize()
    barrier(world)
    torch.cuda.synchronize(dev)
    run_steps()
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    sampler.mark(t_soak + min(0.2, args.soak / 2), t_wall1)
    clocks = sampler.stop()
    elapsed = max_over_ranks(elapsed_of(), world, dev)
    per_launch = elapsed / args.steps
    value = weak_scaling_value(spec, nbytes, flops, per_launch, world)
    st = mha.mha_debug_status(stream)
    if st != mha.MHA_OK:
        raise RuntimeError("device status after timing: %s" % mha.mha_status_string(st))

    # host cost of one call: the C entry point with its arguments already
    # converted (what a C caller pays), and the Python binding (marshalling
    # included); both only enqueue.  Eager: the same K calls launched one by
    # one from the binding, timed on the device.
    qq, kk, vv, oo = sets[0]
    raw_args = [ctypes.c_void_p(t.data_ptr()) for t in (qq, kk, vv, oo)]
    lens_ptr = ctypes.c_void_p(kl.data_ptr() if kl is not None else 0)
    sh = ctypes.c_void_p(stream.cuda_stream)
    n_host = max(args.steps, 50)
    dtype_code = mha.MHA_DTYPE_BF16 if dt == "bf16" else mha.MHA_DTYPE_F32
    lay = 1 if layout == "bshd" else 0
    stream.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_host):
        rc = mha.lib.mha_fwd_ex(*raw_args, B, H, Hkv, Lq, Lk, dk, dv, lay, mask, lens_ptr,
                                ctypes.c_float(scale), dtype_code, sh)
    host_c = (time.perf_counter() - t0) / n_host
    if rc != mha.MHA_OK:
        raise RuntimeError("mha_fwd_ex: %s" % mha.mha_status_string(rc))
    stream.synchronize()
    t0 = time.perf_counter()
    for i in range(n_host):
        step(i, stream)
    host_py = (time.perf_counter() - t0) / n_host
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            step(i, stream)
        e1.record(stream)
    stream.synchronize()
    eager = e0.elapsed_time(e1) / 1e3 / args.steps

    # e2e: pinned host buffers, copies inside the timed region
    pq, pk, pv = hq.pin_memory(), hk.pin_memory(), hv.pin_memory()
    pout = torch.empty(out_shape, dtype=hq.dtype).pin_memory()
    plen = torch.from_numpy(lens).pin_memory() if lens is not None else None
    h2d = sum(t.numel() * t.element_size() for t in (pq, pk, pv))
    h2d += plen.numel() * 4 if plen is not None else 0
    d2h = pout.numel() * pout.element_size()
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    # slot 0 reuses the first timed input set; slot 1 gets its own buffers
    e2e_dev = [list(sets[0]) + [torch.empty_like(kl) if kl is not None else None]]
    e2e_dev.append([torch.empty_like(t) if t is not None else None for t in e2e_dev[0]])
    srcs = (pq, pk, pv)
    slots_in = [[(d[j], srcs[j]) for j in range(3)] + ([(d[4], plen)] if plen is not None else [])
                for d in e2e_dev]
    slots_out = [[(pout, d[3])] for d in e2e_dev]

    def e2e_launch(s, st_):
        d = e2e_dev[s]
        call(d[0], d[1], d[2], d[3], d[4], st_)

    e2e_t = max_over_ranks(e2e_seconds_per_step(slots_in, e2e_launch, slots_out, e2e_steps,
                                                stream, world), world, dev)
    e2e_value = weak_scaling_value(spec, nbytes, flops, e2e_t, world)

    peaks, peak_src = read_peaks()
    if bound_of(spec) == "tensor":
        peak, achieved, runit = peaks["bf16_tflops"], flops / per_launch / 1e12, "TFLOP/s"
    else:
        peak, achieved, runit = peaks["hbm_gbs"], nbytes / per_launch / 1e9, "GB/s"
    roofline = {"bound": bound_of(spec), "achieved": round(achieved, 2), "peak": peak,
                "unit": runit, "frac": round(achieved / peak, 4), "traffic":
                recorded_traffic(name), "kernel": kernel,
                "peak_source": peak_src + " (MEASURED_PEAKS.json)" if peak_src == "measured"
                else "fallback", "algorithmic_bytes": nbytes, "algorithmic_flops": flops}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(spec, q, k, v, lens, budget_s=cpu_budget)
    del sets, e2e_dev
    torch.cuda.empty_cache()
    return {
        "metric": metric, "value": round(value, 3), "unit": unit, "steps": args.steps,
        "ms_per_step": round(per_launch * 1e3, 6),
        "dtype": dt, "data": "synthetic (seeded N(0,1)%s inputs, seed %d)" % (
            "*%g" % spec["amp"] if spec["amp"] != 1.0 else "", args.seed),
        "config": {"workload": name, "B": B, "H": H, "H_kv": Hkv, "layout": layout, "Lq": Lq,
                   "Lk": Lk, "d_k": dk, "d_v": dv, "mask_kind": mask,
                   "len_range": spec["len_range"], "scale": scale,
                   "l2": "inputs rotate over %d device copies (%.0f MB > 3x L2 %.0f MB)"
                         % (n_sets, n_sets * set_bytes / 1e6, l2 / 1e6),
                   "timing": timing,
                   "parallelism": "weak: same workload per rank, no collective" if world > 1
                   else "1 GPU"},
        "e2e": {"value": round(e2e_value, 3), "unit": unit, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "pipeline": E2E_PIPELINE},
        "gpu_launches": args.steps,
        "host_us_per_call": {"c_abi": round(host_c * 1e6, 2), "python_binding":
                             round(host_py * 1e6, 2), "kernel": round(per_launch * 1e6, 2),
                             "eager_device_per_call": round(eager * 1e6, 2),
                             "note": "host time to enqueue one call (no synchronisation), "
                                     "mean of %d; eager: %d calls launched one by one, device "
                                     "time per call" % (n_host, args.steps)},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clocks,
    }


def run_ours(args):
    world, rank, local, dev = gpu_context()
    if args.workload == "all":
        head = measure_forward(HEADLINE_WORKLOAD, args, world, rank, local, dev, args.cpu_budget)
        configs = {}
        for name in CONFIG_WORKLOADS:
            c = measure_forward(name, args, world, rank, local, dev, args.config_cpu_budget)
            configs[name] = {k_: c[k_] for k_ in ("value", "unit", "ms_per_step", "dtype",
                                                  "config", "roofline", "e2e",
                                                  "host_us_per_call", "cpu_baseline", "clocks",
                                                  "gpu_launches")}
            if name == "enc_f32_b2_h8_l32_d64":
                configs[name]["note"] = ("parity configuration (0.5 MB, 4.2 MFLOP): "
                                         "launch-bound, not a throughput target")
        line = dict(head)
        line["metric"] = BASELINE_METRIC
        line["configs"] = configs
        line["gpu_launches"] = head["gpu_launches"]
    else:
        line = measure_forward(args.workload, args, world, rank, local, dev, args.cpu_budget)
    if rank == 0:
        line = {"metric": line["metric"], "value": line["value"], "unit": line["unit"],
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": line["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                **{k_: v_ for k_, v_ in line.items()
                   if k_ not in ("metric", "value", "unit", "steps", "ms_per_step")}}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# multi-head sublayer workloads (projections + attention + output projection)
# ---------------------------------------------------------------------------
def sublayer_flops(spec, lens):
    """Projection flops (2 M K N each, with the realised shapes) plus the
    attention step's algorithmic flops."""
    B, T, S, d = spec["B"], spec["T"], spec["S"], spec["d_model"]
    H, Hkv, dk, dv = spec["H"], spec["H_kv"], spec["dk"], spec["dv"]
    proj = 2 * B * (T * d * H * dk + S * d * Hkv * dk + S * d * Hkv * dv + T * H * dv * d)
    _, att = algorithmic(gen.sublayer_attention_spec(spec), lens)
    return int(proj), int(att)


def sublayer_oracle_time(spec, inp, frac_b):
    """Oracle seconds for the first ceil(frac_b * B) batch elements."""
    import oracle
    nb = max(1, int(math.ceil(spec["B"] * frac_b)))
    sl = slice(0, nb)
    x = inp["x"][sl]
    mem = inp["mem"][sl] if inp["mem"] is not None else x
    lens = inp["lens"][sl] if inp["lens"] is not None else None
    t0 = time.perf_counter()
    oracle.mha_sublayer(x, mem, *inp["w"], *inp["b"], H=spec["H"], H_kv=spec["H_kv"],
                        mask_kind=spec["mask"], key_lengths=lens,
                        scale=gen.default_scale(spec["dk"]))
    return time.perf_counter() - t0, nb / spec["B"]


def sublayer_oracle_baseline(spec, inp, flops, budget_s):
    import oracle
    oracle.build()
    t1, f1 = sublayer_oracle_time(spec, inp, 1.0 / spec["B"])
    frac = min(1.0, budget_s / max(t1 / f1, 1e-9))
    t, frac = sublayer_oracle_time(spec, inp, frac)
    nb = int(round(frac * spec["B"]))
    return {"value": flops * frac / t / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": "the first %d of %d batch elements (%.3g%%), %.1f s; work scaled by the "
                      "sampled share" % (nb, spec["B"], 100 * frac, t)}


def run_sublayer(args):
    import torch

    import transformer_head_scaled_mha_gb300 as mha

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    spec = gen.SUBLAYERS[args.workload]
    inp = gen.make_sublayer_inputs(spec, seed=args.seed)
    lens = inp["lens"]
    proj_flops, att_flops = sublayer_flops(spec, lens)
    flops = proj_flops + att_flops
    B, T, S, d = spec["B"], spec["T"], spec["S"], spec["d_model"]
    H, Hkv, dk, dv = spec["H"], spec["H_kv"], spec["dk"], spec["dv"]
    scale = gen.default_scale(dk)
    mask = spec["mask"]

    def host(a):
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16)

    hx = host(inp["x"])
    hm = host(inp["mem"]) if inp["mem"] is not None else None
    w = [host(a).to(dev) for a in inp["w"]]
    bias = [host(a).to(dev) for a in inp["b"]]
    kl = torch.from_numpy(lens).to(dev) if lens is not None else None
    set_bytes = hx.numel() * 2 * 2 + (hm.numel() * 2 if hm is not None else 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(1, math.ceil(3 * l2 / set_bytes))
    sets = [(hx.to(dev), hm.to(dev) if hm is not None else None,
             torch.empty((B, T, d), dtype=torch.bfloat16, device=dev)) for _ in range(n_sets)]
    ws = torch.empty(mha.mha_sublayer_workspace_size(B, T, S, d, H, Hkv, dk, dv),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i, s):
        xx, mm, oo = sets[i % n_sets]
        mha.mha_sublayer_fwd(xx, *w, *bias, mem=mm, H=H, H_kv=Hkv, mask_kind=mask,
                             key_lengths=kl, scale=scale, workspace=ws, out=oo, stream=s)

    def timed(fn, steps):
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                fn(i, stream)
        stream.synchronize()
        run, elapsed_of, _ = graph_timer(stream, fn, steps)
        run()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize(dev)
        run()
        torch.cuda.synchronize(dev)
        barrier(world)
        return elapsed_of() / steps

    sampler = ClockSampler(local)
    sampler.start()
    t_soak = time.time()
    per_step = timed(step, args.steps)
    per_step = max_over_ranks(per_step, world, dev)
    t_wall1 = time.time()
    sampler.mark(t_soak, t_wall1)
    clocks = sampler.stop()
    value = flops / per_step / 1e12 * world
    st = mha.mha_debug_status(stream)
    if st != mha.MHA_OK:
        raise RuntimeError("device status after timing: %s" % mha.mha_status_string(st))

    # the dominant kernel, the projection, timed alone on the query projection
    xq = [s_[0].view(B * T, d) for s_ in sets]
    yq = torch.empty((B * T, H * dk), dtype=torch.bfloat16, device=dev)

    def lin(i, s):
        mha.mha_linear_fwd(xq[i % n_sets], w[0], bias[0], yq, stream=s)
    lin_t = timed(lin, args.steps)
    lin_flops = 2 * B * T * d * H * dk
    peaks, peak_src = read_peaks()
    achieved = lin_flops / lin_t / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": recorded_traffic(args.workload + ":linear"),
                "kernel": "%s (query projection %dx%dx%d, timed alone)" % (
                    linear_kernel_name(d, H * dk), B * T, d, H * dk),
                "peak_source": peak_src + " (MEASURED_PEAKS.json)" if peak_src == "measured"
                else "fallback", "algorithmic_flops": lin_flops,
                "sublayer_share": {"projections_flops": proj_flops, "attention_flops": att_flops}}

    # e2e: token vectors (and lengths) in, sublayer output back, every step;
    # the weights stay resident like a model's parameters
    px = hx.pin_memory()
    pm = hm.pin_memory() if hm is not None else None
    pl = torch.from_numpy(lens).pin_memory() if lens is not None else None
    pout = torch.empty((B, T, d), dtype=torch.bfloat16).pin_memory()
    h2d = px.numel() * 2 + (pm.numel() * 2 if pm is not None else 0) + (
        pl.numel() * 4 if pl is not None else 0)
    d2h = pout.numel() * 2
    # per slot: x, mem, out, lengths, workspace (slot 0 reuses the first set)
    dx, dm, do = sets[0]
    e2e_dev = [[dx, dm, do, torch.empty_like(kl) if kl is not None else None, ws]]
    e2e_dev.append([torch.empty_like(t) if t is not None else None for t in e2e_dev[0]])
    slots_in = [[(e[0], px)] + ([(e[1], pm)] if pm is not None else []) +
                ([(e[3], pl)] if pl is not None else []) for e in e2e_dev]
    slots_out = [[(pout, e[2])] for e in e2e_dev]

    def e2e_launch(s, st):
        e = e2e_dev[s]
        mha.mha_sublayer_fwd(e[0], *w, *bias, mem=e[1], H=H, H_kv=Hkv, mask_kind=mask,
                             key_lengths=e[3], scale=scale, workspace=e[4], out=e[2], stream=st)

    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    e2e_t = max_over_ranks(e2e_seconds_per_step(slots_in, e2e_launch, slots_out, e2e_steps,
                                                stream, world), world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = sublayer_oracle_baseline(spec, inp, flops, args.cpu_budget)
    if rank == 0:
        line = {
            "metric": "multi-head sublayer TFLOP/s", "value": round(value, 3),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded: x, mem N(0,1); W N(0,1/fan_in); b N(0,0.01); seed %d)"
                    % args.seed,
            "config": {"workload": args.workload, "B": B, "T": T, "S": S, "d_model": d,
                       "H": H, "H_kv": Hkv, "d_k": dk, "d_v": dv, "mask_kind": mask,
                       "len_range": spec["len_range"], "cross": spec["cross"],
                       "l2": "inputs rotate over %d device copies (%.0f MB > 3x L2 %.0f MB)"
                             % (n_sets, n_sets * set_bytes / 1e6, l2 / 1e6),
                       "timing": "CUDA graph of %d calls (3 launches each: the three "
                                 "projections, the attention, the output projection), CUDA "
                                 "events recorded as the graph's first and last nodes"
                                 % args.steps,
                       "parallelism": "weak: same workload per rank, no collective"
                       if world > 1 else "1 GPU"},
            "e2e": {"value": round(flops / e2e_t / 1e12 * world, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "note": "weights resident on the device", "pipeline": E2E_PIPELINE},
            "gpu_launches": 3 * args.steps,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference_sublayer(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    spec = gen.SUBLAYERS[args.workload]
    inp = gen.make_sublayer_inputs(spec, seed=args.seed)
    proj, att = sublayer_flops(spec, inp["lens"])
    flops = proj + att
    import oracle
    oracle.build()
    t1, f1 = sublayer_oracle_time(spec, inp, 1.0 / spec["B"])
    frac = min(1.0, args.ref_step_budget / max(t1 / f1, 1e-9))
    for _ in range(args.warmup):
        sublayer_oracle_time(spec, inp, frac)
    runs = [sublayer_oracle_time(spec, inp, frac) for _ in range(args.steps)]
    t = sum(r[0] for r in runs)
    frac = runs[0][1]
    value = flops * frac * args.steps / t / 1e12
    sample = "each step: the first %d of %d batch elements, scaled by the sampled share" % (
        int(round(frac * spec["B"])), spec["B"])
    line = {"impl": "reference", "metric": "multi-head sublayer TFLOP/s",
            "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * t / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, seed %d)" % args.seed,
            "config": {"workload": args.workload, "B": spec["B"], "T": spec["T"],
                       "S": spec["S"], "d_model": spec["d_model"], "H": spec["H"],
                       "H_kv": spec["H_kv"], "mask_kind": spec["mask"]},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    spec = gen.WORKLOADS[args.workload]
    q, k, v, lens = gen.make_inputs(spec, seed=args.seed)
    metric, unit = metric_of(spec)
    import oracle
    oracle.build()
    nbytes, flops = algorithmic(spec, lens)
    # each step: one bounded random sample of the workload's rows
    budget = args.ref_step_budget
    probe_rows, probe_frac = oracle_sample_rows(spec, lens, 2e8)
    t_probe = time_oracle(spec, q, k, v, lens, probe_rows)
    rate = flops * probe_frac / max(t_probe, 1e-6)
    rows, frac = oracle_sample_rows(spec, lens, rate * budget, seed=2)
    for _ in range(args.warmup):
        time_oracle(spec, q, k, v, lens, rows)
    times = [time_oracle(spec, q, k, v, lens, rows) for _ in range(args.steps)]
    t = sum(times)
    value = throughput(spec, nbytes * frac * args.steps, flops * frac * args.steps, t)
    cores = oracle.max_threads()
    n_rows = spec["B"] * spec["H"] * spec["Lq"] if rows is None else len(rows)
    sample = ("each step: %d of %d query rows (%.4g%%), uniform random, scaled by the sampled "
              "share" % (n_rows, spec["B"] * spec["H"] * spec["Lq"], 100 * frac))
    line = {"impl": "reference", "metric": metric, "value": round(value, 6), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, seed %d)" % args.seed,
            "config": {"workload": args.workload, "B": spec["B"], "H": spec["H"],
                       "Lq": spec["Lq"], "Lk": spec["Lk"], "d_k": spec["dk"], "d_v": spec["dv"],
                       "mask_kind": spec["mask"], "len_range": spec["len_range"]},
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# backward workloads: the gradients dq, dk, dv of a forward workload
# ---------------------------------------------------------------------------
def backward_flops(spec, lens):
    """Algorithmic flops of the backward pass: per allowed (query, key) pair the
    scores recomputed (2 d_k), dP = dout v (2 d_v), dV (2 d_v), dK (2 d_k) and
    dQ (2 d_k) -- 2 (3 d_k + 2 d_v), 2.5 times the forward's 2 (d_k + d_v)."""
    _, fwd = algorithmic(spec, lens)
    dk, dv = spec["dk"], spec["dv"]
    return int(fwd * (3 * dk + 2 * dv) // (dk + dv))


def oracle_backward_time(spec, inp, units, rows):
    """Seconds for the oracle's backward pass over some (batch, key/value head)
    units and a range of query rows in each, and the share of the whole
    workload's allowed (query, key) pairs that sample holds."""
    import oracle
    q, k, v, lens, dout = inp
    scale = gen.default_scale(spec["dk"])
    t0 = time.perf_counter()
    oracle.mha_bwd(q, k, v, dout, mask_kind=spec["mask"], key_lengths=lens, scale=scale,
                   layout=spec.get("layout", "bhsd"), units=units, rows=rows)
    t = time.perf_counter() - t0
    return t, sample_pair_share(spec, lens, units, rows)


def sample_pair_share(spec, lens, units, rows):
    """Share of all allowed (query, key) pairs that lie in the sampled units and rows."""
    B, H, Lq, Lk = spec["B"], spec["H"], spec["Lq"], spec["Lk"]
    Hkv = spec.get("Hkv", H)
    m = spec["mask"]
    L = np.full(B, Lk, dtype=np.int64) if lens is None else np.clip(lens.astype(np.int64), 0, Lk)
    i_lo, i_hi = (0, Lq) if rows is None else rows

    def pairs_of(b, lo, hi):
        kmax = int(L[b]) if m & gen.MASK_KEY_PADDING else Lk
        hi = min(hi, int(L[b])) if m & gen.MASK_QUERY_PADDING else hi
        i = np.arange(lo, max(lo, hi))
        if m & gen.MASK_CAUSAL:
            return int(np.minimum(i + 1, kmax).sum())
        if m & gen.MASK_CAUSAL_TAIL:
            return int(np.clip(kmax - Lq + i + 1, 0, kmax).sum())
        return len(i) * kmax

    total = sum(pairs_of(b, 0, Lq) for b in range(B)) * H
    us = range(B * Hkv) if units is None else units
    part = sum(pairs_of(u // Hkv, i_lo, i_hi) for u in us) * (H // Hkv)
    return part / max(total, 1)


def backward_sample(spec, inp, budget_s):
    """Units and a row range whose oracle backward takes about budget_s."""
    B, Hkv, Lq = spec["B"], spec.get("Hkv", spec["H"]), spec["Lq"]
    # probe: one unit, a row range sized for a fraction of a second
    rows = (max(0, Lq - 64), Lq)
    t, share = oracle_backward_time(spec, inp, [0], rows)
    rate = share / max(t, 1e-6)  # workload share per second
    want = rate * budget_s
    import oracle
    one_unit = sample_pair_share(spec, inp[3], [0], None)
    if want >= one_unit:
        n = max(1, min(B * Hkv, int(want / max(one_unit, 1e-12))))
        return list(range(n)), None
    # less than one unit's work: the last rows of as many units as host
    # threads, so every thread has a unit (the oracle runs one per thread)
    units = list(range(min(B * Hkv, max(1, oracle.max_threads()))))
    per = sample_pair_share(spec, inp[3], units, None)
    n_rows = max(1, min(Lq, int(Lq * want * len(units) / max(per, 1e-12))))
    return units, (max(0, Lq - n_rows), Lq)


def run_backward(args):
    import torch

    import transformer_head_scaled_mha_gb300 as mha

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    fwd_name = BWD_WORKLOADS[args.workload]
    spec = gen.WORKLOADS[fwd_name]
    q, k, v, lens = gen.make_inputs(spec, seed=args.seed)
    dout = gen.make_dout(spec, seed=args.seed)
    flops = backward_flops(spec, lens)
    scale = gen.default_scale(spec["dk"])
    mask = spec["mask"]
    layout = spec.get("layout", "bhsd")
    B, H, Lq, Lk, dk, dv = (spec[x] for x in ("B", "H", "Lq", "Lk", "dk", "dv"))
    Hkv = spec.get("Hkv", H)

    def host(a):
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16)

    hq, hk, hv, hdo = host(q), host(k), host(v), host(dout)
    kl = torch.from_numpy(lens).to(dev) if lens is not None else None
    # the forward output and row statistics the backward reads, from the
    # forward kernel itself (as a training step keeps them)
    out0, lse0 = mha.mha_fwd_lse(hq.to(dev), hk.to(dev), hv.to(dev), layout=layout,
                                 mask_kind=mask, key_lengths=kl, scale=scale)
    hout, hlse = out0.cpu(), lse0.cpu()
    ins = (hq, hk, hv, hout, hdo)
    set_bytes = sum(t.numel() * 2 for t in ins) + (hq.numel() + hk.numel() + hv.numel()) * 2 + \
        hlse.numel() * 4
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(1, math.ceil(3 * l2 / set_bytes))
    sets = [tuple(t.to(dev) for t in ins) + (torch.empty_like(hq, device=dev),
                                             torch.empty_like(hk, device=dev),
                                             torch.empty_like(hv, device=dev), hlse.to(dev))
            for _ in range(n_sets)]
    ws = torch.empty(max(1, mha.mha_bwd_workspace_size(B, H, Lq)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step_with(use_lse):
        def step(i, s):
            qq, kk, vv, oo, gg, dq, dk_, dv_, ls = sets[i % n_sets]
            mha.mha_bwd(qq, kk, vv, oo, gg, layout=layout, mask_kind=mask, key_lengths=kl,
                        scale=scale, workspace=ws, dq=dq, dk=dk_, dv=dv_, stream=s,
                        lse=ls if use_lse else None)
        return step

    # the call without the forward's statistics (a statistics pass first),
    # timed for comparison only
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step_with(False)(i, stream)
    stream.synchronize()
    replay0, elapsed0, _ = graph_timer(stream, step_with(False), args.steps)
    for _ in range(2):  # the first replay uploads the graph
        replay0()
        torch.cuda.synchronize(dev)
    stats_pass_ms = max_over_ranks(elapsed0(), world, dev) / args.steps * 1e3
    del replay0

    step = step_with(True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, stream)
    stream.synchronize()
    replay, elapsed_of, timing = graph_timer(stream, step, args.steps)

    sampler = ClockSampler(local)
    sampler.start()
    t_soak = time.time()
    while time.time() - t_soak < args.soak:
        replay()
        stream.synchronize()
    barrier(world)
    torch.cuda.synchronize(dev)
    replay()
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    sampler.mark(t_soak + min(0.2, args.soak / 2), t_wall1)
    clocks = sampler.stop()
    per_step = max_over_ranks(elapsed_of(), world, dev) / args.steps
    value = flops / per_step / 1e12 * world
    st = mha.mha_debug_status(stream)
    if st != mha.MHA_OK:
        raise RuntimeError("device status after timing: %s" % mha.mha_status_string(st))

    # roofline: the whole backward call (stats, dq and dkdv launches) against
    # the bf16 tensor peak; the ncu launch list splits its time by kernel
    peaks, peak_src = read_peaks()
    achieved = flops / per_step / 1e12
    kernels, traffic_kernel = bwd_kernel_names(dk, Lq, Lk, mask)
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": recorded_traffic(args.workload), "traffic_kernel": traffic_kernel,
                "kernel": kernels,
                "peak_source": peak_src + " (MEASURED_PEAKS.json)" if peak_src == "measured"
                else "fallback", "algorithmic_flops": flops}

    # e2e: q, k, v, out, dout (and lengths) in, dq, dk, dv back, every step
    pins = [t.pin_memory() for t in ins]
    plse = hlse.pin_memory()
    pl = torch.from_numpy(lens).pin_memory() if lens is not None else None
    pouts = [torch.empty_like(t).pin_memory() for t in (hq, hk, hv)]
    h2d = sum(t.numel() * 2 for t in pins) + plse.numel() * 4 + \
        (pl.numel() * 4 if pl is not None else 0)
    d2h = sum(t.numel() * 2 for t in pouts)
    # per slot: q, k, v, out, dout, dq, dk, dv, lse, lengths, workspace (slot
    # 0 reuses the first set)
    e2e_dev = [list(sets[0][:9]) + [torch.empty_like(kl) if kl is not None else None, ws]]
    e2e_dev.append([torch.empty_like(t) if t is not None else None for t in e2e_dev[0]])
    slots_in = [list(zip(e[:5], pins)) + [(e[8], plse)] +
                ([(e[9], pl)] if pl is not None else []) for e in e2e_dev]
    slots_out = [list(zip(pouts, e[5:8])) for e in e2e_dev]

    def e2e_launch(s, st):
        e = e2e_dev[s]
        mha.mha_bwd(*e[:5], layout=layout, mask_kind=mask, key_lengths=e[9], scale=scale,
                    workspace=e[10], dq=e[5], dk=e[6], dv=e[7], stream=st, lse=e[8])

    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    e2e_t = max_over_ranks(e2e_seconds_per_step(slots_in, e2e_launch, slots_out, e2e_steps,
                                                stream, world), world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        inp = (q, k, v, lens, dout)
        units, rows = backward_sample(spec, inp, args.cpu_budget)
        t, share = oracle_backward_time(spec, inp, units, rows)
        cpu = {"value": flops * share / t / 1e12, "unit": "TFLOP/s",
               "cores": min(oracle.max_threads(), len(units)), "kind": "oracle",
               "sample": "%d of %d (batch, key/value head) units, query rows %s; %.4g%% of the "
                         "allowed (query, key) pairs, %.1f s; work scaled by that share" % (
                             len(units), B * Hkv, "all" if rows is None else "%d..%d" % (
                                 rows[0], rows[1] - 1), 100 * share, t)}
    if rank == 0:
        line = {
            "metric": "attention bwd TFLOP/s", "value": round(value, 3), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1)%s q, k, v and dout; out from the forward "
                    "kernel; seed %d)" % ("*%g" % spec["amp"] if spec["amp"] != 1.0 else "",
                                          args.seed),
            "config": {"workload": args.workload, "forward": fwd_name, "B": B, "H": H,
                       "H_kv": Hkv, "layout": layout, "Lq": Lq, "Lk": Lk, "d_k": dk,
                       "d_v": dv, "mask_kind": mask, "len_range": spec["len_range"],
                       "scale": scale,
                       "l2": "inputs rotate over %d device copies (%.0f MB > 3x L2 %.0f MB)"
                             % (n_sets, n_sets * set_bytes / 1e6, l2 / 1e6),
                       "timing": timing.replace("launches", "mha_bwd_lse calls"),
                       "statistics": "the forward's (mha_fwd_lse) row statistics, as a "
                                     "training step keeps them",
                       "ms_per_step_with_statistics_pass": round(stats_pass_ms, 6),
                       "parallelism": "weak: same workload per rank, no collective"
                       if world > 1 else "1 GPU"},
            "e2e": {"value": round(flops / e2e_t / 1e12 * world, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "pipeline": E2E_PIPELINE},
            "gpu_launches": (1 if spec["dk"] == 64 and Lq <= 128 and Lk <= 128 else 3) * args.steps,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference_backward(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    spec = gen.WORKLOADS[BWD_WORKLOADS[args.workload]]
    q, k, v, lens = gen.make_inputs(spec, seed=args.seed)
    dout = gen.make_dout(spec, seed=args.seed)
    flops = backward_flops(spec, lens)
    import oracle
    oracle.build()
    inp = (q, k, v, lens, dout)
    units, rows = backward_sample(spec, inp, args.ref_step_budget)
    for _ in range(args.warmup):
        oracle_backward_time(spec, inp, units, rows)
    runs = [oracle_backward_time(spec, inp, units, rows) for _ in range(args.steps)]
    t = sum(r[0] for r in runs)
    share = runs[0][1]
    value = flops * share * args.steps / t / 1e12
    B, Hkv = spec["B"], spec.get("Hkv", spec["H"])
    sample = ("each step: %d of %d (batch, key/value head) units, query rows %s (%.4g%% of the "
              "allowed pairs), scaled by that share" % (
                  len(units), B * Hkv, "all" if rows is None else "%d..%d" % (rows[0], rows[1] - 1),
                  100 * share))
    line = {"impl": "reference", "metric": "attention bwd TFLOP/s", "value": round(value, 6),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, seed %d)" % args.seed,
            "config": {"workload": args.workload, "forward": BWD_WORKLOADS[args.workload],
                       "B": B, "H": spec["H"], "Lq": spec["Lq"], "Lk": spec["Lk"],
                       "d_k": spec["dk"], "d_v": spec["dv"], "mask_kind": spec["mask"]},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                             "cores": min(oracle.max_threads(), len(units)), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["all"] + sorted(gen.WORKLOADS) + sorted(gen.SUBLAYERS) +
                    sorted(BWD_WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true", help="eager launches instead of a graph")
    ap.add_argument("--soak", type=float, default=1.0, help="untimed load before timing, s")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="oracle baseline budget, s")
    ap.add_argument("--config-cpu-budget", type=float, default=4.0,
                    help="oracle baseline budget of each non-headline configuration, s")
    ap.add_argument("--ref-step-budget", type=float, default=2.0, help="reference arm s/step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    world, _, _ = dist_env()
    if world != args.gpus:
        if not (world == 1 and args.gpus == 1):
            print("warning: --gpus %d but WORLD_SIZE %d; using WORLD_SIZE" % (args.gpus, world),
                  file=sys.stderr)
    if args.workload in BWD_WORKLOADS:
        (run_reference_backward if args.impl == "reference" else run_backward)(args)
        return
    sub = args.workload in gen.SUBLAYERS
    if args.impl == "reference" and args.workload == "all":
        args.workload = HEADLINE_WORKLOAD  # the reference arm times the headline configuration
    if args.impl == "reference":
        (run_reference_sublayer if sub else run_reference)(args)
    else:
        (run_sublayer if sub else run_ours)(args)


if __name__ == "__main__":
    main()
