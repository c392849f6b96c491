#!/usr/bin/env python
"""Benchmark of the paged-KV varlen attention forward on one GB300 (or N replicas).

A step is one pa_varlen_fwd call over one synthetic serving batch (default: the
decode batch -- 64 sequences, q_len 1, sk ~ U[512, 4096], H=32, Hkv=8, D=128,
page 32, bf16).  The headline value is the algorithmic KV GB/s of that step; the
roofline object compares its dominant kernel with the measured HBM copy bandwidth (and,
labelled apart, with the nominal ~7.9 TB/s).  Beside it: `secondary`, the causal-prefill
workload in TFLOP/s against the measured (and nominal) dense bf16 peak, and `workloads`,
the chunked-prefill + decode batch with a sliding window and the long-context split-KV
batches at head_dim 256 and 512, each with its own roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica (the path needs no
exchange); rank 0 prints one JSON line with the whole-job value.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "paged-attn TFLOP/s (prefill) and KV GB/s (decode), % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# nominal GB300 figures: HBM3e ~7.9 TB/s, dense bf16 tensor 2.25 PFLOP/s (the targets' "~8 TB/s"
# and "dense bf16 peak"); reported beside the measured copy / matmul rates, labelled as such
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0
L2_BYTES = 129 * 1024 * 1024
# the serving workloads measured beside the headline (chunked prefill + decode with a window,
# long-context split-KV decode at head_dim 256 and 512, the decode batch with one sequence
# far longer than the rest, and the causal prefill batch at head_dim 256)
EXTRA_WORKLOADS = ("mixed_bf16", "long_bf16", "long_d512_bf16", "skewed_decode_bf16", "prefill_d256_bf16")


# ---- algorithmic work (closed form per query row) -----------------------------------------

def algorithmic(lay, seqs=None):
    """(FLOPs, bytes) of one pass: FLOPs = 4 * D * H * sum over rows of attended keys;
    bytes = K+V of the union of attended keys per sequence and kv head, plus q, out
    (input dtype) and lse (fp32)."""
    elt = 2
    H, Hkv, D = lay.num_heads, lay.num_heads_k, lay.head_dim
    wl, wr = lay.window_left, lay.window_right
    flops = 0
    keys = 0
    rows = 0
    for b in (range(lay.batch) if seqs is None else seqs):
        sq, sk = lay.seqlens_q[b], lay.seqlens_k[b]
        if sq == 0:
            continue
        i = np.arange(sq, dtype=np.int64)
        c = sk - sq
        lo = np.maximum(0, i + c - wl) if wl >= 0 else np.zeros(sq, dtype=np.int64)
        hi = np.minimum(sk - 1, i + c + wr) if wr >= 0 else np.full(sq, sk - 1, dtype=np.int64)
        n = np.maximum(0, hi - lo + 1)
        flops += 4 * D * H * int(n.sum())
        live = n > 0
        if live.any():
            keys += int(hi[live].max() - lo[live].min() + 1)
        rows += sq
    kv = 2 * Hkv * D * elt * keys
    qo = 2 * rows * H * D * elt
    lse = 4 * H * rows
    return flops, kv + qo + lse


def pool_bytes(lay):
    """Bytes of the K and V pools (the data a step re-reads from one call to the next)."""
    return 2 * lay.num_blocks * lay.page_block_size * lay.num_heads_k * lay.head_dim * 2


def l2_label(nbytes, what="K/V"):
    return (f"{what} larger than twice L2 (no flush)" if nbytes > 2 * L2_BYTES
            else f"{what} within twice L2: L2 flushed (a 3x L2 buffer written, another read) before every "
                 "timed call, outside the timed events")


class L2Flush:
    """Before each timed call, when the K/V a step reads is small enough to stay resident in
    L2 between calls (a no-op otherwise): writes a buffer three times the size of L2, then
    reads a second one of that size, so that the call finds neither its own inputs nor the
    flush's dirty lines in L2 (writing those back would otherwise fall inside the timed
    call: 2.7 us of a 34 us split kernel on long_d512_bf16, ~20 us on the 1.1 GB long_bf16
    batch); then holds the GPU for ~0.1 ms with a spin kernel, so that the call is already
    enqueued when the timed region starts and the events measure its device time (the
    host's share of a call is in the e2e figure)."""

    def __init__(self, kv_bytes):
        import torch
        small = kv_bytes <= 2 * L2_BYTES
        self.buf = torch.empty(3 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if small else None
        self.rbuf = torch.zeros(3 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if small else None
        self.acc = torch.empty((), dtype=torch.float32, device="cuda") if small else None

    def __bool__(self):
        return self.buf is not None

    def __call__(self):
        if self.buf is not None:
            import torch
            self.buf.zero_()
            torch.sum(self.rbuf, dim=0, out=self.acc)
            torch.cuda._sleep(200_000)


def timed_calls(step, steps, flush):
    """Average device time (ms) of `steps` calls of `step` on the current stream: one event
    pair around all of them, or, when L2 is flushed, one pair around each call with the
    flush before it outside the events."""
    import torch
    stream = torch.cuda.current_stream()
    if not flush:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    pairs = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs) / steps


def workload_config(lay, flops, nbytes, world):
    """The `config` object of the JSON line (both arms)."""
    return {"workload": lay.name, "batch": lay.batch, "num_heads": lay.num_heads,
            "num_heads_k": lay.num_heads_k, "head_dim": lay.head_dim,
            "page_block_size": lay.page_block_size, "max_seqlen_k": lay.max_seqlen_k,
            "total_keys": lay.total_k, "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
            "l2": l2_label(pool_bytes(lay)),
            "parallelism": f"replicas{world}",
            **({"alibi_slopes": "2^(-8 (h + 1) / H)"} if ALIBI["slopes"] is not None else {})}


def headline_unit(flops, nbytes):
    """("TFLOP/s", 1e12) for a workload above the ridge point of the peaks, else ("GB/s", 1e9),
    with the matching amount of work per step."""
    hbm, bf16, _, _ = peaks()
    if flops / nbytes > (bf16 * 1e12) / (hbm * 1e9):
        return "TFLOP/s", flops / 1e12
    return "GB/s", nbytes / 1e9


def max_over_ranks(value, dist, device):
    """The largest of every rank's value (the slowest rank's time); `dist` None on one GPU."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(work_per_rank, world, ms_max):
    """Whole-job throughput of N replicas: every rank runs the same step on its own GPU (the
    path has no exchange between (sequence, kv head) units), so the job does `world` times
    the per-rank work in the slowest rank's time."""
    return world * work_per_rank / (ms_max * 1e-3)


def kernel_class_seqs(lay):
    """Sequences per kernel class, mirroring the library's dispatch: sequences with more
    than 32 rows (sq * G) go to the tensor-core prefill kernels when they take the call
    (head_dim <= 256, G <= 128, softmax_scale > 0), the rest to the split-KV pass."""
    G = lay.num_heads // lay.num_heads_k
    tc = (lay.head_dim <= 256 and G <= 128 and lay.softmax_scale > 0
          and max(lay.seqlens_q) * G > 32 and not os.environ.get("PA_DISABLE_TC_PREFILL"))
    pre = [b for b in range(lay.batch) if tc and lay.seqlens_q[b] * G > 32]
    split = [b for b in range(lay.batch) if b not in set(pre)]
    return {"prefill": pre, "splitkv": split}


def time_kernels(binding, g, lay, steps, flush=None):
    """Per-kernel device time: the library brackets each launch with CUDA events on the
    stream it is launched on.  Returns {class: (ms per launch, launches per step)}."""
    import torch
    out = torch.empty_like(g.q)
    lse = torch.empty((lay.num_heads, lay.total_q), dtype=torch.float32, device=g.q.device)
    torch.cuda.synchronize()
    binding.kernel_times()  # drop anything recorded earlier
    binding.kernel_timing(True)
    try:
        for _ in range(steps):
            if flush:
                flush()
            _call(binding, g, lay, out, lse)
        torch.cuda.synchronize()
    finally:
        binding.kernel_timing(False)
    t = binding.kernel_times()
    return {k: (ms / n, n / steps) for k, (ms, n) in t.items() if n > 0}


# ---- peaks, profiles, clocks ------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            p = json.load(open(path))
            return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                    float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def csrc_hash():
    """Hash of the kernels and their launch code (csrc/), which determine the traffic."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "paged_kv_varlen_flashattention_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".cpp", ".h")):
            h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def profiled_traffic(workload):
    """DRAM bytes per launch of the workload's dominant kernel from the committed ncu capture
    (profiles/traffic.json: dram__bytes_read.sum + dram__bytes_write.sum, with the hash of the
    kernel sources it was taken on), or None if there is none for the current sources."""
    try:
        entry = json.load(open(TRAFFIC_JSON))["captures"][workload]
    except Exception:
        return None
    if entry.get("csrc_sha256_16") != csrc_hash():
        return None
    return float(entry["dram_read_bytes"]) + float(entry["dram_write_bytes"])


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, val in zip(names, f[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---- the measured arm ----------------------------------------------------------------------------

ALIBI = {"slopes": None}  # set by --alibi: per-head slopes (numpy float32) given to every leg


def alibi_slopes(num_heads):
    """The usual geometric slopes of the linear position bias, 2^(-8 (h + 1) / H)."""
    return np.array([2.0 ** (-8.0 * (h + 1) / num_heads) for h in range(num_heads)], dtype=np.float32)


def set_alibi(args, lay):
    ALIBI.clear()
    ALIBI["slopes"] = alibi_slopes(lay.num_heads) if getattr(args, "alibi", False) else None


def _slopes_on(device):
    import torch
    s = ALIBI["slopes"]
    if s is None:
        return None
    key = f"t_{device}"
    if key not in ALIBI:
        ALIBI[key] = torch.from_numpy(s).to(device)
    return ALIBI[key]


def _call(binding, g, lay, out, lse, stream=None):
    binding.varlen_fwd(g.q, g.k_cache, g.v_cache, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table,
                       max_seqlen_q=lay.max_seqlen_q, max_seqlen_k=lay.max_seqlen_k,
                       softmax_scale=lay.softmax_scale, window_left=lay.window_left,
                       window_right=lay.window_right, out=out, softmax_lse=lse, stream=stream,
                       alibi_slopes=_slopes_on(g.q.device))


def time_device(binding, g, lay, steps, warmup, dist, flush=None):
    import torch
    out = torch.empty_like(g.q)
    lse = torch.empty((lay.num_heads, lay.total_q), dtype=torch.float32, device=g.q.device)
    for _ in range(warmup):
        _call(binding, g, lay, out, lse)
    torch.cuda.synchronize()
    st = binding.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}: {binding.last_error()}")
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = binding.kernel_launches()
    ms = timed_calls(lambda: _call(binding, g, lay, out, lse), steps, flush)
    if dist:
        dist.barrier()
    launches = binding.kernel_launches() - n0
    return ms, launches


def time_e2e(binding, g, lay, steps, warmup):
    """Same step through the public call with host-resident inputs: pinned host -> device
    copies of every input, the call, and device -> host copies of out and lse, all timed.
    The inputs alternate between two device buffer sets, and their copies run on a copy
    stream, so that step i + 1's copies (the host link is the limit: ~210 GB/s pinned, one
    stream or several alike) overlap step i's call; a set is overwritten only after the
    call that read it has finished."""
    import torch
    sl = _slopes_on("cpu")
    host = [t.cpu().pin_memory() if t is not None else None
            for t in (g.q, g.k_cache, g.v_cache, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table, sl)]
    sets = [[torch.empty_like(t, device="cuda") if t is not None else None for t in host] for _ in range(2)]
    out_h = torch.empty(g.q.shape, dtype=g.q.dtype).pin_memory()
    lse_h = torch.empty((lay.num_heads, lay.total_q), dtype=torch.float32).pin_memory()
    outs = [(torch.empty_like(g.q), torch.empty((lay.num_heads, lay.total_q), dtype=torch.float32, device="cuda"))
            for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host if t is not None)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * 4
    main = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    read_done = [None, None]  # event after the last call that read buffer set s

    def step(i):
        s = i % 2
        dev = sets[s]
        with torch.cuda.stream(copy_stream):
            if read_done[s] is not None:
                copy_stream.wait_event(read_done[s])
            for d, h in zip(dev, host):
                if d is not None:
                    d.copy_(h, non_blocking=True)
            copied = torch.cuda.Event()
            copied.record(copy_stream)
        main.wait_event(copied)
        binding.varlen_fwd(dev[0], dev[1], dev[2], dev[3], dev[4], dev[5], max_seqlen_q=lay.max_seqlen_q,
                           max_seqlen_k=lay.max_seqlen_k, softmax_scale=lay.softmax_scale,
                           window_left=lay.window_left, window_right=lay.window_right, out=outs[s][0],
                           softmax_lse=outs[s][1], alibi_slopes=dev[6])
        ev = torch.cuda.Event()
        ev.record(main)
        read_done[s] = ev
        out_h.copy_(outs[s][0], non_blocking=True)
        lse_h.copy_(outs[s][1], non_blocking=True)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    copy_stream.wait_event(e0)  # no copy of the timed steps starts before the start event
    for i in range(steps):
        step(i)
    e1.record(main)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


def cpu_baseline(lay, inp_cpu, budget_s=20.0):
    """The oracle, as it stands, on the host cores over a bounded sample of the workload:
    whole sequences (all heads) in a seeded order, repeated until about half the budget has
    been spent and never past the budget; returns (value in the workload's headline unit,
    unit, seconds, threads, sample text)."""
    import oracle
    order = list(range(lay.batch))
    rng = np.random.default_rng(0)
    rng.shuffle(order)
    cq, _ = lay.cu_seqlens()
    bt = inp_cpu.block_table.numpy() if inp_cpu.block_table is not None else None
    nbytes, nflops, t_total, runs, distinct, passes = 0, 0, 0.0, 0, set(), 0
    while t_total < 0.5 * budget_s:
        progressed = False
        for b in order:
            rows = np.arange(cq[b] * lay.num_heads, cq[b + 1] * lay.num_heads, dtype=np.int64)
            if len(rows) == 0:
                continue
            t0 = time.perf_counter()
            oracle.attention(lay.dtype, inp_cpu.q, inp_cpu.k_cache, inp_cpu.v_cache, inp_cpu.cu_seqlens_q.numpy(),
                             inp_cpu.cu_seqlens_k.numpy(), bt, lay.softmax_scale, lay.window_left,
                             lay.window_right, rows=rows, alibi_slopes=ALIBI["slopes"])
            t_total += time.perf_counter() - t0
            f_b, b_b = algorithmic(lay, [b])
            nflops += f_b
            nbytes += b_b
            runs += 1
            distinct.add(b)
            progressed = True
            if t_total > budget_s:
                break
        passes += 1
        if not progressed or t_total > budget_s:
            break
    sample = (f"{runs} sequence runs ({len(distinct)} of {lay.batch} sequences, all heads; "
              f"{passes} pass(es) in a seeded order), {t_total:.1f} s")
    unit, _ = headline_unit(*algorithmic(lay))
    work = nflops / 1e12 if unit == "TFLOP/s" else nbytes / 1e9
    return work / t_total, unit, t_total, oracle.threads(), sample


def kernel_names(lay):
    """Kernel class -> kernel name for a workload, mirroring the library's choice for the
    split-KV class: rows of at most 32 (q_len x group) go to the warp-sliced decode kernel for
    head_dim up to 256 and to the quarter-column decode kernel above (to the tensor-core decode
    kernel under PA_DECODE_TC=1); longer rows the prefill kernel does not take go to the
    general kernel."""
    G = lay.num_heads // lay.num_heads_k
    rows = max(q for q in lay.seqlens_q) * G if not kernel_class_seqs(lay)["prefill"] else 32
    dp = 64 if lay.head_dim <= 64 else 128 if lay.head_dim <= 128 else 256 if lay.head_dim <= 256 else 512
    tc = dp >= 128 and os.environ.get("PA_DECODE_TC", "") == "1"
    dec = ("splitkv_kernel" if rows > 32 else "decode_tc_kernel" if tc else
           "decode_kernel" if dp <= 256 else "decode512_kernel")
    return {"prefill": "prefill256_kernel" if lay.head_dim > 128 else "prefill_kernel", "combine": "combine_kernel",
            "splitkv": dec}


def roofline_of(binding, g, lay, steps, flush):
    """The roofline object of a workload's dominant kernel: its algorithmic work per launch
    (bytes of its sequences for the split-KV pass, FLOPs for the prefill kernel) over its own
    average launch duration (CUDA events around each launch, on the stream it runs on),
    against the measured peak, and beside it against the nominal GB300 peak."""
    hbm, bf16, _, peak_kind = peaks()
    per_kernel = time_kernels(binding, g, lay, steps, flush)
    # a class without sequences of its own (e.g. the split-KV pass of a prefill-only batch)
    # launches CTAs that exit at once; its events then mostly time the wait for SMs
    classes = kernel_class_seqs(lay)
    with_work = {k: v for k, v in per_kernel.items() if k == "combine" or classes.get(k)}
    dom = max((k for k in with_work if k != "combine"), key=lambda k: with_work[k][0] * with_work[k][1],
              default="combine")
    dom_ms, dom_launches = per_kernel[dom]
    f_d, b_d = algorithmic(lay, classes[dom]) if dom != "combine" else algorithmic(lay)
    dom_tensor = dom == "prefill" or (f_d / max(b_d, 1) > (bf16 * 1e12) / (hbm * 1e9))
    if dom_tensor:
        unit, peak, nominal, work = "TFLOP/s", bf16, NOMINAL_BF16_TFLOPS, f_d / 1e12 / dom_launches
    else:
        unit, peak, nominal, work = "GB/s", hbm, NOMINAL_HBM_GBS, b_d / 1e9 / dom_launches
    achieved = work / (dom_ms * 1e-3)
    total_ms = sum(v[0] * v[1] for v in with_work.values())
    src = ("bf16_tflops" if dom_tensor else "hbm_gbs")
    return {"bound": "tensor" if dom_tensor else "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": profiled_traffic(lay.name),
            "kernel": kernel_names(lay)[dom], "kernel_ms": round(dom_ms, 5),
            "kernel_share": round(dom_ms * dom_launches / total_ms, 4) if total_ms > 0 else None,
            "work_per_launch": work * (1e12 if dom_tensor else 1e9),
            "peak_source": (f"measured (MEASURED_PEAKS.json {src})" if peak_kind == "measured" else
                            ("fallback 1.9 PFLOP/s" if dom_tensor else "fallback 6.8 TB/s")),
            "peak_nominal": nominal, "frac_nominal": round(achieved / nominal, 4),
            "timed": "CUDA events around each launch of the kernel, on its stream"}


def measure(binding, lay, steps, warmup, dist, world):
    """Whole-call device time of one workload (inputs resident in HBM, L2 flushed before every
    call when the K/V pools fit in it), its value in the workload's unit, and its roofline."""
    import torch
    g = workloads_mod().materialize(lay, device="cuda")
    flops, nbytes = algorithmic(lay)
    hbm, bf16, _, _ = peaks()
    flush = L2Flush(pool_bytes(lay))
    ms, launches = time_device(binding, g, lay, steps, warmup, dist, flush)
    ms = max_over_ranks(ms, dist, "cuda")
    tensor_bound = flops / nbytes > (bf16 * 1e12) / (hbm * 1e9)
    unit, work = ("TFLOP/s", flops / 1e12) if tensor_bound else ("GB/s", nbytes / 1e9)
    value = replica_throughput(work, world, ms)
    roof = roofline_of(binding, g, lay, max(3, min(steps, 20)), flush)
    out = {"g": g, "flops": flops, "nbytes": nbytes, "ms": ms, "launches": launches, "unit": unit,
           "value": value, "roofline": roof, "flush": flush}
    torch.cuda.synchronize()
    return out


def workloads_mod():
    from paged_kv_varlen_flashattention_gb300 import workloads
    return workloads


def run_ours(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    else:
        torch.cuda.set_device(0)
    from paged_kv_varlen_flashattention_gb300 import binding, workloads

    lay = workloads.CONFIGS[args.workload]()
    lay.nan_fill = False
    set_alibi(args, lay)
    _, bf16, _, _ = peaks()

    if args.profile:
        args.no_e2e = args.no_secondary = args.no_cpu_baseline = args.no_workloads = True
    sampler = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    sampler.start()
    # a sustained run of the same step while the clock sampler warms up
    g0 = workloads.materialize(lay, device="cuda")
    out = torch.empty_like(g0.q)
    lse = torch.empty((lay.num_heads, lay.total_q), dtype=torch.float32, device="cuda")
    t_end = time.time() + (0.0 if args.profile else 1.0)
    while time.time() < t_end:
        for _ in range(20):
            _call(binding, g0, lay, out, lse)
        torch.cuda.synchronize()
    del g0, out, lse
    m = measure(binding, lay, args.steps, args.warmup, dist, world)
    clocks = sampler.stop()
    g, flops, nbytes = m["g"], m["flops"], m["nbytes"]

    result = {
        "metric": METRIC, "value": round(m["value"], 2), "unit": m["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(m["ms"], 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if lay.dtype == "bf16" else "f16", "data": "synthetic",
        "config": workload_config(lay, flops, nbytes, world),
        "roofline": m["roofline"],
        "gpu_launches": int(m["launches"]),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_e2e:
        ms_e2e, h2d, d2h = time_e2e(binding, g, lay, max(3, min(args.steps, 10)), 2)
        result["e2e"] = {"value": round(nbytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                         "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                         "ms_per_step": round(ms_e2e, 4)}
    if rank == 0 and not args.no_cpu_baseline:
        inp_cpu = g.to("cpu")
        val, cunit, secs, cores, sample = cpu_baseline(lay, inp_cpu, budget_s=args.cpu_budget)
        result["cpu_baseline"] = {"value": round(val, 4), "unit": cunit, "cores": cores, "cpu_model": cpu_model(),
                                  "kind": "oracle", "sample": sample}
        del inp_cpu
    del g, m
    if rank == 0 and not args.no_secondary and lay.name != "prefill_bf16":
        try:
            lay2 = workloads.CONFIGS["prefill_bf16"]()
            lay2.nan_fill = False
            set_alibi(args, lay2)
            m2 = measure(binding, lay2, 3, 3, None, 1)
            roof = m2["roofline"]
            result["secondary"] = {"workload": lay2.name, "value": round(m2["flops"] / (m2["ms"] * 1e-3) / 1e12, 2),
                                   "unit": "TFLOP/s", "ms_per_step": round(m2["ms"], 4),
                                   "algorithmic_flops": m2["flops"], "roofline": roof,
                                   "l2": l2_label(pool_bytes(lay2)), "gpu_launches": int(m2["launches"])}
            del m2
        except Exception as e:  # reported, not hidden
            result["secondary"] = {"error": str(e)[:300]}
        set_alibi(args, lay)
    if rank == 0 and not args.no_workloads:
        result["workloads"] = {}
        for name in EXTRA_WORKLOADS:
            if name == lay.name:
                continue
            try:
                lw = workloads.CONFIGS[name]()
                lw.nan_fill = False
                set_alibi(args, lw)
                mw = measure(binding, lw, 10, 3, None, 1)
                result["workloads"][name] = {
                    "value": round(mw["value"], 2), "unit": mw["unit"], "ms_per_step": round(mw["ms"], 5),
                    "algorithmic_bytes": mw["nbytes"], "algorithmic_flops": mw["flops"],
                    "roofline": mw["roofline"], "l2": l2_label(pool_bytes(lw)), "gpu_launches": int(mw["launches"])}
                del mw
            except Exception as e:  # reported, not hidden
                result["workloads"][name] = {"error": str(e)[:300]}
        set_alibi(args, lay)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_append(args):
    """--op append: pa_kv_append of each sequence's query tokens (the new tokens of a serving
    step: whole prompts for prefill, one token per sequence for decode) into a pool laid out
    like the workload's, timed on the device; GB/s of K and V read plus written."""
    import torch
    from paged_kv_varlen_flashattention_gb300 import binding, workloads
    torch.cuda.set_device(0)
    lay = workloads.CONFIGS[args.workload]()
    lay.nan_fill = False
    g = workloads.materialize(lay, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(17)
    shape = (lay.total_q, lay.num_heads_k, lay.head_dim)
    kn = torch.randn(shape, generator=gen, device="cuda").to(g.k_cache.dtype)
    vn = torch.randn(shape, generator=gen, device="cuda").to(g.k_cache.dtype)
    elt = 2
    nbytes = 2 * 2 * lay.total_q * lay.num_heads_k * lay.head_dim * elt

    def step():
        binding.kv_append(kn, vn, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table, g.k_cache, g.v_cache)

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert binding.device_status() == 0, binding.last_error()
    flush = L2Flush(nbytes)  # the bytes an append step touches (new rows in, their slots out)
    n0 = binding.kernel_launches()
    ms = timed_calls(step, args.steps, flush)
    clocks = sampler.stop()
    launches = binding.kernel_launches() - n0
    binding.kernel_times()
    binding.kernel_timing(True)
    for _ in range(max(3, min(args.steps, 20))):
        flush()
        step()
    torch.cuda.synchronize()
    binding.kernel_timing(False)
    k_ms, k_n = binding.kernel_times()["append"]
    hbm, _, _, peak_kind = peaks()
    value = nbytes / (ms * 1e-3) / 1e9
    achieved = nbytes / (k_ms / k_n * 1e-3) / 1e9
    cfg = workload_config(lay, 0, nbytes, 1)
    cfg.update({"op": "kv_append", "new_tokens": lay.total_q,
                "l2": l2_label(nbytes, "bytes moved")})
    print(json.dumps({
        "metric": "KV append GB/s (K and V read + written), % of GB300 HBM roofline", "value": round(value, 2),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if lay.dtype == "bf16" else "f16", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None, "kernel": "kv_append_kernel",
                     "kernel_ms": round(k_ms / k_n, 5), "work_per_launch": nbytes,
                     "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "timed": "CUDA events around each launch of the kernel, on its stream"},
        "gpu_launches": int(launches), "clocks": clocks,
    }), flush=True)


def run_padded(args):
    """--op padded: pa_fwd_padded on a padded causal batch of 8 x 4096 tokens (H=32, Hkv=8,
    D=128, bf16; the prefill shape at a uniform length), timed on the device; TFLOP/s."""
    import torch
    from paged_kv_varlen_flashattention_gb300 import binding
    torch.cuda.set_device(0)
    B, S, H, Hkv, D = 8, 4096, 32, 8, 128
    g = torch.Generator(device="cuda").manual_seed(19)
    q = torch.randn((B, S, H, D), generator=g, device="cuda").bfloat16()
    k = torch.randn((B, S, Hkv, D), generator=g, device="cuda").bfloat16()
    v = torch.randn((B, S, Hkv, D), generator=g, device="cuda").bfloat16()
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    sl = torch.from_numpy(alibi_slopes(H)).cuda() if args.alibi else None
    flops = 4 * D * H * B * (S * (S + 1) // 2)
    nbytes = 2 * B * S * Hkv * D * 2 + 2 * B * S * H * D * 2 + 4 * B * H * S

    def step():
        binding.fwd_padded(q, k, v, 1.0 / D ** 0.5, -1, 0, alibi_slopes=sl, out=out, softmax_lse=lse)

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert binding.device_status() == 0, binding.last_error()
    kv_bytes = 2 * B * S * Hkv * D * 2
    flush = L2Flush(kv_bytes)
    n0 = binding.kernel_launches()
    ms = timed_calls(step, args.steps, flush)
    clocks = sampler.stop()
    launches = binding.kernel_launches() - n0
    binding.kernel_times()
    binding.kernel_timing(True)
    for _ in range(max(3, min(args.steps, 10))):
        flush()
        step()
    torch.cuda.synchronize()
    binding.kernel_timing(False)
    k_ms, k_n = binding.kernel_times()["prefill"]
    _, bf16, _, peak_kind = peaks()
    value = flops / (ms * 1e-3) / 1e12
    achieved = flops / (k_ms / k_n * 1e-3) / 1e12
    print(json.dumps({
        "metric": "paged-attn TFLOP/s (prefill) and KV GB/s (decode), % of GB300 roofline", "value": round(value, 2),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "padded_causal_bf16", "op": "fwd_padded", "batch": B, "seqlen": S, "num_heads": H,
                   "num_heads_k": Hkv, "head_dim": D, "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
                   "l2": l2_label(kv_bytes), "parallelism": "replicas1",
                   **({"alibi_slopes": "2^(-8 (h + 1) / H)"} if args.alibi else {})},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16, "unit": "TFLOP/s",
                     "frac": round(achieved / bf16, 4), "traffic": None, "kernel": "prefill_kernel",
                     "kernel_ms": round(k_ms / k_n, 5), "work_per_launch": flops,
                     "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops)" if peak_kind == "measured"
                     else "fallback 1.9 PFLOP/s",
                     "timed": "CUDA events around each launch of the kernel, on its stream"},
        "gpu_launches": int(launches), "clocks": clocks,
    }), flush=True)


def run_reference(args):
    """The oracle on the host cores, timed per step over a bounded sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from paged_kv_varlen_flashattention_gb300 import workloads

    lay = workloads.CONFIGS[args.workload]()
    lay.nan_fill = False
    set_alibi(args, lay)
    inp = workloads.materialize(lay, device="cpu")
    cq, _ = lay.cu_seqlens()
    bt = inp.block_table.numpy() if inp.block_table is not None else None
    rng = np.random.default_rng(1)
    n_seq = max(1, min(lay.batch, args.ref_sequences))
    seqs = sorted(rng.choice(lay.batch, size=n_seq, replace=False).tolist())
    rows = np.concatenate([np.arange(cq[b] * lay.num_heads, cq[b + 1] * lay.num_heads) for b in seqs]).astype(np.int64)
    flops_all, bytes_all = algorithmic(lay)
    unit, _ = headline_unit(flops_all, bytes_all)
    f_s, b_s = algorithmic(lay, seqs)
    work = f_s / 1e12 if unit == "TFLOP/s" else b_s / 1e9

    def step():
        oracle.attention(lay.dtype, inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q.numpy(),
                         inp.cu_seqlens_k.numpy(), bt, lay.softmax_scale, lay.window_left, lay.window_right,
                         rows=rows, alibi_slopes=ALIBI["slopes"])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = (time.perf_counter() - t0) / args.steps
    value = work / secs
    sample = f"{n_seq} of {lay.batch} sequences (all heads) per step, seeded choice"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(lay, flops_all, bytes_all, world),
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": oracle.threads(), "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_bf16")
    ap.add_argument("--op", choices=["attention", "append", "padded"], default="attention",
                    help="attention: the forward call (default); append: pa_kv_append of the step's tokens; "
                         "padded: pa_fwd_padded on an 8 x 4096 causal batch")
    ap.add_argument("--alibi", action="store_true",
                    help="run every leg with the linear position bias (geometric per-head slopes)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the mixed / long-context workloads measured beside the headline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-sequences", type=int, default=16)
    ap.add_argument("--profile", action="store_true",
                    help="only warm-up + timed steps (no clock warm-up loop, e2e, secondary or CPU legs): "
                         "the command the ncu summaries are taken with")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "append":
        run_append(args)
    elif args.op == "padded":
        run_padded(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
