#!/usr/bin/env python3
"""Benchmark of the MLA paged latent-cache decode step on B300.

One step = one mla_decode_paged call (split-KV attention pass + log-sum-exp
combine) over the whole batch of the V2-shaped decode workload: 32
sequences x 4096 cached tokens, 128 heads, rows of 512 latent + 64 rotary
bfloat16 numbers in 64-token blocks with a shuffled block table, latent
queries [32, 1, 128, 576].  Inputs are seeded synthetic normal draws.

Prints ONE JSON line (rank 0).  `value` is the algorithmic cache+query bytes
of all ranks' steps divided by the device time of the timed steps (max over
ranks), in GB/s.  Other keys: TFLOP/s, tokens/s, the roofline of the
dominant kernel, an end-to-end figure through the public API with host
buffers, the oracle timed on the host cores, and the SM clocks sampled
during the timed region.

With --workload prefill_b1_t4096_h128 a step is instead one prefill of a
4096-token prompt over keys and values rebuilt from the latent cache
(mla_prefill_kv + mla_prefill_attention, 128 heads), and `value` is its
algorithmic TFLOP/s against the tensor-core roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mla|reference]
                  [--workload NAME]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import shutil
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_inputs as mi  # noqa: E402

METRIC = "MLA decode cache GB/s + TFLOP/s, % of B300 roofline; decode tokens/sec"
L2_BYTES = 126 * 1024 * 1024
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")


# --------------------------------------------------------------------------
# workload arithmetic (algorithmic work, no padding / split / tail waste)
# --------------------------------------------------------------------------

def algorithmic_work(spec: mi.DecodeSpec, seqlens: np.ndarray):
    """Bytes the method must read (every visible cache row once + the latent
    queries) and FLOPs it must do (576-wide score and 512-wide value sum per
    (query row, visible key))."""
    D, elt = spec.D, 2
    L = seqlens.astype(np.int64)
    cache_bytes = int(L.sum()) * D * elt
    q_bytes = spec.B * spec.T_q * spec.H * D * elt
    if spec.causal:
        vis = sum(int(l) - spec.T_q + t + 1 for l in L for t in range(spec.T_q))
    else:
        vis = int(L.sum()) * spec.T_q
    flops = 2 * spec.H * vis * (D + spec.d_c)
    out_bytes = spec.B * spec.T_q * spec.H * (spec.d_c + 1) * 4
    return dict(cache_bytes=cache_bytes, q_bytes=q_bytes, bytes=cache_bytes + q_bytes,
                flops=flops, out_bytes=out_bytes)


def pipelined_e2e(torch, dev, stream, steps, load, compute, store):
    """End-to-end steps through the public API, as a server would run them:
    step i's inputs are copied in from pinned host memory on one stream, step i
    runs on `stream`, and its results are copied back on a third stream.  Two
    device buffer sets (k = i mod 2) let the copies of steps i + 1 and i - 1
    overlap step i.  Every step's copies are inside the timed region.  Returns
    the milliseconds from the first copy in to the last copy out."""
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        k = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_c[k])        # step i - 2 has read buffer set k
            load(k)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if i >= 2:
            stream.wait_event(ev_out[k])        # step i - 2's results are copied out
        compute(i, k)
        ev_c[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[k])
            store(k)
            ev_out[k].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(3, 3 + steps):
        step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in PEAKS_FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def kernel_source_sha(name: str) -> str:
    path = os.path.join(ROOT, "head_latent_attention_28_b300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def profiled_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the kernel source as it is now (else None)."""
    path = os.path.join(PROFILE_DIR, f"{os.path.splitext(kernel_file)[0]}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_tr) or m_sha.group(1) != kernel_source_sha(kernel_file):
        return None
    return float(m_tr.group(1))


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    """Samples the SM clock and the clock-event reasons of one GPU in the
    background (NVML if importable, else `nvidia-smi -lms`), timestamping
    every sample on the host clock.  `mark(start|end)` brackets the timed
    region; the summary keeps the samples inside it (the nearest ones when the
    region is shorter than the sampling period, flagged as such)."""
    REASONS = {  # NVML clocks-event reason bits
        0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
        0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
        0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    SMI_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.dev, self.period = device_index, period_s
        self.samples = []          # (host time, sm MHz, set of reasons)
        self.max_mhz, self.err = None, None
        self.t_start = self.t_end = None
        self._stop = threading.Event()
        self.mode = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:  # noqa: BLE001
            self.err = repr(e)
            if shutil.which("nvidia-smi"):
                self.mode = "nvidia-smi"

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                mhz = nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)
                bits = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                self.samples.append((time.monotonic(), float(mhz),
                                     {n for b, n in self.REASONS.items() if bits & b}))
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.period)

    def _read_smi(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                mhz, self.max_mhz = float(f[0]), float(f[1])
            except ValueError:
                continue
            self.samples.append((time.monotonic(), mhz,
                                 {n for n, v in zip(self.SMI_REASONS, f[4:8]) if v.lower() == "active"}))

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run_nvml, daemon=True)
            self.t.start()
        elif self.mode == "nvidia-smi":
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.SMI_FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(max(1, int(self.period * 1000)))],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read_smi, daemon=True)
            self.t.start()
        # the sampler is live before the timed region starts
        t0 = time.monotonic()
        while self.mode and not self.samples and time.monotonic() - t0 < 5.0:
            time.sleep(0.01)
        return self

    def mark(self, which: str):
        if which == "start":
            self.t_start = time.monotonic()
        else:
            self.t_end = time.monotonic()

    def __exit__(self, *a):
        time.sleep(2 * self.period)
        if self.mode == "nvml":
            self._stop.set()
            self.t.join()
        elif self.mode == "nvidia-smi":
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        if self.mode is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": self.err}
        inside = [x for x in self.samples
                  if self.t_start is not None and self.t_start <= x[0] <= (self.t_end or x[0])]
        where = "timed region"
        if not inside and self.samples and self.t_start is not None:
            mid = 0.5 * (self.t_start + (self.t_end or self.t_start))
            inside = sorted(self.samples, key=lambda x: abs(x[0] - mid))[:2]
            where = "nearest to the timed region (shorter than the sampling period)"
        reasons = set()
        for x in inside:
            reasons |= x[2]
        return {"sm_mhz": statistics.median(x[1] for x in inside) if inside else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(inside), "window": where, "source": self.mode}


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no data-path collective)
# --------------------------------------------------------------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("MLA_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, local, None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm)
# --------------------------------------------------------------------------

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 0) for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001
        pass
    return os.cpu_count() or 1


def time_oracle_sequences(inp, seqs):
    """Run the fp64 oracle on the given sequences; returns (seconds, bytes)."""
    import oracle as orc
    s = inp.spec
    t0 = time.perf_counter()
    orc.decode_paged_logical(inp.q_bits, inp.cache_bits, inp.offsets, s.d_c,
                             s.softmax_scale, s.causal, batch=seqs)
    dt = time.perf_counter() - t0
    nbytes = sum(int(inp.seqlens[b]) * s.D * 2 + s.T_q * s.H * s.D * 2 for b in seqs)
    return dt, nbytes


def cpu_baseline(inp, budget_s: float = 12.0):
    """The oracle as it stands on the host cores, on whole sequences of the
    workload, repeated until about budget_s seconds have passed."""
    done_s, done_b, n, b = 0.0, 0, 0, 0
    while done_s < budget_s:
        dt, nb = time_oracle_sequences(inp, [b % inp.spec.B])
        done_s += dt
        done_b += nb
        n += 1
        b += 1
    return {"value": done_b / done_s / 1e9, "unit": "GB/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"{n} whole sequences ({inp.spec.seqlen or 'mixed'} tokens x {inp.spec.H} "
                      f"heads each) of the {inp.spec.name} batch, fp64 numpy, {done_s:.1f} s"}


def run_reference(args, spec):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    inp = mi.make_decode_inputs(spec, build_pool=False)
    for i in range(args.warmup):
        time_oracle_sequences(inp, [i % spec.B])
    tot_s, tot_b = 0.0, 0
    for i in range(args.steps):
        dt, nb = time_oracle_sequences(inp, [(args.warmup + i) % spec.B])
        tot_s += dt
        tot_b += nb
    value = tot_b / tot_s / 1e9
    cores = blas_threads()
    sample = f"one whole sequence of the {spec.name} batch per step (1/{spec.B} of the batch)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(spec, "fp64 numpy oracle on host cores"),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(spec, l2_note):
    return {"workload": spec.name, "global_batch": spec.B, "seq_len": spec.seqlen,
            "heads": spec.H, "q_tokens": spec.T_q, "d_c": spec.d_c, "d_rope": spec.d_r,
            "page": mi.PAGE, "cache_dtype": "bf16", "softmax_scale": spec.softmax_scale,
            "l2": l2_note, "parallelism": "replicas"}


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

def device_time_ms(fn, K, stream, dev):
    """Mean device time of K back-to-back calls of fn(i), from one pair of
    CUDA events on the launching stream.  A sleep kernel queued first lets
    the host enqueue ahead, so host call overhead stays outside the window."""
    import torch
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(4_000_000)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / K


def host_enqueue_us(fn, K, dev):
    """Host-clock time of one call (argument checks, marshalling, launches),
    with the device busy so that no call waits for it: few enough calls that
    their launches fit the launch queue (a full queue makes the host wait for
    the device, which is not host work)."""
    import torch
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(40_000_000)
    t0 = time.perf_counter()
    for i in range(K):
        fn(i)
    dt = time.perf_counter() - t0
    torch.cuda.synchronize(dev)
    return 1e6 * dt / K


class DecodeBench:
    """One decode workload resident on the device: the cache (with enough
    copies to exceed L2, rotated between steps), queries, block table,
    lengths, workspace and outputs."""

    def __init__(self, spec, dev, rank=0):
        import torch
        import head_latent_attention_28_b300 as mla
        self.mla, self.dev = mla, dev
        self.spec = mi.DecodeSpec(**{**spec.__dict__, "seed": spec.seed + rank})
        self.inp = mi.make_decode_inputs(self.spec)
        self.work = algorithmic_work(self.spec, self.inp.seqlens)

        def up(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)
        self.q = up(self.inp.q_bits)
        pool0 = up(self.inp.pool_bits)
        self.n_copies = max(2, math.ceil(3 * L2_BYTES / (pool0.numel() * 2)))
        self.pools = [pool0] + [pool0.clone() for _ in range(self.n_copies - 1)]
        self.pool_mb = self.n_copies * pool0.numel() * 2 / 1e6
        self.bt = torch.from_numpy(self.inp.block_table).to(dev)
        self.sl = torch.from_numpy(self.inp.seqlens).to(dev)
        B, T_q, H, D = self.q.shape
        s = self.spec
        self.ws = mla.alloc_workspace(B, T_q, H, s.d_c, s.d_r, torch.bfloat16, dev)
        self.o = torch.empty((B, T_q, H, s.d_c), device=dev, dtype=torch.float32)
        self.lse = torch.empty((B, T_q, H), device=dev, dtype=torch.float32)
        self.stream = torch.cuda.current_stream(dev)
        self.kw = dict(d_c=s.d_c, softmax_scale=s.softmax_scale, causal=s.causal,
                       workspace=self.ws, o_lat=self.o, lse=self.lse, stream=self.stream)
        self.tc = mla.lib().mla_decode_path(T_q, H, s.d_c, s.d_r, mla.MLA_BF16) == 1
        self.kernel_file = "decode_tc.cu" if self.tc else "decode_generic.cu"
        self.workers = mla.lib().mla_decode_num_workers(B, T_q, H, s.d_c, s.d_r, mla.MLA_BF16)

    def step(self, i, stage="both"):
        self.mla.mla_decode_paged(self.q, self.pools[i % self.n_copies], self.bt, self.sl,
                                  stage=stage, **self.kw)

    def check(self, what):
        st = self.mla.mla_check_status(self.stream)
        if st != self.mla.MLA_OK:
            raise SystemExit(f"{self.spec.name}: {what}: {self.mla.mla_status_string(st)}")

    def kernel_times(self, K):
        """(decode kernel ms, merge kernel ms, host enqueue us per call), each
        from back-to-back launches of that kernel alone."""
        main_ms = device_time_ms(lambda i: self.step(i, "partial"), K, self.stream, self.dev)
        comb_ms = device_time_ms(lambda i: self.step(i, "combine"), K, self.stream, self.dev)
        host_us = host_enqueue_us(self.step, min(K, 40), self.dev)
        self.check("kernel timing")
        return main_ms, comb_ms, host_us

    def roofline(self, step_ms, main_ms, comb_ms, peaks, peak_src):
        w = self.work
        t_mem = w["bytes"] / (peaks["hbm_gbs"] * 1e9)
        t_tc = w["flops"] / (peaks["bf16_tflops"] * 1e12)
        hbm = t_mem >= t_tc
        achieved = (w["bytes"] / (main_ms / 1e3) / 1e9) if hbm else (w["flops"] / (main_ms / 1e3) / 1e12)
        peak = peaks["hbm_gbs"] if hbm else peaks["bf16_tflops"]
        return {"bound": "hbm" if hbm else "tensor", "achieved": achieved, "peak": peak,
                "unit": "GB/s" if hbm else "TFLOP/s", "frac": achieved / peak,
                "traffic": profiled_traffic(self.kernel_file, self.spec.name),
                "kernel": self.kernel_file, "kernel_ms": main_ms, "combine_ms": comb_ms,
                "split_workers": self.workers,
                "peak_source": peak_src + " (burst; kernel timed alone)",
                "achieved_tflops": w["flops"] / (main_ms / 1e3) / 1e12,
                "tensor_peak_tflops": peaks["bf16_tflops"],
                "roofline_us": 1e6 * max(t_mem, t_tc),
                "step_frac_of_roofline": max(t_mem, t_tc) / (step_ms / 1e3),
                "kernel_time": "one event pair around back-to-back launches of the kernel alone, "
                               "divided by their number"}


def decode_subrecord(spec, dev, args, peaks, peak_src):
    """Step, kernel, roofline and oracle figures of one more decode workload
    (rank 0, one GPU)."""
    db = DecodeBench(spec, dev)
    K = max(args.steps, 20)
    for i in range(args.warmup):
        db.step(i)
    db.check("warm-up")
    step_ms = device_time_ms(db.step, K, db.stream, dev)
    db.check("timed steps")
    main_ms, comb_ms, host_us = db.kernel_times(K)
    rf = db.roofline(step_ms, main_ms, comb_ms, peaks, peak_src)
    w = db.work
    rec = {"step_us": 1e3 * step_ms, "kernel_us": 1e3 * main_ms, "combine_us": 1e3 * comb_ms,
           "host_enqueue_us": host_us, "steps": K,
           "value": w["bytes"] / (step_ms / 1e3) / 1e9, "unit": "GB/s",
           "tflops": w["flops"] / (step_ms / 1e3) / 1e12,
           "tokens_per_s": spec.B * spec.T_q / (step_ms / 1e3),
           "roofline": rf, "config": workload_config(db.spec, f"{db.n_copies} cache copies "
                                                             f"({db.pool_mb:.0f} MB) rotated")}
    # the kernel timed alone can come out a fraction of a percent above the
    # step (kernel + merge) on single-item workloads: timing noise, not a fault
    if main_ms > step_ms * 1.03:
        raise SystemExit(f"{spec.name}: kernel time {main_ms} ms exceeds the step time {step_ms} ms")
    if not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(db.inp, args.cpu_budget / 2)
    del db
    import torch
    torch.cuda.empty_cache()
    return rec


def run_mla(args, spec):
    import torch
    rank, world, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    import head_latent_attention_28_b300 as mla
    dev = torch.device("cuda", local)

    # rank r draws its own batch (same shapes, seed + r)
    db = DecodeBench(spec, dev, rank)
    work, stream = db.work, db.stream
    for i in range(args.warmup):
        db.step(i)
    db.check("warm-up")

    # ---- timed region: K whole steps, back to back on one stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(dist, local)
    torch.cuda.synchronize(dev)
    with sampler:
        torch.cuda._sleep(4_000_000)   # the host enqueues ahead; the window starts at ev0
        sampler.mark("start")
        ev0.record(stream)
        for i in range(args.steps):
            db.step(i)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        sampler.mark("end")
    barrier(dist, local)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(dist, ms)
    db.check("timed region")

    # ---- the dominant kernel and the merge, each timed alone
    main_ms, comb_ms, host_us = db.kernel_times(max(args.steps, 20))
    step_ms = ms / args.steps
    if main_ms > step_ms * 1.03:
        raise SystemExit(f"kernel time {main_ms:.4f} ms exceeds the step time {step_ms:.4f} ms")

    # ---- end to end through the public API with pinned host buffers
    q, bt, sl, o, lse = db.q, db.bt, db.sl, db.o, db.lse
    q_h = q.cpu().pin_memory()
    bt_h = bt.cpu().pin_memory()
    sl_h = sl.cpu().pin_memory()
    o_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    lse_h = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    q_d = [torch.empty_like(q) for _ in range(2)]
    bt_d = [torch.empty_like(bt) for _ in range(2)]
    sl_d = [torch.empty_like(sl) for _ in range(2)]
    o_d, lse_d = [o, torch.empty_like(o)], [lse, torch.empty_like(lse)]
    h2d = q_h.numel() * 2 + bt_h.numel() * 4 + sl_h.numel() * 4
    d2h = o.numel() * 4 + lse.numel() * 4

    def e2e_load(k):
        q_d[k].copy_(q_h, non_blocking=True)
        bt_d[k].copy_(bt_h, non_blocking=True)
        sl_d[k].copy_(sl_h, non_blocking=True)

    def e2e_compute(i, k):
        mla.mla_decode_paged(q_d[k], db.pools[i % db.n_copies], bt_d[k], sl_d[k], d_c=spec.d_c,
                             softmax_scale=spec.softmax_scale, causal=spec.causal,
                             workspace=db.ws, o_lat=o_d[k], lse=lse_d[k], stream=stream)

    def e2e_store(k):
        o_h[k].copy_(o_d[k], non_blocking=True)
        lse_h[k].copy_(lse_d[k], non_blocking=True)

    barrier(dist, local)
    e2e_ms = max_over_ranks(dist, pipelined_e2e(torch, dev, stream, args.steps, e2e_load, e2e_compute,
                                                e2e_store))
    db.check("end-to-end steps")

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    total_bytes = work["bytes"] * world * args.steps
    value = total_bytes / (ms_max / 1e3) / 1e9
    tflops = work["flops"] * world * args.steps / (ms_max / 1e3) / 1e12
    roofline = db.roofline(ms_max / args.steps, main_ms, comb_ms, peaks, peak_src)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal draws, shuffled block table)",
        "config": workload_config(db.spec, f"inputs larger than L2: {db.n_copies} cache copies "
                                           f"({db.pool_mb:.0f} MB) rotated"),
        "tflops": tflops, "tokens_per_s": spec.B * spec.T_q * world * args.steps / (ms_max / 1e3),
        "roofline": roofline,
        "host_enqueue_us": host_us,
        "e2e": {"value": total_bytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps,
                "note": "per step: latent queries, block table and lengths copied in from "
                        "pinned host memory, o_lat and lse copied back; the cache is resident; "
                        "copies in, decode and copies out on three streams, neighbouring "
                        "steps overlapping (two device buffer sets)"},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(db.inp, args.cpu_budget)
    del db, q_d, bt_d, sl_d
    torch.cuda.empty_cache()
    if world == 1 and not args.no_extra:
        # the other workloads of the scope table, from the same run
        extra = {}
        for name in sorted(mi.DECODE_WORKLOADS):
            if name != spec.name:
                extra[name] = decode_subrecord(mi.DECODE_WORKLOADS[name], dev, args, peaks, peak_src)
        for name, pspec in sorted(mi.PREFILL_WORKLOADS.items()):
            extra[name] = prefill_subrecord(pspec, dev, args, peaks, peak_src)
        for name, ospec in sorted(mi.OUT_PROJ_WORKLOADS.items()):
            extra[name] = out_proj_subrecord(ospec, dev, args, peaks, peak_src)
        line["configs"] = extra
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------------
# output projections: W^UV then W^O, or the two merged into one matrix
# --------------------------------------------------------------------------

def out_proj_subrecord(spec, dev, args, peaks, peak_src):
    """Both forms of the output projection at decode size, each timed alone
    (back-to-back calls); HBM-bound at this N, so each gets the HBM roofline
    over its own algorithmic bytes (its weights, o_lat in, out back)."""
    import torch
    import head_latent_attention_28_b300 as mla
    inp = mi.make_out_proj_inputs(spec)
    N, H, d_h, d_c, d = spec.N, spec.H, spec.d_h, spec.d_c, spec.d

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)
    w_uv, w_o = up(inp.w_uv_bits), up(inp.w_o_bits)
    o_lat = torch.from_numpy(inp.o_lat).to(dev)
    out = torch.empty((N, d), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    w_m = mla.mla_merge_output_weights(w_uv, w_o, H)
    torch.cuda.synchronize(dev)
    merge_ms = 1e3 * (time.perf_counter() - t0)
    ws = torch.empty(mla.mla_absorb_output_merged_workspace_size(N, H, d_c, d), device=dev, dtype=torch.uint8)

    def unmerged(i):
        mla.mla_absorb_output(o_lat, w_uv, w_o, out=out, stream=stream)

    def merged(i):
        mla.mla_absorb_output_merged(o_lat, w_m, workspace=ws, out=out, stream=stream)
    for _ in range(args.warmup):
        unmerged(0)
        merged(0)
    K = max(min(args.steps, 50), 10)
    un_ms = device_time_ms(unmerged, K, stream, dev)
    mg_ms = device_time_ms(merged, K, stream, dev)
    if mla.mla_check_status(stream) != mla.MLA_OK:
        raise SystemExit("out_proj: device error")
    act = N * H * d_c * 4 + N * d * 4
    b_un = (H * d_h * d_c + d * H * d_h) * 2 + act
    b_mg = d * H * d_c * 2 + act

    def roof(bytes_, ms, kernel):
        gbs = bytes_ / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": kernel, "kernel_ms": ms,
                "algorithmic_bytes": bytes_, "peak_source": peak_src + " (burst; calls timed alone)",
                "kernel_time": "one event pair around back-to-back calls, divided by their number"}
    rec = {"unmerged_us": 1e3 * un_ms, "merged_us": 1e3 * mg_ms, "merge_weights_ms": merge_ms, "steps": K,
           "value": b_un / (un_ms / 1e3) / 1e9, "unit": "GB/s",
           "adopted": "unmerged (mla_absorb_output): it reads H*d_h*(d_c + d) weights against d*H*d_c merged",
           "roofline": roof(b_un, un_ms, "out_proj_tc.cu (gemm_tn_kernel, unmerged: per-head W^UV, split-K W^O)"),
           "merged": {"value": b_mg / (mg_ms / 1e3) / 1e9, "unit": "GB/s",
                      "roofline": roof(b_mg, mg_ms, "out_proj_tc.cu (gemm_tn_kernel, split-K merged weights)")},
           "config": {"workload": spec.name, "rows": N, "heads": H, "d_h": d_h, "d_c": d_c, "d": d,
                      "weight_dtype": "bf16", "l2": "the weights of each call exceed L2",
                      "parallelism": "replicas"}}
    if not args.no_cpu_baseline:
        import oracle as orc
        w_uv64 = mi.bf16_bits_to_f32(inp.w_uv_bits).reshape(inp.w_uv_bits.shape)
        w_o64 = mi.bf16_bits_to_f32(inp.w_o_bits).reshape(inp.w_o_bits.shape)
        t0, n = time.perf_counter(), 0
        while n < N and (n == 0 or time.perf_counter() - t0 < args.cpu_budget / 4):
            orc.absorb_output(inp.o_lat[n:n + 1], w_uv64, w_o64)
            n += 1
        sec = time.perf_counter() - t0
        # the whole batch at the sample's rate: N rows take N / n times as long
        rec["cpu_baseline"] = {"value": b_un / (sec * N / n) / 1e9, "unit": "GB/s",
                               "cores": blas_threads(), "kind": "oracle",
                               "sample": f"fp64 numpy absorb_output of {n} of the {N} rows, {sec:.1f} s, "
                                         f"scaled to the batch"}
    del w_uv, w_o, w_m, ws, o_lat, out
    torch.cuda.empty_cache()
    return rec


# --------------------------------------------------------------------------
# prefill over rebuilt per-head keys and values
# --------------------------------------------------------------------------

PREFILL_METRIC = "MLA prefill TFLOP/s (rebuild of per-head K/V + causal attention), % of B300 bf16 peak"


def prefill_work(spec: mi.PrefillSpec, seqlens: np.ndarray):
    """FLOPs the method must do: the rebuild of k = W^UK_h c and v = W^UV_h c
    for every cached row and head (2 products of d_c x d_h), and per (query,
    visible key, head) a (d_h + d_r)-wide score and a d_h-wide value sum."""
    L = seqlens.astype(np.int64)
    rebuild = int(L.sum()) * spec.H * 2 * (2 * spec.d_c * spec.d_h)
    vis = sum(int(l) - spec.T_q + t + 1 for l in L for t in range(spec.T_q))
    attn = 2 * spec.H * vis * (spec.d_h + spec.d_r + spec.d_h)
    return dict(rebuild_flops=rebuild, attn_flops=attn, flops=rebuild + attn)


def prefill_config(spec, note):
    return {"workload": spec.name, "global_batch": spec.B, "seq_len": spec.seqlen,
            "heads": spec.H, "q_tokens": spec.T_q, "d_c": spec.d_c, "d_h": spec.d_h,
            "d_rope": spec.d_r, "page": mi.PAGE, "cache_dtype": "bf16",
            "softmax_scale": spec.softmax_scale, "l2": note, "parallelism": "replicas"}


def time_prefill_oracle(inp, queries):
    """The fp64 oracle on the rebuild of the whole prompt and the attention of
    the given query tokens of sequence 0; returns (seconds, flops)."""
    import oracle as orc
    s, c = inp.spec, inp.cache
    f64 = lambda b: mi.bf16_bits_to_f32(b).reshape(b.shape).astype(np.float64)  # noqa: E731
    L = int(c.seqlens[0])
    pos = np.arange(L - s.T_q, L)[queries]
    t0 = time.perf_counter()
    k, v, kr = orc.rebuild_kv(f64(c.seq_rows(0)), s.H, f64(inp.w_uk_bits), f64(inp.w_uv_bits), s.d_c)
    orc.prefill_attention(f64(inp.q_nope_bits[0, queries]), f64(inp.q_rope_bits[0, queries]), pos,
                          k, v, kr, s.softmax_scale, s.rope_base)
    dt = time.perf_counter() - t0
    flops = L * s.H * 4 * s.d_c * s.d_h + 2 * s.H * int((pos + 1).sum()) * (2 * s.d_h + s.d_r)
    return dt, flops


def prefill_cpu_sample(inp, budget_s):
    rng = np.random.default_rng(0)
    done_s, done_f, nq = 0.0, 0, 0
    while done_s < budget_s:
        qs = rng.integers(0, inp.spec.T_q, 64)
        dt, fl = time_prefill_oracle(inp, qs)
        done_s += dt
        done_f += fl
        nq += len(qs)
    return done_s, done_f, nq


def run_prefill_reference(args, spec):
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    inp = mi.make_prefill_inputs(spec)
    for _ in range(args.warmup):
        time_prefill_oracle(inp, np.arange(4))
    tot_s, tot_f = 0.0, 0
    rng = np.random.default_rng(1)
    for _ in range(args.steps):
        dt, fl = time_prefill_oracle(inp, rng.integers(0, spec.T_q, 16))
        tot_s += dt
        tot_f += fl
    value = tot_f / tot_s / 1e12
    sample = (f"per step: the rebuild of all {spec.seqlen} rows x {spec.H} heads and the "
              f"attention of 16 random query tokens of the prompt")
    line = {"impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": prefill_config(spec, "fp64 numpy oracle on host cores"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class PrefillBench:
    """One prefill workload resident on the device: cache, queries, weights,
    rebuilt K/V buffers and outputs."""

    def __init__(self, spec, dev, rank=0):
        import torch
        import head_latent_attention_28_b300 as mla
        self.mla, self.dev = mla, dev
        self.spec = mi.PrefillSpec(**{**spec.__dict__, "seed": spec.seed + rank})
        self.inp = inp = mi.make_prefill_inputs(self.spec)
        self.work = prefill_work(self.spec, inp.cache.seqlens)

        def up(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)
        self.pool, self.qn, self.qr = up(inp.cache.pool_bits), up(inp.q_nope_bits), up(inp.q_rope_bits)
        self.wuk, self.wuv = up(inp.w_uk_bits), up(inp.w_uv_bits)
        self.bt = torch.from_numpy(inp.cache.block_table).to(dev)
        self.sl = torch.from_numpy(inp.cache.seqlens).to(dev)
        self.mb = inp.cache.max_blocks
        R = mla.mla_prefill_kv_rows(self.mb)
        B, T_q, H, d_h = self.qn.shape
        self.H = H
        self.kv = (torch.empty((B, H, R, d_h), device=dev, dtype=torch.bfloat16),
                   torch.empty((B, H, R, d_h), device=dev, dtype=torch.bfloat16),
                   torch.empty((B, R, spec.d_r), device=dev, dtype=torch.bfloat16))
        self.o = torch.empty((B, T_q, H, d_h), device=dev, dtype=torch.float32)
        self.lse = torch.empty((B, T_q, H), device=dev, dtype=torch.float32)
        self.stream = torch.cuda.current_stream(dev)

    def rebuild(self, i=0, sl=None):
        self.mla.mla_prefill_kv(self.pool, self.bt, self.sl if sl is None else sl, self.wuk, self.wuv,
                                H=self.H, out=self.kv, stream=self.stream)

    def attend(self, i=0, q_nope=None, q_rope=None, sl=None, o=None, lse=None):
        s = self.spec
        self.mla.mla_prefill_attention(self.qn if q_nope is None else q_nope,
                                       self.qr if q_rope is None else q_rope, *self.kv,
                                       self.sl if sl is None else sl, max_blocks_per_seq=self.mb,
                                       softmax_scale=s.softmax_scale, rope_base=s.rope_base,
                                       o=self.o if o is None else o, lse=self.lse if lse is None else lse,
                                       stream=self.stream)

    def step(self, i=0):
        self.rebuild()
        self.attend()

    def check(self, what):
        if self.mla.mla_check_status(self.stream) != self.mla.MLA_OK:
            raise SystemExit(f"prefill: {what}: device error")

    def kernel_times(self, K):
        kv_ms = device_time_ms(self.rebuild, K, self.stream, self.dev)
        at_ms = device_time_ms(self.attend, K, self.stream, self.dev)
        self.check("kernel timing")
        return kv_ms, at_ms

    def roofline(self, at_ms, kv_ms, step_ms, peaks, peak_src):
        w = self.work
        at_tflops = w["attn_flops"] / (at_ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": at_tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": at_tflops / peaks["bf16_tflops"],
                "traffic": profiled_traffic("prefill_tc.cu", self.spec.name),
                "kernel": "prefill_tc.cu (prefill_attn_kernel)", "kernel_ms": at_ms,
                "rebuild_ms": kv_ms,
                "rebuild_tflops": w["rebuild_flops"] / (kv_ms / 1e3) / 1e12,
                "peak_source": peak_src + " (burst; kernel timed alone)",
                "step_frac_of_peak": w["flops"] / (step_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                "kernel_time": "one event pair around back-to-back launches of the kernel alone, "
                               "divided by their number"}


def prefill_subrecord(spec, dev, args, peaks, peak_src):
    pb = PrefillBench(spec, dev)
    K = max(min(args.steps, 50), 10)
    for _ in range(args.warmup):
        pb.step()
    pb.check("warm-up")
    step_ms = device_time_ms(pb.step, K, pb.stream, dev)
    kv_ms, at_ms = pb.kernel_times(K)
    w = pb.work
    rec = {"step_us": 1e3 * step_ms, "attention_kernel_us": 1e3 * at_ms, "rebuild_kernel_us": 1e3 * kv_ms,
           "steps": K, "value": w["flops"] / (step_ms / 1e3) / 1e12, "unit": "TFLOP/s",
           "tokens_per_s": spec.B * spec.T_q / (step_ms / 1e3),
           "roofline": pb.roofline(at_ms, kv_ms, step_ms, peaks, peak_src),
           "config": prefill_config(pb.spec, "the rebuilt K/V of each step exceed L2")}
    if not args.no_cpu_baseline:
        sec, fl, nq = prefill_cpu_sample(pb.inp, args.cpu_budget / 2)
        rec["cpu_baseline"] = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
                               "kind": "oracle",
                               "sample": f"fp64 numpy: the rebuild of all rows and the attention "
                                         f"of {nq} random query tokens, {sec:.1f} s"}
    del pb
    import torch
    torch.cuda.empty_cache()
    return rec


def run_prefill(args, spec):
    import torch
    rank, world, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pb = PrefillBench(spec, dev, rank)
    work, stream = pb.work, pb.stream
    for _ in range(args.warmup):
        pb.step()
    pb.check("warm-up")

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(dist, local)
    torch.cuda.synchronize(dev)
    with sampler:
        torch.cuda._sleep(4_000_000)
        sampler.mark("start")
        ev0.record(stream)
        for _ in range(args.steps):
            pb.step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        sampler.mark("end")
    barrier(dist, local)
    ms_max = max_over_ranks(dist, ev0.elapsed_time(ev1))
    pb.check("timed region")
    kv_ms, at_ms = pb.kernel_times(max(args.steps, 10))

    # end to end: the prompt's queries in from pinned host memory, o and lse back
    qn_h, qr_h = pb.qn.cpu().pin_memory(), pb.qr.cpu().pin_memory()
    sl_h = pb.sl.cpu().pin_memory()
    o_h = [torch.empty(pb.o.shape, dtype=pb.o.dtype).pin_memory() for _ in range(2)]
    lse_h = [torch.empty(pb.lse.shape, dtype=pb.lse.dtype).pin_memory() for _ in range(2)]
    qn_d = [torch.empty_like(pb.qn) for _ in range(2)]
    qr_d = [torch.empty_like(pb.qr) for _ in range(2)]
    sl_d = [torch.empty_like(pb.sl) for _ in range(2)]
    o_d, lse_d = [pb.o, torch.empty_like(pb.o)], [pb.lse, torch.empty_like(pb.lse)]
    h2d = (qn_h.numel() + qr_h.numel()) * 2 + sl_h.numel() * 4
    d2h = (pb.o.numel() + pb.lse.numel()) * 4

    def e2e_load(k):
        qn_d[k].copy_(qn_h, non_blocking=True)
        qr_d[k].copy_(qr_h, non_blocking=True)
        sl_d[k].copy_(sl_h, non_blocking=True)

    def e2e_compute(i, k):
        pb.rebuild(sl=sl_d[k])
        pb.attend(q_nope=qn_d[k], q_rope=qr_d[k], sl=sl_d[k], o=o_d[k], lse=lse_d[k])

    def e2e_store(k):
        o_h[k].copy_(o_d[k], non_blocking=True)
        lse_h[k].copy_(lse_d[k], non_blocking=True)

    barrier(dist, local)
    e2e_ms = max_over_ranks(dist, pipelined_e2e(torch, dev, stream, args.steps, e2e_load, e2e_compute,
                                                e2e_store))

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    peaks, peak_src = load_peaks()
    total_flops = work["flops"] * world * args.steps
    value = total_flops / (ms_max / 1e3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal draws, shuffled block table)",
        "config": prefill_config(pb.spec, "the rebuilt K/V of each step (%d MB) exceed L2" %
                                 (sum(x.numel() for x in pb.kv) * 2 // 10**6)),
        "tokens_per_s": spec.B * spec.T_q * world * args.steps / (ms_max / 1e3),
        "roofline": pb.roofline(at_ms, kv_ms, ms_max / args.steps, peaks, peak_src),
        "e2e": {"value": total_flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps,
                "note": "per step: q_nope, q_rope and lengths copied in from pinned host "
                        "memory, o and lse copied back; cache and weights resident; copies in, "
                        "compute and copies out on three streams, neighbouring steps "
                        "overlapping (two device buffer sets)"},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        sec, fl, nq = prefill_cpu_sample(pb.inp, args.cpu_budget)
        line["cpu_baseline"] = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": f"fp64 numpy: the rebuild of all rows and the attention "
                                          f"of {nq} random query tokens, {sec:.1f} s"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["mla", "reference"], default="mla")
    ap.add_argument("--workload", default=mi.RAGGED_SERVING.name,
                    choices=sorted(mi.DECODE_WORKLOADS) + sorted(mi.PREFILL_WORKLOADS) +
                    sorted(mi.OUT_PROJ_WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-workload sub-records of the other configurations")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload in mi.OUT_PROJ_WORKLOADS:
        # the output projections alone (one JSON record, one GPU)
        import torch
        peaks, peak_src = load_peaks()
        rec = out_proj_subrecord(mi.OUT_PROJ_WORKLOADS[args.workload], torch.device("cuda", 0), args, peaks, peak_src)
        if args.impl == "reference":
            rec = {"impl": "reference", "metric": "output projection GB/s", "unit": "GB/s",
                   "value": rec.get("cpu_baseline", {}).get("value"), "config": rec["config"]}
        print(json.dumps(rec), flush=True)
        return 0
    if args.workload in mi.PREFILL_WORKLOADS:
        pspec = mi.PREFILL_WORKLOADS[args.workload]
        return run_prefill_reference(args, pspec) if args.impl == "reference" else run_prefill(args, pspec)
    spec = mi.DECODE_WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, spec)
    return run_mla(args, spec)


if __name__ == "__main__":
    sys.exit(main())
