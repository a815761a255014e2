"""Benchmark: paged GQA decode attention on GB300.

One step = one decode-attention call over the whole batch of the workload
(every (sequence, query head) row), inputs resident in HBM.  Prints ONE JSON
line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Default workload: the LLaMA-3-8B-shaped decode batch (32 sequences, H_q 32,
H_kv 8, head_dim 128, block 16, lengths U[512, 4096], shuffled blocks).
Throughput counts algorithmic bytes: the K and V rows of every attended token
once per KV head, plus q, out and the block-table entries in use.  L2: the
timed calls rotate over replicas of the KV cache whose total size is several
times the 129 MB L2, so every call streams from HBM.

--impl reference times the FP64 CPU oracle (the reference arm of this
project) on the host cores, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode attn µs/step and KV GB/s (% of GB300 HBM peak), 1 GPU"
L2_BYTES = 129 * 10**6
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ byte accounting

def algorithmic_bytes(spec, lens) -> dict:
    """K+V rows once per KV head, q read, out written, block-table entries in use."""
    D, BS, H_kv, H_q = spec.D, spec.block_size, spec.H_kv, spec.H_q
    kv = sum(int(L) for L in lens) * H_kv * 4 * D
    qo = len(lens) * H_q * D * 2 * 2
    bt = sum(-(-int(L) // BS) for L in lens) * 4
    return {"kv": kv, "q_out": qo, "block_table": bt, "total": kv + qo + bt}


def group_bytes(spec, L: int) -> int:
    """Algorithmic bytes of one (sequence, KV head) group of G query rows."""
    return L * 4 * spec.D + spec.G * spec.D * 4 + (-(-L // spec.block_size)) * 4 // spec.H_kv


# ------------------------------------------------------------------ environment

def ctas_per_sm(D: int, BS: int, G: int, fp8: bool) -> int:
    """CTAs per SM of the library's persistent grid for a single-token decode
    (the kernel's own rule, ctas_per_sm in csrc/decode_kernel.cuh): one when a
    bf16 stage is 16 KB or more or head_dim 256 has more than 8 query rows,
    three for FP8 caches of head_dim 128 with 16-token pages and up to 8 query
    rows, two otherwise."""
    if (D >= 256 and G > 8) or (not fp8 and D * BS * 4 >= 16384):
        return 1
    if fp8 and D == 128 and BS == 16 and G <= 8:
        return 3
    return 2


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(config_name: str):
    """DRAM bytes per launch recorded by ncu for this workload, if the kernel
    sources are unchanged since the capture (else None)."""
    from paged_kv_gqa_decode_gb300 import build as pbuild

    path = os.path.join(ROOT, "profiles", f"decode_{config_name}_traffic.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_sha256") != pbuild.source_digest():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device: int):
        self.samples = []  # (monotonic time, fields)
        self.proc = None
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = ["--id=" + (uuid if uuid.startswith("GPU-") else "GPU-" + uuid)]
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            idx = vis.split(",")[device] if vis else str(device)
            sel = ["--id=" + idx]
        cmd = ["nvidia-smi", *sel, f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.monotonic(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed region"
        if len(inside) < 3:
            inside = [s for _, s in self.samples]
            window = "whole run (timed region shorter than 3 samples)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        smax = [num(s[1]) for s in inside if num(s[1]) is not None]
        reasons = set()
        for s in inside:
            for name, v in zip(self.NAMES, s[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (read-only queries,
    libnvidia-ml loaded with ctypes), polled as fast as a background thread can
    while the timed region runs, so that even a region of a millisecond holds
    samples.  Changes no GPU setting."""

    SM = 1  # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: int):
        import ctypes

        self.ok = False
        self.samples = []  # (monotonic time, sm MHz, reason bits)
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.handle = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
                return
            self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) \
                or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = None
            if self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.SM, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.ok = self.sample() is not None
        except Exception:
            self.ok = False
        self._stop = None

    def sample(self):
        import ctypes

        mhz, bits = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, self.SM, ctypes.byref(mhz)) != 0:
            return None
        if self.reasons_fn(self.handle, ctypes.byref(bits)) != 0:
            return None
        s = (time.monotonic(), mhz.value, bits.value)
        self.samples.append(s)
        return s

    def start(self):
        if not self.ok:
            return
        self._stop = threading.Event()

        def poll():
            while not self._stop.is_set():
                self.sample()
                time.sleep(0.0002)

        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()

    def stop(self):
        if self._stop is not None:
            self._stop.set()
            self._thread.join()

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return None
        reasons = set()
        for _, _, bits in inside:
            for b, name in self.REASONS.items():
                if bits & b:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(m for _, m, _ in inside),
                "sm_min_mhz": min(m for _, m, _ in inside),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(inside), "window": "timed region (NVML, ~0.2 ms polling)"}


# ------------------------------------------------------------------ oracle timing

def oracle_sample_run(w_host, spec, groups, threads):
    """Run the FP64 oracle on the listed (s, g) groups; returns (seconds, bytes, flops).

    flops: 4 D per token and query head (q.K and p.V, a multiply and an add each)."""
    import oracle

    inp = oracle.Inputs.from_workload(w_host)
    lens = w_host.lens_list
    pairs = [(s, g * spec.G + r) for (s, g) in groups for r in range(spec.G)]
    t = time.perf_counter()
    oracle.decode(inp, pairs=pairs, num_threads=threads)
    dt = time.perf_counter() - t
    flops = sum(lens[s] * spec.G * 4 * spec.D for s, _ in groups)
    return dt, sum(group_bytes(spec, lens[s]) for s, _ in groups), flops


def all_groups(spec, lens):
    return [(s, g) for s in range(len(lens)) for g in range(spec.H_kv) if lens[s] > 0]


def oracle_baseline(w_host, spec, budget_s: float, threads: int):
    """Time the oracle on whole groups in round-robin order for about budget_s seconds."""
    lens = w_host.lens_list
    groups = all_groups(spec, lens)
    done, secs, nbytes, nflops, i = 0, 0.0, 0, 0, 0
    batch = max(1, min(len(groups), 4 * threads))
    while secs < budget_s and done < 10**7:
        chunk = [groups[(i + k) % len(groups)] for k in range(batch)]
        i += batch
        dt, b, f = oracle_sample_run(w_host, spec, chunk, threads)
        secs += dt
        nbytes += b
        nflops += f
        done += batch
    return secs, nbytes, done, len(groups), nflops


# ------------------------------------------------------------------ arms

def build_and_load():
    from paged_kv_gqa_decode_gb300 import build as pbuild

    pbuild.build()
    import paged_kv_gqa_decode_gb300 as pa

    pa.load()
    return pa


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def run_ours(args, world, rank, local):
    pa = build_and_load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = workloads.spec(args.config)
    seed = workloads.SEEDS[args.config] + rank  # each rank decodes its own batch (weak scaling)
    w = workloads.make(spec, seed=seed, device=dev, poison="zero")
    lens = w.lens_list
    nbytes = algorithmic_bytes(spec, lens)
    fp8 = args.kv == "fp8"
    if fp8:
        # e4m3 caches: one byte per element plus one float per (token, KV head) for K and V
        f = workloads.to_fp8(w)
        w.k_cache = w.v_cache = None
        kv = sum(int(L) for L in lens) * spec.H_kv * (2 * spec.D + 8)
        nbytes = dict(nbytes, kv=kv, total=kv + nbytes["q_out"] + nbytes["block_table"])
        base = (f.k8, f.v8, f.k_scale, f.v_scale)
    elif args.kv == "xpacked":
        # the same bf16 values in the x-packed K / D-major V layout
        x = workloads.to_xpacked(w)
        w.k_cache = w.v_cache = None
        base = (x.kx, x.vt, None, None)
    else:
        base = (w.k_cache, w.v_cache, None, None)
    kv_bytes = sum(t.numel() * t.element_size() for t in base if t is not None)
    reps = max(1, min(8, math.ceil(4 * L2_BYTES / max(1, kv_bytes))))
    caches = [base] + [tuple(t.clone() if t is not None else None for t in base)
                       for _ in range(reps - 1)]
    out = torch.empty_like(w.q)
    stream = torch.cuda.current_stream(dev)

    # --qlen > 1: multi-token decode, the last qlen tokens of every sequence query
    # the cache (causal unless --noncausal); q and out grow to qlen rows per sequence
    qlen = args.qlen
    q_in = w.q
    qo = None
    if qlen > 1:
        gq = torch.Generator(device="cpu").manual_seed(seed + 29)
        q_in = torch.randn(spec.num_seqs * qlen, spec.H_q, spec.D, generator=gq).to(
            torch.bfloat16).to(dev)
        qo = torch.arange(0, spec.num_seqs * qlen + 1, qlen, dtype=torch.int32, device=dev)
        out = torch.empty_like(q_in)
        nbytes = dict(nbytes)
        nbytes["q_out"] = spec.num_seqs * qlen * spec.H_q * spec.D * 2 * 2
        nbytes["total"] = nbytes["kv"] + nbytes["q_out"] + nbytes["block_table"]
    causal = not args.noncausal

    # --op: the decode alone, or with each sequence's new tokens appended to the
    # cache first (fused into the decode launch, or as a separate launch; FP8
    # caches quantize the new rows on the way in)
    op = args.op
    k_new = v_new = None
    if op != "decode":
        gk = torch.Generator(device="cpu").manual_seed(seed + 17)
        new_rows = spec.num_seqs * qlen
        shape = (new_rows, spec.H_kv, spec.D)
        k_new = torch.randn(shape, generator=gk).to(torch.bfloat16).to(dev)
        v_new = torch.randn(shape, generator=gk).to(torch.bfloat16).to(dev)
        rows = sum(min(qlen, L) for L in lens) * spec.H_kv
        written = 2 * (spec.D + 4) if fp8 else 2 * spec.D * 2  # K and V: e4m3 + float, or bf16
        nbytes = dict(nbytes)
        nbytes["append"] = rows * (spec.D * 2 * 2 + written)  # bf16 rows read, cache rows written
        nbytes["total"] += nbytes["append"]

    # Early prologue (include/paged_attn.h): in the plain decode ops the work
    # ahead of a launch (the previous step) writes the output only, never the
    # caches, tables or lengths, so the producer may start before it ends.  The
    # append ops write the cache every step: plain launch.
    early = op == "decode"
    pa.paged_attn_set_launch_flags(pa.FLAG_EARLY_PROLOGUE if early else 0)

    def run_op(q, bt, sl, cache, kn, vn, out=out, st=None, qo=qo):
        st = stream if st is None else st
        kc, vc, ksc, vsc = cache
        if qo is not None:
            if op == "decode":
                pa.paged_attn_decode_multi(q, kc, vc, qo, bt, sl, w.scale, qlen, out=out,
                                           stream=st, causal=causal)
            elif op == "append_decode":
                pa.paged_attn_append_decode_multi(q, kn, vn, kc, vc, qo, bt, sl, w.scale, qlen,
                                                  out=out, stream=st, causal=causal)
            else:
                pa.paged_kv_append_multi(kn, vn, kc, vc, qo, bt, sl, stream=st)
                pa.paged_attn_decode_multi(q, kc, vc, qo, bt, sl, w.scale, qlen, out=out,
                                           stream=st, causal=causal)
        elif fp8:
            if op == "decode":
                pa.paged_attn_decode_fp8(q, kc, vc, ksc, vsc, bt, sl, w.scale, out=out,
                                         stream=st)
            elif op == "append_decode":
                pa.paged_attn_append_decode_fp8(q, kn, vn, kc, vc, ksc, vsc, bt, sl, w.scale,
                                                out=out, stream=st)
            else:
                pa.paged_kv_append_fp8(kn, vn, kc, vc, ksc, vsc, bt, sl, stream=st)
                pa.paged_attn_decode_fp8(q, kc, vc, ksc, vsc, bt, sl, w.scale, out=out,
                                         stream=st)
        elif args.kv == "xpacked":
            pa.paged_attn_decode_xpacked(q, kc, vc, bt, sl, w.scale, out=out, stream=st)
        elif op == "decode":
            pa.paged_attn_decode(q, kc, vc, bt, sl, w.scale, out=out, stream=st)
        elif op == "append_decode":
            pa.paged_attn_append_decode(q, kn, vn, kc, vc, bt, sl, w.scale, out=out,
                                        stream=st)
        else:
            pa.paged_kv_append(kn, vn, kc, vc, bt, sl, stream=st)
            pa.paged_attn_decode(q, kc, vc, bt, sl, w.scale, out=out, stream=st)

    # Kernel launches per step, by the library's rules: one decode launch per
    # 4,096 sequences; the append is a launch of its own for multi-token rows, for
    # --op append_then_decode, for FP8 caches of head_dim 256, and for the fused
    # op when the batch has four or more (sequence, KV head) pieces per CTA of the
    # persistent grid (ctas_per_sm).
    fmt = ("multi-token, %d %s queries per sequence" % (qlen, "causal" if causal else
                                                           "non-causal") if qlen > 1 else
           "FP8 caches" if fp8 else "x-packed caches" if args.kv == "xpacked" else "bf16 caches")
    kernel_desc = {"decode": f"paged_decode_kernel ({fmt}; fused combine)",
                   "append_decode": f"paged_decode_kernel ({fmt}) with the cache append of the "
                                    "new tokens",
                   "append_then_decode": f"append kernel + paged_decode_kernel ({fmt})"}[op]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ctas = sms * ctas_per_sm(spec.D, spec.block_size, spec.G, fp8)
    append_launch = op == "append_then_decode" or (op == "append_decode" and (
        (fp8 and spec.D != 128) or qo is not None or spec.num_seqs * spec.H_kv >= 4 * ctas))
    launches_per_step = -(-len(lens) // 4096) + (1 if append_launch else 0)
    kernel_desc += f" ({launches_per_step} launch{'es' if launches_per_step > 1 else ''} per step)"

    def step(i, st=None):
        run_op(q_in, w.block_tables, w.seq_lens, caches[i % reps], k_new, v_new, st=st)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # steps: as given, else enough for ~2 s of timed work
    if args.steps is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(20):
            step(i)
        e1.record(stream)
        e1.synchronize()
        per = e0.elapsed_time(e1) / 20 / 1e3
        steps = int(min(200000, max(50, 2.0 / max(per, 1e-6))))
    else:
        steps = args.steps

    # The timed steps are issued as CUDA graphs, as a decode loop on this GPU
    # would issue them: groups of up to 64 steps (a multiple of the replica count,
    # so that consecutive steps never read the same replica) captured once and
    # replayed, so host-side call latency stays off the GPU's critical path.  The
    # launches inside are the same kernel launches (programmatic dependent launch
    # kept as graph edges).  Eager issue is timed as well and reported beside it.
    per_graph = max(reps, (min(steps, 64) // reps) * reps)
    graphs = {}
    timing_mode = f"CUDA graphs of {per_graph} steps replayed"
    if not args.eager:
        try:
            for n in sorted({per_graph, steps % per_graph} - {0}):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(n):
                        step(i, st=torch.cuda.current_stream())
                graphs[n] = g
            for g in graphs.values():  # one untimed replay each
                g.replay()
            torch.cuda.synchronize()
        except Exception as exc:  # capture unsupported here: eager issue
            torch.cuda.synchronize()
            graphs = {}
            timing_mode = f"eager issue (graph capture failed: {type(exc).__name__})"
    else:
        timing_mode = "eager issue (--eager)"

    def timed_steps():
        if graphs:
            for _ in range(steps // per_graph):
                graphs[per_graph].replay()
            if steps % per_graph:
                graphs[steps % per_graph].replay()
        else:
            for i in range(steps):
                step(i)

    clocks = ClockSampler(local) if rank == 0 and not args.no_clocks else None
    nvml = NvmlClocks(local) if rank == 0 and not args.no_clocks else None
    time.sleep(0.3 if clocks else 0)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def host_lead():
        # A ~50 us spin on the stream ahead of the start event: the host issues
        # the start event and the timed launches while it runs, so the start is
        # stamped when the first step can begin, not before the host has issued
        # it (the timed region still holds exactly the K steps).
        torch.cuda._sleep(100000)

    barrier(world)
    torch.cuda.synchronize()
    if nvml:
        nvml.start()
    t0 = time.monotonic()
    host_lead()
    ev[0].record(stream)
    timed_steps()
    ev[1].record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    if nvml:
        nvml.stop()
    barrier(world)
    elapsed = ev[0].elapsed_time(ev[1]) / 1e3
    elapsed = reduce_max(elapsed, world)
    # the same K steps issued eagerly, one call after another
    eager_s = None
    if graphs:
        torch.cuda.synchronize()
        host_lead()
        ev[0].record(stream)
        for i in range(steps):
            step(i)
        ev[1].record(stream)
        torch.cuda.synchronize()
        eager_s = reduce_max(ev[0].elapsed_time(ev[1]) / 1e3, world) / steps
    # after the timed region: event pairs around single launches on the launching
    # stream (each pair holds one step alone: no overlap with its neighbours)
    j = min(steps, 2000)
    k_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(j)]
    for i in range(j):
        k_ev[i][0].record(stream)
        step(i)
        k_ev[i][1].record(stream)
    torch.cuda.synchronize()
    kernel_s = sum(a.elapsed_time(b) for a, b in k_ev) / max(1, j) / 1e3
    clock_info = None
    if clocks:
        clocks.stop()
        clock_info = clocks.summary(t0, t1)
    if nvml:
        inside = nvml.summary(t0, t1)
        if inside is not None:
            clock_info = dict(inside, nvidia_smi_whole_run=clock_info)
    per_step = elapsed / steps

    # End to end through the public API with host buffers (the `e2e` figure):
    # every step's inputs -- q, block table, lengths (and the new K/V rows, the
    # query offsets) -- sit in pinned host memory of their own, and its output
    # goes to pinned host memory.  The library's kernels read and write those
    # buffers directly over the host link (NVLink-C2C on GB300; pinned memory is
    # addressable from the device), so the transfers happen inside each call and
    # the decode launches still chain as they do on device buffers.  Groups of
    # 32 steps are captured once in a CUDA graph and replayed; the timed region
    # ends when the last output is in host memory.
    per_graph = 32

    def pinned(t):
        return None if t is None else t.cpu().pin_memory()

    zbufs = [dict(q=pinned(q_in), bt=pinned(w.block_tables), sl=pinned(w.seq_lens),
                  kn=pinned(k_new), vn=pinned(v_new), qo=pinned(qo),
                  out=torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory())
             for _ in range(per_graph)]

    def zero_copy_group(cs):
        for i in range(per_graph):
            b = zbufs[i]
            run_op(b["q"], b["bt"], b["sl"], caches[i % reps], b["kn"], b["vn"], out=b["out"],
                   st=cs, qo=b["qo"])

    zero_copy_group(stream)  # warm-up, outside any capture
    torch.cuda.synchronize()
    # the host buffers give the device buffers' result, bit for bit
    check = torch.empty_like(out)
    run_op(q_in, w.block_tables, w.seq_lens, caches[0], k_new, v_new, out=check)
    torch.cuda.synchronize()
    if op == "decode" and not torch.equal(check.cpu().view(torch.int16),
                                          zbufs[0]["out"].view(torch.int16)):
        raise RuntimeError("zero-copy output differs from the device-buffer output")
    zgraph = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            zero_copy_group(torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        zgraph = g
    except Exception:  # capture unsupported here: issue the groups directly
        torch.cuda.synchronize()
    zgroups = max(3, min(steps, 2000) // per_graph)
    barrier(world)
    t = time.perf_counter()
    for _ in range(zgroups):
        if zgraph is not None:
            zgraph.replay()
        else:
            zero_copy_group(stream)
    torch.cuda.synchronize()
    zc_time = reduce_max((time.perf_counter() - t) / (zgroups * per_graph), world)
    zb = zbufs[0]
    zc_h2d = sum(zb[k].numel() * zb[k].element_size() for k in ("q", "bt", "sl", "kn", "vn", "qo")
                 if zb[k] is not None)
    zc_d2h = zb["out"].numel() * zb["out"].element_size()
    zc_mode = ("kernels read each step's pinned host inputs and write its pinned host output "
               f"(no separate copies); CUDA graph of {per_graph} steps" +
               ("" if zgraph is not None else ", no graph"))

    # The same with explicit copies (`e2e_copies`): every step copies its inputs from
    # pinned host memory to the device and its result back to pinned host
    # memory.  The copies run on two copy streams with double-buffered device
    # inputs and outputs, so step i + 1's inputs go up and step i - 1's result
    # comes down while step i computes (events order each buffer's reuse).
    # Groups of 32 steps are captured once in a CUDA graph and replayed, so the
    # host's per-step launch cost stays off the GPU's critical path (the pipeline
    # fills and drains once per group); the timed region ends when the last
    # result is on the host.
    host_q = q_in.cpu().pin_memory()
    host_bt = w.block_tables.cpu().pin_memory()
    host_sl = w.seq_lens.cpu().pin_memory()
    host_kn = k_new.cpu().pin_memory() if k_new is not None else None
    host_vn = v_new.cpu().pin_memory() if v_new is not None else None
    host_outs = [torch.empty_like(host_q).pin_memory() for _ in range(2)]
    host_out = host_outs[0]
    bufs = [dict(q=torch.empty_like(q_in), bt=torch.empty_like(w.block_tables),
                 sl=torch.empty_like(w.seq_lens),
                 kn=torch.empty_like(k_new) if k_new is not None else None,
                 vn=torch.empty_like(v_new) if v_new is not None else None,
                 out=torch.empty_like(out)) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_start = torch.cuda.Event()
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the buffer uploaded
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the step using the buffer computed
    ev_out = [torch.cuda.Event() for _ in range(2)]   # its result downloaded

    def e2e_group(cs):
        """per_graph steps issued on compute stream cs, the copy streams forked from
        and joined back into it (so the group can be captured as one graph)."""
        ev_start.record(cs)
        up.wait_event(ev_start)
        down.wait_event(ev_start)
        for i in range(per_graph):
            k = i % 2
            b = bufs[k]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(ev_done[k])  # step i - 2 has read these inputs
                b["q"].copy_(host_q, non_blocking=True)
                b["bt"].copy_(host_bt, non_blocking=True)
                b["sl"].copy_(host_sl, non_blocking=True)
                if host_kn is not None:
                    b["kn"].copy_(host_kn, non_blocking=True)
                    b["vn"].copy_(host_vn, non_blocking=True)
                ev_in[k].record(up)
            cs.wait_event(ev_in[k])
            if i >= 2:
                cs.wait_event(ev_out[k])  # step i - 2's result has left this buffer
            run_op(b["q"], b["bt"], b["sl"], caches[i % reps], b["kn"], b["vn"], out=b["out"],
                   st=cs)
            ev_done[k].record(cs)
            with torch.cuda.stream(down):
                down.wait_event(ev_done[k])
                host_outs[k].copy_(b["out"], non_blocking=True)
                ev_out[k].record(down)
        cs.wait_event(ev_out[0])
        cs.wait_event(ev_out[1])

    e2e_group(stream)  # warm-up, outside any capture
    torch.cuda.synchronize()
    graph, e2e_mode = None, f"CUDA graph of {per_graph} steps, copies on two streams"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_group(torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        graph = g
    except Exception as exc:  # capture unsupported here: issue the groups directly
        torch.cuda.synchronize()
        e2e_mode = f"copies on two streams, no graph ({type(exc).__name__})"
    groups = max(3, min(steps, 2000) // per_graph)
    e2e_steps = groups * per_graph
    barrier(world)
    t = time.perf_counter()
    for _ in range(groups):
        if graph is not None:
            graph.replay()
        else:
            e2e_group(stream)
    torch.cuda.synchronize()
    e2e_time = reduce_max((time.perf_counter() - t) / e2e_steps, world)
    h2d = host_q.numel() * 2 + host_bt.numel() * 4 + host_sl.numel() * 4
    if host_kn is not None:
        h2d += (host_kn.numel() + host_vn.numel()) * 2
    d2h = host_out.numel() * 2

    result = None
    if rank == 0:
        peak, peak_src = measured_peaks()
        # The kernel's average launch duration: with one launch per step, the
        # timed region's events over its launches (back-to-back launches overlap
        # one's prologue with the previous one's tail, as in a decode loop);
        # otherwise the event pairs around single launches.  The pairs break that
        # overlap and add the launch latency, so their figure is reported beside
        # it as the isolated duration.
        single = launches_per_step == 1
        launch_s = per_step if single else kernel_s
        achieved = nbytes["total"] / launch_s / 1e9
        plain = op == "decode" and args.kv == "bf16" and qlen == 1
        traffic = profile_traffic(args.config) if plain else None
        cpu = None
        if not args.no_cpu_baseline and args.kv == "bf16" and qlen == 1:  # the baseline leg times the bf16 oracle
            w_host = workloads.host_copy(w)
            threads = len(os.sched_getaffinity(0))
            secs, b, ngroups, total_groups, nflops = oracle_baseline(w_host, spec,
                                                                     args.cpu_budget, threads)
            cpu = {"value": round(b / secs / 1e9, 4), "unit": "GB/s", "cores": threads,
                   "kind": "oracle",
                   "sample": f"{ngroups} (sequence, KV head) groups of the {args.config} "
                             f"workload ({total_groups} per step), round-robin, "
                             f"{secs:.1f} s of FP64 CPU work",
                   "gflop_per_s": round(nflops / secs / 1e9, 3)}
        result = {
            "metric": METRIC,
            "value": round(world * nbytes["total"] / per_step / 1e9, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": steps,
            "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 5),
            "us_per_step": round(per_step * 1e6, 2),
            "kv_gbs": round(nbytes["kv"] / per_step / 1e9, 2),
            "pct_of_hbm_peak": round(100 * achieved / peak, 2),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "e4m3" if fp8 else "bf16",
            "data": "synthetic (seeded; see workloads.py)",
            "config": {
                "workload": spec.description,
                "name": args.config,
                "num_seqs": spec.num_seqs, "H_q": spec.H_q, "H_kv": spec.H_kv,
                "head_dim": spec.D, "block_size": spec.block_size,
                "tokens": int(sum(lens)), "seed": seed, "op": op, "kv": args.kv, "q_len": qlen,
                "bytes_per_step": nbytes,
                "l2": f"inputs larger than L2: {reps} KV-cache replicas rotated "
                      f"({reps * kv_bytes / 1e9:.2f} GB vs 129 MB L2)",
                "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                "launch": "early prologue (the producer starts before the previous launch "
                          "ends; caches, tables and lengths are not written between steps)"
                if early else "plain (each step writes the cache)",
                "issue": timing_mode,
            },
            "roofline": {
                "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_src == "measured" else "fallback 6800 GB/s",
                "kernel": kernel_desc,
                "kernel_us": round(launch_s * 1e6, 2),
                "eager_us_per_step": round(eager_s * 1e6, 2) if eager_s else None,
                "kernel_us_isolated": round(kernel_s * 1e6, 2),
                "frac_isolated": round(nbytes["total"] / kernel_s / 1e9 / peak, 4),
                "timing": (f"CUDA events over the timed region on the launching stream, "
                           f"{steps} launches" if single else
                           f"CUDA events around {j} of the {steps} timed launches") +
                          f"; isolated: event pairs around {j} single launches after it",
            },
            "e2e": {"value": round(world * nbytes["total"] / zc_time / 1e9, 2), "unit": "GB/s",
                    "us_per_step": round(zc_time * 1e6, 2), "mode": zc_mode,
                    "h2d_bytes_per_step": zc_h2d, "d2h_bytes_per_step": zc_d2h},
            "e2e_copies": {"value": round(world * nbytes["total"] / e2e_time / 1e9, 2),
                           "unit": "GB/s", "us_per_step": round(e2e_time * 1e6, 2),
                           "mode": e2e_mode, "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h},
            "gpu_launches": steps * launches_per_step,
            "clocks": clock_info,
        }
        if cpu:
            result["cpu_baseline"] = cpu
    return result


def run_reference(args, world, rank):
    """The FP64 oracle on host cores, each step a bounded sample of the workload."""
    if rank != 0:
        return None
    spec = workloads.spec(args.config)
    seed = workloads.SEEDS[args.config]
    w = workloads.make(spec, seed=seed, device="cpu", poison="zero")
    lens = w.lens_list
    threads = len(os.sched_getaffinity(0))
    groups = all_groups(spec, lens)
    steps = args.steps if args.steps is not None else 20
    budget_total = args.reference_budget
    # size each step so warmup + steps stay within the budget
    per_step_budget = budget_total / max(1, steps + args.warmup)
    dt1, _, _ = oracle_sample_run(w, spec, groups[:threads], threads)
    per_group = dt1 / max(1, min(threads, len(groups)))
    per_step_groups = int(max(1, min(len(groups), per_step_budget / max(per_group, 1e-9))))
    i = 0

    def step():
        nonlocal i
        chunk = [groups[(i + k) % len(groups)] for k in range(per_step_groups)]
        i += per_step_groups
        return oracle_sample_run(w, spec, chunk, threads)

    for _ in range(args.warmup):
        step()
    secs = 0.0
    nbytes = 0
    nflops = 0
    for _ in range(steps):
        dt, b, f = step()
        secs += dt
        nbytes += b
        nflops += f
    value = nbytes / secs / 1e9
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(secs / steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; see workloads.py)",
        "config": {"workload": spec.description, "name": args.config, "seed": seed},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{per_step_groups} of {len(groups)} (sequence, KV head) "
                                   "groups per step, round-robin",
                         "gflop_per_s": round(nflops / secs / 1e9, 3)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="llama8b", choices=sorted(workloads.SPECS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8", "xpacked"],
                    help="cache format: bf16, e4m3 bytes with a float per cache row, or bf16 "
                         "in the x-packed K / D-major V layout")
    ap.add_argument("--op", default="decode",
                    choices=["decode", "append_decode", "append_then_decode"],
                    help="decode alone, or with each sequence's new token appended to the "
                         "cache first (fused into the decode launch, or a separate launch)")
    ap.add_argument("--qlen", type=int, default=1,
                    help="query tokens per sequence: > 1 runs the multi-token (causal) decode")
    ap.add_argument("--noncausal", action="store_true",
                    help="with --qlen > 1: every query row attends all of its sequence's tokens")
    ap.add_argument("--eager", action="store_true",
                    help="issue the timed steps one call at a time instead of as CUDA graphs")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline field")
    ap.add_argument("--reference-budget", type=float, default=90.0,
                    help="seconds of oracle work for --impl reference")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.kv == "xpacked" and args.op != "decode":
        ap.error("--kv xpacked runs the decode alone (--op decode)")
    if args.qlen > 1 and args.kv != "bf16":
        ap.error("--qlen > 1 runs over bf16 caches")
    if args.noncausal and args.qlen < 2:
        ap.error("--noncausal needs --qlen > 1")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
