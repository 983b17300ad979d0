#!/usr/bin/env python
"""Benchmark of LSH-sampled decode attention (MagicPIG's hot path) on GB300.

One step = one whole job of the Llama-3.1-8B-shaped long-context workload: build the
hash tables of 32 layers x 8 KV heads from 96K prefill keys (center, SimHash on
tensor cores, bucket), then 64 decode steps, each appending one key per KV head and
answering all 32 x 32 query heads. Inputs are resident in HBM when timing starts
(12.9 GB of K/V, larger than L2). `value` is queries answered per second by all
ranks; the JSON line also carries per-kernel timings, the roofline of the dominant
kernel, the CPU oracle's throughput on a bounded sample and an end-to-end figure
with host buffers.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LSH-sampled decode attention: μs/step, queries/s, achieved HBM GB/s vs roofline"
L2_FLUSH_BELOW = 512 << 20  # inputs smaller than this are timed job by job with L2 flushed between
DEFAULT_WORKLOAD = 2


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--w-fp32", action="store_true",
                    help="draw W in fp32 (not rounded to bf16): the tensor-core hashing then runs on "
                         "W's three-term bf16 split")
    ap.add_argument("--sweep", action="store_true",
                    help="sampled budget and step time over the pages' (K, L) grid, centering on and off "
                         "(one layer of the workload; one JSON line per grid point)")
    ap.add_argument("--eager", action="store_true",
                    help="launch every call from Python instead of replaying the captured job graph")
    ap.add_argument("--cone", type=float, default=None,
                    help="key cone a in k = a·mu + N(0, I), sink -a·mu (the pages' narrow cones: 40 to 80); "
                         "default: the workload's recipe")
    ap.add_argument("--center-query", action="store_true",
                    help="hash the query centered (q - c) and take p from cos(q - c, k - c)")
    return ap.parse_args()


# ----------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no data-path collective)
# ----------------------------------------------------------------------------------

def dist_setup(use_cuda: bool):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if use_cuda:
        torch.cuda.set_device(local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, use_cuda: bool) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------
# peaks and clocks
# ----------------------------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not self.path:
            return None
        rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        os.unlink(self.path)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------

class Job:
    """Buffers of one workload replica on the current GPU and the ABI calls of one job."""

    def __init__(self, mp, wl, device, stream, center_query: bool = False):
        import torch
        import workloads as WL
        self.mp, self.wl, self.dev, self.stream = mp, wl, device, stream
        t = WL.generate(wl, device=device)
        self.keys, self.values, self.W = t["keys"], t["values"], t["W"].contiguous()
        self.queries = t["queries"]
        self.cfg = mp.make_config(layers=wl.layers, batch=wl.batch, kv_heads=wl.kv_heads, q_heads=wl.q_heads,
                                  head_dim=wl.head_dim, K=wl.K, L=wl.L, n_sink=wl.n_sink, window=wl.window,
                                  capacity=wl.capacity, dtype=wl.dtype, w_per_layer=wl.w_per_layer,
                                  center_query=center_query)
        self.tl = mp.mp_tables_layout_get(self.cfg)
        self.dl = mp.mp_decode_layout_get(self.cfg)
        self.tables = torch.empty(self.tl.total_bytes, dtype=torch.uint8, device=device)
        self.scratch = torch.empty(self.dl.total_bytes, dtype=torch.uint8, device=device)
        self.outs = torch.empty(wl.steps, wl.layers, wl.batch, wl.q_heads, wl.head_dim, dtype=torch.float32,
                                device=device)
        self.sp = stream.cuda_stream
        self.hook = None
        self.graph = None

    def build(self, keys=None, W=None):
        mp = self.mp
        mp.mp_build_tables(self.cfg, self.keys if keys is None else keys, self.wl.n_prefill,
                           self.W if W is None else W, self.tables, stream=self.sp)

    def decode_steps(self, keys=None, values=None, queries=None):
        mp, wl = self.mp, self.wl
        k = self.keys if keys is None else keys
        v = self.values if values is None else values
        qs = self.queries if queries is None else queries
        for s in range(wl.steps):
            n = wl.seq_len(s)
            if wl.append:
                # append token n - 1 and decode over n tokens: one call, one hashing launch
                mp.mp_decode_step(self.cfg, self.tables, k, v, n - 1, qs[s], self.outs[s], self.scratch,
                                  scratch_bytes=self.dl.total_bytes, stream=self.sp)
            else:
                mp.mp_decode_attention(self.cfg, self.tables, k, v, n, qs[s], self.outs[s], self.scratch,
                                       scratch_bytes=self.dl.total_bytes, stream=self.sp)
            if self.hook:
                self.hook(s, n)

    def run(self):
        if self.graph is not None:
            self.graph.replay()
            return
        self.build()
        self.decode_steps()

    def capture(self):
        """Capture one whole job (build + all decode steps: the same ABI calls) into a
        CUDA graph so that replays carry no host launch overhead. Returns an error
        string or None."""
        import torch
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream, capture_error_mode="relaxed"):
                self.build()
                self.decode_steps()
            self.graph = g
            return None
        except Exception as e:  # noqa: BLE001
            self.graph = None
            return f"{type(e).__name__}: {e}"

    @property
    def resident_bytes(self):
        """Device bytes a job reads: K, V, queries, W and the tables."""
        return sum(t.numel() * t.element_size() for t in (self.keys, self.values, self.queries, self.W)) + \
            self.tl.total_bytes

    @property
    def queries_per_job(self):
        wl = self.wl
        return wl.steps * wl.layers * wl.batch * wl.q_heads

    @property
    def launches_per_job(self):
        # prepare_w, the -log u table, center (partial sums, mean, -W^T c), hash keys, csr
        # build; per step: one hash launch (the appended keys, which also marks the appended
        # end, with the queries), match, attend
        return 7 + self.wl.steps * 3


def decode_state_stats(job, torch):
    """Device-side sums used for algorithmic bytes: total list entries and sampled entries,
    and the total bucket entries the match kernel walked (CSR mode)."""
    wl, dl, tl = job.wl, job.dl, job.tl
    Q = wl.layers * wl.batch * wl.q_heads
    U = wl.layers * wl.batch * wl.kv_heads
    ln = job.scratch[dl.list_len: dl.list_len + 4 * Q].view(torch.int32).to(torch.int64)
    ns = job.scratch[dl.sample_count: dl.sample_count + 4 * Q].view(torch.int32).to(torch.int64)
    walked = torch.zeros((), dtype=torch.int64, device=ln.device)
    if tl.csr_offsets:
        qc = (job.scratch[dl.q_codes: dl.q_codes + 2 * Q * wl.L].view(torch.int16).to(torch.int64)
              & 0xFFFF).view(Q, wl.L)
        nb, nseg = tl.n_buckets, -(-wl.capacity // 32768)
        off = (job.tables[tl.csr_offsets: tl.csr_offsets + 2 * U * wl.L * nseg * (nb + 1)].view(torch.int16)
               .to(torch.int64) & 0xFFFF).view(U, wl.L, nb + 1, nseg)  # bucket-major, segments innermost
        unit = torch.arange(Q, device=qc.device) // wl.group
        t = torch.arange(wl.L, device=qc.device)
        used = -(-(wl.n_prefill - min(wl.n_sink, wl.n_prefill)) // 32768)
        for sg in range(used):
            b0 = off[unit[:, None], t[None, :], qc, sg]
            b1 = off[unit[:, None], t[None, :], qc + 1, sg]
            walked = walked + (b1 - b0).sum()
    return torch.stack([ln.sum(), ns.sum(), walked])


def run_ours(args, rank, world, local):
    import torch

    import workloads as WL
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as mp

    dev = torch.device("cuda", local)
    wl = WL.WORKLOADS[args.workload]
    wl = wl.replace(seed=wl.seed + 1000 * rank)  # independent replica per rank
    if args.w_fp32:
        wl = wl.replace(w_bf16=False, name=wl.name + "-fp32W")
    if args.cone is not None:
        wl = wl.replace(cone=args.cone, sink_scale=1.0, name=wl.name + "-cone%g" % args.cone)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        job = Job(mp, wl, dev, stream, center_query=args.center_query)
    torch.cuda.synchronize()

    # warm-up (eager), then capture the job into a CUDA graph unless --eager
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            job.run()
    torch.cuda.synchronize()
    # the W status bit is informational (fp32 W runs on its three-term bf16 split)
    assert (mp.mp_get_status(job.tables, stream=job.sp) & ~mp.MP_STATUS_W_NOT_BF16) == 0
    launch_mode = "eager"
    if not args.eager:
        err = job.capture()
        if err is None:
            launch_mode = "cuda-graph"
            with torch.cuda.stream(stream):
                job.run()  # one replay before timing
            torch.cuda.synchronize()
            assert (mp.mp_get_status(job.tables, stream=job.sp) & ~mp.MP_STATUS_W_NOT_BF16) == 0
        else:
            launch_mode = "eager (graph capture failed: %s)" % err[:120]

    # timed region. Inputs larger than L2 (the long-context jobs): the K jobs back to back
    # between two events. Inputs that fit in L2 (small configurations): each job between
    # its own two events, with a 256 MB write between jobs to flush L2, outside the events.
    resident = job.resident_bytes
    flush = resident < L2_FLUSH_BELOW
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if flush else 1)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            if flush:
                for e0, e1 in evs:
                    flush_buf.fill_(1)
                    e0.record(stream)
                    job.run()
                    e1.record(stream)
            else:
                evs[0][0].record(stream)
                for _ in range(args.steps):
                    job.run()
                evs[0][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    ms_max = max_over_ranks(ms, world, True)
    clocks = clk.summary()

    # per-kernel device time (events around each launch) + algorithmic sizes, one job
    stats = torch.zeros(3, dtype=torch.int64, device=dev)

    def hook(s, n):
        stats.add_(decode_state_stats(job, torch))

    job.hook = hook
    graph, job.graph = job.graph, None  # the per-launch profile runs the calls eagerly
    mp.mp_profile_enable(True)
    with torch.cuda.stream(stream):
        job.run()
    torch.cuda.synchronize()
    prof = mp.mp_profile_read()
    mp.mp_profile_enable(False)
    job.hook = None
    job.graph = graph
    list_entries, sampled_entries, bucket_entries = [int(x) for x in stats.cpu()]

    pk = peaks()
    res = summarize(job, wl, prof, pk, list_entries, sampled_entries, bucket_entries)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(job, stream, args, world)

    queries = job.queries_per_job * args.steps * world
    value = queries / (ms_max / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic: seeded cone keys k=%gmu+N(0,I) with sink k0=-%gmu, queries q=-2mu+N(0,I), " % (
            wl.cone, wl.sink_scale * wl.cone) +
                "values N(0,1), W N(0,1)" + (" rounded to bf16" if wl.w_bf16 else " in fp32"),
        "config": {"workload": wl.name, "layers": wl.layers, "batch": wl.batch, "kv_heads": wl.kv_heads,
                   "q_heads": wl.q_heads, "head_dim": wl.head_dim, "n_prefill": wl.n_prefill,
                   "decode_steps": wl.steps, "K": wl.K, "L": wl.L, "n_sink": wl.n_sink, "window": wl.window,
                   "step": "build tables + %d x (append + decode attention)" % wl.steps,
                   "parallelism": "replicas" if world > 1 else "single",
                   "query": "centered (q - c)" if args.center_query else "as is",
                   "launch": launch_mode,
                   "l2": ("inputs larger than L2 (%.1f GB of K/V and tables resident)" % (resident / 1e9))
                   if not flush else ("inputs fit in L2 (%.0f MB of K/V and tables): 256 MB written between "
                                      "timed jobs, outside the timed events" % (resident / 1e6))},
        "us_per_decode_step": res["us_per_decode_step"],
        "build_ms": res["build_ms"],
        "sampled_fraction": res["sampled_fraction"],
        "closed_form_fraction": res["closed_form_fraction"],
        "roofline": res["roofline"],
        "pipeline_roofline": res["pipeline_roofline"],
        "kernels": res["kernels"],
        "gpu_launches": job.launches_per_job * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": None,
    }
    return line, job


# kernel -> source file whose contents the recorded DRAM counters belong to
KERNEL_SOURCE = {
    "attend": "mp_decode.cu", "match_csr": "mp_decode.cu", "hash_keys_tc": "mp_gemm.cu",
    "hash_query": "mp_gemm.cu", "hash_append": "mp_gemm.cu", "hash_step": "mp_gemm.cu", "csr_build": "mp_csr.cu",
    "center": "mp_hash.cu",
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def measured_traffic(kernel: str, algorithmic_per_launch: float):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu counters:
    the captured launch's traffic per algorithmic byte (or flop), times this launch's
    algorithmic amount. None when no counters are recorded or the kernel's source file
    has changed since they were taken."""
    import hashlib
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)["kernels"][kernel]
        src = os.path.join(ROOT, "lsh_sampled_sparse_centered_gb300", "csrc", KERNEL_SOURCE[kernel])
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        return float(rec["dram_bytes_per_algorithmic_unit"]) * algorithmic_per_launch
    except (OSError, KeyError, ValueError):
        return None


def summarize(job, wl, prof, pk, list_entries, sampled_entries, bucket_entries):
    """Per-kernel average durations and algorithmic work for one job; roofline of the
    kernel with the largest share of device time."""
    esz = 2 if wl.dtype == "bf16" else 4
    U = wl.layers * wl.batch * wl.kv_heads
    Q = wl.layers * wl.batch * wl.q_heads
    d, KL = wl.head_dim, wl.K * wl.L
    n0, s = wl.n_prefill, wl.n_sink
    steps = wl.steps
    hbm = pk["hbm_gbs"]
    tc = pk["bf16_tflops_sustained"]
    work = {
        # name: (kind, amount per job)   kind: "bytes" or "flops"
        "prepare_w": ("bytes", (wl.layers if wl.w_per_layer else 1) * KL * d * (4 + 4 + esz)),
        "center": ("bytes", U * (n0 - s) * d * esz),
        "hash_keys_tc": ("flops", 2.0 * U * n0 * d * KL),
        "hash_keys_simt": ("flops", 2.0 * U * n0 * d * KL),
        "csr_build": ("bytes", U * wl.L * ((n0 - s) * (2 + 2) + -(-(n0 - s) // 32768) * (2 ** wl.K + 1) * 2)),
        "hash_append": ("flops", 2.0 * steps * U * d * KL),
        "hash_step": ("flops", 2.0 * steps * (U + Q) * d * KL),
        "mark_appended": ("bytes", 0),
        "logu_lut": ("bytes", (4096 + 1) * 4),
        "hash_query": ("flops", 2.0 * steps * Q * d * KL),
        "match_csr": ("bytes", bucket_entries * 2 + steps * Q * wl.L * (4 * -(-(n0 - s) // 32768) + 2)
                      + list_entries * 4),
        "attend": ("bytes", list_entries * (2 * d * esz + 4) + steps * Q * d * (esz + 4)),
    }
    kernels = {}
    total = sum(v[1] for v in prof.values())
    for name, (launches, tot_ms) in prof.items():
        kind, amt = work.get(name, ("bytes", 0))
        avg = tot_ms / launches
        rate = amt / (tot_ms / 1e3) if tot_ms > 0 else 0.0
        ent = {"launches": launches, "avg_us": 1e3 * avg, "total_ms": tot_ms, "share": tot_ms / total}
        if kind == "bytes":
            ent.update({"achieved": rate / 1e9, "unit": "GB/s", "frac": rate / 1e9 / hbm})
        else:
            ent.update({"achieved": rate / 1e12, "unit": "TFLOP/s", "frac": rate / 1e12 / tc})
        ent["algorithmic_per_launch"] = amt / launches
        kernels[name] = ent
    dom = max(kernels, key=lambda k: kernels[k]["share"])
    kd = kernels[dom]
    kind = work[dom][0]
    roof = {"kernel": dom, "bound": "hbm" if kind == "bytes" else "tensor", "achieved": kd["achieved"],
            "peak": hbm if kind == "bytes" else tc, "unit": kd["unit"], "frac": kd["frac"],
            "traffic": measured_traffic(dom, kd["algorithmic_per_launch"]),
            "peak_source": pk["source"] + (" (sustained)" if kind != "bytes" else "")}
    # whole-job roofline: bytes at HBM bandwidth + hashing flops at tensor peak
    t_roof = sum(v[1] / (hbm * 1e9) for k, v in work.items() if v[0] == "bytes" and k in prof)
    t_roof += sum(v[1] / (tc * 1e12) for k, v in work.items() if v[0] == "flops" and k in prof)
    build_ms = sum(prof[k][1] for k in ("prepare_w", "logu_lut", "center", "hash_keys_tc", "hash_keys_simt",
                                        "csr_build", "planes_build")
                   if k in prof)
    dec_ms = total - build_ms
    x = 0.5 ** wl.K
    closed = 1 - (1 - x) ** wl.L - wl.L * x * (1 - x) ** (wl.L - 1)
    region = sum(max(0, wl.seq_len(t) - wl.window - min(s, wl.seq_len(t))) for t in range(steps)) * Q
    return {
        "kernels": kernels, "roofline": roof,
        "pipeline_roofline": {"roofline_ms": 1e3 * t_roof, "measured_ms": total,
                              "frac": (1e3 * t_roof) / total if total else None},
        "build_ms": build_ms, "us_per_decode_step": 1e3 * dec_ms / steps,
        "sampled_fraction": sampled_entries / region if region else None,
        "closed_form_fraction": closed,
    }


def e2e_groups(wl):
    """How the end-to-end run splits the job so that compute on one part overlaps the
    host-to-device copy of the next: groups of layers (any number of layers per group
    that divides them, four groups at most), else groups of sequences when there is one
    layer, else one group. Returns (dimension, groups) with dimension "layers",
    "batch" or None. The copies dominate, so the job ends about one group's compute
    after the last copy; smaller groups do not shorten that tail, because a group of few
    layers decodes its steps at the latency of small launches (eight groups of four
    layers measured 68.0 ms against 67.8 ms for four groups of eight)."""
    for dim, size in (("layers", wl.layers), ("batch", wl.batch if wl.layers == 1 else 1)):
        for g in (4, 2):
            if size >= g and size % g == 0:
                return dim, g
    return None, 1


def run_e2e(job, stream, args, world):
    """Same job through the public API with host buffers: pinned host inputs copied in
    and outputs copied back inside the timed region. The job is issued in groups of
    layers (or sequences): one copy stream moves each group's keys and W, then its values
    and queries, in order; each group's build and decode steps start as soon as its own
    inputs have landed, and its outputs go back on a second copy stream while the next
    group computes. Two sets of device buffers let the next job's copies start while
    this job still computes, as a serving loop would run successive jobs."""
    import torch
    mp, wl = job.mp, job.wl
    dim, ng = e2e_groups(wl)
    per = (wl.layers if dim == "layers" else wl.batch if dim == "batch" else 1) // ng

    def part(t, i, lead=0):
        """Group i of a tensor whose layer dimension is `lead` (its batch dimension is
        lead + 1)."""
        if dim is None:
            return t
        return t.narrow(lead if dim == "layers" else lead + 1, i * per, per)

    def pinned(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    w_grouped = dim == "layers" and wl.w_per_layer
    # per group: keys, values (and W) are contiguous slices; queries and outputs get
    # buffers of their own so that every copy is one dense block
    h_keys, h_vals, h_W = pinned(job.keys), pinned(job.values), pinned(job.W)
    h_q = [pinned(part(job.queries, i, lead=1).contiguous()) for i in range(ng)]
    gcfg = mp.make_config(layers=per if dim == "layers" else wl.layers, batch=per if dim == "batch" else wl.batch,
                          kv_heads=wl.kv_heads, q_heads=wl.q_heads, head_dim=wl.head_dim, K=wl.K, L=wl.L,
                          n_sink=wl.n_sink, window=wl.window, capacity=wl.capacity, dtype=wl.dtype,
                          w_per_layer=wl.w_per_layer, center_query=bool(job.cfg.center_query))
    gtl, gdl = mp.mp_tables_layout_get(gcfg), mp.mp_decode_layout_get(gcfg)

    class Set:
        """Device buffers of one job in flight (and its host outputs); two sets let the
        next job's copies run while this job computes."""

        def __init__(self):
            self.keys, self.vals = torch.empty_like(job.keys), torch.empty_like(job.values)
            self.W = torch.empty_like(job.W)
            self.q = [torch.empty(q.shape, dtype=q.dtype, device=job.dev) for q in h_q]
            self.out = [torch.empty(q.shape, dtype=torch.float32, device=job.dev) for q in h_q]
            self.h_out = [torch.empty(q.shape, dtype=torch.float32, pin_memory=True) for q in h_q]
            self.tables = [torch.empty(gtl.total_bytes, dtype=torch.uint8, device=job.dev) for _ in range(ng)]
            self.scratch = [torch.empty(gdl.total_bytes, dtype=torch.uint8, device=job.dev) for _ in range(ng)]
            self.free = None  # event: the last job on this set is done with it

    sets = [Set(), Set()]
    torch.cuda.synchronize()
    up = torch.cuda.Stream(device=job.dev)
    down = torch.cuda.Stream(device=job.dev)

    def copy_on(s, dst, src):
        with torch.cuda.stream(s):
            dst.copy_(src, non_blocking=True)

    def mark(s):
        e = torch.cuda.Event()
        e.record(s)
        return e

    def one(k, compute=True):
        S = sets[k % 2]
        if S.free is not None:
            up.wait_event(S.free)  # the job before the previous one is done with this set
        ev_build, ev_decode = [], []
        for i in range(ng):
            copy_on(up, part(S.keys, i), part(h_keys, i))
            if w_grouped or i == 0:
                copy_on(up, part(S.W, i) if w_grouped else S.W, part(h_W, i) if w_grouped else h_W)
            ev_build.append(mark(up))
            copy_on(up, part(S.vals, i), part(h_vals, i))
            copy_on(up, S.q[i], h_q[i])
            ev_decode.append(mark(up))
        for i in range(ng):
            if not compute:
                stream.wait_event(ev_decode[i])
                down.wait_event(mark(stream))
                copy_on(down, S.h_out[i], S.out[i])
                continue
            keys_i, vals_i = part(S.keys, i), part(S.vals, i)
            stream.wait_event(ev_build[i])
            mp.mp_build_tables(gcfg, keys_i, wl.n_prefill, part(S.W, i) if w_grouped else S.W, S.tables[i],
                               stream=job.sp)
            stream.wait_event(ev_decode[i])
            for s_ in range(wl.steps):
                n = wl.seq_len(s_)
                if wl.append:
                    mp.mp_decode_step(gcfg, S.tables[i], keys_i, vals_i, n - 1, S.q[i][s_], S.out[i][s_],
                                      S.scratch[i], scratch_bytes=gdl.total_bytes, stream=job.sp)
                else:
                    mp.mp_decode_attention(gcfg, S.tables[i], keys_i, vals_i, n, S.q[i][s_], S.out[i][s_],
                                           S.scratch[i], scratch_bytes=gdl.total_bytes, stream=job.sp)
            down.wait_event(mark(stream))
            copy_on(down, S.h_out[i], S.out[i])
        stream.wait_stream(down)
        S.free = mark(stream)

    n = max(1, min(args.steps, 6))
    with torch.cuda.stream(stream):
        one(0)
        one(1)
    torch.cuda.synchronize()
    for S in sets:
        for t in S.tables:
            assert (mp.mp_get_status(t, stream=job.sp) & ~mp.MP_STATUS_W_NOT_BF16) == 0
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        up.wait_event(ev0)
        for k in range(n):
            one(k)
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, True) / n
    # the same copies with no compute: what the host link alone takes per job
    with torch.cuda.stream(stream):
        ev0.record(stream)
        up.wait_event(ev0)
        for k in range(n):
            one(k, compute=False)
        ev1.record(stream)
    torch.cuda.synchronize()
    copy_ms = max_over_ranks(ev0.elapsed_time(ev1), world, True) / n
    bi = sum(t.numel() * t.element_size() for t in [h_keys, h_vals, h_W] + h_q)
    bo = sum(t.numel() * t.element_size() for t in sets[0].h_out)
    del sets
    return {"value": job.queries_per_job * world / (ms / 1e3), "unit": "queries/s", "ms_per_step": ms,
            "steps": n, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "copies_alone_ms": copy_ms, "host_link_gbs": (bi + bo) / (copy_ms / 1e3) / 1e9,
            "overlap": ("%d groups of %s, each built and decoded as soon as its inputs land; two jobs in "
                        "flight (the next job's copies run while this one computes)" % (ng, dim))
            if dim else "two jobs in flight"}


# ----------------------------------------------------------------------------------
# CPU oracle timing (bounded sample of the same workload)
# ----------------------------------------------------------------------------------

def oracle_sample(wl, decode_steps: int = 4):
    """Time the fp64 oracle on one KV head of the workload: its table build (all
    tokens hashed) and `decode_steps` decode steps for each of its query heads; scale
    to the whole job by unit counts. Returns (queries/s, seconds spent, description)."""

    import oracle as O
    import workloads as WL
    cap, d = wl.capacity, wl.head_dim
    k = WL.round_to(WL.keys_block(wl, 0, 0, 0, 0, cap), wl.dtype).double().numpy()
    v = WL.round_to(WL.values_block(wl, 0, 0, 0, 0, cap), wl.dtype).double().numpy()
    W = WL.projection(wl, 0).double().numpy()
    t0 = time.perf_counter()
    tab = O.HeadTables(k, W, wl.K, wl.L, wl.n_sink, wl.n_prefill, n_total=cap)
    t_build = time.perf_counter() - t0
    steps = list(range(min(decode_steps, wl.steps)))
    nq = 0
    t1 = time.perf_counter()
    for s in steps:
        q = WL.round_to(WL.query_block(wl, s, 0, 0), wl.dtype).double().numpy()
        n = wl.seq_len(s)
        for g in range(wl.group):
            O.decode_head(q[g], k[:n], v[:n], tab, n, wl.window)
            nq += 1
    t_dec = time.perf_counter() - t1
    U = wl.layers * wl.batch * wl.kv_heads
    total_q = wl.steps * wl.layers * wl.batch * wl.q_heads
    job_s = t_build * U + t_dec * (total_q / nq)
    desc = (f"one KV head (layer 0, sequence 0, head 0): table build over {cap} tokens "
            f"({t_build:.2f} s) + {len(steps)} decode steps x {wl.group} query heads ({t_dec:.2f} s); "
            f"job time scaled by {U} heads and {total_q} queries; one process: numpy's BLAS "
            f"matrix products may use all {cpu_cores()} cores, everything else runs on one thread")
    return total_q / job_s, t_build + t_dec, desc


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, rank, world):
    import workloads as WL
    wl = WL.WORKLOADS[args.workload]
    if rank != 0:
        return None
    for _ in range(args.warmup):
        oracle_sample(wl, decode_steps=1)
    vals, secs = [], 0.0
    t0 = time.perf_counter()
    desc = ""
    for _ in range(args.steps):
        v, sec, desc = oracle_sample(wl, decode_steps=1)
        vals.append(v)
        secs += sec
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same recipe as the GPU arm)",
        "config": {"workload": wl.name, "step": "bounded sample of the job on the CPU oracle"},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


SWEEP_GRID = [(8, 75), (8, 90), (9, 120), (10, 150), (10, 220), (10, 300), (11, 300)]


def run_sweep(args):
    """(K, L) grid of the pages with centering on and off on one layer of the workload:
    measured sampled fraction (the GPU's |S| / |R|), the isotropic closed form, the
    list entries per query head and the device time per decode step."""
    import torch

    import workloads as WL
    import __graft_entry__
    __graft_entry__.build()
    import lsh_sampled_sparse_centered_gb300 as mp

    dev = torch.device("cuda", 0)
    base = WL.WORKLOADS[args.workload].replace(layers=1, steps=8)
    stream = torch.cuda.Stream(device=dev)
    for K, L in SWEEP_GRID:
        for centering in (True, False):
            wl = base.replace(K=K, L=L, name=f"{base.name}-1L-K{K}-L{L}")
            with torch.cuda.stream(stream):
                job = Job(mp, wl, dev, stream)
                job.cfg.no_centering = 0 if centering else 1
            stats = torch.zeros(3, dtype=torch.int64, device=dev)
            job.hook = lambda s, n: stats.add_(decode_state_stats(job, torch))
            with torch.cuda.stream(stream):
                job.run()  # warm-up, and the sampled-set statistics
            torch.cuda.synchronize()
            assert mp.mp_get_status(job.tables, stream=job.sp) == 0
            job.hook = None
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            with torch.cuda.stream(stream):
                ev[0].record(stream)
                job.build()
                ev[1].record(stream)
                job.decode_steps()
                ev[2].record(stream)
            torch.cuda.synchronize()
            entries, sampled, _ = [int(v) for v in stats.cpu()]
            Q = wl.layers * wl.batch * wl.q_heads
            region = sum(max(0, wl.seq_len(t) - wl.window - min(wl.n_sink, wl.seq_len(t))) for t in range(wl.steps)) * Q
            x = 0.5 ** K
            print(json.dumps({
                "sweep": "budget", "workload": wl.name, "K": K, "L": L, "centering": centering,
                "sampled_fraction": sampled / region, "closed_form_fraction_isotropic":
                    1 - (1 - x) ** L - L * x * (1 - x) ** (L - 1),
                "list_entries_per_query": entries / (Q * wl.steps),
                "build_ms": ev[0].elapsed_time(ev[1]),
                "us_per_decode_step": 1e3 * ev[1].elapsed_time(ev[2]) / wl.steps}), flush=True)
            del job
            torch.cuda.empty_cache()


def main():
    args = parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    rank, world, local = dist_setup(True)
    line, job = run_ours(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import workloads as WL
        v, sec, desc = oracle_sample(WL.WORKLOADS[args.workload], decode_steps=4)
        line["cpu_baseline"] = {"value": v, "unit": "queries/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": desc, "seconds": sec}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
