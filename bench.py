#!/usr/bin/env python
"""Benchmark of the compressed ring allreduce on one GB300 (N simulated ranks).

Default workload (the one the metric is quoted on): block-FP8 compressed ring
allreduce of one 25 MiB DDP-style fp16 gradient bucket, N = 8 simulated ranks,
T = 13,107,200 fp16 elements per rank drawn N(0, 1e-3^2) from seed 1, fp32
accumulation, fp16 output.  One step = one rra_ring_allreduce call (the whole
hot path: chunking, reduce-scatter hops with fused decode + fp32 add + encode,
owner finalise, allgather hops with decode + output cast, byte counters).

Metric: algbw = T * sizeof(input element) / step time (per-rank logical
payload, as nccl-tests count it), reported whole-job (replicas x payload /
max-over-ranks time), plus the dominant kernel's roofline fraction against
the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--impl rra|reference]

--impl reference times the CPU oracle on the machine's host cores instead (a
bounded sample of the same workload per step).  With torchrun (N > 1) every
rank runs an independent replica on its own GPU ("replicas only": the method
simulates all ranks inside one GPU, so nothing is sharded across GPUs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "compressed ring-allreduce algbw GB/s on 1 GB300 (N sim ranks), % of HBM peak"
FALLBACK_HBM_GBS = 6800.0
CONFIG_NAMES = ("bfp8_bucket", "lossless_n4", "sparse_n16", "diloco_n8", "bfp8_allgather",
                "bfp8_broadcast")


# ---------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x: float) -> float:
    """Largest value over the ranks (the slowest replica's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, payload_bytes: int, ms_per_step_max: float) -> float:
    """Whole-job algbw: every replica moves its own payload per step; the job
    takes as long as its slowest replica."""
    return world * payload_bytes / (ms_per_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of this process's GPU during the timed region."""

    def __init__(self, device_index: int, period_ms: int = 50):
        self.path = tempfile.mktemp(prefix="rra_clocks_", suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", str(period_ms)],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                    power.append(float(p[3]))
                except ValueError:
                    continue
                for nm, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ---------------------------------------------------------------- peaks / profiles

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, an earlier GB300 copy measurement)"


# The files each workload's ring kernel is compiled from (host-side launch
# code excluded): a change to another codec's files leaves its summary valid.
RING_KERNEL_COMMON = ("ring_kernel.cuh", "bfp_group.cuh", "rra_device.cuh", "rra_kernels.h")
RING_KERNEL_SOURCES = {
    "bfp8_bucket": ("ring_bfp8.cu", "ring_bfp8_ef.cu"),
    "diloco_n8": ("ring_bfp4.cu", "ring_bfp4_ef.cu"),
    "sparse_n16": ("ring_sparse_chunk.cu", "wire_sparse.cuh"),
    "bfp8_allgather": ("ring_bfp8.cu",),
    "bfp8_broadcast": ("coll_kernels.cu",),
    "lossless_n4": ("ring_none.cu",),
}


def kernel_sources_sha(config: str = "bfp8_bucket") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ring_allreduce_compressed_gb300", "csrc")
    for name in sorted(RING_KERNEL_COMMON + RING_KERNEL_SOURCES[config]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# the kernel each workload times (the ring kernel unless named here)
KERNEL_OF = {"bfp8_broadcast": "broadcast_bfp_kernel"}


def traffic_from_profile(config: str):
    """DRAM bytes per launch of the workload's kernel from the committed ncu
    summary for it, or None when no summary exists or the kernel sources
    changed since it was taken."""
    kernel = KERNEL_OF.get(config, "ring_kernel")
    path = os.path.join(ROOT, "profiles", f"{kernel}_{config}.md")
    try:
        text = open(path).read()
    except OSError:
        return None, "no ncu summary"
    m_sha = re.search(r"kernel_sources_sha:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_sha or not m_tr:
        return None, "summary incomplete"
    if m_sha.group(1) != kernel_sources_sha(config):
        return None, "kernel changed since the ncu capture"
    return int(m_tr.group(1)), os.path.relpath(path, ROOT)


# ---------------------------------------------------------------- workloads

class Workload:
    """One of the configurations, resident in HBM.  With use_lib=False (the
    reference arm) only the inputs are drawn; the CUDA library is not used."""

    def __init__(self, name: str, device="cuda", use_lib: bool = True, scale: int = 1,
                 ef: bool = False):
        rra = None
        if use_lib:
            import ring_allreduce_compressed_gb300 as rra
        self.name = name
        self.base = None
        self.prev = None
        self.codec = None
        c = W.CONFIGS[name]
        # scale > 1: the same workload with T / scale elements per rank (a
        # small case for profiler captures; never a bench line of the metric)
        self.N, self.T = c["N"], c["T"] // scale
        if name == "bfp8_bucket":
            self.inputs = W.bfp_bucket(self.N, self.T, seed=c["seed"], device=device)
            self.out_dtype = torch.float16
            self.codec_name = "bfp8"
            self.desc = ("block-FP8 compressed ring allreduce of one 25 MiB fp16 DDP bucket: "
                         "N=8 simulated ranks x 13,107,200 fp16, N(0,1e-3^2) seed 1, "
                         "128-element blocks, fp32 accumulation, fp16 output")
        elif name == "bfp8_allgather":
            self.inputs = W.bfp_bucket(self.N, self.T, seed=c["seed"], device=device)
            self.out_dtype = torch.float16
            self.codec_name = "bfp8-allgather"
            self.desc = ("block-FP8 compressed allgather, in place (parameters gathered as in "
                         "ZeRO/FSDP): N=8 simulated ranks x 13,107,200 fp16, N(0,1e-3^2) seed 1; "
                         "each owner encodes its chunk once, every rank stores the decoded "
                         "chunks.  Decoding then re-encoding gives the same codes, so every "
                         "step does the same work on the buffers the previous step left")
        elif name == "bfp8_broadcast":
            self.inputs = W.bfp_bucket(self.N, self.T, seed=c["seed"], device=device)
            self.out_dtype = torch.float16
            self.codec_name = "bfp8-broadcast"
            self.desc = ("block-FP8 compressed broadcast from rank 0 over the binomial tree, in "
                         "place: N=8 simulated ranks x 13,107,200 fp16, N(0,1e-3^2) seed 1; the "
                         "root encodes once, every rank stores the decoded buffer.  Decoding "
                         "then re-encoding gives the same codes, so every step does the same "
                         "work")
        elif name == "lossless_n4":
            self.inputs = W.lossless(self.N, self.T, seed=c["seed"], device=device)
            self.out_dtype = torch.float32
            self.codec_name = "none"
            self.desc = "lossless fp32 ring allreduce, N=4 x 4096 fp32, N(0,1) seed 0"
        elif name == "sparse_n16":
            self.inputs = W.sparse(self.N, self.T, seed=c["seed"], device=device)
            self.out_dtype = torch.float32
            self.codec_name = "sparse"
            self.desc = ("sparse-format ring allreduce: N=16 x 64 Mi bf16, zero w.p. 0.6 else "
                         "N(0,0.02^2), seed 2, threshold 0.5, one message per ring chunk and "
                         "hop (values + int32 indices, or dense fp32), fp32 out")
        elif name == "diloco_n8":
            self.inputs, self.prev = W.diloco(self.N, self.T, seed=c["seed"], device=device)
            self.out_dtype = torch.float32
            self.codec_name = "diff+bfp4"
            self.desc = ("DiLoCo outer-step pseudo-gradient: N=8 x 10^9 fp32 deltas, "
                         "difference against the previous round, block-FP4, averaged by 1/N, "
                         "previous result (lossless mean of prev) added back; seed 3")
        else:
            raise ValueError(name)
        self.in_dtype = self.inputs[0].dtype
        # error feedback (BFP workloads): one fp32 residual per rank, from zero
        self.ef = ef
        if ef:
            if self.codec_name not in ("bfp8", "diff+bfp4"):
                raise SystemExit(f"--ef needs a BFP workload, not {name}")
            self.residual = [torch.zeros(self.T, dtype=torch.float32, device=device)
                             for _ in range(self.N)]
            self.desc += "; with error feedback (an fp32 residual per rank, read and written)"
        if use_lib:
            self.comm = rra.Comm(self.N, self.T, self.in_dtype)
            if name in ("bfp8_bucket", "bfp8_allgather", "bfp8_broadcast"):
                self.codec = rra.Codec("bfp", bits=8)
            elif name == "sparse_n16":
                self.codec = rra.Codec("sparse", sparsity_threshold=0.5)
            elif name == "diloco_n8":
                # previous round's result: lossless mean of prev (setup, untimed);
                # reduce-scatter writes chunk r of each output, so one buffer holds it
                self.base = torch.empty(self.T, dtype=torch.float32, device=device)
                self.comm.reduce_scatter(self.prev, [self.base] * self.N,
                                         rra.Codec("none", average=True))
                torch.cuda.synchronize()
                self.codec = rra.Codec("bfp", bits=4, diff_prev=self.prev, diff_base=self.base,
                                       average=True)
            if ef:
                self.codec.residual = self.residual
            self.outputs = [torch.empty(self.T, dtype=self.out_dtype, device=device)
                            for _ in range(self.N)]
        ies = self.inputs[0].element_size()
        oes = torch.empty(0, dtype=self.out_dtype).element_size()
        self.payload = self.T * ies  # per-rank logical payload (algbw numerator)
        diff = self.prev is not None
        extra_in = self.T * 4 * self.N if diff else 0  # the prev streams
        base = self.T * 4 if diff else 0
        self.compulsory = (self.N * self.T * (ies + oes) + extra_in + base +
                           (self.N * self.T * 8 if ef else 0))  # residual read + write
        if name == "bfp8_allgather":  # each rank reads its own chunk, writes its buffer
            n = -(-self.T // self.N)
            self.compulsory = self.N * (n * ies + self.T * oes)
        if name == "bfp8_broadcast":  # the root reads its buffer, every rank writes its own
            self.compulsory = self.T * ies + self.N * self.T * oes
        # algorithmic bytes of one step: the compulsory traffic, plus, for the
        # per-chunk sparse ring, the count pass that reads every input once
        # more before the ring starts (one step = two kernels)
        self.alg_bytes = self.compulsory
        self.kernels = "ring_kernel"
        self.launches_per_step = 1
        if name == "sparse_n16":
            self.alg_bytes += self.N * self.T * ies
            self.kernels = "sparse_chunk_count_kernel + ring_kernel"
            self.launches_per_step = 2

    def step(self, stream=None):
        if self.name == "bfp8_allgather":
            self.comm.allgather(self.inputs, self.codec, stream=stream)
            return
        if self.name == "bfp8_broadcast":
            self.comm.broadcast(self.inputs, 0, self.codec, stream=stream)
            return
        self.comm.ring_allreduce(self.inputs, self.outputs, self.codec, stream=stream)

    def l2_note(self):
        mb = self.compulsory / 1e6
        return (f"inputs+outputs {mb:.0f} MB per step > 129 MB L2: no flush between steps"
                if mb > 129 else f"working set {mb:.2f} MB fits in L2 (latency-bound case)")


# ---------------------------------------------------------------- CPU baseline (oracle)

def oracle_sample_ring(wl_host, N, T, codec_name, slices_per_chunk, in_dt, out_dt, extra,
                       ef=False, first_slice=0):
    """Run the oracle on `slices_per_chunk` 256-element slices of every chunk,
    from slice `first_slice` on (an exact sub-problem: slices are
    independent).  Returns (seconds, payload bytes per rank of the sample)."""
    import oracle as O
    n = T // N
    lo = min(n, first_slice * 256)
    m = min(n - lo, slices_per_chunk * 256)
    idx = np.concatenate([np.arange(c * n + lo, c * n + lo + m) for c in range(N)])
    xs = [np.ascontiguousarray(x[idx]) for x in wl_host]
    kw = {}
    if codec_name == "bfp8":
        kw = dict(codec="bfp", bits=8)
    elif codec_name == "sparse":
        kw = dict(codec="sparse", threshold=0.5)
    elif codec_name == "diff+bfp4":
        kw = dict(codec="bfp", bits=4, diff_prev=[np.ascontiguousarray(p[idx]) for p in extra[0]],
                  diff_base=np.ascontiguousarray(extra[1][idx]), average=True)
    if ef:
        kw["residual"] = [np.zeros(xs[0].size, np.float32) for _ in range(N)]
    t0 = time.perf_counter()
    if codec_name == "bfp8-allgather":
        O.allgather_codec(xs, in_dt, "bfp", 8)
    elif codec_name == "bfp8-broadcast":
        O.broadcast_codec(xs, in_dt, 0, 8)
    else:
        O.ring(xs, in_dt, out_dt, **kw)
    dt = time.perf_counter() - t0
    return dt, N * m * xs[0].itemsize


def host_copy(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


DT_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def cpu_baseline(wl: Workload, budget_s: float = 20.0):
    """The oracle, as it stands, single-threaded on a host core, on a bounded
    sample of the workload sized to about `budget_s` seconds."""
    n = wl.T // wl.N
    hosts = [host_copy(x) for x in wl.inputs]
    extra = None
    if wl.prev is not None:
        extra = ([host_copy(p) for p in wl.prev], host_copy(wl.base))
    # calibrate on a small sample, then size the measured one
    s0 = max(1, min(n // 256, 16))
    dt0, _ = oracle_sample_ring(hosts, wl.N, wl.T, wl.codec_name, s0, DT_NAME[wl.in_dtype],
                                DT_NAME[wl.out_dtype], extra, wl.ef)
    slices = max(1, min(-(-n // 256), int(s0 * budget_s / max(dt0, 1e-6))))
    dt, payload = oracle_sample_ring(hosts, wl.N, wl.T, wl.codec_name, slices,
                                     DT_NAME[wl.in_dtype], DT_NAME[wl.out_dtype], extra, wl.ef)
    full = slices * 256 >= n
    # the same sample on every host core: contiguous groups of slices, each an
    # exact sub-problem, one oracle call per thread (the C oracle runs outside
    # the interpreter lock)
    threads = max(1, min(os.cpu_count() or 1, slices))
    per = -(-slices // threads)
    groups = [(g0, min(per, slices - g0)) for g0 in range(0, slices, per)]

    def one(group):
        return oracle_sample_ring(hosts, wl.N, wl.T, wl.codec_name, group[1],
                                  DT_NAME[wl.in_dtype], DT_NAME[wl.out_dtype], extra, wl.ef,
                                  first_slice=group[0])[1]

    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=len(groups)) as ex:
        t0 = time.perf_counter()
        moved = sum(ex.map(one, groups))
        dt_all = time.perf_counter() - t0
    assert moved == payload
    return {"value": payload / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": dt,
            "all_cores": {"value": payload / dt_all / 1e9, "cores": len(groups),
                          "seconds": dt_all, "split": "contiguous slice groups, one thread each"},
            "sample": ("the full workload" if full else
                       f"first {slices} of {-(-n // 256)} 256-element slices of every chunk "
                       f"({slices * 256 * wl.N} of {wl.T} elements per rank; " +
                       ("run as its own N-rank problem: one sparse message per chunk of the "
                        "sample, so the same work per element as the whole)"
                        if wl.codec_name == "sparse" else
                        "slices are independent, so the sample is an exact sub-problem)"))}


# ---------------------------------------------------------------- arms

def run_rra(args, world, rank, local):
    import ring_allreduce_compressed_gb300 as rra
    rra.build()
    wl = Workload(args.config, scale=args.scale, ef=args.ef)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    sent, recv = wl.comm.get_bytes()
    assert wl.comm.status() == rra.RRA_OK

    K = args.steps
    if K is None:
        # about one second of timed work: the step time from a few more
        # untimed steps, the same K on every rank
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            wl.step()
        e1.record(stream)
        torch.cuda.synchronize()
        t_step = max_over_ranks(world, e0.elapsed_time(e1) / 3) * 1e-3
        K = int(max(20, min(10000, round(1.0 / max(t_step, 1e-7)))))
        args.steps = K
    # The K timed steps are one CUDA graph of K back-to-back calls, so the
    # host's per-call cost (argument marshalling, launch) stays outside the
    # device timeline; the same calls made eagerly, one event pair per step,
    # are timed afterwards for comparison.
    graph = None
    if not args.eager:
        try:
            graph = torch.cuda.CUDAGraph()
            gs = torch.cuda.Stream()
            gs.wait_stream(stream)
            with torch.cuda.stream(gs):
                with torch.cuda.graph(graph, stream=gs):
                    for _ in range(K):
                        wl.step()
            stream.wait_stream(gs)
            graph.replay()  # one untimed replay: the graph's own warm-up
            torch.cuda.synchronize()
            assert wl.comm.status() == rra.RRA_OK
        except RuntimeError:
            graph = None
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    time.sleep(0.15)
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for k in range(K):
            wl.step()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    status = wl.comm.status()
    total_ms = t_start.elapsed_time(t_end)
    ms_step = max_over_ranks(world, total_ms / K)
    # per-step device time (the step's kernels back to back): from the graph,
    # the timed region over K; eagerly, one event pair per step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for k in range(K):
        ev[k][0].record(stream)
        wl.step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    eager = {"ms_mean": statistics.mean(step_ms), "ms_median": statistics.median(step_ms),
             "note": "the same steps launched one by one from Python, one event pair each "
                     "(includes any wait for the host's launch)"}
    graph_used = graph is not None
    if graph_used:
        kern_ms = ms_step
        kern_ms_median = ms_step
        del graph
    else:
        kern_ms = max_over_ranks(world, sum(step_ms) / K)
        kern_ms_median = max_over_ranks(world, statistics.median(step_ms))

    value = whole_job_gbs(world, wl.payload, ms_step)

    # latency-bound workloads: one call's device time without the host's
    # launch cost, from CUDA-graph replays of back-to-back calls (outside the
    # timed region above)
    latency = None
    if wl.compulsory <= 2 ** 26:
        calls, reps = 20, 20
        graph = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            with torch.cuda.graph(graph, stream=gs):
                for _ in range(calls):
                    wl.step()
        stream.wait_stream(gs)
        graph.replay()
        torch.cuda.synchronize()
        per_call = []
        for _ in range(reps):
            a_ev = torch.cuda.Event(enable_timing=True)
            b_ev = torch.cuda.Event(enable_timing=True)
            a_ev.record()
            graph.replay()
            b_ev.record()
            b_ev.synchronize()
            per_call.append(a_ev.elapsed_time(b_ev) * 1e3 / calls)
        del graph
        assert wl.comm.status() == rra.RRA_OK
        latency = {"graph_us_per_call": statistics.median(per_call), "calls_per_graph": calls,
                   "replays": reps, "note": "median over CUDA-graph replays of back-to-back "
                   "calls; excludes the host launch cost that the per-step events include"}
    peak, peak_src = hbm_peak()
    achieved = wl.alg_bytes / (kern_ms * 1e-3) / 1e9
    traffic, traffic_src = traffic_from_profile(args.config)

    # end to end: pinned host inputs in, results out, through the public API.
    # Two buffer sets pipeline the steps as a training loop would: step k+1's
    # inputs go up (one copy stream) while step k's results come down (the
    # other), and the allreduce of a step starts once its inputs are in.
    # Every step still copies all of its inputs in and all of its result out
    # inside the timed region.
    e2e = None
    if args.config in ("bfp8_bucket", "lossless_n4") and args.e2e_steps > 0:
        h_in = [[torch.empty(wl.T, dtype=wl.in_dtype, pin_memory=True) for _ in range(wl.N)]
                for _ in range(2)]
        for hs in h_in:
            for h, d in zip(hs, wl.inputs):
                h.copy_(d)
        h_out = [[torch.empty(wl.T, dtype=wl.out_dtype, pin_memory=True) for _ in range(wl.N)]
                 for _ in range(2)]
        d_in = [[torch.empty_like(x) for x in wl.inputs] for _ in range(2)]
        d_out = [[torch.empty_like(x) for x in wl.outputs] for _ in range(2)]
        s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set b are on the device
        ev_red = [torch.cuda.Event() for _ in range(2)]   # allreduce of set b done
        ev_out = [torch.cuda.Event() for _ in range(2)]   # results of set b are on the host
        for b in range(2):  # every set starts free
            ev_red[b].record(stream)
            ev_out[b].record(stream)
        step_no = [0]

        def e2e_step():
            b = step_no[0] & 1
            step_no[0] += 1
            s_up.wait_event(ev_red[b])  # the previous allreduce of this set has read its inputs
            with torch.cuda.stream(s_up):
                for h, d in zip(h_in[b], d_in[b]):
                    d.copy_(h, non_blocking=True)
                ev_in[b].record(s_up)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])  # this set's previous results are on the host
            wl.comm.ring_allreduce(d_in[b], d_out[b], wl.codec, stream=stream)
            ev_red[b].record(stream)
            s_down.wait_event(ev_red[b])
            with torch.cuda.stream(s_down):
                for h, d in zip(h_out[b], d_out[b]):
                    h.copy_(d, non_blocking=True)
                ev_out[b].record(s_down)

        for _ in range(4):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_up.wait_stream(stream)  # no copy of the timed steps starts before the clock
        s_down.wait_stream(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        stream.wait_stream(s_up)
        stream.wait_stream(s_down)
        b_.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(world, a.elapsed_time(b_) / args.e2e_steps)
        last = (step_no[0] - 1) & 1
        vt = torch.int16 if wl.out_dtype != torch.float32 else torch.int32
        ok = all(torch.equal(h_out[last][r].view(vt), wl.outputs[r].cpu().view(vt))
                 for r in range(wl.N))
        e2e = {"value": whole_job_gbs(world, wl.payload, e2e_ms), "unit": "GB/s",
               "ms_per_step": e2e_ms, "steps": args.e2e_steps,
               "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in h_in[0]),
               "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in h_out[0]),
               "pipelined": "two buffer sets; step k+1's inputs go up while step k's "
                            "results come down",
               "result_matches_device_run": ok}

    others = None
    if args.config == CONFIG_NAMES[0] and args.scale == 1 and not args.ef and args.other_configs:
        others = run_other_configs(world, local, args.other_configs)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, budget_s=args.cpu_budget)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.config}: {wl.desc}" + (f" [T / {args.scale}]" if getattr(args, "scale", 1) > 1 else ""), "N": wl.N, "T": wl.T,
                   "in_dtype": DT_NAME[wl.in_dtype], "out_dtype": DT_NAME[wl.out_dtype],
                   "codec": wl.codec_name, "parallelism": f"replicas x{world}",
                   "l2": wl.l2_note()},
        "hbm_pct": 100.0 * wl.compulsory / (kern_ms * 1e-3) / 1e9 / peak,
        "busbw": value * 2 * (wl.N - 1) / wl.N,
        "bytes_sent_per_rank": sent[0],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": KERNEL_OF.get(args.config, wl.kernels), "kernel_ms": kern_ms,
                     "bytes_per_launch": wl.alg_bytes,
                     "kernel_ms_median": kern_ms_median,
                     "timing": ("CUDA graph of the K timed calls: kernel_ms = timed region / K"
                                if graph_used else "eager: one event pair per step"),
                     "frac_compulsory": wl.compulsory / (kern_ms * 1e-3) / 1e9 / peak,
                     # the slot-materialised model: every wire byte written to a
                     # slot and read back once, beside the compulsory bytes (the
                     # slots live in shared memory here, so this can exceed 1)
                     "bytes_alg_slots": wl.compulsory + 2 * sum(sent),
                     "frac_alg_slots": (wl.compulsory + 2 * sum(sent)) / (kern_ms * 1e-3) / 1e9 / peak,
                     "bytes_model": ("compulsory: N*T*(in+out) (+ diff prev and base)" +
                                     ("; + N*T*in for the count pass" if wl.alg_bytes > wl.compulsory
                                      else "")),
                     "peak_source": peak_src, "traffic_source": traffic_src},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "latency": latency,
        "eager": eager,
        "gpu_launches": K * wl.launches_per_step,
        "other_configs": others,
        "clocks": clk,
        "status": rra.status_string(status),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
        if args.jsonl:
            with open(args.jsonl, "a") as f:
                f.write(json.dumps(line) + "\n")


def run_other_configs(world: int, local: int, seconds: float):
    """Every other workload of the metric, each timed like the headline line:
    3 untimed steps, then K back-to-back steps as one CUDA graph (K for about
    `seconds` of timed work), one untimed replay and one timed replay, with
    the GPU's clocks sampled over the timed replays.  The workloads are built
    and freed one at a time (the DiLoCo one holds about 100 GB)."""
    import ring_allreduce_compressed_gb300 as rra
    peak, _ = hbm_peak()
    res = {}
    for name in CONFIG_NAMES[1:]:
        wl = Workload(name)
        stream = torch.cuda.current_stream()
        for _ in range(3):
            wl.step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            wl.step()
        e1.record(stream)
        torch.cuda.synchronize()
        t_step = max_over_ranks(world, e0.elapsed_time(e1) / 3) * 1e-3
        K = int(max(10, min(2000, round(seconds / max(t_step, 1e-7)))))
        graph = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            with torch.cuda.graph(graph, stream=gs):
                for _ in range(K):
                    wl.step()
        stream.wait_stream(gs)
        graph.replay()
        torch.cuda.synchronize()
        clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
        time.sleep(0.15)
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        clk = clocks.stop()
        ms = max_over_ranks(world, a.elapsed_time(b) / K)
        status = wl.comm.status()
        res[name] = {
            "workload": wl.desc, "N": wl.N, "T": wl.T, "codec": wl.codec_name,
            "value": whole_job_gbs(world, wl.payload, ms), "unit": "GB/s",
            "ms_per_step": ms, "steps": K, "kernels": KERNEL_OF.get(name, wl.kernels),
            "bytes_per_step": wl.alg_bytes,
            "frac": wl.alg_bytes / (ms * 1e-3) / 1e9 / peak,
            "frac_compulsory": wl.compulsory / (ms * 1e-3) / 1e9 / peak,
            "l2": wl.l2_note(), "clocks": clk, "status": rra.status_string(status)}
        del graph, wl
        torch.cuda.empty_cache()
    return res


def run_reference(args, world, rank):
    """The oracle timed on the host cores, one bounded sample per step."""
    if rank != 0:
        return
    if args.steps is None:
        args.steps = 20
    wl = Workload(args.config, use_lib=False, ef=args.ef)
    n = wl.T // wl.N
    hosts = [host_copy(x) for x in wl.inputs]
    extra = None
    if wl.prev is not None:
        import oracle as O
        prev_h = [host_copy(p) for p in wl.prev]
        # the previous result is the lossless mean of prev; the oracle computes
        # it on the positions the samples use (the first slices of each chunk)
        m = min(n, 1 << 20)
        idx = np.concatenate([np.arange(c * n, c * n + m) for c in range(wl.N)])
        mean = O.ring([np.ascontiguousarray(p[idx]) for p in prev_h], average=True)[0][0]
        base = np.zeros(wl.T, np.float32)
        base[idx] = mean
        extra = (prev_h, base)
    s0 = max(1, min(n // 256, 4))
    dt0, _ = oracle_sample_ring(hosts, wl.N, wl.T, wl.codec_name, s0, DT_NAME[wl.in_dtype],
                                DT_NAME[wl.out_dtype], extra, wl.ef)
    per_step = args.ref_budget / max(1, args.steps + args.warmup)
    slices = max(1, min(-(-n // 256), int(s0 * per_step / max(dt0, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample_ring(hosts, wl.N, wl.T, wl.codec_name, slices, DT_NAME[wl.in_dtype],
                           DT_NAME[wl.out_dtype], extra, wl.ef)
    tot, pay = 0.0, 0
    for _ in range(args.steps):
        dt, p = oracle_sample_ring(hosts, wl.N, wl.T, wl.codec_name, slices, DT_NAME[wl.in_dtype],
                                   DT_NAME[wl.out_dtype], extra, wl.ef)
        tot += dt
        pay += p
    value = pay / tot / 1e9
    sample = (f"first {slices} of {-(-n // 256)} 256-element slices of every chunk per step "
              f"({slices * 256 * wl.N} of {wl.T} elements per rank)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{args.config}: {wl.desc}", "N": wl.N, "T": wl.T,
                       "in_dtype": DT_NAME[wl.in_dtype], "out_dtype": DT_NAME[wl.out_dtype],
                       "codec": wl.codec_name, "parallelism": f"replicas x{world}"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ring vs tree sweep

def run_codecs(args, world, rank):
    """The standalone codec entry points on 2^28 elements, each timed on the
    device (time_op: 10 calls in a CUDA graph after 3 warm-ups) against its
    compulsory bytes: the input read once and the output written once (the
    sparse encoder reads its input twice: a count pass and an emit pass)."""
    import ring_allreduce_compressed_gb300 as rra
    rra.build()
    if rank != 0:
        return
    peak, peak_src = hbm_peak()
    n = args.codec_n
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    x16 = (torch.randn(n, generator=g, device="cuda") * 1e-3).half()
    xs = torch.randn(n, generator=g, device="cuda")
    xs[torch.rand(n, generator=g, device="cuda") < 0.6] = 0.0
    xb = xs.bfloat16()
    del xs
    nb = -(-n // 128)
    exps = torch.empty(nb, dtype=torch.int8, device="cuda")
    mants = torch.empty(n, dtype=torch.uint8, device="cuda")
    out32 = torch.zeros(n, device="cuda")
    hdr = torch.empty(2, dtype=torch.int32, device="cuda")
    vals = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(n, dtype=torch.int32, device="cuda")
    rra.sparse_encode(xb, 0.5, hdr, vals, idx)
    # a dense message (45 % zeros is below the threshold) for the dense path
    # of the accumulating decoder
    xd = torch.randn(n, generator=g, device="cuda")
    xd[torch.rand(n, generator=g, device="cuda") < 0.45] = 0.0
    xd = xd.bfloat16()
    hdr_d = torch.empty(2, dtype=torch.int32, device="cuda")
    vals_d = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    rra.sparse_encode(xd, 0.5, hdr_d, vals_d, idx)
    del xd
    torch.cuda.synchronize()
    assert int(hdr_d[0]) == 0
    rra.sparse_encode(xb, 0.5, hdr, vals, idx)  # idx again holds xb's indices
    torch.cuda.synchronize()
    fmt, nnz = [int(v) for v in hdr.cpu()]
    cur = torch.randn(n, generator=g, device="cuda")
    prev = torch.randn(n, generator=g, device="cuda")
    diff = torch.empty(n, device="cuda")

    def bfp_bytes(bits):
        return nb + (n if bits == 8 else n // 2)

    cases = [
        ("bfp8_encode f16", lambda: rra.bfp_encode(x16, 8, exps, mants), 2 * n + bfp_bytes(8)),
        ("bfp4_encode f16", lambda: rra.bfp_encode(x16, 4, exps, mants), 2 * n + bfp_bytes(4)),
        ("bfp8_decode -> f32", lambda: rra.bfp_decode(exps, mants, n, 8, out32), bfp_bytes(8) + 4 * n),
        ("bfp8_decode accumulate f32", lambda: rra.bfp_decode(exps, mants, n, 8, out32, True),
         bfp_bytes(8) + 8 * n),
        ("sparse_encode bf16 (60 % zeros)", lambda: rra.sparse_encode(xb, 0.5, hdr, vals, idx),
         2 * n + (6 * nnz if fmt else 2 * n)),
        ("sparse_decode -> f32", lambda: rra.sparse_decode(hdr, vals, idx, n, out32),
         (6 * nnz if fmt else 2 * n) + 4 * n),
        # the listed values and indices read, acc read and written at each
        ("sparse_decode accumulate f32", lambda: rra.sparse_decode(hdr, vals, idx, n, out32, True),
         14 * nnz if fmt else 10 * n),
        ("sparse_decode accumulate f32, dense message",
         lambda: rra.sparse_decode(hdr_d, vals_d, idx, n, out32, True), 10 * n,
         {"sparse_format": "dense", "nnz": n}),
        ("diff_encode f32", lambda: rra.diff_encode(cur, prev, diff), 12 * n),
    ]
    out = []
    for name, fn, nbytes, *extra in cases:
        us, how = time_op(fn, args.op_warmup, args.op_reps)
        line = {"codec_bench": True, "op": name, "n": n, "us": us, "timing": how, "bytes": nbytes,
                "gbs": nbytes / (us * 1e-6) / 1e9,
                "hbm_frac": nbytes / (us * 1e-6) / 1e9 / peak, "peak_source": peak_src,
                "sparse_format": "sparse" if fmt else "dense", "nnz": nnz}
        line.update(*extra)
        out.append(line)
        print(json.dumps(line), flush=True)
    if args.jsonl:
        with open(args.jsonl, "a") as f:
            for line in out:
                f.write(json.dumps(line) + "\n")


def time_op(fn, warmup: int, reps: int):
    """Device time of one call of fn in microseconds, and how it was taken:
    the reps calls captured back to back in a CUDA graph on a side stream
    (after the warm-up calls on that stream), the graph replayed once as its
    own warm-up and once timed; ops that cannot be captured (a synchronous
    read-back) are timed call by call with CUDA events (median)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warmup):
            fn()
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for _ in range(reps):
                    fn()
        g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        return a.elapsed_time(b) * 1e3 / reps, "CUDA graph of the timed calls"
    except RuntimeError:
        torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    return statistics.median(times), "CUDA events per call (median)"


def run_kernels(args, world, rank):
    """One op per library kernel that the ring workloads do not cover -- the
    plain allgather, broadcast and tree allreduce, and the codec statistics --
    on N=8 ranks of --kernels-T fp32 elements (default 16 Mi: 512 MB in all,
    above the 129 MB L2), each called --op-warmup times untimed and then
    --op-reps times, timed by time_op (a CUDA graph of the calls; the codec
    statistics, which read their counts back to the host, call by call), against
    its algorithmic bytes.  Also the command the ncu summaries of these kernels are captured
    from."""
    import ring_allreduce_compressed_gb300 as rra
    rra.build()
    if rank != 0:
        return
    peak, peak_src = hbm_peak()
    N, T = 8, args.kernels_T
    bufs = W.uniform(N, T, seed=4)
    comm = rra.Comm(N, T)
    n = -(-T // N)
    cases = [
        # each rank reads its own chunk once and writes the N-1 others
        ("allgather_kernel", lambda: comm.allgather(bufs), 4 * N * n + 4 * (N - 1) * n * N),
        # the root's buffer read once, every other buffer written once
        ("broadcast_kernel", lambda: comm.broadcast(bufs, root=0), 4 * T + 4 * (N - 1) * T),
        # every buffer read and written once
        ("tree_kernel", lambda: comm.tree_allreduce(bufs), 8 * N * T),
        # every buffer read once
        ("codec_stats_kernel", lambda: comm.codec_stats(bufs), 4 * N * T),
    ]
    for name, fn, nbytes, *extra in cases:
        us, how = time_op(fn, args.op_warmup, args.op_reps)
        assert comm.status() == rra.RRA_OK
        line = {"kernel_bench": True, "kernel": name, "N": N, "T": T, "us": us, "timing": how,
                "bytes": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9,
                "hbm_frac": nbytes / (us * 1e-6) / 1e9 / peak, "peak_source": peak_src}
        print(json.dumps(line), flush=True)
    comm.close()


def run_sweep(args, world, rank):
    """Lossless fp32 ring vs tree allreduce over T = 256 * 4^k elements
    (1 KiB .. 1 GiB per rank) and N in {2, 4, 8, 16, 64}, in place, values
    U(-1,1) from seed 4 (re-seeded per case).  One JSON line per (N, T, op)
    and a summary line per N with the measured crossover and the alpha-beta
    link model fed by the byte counters."""
    import ring_allreduce_compressed_gb300 as rra
    rra.build()
    Ns = [int(x) for x in args.sweep_n.split(",")]
    Ts = [256 * 4 ** k for k in range(args.sweep_kmax + 1)]
    alpha_us, beta_gbs = args.alpha_us, args.beta_gbs
    peak, _ = hbm_peak()
    out = []
    for N in Ns:
        rows = []
        for case, T in enumerate(Ts):
            free, _ = torch.cuda.mem_get_info()
            if N * T * 4 * 1.1 + 2 ** 30 > free:
                continue
            bufs = W.uniform(N, T, seed=4 + case)
            comm = rra.Comm(N, T)
            res = {}
            for op in ("ring", "tree"):
                fn = (lambda: comm.ring_allreduce(bufs, bufs)) if op == "ring" else \
                    (lambda: comm.tree_allreduce(bufs))
                for _ in range(5):
                    fn()
                torch.cuda.synchronize()
                sent, recv = comm.get_bytes()
                assert comm.status() == rra.RRA_OK
                reps = 20 if N * T * 4 < 2 ** 33 else 5
                times = []
                if N * T * 4 <= 2 ** 26:
                    # small messages: replay a CUDA graph of 20 back-to-back calls
                    # so that the host's launch cost is not part of the time
                    graph = torch.cuda.CUDAGraph()
                    s = torch.cuda.Stream()
                    s.wait_stream(torch.cuda.current_stream())
                    with torch.cuda.stream(s):
                        with torch.cuda.graph(graph, stream=s):
                            for _ in range(20):
                                fn()
                    torch.cuda.current_stream().wait_stream(s)
                    graph.replay()
                    torch.cuda.synchronize()
                    for _ in range(reps):
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        a.record()
                        graph.replay()
                        b.record()
                        b.synchronize()
                        times.append(a.elapsed_time(b) * 1e3 / 20)
                    del graph
                    assert comm.status() == rra.RRA_OK
                else:
                    for _ in range(reps):
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        a.record()
                        fn()
                        b.record()
                        b.synchronize()
                        times.append(a.elapsed_time(b) * 1e3)
                    assert comm.status() == rra.RRA_OK
                us = statistics.median(times)
                res[op] = us
                line = {"sweep": True, "op": op, "N": N, "T": T, "bytes_per_rank": T * 4,
                        "us": us, "algbw_gbs": T * 4 / (us * 1e-6) / 1e9,
                        "busbw_gbs": (T * 4 / (us * 1e-6) / 1e9) * (2 * (N - 1) / N
                                                                      if op == "ring" else 1),
                        "hbm_frac": 8 * N * T / (us * 1e-6) / 1e9 / peak,
                        "sent_max": max(sent), "recv_max": max(recv), "reps": reps}
                out.append(line)
                if rank == 0:
                    print(json.dumps(line), flush=True)
            comm.close()
            del bufs
            torch.cuda.empty_cache()
            rows.append((T, res["ring"], res["tree"]))
        cross = None
        for T, r_us, t_us in rows:
            if r_us < t_us:
                cross = T * 4
                break
        model = alpha_beta_crossover(N, alpha_us, beta_gbs)
        summ = {"sweep_summary": True, "N": N,
                "measured_crossover_bytes": cross if cross is not None else "none in range",
                "model": {"alpha_us": alpha_us, "beta_GBps": beta_gbs,
                          "ring_s": "2(N-1)(alpha + beta*4T/N)", "tree_s": "2L(alpha + beta*4T)",
                          "crossover_bytes_per_rank": model}}
        if rank == 0:
            print(json.dumps(summ), flush=True)
        out.append(summ)
    if args.jsonl and rank == 0:
        with open(args.jsonl, "a") as f:
            for line in out:
                f.write(json.dumps(line) + "\n")


def alpha_beta_times(N: int, nbytes: float, alpha_us: float, beta_gbs: float):
    """Link-model times (seconds) of the ring and the binomial tree for
    nbytes per rank: the ring takes 2(N-1) steps of nbytes/N, the tree
    2*ceil(log2 N) steps of the whole buffer, each step alpha + bytes/beta."""
    L = max(N - 1, 0).bit_length()
    a, b = alpha_us * 1e-6, 1.0 / (beta_gbs * 1e9)
    return 2 * (N - 1) * (a + b * nbytes / N), 2 * L * (a + b * nbytes)


def alpha_beta_crossover(N: int, alpha_us: float, beta_gbs: float):
    """Bytes per rank at which the modelled ring and tree times are equal
    (the ring is faster above it), or None when one is never faster (N <= 2:
    the two schedules coincide)."""
    L = max(N - 1, 0).bit_length()
    slope = L - (N - 1) / N  # extra bytes/beta per byte the tree pays
    if N <= 2 or slope <= 0:
        return None
    return (N - 1 - L) * alpha_us * 1e-6 * beta_gbs * 1e9 / slope


def run_drift(args):
    """Error-feedback drift study: K rounds of the DiLoCo composition (difference
    against the previous round, BFP4, average, base).  Every round draws new
    deltas.  The K compressed results, with and without error feedback, are
    summed and compared with the sum of the lossless ring's results.  Feedback
    keeps what compression lost in the residuals and re-sends it, so its
    accumulated error should stay bounded, while the plain codec's error grows
    with K."""
    import ring_allreduce_compressed_gb300 as rra
    c = W.CONFIGS["diloco_n8"]
    N, T = c["N"], c["T"] // max(1, args.scale)
    comm = rra.Comm(N, T)
    base = torch.zeros(T, device="cuda")
    res = [torch.zeros(T, device="cuda") for _ in range(N)]
    out_l = [torch.empty(T, device="cuda") for _ in range(N)]
    out_p = [torch.empty(T, device="cuda") for _ in range(N)]
    out_e = [torch.empty(T, device="cuda") for _ in range(N)]
    acc = {k: torch.zeros(T, dtype=torch.float64, device="cuda") for k in ("lossless", "plain", "ef")}
    rows = []
    for k in range(args.drift_rounds):
        cur, prev = W.diloco(N, T, seed=1000 + k)
        comm.ring_allreduce(cur, out_l, rra.Codec("none", diff_prev=prev, diff_base=base,
                                                   average=True))
        comm.ring_allreduce(cur, out_p, rra.Codec("bfp", bits=4, diff_prev=prev,
                                                   diff_base=base, average=True))
        comm.ring_allreduce(cur, out_e, rra.Codec("bfp", bits=4, diff_prev=prev, diff_base=base,
                                                   average=True, residual=res))
        assert comm.status() == rra.RRA_OK
        acc["lossless"] += out_l[0].double()
        acc["plain"] += out_p[0].double()
        acc["ef"] += out_e[0].double()
        scale = acc["lossless"].pow(2).mean().sqrt().item()
        row = {"round": k + 1,
               "rms_rel_err_plain": (acc["plain"] - acc["lossless"]).pow(2).mean().sqrt().item() / scale,
               "rms_rel_err_ef": (acc["ef"] - acc["lossless"]).pow(2).mean().sqrt().item() / scale}
        rows.append(row)
    print(json.dumps({"drift_study": True, "N": N, "T": T, "codec": "diff+bfp4, average",
                      "rounds": rows}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about one second of timed work, 20 to 10000 "
                         "steps; the reference arm: 20)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["rra", "reference"], default="rra")
    ap.add_argument("--config", choices=CONFIG_NAMES, default="bfp8_bucket")
    ap.add_argument("--ef", action="store_true",
                    help="BFP workloads: with error feedback (an fp32 residual per rank)")
    ap.add_argument("--drift-rounds", type=int, default=0,
                    help="error-feedback drift study: K DiLoCo rounds (T / --scale per rank), "
                         "compressed with and without feedback against the lossless ring")
    ap.add_argument("--scale", type=int, default=1,
                    help="run the workload with T / scale elements per rank: a small case for "
                         "ncu captures, reported with its own T (not the metric's workload)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--other-configs", type=float, default=0.3, metavar="SECONDS",
                    help="the default line also times every other workload for about this "
                         "many seconds each (0: skip)")
    ap.add_argument("--kernels", action="store_true",
                    help="one timed call of each collective kernel the workloads do not "
                         "cover (plain allgather, broadcast, tree; codec statistics)")
    ap.add_argument("--kernels-T", type=int, default=16 << 20)
    ap.add_argument("--op-warmup", type=int, default=3,
                    help="--codecs / --kernels: untimed calls of each op before its timed ones")
    ap.add_argument("--op-reps", type=int, default=10,
                    help="--codecs / --kernels: timed calls of each op (median reported)")
    ap.add_argument("--codec-n", type=int, default=1 << 28,
                    help="--codecs: elements per codec call (a smaller case for ncu captures)")
    ap.add_argument("--eager", action="store_true",
                    help="time the K steps launched one by one instead of as one CUDA graph")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=60.0)
    ap.add_argument("--jsonl", default=None)
    ap.add_argument("--sweep", action="store_true",
                    help="ring vs tree message-size sweep (lossless fp32) instead of one line")
    ap.add_argument("--codecs", action="store_true",
                    help="time the standalone codec entry points instead of one line")
    ap.add_argument("--sweep-n", default="2,4,8,16,64")
    ap.add_argument("--sweep-kmax", type=int, default=10)
    ap.add_argument("--alpha-us", type=float, default=5.0,
                    help="link latency of the alpha-beta model (microseconds)")
    ap.add_argument("--beta-gbs", type=float, default=5.625,
                    help="link bandwidth of the model, GB/s (45 Gbit/s)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.drift_rounds:
        run_drift(args)
        return
    if args.sweep:
        run_sweep(args, world, rank)
    elif args.codecs:
        run_codecs(args, world, rank)
    elif args.kernels:
        run_kernels(args, world, rank)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_rra(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
