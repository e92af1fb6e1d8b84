"""Benchmark of the batch sampler on GB300.

One step = one pass of the sampling hot path over one batch: read a [B, V]
logits matrix once, Gumbel-max sample every row, write B indices. The headline
workload is the throughput-bound batch: bf16 logits, V = 151936, B = 256,
N(0, 4^2) plus +6 on 32 Zipf(1.1)-ranked token ids per row, T = 1.0, per-row
seeds from splitmix64(7), offset = decode step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. Timing: K steps replayed from CUDA graphs between CUDA
events on the launching stream, barrier + synchronize on both sides, max over
ranks; every step reads a different logits buffer from a pool of more than
4x the L2 size, so no step finds its input in L2. With --gpus N > 1 (under
torchrun) every rank samples its own batch on its own GPU: rows are independent,
so the job is N replicas with no collective on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "sampled rows/sec and µs/step vs V×B; achieved HBM GB/s vs 8 TB/s"
FALLBACK_HBM_GBS = 6800.0
HEADLINE_B = 256
PER_ROW_PARAM_BYTES = 4 + 8 + 8 + 8  # temperature, seed, offset in; index out


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=HEADLINE_B, help="rows of the headline batch")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-workload table")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--quick", action="store_true",
                    help="headline timing only (no CPU baseline, e2e, clocks or table); for "
                         "profiler runs")
    ap.add_argument("--workload", choices=["throughput", "sweep", "hlg", "mixed_greedy",
                                           "filtered"],
                    default="throughput",
                    help="with --quick: time this workload instead of the headline (sweep takes "
                         "--batch and --vocab); prints a short line, for profiler runs")
    ap.add_argument("--vocab", type=int, default=151936, help="V of --workload sweep")
    ap.add_argument("--count-blocks", action="store_true",
                    help="build the block-counting variant of the library and print the Philox "
                         "blocks the sampler computes per launch of the headline batch")
    ap.add_argument("--alu-probe", action="store_true",
                    help="time gsample_debug_philox_alu_mix: Philox alone, ALU work alone and "
                         "both, and print how much of the ALU work adds to the Philox time")
    ap.add_argument("--categorical", action="store_true",
                    help="with --workload: time the categorical (softmax + inverse-CDF) kernel")
    args = ap.parse_args()
    if (args.workload != "throughput" or args.categorical) and not args.quick:
        ap.error("--workload and --categorical time a side case and need --quick")
    return args


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self, gpus: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist

            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist
        self.gpus = gpus

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch

        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate(values_per_rank, times_per_rank):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    return sum(values_per_rank) / max(times_per_rank)


# ---------------------------------------------------------------------------
# measured peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Second roof of the sampler: the Philox4x32-10 blocks it computes, against the
# measured rate of the library's own block code alone
# (gsample_debug_philox_rate), at the best of a few occupancies.
def philox_peak():
    """Measured Philox blocks/s of the kernels' block code on this GPU."""
    import torch

    import token_sampling_logits_gb300 as gs

    L = gs.lib()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    sink = torch.empty(sms * 32 * 32, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    iters = 2000
    best, best_w = 0.0, 0
    for w in (8, 16, 24, 32):
        times = []
        for rep in range(3):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            rc = L.gsample_debug_philox_rate(w, iters, sink.data_ptr(), st)
            e1.record()
            torch.cuda.synchronize()
            if rc != 0:
                raise RuntimeError("gsample_debug_philox_rate: " + gs.status_string(rc))
            times.append(e0.elapsed_time(e1) * 1e-3)
        rate = sms * w * 32 * iters * 4 / min(times)
        if rate > best:
            best, best_w = rate, w
    return best, ("measured: gsample_debug_philox_rate (the kernels' four-way Philox block code "
                  "alone), best of 8/16/24/32 warps per SM (%d), %d SMs" % (best_w, sms))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons around the timed
    region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "gsample_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# The sources that define the headline kernel (sample_kernel) and its launch
# shape: the kernel, the device header it includes, and the planner.
SAMPLE_KERNEL_SOURCES = ("gsample_api.cu", "gsample_device.cuh", "gsample_internal.h",
                         "gsample_sample.cu")


def kernel_source_hash(names=SAMPLE_KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "token_sampling_logits_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profile_figure(profile_name: str, key: str, workload_rows: int,
                   rows_key: str = "captured_rows"):
    """A per-launch figure recorded under profiles/ (`key: value`, with the
    kernel-source hash and the rows of the launch it was taken on, under
    rows_key), scaled to the benchmark's batch; None when the kernel sources
    changed since."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_val = re.search(r"%s:\s*([0-9.eE+]+)" % re.escape(key), text)
    m_rows = re.search(r"%s:\s*(\d+)" % re.escape(rows_key), text)
    if not (m_hash and m_val and m_rows) or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_val.group(1)) * workload_rows / int(m_rows.group(1))


def ncu_traffic(profile_name: str, workload_rows: int):
    """DRAM bytes per launch of one ncu capture, scaled to the batch."""
    return profile_figure(profile_name, "dram_bytes_per_launch", workload_rows)


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on the host cores
# ---------------------------------------------------------------------------
def _oracle_row(args):
    import oracle

    row, dtype, T, seed, rid, off = args
    return oracle.sample_row(row, T, seed, rid, off, dtype=dtype)[0]


def make_pool():
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor

    cores = os.cpu_count() or 1
    return ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")), cores


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, or the Arm implementer
    and part numbers), for the CPU-baseline record."""
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                fields.setdefault(k.strip(), v.strip())
        if fields.get("model name"):
            return fields["model name"]
        if fields.get("CPU implementer"):
            return "Arm implementer %s part %s" % (fields["CPU implementer"],
                                                  fields.get("CPU part", "?"))
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


def oracle_rows_per_sec(pool, batch: W.Batch, rows, step: int) -> float:
    jobs = [(np.ascontiguousarray(batch.logits[r]), batch.dtype, float(batch.temperature[r]),
             int(batch.seed[r]), int(r), step) for r in rows]
    t0 = time.perf_counter()
    list(pool.map(_oracle_row, jobs, chunksize=1))
    return len(rows) / (time.perf_counter() - t0)


# ---------------------------------------------------------------------------
# GPU timing
# ---------------------------------------------------------------------------
def _to_device(x, dtype):
    import torch

    if dtype == W.F32:
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == W.BF16 else torch.float16)


class Runner:
    """Timed decode steps of one workload through the C ABI, replayed from
    captured CUDA graphs (see the module docstring for the buffer pool)."""

    def __init__(self, batch: W.Batch, hlg=None, min_pool_bytes: int = 0, ring: int = 1000,
                 categorical: bool = False, filters=None):
        import ctypes

        import torch

        import token_sampling_logits_gb300 as gs

        self.torch, self.gs, self.ctypes = torch, gs, ctypes
        self.batch, self.hlg = batch, hlg
        self.B, self.V = batch.B, batch.V
        x0 = _to_device(batch.logits, batch.dtype)
        self.bytes_per_step = x0.numel() * x0.element_size()
        # P copies of the batch in one arena, P * bytes > min_pool_bytes, and a
        # graph long enough to visit every copy before coming back to one.
        self.P = max(1, math.ceil(min_pool_bytes / self.bytes_per_step) + 1) if min_pool_bytes else 1
        arena = x0.reshape(-1).repeat(self.P)
        n = x0.numel()
        self.pool = [arena[k * n:(k + 1) * n].view(self.B, self.V) for k in range(self.P)]
        self.ring = max(ring, self.P)
        self.ring = ((self.ring + self.P - 1) // self.P) * self.P
        self.T = torch.from_numpy(batch.temperature.astype(np.float32)).cuda()
        self.S = gs.seeds_as_tensor(batch.seed, "cuda")
        self.offs = torch.zeros((self.ring, self.B), dtype=torch.int64, device="cuda")
        self.out = torch.zeros((self.ring, self.B), dtype=torch.int64, device="cuda")
        self.ws = gs.new_workspace(self.B)
        self.dt, _, _, self.ld = gs._logits_args(self.pool[0])
        self.hp = hlg.to_c() if hlg is not None else None
        self.categorical = categorical
        # (top_k int32[B], top_p float32[B]) for gsample_filtered_gumbel_argmax
        self.filters = None
        if filters is not None:
            self.filters = (torch.from_numpy(np.asarray(filters[0], np.int32)).cuda(),
                            torch.from_numpy(np.asarray(filters[1], np.float32)).cuda())
        self.graphs = {}
        self.launches = 0

    def _launch_range(self, n: int, k0: int):
        L = self.gs.lib()
        st = self.torch.cuda.current_stream().cuda_stream
        B = self.B
        for k in range(n):
            x = self.pool[(k0 + k) % self.P]
            if self.categorical:
                rc = L.gsample_categorical(x.data_ptr(), self.dt, B, self.V, self.ld,
                                           self.T.data_ptr(), self.S.data_ptr(),
                                           self.offs.data_ptr() + 8 * B * k,
                                           self.out.data_ptr() + 8 * B * k, st)
            elif self.filters is not None:
                rc = L.gsample_filtered_gumbel_argmax(
                    x.data_ptr(), self.dt, B, self.V, self.ld, self.T.data_ptr(),
                    self.S.data_ptr(), self.offs.data_ptr() + 8 * B * k,
                    self.filters[0].data_ptr(), self.filters[1].data_ptr(),
                    self.out.data_ptr() + 8 * B * k, self.ws.data_ptr(), st)
            elif self.hp is None:
                rc = L.gsample_gumbel_argmax(x.data_ptr(), self.dt, B, self.V, self.ld,
                                             self.T.data_ptr(), self.S.data_ptr(),
                                             self.offs.data_ptr() + 8 * B * k,
                                             self.out.data_ptr() + 8 * B * k, self.ws.data_ptr(), st)
            else:
                rc = L.gsample_hlg_gumbel_argmax(x.data_ptr(), self.dt, B, self.V, self.ld,
                                                 self.T.data_ptr(), self.S.data_ptr(),
                                                 self.offs.data_ptr() + 8 * B * k,
                                                 self.ctypes.byref(self.hp),
                                                 self.out.data_ptr() + 8 * B * k,
                                                 self.ws.data_ptr(), st)
            if rc != 0:
                raise RuntimeError("sampler launch failed: " + self.gs.status_string(rc))
        self.offs.add_(n)

    def graph(self, n: int):
        torch = self.torch
        if n not in self.graphs:
            # buffers cycle with the step index, so a graph of n launches must
            # start on a step that is a multiple of P to keep the cycle aligned
            self.offs.copy_(torch.arange(self.ring, device="cuda", dtype=torch.int64)[:, None]
                            .expand(self.ring, self.B))
            self._launch_range(n, 0)  # warm-up, outside capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._launch_range(n, 0)
            self.graphs[n] = g
        return self.graphs[n]

    def run(self, steps: int):
        """Enqueue exactly `steps` sampler launches."""
        full, rem = divmod(steps, self.ring)
        if full:
            g = self.graph(self.ring)
            for _ in range(full):
                g.replay()
        if rem:
            self.graph(rem).replay()
        self.launches += steps

    def single_launch_us(self, n: int = 25) -> float:
        """Median of n single launches, each un-captured and bracketed by its own
        pair of CUDA events with the stream idle before it. The span includes
        the host side of the C call (argument checks and the launch itself),
        unlike the graph-replayed µs/step."""
        torch = self.torch
        st = torch.cuda.current_stream().cuda_stream
        L = self.gs.lib()
        B = self.B
        times = []
        for k in range(n):
            x = self.pool[k % self.P]
            out = self.out.data_ptr() + 8 * B * (k % self.ring)
            offs = self.offs.data_ptr() + 8 * B * (k % self.ring)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            if self.categorical:
                rc = L.gsample_categorical(x.data_ptr(), self.dt, B, self.V, self.ld,
                                           self.T.data_ptr(), self.S.data_ptr(), offs, out, st)
            elif self.hp is None:
                rc = L.gsample_gumbel_argmax(x.data_ptr(), self.dt, B, self.V, self.ld,
                                             self.T.data_ptr(), self.S.data_ptr(), offs, out,
                                             self.ws.data_ptr(), st)
            else:
                rc = L.gsample_hlg_gumbel_argmax(x.data_ptr(), self.dt, B, self.V, self.ld,
                                                 self.T.data_ptr(), self.S.data_ptr(), offs,
                                                 self.ctypes.byref(self.hp), out,
                                                 self.ws.data_ptr(), st)
            e1.record()
            torch.cuda.synchronize()
            if rc != 0:
                raise RuntimeError("sampler launch failed: " + self.gs.status_string(rc))
            times.append(e0.elapsed_time(e1) * 1000.0)
        return statistics.median(times)

    def prepare(self, steps: int):
        full, rem = divmod(steps, self.ring)
        if full:
            self.graph(self.ring)
        if rem:
            self.graph(rem)
        self.offs.copy_(self.torch.arange(self.ring, device="cuda", dtype=self.torch.int64)[:, None]
                        .expand(self.ring, self.B))


def time_steps(runner: Runner, steps: int, warmup: int, dist: Dist, clocks: ClockSampler = None):
    torch = runner.torch
    runner.prepare(steps)
    runner.prepare(warmup) if warmup else None
    if warmup:
        runner.run(warmup)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
        # keep the GPU busy while the sampler comes up, so the samples see load
        t_end = time.perf_counter() + 0.3
        while time.perf_counter() < t_end:
            runner.run(min(steps, runner.ring))
            torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    runner.run(steps)
    e1.record()
    torch.cuda.synchronize()
    dist.barrier()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop() if clocks is not None else None
    return ms, clk


def _pinned_batch_copies(batch: W.Batch, n: int):
    import torch

    if batch.dtype == W.F32:
        base = torch.from_numpy(np.ascontiguousarray(batch.logits, dtype=np.float32))
        view = lambda t: t  # noqa: E731
    else:
        base = torch.from_numpy(np.ascontiguousarray(batch.logits).view(np.int16))
        tdt = torch.bfloat16 if batch.dtype == W.BF16 else torch.float16
        view = lambda t: t.view(tdt)  # noqa: E731
    return [view(base.clone().pin_memory()) for _ in range(n)]


def e2e_steps(batch: W.Batch, steps: int, dist: Dist, l2: int):
    """Same metric through the public API with host buffers. Each step the
    sampler reads its logits and per-row parameters from pinned host memory
    over the CPU-GPU link and writes the indices into pinned host memory
    (the C ABI's gsample_gumbel_argmax_host: no staging copy); the host waits
    for them.
    Steps rotate over host buffers larger than 2x L2, so no step finds its
    logits cached. Also timed: the staged path (cudaMemcpyAsync of the inputs
    into device buffers, gsample_gumbel_argmax, copy of the indices back).
    Both call the C ABI directly, as a C caller would."""
    import torch

    import token_sampling_logits_gb300 as gs

    B = batch.B
    nbytes = batch.logits.size * (4 if batch.dtype == W.F32 else 2)
    n_buf = max(2, math.ceil(2 * l2 / nbytes) + 1)
    h_x = _pinned_batch_copies(batch, n_buf)
    h_T = torch.from_numpy(batch.temperature.astype(np.float32)).pin_memory()
    h_S = torch.from_numpy(batch.seed.view(np.int64).copy()).pin_memory()
    h_O = torch.zeros(B, dtype=torch.int64).pin_memory()
    h_out = torch.zeros(B, dtype=torch.int64).pin_memory()
    ws = gs.new_workspace(B)
    h2d = nbytes + B * (4 + 8 + 8)
    d2h = B * 8

    L = gs.lib()
    dt = {W.F32: gs.F32, W.BF16: gs.BF16, W.F16: gs.F16}[batch.dtype]
    V = ld = batch.V
    stream = torch.cuda.current_stream()

    def step_mapped(k):
        h_O.fill_(k)
        rc = L.gsample_gumbel_argmax_host(h_x[k % n_buf].data_ptr(), dt, B, V, ld,
                                          h_T.data_ptr(), h_S.data_ptr(), h_O.data_ptr(),
                                          h_out.data_ptr(), ws.data_ptr(), stream.cuda_stream)
        if rc != 0:
            raise RuntimeError("gsample_gumbel_argmax_host: " + gs.status_string(rc))
        stream.synchronize()  # the caller reads the tokens

    d_x = torch.empty(h_x[0].shape, dtype=h_x[0].dtype, device="cuda")
    d_T = torch.empty(B, dtype=torch.float32, device="cuda")
    d_S = torch.empty(B, dtype=torch.int64, device="cuda")
    d_O = torch.empty(B, dtype=torch.int64, device="cuda")
    d_out = torch.empty(B, dtype=torch.int64, device="cuda")

    def step_staged(k):
        h_O.fill_(k)
        d_x.copy_(h_x[k % n_buf], non_blocking=True)
        d_T.copy_(h_T, non_blocking=True)
        d_S.copy_(h_S, non_blocking=True)
        d_O.copy_(h_O, non_blocking=True)
        rc = L.gsample_gumbel_argmax(d_x.data_ptr(), dt, B, V, ld, d_T.data_ptr(), d_S.data_ptr(),
                                     d_O.data_ptr(), d_out.data_ptr(), ws.data_ptr(),
                                     stream.cuda_stream)
        if rc != 0:
            raise RuntimeError("gsample_gumbel_argmax: " + gs.status_string(rc))
        h_out.copy_(d_out, non_blocking=True)
        stream.synchronize()  # the caller reads the tokens

    secs = {}
    for name, step in (("mapped", step_mapped), ("staged", step_staged)):
        for k in range(3):
            step(k)
        dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(steps):
            step(k)
        torch.cuda.synchronize()
        secs[name] = time.perf_counter() - t0
        dist.barrier()
    return secs, h2d, d2h, n_buf


def extra_table(dist: Dist, l2: int):
    """µs/step of the other workloads (graph-replayed, rotating pools), and the
    latency of one un-captured launch of each."""
    import token_sampling_logits_gb300 as gs

    rows = []
    cases = [("sweep", W.sweep(V, B), None) for V in W.VOCAB_SWEEP for B in W.BATCH_SWEEP]
    cases += [("throughput", W.throughput(B), None) for B in W.THROUGHPUT_B]
    p = W.HLG_PARAMS
    hp = gs.HlgParams(m=p["m"], w=p["w"], beta_t=p["beta_t"], beta_h=p["beta_h"],
                      pivot_offset=p["c"])
    cases.append(("hlg", W.hlg(), hp))
    cases.append(("mixed_greedy", W.mixed_greedy(), None))
    # top-k / top-p on the headline batch: top_k = 50 and top_p = 0.9 on every row
    cases.append(("filtered", W.throughput(HEADLINE_B), None))
    def timed(b, h=None, categorical=False, single=False, filters=None):
        r = Runner(b, hlg=h, min_pool_bytes=4 * l2, ring=500, categorical=categorical,
                   filters=filters)
        steps = r.ring * max(1, (2000 if b.B * b.V < 50_000_000 else 500) // r.ring)
        ms, _ = time_steps(r, steps, 50, dist)
        one = r.single_launch_us() if single else None
        del r
        return (ms * 1000 / steps, one) if single else ms * 1000 / steps

    for kind, b, h in cases:
        filt = ((np.full(b.B, 50, np.int32), np.full(b.B, 0.9, np.float32))
                if kind == "filtered" else None)
        us, one = timed(b, h, single=True, filters=filt) if filt is None else \
            (timed(b, h, filters=filt), None)
        nbytes = b.B * (b.V * (4 if b.dtype == W.F32 else 2) + PER_ROW_PARAM_BYTES)
        row = {"workload": kind, "B": b.B, "V": b.V, "dtype": W.DTYPE_NAMES[b.dtype],
               "us_per_step": round(us, 3), "rows_per_s": round(b.B / us * 1e6, 1),
               "GBps": round(nbytes / us / 1e3, 1),
               "frac_of_8TBps": round(nbytes / us / 1e3 / 8000, 4),
               "single_launch_us": round(one, 3) if one is not None else None}
        if kind == "filtered":
            row["filters"] = "top_k=50, top_p=0.9 on every row (two launches per step: proposal, filter)"
        if kind == "sweep":
            # The issue's comparison: the categorical (softmax + inverse-CDF)
            # path against Gumbel-max on the same V x B grid.
            cu = timed(b, categorical=True)
            row["categorical_us_per_step"] = round(cu, 3)
            row["categorical_over_gumbel"] = round(cu / us, 3)
        rows.append(row)
    return rows


def run_case(args):
    """One side workload (--quick --workload ...), graph-replayed over a pool
    larger than 4x L2, for capturing its kernel under a profiler."""
    import torch

    import token_sampling_logits_gb300 as gs

    gs.lib()
    hp = None
    if args.workload == "sweep":
        b = W.sweep(args.vocab, args.batch)
    elif args.workload == "hlg":
        b = W.hlg()
        p = W.HLG_PARAMS
        hp = gs.HlgParams(m=p["m"], w=p["w"], beta_t=p["beta_t"], beta_h=p["beta_h"],
                          pivot_offset=p["c"])
    elif args.workload == "mixed_greedy":
        b = W.mixed_greedy()
    elif args.workload == "filtered":
        b = W.throughput(args.batch)
    else:
        b = W.throughput(args.batch)
    if hp is not None and args.categorical:
        raise SystemExit("--categorical has no HLG form")
    props = torch.cuda.get_device_properties(0)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    filt = ((np.full(b.B, 50, np.int32), np.full(b.B, 0.9, np.float32))
            if args.workload == "filtered" else None)
    r = Runner(b, hlg=hp, min_pool_bytes=4 * l2, ring=max(1, args.steps),
               categorical=args.categorical, filters=filt)
    ms, _ = time_steps(r, args.steps, max(3, args.warmup), Dist(1))
    print(json.dumps({"workload": args.workload, "B": b.B, "V": b.V,
                      "dtype": W.DTYPE_NAMES[b.dtype], "categorical": args.categorical,
                      "steps": args.steps, "us_per_step": round(ms * 1000 / args.steps, 3)}),
          flush=True)


def headline_config(batch: W.Batch, world: int) -> dict:
    """The workload both arms report (identical keys and values)."""
    return {"workload": "throughput bf16 V=%d B=%d (N(0,4^2) + 32 Zipf(1.1) bumps of +6, "
                        "T=1.0, splitmix64(7) seeds, offset=step)" % (batch.V, batch.B),
            "global_batch": batch.B * world, "vocab": batch.V}


def run_ours(args, dist: Dist):
    import torch

    torch.cuda.set_device(dist.local_rank)
    import token_sampling_logits_gb300 as gs

    gs.lib()
    # CPU baseline pool first (spawned), before the GPU is busy
    pool = cores = None
    batch = W.throughput(args.batch)
    cpu = None
    if dist.rank == 0 and not args.quick:
        pool, cores = make_pool()
        sample_rows = list(range(batch.B))
        rps = []
        for step in range(4):
            rps.append(oracle_rows_per_sec(pool, batch, sample_rows, step))
        cpu = {"value": round(statistics.median(rps), 2), "unit": "rows/s", "cores": cores,
               "cpu": cpu_model(), "kind": "oracle",
               "sample": "%d rows x 4 decode steps of the headline batch (bf16, V=%d), one row "
                         "per task over a spawn pool" % (batch.B, batch.V)}
        pool.shutdown()

    props = torch.cuda.get_device_properties(dist.local_rank)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    runner = Runner(batch, min_pool_bytes=4 * l2)
    clocks = None if args.quick else ClockSampler(dist.local_rank)
    ms, clk = time_steps(runner, args.steps, max(3, args.warmup), dist, clocks)
    ms = dist.max(ms)
    secs = ms / 1000.0
    rows_total = batch.B * args.steps * dist.world
    value = rows_total / secs
    us_step = ms * 1000.0 / args.steps
    alg_bytes = batch.B * (batch.V * 2 + PER_ROW_PARAM_BYTES)
    achieved = alg_bytes / (us_step * 1e-6) / 1e9
    peak, peak_kind = hbm_peak()
    # The method draws one Philox word per element: B * ceil(V / 4) blocks.
    # The sampler computes fewer (exact pruning); a build of the library with
    # -DGSAMPLE_COUNT_BLOCKS counts them (`bench.py --count-blocks`), and the
    # count recorded under profiles/ is used while the kernel sources match.
    alg_blocks = batch.B * ((batch.V + 3) // 4)
    computed = profile_figure("sample_kernel_bf16_throughput.md", "philox_blocks_per_launch",
                              batch.B, rows_key="philox_count_rows")
    ppeak, ppeak_kind = philox_peak() if not args.quick else (None, None)
    hbm_view = {"achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind + " (copy bandwidth)",
                "floor_us": round(alg_bytes / (peak * 1e9) * 1e6, 2)}
    philox_view = None
    if ppeak:
        blocks = computed if computed is not None else float(alg_blocks)
        philox_view = {
            "achieved": round(blocks / (us_step * 1e-6), 1), "peak": round(ppeak, 1),
            "unit": "Philox4x32-10 blocks/s", "frac": round(blocks / (us_step * 1e-6) / ppeak, 4),
            "peak_kind": ppeak_kind,
            "blocks_per_launch": round(blocks),
            "blocks_kind": ("computed (device counter of a -DGSAMPLE_COUNT_BLOCKS build, "
                            "recorded under profiles/)" if computed is not None else
                            "algorithmic B * ceil(V/4) (no count recorded for these sources)"),
            "algorithmic_blocks_per_launch": alg_blocks,
            "floor_us": round(blocks / ppeak * 1e6, 2)}

    e2e = None
    if not args.quick:
        secs, h2d, d2h, n_buf = e2e_steps(batch, args.e2e_steps, dist, l2)
        rows_e2e = batch.B * args.e2e_steps * dist.world
        e2e = {"value": round(rows_e2e / dist.max(secs["mapped"]), 1),
               "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": "gsample_gumbel_argmax_host: the kernel reads pinned host logits and "
                       "parameters over the CPU-GPU link and writes the indices to pinned host "
                       "memory; %d host buffers in rotation" % n_buf,
               "staged_value": round(rows_e2e / dist.max(secs["staged"]), 1),
               "staged_path": "cudaMemcpyAsync of the inputs to device buffers, "
                              "gsample_gumbel_argmax, copy of the indices back"}

    extra = None if args.no_extra or args.quick or dist.rank != 0 else extra_table(Dist(1), l2)

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "rows/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms / args.steps, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        # the arithmetic the path computes in: binary32 scores (the bf16
        # logits widened exactly) and 32-bit integer Philox words
        "dtype": "f32",
        "input_dtype": "bf16",
        "data": "synthetic",
        "config": headline_config(batch, dist.world),
        "setup": {"parallelism": "replicas x%d" % dist.world,
                  "l2": "rotating pool of %d logits buffers (%.0f MB > 4 x L2 %.0f MB): every "
                        "step reads its input from DRAM" % (
                            runner.P, runner.P * runner.bytes_per_step / 1e6, l2 / 1e6),
                  "timing": "CUDA events around the %d timed launches, replayed from captured "
                            "CUDA graphs of up to %d launches" % (args.steps, runner.ring)},
        "us_per_step": round(us_step, 3),
        "GBps": round(achieved, 1),
        "frac_of_8TBps": round(achieved / 8000.0, 4),
        # The path streams each logit once: HBM bytes are the roof (the
        # Philox view below explains the time the sampler spends above it).
        "roofline": {"bound": "hbm", "achieved": hbm_view["achieved"], "peak": peak,
                     "unit": "GB/s", "frac": hbm_view["frac"],
                     "peak_kind": hbm_view["peak_kind"],
                     "traffic": ncu_traffic("sample_kernel_bf16_throughput.md", batch.B),
                     "kernel": "gsample::sample_kernel<bf16, 128-bit>",
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "floor_us": hbm_view["floor_us"],
                     "philox": philox_view},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if extra is not None:
        line["workloads"] = extra
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, dist: Dist):
    """The reference arm: the CPU oracle as it stands, on the host cores, on the
    same workload and metric (each step a bounded sample of rows)."""
    if dist.rank != 0:
        return
    batch = W.throughput(args.batch)
    pool, cores = make_pool()
    # calibrate, then size the per-step sample so the whole run stays in minutes
    rps = oracle_rows_per_sec(pool, batch, list(range(min(batch.B, 2 * cores))), 0)
    total_steps = args.steps + max(3, args.warmup)
    budget_s = 150.0
    rows_per_step = int(max(1, min(batch.B, budget_s * rps / total_steps)))
    rows = list(range(rows_per_step))
    for k in range(max(3, args.warmup)):
        oracle_rows_per_sec(pool, batch, rows[:max(1, min(len(rows), cores))], k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        oracle_rows_per_sec(pool, batch, rows, k)
    secs = time.perf_counter() - t0
    pool.shutdown()
    value = rows_per_step * args.steps / secs
    sample = "%d of %d rows per decode step of the headline batch (bf16, V=%d), one row per " \
             "task over a spawn pool" % (rows_per_step, batch.B, batch.V)
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 2), "unit": "rows/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(secs * 1000 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(batch, dist.world),
        "setup": {"parallelism": "oracle on the host cores (rank 0)"},
        "cpu_baseline": {"value": round(value, 2), "unit": "rows/s", "cores": cores,
                         "cpu": cpu_model(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_alu_probe(args):
    """How much ALU work issued beside the Philox multiplies adds to their time
    (gsample_debug_philox_alu_mix, 16 warps per SM as in the sampler): ns per
    warp-block per SM sub-partition for Philox alone, the ALU updates alone and
    both, and the share of the ALU time that the mixed run adds."""
    import torch

    import token_sampling_logits_gb300 as gs

    L = gs.lib()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    w, iters = 16, 2000
    sink = torch.empty(sms * w * 32, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream

    def ns_per_warp_block(steps, philox):
        times = []
        for rep in range(4):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            rc = L.gsample_debug_philox_alu_mix(w, iters, steps, philox, sink.data_ptr(), st)
            e1.record()
            torch.cuda.synchronize()
            if rc != 0:
                raise RuntimeError("gsample_debug_philox_alu_mix: " + gs.status_string(rc))
            times.append(e0.elapsed_time(e1) * 1e6)
        # each SM sub-partition runs w / 4 warps of iters * 4 blocks
        return min(times[1:]) / (w / 4 * iters * 4)

    res = {"warps_per_sm": w, "iters": iters, "unit": "ns per warp-block per SM sub-partition",
           "philox_only": round(ns_per_warp_block(0, 1), 4)}
    for steps in (2, 4):
        alu = ns_per_warp_block(steps, 0)
        mix = ns_per_warp_block(steps, 1)
        res["alu_steps_%d" % steps] = {"alu_only": round(alu, 4), "mixed": round(mix, 4),
                                       "added_share_of_alu": round((mix - res["philox_only"]) / alu,
                                                                   3)}
    print(json.dumps(res), flush=True)


def run_count_blocks(args):
    """Philox blocks the sampler computes per launch of the headline batch, from
    a build of the library with a device counter (-DGSAMPLE_COUNT_BLOCKS, built
    beside the regular one), at the headline temperature and two others."""
    from token_sampling_logits_gb300 import build as gbuild

    out_dir = os.path.join(ROOT, "token_sampling_logits_gb300", "_build", "count")
    path = gbuild.build(extra_flags=["-DGSAMPLE_COUNT_BLOCKS"], out_dir=out_dir)
    gbuild.LIB = path
    gbuild.is_stale = lambda: False
    import ctypes

    import torch

    import token_sampling_logits_gb300 as gs

    L = gs.lib()
    base = W.throughput(args.batch)
    x = _to_device(base.logits, base.dtype)
    S = gs.seeds_as_tensor(base.seed, "cuda")
    cnt = ctypes.c_uint64(0)
    res = {}
    for T in (1.0, 0.3, 100.0):
        Tt = torch.full((base.B,), T, dtype=torch.float32, device="cuda")
        L.gsample_debug_blocks_computed(ctypes.byref(cnt), 1)
        n = 20
        for k in range(n):
            gs.gumbel_argmax(x, Tt, S, torch.full((base.B,), k, dtype=torch.int64, device="cuda"))
        torch.cuda.synchronize()
        rc = L.gsample_debug_blocks_computed(ctypes.byref(cnt), 1)
        if rc != 0:
            raise RuntimeError("gsample_debug_blocks_computed: " + gs.status_string(rc))
        res["T=%g" % T] = cnt.value / n
    alg = base.B * ((base.V + 3) // 4)
    print(json.dumps({"kernel_source_hash": kernel_source_hash(), "philox_count_rows": base.B,
                      "algorithmic_blocks_per_launch": alg,
                      "philox_blocks_per_launch": res,
                      "share_of_algorithmic": {k: round(v / alg, 4) for k, v in res.items()}}),
          flush=True)


def main():
    args = parse_args()
    if args.count_blocks:
        run_count_blocks(args)
        return
    if args.alu_probe:
        run_alu_probe(args)
        return
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        elif args.workload != "throughput" or args.categorical:
            run_case(args)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
