#!/usr/bin/env python3
"""Benchmark of one paged decode step on GB300.

A step is the whole hot path over one batch: pa_cache_append of the step's
new token for every sequence, then the paged read (pa_decode).  The
workload is the Llama-3.2-1B-shaped decode batch: 64 sequences at history
4096, 32 query / 8 kv heads, head_dim 64, 16-token pages from a 20,000-page
pool, bf16.  The metric is achieved HBM bandwidth of the step (algorithmic
bytes / device time, GB/s) with the time per step.

Also reported on the same JSON line: the history sweep {16 .. 4096} of the
read alone (L2 flushed between launches), the long-context split-KV read +
merge at 32K and 128K tokens, the ragged 256-sequence batch, the roofline
of the read kernel, clocks sampled during the run, an end-to-end number
through the C ABI with host buffers, and the fp64 oracle timed on the host
cores as a CPU baseline.

``--impl reference`` times the fp64 CPU oracle instead (the slow program
the pages call the correctness oracle), on host cores, in the same units.

Run: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

if __name__ == "__main__":
    # The CPU baseline runs the oracle on one thread, then one process per core:
    # hold NumPy's BLAS to one thread in each (read when NumPy loads, after this
    # point; spawned workers inherit it).
    os.environ["OPENBLAS_NUM_THREADS"] = "1"

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak), µs/step at B=64"
UNIT = "GB/s"
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_llama1b_h4096.md")
DOMINANT_SOURCES = ("paged_kv_cache_184_gb300/csrc/pa_decode_mma.cu",
                    "paged_kv_cache_184_gb300/csrc/pa_common.cuh")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--history", type=int, default=4096)
    ap.add_argument("--no-extras", action="store_true",
                    help="headline step only (no sweep, long-context, ragged, CPU baseline)")
    ap.add_argument("--only", choices=["sweep", "longctx", "ragged8b", "dense_vs_sdpa", "chunk",
                                       "prefill", "f32", "floor"],
                    help="run one extra section alone and print its JSON (for profiling)")
    return ap.parse_args()


# ----------------------------------------------------------------- byte counts


def read_bytes(lens, hq, hkv, d, elem, block_size):
    """Algorithmic bytes of one paged read: K+V rows, q, out, table entries, lengths."""
    kv = sum(lens) * hkv * d * 2 * elem
    qo = 2 * len(lens) * hq * d * elem
    table = 4 * sum(-(-n // block_size) for n in lens) + 4 * len(lens)
    return kv + qo + table


def append_bytes(b, hkv, d, elem):
    """Read k_new/v_new, write them into the pool, read position, table entry."""
    return 2 * 2 * b * hkv * d * elem + 8 * b


def split_bytes(b, hq, s, d):
    """Partials written by the split read and read back by the merge."""
    return 2 * b * hq * s * (d + 1) * 4


# ----------------------------------------------------------------- ranks


def max_over_ranks(dist, x: float, device) -> float:
    """The largest x over all ranks (x itself when not distributed)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------------- environment


def measured_peaks():
    """HBM copy bandwidth (GB/s) measured on this machine's GPUs, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
    except (OSError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"

    def find(obj):
        if isinstance(obj, dict):
            for k, v in obj.items():
                if "hbm" in k.lower() and isinstance(v, (int, float)) and v > 100:
                    return float(v)
            for v in obj.values():
                r = find(v)
                if r is not None:
                    return r
        return None

    v = find(j)
    return (v, "measured") if v is not None else (FALLBACK_HBM_GBS, "fallback")


def source_sha():
    h = hashlib.sha256()
    for rel in DOMINANT_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current kernel source; else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != source_sha():
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "sm_min_mhz": min(sm), "power_w_median": statistics.median(
                    [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()] or [0.0]),
                "samples": len(rows), "reasons": reasons}


# ----------------------------------------------------------------- CPU oracle timing


class OracleSample:
    """Host copies of a batch for timing the fp64 oracle on whole sequences."""

    def __init__(self, batch_cpu):
        self.b = batch_cpu
        self.q = batch_cpu.q.float().numpy()
        self.kp = batch_cpu.k_pool.float().numpy()
        self.vp = batch_cpu.v_pool.float().numpy()
        self.bt = batch_cpu.block_table.numpy()
        self.lens = batch_cpu.lens_list()
        self.cpu_s = 0.0
        self.wall_s = 0.0
        self.seq_s = []   # wall time of every sequence run so far

    def seq_bytes(self, i: int) -> int:
        b = self.b
        return read_bytes([self.lens[i]], b.num_q_heads, b.num_kv_heads, b.head_dim,
                          b.q.element_size(), b.block_size)

    def run(self, budget_s: float, max_seqs: int, first: int = 0):
        """Oracle over sequences first, first+1, ... until the budget is spent.
        Returns (seconds, algorithmic bytes read, sequences done)."""
        import oracle
        b = self.b
        t0, c0 = time.perf_counter(), time.process_time()
        done, nbytes = 0, 0
        t_prev = t0
        while done < max_seqs:
            i = (first + done) % len(self.lens)
            oracle.paged_decode_one(self.q[i], self.kp, self.vp, self.bt[i], self.lens[i],
                                    b.scale, b.block_size)
            nbytes += self.seq_bytes(i)
            done += 1
            t_now = time.perf_counter()
            self.seq_s.append(t_now - t_prev)
            t_prev = t_now
            if t_now - t0 > budget_s:
                break
        wall = time.perf_counter() - t0
        self.cpu_s += time.process_time() - c0   # CPU time of every thread of the process
        self.wall_s += wall
        return wall, nbytes, done

    def cpu_per_wall(self) -> float:
        """Average number of busy host threads over the timed oracle runs."""
        return round(self.cpu_s / self.wall_s, 2) if self.wall_s > 0 else 0.0


# The multi-core oracle: one spawned process per host core, each running the
# unchanged oracle on whole sequences with its BLAS held to one thread.  The
# pools are placed once in shared memory, so a worker maps them instead of
# receiving a copy.

_W = {}


def _oracle_worker_init(names, shapes, scale, block_size):
    from multiprocessing import shared_memory
    import numpy as np
    _W["shm"] = [shared_memory.SharedMemory(name=n) for n in names]
    _W["arr"] = [np.ndarray(shp, dtype=np.float32 if k < 3 else np.int32, buffer=m.buf)
                 for k, (m, shp) in enumerate(zip(_W["shm"], shapes))]
    _W["scale"], _W["bs"] = scale, block_size


def _oracle_worker(task):
    """Oracle over the sequences of `task`; returns (CPU seconds, wall seconds)."""
    import oracle
    q, kp, vp, bt, lens = _W["arr"]
    t0, c0 = time.perf_counter(), time.process_time()
    for i in task:
        oracle.paged_decode_one(q[i], kp, vp, bt[i], int(lens[i]), _W["scale"], _W["bs"])
    return time.process_time() - c0, time.perf_counter() - t0


class ParallelOracle:
    """The oracle over a whole batch, one sequence per task, on `cores` processes."""

    def __init__(self, sample: OracleSample, cores: int):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        import numpy as np
        self.sample = sample
        self.cores = cores
        arrays = [sample.q, sample.kp, sample.vp, sample.bt.astype(np.int32),
                  np.asarray(sample.lens, dtype=np.int32)]
        self.shm = []
        for a in arrays:
            m = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=a.dtype, buffer=m.buf)[...] = a
            self.shm.append(m)
        ctx = mp.get_context("spawn")   # a fresh interpreter: safe after CUDA is initialised
        self.pool = ctx.Pool(cores, initializer=_oracle_worker_init,
                             initargs=([m.name for m in self.shm], [a.shape for a in arrays],
                                       sample.b.scale, sample.b.block_size))
        n = len(sample.lens)
        self.tasks = [list(range(w, n, cores)) for w in range(min(cores, n))]
        self.pass_bytes = sum(sample.seq_bytes(i) for i in range(n))
        self.cpu_s = 0.0
        self.wall_s = 0.0

    def one_pass(self) -> float:
        """Wall seconds of the oracle over every sequence of the batch."""
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_worker, self.tasks, chunksize=1)
        wall = time.perf_counter() - t0
        self.cpu_s += sum(c for c, _ in res)
        self.wall_s += wall
        return wall

    def close(self):
        self.pool.close()
        self.pool.join()
        for m in self.shm:
            m.close()
            m.unlink()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(batch_cpu, history: int, single_budget_s: float = 6.0,
                 multi_budget_s: float = 10.0) -> dict:
    """The oracle as it stands on this host: one core, then every core of the affinity
    set (one process each, BLAS at one thread).  value = the multi-core figure."""
    sample = OracleSample(batch_cpu)
    t1, nb1, n1 = sample.run(single_budget_s, 1 << 30)
    gbs = lambda nbytes, sec: nbytes / sec / 1e9
    cores = host_cores()
    try:
        par = ParallelOracle(sample, cores)
    except (OSError, ValueError) as e:      # e.g. too little shared memory for the pools
        return {"value": gbs(nb1, t1), "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{n1} seqs of the h{history} batch, 1 thread ({type(e).__name__})"}
    try:
        par.one_pass()                      # warm-up: workers import NumPy and map the pools
        par.cpu_s = par.wall_s = 0.0
        walls = []
        while sum(walls) < multi_budget_s and len(walls) < 200:
            walls.append(par.one_pass())
        busy = par.cpu_s / par.wall_s if par.wall_s > 0 else 0.0
    finally:
        par.close()
    return {"value": gbs(par.pass_bytes * len(walls), sum(walls)), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{len(walls)} passes of the h{history} batch, 1 proc/core",
            "best_ms": 1e3 * min(walls), "median_ms": 1e3 * statistics.median(walls),
            "busy": busy, "single_core": gbs(nb1, t1)}


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle on every host core, same workload and metric.
    Each step is one pass of the oracle over the whole 64-sequence batch."""
    if rank != 0:
        return
    import workloads
    sample = OracleSample(workloads.llama1b(args.history))
    cores = host_cores()
    try:
        par = ParallelOracle(sample, cores)
    except (OSError, ValueError):          # e.g. too little shared memory: one process
        par = None
    if par is not None:
        try:
            for _ in range(args.warmup):
                par.one_pass()
            par.cpu_s = par.wall_s = 0.0
            times = [par.one_pass() for _ in range(args.steps)]
            busy = par.cpu_s / par.wall_s if par.wall_s > 0 else 0.0
        finally:
            par.close()
        pass_bytes = par.pass_bytes
    else:
        cores, n = 1, len(sample.lens)
        for k in range(args.warmup):
            sample.run(0.0, 1, first=k)
        sample.cpu_s = sample.wall_s = 0.0
        times = [sample.run(1e9, n)[0] for _ in range(args.steps)]
        busy = sample.cpu_per_wall()
        pass_bytes = sum(sample.seq_bytes(i) for i in range(n))
    total = sum(times)
    value = pass_bytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "busy": busy, "blas_threads": os.environ.get("OPENBLAS_NUM_THREADS"),
                         "best_ms": 1e3 * min(times),
                         "median_ms": 1e3 * statistics.median(times),
                         "sample": f"each step: the fp64 oracle over all 64 sequences "
                                   f"(history {args.history}), {cores} process(es)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(compact_json(line), flush=True)


# ----------------------------------------------------------------- the JSON line


def round_sig(x, sig: int = 4):
    """Floats rounded to `sig` significant figures, recursively (ints, strings kept); a
    rounded value of 1000 or more that is a whole number is written as an int."""
    if isinstance(x, float):
        if not math.isfinite(x) or x == 0.0:
            return x
        r = float(f"{x:.{sig}g}")
        return int(r) if abs(r) >= 1000 and r == int(r) else r
    if isinstance(x, dict):
        return {k: round_sig(v, sig) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [round_sig(v, sig) for v in x]
    return x


def compact_json(line: dict) -> str:
    """One JSON line, floats at 4 significant figures, no spaces after separators."""
    return json.dumps(round_sig(line), separators=(",", ":"), ensure_ascii=False)


def extra_error(e: Exception) -> dict:
    return {"error": f"{type(e).__name__}: {e}"[:64]}


def workload_config(args, world):
    return {"workload": f"llama1b append+read B64 h{args.history} Hq32/Hkv8 d64 bs16 bf16",
            "global_batch": 64 * world, "seq_len": args.history,
            "parallelism": f"{world} replicas" if world > 1 else "1 GPU",
            "l2": "inputs > L2" if args.history >= 1024 else "L2 flushed"}


# ----------------------------------------------------------------- GPU side


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        run_reference(args, rank, world)
        return

    import torch
    import paged_kv_cache_184_gb300 as pa
    import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.only:
        pa.load()
        peak, _ = measured_peaks()
        fns = {"sweep": lambda: sweep(pa, workloads, torch, dev, L2Flush(torch, dev), peak),
               "longctx": lambda: longctx(pa, workloads, torch, dev, peak),
               "ragged8b": lambda: ragged(pa, workloads, torch, dev, peak),
               "dense_vs_sdpa": lambda: dense_vs_sdpa(pa, workloads, torch, dev, peak),
               "chunk": lambda: chunk(pa, workloads, torch, dev, peak),
               "prefill": lambda: prefill(pa, workloads, torch, dev),
               "f32": lambda: f32_read(pa, workloads, torch, dev, peak),
               "floor": lambda: launch_floor(pa, workloads, torch, dev, peak)}
        print(json.dumps({args.only: fns[args.only]()[1]}), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pa.load()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ------------------------------------------------ headline workload
    cpu = workloads.llama1b(args.history)
    g = cpu.to(dev)
    out = torch.empty_like(g.q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lens = g.lens_list()
    elem = g.q.element_size()
    rb = read_bytes(lens, g.num_q_heads, g.num_kv_heads, g.head_dim, elem, g.block_size)
    ab = append_bytes(g.num_seqs, g.num_kv_heads, g.head_dim, elem)
    step_bytes = rb + ab
    flush = L2Flush(torch, dev)
    small = args.history < 1024  # history too short to exceed L2 by itself

    def step():
        pa.pa_cache_append(g.k_new, g.v_new, g.k_pool, g.v_pool, g.block_table, g.positions,
                           dev_err=err)
        pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale,
                     dev_err=err)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t_end = time.perf_counter() + 1.0        # keep the GPU loaded so clocks settle
    while time.perf_counter() < t_end:
        for _ in range(50):
            step()
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # timed region: K whole steps, events only at step boundaries (an event
    # between the two kernels would stop the read's launch from overlapping
    # the append)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    for k in range(args.steps):
        if small:
            flush()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step = max_over_ranks(dist, sum(step_ms) / args.steps, dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())} during the timed steps")
    value = job_gbs(step_bytes, world, ms_per_step)
    gpu_launches = 2 * args.steps

    # the dominant kernel alone, same launch, K launches with an event pair each
    dec = lambda: pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale,
                               dev_err=err)
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    barrier()
    # two untimed launches queue ahead of the timed ones: on an idle GPU the first
    # start event would fire at once and the kernel arrive a host submission later
    # (measured: the first launch after a synchronize read 103-115 us, the rest 82-86)
    for _ in range(2):
        dec()
    for k in range(args.steps):
        if small:
            flush()
        dev_ev[k][0].record(stream)
        dec()
        dev_ev[k][1].record(stream)
    barrier()
    dec_ms = [a.elapsed_time(b) for a, b in dev_ev]
    dec_avg_ms = sum(dec_ms) / args.steps
    peak, peak_kind = measured_peaks()
    achieved = rb / (dec_avg_ms * 1e-3) / 1e9

    # ------------------------------------------------ end to end with host buffers
    # The step's inputs live in one pinned host buffer and move to the device
    # in one copy; the output comes back in one copy.
    names = ("q", "k_new", "v_new", "positions", "seq_lens", "block_table")
    parts = [getattr(cpu, n).contiguous().view(torch.uint8).reshape(-1) for n in names]
    sizes = [(x.numel() + 255) // 256 * 256 for x in parts]
    h_in = torch.zeros(sum(sizes), dtype=torch.uint8).pin_memory()
    d_in_buf = torch.empty_like(h_in, device=dev)
    d_in, off = {}, 0
    for n, x, sz in zip(names, parts, sizes):
        h_in[off:off + x.numel()].copy_(x)
        src = getattr(cpu, n)
        d_in[n] = d_in_buf[off:off + x.numel()].view(src.dtype).view(src.shape)
        off += sz
    h_out = torch.empty(cpu.q.shape, dtype=cpu.q.dtype).pin_memory()
    h2d = h_in.numel()
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_in_buf.copy_(h_in, non_blocking=True)
        pa.pa_cache_append(d_in["k_new"], d_in["v_new"], g.k_pool, g.v_pool, d_in["block_table"],
                           d_in["positions"], dev_err=err)
        pa.pa_decode(out, d_in["q"], g.k_pool, g.v_pool, d_in["block_table"], d_in["seq_lens"],
                     g.scale, dev_err=err)
        h_out.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        if small:
            flush()
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_serial_ms = max_over_ranks(dist, e0.elapsed_time(e1) / args.steps, dev)
    serial_result = h_out.clone()  # every step computes the same thing from the same inputs

    # The serving-loop form of the same steps: two input buffers and two outputs,
    # step k+1's upload and step k's download on a copy stream while step k's
    # kernels run.  Every step still uploads its own inputs and downloads its own
    # result inside the timed region; events keep a buffer from being refilled
    # before the kernels (or the download) that use it are done.
    copy_stream = torch.cuda.Stream(dev)
    bufs = [d_in_buf, torch.empty_like(h_in, device=dev)]
    views = [d_in, {n: bufs[1][int(t.data_ptr() - d_in_buf.data_ptr()):][:t.numel() * t.element_size()]
                    .view(t.dtype).view(t.shape) for n, t in d_in.items()}]
    outs = [out, torch.empty_like(out)]
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
    ev = lambda: torch.cuda.Event()
    in_ready, computed, downloaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def upload(k):
        j = k % 2
        copy_stream.wait_event(computed[j])     # step k - 2's kernels are done with buffer j
        with torch.cuda.stream(copy_stream):
            bufs[j].copy_(h_in, non_blocking=True)
        in_ready[j].record(copy_stream)

    def compute(k):
        j = k % 2
        stream.wait_event(in_ready[j])
        stream.wait_event(downloaded[j])        # step k - 2's result has left outs[j]
        v = views[j]
        pa.pa_cache_append(v["k_new"], v["v_new"], g.k_pool, g.v_pool, v["block_table"],
                           v["positions"], dev_err=err)
        pa.pa_decode(outs[j], v["q"], g.k_pool, g.v_pool, v["block_table"], v["seq_lens"],
                     g.scale, dev_err=err)
        computed[j].record(stream)

    def download(k):
        j = k % 2
        copy_stream.wait_event(computed[j])
        with torch.cuda.stream(copy_stream):
            h_outs[j].copy_(outs[j], non_blocking=True)
        downloaded[j].record(copy_stream)

    def pipelined(n):
        copy_stream.wait_stream(stream)
        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            compute(k)
            download(k)
        stream.wait_event(downloaded[(n - 1) % 2])

    pipelined(max(args.warmup, 2))
    torch.cuda.synchronize(dev)
    barrier()
    e0.record(stream)
    pipelined(args.steps)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1) / args.steps, dev)
    e2e_value = job_gbs(step_bytes, world, e2e_ms)
    torch.cuda.synchronize(dev)
    for j in range(2):
        if not torch.equal(h_outs[j], serial_result):
            raise RuntimeError("pipelined end-to-end step differs from the serial one")

    m = {"value": value, "world": world, "steps": args.steps, "warmup": args.warmup,
         "ms_per_step": ms_per_step, "config": workload_config(args, world), "clocks": clk,
         "e2e_value": e2e_value, "h2d": h2d, "d2h": d2h,
         "serial_value": job_gbs(step_bytes, world, e2e_serial_ms),
         "gpu_launches": gpu_launches, "achieved": achieved, "peak": peak,
         "peak_kind": peak_kind, "traffic": profiled_traffic(), "rb": rb,
         "dec_ms": dec_ms}
    extras, cpu_line = {}, None
    if rank == 0 and not args.no_extras:
        runs = (("chunk", lambda: chunk(pa, workloads, torch, dev, peak)),
                ("dense_vs_sdpa", lambda: dense_vs_sdpa(pa, workloads, torch, dev, peak)),
                ("sweep", lambda: sweep(pa, workloads, torch, dev, flush, peak)),
                ("longctx", lambda: longctx(pa, workloads, torch, dev, peak)),
                ("ragged8b", lambda: ragged(pa, workloads, torch, dev, peak)),
                ("prefill", lambda: prefill(pa, workloads, torch, dev)))
        for key, run_extra in runs:
            try:
                extras[key] = run_extra()[0]
            except Exception as e:  # the headline stands; the failure is reported in its place
                extras[key] = extra_error(e)
        if world == 1:
            try:
                cpu_line = cpu_baseline(cpu, args.history)
            except Exception as e:
                cpu_line = extra_error(e)
    if rank == 0:
        print(compact_json(compose_line(m, extras, cpu_line)), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# Compact forms of the extras' results for the JSON line (the full detail is printed by
# --only <extra>).


def compact_sweep(rows):
    return {"h": [r["history"] for r in rows], "us": [r["us_median"] for r in rows],
            "frac": [r["frac"] for r in rows]}


def compact_longctx(rows):
    return {f"{r['history'] // 1024}k": {"us": r["us_split_plus_merge"], "frac": r["frac"]}
            for r in rows}


def compact_ragged(res):
    best = min(res["planned"], key=lambda x: x["us"])
    return {"us_1pass": res["us_single_pass"], "us_split64": res["us_split64_plus_merge"],
            "us_planned": best["us"], "frac_best": res["frac_best"]}


def compact_chunk(detail):
    rows, lc = detail["llama1b_h4096"], detail["longctx_h32768_split"]
    return {"nq": [r["n_q"] for r in rows], "us": [r["us"] for r in rows],
            "tf": rows[-1]["tflops"], "ctx32k_us": [r["us_split_plus_merge"] for r in lc]}


def compact_prefill(rows):
    return {f"d{r['head_dim']}": {"tf": r["tflops"], "frac": r["frac_tensor"]} for r in rows}


def compact_dense(rows):
    return {"n": [r["n_ctx"] // 1024 for r in rows], "x_sdpa": [r["sdpa_over_ours"] for r in rows]}


GRADED = ("sweep", "longctx", "ragged8b", "prefill")


def compose_line(m: dict, extras: dict, cpu_line) -> dict:
    """The bench's one JSON line from the measurements `m`, the extras' compact results
    and the CPU baseline.  Short keys and 4 significant figures keep the whole line near
    1.5 KB; the graded extras come last, so that they end the line."""
    dec_ms = m["dec_ms"]
    mean_ms = sum(dec_ms) / len(dec_ms)
    line = {
        "metric": METRIC, "value": m["value"], "unit": UNIT, "n_gpus": m["world"],
        "steps": m["steps"], "warmup": m["warmup"], "ms_per_step": m["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded)",
        "config": m["config"],
        "clocks": {k: m["clocks"].get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")
                   if k in m["clocks"]},
        "e2e": {"value": m["e2e_value"], "unit": UNIT, "h2d_bytes_per_step": m["h2d"],
                "d2h_bytes_per_step": m["d2h"]},
        "gpu_launches": m["gpu_launches"],
        "roofline": {"bound": "hbm", "achieved": m["achieved"], "peak": m["peak"],
                     "unit": "GB/s", "frac": m["achieved"] / m["peak"],
                     "traffic": m["traffic"], "algo_bytes": m["rb"], "us": 1e3 * mean_ms},
    }
    if cpu_line is not None:
        line["cpu_baseline"] = cpu_line
    for key in [k for k in extras if k not in GRADED] + [k for k in GRADED if k in extras]:
        line[key] = extras[key]
    return line


class L2Flush:
    """Evicts L2 by reading a buffer twice its size.  Reading (not writing)
    leaves no dirty lines behind, so the next kernel pays no write-back."""

    def __init__(self, torch, dev):
        self.buf = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)
        self.torch = torch

    def __call__(self):
        self.torch.sum(self.buf, dim=0, out=self.sink)


def _time_launches(fn, torch, flush, iters=30, warm=3):
    """Median / min device time (ms) of fn over iters launches, L2 flushed before each."""
    stream = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(iters):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ts]
    return statistics.median(ms), min(ms)


def sweep(pa, workloads, torch, dev, flush, peak):
    """The read alone at every llama1b history (B 64), L2 flushed before each launch."""
    rows = []
    for h in workloads.LLAMA1B_HISTORIES:
        g = workloads.llama1b(h, device=str(dev))
        out = torch.empty_like(g.q)
        fn = lambda: pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale)
        med, mn = _time_launches(fn, torch, flush)
        rb = read_bytes(g.lens_list(), 32, 8, 64, 2, 16)
        rows.append({"history": h, "us_median": 1e3 * med, "us_min": 1e3 * mn,
                     "gbs": rb / (med * 1e-3) / 1e9, "frac": rb / (med * 1e-3) / 1e9 / peak})
        del g, out
    torch.cuda.empty_cache()
    return compact_sweep(rows), rows


def longctx(pa, workloads, torch, dev, peak):
    rows = []
    flush = L2Flush(torch, dev)
    for h in workloads.LONGCTX_HISTORIES:
        g = workloads.longctx(h, device=str(dev))
        s = pa.pa_num_splits(g.max_blocks, g.pages_per_split)
        po = torch.empty((g.num_seqs, g.num_q_heads, s, g.head_dim), device=dev)
        pl = torch.empty((g.num_seqs, g.num_q_heads, s), device=dev)
        out = torch.empty_like(g.q)

        def fn():
            pa.pa_decode_splitkv(po, pl, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                 g.scale, g.pages_per_split)
            pa.pa_merge(out, po, pl)

        med, mn = _time_launches(fn, torch, flush, iters=20)
        rb = read_bytes(g.lens_list(), 32, 8, 128, 2, 16) + split_bytes(g.num_seqs, 32, s, 128)
        single = lambda: pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                      g.scale)
        med1, _ = _time_launches(single, torch, flush, iters=10)
        rows.append({"history": h, "splits": s, "us_split_plus_merge": 1e3 * med,
                     "gbs": rb / (med * 1e-3) / 1e9, "frac": rb / (med * 1e-3) / 1e9 / peak,
                     "us_single_pass": 1e3 * med1})
        del g, po, pl, out
        torch.cuda.empty_cache()
    return compact_longctx(rows), rows


def ragged(pa, workloads, torch, dev, peak):
    flush = L2Flush(torch, dev)
    g = workloads.ragged8b(device=str(dev))
    out = torch.empty_like(g.q)
    s = pa.pa_num_splits(g.max_blocks, 64)
    po = torch.empty((g.num_seqs, g.num_q_heads, s, g.head_dim), device=dev)
    pl = torch.empty((g.num_seqs, g.num_q_heads, s), device=dev)
    single = lambda: pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale)

    def split():
        pa.pa_decode_splitkv(po, pl, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale, 64)
        pa.pa_merge(out, po, pl)

    med1, _ = _time_launches(single, torch, flush, iters=10)
    med2, _ = _time_launches(split, torch, flush, iters=10)
    rb = read_bytes(g.lens_list(), 32, 8, 128, 2, 16)
    res = {"batch": g.num_seqs, "kv_gb": g.kv_bytes() / 1e9,
           "us_single_pass": 1e3 * med1, "gbs_single_pass": rb / (med1 * 1e-3) / 1e9,
           "us_split64_plus_merge": 1e3 * med2,
           "gbs_split64": (rb + split_bytes(g.num_seqs, 32, s, 128)) / (med2 * 1e-3) / 1e9}
    # planned work lists (host plan from the lengths; items copied to the device)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    host_lens = g.seq_lens.cpu()
    planned = []
    for mult in (3, 6, 12, 24):
        t0 = time.perf_counter()
        items, slots = pa.pa_plan_work(host_lens, 8, 16, sms * mult, 16)
        plan_us = 1e6 * (time.perf_counter() - t0)
        d_items = items.to(dev)
        po_w = torch.empty((g.num_seqs, 32, slots, 128), device=dev)
        pl_w = torch.empty((g.num_seqs, 32, slots), device=dev)

        def work(d_items=d_items, po_w=po_w, pl_w=pl_w):
            pa.pa_decode_work(po_w, pl_w, d_items, g.q, g.k_pool, g.v_pool, g.block_table,
                              g.seq_lens, g.scale)
            pa.pa_merge(out, po_w, pl_w)

        med3, _ = _time_launches(work, torch, flush, iters=10)
        planned.append({"target_ctas": sms * mult, "items": len(items), "max_slots": slots,
                        "us": 1e3 * med3, "plan_host_us": plan_us,
                        "gbs": (rb + split_bytes(g.num_seqs, 32, slots, 128)) / (med3 * 1e-3) / 1e9})
        del po_w, pl_w, d_items
    res["planned"] = planned
    res["frac_best"] = max([res["gbs_single_pass"], res["gbs_split64"]] +
                           [x["gbs"] for x in planned]) / peak
    del g, out, po, pl
    torch.cuda.empty_cache()
    return compact_ragged(res), res


def chunk(pa, workloads, torch, dev, peak):
    """Chunked multi-query read (pa_decode_chunk) on the llama1b batch at history 4096:
    every sequence brings n_q queries (causal), K/V read once per (sequence, kv head)."""
    flush = L2Flush(torch, dev)
    g = workloads.llama1b(4096, device=str(dev))
    rows = []
    for n_q in (1, 4, 16, 64):
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        q = torch.randn((64, n_q, 32, 64), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        fn = lambda: pa.pa_decode_chunk(out, q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                        g.scale)
        med, _ = _time_launches(fn, torch, flush, iters=20)
        lens = g.lens_list()
        kvb = read_bytes(lens, 32, 8, 64, 2, 16) + 2 * 64 * (n_q - 1) * 32 * 64 * 2
        flops = sum(4 * 32 * 64 * (n - n_q + i + 1) for n in lens for i in range(n_q))
        rows.append({"n_q": n_q, "us": 1e3 * med, "gbs": kvb / (med * 1e-3) / 1e9,
                     "frac_hbm": kvb / (med * 1e-3) / 1e9 / peak,
                     "tflops": flops / (med * 1e-3) / 1e12})
        del q, out
    del g
    torch.cuda.empty_cache()
    lc = chunk_longctx(pa, workloads, torch, dev, peak, flush)
    detail = {"llama1b_h4096": rows, "longctx_h32768_split": lc}
    return compact_chunk(detail), detail


def chunk_longctx(pa, workloads, torch, dev, peak, flush):
    """The chunked read on the long-context batch (8 x 32,768 tokens, head_dim 128): split
    into 64-page runs (pa_decode_chunk_splitkv + pa_merge) against one pass."""
    g = workloads.longctx(32768, device=str(dev))
    lens = g.lens_list()
    pps = g.pages_per_split
    s = pa.pa_num_splits(g.max_blocks, pps)
    rows = []
    for n_q in (1, 4, 16):
        gen = torch.Generator(device=dev)
        gen.manual_seed(9)
        q = torch.randn((8, n_q, 32, 128), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        po = torch.empty((8, n_q, 32, s, 128), device=dev)
        pl = torch.empty((8, n_q, 32, s), device=dev)

        def fn():
            pa.pa_decode_chunk_splitkv(po, pl, q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                       g.scale, pps)
            pa.pa_merge(out, po, pl)

        med, _ = _time_launches(fn, torch, flush, iters=20)
        one = lambda: pa.pa_decode_chunk(out, q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                         g.scale)
        med1, _ = _time_launches(one, torch, flush, iters=5)
        rb = (read_bytes(lens, 32, 8, 128, 2, 16) + 2 * 8 * (n_q - 1) * 32 * 128 * 2 +
              split_bytes(8 * n_q, 32, s, 128))
        rows.append({"n_q": n_q, "splits": s, "us_split_plus_merge": 1e3 * med,
                     "gbs": rb / (med * 1e-3) / 1e9, "frac_hbm": rb / (med * 1e-3) / 1e9 / peak,
                     "us_single_pass": 1e3 * med1})
        del q, out, po, pl
    del g
    torch.cuda.empty_cache()
    return rows


def launch_floor(pa, workloads, torch, dev, peak):
    """The read's fixed cost per launch at history 1024 (B 64): the same batch with every
    length 0 (the same 512-CTA grid, reading only q and the lengths) beside the real read,
    and two events with nothing between them, each after an L2 flush; then the read in a
    loop of back-to-back launches.  Launch order (for an ncu capture of decode_mma): 3 + 30
    empty reads, then 3 + 30 real ones, then 60 warm-up and 20 timed loop launches."""
    flush = L2Flush(torch, dev)
    g = workloads.llama1b(1024, device=str(dev))
    out = torch.empty_like(g.q)
    zero = torch.zeros_like(g.seq_lens)
    empty = lambda: pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, zero, g.scale)
    real = lambda: pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale)
    e_med, e_min = _time_launches(empty, torch, flush)
    r_med, r_min = _time_launches(real, torch, flush)
    n_med, n_min = _time_launches(lambda: None, torch, flush)
    rb = read_bytes(g.lens_list(), 32, 8, 64, 2, 16)
    detail = {"us_events_alone": 1e3 * n_med, "us_empty_read": 1e3 * e_med,
              "us_read_h1024": 1e3 * r_med, "us_read_h1024_min": 1e3 * r_min,
              "frac_read_h1024": rb / (r_med * 1e-3) / 1e9 / peak}
    # A decode loop: the read launched back to back, as a serving step issues it, on two
    # batches in turn (their K/V, 2 x 134.5 MB, exceed L2, so each read comes from DRAM).
    # The timed loop lies between cudaProfilerStart and cudaProfilerStop, so that an ncu
    # range replay (--replay-mode range --profile-from-start off) measures exactly it.
    g2 = workloads.make_batch("llama1b_h1024_second", seed=5, dtype="bf16", lens=[1024] * 64,
                              num_q_heads=32, num_kv_heads=8, head_dim=64, block_size=16,
                              num_pages=20000, device=str(dev))
    out2 = torch.empty_like(g2.q)
    real2 = lambda: pa.pa_decode(out2, g2.q, g2.k_pool, g2.v_pool, g2.block_table,
                                 g2.seq_lens, g2.scale)
    n_loop = 20
    for _ in range(3):
        for i in range(n_loop):
            (real if i % 2 == 0 else real2)()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.profiler.start()
    start.record()
    for i in range(n_loop):
        (real if i % 2 == 0 else real2)()
    stop.record()
    torch.cuda.profiler.stop()
    torch.cuda.synchronize()
    loop_us = 1e3 * start.elapsed_time(stop) / n_loop
    detail.update({"us_read_h1024_in_loop": loop_us, "loop_launches": n_loop,
                   "frac_read_h1024_in_loop": rb / (loop_us * 1e-6) / 1e9 / peak})
    del g, out, g2, out2
    torch.cuda.empty_cache()
    return {k: detail[k] for k in ("us_empty_read", "us_read_h1024",
                                   "us_read_h1024_in_loop")}, detail


def f32_read(pa, workloads, torch, dev, peak):
    """The fp32 read (CUDA cores) on llama1b-shaped batches (B 64, Hq 32 / Hkv 8) at
    head_dim 64 and 128, histories 1024 and 4096, L2 flushed before each launch."""
    flush = L2Flush(torch, dev)
    rows = []
    for d in (64, 128):
        for h in (1024, 4096):
            g = workloads.make_batch(f"f32_d{d}_h{h}", 2, "f32", [h] * 64, 32, 8, d, 16,
                                     64 * (h // 16) + 16, device=str(dev))
            out = torch.empty_like(g.q)
            fn = lambda: pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                      g.scale)
            med, mn = _time_launches(fn, torch, flush, iters=20)
            rb = read_bytes(g.lens_list(), 32, 8, d, 4, 16)
            rows.append({"head_dim": d, "history": h, "us_median": 1e3 * med, "us_min": 1e3 * mn,
                         "gbs": rb / (med * 1e-3) / 1e9, "frac": rb / (med * 1e-3) / 1e9 / peak})
            del g, out
            torch.cuda.empty_cache()
    return {f"d{r['head_dim']}_h{r['history']}": r["frac"] for r in rows}, rows


def measured_bf16_tflops():
    """Dense bf16 tensor peak (TFLOP/s) measured on this machine, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        for key in ("bf16_tflops", "bf16_tflops_burst"):
            if isinstance(j.get(key), (int, float)):
                return float(j[key]), "measured"
    except (OSError, ValueError):
        pass
    return 1900.0, "fallback"


def prefill(pa, workloads, torch, dev):
    """Causal prefill of 8 prompts x 4096 tokens through pa_decode_chunk (chunk = the whole
    prompt, tcgen05 path), head_dim 64 (Llama-3.2-1B heads) and 128 (Llama-3-8B heads)."""
    flush = L2Flush(torch, dev)
    peak_tf, kind = measured_bf16_tflops()
    rows = []
    for d in (64, 128):
        g = workloads.make_batch(f"prefill_d{d}", 6, "bf16", [4096] * 8, 32, 8, d, 16, 8 * 256,
                                 device=str(dev))
        gen = torch.Generator(device=dev)
        gen.manual_seed(8)
        q = torch.randn((8, 4096, 32, d), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        fn = lambda: pa.pa_decode_chunk(out, q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                        g.scale)
        med, mn = _time_launches(fn, torch, flush, iters=10)
        flops = 8 * 4 * 32 * d * (4096 * 4097 // 2)
        tf = flops / (med * 1e-3) / 1e12
        rows.append({"head_dim": d, "batch": 8, "prompt": 4096, "us": 1e3 * med,
                     "tflops": tf, "peak_tflops": peak_tf, "peak_source": kind,
                     "frac_tensor": tf / peak_tf})
        del g, q, out
    torch.cuda.empty_cache()
    return compact_prefill(rows), rows


def dense_vs_sdpa(pa, workloads, torch, dev, peak):
    """Contiguous K/V (B 4, H 16, D 64, fp16) at 1K-16K: our read at every split count of
    the "Three Attention Kernels" sweep against torch SDPA on its own [B,H,N,D] layout."""
    flush = L2Flush(torch, dev)
    rows = []
    for n in workloads.DENSE_CONTEXTS:
        g = workloads.dense(n, device=str(dev))
        out = torch.empty_like(g.q)
        kvb = g.kv_bytes()
        ours = {}
        for splits in workloads.DENSE_SPLITS:
            if splits == 1:
                fn = lambda: pa.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table,
                                          g.seq_lens, g.scale)
            else:
                pps = max(1, g.max_blocks // splits)  # at least one page per split
                s = pa.pa_num_splits(g.max_blocks, pps)
                po = torch.empty((4, 16, s, 64), device=dev)
                pl = torch.empty((4, 16, s), device=dev)

                def fn(po=po, pl=pl, pps=pps):
                    pa.pa_decode_splitkv(po, pl, g.q, g.k_pool, g.v_pool, g.block_table,
                                         g.seq_lens, g.scale, pps)
                    pa.pa_merge(out, po, pl)
            ours[splits] = 1e3 * _time_launches(fn, torch, flush, iters=20)[0]
        k = g.k_pool.reshape(4, n, 16, 64).transpose(1, 2).contiguous()
        v = g.v_pool.reshape(4, n, 16, 64).transpose(1, 2).contiguous()
        q4 = g.q.unsqueeze(2)
        sdpa = lambda: torch.nn.functional.scaled_dot_product_attention(q4, k, v, scale=g.scale)
        t_sdpa = 1e3 * _time_launches(sdpa, torch, flush, iters=20)[0]
        best = min(ours, key=ours.get)
        rows.append({"n_ctx": n, "us_by_splits": {str(k_): round(v_, 2) for k_, v_ in ours.items()},
                     "best_splits": best, "us_best": ours[best], "us_sdpa": t_sdpa,
                     "gbs_best": kvb / (ours[best] * 1e-6) / 1e9,
                     "gbs_sdpa": kvb / (t_sdpa * 1e-6) / 1e9, "sdpa_over_ours": t_sdpa / ours[best]})
        del g, out, k, v
    torch.cuda.empty_cache()
    return compact_dense(rows), rows


if __name__ == "__main__":
    main()
