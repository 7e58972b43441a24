"""Benchmark of the ReplaySSM decode step on GB300.

Workload: one Nemotron-H-like Mamba-2 layer, batch 256 per GPU, 32 heads,
d = 64, n = 128, 8 k/q groups, fp32 checkpoint, bf16 v/k/q, ring buffer
L = 16, sequences starting at random fill levels 0..15.  A step is one
ReplaySSM decode step of the whole batch: output-only decode and, in the
same launch, the flush of every sequence whose buffer filled.  Inputs are seeded synthetic data.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on the host cores instead (bounded sample of the same workload).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from ssm_decode_hybrid_gb300 import workloads as wl  # noqa: E402

METRIC = "SSM decode tokens/s @batch256 (32h,d64,n128,L16); HBM GB/s vs GB300 peak"
WORKLOAD = "nemotron-h mamba-2 layer decode (B=256, H=32, G=8, d=64, n=128, L=16, fp32 state, bf16 v/k/q)"
POOL = 32  # distinct step inputs cycled through the timed steps


# ---------------------------------------------------------------------------
# algorithmic bytes (per sequence)
# ---------------------------------------------------------------------------


def m2_entry_bytes(s: wl.Mamba2Shape) -> int:
    """One ring entry of a sequence: v (H x d) + k (G x n) in the input dtype, dt (H) f32."""
    e = 2 if s.in_dtype == wl.BF16 else 4
    return s.H * s.d * e + s.G * s.n * e + s.H * 4


def m2_decode_bytes(s: wl.Mamba2Shape, h: int) -> int:
    """Bytes one decode step must move for one sequence with h committed entries:
    read S_0, the h buffered entries and this step's v, k, q, dt; write the new
    entry and y (f32)."""
    e = 2 if s.in_dtype == wl.BF16 else 4
    s0 = 4 * s.H * s.d * s.n
    inputs = s.H * s.d * e + 2 * s.G * s.n * e + s.H * 4
    return s0 + h * m2_entry_bytes(s) + inputs + m2_entry_bytes(s) + 4 * s.H * s.d


def m2_flush_bytes(s: wl.Mamba2Shape, c: int) -> int:
    """Flush of one sequence with c entries: read + write S_0, read the entries."""
    return 8 * s.H * s.d * s.n + c * m2_entry_bytes(s)


def m2_fused_flush_extra_bytes(s: wl.Mamba2Shape) -> int:
    """Extra bytes of a flush fused into the decode step: only the S_0 write,
    since S_0 and the entries were already read for the output."""
    return 4 * s.H * s.d * s.n


def m2_baseline_bytes(s: wl.Mamba2Shape) -> int:
    e = 2 if s.in_dtype == wl.BF16 else 4
    return 8 * s.H * s.d * s.n + s.H * s.d * e + 2 * s.G * s.n * e + s.H * 4 + 4 * s.H * s.d


def fill_trace(count0: np.ndarray, L: int, steps: int):
    """Committed count of every sequence at the start of each decode step, and
    the number of entries flushed after it (0 if none), for `steps` steps."""
    h = np.empty((steps, count0.size), dtype=np.int64)
    c = count0.astype(np.int64).copy()
    for t in range(steps):
        h[t] = c
        c = c + 1
        c[c == L] = 0
    return h


# ---------------------------------------------------------------------------
# multi-rank helpers (one process per GPU; ranks hold independent batches)
# ---------------------------------------------------------------------------


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(units_per_rank: int, world: int, elapsed_ms_max: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank * world / (elapsed_ms_max * 1e-3)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


HEADLINE_SOURCES = ("decode_split.cu", "common.cuh", "kernels.cuh")  # the headline kernels and their headers
# the capture the recorded DRAM traffic comes from (run after the same command without ncu exited 0)
HEADLINE_SMALL = "python bench.py --no-cpu-baseline --no-extra --windows 1 --steps 64 --warmup 8 --e2e-steps 16"
TRAFFIC_COMMAND = (f"{HEADLINE_SMALL} && ncu --set full --import-source no --clock-control none "
                   f"-k regex:\"m2_(prep|stream)_kernel\" -s 8 -c 2 -o prof {HEADLINE_SMALL}")


def source_digest(names=None) -> str:
    """Digest of the named sources under csrc/ (default: every .cu/.cuh file)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ssm_decode_hybrid_gb300", "csrc")
    if names is None:
        names = [n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh"))]
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


LAUNCHES_PER_STEP = 2  # replay_decode_step_fused with a workspace: precompute + streaming kernel


def recorded_traffic(*kernels: str):
    """DRAM bytes of one launch of each of `kernels`, summed, from the committed
    ncu summary; None if the summary is missing, lacks one of them, or was
    taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_digest") != source_digest(rec.get("sources")):
        return None
    total = 0.0
    for kernel in kernels:
        k = rec.get("kernels", {}).get(kernel)
        if not k or k.get("dram_bytes_per_launch") is None:
            return None
        total += k["dram_bytes_per_launch"]
    return total


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int | None):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu is not None:
            cmd += ["-i", str(self.gpu)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (spawned workers; never forked after CUDA init)
# ---------------------------------------------------------------------------


def _oracle_worker(args):
    seed, seqs, min_seconds, max_steps = args
    from oracle import mamba2 as om

    shape = wl.Mamba2Shape(B=seqs, H=32, G=8, d=64, n=128, L=16, in_dtype=wl.BF16)
    init = wl.mamba2_init(shape, seed)
    orc = om.Mamba2Replay(init.S0, init.A, init.ring_v, init.ring_k, init.ring_dt, init.start, init.count)
    steps = [wl.mamba2_step(shape, seed, t) for t in range(4)]
    t0 = time.perf_counter()
    n = 0
    while n < max_steps and (n < 2 or time.perf_counter() - t0 < min_seconds):
        st = steps[n % len(steps)]
        orc.decode_step(st.v, st.k, st.q, st.dt)
        orc.flush()
        n += 1
    return n * seqs, time.perf_counter() - t0


def oracle_throughput(seconds: float = 12.0, seqs_per_worker: int = 2):
    """tokens/s of the fp64 oracle (decode step + flush) over all host cores."""
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    jobs = [(5000 + w, seqs_per_worker, seconds, 100000) for w in range(cores)]
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, jobs)
    wall = time.perf_counter() - t0
    tokens = sum(r[0] for r in res)
    slowest = max(r[1] for r in res)
    return {"value": tokens / slowest, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"{cores} spawned processes x {seqs_per_worker} sequences of the B=256 layer shape, "
                       f"fp64 numpy decode step + flush, >= {seconds:.0f} s each; {tokens} sequence-steps, "
                       f"{wall:.1f} s wall")}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


def workload_config(world: int) -> dict:
    """The benchmarked workload, shared by both arms of the benchmark."""
    s = wl.NEMOTRON_H_MAMBA2
    return {"workload": WORKLOAD, "batch_per_gpu": s.B, "H": s.H, "G": s.G, "d": s.d, "n": s.n, "L": s.L,
            "inputs": "bf16 v/k/q, f32 dt/A, f32 S_0", "fill": "random 0..15 at start",
            "l2": "inputs larger than L2 (S_0 is 256 MiB per GPU; no L2 flush)",
            "parallelism": f"replicas x{world} (independent batches, no collective)"}


STEP_DESCRIPTION = ("replay_decode_step_fused with the decode workspace: a precompute launch and an S_0 streaming "
                    "launch (programmatic dependent launch) that also folds full buffers; the K steps of a window "
                    "are captured once in a CUDA graph and the graph is replayed, as a serving loop does")


def graph_windows(step, K: int, reps: int, world: int, dev, sync_ranks):
    """Capture step(t), t = 0..K-1, in one CUDA graph on a side stream, replay
    it once untimed, then `reps` timed windows of exactly K steps, each
    bracketed by a barrier and a device synchronisation, timed with CUDA
    events on the replaying stream; returns each window's milliseconds, the
    maximum over ranks."""
    import torch

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(K):
            step(t)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    out = []
    for _ in range(reps):
        sync_ranks()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(max_over_ranks(e0.elapsed_time(e1), dev))
    del g
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    def sync_ranks():
        if world > 1:
            dist.barrier()

    # the oracle baseline runs before the first CUDA work of this process
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        cpu = oracle_throughput(args.cpu_seconds)

    from ssm_decode_hybrid_gb300 import replayssm as R

    shape = wl.NEMOTRON_H_MAMBA2
    seed = wl.SEED_NEMOTRON + 7919 * rank
    init = wl.mamba2_init(shape, seed)

    def to(x, dt=torch.float32):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dt).to(dev)

    state = R.Mamba2State(to(init.S0), to(init.ring_v, torch.bfloat16), to(init.ring_k, torch.bfloat16),
                          to(init.ring_dt), to(init.start, torch.int32), to(init.count, torch.int32),
                          torch.zeros(shape.B, dtype=torch.int32, device=dev),
                          torch.zeros(shape.B, dtype=torch.int32, device=dev),
                          torch.zeros(1, dtype=torch.int32, device=dev)).add_workspace()
    A = to(init.A)
    host_in = []
    for p in range(POOL):
        st = wl.mamba2_step(shape, seed, p)
        host_in.append(tuple(torch.from_numpy(np.ascontiguousarray(x)).to(dt).pin_memory()
                             for x, dt in ((st.v, torch.bfloat16), (st.k, torch.bfloat16),
                                           (st.q, torch.bfloat16), (st.dt, torch.float32))))
    dev_in = [tuple(x.to(dev) for x in h) for h in host_in]
    y = torch.empty(shape.B, shape.H, shape.d, device=dev)
    stream = torch.cuda.current_stream()

    W, K, REPS = args.warmup, args.steps, args.windows
    # steps run in order: W warm-up, one eager window of K, the graph's untimed
    # replay of K, then REPS timed windows of K
    trace = fill_trace(init.count, shape.L, W + K * (2 + REPS))
    per_h = np.array([m2_decode_bytes(shape, h) for h in range(shape.L)], dtype=np.int64)

    def window_bytes(first):
        h = trace[first:first + K]
        return int(per_h[h].sum()) + int((h + 1 == shape.L).sum()) * m2_fused_flush_extra_bytes(shape)

    for t in range(W):
        R.replay_decode_step_fused(state, *dev_in[t % POOL], A, y=y)
    torch.cuda.synchronize()
    sync_ranks()

    gpu_index = None
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis and vis.split(",")[local_rank].strip().isdigit():
        gpu_index = int(vis.split(",")[local_rank])
    elif vis is None:
        gpu_index = local_rank
    with ClockSampler(gpu_index) as clk:
        # one window with every step launched from the host through the public call
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for t in range(K):
            R.replay_decode_step_fused(state, *dev_in[(W + t) % POOL], A, y=y)
        ev1.record(stream)
        torch.cuda.synchronize()
        eager_ms = max_over_ranks(ev0.elapsed_time(ev1), dev)
        # the headline: the same steps captured once, replayed as timed windows of K steps
        first = W + K
        win_ms = graph_windows(lambda t: R.replay_decode_step_fused(state, *dev_in[(first + t) % POOL], A, y=y),
                               K, REPS, world, dev, sync_ranks)
    sync_ranks()
    clocks = clk.summary()
    err = int(state.err.item())
    win_bytes = [window_bytes(W + K * (2 + r)) for r in range(REPS)]
    order = np.argsort(win_ms)
    med = int(order[len(order) // 2])
    elapsed_ms = win_ms[med]
    step_bytes = win_bytes[med] / K
    achieved = step_bytes / (elapsed_ms / K * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    value = whole_job_throughput(shape.B * K, world, elapsed_ms)
    flushed_share = (win_bytes[med] - int(per_h[trace[W + K * (2 + med):W + K * (3 + med)]].sum())) / win_bytes[med]

    # the same steps as two calls: decode step, then the separate flush
    for t in range(W):
        R.replay_decode_step(state, *dev_in[t % POOL], A, y=y)
        R.replay_flush(state, A)
    torch.cuda.synchronize()

    def unfused(t):
        R.replay_decode_step(state, *dev_in[t % POOL], A, y=y)
        R.replay_flush(state, A)

    unfused_ms = statistics.median(graph_windows(unfused, K, REPS, world, dev, sync_ranks)) / K

    # baseline kernel on the same inputs (reads + writes the whole state), timed the same way
    S = to(init.S0)
    for t in range(W):
        R.ssm_state_update_baseline(S, *dev_in[t % POOL], A, y=y)
    torch.cuda.synchronize()
    base_ms = statistics.median(graph_windows(
        lambda t: R.ssm_state_update_baseline(S, *dev_in[t % POOL], A, y=y), K, REPS, world, dev, sync_ranks)) / K
    base_gbs = m2_baseline_bytes(shape) * shape.B / (base_ms * 1e-3) / 1e9
    del S

    # end to end through the public call with host buffers.  Each step's v, k,
    # q and dt sit back to back in one pinned host buffer and arrive with one
    # H2D copy into a device staging buffer whose typed views the call takes; y
    # goes back with one D2H copy (a copy call costs the host far less than
    # four).  A step's synthetic inputs do not depend on earlier outputs, so the
    # copies run on a stream of their own beside the neighbouring steps'
    # kernels: once step t's kernels are done, its y is read back and step
    # t+2's inputs are copied into the buffer it used (two staging buffers, two
    # y buffers).  Every step's H2D and D2H copy lands inside the timed region,
    # which ends when the copy stream has drained.  The same steps with every
    # copy on the compute stream, in order, are reported beside it.
    sizes = [x.numel() * x.element_size() for x in host_in[0]]
    h2d = sum(sizes)
    offs = [sum(sizes[:i]) for i in range(len(sizes))]
    assert all(o % 16 == 0 for o in offs), "each input view starts on a 16-byte boundary"

    def packed_host(parts):
        buf = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        for x, o, n in zip(parts, offs, sizes):
            buf[o:o + n].copy_(x.reshape(-1).view(torch.uint8))
        return buf

    def typed_views(buf):
        return tuple(buf[o:o + n].view(x.dtype).view(x.shape) for x, o, n in zip(host_in[0], offs, sizes))

    host_packed = [packed_host(h) for h in host_in]
    for h, p in zip(host_in, host_packed):
        assert all(torch.equal(a, b) for a, b in zip(h, typed_views(p))), "packed inputs equal the step's inputs"
    NB, G = 8, 4  # staging and y buffers; the compute stream waits for G steps' copies at once
    staging = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(NB)]
    staged = [typed_views(b) for b in staging]
    ys = [y] + [torch.empty_like(y) for _ in range(NB - 1)]
    y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(NB)]
    d2h = y_host[0].numel() * y_host[0].element_size()
    copy_stream = torch.cuda.Stream(device=dev)
    computed = torch.cuda.Event()
    copied = [torch.cuda.Event() for _ in range(NB)]
    origin = [0]  # the first step after the last inputs_ahead: wait groups start there
    Ke = args.e2e_steps  # its own count: a 20-step window is too short to average the host's per-call costs

    def inputs_ahead(t0):
        # steps t0 .. t0 + NB - 1 find their inputs in place
        origin[0] = t0
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_stream(stream)  # earlier steps are done with every buffer
            for j in range(NB):
                staging[(t0 + j) % NB].copy_(host_packed[(t0 + j) % POOL], non_blocking=True)
                copied[(t0 + j) % NB].record(copy_stream)

    def e2e_step(st, t):
        # called with the copy stream current, so that the copies need no
        # stream switch; the decode call names the compute stream.  A wait on
        # the compute stream between two decode calls costs the programmatic
        # overlap of one step's S_0 stream with the next step's precompute
        # (about 2.5 us), so the compute stream waits once every G steps, for
        # the next G steps' inputs (copied NB - G or more steps earlier) and for
        # the reads of the y buffers those steps overwrite.
        i = t % NB
        if (t - origin[0]) % G == 0:
            for j in range(G):
                stream.wait_event(copied[(t + j) % NB])
        R.replay_decode_step_fused(st, *staged[i], A, y=ys[i], stream=stream)
        computed.record(stream)
        copy_stream.wait_event(computed)
        y_host[i].copy_(ys[i], non_blocking=True)
        staging[i].copy_(host_packed[(t + NB) % POOL], non_blocking=True)
        copied[i].record(copy_stream)

    def serial_step(st, t):
        staging[0].copy_(host_packed[t % POOL], non_blocking=True)
        R.replay_decode_step_fused(st, *staged[0], A, y=ys[0])
        y_host[0].copy_(ys[0], non_blocking=True)

    # 2 NB overlapped steps (no synchronisation between them, every buffer used
    # twice) leave the state and the last NB outputs of as many serial steps,
    # bit for bit
    fields = [f.name for f in dataclasses.fields(state) if getattr(state, f.name) is not None]
    twins = [dataclasses.replace(state, **{f: getattr(state, f).clone() for f in fields}) for _ in range(2)]
    inputs_ahead(0)
    with torch.cuda.stream(copy_stream):
        for t in range(2 * NB):
            e2e_step(twins[0], t)
    stream.wait_stream(copy_stream)
    torch.cuda.synchronize()
    last = [y_host[t % NB].clone() for t in range(NB, 2 * NB)]
    for t in range(2 * NB):
        serial_step(twins[1], t)
        torch.cuda.synchronize()
        if t >= NB:
            assert torch.equal(last[t - NB], y_host[0]), "overlapped copies changed a step's output"
    for f in fields:
        assert torch.equal(getattr(twins[0], f), getattr(twins[1], f)) or f == "work", f"overlapped copies changed {f}"
    del twins

    def e2e_window(step, first, overlapped):
        torch.cuda.synchronize()
        sync_ranks()
        if overlapped:
            inputs_ahead(first)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(copy_stream if overlapped else stream):
            for t in range(Ke):
                step(state, first + t)
        stream.wait_stream(copy_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), dev)

    Wu = max(W, 16)
    inputs_ahead(0)
    with torch.cuda.stream(copy_stream):
        for t in range(Wu):
            e2e_step(state, t)
    stream.wait_stream(copy_stream)
    e2e_ms = e2e_window(e2e_step, Wu, True)
    e2e_value = whole_job_throughput(shape.B * Ke, world, e2e_ms)
    e2e_serial_ms = e2e_window(serial_step, Wu + Ke, False)
    e2e_serial_value = whole_job_throughput(shape.B * Ke, world, e2e_serial_ms)

    # the speculative (B = 512, T = 4) and GDN (B = 256) workloads, short graph-timed runs
    extra = {}
    if not args.no_extra:
        extra = extra_workloads(R, peak)

    if rank == 0:
        traffic = recorded_traffic("m2_prep_kernel<fused>", "m2_stream_kernel<fused>")
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": elapsed_ms / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": workload_config(world),
            "step": STEP_DESCRIPTION,
            "windows": {"count": REPS, "steps_each": K, "reported": "median window",
                        "ms": win_ms, "median_ms": elapsed_ms, "min_ms": min(win_ms), "max_ms": max(win_ms)},
            "hbm_gbs_step": achieved,
            "roofline": {"bound": "hbm",
                         "kernel": "one decode step: m2_prep_kernel<fused> + m2_stream_kernel<fused> "
                                   "(replay_decode_step_fused), timed together",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "traffic": traffic,
                         "algorithmic_bytes_per_launch": step_bytes,
                         "avg_launch_ms": elapsed_ms / K},
            "eager_window": {"calls": "every step launched from the host through the public call",
                             "ms_per_step": eager_ms / K, "tokens_per_s": shape.B * world / (eager_ms / K * 1e-3)},
            "baseline_kernel": {"name": "ssm_state_update_baseline", "ms_per_step": base_ms,
                                "tokens_per_s": shape.B * world / (base_ms * 1e-3), "gbs": base_gbs,
                                "frac": base_gbs / peak},
            "replay_over_baseline": base_ms / (elapsed_ms / K),
            "unfused_two_launch_step": {"calls": "replay_decode_step + replay_flush", "ms_per_step": unfused_ms,
                                        "tokens_per_s": shape.B * world / (unfused_ms * 1e-3),
                                        "replay_over_baseline": base_ms / unfused_ms},
            "flush_share_bytes": flushed_share,
            **extra,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": Ke, "ms_per_step": e2e_ms / Ke,
                    "calls": "each step from the host: replay_decode_step_fused on the compute stream; one H2D "
                             "copy of a later step's packed v/k/q/dt and one D2H copy of y on a copy stream, "
                             "overlapping other steps' kernels (8 staging and y buffers; the compute stream "
                             "waits for the copies once every 4 steps)",
                    "serial": {"value": e2e_serial_value, "ms_per_step": e2e_serial_ms / Ke,
                               "calls": "the same steps with both copies on the compute stream, in order"}},
            "gpu_launches": LAUNCHES_PER_STEP * K,
            "gpu_launches_note": "per timed window of K steps (precompute + stream per step)",
            "clocks": clocks,
            "device_error_word": err,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def extra_workloads(R, peak) -> dict:
    """Keys for the speculative workload (Mamba-2 layer, B = 512, T = 4) and
    the GDN layer (B = 256; decode and T = 4 verify), from short CUDA-graph
    timed runs of the window sweep restricted to T = 4."""
    rows = suite_sweep(R, peak, steps=4, Ts=(4,), emit=False)
    m2 = next(r for r in rows if r["model"] == "mamba2")
    gd = next(r for r in rows if r["model"] == "gdn")
    return {
        "spec_round_b512_t4": {
            "workload": m2["workload"], "calls": m2["calls"],
            "timing": m2["timing"], "rounds": m2["rounds"], "ms_per_round": m2["ms_per_round"],
            "gbs": m2["gbs"], "frac": m2["frac_of_peak"], "accepted_tokens_per_s": m2["accepted_tokens_per_s"],
            "snapshot_baseline_ms_per_round": m2["baseline_ms_per_round"],
            "replay_over_snapshot": m2["replay_over_baseline"], "round_over_decode": m2["round_over_decode"],
            "device_error_word": m2["device_error_word"]},
        "gdn_b256": {
            "workload": "GDN layer B=256, Hv=32, Hk=16, d_k=d_v=128, L=16, u f32",
            "decode_fused_ms_per_step": gd["decode_step_ms"], "decode_gbs": gd["decode_gbs"],
            "decode_frac": gd["decode_gbs"] / peak,
            "baseline_decode_ms_per_step": gd["baseline_decode_step_ms"],
            "decode_replay_over_baseline": gd["baseline_decode_step_ms"] / gd["decode_step_ms"],
            "verify_t4_ms_per_round": gd["ms_per_round"], "verify_round_over_decode": gd["round_over_decode"],
            "verify_gbs": gd["gbs"], "verify_frac": gd["frac_of_peak"],
            "snapshot_baseline_ms_per_round": gd["baseline_ms_per_round"],
            "verify_replay_over_snapshot": gd["replay_over_baseline"],
            "device_error_word": gd["device_error_word"]},
    }


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # each step is a bounded sample: every host core runs the oracle on its own
    # sequences for a fixed slice of time; value is sequence-steps per second
    W, K = args.warmup, args.steps
    per_step = max(0.5, min(2.0, 120.0 / max(1, K + W)))
    vals = []
    for i in range(W + K):
        r = oracle_throughput(per_step, seqs_per_worker=1)
        if i >= W:
            vals.append(r)
    value = statistics.median(v["value"] for v in vals)
    cores = vals[-1]["cores"]
    ms_per_step = 1e3 * wl.NEMOTRON_H_MAMBA2.B / value
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(world),
        "step": "oracle decode step + flush (fp64, CPU, host cores)",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {cores} spawned processes x 1 sequence for {per_step:.1f} s"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# measurement suite (--suite): the other workloads, one JSON line each
# ---------------------------------------------------------------------------


def m2_verify_bytes(s: wl.Mamba2Shape, h: int, T: int) -> int:
    """One verify round of one sequence with h committed entries: S_0, the h
    entries, T drafts' v/k/q/dt, the T tentative entries written, T outputs."""
    e = 2 if s.in_dtype == wl.BF16 else 4
    inputs = s.H * s.d * e + 2 * s.G * s.n * e + s.H * 4
    return 4 * s.H * s.d * s.n + h * m2_entry_bytes(s) + T * (inputs + m2_entry_bytes(s) + 4 * s.H * s.d)


def m2_snapshot_verify_bytes(s: wl.Mamba2Shape, T: int) -> int:
    """Snapshot baseline round: read one state slot, write T slots, T drafts' inputs and outputs."""
    e = 2 if s.in_dtype == wl.BF16 else 4
    inputs = s.H * s.d * e + 2 * s.G * s.n * e + s.H * 4
    return (T + 1) * 4 * s.H * s.d * s.n + T * (inputs + 4 * s.H * s.d)


def gdn_entry_bytes(s: wl.GdnShape) -> int:
    eu = 4 if s.u_dtype == wl.F32 else 2
    ek = 2 if s.in_dtype == wl.BF16 else 4
    return s.Hv * s.dv * eu + s.Hk * s.dk * ek + s.Hv * 4


def gdn_input_bytes(s: wl.GdnShape) -> int:
    e = 2 if s.in_dtype == wl.BF16 else 4
    return 2 * s.Hk * s.dk * e + s.Hv * s.dv * e + 2 * s.Hv * 4


def gdn_decode_bytes(s: wl.GdnShape, h: int) -> int:
    return 4 * s.Hv * s.dv * s.dk + h * gdn_entry_bytes(s) + gdn_input_bytes(s) + gdn_entry_bytes(s) + 4 * s.Hv * s.dv


def gdn_flush_bytes(s: wl.GdnShape, c: int) -> int:
    return 8 * s.Hv * s.dv * s.dk + c * gdn_entry_bytes(s)


def gdn_baseline_bytes(s: wl.GdnShape) -> int:
    return 8 * s.Hv * s.dv * s.dk + gdn_input_bytes(s) + 4 * s.Hv * s.dv


def gdn_verify_bytes(s: wl.GdnShape, h: int, T: int) -> int:
    return 4 * s.Hv * s.dv * s.dk + h * gdn_entry_bytes(s) + T * (gdn_input_bytes(s) + gdn_entry_bytes(s) +
                                                                   4 * s.Hv * s.dv)


def gdn_snapshot_verify_bytes(s: wl.GdnShape, T: int) -> int:
    return (T + 1) * 4 * s.Hv * s.dv * s.dk + T * (gdn_input_bytes(s) + 4 * s.Hv * s.dv)


def _time_graph(fn, K: int, W: int, reps: int = 8) -> float:
    """Milliseconds per call of fn(i), with K calls (i = 0..K-1) captured in one
    CUDA graph and the graph replayed `reps` times after W warm-up replays."""
    import torch

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(K):
                fn(i)
    torch.cuda.synchronize()
    for _ in range(W):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / (reps * K)


def _time_loop(fn, K: int, W: int) -> float:
    """Milliseconds per call of fn(i) over K calls after W warm-up calls (CUDA events)."""
    import torch

    for i in range(W):
        fn(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        fn(W + i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / K


def _dev(x, dt=None):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x))
    return (t.to(dt) if dt is not None else t).cuda()


def suite_layers(R, peak, steps=None):
    """Layer-stack sweep: 23 independent Nemotron-H Mamba-2 layers per step,
    batch B in {1, 8, 64, 256, 512} and ring capacity L in {4, 8, 16, 32}
    (the buffer-capacity trade-off of "Results -- standard decoding", Fig. 7).
    Every variant of a point is a 23-layer step captured in a CUDA graph of 16
    steps (as a serving loop would), replayed until 512 steps are timed; byte
    accounting follows each sequence's fill level through the replays.
    Variants: the fused decode step with a workspace (the reported one), the
    same without a workspace (one launch per layer), the decode step plus a
    separate replay_flush, the decode step alone with every layer's counts
    restored after each step (no buffer ever fills, same mean fill: what the
    step costs without any flush), and the baseline state update.  The flush
    cost share of a point is (decode + flush - decode alone) / (decode +
    flush), and for the fused step (fused - decode alone) / fused, next to
    the share of the bytes the flush moves.  A last line names the best L
    per batch."""
    import torch

    LAYERS, out = 23, []
    K, W = 16, 3
    reps = max(1, (steps or 512) // K)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    best = {}
    for bi, B in enumerate((1, 8, 64, 256, 512)):
        base_ms = None
        for li, L in enumerate((4, 8, 16, 32)):
            shape = wl.Mamba2Shape(B=B, H=32, G=8, d=64, n=128, L=L, in_dtype=wl.BF16)
            seed = wl.SEED_SWEEP + 100 * (bi * 4 + li)
            layers = []
            count_all = torch.empty(LAYERS, B, dtype=torch.int32, device="cuda")
            for layer in range(LAYERS):
                t = wl.mamba2_state_tensors_device(shape, seed + layer, "cuda")
                count_all[layer].copy_(t["count"])
                z = lambda n: torch.zeros(n, dtype=torch.int32, device="cuda")  # noqa: E731
                st = R.Mamba2State(t["S0"], t["ring_v"], t["ring_k"], t["ring_dt"], t["start"], count_all[layer],
                                   z(B), z(B), z(1)).add_workspace()
                layers.append((st, t["A"]))
            g = torch.Generator(device="cuda")
            g.manual_seed(seed + 999)
            pool = [(torch.randn(B, 32, 64, generator=g, device="cuda").to(torch.bfloat16),
                     torch.randn(B, 8, 128, generator=g, device="cuda").to(torch.bfloat16),
                     torch.randn(B, 8, 128, generator=g, device="cuda").to(torch.bfloat16),
                     torch.nn.functional.softplus(torch.randn(B, 32, generator=g, device="cuda")))
                    for _ in range(4)]
            y = torch.empty(B, 32, 64, device="cuda")
            per_h = np.array([m2_decode_bytes(shape, h) for h in range(L)], dtype=np.int64)
            steps_run = 1 + K * (W + reps)  # _time_graph: one eager call, then W + reps replays of K

            def timed_trace():
                """Fill levels of the timed steps, from every layer's counts now."""
                c = count_all.cpu().numpy()
                return [fill_trace(c[layer], L, steps_run)[-reps * K:] for layer in range(LAYERS)]

            def fused(i):
                for st, A in layers:
                    R.replay_decode_step_fused(st, *pool[i % 4], A, y=y)

            trs = timed_trace()
            ms = _time_graph(fused, K, W, reps)
            dec_b = sum(int(per_h[tr].sum()) for tr in trs) / (reps * K)
            fold_b = sum(int((tr + 1 == L).sum()) for tr in trs) * m2_fused_flush_extra_bytes(shape) / (reps * K)
            nbytes = dec_b + fold_b

            def pair(i):
                for st, A in layers:
                    R.replay_decode_step(st, *pool[i % 4], A, y=y)
                    R.replay_flush(st, A)

            trs = timed_trace()
            pair_ms = _time_graph(pair, K, W, reps)
            pair_flush_b = sum(int((tr + 1 == L).sum()) for tr in trs) * m2_flush_bytes(shape, L) / (reps * K)
            pair_dec_b = sum(int(per_h[tr].sum()) for tr in trs) / (reps * K)

            count0 = count_all.clone()

            def frozen(i):
                for st, A in layers:
                    R.replay_decode_step(st, *pool[i % 4], A, y=y)
                count_all.copy_(count0)

            def restore_only(i):
                count_all.copy_(count0)

            dec_ms = _time_graph(frozen, K, W, reps) - _time_graph(restore_only, K, W, reps)
            for st, _ in layers:  # flags the frozen steps left: a full buffer flags every step
                st.flag.zero_()
            # the same step without a workspace: one launch per layer
            works = [st.work for st, _ in layers]
            for st, _ in layers:
                st.work = None
            one_ms = _time_graph(fused, K, W, reps)
            for (st, _), wkt in zip(layers, works):
                st.work = wkt
            err = max(int(st.err.item()) for st, _ in layers)
            if base_ms is None:  # the baseline does not depend on L
                Ss = [st.S0.clone() for st, _ in layers]

                def bstep(i):
                    for S, (_, A) in zip(Ss, layers):
                        R.ssm_state_update_baseline(S, *pool[i % 4], A, y=y)

                base_ms = _time_graph(bstep, K, W, reps)
                del Ss
            gbs = nbytes / (ms * 1e-3) / 1e9
            line = {"suite": "layers", "workload": f"{LAYERS} Mamba-2 layers (H=32, G=8, d=64, n=128), B={B}, L={L}",
                    "B": B, "L": L, "layers": LAYERS, "steps": K * reps,
                    "timing": f"CUDA graph of {K} steps, {reps} replays timed",
                    "ms_per_step": ms, "tokens_per_s": B / (ms * 1e-3), "gbs": gbs, "frac_of_peak": gbs / peak,
                    "decode_plus_flush_ms_per_step": pair_ms, "decode_alone_ms_per_step": dec_ms,
                    "flush_cost_share": (pair_ms - dec_ms) / pair_ms,
                    "flush_byte_share": pair_flush_b / (pair_dec_b + pair_flush_b),
                    "fused_fold_cost_share": (ms - dec_ms) / ms,
                    "fused_fold_byte_share": fold_b / nbytes,
                    "one_launch_ms_per_step": one_ms,
                    "baseline_ms_per_step": base_ms, "replay_over_baseline": base_ms / ms,
                    "state_bytes": LAYERS * B * 32 * 64 * 128 * 4,
                    "state_fits_l2": LAYERS * B * 32 * 64 * 128 * 4 <= l2, "device_error_word": err}
            out.append(line)
            print(json.dumps(line), flush=True)
            if B not in best or line["tokens_per_s"] > best[B]["tokens_per_s"]:
                best[B] = line
            del layers, pool
            torch.cuda.empty_cache()
    summary = {"suite": "layers_best_L", "best_L_per_B": {str(B): r["L"] for B, r in best.items()},
               "tokens_per_s_at_best": {str(B): r["tokens_per_s"] for B, r in best.items()}}
    print(json.dumps(summary), flush=True)
    return out + [summary]


def _spec_pool(shape, seed, T, n):
    steps = [wl.mamba2_step(shape, seed, r, T=T) for r in range(n)]
    inp = [(_dev(s.v, _bf16()), _dev(s.k, _bf16()), _dev(s.q, _bf16()), _dev(s.dt)) for s in steps]
    acc = [_dev(wl.accepted_counts(shape.B, T, seed, r), _i32()) for r in range(n)]
    return inp, acc


def _bf16():
    import torch

    return torch.bfloat16


def _i32():
    import torch

    return torch.int32


def _m2_state(R, init):
    import torch

    B = init.shape.B
    z = lambda n: torch.zeros(n, dtype=torch.int32, device="cuda")  # noqa: E731
    return R.Mamba2State(_dev(init.S0), _dev(init.ring_v, _bf16()), _dev(init.ring_k, _bf16()), _dev(init.ring_dt),
                         _dev(init.start, _i32()), _dev(init.count, _i32()), z(B), z(B), z(1))


def suite_spec(R, peak, steps=None):
    """Speculative verify rounds, B=512, T=4, L=16, accepted ~ U{0..4}: replay
    (verify + device commit + flush of early-flagged sequences) vs the
    snapshot baseline (T+1 state slots)."""
    import torch

    shape, T, seed, P = wl.SPEC_MAMBA2, 4, wl.SEED_SPEC, 8
    init = wl.mamba2_init(shape, seed, fill_max=shape.L - T)
    inp, acc = _spec_pool(shape, seed, T, P)
    mk = lambda: _m2_state(R, init).add_workspace(max_T=T)  # noqa: E731
    A = _dev(init.A)
    y = torch.empty(shape.B, T, shape.H, shape.d, device="cuda")
    W, K = 4, steps or 256

    def make_round(st):
        def rnd(i):
            R.replay_spec_verify(st, *inp[i % P], A, y=y)
            R.replay_spec_commit(acc[i % P], st.count, T, shape.L, st.err)
            R.replay_flush(st, A)
        return rnd

    # the committed-count trace of these rounds, recorded on an untimed copy
    st = mk()
    h_tr, fl_tr, acc_tr = [], [], []
    for i in range(W + K):
        h_tr.append(st.count.cpu().numpy().astype(np.int64))
        R.replay_spec_verify(st, *inp[i % P], A, y=y)
        fl_tr.append(st.flag.cpu().numpy() != 0)
        R.replay_spec_commit(acc[i % P], st.count, T, shape.L, st.err)
        acc_tr.append(acc[i % P].cpu().numpy().astype(np.int64))
        R.replay_flush(st, A)
    del st
    st = mk()
    ms = _time_loop(make_round(st), K, W)
    err = int(st.err.item())
    nbytes = 0
    for i in range(W, W + K):
        h = h_tr[i]
        nbytes += sum(m2_verify_bytes(shape, int(x), T) for x in h)
        c = (h + acc_tr[i])[fl_tr[i]]
        nbytes += sum(m2_flush_bytes(shape, int(x)) for x in c)
    mean_acc = float(np.mean(acc_tr[W:]))
    del st
    torch.cuda.empty_cache()
    slots = torch.zeros(shape.B, T + 1, shape.H, shape.d, shape.n, device="cuda")
    slots[:, 0] = _dev(init.S0)
    cur = torch.zeros(shape.B, dtype=torch.int32, device="cuda")
    berr = torch.zeros(1, dtype=torch.int32, device="cuda")

    def brnd(i):
        R.ssm_spec_verify_baseline(slots, cur, *inp[i % P], A, y=y, err=berr)
        R.ssm_spec_commit_baseline(acc[i % P], cur, T, berr)

    bms = _time_loop(brnd, K, W)
    bbytes = m2_snapshot_verify_bytes(shape, T) * shape.B
    gbs = nbytes / K / (ms * 1e-3) / 1e9
    line = {"suite": "spec", "workload": "Mamba-2 layer B=512, T=4, L=16, accepted ~ U{0..4}",
            "rounds": K, "ms_per_round": ms, "rounds_per_s": 1e3 / ms,
            "accepted_tokens_per_s": shape.B * mean_acc / (ms * 1e-3), "gbs": gbs, "frac_of_peak": gbs / peak,
            "calls_per_round": "replay_spec_verify + replay_spec_commit + replay_flush",
            "baseline_ms_per_round": bms, "baseline_gbs": bbytes / (bms * 1e-3) / 1e9,
            "replay_over_baseline": bms / ms, "device_error_word": err | int(berr.item())}
    print(json.dumps(line), flush=True)
    del slots
    torch.cuda.empty_cache()
    return [line]


def _gdn_state(R, init):
    import torch

    B = init.shape.B
    ut = torch.float32 if init.shape.u_dtype == wl.F32 else torch.bfloat16
    z = lambda n: torch.zeros(n, dtype=torch.int32, device="cuda")  # noqa: E731
    return R.GdnState(_dev(init.S0), _dev(init.ring_u, ut), _dev(init.ring_k, _bf16()), _dev(init.ring_g),
                      _dev(init.start, _i32()), _dev(init.count, _i32()), z(B), z(B), z(1)).add_workspace(4)


def _gdn_inp(st):
    return (_dev(st.q, _bf16()), _dev(st.k, _bf16()), _dev(st.v, _bf16()), _dev(st.beta), _dev(st.g))


def suite_gdn(R, peak, steps=None):
    """GDN layer (B=256, Hv=32, Hk=16, d_k=d_v=128, L=16): decode steps
    (decode + flush) vs the baseline state update, and T=4 verify rounds vs
    the snapshot baseline."""
    import torch

    shape, seed, P = wl.GDN_LAYER, wl.SEED_GDN, 8
    out = []
    init = wl.gdn_init(shape, seed)
    pool = [_gdn_inp(wl.gdn_step(shape, seed, t)) for t in range(P)]
    y = torch.empty(shape.B, shape.Hv, shape.dv, device="cuda")
    st = _gdn_state(R, init)
    W, K = 4, steps or 512

    def step(i):
        R.gdn_replay_decode_fused(st, *pool[i % P], y=y)

    ms = _time_loop(step, K, W)
    err = int(st.err.item())
    per_h = np.array([gdn_decode_bytes(shape, h) for h in range(shape.L)], dtype=np.int64)
    tr = fill_trace(init.count, shape.L, W + K)[W:]
    # a fused fold adds only the S_0 write: S_0 and the entries were read for the output
    nbytes = int(per_h[tr].sum()) + int((tr + 1 == shape.L).sum()) * 4 * shape.Hv * shape.dv * shape.dk
    del st
    st = _gdn_state(R, init)

    def ustep(i):
        R.gdn_replay_decode(st, *pool[i % P], y=y)
        R.gdn_replay_flush(st)

    ums = _time_loop(ustep, K, W)
    err |= int(st.err.item())
    del st
    S = _dev(init.S0)

    def bstep(i):
        R.gdn_state_update_baseline(S, *pool[i % P], y=y)

    bms = _time_loop(bstep, K, W)
    del S
    gbs = nbytes / K / (ms * 1e-3) / 1e9
    out.append({"suite": "gdn_decode", "workload": "GDN layer B=256, Hv=32, Hk=16, d_k=d_v=128, L=16, u f32",
                "steps": K, "ms_per_step": ms, "tokens_per_s": shape.B / (ms * 1e-3), "gbs": gbs,
                "frac_of_peak": gbs / peak, "calls_per_step": "gdn_replay_decode_fused (workspace)",
                "unfused_ms_per_step": ums, "unfused_calls": "gdn_replay_decode + gdn_replay_flush",
                "baseline_ms_per_step": bms,
                "baseline_gbs": gdn_baseline_bytes(shape) * shape.B / (bms * 1e-3) / 1e9,
                "replay_over_baseline": bms / ms, "device_error_word": err})
    print(json.dumps(out[-1]), flush=True)

    T, Kv = 4, steps or 256
    init = wl.gdn_init(shape, seed + 50, fill_max=shape.L - T)
    vpool = [_gdn_inp(wl.gdn_step(shape, seed + 50, r, T=T)) for r in range(P)]
    acc = [_dev(wl.accepted_counts(shape.B, T, seed + 50, r), _i32()) for r in range(P)]
    yv = torch.empty(shape.B, T, shape.Hv, shape.dv, device="cuda")
    st = _gdn_state(R, init)
    h_tr, fl_tr, acc_tr = [], [], []
    for i in range(W + Kv):
        h_tr.append(st.count.cpu().numpy().astype(np.int64))
        R.gdn_replay_verify(st, *vpool[i % P], y=yv)
        fl_tr.append(st.flag.cpu().numpy() != 0)
        R.replay_spec_commit(acc[i % P], st.count, T, shape.L, st.err)
        acc_tr.append(acc[i % P].cpu().numpy().astype(np.int64))
        R.gdn_replay_flush(st)
    del st
    st = _gdn_state(R, init)

    def rnd(i):
        R.gdn_replay_verify(st, *vpool[i % P], y=yv)
        R.replay_spec_commit(acc[i % P], st.count, T, shape.L, st.err)
        R.gdn_replay_flush(st)

    vms = _time_loop(rnd, Kv, W)
    err = int(st.err.item())
    nbytes = 0
    for i in range(W, W + Kv):
        nbytes += sum(gdn_verify_bytes(shape, int(x), T) for x in h_tr[i])
        nbytes += sum(gdn_flush_bytes(shape, int(x)) for x in (h_tr[i] + acc_tr[i])[fl_tr[i]])
    del st
    torch.cuda.empty_cache()
    slots = torch.zeros(shape.B, T + 1, shape.Hv, shape.dv, shape.dk, device="cuda")
    slots[:, 0] = _dev(init.S0)
    cur = torch.zeros(shape.B, dtype=torch.int32, device="cuda")
    berr = torch.zeros(1, dtype=torch.int32, device="cuda")

    def brnd(i):
        R.gdn_spec_verify_baseline(slots, cur, *vpool[i % P], y=yv, err=berr)
        R.ssm_spec_commit_baseline(acc[i % P], cur, T, berr)

    bvms = _time_loop(brnd, Kv, W)
    gbs = nbytes / Kv / (vms * 1e-3) / 1e9
    out.append({"suite": "gdn_verify", "workload": "GDN layer B=256, T=4, L=16, accepted ~ U{0..4}",
                "rounds": Kv, "ms_per_round": vms, "rounds_per_s": 1e3 / vms,
                "accepted_tokens_per_s": shape.B * float(np.mean(acc_tr[W:])) / (vms * 1e-3),
                "gbs": gbs, "frac_of_peak": gbs / peak,
                "calls_per_round": "gdn_replay_verify + replay_spec_commit + gdn_replay_flush",
                "decode_step_ms": ms, "verify_over_decode": vms / ms,
                "baseline_ms_per_round": bvms,
                "baseline_gbs": gdn_snapshot_verify_bytes(shape, T) * shape.B / (bvms * 1e-3) / 1e9,
                "replay_over_baseline": bvms / vms, "device_error_word": err | int(berr.item())})
    print(json.dumps(out[-1]), flush=True)
    del slots
    torch.cuda.empty_cache()
    return out


def spec_trace(count0: np.ndarray, accs: list, T: int, L: int):
    """Committed count h of every sequence at the start of each round of the
    accepted-count sequence `accs`, and the number of entries the flush after
    the round folds (-1 where it does not flush): verify flags h + 2T > L,
    commit adds the accepted count, the flush resets flagged sequences."""
    h = count0.astype(np.int64).copy()
    hs, folds = [], []
    for a in accs:
        hs.append(h.copy())
        flag = h + 2 * T > L
        h = h + a.astype(np.int64)
        folds.append(np.where(flag, h, -1))
        h = np.where(flag, 0, h)
    return hs, folds


SWEEP_ROUNDS = 8  # rounds captured per CUDA graph (each with its own inputs and accepted counts)


def suite_sweep(R, peak, steps=None, Ts=range(1, 7), emit=True):
    """Speculative rounds against the window T = 1..6 (the shape of "Results --
    speculative decoding", Fig. 9): each round is verify + device commit +
    flush of the early-flagged sequences, captured in a CUDA graph with the
    per-round accepted counts in device memory (the sampler is a stub: counts
    drawn U{0..T} beforehand), so one graph covers every sequence's runtime
    branch with no host synchronisation.  Against it, the snapshot baseline
    round (T serial state updates into T + 1 slots, then the slot commit), and
    both relative to the standard decode step of their own kind at the same
    batch.  Mamba-2 layer at B = 512 and GDN layer at B = 256, L = 16."""
    import torch

    reps, W = (steps or 8), 2
    K = SWEEP_ROUNDS
    out = []
    for model in ("mamba2", "gdn"):
        if model == "mamba2":
            shape = wl.SPEC_MAMBA2
            t = wl.mamba2_state_tensors_device(shape, wl.SEED_SPEC + 7, "cuda")
            z = lambda n: torch.zeros(n, dtype=torch.int32, device="cuda")  # noqa: E731
            dst = R.Mamba2State(t["S0"].clone(), t["ring_v"].clone(), t["ring_k"].clone(), t["ring_dt"].clone(),
                                t["start"].clone(), t["count"].clone(), z(shape.B), z(shape.B), z(1)).add_workspace()
            A = t["A"]
            dinp = [tuple(x[:, 0].contiguous() for x in wl.mamba2_round_device(shape, 50 + i, 1, "cuda"))
                    for i in range(K)]
            y1 = torch.empty(shape.B, shape.H, shape.d, device="cuda")
            c0 = dst.count.cpu().numpy()
            dec_ms = _time_graph(lambda i: R.replay_decode_step_fused(dst, *dinp[i % K], A, y=y1), K, W, reps)
            per_h = np.array([m2_decode_bytes(shape, h) for h in range(shape.L)], dtype=np.int64)
            fold_extra = m2_fused_flush_extra_bytes(shape)
            Sb = t["S0"].clone()
            base_dec_ms = _time_graph(lambda i: R.ssm_state_update_baseline(Sb, *dinp[i % K], A, y=y1), K, W, reps)
            del dst, Sb
        else:
            shape = wl.GDN_LAYER
            t = wl.gdn_state_tensors_device(shape, wl.SEED_GDN + 7, "cuda")
            z = lambda n: torch.zeros(n, dtype=torch.int32, device="cuda")  # noqa: E731
            dst = R.GdnState(t["S0"].clone(), t["ring_u"].clone(), t["ring_k"].clone(), t["ring_g"].clone(),
                             t["start"].clone(), t["count"].clone(), z(shape.B), z(shape.B), z(1)).add_workspace(1)
            dinp = [tuple(x[:, 0].contiguous() for x in wl.gdn_round_device(shape, 50 + i, 1, "cuda"))
                    for i in range(K)]
            y1 = torch.empty(shape.B, shape.Hv, shape.dv, device="cuda")
            c0 = dst.count.cpu().numpy()
            dec_ms = _time_graph(lambda i: R.gdn_replay_decode_fused(dst, *dinp[i % K], y=y1), K, W, reps)
            per_h = np.array([gdn_decode_bytes(shape, h) for h in range(shape.L)], dtype=np.int64)
            fold_extra = 4 * shape.Hv * shape.dv * shape.dk
            Sb = t["S0"].clone()
            base_dec_ms = _time_graph(lambda i: R.gdn_state_update_baseline(Sb, *dinp[i % K], y=y1), K, W, reps)
            del dst, Sb
        torch.cuda.empty_cache()
        # decode steps run: one eager, then W + reps replays of K; the last reps x K are timed
        tr = fill_trace(c0, shape.L, 1 + K * (W + reps))[-reps * K:]
        dec_gbs = (int(per_h[tr].sum()) + int((tr + 1 == shape.L).sum()) * fold_extra) / (reps * K) / \
            (dec_ms * 1e-3) / 1e9
        for T in Ts:
            fill = dict(fill_max=shape.L - T)
            accs = [wl.accepted_counts_device(shape.B, T, 900 + 10 * T + i, "cuda") for i in range(K)]
            if model == "mamba2":
                t = wl.mamba2_state_tensors_device(shape, wl.SEED_SPEC + T, "cuda", **fill)
                st = R.Mamba2State(t["S0"], t["ring_v"], t["ring_k"], t["ring_dt"], t["start"], t["count"],
                                   z(shape.B), z(shape.B), z(1)).add_workspace(max_T=T)
                inp = [wl.mamba2_round_device(shape, 100 * T + i, T, "cuda") for i in range(K)]
                y = torch.empty(shape.B, T, shape.H, shape.d, device="cuda")

                def rnd(i):
                    R.replay_spec_verify(st, *inp[i % K], A, y=y)
                    R.replay_spec_commit(accs[i % K], st.count, T, shape.L, st.err)
                    R.replay_flush(st, A)

                vb = lambda h: m2_verify_bytes(shape, h, T)  # noqa: E731
                fb = lambda c: m2_flush_bytes(shape, c)  # noqa: E731
                calls = "replay_spec_verify + replay_spec_commit + replay_flush"
                snap_round_bytes = m2_snapshot_verify_bytes(shape, T) * shape.B
                slot_shape = (shape.B, T + 1, shape.H, shape.d, shape.n)
            else:
                t = wl.gdn_state_tensors_device(shape, wl.SEED_GDN + T, "cuda", **fill)
                st = R.GdnState(t["S0"], t["ring_u"], t["ring_k"], t["ring_g"], t["start"], t["count"],
                                z(shape.B), z(shape.B), z(1)).add_workspace(T)
                inp = [wl.gdn_round_device(shape, 100 * T + i, T, "cuda") for i in range(K)]
                y = torch.empty(shape.B, T, shape.Hv, shape.dv, device="cuda")

                def rnd(i):
                    R.gdn_replay_verify(st, *inp[i % K], y=y)
                    R.replay_spec_commit(accs[i % K], st.count, T, shape.L, st.err)
                    R.gdn_replay_flush(st)

                vb = lambda h: gdn_verify_bytes(shape, h, T)  # noqa: E731
                fb = lambda c: gdn_flush_bytes(shape, c)  # noqa: E731
                calls = "gdn_replay_verify + replay_spec_commit + gdn_replay_flush"
                snap_round_bytes = gdn_snapshot_verify_bytes(shape, T) * shape.B
                slot_shape = (shape.B, T + 1, shape.Hv, shape.dv, shape.dk)
            count0 = st.count.cpu().numpy()
            acc_h = [a.cpu().numpy() for a in accs]
            ms = _time_graph(rnd, K, W, reps)
            err = int(st.err.item())
            # rounds run: one eager, then W + reps replays of the K captured rounds; the last reps x K are timed
            seq = [acc_h[0]] + [acc_h[i] for _ in range(W + reps) for i in range(K)]
            hs, folds = spec_trace(count0, seq, T, shape.L)
            per_h = {x: vb(x) for x in range(shape.L + 1)}
            per_c = {x: fb(x) for x in range(shape.L + 1)}
            nbytes = 0
            for h, f in zip(hs[-reps * K:], folds[-reps * K:]):
                nbytes += sum(per_h[int(x)] for x in h) + sum(per_c[int(x)] for x in f[f >= 0])
            nbytes /= reps * K
            mean_acc = float(np.mean([a.mean() for a in acc_h]))
            del st
            torch.cuda.empty_cache()
            slots = torch.empty(*slot_shape, device="cuda")
            slots[:, 0] = t["S0"]
            del t
            cur = torch.zeros(shape.B, dtype=torch.int32, device="cuda")
            berr = torch.zeros(1, dtype=torch.int32, device="cuda")
            if model == "mamba2":
                def brnd(i):
                    R.ssm_spec_verify_baseline(slots, cur, *inp[i % K], A, y=y, err=berr)
                    R.ssm_spec_commit_baseline(accs[i % K], cur, T, berr)
            else:
                def brnd(i):
                    R.gdn_spec_verify_baseline(slots, cur, *inp[i % K], y=y, err=berr)
                    R.ssm_spec_commit_baseline(accs[i % K], cur, T, berr)
            bms = _time_graph(brnd, K, W, reps)
            err |= int(berr.item())
            gbs = nbytes / (ms * 1e-3) / 1e9
            line = {"suite": "sweep", "model": model,
                    "workload": (f"Mamba-2 layer B={shape.B}, H=32, G=8, d=64, n=128" if model == "mamba2" else
                                 f"GDN layer B={shape.B}, Hv=32, Hk=16, d_k=d_v=128") + f", L=16, T={T}",
                    "T": T, "rounds": reps * K, "timing": f"CUDA graph of {K} rounds", "calls": calls,
                    "ms_per_round": ms, "accepted_tokens_per_s": shape.B * mean_acc / (ms * 1e-3),
                    "gbs": gbs, "frac_of_peak": gbs / peak,
                    "decode_step_ms": dec_ms, "decode_gbs": dec_gbs, "round_over_decode": ms / dec_ms,
                    "baseline_ms_per_round": bms, "baseline_decode_step_ms": base_dec_ms,
                    "baseline_round_over_decode": bms / base_dec_ms,
                    "baseline_gbs": snap_round_bytes / (bms * 1e-3) / 1e9,
                    "replay_over_baseline": bms / ms, "device_error_word": err}
            out.append(line)
            if emit:
                print(json.dumps(line), flush=True)
            del slots, inp, y
            torch.cuda.empty_cache()
    return out


CONCURRENCY_BUDGET = 8 * 2**30  # bytes of HBM per layer for decode state (a 23-layer stack in 184 GiB)


def suite_concurrency(R, peak, steps=None):
    """Maximum decode concurrency at a fixed HBM budget ("Results --
    speculative decoding", Fig. 11).  The library's per-sequence accounting
    (replay: checkpoint, ring, pointers, workspace share; snapshot baseline:
    T + 1 states) gives the largest batch that fits CONCURRENCY_BUDGET per
    layer for T = 0..6; then, at T = 4, one layer is allocated at each of the
    two batches and runs speculative rounds (replay: verify + commit + flush;
    baseline: snapshot verify + commit, CUDA graphs of 8 rounds), measuring
    the accepted-token throughput each layout sustains within the budget."""
    import torch

    reps, W, K = (steps or 4), 2, SWEEP_ROUNDS
    out = []
    for model in ("mamba2", "gdn"):
        base = wl.SPEC_MAMBA2 if model == "mamba2" else wl.GDN_LAYER
        dims = (R.M2Dims(1, base.H, base.G, base.d, base.n, base.L, R.BF16, R.F32) if model == "mamba2" else
                R.GdnDims(1, base.Hv, base.Hk, base.dk, base.dv, base.L, R.BF16, R.F32, R.F32))
        rows = []
        for T in range(0, 7):
            rb, sb = R.seq_bytes(dims, T, R.SEQ_REPLAY), R.seq_bytes(dims, T, R.SEQ_SNAPSHOT)
            rows.append({"T": T, "replay_bytes_per_seq": rb, "snapshot_bytes_per_seq": sb,
                         "replay_max_batch": CONCURRENCY_BUDGET // rb, "snapshot_max_batch": CONCURRENCY_BUDGET // sb,
                         "ratio": (CONCURRENCY_BUDGET // rb) / (CONCURRENCY_BUDGET // sb)})
        T = 4
        Br, Bs = rows[T]["replay_max_batch"], rows[T]["snapshot_max_batch"]
        z = lambda n: torch.zeros(n, dtype=torch.int32, device="cuda")  # noqa: E731
        tput = {}
        for kind, Bk in (("replay", Br), ("snapshot", Bs)):
            shape = dataclasses.replace(base, B=int(Bk))
            accs = [wl.accepted_counts_device(shape.B, T, 700 + i, "cuda") for i in range(K)]
            if model == "mamba2":
                t = wl.mamba2_state_tensors_device(shape, 77, "cuda", fill_max=shape.L - T)
                inp = [wl.mamba2_round_device(shape, 300 + i, T, "cuda") for i in range(K)]
                y = torch.empty(shape.B, T, shape.H, shape.d, device="cuda")
                A = t["A"]
            else:
                t = wl.gdn_state_tensors_device(shape, 77, "cuda", fill_max=shape.L - T)
                inp = [wl.gdn_round_device(shape, 300 + i, T, "cuda") for i in range(K)]
                y = torch.empty(shape.B, T, shape.Hv, shape.dv, device="cuda")
            err = z(1)
            if kind == "replay":
                if model == "mamba2":
                    st = R.Mamba2State(t["S0"], t["ring_v"], t["ring_k"], t["ring_dt"], t["start"], t["count"],
                                       z(shape.B), z(shape.B), err).add_workspace(max_T=T)

                    def rnd(i):
                        R.replay_spec_verify(st, *inp[i % K], A, y=y)
                        R.replay_spec_commit(accs[i % K], st.count, T, shape.L, st.err)
                        R.replay_flush(st, A)
                else:
                    st = R.GdnState(t["S0"], t["ring_u"], t["ring_k"], t["ring_g"], t["start"], t["count"],
                                    z(shape.B), z(shape.B), err).add_workspace(T)

                    def rnd(i):
                        R.gdn_replay_verify(st, *inp[i % K], y=y)
                        R.replay_spec_commit(accs[i % K], st.count, T, shape.L, st.err)
                        R.gdn_replay_flush(st)
                held = sum(x.numel() * x.element_size() for x in
                           (st.S0, st.ring_v if model == "mamba2" else st.ring_u, st.ring_k,
                            st.ring_dt if model == "mamba2" else st.ring_g, st.start, st.count, st.flag, st.sync,
                            st.work))
            else:
                S0 = t["S0"]
                del t
                slots = torch.empty(shape.B, T + 1, *S0.shape[1:], device="cuda")
                slots[:, 0] = S0
                del S0
                cur = z(shape.B)
                if model == "mamba2":
                    def rnd(i):
                        R.ssm_spec_verify_baseline(slots, cur, *inp[i % K], A, y=y, err=err)
                        R.ssm_spec_commit_baseline(accs[i % K], cur, T, err)
                else:
                    def rnd(i):
                        R.gdn_spec_verify_baseline(slots, cur, *inp[i % K], y=y, err=err)
                        R.ssm_spec_commit_baseline(accs[i % K], cur, T, err)
                held = slots.numel() * 4 + cur.numel() * 4
            ms = _time_graph(rnd, K, W, reps)
            mean_acc = float(np.mean([a.float().mean().item() for a in accs]))
            tput[kind] = {"batch": int(Bk), "held_bytes": int(held), "ms_per_round": ms,
                          "accepted_tokens_per_s": shape.B * mean_acc / (ms * 1e-3),
                          "device_error_word": int(err.item())}
            st = slots = t = inp = y = accs = None  # release this layout before allocating the next
            torch.cuda.empty_cache()
        line = {"suite": "concurrency", "model": model,
                "workload": ("Mamba-2 layer H=32, G=8, d=64, n=128" if model == "mamba2" else
                             "GDN layer Hv=32, Hk=16, d_k=d_v=128") + ", L=16",
                "budget_bytes_per_layer": CONCURRENCY_BUDGET, "per_T": rows, "measured_T": T,
                "at_max_batch": tput,
                "throughput_ratio": tput["replay"]["accepted_tokens_per_s"] / tput["snapshot"]["accepted_tokens_per_s"]}
        out.append(line)
        print(json.dumps(line), flush=True)
    return out


def suite_conv(R, peak, steps=None):
    """Convolution-state step of the Nemotron-H layer (x 32 x 64, B and C
    8 x 128, W = 4, bf16) at batch 256, alone and followed by the fused decode
    step it feeds (the layer's decode path from the in-projection's columns to
    y).  The state and inputs (about 17 MB) stay in L2 between steps, so the
    step's GB/s is an L2 figure; the decode step is not."""
    import torch

    K, W, P = steps or 1024, 16, 8
    ms = wl.NEMOTRON_H_MAMBA2
    cs = wl.ConvShape(B=ms.B, dx=ms.H * ms.d, dbc=ms.G * ms.n, W=4, io_dtype=wl.BF16)
    cinit = wl.conv_init(cs, wl.SEED_NEMOTRON + 30)
    state = _dev(cinit.state, _bf16())
    weight, bias = _dev(cinit.weight), _dev(cinit.bias)
    us = [_dev(wl.conv_input(cs, wl.SEED_NEMOTRON + 30, t), _bf16()) for t in range(P)]
    outs = tuple(torch.empty(ms.B, n, dtype=torch.bfloat16, device="cuda") for n in (cs.dx, cs.dbc, cs.dbc))
    conv_ms = _time_loop(lambda i: R.conv_state_update(state, us[i % P], weight, bias, cs.dx, cs.dbc, out=outs), K, W)
    C = cs.dx + 2 * cs.dbc
    conv_bytes = ms.B * C * (2 * 2 * (cs.W - 1) + 2 + 2) + C * (cs.W + 1) * 4
    init = wl.mamba2_init(ms, wl.SEED_NEMOTRON + 31)
    st = _m2_state(R, init).add_workspace()
    A = _dev(init.A)
    g = torch.Generator(device="cuda")
    g.manual_seed(wl.SEED_NEMOTRON + 32)
    dts = [torch.nn.functional.softplus(torch.randn(ms.B, ms.H, generator=g, device="cuda")) for _ in range(P)]
    y = torch.empty(ms.B, ms.H, ms.d, device="cuda")
    v, k, q = outs[0].view(ms.B, ms.H, ms.d), outs[1].view(ms.B, ms.G, ms.n), outs[2].view(ms.B, ms.G, ms.n)

    def layer(i):
        R.conv_state_update(state, us[i % P], weight, bias, cs.dx, cs.dbc, out=outs)
        R.replay_decode_step_fused(st, v, k, q, dts[i % P], A, y=y)

    pair_ms = _time_loop(layer, K, W)
    dec_ms = _time_loop(lambda i: R.replay_decode_step_fused(st, v, k, q, dts[i % P], A, y=y), K, W)
    line = {"suite": "conv", "workload": "Nemotron-H convolution state B=256, x 2048 + B 1024 + C 1024 channels, "
                                         "W=4, bf16; then the fused decode step",
            "steps": K, "conv_ms_per_step": conv_ms, "conv_bytes_per_step": conv_bytes,
            "conv_gbs": conv_bytes / (conv_ms * 1e-3) / 1e9, "conv_state_fits_l2": True,
            "conv_plus_decode_ms_per_step": pair_ms, "decode_ms_per_step": dec_ms,
            "conv_share": (pair_ms - dec_ms) / pair_ms,
            "device_error_word": int(st.err.item())}
    print(json.dumps(line), flush=True)
    return [line]


def record_traffic(report: str, command: str):
    """Write profiles/ncu_traffic.json from an ncu report of the headline
    command (read with `ncu -i`, no GPU needed): DRAM bytes and duration of
    the first captured launch of each fused decode kernel, with the digest of
    the sources that define them."""
    import csv
    import io

    if report.endswith(".csv"):  # the raw page already exported (ncu -i REPORT --page raw --csv)
        with open(report) as f:
            text = f.read()
    else:
        text = subprocess.run(["ncu", "-i", report, "--page", "raw", "--csv"], capture_output=True, text=True,
                              check=True).stdout
    rows = list(csv.reader(io.StringIO(text)))
    head, units = rows[0], rows[1]
    col = {n: i for i, n in enumerate(head)}

    def val(r, name):
        v = float(r[col[name]].replace(",", ""))
        u = units[col[name]]
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "nsecond": 1e-3, "usecond": 1, "msecond": 1e3}
        return v * scale.get(u, 1)

    kernels = {}
    for r in rows[2:]:
        name = r[col["Kernel Name"]]
        for key, pat in (("m2_prep_kernel<fused>", "m2_prep_kernel<128, 1,"),
                         ("m2_stream_kernel<fused>", "m2_stream_kernel<128, 1,")):
            if pat in name and key not in kernels:
                rd, wr = val(r, "dram__bytes_read.sum"), val(r, "dram__bytes_write.sum")
                short = name[name.index(pat.split("<")[0]):].split("(")[0]
                kernels[key] = {"kernel": short.replace("__nv_bfloat16", "bf16"),
                                "dram_bytes_per_launch": rd + wr, "dram_read": rd, "dram_write": wr,
                                "duration_us": val(r, "gpu__time_duration.sum")}
    rec = {"source_digest": source_digest(HEADLINE_SOURCES), "sources": list(HEADLINE_SOURCES), "command": command,
           "kernels": kernels}
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec, indent=1))


def suite_kernels(R, peak, steps=None):
    """A few eager calls of every hot kernel at its benchmark workload, one
    JSON line each with the mean milliseconds per call: the command the ncu
    captures of single kernels run (one kernel per capture, selected with
    -k).  Mamba-2 baseline and fused decode (B = 256), the speculative rounds
    at B = 512 (verify, commit, flush) for T = 4 (CUDA-core verify stream)
    and T = 6 (tensor-core verify), the GDN baseline and fused decode
    (B = 256) and the GDN T = 4 round (pipelined tensor-core verify, flush)."""
    import torch

    n = steps or 3
    z = lambda k: torch.zeros(k, dtype=torch.int32, device="cuda")  # noqa: E731

    def timed(name, fn):
        fn(0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n):
            fn(1 + i)
        e1.record()
        torch.cuda.synchronize()
        print(json.dumps({"suite": "kernels", "workload": name, "calls": n, "ms_per_call": e0.elapsed_time(e1) / n}),
              flush=True)

    def m2(shape, seed, T=None):
        t = wl.mamba2_state_tensors_device(shape, seed, "cuda", fill_max=None if T is None else shape.L - T)
        st = R.Mamba2State(t["S0"], t["ring_v"], t["ring_k"], t["ring_dt"], t["start"], t["count"], z(shape.B),
                           z(shape.B), z(1)).add_workspace(max_T=T or 0)
        return st, t["A"]

    shape = wl.NEMOTRON_H_MAMBA2
    st, A = m2(shape, 11)
    inp = [tuple(x[:, 0].contiguous() for x in wl.mamba2_round_device(shape, 20 + i, 1, "cuda")) for i in range(4)]
    y = torch.empty(shape.B, shape.H, shape.d, device="cuda")
    S = st.S0.clone()
    timed("m2_baseline B=256", lambda i: R.ssm_state_update_baseline(S, *inp[i % 4], A, y=y))
    timed("m2_decode_fused B=256", lambda i: R.replay_decode_step_fused(st, *inp[i % 4], A, y=y))
    del st, S
    shape = wl.SPEC_MAMBA2
    for T in (4, 6):
        st, A = m2(shape, 12 + T, T)
        rin = [wl.mamba2_round_device(shape, 30 + i, T, "cuda") for i in range(4)]
        acc = [wl.accepted_counts_device(shape.B, T, 40 + i, "cuda") for i in range(4)]
        yv = torch.empty(shape.B, T, shape.H, shape.d, device="cuda")

        def rnd(i, st=st, A=A, rin=rin, acc=acc, yv=yv, T=T):
            R.replay_spec_verify(st, *rin[i % 4], A, y=yv)
            R.replay_spec_commit(acc[i % 4], st.count, T, shape.L, st.err)
            R.replay_flush(st, A)

        timed(f"m2_spec_round B=512 T={T}", rnd)
        del st
    shape = wl.GDN_LAYER
    t = wl.gdn_state_tensors_device(shape, 13, "cuda")
    st = R.GdnState(t["S0"], t["ring_u"], t["ring_k"], t["ring_g"], t["start"], t["count"], z(shape.B), z(shape.B),
                    z(1)).add_workspace(4)
    ginp = [tuple(x[:, 0].contiguous() for x in wl.gdn_round_device(shape, 50 + i, 1, "cuda")) for i in range(4)]
    yg = torch.empty(shape.B, shape.Hv, shape.dv, device="cuda")
    Sg = t["S0"].clone()
    timed("gdn_baseline B=256", lambda i: R.gdn_state_update_baseline(Sg, *ginp[i % 4], y=yg))
    timed("gdn_decode_fused B=256", lambda i: R.gdn_replay_decode_fused(st, *ginp[i % 4], y=yg))
    del st, Sg, t
    T = 4
    t = wl.gdn_state_tensors_device(shape, 14, "cuda", fill_max=shape.L - T)
    st = R.GdnState(t["S0"], t["ring_u"], t["ring_k"], t["ring_g"], t["start"], t["count"], z(shape.B), z(shape.B),
                    z(1)).add_workspace(T)
    vin = [wl.gdn_round_device(shape, 60 + i, T, "cuda") for i in range(4)]
    acc = [wl.accepted_counts_device(shape.B, T, 70 + i, "cuda") for i in range(4)]
    yv = torch.empty(shape.B, T, shape.Hv, shape.dv, device="cuda")

    def grnd(i):
        R.gdn_replay_verify(st, *vin[i % 4], y=yv)
        R.replay_spec_commit(acc[i % 4], st.count, T, shape.L, st.err)
        R.gdn_replay_flush(st)

    timed("gdn_verify_round B=256 T=4", grnd)
    return []


def run_suite(args):
    import torch

    torch.cuda.set_device(0)
    from ssm_decode_hybrid_gb300 import replayssm as R

    peak, _ = measured_peaks()
    names = args.suite.split(",")
    for name in names:
        {"layers": suite_layers, "spec": suite_spec, "gdn": suite_gdn, "sweep": suite_sweep,
         "concurrency": suite_concurrency, "conv": suite_conv, "kernels": suite_kernels}[name](R, peak,
                                                                                              args.suite_steps)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=32)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=1024)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--windows", type=int, default=5,
                    help="timed windows of --steps steps each; the line reports the median window")
    ap.add_argument("--no-extra", action="store_true",
                    help="leave out the speculative and GDN keys of the headline line")
    ap.add_argument("--suite", default=None,
                    help="instead of the headline line, print one JSON line per measurement of the other "
                         "workloads: comma-separated subset of layers,spec,gdn,sweep,concurrency,conv,kernels")
    ap.add_argument("--suite-steps", type=int, default=None,
                    help="timed steps (rounds) per suite measurement instead of each suite's own count "
                         "(short runs for profiling; the layer sweep keeps its graph of 16 steps)")
    ap.add_argument("--record-traffic", default=None, metavar="REPORT",
                    help="write profiles/ncu_traffic.json from an ncu report of the headline command and exit")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(args.record_traffic, TRAFFIC_COMMAND)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.suite:
        run_suite(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
