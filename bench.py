"""Benchmark of the decode-step attention hot path on GB300.

A step = one decode step of a seeded synthetic workload through the C ABI:
kvs_decode_step per layer, i.e. the KV-cache scatter of the new rows, the
split plan, the chunk partials and the rescaled merge, all in one kernel
launch.  One run measures every workload of the decode path and prints ONE
JSON line (rank 0):

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--chunk C] [--impl kvs|reference]

The headline (`value`, `config`, `roofline`, `e2e`, `cpu_baseline`) is the
--config workload, by default `ragged`, the largest: 32 sequences of up to
131,072 positions, 34 GB of caches.  `per_config` holds the same
measurements for all five workloads (tiny, small_model as one CUDA graph of
24 layers, 8b_batch, long_context with its chunk sweep, ragged).

value       : algorithmic GB/s of the step (live KV bytes read + Q read + O
              written + positions, plus the scatter's row bytes), inputs
              resident in HBM, device time from CUDA events, max over ranks.
e2e         : the same metric when every step also copies its inputs (q, new
              K/V rows, positions) from pinned host memory and its output
              back, through kvs_decode_step_host_io (one C call per layer:
              one copy in, the step, one copy out); two host buffers in
              alternation, each reused once its previous step's output has
              reached the host.
us_per_call : the step's mean, median, p10 and p90 over the timed steps
              (L2 scrubbed between steps when the working set fits in it),
              the hot mean of back-to-back steps, and for the headline the
              two-launch breakdown.
roofline    : the step kernel (the step's one launch per layer): its
              algorithmic bytes / its mean event-timed duration, against the
              measured HBM copy bandwidth.
cpu_baseline: the f64 CPU oracle on the host cores, all threads and one
              (rank 0, N=1 only), on the headline workload.
--impl reference times that oracle as the reference arm.
Under torchrun every rank runs its own batch (weak scaling, no collective on
the data path; a barrier and a max-reduction of the timings only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from split_flash_decoding_kvcachescatter_gb300 import workloads as W  # noqa: E402

METRIC = "split-K decode attention: KV-cache HBM GB/s (% of GB300 peak) and µs/call"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0  # the 8 TB/s the targets are stated against
FALLBACK_HBM_GBS = 6800.0
HEADLINE = "ragged"  # the largest workload that fits one GPU
# Every workload of the decode path, in the order they are measured.
PER_CONFIG = ("tiny", "small_model", "8b_batch", "long_context", "ragged")
# Timed steps of a per-config leg: at least these, at least --steps.
MIN_STEPS = {"tiny": 200, "small_model": 200, "8b_batch": 100, "long_context": 100,
             "ragged": 20}
CSRC = os.path.join(ROOT, "split_flash_decoding_kvcachescatter_gb300", "csrc")
# Sources of each attention kernel (a recorded ncu capture is used only
# while these are unchanged).
KERNEL_SOURCES = {
    "persistent": ("flash_decode.cu", "fd_tile.cuh", "kvs_device.cuh"),
    "cluster": ("fd_cluster.cu", "fd_tile.cuh", "kvs_device.cuh", "kvs_cluster.cuh"),
}
KERNEL_NAMES = {"persistent": "fd_step_kernel", "cluster": "fd_cluster_kernel"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(w, rank):
    """Each rank decodes its own, independent batch (weak scaling)."""
    return w.seed + 7919 * rank


def percentile(xs, q):
    """Nearest-rank percentile of a list (q in 0..100)."""
    ys = sorted(xs)
    k = max(0, min(len(ys) - 1, int(round(q / 100.0 * (len(ys) - 1)))))
    return ys[k]


def reduce_over_ranks(step_ms, e2e_ms, bytes_timed, bytes_e2e, world, device):
    """Max of the timings and sum of the bytes over all ranks (the only
    communication of a multi-rank run; nothing on the data path)."""
    if world <= 1:
        return float(step_ms), float(e2e_ms), float(bytes_timed), float(bytes_e2e)
    import torch
    import torch.distributed as tdist
    t = torch.tensor([step_ms, e2e_ms], dtype=torch.float64, device=device)
    b = torch.tensor([bytes_timed, bytes_e2e], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    tdist.all_reduce(b, op=tdist.ReduceOp.SUM)
    return float(t[0]), float(t[1]), float(b[0]), float(b[1])


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload, chunk):
    """Per-launch DRAM bytes of the attention kernel from a committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "fd_step_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    key = f"{workload}:{chunk}" if kernel == "persistent" else f"{workload}:{kernel}"
    e = rec.get(key)
    if not e or e.get("source_sha256_16") != kernel_source_hash(kernel):
        return None
    return int(e["dram_bytes_per_launch"])


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo) and core count."""
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                name = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not name:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu model")):
                        name = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"cpu_model": name or "unknown", "nproc": os.cpu_count() or 1}


VOCAB = 152064  # vocabulary of the pages' batched argmax (PAR-062)


def time_stream_read(torch, dev, stream, nbytes=2 << 30, iters=10):
    """A read-only streaming pass measured in the same run, beside the copy
    peak of MEASURED_PEAKS.json: torch's sum over a 2 GiB float32 buffer
    (a library kernel, not one of ours), median of CUDA-event times."""
    x = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        x.sum()
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x.sum()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    del x
    ms = statistics.median(ts)
    return {"read_gbs": nbytes / (ms * 1e-3) / 1e9, "bytes": nbytes,
            "kernel": "torch.sum over a 2 GiB float32 buffer (read-only)"}


def launch_floor(torch, dev, stream, iters=200):
    """What one launch costs with this file's single-launch timing (L2 scrub,
    then events around the call) when the kernel does nothing: a one-element
    add.  The event pair and the launch itself take this much of every
    single-launch figure here (argmax, tiny)."""
    one = torch.zeros(1, device=dev)
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(5):
        one.add_(1.0)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    for a, b in ev:
        scrub.zero_()
        a.record(stream)
        one.add_(1.0)
        b.record(stream)
    torch.cuda.synchronize()
    us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in ev)
    return {"us": us, "kernel": "torch add_ on one float32 element",
            "method": "L2 scrubbed, then CUDA events around the single launch (as argmax and tiny)"}


def time_argmax(B, torch, M, dev, stream, iters=200):
    """The batched argmax of the serving step after attention (kvs_argmax):
    M rows of VOCAB logits, one launch; L2 scrubbed between launches
    (outside the events).  HBM-bound: M*VOCAB*4 bytes read per launch."""
    g = torch.Generator(device=dev).manual_seed(1234)
    logits = torch.randn((M, VOCAB), device=dev, generator=g)
    ids = torch.empty(M, dtype=torch.int32, device=dev)
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(5):
        B.kvs_argmax(logits, ids)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    for a, b in ev:
        scrub.zero_()
        a.record(stream)
        B.kvs_argmax(logits, ids)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    ok = torch.equal(ids.long(), torch.argmax(logits, dim=1))  # finite data: same first-max rule
    nbytes = M * VOCAB * 4 + M * 4
    peak, _ = hbm_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "argmax_cluster_kernel (kvs_argmax)", "M": M, "vocab": VOCAB,
            "us_per_call": 1e3 * ms, "bytes_per_call": nbytes, "gbs": gbs, "frac": gbs / peak,
            "l2": "scrubbed between launches", "matches_torch_argmax": bool(ok)}


PREFILL_SHAPE = (32, 4096, 128)  # heads, sequence length, head_dim of an 8B-class prefill


def tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16 (burst); fp16 has the same rate"
    except Exception:
        return 1900.0, "fallback"


def time_prefill(B, torch, dev, stream, iters=20, shape=PREFILL_SHAPE, causal=True):
    """Tensor-core prefill attention (kvs_prefill_attention), timed as one
    call (all its launches).  At the default shape the inputs (3 x 67 MB)
    and the packed workspace exceed L2."""
    H, S, D = shape
    g = torch.Generator(device=dev).manual_seed(4321)
    q, k, v = (torch.randn((H, S, D), device=dev, generator=g) for _ in range(3))
    out = torch.empty_like(q)
    ws = B.prefill_workspace(H, S, D, device=dev)
    for _ in range(3):
        B.kvs_prefill_attention(q, k, v, out, causal=causal, workspace=ws)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    for a, b in ev:
        a.record(stream)
        B.kvs_prefill_attention(q, k, v, out, causal=causal, workspace=ws)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    # QK^T and PV over the causal triangle, or the full square
    flops = 4.0 * D * H * (S * (S + 1) / 2 if causal else S * S)
    tf = flops / (ms * 1e-3) / 1e12
    peak, kind = tensor_peak()
    return {"kernel": "prefill kernels (kvs_prefill_attention)",
            "heads": H, "seq_len": S, "head_dim": D, "causal": causal,
            "dtype": "f16 x f16 -> f32",
            "us_per_call": 1e3 * ms, "flops_per_call": flops,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "peak_source": kind}}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self, windows):
        """Median SM clock, max clock and throttle reasons over the samples
        taken inside the given (t0, t1) windows (the timed regions)."""
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if any(t0 <= r[0] <= t1 for t0, t1 in windows)]
        window = "timed regions"
        if not inside:  # timed regions shorter than the sampling interval
            t0 = min(w[0] for w in windows) - 1.0
            t1 = max(w[1] for w in windows) + 1.0
            inside = [r for r in rows if t0 <= r[0] <= t1] or rows
            window = "around the timed regions"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3][5:9])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


def _unit_bytes(inp, w, i):
    """Algorithmic step bytes of sequence i, shared equally by its query heads."""
    L = int(inp.positions[i]) + 1
    seq = (2 * w.num_kv_heads * L * w.head_dim * 4 + 2 * w.num_heads * w.head_dim * 4 + 4
           + 4 * w.num_kv_heads * w.head_dim * 4 + 4)
    return seq / w.num_heads


class CpuOracleRunner:
    """Runs the f64 CPU oracle over (sequence, query head) units of the
    workload, in rotation, on `threads` host threads (the C call releases the
    GIL).  A sample is time-bounded: batches of units run until the budget is
    spent."""

    def __init__(self, inp, w, threads=None):
        from concurrent.futures import ThreadPoolExecutor
        import oracle
        oracle.build()
        self.oracle = oracle
        self.inp, self.w = inp, w
        self.threads = threads or os.cpu_count() or 1
        self.pool = ThreadPoolExecutor(max_workers=self.threads) if self.threads > 1 else None
        self.units = [(i, h) for i in range(w.M) for h in range(w.num_heads)]
        self.next = 0
        self.G = w.group

    def _one(self, u):
        i, h = u
        L = int(self.inp.positions[i]) + 1
        g = h // self.G
        self.oracle.attend_row(self.inp.q[i, h], self.inp.k_seq[i][g, :L], self.inp.v_seq[i][g, :L])
        return _unit_bytes(self.inp, self.w, i)

    def sample(self, budget_s):
        """(seconds, bytes, units) of one time-bounded sample."""
        t0 = time.perf_counter()
        done_bytes, n = 0.0, 0
        batch = 2 * self.threads
        while True:
            us = [self.units[(self.next + k) % len(self.units)] for k in range(batch)]
            self.next = (self.next + batch) % len(self.units)
            if self.pool is not None:
                done_bytes += sum(self.pool.map(self._one, us))
            else:
                done_bytes += sum(self._one(u) for u in us)
            n += batch
            if time.perf_counter() - t0 >= budget_s:
                break
        return time.perf_counter() - t0, done_bytes, n

    def describe(self, n_units):
        return (f"{n_units} (sequence, query head) units of the {self.w.name} workload in "
                f"rotation ({len(self.units)} units = the whole batch), f64 C oracle on "
                f"{self.threads} host thread{'s' if self.threads > 1 else ''}")


def run_reference(args, w, inp, rank, world):
    if rank != 0:
        return
    ab = W.algorithmic_bytes(inp, w)
    runner = CpuOracleRunner(inp, w)
    budget = max(0.02, min(3.0, 150.0 / (args.steps + args.warmup)))
    tot_t, tot_b, tot_n = 0.0, 0.0, 0
    for s in range(args.warmup + args.steps):
        dt, b, n = runner.sample(budget)
        if s >= args.warmup:
            tot_t += dt
            tot_b += b
            tot_n += n
    value = tot_b / tot_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "num_heads": w.num_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "max_len": w.max_len, "algorithmic_bytes_per_step": ab["step"],
                   "step": f"a time-bounded sample of about {budget:.2f} s of oracle work"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": runner.threads,
                         "kind": "oracle", "sample": runner.describe(tot_n), **cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class Ctx:
    """What every leg of a run shares: the torch modules, the device, the
    stream, the binding, the rank layout and the timed-region clock."""

    def __init__(self, torch, tdist, B, dev, rank, world):
        self.torch, self.tdist, self.B = torch, tdist, B
        self.dev, self.rank, self.world = dev, rank, world
        self.stream = torch.cuda.current_stream()
        self.windows = []  # wall-clock (t0, t1) of every timed region

    def barrier(self):
        if self.world > 1:
            self.tdist.barrier()


def measure_workload(ctx, w, seed, steps, warmup, chunks, graph=False, full=False,
                     e2e_steps=None, keep_inputs=False):
    """Times one workload's decode step for each chunk size in `chunks` (0 =
    the library rule), on the same inputs.  Returns a list of result dicts,
    one per chunk; the first also carries the e2e leg, and with `full` the
    two-launch breakdown.  Multi-layer workloads (small_model) time all
    layers as one step, eagerly or, with `graph`, as one captured graph."""
    torch, B, dev, stream = ctx.torch, ctx.B, ctx.dev, ctx.stream
    nl = w.layers
    inp = W.make_inputs(w, seed=seed)
    inps = [inp] + [W.make_inputs(w, layer=l, seed=seed, positions=inp.positions)
                    for l in range(1, nl)]
    ts = [W.upload(x, w, dev) for x in inps]
    outs = [torch.empty_like(t["q"]) for t in ts]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ab1 = W.algorithmic_bytes(inp, w)  # one layer; every layer has the same positions
    ab = {k: v * nl for k, v in ab1.items()}
    flush = ab["step"] < 4 * L2_BYTES  # small working sets: scrub L2 between steps
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    kernel = ("cluster" if B.kvs_schedule_for(w.M, w.num_heads, w.num_kv_heads, w.head_dim,
                                               w.max_len) == B.KVS_SCHEDULE_CLUSTER
              else "persistent")
    peak, peak_kind = hbm_peak()
    results = []
    for ci, chunk in enumerate(chunks):
        resolved = chunk if chunk > 0 else B.kvs_choose_chunk_size(
            w.M, w.num_kv_heads, w.head_dim, w.max_len)
        ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len, resolved,
                         device=dev)

        def eager_step():
            for t, out in zip(ts, outs):
                B.kvs_decode_step(t["q"], t["k_rows"], t["v_rows"], t["positions"],
                                  t["k_cache"], t["v_cache"], out, chunk_size=resolved,
                                  workspace=ws, d_status=status)

        sg = None
        if graph:
            eager_step()  # configure the kernels outside the capture
            torch.cuda.synchronize()
            sg = B.kvs_step_graph_create(
                [t["q"] for t in ts], [t["k_rows"] for t in ts], [t["v_rows"] for t in ts],
                ts[0]["positions"], [t["k_cache"] for t in ts], [t["v_cache"] for t in ts],
                outs, chunk_size=resolved, workspace=ws, d_status=status)

        def step():
            if sg is not None:
                sg.launch(stream)
            else:
                eager_step()

        for _ in range(warmup):
            if flush:
                scrub.zero_()
            step()
        torch.cuda.synchronize()
        # events only at step boundaries, so the programmatic launch overlap
        # between the step's kernels is untouched
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ctx.barrier()
        torch.cuda.synchronize()
        wall0 = time.time()
        for k in range(steps):
            if flush:
                scrub.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize()
        ctx.barrier()
        ctx.windows.append((wall0, time.time()))
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        if int(status.item()) != 0:
            raise SystemExit(f"{w.name}: device status {B.strerror(int(status.item()))}")

        # hot: the same step back to back, nothing between steps (L2 warm);
        # eager steps are captured into one CUDA graph of HOT_CHUNK steps and
        # replayed, so that the host's launch rate does not set the time
        HOT_CHUNK = 20
        hot_reps = max(1, min(steps, 200) // HOT_CHUNK)
        hot_mode = "step graph launched back to back"
        if sg is not None:
            hot_run, hot_calls, KH = step, hot_reps * HOT_CHUNK, hot_reps * HOT_CHUNK
        else:
            try:
                hot_graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(hot_graph):
                    for _ in range(HOT_CHUNK):
                        eager_step()
                torch.cuda.synchronize()
                hot_run, hot_calls, KH = hot_graph.replay, hot_reps, hot_reps * HOT_CHUNK
                hot_mode = f"graph of {HOT_CHUNK} eager steps, replayed"
            except RuntimeError as e:  # capture refused: eager steps back to back
                torch.cuda.synchronize()
                hot_run, hot_calls, KH = step, hot_reps * HOT_CHUNK, hot_reps * HOT_CHUNK
                hot_mode = f"eager steps back to back (capture failed: {str(e)[:80]})"
        hot_run()
        torch.cuda.synchronize()
        h0 = torch.cuda.Event(enable_timing=True)
        h1 = torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        for _ in range(hot_calls):
            hot_run()
        h1.record(stream)
        torch.cuda.synchronize()
        hot_ms = h0.elapsed_time(h1) / KH
        if int(status.item()) != 0:
            raise SystemExit(f"{w.name} hot: device status {B.strerror(int(status.item()))}")

        total_ms = sum(step_ms)
        total_ms_max, _, bytes_all, _ = reduce_over_ranks(total_ms, 0.0, ab["step"] * steps, 0.0,
                                                          ctx.world, dev)
        mean_ms = total_ms / steps
        achieved = ab["step"] / (mean_ms * 1e-3) / 1e9
        traffic1 = ncu_traffic(kernel, w.name, resolved)
        res = {
            "workload": w.name, "kernel": KERNEL_NAMES[kernel], "chunk_size": resolved,
            "chunk_rule": "given" if chunk > 0 else "library rule (chunk_size=0)",
            "layers": nl,
            "launch": ("one CUDA graph for all layers" if sg is not None
                       else f"{nl} kvs_decode_step launch(es)"),
            "steps": steps,
            "value": bytes_all / (total_ms_max * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": total_ms_max / steps,
            "us_per_call": {"decode_step": 1e3 * mean_ms,
                            "decode_step_median": 1e3 * statistics.median(step_ms),
                            "decode_step_p10": 1e3 * percentile(step_ms, 10),
                            "decode_step_p90": 1e3 * percentile(step_ms, 90),
                            "decode_step_hot": 1e3 * hot_ms, "hot_steps": KH,
                            "hot_mode": hot_mode},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                         "traffic": traffic1,
                         "kernel": f"{KERNEL_NAMES[kernel]} (kvs_decode_step)",
                         "bytes_per_launch": ab1["step"]},
            "live_kv_bytes": W.kv_bytes(inp, w) * nl,
            "algorithmic_bytes_per_step": ab["step"],
            "cache_bytes_allocated": 2 * w.cache_elems() * 4 * nl,
            "l2": ("L2 scrubbed (2x129 MB write) between timed steps, outside the events"
                   if flush else "inputs larger than L2 (live KV bytes >> 129 MB)"),
            "seed": seed,
        }
        if nl > 1:
            res["us_per_layer"] = 1e3 * mean_ms / nl

        if full:  # the same step as kvs_kv_scatter + kvs_flash_decode, an event between
            KB = min(steps, 500)
            b_start = [torch.cuda.Event(enable_timing=True) for _ in range(KB)]
            b_end = [torch.cuda.Event(enable_timing=True) for _ in range(KB)]
            mids = [torch.cuda.Event(enable_timing=True) for _ in range(KB)]
            torch.cuda.synchronize()
            for k in range(KB):
                if flush:
                    scrub.zero_()
                b_start[k].record(stream)
                for t in ts:
                    B.kvs_kv_scatter(t["k_rows"], t["v_rows"], t["positions"], t["k_cache"],
                                     t["v_cache"], d_status=status)
                mids[k].record(stream)
                for t, out in zip(ts, outs):
                    B.kvs_flash_decode(t["q"], t["k_cache"], t["v_cache"], t["positions"], out,
                                       chunk_size=resolved, workspace=ws, d_status=status)
                b_end[k].record(stream)
            torch.cuda.synchronize()
            scatter_ms = [s.elapsed_time(m) for s, m in zip(b_start, mids)]
            decode_ms = [m.elapsed_time(e) for m, e in zip(mids, b_end)]
            res["us_per_call"].update({"kv_scatter": 1e3 * statistics.mean(scatter_ms),
                                       "flash_decode": 1e3 * statistics.mean(decode_ms),
                                       "breakdown_steps": KB})
            res["attention_gbs"] = ab["attention"] / (statistics.mean(decode_ms) * 1e-3) / 1e9
            if int(status.item()) != 0:
                raise SystemExit(f"{w.name} breakdown: device status "
                                 f"{B.strerror(int(status.item()))}")

        if ci == 0:
            res["e2e"] = measure_e2e(ctx, w, ts, inps, ws, resolved, status, scrub, warmup,
                                     e2e_steps or max(3, min(steps, 500)), ab["step"],
                                     graph=sg is not None)
        if sg is not None:
            sg.destroy()
        del ws
        results.append(res)
    if keep_inputs:  # the host inputs, for the CPU baseline on the same batch
        results[0]["_inputs"] = inp
    del ts, outs, scrub
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return results


def measure_e2e(ctx, w, ts, inps, ws, chunk, status, scrub, warmup, Ke, step_bytes,
                graph=False):
    """The step through the public host-buffer entry points, all inputs
    copied in from pinned host memory and every out copied back each step:
    with `graph` (a multi-layer step launched as one graph), one launch of a
    kvs_step_graph_create_host_io graph (one copy of every layer's q,
    k_rows, v_rows and the positions in, the layers, one copy of every out
    back); otherwise one kvs_decode_step_host_io call per layer (the same for
    one layer).  Two sets of host and device io buffers in alternation: a
    set is reused once the event after its previous step has passed, i.e.
    its output has reached the host (the host waits for it), so step k+1 is
    enqueued while step k runs."""
    torch, B, dev, stream = ctx.torch, ctx.B, ctx.dev, ctx.stream
    M, H, D = ts[0]["q"].shape
    Hkv = w.num_kv_heads
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32))
    sets = []
    for _ in range(2):
        if graph:
            h = B.HostStepIo(len(inps), M, H, Hkv, D)
            for l, x in enumerate(inps):
                h.q[l].copy_(f32(x.q))
                h.k_rows[l].copy_(f32(x.k_rows))
                h.v_rows[l].copy_(f32(x.v_rows))
            h.positions.copy_(torch.from_numpy(np.ascontiguousarray(inps[0].positions, np.int32)))
            io = torch.empty(h.total, dtype=torch.uint8, device=dev)
            # captured on a side stream of the binding's, launched on `stream`
            g = B.kvs_step_graph_create_host_io(h, [t["k_cache"] for t in ts],
                                                [t["v_cache"] for t in ts], chunk_size=chunk,
                                                workspace=ws, io=io, d_status=status)
            sets.append((h, io, g))
        else:
            hios = []
            for x in inps:
                h = B.HostIo(M, H, Hkv, D)
                h.q.copy_(f32(x.q))
                h.k_rows.copy_(f32(x.k_rows))
                h.v_rows.copy_(f32(x.v_rows))
                h.positions.copy_(torch.from_numpy(np.ascontiguousarray(x.positions, np.int32)))
                hios.append(h)
            sets.append((hios, B.step_io(M, H, Hkv, D, device=dev), None))
    if graph:
        h2d, d2h = sets[0][0].in_bytes, sets[0][0].out_bytes
    else:
        h2d = sum(h.in_bytes for h in sets[0][0])
        d2h = sum(h.out_bytes for h in sets[0][0])
    done = [None, None]

    def e2e_step(k):
        b = k % 2
        if done[b] is not None:
            done[b].synchronize()  # that set's previous output is on the host
        hios, io, g = sets[b]
        if g is not None:
            g.launch(stream)
        else:
            for l, t in enumerate(ts):
                B.kvs_decode_step_host_io(hios[l], t["k_cache"], t["v_cache"], chunk_size=chunk,
                                          workspace=ws, io=io, d_status=status, stream=stream)
        ev = torch.cuda.Event()
        ev.record(stream)
        done[b] = ev

    for k in range(warmup):
        e2e_step(k)
    torch.cuda.synchronize()
    done[0] = done[1] = None
    ctx.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record(stream)
    for k in range(Ke):
        if scrub is not None:
            scrub.zero_()
        e2e_step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    ctx.windows.append((wall0, time.time()))
    e2e_ms = e0.elapsed_time(e1) / Ke
    if scrub is not None:  # take the scrub time back out
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(Ke):
            scrub.zero_()
        s1.record(stream)
        torch.cuda.synchronize()
        e2e_ms -= s0.elapsed_time(s1) / Ke
    if int(status.item()) != 0:
        raise SystemExit(f"{w.name} e2e: device status {B.strerror(int(status.item()))}")
    _, e2e_ms_max, _, bytes_all = reduce_over_ranks(0.0, e2e_ms, 0.0, step_bytes * Ke,
                                                    ctx.world, dev)
    return {"value": bytes_all / (e2e_ms_max * Ke * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": e2e_ms_max, "steps": Ke,
            "api": ("kvs_step_graph_create_host_io, one graph launch a step (one copy in, the "
                    "layers, one copy out)" if graph else
                    "kvs_decode_step_host_io, one call per layer") +
                   "; two buffer sets in alternation"}


def brief(res):
    """The per_config view of one measurement."""
    keep = ("kernel", "chunk_size", "chunk_rule", "layers", "launch", "steps", "value", "unit",
            "ms_per_step", "us_per_call", "us_per_layer", "live_kv_bytes",
            "algorithmic_bytes_per_step", "l2", "e2e")
    out = {k: res[k] for k in keep if k in res}
    r = res["roofline"]
    out["roofline"] = {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                         "frac_of_nominal_8tbs", "traffic")}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=HEADLINE, choices=sorted(W.WORKLOADS),
                    help="the headline workload")
    ap.add_argument("--chunk", type=int, default=None, help="override the headline chunk size")
    ap.add_argument("--impl", default="kvs", choices=["kvs", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--graph", action="store_true",
                    help="launch the headline's (multi-layer) step as one captured CUDA graph")
    ap.add_argument("--only-headline", action="store_true",
                    help="measure the headline workload alone (no per_config legs)")
    ap.add_argument("--no-argmax", action="store_true",
                    help="skip the batched argmax measurement")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the tensor-core prefill measurement")
    ap.add_argument("--only", choices=["argmax", "prefill"], default=None,
                    help="run only that measurement and print its JSON object (profiling)")
    ap.add_argument("--prefill-shape", default=None,
                    help="H,S,D of the prefill measurement (default 32,4096,128)")
    ap.add_argument("--prefill-full", action="store_true",
                    help="prefill without the causal mask")
    ap.add_argument("--schedule", default="auto", choices=["auto", "persistent", "cluster"],
                    help="attention kernel (kvs_set_schedule)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank, world, local = dist_env()
    w = W.WORKLOADS[args.config]
    seed = rank_seed(w, rank)

    if args.impl == "reference":
        return run_reference(args, w, W.make_inputs(w, seed=seed), rank, world)

    import torch
    import torch.distributed as tdist

    from split_flash_decoding_kvcachescatter_gb300 import binding as B
    from split_flash_decoding_kvcachescatter_gb300 import build as kbuild

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        tdist.init_process_group("nccl", device_id=dev)
    kbuild.build()
    B.lib()
    if args.only is not None:  # one measurement alone, for profiling
        stream = torch.cuda.current_stream()
        if args.only == "argmax":
            res = time_argmax(B, torch, w.M, dev, stream, iters=args.steps)
        else:
            shape = (tuple(int(v) for v in args.prefill_shape.split(","))
                     if args.prefill_shape else PREFILL_SHAPE)
            res = time_prefill(B, torch, dev, stream, iters=args.steps, shape=shape,
                               causal=not args.prefill_full)
        print(json.dumps(res), flush=True)
        return
    B.kvs_set_schedule({"auto": B.KVS_SCHEDULE_AUTO, "persistent": B.KVS_SCHEDULE_PERSISTENT,
                        "cluster": B.KVS_SCHEDULE_CLUSTER}[args.schedule])
    ctx = Ctx(torch, tdist, B, dev, rank, world)
    sampler = ClockSampler(local)
    sampler.start()

    per_config = {}
    head = None
    legs = [args.config] if args.only_headline else \
        [n for n in PER_CONFIG if n != args.config] + [args.config]
    for name in legs:
        wl = W.WORKLOADS[name]
        is_head = name == args.config
        steps = args.steps if is_head else max(args.steps, MIN_STEPS[name])
        graph = (args.graph if is_head else wl.layers > 1)
        if is_head:
            chunks = [args.chunk if args.chunk is not None else wl.chunk_size]
        else:
            chunks = [wl.chunk_size]
        if wl.chunk_sweep and not (is_head and args.chunk is not None):
            chunks += [c for c in wl.chunk_sweep if c != chunks[0]] + [0]
        res = measure_workload(ctx, wl, rank_seed(wl, rank), steps, args.warmup, chunks,
                               graph=graph, full=is_head, e2e_steps=args.e2e_steps,
                               keep_inputs=is_head)
        entry = brief(res[0])
        if len(res) > 1:
            entry["chunk_sweep"] = [
                {"chunk_size": r["chunk_size"], "chunk_rule": r["chunk_rule"],
                 "us_per_call": r["us_per_call"]["decode_step"],
                 "us_median": r["us_per_call"]["decode_step_median"],
                 "value": r["value"], "frac": r["roofline"]["frac"],
                 "frac_of_nominal_8tbs": r["roofline"]["frac_of_nominal_8tbs"]}
                for r in res]
        per_config[name] = entry
        if is_head:
            head = res[0]

    live_read = time_stream_read(torch, dev, ctx.stream)
    argmax = time_argmax(B, torch, w.M, dev, ctx.stream) if not args.no_argmax else None
    floor = launch_floor(torch, dev, ctx.stream)
    prefill = time_prefill(B, torch, dev, ctx.stream) if not args.no_prefill else None
    sampler.stop()
    clocks = sampler.summary(ctx.windows)

    if rank != 0:
        if world > 1:
            tdist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        inp = head.pop("_inputs")
        runner = CpuOracleRunner(inp, w)
        runner.sample(0.5)  # warm the pool and the page cache
        dt, b, n = runner.sample(8.0)
        one = CpuOracleRunner(inp, w, threads=1)
        dt1, b1, n1 = one.sample(8.0)
        cpu = {"value": b / dt / 1e9, "unit": "GB/s", "cores": runner.threads, "kind": "oracle",
               "sample": runner.describe(n), **cpu_model(),
               "single_core": {"value": b1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                               "sample": one.describe(n1)}}

    roof = dict(head["roofline"])
    roof["live_stream_read"] = live_read
    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world,
        "steps": head["steps"], "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": w.name, "M": w.M, "num_heads": w.num_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "max_len": w.max_len,
            "chunk_size": head["chunk_size"], "chunk_rule": head["chunk_rule"],
            "schedule": args.schedule, "kernel": head["kernel"], "layers": head["layers"],
            "launch": head["launch"], "live_kv_bytes": head["live_kv_bytes"],
            "algorithmic_bytes_per_step": head["algorithmic_bytes_per_step"],
            "cache_bytes_allocated": head["cache_bytes_allocated"], "l2": head["l2"],
            "seed": head["seed"], "parallelism": f"replicas x{world} (independent batches)",
        },
        "us_per_call": head["us_per_call"],
        "attention_gbs": head.get("attention_gbs"),
        "roofline": roof,
        "e2e": head["e2e"],
        "gpu_launches": head["steps"] * head["layers"],
        "clocks": clocks,
        "cpu_baseline": cpu,
        "per_config": per_config,
        "argmax": argmax,
        "prefill": prefill,
        "launch_floor": floor,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
