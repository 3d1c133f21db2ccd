"""Benchmark of one decode step of the attention hot path on GB300.

A step = one layer's decode step of a seeded synthetic workload through the C
ABI: kvs_decode_step, i.e. the KV-cache scatter of the new rows, the split
plan, the chunk partials and the rescaled merge, all in one kernel launch.
The same step as kvs_kv_scatter + kvs_flash_decode (two launches) is timed
beside it for the per-call breakdown.  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--chunk C] [--impl kvs|reference]

value      : algorithmic GB/s of the step (live KV bytes read + Q read + O
             written + positions, plus the scatter's row bytes), inputs resident
             in HBM, device time from CUDA events, max over ranks.
e2e        : the same metric when every step also copies its inputs (q, new K/V
             rows, positions) from pinned host memory and reads the output back,
             all through kvs_decode_step_host (one C call per layer).
us_per_call: the step's mean, median, p10 and p90 over the timed steps
             (L2 scrubbed between steps when the working set fits in it), the
             hot mean of back-to-back steps, and the two-launch breakdown.
roofline   : the step kernel (the step's one launch): its algorithmic bytes /
             its mean event-timed duration, against the measured HBM copy
             bandwidth.
cpu_baseline: the f64 CPU oracle on the host cores (rank 0, N=1 only).
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
FALLBACK_HBM_GBS = 6800.0
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
    """Tensor-core prefill attention (kvs_prefill_attention): the FP16 pack
    launch and the tcgen05 attention launch, timed together.  At the default
    shape the inputs (3 x 67 MB) and the packed workspace exceed L2."""
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
    return {"kernel": "prefill_pack_kernel + prefill_tc_kernel (kvs_prefill_attention)",
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

    def summary(self, t0, t1):
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
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:  # timed region shorter than the sampling interval
            inside = rows
            window = "warmup + timed region"
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
    workload, in rotation, on all host cores (the C call releases the GIL).
    A sample is time-bounded: batches of units run until the budget is spent."""

    def __init__(self, inp, w):
        from concurrent.futures import ThreadPoolExecutor
        import oracle
        oracle.build()
        self.oracle = oracle
        self.inp, self.w = inp, w
        self.threads = os.cpu_count() or 1
        self.pool = ThreadPoolExecutor(max_workers=self.threads)
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
            done_bytes += sum(self.pool.map(self._one, us))
            n += batch
            if time.perf_counter() - t0 >= budget_s:
                break
        return time.perf_counter() - t0, done_bytes, n

    def describe(self, n_units, passes=None):
        return (f"{n_units} (sequence, query head) units of the {self.w.name} workload in "
                f"rotation ({len(self.units)} units = the whole batch), f64 C oracle on "
                f"{self.threads} host threads")


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
                         "kind": "oracle", "sample": runner.describe(tot_n)},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="8b_batch", choices=sorted(W.WORKLOADS))
    ap.add_argument("--chunk", type=int, default=None, help="override the chunk size")
    ap.add_argument("--impl", default="kvs", choices=["kvs", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--graph", action="store_true",
                    help="launch the whole (multi-layer) step as one captured CUDA graph")
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
    inp = W.make_inputs(w, seed=seed)

    if args.impl == "reference":
        return run_reference(args, w, inp, rank, world)

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
    kernel = ("cluster" if B.kvs_schedule_for(w.M, w.num_heads, w.num_kv_heads, w.head_dim,
                                               w.max_len) == B.KVS_SCHEDULE_CLUSTER
              else "persistent")

    def barrier():
        if world > 1:
            tdist.barrier()

    nl = w.layers  # a step covers every layer of the workload (24 for small_model)
    inps = [inp] + [W.make_inputs(w, layer=l, seed=seed, positions=inp.positions)
                    for l in range(1, nl)]
    ts = [W.upload(x, w, dev) for x in inps]
    chunk = args.chunk if args.chunk is not None else w.chunk_size
    resolved_chunk = chunk if chunk > 0 else B.kvs_choose_chunk_size(
        w.M, w.num_kv_heads, w.head_dim, w.max_len)
    ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len, resolved_chunk,
                     device=dev)
    outs = [torch.empty_like(t["q"]) for t in ts]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ab1 = W.algorithmic_bytes(inp, w)  # one layer; every layer has the same positions
    ab = {k: v * nl for k, v in ab1.items()}
    cache_bytes = 2 * w.cache_elems() * 4 * nl
    flush = ab["step"] < 4 * L2_BYTES  # small working sets: scrub L2 between steps
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    stream = torch.cuda.current_stream()

    def eager_step():
        """The whole hot path, one launch per layer: scatter, split plan, chunk
        partials and the rescaled merge (kvs_decode_step)."""
        for t, out in zip(ts, outs):
            B.kvs_decode_step(t["q"], t["k_rows"], t["v_rows"], t["positions"], t["k_cache"],
                              t["v_cache"], out, chunk_size=resolved_chunk, workspace=ws,
                              d_status=status)

    graph = None
    if args.graph:
        eager_step()  # configure the kernels outside the capture
        torch.cuda.synchronize()
        graph = B.kvs_step_graph_create(
            [t["q"] for t in ts], [t["k_rows"] for t in ts], [t["v_rows"] for t in ts],
            ts[0]["positions"], [t["k_cache"] for t in ts], [t["v_cache"] for t in ts], outs,
            chunk_size=resolved_chunk, workspace=ws, d_status=status)
        for t in ts[1:]:  # the graph reads the positions of layer 0 for every layer
            t["positions"] = ts[0]["positions"]

    def step():
        if graph is not None:
            graph.launch(stream)
        else:
            eager_step()

    def two_calls(mid):
        """The same step as the two separate entry points (all layers' scatters,
        an event, then all layers' attention)."""
        for t in ts:
            B.kvs_kv_scatter(t["k_rows"], t["v_rows"], t["positions"], t["k_cache"],
                             t["v_cache"], d_status=status)
        mid.record(stream)
        for t, out in zip(ts, outs):
            B.kvs_flash_decode(t["q"], t["k_cache"], t["v_cache"], t["positions"], out,
                               chunk_size=resolved_chunk, workspace=ws, d_status=status)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        if flush:
            scrub.zero_()
        step()
    torch.cuda.synchronize()

    K = args.steps
    # Region A (the headline): events only at step boundaries, so the
    # programmatic launch overlap between the step's kernels is untouched.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    for k in range(K):
        if flush:
            scrub.zero_()
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall1 = time.time()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    # Region B (breakdown): the step as kvs_kv_scatter + kvs_flash_decode,
    # an event between the two launches.
    KB = min(K, 500)
    b_start = [torch.cuda.Event(enable_timing=True) for _ in range(KB)]
    b_end = [torch.cuda.Event(enable_timing=True) for _ in range(KB)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(KB)]
    torch.cuda.synchronize()
    for k in range(KB):
        if flush:
            scrub.zero_()
        b_start[k].record(stream)
        two_calls(mids[k])
        b_end[k].record(stream)
    torch.cuda.synchronize()
    scatter_ms = [s.elapsed_time(m) for s, m in zip(b_start, mids)]
    decode_ms = [m.elapsed_time(e) for m, e in zip(mids, b_end)]
    if int(status.item()) != 0:
        raise SystemExit(f"device status: {B.strerror(int(status.item()))}")

    # ---- hot: the same step back to back, nothing between steps (L2 warm) ----
    # The eager steps are captured into one CUDA graph of HOT_CHUNK steps and
    # replayed, so that the host's launch rate does not set the time (the
    # step graph of --graph is launched back to back as it is).
    HOT_CHUNK = 20
    hot_reps = max(1, min(K, 200) // HOT_CHUNK)
    torch.cuda.synchronize()
    hot_mode = "step graph launched back to back"
    if graph is not None:
        hot_run, KH = step, hot_reps * HOT_CHUNK
        hot_calls = KH
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
            hot_run, KH = step, hot_reps * HOT_CHUNK
            hot_calls = KH
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

    # ---- e2e: host buffers through the public API ----
    # kvs_decode_step_host: one library call per layer enqueues the copies of
    # that layer's inputs (pinned host memory) to the device, the fused step,
    # and the copy of its output back to the host.
    Ke = args.e2e_steps or max(3, min(K, 500))
    names = ("q", "k_rows", "v_rows", "positions")
    host = [{k: t[k].cpu().pin_memory() for k in names} for t in ts]
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    io = B.step_io(w.M, w.num_heads, w.num_kv_heads, w.head_dim, device=dev)
    h2d = sum(v.numel() * v.element_size() for h in host for v in h.values())
    d2h = sum(o.numel() * o.element_size() for o in host_out)

    def e2e_step():
        for l, t in enumerate(ts):
            B.kvs_decode_step_host(host[l]["q"], host[l]["k_rows"], host[l]["v_rows"],
                                   host[l]["positions"], t["k_cache"], t["v_cache"], host_out[l],
                                   chunk_size=resolved_chunk, workspace=ws, io=io,
                                   d_status=status, stream=stream)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(Ke):
        if flush:
            scrub.zero_()
        e2e_step()
        # the result must be on the host before the step counts as done
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / Ke
    if flush:  # take the scrub time back out
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(Ke):
            scrub.zero_()
        s1.record(stream)
        torch.cuda.synchronize()
        e2e_ms -= s0.elapsed_time(s1) / Ke
    live_read = time_stream_read(torch, dev, stream)
    argmax = time_argmax(B, torch, w.M, dev, stream) if not args.no_argmax else None
    prefill = time_prefill(B, torch, dev, stream) if not args.no_prefill else None
    sampler.stop()
    clocks = sampler.summary(wall0, wall1)

    # ---- reduce over ranks ----
    total_ms_max, e2e_ms_max, bytes_all, bytes_e2e_all = reduce_over_ranks(
        total_ms, e2e_ms, ab["step"] * K, ab["step"] * Ke, world, dev)

    if rank != 0:
        if world > 1:
            tdist.destroy_process_group()
        return

    value = bytes_all / (total_ms_max * 1e-3) / 1e9
    e2e_value = bytes_e2e_all / (e2e_ms_max * Ke * 1e-3) / 1e9
    # A step is one launch of the step kernel per layer and nothing else, so
    # the headline events time exactly those launches: bytes per launch over
    # the mean launch time is the step's bytes over the step's time.
    step_mean_ms = total_ms / K
    achieved = ab["step"] / (step_mean_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    traffic = ncu_traffic(kernel, w.name, resolved_chunk)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        runner = CpuOracleRunner(inp, w)
        runner.sample(0.5)  # warm the pool and the page cache
        dt, b, n = runner.sample(10.0)
        cpu = {"value": b / dt / 1e9, "unit": "GB/s", "cores": runner.threads, "kind": "oracle",
               "sample": runner.describe(n)}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": w.name, "M": w.M, "num_heads": w.num_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "max_len": w.max_len,
            "chunk_size": resolved_chunk,
            "chunk_rule": "given" if chunk > 0 else "library rule (chunk_size=0)",
            "schedule": args.schedule, "kernel": KERNEL_NAMES[kernel],
            "layers": nl, "launch": ("one CUDA graph for all layers" if graph is not None
                                     else f"{nl} kvs_decode_step launch(es)"),
            "live_kv_bytes": W.kv_bytes(inp, w) * nl,
            "algorithmic_bytes_per_step": ab["step"],
            "cache_bytes_allocated": cache_bytes,
            "l2": ("L2 scrubbed (2x129 MB write) between timed steps, outside the events"
                   if flush else "inputs larger than L2 (live KV bytes >> 129 MB)"),
            "seed": seed, "parallelism": f"replicas x{world} (independent batches)",
        },
        "us_per_call": {"decode_step": 1e3 * step_mean_ms,
                        "decode_step_median": 1e3 * statistics.median(step_ms),
                        "decode_step_p10": 1e3 * percentile(step_ms, 10),
                        "decode_step_p90": 1e3 * percentile(step_ms, 90),
                        "decode_step_hot": 1e3 * hot_ms,
                        "hot_steps": KH, "hot_mode": hot_mode,
                        "kv_scatter": 1e3 * statistics.mean(scatter_ms),
                        "flash_decode": 1e3 * statistics.mean(decode_ms),
                        "breakdown_steps": KB},
        "attention_gbs": ab["attention"] / (statistics.mean(decode_ms) * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": f"{KERNEL_NAMES[kernel]} (kvs_decode_step)",
                     "peak_source": peak_kind,
                     "bytes_per_launch": ab1["step"],
                     "live_stream_read": live_read},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_max},
        "gpu_launches": K * nl,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "argmax": argmax,
        "prefill": prefill,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
