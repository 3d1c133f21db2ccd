"""Bounded waits, tested on the GPU: kvs_set_wait_limit_ns lowers the bound on
every pipeline wait of the kernels so that waits run out on purpose.

For each kernel with waits -- the persistent decode kernel, the cluster
decode kernel and the tensor-core prefill kernel -- and for a replayed step
graph, a call under a lowered bound must
  * return KVS_OK from the host call (the kernel gives up, it does not fault),
  * record KVS_ERR_TIMEOUT in d_status when the bound is 0 (calls made under
    a lowered bound run the kernels' polling wait variant, whose first wait
    that does not find its data ready ends at once), or nothing else but
    KVS_ERR_TIMEOUT under a bound of a few microseconds (then waits run out
    at random points of the pipeline, with copies and tensor-core products
    in flight),
  * write nothing outside its output (guard zones on both sides),
and the next call, at the default bound, on the same workspace, must be
parity-green against the oracle: a timed-out call leaves nothing behind that
a later call could take for its own (the workspace counters carry an epoch
that a timed-out call changes, and a step graph writes a fresh one at each
replay).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import gate
from split_flash_decoding_kvcachescatter_gb300 import binding as B
from split_flash_decoding_kvcachescatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GUARD = 4096                # float32 guard elements on each side of an output
GUARD_BITS = 0x7FBADBAD     # a NaN bit pattern no kernel writes
LIMITS_NS = (0, 300, 1000, 3000, 10000)


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from split_flash_decoding_kvcachescatter_gb300 import build
    build.build()
    B.lib()
    yield
    torch.cuda.synchronize()


@pytest.fixture(autouse=True)
def _restore():
    """Every test leaves the default bound and the schedule as it found them."""
    prev_sched = B.kvs_get_schedule()
    yield
    torch.cuda.synchronize()
    B.kvs_set_wait_limit_ns(B.KVS_WAIT_LIMIT_DEFAULT_NS)
    B.kvs_set_schedule(prev_sched)


def guarded(shape):
    """(buffer, view): a float32 view of `shape` with guard zones around it."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), GUARD_BITS, dtype=torch.int32, device=DEV)
    return buf, buf[GUARD:GUARD + n].view(torch.float32).view(*shape)


def guards_intact(buf):
    g = torch.cat([buf[:GUARD], buf[-GUARD:]])
    return bool(torch.all(g == GUARD_BITS).item())


def test_wait_limit_setter_round_trips_and_rejects_out_of_range():
    prev = B.kvs_set_wait_limit_ns(1234)
    assert prev == B.KVS_WAIT_LIMIT_DEFAULT_NS
    assert B.kvs_set_wait_limit_ns(B.KVS_WAIT_LIMIT_DEFAULT_NS) == 1234
    with pytest.raises(B.KvsError) as e:
        B.kvs_set_wait_limit_ns(B.KVS_WAIT_LIMIT_DEFAULT_NS + 1)
    assert e.value.status == B.KVS_ERR_DIMS


def _decode_case(schedule, seed, **kw):
    B.kvs_set_schedule(schedule)
    w = W.custom(positions="uniform", seed=seed, **kw)
    assert B.kvs_schedule_for(w.M, w.num_heads, w.num_kv_heads, w.head_dim,
                              w.max_len) == schedule
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    exp = W.upload(inp, w, DEV, include_new_row=True)
    ref = oracle.decode_sequences(inp.q, inp.k_seq, inp.v_seq, inp.positions)
    return w, t, exp, ref


def _step(w, t, ws, out, status):
    B.kvs_decode_step(t["q"], t["k_rows"], t["v_rows"], t["positions"], t["k_cache"],
                      t["v_cache"], out, chunk_size=w.chunk_size, workspace=ws, d_status=status)


def _timeout_then_recover(w, t, exp, ref, what):
    M, H, D = t["q"].shape
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = B.workspace(M, H, w.num_kv_heads, D, w.max_len, w.chunk_size, device=DEV).fill_(0xFF)
    seen = {}
    for limit in LIMITS_NS:
        B.kvs_set_wait_limit_ns(limit)
        status.zero_()
        buf, out = guarded((M, H, D))
        _step(w, t, ws, out, status)  # the host call itself succeeds
        torch.cuda.synchronize()
        st = int(status.item())
        seen[limit] = st
        assert st in (B.KVS_OK, B.KVS_ERR_TIMEOUT), f"{what} limit={limit}: {B.strerror(st)}"
        assert guards_intact(buf), f"{what} limit={limit}: wrote outside out"
        # back at the default bound, on the same workspace: parity-green
        B.kvs_set_wait_limit_ns(B.KVS_WAIT_LIMIT_DEFAULT_NS)
        status.zero_()
        buf, out = guarded((M, H, D))
        _step(w, t, ws, out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"{what} after limit={limit}"
        assert guards_intact(buf)
        gate(out.cpu().numpy(), ref, where=f"{what} after a call with limit={limit}")
        for name in ("k_cache", "v_cache"):
            assert torch.equal(t[name].view(torch.int32), exp[name].view(torch.int32)), name
    assert seen[0] == B.KVS_ERR_TIMEOUT, f"{what}: a bound of 0 must time out"
    return seen


def test_persistent_kernel_times_out_and_recovers():
    w, t, exp, ref = _decode_case(B.KVS_SCHEDULE_PERSISTENT, seed=61, M=8, num_heads=32,
                                  num_kv_heads=8, head_dim=128, max_len=4096, chunk_size=0)
    _timeout_then_recover(w, t, exp, ref, "persistent")


def test_persistent_kernel_small_group_times_out_and_recovers():
    # head_dim 64 and a group of 7: 16-row stages and an 8-stage ring
    w, t, exp, ref = _decode_case(B.KVS_SCHEDULE_PERSISTENT, seed=62, M=4, num_heads=14,
                                  num_kv_heads=2, head_dim=64, max_len=2048, chunk_size=128)
    _timeout_then_recover(w, t, exp, ref, "persistent D=64 G=7")


def test_cluster_kernel_times_out_and_recovers():
    w, t, exp, ref = _decode_case(B.KVS_SCHEDULE_CLUSTER, seed=63, M=8, num_heads=32,
                                  num_kv_heads=8, head_dim=128, max_len=8192, chunk_size=0)
    _timeout_then_recover(w, t, exp, ref, "cluster")


def test_cluster_kernel_small_model_layer_times_out_and_recovers():
    w, t, exp, ref = _decode_case(B.KVS_SCHEDULE_CLUSTER, seed=64, M=4, num_heads=14,
                                  num_kv_heads=2, head_dim=64, max_len=2048, chunk_size=128)
    _timeout_then_recover(w, t, exp, ref, "cluster small model")


def test_step_graph_replay_after_a_timed_out_replay():
    """A captured step replays frozen kernel arguments, the counters' host tag
    included.  A replay that gives up part-way can leave completion counts
    behind; the graph's epoch write makes the next replay start clean.  The
    graph is captured under a lowered bound, so it holds the kernels' polling
    wait variant, which reads the bound at run time: each replay then runs
    under the bound set just before it."""
    B.kvs_set_schedule(B.KVS_SCHEDULE_PERSISTENT)
    w = W.custom(positions="uniform", seed=65, M=8, num_heads=32, num_kv_heads=8, head_dim=128,
                 max_len=2048, chunk_size=0)
    layers = 2
    pos = W.draw_positions(w)
    ins = [W.make_inputs(w, layer=l, positions=pos) for l in range(layers)]
    ts = [W.upload(x, w, DEV) for x in ins]
    refs = [oracle.decode_sequences(x.q, x.k_seq, x.v_seq, x.positions) for x in ins]
    M, H, D = ts[0]["q"].shape
    outs = [torch.full((M, H, D), float("nan"), device=DEV) for _ in range(layers)]
    ws = B.workspace(M, H, w.num_kv_heads, D, w.max_len, w.chunk_size, device=DEV).fill_(0xFF)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # configure the kernels outside the capture
    _step(w, ts[0], ws, outs[0], status)
    torch.cuda.synchronize()
    B.kvs_set_wait_limit_ns(0)
    g = B.kvs_step_graph_create([t["q"] for t in ts], [t["k_rows"] for t in ts],
                                [t["v_rows"] for t in ts], ts[0]["positions"],
                                [t["k_cache"] for t in ts], [t["v_cache"] for t in ts], outs,
                                chunk_size=w.chunk_size, workspace=ws, d_status=status)
    try:
        seen = []
        for limit in LIMITS_NS:
            B.kvs_set_wait_limit_ns(limit)
            status.zero_()
            g.launch()
            torch.cuda.synchronize()
            seen.append(int(status.item()))
            assert seen[-1] in (B.KVS_OK, B.KVS_ERR_TIMEOUT)
            B.kvs_set_wait_limit_ns(B.KVS_WAIT_LIMIT_DEFAULT_NS)
            for o in outs:
                o.fill_(float("nan"))
            status.zero_()
            g.launch()
            torch.cuda.synchronize()
            assert int(status.item()) == 0, f"replay after limit={limit}"
            for l in range(layers):
                gate(outs[l].cpu().numpy(), refs[l], where=f"layer {l} after limit={limit}")
        assert seen[0] == B.KVS_ERR_TIMEOUT
    finally:
        g.destroy()


def _prefill_inputs(H, S, D, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((H, S, D)).astype(np.float32) for _ in range(3)]


@pytest.mark.parametrize("D,H,S", [(64, 4, 1000), (128, 4, 1000), (128, 2, 2100), (64, 3, 2048)])
def test_prefill_kernel_times_out_and_recovers(D, H, S):
    # S >= 2048 adds the waits of the in-kernel packing: the copy warp's tile
    # flags and the pack warps' staged chunks
    q, k, v = _prefill_inputs(H, S, D, seed=66 + D + S)
    ref = oracle.prefill_attention(q, k, v, True)
    tq, tk, tv = (torch.from_numpy(a).to(DEV) for a in (q, k, v))
    ws = B.prefill_workspace(H, S, D, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # per-element bound of the FP16 products (as in the prefill parity test)
    v16 = np.abs(v.astype(np.float16).astype(np.float64))
    tol = 2.0 ** -11 * np.maximum.accumulate(v16, axis=1) * 1.05 + 1e-5
    seen = {}
    for limit in LIMITS_NS:
        B.kvs_set_wait_limit_ns(limit)
        status.zero_()
        buf, out = guarded((H, S, D))
        B.kvs_prefill_attention(tq, tk, tv, out, causal=True, workspace=ws, d_status=status)
        torch.cuda.synchronize()
        seen[limit] = int(status.item())
        assert seen[limit] in (B.KVS_OK, B.KVS_ERR_TIMEOUT)
        assert guards_intact(buf), f"prefill limit={limit}: wrote outside out"
        B.kvs_set_wait_limit_ns(B.KVS_WAIT_LIMIT_DEFAULT_NS)
        status.zero_()
        buf, out = guarded((H, S, D))
        B.kvs_prefill_attention(tq, tk, tv, out, causal=True, workspace=ws, d_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert guards_intact(buf)
        err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= tol), f"prefill after limit={limit}: max err {err.max():.3e}"
    assert seen[0] == B.KVS_ERR_TIMEOUT
