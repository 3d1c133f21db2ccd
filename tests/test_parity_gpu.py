"""GPU parity: the CUDA path (through the C ABI) against the f64 CPU oracle.

Bar: the scattered caches are bit-identical to the expected caches (every
byte, untouched rows included); attention outputs are within max-abs 2e-5
and max-rel 1e-4 (relative error taken where |oracle| >= 0.2) of the oracle.
Inputs are the seeded synthetic workloads; rows past each position are
poisoned with NaN so any read beyond row p shows up.
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from split_flash_decoding_kvcachescatter_gb300 import build
    build.build()
    B.lib()
    yield
    torch.cuda.synchronize()


@pytest.fixture(autouse=True, params=[B.KVS_SCHEDULE_PERSISTENT, B.KVS_SCHEDULE_CLUSTER],
                ids=["persistent", "cluster"])
def schedule(request, _built):
    """Every test here runs on both kernels: the persistent split-K kernel
    (partials merged through the workspace) and the cluster kernel (partials
    merged in distributed shared memory)."""
    prev = B.kvs_set_schedule(request.param)
    yield request.param
    B.kvs_set_schedule(prev)


def run_step(t, w, chunk, status=None, ws=None, poison_ws=True, fused=False):
    """One decode step through the C ABI; returns out (device).

    fused=False: kvs_kv_scatter then kvs_flash_decode (two launches);
    fused=True:  kvs_decode_step (one launch)."""
    M, H, D = t["q"].shape
    if ws is None:
        ws = B.workspace(M, H, w.num_kv_heads, D, w.max_len, chunk, device=DEV)
    if poison_ws:
        ws.fill_(0xFF)
    out = torch.full((M, H, D), float("nan"), device=DEV)
    if fused:
        B.kvs_decode_step(t["q"], t["k_rows"], t["v_rows"], t["positions"], t["k_cache"],
                          t["v_cache"], out, chunk_size=chunk, workspace=ws, d_status=status)
    else:
        B.kvs_kv_scatter(t["k_rows"], t["v_rows"], t["positions"], t["k_cache"], t["v_cache"],
                         d_status=status)
        B.kvs_flash_decode(t["q"], t["k_cache"], t["v_cache"], t["positions"], out,
                           chunk_size=chunk, workspace=ws, d_status=status)
    return out


def assert_cache_bit_exact(t, expected):
    torch.cuda.synchronize()
    for name in ("k_cache", "v_cache"):
        same = torch.equal(t[name].view(torch.int32), expected[name].view(torch.int32))
        assert same, f"{name} differs from the expected scatter result"


def oracle_out(inp):
    return oracle.decode_sequences(inp.q, inp.k_seq, inp.v_seq, inp.positions)


def check_workload(w, chunks, layer=0, inp=None):
    """Both entry paths (two launches, and the fused step) against the oracle,
    for every chunk size, plus the bit-exact caches."""
    inp = inp if inp is not None else W.make_inputs(w, layer=layer)
    exp = W.upload(inp, w, DEV, include_new_row=True)
    ref = oracle_out(inp)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    results = {}
    for fused in (False, True):
        t = W.upload(inp, w, DEV)
        for c in chunks:
            out = run_step(t, w, c, status, fused=fused)
            torch.cuda.synchronize()
            assert int(status.item()) == 0, B.strerror(int(status.item()))
            results[(fused, c)] = gate(out.cpu().numpy(), ref,
                                       where=f"{w.name} chunk={c} fused={fused}")
        assert_cache_bit_exact(t, exp)
        del t
    del exp
    torch.cuda.empty_cache()
    return results


# ---------------------------------------------------------------- workloads
def test_tiny_full_oracle_layout():
    """tiny: also run the oracle's own scatter on the host cache layout."""
    w = W.WORKLOADS["tiny"]
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    host_k = t["k_cache"].cpu().numpy().copy()
    host_v = t["v_cache"].cpu().numpy().copy()
    assert oracle.kv_scatter(inp.k_rows, inp.v_rows, inp.positions, host_k, host_v) == 0
    ref = oracle.decode(inp.q, host_k, host_v, inp.positions)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_step(t, w, w.chunk_size, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gate(out.cpu().numpy(), ref, where="tiny")
    assert np.array_equal(t["k_cache"].cpu().numpy().view(np.int32), host_k.view(np.int32))
    assert np.array_equal(t["v_cache"].cpu().numpy().view(np.int32), host_v.view(np.int32))


def test_small_model_all_24_layers():
    w = W.WORKLOADS["small_model"]
    pos = W.draw_positions(w)
    for layer in range(w.layers):
        inp = W.make_inputs(w, layer=layer, positions=pos)
        check_workload(w, [w.chunk_size], inp=inp)


@pytest.mark.slow
def test_8b_batch_with_outliers():
    w = W.WORKLOADS["8b_batch"]
    check_workload(w, [0, 256])


@pytest.mark.slow
def test_long_context_chunk_sweep():
    w = W.WORKLOADS["long_context"]
    check_workload(w, list(w.chunk_sweep) + [0])


@pytest.mark.slow
def test_ragged_serving_mix():
    w = W.WORKLOADS["ragged"]
    check_workload(w, [w.chunk_size])


# ---------------------------------------------------------------- shapes
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (6, 2), (8, 2), (10, 2), (12, 2), (14, 2),
                                   (16, 2)])
def test_group_sizes_and_head_dims(D, H, Hkv):
    w = W.custom(M=5, num_heads=H, num_kv_heads=Hkv, head_dim=D, max_len=700, chunk_size=100,
                 positions="uniform", seed=31 + H + D)
    check_workload(w, [1 if H == 4 and Hkv == 4 else 37, 100, 128, 1000])


@pytest.mark.parametrize("chunk", [1, 7, 33, 64, 255, 256, 4096])
def test_chunk_sizes_ragged_tail(chunk):
    w = W.custom(M=3, num_heads=8, num_kv_heads=2, head_dim=128, max_len=1000,
                 chunk_size=chunk, positions="uniform", seed=5)
    check_workload(w, [chunk])


# ---------------------------------------------------------------- edge cases
def test_seq_len_one_returns_v_row_bitwise():
    w = W.custom(M=6, num_heads=8, num_kv_heads=2, head_dim=128, max_len=64,
                 positions="fixed", fixed_position=0, seed=3)
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    out = run_step(t, w, 16).cpu().numpy()
    G = w.group
    for i in range(w.M):
        for h in range(w.num_heads):
            assert np.array_equal(out[i, h].view(np.int32), inp.v_rows[i, h // G].view(np.int32))


def test_last_position_and_mixed_lengths():
    w = W.custom(M=4, num_heads=32, num_kv_heads=8, head_dim=128, max_len=513,
                 positions="uniform", seed=9)
    pos = np.array([512, 0, 1, 300], np.int32)
    inp = W.make_inputs(w, positions=pos)
    check_workload(w, [64, 0], inp=inp)


def test_out_of_range_positions_flag_and_skip():
    w = W.custom(M=4, num_heads=8, num_kv_heads=2, head_dim=64, max_len=128, seed=11)
    pos = np.array([5, 128, -1, 127], np.int32)
    inp = W.make_inputs(w, positions=pos)
    t = W.upload(inp, w, DEV)
    exp = W.upload(inp, w, DEV, include_new_row=True)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_step(t, w, 32, status).cpu().numpy()
    assert int(status.item()) == B.KVS_ERR_POSITION
    assert np.all(np.isnan(out[1])) and np.all(np.isnan(out[2]))
    good = [0, 3]
    ref = oracle.decode_sequences(inp.q[good], [inp.k_seq[i] for i in good],
                                  [inp.v_seq[i] for i in good], pos[good])
    gate(out[good], ref, where="valid sequences beside invalid ones")
    assert_cache_bit_exact(t, exp)


def test_empty_batch_is_a_no_op():
    L = B.lib()
    assert L.kvs_kv_scatter(None, None, None, None, None, 0, 2, 64, 16, None, None) == 0
    assert L.kvs_flash_decode(None, None, None, None, None, 0, 4, 2, 64, 16, 8, None, 0,
                              None, None) == 0


def test_repeatable_and_stream_ordered():
    """Two calls give identical bits; a non-default stream works."""
    w = W.custom(M=8, num_heads=32, num_kv_heads=8, head_dim=128, max_len=2000, seed=13)
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        a = run_step(t, w, 0)
        b = run_step(t, w, 0)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    gate(a.cpu().numpy(), oracle_out(inp), where="side stream")


def test_fused_step_equals_scatter_then_decode_bitwise():
    """kvs_decode_step = kvs_kv_scatter + kvs_flash_decode, bit for bit."""
    w = W.custom(M=6, num_heads=40, num_kv_heads=8, head_dim=128, max_len=1500, seed=17)
    inp = W.make_inputs(w)
    t1 = W.upload(inp, w, DEV)
    t2 = W.upload(inp, w, DEV)
    a = run_step(t1, w, 64)
    b = run_step(t2, w, 64, fused=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    for name in ("k_cache", "v_cache"):
        assert torch.equal(t1[name].view(torch.int32), t2[name].view(torch.int32))


def test_fused_step_bad_position_flags_and_skips():
    w = W.custom(M=3, num_heads=8, num_kv_heads=2, head_dim=128, max_len=64, seed=23)
    pos = np.array([10, 64, 63], np.int32)
    inp = W.make_inputs(w, positions=pos)
    t = W.upload(inp, w, DEV)
    exp = W.upload(inp, w, DEV, include_new_row=True)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_step(t, w, 16, status, fused=True).cpu().numpy()
    assert int(status.item()) == B.KVS_ERR_POSITION
    assert np.all(np.isnan(out[1]))
    good = [0, 2]
    ref = oracle.decode_sequences(inp.q[good], [inp.k_seq[i] for i in good],
                                  [inp.v_seq[i] for i in good], pos[good])
    gate(out[good], ref, where="fused step beside an invalid position")
    assert_cache_bit_exact(t, exp)


def test_workspace_reuse_across_shapes_and_calls():
    """One workspace, garbage-filled, reused by calls of different shapes: the
    tagged counters must never take a stale value as this call's."""
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=DEV)
    ws.fill_(0x5A)
    for seed, (M, H, Hkv, L) in enumerate([(4, 32, 8, 3000), (2, 8, 2, 700), (4, 32, 8, 3000)]):
        w = W.custom(M=M, num_heads=H, num_kv_heads=Hkv, head_dim=128, max_len=L, seed=50 + seed)
        inp = W.make_inputs(w)
        t = W.upload(inp, w, DEV)
        for fused in (False, True, True):
            t = W.upload(inp, w, DEV)
            out = run_step(t, w, 32, ws=ws, poison_ws=False, fused=fused)
            torch.cuda.synchronize()
            gate(out.cpu().numpy(), oracle_out(inp), where=f"reuse {seed} fused={fused}")


def test_workspace_too_small_is_rejected_before_launch():
    w = W.custom(M=2, num_heads=4, num_kv_heads=2, head_dim=64, max_len=256, seed=19)
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    n = B.kvs_flash_decode_workspace_bytes(2, 4, 2, 64, 256, 64)
    small = torch.empty(n - 256, dtype=torch.uint8, device=DEV)
    out = torch.zeros_like(t["q"])
    with pytest.raises(B.KvsError) as e:
        B.kvs_flash_decode(t["q"], t["k_cache"], t["v_cache"], t["positions"], out,
                           chunk_size=64, workspace=small)
    assert e.value.status == B.KVS_ERR_WORKSPACE
    assert torch.count_nonzero(out).item() == 0


def test_graph_replay_with_new_inputs():
    """A captured CUDA graph freezes every kernel argument; replays with new
    inputs copied into the captured buffers must still match the oracle."""
    w = W.custom(M=8, num_heads=32, num_kv_heads=8, head_dim=128, max_len=3000, seed=61)
    inp_a = W.make_inputs(w, seed=61)
    inp_b = W.make_inputs(w, seed=62)
    t = W.upload(inp_a, w, DEV)
    ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len, 0, device=DEV)
    ws.fill_(0x33)
    out = torch.empty_like(t["q"])

    def step():
        B.kvs_decode_step(t["q"], t["k_rows"], t["v_rows"], t["positions"], t["k_cache"],
                          t["v_cache"], out, chunk_size=0, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # first call on the device configures the kernel outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for inp in (inp_a, inp_b, inp_a):
        fresh = W.upload(inp, w, DEV)
        for name in fresh:
            t[name].copy_(fresh[name])
        g.replay()
        torch.cuda.synchronize()
        gate(out.cpu().numpy(), oracle_out(inp), where="graph replay")


def test_step_graph_multi_layer():
    """kvs_step_graph_create: L layers' decode steps in one graph launch, then
    relaunched after new inputs are copied into the same buffers."""
    layers = 4
    w = W.custom(M=4, num_heads=14, num_kv_heads=2, head_dim=64, max_len=900, chunk_size=64,
                 seed=70)
    pos = W.draw_positions(w)
    ins = [W.make_inputs(w, layer=l, positions=pos) for l in range(layers)]
    ts = [W.upload(x, w, DEV) for x in ins]
    exps = [W.upload(x, w, DEV, include_new_row=True) for x in ins]
    outs = [torch.full_like(t["q"], float("nan")) for t in ts]
    ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len, 64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.Stream()
    g = B.kvs_step_graph_create([t["q"] for t in ts], [t["k_rows"] for t in ts],
                                [t["v_rows"] for t in ts], ts[0]["positions"],
                                [t["k_cache"] for t in ts], [t["v_cache"] for t in ts], outs,
                                chunk_size=64, workspace=ws, d_status=status, stream=stream)
    g.launch(stream)
    stream.synchronize()
    assert int(status.item()) == 0
    for l in range(layers):
        gate(outs[l].cpu().numpy(), oracle_out(ins[l]), where=f"graph layer {l}")
        assert_cache_bit_exact(ts[l], exps[l])
    # a second token: new q and rows, next positions, same buffers
    pos2 = np.minimum(pos + 1, w.max_len - 1).astype(np.int32)
    ins2 = [W.make_inputs(w, layer=l, positions=pos2, seed=71) for l in range(layers)]
    for l in range(layers):
        fresh = W.upload(ins2[l], w, DEV)
        for name in ("q", "k_rows", "v_rows", "k_cache", "v_cache"):
            ts[l][name].copy_(fresh[name])
    ts[0]["positions"].copy_(torch.from_numpy(pos2).to(DEV))
    g.launch(stream)
    stream.synchronize()
    for l in range(layers):
        gate(outs[l].cpu().numpy(), oracle_out(ins2[l]), where=f"graph relaunch layer {l}")
    g.destroy()


def test_step_graph_bad_position_and_length_one():
    """A step graph whose shared positions hold a bad position and a
    sequence of one row: every layer flags KVS_ERR_POSITION and leaves NaN
    in the bad sequence's rows, and the others match the oracle (the layers
    after the first read the positions before their dependency wait)."""
    layers = 3
    w = W.custom(M=4, num_heads=14, num_kv_heads=2, head_dim=64, max_len=300, chunk_size=64,
                 seed=72)
    pos = np.array([0, 300, 157, 299], np.int32)
    ins = [W.make_inputs(w, layer=l, positions=pos) for l in range(layers)]
    ts = [W.upload(x, w, DEV) for x in ins]
    exps = [W.upload(x, w, DEV, include_new_row=True) for x in ins]
    outs = [torch.zeros_like(t["q"]) for t in ts]
    ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len, 64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.Stream()
    g = B.kvs_step_graph_create([t["q"] for t in ts], [t["k_rows"] for t in ts],
                                [t["v_rows"] for t in ts], ts[0]["positions"],
                                [t["k_cache"] for t in ts], [t["v_cache"] for t in ts], outs,
                                chunk_size=64, workspace=ws, d_status=status, stream=stream)
    g.launch(stream)
    stream.synchronize()
    assert int(status.item()) == B.KVS_ERR_POSITION
    good = [0, 2, 3]
    for l in range(layers):
        out = outs[l].cpu().numpy()
        assert np.all(np.isnan(out[1])), f"layer {l}: bad sequence not NaN"
        ref = oracle.decode_sequences(ins[l].q[good], [ins[l].k_seq[i] for i in good],
                                      [ins[l].v_seq[i] for i in good], pos[good])
        gate(out[good], ref, where=f"graph layer {l} beside an invalid position")
        assert_cache_bit_exact(ts[l], exps[l])
    g.destroy()


# ---------------------------------------------------------------- schedules
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("max_len", [1, 2, 31, 32, 33, 100, 513, 1200])
def test_cache_lengths_across_cluster_sizes(schedule, D, max_len):
    """Cache lengths that give every cluster size from 1 to 16 (and slices
    of 0, 1 or a few rows per block), with the first and last positions."""
    w = W.custom(M=4, num_heads=8, num_kv_heads=2, head_dim=D, max_len=max_len,
                 positions="uniform", seed=71 + max_len + D)
    assert B.kvs_schedule_for(w.M, w.num_heads, w.num_kv_heads, D, max_len) == schedule
    pos = np.array([max_len - 1, 0, (max_len - 1) // 2, max(0, max_len - 2)], np.int32)
    inp = W.make_inputs(w, positions=pos)
    check_workload(w, [16], inp=inp)


def test_many_pairs_fall_back_to_the_persistent_kernel(schedule):
    """M * Hkv above one grid dimension (65535 clusters) takes the persistent
    kernel under every schedule; with one row per sequence the output is the
    V row itself, bit for bit."""
    w = W.custom(M=8193, num_heads=16, num_kv_heads=8, head_dim=64, max_len=1,
                 positions="fixed", fixed_position=0, seed=17)
    assert B.kvs_schedule_for(w.M, w.num_heads, w.num_kv_heads, 64, 1) == \
        B.KVS_SCHEDULE_PERSISTENT
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_step(t, w, 16, status, fused=True).cpu().numpy()
    assert int(status.item()) == 0
    G = w.group
    for h in range(w.num_heads):
        assert np.array_equal(out[:, h].view(np.int32), inp.v_rows[:, h // G].view(np.int32))


def test_auto_schedule_picks_by_size():
    prev = B.kvs_set_schedule(B.KVS_SCHEDULE_AUTO)
    try:
        tiny, small = W.WORKLOADS["tiny"], W.WORKLOADS["small_model"]
        big = W.WORKLOADS["8b_batch"]
        # 32 (sequence, kv head) pairs need more clusters than stay resident
        many = W.custom(M=4, num_heads=32, num_kv_heads=8, head_dim=128, max_len=2048)
        for w, want in ((tiny, B.KVS_SCHEDULE_CLUSTER), (small, B.KVS_SCHEDULE_CLUSTER),
                        (big, B.KVS_SCHEDULE_PERSISTENT), (many, B.KVS_SCHEDULE_PERSISTENT)):
            got = B.kvs_schedule_for(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len)
            assert got == want, w.name
        check_workload(tiny, [tiny.chunk_size])
    finally:
        B.kvs_set_schedule(prev)



# ---------------------------------------------------------------- pool slots, finished sequences
def _pool_case(w, S, seed, slots=None, done=None):
    """Device pool [S][Hkv][Lmax][D] holding sequence i's live rows in slot
    slots[i] (other slots poisoned), plus the matching numpy arrays."""
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    rng = np.random.default_rng(seed)
    if slots is None:
        slots = rng.permutation(S)[:w.M].astype(np.int32)
    if done is None:
        done = np.zeros(w.M, np.uint8)
    pool_k = W.poisoned_cache(W.custom(M=S, num_heads=w.num_heads, num_kv_heads=w.num_kv_heads,
                                       head_dim=w.head_dim, max_len=w.max_len), DEV)
    pool_v = pool_k.clone()
    ok = [i for i in range(w.M) if 0 <= slots[i] < S]
    idx = torch.tensor([int(slots[i]) for i in ok], dtype=torch.long, device=DEV)
    src = torch.tensor(ok, dtype=torch.long, device=DEV)
    pool_k[idx] = t["k_cache"][src]
    pool_v[idx] = t["v_cache"][src]
    return inp, t, slots, done, pool_k, pool_v


def _oracle_pool_step(inp, slots, done, pool_k, pool_v, out_before):
    kp, vp = pool_k.cpu().numpy().copy(), pool_v.cpu().numpy().copy()
    out = out_before.copy()
    bad = oracle.decode_step_slots(inp.q, inp.k_rows, inp.v_rows, inp.positions, slots, done,
                                   kp, vp, out)
    return out, kp, vp, bad


@pytest.mark.parametrize("D,H,Hkv", [(64, 14, 2), (128, 32, 8), (128, 40, 8)])
def test_pool_slots_and_finished_sequences(schedule, D, H, Hkv):
    w = W.custom(M=6, num_heads=H, num_kv_heads=Hkv, head_dim=D, max_len=300,
                 positions="uniform", seed=101 + D + H)
    S = 9
    done = np.array([0, 1, 0, 0, 1, 0], np.uint8)
    inp, t, slots, done, pk, pv = _pool_case(w, S, seed=5, done=done)
    before = np.random.default_rng(7).standard_normal((w.M, H, D)).astype(np.float32)
    ref, kp_ref, vp_ref, bad = _oracle_pool_step(inp, slots, done, pk, pv, before)
    assert bad == []
    out = torch.from_numpy(before).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = B.workspace(w.M, H, Hkv, D, w.max_len, 32, device=DEV).fill_(0xFF)
    B.kvs_decode_step_slots(t["q"], t["k_rows"], t["v_rows"], t["positions"],
                            torch.from_numpy(slots).to(DEV), torch.from_numpy(done).to(DEV),
                            pk, pv, out, chunk_size=32, workspace=ws, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy()
    live = np.flatnonzero(done == 0)
    fin = np.flatnonzero(done != 0)
    gate(got[live], ref[live], where=f"pool slots D={D} G={H // Hkv}")
    assert np.array_equal(got[fin].view(np.int32), before[fin].view(np.int32))
    assert np.array_equal(pk.cpu().numpy().view(np.int32), kp_ref.view(np.int32))
    assert np.array_equal(pv.cpu().numpy().view(np.int32), vp_ref.view(np.int32))
    # attention only (no new rows) over the scattered pool gives the same bits
    out2 = torch.from_numpy(before).to(DEV)
    B.kvs_decode_step_slots(t["q"], None, None, t["positions"], torch.from_numpy(slots).to(DEV),
                            torch.from_numpy(done).to(DEV), pk, pv, out2, chunk_size=32,
                            workspace=ws, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(out2.cpu().numpy().view(np.int32), got.view(np.int32))
    assert np.array_equal(pk.cpu().numpy().view(np.int32), kp_ref.view(np.int32))


def test_pool_identity_slots_equal_decode_step(schedule):
    """slots None and done None is kvs_decode_step, bit for bit."""
    w = W.custom(M=4, num_heads=8, num_kv_heads=2, head_dim=128, max_len=777, seed=23)
    inp = W.make_inputs(w)
    a, b = W.upload(inp, w, DEV), W.upload(inp, w, DEV)
    ws = B.workspace(w.M, 8, 2, 128, w.max_len, 64, device=DEV)
    out_a = torch.empty_like(a["q"])
    out_b = torch.empty_like(b["q"])
    B.kvs_decode_step(a["q"], a["k_rows"], a["v_rows"], a["positions"], a["k_cache"],
                      a["v_cache"], out_a, chunk_size=64, workspace=ws)
    B.kvs_decode_step_slots(b["q"], b["k_rows"], b["v_rows"], b["positions"], None, None,
                            b["k_cache"], b["v_cache"], out_b, chunk_size=64, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int32), out_b.view(torch.int32))
    assert torch.equal(a["k_cache"].view(torch.int32), b["k_cache"].view(torch.int32))
    assert torch.equal(a["v_cache"].view(torch.int32), b["v_cache"].view(torch.int32))


def test_pool_bad_slot_flags_and_skips(schedule):
    w = W.custom(M=4, num_heads=8, num_kv_heads=2, head_dim=64, max_len=200, seed=29)
    S = 6
    slots = np.array([3, 6, 0, -2], np.int32)   # 6 and -2 are outside the pool
    done = np.array([0, 0, 0, 1], np.uint8)     # the last is finished as well
    inp, t, slots, done, pk, pv = _pool_case(w, S, seed=1, slots=slots, done=done)
    before = np.full((w.M, 8, 64), 7.0, np.float32)
    ref, kp_ref, vp_ref, bad = _oracle_pool_step(inp, slots, done, pk, pv, before)
    assert bad == [1, 3]
    out = torch.from_numpy(before).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = B.workspace(w.M, 8, 2, 64, w.max_len, 16, device=DEV)
    B.kvs_decode_step_slots(t["q"], t["k_rows"], t["v_rows"], t["positions"],
                            torch.from_numpy(slots).to(DEV), torch.from_numpy(done).to(DEV),
                            pk, pv, out, chunk_size=16, workspace=ws, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == B.KVS_ERR_SLOT
    got = out.cpu().numpy()
    assert np.all(np.isnan(got[1]))
    assert np.array_equal(got[3], before[3])     # finished: left as it was
    gate(got[[0, 2]], ref[[0, 2]], where="valid slots beside bad ones")
    assert np.array_equal(pk.cpu().numpy().view(np.int32), kp_ref.view(np.int32))
    assert np.array_equal(pv.cpu().numpy().view(np.int32), vp_ref.view(np.int32))
