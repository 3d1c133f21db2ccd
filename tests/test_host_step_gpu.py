"""GPU parity of kvs_decode_step_host: the decode step called with its inputs
and result in host memory (the library enqueues the copies in and out).

Bar as for the device entry points: bit-identical caches, outputs within
max-abs 2e-5 / max-rel 1e-4 of the f64 oracle, and bit-identical to
kvs_decode_step on the same inputs (the same kernel runs on the copies).
"""
import ctypes

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
    prev = B.kvs_set_schedule(request.param)
    yield request.param
    B.kvs_set_schedule(prev)


def oracle_out(inp):
    return oracle.decode_sequences(inp.q, inp.k_seq, inp.v_seq, inp.positions)


def assert_cache_bit_exact(t, expected):
    torch.cuda.synchronize()
    for name in ("k_cache", "v_cache"):
        assert torch.equal(t[name].view(torch.int32), expected[name].view(torch.int32)), name


def host_inputs(inp, pinned=True):
    h = {"q": torch.from_numpy(np.ascontiguousarray(inp.q, np.float32)),
         "k_rows": torch.from_numpy(np.ascontiguousarray(inp.k_rows, np.float32)),
         "v_rows": torch.from_numpy(np.ascontiguousarray(inp.v_rows, np.float32)),
         "positions": torch.from_numpy(np.ascontiguousarray(inp.positions, np.int32))}
    return {k: v.pin_memory() for k, v in h.items()} if pinned else h


def host_step(w, inp, t, pinned=True, io=None, ws=None, status=None):
    M, H, D = inp.q.shape
    h = host_inputs(inp, pinned)
    out = torch.full((M, H, D), float("nan"))
    if pinned:
        out = out.pin_memory()
    io = io if io is not None else B.step_io(M, H, w.num_kv_heads, D, device=DEV)
    ws = ws if ws is not None else B.workspace(M, H, w.num_kv_heads, D, w.max_len, w.chunk_size,
                                               device=DEV)
    B.kvs_decode_step_host(h["q"], h["k_rows"], h["v_rows"], h["positions"], t["k_cache"],
                           t["v_cache"], out, chunk_size=w.chunk_size, workspace=ws, io=io,
                           d_status=status)
    return out


@pytest.mark.parametrize("name", ["tiny", "small_model"])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_step_matches_oracle(name, pinned):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    exp = W.upload(inp, w, DEV, include_new_row=True)
    t = W.upload(inp, w, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = host_step(w, inp, t, pinned=pinned, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, B.strerror(int(status.item()))
    gate(out.numpy(), oracle.decode_sequences(inp.q, inp.k_seq, inp.v_seq, inp.positions),
         where=f"{name} host step")
    for c in ("k_cache", "v_cache"):
        assert torch.equal(t[c].view(torch.int32), exp[c].view(torch.int32)), c


def test_host_step_equals_device_step_bitwise():
    w = W.custom(M=5, num_heads=40, num_kv_heads=8, head_dim=128, max_len=1300, seed=23)
    inp = W.make_inputs(w)
    t1 = W.upload(inp, w, DEV)
    t2 = W.upload(inp, w, DEV)
    ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len, w.chunk_size,
                     device=DEV)
    out_dev = torch.empty_like(t1["q"])
    B.kvs_decode_step(t1["q"], t1["k_rows"], t1["v_rows"], t1["positions"], t1["k_cache"],
                      t1["v_cache"], out_dev, chunk_size=w.chunk_size, workspace=ws)
    torch.cuda.synchronize()
    out_host = host_step(w, inp, t2)
    torch.cuda.synchronize()
    assert torch.equal(out_dev.cpu().view(torch.int32), out_host.view(torch.int32))
    for c in ("k_cache", "v_cache"):
        assert torch.equal(t1[c].view(torch.int32), t2[c].view(torch.int32)), c


def test_host_steps_in_a_row_share_one_io_buffer():
    """Three steps of one batch enqueued back to back with one io buffer and
    no synchronisation between them: the stream orders each step's copies
    after the previous step's read of out, so each result is its own."""
    w = W.custom(M=3, num_heads=8, num_kv_heads=2, head_dim=64, max_len=600, seed=29)
    inp = W.make_inputs(w, positions=np.array([5, 250, 596], np.int32))  # room for 2 more rows
    t = W.upload(inp, w, DEV)
    io = B.step_io(w.M, w.num_heads, w.num_kv_heads, w.head_dim, device=DEV)
    ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len, w.chunk_size,
                     device=DEV)
    rng = np.random.default_rng(31)
    k_seq = [np.asarray(s, np.float32) for s in inp.k_seq]
    v_seq = [np.asarray(s, np.float32) for s in inp.v_seq]
    outs, refs, keep = [], [], []
    pos = np.asarray(inp.positions, np.int32).copy()
    for step in range(3):
        q = rng.standard_normal(inp.q.shape).astype(np.float32)
        kr = rng.standard_normal(inp.k_rows.shape).astype(np.float32)
        vr = rng.standard_normal(inp.v_rows.shape).astype(np.float32)
        if step > 0:
            pos = pos + 1
            for i in range(w.M):
                k_seq[i] = np.concatenate([k_seq[i], kr[i][:, None, :]], axis=1)
                v_seq[i] = np.concatenate([v_seq[i], vr[i][:, None, :]], axis=1)
        else:
            kr, vr = np.asarray(inp.k_rows, np.float32), np.asarray(inp.v_rows, np.float32)
        h = {n: torch.from_numpy(a).pin_memory() for n, a in
             (("q", q), ("k_rows", kr), ("v_rows", vr), ("positions", pos.copy()))}
        out = torch.full(inp.q.shape, float("nan")).pin_memory()
        B.kvs_decode_step_host(h["q"], h["k_rows"], h["v_rows"], h["positions"], t["k_cache"],
                               t["v_cache"], out, chunk_size=w.chunk_size, workspace=ws, io=io)
        keep.append(h)  # the pinned inputs stay alive until the stream is done
        outs.append(out)
        refs.append(oracle.decode_sequences(q, k_seq, v_seq, pos))
    torch.cuda.synchronize()
    for step, (o, r) in enumerate(zip(outs, refs)):
        gate(o.numpy(), r, where=f"step {step}")


def test_host_step_rejects_device_tensors_in_the_binding():
    w = W.WORKLOADS["tiny"]
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    io = B.step_io(w.M, w.num_heads, w.num_kv_heads, w.head_dim, device=DEV)
    ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len, w.chunk_size,
                     device=DEV)
    with pytest.raises(TypeError):
        B.kvs_decode_step_host(t["q"], t["k_rows"], t["v_rows"], t["positions"], t["k_cache"],
                               t["v_cache"], torch.empty(inp.q.shape), chunk_size=w.chunk_size,
                               workspace=ws, io=io)


def fill_host_io(hio, inp):
    hio.q.copy_(torch.from_numpy(np.ascontiguousarray(inp.q, np.float32)))
    hio.k_rows.copy_(torch.from_numpy(np.ascontiguousarray(inp.k_rows, np.float32)))
    hio.v_rows.copy_(torch.from_numpy(np.ascontiguousarray(inp.v_rows, np.float32)))
    hio.positions.copy_(torch.from_numpy(np.ascontiguousarray(inp.positions, np.int32)))
    hio.out.fill_(float("nan"))


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("name", ["tiny", "small_model", "8b_batch"])
def test_host_io_step_matches_oracle_and_device_step(name, pinned):
    """kvs_decode_step_host_io: one host buffer in the io layout, moved in
    and out by the library's copy kernel (pinned) or by copy engines
    (pageable); the same attention kernel as kvs_decode_step, so the output
    is bit-identical to it, and within the gate of the oracle."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    exp = W.upload(inp, w, DEV, include_new_row=True)
    t = W.upload(inp, w, DEV)
    t_dev = W.upload(inp, w, DEV)
    M, H, D = inp.q.shape
    hio = B.HostIo(M, H, w.num_kv_heads, D, pinned=pinned)
    fill_host_io(hio, inp)
    io = B.step_io(M, H, w.num_kv_heads, D, device=DEV)
    ws = B.workspace(M, H, w.num_kv_heads, D, w.max_len, w.chunk_size, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.kvs_decode_step_host_io(hio, t["k_cache"], t["v_cache"], chunk_size=w.chunk_size,
                              workspace=ws, io=io, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, B.strerror(int(status.item()))
    gate(hio.out.numpy(), oracle.decode_sequences(inp.q, inp.k_seq, inp.v_seq, inp.positions),
         where=f"{name} host io step")
    out_dev = torch.empty_like(t_dev["q"])
    B.kvs_decode_step(t_dev["q"], t_dev["k_rows"], t_dev["v_rows"], t_dev["positions"],
                      t_dev["k_cache"], t_dev["v_cache"], out_dev, chunk_size=w.chunk_size,
                      workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_dev.cpu().view(torch.int32), hio.out.view(torch.int32))
    for c in ("k_cache", "v_cache"):
        assert torch.equal(t[c].view(torch.int32), exp[c].view(torch.int32)), c


def test_host_io_steps_double_buffered_without_synchronisation():
    """Two host buffers and two io buffers used in alternation, six steps of
    one batch enqueued with no host synchronisation between them (each
    buffer's previous step is waited for with an event before it is
    rewritten): every step's result is its own."""
    w = W.custom(M=3, num_heads=8, num_kv_heads=2, head_dim=64, max_len=600, seed=37)
    inp = W.make_inputs(w, positions=np.array([5, 250, 590], np.int32))  # room for 5 more rows
    t = W.upload(inp, w, DEV)
    M, H, D = inp.q.shape
    hios = [B.HostIo(M, H, w.num_kv_heads, D) for _ in range(2)]
    ios = [B.step_io(M, H, w.num_kv_heads, D, device=DEV) for _ in range(2)]
    ws = B.workspace(M, H, w.num_kv_heads, D, w.max_len, w.chunk_size, device=DEV)
    done = [None, None]      # event after each buffer's latest step
    pending = [None, None]   # the oracle's result for that step
    rng = np.random.default_rng(41)
    k_seq = [np.asarray(s, np.float32) for s in inp.k_seq]
    v_seq = [np.asarray(s, np.float32) for s in inp.v_seq]
    pos = np.asarray(inp.positions, np.int32).copy()
    results = []
    for step in range(6):
        b = step % 2
        if done[b] is not None:  # the buffer's previous step: result copied out, inputs read
            done[b].synchronize()
            results.append((hios[b].out.clone(), pending[b]))
        q = rng.standard_normal(inp.q.shape).astype(np.float32)
        if step == 0:
            kr, vr = np.asarray(inp.k_rows, np.float32), np.asarray(inp.v_rows, np.float32)
        else:
            kr = rng.standard_normal(inp.k_rows.shape).astype(np.float32)
            vr = rng.standard_normal(inp.v_rows.shape).astype(np.float32)
            pos = pos + 1
            for i in range(M):
                k_seq[i] = np.concatenate([k_seq[i], kr[i][:, None, :]], axis=1)
                v_seq[i] = np.concatenate([v_seq[i], vr[i][:, None, :]], axis=1)
        h = hios[b]
        h.q.copy_(torch.from_numpy(q))
        h.k_rows.copy_(torch.from_numpy(kr))
        h.v_rows.copy_(torch.from_numpy(vr))
        h.positions.copy_(torch.from_numpy(pos.copy()))
        B.kvs_decode_step_host_io(h, t["k_cache"], t["v_cache"], chunk_size=w.chunk_size,
                                  workspace=ws, io=ios[b])
        ev = torch.cuda.Event()
        ev.record()
        done[b] = ev
        pending[b] = oracle.decode_sequences(q, k_seq, v_seq, pos)
    torch.cuda.synchronize()
    for b in (0, 1):
        results.append((hios[b].out.clone(), pending[b]))
    assert len(results) == 6
    for n, (o, r) in enumerate(results):
        gate(o.numpy(), r, where=f"double-buffered step {n}")


def test_step_graph_host_io_equals_device_step_graph():
    """kvs_step_graph_create_host_io: every layer's inputs in one pinned host
    buffer; outputs bit-identical to kvs_step_graph_create on the same inputs
    (the same kernels run on the copies), within the gate of the oracle, and
    the caches bit-exact; then a second token through the same graphs."""
    layers = 3
    w = W.custom(M=4, num_heads=14, num_kv_heads=2, head_dim=64, max_len=700, chunk_size=64,
                 seed=81)
    pos = W.draw_positions(w)
    ins = [W.make_inputs(w, layer=l, positions=pos) for l in range(layers)]
    M, H, D = ins[0].q.shape
    # the device step graph on one set of caches, the host-io graph on another
    td = [W.upload(x, w, DEV) for x in ins]
    th = [W.upload(x, w, DEV) for x in ins]
    exps = [W.upload(x, w, DEV, include_new_row=True) for x in ins]
    outs = [torch.full_like(t["q"], float("nan")) for t in td]
    ws_d = B.workspace(M, H, w.num_kv_heads, D, w.max_len, 64, device=DEV)
    ws_h = B.workspace(M, H, w.num_kv_heads, D, w.max_len, 64, device=DEV)
    st_d = torch.zeros(1, dtype=torch.int32, device=DEV)
    st_h = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.Stream()
    gd = B.kvs_step_graph_create([t["q"] for t in td], [t["k_rows"] for t in td],
                                 [t["v_rows"] for t in td], td[0]["positions"],
                                 [t["k_cache"] for t in td], [t["v_cache"] for t in td], outs,
                                 chunk_size=64, workspace=ws_d, d_status=st_d, stream=stream)
    hio = B.HostStepIo(layers, M, H, w.num_kv_heads, D)
    io = torch.empty(hio.total, dtype=torch.uint8, device=DEV)
    gh = B.kvs_step_graph_create_host_io(hio, [t["k_cache"] for t in th],
                                         [t["v_cache"] for t in th], chunk_size=64,
                                         workspace=ws_h, io=io, d_status=st_h, stream=stream)

    def fill(inputs, positions):
        for l, x in enumerate(inputs):
            hio.q[l].copy_(torch.from_numpy(np.ascontiguousarray(x.q, np.float32)))
            hio.k_rows[l].copy_(torch.from_numpy(np.ascontiguousarray(x.k_rows, np.float32)))
            hio.v_rows[l].copy_(torch.from_numpy(np.ascontiguousarray(x.v_rows, np.float32)))
            hio.out[l].fill_(float("nan"))
        hio.positions.copy_(torch.from_numpy(np.ascontiguousarray(positions, np.int32)))

    fill(ins, pos)
    gd.launch(stream)
    gh.launch(stream)
    stream.synchronize()
    assert int(st_d.item()) == 0 and int(st_h.item()) == 0
    for l in range(layers):
        assert torch.equal(outs[l].cpu().view(torch.int32), hio.out[l].view(torch.int32)), l
        gate(hio.out[l].numpy(), oracle_out(ins[l]), where=f"host-io graph layer {l}")
        assert_cache_bit_exact(th[l], exps[l])
    # a second token: new inputs at the same addresses, next positions
    pos2 = np.minimum(pos + 1, w.max_len - 1).astype(np.int32)
    ins2 = [W.make_inputs(w, layer=l, positions=pos2, seed=82) for l in range(layers)]
    for l in range(layers):
        for tt in (td[l], th[l]):
            fresh = W.upload(ins2[l], w, DEV)
            for name in ("q", "k_rows", "v_rows", "k_cache", "v_cache"):
                tt[name].copy_(fresh[name])
    td[0]["positions"].copy_(torch.from_numpy(pos2).to(DEV))
    fill(ins2, pos2)
    gd.launch(stream)
    gh.launch(stream)
    stream.synchronize()
    for l in range(layers):
        assert torch.equal(outs[l].cpu().view(torch.int32), hio.out[l].view(torch.int32)), l
        gate(hio.out[l].numpy(), oracle_out(ins2[l]), where=f"host-io graph relaunch layer {l}")
    gd.destroy()
    gh.destroy()


def test_step_graph_host_io_rejects_pageable_memory():
    w = W.custom(M=2, num_heads=4, num_kv_heads=2, head_dim=64, max_len=64, chunk_size=32,
                 seed=83)
    t = W.upload(W.make_inputs(w), w, DEV)
    off = B.kvs_step_graph_io_layout(1, 2, 4, 2, 64)
    pageable = torch.empty(off[-1], dtype=torch.uint8)  # not pinned
    io = torch.empty(off[-1], dtype=torch.uint8, device=DEV)
    ws = B.workspace(2, 4, 2, 64, 64, 32, device=DEV)
    h = ctypes.c_void_p()
    caches_k = (ctypes.c_void_p * 1)(t["k_cache"].data_ptr())
    caches_v = (ctypes.c_void_p * 1)(t["v_cache"].data_ptr())
    stream = torch.cuda.Stream()
    rc = B.lib().kvs_step_graph_create_host_io(
        1, pageable.data_ptr(), io.data_ptr(), off[-1], caches_k, caches_v, 2, 4, 2, 64, 64, 32,
        ws.data_ptr(), ws.numel(), None, stream.cuda_stream, ctypes.byref(h))
    assert rc == B.KVS_ERR_UNSUPPORTED
    assert not h.value
