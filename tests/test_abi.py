"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/kvsdecode.h declares, and rejects bad
arguments with the documented status before touching CUDA."""
import ctypes
import os
import re

import pytest

from split_flash_decoding_kvcachescatter_gb300 import binding as B
from split_flash_decoding_kvcachescatter_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvsdecode.h")


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvs_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert isinstance(getattr(L, name), ctypes._CFuncPtr)


def test_strerror_covers_all_codes(L):
    for code in range(0, 11):
        s = B.strerror(code)
        assert s and "unknown" not in s
    assert "unknown" in B.strerror(99)


P = ctypes.c_void_p
A16 = 1 << 20  # an aligned fake address; never dereferenced (validation fails first)


@pytest.mark.parametrize("args,code", [
    ((None, None, None, None, None, -1, 2, 64, 16), B.KVS_ERR_DIMS),
    ((None, None, None, None, None, 1, 0, 64, 16), B.KVS_ERR_DIMS),
    ((None, None, None, None, None, 1, 2, 64, 0), B.KVS_ERR_DIMS),
    ((None, None, None, None, None, 1, 2, 96, 16), B.KVS_ERR_UNSUPPORTED),
    ((None, None, None, None, None, 1, 2, 64, 16), B.KVS_ERR_NULL),
    ((A16, A16, A16, A16 + 4, A16, 1, 2, 64, 16), B.KVS_ERR_ALIGN),
    ((A16, A16 + 8, A16, A16, A16, 1, 2, 64, 16), B.KVS_ERR_ALIGN),
    ((A16, A16, A16 + 2, A16, A16, 1, 2, 64, 16), B.KVS_ERR_ALIGN),
])
def test_scatter_validation(L, args, code):
    assert L.kvs_kv_scatter(*args, None, None) == code


def test_scatter_empty_batch_ok(L):
    assert L.kvs_kv_scatter(None, None, None, None, None, 0, 2, 64, 16, None, None) == 0


def _fd(L, q=A16, k=A16, v=A16, pos=A16, out=A16, M=1, H=4, Hkv=2, D=64, Lmax=256, C=64,
        ws=A16, wsb=1 << 30):
    return L.kvs_flash_decode(q, k, v, pos, out, M, H, Hkv, D, Lmax, C, ws, wsb, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), B.KVS_ERR_DIMS),
    (dict(H=0), B.KVS_ERR_DIMS),
    (dict(H=6, Hkv=4), B.KVS_ERR_DIMS),
    (dict(Lmax=0), B.KVS_ERR_DIMS),
    (dict(C=-5), B.KVS_ERR_DIMS),
    (dict(D=80), B.KVS_ERR_UNSUPPORTED),
    (dict(D=256), B.KVS_ERR_UNSUPPORTED),
    (dict(H=18, Hkv=2), B.KVS_ERR_UNSUPPORTED),
    (dict(q=None), B.KVS_ERR_NULL),
    (dict(k=None), B.KVS_ERR_NULL),
    (dict(out=None), B.KVS_ERR_NULL),
    (dict(pos=None), B.KVS_ERR_NULL),
    (dict(q=A16 + 4), B.KVS_ERR_ALIGN),
    (dict(v=A16 + 12), B.KVS_ERR_ALIGN),
    (dict(out=A16 + 8), B.KVS_ERR_ALIGN),
    (dict(ws=None), B.KVS_ERR_WORKSPACE),
    (dict(ws=A16 + 16), B.KVS_ERR_ALIGN),
    (dict(wsb=100), B.KVS_ERR_WORKSPACE),
])
def test_flash_decode_validation(L, kw, code):
    assert _fd(L, **kw) == code


def _ds(L, q=A16, kr=A16, vr=A16, pos=A16, k=A16, v=A16, out=A16, M=1, H=4, Hkv=2, D=64,
        Lmax=256, C=64, ws=A16, wsb=1 << 30):
    return L.kvs_decode_step(q, kr, vr, pos, k, v, out, M, H, Hkv, D, Lmax, C, ws, wsb, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), B.KVS_ERR_DIMS),
    (dict(H=6, Hkv=4), B.KVS_ERR_DIMS),
    (dict(D=96), B.KVS_ERR_UNSUPPORTED),
    (dict(kr=None), B.KVS_ERR_NULL),
    (dict(vr=None), B.KVS_ERR_NULL),
    (dict(k=None), B.KVS_ERR_NULL),
    (dict(out=None), B.KVS_ERR_NULL),
    (dict(kr=A16 + 4), B.KVS_ERR_ALIGN),
    (dict(v=A16 + 8), B.KVS_ERR_ALIGN),
    (dict(ws=None), B.KVS_ERR_WORKSPACE),
    (dict(wsb=64), B.KVS_ERR_WORKSPACE),
])
def test_decode_step_validation(L, kw, code):
    assert _ds(L, **kw) == code


def test_flash_decode_empty_batch_ok(L):
    assert _fd(L, M=0, q=None, k=None, v=None, pos=None, out=None, ws=None, wsb=0) == 0


def test_workspace_bytes_formula(L):
    # 256-byte header, one 8-byte completion counter per (sequence, kv head),
    # then per partial slot (M*Hkv + 1024 slots, G query heads each) a float2
    # (m, l) and D floats of accumulator; each section starts on a 256-byte
    # boundary.
    up = lambda x: -(-x // 256) * 256
    for (M, H, Hkv, D, Lmax, C) in [(1, 4, 2, 64, 256, 64), (8, 32, 8, 128, 32768, 128),
                                    (32, 40, 8, 128, 131072, 256), (3, 8, 2, 128, 1000, 7)]:
        G = H // Hkv
        slots = M * Hkv + 1024
        off_ml = up(256 + M * Hkv * 8)
        off_acc = up(off_ml + slots * G * 8)
        assert B.kvs_flash_decode_workspace_bytes(M, H, Hkv, D, Lmax, C) == up(off_acc + slots * G * D * 4)
        # independent of max_len and chunk size
        assert B.kvs_flash_decode_workspace_bytes(M, H, Hkv, D, 7, 1) == \
            B.kvs_flash_decode_workspace_bytes(M, H, Hkv, D, Lmax, C)
    assert B.kvs_flash_decode_workspace_bytes(1, 6, 4, 64, 16, 8) == 0


def test_chunk_rule_is_pow2_in_range(L):
    for sms in (1, 76, 152, 160):
        for (M, Hkv, D, Lmax) in [(1, 2, 64, 256), (32, 8, 128, 8192), (8, 8, 128, 32768),
                                  (32, 8, 128, 131072), (1, 1, 128, 1 << 20)]:
            c = B.kvs_choose_chunk_size(M, Hkv, D, Lmax, sms)
            assert 16 <= c <= 64 and (c & (c - 1)) == 0
    # more SMs never asks for larger chunks
    assert B.kvs_choose_chunk_size(32, 8, 128, 8192, 152) <= \
        B.kvs_choose_chunk_size(32, 8, 128, 8192, 76)
    with pytest.raises(B.KvsError):
        B.kvs_choose_chunk_size(0, 8, 128, 8192, 152)


def test_chunk_rule_matches_its_documented_thresholds(L):
    # r = M * Hkv * max_len // (2 * SMs) cache rows per block: 16 below 4096,
    # 32 below 8192, else 64 (the header's rule); positions play no part
    for sms in (1, 76, 152):
        for (M, Hkv, Lmax) in [(1, 2, 256), (4, 2, 2048), (32, 8, 8192), (8, 8, 32768),
                               (32, 8, 131072), (1, 1, 4096 * 304), (1, 1, 4096 * 304 - 1),
                               (1, 1, 8192 * 304), (1, 1, 8192 * 304 - 1)]:
            r = M * Hkv * Lmax // (2 * sms)
            want = 16 if r < 4096 else (32 if r < 8192 else 64)
            assert B.kvs_choose_chunk_size(M, Hkv, 128, Lmax, sms) == want, (M, Hkv, Lmax, sms)


def test_wait_limit_rejects_values_above_the_default_before_touching_cuda(L):
    prev = ctypes.c_uint64(7)
    assert L.kvs_set_wait_limit_ns(B.KVS_WAIT_LIMIT_DEFAULT_NS + 1, ctypes.byref(prev)) == \
        B.KVS_ERR_DIMS
    assert prev.value == 7  # untouched
    assert L.kvs_set_wait_limit_ns((1 << 64) - 1, None) == B.KVS_ERR_DIMS


def test_step_graph_host_checks(L):
    h = ctypes.c_void_p()
    args = [None] * 7
    # no output handle
    assert L.kvs_step_graph_create(1, *args, 1, 4, 2, 64, 16, 0, None, 0, None, A16, None) == \
        B.KVS_ERR_NULL
    # zero layers, negative chunk, legacy default stream: rejected before any CUDA call
    assert L.kvs_step_graph_create(0, *args, 1, 4, 2, 64, 16, 0, None, 0, None, A16,
                                   ctypes.byref(h)) == B.KVS_ERR_DIMS
    assert L.kvs_step_graph_create(1, *args, 1, 4, 2, 64, 16, -1, None, 0, None, A16,
                                   ctypes.byref(h)) == B.KVS_ERR_DIMS
    assert L.kvs_step_graph_create(1, *args, 1, 4, 2, 64, 16, 0, None, 0, None, None,
                                   ctypes.byref(h)) == B.KVS_ERR_NULL
    assert L.kvs_step_graph_destroy(None) == 0
    assert L.kvs_step_graph_launch(None, None) == B.KVS_ERR_NULL


def test_schedule_set_get_and_rule(L):
    prev = B.kvs_set_schedule(B.KVS_SCHEDULE_AUTO)
    try:
        assert B.kvs_get_schedule() == B.KVS_SCHEDULE_AUTO
        # automatic rule, the part decided before any device query: full
        # caches above 64 MiB of K/V, or more pairs than a grid dimension,
        # always take the persistent kernel
        assert B.kvs_schedule_for(32, 32, 8, 128, 8192) == B.KVS_SCHEDULE_PERSISTENT  # 2 GiB
        assert B.kvs_schedule_for(8, 32, 8, 128, 1025) == B.KVS_SCHEDULE_PERSISTENT
        assert B.kvs_schedule_for(65536, 1, 1, 64, 1) == B.KVS_SCHEDULE_PERSISTENT
        assert B.kvs_set_schedule(B.KVS_SCHEDULE_PERSISTENT) == B.KVS_SCHEDULE_AUTO
        assert B.kvs_schedule_for(1, 4, 2, 64, 256) == B.KVS_SCHEDULE_PERSISTENT
        assert B.kvs_set_schedule(B.KVS_SCHEDULE_CLUSTER) == B.KVS_SCHEDULE_PERSISTENT
        assert B.kvs_schedule_for(32, 32, 8, 128, 8192) == B.KVS_SCHEDULE_CLUSTER
        assert B.kvs_schedule_for(65535, 1, 1, 64, 1) == B.KVS_SCHEDULE_CLUSTER
        assert B.kvs_schedule_for(65536, 1, 1, 64, 1) == B.KVS_SCHEDULE_PERSISTENT
        with pytest.raises(B.KvsError):
            B.kvs_set_schedule(7)
        assert B.kvs_get_schedule() == B.KVS_SCHEDULE_CLUSTER  # unchanged by a bad value
        with pytest.raises(B.KvsError):
            B.kvs_schedule_for(1, 4, 2, 96, 16)
        with pytest.raises(B.KvsError):
            B.kvs_schedule_for(0, 4, 2, 64, 16)
        with pytest.raises(B.KvsError):
            B.kvs_schedule_for(1, 4, 3, 64, 16)
    finally:
        B.kvs_set_schedule(prev)


def test_prepare_validates_before_touching_cuda(L):
    assert L.kvs_prepare(4, 3, 64) == B.KVS_ERR_DIMS
    assert L.kvs_prepare(0, 1, 64) == B.KVS_ERR_DIMS
    assert L.kvs_prepare(4, 2, 96) == B.KVS_ERR_UNSUPPORTED
    assert L.kvs_prepare(18, 2, 64) == B.KVS_ERR_UNSUPPORTED


def _dss(L, q=A16, kr=A16, vr=A16, pos=A16, slots=A16, done=A16, k=A16, v=A16, S=4, out=A16,
         M=2, H=4, Hkv=2, D=64, Lmax=16, C=8, ws=A16, wsb=1 << 30):
    return L.kvs_decode_step_slots(q, kr, vr, pos, slots, done, k, v, S, out, M, H, Hkv, D, Lmax,
                                   C, ws, wsb, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), B.KVS_ERR_DIMS),
    (dict(S=0), B.KVS_ERR_DIMS),
    (dict(slots=None, S=1), B.KVS_ERR_DIMS),       # slot i needs num_slots >= M
    (dict(H=6, Hkv=4), B.KVS_ERR_DIMS),
    (dict(D=96), B.KVS_ERR_UNSUPPORTED),
    (dict(kr=None), B.KVS_ERR_NULL),               # one of the new-row inputs alone
    (dict(vr=None), B.KVS_ERR_NULL),
    (dict(q=None), B.KVS_ERR_NULL),
    (dict(k=None), B.KVS_ERR_NULL),
    (dict(kr=A16 + 4), B.KVS_ERR_ALIGN),
    (dict(slots=A16 + 2), B.KVS_ERR_ALIGN),
    (dict(k=A16 + 8), B.KVS_ERR_ALIGN),
    (dict(ws=None), B.KVS_ERR_WORKSPACE),
    (dict(wsb=64), B.KVS_ERR_WORKSPACE),
])
def test_decode_step_slots_validation(L, kw, code):
    assert _dss(L, **kw) == code


def test_decode_step_slots_empty_batch_ok(L):
    assert _dss(L, M=0, q=None, kr=None, vr=None, pos=None, slots=None, done=None, k=None,
                v=None, out=None, ws=None, wsb=0) == 0


@pytest.mark.parametrize("args,code", [
    ((A16, -1, 10, A16), B.KVS_ERR_DIMS),
    ((A16, 1, 0, A16), B.KVS_ERR_DIMS),
    ((None, 1, 10, A16), B.KVS_ERR_NULL),
    ((A16, 1, 10, None), B.KVS_ERR_NULL),
    ((A16 + 2, 1, 10, A16), B.KVS_ERR_ALIGN),
    ((A16, 1, 10, A16 + 1), B.KVS_ERR_ALIGN),
    ((None, 0, 10, None), B.KVS_OK),
])
def test_argmax_validation(L, args, code):
    assert L.kvs_argmax(*args, None) == code


@pytest.mark.parametrize("args,code", [
    ((A16, A16, A16, A16, -1, 16, 64, 1, A16, 1 << 30), B.KVS_ERR_DIMS),
    ((A16, A16, A16, A16, 2, -1, 64, 1, A16, 1 << 30), B.KVS_ERR_DIMS),
    ((A16, A16, A16, A16, 70000, 16, 64, 1, A16, 1 << 30), B.KVS_ERR_DIMS),
    ((A16, A16, A16, A16, 1, 65535 * 128 + 1, 64, 1, A16, 1 << 62), B.KVS_ERR_DIMS),
    ((A16, A16, A16, A16, 2, 16, 96, 1, A16, 1 << 30), B.KVS_ERR_UNSUPPORTED),
    ((None, A16, A16, A16, 2, 16, 64, 1, A16, 1 << 30), B.KVS_ERR_NULL),
    ((A16, A16, None, A16, 2, 16, 64, 0, A16, 1 << 30), B.KVS_ERR_NULL),
    ((A16, A16 + 4, A16, A16, 2, 16, 64, 1, A16, 1 << 30), B.KVS_ERR_ALIGN),
    ((A16, A16, A16, A16 + 8, 2, 16, 128, 1, A16, 1 << 30), B.KVS_ERR_ALIGN),
    ((A16, A16, A16, A16, 2, 16, 64, 1, None, 1 << 30), B.KVS_ERR_WORKSPACE),
    ((A16, A16, A16, A16, 2, 16, 64, 1, A16 + 16, 1 << 30), B.KVS_ERR_ALIGN),
    ((A16, A16, A16, A16, 2, 16, 64, 1, A16, 3 * 2 * 128 * 64 * 2 - 1), B.KVS_ERR_WORKSPACE),
    ((None, None, None, None, 0, 16, 64, 1, None, 0), B.KVS_OK),
    ((None, None, None, None, 2, 0, 64, 1, None, 0), B.KVS_OK),
])
def test_prefill_validation(L, args, code):
    assert L.kvs_prefill_attention(*args, None, None) == code


def test_prefill_workspace_formula(L):
    # a 4-byte flag per tile and a task counter, padded to 256 bytes, then q,
    # k and v as FP16 tiles of 128 rows: 3 * H * ceil(S / 128) * 128 * D * 2
    for H, S, D in [(1, 1, 64), (2, 128, 64), (3, 129, 128), (32, 4096, 128)]:
        T = -(-S // 128)
        flags = -(-(4 * (3 * H * T + 1)) // 256) * 256
        want = flags + 3 * H * T * 128 * D * 2
        assert L.kvs_prefill_workspace_bytes(H, S, D) == want
    assert L.kvs_prefill_workspace_bytes(0, 16, 64) == 0
    assert L.kvs_prefill_workspace_bytes(2, 16, 96) == 0


def _dsh(L, q=A16, kr=A16, vr=A16, pos=A16, k=A16, v=A16, out=A16, M=1, H=4, Hkv=2, D=64,
         Lmax=256, C=64, io=A16, iob=1 << 30, ws=A16, wsb=1 << 30):
    return L.kvs_decode_step_host(q, kr, vr, pos, k, v, out, M, H, Hkv, D, Lmax, C, io, iob, ws,
                                  wsb, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), B.KVS_ERR_DIMS),
    (dict(H=6, Hkv=4), B.KVS_ERR_DIMS),
    (dict(D=96), B.KVS_ERR_UNSUPPORTED),
    (dict(q=None), B.KVS_ERR_NULL),
    (dict(kr=None), B.KVS_ERR_NULL),
    (dict(pos=None), B.KVS_ERR_NULL),
    (dict(out=None), B.KVS_ERR_NULL),
    (dict(io=None), B.KVS_ERR_NULL),
    (dict(k=None), B.KVS_ERR_NULL),
    (dict(io=A16 + 16), B.KVS_ERR_ALIGN),
    (dict(k=A16 + 8), B.KVS_ERR_ALIGN),
    (dict(iob=64), B.KVS_ERR_WORKSPACE),
    (dict(ws=None), B.KVS_ERR_WORKSPACE),
    (dict(wsb=64), B.KVS_ERR_WORKSPACE),
    # host buffers need no alignment: they are only copied from and to
    (dict(q=A16 + 4, kr=A16 + 4, vr=A16 + 4, pos=A16 + 2, out=A16 + 4, iob=64), B.KVS_ERR_WORKSPACE),
])
def test_decode_step_host_validation(L, kw, code):
    assert _dsh(L, **kw) == code


def test_decode_step_host_empty_batch_ok(L):
    assert _dsh(L, M=0, q=None, kr=None, vr=None, pos=None, k=None, v=None, out=None, io=None,
                iob=0, ws=None, wsb=0) == 0


def test_step_io_bytes_formula(L):
    # q, k_rows, v_rows, positions, out, each rounded up to 256 bytes
    def r(x):
        return -(-x // 256) * 256
    for M, H, Hkv, D in [(1, 4, 2, 64), (3, 14, 2, 64), (32, 32, 8, 128), (5, 40, 8, 128)]:
        qo, kv = M * H * D * 4, M * Hkv * D * 4
        assert L.kvs_step_io_bytes(M, H, Hkv, D) == 2 * r(qo) + 2 * r(kv) + r(4 * M)
    assert L.kvs_step_io_bytes(0, 4, 2, 64) == 0
    assert L.kvs_step_io_bytes(1, 4, 0, 64) == 0


def test_step_io_layout_matches_io_bytes(L):
    def r(x):
        return -(-x // 256) * 256
    for M, H, Hkv, D in [(1, 4, 2, 64), (3, 14, 2, 64), (32, 32, 8, 128), (5, 40, 8, 128)]:
        oq, ok, ov, op, oo, total = B.kvs_step_io_layout(M, H, Hkv, D)
        qo, kv = M * H * D * 4, M * Hkv * D * 4
        assert (oq, ok, ov, op, oo) == (0, r(qo), r(qo) + r(kv), r(qo) + 2 * r(kv),
                                        r(qo) + 2 * r(kv) + r(4 * M))
        assert total == L.kvs_step_io_bytes(M, H, Hkv, D)
    off = (ctypes.c_size_t * 6)()
    assert L.kvs_step_io_layout(0, 4, 2, 64, off) == B.KVS_ERR_DIMS
    assert L.kvs_step_io_layout(1, 4, 2, 64, None) == B.KVS_ERR_NULL


def test_step_graph_io_layout(L):
    """Every layer's q, k_rows, v_rows, then the positions, then every
    layer's out, each 256-byte aligned and in that order."""
    def r(x):
        return -(-x // 256) * 256
    for layers, M, H, Hkv, D in [(1, 1, 4, 2, 64), (3, 4, 14, 2, 64), (24, 4, 14, 2, 64),
                                 (2, 32, 32, 8, 128), (2, 5, 40, 8, 128)]:
        off = B.kvs_step_graph_io_layout(layers, M, H, Hkv, D)
        assert len(off) == 4 * layers + 2
        qo, kv = r(M * H * D * 4), r(M * Hkv * D * 4)
        at = 0
        for l in range(layers):
            assert off[3 * l: 3 * l + 3] == [at, at + qo, at + qo + kv]
            at += qo + 2 * kv
        assert off[3 * layers] == at
        at += r(4 * M)
        for l in range(layers):
            assert off[3 * layers + 1 + l] == at + l * qo
        assert off[4 * layers + 1] == at + layers * qo
    off = (ctypes.c_size_t * 6)()
    assert L.kvs_step_graph_io_layout(0, 1, 4, 2, 64, off) == B.KVS_ERR_DIMS
    assert L.kvs_step_graph_io_layout(1, 1, 4, 0, 64, off) == B.KVS_ERR_DIMS
    assert L.kvs_step_graph_io_layout(1, 1, 4, 2, 64, None) == B.KVS_ERR_NULL


def test_step_graph_create_host_io_rejects_before_any_device_work(L):
    """Argument checks that need no device: a NULL handle pointer, bad sizes,
    NULL buffers, the legacy default stream, a misaligned or short io buffer."""
    h = ctypes.c_void_p()
    caches = (ctypes.c_void_p * 1)(A16)
    def call(**kw):
        a = dict(layers=1, hio=A16, io=A16, iob=1 << 30, k=caches, v=caches, M=1, H=4, Hkv=2,
                 D=64, Lmax=256, C=64, ws=A16, wsb=1 << 30, st=A16, out=ctypes.byref(h))
        a.update(kw)
        return L.kvs_step_graph_create_host_io(a["layers"], a["hio"], a["io"], a["iob"], a["k"],
                                               a["v"], a["M"], a["H"], a["Hkv"], a["D"],
                                               a["Lmax"], a["C"], a["ws"], a["wsb"], None,
                                               a["st"], a["out"])
    assert call(out=None) == B.KVS_ERR_NULL
    assert call(layers=0) == B.KVS_ERR_DIMS
    assert call(M=0) == B.KVS_ERR_DIMS
    assert call(hio=None) == B.KVS_ERR_NULL
    assert call(io=None) == B.KVS_ERR_NULL
    assert call(k=None) == B.KVS_ERR_NULL
    assert call(st=None) == B.KVS_ERR_DIMS
    assert call(io=A16 + 16) == B.KVS_ERR_ALIGN
    assert call(iob=1024) == B.KVS_ERR_WORKSPACE


def _dshio(L, hio=A16, k=A16, v=A16, M=1, H=4, Hkv=2, D=64, Lmax=256, C=64, io=A16,
           iob=1 << 30, ws=A16, wsb=1 << 30):
    return L.kvs_decode_step_host_io(hio, k, v, M, H, Hkv, D, Lmax, C, io, iob, ws, wsb, None,
                                     None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), B.KVS_ERR_DIMS),
    (dict(H=6, Hkv=4), B.KVS_ERR_DIMS),
    (dict(C=-1), B.KVS_ERR_DIMS),
    (dict(D=96), B.KVS_ERR_UNSUPPORTED),
    (dict(hio=None), B.KVS_ERR_NULL),
    (dict(io=None), B.KVS_ERR_NULL),
    (dict(k=None), B.KVS_ERR_NULL),
    (dict(io=A16 + 16), B.KVS_ERR_ALIGN),
    (dict(v=A16 + 8), B.KVS_ERR_ALIGN),
    (dict(iob=64), B.KVS_ERR_WORKSPACE),
    (dict(ws=None), B.KVS_ERR_WORKSPACE),
    (dict(wsb=64), B.KVS_ERR_WORKSPACE),
    # the host buffer needs no alignment: it is only copied from and to
    (dict(hio=A16 + 4, iob=64), B.KVS_ERR_WORKSPACE),
])
def test_decode_step_host_io_validation(L, kw, code):
    assert _dshio(L, **kw) == code


def test_decode_step_host_io_empty_batch_ok(L):
    assert _dshio(L, M=0, hio=None, k=None, v=None, io=None, iob=0, ws=None, wsb=0) == 0
