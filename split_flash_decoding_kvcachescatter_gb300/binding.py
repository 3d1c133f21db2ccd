"""Thin Python binding of libkvsdecode.so: argument marshalling only.

Every function here has the name of the C entry point it calls
(include/kvsdecode.h).  It checks tensor dtype/device/contiguity, reads the
sizes off the tensor shapes, passes raw device pointers and the current
CUDA stream, and raises KvsError on a non-zero status.  All compute runs
in the CUDA kernels of the library; there is no fallback of any kind: if
the library is missing or fails to load, the functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvsdecode.so")

KVS_OK = 0
KVS_ERR_NULL = 1
KVS_ERR_DIMS = 2
KVS_ERR_UNSUPPORTED = 3
KVS_ERR_ALIGN = 4
KVS_ERR_WORKSPACE = 5
KVS_ERR_LAUNCH = 6
KVS_ERR_POSITION = 7
KVS_ERR_TIMEOUT = 8
KVS_ERR_SLOT = 9
KVS_ERR_MEMORY = 10

# Every symbol include/kvsdecode.h declares.
EXPORTS = ("kvs_kv_scatter", "kvs_choose_chunk_size", "kvs_flash_decode_workspace_bytes",
           "kvs_flash_decode", "kvs_decode_step", "kvs_strerror", "kvs_flash_decode_static",
           "kvs_step_graph_create", "kvs_step_graph_launch", "kvs_step_graph_destroy",
           "kvs_set_schedule", "kvs_get_schedule", "kvs_schedule_for", "kvs_prepare",
           "kvs_decode_step_slots", "kvs_argmax", "kvs_prefill_attention",
           "kvs_prefill_workspace_bytes", "kvs_step_io_bytes", "kvs_decode_step_host",
           "kvs_set_wait_limit_ns", "kvs_step_io_layout", "kvs_decode_step_host_io",
           "kvs_step_graph_io_layout", "kvs_step_graph_create_host_io")

# Default bound on each pipeline wait of the kernels (kvs_set_wait_limit_ns).
KVS_WAIT_LIMIT_DEFAULT_NS = 2_000_000_000

# kvs_schedule values (kernel schedule of the attention entry points)
KVS_SCHEDULE_AUTO = 0
KVS_SCHEDULE_PERSISTENT = 1
KVS_SCHEDULE_CLUSTER = 2

# Size of the library's built-in scratch buffer used by kvs_flash_decode_static.
KVS_STATIC_WORKSPACE_BYTES = 32 * 1024 * 1024

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


class KvsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {strerror(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m split_flash_decoding_kvcachescatter_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            L.kvs_kv_scatter.restype = _I
            L.kvs_kv_scatter.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]
            L.kvs_choose_chunk_size.restype = _I
            L.kvs_choose_chunk_size.argtypes = [_I, _I, _I, _I, _I]
            L.kvs_flash_decode_workspace_bytes.restype = _SZ
            L.kvs_flash_decode_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
            L.kvs_flash_decode.restype = _I
            L.kvs_flash_decode.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                           _P, _SZ, _P, _P]
            L.kvs_decode_step.restype = _I
            L.kvs_decode_step.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                          _P, _SZ, _P, _P]
            L.kvs_step_io_bytes.restype = _SZ
            L.kvs_step_io_bytes.argtypes = [_I, _I, _I, _I]
            L.kvs_decode_step_host.restype = _I
            L.kvs_decode_step_host.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                               _I, _P, _SZ, _P, _SZ, _P, _P]
            L.kvs_flash_decode_static.restype = _I
            L.kvs_flash_decode_static.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                  _P, _P]
            L.kvs_step_graph_create.restype = _I
            L.kvs_step_graph_create.argtypes = [_I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                                _I, _I, _P, _SZ, _P, _P, _P]
            L.kvs_step_graph_launch.restype = _I
            L.kvs_step_graph_launch.argtypes = [_P, _P]
            L.kvs_step_graph_io_layout.restype = _I
            L.kvs_step_graph_io_layout.argtypes = [_I, _I, _I, _I, _I, _P]
            L.kvs_step_graph_create_host_io.restype = _I
            L.kvs_step_graph_create_host_io.argtypes = [_I, _P, _P, _SZ, _P, _P, _I, _I, _I, _I,
                                                        _I, _I, _P, _SZ, _P, _P, _P]
            L.kvs_step_graph_destroy.restype = _I
            L.kvs_step_graph_destroy.argtypes = [_P]
            L.kvs_decode_step_slots.restype = _I
            L.kvs_decode_step_slots.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I,
                                                _I, _I, _I, _I, _P, _SZ, _P, _P]
            L.kvs_prefill_attention.restype = _I
            L.kvs_prefill_attention.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _P, _SZ, _P,
                                                _P]
            L.kvs_prefill_workspace_bytes.restype = _SZ
            L.kvs_prefill_workspace_bytes.argtypes = [_I, _I, _I]
            L.kvs_argmax.restype = _I
            L.kvs_argmax.argtypes = [_P, _I, _I, _P, _P]
            L.kvs_set_schedule.restype = _I
            L.kvs_set_schedule.argtypes = [_I]
            L.kvs_get_schedule.restype = _I
            L.kvs_get_schedule.argtypes = []
            L.kvs_schedule_for.restype = _I
            L.kvs_schedule_for.argtypes = [_I, _I, _I, _I, _I]
            L.kvs_prepare.restype = _I
            L.kvs_prepare.argtypes = [_I, _I, _I]
            L.kvs_step_io_layout.restype = _I
            L.kvs_step_io_layout.argtypes = [_I, _I, _I, _I, ctypes.POINTER(_SZ)]
            L.kvs_decode_step_host_io.restype = _I
            L.kvs_decode_step_host_io.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ,
                                                  _P, _SZ, _P, _P]
            L.kvs_set_wait_limit_ns.restype = _I
            L.kvs_set_wait_limit_ns.argtypes = [ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64)]
            L.kvs_strerror.restype = ctypes.c_char_p
            L.kvs_strerror.argtypes = [_I]
            _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().kvs_strerror(int(status)).decode()


def _check(rc: int, where: str) -> None:
    if rc != KVS_OK:
        raise KvsError(rc, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _f32(t: torch.Tensor, name: str, ndim: int) -> int:
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and t.dim() == ndim):
        raise TypeError(f"{name}: need a contiguous float32 CUDA tensor with {ndim} dims, got "
                        f"{tuple(t.shape)} {t.dtype} {t.device}")
    return t.data_ptr()


def _i32(t: torch.Tensor, name: str) -> int:
    if not (t.is_cuda and t.dtype == torch.int32 and t.is_contiguous() and t.dim() == 1):
        raise TypeError(f"{name}: need a contiguous int32 CUDA vector")
    return t.data_ptr()


def _status_ptr(d_status) -> int:
    if d_status is None:
        return 0
    if not (d_status.is_cuda and d_status.dtype == torch.int32):
        raise TypeError("d_status: need an int32 CUDA tensor")
    return d_status.data_ptr()


def kvs_kv_scatter(k_rows, v_rows, positions, k_cache, v_cache, d_status=None, stream=None):
    """Scatter k_rows/v_rows [M,Hkv,D] into caches [M,Hkv,Lmax,D] at positions [M]."""
    M, Hkv, Lmax, D = k_cache.shape
    if tuple(v_cache.shape) != (M, Hkv, Lmax, D) or tuple(k_rows.shape) != (M, Hkv, D) or \
            tuple(v_rows.shape) != (M, Hkv, D) or positions.numel() != M:
        raise ValueError("kvs_kv_scatter: inconsistent shapes")
    rc = lib().kvs_kv_scatter(_f32(k_rows, "k_rows", 3), _f32(v_rows, "v_rows", 3),
                              _i32(positions, "positions"), _f32(k_cache, "k_cache", 4),
                              _f32(v_cache, "v_cache", 4), M, Hkv, D, Lmax,
                              _status_ptr(d_status), _stream(stream))
    _check(rc, "kvs_kv_scatter")


def prefill_workspace(H, S, D, device=None):
    """A device byte buffer large enough for kvs_prefill_attention (allocated by torch)."""
    n = int(lib().kvs_prefill_workspace_bytes(H, S, D))
    if n == 0:
        raise KvsError(KVS_ERR_DIMS, "kvs_prefill_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def kvs_prefill_attention(q, k, v, out, causal=True, workspace=None, d_status=None, stream=None):
    """Tensor-core attention over whole sequences: q, k, v, out [H, S, D] float32 (CUDA)."""
    H, S, D = q.shape
    for name, t in (("k", k), ("v", v), ("out", out)):
        if tuple(t.shape) != (H, S, D):
            raise ValueError(f"kvs_prefill_attention: {name} must be [H, S, D] like q")
    if workspace is None:
        raise ValueError("kvs_prefill_attention: pass a workspace (see binding.prefill_workspace)")
    _check(lib().kvs_prefill_attention(_f32(q, "q", 3), _f32(k, "k", 3), _f32(v, "v", 3),
                                       _f32(out, "out", 3), H, S, D, 1 if causal else 0,
                                       workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(),
                                       _status_ptr(d_status), _stream(stream)),
           "kvs_prefill_attention")
    return out


def kvs_argmax(logits, token_ids=None, stream=None):
    """Greedy token of each row of logits [M, V] (float32, CUDA): int32 [M] on the device."""
    if not (logits.is_cuda and logits.dtype == torch.float32 and logits.dim() == 2 and
            logits.stride(1) == 1 and logits.stride(0) == logits.shape[1]):
        raise TypeError("logits: need a contiguous float32 CUDA matrix [M, V]")
    M, V = logits.shape
    if token_ids is None:
        token_ids = torch.empty(M, dtype=torch.int32, device=logits.device)
    _check(lib().kvs_argmax(logits.data_ptr(), M, V, _i32(token_ids, "token_ids"),
                            _stream(stream)), "kvs_argmax")
    return token_ids


def kvs_set_schedule(schedule: int) -> int:
    """Set the process-wide kernel schedule (KVS_SCHEDULE_*); returns the previous one."""
    prev = lib().kvs_set_schedule(int(schedule))
    if prev < 0:
        raise KvsError(-prev, "kvs_set_schedule")
    return prev


def kvs_get_schedule() -> int:
    return int(lib().kvs_get_schedule())


def kvs_schedule_for(M, num_heads, num_kv_heads, head_dim, max_len) -> int:
    """KVS_SCHEDULE_PERSISTENT or KVS_SCHEDULE_CLUSTER: the kernel such a call would run."""
    r = lib().kvs_schedule_for(M, num_heads, num_kv_heads, head_dim, max_len)
    if r < 0:
        raise KvsError(-r, "kvs_schedule_for")
    return r


def kvs_set_wait_limit_ns(ns: int) -> int:
    """Set the bound on each pipeline wait of the kernels on the current
    device (0 .. KVS_WAIT_LIMIT_DEFAULT_NS); returns the previous bound."""
    prev = ctypes.c_uint64(0)
    _check(lib().kvs_set_wait_limit_ns(int(ns), ctypes.byref(prev)), "kvs_set_wait_limit_ns")
    return int(prev.value)


def kvs_prepare(num_heads, num_kv_heads, head_dim) -> None:
    """Set up both attention kernels for this shape on the current device."""
    _check(lib().kvs_prepare(num_heads, num_kv_heads, head_dim), "kvs_prepare")


def kvs_choose_chunk_size(M, num_kv_heads, head_dim, max_len, num_sms=0) -> int:
    c = lib().kvs_choose_chunk_size(M, num_kv_heads, head_dim, max_len, num_sms)
    if c <= 0:
        raise KvsError(-c, "kvs_choose_chunk_size")
    return c


def kvs_flash_decode_workspace_bytes(M, num_heads, num_kv_heads, head_dim, max_len,
                                     chunk_size) -> int:
    return int(lib().kvs_flash_decode_workspace_bytes(M, num_heads, num_kv_heads, head_dim,
                                                      max_len, chunk_size))


def workspace(M, num_heads, num_kv_heads, head_dim, max_len, chunk_size, device=None):
    """A device byte buffer large enough for kvs_flash_decode (allocated by torch)."""
    n = kvs_flash_decode_workspace_bytes(M, num_heads, num_kv_heads, head_dim, max_len,
                                         chunk_size)
    if n == 0 and M > 0:
        raise KvsError(KVS_ERR_DIMS, "kvs_flash_decode_workspace_bytes")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def _attn_shapes(q, k_cache):
    M, H, D = q.shape
    M2, Hkv, Lmax, D2 = k_cache.shape
    if M2 != M or D2 != D:
        raise ValueError("q and k_cache disagree on M or head_dim")
    return M, H, Hkv, D, Lmax


def kvs_flash_decode(q, k_cache, v_cache, positions, out, chunk_size=0, workspace=None,
                     d_status=None, stream=None):
    """out[M,H,D] = split-K softmax attention of q over cache rows 0..positions[i]."""
    M, H, Hkv, D, Lmax = _attn_shapes(q, k_cache)
    if workspace is None:
        raise ValueError("kvs_flash_decode: pass a workspace (see binding.workspace)")
    rc = lib().kvs_flash_decode(_f32(q, "q", 3), _f32(k_cache, "k_cache", 4),
                                _f32(v_cache, "v_cache", 4), _i32(positions, "positions"),
                                _f32(out, "out", 3), M, H, Hkv, D, Lmax, int(chunk_size),
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _status_ptr(d_status), _stream(stream))
    _check(rc, "kvs_flash_decode")


def kvs_decode_step(q, k_rows, v_rows, positions, k_cache, v_cache, out, chunk_size=0,
                    workspace=None, d_status=None, stream=None):
    """kvs_kv_scatter + kvs_flash_decode of one layer's decode step, in one launch."""
    M, H, Hkv, D, Lmax = _attn_shapes(q, k_cache)
    if workspace is None:
        raise ValueError("kvs_decode_step: pass a workspace (see binding.workspace)")
    if tuple(k_rows.shape) != (M, Hkv, D) or tuple(v_rows.shape) != (M, Hkv, D) or \
            tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("kvs_decode_step: inconsistent shapes")
    rc = lib().kvs_decode_step(_f32(q, "q", 3), _f32(k_rows, "k_rows", 3),
                               _f32(v_rows, "v_rows", 3), _i32(positions, "positions"),
                               _f32(k_cache, "k_cache", 4), _f32(v_cache, "v_cache", 4),
                               _f32(out, "out", 3), M, H, Hkv, D, Lmax, int(chunk_size),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               _status_ptr(d_status), _stream(stream))
    _check(rc, "kvs_decode_step")


def step_io(M, num_heads, num_kv_heads, head_dim, device=None):
    """A device byte buffer large enough for kvs_decode_step_host's copies."""
    n = int(lib().kvs_step_io_bytes(M, num_heads, num_kv_heads, head_dim))
    if n == 0:
        raise KvsError(KVS_ERR_DIMS, "kvs_step_io_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _host(t: torch.Tensor, name: str, dtype, shape) -> int:
    if t.is_cuda or t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise TypeError(f"{name}: need a contiguous {dtype} CPU tensor of shape {tuple(shape)}, "
                        f"got {tuple(t.shape)} {t.dtype} {t.device}")
    return t.data_ptr()


def kvs_decode_step_host(q, k_rows, v_rows, positions, k_cache, v_cache, out, chunk_size=0,
                         workspace=None, io=None, d_status=None, stream=None):
    """kvs_decode_step with q, k_rows, v_rows, positions and out in host memory
    (CPU tensors, pinned for asynchronous copies): the copies in, the fused
    step and the copy of out back, enqueued by one library call.  out is valid
    after the stream is synchronised."""
    M, Hkv, Lmax, D = k_cache.shape
    H = q.shape[1] if q.dim() == 3 else -1
    if workspace is None or io is None:
        raise ValueError("kvs_decode_step_host: pass a workspace and an io buffer "
                         "(see binding.workspace, binding.step_io)")
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("kvs_decode_step_host: inconsistent cache shapes")
    rc = lib().kvs_decode_step_host(
        _host(q, "q", torch.float32, (M, H, D)), _host(k_rows, "k_rows", torch.float32, (M, Hkv, D)),
        _host(v_rows, "v_rows", torch.float32, (M, Hkv, D)),
        _host(positions, "positions", torch.int32, (M,)),
        _f32(k_cache, "k_cache", 4), _f32(v_cache, "v_cache", 4),
        _host(out, "out", torch.float32, (M, H, D)), M, H, Hkv, D, Lmax, int(chunk_size),
        io.data_ptr(), io.numel() * io.element_size(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _status_ptr(d_status), _stream(stream))
    _check(rc, "kvs_decode_step_host")


def kvs_step_io_layout(M, num_heads, num_kv_heads, head_dim):
    """Byte offsets of q, k_rows, v_rows, positions, out and the total size
    of an io buffer (device, or the host buffer of kvs_decode_step_host_io)."""
    off = (_SZ * 6)()
    _check(lib().kvs_step_io_layout(M, num_heads, num_kv_heads, head_dim, off),
           "kvs_step_io_layout")
    return tuple(int(x) for x in off)


class HostIo:
    """A host buffer with the io layout, and views of its arrays: fill q,
    k_rows, v_rows and positions, call kvs_decode_step_host_io, and read out
    once the stream has passed the call.  Pinned by default (the library then
    moves it with its copy kernel); pinned=False gives pageable memory (moved
    by copy engines, the host waiting for them)."""

    def __init__(self, M, num_heads, num_kv_heads, head_dim, pinned=True):
        oq, ok, ov, op, oo, total = kvs_step_io_layout(M, num_heads, num_kv_heads, head_dim)
        self.shape = (M, num_heads, num_kv_heads, head_dim)
        self.buf = torch.empty(total, dtype=torch.uint8, pin_memory=pinned)
        f = lambda off, n, dt: self.buf[off:off + n * 4].view(dt)
        self.q = f(oq, M * num_heads * head_dim, torch.float32).view(M, num_heads, head_dim)
        self.k_rows = f(ok, M * num_kv_heads * head_dim, torch.float32).view(
            M, num_kv_heads, head_dim)
        self.v_rows = f(ov, M * num_kv_heads * head_dim, torch.float32).view(
            M, num_kv_heads, head_dim)
        self.positions = f(op, M, torch.int32)
        self.out = f(oo, M * num_heads * head_dim, torch.float32).view(M, num_heads, head_dim)
        self.in_bytes = op + 4 * M          # what one step copies to the device
        self.out_bytes = M * num_heads * head_dim * 4  # and back


def kvs_decode_step_host_io(host_io, k_cache, v_cache, chunk_size=0, workspace=None, io=None,
                            d_status=None, stream=None):
    """kvs_decode_step with the step's inputs and result in one pinned host
    buffer (a HostIo): one copy in, the fused step, one copy out."""
    M, Hkv, Lmax, D = k_cache.shape
    if not isinstance(host_io, HostIo):
        raise TypeError("host_io: need a binding.HostIo")
    Mh, H, Hkvh, Dh = host_io.shape
    if (Mh, Hkvh, Dh) != (M, Hkv, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("kvs_decode_step_host_io: inconsistent shapes")
    if workspace is None or io is None:
        raise ValueError("kvs_decode_step_host_io: pass a workspace and an io buffer")
    rc = lib().kvs_decode_step_host_io(
        host_io.buf.data_ptr(), _f32(k_cache, "k_cache", 4), _f32(v_cache, "v_cache", 4), M, H,
        Hkv, D, Lmax, int(chunk_size), io.data_ptr(), io.numel() * io.element_size(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _status_ptr(d_status), _stream(stream))
    _check(rc, "kvs_decode_step_host_io")


def kvs_step_graph_io_layout(layers, M, num_heads, num_kv_heads, head_dim):
    """Offsets of kvs_step_graph_io_layout: a list of 4 * layers + 2 ints."""
    off = (ctypes.c_size_t * (4 * layers + 2))()
    _check(lib().kvs_step_graph_io_layout(layers, M, num_heads, num_kv_heads, head_dim, off),
           "kvs_step_graph_io_layout")
    return list(off)


class HostStepIo:
    """A pinned host buffer with the layout of kvs_step_graph_io_layout and
    views of its arrays: q[l], k_rows[l], v_rows[l], out[l] per layer and the
    shared positions.  Fill the inputs, launch the host-io step graph, read
    the outs once the stream has passed the launch."""

    def __init__(self, layers, M, num_heads, num_kv_heads, head_dim):
        off = kvs_step_graph_io_layout(layers, M, num_heads, num_kv_heads, head_dim)
        self.layers, self.shape = layers, (M, num_heads, num_kv_heads, head_dim)
        self.total = off[4 * layers + 1]
        self.buf = torch.empty(self.total, dtype=torch.uint8, pin_memory=True)
        f = lambda o, n, dt: self.buf[o:o + n * 4].view(dt)
        qn, kn = M * num_heads * head_dim, M * num_kv_heads * head_dim
        self.q = [f(off[3 * l], qn, torch.float32).view(M, num_heads, head_dim)
                  for l in range(layers)]
        self.k_rows = [f(off[3 * l + 1], kn, torch.float32).view(M, num_kv_heads, head_dim)
                       for l in range(layers)]
        self.v_rows = [f(off[3 * l + 2], kn, torch.float32).view(M, num_kv_heads, head_dim)
                       for l in range(layers)]
        self.positions = f(off[3 * layers], M, torch.int32)
        self.out = [f(off[3 * layers + 1 + l], qn, torch.float32).view(M, num_heads, head_dim)
                    for l in range(layers)]
        self.in_bytes = off[3 * layers + 1]          # one copy to the device a step
        self.out_bytes = self.total - self.in_bytes  # and one back


def kvs_step_graph_create_host_io(host_io, k_cache, v_cache, chunk_size=0, workspace=None,
                                  io=None, d_status=None, stream=None):
    """A step graph over one pinned host buffer (a HostStepIo): one copy of
    every layer's inputs in, the layers, one copy of every layer's out back."""
    if not isinstance(host_io, HostStepIo):
        raise TypeError("host_io: need a binding.HostStepIo")
    layers = host_io.layers
    if not (len(k_cache) == len(v_cache) == layers):
        raise ValueError("kvs_step_graph_create_host_io: one cache per layer")
    if workspace is None or io is None:
        raise ValueError("kvs_step_graph_create_host_io: pass a workspace and an io buffer")
    M, Hkv, Lmax, D = k_cache[0].shape
    Mh, H, Hkvh, Dh = host_io.shape
    if (Mh, Hkvh, Dh) != (M, Hkv, D):
        raise ValueError("kvs_step_graph_create_host_io: inconsistent shapes")
    arr = lambda ts, name: (ctypes.c_void_p * layers)(*[_f32(t, name, 4) for t in ts])
    s = torch.cuda.Stream() if stream is None else stream
    handle = ctypes.c_void_p()
    rc = lib().kvs_step_graph_create_host_io(
        layers, host_io.buf.data_ptr(), io.data_ptr(), io.numel() * io.element_size(),
        arr(k_cache, "k_cache"), arr(v_cache, "v_cache"), M, H, Hkv, D, Lmax, int(chunk_size),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _status_ptr(d_status), _stream(s), ctypes.byref(handle))
    _check(rc, "kvs_step_graph_create_host_io")
    return StepGraph(handle, (host_io, io, k_cache, v_cache, workspace))


def kvs_decode_step_slots(q, k_rows, v_rows, positions, slots, done, k_pool, v_pool, out,
                          chunk_size=0, workspace=None, d_status=None, stream=None):
    """Decode step over a cache pool [S, Hkv, Lmax, D]: sequence i uses slot
    slots[i] (int32 [M], or None for slot i); done (uint8 [M] or None) marks
    finished sequences, which are scattered but not attended (their out rows
    are left as they are).  k_rows and v_rows both None: attention only."""
    M, H, D = q.shape
    S, Hkv, Lmax, D2 = k_pool.shape
    if D2 != D or tuple(v_pool.shape) != tuple(k_pool.shape) or tuple(out.shape) != (M, H, D):
        raise ValueError("kvs_decode_step_slots: inconsistent shapes")
    if workspace is None:
        raise ValueError("kvs_decode_step_slots: pass a workspace (see binding.workspace)")
    if (k_rows is None) != (v_rows is None):
        raise ValueError("kvs_decode_step_slots: pass both k_rows and v_rows, or neither")
    kr = 0 if k_rows is None else _f32(k_rows, "k_rows", 3)
    vr = 0 if v_rows is None else _f32(v_rows, "v_rows", 3)
    if k_rows is not None and (tuple(k_rows.shape) != (M, Hkv, D) or
                               tuple(v_rows.shape) != (M, Hkv, D)):
        raise ValueError("kvs_decode_step_slots: k_rows / v_rows must be [M, Hkv, D]")
    sl = 0 if slots is None else _i32(slots, "slots")
    if slots is not None and slots.numel() != M:
        raise ValueError("kvs_decode_step_slots: slots must have M entries")
    dn = 0
    if done is not None:
        if not (done.is_cuda and done.dtype == torch.uint8 and done.is_contiguous() and
                done.numel() == M):
            raise TypeError("done: need a contiguous uint8 CUDA vector of M entries")
        dn = done.data_ptr()
    rc = lib().kvs_decode_step_slots(_f32(q, "q", 3), kr, vr, _i32(positions, "positions"), sl,
                                     dn, _f32(k_pool, "k_pool", 4), _f32(v_pool, "v_pool", 4), S,
                                     _f32(out, "out", 3), M, H, Hkv, D, Lmax, int(chunk_size),
                                     workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(),
                                     _status_ptr(d_status), _stream(stream))
    _check(rc, "kvs_decode_step_slots")


def kvs_flash_decode_static(q, k_cache, v_cache, positions, out, chunk_size=0, d_status=None,
                            stream=None):
    """kvs_flash_decode without a workspace argument: the partials go to the
    library's built-in buffer (for callers that cannot allocate device memory;
    calls that may overlap on the GPU must be ordered, see the C header)."""
    M, H, Hkv, D, Lmax = _attn_shapes(q, k_cache)
    rc = lib().kvs_flash_decode_static(_f32(q, "q", 3), _f32(k_cache, "k_cache", 4),
                                       _f32(v_cache, "v_cache", 4),
                                       _i32(positions, "positions"), _f32(out, "out", 3), M, H,
                                       Hkv, D, Lmax, int(chunk_size), _status_ptr(d_status),
                                       _stream(stream))
    _check(rc, "kvs_flash_decode_static")


class StepGraph:
    """Handle of kvs_step_graph_create: a whole multi-layer decode step as one
    CUDA graph over fixed buffers (update their contents, not their
    addresses, between launches)."""

    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep  # the captured tensors must outlive the graph

    def launch(self, stream=None):
        _check(lib().kvs_step_graph_launch(self._h, _stream(stream)), "kvs_step_graph_launch")

    def destroy(self):
        if self._h:
            lib().kvs_step_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def kvs_step_graph_create(q, k_rows, v_rows, positions, k_cache, v_cache, out, chunk_size=0,
                          workspace=None, d_status=None, stream=None):
    """Capture one kvs_decode_step per layer (lists of per-layer tensors)."""
    layers = len(q)
    if not (len(k_rows) == len(v_rows) == len(k_cache) == len(v_cache) == len(out) == layers):
        raise ValueError("kvs_step_graph_create: one tensor per layer in every list")
    if workspace is None:
        raise ValueError("kvs_step_graph_create: pass a workspace")
    M, H, Hkv, D, Lmax = _attn_shapes(q[0], k_cache[0])
    arr = lambda ts, name, nd: (ctypes.c_void_p * layers)(*[_f32(t, name, nd) for t in ts])
    s = torch.cuda.Stream() if stream is None else stream
    handle = ctypes.c_void_p()
    rc = lib().kvs_step_graph_create(
        layers, arr(q, "q", 3), arr(k_rows, "k_rows", 3), arr(v_rows, "v_rows", 3),
        _i32(positions, "positions"), arr(k_cache, "k_cache", 4), arr(v_cache, "v_cache", 4),
        arr(out, "out", 3), M, H, Hkv, D, Lmax, int(chunk_size), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _status_ptr(d_status), _stream(s),
        ctypes.byref(handle))
    _check(rc, "kvs_step_graph_create")
    return StepGraph(handle, (q, k_rows, v_rows, positions, k_cache, v_cache, out, workspace))
