"""CPU oracle for the decode-step attention path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports it and never falls back to it.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, one thread; see
its header for the passages it follows).  This module only builds that file
with gcc and marshals numpy arrays into it.

Pages followed: realizar 0.8.5, src/cuda/executor/head_dim.rs,
``flash_decoding_attention_into`` (PAR-118): doc comment (layouts, split-K
with rescaled merge), Step 1 (scatter before attention), "Update cache
lengths" (seq_len = position + 1), Step 3 (chunk count = ceil(len / chunk)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_F32P = ctypes.POINTER(ctypes.c_float)
_F64P = ctypes.POINTER(ctypes.c_double)
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no FMA contraction)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_kv_scatter.restype = _I64
            lib.oracle_kv_scatter.argtypes = [_F32P, _F32P, _I32P, _F32P, _F32P,
                                              _I64, _I64, _I64, _I64]
            lib.oracle_attend_row_f64.restype = ctypes.c_int
            lib.oracle_attend_row_f64.argtypes = [_F32P, _F32P, _F32P, _I64, _I64,
                                                  ctypes.c_double, _F64P]
            lib.oracle_attend_row.restype = ctypes.c_int
            lib.oracle_attend_row.argtypes = [_F32P, _F32P, _F32P, _I64, _I64,
                                              ctypes.c_double, _F32P]
            lib.oracle_attend_row_split_f64.restype = ctypes.c_int
            lib.oracle_attend_row_split_f64.argtypes = [_F32P, _F32P, _F32P, _I64,
                                                        _I64, ctypes.c_double, _I64,
                                                        _F64P]
            lib.oracle_attend_seq.restype = ctypes.c_int
            lib.oracle_attend_seq.argtypes = [_F32P, _F32P, _F32P, _I64, _I64, _I64,
                                              _I64, _I64, ctypes.c_double, _F32P]
            lib.oracle_decode.restype = _I64
            lib.oracle_decode.argtypes = [_F32P, _F32P, _F32P, _I32P, _F32P, _I64,
                                          _I64, _I64, _I64, _I64]
            _lib = lib
    return _lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(_F32P)


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(_I32P)


def kv_scatter(k_rows, v_rows, positions, k_cache, v_cache):
    """In-place scatter into numpy caches [M][Hkv][Lmax][D] (float32, C order).

    Returns the number of sequences skipped for an out-of-range position.
    """
    lib = _load()
    M, Hkv, Lmax, D = k_cache.shape
    assert v_cache.shape == k_cache.shape
    for c in (k_cache, v_cache):
        assert c.dtype == np.float32 and c.flags.c_contiguous
    kr, krp = _f32(k_rows)
    vr, vrp = _f32(v_rows)
    ps, psp = _i32(positions)
    assert kr.shape == (M, Hkv, D) and vr.shape == (M, Hkv, D) and ps.shape == (M,)
    return int(lib.oracle_kv_scatter(krp, vrp, psp, k_cache.ctypes.data_as(_F32P),
                                     v_cache.ctypes.data_as(_F32P), M, Hkv, D, Lmax))


def attend_row(q, K, V, scale=None, f64=False):
    """Softmax attention of one query row q[D] over K[L][D], V[L][D]."""
    lib = _load()
    qa, qp = _f32(q)
    Ka, Kp = _f32(K)
    Va, Vp = _f32(V)
    L, D = Ka.shape
    assert Va.shape == (L, D) and qa.shape == (D,)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    if f64:
        out = np.empty(D, np.float64)
        rc = lib.oracle_attend_row_f64(qp, Kp, Vp, L, D, scale, out.ctypes.data_as(_F64P))
    else:
        out = np.empty(D, np.float32)
        rc = lib.oracle_attend_row(qp, Kp, Vp, L, D, scale, out.ctypes.data_as(_F32P))
    if rc != 0:
        raise RuntimeError(f"oracle_attend_row failed: {rc}")
    return out


def attend_row_split(q, K, V, chunk, scale=None):
    """The split-K form with chunk size `chunk`, in double (merge-algebra pin)."""
    lib = _load()
    qa, qp = _f32(q)
    Ka, Kp = _f32(K)
    Va, Vp = _f32(V)
    L, D = Ka.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.empty(D, np.float64)
    rc = lib.oracle_attend_row_split_f64(qp, Kp, Vp, L, D, scale, int(chunk),
                                         out.ctypes.data_as(_F64P))
    if rc != 0:
        raise RuntimeError(f"oracle_attend_row_split_f64 failed: {rc}")
    return out


def attend_seq(q, K, V, L, scale=None):
    """All heads of one sequence: q [H][D], K/V [Hkv][rows>=L][D] -> out [H][D]."""
    lib = _load()
    qa, qp = _f32(q)
    Ka, Kp = _f32(K)
    Va, Vp = _f32(V)
    H, D = qa.shape
    Hkv, rows, D2 = Ka.shape
    assert D2 == D and Va.shape == Ka.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.empty((H, D), np.float32)
    rc = lib.oracle_attend_seq(qp, Kp, Vp, int(L), rows, H, Hkv, D, scale,
                               out.ctypes.data_as(_F32P))
    if rc != 0:
        raise RuntimeError(f"oracle_attend_seq failed: {rc}")
    return out


def decode(q, k_cache, v_cache, positions):
    """Attention over the scattered cache layout [M][Hkv][Lmax][D] -> out [M][H][D]."""
    lib = _load()
    qa, qp = _f32(q)
    M, H, D = qa.shape
    Kc, Kcp = _f32(k_cache)
    Vc, Vcp = _f32(v_cache)
    M2, Hkv, Lmax, D2 = Kc.shape
    assert M2 == M and D2 == D and Vc.shape == Kc.shape
    ps, psp = _i32(positions)
    out = np.empty((M, H, D), np.float32)
    rc = lib.oracle_decode(qp, Kcp, Vcp, psp, out.ctypes.data_as(_F32P), M, H, Hkv, D, Lmax)
    if rc < 0:
        raise RuntimeError(f"oracle_decode failed: {-rc}")
    return out


def decode_sequences(q, k_seq, v_seq, positions, threads=None):
    """Attention per sequence from per-sequence live rows.

    q: [M][H][D]; k_seq[i], v_seq[i]: [Hkv][>= p_i + 1][D] holding rows
    0..p_i of sequence i's cache after the scatter.  Sequences run on a
    thread pool (the C call releases the GIL); each call is the
    single-threaded oracle.  Returns out [M][H][D] float32.
    """
    M, H, D = q.shape
    out = np.empty((M, H, D), np.float32)

    def one(i):
        out[i] = attend_seq(q[i], k_seq[i], v_seq[i], int(positions[i]) + 1)

    n = threads or os.cpu_count() or 1
    if n <= 1 or M == 1:
        for i in range(M):
            one(i)
    else:
        with ThreadPoolExecutor(max_workers=n) as ex:
            list(ex.map(one, range(M)))
    return out


def decode_step_slots(q, k_rows, v_rows, positions, slots, done, k_pool, v_pool, out):
    """One decode step over a pool of cache slots with finished sequences.

    Follows realizar 0.8.5, src/cuda/executor/head_dim.rs,
    ``flash_decoding_attention_into``: "Step 2: Build pointer arrays" (each
    sequence's K/V cache is found through a per-sequence pointer; here an
    index into the pool k_pool/v_pool [num_slots][Hkv][Lmax][D]) and the
    PMAT-076 note in the same step (a finished sequence gets seq_len 0, so
    the attention kernels skip it).  Step 1 scatters every sequence before
    any attention runs, finished or not.

    In place: k_pool, v_pool (scatter) and out [M][H][D] (attention).
      slots[i]  pool slot of sequence i (None: slot i)
      done[i]   nonzero: finished -- the scatter still happens, the
                attention does not, and out[i] keeps its contents (None: none)
    A sequence whose position is outside [0, Lmax) or whose slot is outside
    [0, num_slots) is not scattered; unless finished its out rows become NaN.
    Returns the indices of such sequences.
    """
    M, H, D = q.shape
    S, Hkv, Lmax, D2 = k_pool.shape
    assert D2 == D and v_pool.shape == k_pool.shape and out.shape == (M, H, D)
    slots = np.arange(M, dtype=np.int64) if slots is None else np.asarray(slots, np.int64)
    done = np.zeros(M, bool) if done is None else (np.asarray(done) != 0)
    positions = np.asarray(positions, np.int64)
    bad = [i for i in range(M)
           if not (0 <= positions[i] < Lmax) or not (0 <= slots[i] < S)]
    # Step 1: the new rows of every sequence, at its position in its slot
    for i in range(M):
        if i in bad:
            continue
        k_pool[slots[i], :, positions[i], :] = k_rows[i]
        v_pool[slots[i], :, positions[i], :] = v_rows[i]
    # Steps 3-5: attention of every sequence that is not finished
    for i in range(M):
        if done[i]:
            continue
        if i in bad:
            out[i] = np.nan
            continue
        out[i] = attend_seq(q[i], k_pool[slots[i]], v_pool[slots[i]], int(positions[i]) + 1)
    return bad


def argmax_rows(logits):
    """Greedy token of each row of logits [M][V]: the index of the largest
    value, the smallest such index on ties, NaN entries never chosen (a row
    with no value above -inf gives index 0).

    Follows realizar 0.8.5, src/cuda/executor/reduces.rs, PAR-062 /
    PMAT-045 (batched GPU argmax: for each of M logit vectors, the token ID
    with the maximum logit value).  The pages state no rule for ties or NaN;
    this is the plain reading (first maximum, NaN is no value).
    """
    x = np.asarray(logits, dtype=np.float64)
    M, V = x.shape
    out = np.zeros(M, np.int32)
    for i in range(M):
        best, arg = -np.inf, 0
        for j in range(V):
            v = x[i, j]
            if v == v and v > best:  # NaN fails both comparisons
                best, arg = v, j
        out[i] = arg
    return out


def prefill_attention(q, k, v, causal, fp16_inputs=True):
    """Softmax attention of every query row of every head over the keys of
    the same head: q, k, v [n_heads][seq_len][head_dim] -> out (float64).

    Follows realizar 0.8.5, src/cuda/executor/head_dim.rs,
    tensor_core_attention (PARITY-001.3): inputs given as FP32 and converted
    to FP16 on the GPU, softmax(q k^T / sqrt(head_dim)) v per head, FP32
    output, optional causal masking (query i sees keys 0..i).  With
    fp16_inputs the inputs are first rounded to IEEE half (that conversion is
    a step of the method); everything after it is float64.
    """
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    if fp16_inputs:
        q, k, v = (a.astype(np.float16) for a in (q, k, v))
    q, k, v = (a.astype(np.float64) for a in (q, k, v))
    H, S, D = q.shape
    out = np.empty((H, S, D), np.float64)
    scale = 1.0 / np.sqrt(D)
    for h in range(H):
        s = (q[h] @ k[h].T) * scale                  # [S][S] scores
        if causal:
            s = np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        out[h] = (w @ v[h]) / w.sum(axis=1, keepdims=True)
    return out
