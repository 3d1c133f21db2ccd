"""kvs_flash_decode_static: the entry point for callers that cannot allocate
device memory (it keeps its scratch in a buffer built into the library).

Its output must match kvs_flash_decode (which uses a caller workspace) on the
same inputs, on two calls in a row -- the second call runs on different inputs
over whatever the first left in the shared buffer.  This file is collected
last; it builds the library itself so it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import gate
from split_flash_decoding_kvcachescatter_gb300 import binding as B
from split_flash_decoding_kvcachescatter_gb300 import build as kbuild
from split_flash_decoding_kvcachescatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(seed, M, H, Hkv, D, Lmax, chunk):
    w = W.custom(M=M, num_heads=H, num_kv_heads=Hkv, head_dim=D, max_len=Lmax,
                 chunk_size=chunk, positions="uniform", seed=seed)
    inp = W.make_inputs(w)
    t = W.upload(inp, w, DEV)
    B.kvs_kv_scatter(t["k_rows"], t["v_rows"], t["positions"], t["k_cache"], t["v_cache"])
    return w, t


def _static_call(L, t, w, out, status):
    """One call straight through the C ABI (raw pointers, current stream)."""
    M, H, D = t["q"].shape
    return L.kvs_flash_decode_static(
        t["q"].data_ptr(), t["k_cache"].data_ptr(), t["v_cache"].data_ptr(),
        t["positions"].data_ptr(), out.data_ptr(), M, H, w.num_kv_heads, D, w.max_len,
        w.chunk_size, status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_static_workspace_entry_matches_workspace_entry():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    kbuild.build()
    L = B.lib()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cases = [dict(seed=41, M=8, H=32, Hkv=8, D=128, Lmax=3000, chunk=0),
             dict(seed=42, M=5, H=14, Hkv=2, D=64, Lmax=777, chunk=100)]
    for c in cases:  # two calls in a row, different inputs and shapes
        w, t = _case(**c)
        ws = B.workspace(w.M, w.num_heads, w.num_kv_heads, w.head_dim, w.max_len,
                         w.chunk_size, device=DEV)
        ref = torch.empty_like(t["q"])
        B.kvs_flash_decode(t["q"], t["k_cache"], t["v_cache"], t["positions"], ref,
                           chunk_size=w.chunk_size, workspace=ws)
        out = torch.full_like(t["q"], float("nan"))
        assert _static_call(L, t, w, out, status) == B.KVS_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        gate(out.cpu().numpy(), ref.cpu().numpy(), where=f"static vs workspace entry {c}")


def test_static_workspace_entry_rejects_problems_beyond_its_buffer():
    kbuild.build()
    L = B.lib()
    # 1024 sequences x 8 kv heads x 8 query heads per group: ~37 MB of partials
    need = B.kvs_flash_decode_workspace_bytes(1024, 64, 8, 128, 4096, 64)
    assert need > B.KVS_STATIC_WORKSPACE_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = L.kvs_flash_decode_static(fake, fake, fake, fake, fake, 1024, 64, 8, 128, 4096, 64,
                                   None, None)
    assert rc == B.KVS_ERR_WORKSPACE
