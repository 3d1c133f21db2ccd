"""Seeded synthetic workloads for the decode-step attention path.

This module only draws random inputs; it holds none of the method's
arithmetic.  Both the CUDA path's tests/benchmark and the CPU oracle read
the arrays it returns.

The shapes follow the pages' batched decode step (realizar 0.8.5,
src/cuda/executor/head_dim.rs, ``flash_decoding_attention_into``, doc
comment: Q [M, num_heads, head_dim], new K/V rows [M, num_kv_heads,
head_dim]; per-sequence cache [num_kv_heads][max_len][head_dim]).

Recipe (all float32, numpy PCG64):
  * positions   : ``default_rng([seed, 0])``; "uniform" -> integers in
                  [0, max_len); "loguniform" -> p = min(floor(exp(U ln(max_len+1))) - 1,
                  max_len - 1) with U ~ U[0,1), then p_0 forced to 0; "fixed" -> all equal.
  * q           : ``default_rng([seed, 1, layer])``, N(0, std^2), shape [M, H, D].
  * sequence i  : ``default_rng([seed, 2, layer, i])`` draws K rows [Hkv, p_i+1, D],
                  then V rows [Hkv, p_i+1, D] (both N(0, std^2)), then, if the
                  workload has outliers, one Bernoulli(outlier_p) per position; a
                  selected position has its K row multiplied by outlier_scale in
                  every kv head.  Row p_i of these arrays is the sequence's new
                  K/V row (the scatter input); rows 0..p_i-1 are the prefilled cache.
Each sequence has its own generator, so one sequence can be redrawn alone.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    max_len: int
    chunk_size: int  # 0 = let the library choose
    positions: str  # "fixed" | "uniform" | "loguniform"
    fixed_position: int = 0
    layers: int = 1
    std: float = 1.0
    outlier_p: float = 0.0
    outlier_scale: float = 1.0
    seed: int = 0
    chunk_sweep: tuple = ()

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    def cache_elems(self) -> int:
        return self.M * self.num_kv_heads * self.max_len * self.head_dim


# The five workloads the decode path is measured on.  Seeds are 1000 + index.
WORKLOADS = {
    "tiny": Workload("tiny", M=1, num_heads=4, num_kv_heads=2, head_dim=64,
                     max_len=256, chunk_size=64, positions="fixed",
                     fixed_position=255, seed=1001),
    "small_model": Workload("small_model", M=4, num_heads=14, num_kv_heads=2,
                            head_dim=64, max_len=2048, chunk_size=128,
                            positions="uniform", layers=24, seed=1002),
    "8b_batch": Workload("8b_batch", M=32, num_heads=32, num_kv_heads=8,
                         head_dim=128, max_len=8192, chunk_size=0,
                         positions="uniform", outlier_p=0.01, outlier_scale=8.0,
                         seed=1003),
    "long_context": Workload("long_context", M=8, num_heads=32, num_kv_heads=8,
                             head_dim=128, max_len=32768, chunk_size=256,
                             positions="fixed", fixed_position=32767, seed=1004,
                             chunk_sweep=(128, 256, 512)),
    "ragged": Workload("ragged", M=32, num_heads=40, num_kv_heads=8, head_dim=128,
                       max_len=131072, chunk_size=256, positions="loguniform",
                       std=0.5, seed=1005),
}


@dataclasses.dataclass
class DecodeInputs:
    """One layer's inputs for one decode step."""
    positions: np.ndarray  # int32 [M]
    q: np.ndarray  # float32 [M, H, D]
    k_rows: np.ndarray  # float32 [M, Hkv, D]  new rows (scatter input)
    v_rows: np.ndarray  # float32 [M, Hkv, D]
    k_seq: List[np.ndarray]  # per sequence float32 [Hkv, p_i + 1, D]; row p_i == k_rows[i]
    v_seq: List[np.ndarray]

    @property
    def seq_lens(self) -> np.ndarray:
        return self.positions.astype(np.int64) + 1


def draw_positions(w: Workload, seed: Optional[int] = None) -> np.ndarray:
    seed = w.seed if seed is None else seed
    rng = np.random.default_rng([seed, 0])
    if w.positions == "fixed":
        p = np.full(w.M, w.fixed_position, dtype=np.int64)
    elif w.positions == "uniform":
        p = rng.integers(0, w.max_len, size=w.M)
    elif w.positions == "loguniform":
        u = rng.random(w.M)
        p = np.floor(np.exp(u * np.log(w.max_len + 1.0))).astype(np.int64) - 1
        p = np.clip(p, 0, w.max_len - 1)
        p[0] = 0
    else:
        raise ValueError(w.positions)
    return p.astype(np.int32)


def draw_sequence(w: Workload, i: int, position: int, layer: int = 0,
                  seed: Optional[int] = None):
    """Rows 0..position of sequence i (K, V), each [Hkv, position + 1, D]."""
    seed = w.seed if seed is None else seed
    rng = np.random.default_rng([seed, 2, layer, i])
    shape = (w.num_kv_heads, position + 1, w.head_dim)
    K = rng.standard_normal(shape, dtype=np.float32)
    V = rng.standard_normal(shape, dtype=np.float32)
    if w.std != 1.0:
        K *= np.float32(w.std)
        V *= np.float32(w.std)
    if w.outlier_p > 0.0:
        mask = rng.random(position + 1) < w.outlier_p
        K[:, mask, :] *= np.float32(w.outlier_scale)
    return K, V


def make_inputs(w: Workload, layer: int = 0, seed: Optional[int] = None,
                positions: Optional[np.ndarray] = None) -> DecodeInputs:
    seed = w.seed if seed is None else seed
    pos = draw_positions(w, seed) if positions is None else np.asarray(positions, np.int32)
    rng_q = np.random.default_rng([seed, 1, layer])
    q = rng_q.standard_normal((w.M, w.num_heads, w.head_dim), dtype=np.float32)
    if w.std != 1.0:
        q *= np.float32(w.std)
    k_seq, v_seq = [], []
    k_rows = np.empty((w.M, w.num_kv_heads, w.head_dim), np.float32)
    v_rows = np.empty_like(k_rows)
    for i in range(w.M):
        # an out-of-range position still gets one drawn row (never attended)
        p = int(min(max(int(pos[i]), 0), w.max_len - 1))
        K, V = draw_sequence(w, i, p, layer, seed)
        k_seq.append(K)
        v_seq.append(V)
        k_rows[i] = K[:, p, :]
        v_rows[i] = V[:, p, :]
    return DecodeInputs(pos, q, k_rows, v_rows, k_seq, v_seq)


def custom(name="custom", **kw) -> Workload:
    """A workload with explicit fields (used for parity sweeps and edge cases)."""
    base = dict(M=1, num_heads=4, num_kv_heads=2, head_dim=64, max_len=256,
                chunk_size=64, positions="uniform", seed=7)
    base.update(kw)
    return Workload(name, **base)


def kv_bytes(inp: DecodeInputs, w: Workload) -> int:
    """Live K and V bytes one attention call reads (rows 0..p_i, all kv heads)."""
    return int(2 * w.num_kv_heads * w.head_dim * 4 * inp.seq_lens.sum())


def algorithmic_bytes(inp: DecodeInputs, w: Workload) -> dict:
    """Algorithmic bytes of one decode step (one layer).

    attention: live KV bytes read + Q read + O written + positions read.
    scatter:   new K/V rows read + the same bytes written + positions read.
    """
    qo = 2 * w.M * w.num_heads * w.head_dim * 4
    attn = kv_bytes(inp, w) + qo + 4 * w.M
    scat = 4 * w.M * w.num_kv_heads * w.head_dim * 4 + 4 * w.M
    return {"attention": attn, "scatter": scat, "step": attn + scat,
            "chunk_kernel": kv_bytes(inp, w) + w.M * w.num_heads * w.head_dim * 4}


# Bit pattern used to poison cache rows that hold no live data (a NaN).
POISON_BITS = -1  # 0xFFFFFFFF as int32


def poisoned_cache(w: Workload, device):
    """A [M, Hkv, Lmax, D] float32 device tensor whose every element is the
    NaN with bits 0xFFFFFFFF, so reading any row that is not live shows up."""
    import torch
    t = torch.full((w.M, w.num_kv_heads, w.max_len, w.head_dim), POISON_BITS,
                   dtype=torch.int32, device=device)
    return t.view(torch.float32)


def upload(inp: DecodeInputs, w: Workload, device, include_new_row: bool = False):
    """Device tensors for one layer: q, k_rows, v_rows, positions and the two
    caches holding rows 0..p_i-1 of every sequence (rows p_i.. poisoned).

    With include_new_row the caches also hold row p_i, i.e. the state the
    scatter must produce (used as the expected cache; built with plain
    torch copies of the generator's arrays)."""
    import torch
    k_cache = poisoned_cache(w, device)
    v_cache = poisoned_cache(w, device)
    for i in range(w.M):
        p = int(inp.positions[i])
        if p < 0 or p >= w.max_len:
            continue
        n = p + 1 if include_new_row else p
        if n > 0:
            k_cache[i, :, :n, :].copy_(torch.from_numpy(np.ascontiguousarray(inp.k_seq[i][:, :n])))
            v_cache[i, :, :n, :].copy_(torch.from_numpy(np.ascontiguousarray(inp.v_seq[i][:, :n])))
    return {
        "q": torch.from_numpy(inp.q).to(device),
        "k_rows": torch.from_numpy(inp.k_rows).to(device),
        "v_rows": torch.from_numpy(inp.v_rows).to(device),
        "positions": torch.from_numpy(inp.positions.astype(np.int32)).to(device),
        "k_cache": k_cache,
        "v_cache": v_cache,
    }
