"""GPU parity of the tensor-core prefill attention (kvs_prefill_attention,
through the C ABI) against the oracle.

Tolerance, from the arithmetic: q, k and v are rounded to FP16 on both
sides (a step of the method), so the only rounding the oracle does not
share is the kernel's: each probability is rounded to FP16 before the P.V
product (relative error <= 2^-11) while the row sum adds the FP32 values,
and the accumulation is FP32.  Output element (h, i, d) is then
sum_j p_j (1 + e_j) v[j, d] / sum_j p_j, which differs from the exact
attention of the rounded inputs by at most 2^-11 * max_j |v16[h, j, d]| over
the attended keys j; the gate adds 5 % and 1e-5 for FP32 accumulation and
the hardware exp2 (relative error ~2^-22)."""
import numpy as np
import pytest
import torch

import oracle
from split_flash_decoding_kvcachescatter_gb300 import binding as B

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from split_flash_decoding_kvcachescatter_gb300 import build
    build.build()
    B.lib()


def inputs(H, S, D, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((H, S, D)).astype(np.float32) for _ in range(3)]


def bound(v, ref, causal):
    v16 = np.abs(v.astype(np.float16).astype(np.float64))
    H, S, D = v.shape
    b = np.empty_like(ref)
    for h in range(H):
        if causal:  # max |v| over keys 0..i
            b[h] = np.maximum.accumulate(v16[h], axis=0)
        else:
            b[h] = np.broadcast_to(v16[h].max(axis=0), (S, D))
    return 2.0 ** -11 * b * 1.05 + 1e-5


def run(q, k, v, causal):
    H, S, D = q.shape
    tq, tk, tv = (torch.from_numpy(a).to(DEV) for a in (q, k, v))
    # the output sits inside a larger buffer: nothing past it may be written
    buf = torch.full((H * S * D + 64,), 12345.0, device=DEV)
    out = buf[:H * S * D].view(H, S, D)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = B.prefill_workspace(H, S, D, device=DEV).fill_(0xFF)  # stale contents must not matter
    B.kvs_prefill_attention(tq, tk, tv, out, causal=causal, workspace=ws, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, B.strerror(int(status.item()))
    assert torch.all(buf[H * S * D:] == 12345.0)
    return out.cpu().numpy()


def check(H, S, D, causal, seed):
    q, k, v = inputs(H, S, D, seed)
    got = run(q, k, v, causal)
    ref = oracle.prefill_attention(q, k, v, causal)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    lim = bound(v, ref, causal)
    worst = np.unravel_index(np.argmax(err - lim), err.shape)
    assert np.all(err <= lim), (f"H={H} S={S} D={D} causal={causal}: err {err[worst]:.3e} > "
                                f"bound {lim[worst]:.3e} at {worst}")
    return float(err.max())


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_one_tile(D, causal):
    check(1, 128, D, causal, seed=D + causal)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S", [1, 16, 100, 129, 384])
def test_sequence_lengths(S, causal):
    check(2, S, 64, causal, seed=S * 2 + causal)


@pytest.mark.parametrize("causal", [True, False])
def test_several_heads_head_dim_128(causal):
    check(3, 300, 128, causal, seed=7 + causal)


def test_long_sequence_causal():
    check(2, 1000, 128, True, seed=11)


@pytest.mark.parametrize("H,S,D,causal", [(2, 2100, 128, True), (3, 2048, 64, False),
                                          (1, 4096, 128, True), (5, 2500, 64, True)])
def test_tiles_packed_beside_the_attention(H, S, D, causal):
    """From 16 key tiles on, part of the FP16 packing runs in the attention
    kernel's pack warps and reaches the copy warp tile by tile through ready
    flags (zeroed by the call, over a workspace full of 0xFF bytes)."""
    check(H, S, D, causal, seed=H * 31 + S + D + causal)


def test_no_in_kernel_tasks_over_any_workspace_contents():
    """Below 16 key tiles the pack warps get no tasks and the call neither
    zeroes nor reads the flags and the task counter: a workspace whose
    counter word reads negative (0x80 bytes) must not matter."""
    H, S, D = 3, 1000, 128
    q, k, v = inputs(H, S, D, seed=5)
    tq, tk, tv = (torch.from_numpy(a).to(DEV) for a in (q, k, v))
    out = torch.empty((H, S, D), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = B.prefill_workspace(H, S, D, device=DEV).fill_(0x80)
    B.kvs_prefill_attention(tq, tk, tv, out, causal=True, workspace=ws, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.prefill_attention(q, k, v, True)
    assert np.all(np.abs(out.cpu().numpy() - ref) <= bound(v, ref, True))


def test_causal_last_row_equals_full_attention_of_last_query():
    """The last causal row attends every key: it equals the non-causal row."""
    q, k, v = inputs(1, 256, 64, seed=13)
    a = run(q, k, v, True)
    b = run(q, k, v, False)
    assert np.allclose(a[0, -1], b[0, -1], rtol=0, atol=1e-6)


def planted(H, S, D, seed, keys, scale):
    """N(0,1) inputs whose k rows at the given key positions are scaled, so
    that those keys' scores jump far above the rest."""
    q, k, v = inputs(H, S, D, seed)
    for j in keys:
        if j < S:
            k[:, j, :] *= scale
    return q, k, v


def check_inputs(q, k, v, causal, where):
    got = run(q, k, v, causal)
    ref = oracle.prefill_attention(q, k, v, causal)
    assert np.all(np.isfinite(got)), where
    err = np.abs(got - ref)
    lim = bound(v, ref, causal)
    worst = np.unravel_index(np.argmax(err - lim), err.shape)
    assert np.all(err <= lim), f"{where}: err {err[worst]:.3e} > bound {lim[worst]:.3e} at {worst}"


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_score_jump_inside_a_key_tile(D, causal):
    """Keys in the second half of a 128-key tile (64..127) score far above the
    first half: the running maximum moves in the middle of the tile, and the
    FP16 P already written for the first half is rescaled in place."""
    S = 512
    q, k, v = planted(2, S, D, seed=17 + D, keys=[70, 200, 330, 460], scale=6.0)
    check_inputs(q, k, v, causal, f"jump inside a tile D={D} causal={causal}")


@pytest.mark.parametrize("D", [64, 128])
def test_score_jump_across_key_tiles(D):
    """A key far above all earlier ones in a later key tile: the output
    accumulator of the rows that attend it is rescaled."""
    S = 640
    q, k, v = planted(2, S, D, seed=29 + D, keys=[300, 610], scale=8.0)
    check_inputs(q, k, v, True, f"jump across tiles D={D}")
