"""GPU parity of the batched argmax (kvs_argmax, through the C ABI) against
the oracle: token indices must match exactly (integer result; ties, NaN and
infinities included)."""
import numpy as np
import pytest
import torch

import oracle
from split_flash_decoding_kvcachescatter_gb300 import binding as B

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
VOCAB = 152064  # the pages' vocabulary size (PAR-062)


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from split_flash_decoding_kvcachescatter_gb300 import build
    build.build()
    B.lib()


def logit_rows(M, V, seed, ties=True, specials=True):
    """Seeded logits: N(0, 3) values, plus (optionally) planted exact ties of
    the row maximum and NaN / +-inf entries."""
    rng = np.random.default_rng(seed)
    x = (3.0 * rng.standard_normal((M, V))).astype(np.float32)
    for i in range(M):
        if ties and V >= 3:
            j = rng.choice(V, size=3, replace=False)
            x[i, j] = x[i].max() + 1.0          # three equal maxima: the smallest index wins
        if specials and V >= 8:
            k = rng.choice(V, size=4, replace=False)
            x[i, k[0]] = np.nan
            x[i, k[1]] = -np.inf
            x[i, k[2]] = np.nan
    return x


def run(x, offset=0):
    """kvs_argmax on x, optionally with the rows starting `offset` floats into
    the buffer (misaligned for 16-byte loads when offset % 4 != 0)."""
    M, V = x.shape
    buf = torch.empty(offset + M * V, dtype=torch.float32, device=DEV)
    buf[offset:] = torch.from_numpy(x.reshape(-1)).to(DEV)
    logits = buf[offset:].view(M, V)
    ids = torch.full((M,), -7, dtype=torch.int32, device=DEV)
    B.kvs_argmax(logits, ids)
    torch.cuda.synchronize()
    return ids.cpu().numpy()


@pytest.mark.parametrize("M,V", [(1, VOCAB), (4, VOCAB), (3, 1), (5, 3), (2, 1000), (3, 32001),
                                 (7, 4096), (2, 16 * 1024 + 4)])
def test_argmax_matches_oracle(M, V):
    x = logit_rows(M, V, seed=M * 1000 + V)
    assert np.array_equal(run(x), oracle.argmax_rows(x))


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_argmax_misaligned_rows(offset):
    x = logit_rows(3, 40000, seed=offset)
    assert np.array_equal(run(x, offset), oracle.argmax_rows(x))


def test_argmax_special_rows():
    V = 20000
    x = np.zeros((5, V), np.float32)
    x[0, :] = np.nan
    x[1, :] = -np.inf
    x[2, :] = 1.5                         # all equal: index 0
    x[3, :] = np.nan
    x[3, V - 1] = -1e30                   # the only number
    x[4, :] = -np.inf
    x[4, 12345] = np.inf
    x[4, 17] = np.inf                     # two +inf: the first
    want = oracle.argmax_rows(x)
    assert want.tolist() == [0, 0, 0, V - 1, 17]
    assert np.array_equal(run(x), want)


def test_argmax_batch_at_full_size_sampled():
    """M = 32 rows of the full vocabulary in one launch; the oracle checks a
    sample of rows (each row is independent)."""
    M = 32
    x = logit_rows(M, VOCAB, seed=99)
    got = run(x)
    rows = [0, 7, 13, 31]
    assert np.array_equal(got[rows], oracle.argmax_rows(x[rows]))
    # every row: the value at the index is the row's maximum, and no earlier
    # index holds it (checked with numpy, NaN masked)
    xm = np.where(np.isnan(x), -np.inf, x)
    for i in range(M):
        j = got[i]
        assert xm[i, j] == xm[i].max() and not np.any(xm[i, :j] == xm[i, j])


def test_argmax_more_rows_than_one_grid_dimension():
    M, V = 70000, 8
    x = logit_rows(M, V, seed=5, ties=True, specials=False)
    assert np.array_equal(run(x), oracle.argmax_rows(x))


def test_argmax_empty_batch():
    logits = torch.empty((0, 10), dtype=torch.float32, device=DEV)
    assert B.kvs_argmax(logits).numel() == 0
