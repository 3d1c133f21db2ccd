"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each with its
own batch; only the timings (max) and byte counts (sum) are exchanged."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench
from split_flash_decoding_kvcachescatter_gb300 import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as tdist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.WORKLOADS["tiny"]
    inp = W.make_inputs(w, seed=bench.rank_seed(w, rank))
    ab = W.algorithmic_bytes(inp, w)
    step_ms = 10.0 + rank  # rank 1 is the slow one
    e2e_ms = 20.0 - rank
    res = bench.reduce_over_ranks(step_ms, e2e_ms, ab["step"] * 3, ab["step"] * 2, world, "cpu")
    np.save(os.path.join(out_dir, f"r{rank}.npy"),
            np.array(list(res) + [float(inp.q.sum()), ab["step"]]))
    tdist.barrier()
    tdist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r0 = np.load(tmp_path / "r0.npy")
    r1 = np.load(tmp_path / "r1.npy")
    assert np.allclose(r0[:4], r1[:4])  # every rank sees the same reduction
    assert r0[0] == 11.0 and r0[1] == 20.0  # max over ranks
    assert r0[2] == 3 * (r0[5] + r1[5]) and r0[3] == 2 * (r0[5] + r1[5])  # sum of bytes
    assert r0[4] != r1[4]  # independent batches per rank


def test_single_rank_is_identity():
    assert bench.reduce_over_ranks(1.5, 2.5, 10, 20, 1, "cpu") == (1.5, 2.5, 10.0, 20.0)
