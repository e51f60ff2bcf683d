"""Multi-rank host logic on CPU (gloo, world size 2): batch sharding and the max-over-ranks
aggregation that bench.py uses. Sharding the batch needs no exchange on the data path because the
normalization statistics are per sample (GroupNorm, LayerNorm) or per row (row-min)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import synth

WL = synth.CONV_GN.replace(N=2, C_in=8, C_out=32, T=48, groups=4)
WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(WORLD))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        inp = bench.shard_inputs(WL, rank)
        y, _ = oracle.conv1d_norm(oracle.params_of(WL), inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"],
                                  nthreads=1)
        gathered = [torch.zeros(y.shape, dtype=torch.float64) for _ in range(WORLD)]
        dist.all_gather(gathered, torch.from_numpy(y))
        # slowest-rank timing, as bench.py reduces it
        t = torch.tensor([1.0 + rank])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            np.save(os.path.join(out_dir, "y.npy"), torch.cat(gathered).numpy())
            np.save(os.path.join(out_dir, "tmax.npy"), t.numpy())
    finally:
        dist.destroy_process_group()


def test_sharded_batch_equals_unsharded(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(port, str(tmp_path)), nprocs=WORLD, start_method="spawn", join=True)
    y_sharded = np.load(tmp_path / "y.npy")
    # one process over the whole global batch of WORLD * N entries
    full = WL.replace(N=WORLD * WL.N)
    inp = synth.make_inputs(full, seed=0)
    y_full, _ = oracle.conv1d_norm(oracle.params_of(full), inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"],
                                   nthreads=1)
    assert np.array_equal(y_sharded, y_full)
    assert float(np.load(tmp_path / "tmax.npy")[0]) == 2.0


def test_shards_are_disjoint_rows_of_one_batch():
    a = bench.shard_inputs(WL, 0)["x"]
    b = bench.shard_inputs(WL, 1)["x"]
    full = synth.make_inputs(WL.replace(N=2 * WL.N), seed=0)["x"]
    assert np.array_equal(np.concatenate([a, b]), full)
    assert not np.array_equal(a, b)


def test_aggregate_uses_the_slowest_rank():
    value, slowest = bench.aggregate([2.0, 4.0], 1e12, 2)
    assert slowest == 4.0 and abs(value - 2 * 1e12 / 4e-3 / 1e12) < 1e-9


def test_p4_shards_are_disjoint_batch_entries_of_one_batch():
    # the p4 workload shards its batch the same way: rank r draws entries [r N, (r + 1) N) of one
    # global batch, so the ranks together run one bigger model batch (weak scaling)
    wl = synth.CONV_TRANSPOSE3D.replace(N=2, D=2, H=4, W=4)
    full = synth.make_convt3d_inputs(wl.replace(N=4))
    parts = [synth.make_convt3d_inputs(wl, n_rows=wl.N, row_offset=r * wl.N) for r in range(2)]
    assert np.array_equal(np.concatenate([p["x"] for p in parts]), full["x"])
    assert all(np.array_equal(p["w"], full["w"]) and np.array_equal(p["b"], full["b"]) for p in parts)
