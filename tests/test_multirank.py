"""The one exchange of the sharded path, on CPU ranks (gloo, world size 2).

When the activation tensor of a data-parallel step is split by rows across
ranks, the per-tensor global scale ([SAI] "Core architectural changes of the
MVFP4 format": one FP32 scale per tensor) must come from the amax of the
whole tensor: each rank computes its shard's amax, a MAX all-reduce combines
them, and every rank quantises its rows with the combined value.  The
concatenated shards must then equal the unsharded quantisation bit for bit.
This also checks the max-over-ranks reduction the benchmark uses for time.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = synth.normal_bf16((64, 96), 123, 1.0, 0.01, 40.0)
    rows = x.shape[0] // world
    shard = np.ascontiguousarray(x[rank * rows:(rank + 1) * rows])
    local = torch.tensor([oracle.amax(shard)], dtype=torch.float32)
    dist.all_reduce(local, op=dist.ReduceOp.MAX)
    # the shard's rows, quantised within the whole tensor's index space
    q_global_rows = oracle.quantize(x, amax_v=float(local.item()), sr=False,
                                    rows_range=(rank * rows, (rank + 1) * rows))
    q_rne = oracle.quantize(shard, amax_v=float(local.item()), sr=False)
    np.save(os.path.join(out_dir, f"codes{rank}.npy"), q_rne.codes)
    np.save(os.path.join(out_dir, f"scales{rank}.npy"), q_rne.scales_plain)
    np.save(os.path.join(out_dir, f"globalrows{rank}.npy"),
            q_global_rows.codes[rank * rows:(rank + 1) * rows])
    t = torch.tensor([float(rank + 1) * 1.5])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    np.save(os.path.join(out_dir, f"tmax{rank}.npy"), t.numpy())
    np.save(os.path.join(out_dir, f"amax{rank}.npy"), local.numpy())
    dist.destroy_process_group()


def test_sharded_amax_and_quantisation(tmp_path):
    import oracle
    import synth
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    x = synth.normal_bf16((64, 96), 123, 1.0, 0.01, 40.0)
    full = oracle.quantize(x)
    amaxes = [float(np.load(tmp_path / f"amax{r}.npy")[0]) for r in range(world)]
    assert amaxes[0] == amaxes[1] == oracle.amax(x)
    codes = np.concatenate([np.load(tmp_path / f"codes{r}.npy") for r in range(world)])
    scales = np.concatenate([np.load(tmp_path / f"scales{r}.npy") for r in range(world)])
    np.testing.assert_array_equal(codes, full.codes)
    np.testing.assert_array_equal(scales, full.scales_plain)
    glob = np.concatenate([np.load(tmp_path / f"globalrows{r}.npy") for r in range(world)])
    np.testing.assert_array_equal(glob, full.codes)
    for r in range(world):
        assert float(np.load(tmp_path / f"tmax{r}.npy")[0]) == 3.0
