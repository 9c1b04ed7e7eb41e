"""The data-parallel host logic of bench.py on two CPU ranks (gloo).

The library shards by independent batches: every rank runs its own requests
against its own copy of the slot table, with no collective on the data path.
What crosses ranks is the bookkeeping: the whole-job time is the slowest
rank's, and the whole-job token count is the sum over ranks."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r pretends to have run for 10 + r ms (e2e 20 - r ms) and served 100 + r LoRA tokens
        el, e2e, tok = bench.reduce_over_ranks(torch, dist, 10.0 + rank, 20.0 - rank, 100 + rank, "cpu")
        inst = bench.make_workload("decode_qkv", seed_offset=rank)
        np.savez(os.path.join(out_dir, f"r{rank}.npz"), red=np.array([el, e2e, tok]), ts=inst.token_slot,
                 x=inst.x[:4], shape=np.array([inst.num_tokens, inst.d_in, inst.d_out_total, inst.num_slots]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_draw_independent_batches(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r = [np.load(tmp_path / f"r{i}.npz") for i in range(world)]
    for i in range(world):   # every rank sees the same whole-job numbers
        assert r[i]["red"].tolist() == [11.0, 20.0, 201.0]
    assert np.array_equal(r[0]["shape"], r[1]["shape"])          # same workload shape on every rank
    assert not np.array_equal(r[0]["ts"], r[1]["ts"])             # independent batches
    assert not np.array_equal(r[0]["x"], r[1]["x"])


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(torch, None, 3.5, 4.5, 7, "cpu") == (3.5, 4.5, 7.0)
