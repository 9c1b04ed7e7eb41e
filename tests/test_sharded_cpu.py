"""The fully-sharded (S-LoRA rank-split) variant on two CPU ranks (gloo), with the
fp64 oracle: the sharding math of page "vLLM 源码完全拆解(十八): 多 LoRA 服务",
section "S-LoRA 式:把秩也切开".

* Row-parallel layer: rank k holds the d_in shard of x and of A, and the output
  columns shard k of B. Its shrink gives a partial u; the partials are summed by
  an all-reduce; the expand adds u B_k into the columns [k * d_out/2, ...) of
  the rank's partial output (offset_start), and the layer's own all-reduce of
  the partial outputs completes the delta.
* Column-parallel layer: rank k holds the rank columns shard k of A and the
  output columns shard k of B. Its shrink gives u's rank shard; an all-gather
  along the rank dimension rebuilds u; the expand gives the rank's output shard.

Both must equal the unsharded delta (to fp64 rounding: the sums run in another
order). The scale multiplies every partial, which the sums and the
concatenation carry through unchanged."""
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


def _instance():
    import workloads as wl
    # heterogeneous ranks {8,16,32,64} padded to 64, scales alpha/r, 5% no-LoRA rows
    return wl.make_instance("mixed_o_proj", num_tokens=24, d_in=256, out_sizes=[128], num_slots=9, dtype="f32")


def _zero_unwritten(buf):
    return np.where(np.isnan(buf), 0.0, buf)


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    from oracle import lora_oracle as lo
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inst = _instance()
        ads = lo.adapters_f64(inst)
        x = inst.to_f32(inst.x).astype(np.float64)
        T, D, O, R = inst.num_tokens, inst.d_in, inst.d_out_total, inst.r_max
        L, Sl, S = inst.req_lengths, inst.req_slots, inst.num_slots
        D2, O2, R2 = D // world, O // world, R // world
        cols = slice(rank * O2, (rank + 1) * O2)

        # Row-parallel: shrink over the d_in shard, all-reduce u, expand with B's columns shard k
        ads_in = {a: (r, s, [A[0][rank * D2:(rank + 1) * D2]], B) for a, (r, s, A, B) in ads.items()}
        buf, _ = lo.shrink_requests(x[:, rank * D2:(rank + 1) * D2], ads_in, 1, R, L, Sl, S)
        u = torch.from_numpy(_zero_unwritten(buf))
        dist.all_reduce(u)
        ads_out = {a: (r, s, A, [B[0][:, cols]]) for a, (r, s, A, B) in ads.items()}
        part = np.zeros((T, O))
        part[:, cols] = lo.expand_requests(u.numpy(), np.zeros((T, O2)), ads_out, [O2], L, Sl, S)
        y_row = torch.from_numpy(part)
        dist.all_reduce(y_row)

        # Column-parallel, rank split: shrink with A's rank shard, all-gather u along the rank dim
        ads_r = {}
        for a, (r, s, A, B) in ads.items():
            rl = min(max(r - rank * R2, 0), R2)
            ads_r[a] = (rl, s, [A[0][:, rank * R2:(rank + 1) * R2]], [B[0][rank * R2:(rank + 1) * R2]])
        buf_r, _ = lo.shrink_requests(x, ads_r, 1, R2, L, Sl, S)
        shards = [torch.zeros(1, T, R2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(shards, torch.from_numpy(_zero_unwritten(buf_r)))
        u_full = torch.cat(shards, dim=2).numpy()
        y_k = lo.expand_requests(u_full, np.zeros((T, O2)), ads_out, [O2], L, Sl, S)
        outs = [torch.zeros(T, O2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(outs, torch.from_numpy(y_k))
        y_col = torch.cat(outs, dim=1).numpy()
        np.savez(os.path.join(out_dir, f"r{rank}.npz"), row=y_row.numpy(), col=y_col)
    finally:
        dist.destroy_process_group()


def test_fully_sharded_row_and_column_parallel_on_two_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    sys.path.insert(0, ROOT)
    from oracle import lora_oracle as lo
    inst = _instance()
    ads = lo.adapters_f64(inst)
    x = inst.to_f32(inst.x).astype(np.float64)
    ref = lo.apply_requests(x, np.zeros((inst.num_tokens, inst.d_out_total)), ads, inst.out_sizes, inst.r_max,
                            inst.req_lengths, inst.req_slots, inst.num_slots)
    assert np.abs(ref).max() > 0
    assert len({ad[0] for ad in ads.values()}) > 1          # several ranks, some below one shard
    tol = 1e-12 * np.abs(ref).max()
    for i in range(world):
        r = np.load(tmp_path / f"r{i}.npz")
        assert np.allclose(r["row"], ref, rtol=0, atol=tol), "row-parallel sharded delta"
        assert np.allclose(r["col"], ref, rtol=0, atol=tol), "column-parallel sharded delta"
