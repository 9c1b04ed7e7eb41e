"""The fully-sharded variant's two layer kinds through the C ABI on one GPU, two
shards emulated one after the other (section "S-LoRA 式:把秩也切开" of page
"vLLM 源码完全拆解(十八): 多 LoRA 服务"). Each shard is its own slot tables;
x's d_in shard and the output's column range (offset_start) are strided views
passed as pointer + leading dimension; a sum and a concatenation stand in for
the all-reduce and the all-gather. The result must match the fp64 oracle's
unsharded delta within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import rank_adapter_gb300 as ra
import workloads as wl
from gpu_harness import TOL_BF16, lib_dtype, to_dev

pytestmark = pytest.mark.gpu


def _reference(inst):
    ads = oracle.adapters_f64(inst)
    x = inst.to_f32(inst.x).astype(np.float64)
    return oracle.apply_requests(x, np.zeros((inst.num_tokens, inst.d_out_total)), ads, inst.out_sizes,
                                 inst.r_max, inst.req_lengths, inst.req_slots, inst.num_slots)


def _table(inst, d_in, width, r_max, pieces):
    """A single-slice slot table filled from pieces[a] = (rank, A [d_in, r] or None, B [r, width]).
    A table that only expands gets a zero A (a slice's A and B are given together)."""
    t = ra.SlotTable(d_in, [width], inst.num_slots, r_max, lib_dtype(inst))
    for a, (rank, A, B) in pieces.items():
        if rank == 0:
            t.reset_slot(a)
        else:
            if A is None:
                A = np.zeros((d_in, rank), dtype=inst.x.dtype)
            scale = inst.adapters[a].scale
            t.set_slot(a, rank, scale, [to_dev(np.ascontiguousarray(A), inst.dtype)],
                       [to_dev(np.ascontiguousarray(B), inst.dtype)])
    torch.cuda.synchronize()
    return t


def _check(y, ref):
    delta = ref[ref.any(axis=1)]
    rms = np.sqrt(np.mean(delta ** 2))
    err = np.abs(y - ref).max()
    assert err <= TOL_BF16 * rms, f"max err {err:.3e} > {TOL_BF16:.0e} x RMS {rms:.3e}"


@pytest.mark.parametrize("kind_name", ["LORA_BGMV", "LORA_SGMV"])
def test_row_parallel_fully_sharded(lib, kind_name):
    kind = getattr(lib, kind_name)
    inst = wl.make_instance("mixed_o_proj", num_tokens=300, d_in=1024, out_sizes=[512], num_slots=17)
    T, D, O, R = inst.num_tokens, inst.d_in, inst.d_out_total, inst.r_max
    D2, O2 = D // 2, O // 2
    meta = lib.TokenMeta(T, inst.num_slots)
    meta.prepare(torch.from_numpy(inst.token_slot).cuda())
    x = to_dev(inst.x, inst.dtype)
    u = torch.zeros(1, T, R, dtype=torch.float32, device="cuda")
    y = torch.zeros(2, T, O, dtype=torch.float32, device="cuda")   # the two shards' partial outputs
    for k in range(2):
        ad = inst.adapters
        t_in = _table(inst, D2, O, R, {a: (ad[a].rank, ad[a].A[0][k * D2:(k + 1) * D2], ad[a].B[0])
                                       for a in ad})
        part = torch.zeros(1, T, R, dtype=torch.float32, device="cuda")
        lib.shrink(t_in, meta, x[:, k * D2:], part, kind=kind)       # x's d_in shard: pointer + ldx
        u += part                                                    # the all-reduce of u
    for k in range(2):
        ad = inst.adapters
        t_out = _table(inst, D2, O2, R, {a: (ad[a].rank, None, ad[a].B[0][:, k * O2:(k + 1) * O2]) for a in ad})
        lib.expand(t_out, meta, u, y[k][:, k * O2:], kind=kind)      # offset_start = k * O2 columns
    torch.cuda.synchronize()
    _check((y[0] + y[1]).double().cpu().numpy(), _reference(inst))  # the layer's all-reduce


@pytest.mark.parametrize("kind_name", ["LORA_BGMV", "LORA_SGMV"])
def test_column_parallel_rank_split(lib, kind_name):
    kind = getattr(lib, kind_name)
    inst = wl.make_instance("mixed_o_proj", num_tokens=300, d_in=1024, out_sizes=[512], num_slots=17)
    T, D, O, R = inst.num_tokens, inst.d_in, inst.d_out_total, inst.r_max
    R2, O2 = R // 2, O // 2
    meta = lib.TokenMeta(T, inst.num_slots)
    meta.prepare(torch.from_numpy(inst.token_slot).cuda())
    x = to_dev(inst.x, inst.dtype)
    shards = []
    for k in range(2):
        ad = inst.adapters
        pieces = {}
        for a in ad:
            rl = min(max(ad[a].rank - k * R2, 0), R2)
            A = ad[a].A[0][:, k * R2:k * R2 + rl] if rl else None
            B = ad[a].B[0][k * R2:k * R2 + rl] if rl else None
            pieces[a] = (rl, A, B)
        t_in = _table(inst, D, O, R2, pieces)
        part = torch.zeros(1, T, R2, dtype=torch.float32, device="cuda")
        lib.shrink(t_in, meta, x, part, kind=kind)
        shards.append(part)
    u = torch.cat(shards, dim=2).contiguous()                        # the all-gather along the rank dim
    outs = []
    for k in range(2):
        ad = inst.adapters
        t_out = _table(inst, D, O2, R, {a: (ad[a].rank, None, ad[a].B[0][:, k * O2:(k + 1) * O2]) for a in ad})
        y_k = torch.zeros(T, O2, dtype=torch.float32, device="cuda")
        lib.expand(t_out, meta, u, y_k, kind=kind)
        outs.append(y_k)
    torch.cuda.synchronize()
    _check(torch.cat(outs, dim=1).double().cpu().numpy(), _reference(inst))
