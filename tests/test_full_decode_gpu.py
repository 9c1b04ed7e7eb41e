"""The full-model decode step (32 layers x {qkv, o, gate_up, down}, r = 16,
100 resident adapters, 512 tokens uniform over them) against the oracle.

One metadata pass serves every layer, as in a serving step: the groups of
layer 0 and the down projection of layer 1 run through lora_apply with
the same TokenMeta, each checked in full against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_harness import TOL_BF16, bf16_half_ulp, load_table, to_dev

pytestmark = pytest.mark.gpu


def _groups():
    n = len(wl.FULL_DECODE_GROUPS)
    for i, inst in enumerate(wl.full_decode_groups()):
        if i < n or i == 2 * n - 1:       # layer 0 (all groups) and layer 1's down projection
            yield inst
        if i == 2 * n - 1:
            return


def test_full_decode_groups_share_one_metadata_pass(lib):
    meta = None
    seen = 0
    for inst in _groups():
        if meta is None:
            meta = lib.TokenMeta(inst.num_tokens, inst.num_slots)
            meta.prepare(torch.from_numpy(inst.token_slot).cuda())
        t = load_table(inst)
        x = to_dev(inst.x, "bf16")
        y = to_dev(inst.y_in, "bf16")
        lib.apply(t, meta, x, y, kind=lib.LORA_AUTO)
        torch.cuda.synchronize()
        ads = oracle.adapters_f64(inst)
        x64 = inst.to_f32(inst.x).astype(np.float64)
        y64 = inst.to_f32(inst.y_in).astype(np.float64)
        buf, written = oracle.shrink_requests(x64, ads, inst.n_slices, inst.r_max, inst.req_lengths,
                                              inst.req_slots, inst.num_slots)
        y_ref = oracle.expand_requests(buf, y64, ads, inst.out_sizes, inst.req_lengths, inst.req_slots,
                                       inst.num_slots)
        assert written.all()      # every token carries an adapter in this workload
        rms = np.sqrt(np.mean((y_ref - y64) ** 2))
        excess = np.abs(y.float().cpu().numpy().astype(np.float64) - y_ref) - (TOL_BF16 * rms + bf16_half_ulp(y_ref))
        assert excess.max() <= 0, f"{inst.name}: max excess {excess.max():.3e}"
        seen += 1
    assert seen == len(wl.FULL_DECODE_GROUPS) + 1
    st, _ = lib.lora_query_status(meta.c)
    assert st == lib.LORA_OK
