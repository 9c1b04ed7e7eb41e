"""The full-model decode step (32 layers x {qkv, o, gate_up, down}, r = 16,
100 resident adapters, 512 tokens uniform over them) against the oracle.

As in a serving step, every group's slot table is resident, one metadata pass
serves all 128 groups and their lora_apply calls run back to back on one
stream; then each group's output is checked in full (every row and column)
against the oracle. The inputs are drawn twice from the same seeded
generator (once for the device, once for the oracle) so that the host never
holds the whole step's 8.4 GB of weights at once."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_harness import TOL_BF16, bf16_half_ulp, load_table, to_dev

pytestmark = pytest.mark.gpu


def test_full_decode_step_every_group(lib):
    tables, xs, ys, meta = [], [], [], None
    for inst in wl.full_decode_groups():
        if meta is None:
            meta = lib.TokenMeta(inst.num_tokens, inst.num_slots)
            ts = torch.from_numpy(inst.token_slot).cuda()
        tables.append(load_table(inst))
        xs.append(to_dev(inst.x, "bf16"))
        ys.append(to_dev(inst.y_in, "bf16"))
    assert len(tables) == 32 * len(wl.FULL_DECODE_GROUPS)
    meta.prepare(ts)
    for t, x, y in zip(tables, xs, ys):   # the step: one metadata pass, 128 applies, no host sync in between
        lib.apply(t, meta, x, y, kind=lib.LORA_AUTO)
    torch.cuda.synchronize()
    st, _ = lib.lora_query_status(meta.c)
    assert st == lib.LORA_OK
    del tables, xs
    for i, inst in enumerate(wl.full_decode_groups()):
        ads = oracle.adapters_f64(inst)
        x64 = inst.to_f32(inst.x).astype(np.float64)
        y64 = inst.to_f32(inst.y_in).astype(np.float64)
        buf, written = oracle.shrink_requests(x64, ads, inst.n_slices, inst.r_max, inst.req_lengths,
                                              inst.req_slots, inst.num_slots)
        y_ref = oracle.expand_requests(buf, y64, ads, inst.out_sizes, inst.req_lengths, inst.req_slots,
                                       inst.num_slots)
        assert written.all()      # every token carries an adapter in this workload
        rms = np.sqrt(np.mean((y_ref - y64) ** 2))
        y_gpu = ys[i].float().cpu().numpy().astype(np.float64)
        excess = np.abs(y_gpu - y_ref) - (TOL_BF16 * rms + bf16_half_ulp(y_ref))
        assert excess.max() <= 0, f"{inst.name}: max excess {excess.max():.3e}"
        ys[i] = None
