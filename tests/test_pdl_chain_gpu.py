"""Back-to-back steps on one stream against the same steps with a device
synchronisation after each one.

The library's kernels overlap their successors (programmatic dependent
launch): the metadata kernel sorts before it waits and releases the shrink at
its start, and in an AUTO split the SGMV kernels work beside the BGMV kernels
of the same call. Here two request batches alternate on one stream, each with
its own metadata buffers but one shared workspace, and every step recomputes
its metadata and adds its delta into its y again; any read of data that a
still-running kernel writes (metadata, partial rows, y) would change the
fp32 results, which must equal bitwise those of the same steps run one at a
time."""
import numpy as np
import pytest
import torch

import rank_adapter_gb300 as ra
import workloads as wl
from gpu_harness import load_table, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    # decode: one BGMV family (fewer tokens than the AUTO split threshold)
    "decode": lambda seed: wl.make_instance("decode_qkv", seed=seed, num_tokens=200, d_in=2048,
                                            out_sizes=[1024, 256], num_slots=17),
    # mixed: AUTO with short segments on BGMV and long ones on SGMV in every call
    "mixed": lambda seed: wl.make_instance("mixed_o_proj", seed=seed, d_in=1024, out_sizes=[768], num_slots=24),
}


@pytest.mark.parametrize("path", ["apply", "split"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_back_to_back_steps_equal_synchronised_steps(lib, name, path):
    insts = [CASES[name](s) for s in (40, 41)]
    for inst in insts[1:]:
        inst.adapters = insts[0].adapters          # one slot table serves both batches
    table = load_table(insts[0])
    T = max(i.num_tokens for i in insts)
    ws = lib.workspace(table, T, lib.LORA_AUTO)     # shared by both batches
    sets = []
    for inst in insts:
        meta = lib.TokenMeta(inst.num_tokens, inst.num_slots)
        meta.token_slot[:inst.num_tokens].copy_(torch.from_numpy(inst.token_slot).cuda())
        meta.set_num_tokens(inst.num_tokens)
        x = to_dev(inst.x, "bf16")
        y0 = torch.from_numpy(inst.to_f32(inst.y_in)).cuda()
        buf = torch.zeros(inst.n_slices, inst.num_tokens, inst.r_max, dtype=torch.float32, device="cuda")
        sets.append((meta, x, y0, buf))
    torch.cuda.synchronize()
    steps = 6

    def step(k, y):
        meta, x, _, buf = sets[k]
        lib.check(lib.lora_prepare_meta(meta.c, None), "prepare_meta")
        if path == "apply":
            lib.apply(table, meta, x, y, kind=lib.LORA_AUTO, ws=ws)
        else:
            lib.shrink(table, meta, x, buf, lib.LORA_AUTO, ws=ws)
            lib.expand(table, meta, buf, y, lib.LORA_AUTO)

    ref = []
    for k in range(2):
        y = sets[k][2].clone()
        for _ in range(steps):
            step(k, y)
            torch.cuda.synchronize()
        ref.append(y.cpu().numpy())
    ys = [sets[k][2].clone() for k in range(2)]
    torch.cuda.synchronize()
    for i in range(2 * steps):
        step(i % 2, ys[i % 2])
    torch.cuda.synchronize()
    for k in range(2):
        got = ys[k].cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref[k].view(np.uint32)), f"batch {k}"
        assert not np.array_equal(got, insts[k].to_f32(insts[k].y_in))   # the deltas were applied
    for meta, *_ in sets:
        assert lib.lora_query_status(meta.c) == (lib.LORA_OK, 0)
