"""The allocation-free shrink (lora_shrink_noalloc) against lora_shrink.

lora_shrink_noalloc serves callers that cannot allocate device memory where
they run the shrink (inside another framework's memory pool, or on a serving
path that must not call an allocator): it keeps its partial rows in a fixed
device array inside the library. Its output must match lora_shrink's (with a
caller workspace) within the parity tolerance, on two calls in a row (the
array keeps the previous call's contents), and a layer whose partial rows do
not fit the array is refused before anything is launched.

This file is collected last on purpose: it must pass both alone in a fresh
process and after every other test.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_harness import TOL_BF16, load_table, to_dev

pytestmark = pytest.mark.gpu


def _shrink(lib, table, meta, x, ws_kind):
    buf = torch.full((len(table.out_sizes), meta.c.num_tokens, table.r_max), float("nan"), dtype=torch.float32,
                     device="cuda")
    if ws_kind == "noalloc":
        lib.check(lib.lora_shrink_noalloc(table.desc, meta.c, x.data_ptr(), x.stride(0), buf.data_ptr()),
                  "lora_shrink_noalloc")
    else:
        lib.shrink(table, meta, x, buf, kind=lib.LORA_BGMV)
    torch.cuda.synchronize()
    return buf.cpu().numpy()


def test_noalloc_shrink_matches_workspace_shrink_twice(lib):
    # d_in = 4096 spreads the shrink over several chunks, so the partial rows really go through scratch.
    inst = wl.make_instance("decode_qkv", num_tokens=200, d_in=4096, out_sizes=[1024, 256, 256], num_slots=17)
    table = load_table(inst)
    assert 0 < lib.lora_workspace_bytes(table.desc, inst.num_tokens) <= lib.lora_noalloc_scratch_bytes()
    meta = lib.TokenMeta(inst.num_tokens, inst.num_slots)
    meta.prepare(torch.from_numpy(inst.token_slot).cuda())
    x = to_dev(inst.x, "bf16")
    ref = _shrink(lib, table, meta, x, "workspace")
    written = ~np.isnan(ref[0, :, 0])
    assert written.any()
    rms = float(np.sqrt(np.mean(ref[:, written] ** 2)))
    for _ in range(2):
        got = _shrink(lib, table, meta, x, "noalloc")
        assert np.array_equal(np.isnan(got), np.isnan(ref)), "rows written differ"
        err = float(np.max(np.abs(got[:, written] - ref[:, written])))
        assert err <= TOL_BF16 * rms, f"max err {err:.3e} > {TOL_BF16} x RMS {rms:.3e}"
        # same kernels, same arithmetic: the header promises the same results, bit for bit
        assert np.array_equal(got, ref, equal_nan=True)


def test_noalloc_shrink_allocates_nothing(lib):
    """After a first call (which looks up the array's address), further calls leave the
    device's free memory unchanged."""
    inst = wl.make_instance("decode_qkv", seed=13, num_tokens=128, d_in=4096, out_sizes=[512, 128], num_slots=9)
    table = load_table(inst)
    meta = lib.TokenMeta(inst.num_tokens, inst.num_slots)
    meta.prepare(torch.from_numpy(inst.token_slot).cuda())
    x = to_dev(inst.x, "bf16")
    buf = torch.zeros(2, inst.num_tokens, table.r_max, dtype=torch.float32, device="cuda")
    lib.check(lib.lora_shrink_noalloc(table.desc, meta.c, x.data_ptr(), x.stride(0), buf.data_ptr()), "warm-up")
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        lib.check(lib.lora_shrink_noalloc(table.desc, meta.c, x.data_ptr(), x.stride(0), buf.data_ptr()), "call")
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_shrink_after_a_different_layer(lib):
    """A second layer in between leaves other contents in the shared array; results stay right."""
    a = wl.make_instance("decode_qkv", num_tokens=96, d_in=2048, out_sizes=[512], num_slots=9)
    b = wl.make_instance("decode_qkv", seed=11, num_tokens=64, d_in=4096, out_sizes=[256, 256], num_slots=5)
    outs = []
    for inst in (a, b, a):
        table = load_table(inst)
        meta = lib.TokenMeta(inst.num_tokens, inst.num_slots)
        meta.prepare(torch.from_numpy(inst.token_slot).cuda())
        x = to_dev(inst.x, "bf16")
        ref = _shrink(lib, table, meta, x, "workspace")
        got = _shrink(lib, table, meta, x, "noalloc")
        written = ~np.isnan(ref[0, :, 0])
        rms = float(np.sqrt(np.mean(ref[:, written] ** 2)))
        assert float(np.max(np.abs(got[:, written] - ref[:, written]))) <= TOL_BF16 * rms
        outs.append(got)
    assert np.array_equal(outs[0], outs[2], equal_nan=True)


def test_noalloc_shrink_refuses_oversized_scratch(lib):
    table = lib.SlotTable(14336, [8], 3, 128, lib.LORA_BF16)   # partial rows: 112 chunks x 128 ranks per token
    T = 512
    meta = lib.TokenMeta(T, 3)
    meta.set_num_tokens(T)
    assert lib.lora_workspace_bytes(table.desc, T) > lib.lora_noalloc_scratch_bytes()
    x = torch.zeros(T, 14336, dtype=torch.bfloat16, device="cuda")
    buf = torch.zeros(1, T, 128, device="cuda")
    n0 = lib.lora_launch_count()
    st = lib.lora_shrink_noalloc(table.desc, meta.c, x.data_ptr(), x.stride(0), buf.data_ptr())
    assert st == lib.LORA_ERANGE
    assert lib.lora_launch_count() == n0, "a refused call launched a kernel"
