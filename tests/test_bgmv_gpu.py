"""BGMV shrink / expand (CUDA-core decode kernels) against the fp64 oracle.

Every case goes through the C ABI: slots written with lora_set_slot, metadata
from lora_prepare_meta, then lora_shrink and lora_expand. Tolerances are the
ones gpu_harness states (1e-2 x RMS of the oracle delta for bf16 inputs,
1e-5 for the fp32 workload; bf16 stores add half a bf16 ulp)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_harness import load_table, oracle_ref, parity, run_gpu, to_dev

pytestmark = pytest.mark.gpu


def test_toy_fp32_workload(lib):
    """The 53-token toy batch as configured: fp32, d=256, r=16, 8 slots, scale 2."""
    inst = wl.make_instance("toy_fp32")
    for kind in (lib.LORA_BGMV, lib.LORA_AUTO):
        parity(inst, kind=kind)


def test_page_toy_batch_matches_oracle(lib):
    """The page's own toy batch (adapter a in slot a+1) at the page's tolerance."""
    p = wl.toy_page_instance()
    ads = {a + 1: wl.Adapter(16, 2.0, [p["A"][a]], [p["B"][a]]) for a in range(8)}
    lengths = np.asarray(p["lengths"], np.int64)
    inst = wl.Instance(name="toy_page", dtype="f32", d_in=256, out_sizes=[256], num_slots=9, r_max=16,
                       adapters=ads, req_lengths=lengths, req_slots=np.asarray(p["adapters"]) + 1,
                       x=p["x"], y_in=(p["x"].astype(np.float64) @ p["W"].astype(np.float64)).astype(np.float32))
    buf, y, _ = parity(inst, kind=lib.LORA_BGMV)
    _, _, yref = oracle_ref(inst)
    assert np.allclose(y, yref, atol=1e-5)


@pytest.mark.parametrize("y_dtype", ["f32", "bf16"])
def test_decode_qkv_small(lib, y_dtype):
    inst = wl.make_instance("decode_qkv", num_tokens=70, d_in=1032, out_sizes=[512, 128, 1000], num_slots=13)
    parity(inst, kind=lib.LORA_BGMV, y_dtype=y_dtype)


@pytest.mark.parametrize("y_dtype", ["f32", "bf16"])
def test_decode_qkv_full_size(lib, y_dtype):
    """The decode workload at its full size: qkv 4096 -> [4096,1024,1024], r=16, 64 slots, 256 tokens."""
    inst = wl.make_instance("decode_qkv")
    parity(inst, kind=lib.LORA_BGMV, y_dtype=y_dtype)


def test_mixed_heterogeneous_ranks_small(lib):
    inst = wl.make_instance("mixed_o_proj", num_tokens=40, d_in=512, out_sizes=[256], num_slots=20)
    ranks = sorted({a.rank for a in inst.adapters.values()})
    assert len(ranks) > 1
    parity(inst, kind=lib.LORA_BGMV)


def test_mixed_full_size(lib):
    """o_proj 4096->4096, 128 slots, ranks {8,16,32,64} padded to 64, 1024 decode + 4x512 prefill."""
    inst = wl.make_instance("mixed_o_proj")
    parity(inst, kind=lib.LORA_BGMV, y_dtype="bf16")


def test_prefill_long_segments_through_bgmv(lib):
    """Long segments (many token tiles per unit) in the BGMV family."""
    inst = wl.make_instance("prefill_gate_up", num_tokens=1500, d_in=1024, out_sizes=[512, 512], num_slots=8)
    parity(inst, kind=lib.LORA_BGMV)


def test_ragged_shapes_and_strides(lib):
    """d_in not a multiple of the cluster split, widths not a multiple of the column chunk,
    padded leading dimensions, ranks 1..r_max in one table."""
    rng = np.random.default_rng(5)
    inst = wl.make_instance("decode_qkv", num_tokens=37, d_in=4104, out_sizes=[1048, 8, 2056], num_slots=9,
                            r_max=128)
    for k, r in zip(sorted(inst.adapters), [1, 7, 8, 9, 64, 100, 127, 128]):
        ad = inst.adapters[k]
        inst.adapters[k] = wl.Adapter(r, 0.75, [a[:, :r].copy() for a in ad.A], [b[:r].copy() for b in ad.B])
    parity(inst, kind=lib.LORA_BGMV, ldx_pad=24, ldy_pad=8)


def test_slot0_rows_and_negative_zero_untouched(lib):
    inst = wl.make_instance("decode_qkv", num_tokens=64, d_in=256, out_sizes=[64, 32], num_slots=5)
    y_in = inst.y_in.copy()
    rows0 = np.where(inst.token_slot == 0)[0]
    assert len(rows0) > 0
    y_in[rows0, :7] = 0x8000          # bf16 -0.0
    parity(inst, kind=lib.LORA_BGMV, y_in=y_in, y_dtype="bf16")
    parity(inst, kind=lib.LORA_BGMV, y_in=y_in, y_dtype="f32")


@pytest.mark.parametrize("case", ["all0", "single", "distinct", "bad_ids", "empty_slot", "one_token"])
def test_edge_batches(lib, case):
    inst = wl.make_instance("decode_qkv", num_tokens=96, d_in=512, out_sizes=[256, 64], num_slots=17)
    T = inst.num_tokens
    rng = np.random.default_rng(1)
    if case == "all0":
        ts = np.zeros(T, np.int32)
    elif case == "single":
        ts = np.full(T, 7, np.int32)
    elif case == "distinct":
        ts = (1 + np.arange(T) % 16).astype(np.int32)
    elif case == "bad_ids":
        ts = rng.integers(-3, 20, size=T).astype(np.int32)
    elif case == "empty_slot":
        del inst.adapters[5]          # slot 5 is never written: rank 0, zero delta
        ts = rng.integers(0, 17, size=T).astype(np.int32)
        ts[:10] = 5
    else:
        ts = np.zeros(T, np.int32)
        ts[33] = 3
    parity(inst, kind=lib.LORA_BGMV, token_slot=ts)


def test_zero_tokens(lib):
    inst = wl.make_instance("decode_qkv", num_tokens=4, d_in=64, out_sizes=[64], num_slots=4)
    t = load_table(inst)
    m = lib.TokenMeta(8, 4)
    m.prepare(torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert int(m.scalars[0]) == 0 and int(m.scalars[1]) == 1
    x = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    buf = torch.zeros(1, 0, 16, device="cuda")
    lib.shrink(t, m, x, buf, lib.LORA_BGMV)
    lib.expand(t, m, buf, y, lib.LORA_BGMV)
    torch.cuda.synchronize()


def test_reset_slot_gives_zero_delta(lib):
    inst = wl.make_instance("decode_qkv", num_tokens=32, d_in=256, out_sizes=[128], num_slots=4)
    t = load_table(inst)
    for k in range(1, 4):
        t.reset_slot(k)
    ts = np.full(32, 2, np.int32)
    buf, y, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV, token_slot=ts)
    assert np.all(buf == 0.0)
    y_in = inst.to_f32(inst.y_in)
    assert np.array_equal(y, y_in + 0.0)


def test_deterministic_and_permutation_invariant(lib):
    inst = wl.make_instance("decode_qkv", num_tokens=128, d_in=2048, out_sizes=[512, 256], num_slots=9)
    t = load_table(inst)
    b1, y1, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV)
    b2, y2, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV)
    assert np.array_equal(b1, b2, equal_nan=True) and np.array_equal(y1, y2)
    perm = np.random.default_rng(9).permutation(inst.num_tokens)
    inst_p = wl.Instance(name="perm", dtype=inst.dtype, d_in=inst.d_in, out_sizes=inst.out_sizes,
                         num_slots=inst.num_slots, r_max=inst.r_max, adapters=inst.adapters,
                         req_lengths=np.ones(inst.num_tokens, np.int64), req_slots=inst.token_slot[perm],
                         x=inst.x[perm], y_in=inst.y_in[perm])
    b3, y3, _ = run_gpu(inst_p, table=t, kind=lib.LORA_BGMV)
    assert np.array_equal(y3, y1[perm])
    assert np.array_equal(b3, b1[:, perm], equal_nan=True)


def test_high_rank_rows_independent_of_slot_sharing(lib):
    """A high-rank layer (r_max 64: expand column chunks narrower than the block, so a
    slot's token tiles run side by side, up to four at once): each token's y row is
    bitwise the row it gets in a batch where its slot holds far fewer tokens."""
    lengths = [1] * 9 + [14, 6, 23, 2, 9, 40]
    full = wl.make_instance("mixed_o_proj", req_lengths=lengths, d_in=1024, out_sizes=[256], num_slots=6)
    t = load_table(full)
    for path in ("apply", "split"):
        _, y_all, _ = run_gpu(full, table=t, kind=lib.LORA_BGMV, y_dtype="f32", path=path)
        rows = np.arange(0, full.num_tokens, 3)
        solo = wl.make_instance("mixed_o_proj", req_lengths=[1] * len(rows), d_in=1024, out_sizes=[256],
                                num_slots=6)
        solo.adapters = full.adapters
        solo.req_slots = full.token_slot[rows].copy()
        solo.x = full.x[rows].copy()
        solo.y_in = full.y_in[rows].copy()
        assert np.bincount(solo.token_slot).max() < np.bincount(full.token_slot).max()
        _, y_s, _ = run_gpu(solo, table=t, kind=lib.LORA_BGMV, y_dtype="f32", path=path)
        assert np.array_equal(y_s.view(np.uint32), y_all[rows].view(np.uint32)), path


# ----------------------------------------------------------------------------- fused lora_apply

APPLY_CASES = {
    "toy_fp32": lambda: wl.make_instance("toy_fp32"),
    "decode_small": lambda: wl.make_instance("decode_qkv", num_tokens=70, d_in=1032, out_sizes=[512, 128, 1000],
                                             num_slots=13),
    "decode_full": lambda: wl.make_instance("decode_qkv"),
    "mixed_small": lambda: wl.make_instance("mixed_o_proj", num_tokens=40, d_in=512, out_sizes=[256], num_slots=20),
    "long_segments": lambda: wl.make_instance("prefill_gate_up", num_tokens=700, d_in=2048, out_sizes=[3000, 520],
                                              num_slots=6),
    "down_proj_like": lambda: wl.make_instance("decode_qkv", num_tokens=48, d_in=14336, out_sizes=[4096],
                                               num_slots=9),
}


@pytest.mark.parametrize("name", sorted(APPLY_CASES))
@pytest.mark.parametrize("y_dtype", ["f32", "bf16"])
def test_apply_matches_oracle_and_split_path(lib, name, y_dtype):
    inst = APPLY_CASES[name]()
    if inst.dtype == "f32" and y_dtype == "bf16":
        pytest.skip("fp32 tables store fp32 outputs")
    t = load_table(inst)
    buf_a, y_a, _ = parity(inst, kind=lib.LORA_BGMV, y_dtype=y_dtype, table=t, path="apply")
    buf_s, y_s, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV, y_dtype=y_dtype, path="split")
    assert np.array_equal(y_a.view(np.uint32), y_s.view(np.uint32)), "fused and split results differ"
    assert np.array_equal(buf_a, buf_s, equal_nan=True)


def test_apply_without_buffer(lib):
    inst = wl.make_instance("decode_qkv", num_tokens=64, d_in=1024, out_sizes=[256, 64], num_slots=9)
    t = load_table(inst)
    _, y_ref, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV, path="apply")
    T = inst.num_tokens
    m = lib.TokenMeta(T, inst.num_slots)
    m.prepare(torch.from_numpy(inst.token_slot).cuda())
    x = to_dev(inst.x, "bf16")
    y = torch.from_numpy(inst.to_f32(inst.y_in)).cuda()
    lib.apply(t, m, x, y, buf=None, kind=lib.LORA_BGMV)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), y_ref)
