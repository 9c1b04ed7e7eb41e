"""Mixture-of-experts LoRA through the C ABI against the fp64 oracle (page
"vLLM 源码完全拆解(十八): 多 LoRA 服务", section "MoE 的 LoRA:按专家挂载、融合 kernel
与 EP 切片"): the composite slot of every (token, choice) pair bit-exactly,
then the w13 application (x rows shared by a token's top-k pairs: x_row_div =
topk) and the w2 application over the pairs, on both kernel families, with
and without expert parallelism. Tolerance as for the dense layers:
max |diff| <= 1e-2 x RMS of the oracle delta, untouched rows bitwise."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_harness import TOL_BF16, load_table, to_dev

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def test_pair_slots_bit_exact(lib):
    rng = np.random.default_rng(21)
    T, K, E, L, NL = 700, 6, 40, 10, 5
    ts = rng.integers(-1, NL + 2, T).astype(np.int32)                 # includes ids outside [0, NL]
    ids = rng.integers(-2, E + 2, (T, K)).astype(np.int32)             # includes ids outside [0, E)
    emap = np.full(E, -1, np.int32)
    emap[10:20] = np.arange(L)
    emap[33] = L + 3                                                   # an entry past the local experts
    for m in (emap, None):
        want = oracle.moe_pair_slots(ts, ids, NL, E, L if m is not None else E, m)
        got = lib.moe_pair_slots(_i32(ts), _i32(ids), NL, E, L if m is not None else E,
                                 _i32(m) if m is not None else None)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), want)


def _run_layer(lib, inst, layer, x, x_row_div, kind, path):
    """One application (w13 or w2) over the pairs; returns y [P, width] fp32 on the host."""
    t = load_table(layer)
    t.desc.x_row_div = x_row_div
    P = layer.num_tokens
    meta = lib.TokenMeta(P, layer.num_slots)
    meta.prepare(lib.moe_pair_slots(_i32(inst.token_slot), _i32(inst.topk_ids), inst.num_loras, inst.num_experts,
                                    inst.local_experts, _i32(inst.expert_map) if inst.expert_map is not None else None))
    y = torch.from_numpy(layer.to_f32(layer.y_in)).cuda()
    xd = to_dev(x, "bf16")
    if path == "apply":
        lib.apply(t, meta, xd, y, kind=kind)
    else:
        buf = torch.zeros(layer.n_slices, P, layer.r_max, dtype=torch.float32, device="cuda")
        lib.shrink(t, meta, xd, buf, kind)
        lib.expand(t, meta, buf, y, kind)
    torch.cuda.synchronize()
    assert lib.lora_query_status(meta.c) == (lib.LORA_OK, 0)
    return y.cpu().numpy()


def _check(layer, y_gpu, y_ref):
    y_in = layer.to_f32(layer.y_in)
    live = layer.token_slot > 0
    assert live.any() and not live.all()
    assert np.array_equal(y_gpu[~live].view(np.uint32), y_in[~live].view(np.uint32)), "a no-LoRA pair was touched"
    delta = (y_ref - y_in.astype(np.float64))[live]
    rms = np.sqrt(np.mean(delta ** 2))
    err = np.max(np.abs(y_gpu[live].astype(np.float64) - y_ref[live]))
    assert err <= TOL_BF16 * rms, f"err {err:.3e} > 1e-2 x RMS {rms:.3e}"


MOE_CASES = {
    # 40 tokens x top-4 over 16 experts, 8 local (expert parallel rank 1): BGMV sizes
    "ep_small": dict(num_tokens=40, hidden=512, inter=256, num_experts=16, local_experts=8, ep_rank=1, topk=4,
                     num_loras=3, r_max=16),
    # 320 tokens x top-8 = 2560 pairs over 16 experts, all local: AUTO puts the long (adapter, expert) groups on SGMV
    "all_local": dict(num_tokens=320, hidden=1024, inter=512, num_experts=16, local_experts=16, topk=8,
                      num_loras=2, r_max=32),
}


@pytest.mark.parametrize("path", ["apply", "split"])
@pytest.mark.parametrize("kind", ["BGMV", "AUTO"])
@pytest.mark.parametrize("case", sorted(MOE_CASES))
def test_moe_layer_matches_oracle(lib, case, kind, path):
    inst = wl.make_moe_instance(seed=31, **MOE_CASES[case])
    k = getattr(lib, f"LORA_{kind}")
    pair = oracle.moe_pair_slots(inst.token_slot, inst.topk_ids, inst.num_loras, inst.num_experts,
                                 inst.local_experts, inst.expert_map)
    S = inst.w13.num_slots
    # w13: the pairs read their token's row of x
    y13 = _run_layer(lib, inst, inst.w13, inst.w13.x, inst.topk, k, path)
    ref13 = oracle.moe_lora_w13(inst.w13.to_f32(inst.w13.x).astype(np.float64),
                                inst.w13.to_f32(inst.w13.y_in).astype(np.float64), pair, inst.topk,
                                oracle.adapters_f64(inst.w13), inst.w13.out_sizes, S)
    _check(inst.routed(inst.w13, pair), y13, ref13)
    # w2: one input row per pair
    y2 = _run_layer(lib, inst, inst.w2, inst.w2.x, 1, k, path)
    ref2 = oracle.moe_lora_w2(inst.w2.to_f32(inst.w2.x).astype(np.float64),
                              inst.w2.to_f32(inst.w2.y_in).astype(np.float64), pair,
                              oracle.adapters_f64(inst.w2), inst.hidden, S)
    _check(inst.routed(inst.w2, pair), y2, ref2)


def test_moe_sgmv_family_and_bad_ids(lib):
    """The w13 application on the tensor-core family alone, and pairs with bad ids
    (an adapter outside the table) counted by the metadata and left untouched."""
    inst = wl.make_moe_instance(seed=33, **MOE_CASES["all_local"])
    pair = oracle.moe_pair_slots(inst.token_slot, inst.topk_ids, inst.num_loras, inst.num_experts,
                                 inst.local_experts, inst.expert_map)
    y13 = _run_layer(lib, inst, inst.w13, inst.w13.x, inst.topk, lib.LORA_SGMV, "apply")
    ref13 = oracle.moe_lora_w13(inst.w13.to_f32(inst.w13.x).astype(np.float64),
                                inst.w13.to_f32(inst.w13.y_in).astype(np.float64), pair, inst.topk,
                                oracle.adapters_f64(inst.w13), inst.w13.out_sizes, inst.w13.num_slots)
    _check(inst.routed(inst.w13, pair), y13, ref13)
    ts = inst.token_slot.copy()
    ts[:5] = inst.num_loras + 1
    pair = lib.moe_pair_slots(_i32(ts), _i32(inst.topk_ids), inst.num_loras, inst.num_experts, inst.local_experts)
    meta = lib.TokenMeta(int(pair.numel()), inst.w13.num_slots)
    meta.prepare(pair)
    torch.cuda.synchronize()
    assert lib.lora_query_status(meta.c) == (lib.LORA_EBADSLOT, 5 * inst.topk)


@pytest.mark.parametrize("kind", ["BGMV", "SGMV", "AUTO"])
def test_moe_layer_workload_shape(lib, kind):
    """The MoE workload's own layer (hidden 7168, expert intermediate 2048, 256 experts with 8-way
    expert parallelism, top-8, r = 64, 4 adapters), reduced only in token count: 160 tokens give
    1280 pairs, above AUTO's token threshold. The w13 shrink runs 112 K blocks of 64 over d_in 7168,
    the w2 expand 7168-wide outputs. SGMV takes every (adapter, expert) group on the tensor cores."""
    inst = wl.make_moe_instance(seed=35, num_tokens=160)
    assert (inst.hidden, inst.inter, inst.num_experts, inst.local_experts, inst.topk) == (7168, 2048, 256, 32, 8)
    k = getattr(lib, f"LORA_{kind}")
    pair = oracle.moe_pair_slots(inst.token_slot, inst.topk_ids, inst.num_loras, inst.num_experts,
                                 inst.local_experts, inst.expert_map)
    S = inst.w13.num_slots
    y13 = _run_layer(lib, inst, inst.w13, inst.w13.x, inst.topk, k, "apply")
    ref13 = oracle.moe_lora_w13(inst.w13.to_f32(inst.w13.x).astype(np.float64),
                                inst.w13.to_f32(inst.w13.y_in).astype(np.float64), pair, inst.topk,
                                oracle.adapters_f64(inst.w13), inst.w13.out_sizes, S)
    _check(inst.routed(inst.w13, pair), y13, ref13)
    y2 = _run_layer(lib, inst, inst.w2, inst.w2.x, 1, k, "apply")
    ref2 = oracle.moe_lora_w2(inst.w2.to_f32(inst.w2.x).astype(np.float64),
                              inst.w2.to_f32(inst.w2.y_in).astype(np.float64), pair,
                              oracle.adapters_f64(inst.w2), inst.hidden, S)
    _check(inst.routed(inst.w2, pair), y2, ref2)
