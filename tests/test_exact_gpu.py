"""Exact-arithmetic parity on the GPU: small integer inputs, power-of-two scales.

With integer x, A, B, y_in and a power-of-two scale, every product and partial
sum the kernels form is an integer (times the scale) far below 2^24, so fp32
arithmetic is exact in any summation order and the fp64 oracle is exact too.
The device must then match the oracle BITWISE -- buf, y in fp32, and y in bf16
(the exact sum rounded once to nearest even). A wrong row, slice offset, rank
bound or scale cannot hide inside a tolerance here.

The batch shapes follow the definition on the handbook page
"多 LoRA 服务：分段矩阵乘与适配器调度" (section "不合并权重，批量计算"): two packed
slices, mixed ranks, an empty (reset) slot, slot-0 tokens and an id outside the
table (both "no LoRA"). Every family and path runs: BGMV, SGMV (tensor cores;
bf16 tables with r_max >= 16) and AUTO, split (shrink + expand) and fused
(lora_apply with a buf output)."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_harness import load_table, run_gpu

pytestmark = pytest.mark.gpu


def _int_instance(dtype, r_max, d_in, out_sizes, lengths, slots, num_slots, ranks, scales, seed):
    """An instance whose stored values are small integers (exact in bf16 and fp32)."""
    rng = np.random.default_rng(seed)
    enc = (lambda a: wl.bf16_bits_from_f32(a.astype(np.float32))) if dtype == "bf16" else \
        (lambda a: a.astype(np.float32))
    ads = {}
    for k, r in ranks.items():
        A = [enc(rng.integers(-3, 4, size=(d_in, r))) for _ in out_sizes]
        B = [enc(rng.integers(-3, 4, size=(r, d))) for d in out_sizes]
        ads[k] = wl.Adapter(r, scales[k], A, B)
    T = int(sum(lengths))
    x = enc(rng.integers(-4, 5, size=(T, d_in)))
    y_in = enc(rng.integers(-9, 10, size=(T, sum(out_sizes))))
    return wl.Instance(name="exact", dtype=dtype, d_in=d_in, out_sizes=list(out_sizes), num_slots=num_slots,
                       r_max=r_max, adapters=ads, req_lengths=np.asarray(lengths, np.int64),
                       req_slots=np.asarray(slots, np.int32), x=x, y_in=y_in)


def _oracle(inst):
    ads = oracle.adapters_f64(inst)
    x64 = inst.to_f32(inst.x).astype(np.float64)
    y64 = inst.to_f32(inst.y_in).astype(np.float64)
    buf, written = oracle.shrink_requests(x64, ads, inst.n_slices, inst.r_max, inst.req_lengths, inst.req_slots,
                                          inst.num_slots)
    y = oracle.expand_requests(buf, y64, ads, inst.out_sizes, inst.req_lengths, inst.req_slots, inst.num_slots)
    return buf, written, y


def _assert_exact(inst, kind, y_dtype, path, table):
    buf_ref, written, y_ref = _oracle(inst)
    assert np.all(np.abs(y_ref) < 2 ** 24) and np.all(np.abs(buf_ref[:, written]) < 2 ** 24)
    buf, y, _ = run_gpu(inst, table=table, kind=kind, y_dtype=y_dtype, path=path)
    # buf: written rows bitwise (rank tail included: exact zeros), the others untouched (NaN)
    assert np.array_equal(buf[:, written].astype(np.float64), buf_ref[:, written]), "buf differs"
    assert np.isnan(buf[:, ~written]).all(), "a no-LoRA row of buf was written"
    if y_dtype == "f32":
        want = y_ref.astype(np.float32)
    else:   # the exact sum rounded once to bf16 (nearest even)
        want = wl.bf16_bits_to_f32(wl.bf16_bits_from_f32(y_ref.astype(np.float32)))
    assert np.array_equal(y.view(np.uint32), want.view(np.uint32)), \
        f"y differs at {np.argwhere(y != want)[:5].tolist()}"


# T = 8 tokens, d_in 32, slices [16, 40], ranks 2 / 3 / 4; slot 4 holds no adapter, slot 9 is outside
# the table; scales 1/2, 2, 1/4 (powers of two).
TINY = dict(d_in=32, out_sizes=(16, 40), lengths=[2, 1, 1, 2, 1, 1], slots=[2, 0, 4, 1, 9, 3], num_slots=5,
            ranks={1: 2, 2: 3, 3: 4}, scales={1: 0.5, 2: 2.0, 3: 0.25})


@pytest.mark.parametrize("path", ["split", "apply"])
@pytest.mark.parametrize("y_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dtype,r_max,kind", [("f32", 8, "BGMV"), ("bf16", 8, "BGMV"), ("bf16", 16, "BGMV"),
                                               ("bf16", 16, "SGMV"), ("bf16", 16, "AUTO"), ("f32", 8, "AUTO")])
def test_tiny_exact(lib, dtype, r_max, kind, y_dtype, path):
    if dtype == "f32" and y_dtype == "bf16":
        pytest.skip("an fp32 table writes an fp32 y")
    inst = _int_instance(dtype, r_max, seed=r_max, **TINY)
    _assert_exact(inst, getattr(lib, f"LORA_{kind}"), y_dtype, path, load_table(inst))


def test_multichunk_multitile_exact(lib):
    """d_in 2056 (several shrink chunks of d_in rows and a ragged last one), a segment of 70 tokens
    (many token tiles and a ragged tile), four slices of ragged widths; every family, both paths."""
    lengths = [3, 70, 1, 5, 2, 9, 1, 17]
    slots = [1, 2, 0, 3, 5, 4, 2, 1]
    inst = _int_instance("bf16", 16, 2056, (1040, 24, 136, 8), lengths, slots, 6,
                         {1: 16, 2: 5, 3: 1, 4: 9}, {1: 1.0, 2: 2.0, 3: 0.5, 4: 4.0}, seed=7)
    t = load_table(inst)
    for kind in ("BGMV", "SGMV"):
        for path in ("split", "apply"):
            _assert_exact(inst, getattr(lib, f"LORA_{kind}"), "f32", path, t)


def test_auto_split_exact(lib):
    """A batch of >= LORA_AUTO_SGMV_MIN_TOKENS tokens with long and short segments: AUTO runs the long
    ones on the tensor-core family and the short ones on BGMV in one call; both bitwise."""
    rng = np.random.default_rng(12)
    lengths = [int(v) for v in rng.integers(1, 12, size=110)] + [200, 64, 63, 130]
    slots = [int(v) for v in rng.integers(0, 8, size=110)] + [3, 5, 6, 7]
    inst = _int_instance("bf16", 32, 96, (48, 32), lengths, slots, 8,
                         {k: [3, 32, 16, 7, 32, 1, 20][k - 1] for k in range(1, 8)},
                         {k: 2.0 ** (k % 3 - 1) for k in range(1, 8)}, seed=12)
    assert inst.num_tokens >= lib.LORA_AUTO_SGMV_MIN_TOKENS
    t = load_table(inst)
    for path in ("split", "apply"):
        for y_dtype in ("f32", "bf16"):
            _assert_exact(inst, lib.LORA_AUTO, y_dtype, path, t)


@pytest.mark.parametrize("dtype,r_max", [("bf16", 32), ("f32", 16), ("bf16", 64)])
def test_bgmv_grouped_expand_exact(lib, dtype, r_max):
    """The BGMV expand's narrow column chunks (at most 512 columns, so several token tiles of a unit run
    side by side on thread groups) over unit lengths 1..40, 63, 64, 65 and 130, bitwise."""
    sizes = list(range(1, 41)) + [63, 64, 65, 130]
    S = len(sizes) + 1
    rng = np.random.default_rng(r_max)
    slots = list(range(1, S))
    order = rng.permutation(len(sizes))
    lengths = [sizes[i] for i in order]
    slots = [slots[i] for i in order]
    ranks = {k: int(rng.integers(1, r_max + 1)) for k in range(1, S)}
    ranks[1] = r_max
    inst = _int_instance(dtype, r_max, 64, (1040,), lengths, slots, S, ranks,
                         {k: 2.0 ** int(rng.integers(-2, 2)) for k in range(1, S)}, seed=r_max + 1)
    t = load_table(inst)
    for path in ("split", "apply"):
        _assert_exact(inst, lib.LORA_BGMV, "f32", path, t)
