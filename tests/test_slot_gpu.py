"""lora_set_slot / lora_reset_slot: the stacked slot buffers hold exactly the
adapter's values with a zero rank tail, other slots are untouched, a slice
whose sources are both NULL is zeroed, and rank / scale are recorded.
Integer-exact: the buffers are compared bit for bit."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_harness import to_dev

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rank,r_max", [(16, 16), (5, 16), (8, 64), (1, 8), (100, 128)])
def test_set_slot_layout(lib, dtype, rank, r_max):
    rng = np.random.default_rng(rank * 131 + r_max)
    d_in, outs, S = 48, [24, 8, 40], 6
    ldt = lib.LORA_BF16 if dtype == "bf16" else lib.LORA_F32
    t = lib.SlotTable(d_in, outs, S, r_max, ldt)
    mk = lambda shape: (wl.bf16_bits_from_f32(rng.standard_normal(shape).astype(np.float32)) if dtype == "bf16"
                        else rng.standard_normal(shape).astype(np.float32))
    A = [mk((d_in, rank)) for _ in outs]
    B = [mk((rank, d)) for d in outs]
    # fill slot 4 with something first, to see that slot 3's write does not touch it
    A4 = [mk((d_in, rank)) for _ in outs]
    B4 = [mk((rank, d)) for d in outs]
    t.set_slot(4, rank, 0.5, [to_dev(a, dtype) for a in A4], [to_dev(b, dtype) for b in B4])
    before4 = [_bits(a[4]).copy() for a in t.A] + [_bits(b[4]).copy() for b in t.B]
    src = ([to_dev(a, dtype) for a in A], [to_dev(b, dtype) for b in B])
    t.set_slot(3, rank, 1.75, *src)
    torch.cuda.synchronize()
    for s in range(len(outs)):
        exp_a = np.zeros((d_in, r_max), A[s].dtype)
        exp_a[:, :rank] = A[s]
        exp_b = np.zeros((r_max, outs[s]), B[s].dtype)
        exp_b[:rank] = B[s]
        ga, gb = _bits(t.A[s][3]), _bits(t.B[s][3])
        view = np.int16 if dtype == "bf16" else np.uint32
        assert np.array_equal(ga, exp_a.view(view)), f"A slice {s}"
        assert np.array_equal(gb, exp_b.view(view)), f"B slice {s}"
        assert not _bits(t.A[s][0]).any() and not _bits(t.B[s][0]).any(), "slot 0 must stay zero"
    after4 = [_bits(a[4]) for a in t.A] + [_bits(b[4]) for b in t.B]
    assert all(np.array_equal(x, y) for x, y in zip(before4, after4))
    assert t.slot_rank.cpu().tolist() == [0, 0, 0, rank, rank, 0]
    assert t.slot_scale.cpu().tolist() == [0, 0, 0, 1.75, 0.5, 0]

    # a slice the adapter did not train: both sources NULL -> zeroed
    t.set_slot(3, rank, 1.0, [src[0][0], None, src[0][2]], [src[1][0], None, src[1][2]])
    torch.cuda.synchronize()
    assert not _bits(t.A[1][3]).any() and not _bits(t.B[1][3]).any()
    assert _bits(t.A[0][3]).any()

    t.reset_slot(3)
    torch.cuda.synchronize()
    for s in range(len(outs)):
        assert not _bits(t.A[s][3]).any() and not _bits(t.B[s][3]).any()
    assert t.slot_rank.cpu().tolist()[3] == 0 and t.slot_scale.cpu().tolist()[3] == 0.0
    assert all(np.array_equal(x, y) for x, y in zip(before4, [_bits(a[4]) for a in t.A] + [_bits(b[4]) for b in t.B]))


def test_set_slot_rejects_bad_arguments(lib):
    t = lib.SlotTable(16, [8], 4, 8, lib.LORA_BF16)
    a = torch.zeros(16, 8, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    assert lib.lora_set_slot(t.desc, 0, 8, 1.0, [a], [b]) == lib.LORA_ERANGE
    assert lib.lora_set_slot(t.desc, 4, 8, 1.0, [a], [b]) == lib.LORA_ERANGE
    assert lib.lora_set_slot(t.desc, 1, 9, 1.0, [a], [b]) == lib.LORA_ERANGE
    assert lib.lora_set_slot(t.desc, 1, 8, 1.0, [a], [None]) == lib.LORA_EINVAL
    assert lib.lora_reset_slot(t.desc, 0) == lib.LORA_ERANGE
