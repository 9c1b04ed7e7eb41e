"""lora_prepare_meta_unshared: the metadata pass that writes its outputs
without waiting for the previous call's kernels (the caller promises they do
not read this metadata buffer, e.g. two buffers alternating between steps).

Its outputs must equal lora_prepare_meta's bit for bit, and a serving-style
sequence that alternates two metadata buffers between steps, each step a
metadata pass and a fused apply queued back to back with no host sync, must
match the oracle at every step."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_harness import TOL_BF16, check_parity, load_table, oracle_ref, to_dev

pytestmark = pytest.mark.gpu


def _outputs(m, T):
    sc = m.scalars.cpu().numpy()
    return dict(sorted_rows=m.sorted_rows[:T].cpu().numpy(), seg_slot=m.seg_slot.cpu().numpy(),
                seg_count=m.seg_count.cpu().numpy(), seg_start=m.seg_start.cpu().numpy(),
                scalars=sc[:3].copy(), tiles=m.tiles.cpu().numpy())


@pytest.mark.parametrize("T,S,seed", [(1, 2, 0), (53, 8, 1), (256, 64, 2), (3000, 128, 3), (0, 5, 4)])
def test_unshared_outputs_equal_prepare_meta(lib, T, S, seed):
    rng = np.random.default_rng(seed)
    ts = rng.integers(0, S, size=T).astype(np.int32)
    if T > 2:
        ts[1] = S + 3      # an out-of-range id: counted in status, treated as slot 0
    a = lib.TokenMeta(max(T, 1), S)
    b = lib.TokenMeta(max(T, 1), S)
    b.tiles.fill_(-7)      # stale contents must be overwritten exactly as by the normal pass
    dev = torch.from_numpy(ts).cuda()
    a.prepare(dev)
    b.prepare(dev, unshared=True)
    torch.cuda.synchronize()
    ga, gb = _outputs(a, T), _outputs(b, T)
    for k in ga:
        assert np.array_equal(ga[k], gb[k]), k


def test_alternating_buffers_every_step_matches_oracle(lib):
    """Six decode steps of a qkv-shaped layer, each with its own token->slot
    map, metadata in two buffers used by alternate steps; the first step uses
    the normal pass (nothing is known about what ran before it)."""
    base = wl.make_instance("decode_qkv", d_in=512, out_sizes=[512, 128, 128], num_slots=16, num_tokens=96)
    table = load_table(base)
    T = base.num_tokens
    metas = [lib.TokenMeta(T, base.num_slots), lib.TokenMeta(T, base.num_slots)]
    x = to_dev(base.x, "bf16")
    steps = []
    rng = np.random.default_rng(11)
    for i in range(6):
        ts = rng.integers(0, base.num_slots, size=T).astype(np.int32)
        y = to_dev(base.y_in, "bf16")
        buf = torch.full((base.n_slices, T, base.r_max), float("nan"), dtype=torch.float32, device="cuda")
        m = metas[i % 2]
        m.prepare(torch.from_numpy(ts).cuda(), unshared=i > 0)
        lib.apply(table, m, x, y, buf=buf, kind=lib.LORA_AUTO)
        steps.append((ts, y, buf))
    torch.cuda.synchronize()
    for ts, y, buf in steps:
        bref, written, yref = oracle_ref(base, token_slot=ts)
        check_parity(base, buf.cpu().numpy(), y.float().cpu().numpy(), bref, written, yref, TOL_BF16,
                     y_dtype="bf16", token_slot=ts)


def test_back_to_back_steps_without_copies_in_between(lib):
    """The same, with every step's token->slot map written before the loop
    (one metadata buffer per step), so the loop queues only the metadata
    passes and the applies and each unshared pass runs beside the previous
    step's expand."""
    base = wl.make_instance("decode_qkv", d_in=1024, out_sizes=[1024, 256, 256], num_slots=24, num_tokens=160)
    table = load_table(base)
    T = base.num_tokens
    x = to_dev(base.x, "bf16")
    rng = np.random.default_rng(12)
    runs = []
    for i in range(8):
        ts = rng.integers(0, base.num_slots, size=T).astype(np.int32)
        m = lib.TokenMeta(T, base.num_slots)
        m.token_slot[:T].copy_(torch.from_numpy(ts).cuda())
        m.set_num_tokens(T)
        runs.append((ts, m, to_dev(base.y_in, "bf16"),
                     torch.full((base.n_slices, T, base.r_max), float("nan"), dtype=torch.float32, device="cuda")))
    torch.cuda.synchronize()
    for i, (ts, m, y, buf) in enumerate(runs):
        if i == 0:
            lib.check(lib.lora_prepare_meta(m.c, None), "prepare_meta")
        else:
            lib.check(lib.lora_prepare_meta_unshared(m.c, None), "prepare_meta_unshared")
        lib.apply(table, m, x, y, buf=buf, kind=lib.LORA_AUTO)
    torch.cuda.synchronize()
    for ts, m, y, buf in runs:
        bref, written, yref = oracle_ref(base, token_slot=ts)
        check_parity(base, buf.cpu().numpy(), y.float().cpu().numpy(), bref, written, yref, TOL_BF16,
                     y_dtype="bf16", token_slot=ts)
