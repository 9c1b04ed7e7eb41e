"""lora_prepare_meta against the oracle, bit-exactly, through the C ABI.

Covers the page's worked examples, random batches of many sizes, empty and
degenerate batches, out-of-range slot ids, and every workload's token->slot
mapping at full size. The work lists (a private layout the compute kernels
read) are checked against a plain restatement of their definition."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run(ra, ts, S):
    ts = np.asarray(ts, np.int32)
    T = len(ts)
    m = ra.TokenMeta(max(T, 1), S)
    m.prepare(torch.from_numpy(ts).cuda())
    torch.cuda.synchronize()
    sc = m.scalars.cpu().numpy()
    got = dict(sorted_rows=m.sorted_rows[:T].cpu().numpy(), seg_slot=m.seg_slot.cpu().numpy(),
               seg_count=m.seg_count.cpu().numpy(), seg_start=m.seg_start.cpu().numpy(),
               num_segs=int(sc[0]), no_lora=int(sc[1]), status=int(sc[2]),
               tiles=m.tiles.cpu().numpy())
    return got, m


def _work_lists(ref, S):
    """The work lists by their definition: LoRA segments (slot != 0), split at
    LORA_SGMV_MIN_ROWS when some segment has LORA_AUTO_LONG_ROWS or more (else
    all on the small list), as 8-int records {segment, slot, count, start, first 4
    rows (-1 past the count)}, unused records all -1, then the "all" records
    indexed by slot (all -1 for absent slots), then cumulative counts of
    128-row tiles over all LoRA segments and over the large ones, then per
    list the record index of every slot (-1 when absent)."""
    import rank_adapter_gb300 as ra
    n = ref["num_segs"]
    slot, cnt, start, rows = ref["seg_slot"], ref["seg_count"], ref["seg_start"], ref["sorted_rows"]
    segs = [i for i in range(n) if slot[i] != 0]
    has_long = any(cnt[i] >= ra.LORA_AUTO_LONG_ROWS for i in segs)
    large = [i for i in segs if cnt[i] >= ra.LORA_SGMV_MIN_ROWS and has_long]
    small = [i for i in segs if i not in large]

    def rec(i):
        return [i, slot[i], cnt[i], start[i]] + [int(rows[start[i] + j]) if j < cnt[i] else -1 for j in range(4)]

    def lst(L):
        out = []
        for i in L:
            out += rec(i)
        return out + [-1] * 8 * (S - len(L))

    def cum(L):
        c = [0]
        for i in L:
            c.append(c[-1] + (int(cnt[i]) + ra.LORA_SGMV_TILE_M - 1) // ra.LORA_SGMV_TILE_M)
        return c + [c[-1]] * (S + 1 - len(c))

    def slot_index(L):
        idx = [-1] * S
        for j, i in enumerate(L):
            idx[slot[i]] = j
        return idx

    def by_slot():
        out = [-1] * 8 * S
        for i in segs:
            out[8 * slot[i]:8 * slot[i] + 8] = rec(i)
        return out

    ca, cl = cum(segs), cum(large)
    w = [len(segs), len(small), len(large), ca[-1], cl[-1], 0, 0, 0] + lst(segs) + lst(small) + lst(large)
    w += by_slot() + ca + cl
    w += slot_index(segs) + slot_index(small) + slot_index(large)
    return np.asarray(w, np.int32)


def _check(ra, ts, S):
    got, _ = _run(ra, ts, S)
    ref = oracle.prepare_meta(ts, S)
    for k in ("sorted_rows", "seg_slot", "seg_count", "seg_start"):
        assert np.array_equal(got[k], ref[k]), k
    for k in ("num_segs", "no_lora", "status"):
        assert got[k] == ref[k], k
    w = _work_lists(ref, S)
    assert np.array_equal(got["tiles"][:len(w)], w), "work lists"
    return got


def test_meta_walkthrough_example(lib):
    g = json.load(open(os.path.join(GOLDEN, "meta_walkthrough.json")))["page"]
    got = _check(lib, [s + 1 for s in g["token_lora_indices"]], 3)
    assert got["sorted_rows"].tolist() == g["token_indices_sorted_by_lora_ids"]
    assert got["seg_start"][:3].tolist() == g["lora_token_start_loc"]


@pytest.mark.parametrize("T,S,case", [
    (0, 4, "rand"), (1, 4, "rand"), (1, 1, "all0"), (31, 8, "rand"), (32, 8, "rand"), (33, 8, "rand"),
    (53, 8, "rand"), (256, 64, "rand"), (1000, 2, "rand"), (1023, 1024, "distinct"), (4096, 129, "rand"),
    (777, 16, "all0"), (777, 16, "single"), (500, 9, "bad"), (20000, 33, "zipf"), (70000, 256, "rand"),
    (3000, 1024, "rand"), (64, 1024, "bad"),
])
def test_meta_random(lib, T, S, case):
    rng = np.random.default_rng(T * 7 + S)
    if case == "all0":
        ts = np.zeros(T, np.int32)
    elif case == "single":
        ts = np.full(T, S - 1, np.int32)
    elif case == "distinct":
        ts = (np.arange(T) % S).astype(np.int32)
        rng.shuffle(ts)
    elif case == "bad":
        ts = rng.integers(-5, S + 5, size=T).astype(np.int32)
        ts[:3] = [np.iinfo(np.int32).min, np.iinfo(np.int32).max, -1][:min(3, T)]
    elif case == "zipf":
        ts = (1 + rng.choice(S - 1, size=T, p=wl.zipf_probs(S - 1, 1.1))).astype(np.int32)
    else:
        ts = rng.integers(0, S, size=T).astype(np.int32)
    _check(lib, ts, S)


@pytest.mark.parametrize("name", ["toy_fp32", "decode_qkv", "prefill_gate_up", "mixed_o_proj"])
def test_meta_workloads_full_size(lib, name):
    # Only the token->slot mapping is needed: draw it the way the workload does, without weights.
    inst = wl.make_instance(name, d_in=8, out_sizes=[8]) if name != "toy_fp32" else wl.make_instance(name)
    got = _check(lib, inst.token_slot, inst.num_slots)
    assert len(got["sorted_rows"]) == inst.num_tokens


def test_meta_full_decode_mapping(lib):
    g = next(wl.full_decode_groups(groups=(("o", 8, (8,)),), layers=1, pool_size=1 << 12))
    _check(lib, g.token_slot, g.num_slots)


def test_meta_reuse_across_steps(lib):
    """One TokenMeta serves successive steps of different sizes (stale tails are rewritten)."""
    m = lib.TokenMeta(5000, 40)
    rng = np.random.default_rng(3)
    for T in (5000, 17, 0, 1200):
        ts = rng.integers(0, 40, size=T).astype(np.int32)
        m.prepare(torch.from_numpy(ts).cuda())
        ref = oracle.prepare_meta(ts, 40)
        assert np.array_equal(m.sorted_rows[:T].cpu().numpy(), ref["sorted_rows"])
        assert np.array_equal(m.seg_start.cpu().numpy(), ref["seg_start"])
        assert np.array_equal(m.seg_slot.cpu().numpy(), ref["seg_slot"])
        assert int(m.scalars[0]) == ref["num_segs"]


def test_query_status_reports_bad_ids(lib):
    ts = np.array([1, 2, 99, -4, 0, 3], np.int32)
    got, m = _run(lib, ts, 4)
    st, n = lib.lora_query_status(m.c)
    assert st == lib.LORA_EBADSLOT and n == 2
    got, m = _run(lib, np.array([1, 2, 3], np.int32), 4)
    assert lib.lora_query_status(m.c) == (lib.LORA_OK, 0)
