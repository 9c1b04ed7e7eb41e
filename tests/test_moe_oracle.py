"""Pins of the mixture-of-experts oracle (page "vLLM 源码完全拆解(十八): 多 LoRA 服务",
section "MoE 的 LoRA:按专家挂载、融合 kernel 与 EP 切片") against facts that do not
come from the oracle itself: the composite slot layout is a bijection onto the
table, expert-parallel ranks partition the pairs, a single expert with top-1
routing is the dense multi-LoRA delta (pinned separately), relabelling the
experts changes nothing, the ranks' deltas add up to the unsharded delta, and
exact integer brute force on tiny shapes."""
from fractions import Fraction

import numpy as np

import oracle


def _rand_adapters(rng, slots, d_in, out_sizes, r):
    return {int(k): (r, float(rng.choice([0.5, 1.0, 2.0])),
                     [rng.standard_normal((d_in, r)) for _ in out_sizes],
                     [rng.standard_normal((r, w)) for w in out_sizes]) for k in slots}


def test_pair_slots_are_a_bijection_onto_the_table():
    NL, E = 3, 5
    ts = np.repeat(np.arange(1, NL + 1), E).astype(np.int32)          # every (adapter, expert) once
    ids = np.tile(np.arange(E), NL).reshape(-1, 1).astype(np.int32)
    got = oracle.moe_pair_slots(ts, ids, NL, E, E)
    assert sorted(got.tolist()) == list(range(1, 1 + NL * E))
    # the adapter is recovered from the slot's block, the expert from its offset
    assert np.array_equal((got - 1) // E + 1, ts) and np.array_equal((got - 1) % E, ids[:, 0])


def test_pair_slots_special_cases():
    ts = np.array([0, 2, 4, -1, 1, 1], np.int32)
    ids = np.array([[1, 0], [3, 2], [0, 0], [0, 1], [4, 0], [-1, 2]], np.int32)   # E = 4
    emap = np.array([0, 1, -1, 9], np.int32)                                         # expert 3 maps past L = 2
    got = oracle.moe_pair_slots(ts, ids, 3, 4, 2, emap).reshape(6, 2)
    assert got[0].tolist() == [0, 0]            # slot 0: no delta
    assert got[1].tolist() == [-1, 0]           # map entry past the local experts; expert 2 not local
    assert got[2].tolist() == [-1, -1]          # adapter above num_loras
    assert got[3].tolist() == [-1, -1]          # negative adapter
    assert got[4].tolist() == [-1, 1]           # expert id outside [0, E); expert 0 -> slot 1
    assert got[5].tolist() == [-1, 0]           # negative expert id; expert 2 not local


def test_expert_parallel_ranks_partition_the_pairs():
    rng = np.random.default_rng(3)
    T, K, E, R, NL = 50, 4, 16, 4, 3
    L = E // R
    ts = rng.integers(0, NL + 1, T).astype(np.int32)
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)
    live = np.zeros(T * K, np.int64)
    for rank in range(R):
        emap = np.full(E, -1, np.int32)
        emap[rank * L:(rank + 1) * L] = np.arange(L)
        got = oracle.moe_pair_slots(ts, ids, NL, E, L, emap)
        live += got > 0
    lora = np.repeat(ts > 0, K)
    assert np.array_equal(live, lora.astype(np.int64))   # each LoRA pair lives on exactly one rank


def test_single_expert_top1_is_the_dense_delta():
    """E = 1, top-1: composite slot = adapter slot, and both applications equal the
    dense per-request oracle on the same tables (pinned in test_oracle_pins)."""
    rng = np.random.default_rng(5)
    T, H, I, NL, r = 9, 24, 16, 3, 4
    ts = np.array([1, 0, 2, 2, 3, 1, 0, 3, 1], np.int32)
    ids = np.zeros((T, 1), np.int32)
    pair = oracle.moe_pair_slots(ts, ids, NL, 1, 1)
    assert np.array_equal(pair, ts)
    ad13 = _rand_adapters(rng, range(1, NL + 1), H, [I, I], r)
    ad2 = _rand_adapters(rng, range(1, NL + 1), I, [H], r)
    x, h1, h2, h3 = (rng.standard_normal(s) for s in ((T, H), (T, 2 * I), (T, I), (T, H)))
    lengths = np.ones(T, np.int64)
    y13 = oracle.moe_lora_w13(x, h1, pair, 1, ad13, [I, I], NL + 1)
    y13_dense = oracle.apply_requests(x, h1, ad13, [I, I], r, lengths, ts, NL + 1)
    assert np.allclose(y13, y13_dense, rtol=1e-12, atol=1e-12)
    y2 = oracle.moe_lora_w2(h2, h3, pair, ad2, H, NL + 1)
    y2_dense = oracle.apply_requests(h2, h3, ad2, [H], r, lengths, ts, NL + 1)
    assert np.allclose(y2, y2_dense, rtol=1e-12, atol=1e-12)


def _setup(rng, T=12, K=3, E=6, NL=2, H=20, I=12, r=4):
    ts = rng.integers(0, NL + 1, T).astype(np.int32)
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)
    per = {(a, e): _rand_adapters(rng, [0], H, [I, I], r)[0] for a in range(1, NL + 1) for e in range(E)}
    x, h1 = rng.standard_normal((T, H)), rng.standard_normal((T * K, 2 * I))
    return ts, ids, per, x, h1


def _table(per, NL, L, local_of):
    """Composite table of the experts with local index local_of[e] >= 0."""
    tab = {}
    for (a, e), ad in per.items():
        j = local_of[e]
        if j >= 0:
            tab[1 + (a - 1) * L + j] = ad
    return tab


def test_expert_relabelling_changes_nothing():
    rng = np.random.default_rng(7)
    T, K, E, NL, I = 12, 3, 6, 2, 12
    ts, ids, per, x, h1 = _setup(rng, T, K, E, NL, I=I)
    ident = np.arange(E)
    y0 = oracle.moe_lora_w13(x, h1, oracle.moe_pair_slots(ts, ids, NL, E, E), K, _table(per, NL, E, ident),
                             [I, I], 1 + NL * E)
    perm = rng.permutation(E)                       # expert e is called perm[e] from now on
    per_p = {(a, int(perm[e])): ad for (a, e), ad in per.items()}
    ids_p = perm[ids].astype(np.int32)
    y1 = oracle.moe_lora_w13(x, h1, oracle.moe_pair_slots(ts, ids_p, NL, E, E), K, _table(per_p, NL, E, ident),
                             [I, I], 1 + NL * E)
    assert np.allclose(y0, y1, rtol=1e-12, atol=1e-12)


def test_expert_parallel_deltas_add_up_to_the_unsharded_delta():
    rng = np.random.default_rng(9)
    T, K, E, NL, I, R = 12, 3, 6, 2, 12, 3
    ts, ids, per, x, h1 = _setup(rng, T, K, E, NL, I=I)
    full = oracle.moe_lora_w13(x, h1, oracle.moe_pair_slots(ts, ids, NL, E, E), K,
                               _table(per, NL, E, np.arange(E)), [I, I], 1 + NL * E)
    L = E // R
    total = np.zeros_like(h1)
    for rank in range(R):
        emap = np.full(E, -1, np.int64)
        emap[rank * L:(rank + 1) * L] = np.arange(L)
        y = oracle.moe_lora_w13(x, h1, oracle.moe_pair_slots(ts, ids, NL, E, L, emap), K,
                                _table(per, NL, L, emap), [I, I], 1 + NL * L)
        total += y - h1
    assert np.allclose(h1 + total, full, rtol=1e-12, atol=1e-12)


def test_gathered_apply_exact_integer_brute_force():
    """Integer-valued inputs: the fp64 result is exact and equals Fraction arithmetic."""
    rng = np.random.default_rng(11)
    T, K, E, NL, H, I, r = 4, 2, 3, 2, 5, 3, 2
    ts = np.array([1, 0, 2, 1], np.int32)
    ids = np.array([[0, 2], [1, 0], [2, 1], [1, 2]], np.int32)
    pair = oracle.moe_pair_slots(ts, ids, NL, E, E)
    tab = {s: (r, 2.0, [rng.integers(-3, 4, (H, r)).astype(np.float64) for _ in range(2)],
               [rng.integers(-3, 4, (r, I)).astype(np.float64) for _ in range(2)]) for s in range(1, 1 + NL * E)}
    x = rng.integers(-4, 5, (T, H)).astype(np.float64)
    h1 = rng.integers(-4, 5, (T * K, 2 * I)).astype(np.float64)
    got = oracle.moe_lora_w13(x, h1, pair, K, tab, [I, I], 1 + NL * E)
    for p in range(T * K):
        t, s = p // K, int(pair[p])
        for sl in range(2):
            for n in range(I):
                want = Fraction(int(h1[p, sl * I + n]))
                if s > 0:
                    rr, sc, A, B = tab[s]
                    for k in range(rr):
                        u = Fraction(sc) * sum(Fraction(int(x[t, j])) * Fraction(int(A[sl][j, k])) for j in range(H))
                        want += u * Fraction(int(B[sl][k, n]))
                assert Fraction(got[p, sl * I + n]) == want, (p, sl, n)
