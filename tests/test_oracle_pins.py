"""Pins of the CPU oracle to facts that do not come from the oracle itself.

* values the pages print (worked metadata examples, the toy batch's verdict
  and counts) -- fixtures under tests/golden/, each with its citation;
* independent library routines (numpy's stable argsort / unique / cumsum for
  the metadata; torch's bf16 conversion for the input encoding);
* exact integer brute force on tiny shapes, written as explicit Python loops;
* closed forms and invariants: merged weights W + sAB, a single adapter's
  s*X*A*B, zero B, reset slots, untouched slot-0 rows, rank padding,
  request permutation;
* planted mistakes in the oracle, which the brute-force pin must catch.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import lora_oracle as lo
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- metadata

def test_meta_walkthrough_from_page():
    g = _golden("meta_walkthrough.json")["page"]
    token_slot = [s + 1 for s in g["token_lora_indices"]]       # -1 -> 0, k -> k+1
    m = oracle.prepare_meta(token_slot, num_slots=3)
    n = m["num_segs"]
    assert m["sorted_rows"].tolist() == g["token_indices_sorted_by_lora_ids"]
    assert m["seg_slot"][:n].tolist() == [s + 1 for s in g["lora_ids"]]
    assert m["seg_count"][:n].tolist() == g["num_tokens_per_lora"]
    assert m["seg_start"][:n + 1].tolist() == g["lora_token_start_loc"]
    assert m["no_lora"] == 0 and m["status"] == 0


def test_meta_counts_to_starts_from_page():
    g = _golden("meta_segments.json")["page"]
    counts = g["num_tokens_per_lora"]
    rng = np.random.default_rng(7)
    token_slot = np.repeat(np.arange(len(counts)), counts)
    rng.shuffle(token_slot)
    m = oracle.prepare_meta(token_slot, num_slots=len(counts))
    assert m["seg_count"][:m["num_segs"]].tolist() == counts
    assert m["seg_start"][:m["num_segs"] + 1].tolist() == g["lora_token_start_loc"]


def _meta_by_numpy(token_slot, num_slots):
    ts = np.asarray(token_slot, np.int64)
    bad = (ts < 0) | (ts >= num_slots)
    key = np.where(bad, 0, ts)
    order = np.argsort(key, kind="stable")
    ids, counts = np.unique(key, return_counts=True)
    starts = np.concatenate([[0], np.cumsum(counts)]) if len(ids) else np.zeros(1, np.int64)
    return order, ids, counts, starts, int(bad.sum())


@pytest.mark.parametrize("T,num_slots,case", [
    (0, 4, "empty"), (1, 4, "one"), (53, 8, "rand"), (300, 64, "rand"), (257, 3, "rand"),
    (100, 16, "all0"), (100, 16, "single"), (64, 65, "distinct"), (200, 9, "bad"),
    (5000, 128, "rand"), (1000, 1, "all0"),
])
def test_meta_matches_numpy_routines(T, num_slots, case):
    rng = np.random.default_rng(T * 131 + num_slots)
    if case == "all0":
        ts = np.zeros(T, np.int32)
    elif case == "single":
        ts = np.full(T, num_slots - 1, np.int32)
    elif case == "distinct":
        ts = rng.permutation(np.arange(1, T + 1) % num_slots).astype(np.int32)
    elif case == "bad":
        ts = rng.integers(-3, num_slots + 4, size=T).astype(np.int32)
    else:
        ts = rng.integers(0, num_slots, size=T).astype(np.int32)
    m = oracle.prepare_meta(ts, num_slots)
    order, ids, counts, starts, bad = _meta_by_numpy(ts, num_slots)
    n = m["num_segs"]
    assert n == len(ids)
    assert np.array_equal(m["sorted_rows"], order)
    assert np.array_equal(m["seg_slot"][:n], ids)
    assert np.array_equal(m["seg_count"][:n], counts)
    assert np.array_equal(m["seg_start"][:n + 1], starts)
    assert np.all(m["seg_slot"][n:] == -1) and np.all(m["seg_count"][n:] == 0)
    assert np.all(m["seg_start"][n + 1:] == T)
    assert len(m["seg_slot"]) == num_slots and len(m["seg_start"]) == num_slots + 1
    assert m["status"] == bad
    assert m["no_lora"] == int(np.all(np.where((ts < 0) | (ts >= num_slots), 0, ts) == 0))


# ----------------------------------------------------------------------------- the page's toy batch

def test_toy_batch_verdict_and_counts():
    """The three formulations on the page agree, and the printed counts hold."""
    import torch
    g = _golden("toy_verdict.json")
    p = wl.toy_page_instance()
    W, A, B, x = p["W"], p["A"], p["B"], p["x"]
    lengths, adapters, scale = p["lengths"], p["adapters"], p["scale"]
    assert lengths == g["inputs"]["lengths"] and adapters == g["inputs"]["adapters"]
    T = sum(lengths)
    # The oracle under this library's slot convention: adapter a lives in slot a + 1.
    ads = {a + 1: (16, scale, [A[a].astype(np.float64)], [B[a].astype(np.float64)]) for a in range(8)}
    req_slots = [a + 1 for a in adapters]
    x64 = x.astype(np.float64)
    y_base = x64 @ W.astype(np.float64)
    y_oracle = oracle.apply_requests(x64, y_base, ads, [256], 16, lengths, req_slots, num_slots=9)

    # This test's own per-token (gather) and per-segment (sorted) formulations, in fp32 as on the page.
    xt, Wt, At, Bt = (torch.from_numpy(v) for v in (x, W, A, B))
    tok = torch.tensor([a for a, n in zip(adapters, lengths) for _ in range(n)])
    gathered = torch.stack([(xt[t] @ At[tok[t]]) @ Bt[tok[t]] for t in range(T)])
    y_tok = xt @ Wt + scale * gathered
    order = torch.sort(tok, stable=True).indices
    seg_out = torch.zeros(T, 256)
    for a in torch.unique(tok).tolist():
        rows = order[tok[order] == a]
        seg_out[rows] = scale * (xt[rows] @ At[a]) @ Bt[a]
    y_seg = xt @ Wt + seg_out

    ref = torch.from_numpy(y_oracle).float()
    atol = g["printed"]["allclose_atol"]
    assert torch.allclose(y_tok, ref, atol=atol) == g["printed"]["bgmv_matches_per_request"]
    assert torch.allclose(y_seg, ref, atol=atol) == g["printed"]["sgmv_matches_per_request"]
    # printed counts: 53 base rows, 6 per-request calls, 4 segments
    assert T == g["printed"]["base_gemm_rows"]
    assert len(lengths) == g["printed"]["per_request_calls"]
    m = oracle.prepare_meta(np.repeat(req_slots, lengths), num_slots=9)
    assert m["num_segs"] == g["printed"]["sgmv_segments"]
    # Under the slot-0-is-no-LoRA reading the same ids give one no-LoRA segment + 3 LoRA segments.
    m0 = oracle.prepare_meta(np.repeat(adapters, lengths), num_slots=8)
    assert m0["num_segs"] == 4
    assert m0["seg_slot"][:4].tolist() == [0, 3, 5, 7]
    assert m0["seg_count"][:4].tolist() == [1, 38, 2, 12]
    assert m0["seg_start"][:5].tolist() == [0, 1, 39, 41, 53]


# ----------------------------------------------------------------------------- exact brute force

def _tiny_problem(seed):
    rng = np.random.default_rng(seed)
    num_slots, d_in, out_sizes, r_max = 5, 5, [3, 6], 4
    ranks = {1: 2, 2: 3, 3: 4}           # slot 4 is an empty (reset) slot
    scales = {1: 0.5, 2: 2.0, 3: 0.25}
    ads = {}
    for k, r in ranks.items():
        A = [rng.integers(-3, 4, size=(d_in, r)).astype(np.float64) for _ in out_sizes]
        B = [rng.integers(-3, 4, size=(r, d)).astype(np.float64) for d in out_sizes]
        ads[k] = (r, scales[k], A, B)
    lengths = [2, 1, 3, 1, 2, 1, 1]
    slots = [2, 0, 1, 3, 4, 7, 2]        # 7 is outside the table -> no LoRA
    T = sum(lengths)
    x = rng.integers(-4, 5, size=(T, d_in)).astype(np.float64)
    y_in = rng.integers(-9, 10, size=(T, sum(out_sizes))).astype(np.float64)
    return num_slots, d_in, out_sizes, r_max, ads, lengths, slots, x, y_in


def _brute(num_slots, d_in, out_sizes, r_max, ads, lengths, slots, x, y_in):
    """Exact rational arithmetic, element by element."""
    T = sum(lengths)
    tok = [s for s, n in zip(slots, lengths) for _ in range(n)]
    y = [[Fraction(int(v)) for v in row] for row in y_in]
    buf = {}
    for t in range(T):
        a = tok[t]
        if a <= 0 or a >= num_slots:
            continue
        r, sc, A, B = ads.get(a, (0, 0.0, None, None))
        off = 0
        for s, d in enumerate(out_sizes):
            u = []
            for k in range(r_max):
                if k < r:
                    acc = Fraction(0)
                    for j in range(d_in):
                        acc += Fraction(int(x[t][j])) * Fraction(int(A[s][j][k]))
                    u.append(Fraction(sc) * acc)
                else:
                    u.append(Fraction(0))
            buf[(s, t)] = u
            for n in range(d):
                acc = Fraction(0)
                for k in range(r):
                    acc += u[k] * Fraction(int(B[s][k][n]))
                y[t][off + n] = Fraction(int(y_in[t][off + n])) + acc
            off += d
    return buf, y


def _check_against_brute(seed=0):
    num_slots, d_in, out_sizes, r_max, ads, lengths, slots, x, y_in = _tiny_problem(seed)
    buf_ref, y_ref = _brute(num_slots, d_in, out_sizes, r_max, ads, lengths, slots, x, y_in)
    buf, written = oracle.shrink_requests(x, ads, len(out_sizes), r_max, lengths, slots, num_slots)
    y = oracle.apply_requests(x, y_in, ads, out_sizes, r_max, lengths, slots, num_slots)
    T = sum(lengths)
    for t in range(T):
        for s in range(len(out_sizes)):
            if (s, t) in buf_ref:
                assert written[t]
                assert [Fraction(v) for v in buf[s, t]] == buf_ref[(s, t)]
            else:
                assert not written[t]
        assert [Fraction(v) for v in y[t]] == y_ref[t]


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_bruteforce_exact_integers(seed):
    _check_against_brute(seed)


@pytest.mark.parametrize("mutant", ["scale_sign", "slot0_is_real", "rows_off_by_one",
                                    "tail_not_zeroed", "slice_offset"])
def test_planted_mistakes_fail_the_pin(monkeypatch, mutant):
    """Each planted mistake in the oracle must make the brute-force pin fail."""
    if mutant == "scale_sign":
        orig = lo._live_adapter
        monkeypatch.setattr(lo, "_live_adapter",
                            lambda ads, a, n: (lambda v: v if v is None else (v[0], -v[1], v[2], v[3]))(orig(ads, a, n)))
    elif mutant == "slot0_is_real":
        monkeypatch.setattr(lo, "_live_adapter",
                            lambda ads, a, n: ads.get(int(a), (0, 0.0, None, None)) if a < n else None)
    elif mutant == "rows_off_by_one":
        orig_rows = lo._request_rows

        def shifted(req_lengths):
            rows = orig_rows(req_lengths)
            return [(a + 1, b + 1) if i == 0 else (a, b) for i, (a, b) in enumerate(rows)]
        monkeypatch.setattr(lo, "_request_rows", shifted)
    elif mutant == "tail_not_zeroed":
        orig_shrink = lo.shrink_requests

        def shrink(*a, **k):
            buf, w = orig_shrink(*a, **k)
            buf[:, w, -1] += 1.0
            return buf, w
        monkeypatch.setattr(lo, "shrink_requests", shrink)
        monkeypatch.setattr(oracle, "shrink_requests", shrink)
    elif mutant == "slice_offset":
        orig_expand = lo.expand_requests

        def expand(buf, y_in, ads, out_sizes, *rest):
            return orig_expand(buf, y_in, ads, list(reversed(out_sizes)), *rest)
        monkeypatch.setattr(lo, "expand_requests", expand)
    with pytest.raises((AssertionError, IndexError, ValueError)):
        _check_against_brute(0)


# ----------------------------------------------------------------------------- closed forms & invariants

def _rand_problem(seed, T_req=(3, 1, 5, 2, 4), d_in=24, out_sizes=(16, 8), r=4, num_slots=4):
    rng = np.random.default_rng(seed)
    ads = {}
    for k in range(1, num_slots):
        ads[k] = (r, float(rng.choice([0.5, 1.0, 2.0])),
                  [rng.standard_normal((d_in, r)) for _ in out_sizes],
                  [rng.standard_normal((r, d)) for d in out_sizes])
    lengths = list(T_req)
    slots = list(rng.integers(0, num_slots, size=len(lengths)))
    T = sum(lengths)
    x = rng.standard_normal((T, d_in))
    y_in = rng.standard_normal((T, sum(out_sizes)))
    return ads, lengths, slots, x, y_in, list(out_sizes), r, num_slots


def test_merged_weight_equivalence():
    """x W + s (x A) B equals x (W + s A B): the merged form of the LoRA update."""
    ads, lengths, slots, x, _, outs, r, S = _rand_problem(1)
    rng = np.random.default_rng(11)
    W = rng.standard_normal((x.shape[1], sum(outs)))
    y = oracle.apply_requests(x, x @ W, ads, outs, r, lengths, slots, S)
    tok = np.repeat(slots, lengths)
    for t in range(x.shape[0]):
        a = int(tok[t])
        Weff = W.copy()
        if a != 0:
            rk, sc, A, B = ads[a]
            Weff = W + sc * np.concatenate([A[s] @ B[s] for s in range(len(outs))], axis=1)
        ref = x[t] @ Weff
        assert np.max(np.abs(y[t] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_single_adapter_is_one_gemm():
    ads, lengths, _, x, y_in, outs, r, S = _rand_problem(2)
    slots = [2] * len(lengths)
    y = oracle.apply_requests(x, y_in, ads, outs, r, lengths, slots, S)
    rk, sc, A, B = ads[2]
    delta = sc * np.concatenate([x @ (A[s] @ B[s]) for s in range(len(outs))], axis=1)
    assert np.max(np.abs(y - (y_in + delta))) <= 1e-12 * np.max(np.abs(y))


def test_zero_B_and_reset_slot_give_zero_delta():
    ads, lengths, slots, x, y_in, outs, r, S = _rand_problem(3)
    zb = {k: (v[0], v[1], v[2], [np.zeros_like(b) for b in v[3]]) for k, v in ads.items()}
    assert np.array_equal(oracle.apply_requests(x, y_in, zb, outs, r, lengths, slots, S), y_in)
    assert np.array_equal(oracle.apply_requests(x, y_in, {}, outs, r, lengths, [1] * len(lengths), S), y_in)
    buf, w = oracle.shrink_requests(x, {}, len(outs), r, lengths, [1] * len(lengths), S)
    assert w.all() and np.all(buf == 0.0)


def test_slot0_rows_bitwise_untouched():
    ads, lengths, _, x, y_in, outs, r, S = _rand_problem(4)
    slots = [0, 1, 0, 2, 0]
    y_in = y_in.copy()
    y_in[0, :5] = -0.0
    y = oracle.apply_requests(x, y_in, ads, outs, r, lengths, slots, S)
    tok = np.repeat(slots, lengths)
    assert np.array_equal(y[tok == 0].view(np.uint64), y_in[tok == 0].view(np.uint64))
    assert not np.array_equal(y[tok != 0], y_in[tok != 0])
    buf, w = oracle.shrink_requests(x, ads, len(outs), r, lengths, slots, S)
    assert not w[tok == 0].any() and np.isnan(buf[:, tok == 0]).all()


def test_rank_padding_is_exact():
    """A rank-r adapter padded to r_max with a zero tail gives identical results."""
    ads, lengths, slots, x, y_in, outs, r, S = _rand_problem(5)
    b1, w1 = oracle.shrink_requests(x, ads, len(outs), r, lengths, slots, S)
    b2, w2 = oracle.shrink_requests(x, ads, len(outs), 64, lengths, slots, S)
    assert np.array_equal(w1, w2)
    assert np.array_equal(b1[:, w1], b2[:, w2, :r]) and np.all(b2[:, w2, r:] == 0.0)
    y1 = oracle.apply_requests(x, y_in, ads, outs, r, lengths, slots, S)
    y2 = oracle.apply_requests(x, y_in, ads, outs, 64, lengths, slots, S)
    assert np.array_equal(y1, y2)


def test_request_permutation_invariance():
    ads, lengths, slots, x, y_in, outs, r, S = _rand_problem(6)
    y = oracle.apply_requests(x, y_in, ads, outs, r, lengths, slots, S)
    perm = [3, 0, 4, 2, 1]
    starts = np.concatenate([[0], np.cumsum(lengths)])
    rows = np.concatenate([np.arange(starts[i], starts[i + 1]) for i in perm])
    yp = oracle.apply_requests(x[rows], y_in[rows], ads, outs, r,
                               [lengths[i] for i in perm], [slots[i] for i in perm], S)
    assert np.array_equal(yp.view(np.uint64), y[rows].view(np.uint64))


def test_token_runs_equal_requests():
    """Splitting a request into per-token runs changes nothing (tokens are independent)."""
    ads, lengths, slots, x, y_in, outs, r, S = _rand_problem(8)
    y = oracle.apply_requests(x, y_in, ads, outs, r, lengths, slots, S)
    tok = np.repeat(slots, lengths)
    y1 = oracle.apply_requests(x, y_in, ads, outs, r, [1] * len(tok), tok, S)
    assert np.max(np.abs(y - y1)) <= 1e-13 * np.max(np.abs(y))
    L, Sl = oracle.requests_of_token_slots(tok)
    assert np.array_equal(np.repeat(Sl, L), tok)


# ----------------------------------------------------------------------------- input encoding

def test_bf16_encoding_matches_torch():
    import torch
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 7,
                        np.float32([0.0, -0.0, 1.0, 1.00390625, 1.01171875, -3.5e-3, 65504.0])])
    ours = wl.bf16_bits_from_f32(v)
    theirs = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    assert np.array_equal(wl.bf16_bits_to_f32(ours),
                          torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_sampled_rows_mapping_and_restriction():
    """The lm_head LoRA's sampled rows are the last token of every request
    (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section "lm_head / logits"), and
    the oracle's delta on those rows alone equals its delta for the whole batch
    restricted to them (each row's delta uses only its row and slot), to fp64
    rounding: the matrix products may sum in another order for another row count."""
    assert wl.sampled_rows([1, 1, 1]).tolist() == [0, 1, 2]
    assert wl.sampled_rows([3, 1, 5, 2]).tolist() == [2, 3, 8, 10]
    with pytest.raises(ValueError):
        wl.sampled_rows([2, 0])
    lengths = [5, 1, 3, 1, 7]
    inst = wl.make_instance("logits_lm_head", req_lengths=lengths, out_sizes=[96], num_slots=4, d_in=64,
                            dtype="f32")
    ads = lo.adapters_f64(inst)
    x = inst.to_f32(inst.x).astype(np.float64)
    y_in = inst.to_f32(inst.y_in).astype(np.float64)
    y_all = lo.apply_requests(x, y_in, ads, inst.out_sizes, inst.r_max, inst.req_lengths, inst.req_slots,
                              inst.num_slots)
    rows = wl.sampled_rows(inst.req_lengths)
    y_s = lo.apply_requests(x[rows], y_in[rows], ads, inst.out_sizes, inst.r_max, np.ones(len(rows), np.int64),
                            inst.req_slots, inst.num_slots)
    assert np.allclose(y_s, y_all[rows], rtol=0, atol=1e-12 * np.abs(y_all).max())
    live = inst.req_slots != 0
    assert live.any()
    assert not np.array_equal(y_s[live], y_in[rows][live])


def test_embedding_lookup_is_the_one_hot_shrink():
    """The embedding lookup (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section
    "embedding 的 LoRA 是一个查表增量") equals the linear shrink applied to each
    token's one-hot row, exactly, and reads the row the page's flattened table
    gives at token id + slot * vocab; an id outside the vocabulary gives a zero row."""
    vocab = 50
    inst = wl.make_instance("embed_lookup", num_tokens=30, d_in=vocab, out_sizes=[24], num_slots=5, r_max=16,
                            dtype="f32")
    for k, (r, s) in zip(sorted(inst.adapters), [(16, 2.0), (3, 0.5), (9, 1.0), (1, 4.0)]):
        ad = inst.adapters[k]
        inst.adapters[k] = wl.Adapter(r, s, [ad.A[0][:, :r].copy()], [ad.B[0][:r].copy()])
    ids = inst.token_ids.copy()
    ids[3] = vocab + 7          # outside the vocabulary
    ids[4] = -1
    ads = lo.adapters_f64(inst)
    L, Sl, S, R = inst.req_lengths, inst.req_slots, inst.num_slots, inst.r_max
    buf, written = lo.embed_requests(ids, ads, R, L, Sl, S)
    onehot = np.zeros((inst.num_tokens, vocab))
    ok = (ids >= 0) & (ids < vocab)
    onehot[np.arange(inst.num_tokens)[ok], ids[ok]] = 1.0
    ref, w_ref = lo.shrink_requests(onehot, ads, 1, R, L, Sl, S)
    assert np.array_equal(written, w_ref)
    assert np.array_equal(np.nan_to_num(buf, nan=-9.0), np.nan_to_num(ref, nan=-9.0))
    # the page's flattened table: row v + a * vocab of A stacked over all slots
    a_2d = np.zeros((S * vocab, R))
    for a, (r, s, A, _) in ads.items():
        a_2d[a * vocab:(a + 1) * vocab, :r] = A[0][:, :r]
    ts = inst.token_slot
    for t in range(inst.num_tokens):
        a = int(ts[t])
        if a == 0:
            assert not written[t]
        elif ok[t]:
            assert np.array_equal(buf[0, t], ads[a][1] * a_2d[ids[t] + a * vocab])
        else:
            assert np.all(buf[0, t] == 0.0)

