"""The tensor-core (SGMV) family and the AUTO split against the fp64 oracle, through the C ABI.

SGMV runs 128-row tiles of same-adapter segments on tcgen05 (split-K shrink
over d_in, hi + lo bf16 expand). The cases cover tiles that end inside a
segment and segments shorter than a tile, d_in and output widths that are not
multiples of the K block or the column block, every supported r_max, one to
four packed slices, padded leading dimensions, heterogeneous ranks with a
scale, the full-size prefill batch (every row) and the full mixed batch
under AUTO. Tolerances are those of the BGMV tests."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_harness import TOL_BF16, bf16_half_ulp, load_table, parity, run_gpu, to_dev

pytestmark = pytest.mark.gpu


def _status_ok(lib, meta):
    st, n = lib.lora_query_status(meta.c)
    assert st in (lib.LORA_OK, lib.LORA_EBADSLOT), lib.lora_strerror(st)


@pytest.mark.parametrize("path", ["split", "apply"])
@pytest.mark.parametrize("y_dtype", ["f32", "bf16"])
def test_sgmv_prefill_small(lib, path, y_dtype):
    inst = wl.make_instance("prefill_gate_up", num_tokens=1500, d_in=512, out_sizes=[640, 384], num_slots=9)
    _, _, meta = parity(inst, kind=lib.LORA_SGMV, y_dtype=y_dtype, path=path)
    _status_ok(lib, meta)


def _segment_batch(sizes, S, rng):
    """Token slots whose segments have the given sizes, interleaved with slot-0
    tokens and split into several requests each, so sorted rows are not contiguous."""
    reqs = []
    for i, n in enumerate(sizes):
        slot = 1 + i % (S - 1)
        cuts = sorted(rng.choice(np.arange(1, n), size=min(3, n - 1), replace=False)) if n > 1 else []
        for part in np.split(np.arange(n), cuts):
            reqs.append(np.full(len(part), slot, np.int32))
        reqs.append(np.zeros(rng.integers(0, 3), np.int32))
    order = rng.permutation(len(reqs))
    return np.concatenate([reqs[i] for i in order]).astype(np.int32)


def test_sgmv_segment_and_tile_boundaries(lib):
    rng = np.random.default_rng(11)
    sizes = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300]
    ts = _segment_batch(sizes, 13, rng)
    inst = wl.make_instance("decode_qkv", num_tokens=len(ts), d_in=320, out_sizes=[136, 72, 200], num_slots=13,
                            r_max=32)
    for path in ("split", "apply"):
        _, _, meta = parity(inst, kind=lib.LORA_SGMV, token_slot=ts, path=path)
        _status_ok(lib, meta)


@pytest.mark.parametrize("r_max,n_slices", [(16, 1), (16, 4), (32, 2), (64, 3), (128, 1), (128, 2), (128, 4)])
def test_sgmv_ranks_slices_ragged_shapes(lib, r_max, n_slices):
    """d_in = 200 (not a multiple of the 64-wide K block), widths not multiples of the
    128-column block, padded strides; ranks 1..r_max within one table."""
    outs = [72, 200, 136, 64][:n_slices]
    inst = wl.make_instance("decode_qkv", num_tokens=700, d_in=200, out_sizes=outs, num_slots=7, r_max=r_max)
    rng = np.random.default_rng(r_max + n_slices)
    for k, r in zip(sorted(inst.adapters), [1, r_max // 2 + 1, r_max, 7, r_max - 1, r_max]):
        ad = inst.adapters[k]
        inst.adapters[k] = wl.Adapter(r, 0.5 + k / 4, [a[:, :r].copy() for a in ad.A], [b[:r].copy() for b in ad.B])
    ts = _segment_batch([150, 90, 300, 64, 96], 7, rng)
    inst = _with_tokens(inst, ts, rng)
    parity(inst, kind=lib.LORA_SGMV, token_slot=ts, ldx_pad=24, ldy_pad=8, path="apply")
    parity(inst, kind=lib.LORA_SGMV, token_slot=ts, y_dtype="bf16", path="split")


def _with_tokens(inst, ts, rng):
    """The instance re-drawn at len(ts) tokens (x and y_in), adapters kept."""
    T = len(ts)
    inst.x = wl.bf16_bits_from_f32(rng.standard_normal((T, inst.d_in), dtype=np.float32))
    inst.y_in = wl.bf16_bits_from_f32(rng.standard_normal((T, inst.d_out_total), dtype=np.float32))
    inst.req_lengths, inst.req_slots = oracle.requests_of_token_slots(ts)
    return inst


def test_sgmv_heterogeneous_ranks_and_scale(lib):
    """Ranks {8, 16, 32, 64} padded to 64 with scale 2 (the mixed batch's adapters), all through SGMV."""
    inst = wl.make_instance("mixed_o_proj", num_tokens=600, d_in=1024, out_sizes=[768], num_slots=24)
    parity(inst, kind=lib.LORA_SGMV, y_dtype="bf16", path="apply")
    parity(inst, kind=lib.LORA_SGMV, path="split")


def test_sgmv_apply_equals_split_bitwise_and_repeats(lib):
    inst = wl.make_instance("prefill_gate_up", num_tokens=2000, d_in=768, out_sizes=[384, 256], num_slots=6)
    t = load_table(inst)
    b1, y1, _ = run_gpu(inst, table=t, kind=lib.LORA_SGMV, path="split", y_dtype="bf16")
    b2, y2, _ = run_gpu(inst, table=t, kind=lib.LORA_SGMV, path="apply", y_dtype="bf16")
    b3, y3, _ = run_gpu(inst, table=t, kind=lib.LORA_SGMV, path="apply", y_dtype="bf16")
    assert np.array_equal(b1, b2, equal_nan=True) and np.array_equal(y1, y2)
    assert np.array_equal(b2, b3, equal_nan=True) and np.array_equal(y2, y3)


def test_sgmv_permutation_invariant(lib):
    """Reordering requests permutes the outputs bitwise: a token's result does not
    depend on where its row falls in a tile."""
    inst = wl.make_instance("prefill_gate_up", num_tokens=1200, d_in=512, out_sizes=[256, 128], num_slots=5)
    t = load_table(inst)
    _, y1, _ = run_gpu(inst, table=t, kind=lib.LORA_SGMV, path="apply")
    rng = np.random.default_rng(3)
    order = rng.permutation(len(inst.req_lengths))
    starts = np.concatenate([[0], np.cumsum(inst.req_lengths)])
    perm = np.concatenate([np.arange(starts[i], starts[i + 1]) for i in order])
    inst_p = wl.make_instance("prefill_gate_up", num_tokens=1200, d_in=512, out_sizes=[256, 128], num_slots=5)
    inst_p.x, inst_p.y_in = inst.x[perm], inst.y_in[perm]
    inst_p.req_lengths, inst_p.req_slots = inst.req_lengths[order], inst.req_slots[order]
    _, y2, _ = run_gpu(inst_p, table=t, kind=lib.LORA_SGMV, path="apply")
    assert np.array_equal(y1[perm], y2)


def test_auto_mixed_full_size(lib):
    """The mixed batch (3072 tokens, >= LORA_AUTO_SGMV_MIN_TOKENS): long segments on SGMV,
    the rest on BGMV, in one call."""
    inst = wl.make_instance("mixed_o_proj")
    assert inst.num_tokens >= lib.LORA_AUTO_SGMV_MIN_TOKENS
    t = load_table(inst)
    _, y_auto, meta = parity(inst, kind=lib.LORA_AUTO, y_dtype="bf16", table=t, path="apply")
    _status_ok(lib, meta)
    parity(inst, kind=lib.LORA_AUTO, table=t, path="split")
    # The long segments really ran on the tensor-core family: their rows differ
    # (within tolerance) from the all-BGMV result somewhere.
    _, y_bgmv, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV, y_dtype="bf16", path="apply")
    counts = np.bincount(inst.token_slot, minlength=inst.num_slots)
    long_rows = np.where((counts[inst.token_slot] >= lib.LORA_SGMV_MIN_ROWS) & (inst.token_slot > 0))[0]
    assert len(long_rows) > 0
    assert not np.array_equal(y_auto[long_rows], y_bgmv[long_rows])


def test_auto_small_batches_stay_on_bgmv(lib):
    """Below LORA_AUTO_SGMV_MIN_TOKENS, or below LORA_AUTO_SGMV_MIN_AVG tokens per slot, AUTO is
    the BGMV family bitwise; a batch above both with no long segment is too (the SGMV kernels
    find no tiles)."""
    inst = wl.make_instance("prefill_gate_up", num_tokens=900, d_in=512, out_sizes=[256, 128], num_slots=5)
    t = load_table(inst)
    _, ya, _ = run_gpu(inst, table=t, kind=lib.LORA_AUTO, path="apply")
    _, yb, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV, path="apply")
    assert np.array_equal(ya, yb)
    dec = wl.make_instance("decode_qkv", num_tokens=1100, d_in=512, out_sizes=[256], num_slots=64)
    assert np.bincount(dec.token_slot)[1:].max() < lib.LORA_SGMV_MIN_ROWS
    t2 = load_table(dec)
    ba, ya, meta = run_gpu(dec, table=t2, kind=lib.LORA_AUTO, path="split")
    bb, yb, _ = run_gpu(dec, table=t2, kind=lib.LORA_BGMV, path="split")
    assert np.array_equal(ya, yb) and np.array_equal(ba, bb, equal_nan=True)
    _status_ok(lib, meta)
    # 22 tokens on each of 47 slots: at least 1024 tokens and 20 per slot, no segment of 32
    S = 48
    ts = np.tile(np.arange(1, S, dtype=np.int32), 22)
    assert len(ts) >= lib.LORA_AUTO_SGMV_MIN_TOKENS and len(ts) >= lib.LORA_AUTO_SGMV_MIN_AVG * (S - 1)
    assert np.bincount(ts)[1:].max() < lib.LORA_SGMV_MIN_ROWS
    dec2 = wl.make_instance("decode_qkv", num_tokens=len(ts), d_in=512, out_sizes=[256], num_slots=S)
    dec2 = _with_tokens(dec2, ts, np.random.default_rng(5))
    t3 = load_table(dec2)
    for path in ("split", "apply"):
        ba, ya, meta = run_gpu(dec2, table=t3, kind=lib.LORA_AUTO, path=path, token_slot=ts)
        bb, yb, _ = run_gpu(dec2, table=t3, kind=lib.LORA_BGMV, path=path, token_slot=ts)
        assert np.array_equal(ya, yb) and np.array_equal(ba, bb, equal_nan=True)
        _status_ok(lib, meta)


def test_auto_splits_only_with_a_long_segment(lib):
    """AUTO sends segments of LORA_SGMV_MIN_ROWS or more to SGMV only when the batch holds a
    segment of LORA_AUTO_LONG_ROWS or more. A batch of 32..63-token segments (over both token
    thresholds) is the BGMV family bitwise; the same batch with one slot grown past
    LORA_AUTO_LONG_ROWS runs its 32+ segments on SGMV (their rows differ from BGMV's, within
    tolerance of the oracle) and its short ones on BGMV (bitwise)."""
    S = 33
    rng = np.random.default_rng(9)
    counts = rng.integers(10, lib.LORA_AUTO_LONG_ROWS, size=S - 1)
    counts[:4] = [lib.LORA_SGMV_MIN_ROWS, 40, 63, 12]
    ts = np.repeat(np.arange(1, S, dtype=np.int32), counts)
    rng.shuffle(ts)
    assert len(ts) >= lib.LORA_AUTO_SGMV_MIN_TOKENS and len(ts) >= lib.LORA_AUTO_SGMV_MIN_AVG * (S - 1)
    inst = wl.make_instance("decode_qkv", num_tokens=len(ts), d_in=512, out_sizes=[256, 128], num_slots=S)
    inst = _with_tokens(inst, ts, np.random.default_rng(10))
    t = load_table(inst)
    for path in ("split", "apply"):
        ba, ya, meta = run_gpu(inst, table=t, kind=lib.LORA_AUTO, path=path, token_slot=ts)
        bb, yb, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV, path=path, token_slot=ts)
        assert np.array_equal(ya, yb) and np.array_equal(ba, bb, equal_nan=True)
        _status_ok(lib, meta)
    # one slot past LORA_AUTO_LONG_ROWS: the split is on
    ts2 = np.concatenate([ts, np.full(lib.LORA_AUTO_LONG_ROWS, 5, np.int32)])
    inst2 = wl.make_instance("decode_qkv", num_tokens=len(ts2), d_in=512, out_sizes=[256, 128], num_slots=S)
    inst2 = _with_tokens(inst2, ts2, np.random.default_rng(11))
    t2 = load_table(inst2)
    _, ya, meta = parity(inst2, kind=lib.LORA_AUTO, table=t2, path="apply", token_slot=ts2)
    _status_ok(lib, meta)
    _, yb, _ = run_gpu(inst2, table=t2, kind=lib.LORA_BGMV, path="apply", token_slot=ts2)
    c2 = np.bincount(ts2, minlength=S)
    short = np.where((c2[ts2] < lib.LORA_SGMV_MIN_ROWS) & (ts2 > 0))[0]
    long_ = np.where(c2[ts2] >= lib.LORA_SGMV_MIN_ROWS)[0]
    assert len(short) and len(long_)
    assert np.array_equal(ya[short], yb[short])
    assert not np.array_equal(ya[long_], yb[long_])


def test_mixed_kind_small_batch_with_a_prompt(lib):
    """LORA_MIXED below AUTO's token thresholds: a 300-token batch holding one 200-token prompt
    beside one-token decode requests runs the prompt's segment on SGMV and the rest on BGMV,
    within tolerance of the oracle on every row, the short rows bitwise equal to BGMV's; a
    decode batch without a long segment is the BGMV family bitwise."""
    S = 17
    rng = np.random.default_rng(21)
    ts = np.concatenate([rng.integers(0, S, size=100), np.full(200, 3)]).astype(np.int32)
    assert len(ts) < lib.LORA_AUTO_SGMV_MIN_TOKENS
    inst = wl.make_instance("decode_qkv", num_tokens=len(ts), d_in=1024, out_sizes=[512, 256], num_slots=S)
    inst = _with_tokens(inst, ts, np.random.default_rng(22))
    t = load_table(inst)
    for path in ("apply", "split"):
        _, ym, meta = parity(inst, kind=lib.LORA_MIXED, table=t, path=path, token_slot=ts)
        _status_ok(lib, meta)
        _, yb, _ = run_gpu(inst, table=t, kind=lib.LORA_BGMV, path=path, token_slot=ts)
        c = np.bincount(ts, minlength=S)
        short = np.where((c[ts] < lib.LORA_SGMV_MIN_ROWS) & (ts > 0))[0]
        assert np.array_equal(ym[short], yb[short])
        assert not np.array_equal(ym[ts == 3], yb[ts == 3])
        assert np.array_equal(ym[ts == 0], yb[ts == 0])
    dec = wl.make_instance("decode_qkv", num_tokens=256, d_in=512, out_sizes=[256], num_slots=33)
    t2 = load_table(dec)
    for path in ("apply", "split"):
        ba, ya, meta = run_gpu(dec, table=t2, kind=lib.LORA_MIXED, path=path)
        bb, yb, _ = run_gpu(dec, table=t2, kind=lib.LORA_BGMV, path=path)
        assert np.array_equal(ya, yb) and np.array_equal(ba, bb, equal_nan=True)
        _status_ok(lib, meta)


def test_sgmv_prefill_full_size_every_row(lib):
    """The full prefill batch (gate_up 4096 -> 2 x 14336, r = 64, ~14k tokens) through
    lora_apply with AUTO and a bf16 y, every row and column checked against the oracle.
    The oracle runs one request at a time on that request's rows (a token's delta
    depends only on its own row and slot), so the host never holds more than one
    request's fp64 rows; the bound is the stated one over the whole batch's delta."""
    inst = wl.make_instance("prefill_gate_up")
    T, W = inst.num_tokens, inst.d_out_total
    assert W == 28672
    t = load_table(inst)
    x = to_dev(inst.x, "bf16")
    y = to_dev(inst.y_in, "bf16")
    meta = lib.TokenMeta(T, inst.num_slots)
    meta.prepare(torch.from_numpy(inst.token_slot).cuda())
    lib.apply(t, meta, x, y, kind=lib.LORA_AUTO)
    torch.cuda.synchronize()
    _status_ok(lib, meta)
    y_gpu_all = y.float().cpu().numpy()
    ads = oracle.adapters_f64(inst)
    starts = np.concatenate([[0], np.cumsum(inst.req_lengths)])
    sq_sum, n, worst = 0.0, 0, []
    for i, slot in enumerate(inst.req_slots):
        t0, t1 = int(starts[i]), int(starts[i + 1])
        x64 = inst.to_f32(inst.x[t0:t1]).astype(np.float64)
        y64 = inst.to_f32(inst.y_in[t0:t1]).astype(np.float64)
        lengths, slots = np.asarray([t1 - t0], np.int64), np.asarray([slot], np.int64)
        buf, written = oracle.shrink_requests(x64, ads, inst.n_slices, inst.r_max, lengths, slots, inst.num_slots)
        y_ref = oracle.expand_requests(buf, y64, ads, inst.out_sizes, lengths, slots, inst.num_slots)
        assert written.all()
        delta = y_ref - y64
        sq_sum += float(np.sum(delta ** 2))
        n += delta.size
        err = np.abs(y_gpu_all[t0:t1].astype(np.float64) - y_ref)
        # per request: the largest error beyond half a bf16 ulp of the reference value
        worst.append(float(np.max(err - bf16_half_ulp(y_ref))))
    rms = np.sqrt(sq_sum / n)
    assert max(worst) <= TOL_BF16 * rms, f"max excess {max(worst):.3e} > 1e-2 x RMS {rms:.3e}"
