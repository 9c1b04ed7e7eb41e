"""fp64 CPU oracle of the batched multi-LoRA delta -- TEST INFRASTRUCTURE ONLY.

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs; the library never calls it.

What it computes (row-vector orientation, as on the handbook page
"多 LoRA 服务：分段矩阵乘与适配器调度", section "不合并权重，批量计算"):

    y[t] = y_in[t] + s_a * (x[t] A_a) B_a       for every token t of a request
                                                 whose adapter slot a != 0,
    y[t] = y_in[t]                               for slot 0 ("no LoRA").

It is split, as the vLLM page "vLLM 源码完全拆解(十八): 多 LoRA 服务" does in
section "两个低秩 GEMM:shrink、expand 与 fp32 中转缓冲", into

* shrink:  buf[s, t, k] = scale[a] * sum_j x[t, j] A_s[a][j, k]   (k < r_a),
           buf[s, t, k] = 0 for r_a <= k < r_max; slot-0 rows are not written;
* expand:  y[t, off_s + n] = y_in[t, off_s + n] + sum_{k < r_a} buf[s, t, k] B_s[a][k, n],
           off_s = sum of the widths of the slices before s (packed qkv / gate_up);

and the token metadata of section "LoRAKernelMeta:先按槽位排序" (a stable sort
of token indices by slot, the slots present in ascending order, per-slot counts
and start offsets with a leading 0).

Readings where the pages leave a step open:
* slot 0 is the reserved no-LoRA slot (vLLM marks it -1; it sorts first either way);
* the per-slot scale multiplies the shrink result (vLLM page, section
  "PEFTHelper:认清 adapter 文件": the scale is applied in the shrink step);
* a token slot id outside [0, num_slots) is treated as slot 0 and counted;
* ``seg_*`` arrays are padded to ``num_slots`` entries (slot -1, count 0,
  start T) after the ``num_segs`` live ones.

The arithmetic is a per-request loop (the page's "逐个请求调用一次矩阵乘"
formulation) with numpy's fp64 matmul as the only library step. Inputs are the
stored bf16/fp32 values widened exactly to fp64.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np

AdapterF64 = Tuple[int, float, List[np.ndarray], List[np.ndarray]]  # rank, scale, A[s] [d_in,r], B[s] [r,d_out_s]


def adapters_f64(inst) -> Dict[int, AdapterF64]:
    """The instance's adapters as exact fp64 copies of their stored values."""
    out = {}
    for k, a in inst.adapters.items():
        out[int(k)] = (int(a.rank), float(np.float32(a.scale)),
                       [inst.to_f32(m).astype(np.float64) for m in a.A],
                       [inst.to_f32(m).astype(np.float64) for m in a.B])
    return out


def requests_of_token_slots(token_slot: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """Split a per-token slot array into maximal runs of equal slots.

    Each run behaves as one request: the delta of a token depends only on its
    own row and its own slot.
    """
    ts = np.asarray(token_slot, dtype=np.int64)
    lengths, slots = [], []
    t = 0
    while t < len(ts):
        u = t
        while u < len(ts) and ts[u] == ts[t]:
            u += 1
        lengths.append(u - t)
        slots.append(int(ts[t]))
        t = u
    return np.asarray(lengths, np.int64), np.asarray(slots, np.int64)


def prepare_meta(token_slot: Sequence[int], num_slots: int) -> dict:
    """Token metadata: stable slot-sorted row order and segments.

    Follows "LoRAKernelMeta:先按槽位排序" (vLLM page): tokens are ordered by slot
    with ties kept in batch order; each slot present forms one segment; segment
    i covers sorted rows [seg_start[i], seg_start[i] + seg_count[i]) and
    seg_start[0] is 0. ``no_lora`` is 1 when no token uses a real adapter
    (the early exit of the same section). Written as one bucket pass per token,
    then the buckets in ascending slot order.
    """
    T = len(token_slot)
    buckets: List[List[int]] = [[] for _ in range(num_slots)]
    bad = 0
    for t in range(T):
        s = int(token_slot[t])
        if s < 0 or s >= num_slots:
            bad += 1
            s = 0
        buckets[s].append(t)
    sorted_rows: List[int] = []
    seg_slot, seg_count, seg_start = [], [], [0]
    for s in range(num_slots):
        if buckets[s]:
            seg_slot.append(s)
            seg_count.append(len(buckets[s]))
            sorted_rows.extend(buckets[s])
            seg_start.append(len(sorted_rows))
    num_segs = len(seg_slot)
    pad = num_slots - num_segs
    return dict(
        sorted_rows=np.asarray(sorted_rows, np.int32).reshape(T),
        seg_slot=np.asarray(seg_slot + [-1] * pad, np.int32),
        seg_count=np.asarray(seg_count + [0] * pad, np.int32),
        seg_start=np.asarray(seg_start + [T] * pad, np.int32),
        num_segs=num_segs,
        no_lora=int(len(buckets[0]) == T),
        status=bad,
    )


def _request_rows(req_lengths) -> List[Tuple[int, int]]:
    rows, t0 = [], 0
    for n in req_lengths:
        rows.append((t0, t0 + int(n)))
        t0 += int(n)
    return rows


def _live_adapter(adapters: Dict[int, AdapterF64], a: int, num_slots: int):
    """None for no-LoRA rows (slot 0 or an id outside the table); else the adapter.

    A slot inside the table that holds no adapter behaves as a reset slot:
    rank 0, so its delta is the empty sum.
    """
    if a <= 0 or a >= num_slots:
        return None
    return adapters.get(int(a), (0, 0.0, None, None))


def shrink_requests(x: np.ndarray, adapters: Dict[int, AdapterF64], n_slices: int, r_max: int,
                    req_lengths, req_slots, num_slots: int) -> Tuple[np.ndarray, np.ndarray]:
    """buf[s, t, :] for every token of a LoRA request; returns (buf, written).

    buf[s, t, k] = scale * (x[t] @ A_s[:, k]) for k < rank, 0 for the rank
    tail. Rows of no-LoRA tokens are left NaN and ``written[t]`` False: the
    library leaves them unwritten and nothing reads them.
    """
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    buf = np.full((n_slices, T, r_max), np.nan, dtype=np.float64)
    written = np.zeros(T, dtype=bool)
    for (t0, t1), a in zip(_request_rows(req_lengths), req_slots):
        ad = _live_adapter(adapters, int(a), num_slots)
        if ad is None or t1 == t0:
            continue
        r, scale, A, _ = ad
        for s in range(n_slices):
            buf[s, t0:t1, :] = 0.0
            if r > 0:
                buf[s, t0:t1, :r] = scale * (x[t0:t1] @ A[s][:, :r])
        written[t0:t1] = True
    return buf, written


def expand_requests(buf: np.ndarray, y_in: np.ndarray, adapters: Dict[int, AdapterF64],
                    out_sizes: Sequence[int], req_lengths, req_slots, num_slots: int) -> np.ndarray:
    """y = y_in with buf @ B_s added into each slice's columns of LoRA rows.

    Slot-0 rows are copied unchanged (no arithmetic touches them).
    """
    y_in = np.asarray(y_in, dtype=np.float64)
    y = y_in.copy()
    for (t0, t1), a in zip(_request_rows(req_lengths), req_slots):
        ad = _live_adapter(adapters, int(a), num_slots)
        if ad is None or t1 == t0:
            continue
        r, _, _, B = ad
        off = 0
        for s, d_out in enumerate(out_sizes):
            if r > 0:
                delta = np.asarray(buf[s, t0:t1, :r], np.float64) @ B[s][:r, :]
            else:
                delta = np.zeros((t1 - t0, d_out), np.float64)
            y[t0:t1, off:off + d_out] = y_in[t0:t1, off:off + d_out] + delta
            off += d_out
    return y


def embed_requests(token_ids, adapters: Dict[int, AdapterF64], r_max: int, req_lengths, req_slots,
                   num_slots: int) -> Tuple[np.ndarray, np.ndarray]:
    """buf[0, t, :] of an embedding layer's LoRA; returns (buf, written).

    Page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section "embedding 的 LoRA 是一个
    查表增量": the r-vector of token id v under slot a is row v of a's A table, so
        buf[0, t, k] = scale * A[token_ids[t], k]   (k < rank),  0 for the rank tail.
    Rows of no-LoRA tokens are left NaN and not written. A token id outside
    [0, vocab) gets a zero row (no delta): the pages do not say; this reading
    lets one bad id spoil nothing else.
    """
    token_ids = np.asarray(token_ids)
    T = int(token_ids.shape[0])
    buf = np.full((1, T, r_max), np.nan, dtype=np.float64)
    written = np.zeros(T, dtype=bool)
    for (t0, t1), a in zip(_request_rows(req_lengths), req_slots):
        ad = _live_adapter(adapters, int(a), num_slots)
        if ad is None or t1 == t0:
            continue
        r, scale, A, _ = ad
        buf[0, t0:t1, :] = 0.0
        for t in range(t0, t1):
            v = int(token_ids[t])
            if r > 0 and 0 <= v < A[0].shape[0]:
                buf[0, t, :r] = scale * A[0][v, :r]
        written[t0:t1] = True
    return buf, written


def apply_requests(x: np.ndarray, y_in: np.ndarray, adapters: Dict[int, AdapterF64],
                   out_sizes: Sequence[int], r_max: int, req_lengths, req_slots,
                   num_slots: int) -> np.ndarray:
    """The whole delta: expand(shrink(x)) added into the base output y_in."""
    buf, _ = shrink_requests(x, adapters, len(out_sizes), r_max, req_lengths, req_slots, num_slots)
    return expand_requests(buf, y_in, adapters, out_sizes, req_lengths, req_slots, num_slots)
