"""fp64 CPU oracle of the mixture-of-experts LoRA -- TEST INFRASTRUCTURE ONLY.

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU legs; the library never calls it.

What it computes (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section
"MoE 的 LoRA:按专家挂载、融合 kernel 与 EP 切片"): every expert of an MoE layer
has its own low-rank pair per adapter, so a token routed to its top-k experts
gets, for each chosen expert e and the token's adapter a, the delta of the
pair (a, e):

* after w13 and before the activation (subsection "融合计算:add_lora_w13 与
  add_lora_w2"): h1[t, k] += s_a * (x[t] A13_s[a, e]) B13_s[a, e] for the w13
  slices s (gate and up);
* after w2 and before the top-k sum: h3[t, k] += s_a * (h2[t, k] A2[a, e]) B2[a, e].

The pages group the (token, choice) pairs by (adapter, expert)
(``moe_lora_align_block_size``) so that one low-rank product runs per group;
here the grouping is a composite slot per pair (``moe_pair_slots``), after
which each w13 / w2 application is the dense multi-LoRA delta of
``lora_oracle`` over the pairs, with the x row of pair p being token p // topk
for w13 and pair p itself for w2. Expert-parallel ranks hold only their local
experts (subsection "EP 下只装载本地专家的权重"): a pair whose expert is not
local gets no delta on that rank.

Readings where the pages leave a step open:
* adapter slot 0 is "no LoRA", as for the dense layers; adapters are slots
  1..num_loras;
* pairs are numbered token-major, p = t * topk + k (the layout of
  ``topk_ids`` [T, topk]);
* the composite slot of (a, e_local) is 1 + (a - 1) * local_experts + e_local,
  0 for no delta, and -1 (counted as a bad id downstream) for an adapter
  outside [0, num_loras], an expert id outside [0, num_experts) or a map entry
  past the local experts;
* the local index of a global expert id is expert_map[e] (-1: not local), or e
  itself without a map.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from .lora_oracle import AdapterF64


def moe_pair_slots(token_slot: Sequence[int], topk_ids: np.ndarray, num_loras: int, num_experts: int,
                   local_experts: int, expert_map: Optional[Sequence[int]] = None) -> np.ndarray:
    """Composite slot of every (token, choice) pair, token-major (p = t * topk + k)."""
    ts = np.asarray(token_slot, dtype=np.int64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, topk = ids.shape
    out = np.zeros(T * topk, dtype=np.int32)
    for t in range(T):
        a = int(ts[t])
        for k in range(topk):
            e = int(ids[t, k])
            p = t * topk + k
            if a < 0 or a > num_loras or e < 0 or e >= num_experts:
                out[p] = -1
                continue
            el = int(expert_map[e]) if expert_map is not None else e
            if el >= local_experts:
                out[p] = -1
            elif a == 0 or el < 0:
                continue
            else:
                out[p] = 1 + (a - 1) * local_experts + el
    return out


def gathered_apply(x_rows: np.ndarray, x_row_of_pair: np.ndarray, y_in: np.ndarray, pair_slot: Sequence[int],
                   adapters: Dict[int, AdapterF64], out_sizes: Sequence[int], num_slots: int) -> np.ndarray:
    """y[p] = y_in[p] + s * (x_rows[x_row_of_pair[p]] A[slot]) B[slot] for every pair p whose
    composite slot is live (rows of slot 0, of ids outside the table and of empty slots unchanged)."""
    y = np.array(y_in, dtype=np.float64, copy=True)
    offs = np.concatenate([[0], np.cumsum(out_sizes)]).astype(np.int64)
    for p, slot in enumerate(np.asarray(pair_slot, dtype=np.int64)):
        if slot <= 0 or slot >= num_slots or int(slot) not in adapters:
            continue
        r, scale, A, B = adapters[int(slot)]
        if r == 0:
            continue
        xr = x_rows[int(x_row_of_pair[p])]
        for s in range(len(out_sizes)):
            u = scale * (xr @ A[s][:, :r])
            y[p, offs[s]:offs[s + 1]] += u @ B[s][:r]
    return y


def moe_lora_w13(x: np.ndarray, h1_in: np.ndarray, pair_slot, topk: int, adapters13: Dict[int, AdapterF64],
                 out_sizes13: Sequence[int], num_slots: int) -> np.ndarray:
    """h1 [T * topk, sum(out_sizes13)] after the w13 LoRA; x [T, hidden] is shared by a token's choices."""
    T = x.shape[0]
    rows = np.repeat(np.arange(T), topk)
    return gathered_apply(x, rows, h1_in, pair_slot, adapters13, out_sizes13, num_slots)


def moe_lora_w2(h2: np.ndarray, h3_in: np.ndarray, pair_slot, adapters2: Dict[int, AdapterF64],
                hidden: int, num_slots: int) -> np.ndarray:
    """h3 [T * topk, hidden] after the w2 LoRA; h2 [T * topk, inter] holds one row per pair."""
    rows = np.arange(h2.shape[0])
    return gathered_apply(h2, rows, h3_in, pair_slot, adapters2, [hidden], num_slots)
