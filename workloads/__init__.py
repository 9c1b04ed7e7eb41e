"""Seeded synthetic inputs for the batched multi-LoRA delta.

This module is shared by the tests, the benchmark and the oracle's callers. It
holds none of the method's arithmetic: only random draws, the bf16 storage
encoding, and the request/slot layouts of the workloads that the multi-LoRA
serving pages describe.

Workloads (sizes follow the Llama-3-8B-shaped projections the pages use):

* ``toy_fp32``      d=256, r=16, 8 slots, scale 2.0, six requests of lengths
                    [1,1,37,1,12,1] (53 tokens) -- the toy batch of the
                    handbook page "多 LoRA 服务：分段矩阵乘与适配器调度",
                    section "不合并权重，批量计算"; fp32 throughout.
* ``decode_qkv``    qkv_proj, d_in=4096, packed slices [4096,1024,1024], r=16,
                    64 slots, 256 one-token requests, 10% slot 0.
* ``prefill_gate_up`` gate_up_proj, d_in=4096, slices [14336,14336], r=64,
                    32 slots, 16 requests of length U[128,2048], Zipf(1.1).
* ``mixed_o_proj``  o_proj 4096->4096, 128 slots, per-slot rank in
                    {8,16,32,64} padded to 64, scale alpha/r with alpha=2r,
                    1024 decode tokens + 4 prefill chunks of 512, 5% slot 0.
* ``full_decode``   one decode step over 32 layers x {qkv, o, gate_up, down},
                    r=16, 100 resident adapters, 512 tokens.
* ``embed_lookup``  the embedding layer's LoRA (page "vLLM 源码完全拆解(十八):
                    多 LoRA 服务", section "embedding 的 LoRA 是一个查表增量"):
                    vocab 128256 -> hidden 4096, r=16, 64 slots, 256 decode
                    tokens with ids uniform over the vocabulary, 10% slot 0.
* ``moe_decode``    one mixture-of-experts layer's LoRA (page "vLLM 源码完全拆解
                    (十八): 多 LoRA 服务", section "MoE 的 LoRA:按专家挂载、融合 kernel
                    与 EP 切片"), shaped like its DeepSeek-V3 memory example:
                    hidden 7168, expert intermediate 2048, 256 experts with
                    8-way expert parallelism (32 local, rank 0), top-8 routing,
                    r=64, 4 adapters, 256 decode tokens (10% slot 0); the w13
                    (gate, up) and w2 applications over the (token, choice) pairs.
* ``logits_lm_head`` the lm_head LoRA on the rows sampled this step (page
                    "vLLM 源码完全拆解(十八): 多 LoRA 服务", section
                    "lm_head / logits"): hidden 4096 -> vocab 128256, r=16,
                    64 slots, 256 sampled rows (one per request), 10% slot 0.

Slot 0 is the reserved "no LoRA" slot; adapters live in slots 1..num_slots-1.
bf16 tensors are produced as uint16 bit patterns so that every consumer sees
exactly the same stored values.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "bf16_bits_from_f32", "bf16_bits_to_f32", "Adapter", "Instance",
    "make_instance", "toy_page_instance", "zipf_probs", "full_decode_groups",
    "CONFIG_NAMES", "EXTRA_NAMES", "split_requests", "sampled_rows", "MoEInstance", "make_moe_instance",
]

CONFIG_NAMES = ("toy_fp32", "decode_qkv", "prefill_gate_up", "mixed_o_proj", "full_decode")
EXTRA_NAMES = ("logits_lm_head", "embed_lookup", "moe_decode")   # widening beyond the five configurations

_CHUNK = 1 << 24


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Encode float32 values as bf16 bit patterns, rounding to nearest even.

    bf16 is the upper half of an IEEE binary32 word; rounding adds
    0x7FFF plus the lowest kept bit before truncating. Finite inputs only.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    flat = a.reshape(-1).view(np.uint32)
    out = np.empty(flat.shape, dtype=np.uint16)
    for i in range(0, flat.size, _CHUNK):
        u = flat[i:i + _CHUNK]
        bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
        out[i:i + _CHUNK] = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    return out.reshape(a.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def zipf_probs(n: int, alpha: float) -> np.ndarray:
    """P(k) proportional to k^-alpha for k = 1..n (rank k <-> slot k)."""
    k = np.arange(1, n + 1, dtype=np.float64)
    p = k ** (-alpha)
    return p / p.sum()


@dataclass
class Adapter:
    """One adapter as the caller holds it before activation.

    ``A[s]`` is ``[d_in, rank]`` and ``B[s]`` is ``[rank, out_sizes[s]]`` for
    every packed slice ``s`` (row-vector orientation ``y = xW + s(xA)B``).
    Arrays are uint16 bf16 bits or float32, as the instance's dtype says.
    """
    rank: int
    scale: float
    A: List[np.ndarray]
    B: List[np.ndarray]


@dataclass
class Instance:
    """A seeded workload: slot table contents, requests, x and the base output."""
    name: str
    dtype: str                      # "bf16" or "f32": storage of x, A, B, y
    d_in: int
    out_sizes: List[int]
    num_slots: int                  # including the reserved slot 0
    r_max: int
    adapters: dict                  # slot (1..num_slots-1) -> Adapter
    req_lengths: np.ndarray         # int64 [n_requests]
    req_slots: np.ndarray           # int32 [n_requests]; may hold ids outside the table
    x: np.ndarray                   # [T, d_in] (uint16 bits or float32)
    y_in: np.ndarray                # [T, sum(out_sizes)]
    meta: dict = field(default_factory=dict)
    token_ids: Optional[np.ndarray] = None   # int32 [T]: an embedding layer's input (x is then empty)

    @property
    def num_tokens(self) -> int:
        return int(self.req_lengths.sum())

    @property
    def n_slices(self) -> int:
        return len(self.out_sizes)

    @property
    def d_out_total(self) -> int:
        return int(sum(self.out_sizes))

    @property
    def token_slot(self) -> np.ndarray:
        """Per-token slot ids: each request's slot broadcast over its tokens."""
        return np.repeat(self.req_slots.astype(np.int32), self.req_lengths).astype(np.int32)

    def slot_ranks(self) -> np.ndarray:
        r = np.zeros(self.num_slots, dtype=np.int32)
        for k, a in self.adapters.items():
            r[k] = a.rank
        return r

    def slot_scales(self) -> np.ndarray:
        s = np.zeros(self.num_slots, dtype=np.float32)
        for k, a in self.adapters.items():
            s[k] = a.scale
        return s

    def to_f32(self, a: np.ndarray) -> np.ndarray:
        """Stored values as float32 (bf16 bits widened exactly)."""
        return bf16_bits_to_f32(a) if self.dtype == "bf16" else np.asarray(a, dtype=np.float32)


def _normal(rng: np.random.Generator, shape, inv_scale: float, dtype: str) -> np.ndarray:
    v = rng.standard_normal(shape, dtype=np.float32)
    if inv_scale != 1.0:
        v /= np.float32(inv_scale)     # powers of two: exact
    return bf16_bits_from_f32(v) if dtype == "bf16" else v


class _Pool:
    """A pool of N(0,1) draws from which large weight sets take seeded windows.

    Used only where drawing every weight afresh would take minutes on the
    host (the 32-layer decode step holds ~4.2e9 adapter weights).
    """

    def __init__(self, rng: np.random.Generator, size: int, dtype: str):
        self.vals = rng.standard_normal(size, dtype=np.float32)
        self.dtype = dtype
        self.rng = rng
        self._bf16 = {}     # inv_scale -> the whole pool divided by it, encoded once

    def take(self, shape, inv_scale: float) -> np.ndarray:
        n = int(np.prod(shape))
        off = int(self.rng.integers(0, self.vals.size - n + 1))
        if self.dtype == "bf16":
            # Encoding the scaled pool once and copying windows of it gives the
            # same bits as encoding each scaled window.
            enc = self._bf16.get(inv_scale)
            if enc is None:
                enc = self._bf16[inv_scale] = bf16_bits_from_f32(self.vals / np.float32(inv_scale))
            return enc[off:off + n].reshape(shape).copy()
        return (self.vals[off:off + n].reshape(shape) / np.float32(inv_scale)).astype(np.float32)


def _draw_adapters(rng, slots: Sequence[int], d_in: int, out_sizes: Sequence[int],
                   ranks: dict, scales: dict, a_inv: float, b_inv: float, dtype: str,
                   pool: Optional[_Pool] = None) -> dict:
    out = {}
    for k in slots:
        r = int(ranks[k])
        As, Bs = [], []
        for d_out in out_sizes:
            if pool is None:
                As.append(_normal(rng, (d_in, r), a_inv, dtype))
                Bs.append(_normal(rng, (r, d_out), b_inv, dtype))
            else:
                As.append(pool.take((d_in, r), a_inv))
                Bs.append(pool.take((r, d_out), b_inv))
        out[int(k)] = Adapter(rank=r, scale=float(scales[k]), A=As, B=Bs)
    return out


def make_instance(name: str, seed: Optional[int] = None, *, num_tokens: Optional[int] = None,
                  d_in: Optional[int] = None, out_sizes: Optional[Sequence[int]] = None,
                  num_slots: Optional[int] = None, r_max: Optional[int] = None,
                  req_lengths: Optional[Sequence[int]] = None,
                  dtype: Optional[str] = None) -> Instance:
    """Build a seeded instance of one of the named workloads.

    Keyword overrides shrink a workload for tests (fewer tokens, narrower
    projections) while keeping its structure: the slot-0 share, the
    popularity law, the rank mix and the value distributions.
    Config i uses seed i (``toy_fp32`` seed 0) unless ``seed`` is given.
    """
    default_seed = {"toy_fp32": 0, "decode_qkv": 2, "prefill_gate_up": 3,
                    "mixed_o_proj": 4, "full_decode": 5, "logits_lm_head": 6, "embed_lookup": 7}
    if name not in default_seed:
        raise ValueError(f"unknown workload {name!r}")
    rng = np.random.Generator(np.random.PCG64(default_seed[name] if seed is None else seed))

    if name == "toy_fp32":
        dt = dtype or "f32"
        D = d_in or 256
        outs = list(out_sizes or [256])
        S = num_slots or 8
        R = r_max or 16
        lengths = np.asarray(req_lengths if req_lengths is not None else [1, 1, 37, 1, 12, 1], np.int64)
        slots = rng.integers(0, S, size=len(lengths)).astype(np.int32)
        ranks = {k: R for k in range(1, S)}
        scales = {k: 2.0 for k in range(1, S)}
        adapters = _draw_adapters(rng, range(1, S), D, outs, ranks, scales, 16.0, 4.0, dt)
        x_inv, a_note = 1.0, "A~N/16, B~N/4"
    elif name == "decode_qkv":
        dt = dtype or "bf16"
        D = d_in or 4096
        outs = list(out_sizes or [4096, 1024, 1024])
        S = num_slots or 64
        R = r_max or 16
        T = num_tokens or 256
        lengths = np.asarray(req_lengths if req_lengths is not None else np.ones(T), np.int64)
        n = len(lengths)
        none = rng.random(n) < 0.10
        slots = np.where(none, 0, rng.integers(1, S, size=n)).astype(np.int32)
        ranks = {k: R for k in range(1, S)}
        scales = {k: 1.0 for k in range(1, S)}
        adapters = _draw_adapters(rng, range(1, S), D, outs, ranks, scales, 64.0, 16.0, dt)
        x_inv, a_note = 1.0, "A~N/64, B~N/16"
    elif name == "prefill_gate_up":
        dt = dtype or "bf16"
        D = d_in or 4096
        outs = list(out_sizes or [14336, 14336])
        S = num_slots or 32
        R = r_max or 64
        if req_lengths is not None:
            lengths = np.asarray(req_lengths, np.int64)
        else:
            lengths = rng.integers(128, 2049, size=16).astype(np.int64)
            if num_tokens is not None:     # shrink proportionally, keep >= 1 per request
                lengths = np.maximum(1, (lengths * num_tokens) // max(1, int(lengths.sum())))
        p = zipf_probs(S - 1, 1.1)
        slots = (1 + rng.choice(S - 1, size=len(lengths), p=p)).astype(np.int32)
        ranks = {k: R for k in range(1, S)}
        scales = {k: 1.0 for k in range(1, S)}
        adapters = _draw_adapters(rng, range(1, S), D, outs, ranks, scales, 64.0, 16.0, dt)
        x_inv, a_note = 1.0, "A~N/64, B~N/16"
    elif name == "mixed_o_proj":
        dt = dtype or "bf16"
        D = d_in or 4096
        outs = list(out_sizes or [4096])
        S = num_slots or 128
        R = r_max or 64
        if req_lengths is not None:
            lengths = np.asarray(req_lengths, np.int64)
        else:
            n_dec = num_tokens if num_tokens is not None else 1024
            chunk = 512 if num_tokens is None else max(1, num_tokens // 2)
            lengths = np.asarray([1] * n_dec + [chunk] * 4, np.int64)
        p = zipf_probs(S - 1, 1.1)
        n = len(lengths)
        none = rng.random(n) < 0.05
        slots = np.where(none, 0, 1 + rng.choice(S - 1, size=n, p=p)).astype(np.int32)
        rank_choices = [r for r in (8, 16, 32, 64) if r <= R] or [R]
        ranks = {k: int(rank_choices[rng.integers(0, len(rank_choices))]) for k in range(1, S)}
        scales = {k: 2.0 * ranks[k] / ranks[k] for k in range(1, S)}   # alpha/r with alpha = 2r
        adapters = _draw_adapters(rng, range(1, S), D, outs, ranks, scales, 64.0, 16.0, dt)
        x_inv, a_note = 1.0, "A~N/64, B~N/16"
    elif name == "logits_lm_head":
        # The sampled rows' hidden states and logits: one row per request (the
        # last token of a prefill request, the token of a decode request).
        dt = dtype or "bf16"
        D = d_in or 4096
        outs = list(out_sizes or [128256])
        S = num_slots or 64
        R = r_max or 16
        n = num_tokens or 256
        lengths = np.asarray(req_lengths if req_lengths is not None else np.ones(n), np.int64)
        none = rng.random(len(lengths)) < 0.10
        slots = np.where(none, 0, rng.integers(1, S, size=len(lengths))).astype(np.int32)
        ranks = {k: R for k in range(1, S)}
        scales = {k: 1.0 for k in range(1, S)}
        adapters = _draw_adapters(rng, range(1, S), D, outs, ranks, scales, 64.0, 16.0, dt)
        x_inv, a_note = 1.0, "A~N/64, B~N/16"
    elif name == "embed_lookup":
        # d_in is the vocabulary: A[a] holds one r-vector per token id.
        dt = dtype or "bf16"
        D = d_in or 128256
        outs = list(out_sizes or [4096])
        S = num_slots or 64
        R = r_max or 16
        n = num_tokens or 256
        lengths = np.asarray(req_lengths if req_lengths is not None else np.ones(n), np.int64)
        none = rng.random(len(lengths)) < 0.10
        slots = np.where(none, 0, rng.integers(1, S, size=len(lengths))).astype(np.int32)
        ranks = {k: R for k in range(1, S)}
        scales = {k: 1.0 for k in range(1, S)}
        adapters = _draw_adapters(rng, range(1, S), D, outs, ranks, scales, 1.0, 16.0, dt)
        T = int(lengths.sum())
        ids = rng.integers(0, D, size=T).astype(np.int32)
        x = np.zeros((T, 0), np.uint16 if dt == "bf16" else np.float32)
        y_in = _normal(rng, (T, int(sum(outs))), 1.0, dt)
        return Instance(name=name, dtype=dt, d_in=D, out_sizes=outs, num_slots=S, r_max=R, adapters=adapters,
                        req_lengths=lengths, req_slots=slots, x=x, y_in=y_in, token_ids=ids,
                        meta={"seed": default_seed[name] if seed is None else seed,
                              "values": "token ids U[0, vocab), y_in~N(0,1), A~N(0,1), B~N/16"})
    else:  # full_decode: one (layer, group); see full_decode_groups for the whole step
        raise ValueError("full_decode is built per (layer, group) by full_decode_groups()")

    T = int(lengths.sum())
    x = _normal(rng, (T, D), x_inv, dt)
    y_in = _normal(rng, (T, int(sum(outs))), 1.0, dt)
    inst = Instance(name=name, dtype=dt, d_in=D, out_sizes=outs, num_slots=S, r_max=R,
                    adapters=adapters, req_lengths=lengths, req_slots=slots, x=x, y_in=y_in,
                    meta={"seed": default_seed[name] if seed is None else seed,
                          "values": "x~N(0,1), y_in~N(0,1), " + a_note})
    return inst


# The 32-layer decode step: 7 projections run as 4 packed groups per layer.
FULL_DECODE_GROUPS = (
    ("qkv", 4096, (4096, 1024, 1024)),
    ("o", 4096, (4096,)),
    ("gate_up", 4096, (14336, 14336)),
    ("down", 14336, (4096,)),
)


def full_decode_groups(seed: int = 5, *, layers: int = 32, num_tokens: int = 512,
                       num_adapters: int = 100, rank: int = 16, dtype: str = "bf16",
                       groups=FULL_DECODE_GROUPS, pool_size: int = 1 << 26):
    """Yield one Instance per (layer, group) of the full-model decode step.

    All groups share the token->slot mapping (a slot holds the same adapter on
    every layer); x and y_in are fresh per (layer, group). Weights are seeded
    windows of a shared N(0,1) pool (see ``_Pool``).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    S = num_adapters + 1
    slots = rng.integers(1, S, size=num_tokens).astype(np.int32)
    lengths = np.ones(num_tokens, np.int64)
    pool = _Pool(rng, pool_size, dtype)
    ranks = {k: rank for k in range(1, S)}
    scales = {k: 1.0 for k in range(1, S)}
    for layer in range(layers):
        for gname, d_in, outs in groups:
            adapters = _draw_adapters(rng, range(1, S), d_in, outs, ranks, scales, 64.0, 16.0,
                                      dtype, pool=pool)
            x = pool.take((num_tokens, d_in), 1.0)
            y_in = pool.take((num_tokens, int(sum(outs))), 1.0)
            yield Instance(name=f"full_decode/L{layer}/{gname}", dtype=dtype, d_in=d_in,
                           out_sizes=list(outs), num_slots=S, r_max=rank, adapters=adapters,
                           req_lengths=lengths, req_slots=slots, x=x, y_in=y_in,
                           meta={"seed": seed, "layer": layer, "group": gname})


def sampled_rows(req_lengths) -> np.ndarray:
    """Batch indices of the rows sampled this step: the last token of every
    request (for a one-token decode request, its only token), in request order.
    The lm_head LoRA runs on these rows only, each with its request's slot."""
    lengths = np.asarray(req_lengths, np.int64)
    if (lengths < 1).any():
        raise ValueError("every request has at least one token")
    return (np.cumsum(lengths) - 1).astype(np.int64)


def split_requests(req_lengths: np.ndarray, world_size: int, rank: int) -> np.ndarray:
    """Indices of the requests that data-parallel rank ``rank`` of ``world_size`` serves.

    Requests are dealt round-robin, so every rank gets a batch of the same
    shape law; no request is split across ranks.
    """
    if world_size < 1 or not (0 <= rank < world_size):
        raise ValueError("bad world_size/rank")
    return np.arange(len(req_lengths))[rank::world_size]


def toy_page_instance():
    """The toy batch exactly as the handbook page draws it.

    Draw order and shapes follow the page's script (section "不合并权重，批量计算"):
    with torch's CPU generator seeded 0, W [256,256]/16, then A [8,256,16]/16,
    B [8,16,256]/4, then x [53,256]; requests of lengths [1,1,37,1,12,1] use
    adapters [3,5,3,0,7,5] and scale 2.0. Returns float32 numpy arrays.
    On the page adapter 0 is a real adapter.
    """
    import torch
    g = torch.Generator().manual_seed(0)
    W = torch.randn(256, 256, generator=g) / 16
    A = torch.randn(8, 256, 16, generator=g) / 16
    B = torch.randn(8, 16, 256, generator=g) / 4
    lengths = [1, 1, 37, 1, 12, 1]
    adapters = [3, 5, 3, 0, 7, 5]
    x = torch.randn(sum(lengths), 256, generator=g)
    return dict(W=W.numpy(), A=A.numpy(), B=B.numpy(), x=x.numpy(), lengths=lengths,
                adapters=adapters, scale=2.0)


@dataclass
class MoEInstance:
    """One mixture-of-experts layer's LoRA inputs (routing, tables, activations).

    ``w13`` and ``w2`` are the two applications as dense-layer instances over
    the (token, choice) pairs (p = t * topk + k): their slot tables hold the
    composite (adapter, local expert) slots 1 + (a - 1) * local_experts + j,
    ``w2.x`` is the per-pair input h2 and ``w2.y_in`` / ``w13.y_in`` the
    pairs' base outputs; ``w13.x`` holds the token rows [T, hidden] (the w13
    LoRA row of pair p reads token row p // topk). The pairs' composite slots
    are not computed here: ``routed(layer, pair_slot)`` gives a layer whose
    requests are the pairs with the slots the caller computed.
    """
    name: str
    hidden: int
    inter: int
    num_experts: int
    local_experts: int
    ep_rank: int
    topk: int
    num_loras: int
    token_slot: np.ndarray          # int32 [T]: adapter slot of every token (0 = none)
    topk_ids: np.ndarray            # int32 [T, topk]: chosen global expert ids
    expert_map: Optional[np.ndarray]  # int32 [num_experts]: local index or -1 (None: all local)
    w13: Instance                   # requests: the pairs, all with slot 0 until routed()
    w2: Instance

    @property
    def num_tokens(self) -> int:
        return int(self.token_slot.size)

    @staticmethod
    def routed(layer: Instance, pair_slot: np.ndarray) -> Instance:
        """The layer with one request per pair carrying the given composite slot."""
        return Instance(name=layer.name, dtype=layer.dtype, d_in=layer.d_in, out_sizes=layer.out_sizes,
                        num_slots=layer.num_slots, r_max=layer.r_max, adapters=layer.adapters,
                        req_lengths=layer.req_lengths, req_slots=np.asarray(pair_slot, np.int32).copy(),
                        x=layer.x, y_in=layer.y_in, meta=dict(layer.meta))


def make_moe_instance(name: str = "moe_decode", seed: Optional[int] = None, *, num_tokens: Optional[int] = None,
                      hidden: Optional[int] = None, inter: Optional[int] = None,
                      num_experts: Optional[int] = None, local_experts: Optional[int] = None, ep_rank: int = 0,
                      topk: Optional[int] = None, num_loras: Optional[int] = None,
                      r_max: Optional[int] = None) -> MoEInstance:
    """A seeded MoE-layer instance; keyword overrides shrink it for tests.

    Tokens: slot 0 with probability 10%, else uniform over adapters 1..num_loras.
    Routing: each token's topk distinct experts uniform over all experts.
    Expert parallelism: rank ep_rank holds experts [ep_rank * L, (ep_rank + 1) * L).
    Weights: A ~ N(0,1)/64, B ~ N(0,1)/16 (seeded windows of a N(0,1) pool),
    every composite slot rank r_max, scale 1.0; x, h2 and base outputs ~ N(0,1).
    """
    if name != "moe_decode":
        raise ValueError(f"unknown MoE workload {name!r}")
    rng = np.random.Generator(np.random.PCG64(8 if seed is None else seed))
    T = num_tokens or 256
    H, I = hidden or 7168, inter or 2048
    E = num_experts or 256
    L = local_experts or 32
    K = topk or 8
    NL = num_loras or 4
    R = r_max or 64
    dt = "bf16"
    ts = rng.integers(1, NL + 1, size=T).astype(np.int32)
    ts[rng.random(T) < 0.10] = 0
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)
    start = ep_rank * L
    emap = None
    if L < E:
        emap = np.full(E, -1, dtype=np.int32)
        emap[start:start + L] = np.arange(L, dtype=np.int32)
    S = 1 + NL * L
    none = np.zeros(T * K, dtype=np.int32)
    pool = _Pool(rng, min(1 << 26, max(1 << 20, 4 * S * R * (2 * H + I + 2 * I + H))), dt)
    ranks = {k: R for k in range(1, S)}
    scales = {k: 1.0 for k in range(1, S)}
    ad13 = _draw_adapters(rng, range(1, S), H, [I, I], ranks, scales, 64.0, 16.0, dt, pool=pool)
    ad2 = _draw_adapters(rng, range(1, S), I, [H], ranks, scales, 64.0, 16.0, dt, pool=pool)
    ones = np.ones(T * K, np.int64)
    x = pool.take((T, H), 1.0)
    w13 = Instance(name=f"{name}/w13", dtype=dt, d_in=H, out_sizes=[I, I], num_slots=S, r_max=R, adapters=ad13,
                   req_lengths=ones, req_slots=none.copy(), x=x, y_in=pool.take((T * K, 2 * I), 1.0),
                   meta={"x_row_div": K})
    w2 = Instance(name=f"{name}/w2", dtype=dt, d_in=I, out_sizes=[H], num_slots=S, r_max=R, adapters=ad2,
                  req_lengths=ones, req_slots=none.copy(), x=pool.take((T * K, I), 1.0),
                  y_in=pool.take((T * K, H), 1.0))
    return MoEInstance(name=name, hidden=H, inter=I, num_experts=E, local_experts=L, ep_rank=ep_rank, topk=K,
                       num_loras=NL, token_slot=ts, topk_ids=ids, expert_map=emap, w13=w13, w2=w2)
