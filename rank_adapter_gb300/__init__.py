"""Python binding of the rank_adapter_gb300 C ABI (``include/lora.h``).

Argument marshalling only: every step of the multi-LoRA path runs in the
library's sm_103a kernels. PyTorch provides device memory and streams. There
is no CPU fallback: importing this package fails loudly if the shared library
has not been built (``__graft_entry__.build()`` or
``python rank_adapter_gb300/build_lib.py``).

Low-level functions carry the C names and return the C status codes
(``lora_set_slot``, ``lora_reset_slot``, ``lora_prepare_meta``,
``lora_shrink``, ``lora_expand``, ``lora_embed_shrink``, ``lora_workspace_bytes``,
``lora_meta_tiles_bytes``, ``lora_query_status``, ``lora_strerror``,
``lora_last_cuda_error``). ``SlotTable`` and ``TokenMeta`` own torch buffers
laid out as the ABI wants and call those functions; ``shrink`` / ``expand``
raise ``LoraError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

__all__ = [
    "LORA_OK", "LORA_EINVAL", "LORA_ERANGE", "LORA_EALIGN", "LORA_EUNSUPPORTED", "LORA_ECUDA",
    "LORA_EBADSLOT", "LORA_EDEVICE", "LORA_EBADTOKEN", "LORA_F32", "LORA_BF16", "LORA_AUTO", "LORA_BGMV", "LORA_SGMV", "LORA_MIXED",
    "LORA_MAX_SLICES", "LORA_MAX_NUM_SLOTS", "LORA_MAX_RANK", "LORA_SGMV_MIN_ROWS", "LORA_SGMV_TILE_M",
    "LORA_AUTO_SGMV_MIN_TOKENS", "LORA_AUTO_SGMV_MIN_AVG", "LORA_AUTO_LONG_ROWS",
    "LayerDesc", "Meta", "LoraError", "lib_path", "exported_symbols",
    "lora_set_slot", "lora_reset_slot", "lora_prepare_meta", "lora_prepare_meta_unshared", "lora_shrink", "lora_expand", "lora_apply",
    "lora_shrink_noalloc", "lora_noalloc_scratch_bytes", "lora_embed_shrink", "embed_shrink",
    "lora_moe_pair_slots", "moe_pair_slots",
    "lora_workspace_bytes", "lora_meta_tiles_bytes", "lora_query_status", "lora_probe_bounded_wait", "lora_strerror",
    "lora_last_cuda_error", "lora_launch_count", "SlotTable", "TokenMeta", "shrink", "expand", "apply", "workspace", "check",
]

(LORA_OK, LORA_EINVAL, LORA_ERANGE, LORA_EALIGN, LORA_EUNSUPPORTED, LORA_ECUDA, LORA_EBADSLOT, LORA_EDEVICE,
 LORA_EBADTOKEN) = range(9)
LORA_F32, LORA_BF16 = 0, 1
LORA_AUTO, LORA_BGMV, LORA_SGMV, LORA_MIXED = 0, 1, 2, 3
LORA_MAX_SLICES = 4
LORA_MAX_NUM_SLOTS = 1024
LORA_MAX_RANK = 128
LORA_MAX_TOKENS = 1 << 24
LORA_SGMV_MIN_ROWS = 32
LORA_SGMV_TILE_M = 128
LORA_AUTO_SGMV_MIN_TOKENS = 1024
LORA_AUTO_SGMV_MIN_AVG = 20
LORA_AUTO_LONG_ROWS = 64

_HERE = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_HERE, "_lib", "librank_adapter_gb300.so")


if not os.path.exists(lib_path()):
    raise ImportError(
        f"rank_adapter_gb300: {lib_path()} is missing; build it with "
        "`python -c 'import __graft_entry__ as g; g.build()'` (there is no CPU fallback)")

_lib = ctypes.CDLL(lib_path())

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class LayerDesc(ctypes.Structure):
    """lora_layer_desc: one projection's stacked slot table (device pointers)."""
    _fields_ = [
        ("dtype", _i32), ("d_in", _i32), ("n_slices", _i32),
        ("out_sizes", _i32 * LORA_MAX_SLICES), ("num_slots", _i32), ("r_max", _i32),
        ("A", _vp * LORA_MAX_SLICES), ("B", _vp * LORA_MAX_SLICES),
        ("slot_rank", _vp), ("slot_scale", _vp), ("x_row_div", _i32),
    ]


class Meta(ctypes.Structure):
    """lora_meta: per-step token metadata (device pointers)."""
    _fields_ = [
        ("token_slot", _vp), ("num_tokens", _i32), ("num_slots", _i32),
        ("sorted_rows", _vp), ("seg_slot", _vp), ("seg_count", _vp), ("seg_start", _vp),
        ("num_segs", _vp), ("no_lora", _vp), ("status", _vp),
        ("tiles", _vp), ("tiles_bytes", ctypes.c_size_t),
    ]


_P = ctypes.POINTER
_sig = {
    "lora_set_slot": (_i32, [_P(LayerDesc), _i32, _i32, ctypes.c_float, _P(_vp), _P(_vp), _vp]),
    "lora_reset_slot": (_i32, [_P(LayerDesc), _i32, _vp]),
    "lora_prepare_meta": (_i32, [_P(Meta), _vp]),
    "lora_prepare_meta_unshared": (_i32, [_P(Meta), _vp]),
    "lora_shrink": (_i32, [_P(LayerDesc), _P(Meta), _vp, ctypes.c_int64, _vp, _i32, _vp, ctypes.c_size_t, _vp]),
    "lora_expand": (_i32, [_P(LayerDesc), _P(Meta), _vp, _vp, ctypes.c_int64, _i32, _i32, _vp]),
    "lora_apply": (_i32, [_P(LayerDesc), _P(Meta), _vp, ctypes.c_int64, _vp, _vp, ctypes.c_int64, _i32, _i32, _vp,
                          ctypes.c_size_t, _vp]),
    "lora_shrink_noalloc": (_i32, [_P(LayerDesc), _P(Meta), _vp, ctypes.c_int64, _vp, _vp]),
    "lora_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "lora_workspace_bytes": (ctypes.c_size_t, [_P(LayerDesc), _i32, _i32]),
    "lora_meta_tiles_bytes": (ctypes.c_size_t, [_i32]),
    "lora_query_status": (_i32, [_P(Meta), _P(_i32), _vp]),
    "lora_probe_bounded_wait": (_i32, [_P(Meta), ctypes.c_uint32, _vp]),
    "lora_embed_shrink": (_i32, [_P(LayerDesc), _P(Meta), _vp, _vp, _vp]),
    "lora_moe_pair_slots": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "lora_strerror": (ctypes.c_char_p, [_i32]),
    "lora_last_cuda_error": (_i32, []),
    "lora_launch_count": (ctypes.c_uint64, []),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def exported_symbols() -> Sequence[str]:
    """The C entry points this binding resolves from the library."""
    return tuple(_sig)


class LoraError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = lora_strerror(status)
        if status == LORA_ECUDA:
            msg += f" (cudaError {lora_last_cuda_error()})"
        super().__init__(f"{what}: {msg}" if what else msg)


def check(status: int, what: str = "") -> None:
    if status != LORA_OK:
        raise LoraError(status, what)


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptrs(seq, n=LORA_MAX_SLICES):
    arr = (_vp * n)()
    for i, p in enumerate(seq):
        arr[i] = None if p is None else (p.data_ptr() if hasattr(p, "data_ptr") else int(p))
    return arr


# ----------------------------------------------------------------------------- C-named functions

def lora_set_slot(desc: LayerDesc, slot: int, rank: int, scale: float, A_src, B_src, stream=None) -> int:
    return _lib.lora_set_slot(ctypes.byref(desc), slot, rank, scale, _ptrs(A_src), _ptrs(B_src), _stream(stream))


def lora_reset_slot(desc: LayerDesc, slot: int, stream=None) -> int:
    return _lib.lora_reset_slot(ctypes.byref(desc), slot, _stream(stream))


def lora_prepare_meta(meta: Meta, stream=None) -> int:
    return _lib.lora_prepare_meta(ctypes.byref(meta), _stream(stream))


def lora_prepare_meta_unshared(meta: Meta, stream=None) -> int:
    return _lib.lora_prepare_meta_unshared(ctypes.byref(meta), _stream(stream))


def lora_shrink(desc: LayerDesc, meta: Meta, x: int, ldx: int, buf: int, kind: int = LORA_AUTO,
                ws: int = 0, ws_bytes: int = 0, stream=None) -> int:
    return _lib.lora_shrink(ctypes.byref(desc), ctypes.byref(meta), x, ldx, buf, kind, ws or None,
                            ws_bytes, _stream(stream))


def lora_expand(desc: LayerDesc, meta: Meta, buf: int, y: int, ldy: int, y_dtype: int,
                kind: int = LORA_AUTO, stream=None) -> int:
    return _lib.lora_expand(ctypes.byref(desc), ctypes.byref(meta), buf, y, ldy, y_dtype, kind, _stream(stream))


def lora_apply(desc: LayerDesc, meta: Meta, x: int, ldx: int, buf: int, y: int, ldy: int, y_dtype: int,
               kind: int = LORA_AUTO, ws: int = 0, ws_bytes: int = 0, stream=None) -> int:
    return _lib.lora_apply(ctypes.byref(desc), ctypes.byref(meta), x, ldx, buf or None, y, ldy, y_dtype, kind,
                           ws or None, ws_bytes, _stream(stream))


def lora_embed_shrink(desc: LayerDesc, meta: Meta, token_id: int, buf: int, stream=None) -> int:
    """Embedding lookup: buf[0, t] = scale * A[slot t][token_id[t]] for LoRA tokens."""
    return _lib.lora_embed_shrink(ctypes.byref(desc), ctypes.byref(meta), token_id, buf, _stream(stream))


def lora_moe_pair_slots(token_slot: int, topk_ids: int, num_tokens: int, topk: int, num_loras: int,
                        num_experts: int, local_experts: int, expert_map: int, pair_slot: int, stream=None) -> int:
    """Composite (adapter, local expert) slot of every (token, choice) pair (see the header)."""
    return _lib.lora_moe_pair_slots(token_slot, topk_ids, num_tokens, topk, num_loras, num_experts, local_experts,
                                    expert_map, pair_slot, _stream(stream))


def lora_shrink_noalloc(desc: LayerDesc, meta: Meta, x: int, ldx: int, buf: int, stream=None) -> int:
    """lora_shrink (BGMV family) with its scratch in the library's fixed device array; allocates nothing."""
    return _lib.lora_shrink_noalloc(ctypes.byref(desc), ctypes.byref(meta), x, ldx, buf, _stream(stream))


def lora_noalloc_scratch_bytes() -> int:
    return int(_lib.lora_noalloc_scratch_bytes())


def lora_workspace_bytes(desc: LayerDesc, max_tokens: int, kind: int = LORA_AUTO) -> int:
    return int(_lib.lora_workspace_bytes(ctypes.byref(desc), max_tokens, kind))


def lora_meta_tiles_bytes(num_slots: int) -> int:
    return int(_lib.lora_meta_tiles_bytes(num_slots))


def lora_query_status(meta: Meta, stream=None):
    """Returns (status_code, bad_token_count); synchronises the stream."""
    out = _i32(0)
    st = _lib.lora_query_status(ctypes.byref(meta), ctypes.byref(out), _stream(stream))
    return st, int(out.value)


def lora_probe_bounded_wait(meta: Meta, limit_us: int, stream=None) -> int:
    return _lib.lora_probe_bounded_wait(ctypes.byref(meta), limit_us, _stream(stream))


def lora_strerror(status: int) -> str:
    return _lib.lora_strerror(status).decode()


def lora_last_cuda_error() -> int:
    return int(_lib.lora_last_cuda_error())


def lora_launch_count() -> int:
    """Kernels the library has launched in this process (graph captures count once)."""
    return int(_lib.lora_launch_count())


# ----------------------------------------------------------------------------- torch-owned buffers

def _torch_dtype(dtype: int):
    import torch
    return torch.bfloat16 if dtype == LORA_BF16 else torch.float32


class SlotTable:
    """Stacked slot table of one (packed) projection, in caller-owned torch memory.

    ``A[s]``: [num_slots, d_in, r_max]; ``B[s]``: [num_slots, r_max, out_sizes[s]];
    ``slot_rank`` int32 [num_slots]; ``slot_scale`` fp32 [num_slots]. All start
    zeroed, so every slot begins empty (rank 0) and slot 0 stays the no-LoRA slot.
    """

    def __init__(self, d_in: int, out_sizes: Sequence[int], num_slots: int, r_max: int,
                 dtype: int = LORA_BF16, device="cuda", x_row_div: int = 1):
        import torch
        td = _torch_dtype(dtype)
        self.dtype, self.d_in, self.out_sizes = dtype, d_in, list(out_sizes)
        self.num_slots, self.r_max = num_slots, r_max
        self.A = [torch.zeros(num_slots, d_in, r_max, dtype=td, device=device) for _ in out_sizes]
        self.B = [torch.zeros(num_slots, r_max, d, dtype=td, device=device) for d in out_sizes]
        self.slot_rank = torch.zeros(num_slots, dtype=torch.int32, device=device)
        self.slot_scale = torch.zeros(num_slots, dtype=torch.float32, device=device)
        d = LayerDesc()
        d.dtype, d.d_in, d.n_slices = dtype, d_in, len(out_sizes)
        for i, w in enumerate(out_sizes):
            d.out_sizes[i] = w
            d.A[i] = self.A[i].data_ptr()
            d.B[i] = self.B[i].data_ptr()
        d.num_slots, d.r_max = num_slots, r_max
        d.slot_rank, d.slot_scale = self.slot_rank.data_ptr(), self.slot_scale.data_ptr()
        d.x_row_div = x_row_div   # LoRA row i reads x row i // x_row_div (an MoE w13 layer: topk)
        self.desc = d

    @property
    def d_out_total(self) -> int:
        return sum(self.out_sizes)

    def set_slot(self, slot: int, rank: int, scale: float, A_src, B_src, stream=None) -> None:
        check(lora_set_slot(self.desc, slot, rank, scale, A_src, B_src, stream), "lora_set_slot")

    def reset_slot(self, slot: int, stream=None) -> None:
        check(lora_reset_slot(self.desc, slot, stream), "lora_reset_slot")

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.A + self.B)


class TokenMeta:
    """Device buffers of lora_meta for up to ``max_tokens`` tokens and a table of ``num_slots``."""

    def __init__(self, max_tokens: int, num_slots: int, device="cuda"):
        import torch
        i32 = dict(dtype=torch.int32, device=device)
        self.max_tokens, self.num_slots = max_tokens, num_slots
        self.token_slot = torch.zeros(max(1, max_tokens), **i32)
        self.sorted_rows = torch.zeros(max(1, max_tokens), **i32)
        self.seg_slot = torch.zeros(num_slots, **i32)
        self.seg_count = torch.zeros(num_slots, **i32)
        self.seg_start = torch.zeros(num_slots + 1, **i32)
        self.scalars = torch.zeros(4, **i32)        # num_segs, no_lora, status, (pad)
        nb = lora_meta_tiles_bytes(num_slots)
        self.tiles = torch.zeros((nb + 3) // 4, **i32)
        m = Meta()
        m.token_slot = self.token_slot.data_ptr()
        m.num_tokens = 0
        m.num_slots = num_slots
        m.sorted_rows = self.sorted_rows.data_ptr()
        m.seg_slot, m.seg_count, m.seg_start = (self.seg_slot.data_ptr(), self.seg_count.data_ptr(),
                                                self.seg_start.data_ptr())
        base = self.scalars.data_ptr()
        m.num_segs, m.no_lora, m.status = base, base + 4, base + 8
        m.tiles, m.tiles_bytes = self.tiles.data_ptr(), nb
        self.c = m

    def set_num_tokens(self, n: int) -> None:
        if not 0 <= n <= self.max_tokens:
            raise ValueError(f"num_tokens {n} outside [0, {self.max_tokens}]")
        self.c.num_tokens = n

    def prepare(self, token_slot=None, stream=None, unshared=False) -> None:
        """Copy ``token_slot`` (int32 device tensor) in if given, then run lora_prepare_meta
        (lora_prepare_meta_unshared when ``unshared``: no kernel of the previous library call on
        the stream reads this metadata)."""
        if token_slot is not None:
            n = int(token_slot.numel())
            self.set_num_tokens(n)
            if n:
                self.token_slot[:n].copy_(token_slot, non_blocking=True)
        if unshared:
            check(lora_prepare_meta_unshared(self.c, stream), "lora_prepare_meta_unshared")
        else:
            check(lora_prepare_meta(self.c, stream), "lora_prepare_meta")

    @property
    def num_segs(self):
        return self.scalars[0]

    @property
    def no_lora(self):
        return self.scalars[1]

    @property
    def status(self):
        return self.scalars[2]


def workspace(table: SlotTable, max_tokens: int, kind: int = LORA_AUTO, device="cuda"):
    """A caller-owned scratch tensor of lora_workspace_bytes() bytes (None when 0)."""
    import torch
    nb = lora_workspace_bytes(table.desc, max_tokens, kind)
    return torch.empty((nb + 15) // 16 * 4, dtype=torch.float32, device=device) if nb else None


def _ws_args(table, meta, kind, ws):
    if ws is None:
        ws = workspace(table, meta.c.num_tokens, kind)
    if ws is None:
        return 0, 0, None
    return ws.data_ptr(), ws.numel() * ws.element_size(), ws


def shrink(table: SlotTable, meta: TokenMeta, x, buf, kind: int = LORA_AUTO, stream=None,
           ws=None) -> None:
    """buf[s, t, :] = scale * x[t] @ A_s[slot t] for LoRA tokens (see lora_shrink).

    ws: scratch from workspace(); allocated per call when omitted."""
    wsp, wsb, _keep = _ws_args(table, meta, kind, ws)
    check(lora_shrink(table.desc, meta.c, x.data_ptr(), x.stride(0), buf.data_ptr(), kind, wsp, wsb, stream),
          "lora_shrink")


def embed_shrink(table: SlotTable, meta: TokenMeta, token_id, buf, stream=None) -> None:
    """buf[0, t, :] = scale * A[slot t][token_id[t], :] for LoRA tokens (see lora_embed_shrink)."""
    check(lora_embed_shrink(table.desc, meta.c, token_id.data_ptr(), buf.data_ptr(), stream), "lora_embed_shrink")


def moe_pair_slots(token_slot, topk_ids, num_loras: int, num_experts: int, local_experts: int, expert_map=None,
                   pair_slot=None, stream=None):
    """pair_slot [T * topk] int32 (allocated when omitted) for token_slot [T] and topk_ids [T, topk]."""
    import torch
    T, topk = int(topk_ids.shape[0]), int(topk_ids.shape[1])
    if pair_slot is None:
        pair_slot = torch.empty(T * topk, dtype=torch.int32, device=topk_ids.device)
    check(lora_moe_pair_slots(token_slot.data_ptr() if T else 0, topk_ids.data_ptr() if T else 0, T, topk,
                              num_loras, num_experts, local_experts,
                              expert_map.data_ptr() if expert_map is not None else 0,
                              pair_slot.data_ptr() if T else 0, stream), "lora_moe_pair_slots")
    return pair_slot


def expand(table: SlotTable, meta: TokenMeta, buf, y, kind: int = LORA_AUTO, stream=None) -> None:
    """y[t, off_s:] += buf[s, t] @ B_s[slot t] for LoRA tokens (see lora_expand)."""
    import torch
    ydt = LORA_BF16 if y.dtype == torch.bfloat16 else LORA_F32
    check(lora_expand(table.desc, meta.c, buf.data_ptr(), y.data_ptr(), y.stride(0), ydt, kind, stream),
          "lora_expand")


def apply(table: SlotTable, meta: TokenMeta, x, y, buf=None, kind: int = LORA_AUTO, stream=None,
          ws=None) -> None:
    """Fused shrink + expand: y[t, off_s:] += (scale * x[t] @ A_s) @ B_s (see lora_apply).

    ws: scratch from workspace(); allocated per call when omitted."""
    import torch
    ydt = LORA_BF16 if y.dtype == torch.bfloat16 else LORA_F32
    wsp, wsb, _keep = _ws_args(table, meta, kind, ws)
    check(lora_apply(table.desc, meta.c, x.data_ptr(), x.stride(0), buf.data_ptr() if buf is not None else 0,
                     y.data_ptr(), y.stride(0), ydt, kind, wsp, wsb, stream), "lora_apply")
