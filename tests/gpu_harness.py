"""Shared plumbing of the GPU parity tests: move a seeded workload onto the
device through the C ABI, run the library's shrink / expand, and compare with
the fp64 oracle under the tolerances the tests state.

Tolerances (the reading of "max |diff| <= 1e-2 x RMS of the oracle delta" for
bf16 inputs and 1e-5 for the fp32 workload):
* fp32 y: max |y_gpu - y_ref| <= tol * RMS(delta), delta = y_ref - y_in over
  the rows that carry a live adapter;
* bf16 y: the same plus half a bf16 ulp of y_ref (the one rounding of the
  stored result);
* buf: max |buf_gpu - buf_ref| <= tol * RMS(buf_ref) on written rows, the
  rank tail exactly 0, and rows of no-LoRA tokens left untouched.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import rank_adapter_gb300 as ra

TOL_BF16 = 1e-2
TOL_F32 = 1e-5


def to_dev(arr: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Stored values (bf16 bits or fp32) as a device tensor with the same bits."""
    arr = np.ascontiguousarray(arr)
    if dtype == "bf16":
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(arr.astype(np.float32, copy=False)).to(device)


def lib_dtype(inst) -> int:
    return ra.LORA_BF16 if inst.dtype == "bf16" else ra.LORA_F32


def load_table(inst, device="cuda") -> ra.SlotTable:
    """A zeroed slot table filled with the instance's adapters through lora_set_slot."""
    t = ra.SlotTable(inst.d_in, inst.out_sizes, inst.num_slots, inst.r_max, lib_dtype(inst), device)
    keep = []
    for k, ad in sorted(inst.adapters.items()):
        As = [to_dev(a, inst.dtype, device) for a in ad.A]
        Bs = [to_dev(b, inst.dtype, device) for b in ad.B]
        keep.append((As, Bs))
        t.set_slot(k, ad.rank, ad.scale, As, Bs)
    torch.cuda.synchronize()
    return t


def run_gpu(inst, table=None, kind=ra.LORA_AUTO, y_dtype="f32", token_slot=None, ldx_pad=0, ldy_pad=0,
            y_in=None, path="split"):
    """Run prepare_meta + shrink + expand (path "split") or prepare_meta +
    lora_apply (path "apply"); returns (buf, y, meta) on the host.

    buf is pre-filled with NaN so rows the shrink must not write stay NaN.
    """
    table = table or load_table(inst)
    T, D = inst.num_tokens, inst.d_in
    ts = inst.token_slot if token_slot is None else np.asarray(token_slot, np.int32)
    xs = torch.zeros(T, D + ldx_pad, dtype=torch.bfloat16 if inst.dtype == "bf16" else torch.float32,
                     device="cuda")
    xs[:, :D] = to_dev(inst.x, inst.dtype)
    x = xs[:, :D]
    y0 = inst.y_in if y_in is None else y_in
    W = inst.d_out_total
    if y_dtype == "f32":
        ys = torch.zeros(T, W + ldy_pad, dtype=torch.float32, device="cuda")
        ys[:, :W] = torch.from_numpy(inst.to_f32(y0)).cuda()
    else:
        ys = torch.zeros(T, W + ldy_pad, dtype=torch.bfloat16, device="cuda")
        ys[:, :W] = to_dev(y0, "bf16")
    y = ys[:, :W]
    meta = ra.TokenMeta(max(T, 1), inst.num_slots)
    meta.prepare(torch.from_numpy(ts).cuda())
    buf = torch.full((inst.n_slices, T, inst.r_max), float("nan"), dtype=torch.float32, device="cuda")
    if path == "split":
        ra.shrink(table, meta, x, buf, kind)
        ra.expand(table, meta, buf, y, kind)
    else:
        ra.apply(table, meta, x, y, buf=buf, kind=kind)
    torch.cuda.synchronize()
    return buf.cpu().numpy(), y.float().cpu().numpy(), meta


def oracle_ref(inst, token_slot=None, y_in=None):
    """(buf, written, y) from the fp64 oracle on the same stored values."""
    ads = oracle.adapters_f64(inst)
    if token_slot is None:
        lengths, slots = inst.req_lengths, inst.req_slots
    else:
        lengths, slots = oracle.requests_of_token_slots(token_slot)
    x64 = inst.to_f32(inst.x).astype(np.float64)
    y64 = inst.to_f32(inst.y_in if y_in is None else y_in).astype(np.float64)
    buf, written = oracle.shrink_requests(x64, ads, inst.n_slices, inst.r_max, lengths, slots, inst.num_slots)
    y = oracle.expand_requests(buf, y64, ads, inst.out_sizes, lengths, slots, inst.num_slots)
    return buf, written, y


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, e - 9)     # ulp = 2^(e-1-7); half of it


def check_parity(inst, buf_gpu, y_gpu, buf_ref, written, y_ref, tol, y_dtype="f32", y_in=None,
                 token_slot=None):
    y_in_st = inst.to_f32(inst.y_in if y_in is None else y_in)     # stored y_in (what the device held)
    y_in64 = y_in_st.astype(np.float64)
    ts = (inst.token_slot if token_slot is None else np.asarray(token_slot)).astype(np.int64)
    # buf: written rows within tolerance, rank tail exactly zero; others untouched (NaN)
    if written.any():
        bref = buf_ref[:, written]
        bgpu = buf_gpu[:, written].astype(np.float64)
        rms_b = np.sqrt(np.mean(bref ** 2))
        assert not np.isnan(bgpu).any(), "shrink left a LoRA row unwritten"
        err_b = np.max(np.abs(bgpu - bref))
        assert err_b <= tol * rms_b + 1e-30, f"buf err {err_b:.3e} > {tol:.0e} x RMS {rms_b:.3e}"
        ranks = np.zeros(inst.num_slots, np.int64)
        for k, ad in inst.adapters.items():
            ranks[k] = ad.rank
        live = (ts > 0) & (ts < inst.num_slots)
        tok_rank = np.where(live, ranks[np.clip(ts, 0, inst.num_slots - 1)], 0)
        tail = np.arange(inst.r_max)[None, None, :] >= tok_rank[None, :, None]
        tail = np.broadcast_to(tail, buf_gpu.shape) & written[None, :, None]
        assert np.all(buf_gpu[tail] == 0.0), "rank tail not exactly zero"
    assert np.isnan(buf_gpu[:, ~written]).all(), "shrink wrote a no-LoRA row"
    # y: no-LoRA rows bitwise untouched (compared as the fp32 widening of what was stored)
    assert np.array_equal(y_gpu[~written].view(np.uint32), y_in_st[~written].view(np.uint32)), \
        "expand touched a no-LoRA row"
    if written.any():
        delta = (y_ref - y_in64)[written]
        rms = np.sqrt(np.mean(delta ** 2))
        diff = np.abs(y_gpu[written].astype(np.float64) - y_ref[written])
        bound = tol * rms
        if y_dtype == "bf16":
            bound = bound + bf16_half_ulp(y_ref[written])
        worst = np.max(diff - bound)
        assert worst <= 0, f"y err exceeds bound by {worst:.3e} (max err {diff.max():.3e}, RMS delta {rms:.3e})"


def parity(inst, kind=ra.LORA_AUTO, y_dtype="f32", tol=None, table=None, **kw):
    """Run GPU and oracle on one instance and assert parity; returns the GPU results."""
    tol = tol if tol is not None else (TOL_F32 if inst.dtype == "f32" else TOL_BF16)
    buf, y, meta = run_gpu(inst, table=table, kind=kind, y_dtype=y_dtype, **kw)
    ts, y_in = kw.get("token_slot"), kw.get("y_in")
    bref, written, yref = oracle_ref(inst, token_slot=ts, y_in=y_in)
    check_parity(inst, buf, y, bref, written, yref, tol, y_dtype=y_dtype, y_in=y_in, token_slot=ts)
    return buf, y, meta
