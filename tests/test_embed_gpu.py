"""The embedding layer's LoRA through the C ABI (page "vLLM 源码完全拆解(十八):
多 LoRA 服务", section "embedding 的 LoRA 是一个查表增量"): lora_embed_shrink
looks each token's r-vector up in its slot's A table, lora_expand adds it
through B. The lookup makes one fp32 product per value (scale times a stored
weight), so buf must equal that product computed in fp32 on the host, bit for
bit; y is held to the bf16 tolerance against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_harness import TOL_BF16, bf16_half_ulp, load_table, to_dev

pytestmark = pytest.mark.gpu


def _run(lib, inst, ids, y_dtype="bf16"):
    t = load_table(inst)
    meta = lib.TokenMeta(inst.num_tokens, inst.num_slots)
    meta.prepare(torch.from_numpy(inst.token_slot).cuda())
    buf = torch.full((1, inst.num_tokens, inst.r_max), float("nan"), device="cuda")
    lib.embed_shrink(t, meta, torch.from_numpy(ids.astype(np.int32)).cuda(), buf)
    y = to_dev(inst.y_in, inst.dtype)
    if y_dtype == "f32":
        y = y.float()
    lib.expand(t, meta, buf, y, kind=lib.LORA_BGMV)
    torch.cuda.synchronize()
    status, _ = lib.lora_query_status(meta.c)
    return buf.cpu().numpy(), y.float().cpu().numpy().astype(np.float64), status


def _host_buf(inst, ids):
    """buf in fp32 on the host: scale * stored weight, rounded once."""
    T, R = inst.num_tokens, inst.r_max
    out = np.full((T, R), np.nan, np.float32)
    ts = inst.token_slot
    for t in range(T):
        a = int(ts[t])
        if a == 0:
            continue
        out[t] = 0.0
        ad = inst.adapters[a]
        v = int(ids[t])
        if 0 <= v < inst.d_in:
            row = inst.to_f32(ad.A[0][v, :ad.rank])
            out[t, :ad.rank] = np.float32(ad.scale) * row
    return out


def _check_y(inst, ids, y_gpu, y_dtype):
    ads = oracle.adapters_f64(inst)
    buf, _ = oracle.embed_requests(ids, ads, inst.r_max, inst.req_lengths, inst.req_slots, inst.num_slots)
    y_in = inst.to_f32(inst.y_in).astype(np.float64)
    y_ref = oracle.expand_requests(buf, y_in, ads, inst.out_sizes, inst.req_lengths, inst.req_slots,
                                   inst.num_slots)
    live = inst.token_slot != 0
    rms = np.sqrt(np.mean((y_ref[live] - y_in[live]) ** 2))
    bound = TOL_BF16 * rms + (bf16_half_ulp(y_ref) if y_dtype == "bf16" else 0.0)
    assert (np.abs(y_gpu - y_ref) - bound).max() <= 0
    assert np.array_equal(y_gpu[~live], y_in[~live])      # no-LoRA rows untouched


def test_embedding_full_size(lib):
    inst = wl.make_instance("embed_lookup")
    assert inst.d_in == 128256 and inst.num_tokens == 256
    buf, y, status = _run(lib, inst, inst.token_ids)
    assert status == lib.LORA_OK
    ref = _host_buf(inst, inst.token_ids)
    assert np.array_equal(np.isnan(buf[0]), np.isnan(ref))
    assert np.array_equal(np.nan_to_num(buf[0], nan=0.0).view(np.uint32), np.nan_to_num(ref, nan=0.0).view(np.uint32))
    _check_y(inst, inst.token_ids, y, "bf16")


def test_embedding_ranks_scales_and_bad_ids(lib):
    """Heterogeneous ranks and scales; ids outside the vocabulary get a zero row and
    lora_query_status reports LORA_EBADTOKEN."""
    inst = wl.make_instance("embed_lookup", num_tokens=200, d_in=5000, out_sizes=[1032], num_slots=9, r_max=32)
    for k, (r, s) in zip(sorted(inst.adapters), [(32, 2.0), (3, 0.5), (17, 1.0), (1, 4.0), (8, 0.25),
                                                 (32, 1.5), (5, 3.0), (31, 0.75)]):
        ad = inst.adapters[k]
        inst.adapters[k] = wl.Adapter(r, s, [ad.A[0][:, :r].copy()], [ad.B[0][:r].copy()])
    ids = inst.token_ids.copy()
    live = np.where(inst.token_slot != 0)[0]
    ids[live[0]] = inst.d_in          # one past the vocabulary
    ids[live[1]] = -5
    buf, y, status = _run(lib, inst, ids, y_dtype="f32")
    assert status == lib.LORA_EBADTOKEN
    ref = _host_buf(inst, ids)
    assert np.array_equal(np.nan_to_num(buf[0], nan=-1.0).view(np.uint32), np.nan_to_num(ref, nan=-1.0).view(np.uint32))
    assert np.all(buf[0, live[:2]] == 0.0)
    _check_y(inst, ids, y, "f32")
