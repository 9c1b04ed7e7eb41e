"""The C-ABI library builds, loads without a GPU, exports every entry point
include/lora.h declares, and rejects bad arguments on the host before any
CUDA call (these calls launch nothing)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ra():
    import __graft_entry__
    __graft_entry__._load_build_lib().build()
    import rank_adapter_gb300
    return rank_adapter_gb300


def _declared():
    src = open(os.path.join(ROOT, "include", "lora.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(ra):
    names = _declared()
    assert set(names) >= {"lora_set_slot", "lora_reset_slot", "lora_prepare_meta", "lora_shrink",
                          "lora_expand", "lora_workspace_bytes", "lora_query_status", "lora_strerror"}
    lib = ctypes.CDLL(ra.lib_path())
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ra.exported_symbols())


def test_header_constants_match_binding(ra):
    src = open(os.path.join(ROOT, "include", "lora.h")).read()
    for name in ("LORA_MAX_SLICES", "LORA_MAX_NUM_SLOTS", "LORA_MAX_RANK", "LORA_SGMV_MIN_ROWS",
                 "LORA_SGMV_TILE_M", "LORA_AUTO_SGMV_MIN_TOKENS", "LORA_AUTO_SGMV_MIN_AVG",
                 "LORA_AUTO_LONG_ROWS"):
        m = re.search(rf"#define {name} (\d+)", src)
        assert m and int(m.group(1)) == getattr(ra, name), name
    for i, name in enumerate(["LORA_OK", "LORA_EINVAL", "LORA_ERANGE", "LORA_EALIGN", "LORA_EUNSUPPORTED",
                              "LORA_ECUDA", "LORA_EBADSLOT", "LORA_EDEVICE", "LORA_EBADTOKEN"]):
        assert re.search(rf"{name} = {i}\b", src) and getattr(ra, name) == i
    for i, name in enumerate(["LORA_AUTO", "LORA_BGMV", "LORA_SGMV", "LORA_MIXED"]):
        assert re.search(rf"{name} = {i}\b", src) and getattr(ra, name) == i


def test_strerror_and_sizes(ra):
    for s in range(9):
        assert ra.lora_strerror(s) and "unknown" not in ra.lora_strerror(s)
    assert "unknown" in ra.lora_strerror(99)
    assert ra.lora_meta_tiles_bytes(0) == 0
    assert ra.lora_meta_tiles_bytes(64) == (8 + 4 * 8 * 64 + 2 * 65 + 3 * 64) * 4
    assert ra.lora_last_cuda_error() == 0
    import torch
    if not torch.cuda.is_available():       # nothing can launch on a host-only run
        assert ra.lora_launch_count() == 0


def _desc(ra, **kw):
    d = ra.LayerDesc()
    d.dtype, d.d_in, d.n_slices = kw.get("dtype", ra.LORA_BF16), kw.get("d_in", 64), kw.get("n_slices", 2)
    d.num_slots, d.r_max = kw.get("num_slots", 4), kw.get("r_max", 16)
    for i in range(4):
        d.out_sizes[i] = kw.get("out", 32)
        d.A[i] = kw.get("ptr", 0x10000)
        d.B[i] = kw.get("ptr", 0x10000)
    d.slot_rank, d.slot_scale = 0x20000, 0x30000
    return d


@pytest.mark.parametrize("field,value,expect", [
    ("dtype", 7, "LORA_EINVAL"), ("n_slices", 0, "LORA_ERANGE"), ("n_slices", 5, "LORA_ERANGE"),
    ("d_in", 12, "LORA_EINVAL"), ("r_max", 12, "LORA_ERANGE"), ("r_max", 256, "LORA_ERANGE"),
    ("num_slots", 0, "LORA_ERANGE"), ("num_slots", 2000, "LORA_ERANGE"), ("out", 20, "LORA_EINVAL"),
    ("ptr", 0x10008, "LORA_EALIGN"),
])
def test_desc_validation(ra, field, value, expect):
    d = _desc(ra, **{field: value})
    assert ra.lora_reset_slot(d, 1, 0) == getattr(ra, expect)


def test_slot_range_and_sources(ra):
    d = _desc(ra)
    assert ra.lora_reset_slot(d, 0, 0) == ra.LORA_ERANGE        # slot 0 is reserved
    assert ra.lora_reset_slot(d, 4, 0) == ra.LORA_ERANGE
    assert ra.lora_set_slot(d, 1, 0, 1.0, [None] * 4, [None] * 4, 0) == ra.LORA_ERANGE
    assert ra.lora_set_slot(d, 1, 17, 1.0, [None] * 4, [None] * 4, 0) == ra.LORA_ERANGE
    assert ra.lora_set_slot(d, 1, 8, 1.0, [0x40000, None], [None, None], 0) == ra.LORA_EINVAL
    assert ra.lora_set_slot(d, 1, 8, 1.0, [0x40000, None], [0x40008, None], 0) == ra.LORA_EALIGN


def _meta(ra, T=8, S=4):
    m = ra.Meta()
    m.token_slot, m.num_tokens, m.num_slots = 0x1000, T, S
    m.sorted_rows = m.seg_slot = m.seg_count = m.seg_start = 0x2000
    m.num_segs, m.no_lora, m.status = 0x3000, 0x3004, 0x3008
    m.tiles, m.tiles_bytes = 0x4000, ra.lora_meta_tiles_bytes(S)
    return m


def test_meta_validation(ra):
    m = _meta(ra, S=0)
    assert ra.lora_prepare_meta(m, 0) == ra.LORA_ERANGE
    m = _meta(ra, T=-1)
    assert ra.lora_prepare_meta(m, 0) == ra.LORA_ERANGE
    m = _meta(ra)
    m.tiles_bytes -= 4
    assert ra.lora_prepare_meta(m, 0) == ra.LORA_EINVAL
    m = _meta(ra)
    m.token_slot = None
    assert ra.lora_prepare_meta(m, 0) == ra.LORA_EINVAL
    m = _meta(ra)
    m.tiles = 0x4002
    assert ra.lora_prepare_meta(m, 0) == ra.LORA_EALIGN


def test_embed_shrink_validation(ra):
    one = _desc(ra, n_slices=1)
    m = _meta(ra)
    assert ra.lora_embed_shrink(_desc(ra), m, 0x9000, 0x6000, 0) == ra.LORA_EINVAL   # an embedding has one slice
    assert ra.lora_embed_shrink(one, m, 0, 0x6000, 0) == ra.LORA_EINVAL              # no token ids
    assert ra.lora_embed_shrink(one, m, 0x9000, 0, 0) == ra.LORA_EINVAL              # no buf
    assert ra.lora_embed_shrink(one, m, 0x9000, 0x6008, 0) == ra.LORA_EALIGN         # buf not 16-byte aligned
    assert ra.lora_embed_shrink(one, m, 0x9002, 0x6000, 0) == ra.LORA_EALIGN         # ids not int-aligned
    assert ra.lora_embed_shrink(one, _meta(ra, S=5), 0x9000, 0x6000, 0) == ra.LORA_EINVAL  # slot count mismatch
    assert ra.lora_embed_shrink(one, _meta(ra, T=0), 0, 0, 0) == ra.LORA_OK          # T = 0: no-op


def test_moe_pair_slots_validation(ra):
    f = lambda *a: ra.lora_moe_pair_slots(*a, 0)   # noqa: E731
    P = 0x1000
    assert f(0, 0, 0, 2, 1, 4, 4, 0, 0) == ra.LORA_OK                  # no tokens: no-op
    assert f(P, P, 5, 0, 1, 4, 4, 0, P) == ra.LORA_ERANGE              # topk < 1
    assert f(P, P, 5, 65, 1, 4, 4, 0, P) == ra.LORA_ERANGE             # topk > 64
    assert f(P, P, 5, 2, 1, 4, 5, 0, P) == ra.LORA_ERANGE              # more local experts than experts
    assert f(P, P, 5, 2, 2000, 4, 4, 0, P) == ra.LORA_ERANGE           # composite table too large
    assert f(P, P, 5, 2, -1, 4, 4, 0, P) == ra.LORA_ERANGE
    assert f(0, P, 5, 2, 1, 4, 4, 0, P) == ra.LORA_EINVAL              # no token slots
    assert f(P, P, 5, 2, 1, 4, 4, 0, 0) == ra.LORA_EINVAL              # no output
    assert f(P + 2, P, 5, 2, 1, 4, 4, 0, P) == ra.LORA_EALIGN
    assert f(P, P, 5, 2, 1, 4, 4, P + 1, P) == ra.LORA_EALIGN          # expert map misaligned
    d = _desc(ra)
    d.x_row_div = -1
    assert ra.lora_reset_slot(d, 1, 0) == ra.LORA_EINVAL


def test_shrink_expand_validation(ra):
    d, m = _desc(ra), _meta(ra)
    assert ra.lora_shrink(d, m, 0x5000, 64, 0x6000, 9, 0, 0, 0) == ra.LORA_EINVAL       # kind
    assert ra.lora_shrink(d, m, 0x5000, 60, 0x6000, 1, 0, 0, 0) == ra.LORA_EINVAL       # ldx < d_in
    assert ra.lora_shrink(d, m, 0x5008, 64, 0x6000, 1, 0, 0, 0) == ra.LORA_EALIGN
    assert ra.lora_shrink(d, m, 0x5000, 68, 0x6000, 1, 0, 0, 0) == ra.LORA_EALIGN       # ldx*2 % 16
    assert ra.lora_shrink(d, m, 0x5000, 64, 0x6000, 1, 0, 0, 0) == ra.LORA_EINVAL       # no scratch
    m2 = _meta(ra, S=5)
    assert ra.lora_shrink(d, m2, 0x5000, 64, 0x6000, 1, 0, 0, 0) == ra.LORA_EINVAL      # slot count mismatch
    f = _desc(ra, dtype=ra.LORA_F32)
    assert ra.lora_shrink(f, m, 0x5000, 64, 0x6000, ra.LORA_SGMV, 0, 0, 0) == ra.LORA_EUNSUPPORTED
    assert ra.lora_expand(f, m, 0x6000, 0x7000, 64, ra.LORA_BF16, 1, 0) == ra.LORA_EUNSUPPORTED
    r8 = _desc(ra, r_max=8)   # the tensor-core family needs r_max >= 16
    assert ra.lora_shrink(r8, m, 0x5000, 64, 0x6000, ra.LORA_SGMV, 0, 0, 0) == ra.LORA_EUNSUPPORTED
    assert ra.lora_expand(r8, m, 0x6000, 0x7000, 64, ra.LORA_BF16, ra.LORA_SGMV, 0) == ra.LORA_EUNSUPPORTED
    assert ra.lora_apply(r8, m, 0x5000, 64, 0, 0x7000, 64, ra.LORA_BF16, ra.LORA_SGMV, 0, 0, 0) == \
        ra.LORA_EUNSUPPORTED
    assert ra.lora_workspace_bytes(r8, 256, ra.LORA_SGMV) == 0
    assert ra.lora_expand(d, m, 0x6000, 0x7000, 60, ra.LORA_BF16, 1, 0) == ra.LORA_EINVAL  # ldy < sum(out)
    assert ra.lora_expand(d, m, 0x6000, 0x7000, 64, 5, 1, 0) == ra.LORA_EINVAL
    m0 = _meta(ra, T=0)
    assert ra.lora_shrink(d, m0, 0, 64, 0, 1, 0, 0, 0) == ra.LORA_OK                   # T = 0: no-op
    assert ra.lora_expand(d, m0, 0, 0, 64, ra.LORA_BF16, 1, 0) == ra.LORA_OK
    assert ra.lora_workspace_bytes(d, 1024, ra.LORA_BGMV) == 2 * 1024 * 1 * 16 * 4   # d_in = 64: one chunk
    assert ra.lora_workspace_bytes(d, 1000, ra.LORA_AUTO) == 2 * 1000 * 1 * 16 * 4   # < 1024 tokens: BGMV only
    assert ra.lora_workspace_bytes(d, 0, 0) == 0
    assert ra.lora_workspace_bytes(d, 16, 7) == 0                                      # bad kind
    # MIXED is a valid kind; where SGMV does not apply (r_max < 16) it plans BGMV alone
    assert ra.lora_workspace_bytes(r8, 1000, ra.LORA_MIXED) == ra.lora_workspace_bytes(r8, 1000, ra.LORA_BGMV) > 0
    assert ra.lora_workspace_bytes(d, 1000, ra.LORA_MIXED) >= ra.lora_workspace_bytes(d, 1000, ra.LORA_BGMV)
    big = _desc(ra, d_in=4096, n_slices=3)
    nb = ra.lora_workspace_bytes(big, 256, 0)
    assert nb > 0 and nb % 16 == 0
    assert ra.lora_workspace_bytes(_desc(ra, r_max=12), 256, 0) == 0  # invalid desc
    mb = _meta(ra, T=256, S=4)
    assert ra.lora_shrink(big, mb, 0x5000, 4096, 0x6000, 1, 0, 0, 0) == ra.LORA_EINVAL        # no scratch
    assert ra.lora_shrink(big, mb, 0x5000, 4096, 0x6000, 1, 0x7000, nb - 16, 0) == ra.LORA_EINVAL
    assert ra.lora_shrink(big, mb, 0x5000, 4096, 0x6000, 1, 0x7008, nb, 0) == ra.LORA_EALIGN
    assert ra.lora_apply(big, mb, 0x5000, 4096, 0, 0x8000, 16 * 4 * 3, ra.LORA_BF16, 1, 0, 0, 0) == ra.LORA_EINVAL


def test_product_path_has_no_oracle_import():
    """The library package never imports the oracle (no CPU fallback)."""
    pkg = os.path.join(ROOT, "rank_adapter_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", txt, re.M), f
                assert "lora_oracle" not in txt, f
