"""The lm_head LoRA on the rows sampled this step (page "vLLM 源码完全拆解(十八):
多 LoRA 服务", section "lm_head / logits"): one shrink and one expand over the
sampled rows only, each with its request's slot, and d_out = the vocabulary.
Through the C ABI against the fp64 oracle, at the full size (hidden 4096 ->
vocab 128256, r = 16, 64 slots, 256 sampled rows) and on a ragged vocabulary,
plus the property that makes the sampled-row mapping exact: a row's delta
depends only on its own hidden state and slot, so running on the sampled rows
gives bitwise the values the whole batch gives at those rows."""
import numpy as np
import pytest

import workloads as wl
from gpu_harness import load_table, parity, run_gpu

pytestmark = pytest.mark.gpu


def test_logits_full_size(lib):
    inst = wl.make_instance("logits_lm_head")
    assert inst.d_out_total == 128256 and inst.num_tokens == 256
    parity(inst, kind=lib.LORA_BGMV, y_dtype="bf16", path="apply")


@pytest.mark.parametrize("path", ["split", "apply"])
def test_logits_ragged_vocab(lib, path):
    """A vocabulary that is no multiple of the expand's column chunk, fp32 logits."""
    inst = wl.make_instance("logits_lm_head", num_tokens=48, out_sizes=[10248], num_slots=9)
    parity(inst, kind=lib.LORA_AUTO, y_dtype="f32", path=path)


def test_sampled_rows_equal_full_batch_rows(lib):
    """Prefill and decode requests in one batch: the lm_head LoRA on the last token
    of every request equals, bitwise, the delta the whole batch gets at those rows."""
    lengths = [37, 1, 1, 120, 5, 1, 64, 1, 9, 1, 1, 200]
    full = wl.make_instance("logits_lm_head", req_lengths=lengths, out_sizes=[4096], num_slots=7)
    t = load_table(full)
    _, y_all, _ = run_gpu(full, table=t, kind=lib.LORA_BGMV, y_dtype="f32", path="apply")
    rows = wl.sampled_rows(full.req_lengths)
    samp = wl.make_instance("logits_lm_head", req_lengths=[1] * len(rows), out_sizes=[4096], num_slots=7)
    samp.adapters = full.adapters
    samp.req_slots = full.req_slots.copy()
    samp.x = full.x[rows].copy()
    samp.y_in = full.y_in[rows].copy()
    _, y_s, _ = run_gpu(samp, table=t, kind=lib.LORA_BGMV, y_dtype="f32", path="apply")
    assert np.array_equal(y_s.view(np.uint32), y_all[rows].view(np.uint32))
