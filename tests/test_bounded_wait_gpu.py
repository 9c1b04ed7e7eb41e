"""The device-side failure path of the pipeline waits, made to happen without a fault.

The tensor-core kernels wait on their own pipeline barriers with a time limit;
a wait that runs out records a bit in the metadata's device error word, the
kernel winds down, and lora_query_status reports LORA_EDEVICE. Here the same
bounded wait runs (lora_probe_bounded_wait) on a barrier nothing arms, with a
limit of a few milliseconds: the status must come back as LORA_EDEVICE after
about that long, and the context must stay usable -- the next metadata pass
clears the word and a full step still matches the oracle."""
import time

import pytest
import torch

import workloads as wl
from gpu_harness import parity

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_edevice(lib):
    ts = torch.tensor([1, 0, 2, 1, 3, 0, 0, 1], dtype=torch.int32, device="cuda")
    meta = lib.TokenMeta(8, 4)
    meta.prepare(ts)
    assert lib.lora_query_status(meta.c) == (lib.LORA_OK, 0)
    t0 = time.perf_counter()
    assert lib.lora_probe_bounded_wait(meta.c, 3000) == lib.LORA_OK
    st, _ = lib.lora_query_status(meta.c)  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert st == lib.LORA_EDEVICE, lib.lora_strerror(st)
    assert 0.003 <= elapsed < 5.0
    # The context is usable: a new metadata pass clears the error word, and a step is right.
    meta.prepare(ts)
    assert lib.lora_query_status(meta.c) == (lib.LORA_OK, 0)
    inst = wl.make_instance("decode_qkv", num_tokens=40, d_in=512, out_sizes=[256, 128], num_slots=9)
    parity(inst, kind=lib.LORA_AUTO)


def test_probe_limits_are_checked_before_launch(lib):
    meta = lib.TokenMeta(4, 3)
    meta.prepare(torch.zeros(4, dtype=torch.int32, device="cuda"))
    n0 = lib.lora_launch_count()
    assert lib.lora_probe_bounded_wait(meta.c, 0) == lib.LORA_ERANGE
    assert lib.lora_probe_bounded_wait(meta.c, 1_000_001) == lib.LORA_ERANGE
    assert lib.lora_launch_count() == n0
    torch.cuda.synchronize()
    assert lib.lora_query_status(meta.c) == (lib.LORA_OK, 0)
