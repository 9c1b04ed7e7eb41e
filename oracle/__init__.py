"""CPU oracle for the batched multi-LoRA delta -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The
library (``rank_adapter_gb300``) never imports it and has no CPU fallback.

It is a plain, slow, obviously correct restatement of what the pages define,
in fp64 over the same stored (bf16 or fp32) values the GPU path reads. It
shares no code with the CUDA path. See ``lora_oracle`` for the functions and
the passages each follows.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(worked examples printed on the pages, closed forms, invariants, exact integer
brute force, and independent library routines).
"""
from .lora_oracle import (  # noqa: F401
    prepare_meta, shrink_requests, expand_requests, apply_requests, adapters_f64,
    requests_of_token_slots, embed_requests,
)
from .moe_oracle import moe_pair_slots, gathered_apply, moe_lora_w13, moe_lora_w2  # noqa: F401
