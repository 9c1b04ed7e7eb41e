"""The MoE workload's table shapes against the memory example the page prints
(tests/golden/moe_memory.json): per (adapter, expert) pair the w13 and w2 A/B
hold 64 x 27648 elements, 454 MB for 4 adapters x 32 local experts in bf16,
3.6 GB without expert parallelism, and sharing w13's A and w2's B across the
experts keeps about a quarter of it."""
import json
import os

import workloads as wl

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "moe_memory.json")))["page"]


def _elements(hidden, inter, r):
    a13, b13 = 2 * hidden * r, 2 * r * inter       # gate and up slices
    a2, b2 = inter * r, r * hidden
    return a13 + b13 + a2 + b2


def _close(a, b, rel=0.006):
    return abs(a - b) <= rel * abs(b)


def test_workload_shapes_match_the_printed_example():
    H, I, E, L, NL, R = 7168, 2048, 256, 32, 4, 64      # the workload's defaults (checked below)
    per = _elements(H, I, R)
    assert per == 64 * 27648
    assert _close(per, GOLD["elements_per_expert_per_slot"])
    total = per * L * NL
    assert _close(total, GOLD["elements_total_ep8"])
    assert _close(total * 2 / 1e6, GOLD["bytes_total_ep8_mb"])
    assert _close(per * E * NL * 2 / 1e9, GOLD["bytes_total_no_ep_gb"], rel=0.02)
    # shared w13 A and w2 B: one copy per slot instead of one per expert
    shared = L * (2 * R * I + I * R) + (2 * H * R + R * H)
    assert _close(shared / (per * L), GOLD["shared_ab_fraction"], rel=0.02)


def test_generator_defaults_are_the_example():
    import inspect
    src = inspect.getsource(wl.make_moe_instance)
    for frag in ("hidden or 7168", "inter or 2048", "num_experts or 256", "local_experts or 32", "topk or 8",
                 "num_loras or 4", "r_max or 64"):
        assert frag in src, frag
