"""The bench's algorithmic byte model (the roofline's numerator) against direct
counts over a tiny batch: each active adapter's weights once, LoRA rows of x once,
LoRA rows of y read and written once; for the MoE layer, each active composite
slot's w13 and w2 weights once and each token's x row once however many of its
pairs are live."""
import numpy as np

import bench
import oracle
import workloads as wl


def test_dense_step_bytes_by_direct_count():
    inst = wl.make_instance("decode_qkv", num_tokens=37, d_in=256, out_sizes=[128, 64], num_slots=6)
    alg = bench.algorithmic(inst)
    ts = inst.token_slot
    want_w = 0
    for a in sorted(set(ts[ts > 0].tolist())):
        ad = inst.adapters[a]
        want_w += sum(A.size * 2 for A in ad.A) + sum(B.size * 2 for B in ad.B)
    n = int((ts > 0).sum())
    want = want_w + n * inst.d_in * 2 + 2 * n * inst.d_out_total * 2
    assert alg["step_bytes"] == want and alg["T_L"] == n


def test_moe_step_bytes_by_direct_count():
    m = wl.make_moe_instance(seed=5, num_tokens=30, hidden=64, inter=32, num_experts=8, local_experts=4, ep_rank=1,
                             topk=3, num_loras=2, r_max=8)
    pair = oracle.moe_pair_slots(m.token_slot, m.topk_ids, m.num_loras, m.num_experts, m.local_experts, m.expert_map)
    alg = bench.moe_algorithmic(m, pair)
    want, toks = 0, set()
    for s in sorted(set(pair[pair > 0].tolist())):
        for ad in (m.w13.adapters[s], m.w2.adapters[s]):
            want += sum(A.size * 2 for A in ad.A) + sum(B.size * 2 for B in ad.B)
    for p in np.nonzero(pair > 0)[0]:
        toks.add(int(p) // m.topk)
        want += 2 * m.inter + 2 * 2 * (2 * m.inter) + 2 * 2 * m.hidden   # h2 read; h1, h3 read + written
    want += len(toks) * m.hidden * 2 + 4 * m.num_tokens * (1 + 2 * m.topk)
    assert alg["step_bytes"] == want
    assert alg["pairs_live"] == int((pair > 0).sum()) and alg["T_L"] == int((m.token_slot > 0).sum())
