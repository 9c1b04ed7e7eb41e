#!/usr/bin/env python
"""Benchmark of the multi-LoRA hot path on one GB300 per rank.

One step = one pass of the whole per-step path over one batch:
lora_prepare_meta (token metadata) + lora_shrink + lora_expand, through the
library's C ABI. The default workload is the decode batch the headline metric
is quoted on: qkv_proj d_in=4096, packed slices [4096,1024,1024], r=16,
64 slots, 256 one-token requests (10% slot 0), bf16.

Timing: the step's inputs (slot table, x, y, token slots, metadata) are
replicated on the device R times so that the rotation touches more than
3x the 129 MB L2 between visits to a replica ("inputs larger than L2").
Warm-up steps run eagerly; a timed region is exactly K steps as CUDA-graph
replays bracketed by CUDA events on the launching stream. Regions repeat
back to back until at least --min-seconds of device time has been timed
(so the clock sampler sees the load), with a barrier and
torch.cuda.synchronize() on both sides of the whole set; the value is the
median region (min and max reported beside it), max over ranks.
Per-call durations come from graphs of G launches of one call alone (on
inputs the steps prepared), timed around their replays. The end-to-end figure repeats the step through
the same ABI with pinned host buffers: the copies in and out are inside its
timed region.

The default run (decode batch, one GPU) also measures the other workloads of
the same family -- the toy fp32 batch, the prefill batch, the mixed batch and
the 32-layer decode step -- and reports them under "configs" with their own
roofline fractions and oracle baselines.

Multi-GPU (torchrun): data parallel over independent batches, one replica of
the slot table per rank, no collective on the data path ("scaling": "weak").

``--impl reference`` times the fp64 CPU oracle on the same workload (the
only other place besides the cpu_baseline leg that runs ``oracle/``).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-delta tokens/s and achieved HBM GB/s (decode) / TC TFLOP/s (prefill) vs peak"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

WORKLOADS = {
    "decode_qkv": "decode BGMV: qkv_proj 4096->[4096,1024,1024], r=16, 64 slots, 256 tokens (10% slot 0)",
    "prefill_gate_up": "prefill SGMV: gate_up_proj 4096->[14336,14336], r=64, 32 slots, 16 requests U[128,2048]",
    "mixed_o_proj": "mixed: o_proj 4096->4096, 128 slots, ranks {8..64} pad 64, 1024 decode + 4x512 prefill",
    "toy_fp32": "toy fp32: d=256, r=16, 8 slots, 6 requests (53 tokens)",
    "full_decode": "full-model decode step: 32 layers x {qkv, o, gate_up, down}, r=16, 100 resident adapters "
                   "(~84 MB each), 512 tokens uniform over them; one metadata pass, 128 lora_apply calls",
    "logits_lm_head": "lm_head LoRA on sampled rows: hidden 4096 -> vocab 128256, r=16, 64 slots, "
                      "256 sampled rows (one per request, 10% slot 0)",
    "embed_lookup": "embedding LoRA: vocab 128256 -> hidden 4096, r=16, 64 slots, 256 decode tokens "
                    "(ids uniform over the vocabulary, 10% slot 0); lookup + expand",
    "moe_decode": "MoE layer LoRA: hidden 7168, expert inter 2048, 256 experts / EP8 (32 local), top-8, r=64, "
                  "4 adapters (128 composite slots, ~457 MB), 256 decode tokens (10% slot 0); pair slots + metadata "
                  "over the 2048 pairs + w13 (gate, up; x rows shared by a token's pairs) + w2",
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="decode_qkv")
    p.add_argument("--kind", choices=["auto", "bgmv", "sgmv", "mixed"], default="auto")
    p.add_argument("--path", choices=["fused", "split"], default="fused",
                   help="fused: prepare_meta + lora_apply; split: prepare_meta + lora_shrink + lora_expand")
    p.add_argument("--replicas", type=int, default=0, help="device replicas (0: enough for 3x L2)")
    p.add_argument("--graph-steps", type=int, default=0, help="steps per captured graph (0: auto)")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--min-seconds", type=float, default=0.5,
                   help="device time to accumulate over repeated K-step regions")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads' sub-records of the default run")
    p.add_argument("--sub-cpu-seconds", type=float, default=4.0,
                   help="oracle time per sub-record's cpu_baseline")
    p.add_argument("--cpu-threads", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--cpu-child", action="store_true", help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ----------------------------------------------------------------------------- algorithmic model

def algorithmic(inst, y_bytes_per_elem=2):
    """Bytes and flops the method must move / do for one step on this batch.

    Weights of every active adapter are read once (rank-aware), x rows of LoRA
    tokens are read once, y rows of LoRA tokens are read and written once.
    The fp32 shrink buffer is counted per kernel (it is the shrink's output and
    the expand's input) but not in the step total.
    """
    import numpy as np
    es = 2 if inst.dtype == "bf16" else 4
    ts = inst.token_slot.astype(np.int64)
    live = (ts > 0) & (ts < inst.num_slots)
    T_L = int(live.sum())
    ranks = np.zeros(inst.num_slots, np.int64)
    for k, ad in inst.adapters.items():
        ranks[k] = ad.rank
    active = np.unique(ts[live])
    n_s, d_in, d_out = inst.n_slices, inst.d_in, inst.d_out_total
    w_a = int(sum(es * ranks[a] * n_s * d_in for a in active))
    w_b = int(sum(es * ranks[a] * d_out for a in active))
    x_b = es * T_L * d_in
    if inst.token_ids is not None:
        # embedding: the lookup reads one r-vector per distinct (slot, token id) and the ids
        pairs = {(int(a), int(v)) for a, v in zip(ts[live], inst.token_ids[live])}
        w_a = int(sum(es * ranks[a] for a, _ in pairs))
        x_b = 4 * len(ts)
    y_b = 2 * y_bytes_per_elem * T_L * d_out
    buf_b = 4 * n_s * T_L * inst.r_max
    shrink_d = 0 if inst.token_ids is not None else n_s * d_in   # a lookup does no products
    flops = int(sum(2 * ranks[a] * (shrink_d + d_out) * int((ts == a).sum()) for a in active))
    return dict(T=int(len(ts)), T_L=T_L, active=int(len(active)), shrink_bytes=w_a + x_b + buf_b,
                expand_bytes=w_b + buf_b + y_b, step_bytes=w_a + w_b + x_b + y_b, flops=flops,
                shrink_flops=int(sum(2 * ranks[a] * shrink_d * int((ts == a).sum()) for a in active)),
                expand_flops=int(sum(2 * ranks[a] * d_out * int((ts == a).sum()) for a in active)))


def make_workload(name, seed_offset=0):
    import workloads as wl
    base = {"toy_fp32": 0, "decode_qkv": 2, "prefill_gate_up": 3, "mixed_o_proj": 4, "logits_lm_head": 6,
            "embed_lookup": 7}[name]
    return wl.make_instance(name, seed=base + 1000 * seed_offset if seed_offset else None)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rank_adapter_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload, {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU legs (oracle)

def cpu_child(args):
    """Time the oracle as it stands on this host's cores; prints one JSON line."""
    import numpy as np
    import oracle
    if args.cpu_threads == 1:   # the single-thread figure: one core
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    inst = make_workload(args.workload)
    alg = algorithmic(inst)
    ads = oracle.adapters_f64(inst)
    x = inst.to_f32(inst.x).astype(np.float64)
    y = inst.to_f32(inst.y_in).astype(np.float64)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.prepare_meta(inst.token_slot, inst.num_slots)
        if inst.token_ids is not None:   # embedding: lookup, then expand
            buf, _ = oracle.embed_requests(inst.token_ids, ads, inst.r_max, inst.req_lengths, inst.req_slots,
                                           inst.num_slots)
            oracle.expand_requests(buf, y, ads, inst.out_sizes, inst.req_lengths, inst.req_slots, inst.num_slots)
        else:
            oracle.apply_requests(x, y, ads, inst.out_sizes, inst.r_max, inst.req_lengths, inst.req_slots,
                                  inst.num_slots)
        reps += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds:
            break
    print(json.dumps({"value": reps * alg["T_L"] / el, "seconds": el, "reps": reps,
                      "sec_per_step": el / reps, "T_L": alg["T_L"], "active": alg["active"],
                      "T": alg["T"]}))


def run_cpu_baseline(workload, seconds, threads=None):
    """The oracle on this host's cores (all of them, or one) in a child process; a cpu_baseline record."""
    cores = len(os.sched_getaffinity(0)) if threads is None else threads
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-child", "--workload", workload,
           "--cpu-seconds", str(seconds), "--cpu-threads", str(threads or 0)]
    p = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT)
    if p.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "error": p.stderr.strip().splitlines()[-1:] }
    r = json.loads(p.stdout.strip().splitlines()[-1])
    what = {"full_decode": f"{r['reps']} x one layer (4 groups) of the full-model step, scaled x32 ",
            "moe_decode": f"{r['reps']} full MoE-layer steps (pair slots, metadata, w13, w2) "}.get(
        workload, f"{r['reps']} full steps of the {workload} batch ")
    rec = {"value": r["value"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": what + f"(fp64 per-request loop, numpy BLAS with {cores} thread{'s' if cores > 1 else ''}), "
                            f"{r['seconds']:.1f} s",
           "sec_per_step": r["sec_per_step"]}
    for k in ("T_L", "active", "T", "pairs", "live_pairs", "active_composite_slots"):
        if k in r:
            rec[k] = r[k]
    return rec


def workload_config(name, kind, path, world, T, T_L, active=None, extra=None):
    """The config dict both arms print for a workload (the same keys and values on both)."""
    cfg = {"workload": name, "desc": WORKLOADS[name], "kind": kind, "path": path, "global_batch": T * world,
           "lora_tokens_per_gpu": T_L, "parallelism": f"dp{world}"}
    if active is not None:
        cfg["active_adapters"] = active
    cfg["l2"] = L2_NOTES.get(name, "inputs larger than L2: device replicas of the step's inputs, "
                                   "rotated so that > 3x the 129 MiB L2 lies between visits to one")
    if extra:
        cfg.update(extra)
    return cfg


L2_NOTES = {
    "full_decode": "inputs larger than L2: ~12 GB of distinct weights and activations touched per step",
    "moe_decode": "inputs larger than L2: ~377 MB touched per step, tables of 457 MB",
}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cpu = run_cpu_baseline(args.workload, max(1.0, args.cpu_seconds))
    v = cpu.get("value")
    T = cpu.get("T") or {"full_decode": 512, "moe_decode": 256}.get(args.workload, 0)
    path = "fused" if args.workload in ("full_decode", "moe_decode") else args.path
    if args.workload == "moe_decode":
        cfg = workload_config(args.workload, args.kind, path, args.gpus, T, cpu.get("T_L"), None,
                              {k: cpu.get(k) for k in ("pairs", "live_pairs", "active_composite_slots")})
    else:
        cfg = workload_config(args.workload, args.kind, path, args.gpus, T, cpu.get("T_L"), cpu.get("active"))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "ms_per_step": (cpu["sec_per_step"] * 1e3) if v else None,
            "cpu_baseline": cpu, "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                         "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- GPU leg

class Replica:
    """One device copy of every input of a step, plus its metadata buffers and ctypes arguments."""

    def __init__(self, ra, torch, inst, table_src, x_src, y_src, ts_src, kind):
        self.table = ra.SlotTable(inst.d_in, inst.out_sizes, inst.num_slots, inst.r_max,
                                  ra.LORA_BF16 if inst.dtype == "bf16" else ra.LORA_F32)
        for dst, src in zip(self.table.A + self.table.B, table_src.A + table_src.B):
            dst.copy_(src)
        self.table.slot_rank.copy_(table_src.slot_rank)
        self.table.slot_scale.copy_(table_src.slot_scale)
        self.x = x_src.clone()
        self.y = y_src.clone()
        T = inst.num_tokens
        self.meta = ra.TokenMeta(T, inst.num_slots)
        self.meta.token_slot[:T].copy_(ts_src)
        self.meta.set_num_tokens(T)
        self.buf = torch.zeros(inst.n_slices, T, inst.r_max, dtype=torch.float32, device="cuda")
        self.ws = ra.workspace(self.table, T, kind)
        self.ws_ptr = self.ws.data_ptr() if self.ws is not None else 0
        self.ws_bytes = self.ws.numel() * 4 if self.ws is not None else 0
        self.kind = kind
        self.ydt = ra.LORA_BF16 if self.y.dtype == torch.bfloat16 else ra.LORA_F32
        self.embed = inst.token_ids is not None   # x holds token ids: the shrink is the embedding lookup

    def bytes(self):
        return self.table.nbytes() + self.x.numel() * self.x.element_size() + \
            self.y.numel() * self.y.element_size()

    def launch(self, ra, i, ev=None, path="fused", only=None, unshared=False):
        """Enqueue one step on the current stream: prepare_meta then lora_apply (path "fused")
        or lora_shrink + lora_expand (path "split"). ev: optional events around each call.
        only: enqueue just that call ("meta", "apply", "shrink" or "expand"; the metadata and
        buffers it reads were prepared by earlier steps). unshared: the previous step on the
        stream used another replica's metadata, so lora_prepare_meta_unshared may write this
        step's metadata without waiting for that step's kernels."""
        st = None
        if only is not None:
            if only == "meta":
                ra.check(ra.lora_prepare_meta(self.meta.c, st), "prepare_meta")
            elif only == "apply" and self.embed:
                self._embed_step(ra, st)
            elif only == "apply":
                ra.check(ra.lora_apply(self.table.desc, self.meta.c, self.x.data_ptr(), self.x.stride(0), 0,
                                       self.y.data_ptr(), self.y.stride(0), self.ydt, self.kind, self.ws_ptr,
                                       self.ws_bytes, st), "apply")
            elif only == "shrink" and self.embed:
                ra.check(ra.lora_embed_shrink(self.table.desc, self.meta.c, self.x.data_ptr(), self.buf.data_ptr(),
                                              st), "embed_shrink")
            elif only == "shrink":
                ra.check(ra.lora_shrink(self.table.desc, self.meta.c, self.x.data_ptr(), self.x.stride(0),
                                        self.buf.data_ptr(), self.kind, self.ws_ptr, self.ws_bytes, st), "shrink")
            else:
                ra.check(ra.lora_expand(self.table.desc, self.meta.c, self.buf.data_ptr(), self.y.data_ptr(),
                                        self.y.stride(0), self.ydt, self.kind, st), "expand")
            return
        if ev is not None:
            ev[0].record()
        if unshared:
            ra.check(ra.lora_prepare_meta_unshared(self.meta.c, st), "prepare_meta_unshared")
        else:
            ra.check(ra.lora_prepare_meta(self.meta.c, st), "prepare_meta")
        if ev is not None:
            ev[1].record()
        if self.embed:  # both paths: the lookup, then the expand
            ra.check(ra.lora_embed_shrink(self.table.desc, self.meta.c, self.x.data_ptr(), self.buf.data_ptr(),
                                          st), "embed_shrink")
            if ev is not None:
                ev[2].record()
            ra.check(ra.lora_expand(self.table.desc, self.meta.c, self.buf.data_ptr(), self.y.data_ptr(),
                                    self.y.stride(0), self.ydt, self.kind, st), "expand")
            if ev is not None:
                ev[len(ev) - 1].record()
            return
        if path == "fused":
            # The fused step keeps the rank-r intermediate in the workspace; no buf output is asked for.
            ra.check(ra.lora_apply(self.table.desc, self.meta.c, self.x.data_ptr(), self.x.stride(0), 0,
                                   self.y.data_ptr(), self.y.stride(0), self.ydt, self.kind, self.ws_ptr,
                                   self.ws_bytes, st), "apply")
            if ev is not None:
                ev[2].record()
            return
        ra.check(ra.lora_shrink(self.table.desc, self.meta.c, self.x.data_ptr(), self.x.stride(0),
                                self.buf.data_ptr(), self.kind, self.ws_ptr, self.ws_bytes, st), "shrink")
        if ev is not None:
            ev[2].record()
        ra.check(ra.lora_expand(self.table.desc, self.meta.c, self.buf.data_ptr(), self.y.data_ptr(),
                                self.y.stride(0), self.ydt, self.kind, st), "expand")
        if ev is not None:
            ev[3].record()


    def _embed_step(self, ra, st):
        ra.check(ra.lora_embed_shrink(self.table.desc, self.meta.c, self.x.data_ptr(), self.buf.data_ptr(), st),
                 "embed_shrink")
        ra.check(ra.lora_expand(self.table.desc, self.meta.c, self.buf.data_ptr(), self.y.data_ptr(),
                                self.y.stride(0), self.ydt, self.kind, st), "expand")


KERNELS = {"fused": ("meta", "apply"), "split": ("meta", "shrink", "expand")}


def time_regions(torch, stream, run_region, min_seconds, min_regions=3):
    """Device time of repeated regions, each one call of run_region() (which enqueues exactly K
    steps) between its own CUDA events on `stream`; regions run back to back until at least
    min_seconds of device time is covered. Returns the regions' durations in ms."""
    def batch(n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                e0.record()
                run_region()
                e1.record()
        stream.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in evs]
    first = batch(1)
    n = int(math.ceil(min_seconds * 1e3 / max(first[0], 1e-3)))
    n = min(max(n, min_regions) - 1, 200000)
    return first + batch(n) if n > 0 else first


def region_stats(ms):
    return {"median_ms": statistics.median(ms), "min_ms": min(ms), "max_ms": max(ms), "regions": len(ms),
            "timed_s": sum(ms) * 1e-3}


def time_path(torch, ra, reps, stream, path, steps, G, min_seconds, clocks=None, dist=None):
    """Time regions of exactly `steps` steps of one path as replays of CUDA graphs of G steps (rotating
    replicas), repeated until min_seconds of device time; see time_regions.

    The timed graphs hold only the library's launches. Per-call durations come
    afterwards from graphs of G launches of one call alone. Returns (region durations in ms, per-call
    mean ms, how, kernels launched per step).
    """
    R = len(reps)
    names = KERNELS[path]

    def capture(n):
        # Consecutive steps use different replicas (R >= 2), so every step but a graph's first
        # prepares its metadata with lora_prepare_meta_unshared: the previous step's kernels read
        # the other replica's metadata (a serving loop alternating two metadata buffers).
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(n):
                reps[i % R].launch(ra, i, path=path, unshared=i > 0 and R > 1)
        return gr

    n0 = ra.lora_launch_count()
    graph = capture(G)
    per_step = (ra.lora_launch_count() - n0) / G  # kernels the library launches per step
    tail = steps % G
    graph_tail = capture(tail) if tail else None
    with torch.cuda.stream(stream):
        for _ in range(2):
            graph.replay()
    stream.synchronize()

    def region():
        for _ in range(steps // G):
            graph.replay()
        if graph_tail is not None:
            graph_tail.replay()

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    ms = time_regions(torch, stream, region, min_seconds)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.stop()

    # Per call: a graph of G launches of that call alone (on metadata and
    # buffers the steps above prepared), timed around its replays. No event
    # sits between the kernels, so these are the calls' own durations.
    durs = {}
    for name in names:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(G):
                reps[i % R].launch(ra, i, path=path, only=name)
        with torch.cuda.stream(stream):
            gr.replay()
        stream.synchronize()
        reps_n = max(3, int(math.ceil(0.05e3 / max(1e-3, statistics.median(ms) * G / steps))))
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            c0.record()
            for _ in range(reps_n):
                gr.replay()
            c1.record()
        stream.synchronize()
        durs[name] = c0.elapsed_time(c1) / (reps_n * G)
    how = (f"each call alone: CUDA-graph replays of {G} launches of that call on prepared inputs, "
           f"CUDA events around the replays")
    return ms, durs, how, per_step


def reduce_over_ranks(torch, dist, elapsed_ms, e2e_ms, lora_tokens, device):
    """Whole-job numbers of a data-parallel run: the slowest rank's timings (max)
    and the LoRA tokens of all ranks (sum). dist is None for a single process."""
    if dist is None:
        return float(elapsed_ms), float(e2e_ms), float(lora_tokens)
    vals = torch.tensor([elapsed_ms, e2e_ms, float(lora_tokens)], dtype=torch.float64, device=device)
    mx = vals.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    tl = vals.clone()
    dist.all_reduce(tl, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(mx[1]), float(tl[2])


def init_dist():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    return world, rank, local, dist


def clock_sampler(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    return ClockSampler(vis.split(",")[local].strip() if vis else str(local))


def replica_bytes(inst):
    """Device bytes of one replica of a step's inputs (slot table, x, y)."""
    es = 2 if inst.dtype == "bf16" else 4
    table = es * inst.num_slots * inst.r_max * (inst.n_slices * inst.d_in + inst.d_out_total)
    x = 4 * inst.num_tokens if inst.token_ids is not None else es * inst.num_tokens * inst.d_in
    return table + x + es * inst.num_tokens * inst.d_out_total


def measure_dense(name, args, world=1, rank=0, local=0, dist=None, with_e2e=True, min_seconds=None,
                  with_other_path=True):
    """Everything the bench reports for one single-projection workload (decode, prefill, mixed, toy,
    lm_head, embedding): the timed step, per-call durations, roofline, e2e. Returns a dict of line
    fields on every rank (rank 0 prints)."""
    import numpy as np
    import torch
    import rank_adapter_gb300 as ra

    kind = {"auto": ra.LORA_AUTO, "bgmv": ra.LORA_BGMV, "sgmv": ra.LORA_SGMV, "mixed": ra.LORA_MIXED}[args.kind]
    inst = make_workload(name, seed_offset=rank)
    alg = algorithmic(inst)
    min_seconds = args.min_seconds if min_seconds is None else min_seconds

    def dev(a, dt):
        a = np.ascontiguousarray(a)
        if dt == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a.astype(np.float32)).cuda()

    # Master copy of the slot table, written through lora_set_slot.
    master = ra.SlotTable(inst.d_in, inst.out_sizes, inst.num_slots, inst.r_max,
                          ra.LORA_BF16 if inst.dtype == "bf16" else ra.LORA_F32)
    for k, ad in sorted(inst.adapters.items()):
        master.set_slot(k, ad.rank, ad.scale, [dev(a, inst.dtype) for a in ad.A], [dev(b, inst.dtype) for b in ad.B])
        torch.cuda.synchronize()
    x0 = dev(inst.x, inst.dtype) if inst.token_ids is None else torch.from_numpy(inst.token_ids).cuda()
    y0 = dev(inst.y_in, inst.dtype)
    ts0 = torch.from_numpy(inst.token_slot).cuda()

    per = replica_bytes(inst)
    R = args.replicas or max(2, int(np.ceil(3 * L2_BYTES / per)))
    reps = [Replica(ra, torch, inst, master, x0, y0, ts0, kind) for _ in range(R)]
    del master
    torch.cuda.synchronize()

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            reps[i % R].launch(ra, i, path=args.path)
    stream.synchronize()

    G = args.graph_steps or R * max(1, 64 // R)
    G = min(G, max(1, args.steps))
    clocks = clock_sampler(local)
    ms, avg, kernel_timing, per_step = time_path(torch, ra, reps, stream, args.path, args.steps, G, min_seconds,
                                                 clocks, dist)
    st = region_stats(ms)
    out = {"alg": alg, "inst": inst, "regions": st, "kernel_ms": avg, "kernel_timing": kernel_timing,
           "per_step_launches": per_step, "clocks": clocks.summary(), "G": G, "R": R, "per": per}
    if with_other_path:
        other = "split" if args.path == "fused" else "fused"
        other_steps = min(args.steps, 20 * G)
        o_ms, o_avg, _, _ = time_path(torch, ra, reps, stream, other, other_steps, G, min(0.1, min_seconds))
        out["other"] = (other, statistics.median(o_ms) / other_steps, o_avg, other_steps)
    med_ms, _, total_TL = reduce_over_ranks(torch, dist, st["median_ms"], 0.0, alg["T_L"], "cuda")
    out["median_ms_all"] = med_ms
    out["total_TL"] = total_TL
    if not with_e2e:
        del reps
        torch.cuda.empty_cache()
        return out

    # End to end: every step copies its inputs in from pinned host memory, runs through the ABI and
    # copies its result back to pinned host memory. A serving loop keeps several steps in flight: up to
    # four replicas on four streams take turns, so one step's copies overlap other steps' kernels and
    # copies (the host link moves ~200 GB/s in either direction but not both at once, so the copies
    # bound the step); each step is one replay of a CUDA graph holding its copies and library calls.
    h_x = torch.empty_like(x0, device="cpu").pin_memory()
    h_x.copy_(x0)
    h_y = torch.empty_like(y0, device="cpu").pin_memory()
    h_y.copy_(y0)
    h_ts = torch.empty_like(ts0, device="cpu").pin_memory()
    h_ts.copy_(ts0)
    nbuf = min(4, R)
    pair = [reps[j] for j in range(nbuf)]
    h_out = [torch.empty_like(y0, device="cpu").pin_memory() for _ in range(nbuf)]
    h2d = h_x.numel() * h_x.element_size() + h_y.numel() * h_y.element_size() + h_ts.numel() * 4
    d2h = h_out[0].numel() * h_out[0].element_size()
    ne = max(3, args.e2e_steps)
    T = inst.num_tokens
    streams = [stream] + [torch.cuda.Stream() for _ in range(nbuf - 1)]

    def e2e_step(j):
        rep = pair[j]
        rep.x.copy_(h_x, non_blocking=True)
        rep.y.copy_(h_y, non_blocking=True)
        rep.meta.token_slot[:T].copy_(h_ts, non_blocking=True)
        rep.launch(ra, j, path=args.path)
        h_out[j].copy_(rep.y, non_blocking=True)

    e2e_graphs = []
    for j in range(nbuf):
        with torch.cuda.stream(streams[j]):
            e2e_step(j)  # warm (eager) before capture
        streams[j].synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=streams[j]):
            e2e_step(j)
        e2e_graphs.append(gr)
    for i in range(3 * nbuf):
        with torch.cuda.stream(streams[i % nbuf]):
            e2e_graphs[i % nbuf].replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    joins = [torch.cuda.Event() for _ in range(nbuf)]
    t0 = time.perf_counter()
    with torch.cuda.stream(streams[0]):
        e0.record()
    for j in range(1, nbuf):
        streams[j].wait_event(e0)
    for i in range(ne):
        with torch.cuda.stream(streams[i % nbuf]):
            e2e_graphs[i % nbuf].replay()
    for j in range(1, nbuf):
        joins[j].record(streams[j])
        streams[0].wait_event(joins[j])
    with torch.cuda.stream(streams[0]):
        e1.record()
    streams[0].synchronize()
    e2e_wall = time.perf_counter() - t0
    e2e_ms = e0.elapsed_time(e1)
    torch.cuda.synchronize()
    # The result the last step brought back is the full step's result (checked against a device step).
    last = (ne - 1) % nbuf
    ref_y = pair[last].y.cpu()
    if not torch.equal(h_out[last], ref_y):
        raise RuntimeError("end-to-end step: the host copy of y differs from the device result")
    _, e2e_ms, _ = reduce_over_ranks(torch, dist, 0.0, e2e_ms, alg["T_L"], "cuda")
    out["e2e"] = {"value": total_TL * ne / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / ne, "wall_s": e2e_wall,
                  "path": f"per step: pinned host x, y_in, token_slot -> device; one step; y -> host; "
                          f"{nbuf} replica(s) on {nbuf} stream(s) taking turns, each step one CUDA-graph replay"}
    del reps, pair, e2e_graphs
    torch.cuda.empty_cache()
    return out


def dense_roofline(name, m, path):
    """Roofline record of the dominant call of a measured dense workload."""
    hbm, tc, src = load_peaks()
    alg, avg = m["alg"], m["kernel_ms"]
    kbytes = {"apply": alg["step_bytes"], "shrink": alg["shrink_bytes"], "expand": alg["expand_bytes"]}
    kflops = {"apply": alg["flops"], "shrink": alg["shrink_flops"], "expand": alg["expand_flops"]}
    kern = max((k for k in avg if k != "meta"), key=lambda k: avg[k])
    kb = kbytes[kern]
    ach = kb / (avg[kern] * 1e-3) / 1e9
    rl = {"bound": "hbm", "kernel": kern, "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
          "peak_source": src, "algorithmic_bytes_per_launch": kb, "traffic": profiled_traffic(name, kern)}
    # The tensor pipe's share where the dense contraction runs on it, next to the ceiling the
    # arithmetic intensity allows when HBM is saturated.
    tflops = kflops[kern] / (avg[kern] * 1e-3) / 1e12
    rl["tensor"] = {"achieved_tflops": tflops, "peak_tflops": tc, "frac": tflops / tc,
                    "ceiling_frac_at_hbm_peak": min(1.0, (kflops[kern] / kb) * hbm * 1e9 / (tc * 1e12))}
    return rl


def sub_record(name, m, args, cpu=None):
    """The compact per-workload record of the default run's "configs"."""
    hbm, _, _ = load_peaks()
    alg, st = m["alg"], m["regions"]
    step_s = st["median_ms"] / args.steps * 1e-3
    rl = dense_roofline(name, m, args.path)
    rec = {"desc": WORKLOADS[name], "dtype": m["inst"].dtype, "T": alg["T"], "lora_tokens": alg["T_L"],
           "active_adapters": alg["active"], "tokens_per_s": alg["T_L"] / step_s,
           "step_us": st["median_ms"] / args.steps * 1e3, "step_us_min": st["min_ms"] / args.steps * 1e3,
           "step_us_max": st["max_ms"] / args.steps * 1e3, "regions": st["regions"],
           "kernel_us": {k: v * 1e3 for k, v in m["kernel_ms"].items()},
           "step_algorithmic_bytes": alg["step_bytes"],
           "step_frac_of_hbm": alg["step_bytes"] / step_s / 1e9 / hbm,
           "roofline": rl, "gpu_launches_per_step": m["per_step_launches"],
           "l2": f"rotating {m['R']} device replicas x {m['per'] / 2**20:.1f} MiB (> 3x {L2_BYTES >> 20} MiB L2)",
           "clocks": m["clocks"]}
    if cpu is not None:
        rec["cpu_baseline"] = cpu
    return rec


def run_ours(args):
    world, rank, local, dist = init_dist()
    m = measure_dense(args.workload, args, world, rank, local, dist)
    launches = int(round(m["per_step_launches"] * args.steps))  # counted by the library while capturing the step graph
    sub = {}
    if args.workload == "decode_qkv" and world == 1 and not args.no_configs:
        for name in ("toy_fp32", "prefill_gate_up", "mixed_o_proj"):
            ms = measure_dense(name, args, with_e2e=False, with_other_path=False)
            cpu = None if args.no_cpu_baseline else run_cpu_baseline(name, args.sub_cpu_seconds)
            sub[name] = sub_record(name, ms, args, cpu)
            del ms
        fd = measure_full_decode(args, min_seconds=args.min_seconds, with_e2e=False)
        sub["full_decode"] = fd["record"]
        if not args.no_cpu_baseline:
            sub["full_decode"]["cpu_baseline"] = run_cpu_baseline("full_decode", args.sub_cpu_seconds)

    if rank == 0:
        hbm, tc, src = load_peaks()
        alg, st = m["alg"], m["regions"]
        med_ms = m["median_ms_all"]
        step_ms = med_ms / args.steps
        other, o_ms, o_avg, other_steps = m["other"]
        line = {
            "metric": METRIC, "value": m["total_TL"] * args.steps / (med_ms * 1e-3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "ms_per_step_min": st["min_ms"] / args.steps, "ms_per_step_max": st["max_ms"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": m["inst"].dtype, "data": "synthetic",
            "config": workload_config(args.workload, args.kind, args.path, world, m["inst"].num_tokens, alg["T_L"],
                                      alg["active"]),
            "timing": f"{st['regions']} regions of exactly {args.steps} steps each ({st['timed_s']:.2f} s of device "
                      f"time), each region CUDA-graph replays of {m['G']} steps (library launches only) between "
                      f"CUDA events on the launching stream; value and ms_per_step from the median region; inputs: "
                      f"{m['R']} rotating device replicas x {m['per'] / 2**20:.1f} MiB (> 3x {L2_BYTES >> 20} MiB L2), "
                      f"each with its own metadata buffers, so every step but a graph's first prepares its "
                      f"metadata with lora_prepare_meta_unshared",
            "gpu_launches": launches,
            "step_algorithmic_bytes": alg["step_bytes"],
            "step_hbm_gbs": alg["step_bytes"] / (step_ms * 1e-3) / 1e9,
            "step_frac_of_hbm": alg["step_bytes"] / (step_ms * 1e-3) / 1e9 / hbm,
            "kernel_us": {k: v * 1e3 for k, v in m["kernel_ms"].items()},
            "kernel_timing": m["kernel_timing"],
            f"{other}_path": {"ms_per_step": o_ms, "kernel_us": {k: v * 1e3 for k, v in o_avg.items()},
                              "steps": other_steps},
            "roofline": dense_roofline(args.workload, m, args.path),
            "clocks": m["clocks"],
            "e2e": m["e2e"],
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = run_cpu_baseline(args.workload, args.cpu_seconds)
            line["cpu_baseline_single_thread"] = run_cpu_baseline(args.workload, args.sub_cpu_seconds, threads=1)
        if sub:
            line["configs"] = sub
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def full_decode_cpu(args):
    """The oracle on one layer (4 groups) of the full-model step, scaled to the step; one JSON line."""
    import numpy as np
    import oracle
    import workloads as wl
    if args.cpu_threads == 1:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    groups = []
    for inst in wl.full_decode_groups():
        groups.append(inst)
        if len(groups) == len(wl.FULL_DECODE_GROUPS):
            break
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.prepare_meta(groups[0].token_slot, groups[0].num_slots)
        for inst in groups:
            oracle.apply_requests(inst.to_f32(inst.x).astype(np.float64), inst.to_f32(inst.y_in).astype(np.float64),
                                  oracle.adapters_f64(inst), inst.out_sizes, inst.r_max, inst.req_lengths,
                                  inst.req_slots, inst.num_slots)
        reps += 1
        if time.perf_counter() - t0 >= args.cpu_seconds:
            break
    el = time.perf_counter() - t0
    sec_per_step = el / reps * 32          # 32 layers per step
    ts = groups[0].token_slot
    T_L = int((ts > 0).sum())
    print(json.dumps({"value": T_L / sec_per_step, "seconds": el, "reps": reps, "sec_per_step": sec_per_step,
                      "T_L": T_L, "T": int(len(ts)), "active": int(len(np.unique(ts[ts > 0])))}))


def measure_full_decode(args, world=1, rank=0, local=0, dist=None, min_seconds=None, with_e2e=True):
    """Full-model decode step: one lora_prepare_meta, then lora_apply for each of the 32 x 4 projection
    groups (own slot table, x and y each). Returns {"record": the sub-record, ...line fields}."""
    import numpy as np
    import torch
    import workloads as wl
    import rank_adapter_gb300 as ra
    kind = {"auto": ra.LORA_AUTO, "bgmv": ra.LORA_BGMV, "sgmv": ra.LORA_SGMV, "mixed": ra.LORA_MIXED}[args.kind]
    min_seconds = args.min_seconds if min_seconds is None else min_seconds

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    tables, xs, ys, step_bytes, T_L, ts, active = [], [], [], 0, 0, None, 0
    for inst in wl.full_decode_groups(seed=5 + 1000 * rank):
        t = ra.SlotTable(inst.d_in, inst.out_sizes, inst.num_slots, inst.r_max, ra.LORA_BF16)
        for k, ad in sorted(inst.adapters.items()):
            t.set_slot(k, ad.rank, ad.scale, [dev(m) for m in ad.A], [dev(m) for m in ad.B])
        tables.append(t)
        xs.append(dev(inst.x))
        ys.append(dev(inst.y_in))
        alg = algorithmic(inst)
        step_bytes += alg["step_bytes"]
        T_L, ts, S, active = alg["T_L"], inst.token_slot, inst.num_slots, alg["active"]
    torch.cuda.synchronize()
    T = len(ts)
    meta = ra.TokenMeta(T, S)
    meta.token_slot[:T].copy_(torch.from_numpy(ts))
    meta.set_num_tokens(T)
    ws = ra.workspace(max(tables, key=lambda t: ra.lora_workspace_bytes(t.desc, T, kind)), T, kind)
    ws_ptr, ws_bytes = (ws.data_ptr(), ws.numel() * 4) if ws is not None else (0, 0)

    def step(st):
        ra.check(ra.lora_prepare_meta(meta.c, st), "prepare_meta")
        for t, x, y in zip(tables, xs, ys):
            ra.check(ra.lora_apply(t.desc, meta.c, x.data_ptr(), x.stride(0), 0, y.data_ptr(), y.stride(0),
                                   ra.LORA_BF16, kind, ws_ptr, ws_bytes, st), "apply")

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(None)
    stream.synchronize()
    n0 = ra.lora_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(None)
    per_step = ra.lora_launch_count() - n0
    with torch.cuda.stream(stream):
        for _ in range(2):
            graph.replay()
    stream.synchronize()
    clocks = clock_sampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)

    def region():
        for _ in range(args.steps):
            graph.replay()

    ms = time_regions(torch, stream, region, min_seconds)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.stop()
    st = region_stats(ms)
    hbm, tc, src = load_peaks()
    step_ms = st["median_ms"] / args.steps
    ach = step_bytes / (step_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": "step (1 metadata + 128 lora_apply)", "achieved": ach,
            "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "peak_source": src,
            "algorithmic_bytes_per_launch": step_bytes, "traffic": None}
    out = {"regions": st, "clocks": clocks.summary(), "per_step": per_step, "T": T, "T_L": T_L, "active": active,
           "step_bytes": step_bytes, "roofline": roof, "groups": len(tables)}
    out["record"] = {"desc": WORKLOADS["full_decode"], "dtype": "bf16", "T": T, "lora_tokens": T_L,
                     "active_adapters": active, "tokens_per_s": T_L / (step_ms * 1e-3), "step_us": step_ms * 1e3,
                     "step_us_min": st["min_ms"] / args.steps * 1e3, "step_us_max": st["max_ms"] / args.steps * 1e3,
                     "regions": st["regions"], "step_algorithmic_bytes": step_bytes, "step_frac_of_hbm": ach / hbm,
                     "roofline": roof, "gpu_launches_per_step": per_step,
                     "l2": L2_NOTES["full_decode"], "clocks": out["clocks"]}
    if not with_e2e:
        del graph, tables, xs, ys, ws
        torch.cuda.empty_cache()
        return out

    # End to end: token slots and every group's x and y_in in from pinned host memory, every y out.
    hx = [torch.empty_like(x, device="cpu").pin_memory().copy_(x) for x in xs]
    hy = [torch.empty_like(y, device="cpu").pin_memory().copy_(y) for y in ys]
    hout = [torch.empty_like(y, device="cpu").pin_memory() for y in ys]
    hts = torch.from_numpy(ts).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hx + hy) + hts.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in hout)

    def e2e_step():
        meta.token_slot[:T].copy_(hts, non_blocking=True)
        for x, y, a, b in zip(xs, ys, hx, hy):
            x.copy_(a, non_blocking=True)
            y.copy_(b, non_blocking=True)
        step(None)
        for y, o in zip(ys, hout):
            o.copy_(y, non_blocking=True)

    ne = max(2, args.e2e_steps)
    with torch.cuda.stream(stream):
        e2e_step()
    stream.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()  # the step's copies and calls, replayed as one graph per step
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_step()
    with torch.cuda.stream(stream):
        e2e_graph.replay()
    stream.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record()
        for _ in range(ne):
            e2e_graph.replay()
        f1.record()
    stream.synchronize()
    e2e_ms = f0.elapsed_time(f1)
    med_ms, e2e_ms, total_TL = reduce_over_ranks(torch, dist, st["median_ms"], e2e_ms, T_L, "cuda")
    out.update(median_ms_all=med_ms, total_TL=total_TL)
    out["e2e"] = {"value": total_TL * ne / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / ne,
                  "path": "pinned host token slots and every group's x, y_in -> device; one step; every y -> host; "
                          "each step one CUDA-graph replay"}
    return out


def run_full_decode(args):
    world, rank, local, dist = init_dist()
    m = measure_full_decode(args, world, rank, local, dist)
    if rank == 0:
        st = m["regions"]
        step_ms = m["median_ms_all"] / args.steps
        line = {
            "metric": METRIC, "value": m["total_TL"] * args.steps / (m["median_ms_all"] * 1e-3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "ms_per_step_min": st["min_ms"] / args.steps, "ms_per_step_max": st["max_ms"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": workload_config("full_decode", args.kind, "fused", world, m["T"], m["T_L"], m["active"]),
            "timing": f"{st['regions']} regions of exactly {args.steps} steps ({st['timed_s']:.2f} s of device time), "
                      f"each step one CUDA-graph replay (library launches only), CUDA events; median region",
            "gpu_launches": m["per_step"] * args.steps,
            "step_algorithmic_bytes": m["step_bytes"],
            "roofline": m["roofline"],
            "clocks": m["clocks"],
            "e2e": m["e2e"],
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = run_cpu_baseline("full_decode", args.cpu_seconds)
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def moe_algorithmic(m, pair_slot):
    """Bytes of one MoE-layer step: every active composite slot's w13 and w2 weights once, the token
    rows x of tokens with a live pair once, h2 of live pairs once, h1 and h3 of live pairs read and
    written once (bf16), and the routing ints. pair_slot: the pairs' composite slots (from the step)."""
    import numpy as np
    pair_slot = np.asarray(pair_slot)
    live = pair_slot > 0
    active = np.unique(pair_slot[live])
    r = m.w13.r_max
    w = int(len(active)) * 2 * r * (2 * m.hidden + 2 * m.inter + m.inter + m.hidden)
    tok = int(np.unique(np.nonzero(live)[0] // m.topk).size)
    P_L = int(live.sum())
    act = 2 * tok * m.hidden + 2 * P_L * m.inter + 2 * 2 * P_L * 2 * m.inter + 2 * 2 * P_L * m.hidden
    ints = 4 * m.num_tokens * (1 + 2 * m.topk)
    return dict(step_bytes=w + act + ints, T_L=int((m.token_slot > 0).sum()), pairs_live=P_L, active=int(len(active)))


def moe_cpu(args):
    """The oracle on the MoE-layer step (pair slots, metadata, w13, w2); one JSON line."""
    import numpy as np
    import oracle
    import workloads as wl
    if args.cpu_threads == 1:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    m = wl.make_moe_instance()
    a13, a2 = oracle.adapters_f64(m.w13), oracle.adapters_f64(m.w2)
    x = m.w13.to_f32(m.w13.x).astype(np.float64)
    h1 = m.w13.to_f32(m.w13.y_in).astype(np.float64)
    h2 = m.w2.to_f32(m.w2.x).astype(np.float64)
    h3 = m.w2.to_f32(m.w2.y_in).astype(np.float64)
    S = m.w13.num_slots
    reps, t0 = 0, time.perf_counter()
    while True:
        pair = oracle.moe_pair_slots(m.token_slot, m.topk_ids, m.num_loras, m.num_experts, m.local_experts,
                                     m.expert_map)
        oracle.prepare_meta(pair, S)
        oracle.moe_lora_w13(x, h1, pair, m.topk, a13, m.w13.out_sizes, S)
        oracle.moe_lora_w2(h2, h3, pair, a2, m.hidden, S)
        reps += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds:
            break
    alg = moe_algorithmic(m, pair)
    print(json.dumps({"value": reps * alg["T_L"] / el, "seconds": el, "reps": reps, "sec_per_step": el / reps,
                      "T_L": alg["T_L"], "T": m.num_tokens, "pairs": m.num_tokens * m.topk,
                      "live_pairs": alg["pairs_live"], "active_composite_slots": alg["active"]}))


def run_moe(args):
    """One mixture-of-experts layer's LoRA per step: the pairs' composite slots, the metadata over the
    pairs, the w13 application (x rows shared by a token's top-k pairs) and the w2 application."""
    import numpy as np
    import torch
    import workloads as wl
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import rank_adapter_gb300 as ra
    kind = {"auto": ra.LORA_AUTO, "bgmv": ra.LORA_BGMV, "sgmv": ra.LORA_SGMV, "mixed": ra.LORA_MIXED}[args.kind]
    m = wl.make_moe_instance(seed=8 + 1000 * rank)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    def table(layer, x_row_div):
        t = ra.SlotTable(layer.d_in, layer.out_sizes, layer.num_slots, layer.r_max, ra.LORA_BF16,
                         x_row_div=x_row_div)
        for k, ad in sorted(layer.adapters.items()):
            t.set_slot(k, ad.rank, ad.scale, [dev(w) for w in ad.A], [dev(w) for w in ad.B])
        return t

    t13, t2 = table(m.w13, m.topk), table(m.w2, 1)
    T, K, S = m.num_tokens, m.topk, m.w13.num_slots
    P = T * K
    ts = torch.from_numpy(m.token_slot).cuda()
    ids = torch.from_numpy(np.ascontiguousarray(m.topk_ids)).cuda()
    emap = torch.from_numpy(m.expert_map).cuda() if m.expert_map is not None else None
    x, h1, h2, h3 = dev(m.w13.x), dev(m.w13.y_in), dev(m.w2.x), dev(m.w2.y_in)
    meta = ra.TokenMeta(P, S)
    meta.set_num_tokens(P)
    ws = ra.workspace(max((t13, t2), key=lambda t: ra.lora_workspace_bytes(t.desc, P, kind)), P, kind)
    ws_ptr, ws_bytes = (ws.data_ptr(), ws.numel() * 4) if ws is not None else (0, 0)
    torch.cuda.synchronize()

    def step(st):
        ra.check(ra.lora_moe_pair_slots(ts.data_ptr(), ids.data_ptr(), T, K, m.num_loras, m.num_experts,
                                        m.local_experts, emap.data_ptr() if emap is not None else 0,
                                        meta.token_slot.data_ptr(), st), "moe_pair_slots")
        ra.check(ra.lora_prepare_meta(meta.c, st), "prepare_meta")
        ra.check(ra.lora_apply(t13.desc, meta.c, x.data_ptr(), x.stride(0), 0, h1.data_ptr(), h1.stride(0),
                               ra.LORA_BF16, kind, ws_ptr, ws_bytes, st), "apply w13")
        ra.check(ra.lora_apply(t2.desc, meta.c, h2.data_ptr(), h2.stride(0), 0, h3.data_ptr(), h3.stride(0),
                               ra.LORA_BF16, kind, ws_ptr, ws_bytes, st), "apply w2")

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(None)
    stream.synchronize()
    alg = moe_algorithmic(m, meta.token_slot[:P].cpu().numpy())   # the pairs' slots as the step computed them
    n0 = ra.lora_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(None)
    per_step = ra.lora_launch_count() - n0
    with torch.cuda.stream(stream):
        for _ in range(2):
            graph.replay()
    stream.synchronize()
    clocks = clock_sampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)

    def region():
        for _ in range(args.steps):
            graph.replay()

    ms = time_regions(torch, stream, region, args.min_seconds)
    st = region_stats(ms)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.stop()
    elapsed_ms = st["median_ms"]

    # End to end: routing, x and the base outputs h1, h2, h3 in from pinned host memory, h1 and h3 out;
    # each step one CUDA-graph replay of its copies and calls.
    pin = lambda t: torch.empty_like(t, device="cpu").pin_memory().copy_(t)   # noqa: E731
    h_in = [(d, pin(d)) for d in (ts, ids, x, h1, h2, h3)]
    h_out = [(d, torch.empty_like(d, device="cpu").pin_memory()) for d in (h1, h3)]
    h2d = sum(h.numel() * h.element_size() for _, h in h_in)
    d2h = sum(h.numel() * h.element_size() for _, h in h_out)

    def e2e_step():
        for d, h in h_in:
            d.copy_(h, non_blocking=True)
        step(None)
        for d, h in h_out:
            h.copy_(d, non_blocking=True)

    ne = max(3, args.e2e_steps)
    with torch.cuda.stream(stream):
        e2e_step()
    stream.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_step()
    with torch.cuda.stream(stream):
        e2e_graph.replay()
    stream.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record()
        for _ in range(ne):
            e2e_graph.replay()
        f1.record()
    stream.synchronize()
    e2e_ms = f0.elapsed_time(f1)
    elapsed_ms, e2e_ms, total_TL = reduce_over_ranks(torch, dist, elapsed_ms, e2e_ms, alg["T_L"], "cuda")
    if rank == 0:
        hbm, _, src = load_peaks()
        step_ms = elapsed_ms / args.steps
        ach = alg["step_bytes"] / (step_ms * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": total_TL * args.steps / (elapsed_ms * 1e-3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "ms_per_step_min": st["min_ms"] / args.steps, "ms_per_step_max": st["max_ms"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": workload_config("moe_decode", args.kind, "fused", world, T, alg["T_L"], None,
                                      {"pairs": P, "live_pairs": alg["pairs_live"],
                                       "active_composite_slots": alg["active"]}),
            "timing": f"{st['regions']} regions of exactly {args.steps} steps ({st['timed_s']:.2f} s of device time), "
                      f"each step one CUDA-graph replay (library launches only), CUDA events; median region",
            "gpu_launches": per_step * args.steps,
            "step_algorithmic_bytes": alg["step_bytes"],
            "roofline": {"bound": "hbm", "kernel": "step (pair slots + metadata + w13 and w2 lora_apply)",
                         "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "peak_source": src,
                         "algorithmic_bytes_per_launch": alg["step_bytes"], "traffic": None},
            "clocks": clocks.summary(),
            "e2e": {"value": total_TL * ne / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / ne,
                    "path": "pinned host token slots, top-k ids, x, h1, h2, h3 -> device; one step; h1, h3 -> host; "
                            "each step one CUDA-graph replay"},
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = run_cpu_baseline("moe_decode", args.cpu_seconds)
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_child:
        if args.workload == "full_decode":
            full_decode_cpu(args)
        elif args.workload == "moe_decode":
            moe_cpu(args)
        else:
            cpu_child(args)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "full_decode":
        return run_full_decode(args)
    if args.workload == "moe_decode":
        return run_moe(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
