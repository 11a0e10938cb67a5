#!/usr/bin/env python3
"""Throughput of the DSA + IndexShare hot path on one GB300 (or N replicas).

A step is one F,S,S,S group forward over a 131,072-token causal prefill (FP8 e4m3 indexer
with H_I=64, d_I=128, top-2048; four layers of 64-head sparse MQA over a 576-dim latent
KV), through ``indexshare_group_forward``: the full layer's indexer + top-k, then four
attention layers over its index buffer.  Inputs are seeded synthetic tensors of that shape
(see ``synth``), far larger than L2.

Prints one JSON line (rank 0).  ``value`` is group-prefill tokens/s summed over ranks;
``indexer_topk`` gives the indexer+top-k query rows/s of the same workload.  ``--impl
reference`` times the CPU oracle instead, on sampled rows of the same workload.
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from long_context_sparse_tcgen05_gb300 import synth  # noqa: E402

METRIC = "indexer+top-k query rows/s at L=128K; FSSS 4-layer group prefill tokens/s"
UNIT = "tokens/s"
GROUP = "FSSS"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_128k")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other configurations after the headline")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target oracle CPU time")
    ap.add_argument("--kernel", choices=["attn", "indexer", "topk", "ixtopk", "quant"], default=None,
                    help="time one call on a single-kernel case instead of the group step "
                         "(the case the committed ncu summaries are captured on)")
    ap.add_argument("--rows", type=int, default=2048, help="--kernel: query rows (the last rows of the sequence)")
    ap.add_argument("--keys", type=int, default=131072, help="--kernel/--heatmap: sequence length")
    ap.add_argument("--varlen", action="store_true",
                    help="one F,S,S,S group over eight packed prompts of 1K..64K tokens "
                         "(indexshare_group_forward_varlen) against the same prompts one call each")
    ap.add_argument("--peaks", action="store_true",
                    help="measure the dense FP8 tensor peak (cuBLAS e4m3 GEMM) and print it")
    ap.add_argument("--heatmap", action="store_true",
                    help="all-F pass over the 16 layers of heatmap_128k, the layer-overlap matrix, "
                         "the best schedule per number of full layers and measured group times")
    return ap.parse_args()


# --- distributed plumbing (replicas: each rank runs its own group; barrier + max time) ---

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --- clocks ---------------------------------------------------------------------------

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
                power.append(float(p[3]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# --- algorithmic work -------------------------------------------------------------------

def visible_counts(wl) -> np.ndarray:
    t = np.arange(wl.T, dtype=np.int64)
    return np.tile(np.clip(wl.q_pos0 + t + wl.diag, 0, wl.S), wl.B)


def attn_bytes(wl) -> float:
    """Algorithmic HBM bytes of one sparse-attention launch: per query row, the gathered
    latent rows (2*d_qk bytes each, min(k, n_t) of them), Q, O, the index row and LSE."""
    n = visible_counts(wl)
    kk = np.minimum(n, wl.k).astype(np.float64)
    per_row_fixed = wl.H * wl.DQK * 2 + wl.H * wl.DV * 2 + wl.k * 4 + wl.H * 4
    return float(np.sum(kk * wl.DQK * 2) + len(n) * per_row_fixed)


def attn_flops(wl) -> float:
    n = visible_counts(wl)
    kk = np.minimum(n, wl.k).astype(np.float64)
    return float(np.sum(kk) * 2 * wl.H * (wl.DQK + wl.DV))


def indexer_flops(wl) -> float:
    return float(np.sum(visible_counts(wl).astype(np.float64)) * 2 * wl.HI * wl.DI)


def stores_scores(wl) -> bool:
    """Whether dsa_topk from indexer operands passes this workload's scores through a score
    buffer (few query rows, 4 indexer heads or k > 2,048) rather than keeping candidates only."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    return wl.HI != 64 or wl.k > 2048 or wl.B * ((wl.T + 3) // 4) < 4 * sms


def indexer_bytes(wl) -> float:
    """Algorithmic HBM bytes of one indexer call: the key cache and its scales, the queries, head
    weights and scales, and -- where the path stores scores (decode's few rows) -- the fp32 score
    of every visible pair written once."""
    elt = 1 if wl.idx_dtype == "e4m3" else 2
    keys = wl.B * wl.S * (wl.DI * elt + 4)
    queries = wl.B * wl.T * (wl.HI * wl.DI * elt + wl.HI * 4 + 4)
    scores = np.sum(visible_counts(wl).astype(np.float64)) * 4 if stores_scores(wl) else 0.0
    return float(keys + queries + scores)


def captured_traffic(kernel: str, units: int):
    """DRAM bytes (read + write) per launch of `kernel` over `units` query rows, scaled from
    the ncu capture recorded in profiles/traffic.json -- or None when the kernel's source has
    changed since that capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, "no capture"
    rec = json.load(open(p)).get(kernel)
    if rec is None:
        return None, "no capture"
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != rec["sha256"]:
        return None, "kernel changed since " + rec["capture"]
    return round(rec["dram_bytes_per_query_row"] * units), (
        f"{rec['capture']}: {rec['dram_bytes'] / 1e9:.2f} GB over {rec['query_rows']} query rows, scaled by rows")


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def fp8_peak(dev, sustain_s: float = 3.0) -> dict:
    """Dense FP8 e4m3 tensor throughput of this GPU, measured the way the bf16 figure in
    MEASURED_PEAKS.json is: a cuBLAS GEMM (torch._scaled_mm, e4m3 x e4m3 -> bf16, unit scales)
    at 8192^3 counted as 2*N^3 flop, best of 10 (burst) and back to back for `sustain_s`
    seconds (sustained, under the power cap)."""
    n = 8192
    g = torch.Generator(device=dev)
    g.manual_seed(synth.SEED_BASE + 99)
    a = torch.randn((n, n), generator=g, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn((n, n), generator=g, device=dev).to(torch.float8_e4m3fn)
    one = torch.ones((), dtype=torch.float32, device=dev)
    out = torch.empty((n, n), dtype=torch.bfloat16, device=dev)

    def mm():
        torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16, out=out)

    for _ in range(3):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    flop = 2.0 * n ** 3
    reps = max(1, int(sustain_s / (best * 1e-3)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        mm()
    e1.record()
    torch.cuda.synchronize()
    sus = e0.elapsed_time(e1) / reps
    del a, b, out
    return {"fp8_tflops": round(flop / (best * 1e-3) / 1e12, 1),
            "fp8_tflops_sustained": round(flop / (sus * 1e-3) / 1e12, 1),
            "how": "torch._scaled_mm e4m3 8192^3 (2*N^3): best of 10 (burst) and back to back for "
                   f"{sustain_s:g} s (sustained), measured in this run"}


# --- timing helpers ---------------------------------------------------------------------

def time_loop(fn, steps, warmup, world=1):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        fn()
    e1.record(st)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / steps


# --- CPU oracle on sampled rows --------------------------------------------------------

def oracle_sample(wl, host_ix, host_ats, rows, k):
    """Oracle time for the sampled rows of one group: (indexer+top-k s, attention s)."""
    import oracle
    t0 = time.perf_counter()
    idx = oracle.indexer_topk(host_ix, k, rows)
    t1 = time.perf_counter()
    for at in host_ats:
        oracle.sparse_attn(at, idx, rows)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def host_sample(wl, ix, ats, rows):
    """Host copies of what the sampled rows read: their query rows, all keys / KV."""
    r = torch.as_tensor(rows, device=ix["q"].device)

    def take(t, lead):
        return None if t is None else t.reshape((-1,) + tuple(t.shape[lead:]))[r].cpu()

    hix = dict(q_rows=take(ix["q"], 2), w_rows=take(ix["w"], 2), q_scale_rows=take(ix.get("q_scale"), 2),
               k=ix["k"].cpu(), k_scale=None if ix.get("k_scale") is None else ix["k_scale"].cpu(),
               T=wl.T, S=wl.S, q_pos0=wl.q_pos0, diag=wl.diag)
    hats = [dict(q_rows=take(at["q"], 2), k=at["k"].cpu(), v=None if at.get("v") is None else at["v"].cpu(),
                 d_v=at["d_v"], scale=at["scale"], T=wl.T) for at in ats]
    return hix, hats


def extrapolate(wl, rows, t_ix, t_at):
    n = visible_counts(wl).astype(np.float64)
    ns = n[np.asarray(rows)]
    kk, kks = np.minimum(n, wl.k), np.minimum(ns, wl.k)
    tot_ix = t_ix * n.sum() / max(ns.sum(), 1.0)
    tot_at = t_at * kk.sum() / max(kks.sum(), 1.0)
    return tot_ix, tot_at


def pick_rows(wl, n_rows, seed=5):
    g = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([g.integers(0, wl.B * wl.T, n_rows), [wl.B * wl.T - 1]]))
    return rows.tolist()


def cpu_baseline(wl, ix, ats, target_s):
    """Time the oracle as it stands on a bounded row sample; extrapolate to tokens/s."""
    import oracle
    probe = pick_rows(wl, 4, seed=1)
    hix, hats = host_sample(wl, ix, ats, probe)
    a, b = oracle_sample(wl, hix, hats, probe, wl.k)
    n_rows = int(max(4, min(512, len(probe) * target_s / max(a + b, 1e-3))))
    rows = pick_rows(wl, n_rows)
    hix, hats = host_sample(wl, ix, ats, rows)
    t_ix, t_at = oracle_sample(wl, hix, hats, rows, wl.k)
    tot_ix, tot_at = extrapolate(wl, rows, t_ix, t_at)
    return {"value": wl.B * wl.T / (tot_ix + tot_at), "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{len(rows)} query rows of {wl.name} (indexer+top-k and 4 attention layers); "
                      f"{t_ix + t_at:.1f} s measured, extrapolated by visible-key and selected-key counts",
            "indexer_topk_rows_per_s": wl.B * wl.T / tot_ix}


# --- our arm ----------------------------------------------------------------------------

def run_ours(args, rank, world, local):
    import long_context_sparse_tcgen05_gb300 as dsa
    from long_context_sparse_tcgen05_gb300 import build
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    dsa.load_library()
    wl = synth.WORKLOADS[args.workload]
    layers = synth.group_inputs(wl, 4, dev, with_indexer=True)
    group = [dict(ix=layers[0]["ix"], at=layers[l]["at"]) for l in range(4)]
    ws_need = dsa.workspace_size(layers[0]["ix"], wl.k)
    dsa.workspace(ws_need, dev)
    outs = [torch.empty(wl.B, wl.T, wl.H, wl.DV, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    lses = [torch.empty(wl.B, wl.T, wl.H, dtype=torch.float32, device=dev) for _ in range(4)]
    bufs = [torch.empty(wl.B, wl.T, wl.k, dtype=torch.int32, device=dev) for _ in range(4)]

    def step():
        dsa.indexshare_group_forward(group, GROUP, wl.k, outs=outs, lses=lses, idx_bufs=bufs[:1])

    clocks = Clocks(local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    n0 = dsa.launch_count()
    clocks.start()
    # every launch of the timed steps is bracketed by CUDA events on its stream, so each
    # kernel's device time is measured inside the timed region itself
    dsa.trace_enable(256 * args.steps + 64)
    ms = time_loop(step, args.steps, 0, world)
    clk = clocks.stop()
    launches = dsa.launch_count() - n0
    trace = dsa.trace_read()
    dsa.trace_disable()
    by_kind = {}
    for kind, t in trace:
        by_kind.setdefault(kind, []).append(t)
    ms = max_over_ranks(ms, world)
    tokens = wl.B * wl.T
    value = tokens * world / (ms / 1e3)

    # components, each timed alone with the same launches the step makes
    at_ms = time_loop(lambda: dsa.dsa_sparse_attn(group[1]["at"], bufs[0], out=outs[1], lse=lses[1]),
                      max(3, args.steps // 2), 1)
    ix_ms = time_loop(lambda: dsa.dsa_topk(wl.k, ix=layers[0]["ix"], idx=bufs[0]), max(3, args.steps // 2), 1)
    ffff = [dict(ix=layers[l]["ix"], at=layers[l]["at"]) for l in range(4)]
    ffff_ms = time_loop(lambda: dsa.indexshare_group_forward(ffff, "FFFF", wl.k, outs=outs, lses=lses, idx_bufs=bufs),
                        max(2, args.steps // 3), 1)
    _, overlap01 = dsa.topk_overlap(bufs[0], bufs[1], per_row=False)
    flags = dsa.read_device_flags(dev)

    peaks = load_peaks()
    a_bytes = attn_bytes(wl)
    att_launch_ms = float(np.mean(by_kind["attention"]))  # mean device time in the timed region
    att_gbs = a_bytes / (att_launch_ms / 1e3) / 1e9
    ix_tf = indexer_flops(wl) / (ix_ms / 1e3) / 1e12
    fp8 = fp8_peak(dev)  # measured in this run: the indexer's tensor roof
    fp8_peak_tf = fp8["fp8_tflops"]
    attn_total = 4 * at_ms
    if attn_total >= ix_ms:
        traffic, traffic_src = captured_traffic("k_sparse_mla_tc", wl.B * wl.T)
        roof = {"kernel": "sparse MLA attention (k_sparse_mla_tc)", "bound": "hbm", "achieved": round(att_gbs, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(att_gbs / peaks["hbm_gbs"], 4),
                "traffic": traffic, "traffic_src": traffic_src, "algorithmic_bytes_per_launch": a_bytes,
                "launch_ms": round(att_launch_ms, 3), "launches_timed": len(by_kind["attention"]),
                "peak_src": peaks["src"]}
    else:
        ixk_ms = float(np.sum(by_kind.get("indexer", [0.0]))) / args.steps
        ix_tf = indexer_flops(wl) / (ixk_ms / 1e3) / 1e12
        ix_gbs = indexer_bytes(wl) / (ixk_ms / 1e3) / 1e9
        # the bound is the roof the indexer's arithmetic intensity meets first (decode reads
        # the whole key cache for a few queries: about 124 flop per byte, under the FP8 ridge)
        if indexer_flops(wl) / indexer_bytes(wl) >= fp8_peak_tf * 1e12 / (peaks["hbm_gbs"] * 1e9):
            roof = {"kernel": "indexer (k_indexer_tc, FP8)", "bound": "tensor", "achieved": round(ix_tf, 1),
                    "peak": fp8_peak_tf, "unit": "TFLOP/s", "frac": round(ix_tf / fp8_peak_tf, 4), "traffic": None,
                    "algorithmic_flops_per_call": indexer_flops(wl), "call_ms": round(ixk_ms, 3),
                    "peak_src": "measured in this run (cuBLAS e4m3 GEMM, burst)"}
        else:
            roof = {"kernel": "indexer (k_indexer_tc, FP8)", "bound": "hbm", "achieved": round(ix_gbs, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ix_gbs / peaks["hbm_gbs"], 4),
                    "traffic": None, "algorithmic_bytes_per_call": indexer_bytes(wl),
                    "call_ms": round(ixk_ms, 3), "peak_src": peaks["src"]}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3+bf16", "data": "synthetic",
        "config": {"workload": wl.name, "L": wl.S, "query_rows": wl.B * wl.T, "k": wl.k, "schedule": GROUP,
                   "H_I": wl.HI, "d_I": wl.DI, "indexer_dtype": wl.idx_dtype, "H": wl.H, "d_qk": wl.DQK,
                   "d_v": wl.DV, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (%.1f GB read per step)" % (
                       (sum(t.numel() * t.element_size() for t in (layers[0]["ix"]["q"], layers[0]["ix"]["k"])) +
                        4 * layers[0]["at"]["q"].numel() * 2) / 1e9)},
        "indexer_topk": {"value": round(tokens * world / (ix_ms / 1e3), 1), "unit": "rows/s", "ms": round(ix_ms, 3),
                         "tflops": round(ix_tf, 1)},
        "fp8_peak": fp8,
        "indexer_kernel": _indexer_kernel_line(wl, by_kind, args.steps, fp8_peak_tf),
        "attention_layer_ms": round(at_ms, 3), "attention_gbs": round(att_gbs, 1),
        "attention_tflops": round(attn_flops(wl) / (at_ms / 1e3) / 1e12, 1),
        "fsss_vs_ffff": {"fsss_ms": round(ms, 3), "ffff_ms": round(ffff_ms, 3), "speedup": round(ffff_ms / ms, 3),
                         "adjacent_layer_overlap": round(overlap01, 4)},
        "roofline": roof, "gpu_launches": int(launches), "clocks": clk, "device_flags": flags,
        "kernel_ms_per_step": {k: round(float(np.sum(v)) / args.steps, 3) for k, v in sorted(by_kind.items())},
    }

    if not args.no_e2e:
        line["e2e"] = run_e2e(dsa, wl, layers, group, outs, lses, bufs, args, world)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(wl, layers[0]["ix"], [g["at"] for g in group], args.cpu_seconds)
    if not args.no_workloads:
        del layers, group, ffff, outs, lses, bufs
        torch.cuda.empty_cache()
        line["workloads"] = run_workloads(dsa, dev, peaks, fp8_peak_tf, world)
    return line


def run_workloads(dsa, dev, peaks, fp8_tf, world, steps=3):
    """The project's other configurations after the headline step, a few steps each through the
    same call (one F,S,S,S group of the workload's first four layers): group ms and tokens/s;
    for the three large ones also the all-full (F,F,F,F) group and the speedup of F,S,S,S over
    it, and the roofline fraction of the kernel that dominates the F,S,S,S step (attention
    against measured HBM; the indexer against the tensor peak of its dtype -- FP8 measured in
    this run, bf16 from the measured peaks -- or HBM where its arithmetic intensity is below the
    ridge, as in decode)."""
    res = {}
    for name in ("tiny_l1k", "prefill_16k", "decode_b32_200k", "chunked_prefill_1m"):
        wl = synth.WORKLOADS[name]
        layers = synth.group_inputs(wl, 4, dev, with_indexer=True)
        fsss = [dict(ix=layers[0]["ix"], at=layers[l]["at"]) for l in range(4)]
        ffff = [dict(ix=layers[l]["ix"], at=layers[l]["at"]) for l in range(4)]
        outs = [torch.empty(wl.B, wl.T, wl.H, wl.DV, dtype=torch.bfloat16, device=dev) for _ in range(4)]
        lses = [torch.empty(wl.B, wl.T, wl.H, dtype=torch.float32, device=dev) for _ in range(4)]
        bufs = [torch.empty(wl.B, wl.T, wl.k, dtype=torch.int32, device=dev) for _ in range(4)]

        def step():
            dsa.indexshare_group_forward(fsss, "FSSS", wl.k, outs=outs, lses=lses, idx_bufs=bufs[:1])

        for _ in range(2):
            step()
        torch.cuda.synchronize()
        dsa.trace_enable(256 * steps + 64)
        ms = time_loop(step, steps, 0, world)
        trace = dsa.trace_read()
        dsa.trace_disable()
        by_kind = {}
        for kind, t in trace:
            by_kind[kind] = by_kind.get(kind, 0.0) + t / steps
        ent = {"group_ms": round(ms, 3), "tokens_per_s": round(wl.B * wl.T * world / (ms / 1e3), 1),
               "kernel_ms_per_step": {k: round(v, 3) for k, v in sorted(by_kind.items())}}
        if name != "tiny_l1k":
            ffff_ms = time_loop(lambda: dsa.indexshare_group_forward(ffff, "FFFF", wl.k, outs=outs, lses=lses,
                                                                      idx_bufs=bufs), 2, 1, world)
            ent["ffff_ms"] = round(ffff_ms, 3)
            ent["fsss_vs_ffff"] = round(ffff_ms / ms, 3)
            att, ixt = by_kind.get("attention", 0.0), by_kind.get("indexer", 0.0) + by_kind.get("topk", 0.0)
            if att >= ixt:
                gbs = 4 * attn_bytes(wl) / (att / 1e3) / 1e9
                ent["roofline"] = {"kernel": "sparse MLA attention", "bound": "hbm", "achieved": round(gbs, 1),
                                   "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4)}
            else:
                ix_ms = by_kind.get("indexer", 0.0)
                fp8 = wl.idx_dtype == "e4m3"
                tpeak = fp8_tf if fp8 else peaks["bf16_tflops"]
                kern = "indexer (%s)" % ("FP8" if fp8 else "bf16")
                if indexer_flops(wl) / indexer_bytes(wl) >= tpeak * 1e12 / (peaks["hbm_gbs"] * 1e9):
                    tf = indexer_flops(wl) / (ix_ms / 1e3) / 1e12
                    ent["roofline"] = {"kernel": kern, "bound": "tensor", "achieved": round(tf, 1),
                                       "peak": tpeak, "unit": "TFLOP/s", "frac": round(tf / tpeak, 4)}
                else:
                    gbs = indexer_bytes(wl) / (ix_ms / 1e3) / 1e9
                    ent["roofline"] = {"kernel": kern, "bound": "hbm", "achieved": round(gbs, 1),
                                       "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4)}
        res[name] = ent
        del layers, fsss, ffff, outs, lses, bufs
        torch.cuda.empty_cache()
    res["mtp_draft_b32_200k"] = run_draft(dsa, dev, world, steps)
    return res


def run_draft(dsa, dev, world, steps=3):
    """The four draft steps of a multi-token-prediction layer over the batch-32 200K decode
    cache: one indexshare_draft_forward call (the first step's indexer + top-k, then one
    attention launch for all steps over its index row) beside the same steps run as an F,S,S,S
    group (whose layers reading one index buffer also share an attention launch when they have
    few rows); ms of each and their ratio."""
    wl = synth.WORKLOADS["mtp_draft_b32_200k"]
    layers = synth.group_inputs(wl, 4, dev, with_indexer=True)
    group = [dict(ix=layers[0]["ix"], at=layers[l]["at"]) for l in range(4)]
    at = dict(layers[0]["at"])
    at["q"] = torch.cat([l["at"]["q"] for l in layers], dim=1).contiguous()
    out = torch.empty(wl.B, 4, wl.H, wl.DV, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(wl.B, 4, wl.H, dtype=torch.float32, device=dev)
    idx = torch.empty(wl.B, 1, wl.k, dtype=torch.int32, device=dev)
    outs = [torch.empty(wl.B, 1, wl.H, wl.DV, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    lses = [torch.empty(wl.B, 1, wl.H, dtype=torch.float32, device=dev) for _ in range(4)]
    bufs = [torch.empty(wl.B, 1, wl.k, dtype=torch.int32, device=dev)]

    def draft():
        dsa.indexshare_draft_forward(layers[0]["ix"], at, wl.k, out=out, lse=lse, idx=idx)

    def walk():
        dsa.indexshare_group_forward(group, "FSSS", wl.k, outs=outs, lses=lses, idx_bufs=bufs)

    for _ in range(3):
        draft()
        walk()
    torch.cuda.synchronize()
    dsa.trace_enable(64 * steps + 64)
    d_ms = time_loop(draft, steps, 0, world)
    trace = dsa.trace_read()
    dsa.trace_disable()
    g_ms = time_loop(walk, steps, 0, world)
    by_kind = {}
    for kind, t in trace:
        by_kind[kind] = by_kind.get(kind, 0.0) + t / steps
    ent = {"draft_ms": round(d_ms, 3), "group_ms": round(g_ms, 3), "draft_vs_group": round(g_ms / d_ms, 3),
           "draft_kernel_ms": {k: round(v, 3) for k, v in sorted(by_kind.items())},
           "tokens_per_s": round(wl.B * 4 * world / (d_ms / 1e3), 1)}
    del layers, group, at, out, lse, idx, outs, lses, bufs
    torch.cuda.empty_cache()
    return ent


def _indexer_kernel_line(wl, by_kind, steps, fp8_tf):
    """The FP8 indexer kernel inside the timed steps: its device time per F layer (the launch
    tracer's events), its algorithmic flops per second and the fraction of the measured FP8
    tensor peak."""
    if not by_kind.get("indexer"):
        return None
    ms = float(np.sum(by_kind["indexer"])) / steps
    tf = indexer_flops(wl) / (ms / 1e3) / 1e12
    return {"ms_per_f_layer": round(ms, 3), "tflops": round(tf, 1), "frac_of_measured_fp8": round(tf / fp8_tf, 4),
            "launches_per_step": len(by_kind["indexer"]) // steps}


def run_e2e(dsa, wl, layers, group, outs, lses, bufs, args, world):
    """The same F,S,S,S group through the public calls, with every input copied in from pinned
    host memory and every output copied back inside the timed region.  The layers consume
    their inputs in order, so the copies are pipelined against the compute: each layer's
    inputs go in on a copy stream ahead of its attention call and each layer's output goes
    back on a second copy stream as soon as it is written.  Alternate steps use two sets of
    device input and output buffers, so one step's copies also overlap its neighbours'
    compute (the next step's inputs stream in while this one computes; its outputs drain
    while the next one computes).  A step ends when its last output is on the host.  The
    calls are the ones indexshare_group_forward makes (the F layer's top-k from indexer
    operands, then one attention call per layer over its index buffer)."""
    ix = layers[0]["ix"]
    ix_keys = ["q", "k", "w", "q_scale", "k_scale"]
    # each distinct device tensor goes in once, before the first layer that reads it (the
    # draft steps of a multi-token-prediction layer share one cache)
    seen = {ix["k"].data_ptr()}
    at_dev = []
    for g in group:
        at_dev.append([t for t in (g["at"]["q"], g["at"]["k"]) if t.data_ptr() not in seen])
        seen.update(t.data_ptr() for t in at_dev[-1])
    ix_dev = [ix[key] for key in ix_keys]

    # the second set of device buffers: every copied tensor and every output, cloned
    twin = {}
    for t in ix_dev + [t for ts in at_dev for t in ts]:
        twin.setdefault(t.data_ptr(), torch.empty_like(t))
    swap = lambda t: twin.get(t.data_ptr(), t) if torch.is_tensor(t) else t
    sets = [dict(ix=ix, ix_dev=ix_dev, at=[g["at"] for g in group], at_dev=at_dev, outs=outs, lses=lses)]
    sets.append(dict(ix={key: swap(v) for key, v in ix.items()}, ix_dev=[swap(t) for t in ix_dev],
                     at=[{key: swap(v) for key, v in g["at"].items()} for g in group],
                     at_dev=[[swap(t) for t in ts] for ts in at_dev],
                     outs=[torch.empty_like(o) for o in outs], lses=[torch.empty_like(x) for x in lses]))

    # page-locked host buffers of exactly the tensors' sizes, allocated by the CUDA driver
    # (cuMemHostAlloc); torch's caching pinned allocator would round each one up to a power of
    # two (131 GB locked instead of 75 GB).  Registering malloc'd pages in place instead
    # (cudaHostRegister) was measured too: host-to-device copies from them fell to 20 GB/s.
    pinned = HostPinned()

    def host_like(t, fill):
        h = pinned.empty(t.shape, t.dtype)
        return h.copy_(t) if fill else h

    ix_host = [host_like(t, True) for t in ix_dev]
    at_host = [[host_like(t, True) for t in ts] for ts in at_dev]
    out_host = [[host_like(outs[l], False), host_like(lses[l], False)] for l in range(4)]
    h2d = sum(t.numel() * t.element_size() for t in ix_host) + sum(t.numel() * t.element_size() for ts in at_host for t in ts)
    d2h = sum(t.numel() * t.element_size() for ts in out_host for t in ts)
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()

    # the last layer runs in row chunks so that only its last chunk's copy-back trails the compute
    nchunk = 4 if wl.T % 4 == 0 else 1
    rc = wl.T // nchunk
    computed = [None, None]   # per set: the compute of the last step that used it
    drained = [None, None]    # per set: the copy-back of the last step that used it

    def step(i):
        S = sets[i % 2]
        if computed[i % 2] is not None:
            cin.wait_event(computed[i % 2])  # that step no longer reads these input buffers
        ready = []
        with torch.cuda.stream(cin):
            for h, d in zip(ix_host, S["ix_dev"]):
                d.copy_(h, non_blocking=True)
            ready_ix = torch.cuda.Event()
            ready_ix.record(cin)
            for l in range(4):
                for h, d in zip(at_host[l], S["at_dev"][l]):
                    d.copy_(h, non_blocking=True)
                ready.append(torch.cuda.Event())
                ready[-1].record(cin)
        comp.wait_event(ready_ix)  # the F layer's indexer starts while the attention inputs stream in
        dsa.dsa_topk(wl.k, ix=S["ix"], idx=bufs[0])
        if drained[i % 2] is not None:
            comp.wait_event(drained[i % 2])  # that step's outputs have left these buffers
        for l in range(4):
            comp.wait_event(ready[l])
            parts = [(0, wl.T)] if l < 3 else [(c * rc, (c + 1) * rc) for c in range(nchunk)]
            for r0, r1 in parts:
                at = S["at"][l]
                if (r0, r1) != (0, wl.T):
                    at = dict(at, q=at["q"][:, r0:r1])
                o, x = S["outs"][l], S["lses"][l]
                dsa.dsa_sparse_attn(at, bufs[0][:, r0:r1], out=o[:, r0:r1], lse=x[:, r0:r1])
                done = torch.cuda.Event()
                done.record(comp)
                cout.wait_event(done)
                with torch.cuda.stream(cout):
                    for h, d in zip(out_host[l], (o, x)):
                        h[:, r0:r1].copy_(d[:, r0:r1], non_blocking=True)
        computed[i % 2] = torch.cuda.Event()
        computed[i % 2].record(comp)
        drained[i % 2] = torch.cuda.Event(enable_timing=True)
        drained[i % 2].record(cout)
        return drained[i % 2]

    link0 = host_copy_gbs(at_host[0][0], at_dev[0][0], out_host[0][0], outs[0], cin, cout)
    # two warm-up steps (both buffer sets), then timed steps; a step's end is the event after
    # its last copy-back, so consecutive ends bound single steps of the running pipeline
    steps = max(3, args.steps // 2)
    step(0)
    step(1)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    cin.wait_stream(comp)
    cout.wait_stream(comp)
    ends = [step(i) for i in range(steps)]
    comp.wait_stream(cout)
    comp.wait_stream(cin)
    e1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    per_step = [e0.elapsed_time(ends[0])] + [ends[i - 1].elapsed_time(ends[i]) for i in range(1, steps)]
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    link1 = host_copy_gbs(at_host[0][0], at_dev[0][0], out_host[0][0], outs[0], cin, cout)
    torch.cuda.synchronize()
    del ix_host, at_host, out_host, sets, twin
    host_alloc = pinned.kind
    pinned.free()
    return {"value": round(wl.B * wl.T * world / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "overlap": "per-layer inputs in and outputs out on two copy streams, pipelined against compute; "
                       "alternate steps on two device buffer sets",
            "step_ms": [round(x, 1) for x in per_step], "host_alloc": host_alloc,
            "host_copy_gbs": {"before": link0, "after": link1},
            "copy_bound_ms": round((h2d + d2h) / (min(link0["both"], link1["both"]) * 1e9) * 1e3, 1)}


class HostPinned:
    """Page-locked host tensors of exact size from the CUDA driver (cuMemHostAlloc in the
    current context), or torch's pinned allocator when the driver call is unavailable."""

    def __init__(self):
        import ctypes
        self._ct = ctypes
        self._ptrs = []
        self.kind = "cuMemHostAlloc"
        try:
            self._cuda = ctypes.CDLL("libcuda.so.1")
            self._cuda.cuMemHostAlloc.restype = ctypes.c_int
            self._cuda.cuMemHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
            self._cuda.cuMemFreeHost.restype = ctypes.c_int
            self._cuda.cuMemFreeHost.argtypes = [ctypes.c_void_p]
        except OSError:
            self._cuda, self.kind = None, "torch pinned"

    def empty(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        if self._cuda is not None and n > 0:
            p = self._ct.c_void_p()
            if self._cuda.cuMemHostAlloc(self._ct.byref(p), n, 0) == 0:
                self._ptrs.append(p.value)
                buf = (self._ct.c_uint8 * n).from_address(p.value)
                return torch.frombuffer(buf, dtype=torch.uint8).view(dtype).view(shape)
            self.kind = "torch pinned"
        return torch.empty(shape, dtype=dtype, pin_memory=True)

    def free(self):
        torch.cuda.synchronize()
        for p in self._ptrs:
            self._cuda.cuMemFreeHost(p)
        self._ptrs = []


def host_copy_gbs(h_in, d_in, h_out, d_out, cin, cout, nbytes=1 << 30, reps=3):
    """Pinned host <-> device copy rates of this machine (GB/s, median of reps): in alone, out
    alone, and both directions at once on the two copy streams the end-to-end step uses.  The
    host link differs between machines, and it bounds the end-to-end step from below."""
    hi, di = h_in.view(-1)[:nbytes // h_in.element_size()], d_in.view(-1)[:nbytes // h_in.element_size()]
    ho, do = h_out.view(-1)[:nbytes // h_out.element_size()], d_out.view(-1)[:nbytes // h_out.element_size()]
    b_in, b_out = hi.numel() * hi.element_size(), ho.numel() * ho.element_size()
    comp = torch.cuda.current_stream()
    res = {}
    for name in ("h2d", "d2h", "both"):
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(comp)
            cin.wait_stream(comp)
            cout.wait_stream(comp)
            for st, go, dst, src in ((cin, name != "d2h", di, hi), (cout, name != "h2d", ho, do)):
                if go:
                    with torch.cuda.stream(st):
                        dst.copy_(src, non_blocking=True)
            comp.wait_stream(cin)
            comp.wait_stream(cout)
            e1.record(comp)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3)
        moved = (b_in if name != "d2h" else 0) + (b_out if name != "h2d" else 0)
        res[name] = round(moved / sorted(ts)[len(ts) // 2] / 1e9, 1)
    return res


# --- reference arm: the CPU oracle -------------------------------------------------------

def run_reference(args, rank, world, local):
    import oracle
    oracle.build()
    wl = synth.WORKLOADS[args.workload]
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    # one sampled row per oracle thread (rows are the oracle's unit of parallel work)
    rows = pick_rows(wl, max(1, oracle.num_threads() - 1), seed=3)
    # inputs: the same seeded tensors; only what the sampled rows read is moved to the host
    ix = synth.indexer_inputs(wl, 0, dev)
    hix, _ = host_sample(wl, ix, [], rows)
    del ix
    hats = []
    for l in range(4):
        at = synth.attn_inputs(wl, l, dev)
        hats += host_sample(wl, dict(q=at["q"], w=at["q"], k=at["k"]), [at], rows)[1]
        del at
    if dev.type == "cuda":
        torch.cuda.empty_cache()

    def step():
        a, b = oracle_sample(wl, hix, hats, rows, wl.k)
        return extrapolate(wl, rows, a, b)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    tot = [step() for _ in range(args.steps)]
    wall = (time.perf_counter() - t0) / args.steps
    ext = float(np.mean([a + b for a, b in tot]))
    value = wl.B * wl.T / ext
    cores = oracle.num_threads()
    sample = f"{len(rows)} query rows of {wl.name} per step (indexer+top-k and 4 attention layers), " \
             f"extrapolated by visible-key and selected-key counts"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ext * 1e3, 1),
            "sample_wall_ms_per_step": round(wall * 1e3, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "L": wl.S, "query_rows": wl.B * wl.T, "k": wl.k, "schedule": GROUP},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_kernel_case(args):
    """One public call on a synthetic single-kernel case: the last `rows` query rows of a
    `keys`-token sequence.  attn: sparse MLA attention (k=2048) over index rows from a top-k
    of Gaussian scores; indexer: FP8 materialised indexer scores; topk: top-2048 over those
    scores (computed once, outside the timed call); ixtopk: FP8 indexer + top-k; quant: e4m3
    quantisation of `rows` query tokens of the indexer (64 heads x 128 dims, one scale per
    token) into a cache."""
    import long_context_sparse_tcgen05_gb300 as dsa
    from long_context_sparse_tcgen05_gb300 import build
    build.build()
    dsa.load_library()
    dev = torch.device("cuda:0")
    T, S = args.rows, args.keys
    if args.kernel == "quant":
        width = 64 * 128
        g = torch.Generator(device=dev)
        g.manual_seed(synth.SEED_BASE + 17)
        x = torch.randn((1, T, width), generator=g, device=dev).to(torch.bfloat16)
        codes = torch.empty((1, T, width), dtype=torch.uint8, device=dev)
        scales = torch.empty((1, T), dtype=torch.float32, device=dev)
        fn = lambda: dsa.dsa_quantize_e4m3_append(x, codes, scales)
        work = f"{T * (3 * width + 4) / 1e9:.3f} GB moved"
    elif args.kernel == "attn":
        wl = synth.WORKLOADS["prefill_16k"].replace(T=T, S=S, q_pos0=S - T)
        at = synth.attn_inputs(wl, 0, dev)
        sc = synth.scores_input(T, S, dev, "normal", seed=5)
        idx = dsa.dsa_topk(2048, scores=sc[None], q_pos0=S - T)
        del sc
        out = torch.empty(1, T, 64, 512, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(1, T, 64, dtype=torch.float32, device=dev)
        fn = lambda: dsa.dsa_sparse_attn(at, idx, out=out, lse=lse)
        work = f"{T * 2048 * 1152 / 1e9:.2f} GB gathered"
    else:
        wl = synth.WORKLOADS["prefill_128k"].replace(T=T, S=S, q_pos0=S - T, values="gauss")
        ix = synth.indexer_inputs(wl, 0, dev)
        flops = sum(min(S, S - T + t) for t in range(T)) * 2 * 64 * 128
        work = f"{flops / 1e12:.2f} TFLOP"
        if args.kernel in ("indexer", "topk"):
            out = torch.empty(1, T, S, dtype=torch.float32, device=dev)
            fn = lambda: dsa.indexer_scores(ix, out=out)
            if args.kernel == "topk":
                fn()
                idx = torch.empty(1, T, 2048, dtype=torch.int32, device=dev)
                fn = lambda: dsa.dsa_topk(2048, scores=out, q_pos0=S - T, diag=wl.diag, idx=idx)
                work = f"{sum(min(S, S - T + t + wl.diag) for t in range(T)) * 4 / 1e9:.2f} GB of scores read"
        else:
            fn = lambda: dsa.dsa_topk(2048, ix=ix)
    torch.cuda.synchronize()
    times = []
    for r in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
        print(json.dumps({"kernel_case": args.kernel, "rows": T, "keys": S, "rep": r,
                          "ms": round(times[-1], 4), "work": work}))
    if args.kernel == "quant" and len(times) > 1:
        # HBM roofline of the warm launches, and the oracle's quantiser on a sample beside it
        import oracle
        ms = statistics.median(times[1:])
        nbytes = T * (3 * width + 4)
        peaks = load_peaks()
        sample = min(T, 256)
        xs = x[0, :sample].cpu()
        t0 = time.perf_counter()
        oracle.quantize_e4m3_rows(xs, width)
        cpu_s = time.perf_counter() - t0
        print(json.dumps({"kernel_case": "quant", "tokens_per_s": round(T / (ms * 1e-3), 1), "ms": round(ms, 4),
                          "roofline": {"bound": "hbm", "achieved": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                       "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                       "frac": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                       "peak_src": peaks["src"]},
                          "cpu_baseline": {"value": round(sample / cpu_s, 1), "unit": "tokens/s", "cores": 1,
                                           "kind": "oracle", "sample": f"{sample} tokens of {width} values"}}))
    print(json.dumps({"device_flags": dsa.read_device_flags(dev)}))


def run_heatmap(args):
    """The layer-overlap heatmap of an all-F pass and the schedules it suggests.  Every layer
    of heatmap_128k runs its own indexer + top-k (dsa_topk), topk_overlap_matrix gives the mean
    overlap of every pair of layers, indexshare_schedule_search the best schedule for each
    number of full layers, and indexshare_group_forward times the uniform F,S,S,S x 4 schedule
    against the best one with as many full layers.  The layers' attention operands are one
    shared set (attention time does not depend on which rows are selected), so the group times
    hold 16 layers of attention without 16 copies of Q and the latent KV."""
    import long_context_sparse_tcgen05_gb300 as dsa
    from long_context_sparse_tcgen05_gb300 import build
    build.build()
    dsa.load_library()
    dev = torch.device("cuda:0")
    wl = synth.WORKLOADS["heatmap_128k"]
    if args.keys != wl.S:
        wl = wl.replace(T=args.keys, S=args.keys)
    n, T, k = wl.n_layers, wl.B * wl.T, wl.k

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    # all-F pass: one indexer + top-k per layer, each into its own index buffer
    bufs = [torch.empty((wl.B, wl.T, k), dtype=torch.int32, device=dev) for _ in range(n)]
    f_ms = []
    for l in range(n):
        ix = synth.indexer_inputs(wl, l, dev)
        if l == 0:
            dsa.dsa_topk(k, ix=ix, idx=bufs[0])  # warm-up
        f_ms.append(timed(lambda: dsa.dsa_topk(k, ix=ix, idx=bufs[l])))
        del ix
    torch.cuda.empty_cache()

    # the overlap matrix, timed by the launch tracer (its kernels on the current stream)
    M, _ = dsa.topk_overlap_matrix(bufs)
    dsa.trace_enable(64)
    for _ in range(3):
        M, _ = dsa.topk_overlap_matrix(bufs)
    m_ms = statistics.median(ms for kind, ms in dsa.trace_read() if kind == "overlap")
    dsa.trace_disable()
    idx_bytes = n * T * k * 4

    # attention time of one layer, then the schedules
    at = synth.attn_inputs(wl, 0, dev)
    out = torch.empty((wl.B, wl.T, wl.H, wl.DV), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.B, wl.T, wl.H), dtype=torch.float32, device=dev)
    dsa.dsa_sparse_attn(at, bufs[0], out=out, lse=lse)
    a_ms = timed(lambda: dsa.dsa_sparse_attn(at, bufs[0], out=out, lse=lse))
    t_f = statistics.mean(f_ms)
    schedules = []
    for m in range(1, n + 1):
        sched, score = dsa.indexshare_schedule_search(M, m)
        schedules.append({"n_full": m, "schedule": sched, "score": round(score, 4),
                          "model_ms": round(m * t_f + n * a_ms, 1)})
    uniform = "FSSS" * (n // 4)
    best = schedules[uniform.count("F") - 1]["schedule"]
    bufs_keep = [b.reshape(T, k)[torch.linspace(0, T - 1, min(T, 512)).long().to(dev)].clone() for b in bufs]
    del bufs
    torch.cuda.empty_cache()

    def group_ms(sched):
        layers = [dict(ix=synth.indexer_inputs(wl, l, dev) if sched[l] == "F" else None, at=at)
                  for l in range(n)]
        run = lambda: dsa.indexshare_group_forward(layers, sched, k, outs=[out] * n, lses=[lse] * n)
        run()
        ms = statistics.median(timed(run) for _ in range(2))
        del layers
        torch.cuda.empty_cache()
        return round(ms, 1)

    groups = {s: group_ms(s) for s in dict.fromkeys([uniform, best, "F" * n])}
    # the oracle's all-pairs overlap on a row sample beside the kernel
    import oracle
    sample = min(T, 512)
    host = [b.cpu().numpy() for b in bufs_keep]
    t0 = time.perf_counter()
    oracle.overlap_matrix(host)
    cpu_s = time.perf_counter() - t0
    del bufs_keep
    peaks = load_peaks()
    line = {
        "workload": wl.name, "L": wl.S, "query_rows": T, "k": k, "layers": n,
        "clusters": list(wl.clusters), "cluster_share": synth.CLUSTER_SHARE,
        "heatmap": [[round(v, 4) for v in row] for row in M],
        "adjacent_overlap": [round(M[l][l + 1], 4) for l in range(n - 1)],
        "indexer_topk_ms_per_layer": round(t_f, 2), "attention_ms_per_layer": round(a_ms, 2),
        "overlap_matrix": {"ms": round(m_ms, 3), "idx_bytes": idx_bytes,
                           "gbs": round(idx_bytes / (m_ms * 1e-3) / 1e9, 1),
                           "rows_per_s": round(T / (m_ms * 1e-3), 1),
                           "roofline": {"bound": "hbm", "achieved": round(idx_bytes / (m_ms * 1e-3) / 1e9, 1),
                                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                        "frac": round(idx_bytes / (m_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                        "note": "HBM floor; the kernel is bound by shared-memory issue"},
                           "cpu_baseline": {"value": round(sample / cpu_s, 1), "unit": "rows/s",
                                            "cores": oracle.num_threads(), "kind": "oracle",
                                            "sample": f"{sample} rows of the {n} buffers, every ordered pair"}},
        "schedules": schedules,
        "measured_group_ms": {s: groups[s] for s in groups},
        "uniform": {"schedule": uniform, "score": round(dsa.indexshare_schedule_score(M, uniform), 4)},
        "device_flags": dsa.read_device_flags(dev),
    }
    print(json.dumps(line), flush=True)


def run_varlen(args):
    """Packed prompts of different lengths through one indexshare_group_forward_varlen call:
    eight prefills of 64K, 32K, 16K, 8K, 8K, 4K, 2K and 1K tokens with the 128K workload's
    operands (FP8 indexer, top-2,048, 64-head MLA), against one indexshare_group_forward call
    per prompt."""
    import long_context_sparse_tcgen05_gb300 as dsa
    from long_context_sparse_tcgen05_gb300 import build
    build.build()
    dsa.load_library()
    dev = torch.device("cuda:0")
    lens = [65536, 32768, 16384, 8192, 8192, 4096, 2048, 1024]
    base = synth.WORKLOADS["prefill_128k"]
    wls = [base.replace(T=n, S=n, q_pos0=0, wid=30 + i) for i, n in enumerate(lens)]
    per_seq = [synth.group_inputs(wl, 4, dev) for wl in wls]
    packed = []
    for l in range(4):
        at = dict(per_seq[0][l]["at"])
        at["q"] = torch.cat([p[l]["at"]["q"] for p in per_seq], dim=1)
        at["k"] = torch.cat([p[l]["at"]["k"] for p in per_seq], dim=1)
        ix = None
        if GROUP[l] == "F":
            ix = dict(per_seq[0][l]["ix"])
            for key in ("q", "w", "q_scale", "k", "k_scale"):
                ix[key] = torch.cat([p[l]["ix"][key] for p in per_seq], dim=1)
        packed.append(dict(ix=ix, at=at))
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    q0 = [0] * len(lens)
    packed_run = lambda: dsa.indexshare_group_forward_varlen(packed, GROUP, base.k, cu, cu, q0)
    outs = [dsa.indexshare_group_forward(p, GROUP, base.k) for p in per_seq]  # buffers for the loop
    loop_run = lambda: [dsa.indexshare_group_forward(p, GROUP, base.k, outs=o[0], lses=o[1], idx_bufs=o[2])
                        for p, o in zip(per_seq, outs)]
    t_packed = time_loop(packed_run, args.steps, max(3, args.warmup))
    t_loop = time_loop(loop_run, args.steps, max(3, args.warmup))
    tokens = sum(lens)
    print(json.dumps({"varlen": {"lengths": lens, "tokens": tokens, "schedule": GROUP,
                                 "packed_ms": round(t_packed, 3), "packed_tokens_per_s": round(tokens / t_packed * 1e3, 1),
                                 "one_call_per_prompt_ms": round(t_loop, 3),
                                 "device_flags": dsa.read_device_flags(dev)}}), flush=True)


def main():
    args = parse()
    if args.kernel:
        run_kernel_case(args)
        return
    if args.peaks:
        print(json.dumps(fp8_peak(torch.device("cuda:0"))), flush=True)
        return
    if args.heatmap:
        run_heatmap(args)
        return
    if args.varlen:
        run_varlen(args)
        return
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank != 0:
            return
        line = run_reference(args, rank, world, local)
        line["n_gpus"] = world
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
