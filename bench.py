#!/usr/bin/env python3
"""Benchmark of one paged gated-MLA decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl plmla|reference]
                    [--workload long|steady|agentic|spec|extend|tiny] [--kv bf16|fp8]

A step is one pass of the whole hot path (split plan -> split decode -> LSE
combine + sigmoid gate) for every MLA layer of the workload.  The default is
the largest single-GPU workload: 4 requests x 1 query token at 1,000,000-token
histories, 64 heads, 576-wide bf16 latent rows (512 latent + 64 rope), 24 MLA
layer slabs sharing one page table of 652 scattered 1,536-token pages per
request, at least 128 KV splits per request (seed 4); all 24 layers are decoded
in turn.  The metric is achieved HBM bandwidth on the KV bytes a step must read
(sum of histories x 1,152 bytes x layers), also given as request-steps/s.

Prints ONE JSON line on rank 0.  Multi-GPU runs (torchrun, one rank per GPU)
are weak-scaling replicas: every rank decodes its own copy of the workload, no
data moves between GPUs, and the value is the total over ranks divided by the
slowest rank's time.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged MLA decode: achieved HBM GB/s (% of GB300 peak), request-steps/s"
UNIT = "GB/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
KV_SCALE_FP8 = 6.0 / 448.0    # the synthetic FP8 cache's scale
DECODE_SOURCES = ["plmla_decode_tc.cu", "plmla_internal.cuh"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["plmla", "reference"], default="plmla")
    ap.add_argument("--op", choices=["decode", "append", "dcp"], default="decode",
                    help="decode: the hot path (default); append: the KV append kernel "
                         "writing a block of new rows per request into the same pool; dcp: "
                         "decode context parallelism's device work (shard, each rank's "
                         "decode, merge) for one layer, the ranks run one after another")
    ap.add_argument("--dcp-world", type=int, default=4,
                    help="ranks of the decode context parallelism group for --op dcp")
    ap.add_argument("--append-tokens", type=int, default=4096,
                    help="new tokens per request for --op append")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="cache format: bf16 pages (the default workload) or E4M3 pages "
                         "(the deployment's FP8 cache, 576 bytes per token row)")
    ap.add_argument("--workload", default="long",
                    choices=["tiny", "steady", "agentic", "spec", "long", "extend"])
    ap.add_argument("--split", choices=["per-request", "uniform"], default="per-request",
                    help="split rule of the planner: per-request split counts (the library's "
                         "default) or the uniform baseline the pages compare it with")
    ap.add_argument("--control", action="store_true",
                    help="the workload's equal-length control: same requests and total KV "
                         "tokens, every history at the average length")
    ap.add_argument("--layers", type=int, default=None,
                    help="decode only the first N layer slabs of a multi-layer workload: a "
                         "smaller case of the same per-layer launch for ncu captures (each "
                         "layer's launch is the same work on its own slab); the line then "
                         "names N layers and is not the workload's measurement")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time plain back-to-back calls instead of replays of a captured step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# distributed plumbing (weak-scaling replicas; the only collectives are the
# barrier and the max/sum of timing scalars)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate(dist, local_ms, local_units, device="cpu"):
    """(max time over ranks, total units over ranks)."""
    if dist is None:
        return local_ms, local_units
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed region"
        if len(inside) < 2:
            # a short timed region: widen to the surrounding busy period
            inside = [p for (t, p) in self.samples if t0 - 2.0 <= t <= t1 + 2.0]
            window = "timed region +/- 2 s"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower() == "active"})
        power = [num(p[3]) for p in inside if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside), "window": window,
                "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------
# peaks and profile-derived traffic
# --------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s): the burst figure, for a kernel timed in
    a short step."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def decode_source_hash():
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "paged_latent_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kv_bytes, fp8=False):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source; else None."""
    name = f"decode_{workload}_fp8_traffic.json" if fp8 else f"decode_{workload}_traffic.json"
    path = os.path.join(ROOT, "profiles", name)
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("decode_source_hash") != decode_source_hash():
        return None
    per_unit = rec.get("dram_bytes_per_kv_byte")
    return None if per_unit is None else per_unit * kv_bytes


# --------------------------------------------------------------------------
# CPU oracle baseline (a bounded sample of the same workload)
# --------------------------------------------------------------------------

def oracle_sample(w, qn, qr, gate, slab_dev, req_ids):
    """Host inputs for the oracle restricted to `req_ids` (pages remapped)."""
    import numpy as np
    import torch
    pages_per_req = [-(-int(w.seq_lens[r]) // w.page_tokens) for r in req_ids]
    phys = [int(p) for r, n in zip(req_ids, pages_per_req) for p in w.page_table[r, :n]]
    idx = torch.as_tensor(phys, dtype=torch.long, device=slab_dev.device)
    host_slab = slab_dev.index_select(0, idx).cpu()
    table = np.zeros((len(req_ids), max(1, max(pages_per_req))), dtype=np.int32)
    pos = 0
    for i, n in enumerate(pages_per_req):
        table[i, :n] = np.arange(pos, pos + n)
        pos += n
    rows_q = torch.cat([torch.arange(r * w.n_q, (r + 1) * w.n_q) for r in req_ids])
    lens = w.seq_lens[list(req_ids)].astype(np.int32)
    return (qn[rows_q].cpu(), qr[rows_q].cpu(), gate[rows_q].cpu(), host_slab, table, lens,
            len(phys))


def row_sample(w, n_reqs):
    """Output rows the oracle computes for a sample of n_reqs requests, and the
    fraction of the requests' rows they are.  Workloads with many query rows per
    request (a chunked extend) take the first, middle and last new token, four
    heads each; the others take every row."""
    rows_per_req = w.n_q * w.num_heads
    if rows_per_req <= 256:
        return None, 1.0
    toks = sorted({0, w.n_q // 2, w.n_q - 1})
    heads = range(min(4, w.num_heads))
    rows = [(i * w.n_q + j) * w.num_heads + h for i in range(n_reqs) for j in toks for h in heads]
    return rows, len(toks) * len(heads) / rows_per_req


def run_oracle(w, sample, kv_scale=None, rows=None):
    import oracle
    qn, qr, gate, slab, table, lens, npages = sample
    t = time.perf_counter()
    if kv_scale is None:
        oracle.mla_decode_reference(qn, qr, gate, slab, table, lens, w.n_q, w.num_heads,
                                    1.0 / math.sqrt(192.0), num_pages=npages,
                                    page_stride=w.page_stride, rows=rows)
    else:
        oracle.mla_decode_e4m3_reference(qn, qr, gate, slab, kv_scale, table, lens, w.n_q,
                                         w.num_heads, 1.0 / math.sqrt(192.0), num_pages=npages,
                                         page_stride=w.page_stride, rows=rows)
    return time.perf_counter() - t


def kv_row_bytes(w, fp8):
    return (w.dc + w.dr) * (1 if fp8 else 2)


def cpu_baseline(w, qn, qr, gate, slab_dev, target_s, kv_scale=None):
    import oracle
    cores = oracle.oracle.default_threads()
    order = list(range(w.num_reqs))
    one = oracle_sample(w, qn, qr, gate, slab_dev, order[:1])
    t1 = run_oracle(w, one, kv_scale, row_sample(w, 1)[0])
    n = max(1, min(w.num_reqs, int(target_s / max(t1, 1e-3))))
    sample = oracle_sample(w, qn, qr, gate, slab_dev, order[:n])
    rows, frac = row_sample(w, n)
    elapsed, reps = 0.0, 0
    while elapsed < 0.5 * target_s or reps == 0:
        elapsed += run_oracle(w, sample, kv_scale, rows)
        reps += 1
    # KV bytes credited in proportion to the rows computed
    kv = int(sum(int(w.seq_lens[r]) for r in order[:n])) * kv_row_bytes(w, kv_scale is not None)
    gbs = frac * kv * reps / elapsed / 1e9
    what = ("all {} heads".format(w.num_heads) if rows is None else
            f"{frac:.4f} of the rows (first, middle and last new token, 4 heads)")
    layer = (f" of layer 0 (of {w.num_slabs}; every layer is the same work, so the rate "
             f"is the step's)" if w.num_slabs > 1 else "")
    return {"value": gbs, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.num_reqs} requests x {what}{layer}, {reps} pass(es), "
                      f"{elapsed:.1f} s of double-precision oracle time, KV bytes credited "
                      f"in proportion to the rows",
            "request_steps_per_s": frac * n * reps / elapsed}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def workload_description(w, fp8=False):
    lens = w.seq_lens
    fmt = (f"E4M3 (FP8 cache, kv_scale {KV_SCALE_FP8:.6g})" if fp8 else "bf16")
    return (f"{w.name} decode: {w.num_reqs} requests x {w.n_q} query token(s), {w.num_heads} "
            f"heads, 512 latent + 64 rope {fmt}, histories {int(lens.min())}..{int(lens.max())} "
            f"tokens (sum {int(lens.sum())}), {w.num_pages} pages of 1536 tokens, "
            f"{w.num_slabs} slab(s), seed {w.seed}")


def run_gpu(args):
    import torch
    import paged_latent_attention_gb300 as plmla
    from paged_latent_attention_gb300 import inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, "nccl")

    w = inputs.make_workload(args.workload)
    if args.control:
        w = inputs.equal_length_control(w)
    plmla.set_split_mode(args.split)
    if args.layers is not None:
        if not 1 <= args.layers <= w.num_slabs:
            raise SystemExit(f"--layers must lie in [1, {w.num_slabs}]")
        w.num_slabs = args.layers
    fp8 = args.kv == "fp8"
    layers = w.num_slabs
    qs = [inputs.make_queries(w, device, layer=l) for l in range(layers)]
    if fp8:
        slabs = [inputs.make_slab_e4m3(w, device, layer=l, kv_scale=KV_SCALE_FP8)
                 for l in range(layers)]
    else:
        slabs = [inputs.make_slab(w, device, layer=l) for l in range(layers)]
    table = torch.as_tensor(w.page_table, device=device)
    lens = torch.as_tensor(w.seq_lens, device=device)
    ws = plmla.allocate_workspace(w.num_reqs, w.n_q, w.num_heads, 0, w.min_splits, device,
                                  fp8=fp8)
    outs = [torch.empty_like(q[0]) for q in qs]
    lses = [torch.empty(w.num_tokens, w.num_heads, dtype=torch.float32, device=device)
            for _ in qs]
    kv_bytes_layer = w.kv_tokens * kv_row_bytes(w, fp8)
    kv_bytes_step = kv_bytes_layer * layers
    decode = decoder(plmla, fp8)
    decode_layers = layers_decoder(plmla, fp8)

    K, W = args.steps, args.warmup
    n_ev = K * layers
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_ev)]
    stream = torch.cuda.current_stream(device)
    for quad in evs:           # create every event handle before the timed region
        for e in quad:
            e.record(stream)

    def call_step(q_layers, tbl, ln, out_layers, lse_layers):
        # the user's call for a step of every layer: one split plan, then each
        # layer's split decode and combine (one layer: the plain decode call)
        if layers == 1:
            decode(*q_layers[0], slabs[0], tbl, ln, n_q=w.n_q, out=out_layers[0],
                   lse=lse_layers[0], workspace=ws, min_splits=w.min_splits)
        else:
            decode_layers([q[0] for q in q_layers], [q[1] for q in q_layers],
                          [q[2] for q in q_layers], slabs, tbl, ln, n_q=w.n_q, out=out_layers,
                          lse=lse_layers, workspace=ws, min_splits=w.min_splits)

    def step():
        call_step(qs, table, lens, outs, lses)

    def step_staged(ev_base):
        # per-layer calls with events between the kernels (plan, decode, combine)
        for l in range(layers):
            qn, qr, gate = qs[l]
            decode(qn, qr, gate, slabs[l], table, lens, n_q=w.n_q, out=outs[l],
                   lse=lses[l], workspace=ws, min_splits=w.min_splits,
                   events=evs[ev_base + l])

    for _ in range(W):
        step()
        step_staged(0)
    torch.cuda.synchronize(device)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    # timed region 1 (the reported value): K steps of the user's step call,
    # captured in a CUDA graph and replayed (as a decode loop runs it: no host
    # work per step), or with --no-graph the plain calls back to back; plan,
    # decodes and combines overlap through programmatic launch either way
    def run_steps():
        for _ in range(K):
            step()
    if not args.no_graph:
        # all K steps in one graph, so that each step's plan still overlaps the
        # previous step's combine (programmatic edges inside the graph); captured
        # and replayed once before the timed region
        graph = torch.cuda.CUDAGraph()
        # thread-local capture: other threads (a process group's) may use CUDA meanwhile
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            run_steps()
        graph.replay()
        torch.cuda.synchronize(device)
        run_steps = graph.replay
    sampler = ClockSampler(uuid).start()
    time.sleep(0.3)
    barrier(dist, device)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    host_t0 = time.time()
    start.record(stream)
    run_steps()
    end.record(stream)
    torch.cuda.synchronize(device)
    # timed region 2 (per-kernel durations for the roofline): the same K steps as
    # per-layer calls with stage events recorded between the kernels, which
    # serialises them
    start2, end2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start2.record(stream)
    for k in range(K):
        step_staged(k * layers)
    end2.record(stream)
    torch.cuda.synchronize(device)
    host_t1 = time.time()
    barrier(dist, device)
    local_ms = start.elapsed_time(end)
    staged_ms = start2.elapsed_time(end2)
    decode_ms = [q[1].elapsed_time(q[2]) for q in evs]
    plan_ms = [q[0].elapsed_time(q[1]) for q in evs]
    combine_ms = [q[2].elapsed_time(q[3]) for q in evs]
    max_ms, total_units = aggregate(dist, local_ms, kv_bytes_step * K, device)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, qs, table, lens, device, dist, call_step, kv_bytes_layer)
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(host_t0, host_t1)

    if rank != 0:
        return None
    ms_per_step = max_ms / K
    value = total_units / (max_ms / 1e3) / 1e9
    peak, peak_src = hbm_peak()
    dec_avg = statistics.mean(decode_ms)
    achieved = kv_bytes_layer / (dec_avg / 1e3) / 1e9
    traffic = profiled_traffic(args.workload, kv_bytes_layer, fp8)
    # Which roofline bounds the decode: 2 * (576 + 512) flop per (query row, KV
    # token) against 1,152 bytes per KV token, compared with the measured ridge.
    tpeak, tpeak_src = tensor_peak()
    if fp8:
        # E4M3 MMAs run at twice the bf16 rate (nominal 4.5 vs 2.25 PFLOP/s dense)
        tpeak, tpeak_src = 2.0 * tpeak, tpeak_src + " x 2 (nominal E4M3 / bf16 ratio)"
    flops_layer = 2.0 * (w.dc + w.dr + w.dc) * w.visible_pairs
    intensity = flops_layer / kv_bytes_layer
    ridge = tpeak * 1e12 / (peak * 1e9)
    if intensity > ridge:
        achieved_t = flops_layer / (dec_avg / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": "split decode", "achieved": achieved_t,
                    "peak": tpeak, "peak_source": tpeak_src, "unit": "TFLOP/s",
                    "frac": achieved_t / tpeak, "traffic": traffic,
                    "algorithmic_flops_per_launch": flops_layer,
                    "flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                    "hbm_achieved_gbs": achieved, "hbm_frac": achieved / peak}
    else:
        roofline = {"bound": "hbm", "kernel": "split decode", "achieved": achieved,
                    "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "algorithmic_bytes_per_launch": kv_bytes_layer,
                    "flop_per_byte": intensity, "ridge_flop_per_byte": ridge}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": workload_description(w, fp8), "requests": w.num_reqs,
                   "n_q": w.n_q, "heads": w.num_heads, "layers": layers,
                   "kv_tokens": w.kv_tokens, "kv_bytes_per_step": kv_bytes_step,
                   "l2": "inputs larger than L2 (KV per step >> 129 MB L2), no flush",
                   "split": args.split, "parallelism": f"replicas x{world}",
                   "call": ("mla_decode_layers per step (one split plan, then each layer's "
                            "decode and combine)" if layers > 1 else "mla_decode per step"),
                   "timing": ("plain back-to-back calls" if args.no_graph else
                              "the K step calls captured in one CUDA graph and replayed")},
        "pct_of_hbm_peak": 100.0 * value / world / peak,
        "pct_of_nominal_8tbs": 100.0 * value / world / NOMINAL_HBM_GBS,
        "request_steps_per_s": w.num_reqs * world / (max_ms / K / 1e3),
        "kernel_ms": {"plan": statistics.mean(plan_ms), "decode": dec_avg,
                      "combine": statistics.mean(combine_ms),
                      "staged_ms_per_step": staged_ms / K,
                      "note": "from a second timed pass of the same K steps as per-layer "
                              "mla_decode calls (a plan per layer) with CUDA events recorded "
                              "between the kernels (which stops them overlapping); the "
                              "reported value comes from the first pass, without them"},
        "roofline": roofline,
        "gpu_launches": K * launches_per_step(layers, fp8),
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, qs[0][0], qs[0][1], qs[0][2], slabs[0],
                                            args.cpu_seconds, KV_SCALE_FP8 if fp8 else None)
    return line


def launches_per_step(layers, fp8):
    """Kernels of one mla_decode_layers step: the plan, each layer's decode and
    combine, and for E4M3 pages the query quantiser of every layer after the
    first (the plan grid quantises the first)."""
    return 1 + 2 * layers + (layers - 1 if fp8 else 0) if layers > 1 else 3


def layers_decoder(plmla, fp8):
    """The public step call for every layer, for the cache format."""
    if not fp8:
        return plmla.mla_decode_layers

    def decode_layers_fp8(*a, **k):
        return plmla.mla_decode_layers(*a, kv_scale=KV_SCALE_FP8, **k)
    return decode_layers_fp8


def decoder(plmla, fp8):
    """The public decode call for the cache format."""
    if not fp8:
        return plmla.mla_decode

    def decode_fp8(*a, **k):
        return plmla.mla_decode_fp8(*a, kv_scale=KV_SCALE_FP8, **k)
    return decode_fp8


def run_e2e(args, w, qs, table, lens, device, dist, call_step, kv_bytes_layer):
    """Same metric through the public call with pinned host buffers: each step
    copies its inputs host->device, decodes, and reads the result back.  As a
    serving loop would, the copies run on their own streams with two buffer
    sets, so step k+1's inputs travel while step k decodes and step k's results
    return while step k+1 decodes; every step's copies are inside the timed
    region."""
    import torch
    layers = w.num_slabs
    nbuf = 2
    host_q = [[t.cpu().pin_memory() for t in q] for q in qs]
    host_table = table.cpu().pin_memory()
    host_lens = lens.cpu().pin_memory()
    dev_q = [[[torch.empty_like(t) for t in q] for q in qs] for _ in range(nbuf)]
    dev_table = [torch.empty_like(table) for _ in range(nbuf)]
    dev_lens = [torch.empty_like(lens) for _ in range(nbuf)]
    host_out = [[torch.empty(q[0].shape, dtype=q[0].dtype).pin_memory() for q in qs]
                for _ in range(nbuf)]
    host_lse = [[torch.empty(w.num_tokens, w.num_heads, dtype=torch.float32).pin_memory()
                 for _ in qs] for _ in range(nbuf)]
    dev_out = [[torch.empty_like(q[0]) for q in qs] for _ in range(nbuf)]
    dev_lse = [[torch.empty(w.num_tokens, w.num_heads, dtype=torch.float32, device=device)
                for _ in qs] for _ in range(nbuf)]
    h2d = sum(t.numel() * t.element_size() for q in host_q for t in q)
    h2d += host_table.numel() * 4 + host_lens.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in host_out[0] + host_lse[0])
    stream = torch.cuda.current_stream(device)
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_ready = [ev() for _ in range(nbuf)]      # buffer b's inputs are on the device
    in_free = [ev() for _ in range(nbuf)]       # buffer b's inputs were consumed
    out_ready = [ev() for _ in range(nbuf)]     # buffer b's results were written
    out_free = [ev() for _ in range(nbuf)]      # buffer b's results were read back
    for b in range(nbuf):
        for e in (in_free[b], out_free[b]):
            e.record(stream)
    counter = [0]

    def step():
        b = counter[0] % nbuf
        counter[0] += 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(in_free[b])
            dev_table[b].copy_(host_table, non_blocking=True)
            dev_lens[b].copy_(host_lens, non_blocking=True)
            for l in range(layers):
                for d, h in zip(dev_q[b][l], host_q[l]):
                    d.copy_(h, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_free[b])
        call_step(dev_q[b], dev_table[b], dev_lens[b], dev_out[b], dev_lse[b])
        in_free[b].record(stream)
        out_ready[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[b])
            for l in range(layers):
                host_out[b][l].copy_(dev_out[b][l], non_blocking=True)
                host_lse[b][l].copy_(dev_lse[b][l], non_blocking=True)
            out_free[b].record(s_out)

    def join():
        # the compute stream waits for both copy streams' last work
        done_in, done_out = ev(), ev()
        done_in.record(s_in)
        done_out.record(s_out)
        stream.wait_event(done_in)
        stream.wait_event(done_out)

    for _ in range(args.warmup):
        step()
    join()
    torch.cuda.synchronize(device)
    barrier(dist, device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    s_in.wait_event(start)
    s_out.wait_event(start)
    for _ in range(args.steps):
        step()
    join()
    end.record(stream)
    torch.cuda.synchronize(device)
    ms = start.elapsed_time(end)
    max_ms, units = aggregate(dist, ms, kv_bytes_layer * layers * args.steps, device)
    return {"value": units / (max_ms / 1e3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": max_ms / args.steps,
            "note": "KV pool resident in HBM (it is the cache); per-step queries, gates, "
                    "page table and lengths copied in from pinned host memory, outputs and LSE "
                    "copied back, on their own streams with two buffer sets (step k+1's inputs "
                    "and step k's results travel while step k, k+1 decode)"}


# --------------------------------------------------------------------------
# KV append (the step before the hot path): n_new rows per request written into
# the steady workload's pool
# --------------------------------------------------------------------------

APPEND_METRIC = "paged KV append: achieved HBM GB/s on row bytes read + written"


def append_rows(w, n_new, device, seed=11):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    lat = torch.empty(w.num_reqs * n_new, w.dc, dtype=torch.bfloat16,
                      device=device).normal_(generator=g)
    rope = torch.empty(w.num_reqs * n_new, w.dr, dtype=torch.bfloat16,
                       device=device).normal_(generator=g)
    return lat, rope


def time_appends(plmla, lat, rope, slab, table, lens, n_new, K, W, stream):
    import torch
    for _ in range(W):
        plmla.mla_kv_append(lat, rope, slab, table, lens, n_new)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(K):
        plmla.mla_kv_append(lat, rope, slab, table, lens, n_new)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / K


def time_append_graph(plmla, lat, rope, slab, table, lens, n_new, stream, per_graph=20,
                      replays=10):
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        plmla.mla_kv_append(lat, rope, slab, table, lens, n_new)
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(per_graph):
            plmla.mla_kv_append(lat, rope, slab, table, lens, n_new)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(replays):
        graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / (replays * per_graph)


DCP_METRIC = ("decode context parallelism, ranks serialised on one GPU: projected step time "
              "(slowest rank's shard + decode, plus the merge), KV GB/s")


def run_dcp(args):
    """Decode context parallelism's device work for one layer of the workload:
    every rank's page shard (mla_dcp_shard) and decode on its pages, then the
    merge of the ranks' gated outputs (mla_merge_partials).  The ranks run one
    after another on this GPU, each timed alone; the projected step of a group
    of GPUs is the slowest rank plus the merge.  The all-gather between them is
    not measured (one GPU), and no rank waits on another."""
    import torch
    import paged_latent_attention_gb300 as plmla
    from paged_latent_attention_gb300 import inputs

    world_procs, rank_proc, local = dist_env()
    if world_procs > 1:
        raise SystemExit("--op dcp runs in one process (the ranks are serialised)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    G = args.dcp_world
    if not 1 <= G <= 64:
        raise SystemExit("--dcp-world must lie in [1, 64]")
    w = inputs.make_workload(args.workload)
    qn, qr, gate = inputs.make_queries(w, device)
    slab = inputs.make_slab(w, device)
    table = torch.as_tensor(w.page_table, device=device)
    lens = torch.as_tensor(w.seq_lens, device=device)
    T, H = w.num_tokens, w.num_heads
    ws = plmla.allocate_workspace(w.num_reqs, w.n_q, H, 0, 1, device)
    out_parts = torch.empty(G, T, H, 512, dtype=torch.bfloat16, device=device)
    lse_parts = torch.empty(G, T, H, dtype=torch.float32, device=device)
    shards = [plmla.mla_dcp_shard(table, lens, G, k) for k in range(G)]
    stream = torch.cuda.current_stream(device)
    K, W = args.steps, max(3, args.warmup)

    def timed(fn):
        for _ in range(W):
            fn()
        torch.cuda.synchronize(device)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(K):
            fn()
        end.record(stream)
        torch.cuda.synchronize(device)
        return start.elapsed_time(end) / K

    def rank_step(k):
        def fn():
            t_k, l_k = plmla.mla_dcp_shard(table, lens, G, k)
            plmla.mla_decode(qn, qr, gate, slab, t_k, l_k, n_q=w.n_q, out=out_parts[k],
                             lse=lse_parts[k], workspace=ws)
        return fn

    rank_ms = [timed(rank_step(k)) for k in range(G)]
    merge_ms = timed(lambda: plmla.mla_merge_partials(out_parts, lse_parts))
    whole_out = torch.empty_like(qn)
    whole_lse = torch.empty(T, H, dtype=torch.float32, device=device)
    whole_ms = timed(lambda: plmla.mla_decode(qn, qr, gate, slab, table, lens, n_q=w.n_q,
                                              out=whole_out, lse=whole_lse, workspace=ws))
    merged_out, merged_lse = plmla.mla_merge_partials(out_parts, lse_parts)
    torch.cuda.synchronize(device)
    lse_err = float((merged_lse - whole_lse).abs().max())
    rank_tokens = [int(l_k.sum()) for _, l_k in shards]
    kv_bytes = w.kv_tokens * kv_row_bytes(w, False)
    step_ms = max(rank_ms) + merge_ms
    parts_bytes = G * T * H * (512 * 2 + 4) + T * H * (512 * 2 + 4)
    return {
        "metric": DCP_METRIC, "value": kv_bytes / (step_ms / 1e3) / 1e9, "unit": UNIT,
        "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_description(w) + " (layer 0)", "dcp_world": G,
                   "parallelism": f"dcp{G}, ranks serialised on one GPU"},
        "rank_ms": rank_ms, "rank_kv_tokens": rank_tokens,
        "rank_balance": max(rank_ms) / (sum(rank_ms) / G),
        "merge_ms": merge_ms, "merge_gbs": parts_bytes / (merge_ms / 1e3) / 1e9,
        "unsharded_decode_ms": whole_ms,
        "projected_speedup_vs_one_gpu": whole_ms / step_ms,
        "merged_vs_unsharded_max_lse_diff": lse_err,
        "note": "each rank's shard and decode timed alone on one GPU; the projected step is the "
                "slowest rank plus the merge, without the all-gather of T x H x 1,028 bytes per "
                "rank (not measurable on one GPU)",
        "gpu_launches": K * (G * 4 + 1),
    }


def run_append(args):
    import torch
    import paged_latent_attention_gb300 as plmla
    from paged_latent_attention_gb300 import inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, "nccl")
    w = inputs.make_workload("steady")
    n_new = args.append_tokens
    if n_new < 1 or n_new > int(w.seq_lens.min()):
        raise SystemExit(f"--append-tokens must lie in [1, {int(w.seq_lens.min())}]")
    slab = inputs.make_slab(w, device)
    table = torch.as_tensor(w.page_table, device=device)
    lens = torch.as_tensor(w.seq_lens, device=device)
    lat, rope = append_rows(w, n_new, device)
    rows = w.num_reqs * n_new
    row_bytes = (w.dc + w.dr) * 2
    # algorithmic bytes: each new row read once and written once, plus the
    # lengths and one table entry per row
    bytes_step = 2 * rows * row_bytes + w.num_reqs * 4 + rows * 4
    stream = torch.cuda.current_stream(device)
    K, W = args.steps, max(3, args.warmup)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid).start()
    time.sleep(0.3)
    barrier(dist, device)
    host_t0 = time.time()
    ms = time_appends(plmla, lat, rope, slab, table, lens, n_new, K, W, stream)
    host_t1 = time.time()
    # the decode step's own append: one new row per request, timed as CUDA-graph
    # replays of 20 launches so the host's launch cost stays out
    lat1, rope1 = append_rows(w, 1, device, seed=12)
    ms_one = time_append_graph(plmla, lat1, rope1, slab, table, lens, 1, stream)
    barrier(dist, device)
    max_ms, units = aggregate(dist, ms, bytes_step, device)

    e2e = None
    if not args.no_e2e:
        host_lat, host_rope = lat.cpu().pin_memory(), rope.cpu().pin_memory()
        host_lens = lens.cpu().pin_memory()
        dev_lat, dev_rope, dev_lens = (torch.empty_like(lat), torch.empty_like(rope),
                                       torch.empty_like(lens))
        host_status = torch.zeros(1, dtype=torch.int32).pin_memory()
        status = torch.zeros(1, dtype=torch.int32, device=device)

        def e2e_step():
            dev_lat.copy_(host_lat, non_blocking=True)
            dev_rope.copy_(host_rope, non_blocking=True)
            dev_lens.copy_(host_lens, non_blocking=True)
            plmla.mla_kv_append(dev_lat, dev_rope, slab, table, dev_lens, n_new, status=status)
            host_status.copy_(status, non_blocking=True)

        for _ in range(W):
            e2e_step()
        torch.cuda.synchronize(device)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(K):
            e2e_step()
        end.record(stream)
        torch.cuda.synchronize(device)
        e_ms, e_units = aggregate(dist, start.elapsed_time(end) / K, bytes_step, device)
        e2e = {"value": e_units / (e_ms / 1e3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": host_lat.numel() * 2 + host_rope.numel() * 2 + 4 * w.num_reqs,
               "d2h_bytes_per_step": 4, "ms_per_step": e_ms,
               "note": "new rows and lengths copied in from pinned host memory, the status "
                       "word copied out; the pool stays resident"}
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(host_t0, host_t1)
    if rank != 0:
        return None
    peak, peak_src = hbm_peak()
    achieved = bytes_step / (ms / 1e3) / 1e9
    line = {
        "metric": APPEND_METRIC, "value": units / (max_ms / 1e3) / 1e9, "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": max_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"KV append: {w.num_reqs} requests x {n_new} new tokens "
                               f"({rows} rows of 512 latent + 64 rope bf16) into the steady "
                               f"decode pool ({w.num_pages} pages of 1536 tokens), positions "
                               f"seq_lens - {n_new} .. seq_lens - 1",
                   "rows": rows, "bytes_per_step": bytes_step,
                   "l2": "rows read + written per step exceed the 129 MB L2"
                         if 2 * rows * row_bytes > 129e6 else "fits in L2 (no flush)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "kv append", "achieved": achieved,
                     "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": bytes_step},
        "decode_step_append_us": 1e3 * ms_one,
        "gpu_launches": K + (K if e2e is not None else 0),
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = append_cpu_baseline(w, slab, lat, rope, n_new, args.cpu_seconds)
    return line


def append_cpu_baseline(w, slab_dev, lat, rope, n_new, target_s):
    """The oracle's kv_append on the pages of the first few requests (remapped
    into a small host pool), timed on the host."""
    import numpy as np
    import torch
    import oracle
    ids = list(range(min(8, w.num_reqs)))
    per = [-(-int(w.seq_lens[r]) // w.page_tokens) for r in ids]
    phys = [int(p) for r, n in zip(ids, per) for p in w.page_table[r, :n]]
    host = slab_dev.index_select(0, torch.as_tensor(phys, device=slab_dev.device)).cpu()
    table = np.zeros((len(ids), max(per)), dtype=np.int32)
    pos = 0
    for i, n in enumerate(per):
        table[i, :n] = np.arange(pos, pos + n)
        pos += n
    lens = w.seq_lens[ids].astype(np.int32)
    lat_h, rope_h = lat[:len(ids) * n_new].cpu(), rope[:len(ids) * n_new].cpu()
    elapsed, reps = 0.0, 0
    while elapsed < 0.5 * target_s or reps == 0:
        t = time.perf_counter()
        oracle.kv_append(host, table, lens, lat_h, rope_h, n_new, page_stride=w.page_stride)
        elapsed += time.perf_counter() - t
        reps += 1
    rows = len(ids) * n_new
    gbs = 2 * rows * (w.dc + w.dr) * 2 * reps / elapsed / 1e9
    return {"value": gbs, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{len(ids)} of {w.num_reqs} requests x {n_new} new rows, {reps} pass(es) "
                      f"over a {len(phys)}-page host pool, {elapsed:.1f} s"}


# --------------------------------------------------------------------------
# reference arm: the oracle as it stands, on host cores
# --------------------------------------------------------------------------

def run_reference(args):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    workload: each step decodes a few requests (in rotation) of one layer, with
    all heads; the pages the sample reads are drawn on the host
    (inputs.make_host_pages).  KV bytes are credited per row computed, and for a
    multi-layer workload the step time is the sample's time per layer times the
    layer count (every layer is the same work)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    from paged_latent_attention_gb300 import inputs
    w = inputs.make_workload(args.workload)
    if args.control:
        w = inputs.equal_length_control(w)
    fp8 = args.kv == "fp8"
    kv_scale = KV_SCALE_FP8 if fp8 else None
    qn, qr, gate = inputs.make_queries(w, "cpu")
    cores = oracle.oracle.default_threads()
    total = args.steps + args.warmup
    budget_s = 150.0

    def sample(ids):
        slab, table, lens = inputs.make_host_pages(w, ids, fp8=fp8, kv_scale=kv_scale)
        rows_q = [r * w.n_q + j for r in ids for j in range(w.n_q)]
        return (qn[rows_q], qr[rows_q], gate[rows_q], slab, table, lens, slab.shape[0])

    t1 = run_oracle(w, sample([0]), kv_scale, row_sample(w, 1)[0])
    per_step = max(1, min(w.num_reqs, int(budget_s / total / max(t1, 1e-3))))
    rows, frac = row_sample(w, per_step)
    times, kv = [], []
    cache = {}                    # every distinct sample, drawn once (a few GB at most)
    for s in range(total):
        ids = tuple((s * per_step + i) % w.num_reqs for i in range(per_step))
        if ids not in cache:
            cache[ids] = sample(list(ids))
        dt = run_oracle(w, cache[ids], kv_scale, rows)
        if s >= args.warmup:
            times.append(dt)
            kv.append(frac * sum(int(w.seq_lens[r]) for r in ids) * kv_row_bytes(w, fp8))
    elapsed = sum(times)
    value = sum(kv) / elapsed / 1e9
    layers = w.num_slabs
    what = (f"all {w.num_heads} heads" if rows is None else
            f"{frac:.4f} of the rows (first, middle and last new token, 4 heads; KV bytes "
            f"credited in proportion)")
    desc = (f"{per_step} of {w.num_reqs} requests x {what} of one layer per step "
            f"(requests taken in rotation), double-precision oracle; pages drawn on the host "
            f"(copies of {inputs.HOST_PAGE_BANK} N(0,1) pages: the oracle's work does not "
            f"depend on the values)")
    # the whole step (every request, every layer) at the sample's rate
    ms_step = 1e3 * w.kv_tokens * kv_row_bytes(w, fp8) * layers / (value * 1e9)
    desc += (f"; ms_per_step = the full step's KV bytes ({layers} layer(s)) at the sample's "
             f"rate")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_description(w, fp8)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        line = run_reference(args)
    elif args.op == "append":
        line = run_append(args)
    elif args.op == "dcp":
        line = run_dcp(args)
    else:
        line = run_gpu(args)
    if line is not None:
        text = json.dumps(line)
        print(text, flush=True)
        if args.out:
            with open(args.out, "a") as f:
                f.write(text + "\n")
    world, _, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
