#!/usr/bin/env python3
"""Benchmark the MLA latent-cache decode step on B300.

A step is one pass of the whole hot path over one batch: compress-and-append
the B*n_q new tokens (mla_append_kv), then decode (absorb q, split-KV
attention over the paged latent cache, log-sum-exp combine, W_uv
up-projection).

The JSON line is headed by the DeepSeek-V2-shape ragged workload (batch 64,
cached lengths uniform in [512, 32768], 1 query token, bf16 cache), the
largest DeepSeek-V2-shape decode workload on one GPU. The same run times the
other bf16 workloads (batch 16 x 4096; batch 4 x 131072 with 2 query tokens;
16 heads, batch 256 x [1024, 8192]) and reports each under ``per_config``:
tokens/s, cache GB/s, the attention kernel's roofline fraction and the whole
step's roofline fraction.

L2 hygiene: the timed steps cycle through several layer-sized input sets
(cache, page table, weights, queries, hidden states). Their total is more
than 3x the L2 size, so no step finds its inputs in L2.

``--gpus N`` without a torchrun environment starts N local processes
through torch.distributed.run, one replica per GPU (sequences shard across
replicas with no collective on the data path).

Prints one JSON line. --impl reference times the fp64 CPU oracle on a
bounded sample of the headline workload instead.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s and latent-cache GB/s at 1 B300, % of roofline"
# The largest DeepSeek-V2-shape workload that fits one GPU heads the line;
# the other bf16 workloads are timed in the same run (per_config).
DEFAULT_WORKLOAD = "dsv2_b64_ragged"
PER_CONFIG = ["dsv2_b64_ragged", "dsv2_b16_l4096", "dsv2_b4_l131072_nq2", "nh16_b256_ragged"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the fp8-cache rows (per_config_fp8)")
    ap.add_argument("--only", action="store_true",
                    help="time the --workload alone (no per_config rows for the others)")
    ap.add_argument("--cpu-sample-heads", type=int, default=0,
                    help="(b, h) pairs in the oracle sample (0: about 10 s worth)")
    ap.add_argument("--variant", choices=["per_head", "full_fold", "layer"], default="per_head",
                    help="full_fold: time the folded layer (x_q in, y out); layer: time "
                         "append + decode + W_o (mla_decode_layer)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed helpers (one process per GPU; replicas, no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(value, dist, device="cpu"):
    """Max of a float over all ranks (identity when not distributed)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, dist, device="cpu"):
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def whole_job_rate(units, ms, dist, device="cpu"):
    """(units of all ranks per second over the slowest rank's time, that time
    in ms). Every rank gets the same pair."""
    ms_max = max_over_ranks(ms, dist, device)
    return sum_over_ranks(units, dist, device) / (ms_max / 1e3), ms_max


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------

def algorithmic(w, lens):
    """Cache bytes and attention FLOPs of one decode call."""
    rows = int(np.sum(lens))
    cache_bytes = rows * w.R * w.elem_bytes
    # per visible (row, query): 2*(R + d_c) FLOPs per head. Visible rows of query i
    # are L - n_q + i + 1.
    vis = sum(int(L) - w.n_q + i + 1 for L in lens for i in range(w.n_q))
    attn_flops = 2.0 * w.n_h * (w.R + w.d_c) * vis
    return cache_bytes, attn_flops


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


def kernel_source_hash():
    src = os.path.join(ROOT, "mla_latent_kv_73_b300", "csrc", "attend_tc.cu")
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "attend_tc_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_sha") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        # the raw samples go to MLA_CLOCKS_CSV if set (to keep them), else to
        # a temporary file; the JSON line carries their summary either way
        self.path = os.environ.get("MLA_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), f"mla_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, t_start, t_end):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------

def step_algorithmic(w, lens):
    """Bytes and FLOPs of one whole step (append of the B*n_q new tokens, then
    the decode), counting each input once and each output once.

    Bytes: the cache, the append's packed W_dkv||W_kr, W_uk and W_uv, the new
    tokens' hidden states and cache rows, the queries and the fp32 output.
    FLOPs: the attention's, plus the append (d_model x R per token), the
    query absorption (d_c x d_nope per head and token) and the value
    up-projection (d_c x d_v per head and token).
    """
    cache_bytes, attn_flops = algorithmic(w, lens)
    eb = w.elem_bytes
    Tq = w.batch * w.n_q
    weight_bytes = (w.R * w.d_model + w.n_h * w.d_c * (w.d_nope + w.d_v)) * eb
    act_bytes = Tq * (w.d_model + w.R + w.n_h * (w.d_nope + w.d_r)) * eb + Tq * w.n_h * w.d_v * 4
    flops = attn_flops + 2.0 * Tq * (w.d_model * w.R + w.n_h * w.d_c * (w.d_nope + w.d_v))
    return cache_bytes + weight_bytes + act_bytes, flops


def roofline_entry(nbytes, flops, ms, hbm, tflops):
    """Roofline of work that moves nbytes and does flops in ms: the slower of
    the bytes at the HBM peak and the FLOPs at the bf16 peak."""
    t_mem = nbytes / (hbm * 1e9)
    t_ten = flops / (tflops * 1e12)
    gbs = nbytes / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    if t_mem >= t_ten:
        e = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
             "frac": round(gbs / hbm, 4)}
    else:
        e = {"bound": "tensor", "achieved": round(tfs, 1), "peak": tflops, "unit": "TFLOP/s",
             "frac": round(tfs / tflops, 4)}
    e["roofline_ms"] = round(max(t_mem, t_ten) * 1e3, 5)
    e["gbs"] = round(gbs, 1)
    e["tflops"] = round(tfs, 1)
    return e


def measure_workload(args, w, K, warmup, world, rank, local, dist, headline, min_steps=1):
    """Time one workload's whole step (append + absorb + attention + combine)
    from CUDA graphs over rotating input sets. Returns a dict; the headline
    workload also gets the clock record, the end-to-end figures and the
    host enqueue cost."""
    import torch
    from mla_latent_kv_73_b300 import _lib, synth
    from mla_latent_kv_73_b300.device_inputs import DeviceWeights, config_for, to_device

    lens = synth.seq_lens(w)
    B, n_q = w.batch, w.n_q
    Tq = B * n_q
    cfg = config_for(w)
    impl = _lib.mla_decode_impl(cfg)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    pt_np, num_blocks = synth.page_table(w, lens)
    max_blocks = pt_np.shape[1]
    cache_bytes, attn_flops = algorithmic(w, lens)
    step_bytes, step_flops = step_algorithmic(w, lens)

    # input sets: one per simulated layer, together more than 3x L2
    wts = synth.weights(w)
    set_bytes = cache_bytes + (w.R * w.d_model + 2 * w.n_h * w.d_c * w.d_nope) * w.elem_bytes
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    n_sets = max(2, math.ceil(3 * l2 / set_bytes))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + 17 * rank + w.seed)
    sets = []
    for k in range(n_sets):
        s = {}
        s["w"] = DeviceWeights(w, wts, cfg)
        s["cache"] = torch.randn((num_blocks, w.block_size, w.R), generator=gen,
                                 device="cuda").to(dt)
        s["pt"] = to_device(pt_np, "i32")
        s["x"] = torch.randn((Tq, w.d_model), generator=gen, device="cuda").to(dt)
        s["q"] = torch.randn((B, n_q, w.n_h, w.d_nope + w.d_r), generator=gen,
                             device="cuda").to(dt)
        s["sl"] = to_device(lens, "i32")  # per-set copies for the pipelined end-to-end run
        s["out"] = torch.empty((B, n_q, w.n_h, w.d_v), device="cuda")
        sets.append(s)
    seq_lens = to_device(lens, "i32")
    seq_idx = to_device(np.repeat(np.arange(B), n_q).astype(np.int32), "i32")
    pos = to_device(np.concatenate([np.arange(L - n_q, L) for L in lens]).astype(np.int32),
                    "i32")
    out = torch.empty((B, n_q, w.n_h, w.d_v), device="cuda")
    ws = torch.empty(_lib.mla_decode_workspace_size(cfg, B, n_q, int(lens.sum())),
                     dtype=torch.uint8, device="cuda")

    def step(s, st):
        _lib.mla_append_kv(cfg, s["w"].handle, s["x"], seq_idx, pos, s["pt"], s["cache"], st)
        _lib.mla_decode_absorb_q(cfg, s["w"].handle, s["q"], seq_lens, max_blocks, ws, st)
        _lib.mla_decode_attend(cfg, s["cache"], s["pt"], seq_lens, B, n_q, ws, st)
        _lib.mla_decode_combine(cfg, s["w"].handle, seq_lens, B, n_q, out, ws, st)

    stream = torch.cuda.current_stream()
    for i in range(warmup):
        step(sets[i % n_sets], stream)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"{w.name}: device error word {code:#x} after warm-up")

    # One CUDA graph per input set: a whole step; and a whole step with
    # timing events between its four stages.
    n_stage_ev = 8
    stage_ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
                for _ in range(n_sets * n_stage_ev)]

    def step_timed(s, st, ev):
        ev[0].record(st)
        _lib.mla_append_kv(cfg, s["w"].handle, s["x"], seq_idx, pos, s["pt"], s["cache"], st)
        ev[1].record(st)
        _lib.mla_decode_absorb_q(cfg, s["w"].handle, s["q"], seq_lens, max_blocks, ws, st)
        ev[2].record(st)
        _lib.mla_decode_attend(cfg, s["cache"], s["pt"], seq_lens, B, n_q, ws, st)
        ev[3].record(st)
        _lib.mla_decode_combine(cfg, s["w"].handle, seq_lens, B, n_q, out, ws, st)
        ev[4].record(st)

    g_step, g_prof = [], []
    for k in range(n_sets * n_stage_ev):
        s = sets[k % n_sets]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step_timed(s, torch.cuda.current_stream(), stage_ev[k])
        g_prof.append(g)
    for s in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(s, torch.cuda.current_stream())
        g_step.append(g)
    for i in range(3 * n_sets):
        g_step[i % n_sets].replay()
    torch.cuda.synchronize()

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if K is None:
        t0.record()
        for i in range(4 * n_sets):
            g_step[i % n_sets].replay()
        t1.record()
        torch.cuda.synchronize()
        est = t0.elapsed_time(t1) / (4 * n_sets)
        K = int(min(3000, max(min_steps, 300.0 / max(est, 1e-3))))
        K = int(max_over_ranks(K, dist, "cuda"))
    clk = ClockSampler(local) if headline else contextlib.nullcontext()
    with clk:
        barrier(dist)
        torch.cuda.synchronize()
        wall0 = time.time()
        t0.record()
        h0 = time.perf_counter()
        for i in range(K):
            g_step[i % n_sets].replay()
        host_us = (time.perf_counter() - h0) * 1e6 / K
        t1.record()
        torch.cuda.synchronize()
        barrier(dist)
        wall1 = time.time()
    clocks = clk.summary(wall0, wall1) if headline else None
    total_ms = t0.elapsed_time(t1)
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"{w.name}: device error word {code:#x} in the timed region")
    value, total_ms_max = whole_job_rate(Tq * K, total_ms, dist, "cuda")
    ms_per_step = total_ms_max / K

    # the attention kernel on its own: one CUDA graph of R launches back to
    # back on the stream, cycling through the input sets (each launch finds
    # its cache cold), timed with events around the graph; per launch =
    # total / R. (One graph per launch would add a graph launch to every
    # kernel; events between the kernels of a step graph serialise the
    # programmatic launch chain.)
    R = max(16, 4 * n_sets)
    g_att_r = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_att_r):
        for i in range(R):
            s_ = sets[i % n_sets]
            _lib.mla_decode_attend(cfg, s_["cache"], s_["pt"], seq_lens, B, n_q, ws,
                                   torch.cuda.current_stream())
    g_att_r.replay()
    torch.cuda.synchronize()
    Ka = max(3, min(50, (K + R - 1) // R))
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record()
    for i in range(Ka):
        g_att_r.replay()
    a1.record()
    torch.cuda.synchronize()
    attend_ms = [a0.elapsed_time(a1) / (Ka * R)]

    # the attention core a3 + a4 (mla_decode_latent: latent queries in, the
    # merged o_lat out), timed the same way
    q_lat_abs = torch.randn((B, n_q, w.n_h, w.R), generator=gen, device="cuda").to(dt)
    o_lat = torch.empty((B, n_q, w.n_h, w.d_c), device="cuda")
    g_core = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_core):
        for i in range(R):
            s_ = sets[i % n_sets]
            _lib.mla_decode_latent(cfg, q_lat_abs, s_["cache"], s_["pt"], seq_lens, o_lat, ws,
                                   torch.cuda.current_stream())
    g_core.replay()
    torch.cuda.synchronize()
    a0.record()
    for i in range(Ka):
        g_core.replay()
    a1.record()
    torch.cuda.synchronize()
    core_ms = a0.elapsed_time(a1) / (Ka * R)
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"{w.name}: device error word {code:#x} in the core timing")
    del q_lat_abs, o_lat, g_core

    # the four stages inside whole-step graph replays (events between them)
    for g in g_prof:
        g.replay()
    torch.cuda.synchronize()
    names = ["append", "absorb_q", "attend", "combine"]
    acc = {n: [] for n in names}
    for rep in range(3):
        for g in g_prof:
            g.replay()
        torch.cuda.synchronize()
        for ev in stage_ev:
            for j, n in enumerate(names):
                acc[n].append(ev[j].elapsed_time(ev[j + 1]))
    stages = {n: round(1e3 * statistics.mean(v), 2) for n, v in acc.items()}
    stages["attend_alone"] = round(1e3 * statistics.mean(attend_ms), 2)
    stages["note"] = ("us per stage inside whole-step graphs split by events; attend_alone: "
                      "average launch of the attention kernel in a graph of back-to-back launches")

    hbm, tflops, tflops_sus, src = measured_peaks()
    # the attention kernel's time: its average launch in a graph of
    # back-to-back launches on cold input sets (above)
    att_ms = statistics.mean(attend_ms)
    att = roofline_entry(cache_bytes, attn_flops, att_ms, hbm, tflops)
    att["kernel"] = "attend_tc_kernel" if impl == 2 else "attend_simt_kernel"
    att["kernel_ms"] = round(att_ms, 5)
    core = roofline_entry(cache_bytes, attn_flops, core_ms, hbm, tflops)
    core["kernel_ms"] = round(core_ms, 5)
    core["what"] = ("attention core a3 + a4 (mla_decode_latent: query copy and plan, "
                    "attention, log-sum-exp merge into o_lat) against the cache roofline")
    step_roof = roofline_entry(step_bytes, step_flops, ms_per_step, hbm, tflops)
    step_roof["bytes"] = int(step_bytes)
    step_roof["flops"] = float(step_flops)
    step_roof["what"] = ("whole step (append + absorb + attention + combine): cache + "
                         "W_dkv||W_kr + W_uk + W_uv + x + new rows + q + out")
    res = {
        "workload": w.name, "value": value, "ms_per_step": ms_per_step, "steps": K,
        "tokens_per_s": round(value, 1),
        "cache_gbs": round(cache_bytes * K / (total_ms_max / 1e3) / 1e9, 1),
        "cache_bytes": int(cache_bytes), "attention_flops": float(attn_flops),
        "attention_roofline": att, "core_roofline": core, "step_roofline": step_roof,
        "stage_us": stages,
        "impl": impl, "peak_source": src, "lens": lens, "n_sets": n_sets,
        "set_bytes": set_bytes, "l2": l2, "clocks": clocks, "host_us": host_us,
    }

    if headline:
        res["e2e"] = e2e_figures(w, lens, sets, n_sets, K, step, seq_lens, seq_idx, pos, out,
                                 max_blocks, cfg, ws, dist, stream)
    for s in sets:
        s["w"].free()
    del sets, ws
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def e2e_figures(w, lens, sets, n_sets, K, step, seq_lens, seq_idx, pos, out, max_blocks, cfg,
                ws, dist, stream):
    """The same step through the C ABI with its inputs copied up from pinned
    host memory and its result read back, every step, inside the timed
    region: serial (one stream), pipelined (copies on two side streams while
    the previous step computes) and issued call by call from Python."""
    import torch
    from mla_latent_kv_73_b300 import _lib
    B, n_q = w.batch, w.n_q
    Tq = B * n_q
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    pin_x = torch.empty((Tq, w.d_model), dtype=dt, pin_memory=True)
    pin_q = torch.empty((B, n_q, w.n_h, w.d_nope + w.d_r), dtype=dt, pin_memory=True)
    pin_lens = torch.from_numpy(lens.astype(np.int32)).pin_memory()
    pin_out = torch.empty((B, n_q, w.n_h, w.d_v), pin_memory=True)
    pin_x.copy_(sets[0]["x"].cpu())
    pin_q.copy_(sets[0]["q"].cpu())

    def e2e_step(s, st):
        s["x"].copy_(pin_x, non_blocking=True)
        s["q"].copy_(pin_q, non_blocking=True)
        seq_lens.copy_(pin_lens, non_blocking=True)
        step(s, st)
        pin_out.copy_(out, non_blocking=True)

    g_e2e = []
    for s in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_step(s, torch.cuda.current_stream())
        g_e2e.append(g)
    for i in range(2 * n_sets):
        g_e2e[i % n_sets].replay()
    torch.cuda.synchronize()
    Ke = max(n_sets, K // 2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    e0.record()
    for i in range(Ke):
        g_e2e[i % n_sets].replay()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
    e2e_value = sum_over_ranks(Tq * Ke, dist, "cuda") / (e2e_ms / 1e3)
    h2d = pin_x.numel() * pin_x.element_size() + pin_q.numel() * pin_q.element_size() + \
        pin_lens.numel() * 4
    d2h = pin_out.numel() * 4

    # Pipelined: step i+1's inputs go up on one copy stream and step i's
    # result comes down on another while step i computes. Each step still
    # uploads its own inputs and reads back its own result; a graph of
    # 8 * n_sets steps holds the copies, the steps and the cross-stream
    # dependencies (a set's inputs are overwritten only after the step that
    # read them, its output only after its read-back).
    def step_io(s, st):
        _lib.mla_append_kv(cfg, s["w"].handle, s["x"], seq_idx, pos, s["pt"], s["cache"], st)
        _lib.mla_decode_absorb_q(cfg, s["w"].handle, s["q"], s["sl"], max_blocks, ws, st)
        _lib.mla_decode_attend(cfg, s["cache"], s["pt"], s["sl"], B, n_q, ws, st)
        _lib.mla_decode_combine(cfg, s["w"].handle, s["sl"], B, n_q, s["out"], ws, st)

    P = 8 * n_sets
    c_in, c_out = torch.cuda.Stream(), torch.cuda.Stream()
    g_pipe = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pipe):
        cs = torch.cuda.current_stream()
        c_in.wait_stream(cs)
        c_out.wait_stream(cs)
        ev_in = [torch.cuda.Event() for _ in range(P)]
        ev_comp = [torch.cuda.Event() for _ in range(P)]
        ev_out = [torch.cuda.Event() for _ in range(P)]
        for i in range(P):
            s = sets[i % n_sets]
            if i >= n_sets:
                c_in.wait_event(ev_comp[i - n_sets])
            with torch.cuda.stream(c_in):
                s["x"].copy_(pin_x, non_blocking=True)
                s["q"].copy_(pin_q, non_blocking=True)
                s["sl"].copy_(pin_lens, non_blocking=True)
            ev_in[i].record(c_in)
            cs.wait_event(ev_in[i])
            if i >= n_sets:
                cs.wait_event(ev_out[i - n_sets])
            step_io(s, cs)
            ev_comp[i].record(cs)
            c_out.wait_event(ev_comp[i])
            with torch.cuda.stream(c_out):
                pin_out.copy_(s["out"], non_blocking=True)
            ev_out[i].record(c_out)
        cs.wait_stream(c_in)
        cs.wait_stream(c_out)
    for _ in range(2):
        g_pipe.replay()
    torch.cuda.synchronize()
    Rp = max(1, Ke // P)
    barrier(dist)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(Rp):
        g_pipe.replay()
    e1.record()
    torch.cuda.synchronize()
    pipe_ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
    pipe_value = sum_over_ranks(Tq * P * Rp, dist, "cuda") / (pipe_ms / 1e3)
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"device error word {code:#x} in the pipelined end-to-end run")

    # the same, issuing every call from Python each step (no graph)
    Kd = min(Ke, 500)
    e0.record()
    for i in range(Kd):
        e2e_step(sets[i % n_sets], stream)
    e1.record()
    torch.cuda.synchronize()
    e2e_direct = Tq * Kd / (e0.elapsed_time(e1) / 1e3)
    return {"value": round(pipe_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": P * Rp, "graph": True,
            "pipelined": "inputs of step i+1 up and result of step i down on two copy "
                         "streams while step i computes",
            "serial_value": round(e2e_value, 1), "serial_steps": Ke,
            "no_graph_value": round(e2e_direct, 1)}


def fp8_algorithmic(w, lens):
    """Bytes of an fp8 cache (one e4m3 code per element and one fp32 scale
    per row) and of the fp8 step: the cache, W_dkv||W_kr (bf16), W_uk,
    W_uv, x, the new rows' codes and scales, q and the fp32 output. FLOPs
    as for the bf16 step."""
    rows = int(np.sum(lens))
    cache_bytes = rows * (w.R + 4)
    Tq = w.batch * w.n_q
    eb = w.elem_bytes
    step_bytes = (cache_bytes + (w.R * w.d_model + w.n_h * w.d_c * (w.d_nope + w.d_v)) * eb
                  + Tq * (w.d_model + w.n_h * (w.d_nope + w.d_r)) * eb + Tq * (w.R + 4)
                  + Tq * w.n_h * w.d_v * 4)
    _, step_flops = step_algorithmic(w, lens)
    return cache_bytes, step_bytes, step_flops


def measure_workload_fp8(w, warmup, world, rank, local, dist, min_steps):
    """The same step over an fp8 (e4m3) cache: mla_append_kv_fp8 of the new
    tokens, then mla_decode_fp8 (absorb into fp16, attention over the codes,
    combine). Timed from CUDA graphs over rotating input sets larger than
    3x L2, about 0.3 s of steps (at least min_steps)."""
    import torch
    from mla_latent_kv_73_b300 import _lib, synth
    from mla_latent_kv_73_b300.device_inputs import DeviceWeights, config_for, to_device

    lens = synth.seq_lens(w)
    B, n_q = w.batch, w.n_q
    Tq = B * n_q
    cfg = config_for(w)
    pt_np, num_blocks = synth.page_table(w, lens)
    cache_bytes, step_bytes, step_flops = fp8_algorithmic(w, lens)
    wts = synth.weights(w)
    set_bytes = cache_bytes + (w.R * w.d_model + 2 * w.n_h * w.d_c * w.d_nope) * w.elem_bytes
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    n_sets = max(2, math.ceil(3 * l2 / set_bytes))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5000 + 17 * rank + w.seed)
    sets = []
    for _ in range(n_sets):
        s = {"w": DeviceWeights(w, wts, cfg), "pt": to_device(pt_np, "i32")}
        # random e4m3 bytes 0..126 with a random sign: never a NaN pattern
        c = torch.randint(0, 127, (num_blocks, w.block_size, w.R), generator=gen, device="cuda",
                          dtype=torch.uint8)
        c |= torch.randint(0, 2, c.shape, generator=gen, device="cuda", dtype=torch.uint8) << 7
        s["cache"] = c
        s["scale"] = torch.rand((num_blocks, w.block_size), generator=gen, device="cuda") * 0.01
        s["x"] = torch.randn((Tq, w.d_model), generator=gen, device="cuda").to(torch.bfloat16)
        s["q"] = torch.randn((B, n_q, w.n_h, w.d_nope + w.d_r), generator=gen,
                             device="cuda").to(torch.bfloat16)
        sets.append(s)
    seq_lens = to_device(lens, "i32")
    seq_idx = to_device(np.repeat(np.arange(B), n_q).astype(np.int32), "i32")
    pos = to_device(np.concatenate([np.arange(L - n_q, L) for L in lens]).astype(np.int32),
                    "i32")
    out = torch.empty((B, n_q, w.n_h, w.d_v), device="cuda")
    ws = torch.empty(_lib.mla_decode_workspace_size(cfg, B, n_q), dtype=torch.uint8,
                     device="cuda")
    ws_a = torch.empty(_lib.mla_append_kv_fp8_workspace_size(cfg, Tq), dtype=torch.uint8,
                       device="cuda")

    def step(s, st, ev=None):
        if ev is not None:
            ev[0].record(st)
        _lib.mla_append_kv_fp8(cfg, s["w"].handle, s["x"], seq_idx, pos, s["pt"], s["cache"],
                               s["scale"], ws_a, st)
        if ev is not None:
            ev[1].record(st)
        _lib.mla_decode_fp8(cfg, s["w"].handle, s["q"], s["cache"], s["scale"], s["pt"],
                            seq_lens, out, ws, st)
        if ev is not None:
            ev[2].record(st)

    stream = torch.cuda.current_stream()
    for i in range(warmup):
        step(sets[i % n_sets], stream)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"{w.name} fp8: device error word {code:#x} after warm-up")
    stage_ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
                for _ in range(4 * n_sets)]
    g_step, g_prof = [], []
    for k, s in enumerate(sets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(s, torch.cuda.current_stream())
        g_step.append(g)
    for k in range(4 * n_sets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(sets[k % n_sets], torch.cuda.current_stream(), stage_ev[k])
        g_prof.append(g)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(4 * n_sets):
        g_step[i % n_sets].replay()
    t1.record()
    torch.cuda.synchronize()
    est = t0.elapsed_time(t1) / (4 * n_sets)
    K = int(max_over_ranks(int(min(3000, max(min_steps, 300.0 / max(est, 1e-3)))), dist, "cuda"))
    barrier(dist)
    torch.cuda.synchronize()
    t0.record()
    for i in range(K):
        g_step[i % n_sets].replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(dist)
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"{w.name} fp8: device error word {code:#x} in the timed region")
    value, total_ms_max = whole_job_rate(Tq * K, t0.elapsed_time(t1), dist, "cuda")
    ms = total_ms_max / K
    acc = {"append": [], "decode": []}
    for rep in range(3):
        for g in g_prof:
            g.replay()
        torch.cuda.synchronize()
        if rep == 0:
            continue
        for ev in stage_ev:
            acc["append"].append(ev[0].elapsed_time(ev[1]))
            acc["decode"].append(ev[1].elapsed_time(ev[2]))
    hbm, tflops, _, _ = measured_peaks()
    dec_ms = statistics.mean(acc["decode"])
    rows = int(np.sum(lens))
    dec_bytes = cache_bytes + w.n_h * w.d_c * (w.d_nope + w.d_v) * w.elem_bytes + \
        Tq * w.n_h * ((w.d_nope + w.d_r) * w.elem_bytes + w.d_v * 4)
    _, attn_flops = algorithmic(w, lens)
    dec_flops = attn_flops + 2.0 * Tq * w.n_h * w.d_c * (w.d_nope + w.d_v)
    dec = roofline_entry(dec_bytes, dec_flops, dec_ms, hbm, tflops)
    dec["kernel_ms"] = round(dec_ms, 5)
    step_roof = roofline_entry(step_bytes, step_flops, ms, hbm, tflops)
    for s in sets:
        s["w"].free()
    del sets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {"tokens_per_s": round(value, 1), "ms_per_step": round(ms, 5), "steps": K,
            "cache_bytes": int(cache_bytes),
            "cache_bytes_per_token": w.R + 4,
            "cache_gbs": round(cache_bytes / (ms / 1e3) / 1e9, 1),
            "decode_call": {k: dec[k] for k in ("bound", "achieved", "unit", "frac", "kernel_ms",
                                                "roofline_ms", "gbs", "tflops")},
            "step": {k: step_roof[k] for k in ("bound", "achieved", "unit", "frac",
                                               "roofline_ms", "gbs", "tflops")},
            "stage_us": {k: round(1e3 * statistics.mean(v), 2) for k, v in acc.items()},
            "what": "mla_append_kv_fp8 + mla_decode_fp8 over an e4m3 cache with one fp32 scale "
                    "per row; decode_call = absorb + attention + combine in one call"}


def per_config_row(r):
    a, s = r["attention_roofline"], r["step_roofline"]
    return {"tokens_per_s": r["tokens_per_s"], "ms_per_step": round(r["ms_per_step"], 5),
            "steps": r["steps"], "cache_gbs": r["cache_gbs"],
            "attention": {k: a[k] for k in ("bound", "achieved", "unit", "frac", "kernel_ms",
                                            "roofline_ms", "gbs", "tflops")},
            "core_a3_a4": {k: r["core_roofline"][k] for k in ("bound", "achieved", "unit", "frac",
                                                             "kernel_ms", "roofline_ms")},
            "step": {k: s[k] for k in ("bound", "achieved", "unit", "frac", "roofline_ms",
                                       "gbs", "tflops")},
            "stage_us": r["stage_us"]}


def run_ours(args, world, rank, local):
    import torch
    from mla_latent_kv_73_b300 import _lib, synth

    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    _lib.load()
    head = synth.WORKLOADS[args.workload]
    others = [] if args.only else [n for n in PER_CONFIG if n != head.name]
    K = args.steps
    r = measure_workload(args, head, K, args.warmup, world, rank, local, dist, headline=True)
    rows = {head.name: per_config_row(r)} if head.dtype == "bf16" else {}
    for name in others:
        # K steps, or about 0.3 s of them if that is more (K=None: chosen
        # from a short probe after the warm-up)
        rc = measure_workload(args, synth.WORKLOADS[name], None, args.warmup, world, rank,
                              local, dist, headline=False, min_steps=K)
        rows[name] = per_config_row(rc)

    rows_fp8 = {}
    if not args.only and not args.no_fp8:
        for name in PER_CONFIG:
            rows_fp8[name] = measure_workload_fp8(synth.WORKLOADS[name], args.warmup, world, rank,
                                                  local, dist, min_steps=K)
    w = head
    lens = r["lens"]
    att = dict(r["attention_roofline"])
    roof = {k: att[k] for k in ("bound", "achieved", "peak", "unit", "frac")}
    roof["traffic"] = profiled_traffic(w.name)
    roof["peak_source"] = r["peak_source"]
    roof["kernel"] = att["kernel"]
    roof["kernel_ms"] = att["kernel_ms"]
    roof["roofline_ms"] = att["roofline_ms"]
    roof["what"] = "attention kernel only (a3): the latent cache against HBM, its FLOPs " \
                   "against the bf16 tensor peak"
    roof["tensor_tflops"] = att["tflops"]
    line = {
        "metric": METRIC,
        "value": round(r["value"], 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(r["ms_per_step"], 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) cache rows, hidden states and queries; "
                "N(0,1/fan_in) weights)",
        "config": {"workload": w.name, "batch": w.batch,
                   "seq_len": int(lens[0]) if w.len_lo == w.len_hi else [w.len_lo, w.len_hi],
                   "total_cached_tokens": int(np.sum(lens)), "n_q": w.n_q, "n_h": w.n_h,
                   "d_model": w.d_model, "d_c": w.d_c, "d_r": w.d_r,
                   "block_size": w.block_size, "parallelism": f"replicas x{world}",
                   "l2": f"{r['n_sets']} rotating layer-sized input sets, "
                         f"{r['n_sets'] * r['set_bytes'] / 2**20:.0f} MiB > 3x L2 "
                         f"({r['l2'] / 2**20:.0f} MiB)",
                   "decode_kernel": "tensor_core" if r["impl"] == 2 else "cuda_core"},
        "cache_gbs": r["cache_gbs"],
        "roofline": roof,
        "core_roofline": r["core_roofline"],
        "step_roofline": r["step_roofline"],
        "per_config": rows,
        "per_config_fp8": rows_fp8,
        "e2e": r["e2e"],
        "gpu_launches": 4 * K,
        "stage_us": r["stage_us"],
        "host_enqueue_us_per_step": round(r["host_us"], 2),
        "clocks": r["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, lens, args.cpu_sample_heads)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_full_fold(args, world, rank, local):
    """The full-fold layer: a step appends the new tokens and runs
    mla_decode_full (hidden states in, layer output out). Every stage streams
    from HBM, so the roofline is the whole call's algorithmic bytes (folded
    fp32 weights, cache, activations) over its time. The per-head step on
    the same inputs is timed beside it."""
    import torch
    from mla_latent_kv_73_b300 import _lib, synth
    from mla_latent_kv_73_b300.device_inputs import DeviceWeights, config_for, to_device

    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    _lib.load()
    w = synth.WORKLOADS[args.workload]
    lens = synth.seq_lens(w)
    B, n_q = w.batch, w.n_q
    Tq = B * n_q
    cfg = config_for(w)
    impl = _lib.mla_decode_impl(cfg)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    pt_np, num_blocks = synth.page_table(w, lens)
    cache_bytes, _ = algorithmic(w, lens)
    wts = synth.weights(w)
    raw = {k: to_device(v, w.dtype) for k, v in wts.raw.items()}
    fw = _lib.mla_fold_full(cfg, raw["W_q"], raw["W_uk"], raw["W_uv"], raw["W_o"])
    dw = DeviceWeights(w, wts, cfg)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2000 + rank)
    cache = torch.randn((num_blocks, w.block_size, w.R), generator=gen, device="cuda").to(dt)
    pt = to_device(pt_np, "i32")
    x = torch.randn((Tq, w.d_model), generator=gen, device="cuda").to(dt)
    q = torch.randn((B, n_q, w.n_h, w.d_nope + w.d_r), generator=gen, device="cuda").to(dt)
    seq_lens = to_device(lens, "i32")
    seq_idx = to_device(np.repeat(np.arange(B), n_q).astype(np.int32), "i32")
    pos = to_device(np.concatenate([np.arange(L - n_q, L) for L in lens]).astype(np.int32), "i32")
    y = torch.empty((B, n_q, w.d_model), device="cuda")
    out = torch.empty((B, n_q, w.n_h, w.d_v), device="cuda")
    ws_f = torch.empty(_lib.mla_decode_full_workspace_size(cfg, B, n_q), dtype=torch.uint8,
                       device="cuda")
    ws_h = torch.empty(_lib.mla_decode_workspace_size(cfg, B, n_q, int(lens.sum())),
                       dtype=torch.uint8, device="cuda")

    def full(st):
        _lib.mla_append_kv(cfg, dw.handle, x, seq_idx, pos, pt, cache, st)
        _lib.mla_decode_full(cfg, fw, x.view(B, n_q, w.d_model), cache, pt, seq_lens, y, ws_f, st)

    def per_head(st):
        _lib.mla_append_kv(cfg, dw.handle, x, seq_idx, pos, pt, cache, st)
        _lib.mla_decode(cfg, dw.handle, q, cache, pt, seq_lens, out, ws_h, st)

    stream = torch.cuda.current_stream()
    graphs = {}
    for name, fn in (("full", full), ("per_head", per_head)):
        for _ in range(args.warmup):
            fn(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream())
        graphs[name] = g
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"device error word {code:#x} after warm-up")
    K = args.steps
    times = {}
    clocks = None
    for name in ("per_head", "full"):
        for _ in range(3):
            graphs[name].replay()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            barrier(dist)
            torch.cuda.synchronize()
            wall0 = time.time()
            t0.record()
            for _ in range(K):
                graphs[name].replay()
            t1.record()
            torch.cuda.synchronize()
            barrier(dist)
            wall1 = time.time()
        if name == "full":
            clocks = clk.summary(wall0, wall1)
        times[name] = max_over_ranks(t0.elapsed_time(t1), dist, "cuda") / K
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"device error word {code:#x} in the timed region")
    ms = times["full"]
    folded = 4 * (w.d_model * w.n_h * w.R + w.n_h * w.d_c * w.d_model)
    step_bytes = folded + cache_bytes + (w.R * w.d_model) * w.elem_bytes  # + append's weights
    hbm, _, _, src = measured_peaks()
    achieved = step_bytes / (ms / 1e3) / 1e9
    line = {
        "metric": "full-fold layer tokens/s (hidden state in, layer output out)",
        "variant": "full_fold",
        "value": round(sum_over_ranks(Tq, dist, "cuda") / (ms / 1e3), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) cache rows and hidden states; N(0,1/fan_in) weights)",
        "config": {"workload": w.name, "batch": B, "n_q": n_q, "n_h": w.n_h,
                   "d_model": w.d_model, "d_c": w.d_c, "d_r": w.d_r,
                   "decode_kernel": "tensor_core" if impl == 2 else "cuda_core",
                   "l2": f"one input set; {folded / 2**20:.0f} MiB of folded weights stream "
                         f"through L2 every step"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None, "peak_source": src,
                     "kernel": "mla_decode_full + append (all stages HBM-bound)",
                     "bytes_per_step": step_bytes, "folded_weight_bytes": folded},
        "per_head_ms_per_step": round(times["per_head"], 5),
        "full_over_per_head": round(ms / times["per_head"], 2),
        "clocks": clocks,
    }
    _lib.mla_full_weights_free(fw)
    dw.free()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_layer_step(args, world, rank, local):
    """One layer's decode step (mla_decode_layer: append, decode, W_o
    projection) as a per-layer latency, beside the per-head step (append +
    decode) on the same inputs. Every stage streams from HBM; the roofline is
    the call's algorithmic bytes over its time. W_o (168 MB at DeepSeek-V2
    widths) is larger than L2, so the step's inputs do not stay in L2."""
    import torch
    from mla_latent_kv_73_b300 import _lib, synth
    from mla_latent_kv_73_b300.device_inputs import DeviceWeights, config_for, to_device

    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    _lib.load()
    w = synth.WORKLOADS[args.workload]
    lens = synth.seq_lens(w)
    B, n_q = w.batch, w.n_q
    Tq = B * n_q
    cfg = config_for(w)
    impl = _lib.mla_decode_impl(cfg)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    pt_np, num_blocks = synth.page_table(w, lens)
    cache_bytes, _ = algorithmic(w, lens)
    wts = synth.weights(w)
    dw = DeviceWeights(w, wts, cfg)
    W_o = to_device(wts.raw["W_o"], w.dtype)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(3000 + rank)
    cache = torch.randn((num_blocks, w.block_size, w.R), generator=gen, device="cuda").to(dt)
    pt = to_device(pt_np, "i32")
    x = torch.randn((Tq, w.d_model), generator=gen, device="cuda").to(dt)
    q = torch.randn((B, n_q, w.n_h, w.d_nope + w.d_r), generator=gen, device="cuda").to(dt)
    seq_lens = to_device(lens, "i32")
    seq_idx = to_device(np.repeat(np.arange(B), n_q).astype(np.int32), "i32")
    pos = to_device(np.concatenate([np.arange(L - n_q, L) for L in lens]).astype(np.int32), "i32")
    out = torch.empty((B, n_q, w.n_h, w.d_v), device="cuda")
    y = torch.empty((B, n_q, w.d_model), device="cuda")
    ws_l = torch.empty(_lib.mla_decode_layer_workspace_size(cfg, B, n_q), dtype=torch.uint8,
                       device="cuda")
    ws_h = torch.empty(_lib.mla_decode_workspace_size(cfg, B, n_q, int(lens.sum())),
                       dtype=torch.uint8, device="cuda")

    def layer(st):
        _lib.mla_decode_layer(cfg, dw.handle, W_o, x, seq_idx, pos, q, cache, pt, seq_lens, out,
                              y, ws_l, st)

    def per_head(st):
        _lib.mla_append_kv(cfg, dw.handle, x, seq_idx, pos, pt, cache, st)
        _lib.mla_decode(cfg, dw.handle, q, cache, pt, seq_lens, out, ws_h, st)

    stream = torch.cuda.current_stream()
    graphs = {}
    for name, fn in (("layer", layer), ("per_head", per_head)):
        for _ in range(args.warmup):
            fn(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream())
        graphs[name] = g
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"device error word {code:#x} after warm-up")
    K = args.steps
    times, clocks = {}, None
    for name in ("per_head", "layer"):
        for _ in range(3):
            graphs[name].replay()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            barrier(dist)
            torch.cuda.synchronize()
            wall0 = time.time()
            t0.record()
            for _ in range(K):
                graphs[name].replay()
            t1.record()
            torch.cuda.synchronize()
            barrier(dist)
            wall1 = time.time()
        if name == "layer":
            clocks = clk.summary(wall0, wall1)
        times[name] = max_over_ranks(t0.elapsed_time(t1), dist, "cuda") / K
    st, code = _lib.mla_get_last_device_error(stream)
    if code:
        raise RuntimeError(f"device error word {code:#x} in the timed region")
    ms = times["layer"]
    eb = w.elem_bytes
    weight_bytes = (w.R * w.d_model + 2 * w.n_h * w.d_c * w.d_nope
                    + w.n_h * w.d_v * w.d_model) * eb
    step_bytes = cache_bytes + weight_bytes
    hbm, _, _, src = measured_peaks()
    achieved = step_bytes / (ms / 1e3) / 1e9
    value, _ = whole_job_rate(Tq, ms, dist, "cuda")
    line = {
        "metric": "per-layer decode latency (append + decode + W_o)",
        "variant": "layer",
        "value": round(1e3 * ms, 2),
        "unit": "us per layer step",
        "tokens_per_s": round(value, 1),
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) cache rows, hidden states and queries; "
                "N(0,1/fan_in) weights)",
        "config": {"workload": w.name, "batch": B, "n_q": n_q, "n_h": w.n_h,
                   "d_model": w.d_model, "d_c": w.d_c, "d_r": w.d_r,
                   "decode_kernel": "tensor_core" if impl == 2 else "cuda_core",
                   "l2": f"one input set; W_o alone is {w.n_h * w.d_v * w.d_model * eb / 2**20:.0f}"
                         f" MiB, above L2"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None, "peak_source": src,
                     "kernel": "mla_decode_layer (all stages HBM-bound)",
                     "bytes_per_step": step_bytes},
        "per_head_step_us": round(1e3 * times["per_head"], 2),
        "w_o_projection_us": round(1e3 * (ms - times["per_head"]), 2),
        "clocks": clocks,
    }
    dw.free()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the oracle (CPU) arm
# ---------------------------------------------------------------------------

def oracle_sample(w, lens, n_pairs):
    """The (b, i, h) triples of a bounded oracle sample: whole sequences first."""
    from mla_latent_kv_73_b300 import synth
    trip = [(b, i, h) for b in range(w.batch) for i in range(w.n_q) for h in range(w.n_h)]
    return trip[:n_pairs]


def time_oracle(w, lens, n_pairs):
    from mla_latent_kv_73_b300 import synth
    from oracle import mla_oracle as O
    wts = synth.weights(w)
    qv, _ = synth.queries(w)
    samples = oracle_sample(w, lens, n_pairs)
    need = sorted({b for b, _, _ in samples})
    rows = [None] * w.batch
    for b in need:
        rows[b] = synth.sequence_rows(w, b, lens[b])[0]
    t0 = time.perf_counter()
    O.decode_materialised(qv, rows, lens, wts.W_uk, wts.W_uv, w.d_c, w.d_nope, w.d_v, w.scale,
                          w.rope_base, samples=samples)
    dt = time.perf_counter() - t0
    # a query token is done when all its heads are: tokens = (b,i,h) triples / n_h
    return dt, len(samples) / w.n_h


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def cpu_baseline(w, lens, n_pairs):
    if n_pairs <= 0:
        # calibrate: time one head, then aim for about 10 s
        dt1, _ = time_oracle(w, lens, 1)
        n_pairs = int(min(w.batch * w.n_q * w.n_h, max(w.n_h, 10.0 / max(dt1, 1e-4))))
    dt, toks = time_oracle(w, lens, n_pairs)
    return {"value": round(toks / dt, 4), "unit": "tokens/s", "cores": blas_threads(),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{n_pairs} (sequence, query, head) triples of {w.name} "
                      f"(= {toks:.3f} query tokens), fp64 NumPy, keys/values materialised"}


def run_reference(args, world, rank):
    from mla_latent_kv_73_b300 import synth
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    lens = synth.seq_lens(w)
    dt1, _ = time_oracle(w, lens, 1)
    # each step: a bounded sample sized so that warmup + steps stay within minutes
    per_step_pairs = int(max(1, min(w.n_h, 8.0 / max(dt1, 1e-4))))
    for _ in range(args.warmup):
        time_oracle(w, lens, 1)
    times, toks = [], 0.0
    for _ in range(args.steps if args.steps <= 20 else 20):
        dt, t = time_oracle(w, lens, per_step_pairs)
        times.append(dt)
        toks += t
    total = sum(times)
    value = toks / total
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": world, "steps": len(times), "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "n_q": w.n_q, "n_h": w.n_h},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"{per_step_pairs} (sequence, query, head) triples per step"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def self_launch(n, argv):
    """Run this script on n local ranks through torch.distributed.run (one
    process per GPU, rendezvous on 127.0.0.1). Returns its exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def main():
    args = parse()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(self_launch(args.gpus, sys.argv[1:]))
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.variant == "full_fold":
        run_full_fold(args, world, rank, local)
        return
    if args.variant == "layer":
        run_layer_step(args, world, rank, local)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
