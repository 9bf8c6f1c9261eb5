#!/usr/bin/env python3
"""Benchmark of the quantized MoE decode layer on GB300.

Workload (one step): one forward of the 40-layer stack of 35B-A3B-shaped MoE
FFN layers (H=2048, E=256, top-8, I=512, 6-bit routed experts, 8-bit shared
expert and router, group 64) at M=1 token row, each layer with its own
weights (40 distinct layer sets, 26.3 GB resident in HBM, so L2 cannot hold
the working set).  The stack runs as one persistent kernel launch.

Metric: achieved HBM GB/s on the unique bytes a step touches (each selected
expert once, shared expert, router, gamma, activations) and microseconds per
layer.  M=4 (1 token + 3 correlated draft rows) is reported alongside.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the reference arm of this tier).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer µs/token & achieved HBM GB/s vs 8 TB/s (35B-A3B shape, M=1 and M=4)"
LAYERS = 40
CORR_M4 = 0.6


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--layers", type=int, default=LAYERS)
    p.add_argument("--no-m4", action="store_true", help="M=1 only: no M=4 line and no M sweep")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--routing-out", default=None, help="write per-layer routing statistics (JSON) here")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(v: float, dev=None) -> float:
    """The largest v over the ranks of the default process group (v itself
    when there is no group, or a group of one): the slowest rank's time is the
    job's time."""
    import torch
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()) or td.get_world_size() == 1:
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_step: int, steps: int, seconds: float) -> float:
    """Whole-job throughput of `world` replicas that each processed `steps`
    steps of `bytes_per_step` algorithmic bytes in `seconds` (max over ranks)."""
    return world * bytes_per_step * steps / seconds / 1e9


def unique_bytes(shape, U: int, M: int) -> int:
    """Algorithmic bytes of one layer call (see accounting.unique_bytes)."""
    from quantized_moe_decode_layer_gb300.accounting import unique_bytes as ub
    return ub(shape, U, M)


# The sources of moe_decode_kernel (the kernel the roofline and the traffic
# figure describe): its translation unit and the headers it includes.
KERNEL_SOURCES = ("moe_layer.cu", "moe_internal.h", "moe_unpack.cuh")


def source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_moe_decode_layer_gb300", "csrc")
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source."""
    try:
        t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
        if t.get("source_hash") == source_hash():
            return t
    except Exception:
        pass
    return None


def traffic_for(record, layers: int):
    """The record's DRAM bytes of one stack launch, scaled from its own layer
    count to `layers` (at M=1 every layer reads the same bytes: U = 8 experts
    per layer), or None without a record."""
    if not record:
        return None
    return int(round(record["bytes_per_launch"] * layers / record.get("layers", LAYERS)))


class Clocks:
    """nvidia-smi samples during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = f"/tmp/moe_clocks_{os.getpid()}.csv"

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].isdigit():
                    rows.append(parts)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        mhz = sorted(int(r[1]) for r in rows)
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": int(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows)}


def build_stack(shape, n_layers, dev, seed0=1000):
    import torch
    import synth
    import quantized_moe_decode_layer_gb300 as moe
    desc = moe.desc_from_shape(shape)
    layers = []
    for l in range(n_layers):
        L = synth.make_layer(shape, seed0 + l, device=dev)
        layers.append(moe.Layer(desc, moe.layer_src_from_synth(L)))
        del L
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return desc, layers


def measure_U(layers, x, ws, selections=None):
    """Distinct experts per layer along the stack for input x (untimed).  With
    a list `selections`, appends each layer's expert ids [M, k] (numpy)."""
    import torch
    import quantized_moe_decode_layer_gb300 as moe
    Us = []
    h = x
    for lyr in layers:
        idx, _ = moe.router_topk(lyr, h, ws)
        Us.append(int(torch.unique(idx).numel()))
        if selections is not None:
            selections.append(idx.cpu().numpy())
        h = moe.decode_layer(lyr, h, ws)
    return Us


def routing_stats(selections, E: int):
    """Per-layer distinct experts U, the fraction of them chosen by two or
    more rows, and the expert-selection histogram summed over the layers."""
    import numpy as np
    U, shared, hist = [], [], np.zeros(E, dtype=np.int64)
    for idx in selections:
        ids, counts = np.unique(idx, return_counts=True)
        rows_per = np.array([int((idx == e).any(axis=1).sum()) for e in ids])
        U.append(int(ids.size))
        shared.append(round(float((rows_per >= 2).sum()) / ids.size, 3))
        hist[ids] += counts
    return {"U_per_layer": U, "shared_frac_per_layer": shared, "selection_hist": hist.tolist()}


def percentiles(per_ms):
    """p10 / median / p90 of per-step times (ms)."""
    import numpy as np
    a = np.asarray(per_ms)
    return {"p10_ms": round(float(np.percentile(a, 10)), 5), "median_ms": round(float(np.percentile(a, 50)), 5),
            "p90_ms": round(float(np.percentile(a, 90)), 5), "n": int(a.size)}


def time_stack(st, x, ws, steps, warmup, stream):
    import torch
    import quantized_moe_decode_layer_gb300 as moe
    out = torch.empty_like(x)
    for _ in range(warmup):
        st.forward(x, ws, out=out, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    moe.launch_count(reset=True)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        st.forward(x, ws, out=out, stream=stream)
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    launches = moe.launch_count(reset=True)
    per = sorted(a.elapsed_time(b) for a, b in ev)
    total_ms = t0.elapsed_time(t1)
    assert ws.status(stream) == 0
    return total_ms, per, launches


def tc_measure(layers, desc, shape, dev, M, warmup):
    """Time moe_gate_up_tc over the layer sets for M routed rows: one call per
    layer (its distinct experts with their row masks), CUDA events around the
    whole pass.  Bytes: the gate/up rows of each call's experts once; flops:
    2 * 2I * H per (expert, row) pair."""
    import numpy as np
    import torch
    import synth
    import quantized_moe_decode_layer_gb300 as moe
    ws = moe.Workspace(desc, M)
    x = synth.make_rows(shape, 40 + M, M).to(dev)
    from quantized_moe_decode_layer_gb300.profile_case import tc_routing
    cases = tc_routing(layers, x, ws)
    acts = [torch.zeros((int(ex.numel()), M, shape.I), dtype=torch.float32, device=dev) for ex, _, _ in cases]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(max(1, warmup)):
        for (ex, mk, hn), act, lyr in zip(cases, acts, layers):
            moe.gate_up_tc(lyr, hn, ex, mk, act=act, err=err)
    torch.cuda.synchronize()
    ys = [torch.zeros((int(ex.numel()), M, shape.H), dtype=torch.float32, device=dev) for ex, _, _ in cases]
    for (ex, mk, _), act, y, lyr in zip(cases, acts, ys, layers):
        moe.down_tc(lyr, act, ex, mk, y=y, err=err)
    reps = 5
    a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    a.record()
    for _ in range(reps):
        for (ex, mk, hn), act, lyr in zip(cases, acts, layers):
            moe.gate_up_tc(lyr, hn, ex, mk, act=act, err=err)
    b.record()
    for _ in range(reps):
        for (ex, mk, _), act, y, lyr in zip(cases, acts, ys, layers):
            moe.down_tc(lyr, act, ex, mk, y=y, err=err)
    c.record()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    per_call_s = a.elapsed_time(b) * 1e-3 / (reps * len(layers))
    down_s = b.elapsed_time(c) * 1e-3 / (reps * len(layers))
    U = np.array([int(ex.numel()) for ex, _, _ in cases])
    pairs = np.array([sum(bin(int(m) & 0xFFFFFFFF).count("1") for m in mk.cpu().tolist()) for _, mk, _ in cases])
    unit_bytes = 2 * (shape.H * shape.routed_bits // 8 + shape.H // 64 * 4)
    bytes_call = float(np.mean(U)) * shape.I * unit_bytes
    down_bytes = float(np.mean(U)) * shape.H * (shape.I * shape.routed_bits // 8 + shape.I // 64 * 4)
    flops_call = float(np.mean(pairs)) * 2 * (2 * shape.I) * shape.H
    return {"M": M, "us_per_call": round(per_call_s * 1e6, 3), "mean_U": round(float(np.mean(U)), 2),
            "rows_per_expert": round(float(np.mean(pairs / U)), 2),
            "gbs": round(bytes_call / per_call_s / 1e9, 1), "tflops": round(flops_call / per_call_s / 1e12, 2),
            "down_us_per_call": round(down_s * 1e6, 3),
            "down_gbs": round(down_bytes / down_s / 1e9, 1),
            "calls": reps * len(layers)}


def qkv_measure(shape, dev, n_sets, warmup):
    """Time moe_qkv_forward over n_sets distinct projections.  One pass over
    the sets is captured in a CUDA graph (the calls are a few microseconds
    each, shorter than a Python-side launch), replayed, and timed with CUDA
    events; bytes = the packed rows of a call (read once) plus its input and
    output."""
    import torch
    import quantized_moe_decode_layer_gb300 as moe
    import synth
    H, rows = shape.H, (4096, 512, 512)
    sets = []
    for i in range(n_sets):
        g = torch.Generator(device=dev).manual_seed(7000 + i)
        mats = [synth.quant_matrix(g, (n,), H, 8, dev) for n in rows]
        sets.append(moe.QKV(H, *mats, bits=8))
        del mats
    torch.cuda.empty_cache()
    res = {}
    for M in (1, 4):
        x = synth.make_rows(shape, 60 + M, M).to(dev)
        y = torch.empty((M, sum(rows)), dtype=torch.float32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            for _ in range(max(1, warmup)):
                for q in sets:
                    q.forward(x, out=y, err=err)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for q in sets:
                q.forward(x, out=y, err=err)
        graph.replay()
        torch.cuda.synchronize()
        reps = 10
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        per = a.elapsed_time(b) * 1e-3 / (reps * len(sets))
        nbytes = sets[0].nbytes + x.numel() * 2 + y.numel() * 4
        res[str(M)] = {"us_per_call": round(per * 1e6, 3), "gbs": round(nbytes / per / 1e9, 1),
                       "bytes_per_call": nbytes, "calls": reps * len(sets), "timing": "CUDA graph replay"}
        del graph
    res["shape"] = "H 2048, Q 4096 + K 512 + V 512 rows, 8-bit groups of 64"
    del sets
    torch.cuda.empty_cache()
    return res


def attn_measure(dev, peaks, warmup):
    """Time moe_attn_decode (16 query heads, 2 KV heads, head dim 256, bf16
    cache) at a 32K-position cache (64 MB of keys and values: L2 could hold
    it, so a 256 MB buffer is written before every call) and at 128K
    positions (256 MB, above L2), for 1 and 3 rows.  Each call is timed with
    CUDA events on its own stream around the replay of a CUDA graph of the
    call (its two kernels go out together; timing the Python-level call
    would count the host's tensor-map encoding and launches while the GPU
    waits); bytes = the valid keys and values (read once) plus the queries
    and the fp32 output."""
    import torch
    import quantized_moe_decode_layer_gb300 as moe
    import synth
    res = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream()
    for T, do_flush, calls in ((32768, True, 40), (131072, False, 40)):
        q_all, k, vt = synth.make_attn(T, T, 3, 5, device=dev)
        cache = moe.AttnCache(T, device=dev)
        cache.k.copy_(k)
        cache.vt.copy_(vt)
        del k, vt
        for M in (1, 3):
            q = q_all[:M].contiguous()
            out = torch.empty((M, 16, 256), dtype=torch.float32, device=dev)
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            with torch.cuda.stream(st):
                for _ in range(max(3, warmup)):
                    cache.attend(q, T - M, out=out, err=err, stream=st)
            st.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=st):
                cache.attend(q, T - M, out=out, err=err, stream=st)
            evs = []
            with torch.cuda.stream(st):
                for _ in range(3):
                    graph.replay()
                for _ in range(calls):
                    if do_flush:
                        flush.fill_(1)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(st)
                    graph.replay()
                    b.record(st)
                    evs.append((a, b))
            st.synchronize()
            assert int(err.item()) == 0
            ts = sorted(a.elapsed_time(b) * 1e-3 for a, b in evs)
            per = sum(ts) / len(ts)
            nbytes = T * 2 * 256 * 2 * 2 + M * 16 * 256 * (2 + 4)
            res[f"T{T}_M{M}"] = {"us_per_call": round(per * 1e6, 2), "median_us": round(ts[len(ts) // 2] * 1e6, 2),
                                 "gbs": round(nbytes / per / 1e9, 1),
                                 "frac": round(nbytes / per / 1e9 / peaks["hbm_gbs"], 4),
                                 "bytes_per_call": nbytes, "calls": calls,
                                 "l2": "256 MB written before each call" if do_flush else "cache > L2",
                                 "timing": "CUDA graph replay, one call per replay"}
        del cache
        torch.cuda.empty_cache()
    res["shape"] = "16 query heads, 2 KV heads, head dim 256, bf16 cache, chunks of 512 positions"
    return res


def streamed_measure(shape, dev, peaks, n_layers=8, n_slots=16, tokens=24, warm_tokens=4, corr=0.6):
    """moe_streamed_forward over n_layers streamed layers (experts in pinned
    host memory, an HBM cache of n_slots experts per layer) for a sequence of
    token rows, x_{t+1} = a x_t + sqrt(1 - a^2) n_t (a = corr), with and
    without next-layer prediction.  Reports wall time per layer (the runtime
    waits for each layer's routing on the host), cache hits, the bytes
    fetched over the host link and their rate, and the share of selected
    experts the prediction named."""
    import math
    import torch
    import quantized_moe_decode_layer_gb300 as moe
    import synth
    desc = moe.desc_from_shape(shape)
    res = {"layers": n_layers, "slots_per_layer": n_slots, "tokens": tokens, "token_correlation": corr,
           "host_blob_GB": None}
    g = torch.Generator().manual_seed(123)
    xs = [torch.randn(shape.H, generator=g)]
    for _ in range(warm_tokens + tokens - 1):
        xs.append(corr * xs[-1] + math.sqrt(1 - corr * corr) * torch.randn(shape.H, generator=g))
    zc = synth.zipf_component(shape).float()
    xs = [(x + zc).to(torch.bfloat16).view(1, -1).to(dev) for x in xs]
    ws = moe.Workspace(desc, 1)
    cs = torch.cuda.Stream()
    for predict in (False, True):
        st = []
        for l in range(n_layers):
            lay = moe.Layer(desc, moe.layer_src_from_synth(synth.make_layer(shape, 5000 + l, device=dev)))
            st.append(moe.StreamedLayer(lay, n_slots=n_slots))
            del lay
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        res["host_blob_GB"] = round(sum(s.host.numel() for s in st) / 1e9, 2)
        out = torch.empty_like(xs[0])
        for t in range(warm_tokens):
            moe.streamed_forward(st, xs[t], ws, out=out, predict=predict, copy_stream=cs)
        torch.cuda.synchronize()
        before = [s.stats() for s in st]
        t0 = time.perf_counter()
        for t in range(warm_tokens, warm_tokens + tokens):
            moe.streamed_forward(st, xs[t], ws, out=out, predict=predict, copy_stream=cs)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert ws.status() == 0
        after = [s.stats() for s in st]
        d = {k: sum(a[k] - b[k] for a, b in zip(after, before)) for k in after[0]}
        sel = d["hits"] + d["misses"]
        res["predict" if predict else "lru_only"] = {
            "us_per_layer": round(dt / (tokens * n_layers) * 1e6, 2),
            "tokens_per_s": round(tokens / dt, 1),
            "hit_rate": round(d["hits"] / max(1, sel), 4),
            "fetched_experts_per_token": round(d["fetched"] / tokens, 2),
            "fetched_GB_per_s": round(d["bytes"] / dt / 1e9, 2),
            "prediction_named": round(d["predicted_used"] / max(1, sel), 4) if predict else None}
        del st
        torch.cuda.empty_cache()
    return res


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as td
    import synth
    import quantized_moe_decode_layer_gb300 as moe

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        td.init_process_group("nccl", device_id=dev)
    shape = synth.A35B
    desc, layers = build_stack(shape, args.layers, dev)
    st = moe.Stack(layers)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            td.barrier()
        torch.cuda.synchronize()

    # M = 1 (headline)
    x1 = synth.make_rows(shape, 5, 1, gamma=None).to(dev)
    ws = moe.Workspace(desc, 4)
    sel1 = []
    U1 = measure_U(layers, x1, ws, sel1)
    routing = {"M1": routing_stats(sel1, shape.E)}
    bytes1 = sum(unique_bytes(shape, u, 1) for u in U1)
    barrier()
    with Clocks(local) as clk:
        barrier()
        total_ms, per, launches = time_stack(st, x1, ws, args.steps, args.warmup, stream)
        barrier()
    clocks = clk.summary()
    total_ms = reduce_max(total_ms, dev)
    ms_step = total_ms / args.steps
    value = whole_job_gbs(world, bytes1, args.steps, total_ms * 1e-3)
    us_layer = ms_step * 1e3 / args.layers

    # roofline of the dominant (only) kernel: one launch per step
    peaks, peak_kind = load_peaks()
    med_ms = per[len(per) // 2]
    mean_ms = sum(per) / len(per)
    achieved = bytes1 / (mean_ms * 1e-3) / 1e9
    traffic = load_traffic()
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_kind": peak_kind,
            "traffic": traffic_for(traffic, args.layers),
            "algorithmic_bytes": bytes1, "launch_ms_mean": round(mean_ms, 5), "launch_ms_median": round(med_ms, 5)}
    # the launch-time distribution over at least 200 launches (after the
    # timed region, so the timed region stays exactly `steps` steps)
    if args.steps >= 200:
        roof["launch_percentiles"] = percentiles(per)
    else:
        _, per_more, _ = time_stack(st, x1, ws, 200, 2, stream)
        roof["launch_percentiles"] = percentiles(per_more)

    # end to end through the C ABI with host buffers (copies inside the call)
    xh = x1.cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    for _ in range(args.warmup):
        st.forward_host(xh, oh, ws)
    e_steps = max(10, args.steps // 4)
    barrier()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        st.forward_host(xh, oh, ws)
    e_s = time.perf_counter() - t0
    e_s = reduce_max(e_s, dev)
    e2e = {"value": round(whole_job_gbs(world, bytes1, e_steps, e_s), 1), "unit": "GB/s",
           "h2d_bytes_per_step": int(x1.numel() * 2), "d2h_bytes_per_step": int(x1.numel() * 2),
           "us_per_layer": round(e_s / e_steps * 1e6 / args.layers, 3)}

    # M = 4: one token + 3 correlated draft rows
    m4 = None
    if not args.no_m4:
        x4 = synth.make_rows(shape, 6, 4, correlation=CORR_M4).to(dev)
        sel4 = []
        U4 = measure_U(layers, x4, ws, sel4)
        routing["M4"] = routing_stats(sel4, shape.E)
        bytes4 = sum(unique_bytes(shape, u, 4) for u in U4)
        s4 = max(200, args.steps // 2)
        tm4, per4, l4 = time_stack(st, x4, ws, s4, args.warmup, stream)
        mean4 = sum(per4) / len(per4)
        m4 = {"us_per_layer": round(tm4 / s4 * 1e3 / args.layers, 3),
              "gbs": round(bytes4 / (mean4 * 1e-3) / 1e9, 1),
              "frac": round(bytes4 / (mean4 * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
              "mean_U": round(float(np.mean(U4)), 2), "bytes_per_step": bytes4,
              "rows": "1 token + 3 draft rows, correlation %.1f at the stack input" % CORR_M4,
              "shared_frac_layer0": routing["M4"]["shared_frac_per_layer"][0],
              "launches_per_step": l4 / s4, "percentiles": percentiles(per4)}

    # the stack over M in {1, 2, 4, 8, 16, 32} independent token rows: up to 8
    # rows one persistent launch per step; above, grouped mode (each selected
    # expert read once per group of up to 32 rows, its products on the
    # tensor cores); 32 rows also on the FMA path alone (4 launches of 8 rows)
    sweep = None
    if not args.no_m4:
        sweep = {}
        wsw = moe.Workspace(desc, 32)
        R = min(8, 16384 // shape.H)
        for M, key, grouped in ((1, "1", 1), (2, "2", 1), (4, "4", 1), (8, "8", 1), (16, "16", 1),
                                (16, "16_fma", 0), (32, "32", 1), (32, "32_fma", 0)):
            moe.set_grouped(grouped)
            try:
                xm = synth.make_rows(shape, 40 + M, M).to(dev)
                selm = []
                Um = measure_U(layers, xm, wsw, selm)
                if key == "32":
                    routing["M32"] = routing_stats(selm, shape.E)
                bm = sum(unique_bytes(shape, u, M) for u in Um)
                sm = max(10, args.steps // 10)
                tmm, perm, lm = time_stack(st, xm, wsw, sm, args.warmup, stream)
            finally:
                moe.set_grouped(1)
            s_step = tmm / sm * 1e-3
            sweep[key] = {"tokens_per_s": round(M / s_step, 1), "us_per_layer": round(s_step * 1e6 / args.layers, 3),
                          "gbs": round(bm / s_step / 1e9, 1), "mean_U": round(float(np.mean(Um)), 2),
                          "mode": "grouped" if (M > R and grouped and M >= grouped) else "persistent",
                          "launches_per_step": lm / sm}
        del wsw

    # the grouped gate/up on the tensor cores (moe_gate_up_tc) for the M=32
    # rows' experts, layer after layer over the 40 layer sets (2 GB of gate/up
    # weights in all, so L2 holds none of a call's weights from the call before)
    tc = None
    if not args.no_m4:
        tc = {str(M): tc_measure(layers, desc, shape, dev, M, args.warmup) for M in (8, 32)}

    # the fused Q/K/V projection (8-bit, Q 16 heads x 256, K and V 2 heads x
    # 256 over H = 2048) over 40 distinct weight sets (445 MB, L2 cannot hold
    # them), one call per set, at 1 and 4 rows
    qkv = None
    if not args.no_m4:
        qkv = qkv_measure(shape, dev, args.layers, args.warmup)

    # the split-K decode attention with grouped query heads
    attn = None
    if not args.no_m4:
        attn = attn_measure(dev, peaks, args.warmup)

    # streamed layers: experts in host memory behind an HBM cache
    streamed = None
    if not args.no_m4:
        streamed = streamed_measure(shape, dev, peaks)

    # the 397B-shaped layer at M=1: a stack over 15 distinct layer sets (55 GB)
    b397 = None
    if not args.no_m4:
        shb = synth.B397
        descb, layb = build_stack(shb, 15, dev, seed0=3000)
        stb = moe.Stack(layb)
        xb = synth.make_rows(shb, 8, 1).to(dev)
        wsb = moe.Workspace(descb, 1)
        Ub = measure_U(layb, xb, wsb)
        bb = sum(unique_bytes(shb, u, 1) for u in Ub)
        sb = max(20, args.steps // 4)
        tmb, perb, _ = time_stack(stb, xb, wsb, sb, args.warmup, stream)
        meanb = sum(perb) / len(perb)
        b397 = {"layers": 15, "us_per_layer": round(tmb / sb * 1e3 / 15, 3),
                "gbs": round(bb / (meanb * 1e-3) / 1e9, 1),
                "frac": round(bb / (meanb * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "resident_weight_GB": round(sum(l.nbytes for l in layb) / 1e9, 2), "bytes_per_step": bb}
        del stb, layb, wsb
        torch.cuda.empty_cache()

    # single-layer calls (one launch per layer) over the 40 rotating layer sets
    single = None
    if rank == 0:
        out = torch.empty_like(x1)
        for lyr in layers[:4]:
            moe.decode_layer(lyr, x1, ws, out=out)
        torch.cuda.synchronize()
        reps = 5
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            for lyr in layers:
                moe.decode_layer(lyr, x1, ws, out=out)
        b.record()
        torch.cuda.synchronize()
        single = round(a.elapsed_time(b) * 1e3 / (reps * len(layers)), 3)

    if rank == 0 and args.routing_out:
        with open(args.routing_out, "w") as f:
            json.dump({"workload": f"a35b stack, {args.layers} layer sets", **routing}, f)
    cpu = cpu_baseline(args, shape, dev) if rank == 0 else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"35B-A3B-shaped MoE FFN stack, {args.layers} distinct layer sets, M=1",
                       "H": 2048, "E": 256, "k": 8, "I": 512, "I_shared": 512, "routed_bits": 6,
                       "shared_bits": 8, "router_bits": 8, "group": 64, "M": 1, "layers": args.layers,
                       "resident_weight_GB": round(sum(l.nbytes for l in layers) / 1e9, 2),
                       "l2": (f"weights rotate over {args.layers} layer sets "
                              f"({sum(l.nbytes for l in layers) / 1e9:.1f} GB) > L2; no flush"),
                       "parallelism": f"replicas x{world}"},
            "us_per_layer": round(us_layer, 3), "fraction_of_8TBs": round(value / world / 8000.0, 4),
            "single_layer_call_us": single, "m4": m4, "sweep": sweep, "tc_gate_up": tc, "b397": b397, "qkv": qkv,
            "attn": attn, "streamed": streamed,
            "roofline": roof, "e2e": e2e,
            "gpu_launches": launches, "launches_per_step": launches / args.steps, "clocks": clocks,
            "cpu_baseline": cpu,
            "routing": {k: {"mean_U": round(float(np.mean(v["U_per_layer"])), 2),
                            "U_per_layer": v["U_per_layer"]} for k, v in routing.items()},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        td.barrier()
        td.destroy_process_group()


def host_cpu():
    """(logical cores, CPU model name) of this host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return os.cpu_count(), model or "unknown"


def cpu_baseline(args, shape, dev=None):
    """The oracle, as it stands, on a bounded sample of the workload: chained
    layers of the stack at M=1 in fp64, first on one host core (the parity
    reference), then the same layer calls again with the oracle's mat-vec
    output rows spread over every host core (OpenMP; the same bits), cycling
    over the prepared layers until its time budget is spent."""
    import numpy as np
    import torch
    import oracle
    import synth
    cores, model = host_cpu()
    budget1, budget_all = args.cpu_seconds * 2 / 3, args.cpu_seconds / 3
    x = synth.bf16_bits(synth.make_rows(shape, 5, 1)).numpy().view(np.uint16)
    calls = []   # (oracle layer, its input, unique bytes)
    n1, b1, e1 = 0, 0, 0.0
    oracle.set_threads(1)
    l = 0
    while e1 < budget1 and l < args.layers:
        L = synth.make_layer(shape, 1000 + l, device=dev if dev is not None else "cpu")
        lay = oracle.Layer(L)
        r = lay.route(x)
        for e in set(int(v) for v in r["idx"].ravel()):
            lay.expert(e)
        del L
        if dev is not None:
            torch.cuda.empty_cache()
        t0 = time.perf_counter()
        res = lay.forward(x, normed=False)
        e1 += time.perf_counter() - t0
        ub = unique_bytes(shape, len(set(res["idx"].ravel().tolist())), 1)
        b1 += ub
        n1 += 1
        calls.append((lay, x, ub))
        x = res["out"]
        l += 1
    nthreads = oracle.max_threads()
    nm, bm, em = 0, 0, 0.0
    oracle.set_threads(nthreads)
    try:
        while em < budget_all:
            lay, xin, ub = calls[nm % len(calls)]
            t0 = time.perf_counter()
            lay.forward(xin, normed=False)
            em += time.perf_counter() - t0
            bm += ub
            nm += 1
    finally:
        oracle.set_threads(1)
    return {"value": round(b1 / e1 / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n1} chained layers of the a35b stack at M=1 ({e1:.1f} s of oracle time)",
            "us_per_layer": round(e1 / n1 * 1e6, 1), "host_cores": cores, "cpu_model": model,
            "all_cores": {"value": round(bm / em / 1e9, 6), "unit": "GB/s", "cores": nthreads,
                          "sample": f"{nm} layer calls cycling over those {len(calls)} layers "
                                    f"({em:.1f} s of oracle time)",
                          "us_per_layer": round(em / nm * 1e6, 1)}}


def oracle_steps(shape, n_layers, steps, warmup, dev=None, prepared=4):
    """The oracle, as it stands, stepped like the bench: one step is one layer
    of the stack at M=1 (fp64, one host core).  `prepared` distinct layer sets
    are built first (the stack's first layers, the input chained through them
    once, untimed); step s runs layer s mod `prepared` on its chained input.
    `warmup` steps are untimed, then exactly `steps` steps are timed."""
    import numpy as np
    import torch
    import oracle
    import synth
    P = max(1, min(prepared, n_layers))
    x = synth.bf16_bits(synth.make_rows(shape, 5, 1)).numpy().view(np.uint16)
    lays, xs, ubytes = [], [], []
    for l in range(P):
        L = synth.make_layer(shape, 1000 + l, device=dev if dev is not None else "cpu")
        lay = oracle.Layer(L)
        del L
        if dev is not None:
            torch.cuda.empty_cache()
        res = lay.forward(x, normed=False)
        lays.append(lay)
        xs.append(x)
        ubytes.append(unique_bytes(shape, len(set(res["idx"].ravel().tolist())), 1))
        x = res["out"]
    for s in range(warmup):
        lays[s % P].forward(xs[s % P], normed=False)
    done = 0
    t0 = time.perf_counter()
    for s in range(steps):
        lays[s % P].forward(xs[s % P], normed=False)
        done += ubytes[s % P]
    elapsed = time.perf_counter() - t0
    return {"value": round(done / elapsed / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps} timed steps of one {shape.name} layer at M=1 each, cycling over the stack's first {P} "
                      f"layer sets ({elapsed:.1f} s of oracle time, {warmup} untimed warm-up steps)",
            "s_per_step": elapsed / max(1, steps)}


def run_reference(args):
    """The reference arm: the oracle on the host cores, on this arm's metric
    and unit.  Under torchrun only rank 0 runs it; the other ranks exit."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    import synth
    import torch
    dev = None
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
    cb = oracle_steps(synth.A35B, args.layers, args.steps, args.warmup, dev)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(cb["s_per_step"] * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"35B-A3B-shaped MoE FFN stack, {args.layers} distinct layer sets, M=1",
                       "M": 1, "layers": args.layers, "step": "one layer of the stack (a bounded sample)"},
            "cpu_baseline": {k: v for k, v in cb.items() if k != "s_per_step"},
            "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
