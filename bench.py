"""Benchmark of the NVFP4 paged-KV decode hot path on GB300.

One step = the hot path of one serving step over one batch: the NVFP4
quantized write of the step's new tokens and the paged GQA decode attention
over the whole batch (plus the chunked-extend pass where the workload has one).
Default workload: mixed28_b70 (the 28-layer mixed-precision model, layers 0,
25, 26, 27 in FP8 and the rest NVFP4, 70 sequences x 4096 tokens, 32 q / 8 KV
heads, head_dim 128, page 64, per-channel lognormal scales), the largest
single-GPU decode configuration.  The same line carries, measured in the same
run, the NVFP4 decode roofline and FP8 ratio of longctx_b2_ctx128k (2 x 131072
tokens, 64 split-KV partitions) and serving_mix_b256 (256 ragged sequences
plus a chunked-extend pass), and pass/fail against the targets (decode at
>= 75 % of 8 TB/s, step >= 1.5x faster than the FP8 cache).

Prints ONE JSON line (rank 0).  ``value`` is the algorithmic HBM throughput of
the step (GB/s; bytes of NVFP4/FP8 K/V codes + scales read, Q read, output
written, new tokens read and their codes written) over the device-timed step;
``roofline`` times the NVFP4 layers' decode calls alone;
``e2e`` is the same metric with the step's inputs copied from pinned host
memory and the output copied back inside the timed region (one copy in and
one copy out per layer and step, on two copy streams, each ordered against
its layer's step by events so that copies overlap other layers' steps).  The FP8-KV
variant of the same workload is timed beside it as the comparator.  Between
timed steps the caches rotate over replicas whose total exceeds L2.

Multi-GPU: replicas only (one independent copy of the workload per rank, no
collective on the data path); the barrier and max-over-ranks timing use
torch.distributed.

--workload extend_b4_chunk2k: the chunked-extend pass instead (the chunk's
FP8 workspace append and the causal FP8 extend attention), metric TFLOP/s.

--workload prefill_write_b4_16k: the initial-prefill write (FP8 K/V
requantized into the NVFP4 cache), metric HBM GB/s.

--workload capacity_mixed28: equal-memory capacity (the page pool admits as
many 4096-token sequences as the KV budget of 44 all-FP8 ones holds, under
FP8 / mixed / NVFP4 layer maps) and the 28-layer decode step at each batch.

--workload calibration_study: the synthetic calibration study (attention
output error of NVFP4 / FP8 caches against FP32, global-scale factors).

--impl reference: the CPU oracle (scalar C, one thread) on a bounded sample of
the same workload, as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 paged decode attn: HBM GB/s & % of 8 TB/s peak; decode tokens/s"
NOMINAL_HBM_GBS = 8000.0
DEFAULT_WORKLOAD = "mixed28_b70"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, rank, ws, local
    return None, rank, ws, local


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, x, device):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(dist, x, device):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.path = index, None, None

    def __enter__(self):
        self.path = os.path.join("/tmp", f"nvkv_clocks_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
        try:
            rows = [l.split(",") for l in open(self.path).read().strip().splitlines() if l.strip()]
            sm = [float(r[0]) for r in rows]
            out["sm_mhz"] = statistics.median(sm) if sm else None
            out["sm_max_mhz"] = float(rows[0][1]) if rows else None
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for j, n in enumerate(names):
                if any(r[2 + j].strip().lower() == "active" for r in rows):
                    out["reasons"].append(n)
            out["samples"] = len(rows)
        except Exception:
            pass
        return out


def _graph(fn):
    """A CUDA graph of fn()'s launches (captured on a side stream)."""
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            fn()
    torch.cuda.current_stream().wait_stream(cs)
    torch.cuda.synchronize()
    return g


def _steps_fn(sets, steps):
    """The launches of `steps` steps, rotating over the cache replicas: per
    layer the step (the new tokens' write and the decode, one launch with one
    new token per sequence) and the extend pass (where the workload has one)."""
    def fn():
        for i in range(steps):
            for lay in sets[i % len(sets)]:
                lay.step()
    return fn


def _time_graph(g, stream, label="bench_timed"):
    """Device time of one replay of g (ms), CUDA events on `stream`.  The
    replay sits in an NVTX range (`label`) so a profiler can keep only the
    timed launches (ncu --nvtx --nvtx-include "bench_timed/")."""
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push(label)
    t0.record(stream)
    g.replay()
    t1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def step_bytes(lay) -> dict:
    """Algorithmic bytes of one step of one layer."""
    s = lay.wl.spec
    kv = lay.kv_bytes_read()
    qo = lay.qo_bytes()
    per_tok_write = (144 if lay.prec == 0 else 256)
    w = 0
    if lay.k_new is not None:
        n = lay.k_new.shape[0] * s.Hkv
        w += n * (2 * 128 * 4 + per_tok_write)
    if lay.ext is not None:
        rows = int(lay.ext["prefix_lens"].sum().item()) * s.Hkv
        w += rows * (144 + 256)                                    # workspace dequant: read NVFP4, write FP8
        n = lay.ext["k"].shape[0] * s.Hkv
        w += n * (2 * 128 * 4 + per_tok_write)
        if "q" in lay.ext:  # chunk append (FP32 in, E4M3 out); the attention's work is FLOPs, not counted here
            w += n * (2 * 128 * 4 + 256)
    return dict(kv=kv, qo=qo, write=w, total=kv + qo + w)


DTYPE = ("QK^T: tcgen05 kind::mxf4nvf4 block-scaled MMA on the stored E2M1 codes and E4M3 scales of K, the BF16 "
         "query written as 8 NVFP4 terms (6 at 8 heads per KV head; FP8 layers: kind::f8f6f4, 4 E4M3 terms), "
         "FP32 accumulate; softmax FP32; P.V: f16 x f16 -> f32 mma.sync on V dequantized exactly to f16")
HEADLINE = "mixed28_b70"
EXTRA_WORKLOADS = ("longctx_b2_ctx128k", "serving_mix_b256")
TARGET_FRAC_OF_8TBPS = 0.75
TARGET_FP8_SPEEDUP = 1.5


def workload_config(spec, ws=1, extend_attention=False):
    """The `config` dict of a decode workload (both arms print the same one)."""
    return {
        "workload": spec.name, "B": spec.B, "Hq": spec.Hq, "Hkv": spec.Hkv, "D": spec.D,
        "L": spec.L or "ragged (lognormal)", "page": spec.P, "layers": spec.layers,
        "fp8_layers": list(spec.fp8_layers), "step_write_tokens_per_seq": spec.step_write,
        "extend": {"seqs": list(spec.extend_seqs), "tokens": spec.extend_tokens,
                   "attention": bool(extend_attention)} if spec.extend_seqs else None,
        "l2": "inputs rotate over cache replicas totalling >= 3x L2 (or one set larger than that)",
        "parallelism": f"replicas x{ws}",
        "launch": "one CUDA graph of the K timed steps",
    }


def _build_sets(wl, layers, dev, l2, prec=None, extend_attention=False):
    """Cache replicas of the workload's layers whose total exceeds 3x L2."""
    from nvfp4_quantized_paged_gb300.runner import Layer
    mk = lambda l: Layer(wl, l, dev, prec=prec, extend_attention=extend_attention)
    first = [mk(l) for l in layers]
    per = sum(step_bytes(x)["kv"] for x in first)
    reps = max(1, -(-3 * l2 // max(per, 1)))
    return [first] + [[mk(l) for l in layers] for _ in range(reps - 1)]


def _decode_graph(sets, steps, keep):
    """A graph of `steps` rounds of decode calls on the layers `keep` selects."""
    def fn():
        for i in range(steps):
            for lay in sets[i % len(sets)]:
                if keep(lay):
                    lay.decode()
    return _graph(fn)


def measure_workload(name, args, dev, dist, stream, full=True):
    """Device-timed step, NVFP4 decode roofline and FP8 comparator of one
    workload (and, with full=True, the e2e step through the C ABI)."""
    import nvfp4_quantized_paged_gb300 as nv
    from nvfp4_quantized_paged_gb300.workloads import SPECS, Workload
    spec = SPECS[name]
    wl = Workload(spec, seed=0, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    layers = list(range(spec.layers)) if not args.layers else [int(x) for x in args.layers.split(",")]
    sets = _build_sets(wl, layers, dev, l2, extend_attention=args.extend_attention)
    bytes_step = sum(step_bytes(x)["total"] for x in sets[0])
    nv_layers = [x for x in sets[0] if x.prec == nv.PREC_NVFP4]
    dec_bytes = sum(x.kv_bytes_read() + x.qo_bytes() for x in nv_layers)  # per round of NVFP4 decodes

    for i in range(args.warmup):
        for lay in sets[i % len(sets)]:
            lay.step()
    torch.cuda.synchronize()
    # The timed region replays one CUDA graph of the K steps: eager launches
    # cost more host time than their GPU time and would leave the GPU idle
    # between kernels.  A second graph of the NVFP4 layers' decode calls alone
    # (same replicas, same stream) gives the decode kernel's own duration.
    g_step = _graph(_steps_fn(sets, args.steps))
    g_dec = _decode_graph(sets, args.steps, lambda x: x.prec == nv.PREC_NVFP4)
    g_step.replay()  # untimed: uploads the graphs
    g_dec.replay()
    torch.cuda.synchronize()
    _barrier(dist)
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = "0"
    with Clocks(gpu_id) as clk:
        step_ms = _time_graph(g_step, stream)
        dec_total_ms = _time_graph(g_dec, stream)
    _barrier(dist)
    ms = _max_over_ranks(dist, step_ms / args.steps, dev)
    dec_avg_ms = dec_total_ms / (args.steps * max(1, len(nv_layers)))
    # per layer: the step (write + decode, one launch, split-KV merge inside)
    # and (serving mix) the prefix dequant and the extend write
    launches_per_step = sum(x.launches_per_step() for x in sets[0])
    del g_step, g_dec
    res = dict(spec=spec, ms=ms, bytes_step=bytes_step, launches_per_step=launches_per_step, clocks=clk.summary(),
               dec_avg_us=dec_avg_ms * 1e3, dec_bytes_per_launch=dec_bytes / max(1, len(nv_layers)),
               nv_layers=len(nv_layers), l2=l2, extend_attention=args.extend_attention)
    res["dec_gbs"] = res["dec_bytes_per_launch"] / (dec_avg_ms * 1e-3) / 1e9

    if full:
        # e2e: inputs from pinned host memory, output back to the host, through
        # the C ABI.  A layer's step inputs (queries, new K/V, their slots) live
        # in one device buffer that the layer's tensors view, so a step copies
        # them in with one host-to-device copy and the output back with one copy.
        def stage(lay):
            parts = lay.step_inputs()
            sizes = [t.numel() * t.element_size() for t in parts]
            buf = torch.empty(sum(sizes), dtype=torch.uint8, device=dev)
            views, off = [], 0
            for t, n in zip(parts, sizes):  # each part's size is a multiple of 16 bytes but the last
                v = buf[off:off + n].view(t.dtype).view(t.shape)
                v.copy_(t)
                views.append(v)
                off += n
            lay.set_step_inputs(views)
            return buf

        bufs = [[stage(lay) for lay in lays] for lays in sets]
        host = [dict(inp=b.cpu().pin_memory(), out=torch.empty(lay.out.shape, dtype=lay.out.dtype).pin_memory())
                for b, lay in zip(bufs[0], sets[0])]
        h2d = sum(h["inp"].numel() for h in host)
        d2h = sum(h["out"].numel() * 2 for h in host)

        # The copies run on two copy streams, a layer's input copy and its
        # output copy ordered against that layer's step by events, so the
        # copies of one layer overlap the steps of the others (as a serving
        # loop pipelines them).  Every step still copies every input in and
        # every output out inside the timed region.
        h2d_stream, d2h_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        in_free = [[None] * len(host) for _ in sets]   # the layer's last step that read this input buffer
        out_free = [[None] * len(host) for _ in sets]  # the copy-out that last read this output

        def e2e_step(i):
            r = i % len(sets)
            ready = []
            with torch.cuda.stream(h2d_stream):
                for j, (buf, h) in enumerate(zip(bufs[r], host)):
                    if in_free[r][j] is not None:
                        h2d_stream.wait_event(in_free[r][j])
                    buf.copy_(h["inp"], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(h2d_stream)
                    ready.append(ev)
            for j, (lay, h) in enumerate(zip(sets[r], host)):
                stream.wait_event(ready[j])
                if out_free[r][j] is not None:
                    stream.wait_event(out_free[r][j])
                lay.step()
                ev = torch.cuda.Event()
                ev.record(stream)
                in_free[r][j] = ev
                with torch.cuda.stream(d2h_stream):
                    d2h_stream.wait_event(ev)
                    h["out"].copy_(lay.out, non_blocking=True)
                    ev_out = torch.cuda.Event()
                    ev_out.record(d2h_stream)
                    out_free[r][j] = ev_out

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        _barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)  # no copy of the timed steps starts before the region does
        for i in range(args.steps):
            e2e_step(i)
        stream.wait_stream(d2h_stream)  # the region ends after the last copy-out
        e1.record(stream)
        torch.cuda.synchronize()
        res.update(e2e_ms=_max_over_ranks(dist, e0.elapsed_time(e1) / args.steps, dev), h2d=h2d, d2h=d2h)
        del bufs, host

    # FP8-KV comparator: the same workload with every layer in FP8
    res["fp8_ms"] = res["fp8_dec_us"] = None
    if not args.no_fp8:
        del sets
        torch.cuda.empty_cache()
        fsets = _build_sets(wl, layers, dev, l2, prec=nv.PREC_FP8)
        for i in range(args.warmup):
            for lay in fsets[i % len(fsets)]:
                lay.step()
        torch.cuda.synchronize()
        fg = _graph(_steps_fn(fsets, args.steps))
        fd = _decode_graph(fsets, args.steps, lambda x: x.layer in {y.layer for y in nv_layers})
        fg.replay()
        fd.replay()
        torch.cuda.synchronize()
        res["fp8_ms"] = _max_over_ranks(dist, _time_graph(fg, stream) / args.steps, dev)
        res["fp8_dec_us"] = _time_graph(fd, stream) / (args.steps * max(1, len(nv_layers))) * 1e3
        del fg, fd, fsets
    torch.cuda.empty_cache()
    return res


def _targets(res):
    frac8 = res["dec_gbs"] / NOMINAL_HBM_GBS
    sp = None if res["fp8_ms"] is None else res["fp8_ms"] / res["ms"]
    return {"decode_frac_of_8TBps": round(frac8, 4), "decode_ge_75pct_of_8TBps": bool(frac8 >= TARGET_FRAC_OF_8TBPS),
            "step_speedup_over_fp8": None if sp is None else round(sp, 3),
            "fp8_speedup_ge_1.5": None if sp is None else bool(sp >= TARGET_FP8_SPEEDUP)}


def _extra_line(res, peak):
    """The decode roofline and FP8 ratio of an extra workload (same run)."""
    return {
        "config": workload_config(res["spec"], 1, res["extend_attention"]),
        "ms_per_step": round(res["ms"], 5),
        "step_gbs": round(res["bytes_step"] / (res["ms"] * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "kernel": "decode_kernel<NVFP4>", "achieved": round(res["dec_gbs"], 1),
                     "peak": peak, "unit": "GB/s", "frac": round(res["dec_gbs"] / peak, 4),
                     "traffic": _traffic_from_profile(res["spec"].name),
                     "algorithmic_bytes_per_launch": int(res["dec_bytes_per_launch"]),
                     "avg_launch_us": round(res["dec_avg_us"], 3)},
        "fp8_comparator": None if res["fp8_ms"] is None else {
            "ms_per_step": round(res["fp8_ms"], 5), "speedup_nvfp4_over_fp8": round(res["fp8_ms"] / res["ms"], 3),
            "decode_us": round(res["fp8_dec_us"], 3),
            "decode_speedup_nvfp4_over_fp8": round(res["fp8_dec_us"] / res["dec_avg_us"], 3)},
        "targets": _targets(res),
        "clocks": res["clocks"],
    }


def run_ours(args):
    dist, rank, ws, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import nvfp4_quantized_paged_gb300 as nv
    nv.lib()
    stream = torch.cuda.current_stream()
    res = measure_workload(args.workload, args, dev, dist, stream, full=True)
    spec = res["spec"]
    peak, peak_kind = _peaks()
    extras = {}
    if not args.no_extra and args.workload == HEADLINE:
        for name in EXTRA_WORKLOADS:
            extras[name] = _extra_line(measure_workload(name, args, dev, dist, stream, full=False), peak)
    total_bytes = _sum_over_ranks(dist, float(res["bytes_step"]), dev)
    ms = res["ms"]
    gbs = total_bytes / (ms * 1e-3) / 1e9
    traffic = _traffic_from_profile(args.workload)
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(gbs, 1),
            "unit": "GB/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": DTYPE,
            "data": "synthetic (seeded; no dataset or weights)",
            "config": workload_config(spec, ws, args.extend_attention),
            "pct_of_8TBps": round(100.0 * gbs / ws / NOMINAL_HBM_GBS, 2),
            "pct_of_measured_hbm": round(100.0 * gbs / ws / peak, 2),
            "decode_tokens_per_s": round(_sum_over_ranks(dist, spec.B, dev) / (ms * 1e-3), 1),
            "us_per_layer": round(ms * 1e3 / spec.layers, 2),
            "e2e": {"value": round(total_bytes / (res["e2e_ms"] * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "ms_per_step": round(res["e2e_ms"], 5), "h2d_bytes_per_step": int(res["h2d"]),
                    "d2h_bytes_per_step": int(res["d2h"])},
            "gpu_launches": int(res["launches_per_step"] * args.steps),
            "roofline": {"bound": "hbm", "kernel": "decode_kernel<NVFP4> (split-KV merge in the same launch)",
                         "achieved": round(res["dec_gbs"], 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(res["dec_gbs"] / peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": int(res["dec_bytes_per_launch"]),
                         "avg_launch_us": round(res["dec_avg_us"], 3),
                         "layers_timed": f"the {res['nv_layers']} NVFP4 layers",
                         "timed": "CUDA events around one graph of K rounds of the NVFP4 layers' decode calls "
                                  "(one launch each), cache replicas rotated"},
            "fp8_comparator": None if res["fp8_ms"] is None else {
                "ms_per_step": round(res["fp8_ms"], 5), "speedup_nvfp4_over_fp8": round(res["fp8_ms"] / ms, 3),
                "decode_us": round(res["fp8_dec_us"], 3),
                "decode_speedup_nvfp4_over_fp8": round(res["fp8_dec_us"] / res["dec_avg_us"], 3)},
            "targets": _targets(res),
            "clocks": res["clocks"],
        }
        if extras:
            line["extra_workloads"] = extras
            ok_frac = [line["targets"]["decode_ge_75pct_of_8TBps"]] + [
                e["targets"]["decode_ge_75pct_of_8TBps"] for e in extras.values()]
            ok_fp8 = [line["targets"]["fp8_speedup_ge_1.5"]] + [e["targets"]["fp8_speedup_ge_1.5"] for e in extras.values()]
            line["targets_summary"] = {"decode_ge_75pct_of_8TBps_all": all(ok_frac),
                                       "fp8_speedup_ge_1.5_all": all(x is True for x in ok_fp8)}
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(spec, args.workload, budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


EXTEND_METRIC = "chunked-extend FP8 attention: TFLOP/s (causal, algorithmic)"


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 burst; f16 has the same dense rate)"
    except Exception:
        return 1900.0, "fallback"


def extend_flops(prefixes, chunks, Hq, D=128):
    """Algorithmic FLOPs of the causal extend attention: query j of a chunk
    over prefix p sees p + j + 1 keys; QK^T and P.V each 2 D per key and head."""
    keys = sum(p * c + c * (c + 1) // 2 for p, c in zip(prefixes, chunks))
    return 4 * D * Hq * keys


def run_extend(args):
    """The chunked-extend pass of one layer: the chunk's K/V appended to the
    FP8 workspace behind the (already dequantized) prefix, then the causal
    FP8 attention of the chunk's queries over [prefix || chunk]."""
    dist, rank, ws, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import nvfp4_quantized_paged_gb300 as nv
    from nvfp4_quantized_paged_gb300.workloads import EXTEND_SPECS, extend_inputs
    nv.lib()
    c = EXTEND_SPECS[args.workload]
    x = extend_inputs(0, **c)
    Hq, Hkv = c["Hq"], c["Hkv"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    k_all = torch.from_numpy(x["k"]).to(dev)
    v_all = torch.from_numpy(x["v"]).to(dev)
    ws_scale = torch.zeros(2, dtype=torch.float32, device=dev)
    nv.nvkv_global_scale(k_all, ws_scale[0:1], nv.FP8_GLOBAL_DIVISOR)
    nv.nvkv_global_scale(v_all, ws_scale[1:2], nv.FP8_GLOBAL_DIVISOR)
    ci = torch.from_numpy(x["chunk_idx"]).to(dev)
    k_chunk, v_chunk = k_all[ci].contiguous(), v_all[ci].contiguous()
    chunk_rows = torch.from_numpy(x["chunk_rows"]).to(dev)
    cu_q = torch.from_numpy(x["cu_q"]).to(dev)
    cu_kv = torch.from_numpy(x["cu_kv"]).to(dev)
    kv_lens = torch.from_numpy(x["kv_lens"]).to(dev)
    max_q = max(c["chunks"])
    per = 6 * x["ws_rows"] * Hkv * 128 + x["q"].numel() * 2  # FP8 workspace, its FP16 tiles, queries
    reps = max(2, -(-3 * l2 // per))  # workspace + queries rotate over >= 3x L2
    sets = []
    for _ in range(reps):
        wk = torch.zeros(x["ws_rows"], Hkv, 128, dtype=torch.uint8, device=dev)
        wv = torch.zeros_like(wk)
        nv.fp8_workspace_append_chunk(k_all, v_all, torch.from_numpy(x["rows"]).to(dev), ws_scale, wk, wv)
        sets.append(dict(wk=wk, wv=wv, q=x["q"].to(dev), scratch=nv.alloc_extend_scratch(wk),
                         out=torch.empty(x["q"].shape, dtype=torch.bfloat16, device=dev)))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def attend(r):
        nv.fp8_chunked_extend_attention(r["q"], cu_q, max_q, r["wk"], r["wv"], cu_kv, kv_lens, ws_scale, r["out"],
                                        r["scratch"], err=err)

    def step(i):
        r = sets[i % reps]
        nv.fp8_workspace_append_chunk(k_chunk, v_chunk, chunk_rows, ws_scale, r["wk"], r["wv"], err=err)
        attend(r)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert err.item() == 0, err.item()
    g_step = _graph(lambda: [step(i) for i in range(args.steps)])
    g_att = _graph(lambda: [attend(sets[i % reps]) for i in range(args.steps)])
    g_step.replay()
    g_att.replay()
    torch.cuda.synchronize()
    _barrier(dist)
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    with Clocks(gpu_id) as clk:
        step_ms = _time_graph(g_step, stream) / args.steps
        att_ms = _time_graph(g_att, stream) / args.steps
    _barrier(dist)
    ms = _max_over_ranks(dist, step_ms, dev)
    del g_step, g_att
    flops = extend_flops(c["prefixes"], c["chunks"], Hq)
    # e2e: the chunk's K/V and queries from pinned host memory, the output back
    hk, hv = k_chunk.cpu().pin_memory(), v_chunk.cpu().pin_memory()
    hq = x["q"].pin_memory()
    hout = torch.empty(x["q"].shape, dtype=torch.bfloat16).pin_memory()
    dk, dv = torch.empty_like(k_chunk), torch.empty_like(v_chunk)

    def e2e_step(i):
        r = sets[i % reps]
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        r["q"].copy_(hq, non_blocking=True)
        nv.fp8_workspace_append_chunk(dk, dv, chunk_rows, ws_scale, r["wk"], r["wv"], err=err)
        attend(r)
        hout.copy_(r["out"], non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(dist, e0.elapsed_time(e1) / args.steps, dev)
    peak, peak_kind = _tensor_peak()
    tot = _sum_over_ranks(dist, float(flops), dev)
    if rank == 0:
        line = {
            "metric": EXTEND_METRIC, "value": round(tot / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f16xf16->f32 (E4M3 K/V exact in f16, BF16 queries in f16, P in f16)",
            "data": "synthetic (seeded; no dataset or weights)",
            "config": {"workload": args.workload, "prefixes": list(c["prefixes"]), "chunks": list(c["chunks"]),
                       "Hq": Hq, "Hkv": Hkv, "D": 128,
                       "l2": f"workspace and queries rotate over {reps} replicas (>= 3x L2, {l2 >> 20} MiB)",
                       "parallelism": f"replicas x{ws}", "launch": "one CUDA graph of the K timed steps"},
            "e2e": {"value": round(tot / (e2e_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 5),
                    "h2d_bytes_per_step": int(hk.numel() * 4 * 2 + hq.numel() * 2),
                    "d2h_bytes_per_step": int(hout.numel() * 2)},
            "gpu_launches": 3 * args.steps,
            "roofline": {"bound": "tensor", "kernel": "extend_attention_kernel (+ its tile expansion)",
                         "unit": "TFLOP/s",
                         "achieved": round(flops / (att_ms * 1e-3) / 1e12, 1), "peak": peak, "peak_kind": peak_kind,
                         "frac": round(flops / (att_ms * 1e-3) / 1e12 / peak, 4), "traffic": None,
                         "algorithmic_flops_per_launch": int(flops), "avg_launch_us": round(att_ms * 1e3, 2),
                         "timed": "CUDA events around one graph of K attention calls (tile expansion + "
                                  "attention kernel), replicas rotated"},
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = extend_cpu_baseline(x, ws_scale.cpu().numpy(), Hq, budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def extend_cpu_baseline(x, ws_scale, Hq, budget_s=10.0):
    """The oracle (scalar C, 1 thread) on a bounded sample: single queries
    of the last sequence, each a one-query problem over its visible keys."""
    import oracle
    wk = np.zeros((x["ws_rows"], x["k"].shape[1], 128), np.uint8)
    wv = np.zeros_like(wk)
    oracle.fp8_workspace_append(wk, wv, x["k"], x["v"], x["rows"], ws_scale)
    qb = x["q"].view(torch.int16).numpy().view(np.uint16)
    i = len(x["chunks"]) - 1
    done, t, nq = 0, 0.0, 0
    for j in range(0, x["chunks"][i], 97):
        pos = x["prefixes"][i] + j
        row = int(x["cu_q"][i]) + j
        t0 = time.perf_counter()
        oracle.fp8_extend_attention(qb[row:row + 1], [0, 1], wk, wv, [int(x["cu_kv"][i])], [pos + 1], ws_scale)
        t += time.perf_counter() - t0
        done += 4 * 128 * Hq * (pos + 1)
        nq += 1
        if t >= budget_s:
            break
    return {"value": round(done / t / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{nq} queries (all heads) of the last sequence, {t:.1f} s", "cpu": _cpu_name(),
            "host_cores": os.cpu_count()}


PREFILL_METRIC = "prefill FP8 -> NVFP4 requantize-write: HBM GB/s"
PREFILL_SPECS = {"prefill_write_b4_16k": dict(tokens=4 * 16384, Hkv=8, P=64)}


def run_prefill_write(args):
    """The initial-prefill write: FP8 K/V of a batch of prompts (4 x 16384
    tokens, 8 KV heads) requantized into the NVFP4 paged cache."""
    dist, rank, ws, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import nvfp4_quantized_paged_gb300 as nv
    nv.lib()
    c = PREFILL_SPECS[args.workload]
    T, Hkv, P = c["tokens"], c["Hkv"], c["P"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per = T * Hkv * (2 * 128 + 144)
    reps = max(2, -(-3 * l2 // per))
    sets = []
    for _ in range(reps):
        k = torch.randn(T, Hkv, 128, device=dev, generator=gen)
        v = torch.randn(T, Hkv, 128, device=dev, generator=gen)
        s8 = torch.stack([k.abs().max(), v.abs().max()]).float() / 448.0
        k8 = (k / s8[0]).to(torch.float8_e4m3fn).view(torch.uint8)  # the prefill's FP8 K/V (input)
        v8 = (v / s8[1]).to(torch.float8_e4m3fn).view(torch.uint8)
        g = torch.zeros(2, dtype=torch.float32, device=dev)
        nv.nvkv_global_scale((k8.view(torch.float8_e4m3fn).float() * s8[0]).contiguous(), g[0:1], nv.NVFP4_GLOBAL_DIVISOR)
        nv.nvkv_global_scale((v8.view(torch.float8_e4m3fn).float() * s8[1]).contiguous(), g[1:2], nv.NVFP4_GLOBAL_DIVISOR)
        cache = nv.Cache(nv.PREC_NVFP4, T // P, Hkv, P, device=dev, kv_scale=g)
        pages = torch.randperm(T // P, device=dev, generator=gen)  # each prompt fills its pages in order,
        t = torch.arange(T, device=dev)                              # the pages themselves permuted
        slots = pages[t // P] * P + t % P
        sets.append(dict(k8=k8, v8=v8, s8=s8, g=g, cache=cache, slots=slots))
        del k, v
    stream = torch.cuda.current_stream()

    def step(i):
        r = sets[i % reps]
        nv.nvfp4_kv_requantize_write_fp8(r["k8"], r["v8"], r["s8"], r["slots"], r["g"], r["cache"])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    g_step = _graph(lambda: [step(i) for i in range(args.steps)])
    g_step.replay()
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    with Clocks(gpu_id) as clk:
        ms = _time_graph(g_step, stream) / args.steps
    ms = _max_over_ranks(dist, ms, dev)
    # e2e: FP8 K/V from pinned host memory, a cache page block back
    hk, hv = sets[0]["k8"].cpu().pin_memory(), sets[0]["v8"].cpu().pin_memory()
    hb = torch.empty(sets[0]["cache"].data[0].shape, dtype=torch.uint8).pin_memory()

    def e2e_step(i):
        r = sets[i % reps]
        r["k8"].copy_(hk, non_blocking=True)
        r["v8"].copy_(hv, non_blocking=True)
        step(i)
        hb.copy_(r["cache"].data[0], non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    peak, peak_kind = _peaks()
    gbs = per / (ms * 1e-3) / 1e9
    if rank == 0:
        line = {"metric": PREFILL_METRIC, "value": round(ws * gbs, 1), "unit": "GB/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32 (E4M3 decode x scale, NVFP4 quantizer)",
                "data": "synthetic (seeded N(0,1) K/V quantized to FP8 by torch as the input)",
                "config": {"workload": args.workload, "tokens": T, "Hkv": Hkv, "D": 128, "page": P,
                           "l2": f"inputs and caches rotate over {reps} replicas (>= 3x L2)",
                           "parallelism": f"replicas x{ws}", "launch": "one CUDA graph of the K timed steps"},
                "e2e": {"value": round(per / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                        "h2d_bytes_per_step": int(hk.numel() * 2), "d2h_bytes_per_step": int(hb.numel())},
                "gpu_launches": args.steps,
                "roofline": {"bound": "hbm", "kernel": "nvfp4_requant_kernel", "achieved": round(gbs, 1),
                             "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(gbs / peak, 4),
                             "traffic": _prefill_traffic(args.workload), "algorithmic_bytes_per_launch": int(per),
                             "avg_launch_us": round(ms * 1e3, 2),
                             "timed": "CUDA events around one graph of K write launches, replicas rotated"},
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


CAPACITY_METRIC = "decode tokens/s at equal KV-cache memory (28-layer model, 44 FP8 sequences' budget)"
CAPACITY_SPECS = {"capacity_mixed28": dict(base="mixed28_b44", fp8_sequences=44)}


def run_capacity(args):
    """Equal-memory capacity: the KV budget of 44 all-FP8 sequences (4096
    tokens, 28 layers) handed to the library's page pool under three
    precision maps (all FP8, the mixed map with layers 0, 25, 26, 27 in FP8,
    all NVFP4); as many sequences as the pool holds are admitted and the
    28-layer decode step (quantized write + decode per layer) is timed at
    that batch."""
    dist, rank, ws, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import nvfp4_quantized_paged_gb300 as nv
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import SPECS, Workload, scaled
    nv.lib()
    c = CAPACITY_SPECS[args.workload]
    base = SPECS[c["base"]]
    layers, P, Hkv, L = base.layers, base.P, base.Hkv, base.L
    pps = -(-L // P)
    budget = c["fp8_sequences"] * pps * layers * nv.nvkv_cache_page_bytes(nv.PREC_FP8, P, Hkv)
    maps = {"fp8": tuple(range(layers)), "mixed": tuple(base.fp8_layers), "nvfp4": ()}
    stream = torch.cuda.current_stream()
    res = {}
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    with Clocks(gpu_id) as clk:
        for name, fp8_layers in maps.items():
            prec_map = [nv.PREC_FP8 if l in fp8_layers else nv.PREC_NVFP4 for l in range(layers)]
            npages = nv.nvkv_pool_pages_for_budget(budget, prec_map, P, Hkv)
            pool = nv.PagePool(npages)
            tables = []
            while True:
                ids = pool.alloc(pps)
                if ids is None:
                    break
                tables.append(ids)
            B = len(tables)
            wl = Workload(scaled(base, name=f"capacity_{name}", B=B, fp8_layers=fp8_layers), seed=0, device=dev)
            wl.block_table = np.array(tables, np.int32)  # the pool's pages
            wl.num_pages = npages
            lays = [Layer(wl, l, dev) for l in range(layers)]
            for _ in range(args.warmup):
                for x in lays:
                    x.step()
            torch.cuda.synchronize()
            g = _graph(_steps_fn([lays], args.steps))
            g.replay()
            torch.cuda.synchronize()
            ms = _max_over_ranks(dist, _time_graph(g, stream) / args.steps, dev)
            kv = sum(step_bytes(x)["total"] for x in lays)
            res[name] = {"sequences": B, "pages": npages, "cache_bytes": int(sum(x.cache.nbytes for x in lays)),
                         "ms_per_step": round(ms, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
                         "step_gbs": round(kv / (ms * 1e-3) / 1e9, 1)}
            del g, lays, wl, pool
            torch.cuda.empty_cache()
    peak, peak_kind = _peaks()
    if rank == 0:
        m = res["mixed"]
        line = {"metric": CAPACITY_METRIC, "value": round(ws * m["tokens_per_s"], 1), "unit": "tokens/s",
                "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": DTYPE,
                "data": "synthetic (seeded; no dataset or weights)",
                "config": {"workload": args.workload, "layers": layers, "Hkv": Hkv, "Hq": base.Hq, "L": L, "page": P,
                           "kv_budget_bytes": int(budget), "mixed_fp8_layers": list(base.fp8_layers),
                           "parallelism": f"replicas x{ws}", "launch": "one CUDA graph of the K timed steps",
                           "l2": "caches of 10 GB per map (far above L2)"},
                "capacity": res,
                "vs_fp8": {k: {"sequences": round(v["sequences"] / res["fp8"]["sequences"], 3),
                               "tokens_per_s": round(v["tokens_per_s"] / res["fp8"]["tokens_per_s"], 3)}
                           for k, v in res.items()},
                "gpu_launches": layers * args.steps,  # one decode-step launch per layer
                "roofline": {"bound": "hbm", "kernel": "28-layer decode step (one write + decode launch per layer), mixed map",
                             "achieved": m["step_gbs"], "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                             "frac": round(m["step_gbs"] / peak, 4), "traffic": None},
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


CALIB_METRIC = "attention-output relative L2 error vs FP32, NVFP4 cache at the amax/2688 global scale (element outliers)"


def run_calibration(args):
    """The synthetic calibration study (nvfp4_quantized_paged_gb300.calibration):
    one JSON line, the table of errors under `rows`."""
    dist, rank, ws, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import nvfp4_quantized_paged_gb300 as nv
    from nvfp4_quantized_paged_gb300.calibration import study
    nv.lib()
    t0 = time.perf_counter()
    rows = study(device=dev)
    elapsed = time.perf_counter() - t0
    main = next(r for r in rows if r["dist"] == "element_outliers" and r["prec"] == "nvfp4" and r["factor"] == 1.0)
    if rank == 0:
        line = {"metric": CALIB_METRIC, "value": round(main["rel_l2"], 6), "unit": "relative L2", "n_gpus": ws,
                "steps": 1, "warmup": 0, "ms_per_step": round(elapsed * 1e3, 1), "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32 kernels vs f32 torch reference",
                "data": "synthetic (seeded; four value distributions)",
                "config": {"workload": args.workload, "B": 4, "L": 4096, "Hq": 32, "Hkv": 8, "D": 128,
                           "factors": [0.25, 0.5, 1.0, 2.0, 4.0]},
                "rows": rows}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


DECODE_SOURCES = ("decode.cu", "nvkv_device.cuh", "nvkv_host.h")
WRITE_SOURCES = ("quantize.cu", "nvkv_device.cuh", "nvkv_host.h")


def decode_sources_sha256(names=DECODE_SOURCES):
    """Hash of a kernel's sources (the kernel file and the headers it includes)."""
    import hashlib
    h = hashlib.sha256()
    for name in names:
        h.update(open(os.path.join(ROOT, "nvfp4_quantized_paged_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def _prefill_traffic(workload):
    """DRAM bytes per prefill-write launch from the committed ncu summary, if it
    was taken on the current write kernel sources (else None)."""
    try:
        prof = json.load(open(os.path.join(ROOT, "profiles", f"prefill_write_{workload}.json")))
        if prof.get("write_sources_sha256") != decode_sources_sha256(WRITE_SOURCES):
            return None
        return prof.get("dram_bytes_per_launch")
    except Exception:
        return None


def _traffic_from_profile(workload):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"decode_nvfp4_{workload}.json")
    try:
        prof = json.load(open(path))
        if prof.get("decode_sources_sha256") != decode_sources_sha256():
            return None
        return prof.get("dram_bytes_per_launch")
    except Exception:
        return None


def cpu_baseline(spec, workload, budget_s=15.0):
    """The oracle (scalar C, 1 thread) on a bounded sample: whole sequences of
    the workload, each = its step write + decode attention over all heads."""
    import oracle
    from nvfp4_quantized_paged_gb300.workloads import Workload
    wl = Workload(spec, seed=0, device="cpu")
    per_tok = 144
    layer = next(l for l in range(spec.layers) if not wl.is_fp8(l))  # an NVFP4 layer
    done_bytes, t_total, seqs = 0, 0.0, 0
    for b in range(spec.B):
        L = int(wl.seq_lens[b])
        k = wl.kv(layer, 0, b).numpy()
        v = wl.kv(layer, 1, b).numpy()
        g = np.array([oracle.global_scale(k), oracle.global_scale(v)], np.float32)
        npages = (L + spec.P - 1) // spec.P
        c = oracle.Cache(oracle.PREC_NVFP4, npages, spec.Hkv, spec.P, spec.D, g)
        t = np.arange(L)
        oracle.quantize_write(c, k[:L], v[:L], (t // spec.P) * spec.P + t % spec.P)
        bt = np.arange(npages, dtype=np.int32)[None]
        q = wl.q_bf16(layer)[b:b + 1].view(torch.int16).numpy().view(np.uint16)
        nw = max(spec.step_write, 0)
        t0 = time.perf_counter()
        if nw:
            tt = np.arange(L - nw, L)
            oracle.quantize_write(c, k[L - nw:L], v[L - nw:L], (tt // spec.P) * spec.P + tt % spec.P)
        oracle.paged_decode_attention(c, q, bt, np.array([L], np.int32))
        t_total += time.perf_counter() - t0
        done_bytes += L * spec.Hkv * per_tok + 2 * spec.Hq * spec.D * 2 + nw * spec.Hkv * (2 * 128 * 4 + per_tok)
        seqs += 1
        if t_total >= budget_s:
            break
    return {"value": round(done_bytes / t_total / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{seqs} of {spec.B} sequences of NVFP4 layer {layer} (step write + decode of all heads), "
                      f"{t_total:.1f} s",
            "cpu": _cpu_name(), "host_cores": os.cpu_count()}


def _cpu_name():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from nvfp4_quantized_paged_gb300.workloads import EXTEND_SPECS, SPECS, extend_inputs
    if args.workload in EXTEND_SPECS:  # the oracle's extend attention on bounded samples
        c = EXTEND_SPECS[args.workload]
        x = extend_inputs(0, **c)
        ws_scale = np.array([np.abs(x["k"]).max() / 448.0, np.abs(x["v"]).max() / 448.0], np.float32)
        t0 = time.perf_counter()
        vals = [extend_cpu_baseline(x, ws_scale, c["Hq"], budget_s=args.cpu_budget / max(1, args.steps))
                for _ in range(args.steps)]
        elapsed = time.perf_counter() - t0
        v = statistics.median(cb["value"] for cb in vals)
        print(json.dumps({"metric": EXTEND_METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": round(1e3 * elapsed / args.steps, 3),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f64 (oracle attention)", "data": "synthetic (seeded)", "impl": "reference",
                          "config": {"workload": args.workload, **{k: list(v2) if isinstance(v2, tuple) else v2
                                                                   for k, v2 in c.items()}},
                          "cpu_baseline": dict(vals[-1], value=v),
                          "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    if args.workload not in SPECS:
        print(json.dumps({"impl": "reference", "unavailable": f"no oracle arm for the {args.workload} measurement"}),
              flush=True)
        return
    spec = SPECS[args.workload]
    # each step: a bounded oracle sample of the workload
    for _ in range(args.warmup):
        pass
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cb = cpu_baseline(spec, args.workload, budget_s=args.cpu_budget / max(1, args.steps))
        vals.append(cb["value"])
    elapsed = time.perf_counter() - t0
    v = statistics.median(vals)
    line = {"metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * elapsed / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle attention), f32 (oracle quantizer)",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": workload_config(spec, 1, args.extend_attention),
            "cpu_baseline": dict(cb, value=v),
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline only: skip the long-context and serving-mix keys")
    ap.add_argument("--layers", default="", help="comma list of layer indices to build (profiling runs)")
    ap.add_argument("--extend-attention", action="store_true",
                    help="serving mix: the extend pass also appends the chunk and runs its FP8 attention")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from nvfp4_quantized_paged_gb300.workloads import EXTEND_SPECS
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in EXTEND_SPECS:
        run_extend(args)
    elif args.workload in PREFILL_SPECS:
        run_prefill_write(args)
    elif args.workload in CAPACITY_SPECS:
        run_capacity(args)
    elif args.workload == "calibration_study":
        run_calibration(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
