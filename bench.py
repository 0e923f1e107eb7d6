#!/usr/bin/env python
"""Benchmark of one decode step of the paged, absorbed MLA path on GB300.

A step is one pass of the whole path over one batch (one attention layer):
  mla_absorb_q -> mla_decode_paged (+ split combine) -> mla_out_proj
Default workload: multi-token (speculative) decode with a causal mask, the
largest single-GPU configuration of the path (B = 132 sequences, s_q = 2 query
tokens each, 128 heads, every cache_seqlen 4096, 64-token bf16 pages, d_c 512 +
rope 64), on seeded synthetic inputs (no datasets or trained weights exist here).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-workloads]

The split schedule (mla_get_metadata) depends only on cache_seqlens: a model
computes it once per decoding step and shares it between its layers, so it is
built once per input set outside the timed loop and timed on its own
(`metadata_us`); the end-to-end loop (`e2e`) still builds it every step.

Prints one JSON line on rank 0. `value` is microseconds per step (lower is
better); with N > 1 every rank runs its own replica of the workload (the path
shards by sequence with no collective) and the step time is the max over ranks.
Inputs stay resident in HBM; several independent input sets (one per emulated
layer) rotate so that the bytes touched between two uses of a set exceed
twice the L2 size, so the KV cache streams from HBM.

The timed region is one CUDA graph of the K steps' C-ABI calls (captured on
a stream of its own from pre-marshalled arguments after the warm-up steps,
replayed once untimed), so that the host's launch cost and jitter stay out of
a device-timed number; CUDA events bracket the region. The decode call's
launch duration (the roofline of the dominant kernel) comes from a second
graph of decode calls alone, bracketed the same way. The `workloads` object
repeats that decode-only measurement on the other named workloads (DeepSeek-V3
batch 128 x 512 tokens, variable lengths, long context), each with its own
rotating input sets, roofline bound and fraction. `e2e` repeats the step
through the same C ABI with the step's inputs copied from pinned host buffers
and the result copied back and read by the host every step. `--impl
reference` times the CPU oracle (the reference implementation of this path)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged MLA decode µs/call, achieved HBM GB/s & TFLOPS vs GB300 roofline"
UNIT = "us/call"
WORKLOAD = "spec"
DECODE_WORKLOADS = ["dsv3", "varlen", "long"]
Q8_WORKLOADS = ["dsv3", "varlen", "long", "spec"]  # decode-only lines over the INT8 cache
FLOP_PER_PAIR = 2 * (576 + 512)          # score + value MACs per visible (query row, key)
FLOP_PROJ_PER_ROW = 2 * 128 * 512        # absorb or out-proj MACs per (b, s, h), x2 flops


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--sets", type=int, default=0, help="input sets to rotate (0: enough to exceed 2x L2)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--profile", action="store_true", help="short run for a profiler: no clocks, e2e or cpu leg")
    p.add_argument("--eager", action="store_true", help="time eager C-ABI calls instead of replaying a CUDA graph")
    p.add_argument("--no-workloads", action="store_true", help="skip the decode-only lines of the other workloads")
    p.add_argument("--decode-calls", type=int, default=400, help="decode calls per workload in `workloads`")
    p.add_argument("--prefill-only", action="store_true",
                   help="time only the prefill workload and print its object (a short run for a profiler)")
    p.add_argument("--prefill-batch", type=int, default=8, help="prompts in the prefill workload")
    p.add_argument("--prefill-calls", type=int, default=5)
    p.add_argument("--int8", action="store_true",
                   help="with --profile: the step decodes over the INT8 cache (mla_decode_paged_q8)")
    return p.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------- distributed --

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("MLA_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# -------------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _strip_comments(src):
    """C++ source without its comments, whitespace runs collapsed to one space
    (string and character literals kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_code_sha256():
    """sha256 of the decode kernel's code (csrc/decode.cu followed by
    csrc/ptx.cuh, comments removed and whitespace collapsed), the key under
    which a traffic capture is recorded: a comment edit keeps it, any code
    change voids it."""
    import hashlib
    h = hashlib.sha256()
    for name in ("decode.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "mla_paged_kv_absorbed_gb300", "csrc", name)) as f:
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()


def recorded_traffic(workload):
    """DRAM bytes (read + write) per decode_kernel launch on `workload` from the
    committed ncu summary, or None when there is none or the kernel code
    changed since that capture."""
    path = os.path.join(ROOT, "profiles", f"decode_traffic_{workload}.txt")
    try:
        vals = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
        if kernel_code_sha256() != vals.get("code_sha256"):
            return None
        return int(vals["dram_bytes_read"]) + int(vals["dram_bytes_write"])
    except Exception:
        return None


# --------------------------------------------------------------- our kernels --

class StepArgs:
    """Pre-marshalled C-ABI arguments of one step over one resident input set.
    Decode-only workloads (q_abs drawn directly) have no absorb or out-proj."""

    def __init__(self, api, inp, num_parts, workspace, stream_ptr, q8=None):
        import torch
        d = inp
        self.inp = d
        B, s_q, H = d.B, d.s_q, d.H
        dev = d.kv_cache.device
        self.tm = torch.empty((num_parts, 8), dtype=torch.int32, device=dev)
        self.ns = torch.empty((B + 1,), dtype=torch.int32, device=dev)
        self.q_abs = d.q_abs if d.q is None else torch.empty((B, s_q, H, 576), dtype=torch.bfloat16, device=dev)
        self.o_lat = torch.empty((B, s_q, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, s_q, H), dtype=torch.float32, device=dev)
        self.out = torch.empty((B, s_q, H, 128), dtype=torch.bfloat16, device=dev) if d.w_uv is not None else None
        P = ctypes.c_void_p
        st = P(stream_ptr)
        self.meta = (P(d.seqlens.data_ptr()), B, s_q, H, 1, num_parts, P(self.tm.data_ptr()), P(self.ns.data_ptr()), st)
        self.absorb = None if d.q is None else (P(d.q.data_ptr()), P(d.w_uk.data_ptr()), P(self.q_abs.data_ptr()),
                                                B, s_q, H, st)
        self.decode = (P(self.q_abs.data_ptr()), P(d.kv_cache.data_ptr()), d.kv_cache.shape[0],
                       P(d.block_table.data_ptr()), d.block_table.shape[1], P(d.seqlens.data_ptr()), B, s_q, H,
                       P(self.tm.data_ptr()), P(self.ns.data_ptr()), num_parts, ctypes.c_float(d.scale),
                       int(d.causal), P(self.o_lat.data_ptr()), P(self.lse.data_ptr()), P(workspace.data_ptr()),
                       workspace.numel(), st)
        self.proj = None if self.out is None else (P(self.o_lat.data_ptr()), P(d.w_uv.data_ptr()),
                                                   P(self.out.data_ptr()), B, s_q, H, st)
        # INT8 cache (records, scales) of the same input set, when given
        self.q8 = q8
        self.decode_q8 = None if q8 is None else (
            P(self.q_abs.data_ptr()), P(q8[0].data_ptr()), P(q8[1].data_ptr()), d.kv_cache.shape[0],
            P(d.block_table.data_ptr()), d.block_table.shape[1], P(d.seqlens.data_ptr()), B, s_q, H,
            P(self.tm.data_ptr()), P(self.ns.data_ptr()), num_parts, ctypes.c_float(d.scale), int(d.causal),
            P(self.o_lat.data_ptr()), P(self.lse.data_ptr()), P(workspace.data_ptr()), workspace.numel(), st)


def run_step(L, a: StepArgs, ev=None, meta=False):
    rc = L.mla_get_metadata(*a.meta) if meta else 0
    if a.absorb is not None:
        rc |= L.mla_absorb_q(*a.absorb)
    if ev is not None:
        ev[0].record()
    rc |= L.mla_decode_paged_q8(*a.decode_q8) if a.decode_q8 is not None else L.mla_decode_paged(*a.decode)
    if ev is not None:
        ev[1].record()
    if a.proj is not None:
        rc |= L.mla_out_proj(*a.proj)
    return rc


def capture(torch, stream, body):
    """A CUDA graph of `body()` captured on `stream`, replayed once untimed; None if refused."""
    try:
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                rc = body()
            g.replay()
            stream.synchronize()
        return g if rc == 0 else None
    except Exception:
        return None


def time_graph(torch, g, stream, reps=1):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps  # ms


def workload_flops(inp):
    s = inp.seqlens.clamp(min=0).long()
    if inp.causal and inp.s_q > 1:
        pairs = sum(int(((s - inp.s_q + q + 1).clamp(min=0)).sum()) for q in range(inp.s_q)) * inp.H
    else:
        pairs = int(s.sum()) * inp.s_q * inp.H
    attn = pairs * FLOP_PER_PAIR
    proj = 2 * inp.B * inp.s_q * inp.H * FLOP_PROJ_PER_ROW
    return attn, proj


Q8_TOKEN_BYTES = 640 + 4  # INT8 cache: a token's record plus its scale


def roofline_of(inp, dec_ms, peaks, kv_bytes=None):
    """Roofline of one decode call on `inp` lasting dec_ms: the binding bound is
    the slower of the latent-cache bytes at the measured HBM copy rate and the
    attention FLOPs at the measured dense bf16 rate (burst: the call is timed
    alone); the fraction against the sustained bf16 rate is reported beside it."""
    hbm_peak, tc_peak, tc_sustained, peak_src = peaks
    kv_bytes = inp.kv_bytes() if kv_bytes is None else kv_bytes
    attn_flops, _ = workload_flops(inp)
    gbs = kv_bytes / (dec_ms * 1e-3) / 1e9
    tflops = attn_flops / (dec_ms * 1e-3) / 1e12
    t_mem = kv_bytes / (hbm_peak * 1e9)
    t_tc = attn_flops / (tc_peak * 1e12)
    if t_mem >= t_tc:
        r = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4)}
    else:
        r = {"bound": "tensor", "achieved": round(tflops, 1), "peak": tc_peak, "unit": "TFLOP/s",
             "frac": round(tflops / tc_peak, 4)}
    r.update({"algorithmic_bytes_per_launch": kv_bytes, "algorithmic_flops_per_launch": attn_flops,
              "avg_launch_us": round(dec_ms * 1e3, 3), "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
              "tensor_tflops": round(tflops, 1), "tensor_frac_of_burst": round(tflops / tc_peak, 4),
              "tensor_frac_of_sustained": round(tflops / tc_sustained, 4),
              "binding_roofline_us": round(max(t_mem, t_tc) * 1e6, 3), "peak_source": peak_src})
    return r


def input_sets(gen, name, rank, dev, l2, n_sets=0):
    """Resident input sets of `name`, enough that the bytes between two uses of
    a set exceed twice the L2 size."""
    probe = gen.make_workload(name, rep=1000 * rank)
    per_set = probe.kv_bytes() + sum(t.numel() * t.element_size() for t in (probe.q, probe.q_abs, probe.w_uk,
                                                                          probe.w_uv) if t is not None)
    n = n_sets if n_sets > 0 else max(2, math.ceil(2.0 * l2 / per_set) + 1)
    sets = [probe.to(dev)] + [gen.make_workload(name, rep=1000 * rank + i).to(dev) for i in range(1, n)]
    return sets, per_set


def decode_only(torch, api, L, gen, name, rank, dev, l2, peaks, calls, q8=False):
    """Decode-call duration on workload `name` (graph of `calls` decode calls
    over rotating input sets; the absorbed query of end-to-end workloads is
    made once per set beforehand) and its roofline. q8: the same workload with
    its cache quantised to the INT8 format (mla_quantize_cache, before timing)
    and decoded by mla_decode_paged_q8."""
    n_sets = 0
    if q8:
        probe = gen.make_workload(name, rep=1000 * rank)
        q_bytes = probe.B * probe.s_q * probe.H * 576 * 2
        per = int(probe.seqlens.clamp(min=0).sum()) * Q8_TOKEN_BYTES + q_bytes
        n_sets = max(2, math.ceil(2.0 * l2 / per) + 1)
        del probe
    sets, per_set = input_sets(gen, name, rank, dev, l2, n_sets)
    B, s_q, H = sets[0].B, sets[0].s_q, sets[0].H
    num_parts = api.mla_default_num_parts(dev.index, s_q)
    ws = api.make_workspace(B, s_q, H, num_parts, dev)
    stream = torch.cuda.Stream(dev)
    q8c = [api.mla_quantize_cache(s.kv_cache) for s in sets] if q8 else [None] * len(sets)
    torch.cuda.synchronize()
    steps = [StepArgs(api, s, num_parts, ws, stream.cuda_stream, q) for s, q in zip(sets, q8c)]
    call = L.mla_decode_paged_q8 if q8 else L.mla_decode_paged

    def args_of(a):
        return a.decode_q8 if q8 else a.decode
    rc = 0
    with torch.cuda.stream(stream):
        for a in steps:
            rc |= L.mla_get_metadata(*a.meta)
            if a.absorb is not None:
                rc |= L.mla_absorb_q(*a.absorb)
        for i in range(3 * len(steps)):
            rc |= call(*args_of(steps[i % len(steps)]))
        stream.synchronize()
    if rc != 0 or api.mla_read_device_error(ws) != 0:
        raise RuntimeError(f"decode failed on {name}")

    def body():
        r = 0
        for i in range(calls):
            r |= call(*args_of(steps[i % len(steps)]))
        return r
    g = capture(torch, stream, body)
    if g is None:
        raise RuntimeError(f"graph capture failed on {name}")
    ms = time_graph(torch, g, stream) / calls
    st = api.mla_read_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error on {name}: {api.status_string(st)}")
    kvb = int(sets[0].seqlens.clamp(min=0).sum()) * Q8_TOKEN_BYTES if q8 else None
    r = roofline_of(sets[0], ms, peaks, kvb)
    if q8:
        q_bytes = B * s_q * H * 576 * 2
        per_set = kvb + q_bytes
        r.update({"cache": "INT8 records (512 codes + 64 bf16 rope) + fp32 scale per token, 644 bytes"})
    r.update({"workload": describe(sets[0]), "num_parts": num_parts, "calls": calls,
              "l2": f"rotate {len(sets)} input sets, {len(sets) * per_set / 1e6:.0f} MB > 2 x L2",
              "traffic": None if q8 else recorded_traffic(name)})
    del g, steps, sets, ws, q8c
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return r


def fused_step_only(torch, api, L, gen, rank, dev, l2, calls):
    """The spec step with the split merge and the output projection fused into
    one finalize kernel (absorb + mla_decode_out_proj, three launches instead of
    four): graph of `calls` steps over rotating input sets."""
    sets, per_set = input_sets(gen, "spec", rank, dev, l2)
    B, s_q, H = sets[0].B, sets[0].s_q, sets[0].H
    num_parts = api.mla_default_num_parts(dev.index, s_q)
    ws = api.make_workspace(B, s_q, H, num_parts, dev)
    stream = torch.cuda.Stream(dev)
    steps = [StepArgs(api, s, num_parts, ws, stream.cuda_stream) for s in sets]
    P = ctypes.c_void_p

    def fused(a):
        d = a.inp
        return a.decode[:14] + (P(d.w_uv.data_ptr()), P(a.o_lat.data_ptr()), P(a.out.data_ptr())) + a.decode[15:]
    fargs = [fused(a) for a in steps]

    def body():
        r = 0
        for i in range(calls):
            a = steps[i % len(steps)]
            r |= L.mla_absorb_q(*a.absorb)
            r |= L.mla_decode_out_proj(*fargs[i % len(steps)])
        return r
    rc = 0
    with torch.cuda.stream(stream):
        for a in steps:
            rc |= L.mla_get_metadata(*a.meta)
        stream.synchronize()
    g = capture(torch, stream, body) if rc == 0 else None
    if g is None or api.mla_read_device_error(ws) != 0:
        raise RuntimeError("fused step failed")
    ms = time_graph(torch, g, stream) / calls
    st = api.mla_read_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error in the fused step: {api.status_string(st)}")
    r = {"workload": describe(sets[0]), "avg_step_us": round(ms * 1e3, 3), "launches_per_step": 3,
         "calls": calls, "num_parts": num_parts,
         "l2": f"rotate {len(sets)} input sets, {len(sets) * per_set / 1e6:.0f} MB > 2 x L2",
         "note": "absorb + decode + finalize (split merge fused with the output projection); "
                 "slower than the unfused step, which is the headline"}
    del g, steps, sets, ws
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return r


def prefill_flops(inp):
    """Algorithmic FLOPs of one naive-form prefill call: per visible (query row,
    key) pair 2 x (192 + 128) (score over [k_nope | k_rope], then V), plus the
    per-head decompression of every cached token, 2 x H x 512 x (128 + 128)."""
    s = inp.seqlens.clamp(min=0).long()
    if inp.causal:
        pairs = sum(int((s - inp.s_q + q + 1).clamp(min=0).sum()) for q in range(inp.s_q))
    else:
        pairs = int(s.sum()) * inp.s_q
    attn = pairs * inp.H * 2 * (192 + 128)
    decomp = int(s.sum()) * inp.H * 2 * 512 * (128 + 128)
    return attn, decomp


def prefill_only(torch, api, gen, rank, dev, peaks, calls=5, batch=8):
    """Duration of one mla_prefill_paged call (gather, two decompression GEMMs,
    causal attention) on the prefill workload, timed with CUDA events over
    `calls` back-to-back calls on one stream; q alone (800 MB) exceeds the L2,
    so every call streams its inputs from HBM."""
    inp = gen.make_workload("prefill", rep=1000 * rank, B=batch)
    d = inp.to(dev)
    stream = torch.cuda.Stream(dev)
    n = api.mla_prefill_workspace_size(inp.B, inp.H, inp.max_blocks_per_seq)
    ws = torch.empty(n + 1024, dtype=torch.uint8, device=dev)
    off = (-ws.data_ptr()) % 1024
    ws = ws[off:off + n]
    out = torch.empty((inp.B, inp.s_q, inp.H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((inp.B, inp.s_q, inp.H), dtype=torch.float32, device=dev)

    def call():
        api.mla_prefill_paged(d.q, d.kv_cache, d.block_table, d.seqlens, d.w_uk, d.w_uv, d.scale, True, out=out,
                              lse=lse, workspace=ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(calls):
            call()
        b.record(stream)
        b.synchronize()
    ms = a.elapsed_time(b) / calls
    st = api.mla_read_device_error()
    if st != 0:
        raise RuntimeError(f"device error on prefill: {api.status_string(st)}")
    attn, decomp = prefill_flops(inp)
    tc_peak = peaks[1]
    tflops = (attn + decomp) / (ms * 1e-3) / 1e12
    r = {"workload": (f"prefill: B={inp.B} whole prompts of {int(inp.seqlens[0])} tokens (s_q = seqlen), H={inp.H}, "
                      f"causal, naive form (gather, per-head K and V decompression GEMMs, flash attention)"),
         "bound": "tensor", "avg_call_us": round(ms * 1e3, 1), "achieved": round(tflops, 1), "peak": tc_peak,
         "unit": "TFLOP/s", "frac": round(tflops / tc_peak, 4), "algorithmic_flops_per_call": attn + decomp,
         "attention_flops": attn, "decompression_flops": decomp, "calls": calls,
         "binding_roofline_us": round((attn + decomp) / (tc_peak * 1e12) * 1e6, 1),
         "l2": f"inputs larger than L2 (q {d.q.numel() * 2 / 1e6:.0f} MB)", "launches_per_call": 4}
    del d, ws, out, lse
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return r


def rope_append_only(torch, L, api, rank, dev, peaks, l2, calls=400, q8=False):
    """Duration of one mla_rope_append call (mla_rope_append_q8 with q8) on the
    multi-token workload's shape: B=132 sequences of 4096 tokens whose last two
    (s_q = 2) are new, H=128. Every head's rope part of q is rotated in place and
    each new token's row is written into its page. A graph of `calls` calls over
    rotating input sets whose touched bytes exceed 2 x L2, seeded N(0,1) bf16.
    Only each sequence's last page is written, so the block table points every
    page of sequence b at block b and the cache holds B blocks."""
    B, s_q, H, n_tok = 132, 2, 128, 4096
    mbps = n_tok // 64
    row_bytes = 640 + 4 if q8 else 576 * 2
    # algorithmic bytes: rope parts of q read and written, new rows read and written
    alg = 2 * B * s_q * H * 64 * 2 + B * s_q * 576 * 2 + B * s_q * row_bytes
    n_sets = max(2, math.ceil(2.0 * l2 / alg) + 1)
    g = torch.Generator(device=dev)
    g.manual_seed(4242 + 1000 * rank)
    qs = [torch.randn((B, s_q, H, 192), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_sets)]
    kvn = [torch.randn((B, s_q, 576), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_sets)]
    seqlens = torch.full((B,), n_tok, dtype=torch.int32, device=dev)
    table = torch.arange(B, dtype=torch.int32, device=dev).repeat_interleave(mbps).view(B, mbps).contiguous()
    if q8:
        cache = torch.zeros((B, 64, 640), dtype=torch.uint8, device=dev)
        scale = torch.ones((B, 64), dtype=torch.float32, device=dev)
    else:
        cache = torch.zeros((B, 64, 576), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    P = ctypes.c_void_p
    st = P(stream.cuda_stream)
    if q8:
        args = [(P(q.data_ptr()), P(k.data_ptr()), P(seqlens.data_ptr()), P(table.data_ptr()), mbps,
                 P(cache.data_ptr()), P(scale.data_ptr()), B, B, s_q, H, ctypes.c_float(10000.0), st)
                for q, k in zip(qs, kvn)]
        call = L.mla_rope_append_q8
    else:
        args = [(P(q.data_ptr()), P(k.data_ptr()), P(seqlens.data_ptr()), P(table.data_ptr()), mbps,
                 P(cache.data_ptr()), B, B, s_q, H, ctypes.c_float(10000.0), st) for q, k in zip(qs, kvn)]
        call = L.mla_rope_append
    torch.cuda.synchronize()
    rc = 0
    with torch.cuda.stream(stream):
        for i in range(2 * n_sets):
            rc |= call(*args[i % n_sets])
        stream.synchronize()
    if rc != 0:
        raise RuntimeError("rope append failed")

    def body():
        r = 0
        for i in range(calls):
            r |= call(*args[i % n_sets])
        return r
    gr = capture(torch, stream, body)
    if gr is None:
        raise RuntimeError("graph capture failed on the rope append")
    ms = time_graph(torch, gr, stream) / calls
    err = api.mla_read_device_error()
    if err != 0:
        raise RuntimeError(f"device error on the rope append: {api.status_string(err)}")
    gbs = alg / (ms * 1e-3) / 1e9
    r = {"workload": (f"rope_append{'_q8' if q8 else ''}: B={B} s_q={s_q} H={H}, the new tokens at positions "
                      f"{n_tok - s_q}..{n_tok - 1}, rope base 10000"
                      + (", INT8 records + scales" if q8 else ", bf16 rows")),
         "bound": "hbm", "avg_call_us": round(ms * 1e3, 3), "achieved": round(gbs, 1), "peak": peaks[0],
         "unit": "GB/s", "frac": round(gbs / peaks[0], 4), "algorithmic_bytes_per_call": alg,
         "binding_roofline_us": round(alg / (peaks[0] * 1e9) * 1e6, 3), "calls": calls,
         "l2": f"rotate {n_sets} input sets, {n_sets * alg / 1e6:.0f} MB touched > 2 x L2", "launches_per_call": 1}
    del gr, qs, kvn, cache, table, seqlens
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return r


def describe(inp):
    sl = inp.seqlens
    lens = f"seqlen {int(sl[0])}" if bool((sl == sl[0]).all()) else f"seqlens {int(sl.min())}..{int(sl.max())}"
    mode = "end to end (absorb, decode, out-proj)" if inp.q is not None else "decode only (q_abs drawn)"
    causal = ", causal" if inp.causal and inp.s_q > 1 else ""
    return (f"{inp.name}: B={inp.B} s_q={inp.s_q} H={inp.H} {lens}{causal}, d_c 512 + rope 64, 64-token bf16 "
            f"pages, {mode}")


def run_ours(args, world, rank, local):
    import torch

    from mla_paged_kv_absorbed_gb300 import _build
    _build.build()
    from mla_paged_kv_absorbed_gb300 import api
    from mla_paged_kv_absorbed_gb300 import inputs as gen

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L = api.lib()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20)
    peaks = measured_peaks()
    if args.prefill_only:
        return prefill_only(torch, api, gen, rank, dev, peaks, args.prefill_calls, args.prefill_batch)

    sets, per_set = input_sets(gen, args.workload, rank, dev, l2, args.sets)
    n_sets = len(sets)
    B, s_q, H = sets[0].B, sets[0].s_q, sets[0].H
    num_parts = api.mla_default_num_parts(local, s_q)
    ws = api.make_workspace(B, s_q, H, num_parts, dev)
    stream = torch.cuda.current_stream(dev)
    if args.int8 and not args.profile:
        raise SystemExit("--int8 is a profiling option: use it with --profile")
    q8c = [api.mla_quantize_cache(s.kv_cache) for s in sets] if args.int8 else [None] * n_sets
    steps = [StepArgs(api, s, num_parts, ws, stream.cuda_stream, q) for s, q in zip(sets, q8c)]
    launches_per_step = sum(x is not None for x in (steps[0].absorb, steps[0].proj)) + 2  # + decode, combine

    # the schedule of each input set (fixed lengths), then warm-up and a
    # correctness gate: the device error word must be clear
    for a in steps:
        if L.mla_get_metadata(*a.meta) != 0:
            raise RuntimeError("mla_get_metadata failed")
    for i in range(max(args.warmup, 3)):
        if run_step(L, steps[i % n_sets]) != 0:
            raise RuntimeError("a C-ABI call returned an error during warm-up")
    torch.cuda.synchronize()
    st = api.mla_read_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {api.status_string(st)}")

    # the schedule on its own (once per model step, shared by the layers); not
    # in --profile runs, whose launch lists count only step launches
    meta_us = None
    if not args.profile:
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record()
        for i in range(200):
            L.mla_get_metadata(*steps[i % n_sets].meta)
        m1.record()
        torch.cuda.synchronize()
        meta_us = m0.elapsed_time(m1) * 1e3 / 200

    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    use_graph = not (args.profile or args.eager) and K <= 8192
    g = gd = None
    if use_graph:
        gstream = torch.cuda.Stream(dev)
        gsteps = [StepArgs(api, s, num_parts, ws, gstream.cuda_stream) for s in sets]
        with torch.cuda.stream(gstream):
            for a in gsteps:
                L.mla_get_metadata(*a.meta)
            for i in range(2 * n_sets):
                run_step(L, gsteps[i % n_sets])
            gstream.synchronize()
        g = capture(torch, gstream, lambda: sum(run_step(L, gsteps[i % n_sets]) for i in range(K)))
        gd = capture(torch, gstream, lambda: sum(L.mla_decode_paged(*gsteps[i % n_sets].decode) for i in range(K)))
        if g is None or gd is None or api.mla_read_device_error(ws) != 0:
            g = gd = None
    if g is not None:
        # The K steps (absorb, decode + combine, out-proj over the rotating input
        # sets) as one CUDA graph, replayed once untimed and once timed: the
        # host's launch cost and jitter stay out of the device timing.
        clocks.start()
        time.sleep(0.3)
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(gstream):
            t_start.record()
            g.replay()
            t_end.record()
        torch.cuda.synchronize()
        barrier(world)
        clk = clocks.stop()
        # the decode call's launch duration: the K decode calls alone, replayed
        dec_ms = [time_graph(torch, gd, gstream) / K]
        timed = ("one CUDA graph of the K steps' C-ABI calls, replayed, CUDA events around it; the decode "
                 "launch duration from a graph of the K decode calls alone")
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        if not args.profile:
            clocks.start()
            time.sleep(0.3)
        barrier(world)
        torch.cuda.synchronize()
        t_start.record()
        rc = 0
        for i in range(K):
            rc |= run_step(L, steps[i % n_sets], ev[i])
        t_end.record()
        torch.cuda.synchronize()
        barrier(world)
        clk = clocks.stop() if not args.profile else {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if rc != 0:
            raise RuntimeError("a C-ABI call returned an error in the timed region")
        dec_ms = [e[0].elapsed_time(e[1]) for e in ev]
        timed = "C-ABI calls, CUDA events on the launching stream"
    st = api.mla_read_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {api.status_string(st)}")
    total_ms = t_start.elapsed_time(t_end)
    ms_step = max_over_ranks(total_ms / K, world, dev)
    dec_avg_ms = statistics.mean(dec_ms)

    attn_flops, proj_flops = workload_flops(sets[0])
    roof = roofline_of(sets[0], dec_avg_ms, peaks)
    roof.update({"traffic": recorded_traffic(args.workload), "kernel": "mla_decode_paged (decode + combine launches)"})
    if len(dec_ms) > 1:
        roof["median_launch_us"] = round(statistics.median(dec_ms) * 1e3, 3)

    result = {
        "metric": METRIC, "value": round(ms_step * 1e3, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 activations and cache, "
        "N(0,1/512) weights, randomly permuted pages)",
        "config": {"workload": describe(sets[0]), "global_batch": B * world, "seq_len": int(sets[0].seqlens.max()),
                   "parallelism": f"replicas x{world} (sequences shard, no collective)",
                   "l2": f"rotate {n_sets} resident input sets, {n_sets * per_set / 1e6:.0f} MB > 2 x L2 "
                         f"({l2 / 1e6:.0f} MB)",
                   "num_parts": num_parts, "timed": timed},
        "roofline": roof,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")} | {"samples": clk.get("samples", 0)},
        "gpu_launches": launches_per_step * K,
        "metadata_us": None if meta_us is None else round(meta_us, 2),
        "throughput": {"decode_steps_per_s": round(world * 1e3 / ms_step, 1),
                       "tokens_per_s": round(world * B * s_q * 1e3 / ms_step, 1),
                       "step_tflops": round((attn_flops + proj_flops) / (ms_step * 1e-3) / 1e12, 2)},
    }
    if not args.no_e2e and not args.profile:
        result["e2e"] = run_e2e(args, api, L, sets, num_parts, ws, dev, world)
    del g, gd
    if not args.no_workloads and not args.profile:
        del steps, sets
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        wl = {args.workload: {k: roof[k] for k in ("bound", "frac", "avg_launch_us", "hbm_frac",
                                                   "tensor_frac_of_burst", "algorithmic_bytes_per_launch",
                                                   "algorithmic_flops_per_launch", "binding_roofline_us")}}
        for name in DECODE_WORKLOADS:
            if name != args.workload:
                wl[name] = decode_only(torch, api, L, gen, name, rank, dev, l2, peaks, args.decode_calls)
        for name in Q8_WORKLOADS:
            wl[name + "_int8"] = decode_only(torch, api, L, gen, name, rank, dev, l2, peaks, args.decode_calls, q8=True)
        wl["prefill"] = prefill_only(torch, api, gen, rank, dev, peaks, args.prefill_calls, args.prefill_batch)
        wl["spec_fused_step"] = fused_step_only(torch, api, L, gen, rank, dev, l2, 200)
        for q8 in (False, True):
            key = "rope_append_int8" if q8 else "rope_append"
            try:
                wl[key] = rope_append_only(torch, L, api, rank, dev, peaks, l2, 400, q8)
            except Exception as e:  # a side measurement: recorded, it does not void the headline
                wl[key] = {"error": f"{type(e).__name__}: {e}"}
        result["workloads"] = wl
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile:
        result["cpu_baseline"] = cpu_baseline(args.workload, budget_s=12.0)
    return result


def run_e2e(args, api, L, sets, num_parts, ws, dev, world):
    """The step through the C ABI with the step's inputs in pinned host memory,
    pipelined as a serving loop would run it: step i's queries, lengths and
    page table go up on a copy stream while step i - 1 computes; the four calls
    (schedule included) run on a compute stream; the projected output and lse
    come back on a third stream, and the host waits for step i - 1's result
    (reads it) before it enqueues step i + 1. Every step's copies and the
    host's read of every result are inside the timed region."""
    import torch
    n = len(sets)
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    steps = [StepArgs(api, s, num_parts, ws, s_comp.cuda_stream) for s in sets]
    host = []
    for s, a in zip(sets, steps):
        res = a.out if a.out is not None else a.o_lat
        host.append({
            "q": (s.q if s.q is not None else s.q_abs).cpu().pin_memory(),
            "seqlens": s.seqlens.cpu().pin_memory(), "table": s.block_table.cpu().pin_memory(),
            "out": torch.empty(res.shape, dtype=res.dtype).pin_memory(),
            "lse": torch.empty(a.lse.shape, dtype=a.lse.dtype).pin_memory(),
        })
    h2d = host[0]["q"].numel() * 2 + host[0]["seqlens"].numel() * 4 + host[0]["table"].numel() * 4
    d2h = host[0]["out"].numel() * 2 + host[0]["lse"].numel() * 4
    K = args.e2e_steps
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_comp = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    started = [False] * n

    def enqueue(i):
        j = i % n
        s, a, h = sets[j], steps[j], host[j]
        dst_q = s.q if s.q is not None else s.q_abs
        res = a.out if a.out is not None else a.o_lat
        with torch.cuda.stream(s_in):
            if started[j]:
                s_in.wait_event(ev_comp[j])  # set j's previous step has consumed its inputs
            dst_q.copy_(h["q"], non_blocking=True)
            s.seqlens.copy_(h["seqlens"], non_blocking=True)
            s.block_table.copy_(h["table"], non_blocking=True)
            ev_in[j].record(s_in)
        s_comp.wait_event(ev_in[j])
        if started[j]:
            s_comp.wait_event(ev_out[j])  # set j's previous result has left the device
        rc = run_step(L, a, meta=True)
        ev_comp[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[j])
            h["out"].copy_(res, non_blocking=True)
            h["lse"].copy_(a.lse, non_blocking=True)
            ev_out[j].record(s_out)
        started[j] = True
        return rc

    def loop(count):
        rc = 0
        for i in range(count):
            rc |= enqueue(i)
            if i >= 1:
                ev_out[(i - 1) % n].synchronize()
                _ = float(host[(i - 1) % n]["lse"][0, 0, 0])  # the host reads the result
        ev_out[(count - 1) % n].synchronize()
        _ = float(host[(count - 1) % n]["lse"][0, 0, 0])
        return rc

    rc = loop(5)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    rc |= loop(K)
    t1 = time.perf_counter()
    barrier(world)
    if rc != 0:
        raise RuntimeError("C-ABI error in the e2e loop")
    us = max_over_ranks((t1 - t0) / K * 1e6, world, dev)
    return {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "mode": "eager C-ABI calls; H2D, compute and D2H on three streams, two steps in flight, the host "
                    "reads every step's result", "steps": K,
            "note": "KV cache and weights stay resident (model state); per step the queries, lengths and page "
                    "table go up and the projected output and lse come back"}


# ------------------------------------------------------------ oracle timing --

def oracle_step(inp, batches):
    """The oracle's chain on the listed sequences: absorb -> attend -> out-proj
    (or attend alone for a workload whose absorbed query is drawn directly)."""
    import oracle
    from mla_paged_kv_absorbed_gb300 import inputs as gen
    sub = gen.sample_batches(inp, batches)
    f = lambda t: t.float().numpy()
    qa = f(sub.q_abs) if sub.q is None else oracle.absorb_q(f(sub.q), f(sub.w_uk))
    o, lse = oracle.attend_absorbed(qa, f(sub.kv_cache), sub.block_table, sub.seqlens, sub.scale, sub.causal)
    return o if sub.w_uv is None else oracle.out_proj(o, f(sub.w_uv))


def cpu_baseline(workload, budget_s=12.0):
    """Time the oracle as it stands on the host cores on a bounded sample of the
    workload and scale it to one full step (us/call)."""
    import oracle
    from mla_paged_kv_absorbed_gb300 import inputs as gen
    oracle.build()
    inp = gen.make_workload(workload)
    t0 = time.perf_counter()
    oracle_step(inp, [0])
    t1 = time.perf_counter()
    per_batch = max(t1 - t0, 1e-4)
    n = int(max(1, min(inp.B, budget_s / per_batch)))
    batches = list(range(n))
    t0 = time.perf_counter()
    oracle_step(inp, batches)
    dt = time.perf_counter() - t0
    return {"value": round(dt / n * inp.B * 1e6, 1), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of {inp.B} sequences of the {workload} workload, the whole chain of the step in "
                      f"fp64; {dt:.1f} s scaled by {inp.B}/{n}"}


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step runs a bounded sample of the
    workload on the host cores; value is scaled to a full step."""
    if rank != 0:
        return None
    import oracle
    from mla_paged_kv_absorbed_gb300 import inputs as gen
    oracle.build()
    inp = gen.make_workload(args.workload)
    t0 = time.perf_counter()
    oracle_step(inp, [0])
    per_batch = max(time.perf_counter() - t0, 1e-4)
    # keep the whole --steps K --warmup W run near two minutes
    per_step_budget = 120.0 / max(args.steps + args.warmup, 1)
    n = int(max(1, min(inp.B, per_step_budget / per_batch)))
    batches = list(range(n))
    for _ in range(args.warmup):
        oracle_step(inp, batches)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(inp, batches)
        times.append(time.perf_counter() - t0)
    us = statistics.mean(times) / n * inp.B * 1e6
    sample = f"{n} of {inp.B} sequences per step, the whole chain of the step in fp64, scaled by {inp.B}/{n}"
    return {"metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": describe(inp), "global_batch": inp.B * world,
                       "seq_len": int(inp.seqlens.max()), "parallelism": "oracle on the host cores (rank 0)"},
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "kind": "oracle", "cores": oracle.num_threads(),
                             "sample": sample},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
