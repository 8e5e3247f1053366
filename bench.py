"""Benchmark of the PaTH attention hot path on GB300.

Headline: PaTH prefill forward, B8 H12 L4096 d128 bf16 (one step = the UT
prep kernel + the tensor-core scan kernel over one batch).  The same line
also reports, as nested objects, the PaTH-FoX prefill (same shape), the
long-context prefill (B1 H12 L32768, beta mostly near 2) and the decode
workload (B16 H12 d128, 65536 cached tokens, 256 steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the workload on
its own GPU (weak scaling, no data-path collective); the elapsed time is the
max over ranks.  `--impl reference` times the fp64 CPU oracle on sampled
query rows of the headline workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import threading
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import dependent_positional_attention_gb300 as pa  # noqa: E402
from dependent_positional_attention_gb300 import workloads as wl  # noqa: E402

METRIC = "PaTH prefill tokens/s & TFLOP/s (L=4K,d=128,bf16); decode HBM GB/s"
CHUNK = 128


def prefill_flops(B, H, L, d, C=CHUNK):
    """Algorithmic FLOPs per head, split by kernel.
    scan: QK^T + PV over the off-diagonal chunk pairs (4 C^2 d per pair,
    N (N-1) / 2 pairs) plus the carried-query update (one C x d x d product
    with a chunk's d x d transition matrix per pair (b, c) with c >= 1:
    2 C d^2 (N-1)(N-2)/2).
    prep: the chunk UT transform (16 L C d: G, T and the boundary products) plus each
    chunk's own causal block (QK^T + PV over its lower triangle, 2 C^2 d).
    Returns (scan_flops, prep_flops)."""
    N = math.ceil(L / C)
    scan = (4 * C * C * d * N * (N - 1) / 2 + 2 * C * d * d * (N - 1) * (N - 2) / 2) * B * H
    prep = (16 * L * C * d + 2 * C * C * d * N) * B * H
    return scan, prep


def backward_flops(B, H, L, d, C=CHUNK):
    """MMA FLOPs of one backward call on the tensor-core route (bf16,
    d = C = 128), 2 C^2 d per 128 x 128 x 128 contraction.  Per (query chunk,
    earlier key chunk) pair the scan runs nine: the carried-row chain product,
    S, dP, dV, dKh, dA and the two of the carried-gradient update.  Per chunk
    the recomputed prep runs twelve (its eleven plus P V) and the backward
    prep thirty-seven (the products of its 22 batched contractions)."""
    N = math.ceil(L / C)
    pairs = N * (N - 1) / 2
    return 2 * C * C * d * (9 * pairs + 49 * N) * B * H


# DRAM read + write bytes per cached key of decode_split_kernel<128, fox>, from
# ncu on B16 H12 with 8195 cached tokens (1,573,440 keys per launch)
DECODE_TRAFFIC_PER_KEY = {False: (805.738240e6 + 354.663424e6) / 1573440,
                          True: (812.037376e6 + 349.548032e6) / 1573440}

# DRAM read + write (bytes) of one scan launch of the headline workload (B8 H12 L4096 d128),
# from a one-pass ncu capture of that launch
SCAN_TRAFFIC_B8 = 507.67e6 + 88.50e6


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during a timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.lines = []
        self.reader = None

    def start(self):
        """Starts sampling every 20 ms and returns once the first sample is in,
        so that the samples that follow fall inside the timed region."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        first = threading.Event()

        def read():
            for line in self.proc.stdout:
                self.lines.append(line)
                first.set()
            first.set()

        self.reader = threading.Thread(target=read, daemon=True)
        self.reader.start()
        first.wait(timeout=5.0)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.03)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.reader is not None:
            self.reader.join(timeout=5)
        out = "".join(self.lines)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- helpers

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def _collective_device():
    # NCCL reduces CUDA tensors; gloo (the CPU tests of this path) host tensors
    return "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"


def max_over_ranks(x, ws):
    """The slowest rank's time: every rank times the same number of steps."""
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=_collective_device())
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, ms_per_step_max, ws):
    """Whole-job rate: every rank processes its own units (weak scaling, no
    data-path collective); the job takes as long as its slowest rank."""
    return ws * units_per_rank / (ms_per_step_max * 1e-3)


def timed_prefill(x, steps, warmup, ws, fox=False, sampler=None):
    """Times K prefill steps with CUDA events on the launching stream.  A step
    is one path_attn_prefill_fwd call, in which the scan starts on the SMs the
    prep's last chunks leave idle.  A second pass of K steps calls the two
    stages separately, with an event between them, for the per-kernel times
    (prep, scan) that the roofline uses.  Returns (ms_per_step, prep_ms,
    scan_ms, clocks)."""
    q, k, v, w, beta = (x[n] for n in ("q", "k", "v", "w", "beta"))
    log_f = x.get("log_f") if fox else None
    stream = torch.cuda.current_stream()
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
    ws_t = pa.path_attn_prefill_prep(q, k, v, w, beta, log_f=log_f)

    def step():
        pa.path_attn_prefill_fwd(q, k, v, w, beta, log_f=log_f, out=out, lse=lse,
                                 workspace=ws_t)

    for _ in range(warmup):
        step()
    barrier(ws)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(ws)
    total = t0.elapsed_time(t1) / steps
    # per-kernel breakdown: the same work as separate stage calls
    for _ in range(warmup):
        pa.path_attn_prefill_prep(q, k, v, w, beta, log_f=log_f, workspace=ws_t)
        pa.path_attn_prefill_scan(q, w, v, ws_t, log_f=log_f, out=out, lse=lse)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        ev[i][0].record(stream)
        pa.path_attn_prefill_prep(q, k, v, w, beta, log_f=log_f, workspace=ws_t)
        ev[i][1].record(stream)
        pa.path_attn_prefill_scan(q, w, v, ws_t, log_f=log_f, out=out, lse=lse)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    prep = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    scan = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    if pa.path_attn_device_status() != 0:
        raise RuntimeError("device error flag set during prefill timing")
    return total, prep, scan, clocks


def prefill_block(wlk, steps, warmup, ws, peaks, seed=0, sampler=None):
    x = wl.workload_inputs(wlk, seed=seed, device="cuda")
    B, H, L, d = wlk.batch, wlk.heads, wlk.seq_len, wlk.head_dim
    ms, prep_ms, scan_ms, clocks = timed_prefill(x, steps, warmup, ws, fox=wlk.fox,
                                                 sampler=sampler)
    ms = max_over_ranks(ms, ws)
    scan_f, prep_f = prefill_flops(B, H, L, d)
    tflops = job_throughput(scan_f + prep_f, ms, ws) / 1e12
    scan_tf = scan_f / (scan_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    res = {
        "workload": wlk.name, "tokens_per_s": job_throughput(B * L, ms, ws), "tflops": tflops,
        "ms_per_step": ms, "prep_ms": prep_ms, "scan_ms": scan_ms,
        "flops_per_step": scan_f + prep_f,
        "roofline": {"kernel": "flash_tc_kernel (tensor-core scan)", "bound": "tensor",
                     "achieved": scan_tf, "peak": peak, "unit": "TFLOP/s",
                     "frac": scan_tf / peak,
                     # DRAM bytes per launch: ncu read + write of this kernel's headline
                     # launch (B8 H12 L4096 d128, not FoX); null for the other workloads
                     "traffic": (SCAN_TRAFFIC_B8
                                 if (B, H, L, d) == (8, 12, 4096, 128) and not wlk.fox else None),
                     "peak_source": peaks["source"] + " bf16 dense (burst)"},
    }
    del x
    torch.cuda.empty_cache()
    return res, clocks


def e2e_prefill(wlk, steps, warmup, ws, seed=0):
    """Same metric through the public API with pinned host buffers: every step
    copies its inputs host->device, runs the prefill and copies its output
    back, all inside the timed region.  Steps are pipelined the way a serving
    loop would run them: three streams (host->device copies, compute,
    device->host copies) and two device buffer sets, so that step i+1's input
    copy and step i-1's output copy overlap step i's kernels.  Events order
    each buffer's reuse after its previous reader."""
    xh = wl.workload_inputs(wlk, seed=seed, device="cpu")
    xh = {n: t.pin_memory() for n, t in xh.items()}
    sets = [{n: torch.empty_like(t, device="cuda") for n, t in xh.items()} for _ in range(2)]
    outs = [torch.empty_like(sets[0]["q"]) for _ in range(2)]
    out_h = torch.empty_like(xh["q"]).pin_memory()
    q = sets[0]["q"]
    ws_t = torch.empty(pa.path_attn_prefill_workspace_size(pa._prefill_desc(q, None, 0)),
                       device="cuda", dtype=torch.uint8)
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    # one extra copy stream per further input tensor, so that several copy
    # engines move a step's inputs at once
    names = list(xh)
    s_ins = [s_in] + [torch.cuda.Stream() for _ in names[1:]]
    ev = lambda: torch.cuda.Event()
    in_done = [[ev() for _ in names] for _ in range(2)]   # each input of the set landed
    cmp_done = [ev(), ev()]      # prefill that read the set (and wrote outs[set]) finished
    out_done = [ev(), ev()]      # output of the set copied back
    used = [False, False]

    def step(i):
        j = i % 2
        xd, od = sets[j], outs[j]
        for n, si, e in zip(names, s_ins, in_done[j]):
            with torch.cuda.stream(si):
                if used[j]:
                    si.wait_event(cmp_done[j])
                xd[n].copy_(xh[n], non_blocking=True)
                e.record(si)
        with torch.cuda.stream(s_cmp):
            for e in in_done[j]:
                s_cmp.wait_event(e)
            if used[j]:
                s_cmp.wait_event(out_done[j])
            pa.path_attn_prefill_fwd(xd["q"], xd["k"], xd["v"], xd["w"], xd["beta"],
                                     log_f=xd.get("log_f"), out=od, workspace=ws_t,
                                     want_lse=False, stream=s_cmp)
            cmp_done[j].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[j])
            out_h.copy_(od, non_blocking=True)
            out_done[j].record(s_out)
        used[j] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    # device time from the first input copy to the last output copy: the last
    # device->host copy waits (through the events) for every earlier step
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(warmup + i)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / steps, ws)
    if pa.path_attn_device_status() != 0:
        raise RuntimeError("device error flag set during end-to-end timing")
    h2d = sum(t.numel() * t.element_size() for t in xh.values())
    d2h = out_h.numel() * out_h.element_size()
    return {"value": job_throughput(wlk.batch * wlk.seq_len, ms, ws), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "pipelined": "%d input-copy streams, compute stream, output-copy stream; "
                         "2 buffer sets" % len(s_ins)}


def decode_block(wlk, steps, warmup, ws, peaks, seed=0, fox=False):
    """Decode steps over a prefilled cache; with fox, the PaTH-FoX step (the
    forget-gate prefixes of the cached tokens built by path_attn_fox_prefix)."""
    B, H, d, L0 = wlk.batch, wlk.heads, wlk.head_dim, wlk.prefix_len
    nsteps = steps if steps > 0 else wlk.steps
    cap = L0 + warmup + nsteps
    x = wl.prefill_inputs(B, H, L0, d, "bf16", seed=seed, fox=fox, device="cuda")
    kc = torch.zeros((B, H, cap, d), device="cuda", dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    pa.path_attn_build_kcache(x["k"], x["w"], x["beta"], kc)
    vc[:, :, :L0] = x["v"]
    fc = None
    if fox:
        fc = torch.zeros((B, H, cap), device="cuda", dtype=torch.float32)
        pa.path_attn_fox_prefix(x["log_f"], fc)
    del x
    torch.cuda.empty_cache()
    toks = [wl.decode_token(B, H, d, "bf16", seed=10_000 + seed + t, device="cuda", fox=fox)
            for t in range(warmup + nsteps)]

    def step(g, t):
        if fox:
            pa.path_attn_decode_step_fox(kc, vc, fc, t, g["q"], g["k"], g["v"], g["w"],
                                         g["beta"], g["log_f"], out=out, workspace=wsp)
        else:
            pa.path_attn_decode_step(kc, vc, t, g["q"], g["k"], g["v"], g["w"], g["beta"],
                                     out=out, workspace=wsp)
    out = torch.empty((B, H, d), device="cuda", dtype=torch.bfloat16)
    wsz = pa.path_attn_decode_workspace_size(pa.decode_desc(kc))
    wsp = torch.empty(max(wsz, 16), device="cuda", dtype=torch.uint8)
    t = L0
    for i in range(warmup):
        step(toks[i], t)
        t += 1
    stream = torch.cuda.current_stream()
    barrier(ws)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nsteps + 1)]
    evs[0].record(stream)
    bytes_total = 0
    keys_total = 0
    for i in range(nsteps):
        step(toks[warmup + i], t)
        bytes_total += 3 * B * H * t * d * 2  # read K, write K, read V
        keys_total += B * H * t
        if fox:
            bytes_total += B * H * t * 4  # read each key's forget-gate prefix
        t += 1
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    total_ms = evs[0].elapsed_time(evs[-1])
    if pa.path_attn_device_status() != 0:
        raise RuntimeError("device error flag set during decode timing")
    ms = max_over_ranks(total_ms / nsteps, ws)
    gbs = bytes_total / nsteps / (ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    name = wlk.name.replace("PaTH decode", "PaTH-FoX decode") if fox else wlk.name
    res = {"workload": name, "tokens_per_s": ws * B / (ms * 1e-3), "ms_per_step": ms,
           "steps": nsteps, "hbm_gbs": gbs * ws,
           "roofline": {"kernel": "decode_split_kernel + decode_combine_kernel",
                        "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                        "frac": gbs / peak,
                        # ncu dram read + write per key of decode_split_kernel (B16 H12,
                        # cache 8192) times the mean keys of one timed step
                        "traffic": (DECODE_TRAFFIC_PER_KEY[fox] * keys_total / nsteps
                                    if d == 128 and DECODE_TRAFFIC_PER_KEY[fox] else None),
                        "peak_source": peaks["source"] + " copy bandwidth"}}
    del kc, vc, fc
    torch.cuda.empty_cache()
    return res


def backward_block(wlk, steps, warmup, ws, peaks, workspace_bytes=None):
    """path_attn_prefill_bwd on the forward's inputs and outputs, device-timed
    with CUDA events; the launches of one call form one step.  With
    workspace_bytes the call gets that much workspace (at least its minimum)
    and runs the (batch, head) slices in passes."""
    x = wl.workload_inputs(wlk, seed=0, device="cuda")
    q, k, v, w, beta = (x[n] for n in ("q", "k", "v", "w", "beta"))
    log_f = x.get("log_f") if wlk.fox else None
    out, lse = pa.path_attn_prefill_fwd(q, k, v, w, beta, log_f=log_f)
    dout = torch.randn(q.shape, generator=torch.Generator("cuda").manual_seed(7), device="cuda",
                       dtype=torch.float32).to(q.dtype)
    desc = pa._prefill_desc(q, None, 0)
    ws_bytes = pa.path_attn_prefill_bwd_workspace_size(desc)
    if workspace_bytes is not None:
        ws_bytes = min(ws_bytes, max(workspace_bytes, pa.path_attn_prefill_bwd_workspace_min(desc)))
    ws_t = torch.empty(ws_bytes, device="cuda", dtype=torch.uint8)
    run = lambda: pa.path_attn_prefill_bwd(q, k, v, w, beta, out, lse, dout, log_f=log_f,
                                           workspace=ws_t)
    for _ in range(warmup):
        run()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        run()
    t1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / steps, ws)
    B, H, L, d = wlk.batch, wlk.heads, wlk.seq_len, wlk.head_dim
    flops = backward_flops(B, H, L, d)
    tf = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"] or peaks["bf16_tflops"]
    res = {"workload": "%s prefill backward (dq, dk, dv, dw, dbeta%s) B%d H%d L%d d%d %s%s"
                       % ("PaTH-FoX" if wlk.fox else "PaTH", ", dlog_f" if wlk.fox else "",
                          B, H, L, d, wlk.dtype,
                          ", workspace %.2f GB (slices in passes)" % (ws_bytes / 1e9)
                          if workspace_bytes is not None else ""),
           "tokens_per_s": job_throughput(B * L, ms, ws), "ms_per_step": ms,
           "flops_per_step": flops, "tflops": tf, "workspace_bytes": ws_t.numel(),
           "roofline": {"kernel": "whole backward call: prep_tc_kernel + bwd_scan_tc_kernel + "
                                  "chunk_gemm_tc_kernel x23 + solve/diag/cvt/dbeta",
                        "bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                        "frac": tf / peak, "traffic": None,
                        "peak_source": peaks["source"] + " bf16 dense (sustained: a step of "
                                       "about 30 launches)"}}
    del x, out, lse, dout, ws_t, log_f
    torch.cuda.empty_cache()
    return res


def autotune_block(wlk):
    """Chunk-size autotune on the CUDA-core route: the chosen chunk and its
    time against the default chunk."""
    from dependent_positional_attention_gb300 import autotune
    best, times = autotune.autotune_chunk(wlk.batch, wlk.heads, wlk.seq_len, wlk.head_dim,
                                          wlk.dtype)
    return {"workload": wlk.name, "best_chunk": best,
            "ms_by_chunk": {str(c): t for c, t in sorted(times.items()) if c},
            "ms_library_default": times[0], "speedup_vs_default": times[0] / times[best]}


def scan_group_block(wlk):
    """Tensor-core route: the scan's head-group size (the one tensor-core
    launch parameter; the chunk is 128 there) swept on the one-call forward,
    against the library's automatic size (key "0")."""
    from dependent_positional_attention_gb300 import autotune
    best, times = autotune.autotune_scan_group(wlk.batch, wlk.heads, wlk.seq_len,
                                               wlk.head_dim, wlk.dtype)
    return {"workload": wlk.name, "best_scan_group": best,
            "ms_by_scan_group": {str(g): t for g, t in sorted(times.items())},
            "ms_library_default": times[0], "speedup_vs_default": times[0] / times[best]}


class OracleSampler:
    """fp64 oracle on uniformly sampled query rows of a few heads of a
    workload (inputs drawn once, with the workload's seeded generator)."""

    def __init__(self, wlk, heads=8, seed=3):
        x = wl.workload_inputs(wlk, seed=0, device="cpu")
        BH = wlk.batch * wlk.heads
        self.g = torch.Generator().manual_seed(seed)
        sel = torch.randperm(BH, generator=self.g)[:heads].tolist()
        flat = {n: t.reshape((BH,) + tuple(t.shape[2:]))[sel].double().numpy()
                for n, t in x.items()}
        self.args = [flat[n] for n in ("q", "k", "v", "w", "beta")]
        self.log_f = flat.get("log_f")
        self.heads, self.L = heads, wlk.seq_len
        self.threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))

    def run(self, rows_per_head):
        import oracle
        rows = torch.randint(0, self.L, (rows_per_head,), generator=self.g).tolist()
        t0 = time.perf_counter()
        oracle.prefill(*self.args, log_f=self.log_f, rows=rows)
        return time.perf_counter() - t0, rows_per_head * self.heads

    def calibrated(self, target_s):
        dt, n = self.run(8)
        return max(8, min(4096, int(target_s / max(dt / n, 1e-7) / self.heads)))


# ----------------------------------------------------------------- main

def workload_config(head, ws):
    """The `config` object of the JSON line (both arms report the same one)."""
    return {"workload": head.name, "batch_per_gpu": head.batch, "heads": head.heads,
            "seq_len": head.seq_len, "head_dim": head.head_dim, "chunk": CHUNK,
            "l2": "inputs larger than L2 (%.0f MB read per step)"
                  % (5 * head.batch * head.heads * head.seq_len * head.head_dim * 2 / 1e6),
            "parallelism": "replicas" if ws > 1 else "single"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-extra", action="store_true",
                    help="headline workload only (no FoX / long / decode objects)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the prefill backward on the headline shape and print its "
                         "object (for profiler captures; not the bench line)")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode workload (PaTH, or PaTH-FoX with --fox) and "
                         "print its object (for profiler captures; not the bench line)")
    ap.add_argument("--fox", action="store_true", help="with --decode-only: the PaTH-FoX step")
    ap.add_argument("--decode-prefix", type=int, default=None,
                    help="override the decode workload's cached tokens (smaller cases for "
                         "profiler captures; the default is 65536)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the headline workload's batch (smaller cases for "
                         "profiler captures; the default is the headline B8)")
    args = ap.parse_args()
    ws, rank, local = dist_info()
    head = wl.PREFILL_4K
    if args.batch:
        head = dataclasses.replace(head, batch=args.batch,
                                   name=head.name.replace("B%d " % head.batch,
                                                          "B%d " % args.batch))

    if args.impl == "reference":
        if rank != 0:
            return
        steps, warm = args.steps, max(args.warmup, 0)
        import oracle
        oracle.build()
        smp = OracleSampler(head, heads=2, seed=100)
        per_step = smp.calibrated(0.5)
        threads = smp.threads
        rates = []
        for i in range(warm + steps):
            dt, n = smp.run(per_step)
            if i >= warm:
                rates.append((n, dt))
        n_tot = sum(n for n, _ in rates)
        t_tot = sum(dt for _, dt in rates)
        value = n_tot / t_tot
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": steps, "warmup": warm,
                "ms_per_step": 1e3 * t_tot / steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": workload_config(head, ws),
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                                 "kind": "oracle",
                                 "sample": "%d uniformly sampled query rows of 2 heads per step"
                                           % (n_tot // max(steps, 1))},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    from dependent_positional_attention_gb300 import build as pa_build
    pa_build.build()
    pa.load_library()
    peaks = load_peaks()
    warmup = max(3, args.warmup)
    steps = max(1, args.steps)

    if args.decode_only:
        dw = wl.DECODE_64K
        if args.decode_prefix:
            dw = dataclasses.replace(dw, prefix_len=args.decode_prefix,
                                     name=dw.name.replace("65536", str(args.decode_prefix)))
        res = decode_block(dw, steps, warmup, ws, peaks, fox=args.fox)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    if args.backward_only:
        res = backward_block(head, steps, warmup, ws, peaks)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    sampler = ClockSampler() if rank == 0 else None
    main_res, clocks = prefill_block(head, steps, warmup, ws, peaks, sampler=sampler)
    e2e = e2e_prefill(head, max(3, steps // 2), 2, ws)
    extra = {}
    if not args.skip_extra:
        extra["fox_4k"], _ = prefill_block(wl.FOX_4K, steps, warmup, ws, peaks)
        extra["long_32k"], _ = prefill_block(wl.PREFILL_32K, max(3, steps // 4), 3, ws, peaks)
        extra["decode_64k"] = decode_block(wl.DECODE_64K, wl.DECODE_64K.steps, warmup, ws, peaks)
        extra["decode_fox_64k"] = decode_block(wl.DECODE_64K, wl.DECODE_64K.steps, warmup, ws,
                                               peaks, fox=True)
        extra["backward_4k"] = backward_block(head, max(3, steps // 2), 3, ws, peaks)
        extra["backward_fox_4k"] = backward_block(wl.FOX_4K, max(3, steps // 2), 3, ws, peaks)
        extra["backward_4k_ws1gb"] = backward_block(head, max(3, steps // 2), 3, ws, peaks,
                                                    workspace_bytes=10 ** 9)
        extra["scan_group_autotune_4k"] = scan_group_block(head)
        extra["chunk_autotune_f32_tiny"] = autotune_block(wl.TINY_F32)
        extra["chunk_autotune_bf16_d64"] = autotune_block(
            wl.PrefillWorkload("PaTH prefill fwd B8 H12 L4096 d64 bf16 (chunks 16-64 on the CUDA "
                               "cores; 128 and the default on the tensor cores, head_dim-64 scan)",
                               8, 12, 4096, 64, "bf16"))
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        # every head, so that about 10 s of oracle work fits under the cap of
        # one sequence's worth of rows per head
        nh = head.batch * head.heads
        smp = OracleSampler(head, heads=nh)
        dt, n = smp.run(smp.calibrated(10.0))
        threads = smp.threads
        cpu = {"value": n / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": "%d uniformly sampled query rows (%d heads) of the %s workload, %.1f s"
                         % (n, nh, head.name, dt)}
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": main_res["tokens_per_s"], "unit": "tokens/s",
        "n_gpus": ws, "steps": steps, "warmup": warmup, "ms_per_step": main_res["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(head, ws),
        "tflops": main_res["tflops"], "prep_ms": main_res["prep_ms"],
        "scan_ms": main_res["scan_ms"], "roofline": main_res["roofline"],
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": 2 * steps,
        "workloads": extra,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
