"""Prefill autotune (per batch, heads, seq_len, head_dim, dtype): the chunk
size on the CUDA-core route, and the tensor-core scan's head-group size.

The chunk size C is a free parameter of the blockwise algorithm (the PaTH
lecture notes, hands-on item 3, sweep it against wallclock).  The
tensor-core route fixes C = head_dim = 128 (one chunk fills an MMA tile), so
only the CUDA-core route (fp32, or bf16 with head_dim other than 128) has a
choice: 16, 32, 64 or 128.  Each candidate, and the library's own default
(chunk 0), is timed once per shape on seeded synthetic inputs of that shape,
through path_attn_prefill_fwd, and the fastest candidate is cached for the
process.  This module only chooses a parameter; the computation is the
library's.

On the tensor-core route the chunk stays 128, and what there is to choose is
the order of the scan's query tiles: the heads per group
(path_prefill_desc_t.scan_group).  The tiles of one group of heads go out,
heaviest first, before the next group's, so that the CTAs on a head read key
chunks another CTA has just brought into L2; the library's automatic size
is about SM count / 10 heads.  autotune_scan_group times it against a few
fixed sizes; every size gives identical results.
"""
from __future__ import annotations

import statistics

from . import path_attn_prefill_fwd
from . import workloads as wl

CUDA_CORE_CHUNKS = (16, 32, 64, 128)
_cache: dict = {}


def candidates(head_dim: int, dtype: str):
    if dtype == "bf16" and head_dim == 128:
        return (128,)
    return CUDA_CORE_CHUNKS


def _median_ms(run, reps):
    import torch

    run()
    torch.cuda.synchronize()
    samples = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        samples.append(e0.elapsed_time(e1))
    return statistics.median(samples)


def autotune_chunk(batch: int, heads: int, seq_len: int, head_dim: int, dtype: str = "f32",
                   reps: int = 5, device: str = "cuda"):
    """Returns (best_chunk, {chunk: median milliseconds}) for this shape; the
    key 0 holds the time of the library's default chunk."""
    key = (batch, heads, seq_len, head_dim, dtype)
    if key in _cache:
        return _cache[key]
    x = wl.prefill_inputs(batch, heads, seq_len, head_dim, dtype, seed=0, device=device)
    times = {}
    for c in (0,) + tuple(candidates(head_dim, dtype)):
        times[c] = _median_ms(lambda: path_attn_prefill_fwd(
            x["q"], x["k"], x["v"], x["w"], x["beta"], chunk=c, want_lse=False), reps)
    best = min((c for c in times if c), key=times.get)
    _cache[key] = (best, times)
    return best, times


_group_cache: dict = {}


def scan_group_candidates(batch: int, heads: int):
    """0 (the library's automatic size), powers of two below batch*heads,
    and batch*heads (one group: every head interleaved)."""
    bh = batch * heads
    c = [0]
    g = 4
    while g < bh:
        c.append(g)
        g *= 2
    c.append(bh)
    return tuple(c)


def autotune_scan_group(batch: int, heads: int, seq_len: int, head_dim: int = 128,
                        dtype: str = "bf16", reps: int = 5, device: str = "cuda"):
    """Returns (best_group, {group: median milliseconds}) of the one-call
    forward on the tensor-core route for this shape; key 0 is the automatic
    size.  Cached per process."""
    key = (batch, heads, seq_len, head_dim, dtype)
    if key in _group_cache:
        return _group_cache[key]
    import torch

    x = wl.prefill_inputs(batch, heads, seq_len, head_dim, dtype, seed=0, device=device)
    out = torch.empty_like(x["q"])
    times = {}
    for g in scan_group_candidates(batch, heads):
        times[g] = _median_ms(lambda: path_attn_prefill_fwd(
            x["q"], x["k"], x["v"], x["w"], x["beta"], out=out, want_lse=False,
            scan_group=g), reps)
    best = min(times, key=times.get)
    _group_cache[key] = (best, times)
    return best, times
