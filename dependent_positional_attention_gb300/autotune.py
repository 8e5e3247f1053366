"""Chunk-size autotune for the prefill (per batch, heads, seq_len, head_dim,
dtype).

The chunk size C is a free parameter of the blockwise algorithm (the PaTH
lecture notes, hands-on item 3, sweep it against wallclock).  The
tensor-core route fixes C = head_dim = 128 (one chunk fills an MMA tile), so
only the CUDA-core route (fp32, or bf16 with head_dim other than 128) has a
choice: 16, 32, 64 or 128.  Each candidate, and the library's own default
(chunk 0), is timed once per shape on seeded synthetic inputs of that shape,
through path_attn_prefill_fwd, and the fastest candidate is cached for the
process.  This module only chooses a parameter; the computation is the
library's.
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
