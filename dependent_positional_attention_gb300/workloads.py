"""Seeded synthetic inputs for PaTH attention.

This module only draws random inputs; it holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle can be fed from it.

Draw order per call (one ``torch.Generator`` seeded with ``seed``):
q, k, v, w, beta-logits, then log-f-logits (PaTH-FoX only).  Each draw is an
fp32 standard normal; w is L2-normalised in fp32 and then cast; beta is
2*sigmoid(z + beta_mu) in fp32; log f = logsigmoid(z + 3) in fp32.  These
follow the parametrisation on the PaTH page (beta = 2*sigmoid(.), unit w) and
the workload shapes of the language-model experiments (4K training length,
32K extrapolation length); the public corpora of those experiments are not
used — these draws stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    batch: int
    heads: int
    seq_len: int
    head_dim: int
    dtype: str            # "f32" or "bf16"
    beta_mu: float = 0.0  # beta = 2*sigmoid(N(beta_mu, 1))
    fox: bool = False     # draw a PaTH-FoX forget gate
    sampled_rows: int = 0  # 0: check every row; else rows checked per head


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    heads: int
    head_dim: int
    prefix_len: int       # tokens already in the cache (built by prefill)
    steps: int            # decode steps, each appending one token
    dtype: str = "bf16"


TINY_F32 = PrefillWorkload("tiny PaTH fwd B1 H1 L256 d64 fp32", 1, 1, 256, 64, "f32")
PREFILL_4K = PrefillWorkload("PaTH prefill fwd B8 H12 L4096 d128 bf16", 8, 12, 4096, 128, "bf16")
PREFILL_32K = PrefillWorkload("long-context PaTH prefill fwd B1 H12 L32768 d128 bf16 beta~2",
                              1, 12, 32768, 128, "bf16", beta_mu=2.0, sampled_rows=512)
FOX_4K = PrefillWorkload("PaTH-FoX prefill fwd B8 H12 L4096 d128 bf16", 8, 12, 4096, 128,
                         "bf16", fox=True)
DECODE_64K = DecodeWorkload("PaTH decode B16 H12 d128 bf16 cache 65536 x 256 steps",
                            16, 12, 128, 65536, 256)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(g, shape, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def prefill_inputs(batch, heads, seq_len, head_dim, dtype="bf16", seed=0,
                   beta_mu=0.0, fox=False, device="cpu"):
    """Draw q, k, v, w ([B,H,L,d], ``dtype``), beta ([B,H,L] fp32) and, for
    PaTH-FoX, log_f ([B,H,L] fp32).  Returns a dict of tensors on ``device``."""
    tdt = DTYPES[dtype]
    g = _gen(seed, device)
    shape = (batch, heads, seq_len, head_dim)
    q = _normal(g, shape, device).to(tdt)
    k = _normal(g, shape, device).to(tdt)
    v = _normal(g, shape, device).to(tdt)
    w = _normal(g, shape, device)
    w = (w / w.norm(dim=-1, keepdim=True)).to(tdt)
    beta = 2.0 * torch.sigmoid(_normal(g, shape[:3], device) + beta_mu)
    out = {"q": q, "k": k, "v": v, "w": w, "beta": beta.contiguous()}
    if fox:
        out["log_f"] = torch.nn.functional.logsigmoid(_normal(g, shape[:3], device) + 3.0)
    return out


def workload_inputs(wl: PrefillWorkload, seed=0, device="cpu"):
    return prefill_inputs(wl.batch, wl.heads, wl.seq_len, wl.head_dim, wl.dtype, seed,
                          wl.beta_mu, wl.fox, device)


def decode_token(batch, heads, head_dim, dtype="bf16", seed=0, device="cpu", fox=False):
    """One decode step's q_t, k_t, v_t, w_t ([B,H,d]), beta_t ([B,H]) and,
    for PaTH-FoX, log_f_t ([B,H])."""
    d = prefill_inputs(batch, heads, 1, head_dim, dtype, seed, fox=fox, device=device)
    return {n: t.squeeze(2).contiguous() for n, t in d.items()}


def sampled_rows(seq_len, n, chunk=128, seed=1):
    """Query positions checked on long sequences: always 0, chunk-1, chunk,
    seq_len-1, plus distinct uniform draws (seed 1), sorted."""
    fixed = {0, min(chunk - 1, seq_len - 1), min(chunk, seq_len - 1), seq_len - 1}
    g = _gen(seed, "cpu")
    perm = torch.randperm(seq_len, generator=g).tolist()
    rows = set(fixed)
    for p in perm:
        if len(rows) >= n:
            break
        rows.add(p)
    return sorted(rows)
