"""Shared test helpers: run the CUDA path through the binding and the fp64
oracle on the same seeded inputs (the oracle sees exactly the values the GPU
receives, upcast to float64)."""
import numpy as np
import torch

import oracle
import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import workloads as wl

NAMES = ("q", "k", "v", "w", "beta")


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def gpu_prefill(x, chunk=0, scale=None):
    dev = torch.device("cuda:0")
    g = {n: t.to(dev) for n, t in x.items()}
    out, lse = pa.path_attn_prefill_fwd(g["q"], g["k"], g["v"], g["w"], g["beta"],
                                        log_f=g.get("log_f"), chunk=chunk, scale=scale)
    torch.cuda.synchronize()
    assert pa.path_attn_device_status() == 0
    return to64(out), to64(lse)


def oracle_prefill(x, rows=None, scale=None):
    args = [to64(x[n]) for n in NAMES]
    lf = to64(x["log_f"]) if "log_f" in x else None
    return oracle.prefill(*args, log_f=lf, rows=rows, scale=scale)


def max_err(a, b):
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def record_margin(test, **values):
    """Prints a measured parity margin (the largest error a test saw next to
    its tolerance) and, when the environment variable PATH_ATTN_MARGINS
    names a file, appends it there as one JSON line."""
    import json
    import os
    line = json.dumps({"test": test, **values}, sort_keys=True)
    print("margin", line, flush=True)
    path = os.environ.get("PATH_ATTN_MARGINS")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")
