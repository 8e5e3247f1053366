"""GPU parity of the decode step and the key-cache build against the fp64
oracle.  The oracle builds its own cache in fp64 from the same bf16 inputs
(it never sees a GPU result) and never re-rounds it; the GPU cache is
re-rounded to bf16 after every update.  Tolerance: max|dout| <= 2e-2."""
import numpy as np
import pytest
import torch

import oracle
import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import workloads as wl
from helpers import max_err, record_margin, to64

pytestmark = pytest.mark.gpu
TOL = 2e-2
DEV = torch.device("cuda:0")


def run_case(B, H, d, L0, steps, seed, cap=None, heads=None, gen_device="cpu"):
    """Builds GPU and oracle caches for L0 prefilled tokens, runs `steps`
    decode steps on both and returns (cache build error in bf16 ulps, the
    max|dout| of every step, GPU k cache, GPU v cache, tokens, oracle k
    cache)."""
    cap = cap or (L0 + steps)
    x = wl.prefill_inputs(B, H, max(L0, 1), d, "bf16", seed=seed, device=gen_device)
    toks = [wl.decode_token(B, H, d, "bf16", seed=10_000 + seed + t, device=gen_device)
            for t in range(steps)]
    kc = torch.zeros((B, H, cap, d), device=DEV, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    if L0 > 0:
        pa.path_attn_build_kcache(x["k"].to(DEV), x["w"].to(DEV), x["beta"].to(DEV), kc)
        vc[:, :, :L0] = x["v"].to(DEV)
    torch.cuda.synchronize()
    assert pa.path_attn_device_status() == 0
    BH = B * H
    sel = list(range(BH)) if heads is None else list(heads)
    flat = lambda t: t.reshape((BH,) + tuple(t.shape[2:]))
    # oracle: own fp64 cache from the same bf16 inputs, selected heads only
    if L0 > 0:
        ok = oracle.build_kcache(to64(flat(x["k"])[sel]), to64(flat(x["w"])[sel]),
                                 to64(flat(x["beta"])[sel]), cap=cap)
        ov = np.zeros_like(ok)
        ov[:, :L0] = to64(flat(x["v"])[sel])
        gk = to64(flat(kc[:, :, :L0])[sel])
        cache_err = float(np.max(np.abs(gk - ok[:, :L0]) / (np.abs(ok[:, :L0]) * 2 ** -8 + 1e-3)))
    else:
        ok = np.zeros((len(sel), cap, d))
        ov = np.zeros_like(ok)
        cache_err = 0.0
    errs = []
    for t in range(steps):
        g = {n: v.to(DEV) for n, v in toks[t].items()}
        out = pa.path_attn_decode_step(kc, vc, L0 + t, g["q"], g["k"], g["v"], g["w"], g["beta"])
        ro = oracle.decode_step(ok, ov, L0 + t, *(to64(flat(toks[t][n])[sel])
                                                 for n in ("q", "k", "v", "w", "beta")))
        torch.cuda.synchronize()
        errs.append(max_err(to64(flat(out)[sel]), ro))
    assert pa.path_attn_device_status() == 0
    return cache_err, errs, kc, vc, toks, ok


@pytest.mark.parametrize("L0", [1, 63, 1000, 2100])
def test_decode_small(L0):
    cache_err, errs, *_ = run_case(2, 3, 128, L0, 4, seed=L0)
    assert cache_err <= 1.0, cache_err
    assert max(errs) <= TOL, errs


def test_decode_head_dim_64():
    cache_err, errs, *_ = run_case(1, 2, 64, 777, 3, seed=5)
    assert cache_err <= 1.0 and max(errs) <= TOL, (cache_err, errs)


def test_decode_empty_cache_returns_v():
    _, errs, kc, vc, toks, _ = run_case(1, 2, 128, 0, 1, seed=6, cap=4)
    assert max(errs) <= TOL
    # softmax over the single new key: out == v_t, and slot 0 holds k_t / v_t
    v = toks[0]["v"].to(DEV)
    assert torch.equal(vc[:, :, 0], v) and torch.equal(kc[:, :, 0], toks[0]["k"].to(DEV))


def test_decode_fills_last_slot():
    cache_err, errs, kc, *_ = run_case(1, 1, 128, 300, 2, seed=7, cap=302)
    assert max(errs) <= TOL


def test_decode_rejects_full_cache():
    kc = torch.zeros((1, 1, 8, 128), device=DEV, dtype=torch.bfloat16)
    t = torch.zeros((1, 1, 128), device=DEV, dtype=torch.bfloat16)
    b = torch.zeros((1, 1), device=DEV, dtype=torch.float32)
    with pytest.raises(pa.PathAttnError):
        pa.path_attn_decode_step(kc, kc.clone(), 8, t, t, t, t, b)


def cache_drift(kc, ok, heads, n):
    """Drift of the GPU key cache (re-rounded to bf16 after every update) from
    the oracle's fp64 cache over the first n slots of the given heads: the
    largest absolute difference and the largest per-key relative difference
    |k_gpu - k_ref| / |k_ref|."""
    BH = kc.shape[0] * kc.shape[1]
    gk = to64(kc.reshape((BH,) + tuple(kc.shape[2:]))[heads][:, :n])
    rk = ok[:, :n]
    diff = np.abs(gk - rk)
    rel = np.linalg.norm(gk - rk, axis=-1) / np.maximum(np.linalg.norm(rk, axis=-1), 1e-30)
    return float(diff.max()), float(rel.max())


@pytest.mark.slow
def test_decode_full_size_all_steps_sampled_heads():
    """The decode workload in full: B16 H12 d128, 65536 cached tokens built by
    the prefill-state builder, then all 256 steps with the benchmark's seeds;
    8 sampled (b, h) heads compared with the oracle at every step.  The GPU
    re-rounds every cached key to bf16 after each in-place update while the
    oracle keeps fp64, so the error can grow with the step count; the
    largest error over the 256 steps and the final cache drift are
    recorded."""
    w = wl.DECODE_64K
    g = torch.Generator().manual_seed(1)
    heads = sorted(torch.randperm(w.batch * w.heads, generator=g)[:8].tolist())
    cache_err, errs, kc, _, _, ok = run_case(w.batch, w.heads, w.head_dim, w.prefix_len,
                                             w.steps, seed=0, cap=w.prefix_len + w.steps,
                                             heads=heads, gen_device="cuda")
    drift_abs, drift_rel = cache_drift(kc, ok, heads, w.prefix_len + w.steps)
    record_margin("decode_64k_256_steps", max_dout=max(errs), tol_out=TOL,
                  dout_first_step=errs[0], dout_last_step=errs[-1],
                  worst_step=int(np.argmax(errs)), cache_build_ulp=cache_err,
                  final_cache_drift_abs=drift_abs, final_cache_drift_rel=drift_rel)
    assert cache_err <= 1.0, cache_err
    assert len(errs) == w.steps
    assert max(errs) <= TOL, (int(np.argmax(errs)), max(errs))
