"""GPU parity of the PaTH-FoX decode step against the fp64 oracle.

The oracle sums the forget-gate logs of each cached key straight from a log f
history (sum_{s=j+1}^{t} log f_s); the GPU keeps per-key prefixes F_j and adds
F_t - F_j.  Tolerance, as for the PaTH decode: max|dout| <= 2e-2."""
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


def setup_cache(B, H, d, L0, cap, seed):
    """GPU caches (keys, values, forget-gate prefixes) after a FoX prefill of
    L0 tokens, and the oracle's own fp64 copies from the same inputs."""
    x = wl.prefill_inputs(B, H, L0, d, "bf16", seed=seed, fox=True)
    kc = torch.zeros((B, H, cap, d), device=DEV, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    fc = torch.zeros((B, H, cap), device=DEV, dtype=torch.float32)
    pa.path_attn_build_kcache(x["k"].to(DEV), x["w"].to(DEV), x["beta"].to(DEV), kc)
    vc[:, :, :L0] = x["v"].to(DEV)
    pa.path_attn_fox_prefix(x["log_f"].to(DEV), fc)
    BH = B * H
    flat = lambda t: t.reshape((BH,) + tuple(t.shape[2:]))
    ok = oracle.build_kcache(to64(flat(x["k"])), to64(flat(x["w"])), to64(flat(x["beta"])),
                             cap=cap)
    ov = np.zeros_like(ok)
    ov[:, :L0] = to64(flat(x["v"]))
    lf = np.zeros((BH, cap))
    lf[:, :L0] = to64(flat(x["log_f"]))
    torch.cuda.synchronize()
    assert pa.path_attn_device_status() == 0
    return (kc, vc, fc), (ok, ov, lf), x


@pytest.mark.parametrize("L0", [1, 700, 2100])
def test_fox_decode_matches_oracle(L0):
    B, H, d, steps = 2, 3, 128, 3
    (kc, vc, fc), (ok, ov, lf), x = setup_cache(B, H, d, L0, L0 + steps, seed=L0)
    flat = lambda t: t.reshape((B * H,) + tuple(t.shape[2:]))
    # the prefix written by path_attn_fox_prefix
    F_ref = np.cumsum(to64(flat(x["log_f"])), axis=1)
    F_gpu = to64(flat(fc[:, :, :L0]))
    assert np.max(np.abs(F_gpu - F_ref)) <= 1e-5 * max(1.0, np.max(np.abs(F_ref)))
    for t in range(steps):
        tok = wl.decode_token(B, H, d, "bf16", seed=20_000 + L0 + t, fox=True)
        g = {n: v.to(DEV) for n, v in tok.items()}
        out = pa.path_attn_decode_step_fox(kc, vc, fc, L0 + t, g["q"], g["k"], g["v"], g["w"],
                                           g["beta"], g["log_f"])
        ro = oracle.decode_step_fox(ok, ov, lf, L0 + t,
                                    *(to64(flat(tok[n])) for n in ("q", "k", "v", "w", "beta")),
                                    to64(flat(tok["log_f"])))
        torch.cuda.synchronize()
        err = max_err(to64(flat(out)), ro)
        assert err <= TOL, (t, err)
    # the step appended F_t at each slot
    F_all = np.cumsum(lf, axis=1)[:, :L0 + steps]
    F_gpu = to64(flat(fc[:, :, :L0 + steps]))
    assert np.max(np.abs(F_gpu - F_all)) <= 1e-5 * max(1.0, np.max(np.abs(F_all)))
    assert pa.path_attn_device_status() == 0


def test_fox_decode_from_empty_reproduces_fox_prefill():
    """Decoding a whole sequence token by token from an empty cache gives the
    PaTH-FoX prefill rows of the oracle (inference bullet of section 3)."""
    B, H, L, d = 1, 2, 96, 128
    x = wl.prefill_inputs(B, H, L, d, "bf16", seed=31, fox=True)
    kc = torch.zeros((B, H, L, d), device=DEV, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    fc = torch.zeros((B, H, L), device=DEV, dtype=torch.float32)
    xs = {n: v.to(DEV) for n, v in x.items()}
    outs = []
    for t in range(L):
        sl = lambda n: xs[n][:, :, t].contiguous()
        outs.append(pa.path_attn_decode_step_fox(kc, vc, fc, t, sl("q"), sl("k"), sl("v"),
                                                 sl("w"), sl("beta"), sl("log_f")))
    torch.cuda.synchronize()
    assert pa.path_attn_device_status() == 0
    flat = lambda t: t.reshape((B * H,) + tuple(t.shape[2:]))
    ref, _ = oracle.prefill(*(to64(flat(x[n])) for n in ("q", "k", "v", "w", "beta")),
                            log_f=to64(flat(x["log_f"])))
    got = np.stack([to64(flat(o)) for o in outs], axis=1)
    assert max_err(got, ref) <= TOL


def test_fox_decode_with_open_gates_is_the_path_step():
    """log f = 0 (forget gates fully open): bit-identical to the PaTH step."""
    B, H, d, L0 = 1, 2, 128, 1500
    (kc, vc, fc), _, _ = setup_cache(B, H, d, L0, L0 + 1, seed=9)
    fc.zero_()
    kc2, vc2 = kc.clone(), vc.clone()
    tok = {n: v.to(DEV) for n, v in wl.decode_token(B, H, d, "bf16", seed=77).items()}
    zero = torch.zeros((B, H), device=DEV, dtype=torch.float32)
    a = pa.path_attn_decode_step_fox(kc, vc, fc, L0, tok["q"], tok["k"], tok["v"], tok["w"],
                                     tok["beta"], zero)
    b = pa.path_attn_decode_step(kc2, vc2, L0, tok["q"], tok["k"], tok["v"], tok["w"], tok["beta"])
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(kc, kc2) and torch.equal(vc, vc2)


@pytest.mark.slow
def test_fox_decode_full_size_all_steps_sampled_heads():
    """The decode workload with forget gates: B16 H12 d128, a PaTH-FoX cache of
    65536 tokens (keys by the prefill-state builder, prefixes by
    path_attn_fox_prefix), then all 256 steps with the benchmark's seeds; 8
    sampled (b, h) heads compared with the oracle's FoX decode at every step.
    The largest error over the steps and the final key-cache drift are
    recorded."""
    w = wl.DECODE_64K
    B, H, d, L0, steps = w.batch, w.heads, w.head_dim, w.prefix_len, w.steps
    cap = L0 + steps
    BH = B * H
    heads = sorted(torch.randperm(BH, generator=torch.Generator().manual_seed(2))[:8].tolist())
    x = wl.prefill_inputs(B, H, L0, d, "bf16", seed=0, fox=True, device="cuda")
    kc = torch.zeros((B, H, cap, d), device=DEV, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    fc = torch.zeros((B, H, cap), device=DEV, dtype=torch.float32)
    pa.path_attn_build_kcache(x["k"], x["w"], x["beta"], kc)
    vc[:, :, :L0] = x["v"]
    pa.path_attn_fox_prefix(x["log_f"], fc)
    flat = lambda t: t.reshape((BH,) + tuple(t.shape[2:]))
    sel = lambda t: to64(flat(t)[heads])
    ok = oracle.build_kcache(sel(x["k"]), sel(x["w"]), sel(x["beta"]), cap=cap)
    ov = np.zeros_like(ok)
    ov[:, :L0] = sel(x["v"])
    lf = np.zeros((len(heads), cap))
    lf[:, :L0] = sel(x["log_f"])
    del x
    errs = []
    for t in range(steps):
        g = wl.decode_token(B, H, d, "bf16", seed=10_000 + t, device="cuda", fox=True)
        out = pa.path_attn_decode_step_fox(kc, vc, fc, L0 + t, g["q"], g["k"], g["v"], g["w"],
                                           g["beta"], g["log_f"])
        ro = oracle.decode_step_fox(ok, ov, lf, L0 + t,
                                    *(sel(g[n]) for n in ("q", "k", "v", "w", "beta")),
                                    sel(g["log_f"]))
        torch.cuda.synchronize()
        errs.append(max_err(sel(out), ro))
    assert pa.path_attn_device_status() == 0
    gk = sel(kc)
    drift_abs = float(np.max(np.abs(gk - ok)))
    drift_rel = float(np.max(np.linalg.norm(gk - ok, axis=-1)
                             / np.maximum(np.linalg.norm(ok, axis=-1), 1e-30)))
    F_ref = np.cumsum(lf, axis=1)
    F_err = float(np.max(np.abs(sel(fc) - F_ref)))
    record_margin("fox_decode_64k_256_steps", max_dout=max(errs), tol_out=TOL,
                  dout_first_step=errs[0], dout_last_step=errs[-1],
                  worst_step=int(np.argmax(errs)), final_cache_drift_abs=drift_abs,
                  final_cache_drift_rel=drift_rel, prefix_abs_err=F_err)
    assert len(errs) == steps
    assert max(errs) <= TOL, (int(np.argmax(errs)), max(errs))
    assert F_err <= 1e-5 * max(1.0, float(np.max(np.abs(F_ref))))
