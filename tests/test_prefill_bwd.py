"""Parity of the prefill backward (path_attn_prefill_bwd, CUDA cores, fp32
arithmetic) with the fp64 oracle's reverse-mode gradients, on the same
seeded inputs (the oracle sees exactly the values the GPU receives).

Tolerance: every gradient G is compared as max|G_gpu - G_ref| / max(1, max|G_ref|).
fp32 outputs: 1e-4 (fp32 accumulation over at most a few thousand terms,
relative error ~1e-6 per term).  bf16 outputs: 2e-2, from the bf16 rounding
of the output itself (2^-9 relative) plus the rounding of the forward's bf16
`out` that enters D = dout . out, whose error reaches every dlogit through
P (D + ...) and is then amplified by at most the row length's worth of
cancellation in the key-side sums; measured errors sit well inside it.
"""
import numpy as np
import pytest
import torch

import oracle
import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import workloads as wl
from helpers import record_margin, to64

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dw", "dbeta")


def run(x, chunk=0, use_dlse=False, fwd_chunk=0, heads=None, scale=None, workspace_bytes=None):
    dev = torch.device("cuda:0")
    g = {n: t.to(dev) for n, t in x.items()}
    gen = torch.Generator().manual_seed(1234)
    dout = torch.randn(g["q"].shape, generator=gen).to(g["q"].dtype)
    dlse = torch.randn(g["beta"].shape, generator=gen) if use_dlse else None
    out, lse = pa.path_attn_prefill_fwd(g["q"], g["k"], g["v"], g["w"], g["beta"],
                                        log_f=g.get("log_f"), chunk=fwd_chunk, scale=scale)
    got = pa.path_attn_prefill_bwd(g["q"], g["k"], g["v"], g["w"], g["beta"], out, lse,
                                   dout.to(dev), log_f=g.get("log_f"),
                                   dlse=dlse.to(dev) if dlse is not None else None, chunk=chunk,
                                   scale=scale, workspace_bytes=workspace_bytes)
    torch.cuda.synchronize()
    assert pa.path_attn_device_status() == 0
    sel = slice(None) if heads is None else heads

    def pick(t):
        B, H = t.shape[:2]
        return to64(t.reshape((B * H,) + tuple(t.shape[2:]))[sel])

    args = [pick(x[n]) for n in ("q", "k", "v", "w", "beta")]
    ref = oracle.prefill_bwd(*args, pick(dout), log_f=pick(x["log_f"]) if "log_f" in x else None,
                             dlse=pick(dlse) if dlse is not None else None, scale=scale)
    return {n: pick(t) for n, t in got.items()}, ref


def check(got, ref, tol):
    """Asserts every gradient's normalised error; returns, per gradient, the
    raw elementwise max|G_gpu - G_ref|, the normalised error and max|G_ref|."""
    assert set(got) == set(ref)
    res = {}
    for n in ref:
        raw = float(np.max(np.abs(got[n] - ref[n])))
        top = float(np.max(np.abs(ref[n])))
        err = raw / max(1.0, top)
        res[n] = {"raw": raw, "normalised": err, "max_ref": top}
        assert err <= tol, "%s: normalised error %.3g > %.3g" % (n, err, tol)
    return res


def record_grads(test, res, tol):
    record_margin(test, tol_normalised=tol,
                  **{"%s_%s" % (n, k): v for n, r in res.items() for k, v in r.items()})


def test_tiny_fp32():
    got, ref = run(wl.prefill_inputs(1, 1, 256, 64, "f32", seed=0))
    check(got, ref, 1e-4)


def test_tiny_fp32_with_dlse_and_fox():
    got, ref = run(wl.prefill_inputs(1, 2, 256, 64, "f32", seed=2, fox=True), use_dlse=True)
    assert "dlog_f" in got
    check(got, ref, 1e-4)


@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
@pytest.mark.parametrize("L", [1, 100, 300])
def test_chunks_and_ragged_tails(chunk, L):
    got, ref = run(wl.prefill_inputs(2, 2, L, 32, "f32", seed=L + chunk), chunk=chunk,
                   use_dlse=True)
    check(got, ref, 1e-4)


@pytest.mark.parametrize("d", [4, 96, 128])
def test_head_dims(d):
    got, ref = run(wl.prefill_inputs(1, 2, 200, d, "f32", seed=d), chunk=64)
    check(got, ref, 1e-4)


def test_beta_near_two_fox():
    x = wl.prefill_inputs(1, 2, 384, 64, "f32", seed=8, beta_mu=2.0, fox=True)
    got, ref = run(x, chunk=128, use_dlse=True)
    check(got, ref, 1e-4)


def test_bf16_inputs_tensor_core_forward():
    """bf16, head_dim 128: the forward runs on the tensor cores, the backward
    (chunk 128) on the CUDA cores."""
    got, ref = run(wl.prefill_inputs(1, 2, 520, 128, "bf16", seed=4))
    check(got, ref, 2e-2)


def test_bf16_fox_other_chunk():
    got, ref = run(wl.prefill_inputs(1, 2, 300, 64, "bf16", seed=6, fox=True), chunk=32,
                   use_dlse=True)
    check(got, ref, 2e-2)


def test_headline_shape_sampled_heads():
    """B8 H12 L4096 d128 bf16, the shape of the forward benchmark; two heads
    (first and last) checked in full against the oracle."""
    x = wl.prefill_inputs(8, 12, 4096, 128, "bf16", seed=0)
    got, ref = run(x, heads=[0, 95])
    record_grads("backward_4k_heads_0_95", check(got, ref, 2e-2), 2e-2)


@pytest.mark.parametrize("L", [1, 128, 129, 700])
def test_tensor_core_scan_ragged(L):
    """bf16, head_dim 128, chunk 128: the backward scan on the tensor cores
    (L <= 128 has no earlier key chunk and skips it)."""
    got, ref = run(wl.prefill_inputs(1, 3, L, 128, "bf16", seed=L), use_dlse=True)
    check(got, ref, 2e-2)


def test_bf16_d128_cuda_core_route():
    """chunk 64 keeps bf16 head_dim 128 on the CUDA-core scan."""
    got, ref = run(wl.prefill_inputs(1, 2, 300, 128, "bf16", seed=12), chunk=64)
    check(got, ref, 2e-2)


def test_autograd_function_matches_the_oracle():
    """path_attention under torch autograd: loss.backward() runs the library's
    backward; the gradients (FoX included) match the oracle's."""
    x = wl.prefill_inputs(1, 2, 200, 64, "f32", seed=21, fox=True)
    dev = torch.device("cuda:0")
    t = {n: a.to(dev).requires_grad_(True) for n, a in x.items()}
    out = pa.path_attention(t["q"], t["k"], t["v"], t["w"], t["beta"], log_f=t["log_f"])
    dout = torch.randn(out.shape, generator=torch.Generator().manual_seed(3)).to(dev)
    (out * dout).sum().backward()
    torch.cuda.synchronize()
    ref = oracle.prefill_bwd(*(to64(x[n]) for n in ("q", "k", "v", "w", "beta")), to64(dout),
                             log_f=to64(x["log_f"]))
    got = {"d" + n: to64(t[n].grad) for n in ("q", "k", "v", "w", "beta", "log_f")}
    check(got, ref, 1e-4)


@pytest.mark.parametrize("L", [1, 129, 700])
def test_tensor_core_route_fox(L):
    """PaTH-FoX, bf16, head_dim 128: the forget-gate bias and dlog_f on the
    tensor-core route."""
    got, ref = run(wl.prefill_inputs(1, 3, L, 128, "bf16", seed=40 + L, fox=True), use_dlse=True)
    assert "dlog_f" in got
    check(got, ref, 2e-2)


def test_fox_headline_shape_sampled_heads():
    """PaTH-FoX B8 H12 L4096 d128 bf16 (the FoX benchmark's shape); two heads
    checked in full."""
    x = wl.prefill_inputs(8, 12, 4096, 128, "bf16", seed=0, fox=True)
    got, ref = run(x, heads=[3, 90])
    record_grads("backward_fox_4k_heads_3_90", check(got, ref, 2e-2), 2e-2)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_custom_scale(dtype, d):
    """A scale other than 1/sqrt(d), on both routes."""
    got, ref = run(wl.prefill_inputs(1, 2, 300, d, dtype, seed=17), use_dlse=True, scale=0.37)
    check(got, ref, 1e-4 if dtype == "f32" else 2e-2)


def test_fox_zero_scale_takes_the_cuda_core_route():
    """scale = 0: the logits are the forget-gate bias alone; bf16 d = 128
    PaTH-FoX then runs on the CUDA cores and still matches the oracle."""
    got, ref = run(wl.prefill_inputs(1, 2, 260, 128, "bf16", seed=19, fox=True), use_dlse=True,
                   scale=0.0)
    check(got, ref, 2e-2)


@pytest.mark.parametrize("fox", [False, True])
def test_bounded_workspace_in_passes(fox):
    """A workspace below the one-pass size: the (batch, head) slices run in
    passes (one per pass at the minimum, two and three at a time in between)
    on the tensor-core route; every variant matches the oracle."""
    x = wl.prefill_inputs(2, 3, 700, 128, "bf16", seed=81 + fox, fox=fox)
    desc = pa.PrefillDesc(2, 3, 700, 128, pa.PATH_BF16, 128 ** -0.5, 0)
    least = pa.path_attn_prefill_bwd_workspace_min(desc)
    for ws in (least, int(2.5 * least), 3 * least):
        got, ref = run(x, use_dlse=True, workspace_bytes=ws)
        check(got, ref, 2e-2)


def test_bounded_workspace_cuda_core_route():
    got, ref = run(wl.prefill_inputs(2, 2, 300, 64, "f32", seed=83, fox=True), chunk=64,
                   use_dlse=True, workspace_bytes=1)
    check(got, ref, 1e-4)


@pytest.mark.slow
def test_long_context_shape_bounded_workspace():
    """The long-context shape (B1 H12 L32768, beta mostly near 2) with the
    smallest workspace (one slice per pass, about 1.5 GB against 17 GB in one
    pass); heads 0 and 11 checked in full against the oracle's gradients."""
    w = wl.PREFILL_32K
    x = wl.workload_inputs(w, seed=0, device="cuda")
    desc = pa.PrefillDesc(1, 12, w.seq_len, 128, pa.PATH_BF16, 128 ** -0.5, 0)
    least = pa.path_attn_prefill_bwd_workspace_min(desc)
    assert least < 2e9 < pa.path_attn_prefill_bwd_workspace_size(desc)
    got, ref = run(x, heads=[0, 11], workspace_bytes=least)
    record_grads("backward_32k_heads_0_11_min_workspace", check(got, ref, 2e-2), 2e-2)
