"""GPU parity of the bf16 tensor-core prefill against the fp64 oracle.

Tolerance (bf16 inputs and outputs, fp32 accumulation): max|dout| <= 2e-2 and
max|dlse| <= 1e-2, elementwise over every checked row.  Small cases check
every row; the full-size workloads check sampled query rows, computed by the
oracle one row at a time."""
import pytest
import torch

import oracle
import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import workloads as wl
from helpers import NAMES, max_err, record_margin, to64

pytestmark = pytest.mark.gpu
TOL_OUT, TOL_LSE = 2e-2, 1e-2
DEV = torch.device("cuda:0")


def run(x, rows=None, chunk=0):
    g = {n: t.to(DEV) for n, t in x.items()}
    out, lse = pa.path_attn_prefill_fwd(g["q"], g["k"], g["v"], g["w"], g["beta"],
                                        log_f=g.get("log_f"), chunk=chunk)
    torch.cuda.synchronize()
    assert pa.path_attn_device_status() == 0
    B, H, L, d = x["q"].shape
    flat = lambda t: t.reshape((B * H,) + tuple(t.shape[2:]))
    args = [to64(flat(x[n])) for n in NAMES]
    lf = to64(flat(x["log_f"])) if "log_f" in x else None
    ro, rl = oracle.prefill(*args, log_f=lf, rows=rows)
    go, gl = to64(flat(out)), to64(flat(lse))
    if rows is not None:
        go, gl = go[:, rows], gl[:, rows]
    return max_err(go, ro), max_err(gl, rl)


@pytest.mark.parametrize("L", [1, 128, 200, 1000])
def test_small_all_rows(L):
    eo, el = run(wl.prefill_inputs(1, 2, L, 128, "bf16", seed=L))
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


def test_multi_batch_ragged():
    eo, el = run(wl.prefill_inputs(3, 2, 700, 128, "bf16", seed=11))
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


def test_beta_near_two():
    eo, el = run(wl.prefill_inputs(1, 2, 1500, 128, "bf16", seed=12, beta_mu=2.0))
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


def test_fox_small():
    eo, el = run(wl.prefill_inputs(2, 2, 1000, 128, "bf16", seed=13, fox=True))
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


def test_beta_zero_is_causal_attention():
    x = wl.prefill_inputs(1, 2, 600, 128, "bf16", seed=14)
    x["beta"] = torch.zeros_like(x["beta"])
    eo, el = run(x)
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


def test_repeat_calls_are_deterministic():
    x = wl.prefill_inputs(1, 3, 900, 128, "bf16", seed=15)
    g = {n: t.to(DEV) for n, t in x.items()}
    o1, l1 = pa.path_attn_prefill_fwd(g["q"], g["k"], g["v"], g["w"], g["beta"])
    o2, l2 = pa.path_attn_prefill_fwd(g["q"], g["k"], g["v"], g["w"], g["beta"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def stages(g, out, lse):
    """The prep and the scan as two calls: the scan starts after the prep has
    finished."""
    ws = pa.path_attn_prefill_prep(g["q"], g["k"], g["v"], g["w"], g["beta"],
                                   log_f=g.get("log_f"))
    pa.path_attn_prefill_scan(g["q"], g["w"], g["v"], ws, log_f=g.get("log_f"), out=out,
                              lse=lse)
    return ws


@pytest.mark.slow
@pytest.mark.parametrize("shape", [(8, 12, 4096, 128, False), (8, 12, 4096, 128, True),
                                   (8, 12, 4096, 64, False), (3, 2, 700, 128, False),
                                   (2, 3, 1000, 96, True)])
def test_fused_call_equals_stages(shape):
    """In the one-call forward the scan's tiles start while the prep still
    runs, each once the prep's counter for its head is complete.  Every tile
    does the same arithmetic as in the two-call form, so the outputs must be
    identical bit for bit, on every repeat; a tile that read a row, chunk
    product or own-chunk output before it was written would differ."""
    B, H, L, d, fox = shape
    x = wl.prefill_inputs(B, H, L, d, "bf16", seed=90 + L + d, fox=fox, device="cuda")
    out0, lse0 = torch.empty_like(x["q"]), torch.empty(B, H, L, device=DEV)
    ws = stages(x, out0, lse0)
    out, lse = torch.empty_like(out0), torch.empty_like(lse0)
    for _ in range(8):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        pa.path_attn_prefill_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"],
                                 log_f=x.get("log_f"), out=out, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        assert pa.path_attn_device_status() == 0
        assert torch.equal(out, out0) and torch.equal(lse, lse0)


@pytest.mark.slow
@pytest.mark.parametrize("B,H,L,fox", [(4, 32, 2048, False), (1, 73, 2000, True)])
def test_uneven_head_groups(B, H, L, fox):
    """The scan hands out its tiles by groups of heads; 128 heads of 16 chunks
    go in groups of 26 (the last of 24), 73 heads of 16 chunks (the last one
    ragged) in groups of 25 (the last of 23): every tile of every head must be
    computed once, checked on sampled rows of every head."""
    x = wl.prefill_inputs(B, H, L, 128, "bf16", seed=B * H + L, fox=fox)
    rows = wl.sampled_rows(L, 48)
    eo, el = run(x, rows=rows)
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


@pytest.mark.slow
@pytest.mark.parametrize("wname", ["PREFILL_4K", "FOX_4K", "PREFILL_32K"])
def test_full_size_sampled_rows(wname):
    """The full-size prefill workloads (B8 H12 L4096; PaTH-FoX; B1 H12 L32768
    with beta mostly near 2) in the launch configuration the benchmark times,
    checked on sampled query rows of every head (512 rows for the long
    context, 64 per head otherwise)."""
    w = getattr(wl, wname)
    x = wl.workload_inputs(w, seed=0, device="cuda")
    n = w.sampled_rows or 64
    rows = wl.sampled_rows(w.seq_len, n)
    eo, el = run(x, rows=rows)
    record_margin("prefill_" + wname.lower(), max_dout=eo, tol_out=TOL_OUT, max_dlse=el,
                  tol_lse=TOL_LSE, rows_per_head=len(rows), heads=w.batch * w.heads)
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


@pytest.mark.parametrize("d,L,chunk,fox", [(64, 257, 32, True), (32, 190, 16, False),
                                           (96, 129, 64, False), (36, 200, 0, False)])
def test_cuda_core_route_other_head_dims(d, L, chunk, fox):
    """bf16 with a chunk other than 128 (or a head_dim not a multiple of 8)
    runs on the CUDA cores (fp32 inside, bf16 in and out); same tolerance."""
    eo, el = run(wl.prefill_inputs(2, 2, L, d, "bf16", seed=d + L, fox=fox), chunk=chunk)
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


@pytest.mark.slow
@pytest.mark.parametrize("fox", [False, True])
def test_head_dim_64_full_size(fox):
    """B8 H12 L4096 head_dim 64 (the head_dim-64 scan, the prep reading the
    64-wide tensors directly), 64 sampled rows of every head."""
    x = wl.prefill_inputs(8, 12, 4096, 64, "bf16", seed=0, fox=fox, device="cuda")
    rows = wl.sampled_rows(4096, 64)
    eo, el = run(x, rows=rows)
    record_margin("prefill_d64_4k" + ("_fox" if fox else ""), max_dout=eo, tol_out=TOL_OUT,
                  max_dlse=el, tol_lse=TOL_LSE)
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


@pytest.mark.parametrize("d,L,chunk,fox", [(64, 300, 0, False), (64, 700, 128, True),
                                           (64, 1, 0, True), (64, 129, 0, False),
                                           (32, 129, 0, False), (96, 1, 0, True),
                                           (120, 260, 0, False)])
def test_padded_tensor_core_route(d, L, chunk, fox):
    """bf16 with head_dim a multiple of 8 below 128 and chunk 128 (the
    default) on the tensor cores: head_dim 64 on its own scan, the others on
    zero-padded copies; the caller's scale kept; same tolerance."""
    eo, el = run(wl.prefill_inputs(2, 3, L, d, "bf16", seed=d + L + 1, fox=fox), chunk=chunk)
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)


def test_maximum_batch_heads():
    """batch * heads at its limit of 65535, one token each: 65535 prep jobs
    and scan tiles spread over the persistent grids (every tile is a first
    chunk, whose result is the prep's own block)."""
    L = 1
    B, H = 65535 // 5, 5
    x = wl.prefill_inputs(B, H, L, 128, "bf16", seed=40 + L)
    g = {n: t.to(DEV) for n, t in x.items()}
    out, lse = pa.path_attn_prefill_fwd(g["q"], g["k"], g["v"], g["w"], g["beta"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status() == 0
    # every head is independent: check a spread of heads with the oracle
    flat = lambda t: t.reshape((B * H,) + tuple(t.shape[2:]))
    heads = [0, 1, 777, 32768, B * H - 2, B * H - 1]
    args = [to64(flat(x[n])[heads]) for n in NAMES]
    ro, rl = oracle.prefill(*args)
    assert max_err(to64(flat(out)[heads]), ro) <= TOL_OUT
    assert max_err(to64(flat(lse)[heads]), rl) <= TOL_LSE
    too_many = pa.PrefillDesc(65536, 1, L, 128, pa.PATH_BF16, 0.088, 0)
    assert pa.path_attn_prefill_workspace_size(too_many) == 0
