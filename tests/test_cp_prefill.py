"""GPU parity of the sequence-sharded prefill (path_attn_cp_prep /
path_attn_cp_scan).  The ranks run one after another on one GPU and the
all-gather of their exchange blocks is a concatenation in rank order, which is
what ncclAllGather produces.  The gathered result must equal the unsharded
prefill bit for bit (same kernels, same operands, same order of operations per
query tile) and match the fp64 oracle within the bf16 tolerance (max|dout| <=
2e-2, max|dlse| <= 1e-2) on sampled rows."""
import pytest
import torch

import oracle
import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import workloads as wl
from helpers import NAMES, max_err, record_margin, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL_OUT, TOL_LSE = 2e-2, 1e-2


def sharded_prefill(g, world, seq_len):
    """All ranks of a sharded prefill on this GPU; returns (out, lse) in
    global row order and the local row counts."""
    B, H, L, d = g["q"].shape
    log_f = g.get("log_f")
    out = torch.full_like(g["q"], float("nan"))
    lse = torch.full(g["beta"].shape, float("nan"), device=DEV)
    shards = []
    for r in range(world):
        rows = pa.path_attn_cp_rows(B, H, seq_len, world, r).to(DEV)
        loc = {n: g[n].index_select(2, rows).contiguous() for n in NAMES}
        ex, ws = pa.path_attn_cp_prep(loc["q"], loc["k"], loc["v"], loc["w"], loc["beta"],
                                      seq_len, world, r, log_f=log_f)
        shards.append((rows, ex, ws))
    gathered = torch.cat([ex for _, ex, _ in shards])
    for r, (rows, _, ws) in enumerate(shards):
        o, l = pa.path_attn_cp_scan(gathered, ws, B, H, seq_len, world, r, log_f=log_f)
        out.index_copy_(2, rows, o)
        lse.index_copy_(2, rows, l)
    torch.cuda.synchronize()
    assert pa.path_attn_device_status() == 0
    return out, lse, [len(s[0]) for s in shards]


def check(x, world, rows=None, name=None):
    g = {n: t.to(DEV) for n, t in x.items()}
    B, H, L, d = g["q"].shape
    out, lse, counts = sharded_prefill(g, world, L)
    ref_out, ref_lse = pa.path_attn_prefill_fwd(g["q"], g["k"], g["v"], g["w"], g["beta"],
                                                log_f=g.get("log_f"))
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), (
        (out.float() - ref_out.float()).abs().max().item())
    flat = lambda t: t.reshape((B * H,) + tuple(t.shape[2:]))
    args = [to64(flat(x[n])) for n in NAMES]
    lf = to64(flat(x["log_f"])) if "log_f" in x else None
    ro, rl = oracle.prefill(*args, log_f=lf, rows=rows)
    go, gl = to64(flat(out)), to64(flat(lse))
    if rows is not None:
        go, gl = go[:, rows], gl[:, rows]
    eo, el = max_err(go, ro), max_err(gl, rl)
    if name:
        record_margin(name, max_dout=eo, tol_out=TOL_OUT, max_dlse=el, tol_lse=TOL_LSE,
                      world=world, rows_per_rank=counts)
    assert eo <= TOL_OUT and el <= TOL_LSE, (eo, el)
    return counts


@pytest.mark.parametrize("world", [1, 2, 3])
def test_sharded_equals_unsharded_ragged(world):
    counts = check(wl.prefill_inputs(2, 3, 1000, 128, "bf16", seed=61 + world), world)
    assert sum(counts) == 1000


def test_sharded_fox():
    check(wl.prefill_inputs(1, 2, 1500, 128, "bf16", seed=71, fox=True), world=2)


def test_rank_without_rows():
    """Three chunks over four ranks: rank 3 holds nothing, its calls read no
    input, yet its (unused) exchange block takes part in the gather."""
    counts = check(wl.prefill_inputs(1, 2, 300, 128, "bf16", seed=72), world=4)
    assert counts[3] == 0 and sum(counts) == 300


def test_single_position():
    check(wl.prefill_inputs(1, 1, 1, 128, "bf16", seed=73), world=2)


@pytest.mark.slow
def test_long_context_over_eight_ranks():
    """The long-context workload (B1 H12 L32768, beta mostly near 2) sharded
    over eight ranks; 512 sampled rows per head against the oracle."""
    w = wl.PREFILL_32K
    x = wl.workload_inputs(w, seed=0, device="cuda")
    rows = wl.sampled_rows(w.seq_len, w.sampled_rows)
    check(x, world=8, rows=rows, name="cp_prefill_32k_world8")


@pytest.mark.slow
def test_fox_4k_over_four_ranks():
    w = wl.FOX_4K
    x = wl.workload_inputs(w, seed=0, device="cuda")
    check(x, world=4, rows=wl.sampled_rows(w.seq_len, 64), name="cp_prefill_fox_4k_world4")
