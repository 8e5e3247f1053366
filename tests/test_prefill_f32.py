"""GPU parity of the fp32 prefill path against the fp64 oracle.

Tolerance: max|dout| <= 1e-4 and max|dlse| <= 1e-4 (fp32 path), elementwise
over every row."""
import pytest
import torch

from dependent_positional_attention_gb300 import workloads as wl
from helpers import gpu_prefill, max_err, oracle_prefill, record_margin

pytestmark = pytest.mark.gpu
TOL = 1e-4


def check(x, chunk=0, scale=None):
    out, lse = gpu_prefill(x, chunk, scale)
    ro, rl = oracle_prefill(x, scale=scale)
    e_out, e_lse = max_err(out, ro), max_err(lse, rl)
    assert e_out <= TOL and e_lse <= TOL, (e_out, e_lse)
    return e_out, e_lse


def test_tiny_config_exact():
    """B1 H1 L256 d64 fp32, seed 0 (the tiny PaTH forward workload)."""
    e_out, e_lse = check(wl.workload_inputs(wl.TINY_F32, seed=0))
    record_margin("prefill_tiny_f32", max_dout=e_out, max_dlse=e_lse, tol_out=TOL, tol_lse=TOL)


@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
@pytest.mark.parametrize("L", [1, 63, 200])
def test_chunk_invariance_and_ragged_tail(chunk, L):
    check(wl.prefill_inputs(2, 2, L, 64, "f32", seed=L), chunk=chunk)


def test_head_dim_128_and_multi_head():
    check(wl.prefill_inputs(1, 3, 300, 128, "f32", seed=3), chunk=64)


def test_fox_f32():
    check(wl.prefill_inputs(2, 1, 256, 64, "f32", seed=4, fox=True), chunk=32)


def test_beta_near_two():
    check(wl.prefill_inputs(1, 2, 384, 64, "f32", seed=5, beta_mu=2.0), chunk=64)


def test_custom_scale():
    check(wl.prefill_inputs(1, 1, 130, 32, "f32", seed=6), chunk=16, scale=0.37)


def test_bounded_wait_reports_timeout():
    """A wait that can never complete gives up after its limit and the host
    reads PATH_ERR_TIMEOUT; the context stays usable afterwards."""
    import dependent_positional_attention_gb300 as pa
    assert pa.path_attn_device_status() == 0
    pa.path_attn_selftest_bounded_wait(2000)
    assert pa.path_attn_device_status() == pa.PATH_ERR_TIMEOUT
    assert pa.path_attn_device_status() == 0
    check(wl.prefill_inputs(1, 1, 64, 64, "f32", seed=7), chunk=64)
