"""Chunk-size autotune (CUDA-core route): the chosen chunk is one of the
allowed sizes, the choice is cached, and the prefill with that chunk matches
the fp64 oracle (fp32 tolerance 1e-4).  Tensor-core route: the scan's
head-group size changes no result, bit for bit, and its autotune picks one
of its candidates."""
import pytest
import torch

import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import autotune
from dependent_positional_attention_gb300 import workloads as wl
from helpers import gpu_prefill, max_err, oracle_prefill

pytestmark = pytest.mark.gpu


def test_autotune_chooses_an_allowed_chunk_and_matches_the_oracle():
    best, times = autotune.autotune_chunk(1, 2, 600, 64, "f32", reps=3)
    assert best in autotune.CUDA_CORE_CHUNKS
    assert set(times) == {0, *autotune.CUDA_CORE_CHUNKS} and all(t > 0 for t in times.values())
    assert autotune.autotune_chunk(1, 2, 600, 64, "f32")[0] == best  # cached
    x = wl.prefill_inputs(1, 2, 600, 64, "f32", seed=5)
    go, gl = gpu_prefill(x, chunk=best)
    ro, rl = oracle_prefill(x)
    assert max_err(go, ro) <= 1e-4 and max_err(gl, rl) <= 1e-4


def test_tensor_core_route_has_one_candidate():
    assert autotune.candidates(128, "bf16") == (128,)
    assert autotune.candidates(64, "bf16") == autotune.CUDA_CORE_CHUNKS


def test_scan_group_changes_no_result():
    """Every head-group size (automatic, one head, uneven groups, all heads,
    more than there are) computes every tile the same way."""
    x = wl.prefill_inputs(2, 12, 2000, 128, "bf16", seed=9, fox=True, device="cuda")
    ref = None
    for g in (0, 1, 5, 7, 24, 1000):
        out, lse = pa.path_attn_prefill_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"],
                                            log_f=x["log_f"], scan_group=g)
        torch.cuda.synchronize()
        assert pa.path_attn_device_status() == 0
        if ref is None:
            ref = (out, lse)
        else:
            assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1]), g


def test_scan_group_autotune_picks_a_candidate():
    best, times = autotune.autotune_scan_group(2, 12, 2048, reps=3)
    assert best in autotune.scan_group_candidates(2, 12) and set(times) == set(
        autotune.scan_group_candidates(2, 12))
    assert all(t > 0 for t in times.values())
    assert autotune.autotune_scan_group(2, 12, 2048)[0] == best  # cached
