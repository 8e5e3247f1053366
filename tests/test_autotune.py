"""Chunk-size autotune (CUDA-core route): the chosen chunk is one of the
allowed sizes, the choice is cached, and the prefill with that chunk matches
the fp64 oracle (fp32 tolerance 1e-4)."""
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
