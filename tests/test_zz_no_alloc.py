"""The decode step that allocates nothing (path_attn_decode_step_noalloc).

This entry point exists for callers that cannot give the library device
memory: plugins inside a host framework that owns every GPU allocation and
hands its plugins no allocator, and token loops that must not call
cudaMalloc mid-generation (an allocation can synchronise the device).  It
keeps its split-KV partials in a fixed 8 MiB device array instead of a caller
workspace.  The kernels are those of path_attn_decode_step, so on the same
inputs both entry points must give bit-identical outputs and caches; that is
checked here through the C ABI (ctypes, raw device pointers) and through the
Python wrapper, on two consecutive decode steps per case.
The file sorts last so a stop-at-first-failure run has already run the rest.
"""
import ctypes

import pytest
import torch

import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SCRATCH_FLOATS = 1 << 21  # the fixed scratch: 8 MiB of fp32
KEYS_PER_SPLIT = 1024


def _lib():
    from dependent_positional_attention_gb300 import build as pa_build
    pa_build.build()
    return pa.load_library()


def _random_caches(B, H, cap, d, filled, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    kc = torch.zeros((B, H, cap, d), device=DEV, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    if filled:
        kc[:, :, :filled] = torch.randn((B, H, filled, d), generator=g, device=DEV).to(kc.dtype)
        vc[:, :, :filled] = torch.randn((B, H, filled, d), generator=g, device=DEV).to(kc.dtype)
    return kc, vc


def _two_steps(lib, kc, vc, L0, seed, via_wrapper):
    """Runs decode steps at cache_len L0 and L0 + 1 through the workspace
    entry point on a copy of the caches and through the allocation-free one
    on the caches themselves; both must agree bit for bit after each step."""
    B, H, cap, d = kc.shape
    kc_ref, vc_ref = kc.clone(), vc.clone()
    desc = pa.decode_desc(kc)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for s in range(2):
        g = wl.decode_token(B, H, d, "bf16", seed=seed + s, device="cuda")
        ref = pa.path_attn_decode_step(kc_ref, vc_ref, L0 + s, g["q"], g["k"], g["v"], g["w"],
                                       g["beta"])
        out = torch.full_like(g["q"], float("nan"))
        if via_wrapper:
            pa.path_attn_decode_step_noalloc(kc, vc, L0 + s, g["q"], g["k"], g["v"], g["w"],
                                             g["beta"], out)
        else:
            rc = lib.path_attn_decode_step_noalloc(
                ctypes.byref(desc), p(kc), p(vc), L0 + s, p(g["q"]), p(g["k"]), p(g["v"]),
                p(g["w"]), p(g["beta"]), p(out), stream)
            assert rc == pa.PATH_OK, lib.path_attn_last_error()
        torch.cuda.synchronize()
        assert torch.equal(out, ref), (s, (out.float() - ref.float()).abs().max().item())
        assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref), s
    assert pa.path_attn_device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("via_wrapper", [False, True])
def test_noalloc_decode_equals_workspace_decode(d, via_wrapper):
    """A cache built by the prefill-state builder, 2500 tokens: three splits."""
    lib = _lib()
    B, H, L0 = 2, 3, 2500
    x = wl.prefill_inputs(B, H, L0, d, "bf16", seed=21, device="cuda")
    kc = torch.zeros((B, H, L0 + 2, d), device=DEV, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    pa.path_attn_build_kcache(x["k"], x["w"], x["beta"], kc)
    vc[:, :, :L0] = x["v"]
    _two_steps(lib, kc, vc, L0, 500 + d, via_wrapper)


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_decode_from_an_empty_cache(d):
    """cache_len 0 (no split runs, the new token alone) and then 1."""
    lib = _lib()
    kc, vc = _random_caches(2, 2, 4, d, 0, seed=3)
    _two_steps(lib, kc, vc, 0, 700 + d, via_wrapper=False)


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_decode_next_to_the_scratch_limit(d):
    """A step whose partials fill the fixed scratch to within one split of a
    head: batch*heads*splits*(head_dim + 2) floats just below 2^21, the
    second step crossing from one split per head to two."""
    lib = _lib()
    BH = SCRATCH_FLOATS // (2 * (d + 2))
    assert BH * 2 * (d + 2) <= SCRATCH_FLOATS < (BH + 1) * 2 * (d + 2)
    L0 = KEYS_PER_SPLIT
    kc, vc = _random_caches(1, BH, L0 + 2, d, L0, seed=5)
    _two_steps(lib, kc, vc, L0, 900 + d, via_wrapper=False)


def test_noalloc_decode_rejects_a_step_beyond_the_scratch():
    """One head more than fits: PATH_ERR_INVALID_ARG before any launch, with
    both sizes in the message; the caches are left untouched."""
    lib = _lib()
    d = 128
    BH = SCRATCH_FLOATS // (2 * (d + 2)) + 1
    L0 = KEYS_PER_SPLIT + 1
    kc, vc = _random_caches(1, BH, L0 + 1, d, 0, seed=6)
    g = wl.decode_token(1, BH, d, "bf16", seed=11, device="cuda")
    out = torch.empty_like(g["q"])
    with pytest.raises(pa.PathAttnError) as e:
        pa.path_attn_decode_step_noalloc(kc, vc, L0, g["q"], g["k"], g["v"], g["w"], g["beta"],
                                         out)
    assert e.value.status == pa.PATH_ERR_INVALID_ARG
    assert "8388608" in str(e.value)
    torch.cuda.synchronize()
    assert int(kc.abs().sum().item()) == 0 and pa.path_attn_device_status() == 0
