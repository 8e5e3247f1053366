"""The decode step that allocates nothing (path_attn_decode_step_noalloc).

This entry point exists for callers that cannot give the library device
memory: plugins inside a host framework that owns every GPU allocation, and
token loops that must not call cudaMalloc mid-generation.  It keeps its
split-KV partials in a fixed device array instead of a caller workspace.
Here it is called through the C ABI (ctypes, raw device pointers) for two
consecutive decode steps and must agree with path_attn_decode_step on the
same inputs, within the decode tolerance used elsewhere (max|dout| <= 2e-2).
The file sorts last so a stop-at-first-failure run has already run the rest.
"""
import ctypes

import pytest
import torch

import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 2e-2
DEV = torch.device("cuda:0")


def test_noalloc_decode_matches_workspace_decode_on_two_steps():
    from dependent_positional_attention_gb300 import build as pa_build
    pa_build.build()
    lib = pa.load_library()
    B, H, d, L0, steps = 2, 3, 128, 2500, 2
    cap = L0 + steps
    x = wl.prefill_inputs(B, H, L0, d, "bf16", seed=21, device="cuda")
    kc = torch.zeros((B, H, cap, d), device=DEV, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    pa.path_attn_build_kcache(x["k"], x["w"], x["beta"], kc)
    vc[:, :, :L0] = x["v"]
    kc_ref, vc_ref = kc.clone(), vc.clone()
    desc = pa.decode_desc(kc)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for s in range(steps):
        g = wl.decode_token(B, H, d, "bf16", seed=500 + s, device="cuda")
        ref = pa.path_attn_decode_step(kc_ref, vc_ref, L0 + s, g["q"], g["k"], g["v"], g["w"],
                                       g["beta"])
        out = torch.empty_like(g["q"])
        rc = lib.path_attn_decode_step_noalloc(
            ctypes.byref(desc), p(kc), p(vc), L0 + s, p(g["q"]), p(g["k"]), p(g["v"]),
            p(g["w"]), p(g["beta"]), p(out), stream)
        assert rc == pa.PATH_OK, lib.path_attn_last_error()
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= TOL, (s, err)
        # the in-place key update and the appended slot agree as well
        assert (kc.float() - kc_ref.float()).abs().max().item() <= TOL
        assert torch.equal(vc, vc_ref)
    assert pa.path_attn_device_status() == 0
