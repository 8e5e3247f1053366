"""C-ABI checks that need no GPU: the library builds, loads on a host
without a driver, exports every entry point include/path_attn.h declares,
and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pa.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "path_attn.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(path_attn_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), "missing export %s" % n
    assert sorted(pa.EXPORTED_SYMBOLS) == names


def test_status_strings(lib):
    assert lib.path_attn_status_string(0) == b"PATH_OK"
    assert lib.path_attn_status_string(4) == b"PATH_ERR_TIMEOUT"
    assert lib.path_attn_version() >= 100


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)       # 8-byte aligned only


def prefill(lib, desc, ws_bytes=1 << 40, ptrs=None, log_f=None):
    p = ptrs or [FAKE] * 5
    return lib.path_attn_prefill_fwd(ctypes.byref(desc), p[0], p[1], p[2], p[3], p[4], log_f,
                                     FAKE, None, FAKE, ws_bytes, None)


def test_prefill_rejects_bad_descriptors(lib):
    D = pa.PrefillDesc
    assert prefill(lib, D(0, 1, 16, 64, 0, 0.1, 0)) == pa.PATH_ERR_INVALID_ARG
    assert prefill(lib, D(1, 1, 0, 64, 0, 0.1, 0)) == pa.PATH_ERR_INVALID_ARG
    assert prefill(lib, D(1, 1, 16, 64, 7, 0.1, 0)) == pa.PATH_ERR_INVALID_ARG
    assert prefill(lib, D(1, 1, 16, 64, 0, float("nan"), 0)) == pa.PATH_ERR_INVALID_ARG
    assert prefill(lib, D(1, 1, 16, 66, 1, 0.1, 0)) == pa.PATH_ERR_UNSUPPORTED  # bf16 d=66
    # bf16 with a head_dim other than 128 takes the CUDA-core route: a valid
    # descriptor, rejected here only for the (deliberately tiny) workspace
    assert prefill(lib, D(1, 1, 16, 64, 1, 0.1, 0), ws_bytes=16) == pa.PATH_ERR_INVALID_ARG
    assert b"workspace" in lib.path_attn_last_error()
    assert prefill(lib, D(1, 1, 16, 130, 0, 0.1, 0)) == pa.PATH_ERR_UNSUPPORTED
    assert prefill(lib, D(1, 1, 16, 64, 0, 0.1, 48)) == pa.PATH_ERR_UNSUPPORTED
    assert prefill(lib, D(1, 1, 16, 128, 1, 0.1, 64)) == pa.PATH_ERR_UNSUPPORTED
    assert lib.path_attn_prefill_workspace_size(ctypes.byref(D(0, 1, 16, 64, 0, 0.1, 0))) == 0
    assert b"batch" in lib.path_attn_last_error()
    # the tensor-core scan's head-group size: >= 0 (0 = automatic)
    assert lib.path_attn_prefill_workspace_size(ctypes.byref(D(1, 1, 16, 128, 1, 0.1, 0, -1))) == 0
    assert b"scan_group" in lib.path_attn_last_error()
    assert (lib.path_attn_prefill_workspace_size(ctypes.byref(D(1, 1, 16, 128, 1, 0.1, 0, 7))) ==
            lib.path_attn_prefill_workspace_size(ctypes.byref(D(1, 1, 16, 128, 1, 0.1, 0, 0))))


def test_prefill_rejects_bad_pointers_and_workspace(lib):
    D = pa.PrefillDesc
    desc = D(2, 3, 100, 64, 0, 0.125, 32)
    need = lib.path_attn_prefill_workspace_size(ctypes.byref(desc))
    assert need > 0
    assert prefill(lib, desc, ws_bytes=need - 1) == pa.PATH_ERR_INVALID_ARG
    assert b"workspace" in lib.path_attn_last_error()
    for i in range(5):
        p = [FAKE] * 5
        p[i] = None
        assert prefill(lib, desc, ptrs=p) == pa.PATH_ERR_INVALID_ARG
        p[i] = ODD
        assert prefill(lib, desc, ptrs=p) == pa.PATH_ERR_INVALID_ARG
    assert prefill(lib, desc, log_f=ODD) == pa.PATH_ERR_INVALID_ARG


def test_workspace_grows_with_problem(lib):
    D = pa.PrefillDesc
    a = lib.path_attn_prefill_workspace_size(ctypes.byref(D(1, 1, 128, 128, 1, 0.1, 0)))
    b = lib.path_attn_prefill_workspace_size(ctypes.byref(D(2, 1, 128, 128, 1, 0.1, 0)))
    c = lib.path_attn_prefill_workspace_size(ctypes.byref(D(1, 1, 129, 128, 1, 0.1, 0)))
    assert 0 < a < b and a < c


def test_noalloc_decode_rejects_steps_beyond_its_fixed_scratch(lib):
    """Rejected before any CUDA call, so this runs without a GPU."""
    desc = pa.DecodeDesc(64, 64, 128, 1 << 20, 1, 0.088)
    rc = lib.path_attn_decode_step_noalloc(ctypes.byref(desc), FAKE, FAKE, 500000, FAKE, FAKE,
                                           FAKE, FAKE, FAKE, FAKE, None)
    assert rc == pa.PATH_ERR_INVALID_ARG
    msg = lib.path_attn_last_error()
    assert b"scratch" in msg and b"8388608" in msg
    small = pa.DecodeDesc(1, 1, 128, 16, 1, 0.088)
    assert lib.path_attn_decode_step_noalloc(ctypes.byref(small), FAKE, FAKE, 16, FAKE, FAKE,
                                             FAKE, FAKE, FAKE, FAKE, None) == pa.PATH_ERR_INVALID_ARG


def test_fox_decode_and_prefix_reject_bad_arguments(lib):
    """Rejected before any CUDA call, so this runs without a GPU."""
    desc = pa.DecodeDesc(1, 2, 128, 64, 1, 0.088)
    ws = lib.path_attn_decode_workspace_size(ctypes.byref(desc))
    args = [FAKE, FAKE, FAKE, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None]
    for i, name in ((2, b"f_cache"), (9, b"log_f_t")):
        bad = list(args)
        bad[i] = None
        assert lib.path_attn_decode_step_fox(ctypes.byref(desc), *bad) == pa.PATH_ERR_INVALID_ARG
        assert name in lib.path_attn_last_error()
    bad = list(args)
    bad[3] = 64  # cache full: no slot for the new token
    assert lib.path_attn_decode_step_fox(ctypes.byref(desc), *bad) == pa.PATH_ERR_INVALID_ARG
    assert lib.path_attn_fox_prefix(FAKE, FAKE, 2, 10, 5, None) == pa.PATH_ERR_INVALID_ARG
    assert lib.path_attn_fox_prefix(None, FAKE, 2, 10, 10, None) == pa.PATH_ERR_INVALID_ARG
    assert lib.path_attn_fox_prefix(FAKE, FAKE, 0, 10, 10, None) == pa.PATH_ERR_INVALID_ARG


def bwd(lib, desc, ptrs, ws_bytes=1 << 40):
    return lib.path_attn_prefill_bwd(ctypes.byref(desc), *ptrs, ws_bytes, None)


def test_backward_workspace_sizes(lib):
    """One slice per pass is the minimum; with a single slice the minimum is
    the whole size; the tensor-core route sizes its regions for bf16."""
    D = pa.PrefillDesc
    one = D(1, 1, 4096, 128, pa.PATH_BF16, 0.088, 0)
    assert lib.path_attn_prefill_bwd_workspace_min(ctypes.byref(one)) == \
        lib.path_attn_prefill_bwd_workspace_size(ctypes.byref(one)) > 0
    head = D(8, 12, 4096, 128, pa.PATH_BF16, 0.088, 0)
    full = lib.path_attn_prefill_bwd_workspace_size(ctypes.byref(head))
    least = lib.path_attn_prefill_bwd_workspace_min(ctypes.byref(head))
    assert full < 6.5e9 and least * 90 < full
    # PaTH-FoX with scale 0 may take the CUDA-core route: fp32-sized regions
    zero = D(8, 12, 4096, 128, pa.PATH_BF16, 0.0, 0)
    assert lib.path_attn_prefill_bwd_workspace_size(ctypes.byref(zero)) > full
    assert lib.path_attn_prefill_bwd_workspace_min(ctypes.byref(D(0, 1, 16, 64, 0, 0.1, 0))) == 0


def test_backward_rejects_bad_arguments(lib):
    """Rejected before any CUDA call, so this runs without a GPU."""
    D = pa.PrefillDesc
    desc = D(2, 3, 100, 64, 0, 0.125, 0)
    need = lib.path_attn_prefill_bwd_workspace_size(ctypes.byref(desc))
    least = lib.path_attn_prefill_bwd_workspace_min(ctypes.byref(desc))
    assert need > lib.path_attn_prefill_workspace_size(ctypes.byref(desc)) > 0
    # six (batch, head) slices: one per pass needs about a sixth of all at once
    assert 0 < least < need and least * 5 < need
    # q k v w beta log_f out lse dout dlse dq dk dv dw dbeta dlog_f workspace
    good = [FAKE] * 5 + [None] + [FAKE] * 3 + [None] + [FAKE] * 5 + [None, FAKE]
    assert bwd(lib, desc, good, ws_bytes=least - 1) == pa.PATH_ERR_INVALID_ARG
    assert b"workspace" in lib.path_attn_last_error()
    required = [0, 1, 2, 3, 4, 6, 7, 8, 10, 11, 12, 13, 14, 16]
    for i in required:
        for bad in (None, ODD):
            p = list(good)
            p[i] = bad
            assert bwd(lib, desc, p) == pa.PATH_ERR_INVALID_ARG, i
    p = list(good)
    p[5] = FAKE  # log_f without dlog_f
    assert bwd(lib, desc, p) == pa.PATH_ERR_INVALID_ARG
    assert b"dlog_f" in lib.path_attn_last_error()
    p[5], p[15] = None, FAKE  # dlog_f without log_f
    assert bwd(lib, desc, p) == pa.PATH_ERR_INVALID_ARG
    p = list(good)
    p[9] = ODD
    assert bwd(lib, desc, p) == pa.PATH_ERR_INVALID_ARG
    assert bwd(lib, D(1, 1, 16, 130, 0, 0.1, 0), good) == pa.PATH_ERR_UNSUPPORTED
    assert bwd(lib, D(1, 1, 16, 64, 0, 0.1, 48), good) == pa.PATH_ERR_UNSUPPORTED
    # bf16 with head_dim 128 accepts any chunk here (the CUDA-core route)
    d128 = D(1, 1, 300, 128, 1, 0.1, 32)
    assert lib.path_attn_prefill_bwd_workspace_size(ctypes.byref(d128)) > 0
    # the carried-row store grows as L^2: doubling L roughly quadruples it
    a = lib.path_attn_prefill_bwd_workspace_size(ctypes.byref(D(1, 1, 4096, 64, 0, 0.1, 64)))
    b = lib.path_attn_prefill_bwd_workspace_size(ctypes.byref(D(1, 1, 8192, 64, 0, 0.1, 64)))
    assert 3.0 < b / a < 4.2


def test_padded_route_workspace(lib):
    """bf16 with head_dim a multiple of 8 below 128 (64 excepted) and the
    default chunk is planned on the tensor-core route with zero-padded copies:
    its workspace holds the 128-wide padded q, k, w, v and out on top of the
    head_dim-128 layout.  Head_dim 64 reads its tensors directly (no copies):
    the head_dim-128 layout alone.  An explicit chunk other than 128 plans the
    CUDA-core route."""
    D = pa.PrefillDesc
    B, H, L = 2, 3, 300
    ws = lambda d, dtype, chunk: lib.path_attn_prefill_workspace_size(
        ctypes.byref(D(B, H, L, d, dtype, 0.1, chunk)))
    full = ws(128, 1, 0)
    padded = ws(96, 1, 0)
    assert padded >= full + 5 * B * H * L * 128 * 2
    assert ws(64, 1, 0) == full == ws(64, 1, 128)
    # chunk 64 on the CUDA-core route: fp32 workspace of head_dim 64, no padded copies
    assert 0 < ws(64, 1, 64) != full
    # head_dim 36 (not a multiple of 8) stays on the CUDA cores
    assert ws(36, 1, 0) > 0
