"""Python binding of libpath_attn (PaTH attention on GB300, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libpath_attn.so``; PyTorch supplies device memory and streams.
The functions carry the names of the C entry points in ``include/path_attn.h``.
There is no fallback: if the library is missing or a call fails, a
``PathAttnError`` is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "PathAttnError", "load_library", "path_attn_prefill_fwd", "path_attn_prefill_prep",
    "path_attn_prefill_scan", "path_attn_prefill_bwd", "path_attn_prefill_bwd_workspace_size",
    "path_attention",
    "path_attn_decode_step", "path_attn_decode_step_fox",
    "path_attn_fox_prefix",
    "path_attn_build_kcache", "path_attn_prefill_workspace_size",
    "path_attn_decode_workspace_size", "path_attn_build_kcache_workspace_size",
    "path_attn_device_status", "path_attn_selftest_bounded_wait", "EXPORTED_SYMBOLS",
    "path_attn_cp_local_len", "path_attn_cp_rows", "path_attn_cp_exchange_bytes",
    "path_attn_cp_workspace_size", "path_attn_cp_prep", "path_attn_cp_scan", "cp_all_gather",
    "path_attention_cp",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpath_attn.so")

PATH_OK, PATH_ERR_INVALID_ARG, PATH_ERR_UNSUPPORTED, PATH_ERR_CUDA, PATH_ERR_TIMEOUT = range(5)
PATH_F32, PATH_BF16 = 0, 1

EXPORTED_SYMBOLS = (
    "path_attn_prefill_workspace_size", "path_attn_prefill_fwd", "path_attn_prefill_prep",
    "path_attn_prefill_scan", "path_attn_prefill_bwd_workspace_size", "path_attn_prefill_bwd",
    "path_attn_prefill_bwd_workspace_min", "path_attn_decode_workspace_size", "path_attn_decode_step", "path_attn_decode_step_noalloc",
    "path_attn_decode_step_fox", "path_attn_fox_prefix",
    "path_attn_build_kcache_workspace_size", "path_attn_build_kcache",
    "path_attn_device_status", "path_attn_selftest_bounded_wait",
    "path_attn_status_string", "path_attn_last_error", "path_attn_version",
    "path_attn_cp_local_len", "path_attn_cp_rows", "path_attn_cp_exchange_bytes",
    "path_attn_cp_workspace_size", "path_attn_cp_prep", "path_attn_cp_scan",
)


class PathAttnError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (_STATUS.get(status, status), message))
        self.status = status


_STATUS = {PATH_OK: "PATH_OK", PATH_ERR_INVALID_ARG: "PATH_ERR_INVALID_ARG",
           PATH_ERR_UNSUPPORTED: "PATH_ERR_UNSUPPORTED", PATH_ERR_CUDA: "PATH_ERR_CUDA",
           PATH_ERR_TIMEOUT: "PATH_ERR_TIMEOUT"}


class PrefillDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("seq_len", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("chunk", ctypes.c_int32), ("scan_group", ctypes.c_int32)]


class DecodeDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("cache_capacity", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float)]


_lib = None
_lock = threading.Lock()
_VP = ctypes.c_void_p
_SZ = ctypes.c_size_t


def load_library(path: str | None = None):
    """Load libpath_attn.so (built by ``build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise PathAttnError(PATH_ERR_CUDA, "libpath_attn.so not built (%s); run "
                                "dependent_positional_attention_gb300.build.build()" % p)
        lib = ctypes.CDLL(p)
        pd, dd = ctypes.POINTER(PrefillDesc), ctypes.POINTER(DecodeDesc)
        lib.path_attn_prefill_workspace_size.argtypes = [pd]
        lib.path_attn_prefill_workspace_size.restype = _SZ
        lib.path_attn_prefill_fwd.argtypes = [pd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                              _VP, _SZ, _VP]
        lib.path_attn_prefill_prep.argtypes = [pd, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]
        lib.path_attn_prefill_scan.argtypes = [pd, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]
        lib.path_attn_prefill_bwd_workspace_size.argtypes = [pd]
        lib.path_attn_prefill_bwd_workspace_size.restype = _SZ
        lib.path_attn_prefill_bwd_workspace_min.argtypes = [pd]
        lib.path_attn_prefill_bwd_workspace_min.restype = _SZ
        lib.path_attn_prefill_bwd.argtypes = [pd] + [_VP] * 17 + [_SZ, _VP]
        lib.path_attn_decode_workspace_size.argtypes = [dd]
        lib.path_attn_decode_workspace_size.restype = _SZ
        lib.path_attn_decode_step.argtypes = [dd, _VP, _VP, ctypes.c_int32, _VP, _VP, _VP,
                                              _VP, _VP, _VP, _VP, _SZ, _VP]
        lib.path_attn_decode_step_noalloc.argtypes = [dd, _VP, _VP, ctypes.c_int32, _VP, _VP,
                                                      _VP, _VP, _VP, _VP, _VP]
        lib.path_attn_decode_step_fox.argtypes = [dd, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP,
                                                  _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]
        lib.path_attn_fox_prefix.argtypes = [_VP, _VP, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, _VP]
        lib.path_attn_build_kcache_workspace_size.argtypes = [pd]
        lib.path_attn_build_kcache_workspace_size.restype = _SZ
        lib.path_attn_build_kcache.argtypes = [pd, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP,
                                               _SZ, _VP]
        i32 = ctypes.c_int32
        lib.path_attn_cp_local_len.argtypes = [pd, i32, i32]
        lib.path_attn_cp_local_len.restype = i32
        lib.path_attn_cp_rows.argtypes = [pd, i32, i32, ctypes.POINTER(i32), i32]
        lib.path_attn_cp_exchange_bytes.argtypes = [pd, i32]
        lib.path_attn_cp_exchange_bytes.restype = _SZ
        lib.path_attn_cp_workspace_size.argtypes = [pd, i32]
        lib.path_attn_cp_workspace_size.restype = _SZ
        lib.path_attn_cp_prep.argtypes = [pd, i32, i32] + [_VP] * 8 + [_SZ, _VP]
        lib.path_attn_cp_scan.argtypes = [pd, i32, i32] + [_VP] * 5 + [_SZ, _VP]
        lib.path_attn_device_status.argtypes = [ctypes.c_int32]
        lib.path_attn_selftest_bounded_wait.argtypes = [ctypes.c_uint32, _VP]
        lib.path_attn_status_string.restype = ctypes.c_char_p
        lib.path_attn_last_error.restype = ctypes.c_char_p
        lib.path_attn_version.restype = ctypes.c_int32
        for f in ("path_attn_prefill_fwd", "path_attn_prefill_prep", "path_attn_prefill_scan",
                  "path_attn_prefill_bwd",
                  "path_attn_decode_step", "path_attn_decode_step_noalloc",
                  "path_attn_build_kcache", "path_attn_cp_rows", "path_attn_cp_prep",
                  "path_attn_cp_scan",
                  "path_attn_device_status", "path_attn_selftest_bounded_wait"):
            getattr(lib, f).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(status):
    if status != PATH_OK:
        raise PathAttnError(status, load_library().path_attn_last_error().decode())


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return PATH_F32
    if t.dtype == torch.bfloat16:
        return PATH_BF16
    raise PathAttnError(PATH_ERR_UNSUPPORTED, "dtype %s not supported" % t.dtype)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, shape=None, dtype=None):
    if not t.is_cuda or not t.is_contiguous():
        raise PathAttnError(PATH_ERR_INVALID_ARG, "%s must be a contiguous CUDA tensor" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise PathAttnError(PATH_ERR_INVALID_ARG, "%s has shape %s, expected %s"
                            % (name, tuple(t.shape), tuple(shape)))
    if dtype is not None and t.dtype != dtype:
        raise PathAttnError(PATH_ERR_INVALID_ARG, "%s has dtype %s, expected %s"
                            % (name, t.dtype, dtype))


def _prefill_desc(q, scale, chunk, scan_group=0):
    B, H, L, d = q.shape
    if scale is None:
        scale = d ** -0.5
    return PrefillDesc(B, H, L, d, _dtype_code(q), float(scale), int(chunk), int(scan_group))


def path_attn_prefill_workspace_size(desc: PrefillDesc) -> int:
    return int(load_library().path_attn_prefill_workspace_size(ctypes.byref(desc)))


def path_attn_prefill_fwd(q, k, v, w, beta, log_f=None, out=None, lse=None, scale=None,
                          chunk=0, workspace=None, stream=None, want_lse=True, scan_group=0):
    """Causal PaTH / PaTH-FoX attention forward (see path_attn_prefill_fwd in
    include/path_attn.h).  q, k, v, w: [B, H, L, d] CUDA tensors (float32 or
    bfloat16); beta, log_f: float32 [B, H, L].  scan_group: heads per group
    of the tensor-core scan's tile order (0 = automatic; speed only).
    Returns (out, lse)."""
    import torch
    lib = load_library()
    B, H, L, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (w, "w")):
        _need(t, n, (B, H, L, d), q.dtype)
    _need(beta, "beta", (B, H, L), torch.float32)
    if log_f is not None:
        _need(log_f, "log_f", (B, H, L), torch.float32)
    desc = _prefill_desc(q, scale, chunk, scan_group)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (B, H, L, d), q.dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, H, L), device=q.device, dtype=torch.float32)
    if lse is not None:
        _need(lse, "lse", (B, H, L), torch.float32)
    ws_bytes = path_attn_prefill_workspace_size(desc)
    if ws_bytes == 0:
        _check(lib.path_attn_prefill_fwd(ctypes.byref(desc), *([None] * 9), 0, None))
    if workspace is None:
        workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
    _check(lib.path_attn_prefill_fwd(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(log_f),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out, lse


def path_attn_prefill_prep(q, k, v, w, beta, log_f=None, scale=None, chunk=0, workspace=None,
                          stream=None):
    """Stage 1 of the prefill (see path_attn_prefill_prep in include/path_attn.h).
    Returns the workspace tensor to pass to path_attn_prefill_scan."""
    import torch
    lib = load_library()
    desc = _prefill_desc(q, scale, chunk)
    if workspace is None:
        workspace = torch.empty(max(path_attn_prefill_workspace_size(desc), 16),
                                device=q.device, dtype=torch.uint8)
    _check(lib.path_attn_prefill_prep(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(log_f),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return workspace


def path_attn_prefill_scan(q, w, v, workspace, log_f=None, out=None, lse=None, scale=None,
                          chunk=0, stream=None, scan_group=0):
    """Stage 2 of the prefill (see path_attn_prefill_scan in include/path_attn.h);
    q is used for its shape and dtype only.  Returns (out, lse)."""
    import torch
    lib = load_library()
    desc = _prefill_desc(q, scale, chunk, scan_group)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
    _check(lib.path_attn_prefill_scan(
        ctypes.byref(desc), _ptr(w), _ptr(v), _ptr(log_f), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def path_attn_prefill_bwd_workspace_size(desc: PrefillDesc) -> int:
    return int(load_library().path_attn_prefill_bwd_workspace_size(ctypes.byref(desc)))


def path_attn_prefill_bwd_workspace_min(desc: PrefillDesc) -> int:
    return int(load_library().path_attn_prefill_bwd_workspace_min(ctypes.byref(desc)))


def path_attn_prefill_bwd(q, k, v, w, beta, out, lse, dout, log_f=None, dlse=None, scale=None,
                          chunk=0, workspace=None, stream=None, workspace_bytes=None):
    """Backward of path_attn_prefill_fwd (see path_attn_prefill_bwd in
    include/path_attn.h): gradients of sum(dout * out) + sum(dlse * lse).
    Tensors as for the forward; out and lse are the forward's outputs.
    workspace_bytes bounds the workspace allocated here (between
    path_attn_prefill_bwd_workspace_min and _size; the call then runs the
    (batch, head) slices in passes).  Returns a dict with dq, dk, dv, dw
    (dtype of q), dbeta and, for PaTH-FoX, dlog_f (float32)."""
    import torch
    lib = load_library()
    B, H, L, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (w, "w"), (out, "out"), (dout, "dout")):
        _need(t, n, (B, H, L, d), q.dtype)
    _need(beta, "beta", (B, H, L), torch.float32)
    _need(lse, "lse", (B, H, L), torch.float32)
    for t, n in ((log_f, "log_f"), (dlse, "dlse")):
        if t is not None:
            _need(t, n, (B, H, L), torch.float32)
    desc = _prefill_desc(q, scale, chunk)
    g = {n: torch.empty_like(q) for n in ("dq", "dk", "dv", "dw")}
    g["dbeta"] = torch.empty((B, H, L), device=q.device, dtype=torch.float32)
    if log_f is not None:
        g["dlog_f"] = torch.empty((B, H, L), device=q.device, dtype=torch.float32)
    ws_bytes = path_attn_prefill_bwd_workspace_size(desc)
    if ws_bytes == 0:
        _check(lib.path_attn_prefill_bwd(ctypes.byref(desc), *([None] * 17), 0, None))
    if workspace_bytes is not None:
        ws_bytes = min(ws_bytes, max(int(workspace_bytes), path_attn_prefill_bwd_workspace_min(desc)))
    if workspace is None:
        workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
    _check(lib.path_attn_prefill_bwd(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(log_f),
        _ptr(out), _ptr(lse), _ptr(dout), _ptr(dlse), _ptr(g["dq"]), _ptr(g["dk"]),
        _ptr(g["dv"]), _ptr(g["dw"]), _ptr(g["dbeta"]), _ptr(g.get("dlog_f")),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return g


def path_attention(q, k, v, w, beta, log_f=None, scale=None):
    """Differentiable PaTH / PaTH-FoX prefill for torch autograd: forward by
    path_attn_prefill_fwd, backward by path_attn_prefill_bwd (both in the
    library).  Returns out; gradients flow to q, k, v, w, beta and log_f."""
    return _PathAttentionFn.apply(q, k, v, w, beta, log_f, scale)


def _autograd_fn():
    import torch

    class PathAttentionFn(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, w, beta, log_f, scale):
            q, k, v, w, beta = (t.contiguous() for t in (q, k, v, w, beta))
            log_f = log_f.contiguous() if log_f is not None else None
            out, lse = path_attn_prefill_fwd(q, k, v, w, beta, log_f=log_f, scale=scale)
            ctx.save_for_backward(q, k, v, w, beta, out, lse,
                                  log_f if log_f is not None else torch.empty(0))
            ctx.fox = log_f is not None
            ctx.scale = scale
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, w, beta, out, lse, log_f = ctx.saved_tensors
            g = path_attn_prefill_bwd(q, k, v, w, beta, out, lse, dout.contiguous(),
                                      log_f=log_f if ctx.fox else None, scale=ctx.scale)
            return (g["dq"], g["dk"], g["dv"], g["dw"], g["dbeta"], g.get("dlog_f"), None)

    return PathAttentionFn


class _LazyFn:
    _fn = None

    def apply(self, *args):
        if _LazyFn._fn is None:
            _LazyFn._fn = _autograd_fn()
        return _LazyFn._fn.apply(*args)


_PathAttentionFn = _LazyFn()


def path_attn_decode_workspace_size(desc: DecodeDesc) -> int:
    return int(load_library().path_attn_decode_workspace_size(ctypes.byref(desc)))


def decode_desc(k_cache, scale=None):
    B, H, cap, d = k_cache.shape
    if scale is None:
        scale = d ** -0.5
    return DecodeDesc(B, H, d, cap, _dtype_code(k_cache), float(scale))


def path_attn_decode_step(k_cache, v_cache, cache_len, q_t, k_t, v_t, w_t, beta_t, out=None,
                          scale=None, workspace=None, stream=None):
    """One PaTH decode step (see path_attn_decode_step in include/path_attn.h).
    k_cache, v_cache: [B, H, capacity, d]; q_t .. w_t: [B, H, d]; beta_t:
    float32 [B, H].  Updates k_cache in place, writes slot cache_len of both
    caches, returns out [B, H, d]."""
    import torch
    lib = load_library()
    B, H, cap, d = k_cache.shape
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", (B, H, cap, d), k_cache.dtype)
    for t, n in ((q_t, "q_t"), (k_t, "k_t"), (v_t, "v_t"), (w_t, "w_t")):
        _need(t, n, (B, H, d), k_cache.dtype)
    _need(beta_t, "beta_t", (B, H), torch.float32)
    desc = decode_desc(k_cache, scale)
    if out is None:
        out = torch.empty_like(q_t)
    _need(out, "out", (B, H, d), k_cache.dtype)
    if workspace is None:
        n = path_attn_decode_workspace_size(desc)
        workspace = torch.empty(max(n, 16), device=k_cache.device, dtype=torch.uint8)
    _check(lib.path_attn_decode_step(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), int(cache_len), _ptr(q_t), _ptr(k_t),
        _ptr(v_t), _ptr(w_t), _ptr(beta_t), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def path_attn_decode_step_fox(k_cache, v_cache, f_cache, cache_len, q_t, k_t, v_t, w_t, beta_t,
                              log_f_t, out=None, scale=None, workspace=None, stream=None):
    """One PaTH-FoX decode step (see path_attn_decode_step_fox in
    include/path_attn.h).  As path_attn_decode_step, plus f_cache: float32
    [B, H, capacity] of forget-gate log prefixes (slot cache_len is written)
    and log_f_t: float32 [B, H]."""
    import torch
    lib = load_library()
    B, H, cap, d = k_cache.shape
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", (B, H, cap, d), k_cache.dtype)
    _need(f_cache, "f_cache", (B, H, cap), torch.float32)
    for t, n in ((q_t, "q_t"), (k_t, "k_t"), (v_t, "v_t"), (w_t, "w_t")):
        _need(t, n, (B, H, d), k_cache.dtype)
    _need(beta_t, "beta_t", (B, H), torch.float32)
    _need(log_f_t, "log_f_t", (B, H), torch.float32)
    desc = decode_desc(k_cache, scale)
    if out is None:
        out = torch.empty_like(q_t)
    _need(out, "out", (B, H, d), k_cache.dtype)
    if workspace is None:
        n = path_attn_decode_workspace_size(desc)
        workspace = torch.empty(max(n, 16), device=k_cache.device, dtype=torch.uint8)
    _check(lib.path_attn_decode_step_fox(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(f_cache), int(cache_len),
        _ptr(q_t), _ptr(k_t), _ptr(v_t), _ptr(w_t), _ptr(beta_t), _ptr(log_f_t), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def path_attn_fox_prefix(log_f, f_out, stream=None):
    """f_out[b, h, i] = sum_{s<=i} log_f[b, h, s] for i < L, the last value
    repeated beyond (see path_attn_fox_prefix in include/path_attn.h).
    log_f: float32 [B, H, L]; f_out: float32 [B, H, capacity >= L]."""
    import torch
    lib = load_library()
    B, H, L = log_f.shape
    _need(log_f, "log_f", (B, H, L), torch.float32)
    cap = f_out.shape[2]
    _need(f_out, "f_out", (B, H, cap), torch.float32)
    _check(lib.path_attn_fox_prefix(_ptr(log_f), _ptr(f_out), B * H, L, cap, _stream(stream)))
    return f_out


def path_attn_decode_step_noalloc(k_cache, v_cache, cache_len, q_t, k_t, v_t, w_t, beta_t,
                                  out, scale=None, stream=None):
    """path_attn_decode_step without a workspace (see include/path_attn.h):
    for callers that cannot allocate device memory.  `out` must be given;
    the tensors are checked as for path_attn_decode_step."""
    import torch
    lib = load_library()
    B, H, cap, d = k_cache.shape
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", (B, H, cap, d), k_cache.dtype)
    for t, n in ((q_t, "q_t"), (k_t, "k_t"), (v_t, "v_t"), (w_t, "w_t"), (out, "out")):
        _need(t, n, (B, H, d), k_cache.dtype)
    _need(beta_t, "beta_t", (B, H), torch.float32)
    desc = decode_desc(k_cache, scale)
    _check(lib.path_attn_decode_step_noalloc(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), int(cache_len), _ptr(q_t), _ptr(k_t),
        _ptr(v_t), _ptr(w_t), _ptr(beta_t), _ptr(out), _stream(stream)))
    return out


def path_attn_build_kcache_workspace_size(desc: PrefillDesc) -> int:
    return int(load_library().path_attn_build_kcache_workspace_size(ctypes.byref(desc)))


def path_attn_build_kcache(k, w, beta, k_cache, workspace=None, stream=None):
    """Write k_cache[:, :, j] = H_{L-1} ... H_{j+1} k_j for j < L (see
    path_attn_build_kcache in include/path_attn.h)."""
    import torch
    lib = load_library()
    B, H, L, d = k.shape
    _need(k, "k")
    _need(w, "w", (B, H, L, d), k.dtype)
    _need(beta, "beta", (B, H, L), torch.float32)
    _need(k_cache, "k_cache")
    desc = _prefill_desc(k, None, 0)
    if workspace is None:
        n = path_attn_build_kcache_workspace_size(desc)
        workspace = torch.empty(max(n, 16), device=k.device, dtype=torch.uint8)
    _check(lib.path_attn_build_kcache(
        ctypes.byref(desc), _ptr(k), _ptr(w), _ptr(beta), _ptr(k_cache), k_cache.shape[2],
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return k_cache


def path_attn_device_status(clear=True):
    """Synchronise and return the device error status code (PATH_OK or
    PATH_ERR_TIMEOUT); clears the flag by default."""
    return int(load_library().path_attn_device_status(1 if clear else 0))


def path_attn_selftest_bounded_wait(limit_us=1000, stream=None):
    _check(load_library().path_attn_selftest_bounded_wait(int(limit_us), _stream(stream)))


# ------------------------------------------------------ sequence-sharded prefill

def _cp_desc(batch, heads, seq_len, scale):
    if scale is None:
        scale = 128 ** -0.5
    return PrefillDesc(batch, heads, seq_len, 128, PATH_BF16, float(scale), 0)


def path_attn_cp_local_len(batch, heads, seq_len, world, rank):
    """Rows of the sequence that rank `rank` of `world` holds (see
    path_attn_cp_local_len in include/path_attn.h)."""
    n = load_library().path_attn_cp_local_len(ctypes.byref(_cp_desc(batch, heads, seq_len, None)),
                                              int(world), int(rank))
    if n < 0:
        _check(PATH_ERR_INVALID_ARG)
    return int(n)


def path_attn_cp_rows(batch, heads, seq_len, world, rank):
    """Global positions of the rank's local rows, in local order (a CPU int64
    tensor); index the sequence dimension with it to shard a tensor."""
    import torch
    lib = load_library()
    desc = _cp_desc(batch, heads, seq_len, None)
    n = path_attn_cp_local_len(batch, heads, seq_len, world, rank)
    buf = (ctypes.c_int32 * max(n, 1))()
    _check(lib.path_attn_cp_rows(ctypes.byref(desc), int(world), int(rank), buf, n))
    return torch.tensor(list(buf)[:n], dtype=torch.int64)


def path_attn_cp_exchange_bytes(batch, heads, seq_len, world):
    return int(load_library().path_attn_cp_exchange_bytes(
        ctypes.byref(_cp_desc(batch, heads, seq_len, None)), int(world)))


def path_attn_cp_workspace_size(batch, heads, seq_len, world):
    return int(load_library().path_attn_cp_workspace_size(
        ctypes.byref(_cp_desc(batch, heads, seq_len, None)), int(world)))


def path_attn_cp_prep(q, k, v, w, beta, seq_len, world, rank, log_f=None, scale=None,
                      exchange=None, workspace=None, stream=None):
    """Step 1 of the sharded prefill (see path_attn_cp_prep in
    include/path_attn.h).  q, k, v, w: the rank's local rows [B, H, Lr, 128]
    bf16; beta: float32 [B, H, Lr]; log_f: float32 [B, H, seq_len] of the
    whole sequence (PaTH-FoX) or None.  Returns (exchange, workspace): the
    rank's exchange block (uint8) to all-gather, and the workspace to hand to
    path_attn_cp_scan."""
    import torch
    lib = load_library()
    B, H, Lr, d = q.shape
    n = path_attn_cp_local_len(B, H, seq_len, world, rank)
    if Lr != n or d != 128:
        raise PathAttnError(PATH_ERR_INVALID_ARG, "q has shape %s, rank %d of %d holds [%d, %d, "
                            "%d, 128]" % (tuple(q.shape), rank, world, B, H, n))
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (w, "w")):
        _need(t, nm, (B, H, Lr, 128), torch.bfloat16)
    _need(beta, "beta", (B, H, Lr), torch.float32)
    if log_f is not None:
        _need(log_f, "log_f", (B, H, seq_len), torch.float32)
    desc = _cp_desc(B, H, seq_len, scale)
    if exchange is None:
        exchange = torch.empty(path_attn_cp_exchange_bytes(B, H, seq_len, world),
                               device=q.device, dtype=torch.uint8)
    if workspace is None:
        workspace = torch.empty(path_attn_cp_workspace_size(B, H, seq_len, world),
                                device=q.device, dtype=torch.uint8)
    ptr = (lambda t: _ptr(t) if t.numel() else None)
    _check(lib.path_attn_cp_prep(
        ctypes.byref(desc), int(world), int(rank), ptr(q), ptr(k), ptr(v), ptr(w), ptr(beta),
        _ptr(log_f), _ptr(exchange), _ptr(workspace), workspace.numel(), _stream(stream)))
    return exchange, workspace


def path_attn_cp_scan(exchange_all, workspace, batch, heads, seq_len, world, rank, log_f=None,
                      out=None, lse=None, scale=None, stream=None):
    """Step 3 of the sharded prefill (see path_attn_cp_scan in
    include/path_attn.h): exchange_all holds the world exchange blocks in rank
    order.  Returns (out [B, H, Lr, 128] bf16, lse [B, H, Lr] float32)."""
    import torch
    lib = load_library()
    n = path_attn_cp_local_len(batch, heads, seq_len, world, rank)
    exb = path_attn_cp_exchange_bytes(batch, heads, seq_len, world)
    if exchange_all.numel() * exchange_all.element_size() != world * exb:
        raise PathAttnError(PATH_ERR_INVALID_ARG, "exchange_all must hold %d bytes" % (world * exb))
    dev = exchange_all.device
    if out is None:
        out = torch.empty((batch, heads, n, 128), device=dev, dtype=torch.bfloat16)
    if lse is None:
        lse = torch.empty((batch, heads, n), device=dev, dtype=torch.float32)
    if n:
        _need(out, "out", (batch, heads, n, 128), torch.bfloat16)
        _need(lse, "lse", (batch, heads, n), torch.float32)
    if log_f is not None:
        _need(log_f, "log_f", (batch, heads, seq_len), torch.float32)
    desc = _cp_desc(batch, heads, seq_len, scale)
    _check(lib.path_attn_cp_scan(
        ctypes.byref(desc), int(world), int(rank), _ptr(log_f), _ptr(exchange_all),
        _ptr(out) if n else None, _ptr(lse) if n else None, _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out, lse


def cp_all_gather(exchange, world, group=None):
    """The exchange step of the sharded prefill: every rank's exchange block,
    gathered in rank order into one buffer (torch.distributed all-gather; over
    NCCL for CUDA tensors)."""
    import torch
    import torch.distributed as dist
    buf = torch.empty(world * exchange.numel(), device=exchange.device, dtype=exchange.dtype)
    if world == 1:
        buf.copy_(exchange)
        return buf
    try:
        dist.all_gather_into_tensor(buf, exchange, group=group)
    except (RuntimeError, NotImplementedError):
        # backends without a flat all-gather: the list form into views of buf
        dist.all_gather(list(buf.chunk(world)), exchange, group=group)
    return buf


def path_attention_cp(q, k, v, w, beta, seq_len, log_f=None, scale=None, group=None):
    """Sequence-sharded PaTH / PaTH-FoX prefill on the ranks of a
    torch.distributed process group (one GPU per rank): each rank passes its
    local rows (path_attn_cp_rows) and gets their outputs back.  Returns
    (out, lse) for the local rows."""
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    B, H = q.shape[:2]
    exchange, ws = path_attn_cp_prep(q, k, v, w, beta, seq_len, world, rank, log_f=log_f,
                                     scale=scale)
    gathered = cp_all_gather(exchange, world, group)
    return path_attn_cp_scan(gathered, ws, B, H, seq_len, world, rank, log_f=log_f, scale=scale)
