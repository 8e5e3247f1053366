"""fp64 CPU oracle for PaTH attention — TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library (libpath_attn)
never imports, links or calls it, and it shares no code with the product.

The arithmetic lives in ``path_oracle.c`` (plain C, fp64, one reflection at a
time, explicit softmax).  This module compiles it with gcc on first use and
wraps it with numpy-friendly functions.  Each function states the passage of
the PaTH pages it follows; see ``path_oracle.c`` for the full citations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "path_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libpath_oracle.so")
_lock = threading.Lock()
_lib = None

_I64 = ctypes.c_int64
_DBL = ctypes.c_double
_PD = ctypes.POINTER(ctypes.c_double)
_PI64 = ctypes.POINTER(ctypes.c_int64)


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the oracle into a shared library with gcc (-O2, OpenMP, IEEE fp)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    lib.path_oracle_prefill.argtypes = [_I64, _I64, _I64, _DBL, _PD, _PD, _PD, _PD,
                                        _PD, _PD, _I64, _PI64, _PD, _PD, ctypes.c_int]
    lib.path_oracle_logits.argtypes = [_I64, _I64, _DBL, _PD, _PD, _PD, _PD, _PD, _PD]
    lib.path_oracle_decode_step.argtypes = [_I64, _I64, _I64, _I64, _DBL, _PD, _PD,
                                            _PD, _PD, _PD, _PD, _PD, _PD, ctypes.c_int]
    lib.path_oracle_decode_step_fox.argtypes = [_I64, _I64, _I64, _I64, _DBL, _PD, _PD,
                                                _PD, _PD, _PD, _PD, _PD, _PD, _PD, _PD,
                                                ctypes.c_int]
    lib.path_oracle_build_kcache.argtypes = [_I64, _I64, _I64, _I64, _PD, _PD, _PD,
                                             _PD, ctypes.c_int]
    lib.path_oracle_boundary_rows.argtypes = [_I64, _I64, _I64, _PD, _PD, _PD, _PD,
                                              _PD, _PD]
    lib.path_oracle_prefill_bwd.argtypes = [_I64, _I64, _I64, _DBL] + [_PD] * 14 + [ctypes.c_int]
    for f in (lib.path_oracle_prefill, lib.path_oracle_prefill_bwd, lib.path_oracle_logits,
              lib.path_oracle_decode_step, lib.path_oracle_decode_step_fox,
              lib.path_oracle_build_kcache,
              lib.path_oracle_boundary_rows):
        f.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.  ``path`` loads a
    specific build instead, e.g. a deliberately mutated copy in a test."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            # PATH_ORACLE_LIB points the pin tests at a deliberately mutated
            # build (tests/test_oracle_mutants.py); unset in normal use.
            alt = os.environ.get("PATH_ORACLE_LIB")
            _lib = _declare(ctypes.CDLL(alt if alt else build()))
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return a.ctypes.data_as(_PD) if a is not None else None


def _bh(x, tail):
    """Flatten leading dims to one [BH] axis; returns (flat, leading shape)."""
    x = _f64(x)
    lead = x.shape[:x.ndim - tail]
    return x.reshape((-1,) + x.shape[x.ndim - tail:]), lead


def prefill(q, k, v, w, beta, log_f=None, scale=None, rows=None, nthreads=0,
            lib=None):
    """PaTH (or PaTH-FoX when ``log_f`` is given) causal attention forward.

    Follows the attention-logit equation and H_s definition of the PaTH
    Attention summary (section 2, 핵심 메커니즘) and the FoX extension
    (section 확장: PaTH-FoX).  q, k, v, w: [..., L, d]; beta, log_f: [..., L].
    Returns (out [..., R, d], lse [..., R]) with R = L or len(rows).
    """
    lib = lib or load()
    qf, lead = _bh(q, 2)
    kf, _ = _bh(k, 2)
    vf, _ = _bh(v, 2)
    wf, _ = _bh(w, 2)
    bf, _ = _bh(beta, 1)
    ff = _bh(log_f, 1)[0] if log_f is not None else None
    BH, L, d = qf.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if rows is None:
        r = None
        nrows = L
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = r.size
    out = np.empty((BH, nrows, d), dtype=np.float64)
    lse = np.empty((BH, nrows), dtype=np.float64)
    rc = lib.path_oracle_prefill(BH, L, d, float(scale), _p(qf), _p(kf), _p(vf),
                                 _p(wf), _p(bf), _p(ff), nrows,
                                 r.ctypes.data_as(_PI64) if r is not None else None,
                                 _p(out), _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("path_oracle_prefill failed: %d" % rc)
    return out.reshape(lead + (nrows, d)), lse.reshape(lead + (nrows,))


def prefill_bwd(q, k, v, w, beta, dout, log_f=None, dlse=None, scale=None, nthreads=0,
                lib=None):
    """Gradients of sum(dout * out) + sum(dlse * lse) of the PaTH (PaTH-FoX
    with ``log_f``) forward with respect to every input, by reverse-mode
    differentiation of the attention-logit equation (section 2, 핵심
    메커니즘), one transition at a time.  Shapes as ``prefill``; dout:
    [..., L, d], dlse: [..., L] or None.  Returns a dict with dq, dk, dv, dw,
    dbeta and (PaTH-FoX) dlog_f."""
    lib = lib or load()
    qf, lead = _bh(q, 2)
    kf, _ = _bh(k, 2)
    vf, _ = _bh(v, 2)
    wf, _ = _bh(w, 2)
    bf, _ = _bh(beta, 1)
    of, _ = _bh(dout, 2)
    ff = _bh(log_f, 1)[0] if log_f is not None else None
    lf = _bh(dlse, 1)[0] if dlse is not None else None
    BH, L, d = qf.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    g = {n: np.empty((BH, L, d), dtype=np.float64) for n in ("dq", "dk", "dv", "dw")}
    g["dbeta"] = np.empty((BH, L), dtype=np.float64)
    if ff is not None:
        g["dlog_f"] = np.empty((BH, L), dtype=np.float64)
    rc = lib.path_oracle_prefill_bwd(BH, L, d, float(scale), _p(qf), _p(kf), _p(vf), _p(wf),
                                     _p(bf), _p(ff), _p(of), _p(lf), _p(g["dq"]), _p(g["dk"]),
                                     _p(g["dv"]), _p(g["dw"]), _p(g["dbeta"]),
                                     _p(g.get("dlog_f")), int(nthreads))
    if rc != 0:
        raise ValueError("path_oracle_prefill_bwd failed: %d" % rc)
    return {n: a.reshape(lead + a.shape[1:]) for n, a in g.items()}


def logits(q, k, w, beta, log_f=None, scale=None, lib=None):
    """Full [L, L] logit matrix of one head (tiny inputs); -inf above the diagonal."""
    lib = lib or load()
    q, k, w, beta = _f64(q), _f64(k), _f64(w), _f64(beta)
    ff = _f64(log_f) if log_f is not None else None
    L, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty((L, L), dtype=np.float64)
    rc = lib.path_oracle_logits(L, d, float(scale), _p(q), _p(k), _p(w), _p(beta),
                                _p(ff), _p(out))
    if rc != 0:
        raise ValueError("path_oracle_logits failed: %d" % rc)
    return out


def decode_step(k_cache, v_cache, t, q_t, k_t, v_t, w_t, beta_t, scale=None,
                nthreads=0, lib=None):
    """One inference step (section 3, bullet 추론): keys j < t are updated in
    place by H_t, (k_t, v_t) is written at slot t, then softmax attention of
    q_t over slots 0..t.  k_cache, v_cache: float64 [BH, cap, d], modified in
    place.  q_t ... w_t: [BH, d]; beta_t: [BH].  Returns out [BH, d]."""
    lib = lib or load()
    assert k_cache.dtype == np.float64 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.float64 and v_cache.flags.c_contiguous
    BH, cap, d = k_cache.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q_t, k_t, v_t, w_t, beta_t = (_f64(x) for x in (q_t, k_t, v_t, w_t, beta_t))
    out = np.empty((BH, d), dtype=np.float64)
    rc = lib.path_oracle_decode_step(BH, cap, int(t), d, float(scale), _p(k_cache),
                                     _p(v_cache), _p(q_t), _p(k_t), _p(v_t),
                                     _p(w_t), _p(beta_t), _p(out), int(nthreads))
    if rc != 0:
        raise ValueError("path_oracle_decode_step failed: %d" % rc)
    return out


def decode_step_fox(k_cache, v_cache, lf_hist, t, q_t, k_t, v_t, w_t, beta_t, log_f_t,
                    scale=None, nthreads=0, lib=None):
    """One PaTH-FoX inference step: decode_step, plus the forget-gate bias
    sum_{s=j+1}^{t} log f_s on the logit of cached key j (section 2, the
    PaTH-FoX combination; section 3, inference).  lf_hist: float64 [BH, cap]
    holding log f of tokens 0..t-1; log_f_t ([BH]) is stored at slot t.
    Returns out [BH, d]."""
    lib = lib or load()
    assert k_cache.dtype == np.float64 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.float64 and v_cache.flags.c_contiguous
    assert lf_hist.dtype == np.float64 and lf_hist.flags.c_contiguous
    BH, cap, d = k_cache.shape
    assert lf_hist.shape == (BH, cap)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q_t, k_t, v_t, w_t, beta_t, log_f_t = (_f64(x) for x in (q_t, k_t, v_t, w_t, beta_t,
                                                             log_f_t))
    out = np.empty((BH, d), dtype=np.float64)
    rc = lib.path_oracle_decode_step_fox(BH, cap, int(t), d, float(scale), _p(k_cache),
                                         _p(v_cache), _p(lf_hist), _p(q_t), _p(k_t),
                                         _p(v_t), _p(w_t), _p(beta_t), _p(log_f_t), _p(out),
                                         int(nthreads))
    if rc != 0:
        raise ValueError("path_oracle_decode_step_fox failed: %d" % rc)
    return out


def build_kcache(k, w, beta, cap=None, nthreads=0, lib=None):
    """Key cache after decoding tokens 0..L0-1 (kc_j = H_{L0-1}...H_{j+1} k_j),
    by an explicit d x d product swept from the right.  k, w: [BH, L0, d];
    beta: [BH, L0].  Returns float64 [BH, cap, d] (rows >= L0 zero)."""
    lib = lib or load()
    k, w, beta = _f64(k), _f64(w), _f64(beta)
    BH, L0, d = k.shape
    cap = L0 if cap is None else int(cap)
    kc = np.zeros((BH, cap, d), dtype=np.float64)
    rc = lib.path_oracle_build_kcache(BH, L0, cap, d, _p(k), _p(w), _p(beta),
                                      _p(kc), int(nthreads))
    if rc != 0:
        raise ValueError("path_oracle_build_kcache failed: %d" % rc)
    return kc


def boundary_rows(q, k, w, beta, C, lib=None):
    """Boundary-adjusted query and key rows of one head for chunk length C
    (section 3, FlashAttention-style algorithm, first bullet).  Returns
    (qb [L, d], kb [L, d])."""
    lib = lib or load()
    q, k, w, beta = _f64(q), _f64(k), _f64(w), _f64(beta)
    L, d = q.shape
    qb = np.empty_like(q)
    kb = np.empty_like(k)
    rc = lib.path_oracle_boundary_rows(L, d, int(C), _p(q), _p(k), _p(w), _p(beta),
                                       _p(qb), _p(kb))
    if rc != 0:
        raise ValueError("path_oracle_boundary_rows failed: %d" % rc)
    return qb, kb
