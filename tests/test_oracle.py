"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: the
hand-derived examples under tests/golden/, brute-force explicit d x d matrix
products, textbook softmax attention, closed forms and invariants that the
PaTH definition fixes.  Definition: PaTH Attention summary
(gist.science/ko/paper/2505.16381), section 2 핵심 메커니즘 (logit equation,
H_s = I - beta_s w_s w_s^T), section 확장: PaTH-FoX, and section 3 (UT
transform, boundary-adjusted rows, inference with in-place key updates).
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            rows = [[float(x) for x in r.split()] for r in rest.split("|")]
            vals[key] = rows
    return vals


def unit_rows(rng, n, d):
    w = rng.standard_normal((n, d))
    return w / np.linalg.norm(w, axis=1, keepdims=True)


def rand_case(rng, L, d, beta_lo=0.0, beta_hi=2.0):
    q, k, v = (rng.standard_normal((L, d)) for _ in range(3))
    w = unit_rows(rng, L, d)
    beta = rng.uniform(beta_lo, beta_hi, L)
    return q, k, v, w, beta


def H(w, b):
    return np.eye(w.size) - b * np.outer(w, w)


def brute_logits(q, k, w, beta, scale, log_f=None):
    """Explicit d x d products per (i, j): k_j^T (H_{j+1} ... H_i) q_i."""
    L, d = q.shape
    out = np.full((L, L), -np.inf)
    for i in range(L):
        for j in range(i + 1):
            P = np.eye(d)
            for s in range(j + 1, i + 1):
                P = P @ H(w[s], beta[s])
            out[i, j] = scale * k[j] @ P @ q[i]
            if log_f is not None:
                out[i, j] += sum(log_f[j + 1:i + 1])
    return out


def softmax_attention(logits, v):
    """Textbook row softmax of a (causally masked) logit matrix."""
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    s = e.sum(axis=1, keepdims=True)
    return (e / s) @ v, (m + np.log(s))[:, 0]


# ---------------------------------------------------------------- golden

@pytest.mark.parametrize("name", ["hand_d2_L3.txt", "hand_d2_L2_halfbeta.txt"])
def test_golden_logits(name):
    g = read_golden(name)
    q, k, v, w = (np.array(g[n]) for n in "qkvw")
    beta = np.array(g["beta"][0])
    want = g["logits"]
    got = oracle.logits(q, k, w, beta, scale=1.0)
    for i, row in enumerate(want):
        np.testing.assert_allclose(got[i, :i + 1], row, rtol=0, atol=1e-12)
        assert np.all(np.isneginf(got[i, i + 1:]))
    # out / lse against the closed-form softmax of the hand-derived logits
    out, lse = oracle.prefill(q, k, v, w, beta, scale=1.0)
    for i, row in enumerate(want):
        e = [math.exp(x) for x in row]
        s = sum(e)
        np.testing.assert_allclose(lse[i], math.log(s), atol=1e-12)
        ref = sum(e[j] * v[j] for j in range(i + 1)) / s
        np.testing.assert_allclose(out[i], ref, atol=1e-12)


def test_golden_fox_logits():
    g = read_golden("hand_d2_L3.txt")
    q, k, v, w = (np.array(g[n]) for n in "qkvw")
    beta, log_f = np.array(g["beta"][0]), np.array(g["log_f"][0])
    got = oracle.logits(q, k, w, beta, log_f=log_f, scale=1.0)
    for i, row in enumerate(g["fox_logits"]):
        np.testing.assert_allclose(got[i, :i + 1], row, atol=1e-12)


def test_golden_decode_cache():
    g = read_golden("hand_d2_L3.txt")
    q, k, v, w = (np.array(g[n]) for n in "qkvw")
    beta = np.array(g["beta"][0])
    kc = oracle.build_kcache(k[None, :2], w[None, :2], beta[None, :2], cap=3)
    np.testing.assert_allclose(kc[0, :2], g["kcache_L0_2"], atol=1e-12)
    vc = np.zeros_like(kc)
    vc[0, :2] = v[:2]
    out = oracle.decode_step(kc, vc, 2, q[None, 2], k[None, 2], v[None, 2], w[None, 2],
                             beta[None, 2], scale=1.0)
    np.testing.assert_allclose(kc[0], g["kcache_after_t2"], atol=1e-12)
    e = [math.exp(x) for x in g["logits"][2]]
    ref = sum(e[j] * v[j] for j in range(3)) / sum(e)
    np.testing.assert_allclose(out[0], ref, atol=1e-12)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("fox", [False, True])
def test_brute_force_explicit_products(fox):
    rng = np.random.default_rng(1)
    L, d = 12, 6
    q, k, v, w, beta = rand_case(rng, L, d)
    log_f = np.log(rng.uniform(0.3, 1.0, L)) if fox else None
    scale = 1 / math.sqrt(d)
    ref = brute_logits(q, k, w, beta, scale, log_f)
    got = oracle.logits(q, k, w, beta, log_f=log_f, scale=scale)
    np.testing.assert_allclose(got[np.tril_indices(L)], ref[np.tril_indices(L)],
                               rtol=1e-12, atol=1e-12)
    out, lse = oracle.prefill(q, k, v, w, beta, log_f=log_f, scale=scale)
    ref_out, ref_lse = softmax_attention(ref, v)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_batched_heads_and_row_subset():
    rng = np.random.default_rng(2)
    B, Hh, L, d = 2, 3, 40, 8
    q, k, v = (rng.standard_normal((B, Hh, L, d)) for _ in range(3))
    w = rng.standard_normal((B, Hh, L, d))
    w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, (B, Hh, L))
    out, lse = oracle.prefill(q, k, v, w, beta)
    for b in range(B):
        for h in range(Hh):
            ref = brute_logits(q[b, h], k[b, h], w[b, h], beta[b, h], 1 / math.sqrt(d))
            ro, rl = softmax_attention(ref, v[b, h])
            np.testing.assert_allclose(out[b, h], ro, atol=1e-11)
            np.testing.assert_allclose(lse[b, h], rl, atol=1e-11)
    rows = [0, 7, 39, 13]
    o2, l2 = oracle.prefill(q, k, v, w, beta, rows=rows)
    np.testing.assert_array_equal(o2, out[:, :, rows])
    np.testing.assert_array_equal(l2, lse[:, :, rows])


# ---------------------------------------------------------------- reductions

def test_beta_zero_is_plain_causal_attention():
    rng = np.random.default_rng(3)
    L, d = 50, 16
    q, k, v, w, _ = rand_case(rng, L, d)
    beta = np.zeros(L)
    scale = 1 / math.sqrt(d)
    logits = np.where(np.tril(np.ones((L, L))) > 0, scale * q @ k.T, -np.inf)
    ref_out, ref_lse = softmax_attention(logits, v)
    out, lse = oracle.prefill(q, k, v, w, beta, scale=scale)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_fox_reductions():
    rng = np.random.default_rng(4)
    L, d = 30, 8
    q, k, v, w, beta = rand_case(rng, L, d)
    scale = 1 / math.sqrt(d)
    # log f == 0 -> plain PaTH, exactly
    o1, l1 = oracle.prefill(q, k, v, w, beta, log_f=np.zeros(L), scale=scale)
    o0, l0 = oracle.prefill(q, k, v, w, beta, scale=scale)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)
    # beta == 0 -> FoX: softmax(scale q.k + F_i - F_j) with F the inclusive cumsum
    log_f = np.log(rng.uniform(0.2, 1.0, L))
    F = np.cumsum(log_f)
    logits = scale * q @ k.T + F[:, None] - F[None, :]
    logits = np.where(np.tril(np.ones((L, L))) > 0, logits, -np.inf)
    ref_out, ref_lse = softmax_attention(logits, v)
    out, lse = oracle.prefill(q, k, v, w, np.zeros(L), log_f=log_f, scale=scale)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_beta_two_is_orthogonal_and_preserves_norms():
    """beta = 2 with exactly unit w: H is orthogonal, so the transported query
    keeps its norm.  Read the transported vector out of the logits by using
    basis vectors as key 0 (logit(i, 0) = e_m^T (H_1...H_i) q_i)."""
    rng = np.random.default_rng(5)
    L, d = 9, 5
    q, _, _, w, _ = rand_case(rng, L, d)
    beta = np.full(L, 2.0)
    transported = np.zeros((L, d))
    for m in range(d):
        k = rng.standard_normal((L, d))
        k[0] = np.eye(d)[m]
        transported[:, m] = oracle.logits(q, k, w, beta, scale=1.0)[:, 0]
    np.testing.assert_allclose(np.linalg.norm(transported, axis=1),
                               np.linalg.norm(q, axis=1), rtol=1e-12)
    # and the map q_i -> transported_i is the orthogonal matrix H_1 ... H_i
    for i in range(L):
        P = np.eye(d)
        for s in range(1, i + 1):
            P = P @ H(w[s], 2.0)
        np.testing.assert_allclose(P.T @ P, np.eye(d), atol=1e-12)
        np.testing.assert_allclose(transported[i], P @ q[i], atol=1e-12)


def test_contraction_bound():
    """beta in [0, 2] and unit w give eigenvalues {1, 1-beta} in [-1, 1], so
    |logit(i, j)| <= scale |k_j| |q_i|."""
    rng = np.random.default_rng(6)
    L, d = 64, 8
    q, k, _, w, beta = rand_case(rng, L, d)
    scale = 0.3
    lg = oracle.logits(q, k, w, beta, scale=scale)
    bound = scale * np.linalg.norm(q, axis=1)[:, None] * np.linalg.norm(k, axis=1)[None, :]
    il = np.tril_indices(L)
    assert np.all(np.abs(lg[il]) <= bound[il] * (1 + 1e-12))


def test_shared_direction_closed_form():
    """All w_s = w: the transitions commute and
    H_{j+1}...H_i = I - (1 - prod_s (1 - beta_s)) w w^T."""
    rng = np.random.default_rng(7)
    L, d = 20, 7
    q, k, _, _, beta = rand_case(rng, L, d)
    w1 = unit_rows(rng, 1, d)[0]
    w = np.tile(w1, (L, 1))
    lg = oracle.logits(q, k, w, beta, scale=1.0)
    for i in range(L):
        for j in range(i + 1):
            c = 1 - np.prod(1 - beta[j + 1:i + 1])
            ref = k[j] @ (q[i] - c * w1 * (w1 @ q[i]))
            assert abs(lg[i, j] - ref) < 1e-12


def test_coordinate_reflections_flip_signs():
    """w_s = e_{pi(s)}, beta = 2: the product is diagonal with entry m equal to
    (-1)^(number of s in (j, i] with pi(s) = m)."""
    rng = np.random.default_rng(8)
    L, d = 16, 4
    q, k, _, _, _ = rand_case(rng, L, d)
    pi = rng.integers(0, d, L)
    w = np.eye(d)[pi]
    lg = oracle.logits(q, k, w, np.full(L, 2.0), scale=1.0)
    for i in range(L):
        for j in range(i + 1):
            sign = np.array([(-1.0) ** np.sum(pi[j + 1:i + 1] == m) for m in range(d)])
            assert abs(lg[i, j] - k[j] @ (sign * q[i])) < 1e-13


# ------------------------------------------- chunk algebra used by the kernels

def ut_T(W, beta):
    """T = (I + strict_lower(diag(beta) W W^T))^{-1} diag(beta)."""
    n = W.shape[0]
    A = np.tril(beta[:, None] * (W @ W.T), -1)
    return np.linalg.solve(np.eye(n) + A, np.diag(beta))


def test_ut_transform_equals_explicit_product():
    """The lecture's exercise: n = 16 random unit vectors, the product of the
    transitions computed directly and from the compact (UT) form agree, in both
    orders: H_1 ... H_n = I - W^T T^T W and H_n ... H_1 = I - W^T T W
    (UT representation, section 3 of the PaTH summary)."""
    rng = np.random.default_rng(9)
    n, d = 16, 24
    W = unit_rows(rng, n, d)
    beta = rng.uniform(0, 2, n)
    fwd = np.eye(d)
    for s in range(n):
        fwd = fwd @ H(W[s], beta[s])
    rev = np.eye(d)
    for s in reversed(range(n)):
        rev = rev @ H(W[s], beta[s])
    T = ut_T(W, beta)
    assert np.allclose(T, np.tril(T))
    np.testing.assert_allclose(fwd, np.eye(d) - W.T @ T.T @ W, atol=1e-13)
    np.testing.assert_allclose(rev, np.eye(d) - W.T @ T @ W, atol=1e-13)


@pytest.mark.parametrize("L,C", [(24, 8), (21, 8), (16, 16)])
def test_chunked_decomposition_matches_oracle(L, C):
    """Boundary-adjusted rows + whole-chunk products reproduce every logit the
    oracle gives: across chunks logit = k_b^T P_{c+1} ... P_{b-1} q_b with
    P_c = I - W_c^T T_c^T W_c; inside a chunk
    S = Q K^T - (M_le * Q W^T) T (M_gt * K W^T)^T (the diagonal-block form)."""
    rng = np.random.default_rng(10)
    d = 6
    q, k, _, w, beta = rand_case(rng, L, d)
    ref = oracle.logits(q, k, w, beta, scale=1.0)
    qb, kb = oracle.boundary_rows(q, k, w, beta, C)
    N = (L + C - 1) // C
    P, T = [], []
    for c in range(N):
        sl = slice(c * C, min(c * C + C, L))
        Tc = ut_T(w[sl], beta[sl])
        T.append(Tc)
        P.append(np.eye(d) - w[sl].T @ Tc.T @ w[sl])
    for i in range(L):
        b = i // C
        for j in range(i + 1):
            c = j // C
            if c == b:
                continue
            M = np.eye(d)
            for cc in range(c + 1, b):
                M = M @ P[cc]
            assert abs(kb[j] @ M @ qb[i] - ref[i, j]) < 1e-12
    for c in range(N):
        sl = slice(c * C, min(c * C + C, L))
        n = sl.stop - sl.start
        Q, K, W = q[sl], k[sl], w[sl]
        r = np.arange(n)
        Mle = (r[None, :] <= r[:, None]).astype(float)
        Mgt = (r[None, :] > r[:, None]).astype(float)
        S = Q @ K.T - (Mle * (Q @ W.T)) @ T[c] @ (Mgt * (K @ W.T)).T
        il = np.tril_indices(n)
        np.testing.assert_allclose(S[il], ref[sl, sl][il], atol=1e-12)
        # boundary-adjusted rows from the same T
        Wt = T[c] @ W
        np.testing.assert_allclose(qb[sl], Q - (Mle * (Q @ W.T)) @ Wt, atol=1e-12)
        np.testing.assert_allclose(kb[sl], K - (Mgt * (K @ W.T)) @ (T[c].T @ W), atol=1e-12)


# ---------------------------------------------------------------- decode

def test_build_kcache_brute_force():
    rng = np.random.default_rng(11)
    L0, d = 10, 5
    _, k, _, w, beta = rand_case(rng, L0, d)
    kc = oracle.build_kcache(k[None], w[None], beta[None], cap=L0 + 2)
    for j in range(L0):
        P = np.eye(d)
        for s in range(L0 - 1, j, -1):
            P = P @ H(w[s], beta[s])
        np.testing.assert_allclose(kc[0, j], P @ k[j], atol=1e-12)
    assert np.all(kc[0, L0:] == 0)


def test_decode_steps_reproduce_prefill():
    """Inference bullet of section 3: updating cached keys in place with the
    current transition reproduces the prefill attention rows."""
    rng = np.random.default_rng(12)
    BH, L, L0, d = 3, 40, 25, 8
    q, k, v = (rng.standard_normal((BH, L, d)) for _ in range(3))
    w = rng.standard_normal((BH, L, d))
    w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, (BH, L))
    out_ref, _ = oracle.prefill(q, k, v, w, beta)
    kc = oracle.build_kcache(k[:, :L0], w[:, :L0], beta[:, :L0], cap=L)
    vc = np.zeros((BH, L, d))
    vc[:, :L0] = v[:, :L0]
    for t in range(L0, L):
        o = oracle.decode_step(kc, vc, t, q[:, t], k[:, t], v[:, t], w[:, t], beta[:, t])
        np.testing.assert_allclose(o, out_ref[:, t], atol=1e-12)
    # after the last step the cache equals a fresh build over all L tokens
    np.testing.assert_allclose(kc, oracle.build_kcache(k, w, beta), atol=1e-12)


def test_fox_decode_steps_reproduce_fox_prefill():
    """PaTH-FoX at inference (section 2, the FoX combination; section 3,
    inference): decoding with the forget-gate history reproduces the PaTH-FoX
    prefill rows, whose bias the prefill oracle sums along each query's
    reflection sweep; with log f = 0 it is the PaTH decode step."""
    rng = np.random.default_rng(21)
    BH, L, L0, d = 3, 36, 20, 8
    q, k, v = (rng.standard_normal((BH, L, d)) for _ in range(3))
    w = rng.standard_normal((BH, L, d))
    w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, (BH, L))
    log_f = np.log(1.0 / (1.0 + np.exp(-rng.normal(1.0, 1.0, (BH, L)))))
    out_ref, _ = oracle.prefill(q, k, v, w, beta, log_f=log_f)
    kc = oracle.build_kcache(k[:, :L0], w[:, :L0], beta[:, :L0], cap=L)
    vc = np.zeros((BH, L, d))
    vc[:, :L0] = v[:, :L0]
    lf = np.zeros((BH, L))
    lf[:, :L0] = log_f[:, :L0]
    kc0, vc0 = kc.copy(), vc.copy()
    for t in range(L0, L):
        o = oracle.decode_step_fox(kc, vc, lf, t, q[:, t], k[:, t], v[:, t], w[:, t],
                                   beta[:, t], log_f[:, t])
        np.testing.assert_allclose(o, out_ref[:, t], atol=1e-12)
    np.testing.assert_allclose(lf, log_f, atol=0)
    # zero forget-gate logits: exactly the PaTH step, on the same cache
    kcA, vcA = kc0.copy(), vc0.copy()
    kcB, vcB = kc0.copy(), vc0.copy()
    lfz = np.zeros((BH, L))
    t = L0 + 1
    oA = oracle.decode_step_fox(kcA, vcA, lfz, t, q[:, t], k[:, t], v[:, t], w[:, t],
                                beta[:, t], np.zeros(BH))
    oB = oracle.decode_step(kcB, vcB, t, q[:, t], k[:, t], v[:, t], w[:, t], beta[:, t])
    np.testing.assert_allclose(oA, oB, atol=0)
    np.testing.assert_allclose(kcA, kcB, atol=0)


def test_oracle_rejects_bad_arguments():
    lib = oracle.load()
    assert lib.path_oracle_prefill(1, 4, 0, 1.0, None, None, None, None, None, None,
                                   4, None, None, None, 1) != 0
    assert lib.path_oracle_decode_step(1, 4, 4, 2, 1.0, None, None, None, None, None,
                                       None, None, None, 1) != 0
