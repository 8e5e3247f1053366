"""Pins of the oracle's prefill backward (CPU only, fp64).

The pages print no gradient, so the backward is pinned to things other than
itself:
  * torch autograd through a brute-force forward that forms every
    H_{j+1} ... H_i as an explicit d x d product (an independent program for
    the attention-logit equation of the PaTH summary, section 2);
  * central finite differences of the oracle's own forward;
  * beta = 0, where PaTH is plain causal softmax attention and the gradient is
    the library's (torch scaled_dot_product_attention under autograd).
"""
import numpy as np
import pytest
import torch

import oracle


def draw(BH, L, d, seed, fox=False, beta_fixed=None):
    rng = np.random.default_rng(seed)
    q, k, v, dout = (rng.standard_normal((BH, L, d)) for _ in range(4))
    w = rng.standard_normal((BH, L, d))
    w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = 2.0 / (1.0 + np.exp(-rng.standard_normal((BH, L))))
    if beta_fixed is not None:
        beta = np.full((BH, L), float(beta_fixed))
    x = dict(q=q, k=k, v=v, w=w, beta=beta, dout=dout, dlse=rng.standard_normal((BH, L)))
    if fox:
        x["log_f"] = -np.log1p(np.exp(-(rng.standard_normal((BH, L)) + 3.0)))
    return x


def brute_force_grads(x, use_dlse, fox):
    """Autograd through explicit d x d products, one head at a time."""
    names = ["q", "k", "v", "w", "beta"] + (["log_f"] if fox else [])
    t = {n: torch.tensor(x[n], dtype=torch.float64, requires_grad=True) for n in names}
    BH, L, d = x["q"].shape
    scale = 1.0 / np.sqrt(d)
    eye = torch.eye(d, dtype=torch.float64)
    loss = 0.0
    for h in range(BH):
        H = [eye - t["beta"][h, s] * torch.outer(t["w"][h, s], t["w"][h, s]) for s in range(L)]
        rows = []
        for i in range(L):
            row = []
            for j in range(L):
                if j > i:
                    row.append(torch.tensor(-np.inf, dtype=torch.float64))
                    continue
                M = eye
                for s in range(j + 1, i + 1):
                    M = M @ H[s]
                lg = scale * (t["k"][h, j] @ M @ t["q"][h, i])
                if fox:
                    lg = lg + t["log_f"][h, j + 1:i + 1].sum()
                row.append(lg)
            rows.append(torch.stack(row))
        S = torch.stack(rows)
        out = torch.softmax(S, dim=-1) @ t["v"][h]
        lse = torch.logsumexp(S, dim=-1)
        loss = loss + (out * torch.tensor(x["dout"][h])).sum()
        if use_dlse:
            loss = loss + (lse * torch.tensor(x["dlse"][h])).sum()
    loss.backward()
    return {"d" + n: t[n].grad.numpy() for n in names}


def oracle_grads(x, use_dlse, fox):
    return oracle.prefill_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["dout"],
                              log_f=x["log_f"] if fox else None,
                              dlse=x["dlse"] if use_dlse else None)


@pytest.mark.parametrize("fox", [False, True])
@pytest.mark.parametrize("use_dlse", [False, True])
def test_matches_autograd_of_explicit_products(fox, use_dlse):
    x = draw(2, 7, 5, seed=11 + fox + 2 * use_dlse, fox=fox)
    ref = brute_force_grads(x, use_dlse, fox)
    got = oracle_grads(x, use_dlse, fox)
    assert set(got) == set(ref)
    for n in ref:
        np.testing.assert_allclose(got[n], ref[n], rtol=0, atol=1e-11, err_msg=n)


@pytest.mark.parametrize("beta_fixed", [1.0, 2.0])
def test_matches_autograd_at_singular_and_orthogonal_beta(beta_fixed):
    """beta = 1 makes H singular (a projection); beta = 2 makes it orthogonal."""
    x = draw(1, 6, 4, seed=21, beta_fixed=beta_fixed)
    ref = brute_force_grads(x, True, False)
    got = oracle_grads(x, True, False)
    for n in ref:
        np.testing.assert_allclose(got[n], ref[n], rtol=0, atol=1e-11, err_msg=n)


def test_single_token():
    """L = 1: out = v_0, so dv = dout, and the only logit carries dlse alone."""
    x = draw(1, 1, 6, seed=3)
    g = oracle_grads(x, True, False)
    np.testing.assert_allclose(g["dv"], x["dout"], atol=1e-15)
    np.testing.assert_allclose(g["dq"][0, 0], x["dlse"][0, 0] * x["k"][0, 0] / np.sqrt(6),
                               atol=1e-15)
    assert np.all(g["dw"] == 0) and np.all(g["dbeta"] == 0)


def test_central_differences_of_the_forward_oracle():
    x = draw(1, 9, 6, seed=5, fox=True)
    g = oracle_grads(x, True, True)

    def loss(y):
        out, lse = oracle.prefill(y["q"], y["k"], y["v"], y["w"], y["beta"], log_f=y["log_f"])
        return float((out * x["dout"]).sum() + (lse * x["dlse"]).sum())

    rng = np.random.default_rng(0)
    h = 1e-6
    for n in ("q", "k", "v", "w", "beta", "log_f"):
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in x[n].shape)
            yp = {m: a.copy() for m, a in x.items()}
            ym = {m: a.copy() for m, a in x.items()}
            yp[n][idx] += h
            ym[n][idx] -= h
            fd = (loss(yp) - loss(ym)) / (2 * h)
            assert abs(fd - g["d" + n][idx]) <= 1e-7 * max(1.0, abs(fd)), (n, idx)


def test_beta_zero_is_softmax_attention():
    x = draw(2, 12, 8, seed=9, beta_fixed=0.0)
    g = oracle_grads(x, False, False)
    t = {n: torch.tensor(x[n], requires_grad=True) for n in ("q", "k", "v")}
    out = torch.nn.functional.scaled_dot_product_attention(t["q"], t["k"], t["v"], is_causal=True)
    (out * torch.tensor(x["dout"])).sum().backward()
    for n in ("q", "k", "v"):
        np.testing.assert_allclose(g["d" + n], t[n].grad.numpy(), rtol=0, atol=1e-12)
    assert np.all(g["dw"] == 0)
