"""Pins of the oracle's reverse mode (``oracle.token_backward``) against facts that do not come
from it: central finite differences of the pinned forward, linearity in the cotangents, the
beta = 0 closed form, and the grouped-query sum.

The loss is L = <dout, out> + <dh_final, h_final> for the recurrence
h_t = exp(g_t)(I - beta_t k_t k_t^T) h_{t-1} + beta_t k_t v_t^T, o_t = h_t^T q_t (the per-token
rule behind the chunk map of "Add context parallelism to the Gated Delta Net", section "Why";
the page's section "Tests" and "Measured results" report backward parity of the sharded layer
against the single-device one, which is what the GPU backward is held to here).
"""
import numpy as np
import pytest

import oracle

NAMES = (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), ("h0", "dh0"))


def problem(seed, T=11, hk=1, hv=2, K=4, V=3, lengths=(5, 6)):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, hk, K))
    k = rng.standard_normal((T, hk, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, hv, V))
    g = -0.4 * rng.random((T, hv))
    beta = rng.random((T, hv))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    h0 = rng.standard_normal((len(lengths), hv, K, V))
    dout = rng.standard_normal((T, hv, V))
    dhf = rng.standard_normal((len(lengths), hv, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu_seqlens=cu), dout, dhf


def loss(x, dout, dhf):
    o, hf = oracle.token(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["cu_seqlens"])
    return float(np.sum(o * dout) + np.sum(hf * dhf))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gradients_match_central_differences(seed):
    x, dout, dhf = problem(seed)
    r = oracle.token_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], dout, x["h0"], dhf,
                              x["cu_seqlens"])
    rng = np.random.default_rng(100 + seed)
    eps = 1e-6
    for name, gname in NAMES:
        e = rng.standard_normal(x[name].shape)
        fd = (loss(dict(x, **{name: x[name] + eps * e}), dout, dhf)
              - loss(dict(x, **{name: x[name] - eps * e}), dout, dhf)) / (2 * eps)
        an = float(np.sum(r[gname] * e))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def test_linear_in_the_cotangents():
    x, d1, h1 = problem(5)
    _, d2, h2 = problem(6)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"])
    r1 = oracle.token_backward(*args, d1, x["h0"], h1, x["cu_seqlens"])
    r2 = oracle.token_backward(*args, d2, x["h0"], h2, x["cu_seqlens"])
    r3 = oracle.token_backward(*args, 2 * d1 - 3 * d2, x["h0"], 2 * h1 - 3 * h2, x["cu_seqlens"])
    for _, gname in NAMES:
        assert np.max(np.abs(r3[gname] - (2 * r1[gname] - 3 * r2[gname]))) < 1e-10


def test_beta_zero_closed_form():
    """beta = 0: h_t = exp(G_t) h0 with G the running sum of g, so o_t = exp(G_t) h0^T q_t and
    dq_t = exp(G_t) h0 dout_t, dk = dv = 0, dh0 = sum_t exp(G_t) q_t dout_t^T + exp(G_T) dh_f,
    dg_s = sum_{t >= s} exp(G_t) dout_t . (h0^T q_t) + exp(G_T) <dh_f, h0>."""
    x, dout, dhf = problem(7, T=6, hk=1, hv=1, lengths=(6,))
    x["beta"] = np.zeros_like(x["beta"])
    r = oracle.token_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], dout, x["h0"], dhf,
                              x["cu_seqlens"])
    G = np.cumsum(x["g"][:, 0])
    h0, q = x["h0"][0, 0], x["q"][:, 0]
    dq = np.stack([np.exp(G[t]) * h0 @ dout[t, 0] for t in range(6)])
    dh0 = sum(np.exp(G[t]) * np.outer(q[t], dout[t, 0]) for t in range(6)) + np.exp(G[-1]) * dhf[0, 0]
    a = np.array([np.exp(G[t]) * dout[t, 0] @ (h0.T @ q[t]) for t in range(6)])
    dg = np.array([a[s:].sum() for s in range(6)]) + np.exp(G[-1]) * np.sum(dhf[0, 0] * h0)
    assert np.max(np.abs(r["dq"][:, 0] - dq)) < 1e-12
    assert np.max(np.abs(r["dh0"][0, 0] - dh0)) < 1e-12
    assert np.max(np.abs(r["dg"][:, 0] - dg)) < 1e-12
    assert np.max(np.abs(r["dk"])) < 1e-15 and np.max(np.abs(r["dv"])) < 1e-15


def test_grouped_query_gradients_sum_over_the_group():
    """Two value heads reading one key head: dq, dk of the key head are the sums of what each
    value head alone (with its own copy of q, k) receives; the per-value-head gradients are
    unchanged."""
    x, dout, dhf = problem(9, lengths=(11,), T=11)
    r = oracle.token_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], dout, x["h0"], dhf,
                              x["cu_seqlens"])
    parts = [oracle.token_backward(x["q"], x["k"], x["v"][:, j:j + 1], x["g"][:, j:j + 1],
                                   x["beta"][:, j:j + 1], dout[:, j:j + 1], x["h0"][:, j:j + 1],
                                   dhf[:, j:j + 1], x["cu_seqlens"]) for j in range(2)]
    for gname in ("dq", "dk"):
        assert np.max(np.abs(r[gname] - parts[0][gname] - parts[1][gname])) < 1e-12
    for j in range(2):
        for gname, sl in (("dv", np.s_[:, j:j + 1]), ("dg", np.s_[:, j:j + 1]),
                          ("dbeta", np.s_[:, j:j + 1]), ("dh0", np.s_[:, j:j + 1])):
            assert np.max(np.abs(r[gname][sl] - parts[j][gname])) < 1e-12
