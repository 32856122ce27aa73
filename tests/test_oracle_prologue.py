"""Pins of the oracle's prologue (``oracle.prologue``) against library routines and invariants.

The pages fix a causal depthwise conv over the q | k | v channels with a halo of
conv_kernel_dim - 1 tokens ("Add context parallelism to the Gated Delta Net", "Implementation")
and a per-request conv state of qkv_dim x (conv_kernel_dim - 1) inputs ("RFC(qwen35): TP
Phase2", "Partition Contract").  The rest (optional SiLU, L2 normalisation of q and k, the g and
beta maps) are readings, pinned here to their plain definitions.
"""
import numpy as np
import pytest

import oracle

HK, HV, K, V, W = 2, 4, 8, 6, 4
CH = 2 * HK * K + HV * V


def problem(seed, T=23, lengths=(9, 14), state=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, CH))
    w = rng.standard_normal((CH, W))
    a = rng.standard_normal((T, HV))
    b = rng.standard_normal((T, HV))
    A_log = rng.standard_normal(HV) * 0.3
    dt = rng.standard_normal(HV) * 0.3
    cu = np.concatenate([[0], np.cumsum(lengths)])
    st = rng.standard_normal((len(lengths), CH, W - 1)) if state else None
    return x, w, a, b, A_log, dt, cu, st


def test_conv_is_a_causal_convolution_per_channel():
    """Before the L2 norm: the v channels equal numpy's full convolution of the carried inputs
    followed by the sequence, with the kernel reversed (a causal correlation), read at the
    sequence's positions."""
    x, w, a, b, A_log, dt, cu, st = problem(0)
    _, _, v, _, _, _ = oracle.prologue(x, w, a, b, A_log, dt, HK, HV, K, V, st, cu)
    for n in range(len(cu) - 1):
        for c in range(2 * HK * K, CH):
            seq = np.concatenate([st[n, c], x[cu[n]:cu[n + 1], c]])
            full = np.convolve(seq, w[c, ::-1])  # correlation with w: y_t = sum_i w_i x_{t-3+i}
            ref = full[W - 1:len(seq)]
            vv = v[cu[n]:cu[n + 1]].reshape(-1, HV * V)[:, c - 2 * HK * K]
            assert np.max(np.abs(vv - ref)) < 1e-12


def test_state_carried_across_calls_equals_one_call():
    """A sequence cut in two calls (the second starting from the first's new conv state) gives
    the first call's outputs and then the second's, exactly as one call over the whole."""
    x, w, a, b, A_log, dt, _, st = problem(1, lengths=(23,))
    whole = oracle.prologue(x, w, a, b, A_log, dt, HK, HV, K, V, st[:1], None)
    for cut in (1, 2, 3, 10):
        p1 = oracle.prologue(x[:cut], w, a[:cut], b[:cut], A_log, dt, HK, HV, K, V, st[:1], None)
        p2 = oracle.prologue(x[cut:], w, a[cut:], b[cut:], A_log, dt, HK, HV, K, V, p1[5], None)
        for i in range(5):
            assert np.max(np.abs(np.concatenate([p1[i], p2[i]]) - whole[i])) < 1e-12
        assert np.max(np.abs(p2[5] - whole[5])) < 1e-12


def test_short_sequences_shift_the_old_state_in():
    x, w, a, b, A_log, dt, cu, st = problem(2, T=3, lengths=(1, 0, 2))
    *_, new = oracle.prologue(x, w, a, b, A_log, dt, HK, HV, K, V, st, cu)
    assert np.array_equal(new[0], np.concatenate([st[0][:, 1:], x[0:1].T], axis=1))
    assert np.array_equal(new[1], st[1])                       # empty: unchanged
    assert np.array_equal(new[2], np.concatenate([st[2][:, 2:], x[1:3].T], axis=1))


def test_norms_maps_and_activation():
    x, w, a, b, A_log, dt, cu, st = problem(3)
    q, k, v, g, beta, _ = oracle.prologue(x, w, a, b, A_log, dt, HK, HV, K, V, st, cu)
    assert np.allclose(np.linalg.norm(q, axis=-1), 1) and np.allclose(np.linalg.norm(k, axis=-1), 1)
    # g = -exp(A_log) softplus(a + dt_bias): with A_log = log 0.1 and dt_bias = 0 this is the
    # workloads' recipe -softplus(a) * 0.1
    _, _, _, g1, _, _ = oracle.prologue(x, w, a, b, np.full(HV, np.log(0.1)), np.zeros(HV),
                                        HK, HV, K, V, st, cu)
    assert np.max(np.abs(g1 + 0.1 * np.log1p(np.exp(a)))) < 1e-14
    assert np.max(np.abs(beta - 1 / (1 + np.exp(-b)))) < 1e-15 and np.all(g < 0)
    _, _, vs, _, _, _ = oracle.prologue(x, w, a, b, A_log, dt, HK, HV, K, V, st, cu, "silu")
    assert np.max(np.abs(vs - v / (1 + np.exp(-v)))) < 1e-12
    with pytest.raises(ValueError):
        oracle.prologue(x, w, a, b, A_log, dt, HK, HV, K, V, st, cu, "relu")
