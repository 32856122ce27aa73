"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

The recurrence is h_t = exp(g_t)(I - beta_t k_t k_t^T) h_{t-1} + beta_t k_t v_t^T and
o_t = h_t^T q_t (the per-token rule behind the chunk map of "Add context parallelism to
the Gated Delta Net", section "Why").  Pins here:
  * exact rational brute force of that dense matrix form (Fractions, no rounding);
  * a hand-worked 2x2 example;
  * numpy dense-form brute force on small random problems (GQA, several sequences,
    ragged tails) for the token, chunked and segmented forms;
  * beta = 0 closed form; orthonormal-key closed form (decayed, beta-weighted linear
    attention); the overwrite property (g = 0, beta = 1);
  * padding no-op ("Implementation", chunk padding bullet), segment-count invariance and
    associativity ("Why"), split-call resume, linearity in (h0, v), the contraction bound;
  * UT residual and the WY factors against a library linear solve; low-rank M_r against the
    dense product of per-token transitions.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


# ----------------------------------------------------------------------------- helpers

def rand_problem(seed, T=40, hk=2, hv=4, K=8, V=6, lengths=None, h0=True, unit_keys=True,
                 g_scale=0.3):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, hk, K))
    k = rng.standard_normal((T, hk, K))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, hv, V))
    g = -g_scale * rng.random((T, hv))
    beta = rng.random((T, hv))
    if lengths is None:
        lengths = [T]
    assert sum(lengths) == T
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    h0a = rng.standard_normal((len(lengths), hv, K, V)) * 0.5 if h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0a, cu_seqlens=cu)


def dense_reference(q, k, v, g, beta, h0, cu_seqlens):
    """The recurrence in its dense matrix form, written directly with numpy matrices."""
    T, hk, K = k.shape
    hv, V = v.shape[1], v.shape[2]
    N = len(cu_seqlens) - 1
    out = np.zeros((T, hv, V))
    hf = np.zeros((N, hv, K, V))
    for n in range(N):
        for j in range(hv):
            kh = j // (hv // hk)
            h = np.zeros((K, V)) if h0 is None else h0[n, j].copy()
            for t in range(cu_seqlens[n], cu_seqlens[n + 1]):
                kt = k[t, kh][:, None]
                trans = np.exp(g[t, j]) * (np.eye(K) - beta[t, j] * kt @ kt.T)
                h = trans @ h + beta[t, j] * kt @ v[t, j][None, :]
                out[t, j] = h.T @ q[t, kh]
            hf[n, j] = h
    return out, hf


def maxdiff(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0


# ------------------------------------------------------------ exact and hand-worked pins

def test_exact_rational_brute_force():
    """Dense form evaluated in exact rational arithmetic; the oracle must agree to 1e-13.
    The decay factors are rationals alpha_t and the oracle gets g_t = log(alpha_t)."""
    rng = np.random.default_rng(7)
    T, K, V = 7, 3, 2

    def frac():
        return Fraction(int(rng.integers(-9, 10)), int(rng.integers(1, 7)))

    k = [[frac() for _ in range(K)] for _ in range(T)]
    q = [[frac() for _ in range(K)] for _ in range(T)]
    v = [[frac() for _ in range(V)] for _ in range(T)]
    alpha = [Fraction(int(rng.integers(1, 9)), 8) for _ in range(T)]
    beta = [Fraction(int(rng.integers(0, 9)), 8) for _ in range(T)]
    h = [[frac() for _ in range(V)] for _ in range(K)]
    h0 = [row[:] for row in h]
    outs = []
    for t in range(T):
        trans = [[alpha[t] * ((1 if a == b else 0) - beta[t] * k[t][a] * k[t][b])
                  for b in range(K)] for a in range(K)]
        h = [[sum(trans[a][i] * h[i][c] for i in range(K)) + beta[t] * k[t][a] * v[t][c]
              for c in range(V)] for a in range(K)]
        outs.append([sum(h[i][c] * q[t][i] for i in range(K)) for c in range(V)])

    def arr(x):
        return np.array([[float(e) for e in row] for row in x])

    args = dict(q=arr(q)[:, None, :], k=arr(k)[:, None, :], v=arr(v)[:, None, :],
                g=np.log(np.array([float(a) for a in alpha]))[:, None],
                beta=np.array([float(b) for b in beta])[:, None], h0=arr(h0)[None, None])
    exp_out, exp_h = arr(outs), arr(h)
    scale = max(1.0, np.abs(exp_out).max(), np.abs(exp_h).max())
    o, hf = oracle.token(**args)
    assert maxdiff(o[:, 0], exp_out) <= 1e-13 * scale
    assert maxdiff(hf[0, 0], exp_h) <= 1e-13 * scale
    for C in (2, 3, 64):
        o, hf = oracle.chunked(**args, C=C)
        assert maxdiff(o[:, 0], exp_out) <= 1e-12 * scale
        assert maxdiff(hf[0, 0], exp_h) <= 1e-12 * scale
        for P in (1, 2, 3):
            o, hf = oracle.segmented(**args, C=C, P=P)
            assert maxdiff(o[:, 0], exp_out) <= 1e-12 * scale
            assert maxdiff(hf[0, 0], exp_h) <= 1e-12 * scale


def test_hand_worked_2x2():
    """Three tokens worked by hand (K = V = 2, h0 = 0).
    t1: alpha=1, beta=1/2, k=(1,0), v=(2,4):  h1 = [[1,2],[0,0]],  q=(1,0) -> o1=(1,2).
    t2: alpha=1/2, beta=1, k=(0,1), v=(6,0): h2 = 1/2 h1 + e2 (6,0) = [[.5,1],[6,0]],
        q=(1,1) -> o2=(6.5,1).
    t3: alpha=1, beta=1, k=(1,0), v=(0,0):   h3 = (I - e1 e1^T) h2 = [[0,0],[6,0]]
        (row 1 erased), q=(0,1) -> o3=(6,0)."""
    q = np.array([[1, 0], [1, 1], [0, 1]], float)[:, None]
    k = np.array([[1, 0], [0, 1], [1, 0]], float)[:, None]
    v = np.array([[2, 4], [6, 0], [0, 0]], float)[:, None]
    g = np.log(np.array([1.0, 0.5, 1.0]))[:, None]
    beta = np.array([0.5, 1.0, 1.0])[:, None]
    expect_o = np.array([[1, 2], [6.5, 1], [6, 0]], float)
    expect_h = np.array([[0, 0], [6, 0]], float)
    for fn in (oracle.token, lambda *a: oracle.chunked(*a, C=2),
               lambda *a: oracle.segmented(*a, C=1, P=3)):
        o, hf = fn(q, k, v, g, beta)
        assert maxdiff(o[:, 0], expect_o) < 1e-14
        assert maxdiff(hf[0, 0], expect_h) < 1e-14


# ------------------------------------------------------------------- brute-force pins

@pytest.mark.parametrize("seed,lengths,C", [
    (0, [40], 8), (1, [13, 27], 8), (2, [5, 1, 34], 16), (3, [40], 64), (4, [0, 40], 8)])
def test_forms_match_dense_brute_force(seed, lengths, C):
    p = rand_problem(seed, lengths=lengths)
    ref_o, ref_h = dense_reference(**p)
    o, hf = oracle.token(**p)
    assert maxdiff(o, ref_o) < 1e-12 and maxdiff(hf, ref_h) < 1e-12
    o, hf = oracle.chunked(**p, C=C)
    assert maxdiff(o, ref_o) < 1e-12 and maxdiff(hf, ref_h) < 1e-12
    for P in (1, 2, 3, 7):
        o, hf = oracle.segmented(**p, C=C, P=P)
        assert maxdiff(o, ref_o) < 1e-12, P
        assert maxdiff(hf, ref_h) < 1e-12, P


def test_gqa_grouped_order():
    """Value head j reads key head j // (hv // hk); a tiled map (j % hk) must differ."""
    p = rand_problem(11, hk=2, hv=4)
    o, _ = oracle.token(**p)
    for j in range(4):
        sub = dict(p, q=p["q"][:, j // 2:j // 2 + 1], k=p["k"][:, j // 2:j // 2 + 1],
                   v=p["v"][:, j:j + 1], g=p["g"][:, j:j + 1], beta=p["beta"][:, j:j + 1],
                   h0=p["h0"][:, j:j + 1])
        o1, _ = oracle.token(**sub)
        assert maxdiff(o1[:, 0], o[:, j]) == 0.0
    tiled = dict(p, q=p["q"][:, [0, 1]][:, [1, 0]], k=p["k"][:, [1, 0]])
    o2, _ = oracle.token(**tiled)
    assert maxdiff(o2, o) > 1e-3


# ------------------------------------------------------------------ closed-form pins

def test_beta_zero_is_pure_decay():
    """beta = 0: no write, no erase: h_T = exp(sum g) h0 and o_t = exp(G_t) h0^T q_t."""
    p = rand_problem(21, lengths=[40])
    p["beta"][:] = 0.0
    G = np.cumsum(p["g"], axis=0)
    exp_h = np.exp(G[-1])[None, :, None, None] * p["h0"]
    exp_o = np.einsum("tj,jkv,tjk->tjv", np.exp(G), p["h0"][0],
                      np.repeat(p["q"], 2, axis=1))
    for fn in (oracle.token, lambda **a: oracle.chunked(**a, C=8),
               lambda **a: oracle.segmented(**a, C=8, P=3)):
        o, hf = fn(**p)
        assert maxdiff(hf, exp_h) < 1e-12
        assert maxdiff(o, exp_o) < 1e-12


def orthonormal_keys(rng, T, K):
    Q, _ = np.linalg.qr(rng.standard_normal((K, K)))
    return Q[:T]


def test_orthonormal_keys_is_decayed_linear_attention():
    """Mutually orthogonal unit keys and h0 = 0: the erase term never fires and
    o_t = sum_{j<=t} exp(G_t - G_j) beta_j (q_t . k_j) v_j for any g and beta."""
    rng = np.random.default_rng(5)
    T, K, V = 12, 16, 5
    k = orthonormal_keys(rng, T, K)[:, None]
    q = rng.standard_normal((T, 1, K))
    v = rng.standard_normal((T, 1, V))
    g = -rng.random((T, 1))
    beta = rng.random((T, 1)) * 2
    G = np.cumsum(g[:, 0])
    exp_o = np.zeros((T, V))
    for t in range(T):
        for j in range(t + 1):
            exp_o[t] += np.exp(G[t] - G[j]) * beta[j, 0] * (q[t, 0] @ k[j, 0]) * v[j, 0]
    for fn in (oracle.token, lambda *a: oracle.chunked(*a, C=5),
               lambda *a: oracle.segmented(*a, C=4, P=2)):
        o, _ = fn(q, k, v, g, beta)
        assert maxdiff(o[:, 0], exp_o) < 1e-12


def test_overwrite_with_repeated_orthonormal_keys():
    """g = 0, beta = 1: writing v with key k_i replaces row k_i of the state; reading with
    q = k_i returns the last v written there; unwritten directions keep h0."""
    rng = np.random.default_rng(9)
    K, V, T = 8, 4, 20
    basis = orthonormal_keys(rng, K, K)
    idx = rng.integers(0, 5, size=T)          # keys 0..4 written, 5..7 never
    k = basis[idx][:, None]
    v = rng.standard_normal((T, 1, V))
    q = k.copy()
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    h0 = rng.standard_normal((1, 1, K, V))
    for fn in (oracle.token, lambda *a, **kw: oracle.chunked(*a, **kw, C=6),
               lambda *a, **kw: oracle.segmented(*a, **kw, C=3, P=4)):
        o, hf = fn(q, k, v, g, beta, h0=h0)
        assert maxdiff(o[:, 0], v[:, 0]) < 1e-12          # read-back of what was just written
        for i in range(K):
            read = hf[0, 0].T @ basis[i]
            if i in idx:
                last = np.where(idx == i)[0][-1]
                assert maxdiff(read, v[last, 0]) < 1e-12
            else:
                assert maxdiff(read, h0[0, 0].T @ basis[i]) < 1e-12


# --------------------------------------------------------------------- invariants

def test_padding_is_a_no_op():
    """Tokens with g = 0 and q = k = v = 0 (any beta) leave the state untouched and read 0."""
    p = rand_problem(31, T=30, lengths=[30])
    rng = np.random.default_rng(1)
    pos = np.sort(rng.choice(np.arange(0, 45), size=15, replace=False))
    keep = np.setdiff1d(np.arange(45), pos)
    padded = {}
    for name, z in (("q", 0), ("k", 0), ("v", 0), ("g", 0), ("beta", None)):
        a = p[name]
        b = np.zeros((45,) + a.shape[1:])
        b[keep] = a
        if z is None:
            b[pos] = rng.random((len(pos),) + a.shape[1:])
        padded[name] = b
    o0, h0f = oracle.token(**p)
    o1, h1f = oracle.token(**padded, h0=p["h0"], cu_seqlens=[0, 45])
    assert np.array_equal(o1[keep], o0) and np.array_equal(h1f, h0f)   # bit-identical
    assert np.all(o1[pos] == 0.0)
    oc, hc = oracle.chunked(**padded, h0=p["h0"], cu_seqlens=[0, 45], C=8)
    assert np.all(oc[pos] == 0.0)
    assert maxdiff(oc[keep], o0) < 1e-12 and maxdiff(hc, h0f) < 1e-12


def test_segment_count_invariance_and_empty_segments():
    p = rand_problem(41, T=70, lengths=[70])
    ref_o, ref_h = oracle.chunked(**p, C=8)
    for P in (1, 2, 4, 9, 12):   # 9 chunks: P=12 leaves three segments empty
        o, hf = oracle.segmented(**p, C=8, P=P)
        assert maxdiff(o, ref_o) < 1e-12 and maxdiff(hf, ref_h) < 1e-12


def test_split_call_resume():
    p = rand_problem(51, T=50, lengths=[50])
    o, hf = oracle.token(**p)
    T1 = 23
    a = {n: p[n][:T1] for n in ("q", "k", "v", "g", "beta")}
    b = {n: p[n][T1:] for n in ("q", "k", "v", "g", "beta")}
    oa, ha = oracle.token(**a, h0=p["h0"])
    ob, hb = oracle.token(**b, h0=ha)
    assert np.array_equal(np.concatenate([oa, ob]), o) and np.array_equal(hb, hf)
    oa, ha = oracle.chunked(**a, h0=p["h0"], C=8)
    ob, hb = oracle.chunked(**b, h0=ha, C=8)
    assert maxdiff(np.concatenate([oa, ob]), o) < 1e-12 and maxdiff(hb, hf) < 1e-12


def test_linearity_in_h0_and_v():
    p = rand_problem(61, T=33, lengths=[33])
    o, hf = oracle.segmented(**p, C=8, P=2)
    o1, h1 = oracle.segmented(**dict(p, v=np.zeros_like(p["v"])), C=8, P=2)
    o2, h2 = oracle.segmented(**dict(p, h0=np.zeros_like(p["h0"])), C=8, P=2)
    assert maxdiff(o, o1 + o2) < 1e-12 and maxdiff(hf, h1 + h2) < 1e-12
    o3, h3 = oracle.segmented(**dict(p, v=3 * p["v"], h0=3 * p["h0"]), C=8, P=2)
    assert maxdiff(o3, 3 * o) < 1e-11 and maxdiff(h3, 3 * hf) < 1e-11


def test_contraction_bound():
    """Unit keys, beta in [0, 2]: (I - beta k k^T) has spectral norm <= 1, so
    ||h_t||_2 <= alpha_t ||h_{t-1}||_2 + beta_t ||v_t||_2 (states taken by split calls)."""
    p = rand_problem(71, T=24, hk=1, hv=1, lengths=[24])
    p["beta"] = np.random.default_rng(2).random((24, 1)) * 2
    h = p["h0"]
    for t in range(24):
        _, hn = oracle.token(q=p["q"][t:t + 1], k=p["k"][t:t + 1], v=p["v"][t:t + 1],
                             g=p["g"][t:t + 1], beta=p["beta"][t:t + 1], h0=h)
        lhs = np.linalg.norm(hn[0, 0], 2)
        rhs = (np.exp(p["g"][t, 0]) * np.linalg.norm(h[0, 0], 2)
               + p["beta"][t, 0] * np.linalg.norm(p["v"][t, 0]))
        assert lhs <= rhs * (1 + 1e-12)
        h = hn


# ---------------------------------------------------------------------- stage pins

def test_chunk_factors_against_linear_solve():
    """UT residual ||(I + A) T - I|| and w, u against numpy's solve of (I + A) X = B."""
    rng = np.random.default_rng(81)
    L, K, V = 64, 32, 24
    kc = rng.standard_normal((L, K))
    kc /= np.linalg.norm(kc, axis=1, keepdims=True)
    vc = rng.standard_normal((L, V))
    gc = -0.1 * rng.random(L)
    bc = rng.random(L)
    f = oracle.chunk_factors(kc, vc, gc, bc)
    G = np.cumsum(gc)
    assert maxdiff(f["G"], G) < 1e-14
    IA = np.eye(L) + f["A"]
    assert maxdiff(IA @ f["T"], np.eye(L)) < 1e-12
    assert maxdiff(np.triu(f["A"]), 0) == 0.0
    A_def = np.tril(bc[:, None] * np.exp(G[:, None] - G[None, :]) * (kc @ kc.T), -1)
    assert maxdiff(f["A"], A_def) < 1e-14
    assert maxdiff(f["w"], np.linalg.solve(IA, (bc * np.exp(G))[:, None] * kc)) < 1e-12
    assert maxdiff(f["u"], np.linalg.solve(IA, bc[:, None] * vc)) < 1e-12
    assert maxdiff(f["ktilde"], np.exp(G[-1] - G)[:, None] * kc) < 1e-14
    assert abs(f["gamma"] - np.exp(G[-1])) < 1e-15


def test_chunk_map_is_one_chunk_of_the_recurrence():
    """h_out = (gamma I - k_tilde^T w) h + k_tilde^T u reproduces L token steps exactly."""
    rng = np.random.default_rng(83)
    L, K, V = 16, 8, 5
    kc = rng.standard_normal((L, K))
    kc /= np.linalg.norm(kc, axis=1, keepdims=True)
    vc, gc, bc = rng.standard_normal((L, V)), -rng.random(L), rng.random(L)
    h = rng.standard_normal((K, V))
    f = oracle.chunk_factors(kc, vc, gc, bc)
    Mc = f["gamma"] * np.eye(K) - f["ktilde"].T @ f["w"]
    Uc = f["ktilde"].T @ f["u"]
    _, hf = dense_reference(kc[:, None], kc[:, None], vc[:, None], gc[:, None], bc[:, None],
                            h[None, None], [0, L])
    assert maxdiff(Mc @ h + Uc, hf[0, 0]) < 1e-12


def test_low_rank_summary_equals_dense_transition():
    p = rand_problem(91, T=45, hk=1, hv=2, lengths=[45])
    C, P = 8, 4   # 6 chunks over 4 segments: the first two get the extra chunk
    M, U = oracle.summary(p["k"], p["v"], p["g"], p["beta"], C=C, P=P)
    bounds = oracle.segment_bounds([0, 45], C, P)
    for r, (c0, c1) in enumerate(bounds):
        t0, t1 = c0 * C, min(c1 * C, 45)
        for j in range(2):
            Md = oracle.dense_transition(p["k"], p["g"], p["beta"], t0, t1, j, hv=2)
            assert maxdiff(M[r, j], Md) < 1e-12
            # U_r is the zero-state end of the segment
            sub = {n: p[n][t0:t1] for n in ("q", "k", "v", "g", "beta")}
            _, hz = oracle.token(**sub)
            assert maxdiff(U[r, j], hz[0, j]) < 1e-12


def test_scan_is_exclusive_and_ordered():
    """h_in[0] = h0; h_in[r+1] = M_r h_in[r] + U_r; and the scan is order sensitive: feeding
    the segments in a different order (a load-balancing reorder) gives a different state."""
    p = rand_problem(93, T=64, hk=1, hv=1, lengths=[64])
    M, U = oracle.summary(p["k"], p["v"], p["g"], p["beta"], C=8, P=4)
    h_in, hf = oracle.scan(M, U, p["h0"], N=1, P=4)
    assert np.array_equal(h_in[0], p["h0"][0])
    _, ref = oracle.token(**p)
    assert maxdiff(hf, ref) < 1e-12
    for r in range(4):
        _, hr = oracle.token(**{n: p[n][:16 * r] for n in ("q", "k", "v", "g", "beta")},
                             h0=p["h0"])
        assert maxdiff(h_in[r], hr[0]) < 1e-12
    perm = [0, 3, 1, 2]   # a zig-zag style reorder of the segments
    _, hbad = oracle.scan(M[perm], U[perm], p["h0"], N=1, P=4)
    assert maxdiff(hbad, ref) > 1e-3


def test_prepare_and_emit_stages_compose():
    p = rand_problem(95, T=50, lengths=[20, 30])
    w, u, gcum = oracle.prepare(p["k"], p["v"], p["g"], p["beta"], p["cu_seqlens"], C=8)
    # prepare is token aligned: chunk-by-chunk factors
    for n, (a, b) in enumerate([(0, 20), (20, 50)]):
        for t0 in range(a, b, 8):
            L = min(8, b - t0)
            for j in range(4):
                f = oracle.chunk_factors(p["k"][t0:t0 + L, j // 2], p["v"][t0:t0 + L, j],
                                         p["g"][t0:t0 + L, j], p["beta"][t0:t0 + L, j])
                assert maxdiff(w[t0:t0 + L, j], f["w"]) == 0.0
                assert maxdiff(u[t0:t0 + L, j], f["u"]) == 0.0
                assert maxdiff(gcum[t0:t0 + L, j], np.cumsum(p["g"][t0:t0 + L, j])) < 1e-15
    M, U = oracle.summary(p["k"], p["v"], p["g"], p["beta"], p["cu_seqlens"], C=8, P=2)
    h_in, hf = oracle.scan(M, U, p["h0"], N=2, P=2)
    o = oracle.emit(p["q"], p["k"], p["v"], p["g"], p["beta"], h_in, p["cu_seqlens"], C=8, P=2)
    ref_o, ref_h = dense_reference(**p)
    assert maxdiff(o, ref_o) < 1e-12 and maxdiff(hf, ref_h) < 1e-12


def test_oracle_rejects_bad_geometry():
    p = rand_problem(97)
    with pytest.raises(ValueError):
        oracle.token(**dict(p, cu_seqlens=[0, 10]))          # cu[N] != T
    with pytest.raises(ValueError):
        oracle.token(**dict(p, cu_seqlens=[0, 30, 20, 40]))  # decreasing


# ------------------------------------------------------------------------ decode over slots

def test_decode_steps_over_a_slot_pool_equal_the_recurrence():
    """Three requests in a pool of five slots, decoded token by token in an interleaved order
    with padding rows, equal the dense recurrence of each request's own sequence; the slots
    no request uses keep their states ("RFC(qwen35): TP Phase2", "Request-State
    Lifecycle": one request's state is never touched by another's work)."""
    rng = np.random.default_rng(11)
    hk, hv, K, V, S = 1, 2, 4, 3, 5
    lengths = [4, 6, 3]
    home = [3, 0, 4]  # slot of each request
    seqs = [rand_problem(20 + i, T=L, hk=hk, hv=hv, K=K, V=V) for i, L in enumerate(lengths)]
    state = rng.standard_normal((S, hv, K, V))
    start = state.copy()
    for i, sl in enumerate(home):
        state[sl] = seqs[i]["h0"][0]
    pos = [0, 0, 0]
    outs = [np.zeros((L, hv, V)) for L in lengths]
    while any(pos[i] < lengths[i] for i in range(3)):
        rows = [i for i in range(3) if pos[i] < lengths[i] and rng.random() < 0.7]
        if not rows:
            continue
        order = list(rng.permutation(rows))
        pad = int(rng.integers(0, 2))
        B = len(order) + pad
        q = np.zeros((B, hk, K)); k = np.zeros((B, hk, K)); v = np.zeros((B, hv, V))
        g = np.zeros((B, hv)); beta = np.zeros((B, hv)); slot = -np.ones(B, dtype=np.int64)
        for b, i in enumerate(order):
            t = pos[i]
            q[b], k[b], v[b] = seqs[i]["q"][t], seqs[i]["k"][t], seqs[i]["v"][t]
            g[b], beta[b], slot[b] = seqs[i]["g"][t], seqs[i]["beta"][t], home[i]
        o, state = oracle.decode(q, k, v, g, beta, state, slot)
        for b, i in enumerate(order):
            outs[i][pos[i]] = o[b]
            pos[i] += 1
        assert np.all(o[len(order):] == 0)  # padding rows
    for i, sl in enumerate(home):
        ref_o, ref_h = dense_reference(**seqs[i])
        assert maxdiff(outs[i], ref_o) < 1e-12 and maxdiff(state[sl], ref_h[0]) < 1e-12
    for sl in set(range(S)) - set(home):
        assert np.array_equal(state[sl], start[sl])


def test_decode_rejects_shared_or_out_of_range_slots():
    z = lambda *s: np.zeros(s)
    with pytest.raises(ValueError):
        oracle.decode(z(2, 1, 4), z(2, 1, 4), z(2, 1, 4), z(2, 1), z(2, 1), z(3, 1, 4, 4), [1, 1])
    with pytest.raises(ValueError):
        oracle.decode(z(1, 1, 4), z(1, 1, 4), z(1, 1, 4), z(1, 1), z(1, 1), z(3, 1, 4, 4), [3])
