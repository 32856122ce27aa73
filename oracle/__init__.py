"""fp64 CPU oracle for the gated delta rule forward and its reverse mode -- TEST
INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library never imports, links or calls it, and it imports
nothing from the CUDA library.  The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64);
this module compiles it with gcc, loads it with ctypes and marshals numpy arrays.

Sources (web pages, by title and section):
  * "Add context parallelism to the Gated Delta Net (Qwen3-Next / Qwen3.5)", MaxText PR
    #5040 -- "Why" (affine chunk map h_out = M h + U, o = (q_g - attn_i w) h + attn_i u),
    "Implementation" (three phases, low-rank M composition, chunk padding is a no-op).
  * "RFC(qwen35): TP Phase2", pegainfer issue #694 -- "Partition Contract": recurrent
    state [Hv, K, V] f32.

Layouts: q, k [T, Hk, K]; v [T, Hv, V]; g, beta [T, Hv]; h0, h_final [N, Hv, K, V];
out [T, Hv, V]; cu_seqlens [N+1].  Value head j reads key head j // (Hv // Hk).

Parity notes: every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, exact rational brute force and invariants; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False, src: str | None = None, out: str | None = None,
          extra_flags: tuple = ()) -> str:
    """Compiles the oracle with gcc (portable flags: it runs on x86_64 and aarch64 hosts)."""
    src = src or _SRC
    out = out or _LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", *extra_flags,
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    i, i64, d = ctypes.c_int, ctypes.c_int64, _dp
    lib.gdn_oracle_token.argtypes = [d, d, d, d, d, d, i64, i, _i64p, i, i, i, i, i, d, d]
    lib.gdn_oracle_chunk_factors.argtypes = [i, i, i, d, d, d, d, d, d, d, d, d, d, d]
    lib.gdn_oracle_prepare.argtypes = [d, d, d, d, i64, i, _i64p, i, i, i, i, i, i, d, d, d]
    lib.gdn_oracle_chunked.argtypes = [d, d, d, d, d, d, i64, i, _i64p, i, i, i, i, i, i, d, d]
    lib.gdn_oracle_summary.argtypes = [d, d, d, d, i64, i, _i64p, i, i, i, i, i, i, i, d, d]
    lib.gdn_oracle_dense_transition.argtypes = [d, d, d, i64, i64, i, i, i, i, d]
    lib.gdn_oracle_scan.argtypes = [d, d, d, i, i, i, i, i, d, d]
    lib.gdn_oracle_emit.argtypes = [d, d, d, d, d, d, i64, i, _i64p, i, i, i, i, i, i, i, d]
    lib.gdn_oracle_segmented.argtypes = [d, d, d, d, d, d, i64, i, _i64p, i, i, i, i, i, i, i,
                                         d, d]
    lib.gdn_oracle_token_backward.argtypes = [d, d, d, d, d, d, d, d, i64, i, _i64p, i, i, i, i,
                                              i, d, d, d, d, d, d]
    for name in ("gdn_oracle_token", "gdn_oracle_chunk_factors", "gdn_oracle_prepare",
                 "gdn_oracle_chunked", "gdn_oracle_summary", "gdn_oracle_dense_transition",
                 "gdn_oracle_scan", "gdn_oracle_emit", "gdn_oracle_segmented",
                 "gdn_oracle_token_backward"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Builds (if stale) and loads the oracle library; ``path`` loads a given build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


class use_library:
    """Context manager that routes every call of this module to another build of the
    oracle (the mutation tests load deliberately broken copies this way)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = _lib
        _lib = load(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> exact widening on the CPU
        x = x.detach().to("cpu")
        x = x.double().numpy() if x.is_floating_point() else x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _cu(cu, T):
    if cu is None:
        return np.array([0, T], dtype=np.int64)
    if hasattr(cu, "detach"):
        cu = cu.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int64))


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: oracle rejected its arguments (code {rc})")


class Problem:
    """Shapes of one call, read off the input arrays."""

    def __init__(self, q, k, v, g, beta, cu):
        self.T, self.hk, self.K = k.shape
        self.hv, self.V = v.shape[1], v.shape[2]
        if q is not None:
            assert q.shape == k.shape
        assert v.shape[0] == self.T and g.shape == (self.T, self.hv) == beta.shape
        self.cu = _cu(cu, self.T)
        self.N = len(self.cu) - 1


def token(q, k, v, g, beta, h0=None, cu_seqlens=None, nthreads=None):
    """The plain definition: the per-token recurrence.  Returns (out, h_final) in fp64."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    p = Problem(q, k, v, g, beta, cu_seqlens)
    out = np.zeros((p.T, p.hv, p.V))
    hf = np.zeros((p.N, p.hv, p.K, p.V))
    rc = load().gdn_oracle_token(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), p.T,
                                 p.N, p.cu.ctypes.data_as(_i64p), p.hk, p.hv, p.K, p.V,
                                 _threads(nthreads), _ptr(out), _ptr(hf))
    _check(rc, "token")
    return out, hf


def token_backward(q, k, v, g, beta, dout, h0=None, dh_final=None, cu_seqlens=None,
                   nthreads=None):
    """Reverse mode of the per-token recurrence: the gradients of
    L = <dout, out> + <dh_final, h_final> with respect to q, k, v, g, beta and h0, in fp64.
    The pages state no backward formulas; this follows from the recurrence alone (the
    derivation is in gdn_oracle.c, section 7).  Returns a dict of dq, dk [T, hk, K],
    dv [T, hv, V], dg, dbeta [T, hv] and dh0 [N, hv, K, V]."""
    q, k, v, g, beta, dout, h0, dh_final = map(_f64, (q, k, v, g, beta, dout, h0, dh_final))
    p = Problem(q, k, v, g, beta, cu_seqlens)
    assert dout.shape == v.shape
    r = {"dq": np.zeros((p.T, p.hk, p.K)), "dk": np.zeros((p.T, p.hk, p.K)),
         "dv": np.zeros((p.T, p.hv, p.V)), "dg": np.zeros((p.T, p.hv)),
         "dbeta": np.zeros((p.T, p.hv)), "dh0": np.zeros((p.N, p.hv, p.K, p.V))}
    rc = load().gdn_oracle_token_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(dout), _ptr(dh_final),
        p.T, p.N, p.cu.ctypes.data_as(_i64p), p.hk, p.hv, p.K, p.V, _threads(nthreads),
        _ptr(r["dq"]), _ptr(r["dk"]), _ptr(r["dv"]), _ptr(r["dg"]), _ptr(r["dbeta"]),
        _ptr(r["dh0"]))
    _check(rc, "token_backward")
    return r


def prologue(x, conv_w, a, b, A_log, dt_bias, hk, hv, K, V, conv_state=None, cu_seqlens=None,
             activation="none"):
    """The layer-side steps ahead of the recurrence, in fp64 (page "Add context parallelism to
    the Gated Delta Net", section "Implementation", layer-side bullets: a causal depthwise conv
    over the q | k | v channels whose halo is conv_kernel_dim - 1 tokens; page "RFC(qwen35): TP
    Phase2", section "Partition Contract": a per-request conv state of qkv_dim x
    (conv_kernel_dim - 1) inputs).  Readings where the pages are silent: the conv output may
    pass through SiLU (``activation``); q and k are L2-normalised per (token, head); g =
    -exp(A_log) softplus(a + dt_bias) and beta = sigmoid(b) per value head.
      x [T, 2 hk K + hv V] (q channels, then k, then v); conv_w [channels, W];
      conv_state [N, channels, W - 1] (the inputs before each sequence, oldest first; None =
      zeros); a, b [T, hv]; A_log, dt_bias [hv].
    Returns q, k [T, hk, K], v [T, hv, V], g, beta [T, hv], new conv state [N, channels, W - 1]
    (the last W - 1 inputs of each sequence, older state entries shifting in when a sequence is
    shorter than W - 1)."""
    x, conv_w, a, b, A_log, dt_bias = map(_f64, (x, conv_w, a, b, A_log, dt_bias))
    T, Ch = x.shape
    W = conv_w.shape[1]
    cu = _cu(cu_seqlens, T)
    N = len(cu) - 1
    st = np.zeros((N, Ch, W - 1)) if conv_state is None else _f64(conv_state)
    y = np.zeros((T, Ch))
    new_state = np.zeros((N, Ch, W - 1))
    for n in range(N):
        # the sequence's inputs with the W - 1 carried ones in front: ext[s + W - 1] = x[cu[n] + s]
        ext = np.concatenate([st[n].T, x[cu[n]:cu[n + 1]]], axis=0)
        L = cu[n + 1] - cu[n]
        for t in range(L):
            y[cu[n] + t] = np.sum(ext[t:t + W] * conv_w.T, axis=0)
        new_state[n] = ext[len(ext) - (W - 1):].T if W > 1 else new_state[n]
    if activation == "silu":
        y = y / (1.0 + np.exp(-y))
    elif activation != "none":
        raise ValueError(activation)
    q = y[:, :hk * K].reshape(T, hk, K)
    k = y[:, hk * K:2 * hk * K].reshape(T, hk, K)
    v = y[:, 2 * hk * K:].reshape(T, hv, V)
    q = q / np.sqrt(np.maximum(np.sum(q * q, -1, keepdims=True), 1e-12))
    k = k / np.sqrt(np.maximum(np.sum(k * k, -1, keepdims=True), 1e-12))
    g = -np.exp(A_log)[None, :] * np.logaddexp(0.0, a + dt_bias[None, :])
    beta = 1.0 / (1.0 + np.exp(-b))
    return q, k, v, g, beta, new_state


def decode(q, k, v, g, beta, state, slot, nthreads=None):
    """One decode step over a pool of per-slot states ("RFC(qwen35): TP Phase2", sections
    "Execution Contract" -- decode updates only the request's own recurrent state -- and
    "Request-State Lifecycle" -- requests live in reusable slots).  Row b continues the request
    whose state is state[slot[b]] by one token of the recurrence: ``token`` on a one-token
    sequence per row, with that state as h0.  A negative slot is a padding row (output 0, no
    state).  Slots must be distinct and in range (ValueError otherwise).  Returns
    (out [B, hv, V], new_state [S, hv, K, V]) in fp64; `state` itself is not modified."""
    q, k, v, g, beta, state = map(_f64, (q, k, v, g, beta, state))
    slot = np.asarray(slot, dtype=np.int64)
    B, hv, V = v.shape
    live = np.nonzero(slot >= 0)[0]
    sl = slot[live]
    if np.any(sl >= state.shape[0]) or len(set(sl.tolist())) != len(sl):
        raise ValueError("slots must be distinct and below the pool size")
    out = np.zeros((B, hv, V))
    new_state = state.copy()
    if len(live):
        o, hf = token(q[live], k[live], v[live], g[live], beta[live], state[sl],
                      np.arange(len(live) + 1, dtype=np.int64), nthreads=nthreads)
        out[live] = o
        new_state[sl] = hf
    return out, new_state


def chunk_factors(kc, vc, gc, bc):
    """WY/UT factors of one chunk of L rows: dict of G, A, T, w, u, ktilde, gamma."""
    kc, vc, gc, bc = map(_f64, (kc, vc, gc, bc))
    L, K = kc.shape
    V = vc.shape[1]
    o = {"G": np.zeros(L), "A": np.zeros((L, L)), "T": np.zeros((L, L)),
         "w": np.zeros((L, K)), "u": np.zeros((L, V)), "ktilde": np.zeros((L, K)),
         "gamma": np.zeros(1)}
    rc = load().gdn_oracle_chunk_factors(L, K, V, _ptr(kc), _ptr(vc), _ptr(gc), _ptr(bc),
                                         *(_ptr(o[n]) for n in ("G", "A", "T", "w", "u",
                                                                 "ktilde", "gamma")))
    _check(rc, "chunk_factors")
    o["gamma"] = float(o["gamma"][0])
    return o


def prepare(k, v, g, beta, cu_seqlens=None, C=64, nthreads=None):
    """WY factors of every chunk, token-aligned: (w [T,Hv,K], u [T,Hv,V], gcum [T,Hv])."""
    k, v, g, beta = map(_f64, (k, v, g, beta))
    p = Problem(None, k, v, g, beta, cu_seqlens)
    w = np.zeros((p.T, p.hv, p.K))
    u = np.zeros((p.T, p.hv, p.V))
    gc = np.zeros((p.T, p.hv))
    rc = load().gdn_oracle_prepare(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), p.T, p.N,
                                   p.cu.ctypes.data_as(_i64p), p.hk, p.hv, p.K, p.V, C,
                                   _threads(nthreads), _ptr(w), _ptr(u), _ptr(gc))
    _check(rc, "prepare")
    return w, u, gc


def chunked(q, k, v, g, beta, h0=None, cu_seqlens=None, C=64, nthreads=None):
    """Single-pass chunked form (chunk map applied chunk after chunk): (out, h_final)."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    p = Problem(q, k, v, g, beta, cu_seqlens)
    out = np.zeros((p.T, p.hv, p.V))
    hf = np.zeros((p.N, p.hv, p.K, p.V))
    rc = load().gdn_oracle_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                   p.T, p.N, p.cu.ctypes.data_as(_i64p), p.hk, p.hv, p.K, p.V, C,
                                   _threads(nthreads), _ptr(out), _ptr(hf))
    _check(rc, "chunked")
    return out, hf


def summary(k, v, g, beta, cu_seqlens=None, C=64, P=1, nthreads=None):
    """Phase 1: (M [N*P,Hv,K,K], U [N*P,Hv,K,V]) from a zero state, low-rank composed."""
    k, v, g, beta = map(_f64, (k, v, g, beta))
    p = Problem(None, k, v, g, beta, cu_seqlens)
    M = np.zeros((p.N * P, p.hv, p.K, p.K))
    U = np.zeros((p.N * P, p.hv, p.K, p.V))
    rc = load().gdn_oracle_summary(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), p.T, p.N,
                                   p.cu.ctypes.data_as(_i64p), p.hk, p.hv, p.K, p.V, C, P,
                                   _threads(nthreads), _ptr(M), _ptr(U))
    _check(rc, "summary")
    return M, U


def dense_transition(k, g, beta, t0, t1, j, hv):
    """Dense product of the per-token maps of tokens [t0, t1) for value head j."""
    k, g, beta = map(_f64, (k, g, beta))
    T, hk, K = k.shape
    M = np.zeros((K, K))
    rc = load().gdn_oracle_dense_transition(_ptr(k), _ptr(g), _ptr(beta), int(t0), int(t1), hk,
                                            hv, K, int(j), _ptr(M))
    _check(rc, "dense_transition")
    return M


def scan(M, U, h0=None, N=1, P=1):
    """Phase 2: exclusive scan -> (h_in [N*P,Hv,K,V], h_final [N,Hv,K,V])."""
    M, U, h0 = map(_f64, (M, U, h0))
    _, hv, K, V = U.shape
    h_in = np.zeros((N * P, hv, K, V))
    hf = np.zeros((N, hv, K, V))
    rc = load().gdn_oracle_scan(_ptr(M), _ptr(U), _ptr(h0), N, P, hv, K, V, _ptr(h_in), _ptr(hf))
    _check(rc, "scan")
    return h_in, hf


def emit(q, k, v, g, beta, h_in, cu_seqlens=None, C=64, P=1, nthreads=None):
    """Phase 3: re-run every segment from its incoming state, emitting out [T,Hv,V]."""
    q, k, v, g, beta, h_in = map(_f64, (q, k, v, g, beta, h_in))
    p = Problem(q, k, v, g, beta, cu_seqlens)
    out = np.zeros((p.T, p.hv, p.V))
    rc = load().gdn_oracle_emit(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h_in),
                                p.T, p.N, p.cu.ctypes.data_as(_i64p), p.hk, p.hv, p.K, p.V, C, P,
                                _threads(nthreads), _ptr(out))
    _check(rc, "emit")
    return out


def segmented(q, k, v, g, beta, h0=None, cu_seqlens=None, C=64, P=1, nthreads=None):
    """The three phases end to end: (out, h_final)."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    p = Problem(q, k, v, g, beta, cu_seqlens)
    out = np.zeros((p.T, p.hv, p.V))
    hf = np.zeros((p.N, p.hv, p.K, p.V))
    rc = load().gdn_oracle_segmented(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                     p.T, p.N, p.cu.ctypes.data_as(_i64p), p.hk, p.hv, p.K, p.V,
                                     C, P, _threads(nthreads), _ptr(out), _ptr(hf))
    _check(rc, "segmented")
    return out, hf


def segment_bounds(cu_seqlens, C, P):
    """Chunk ranges [(c0, c1)] of the P segments of each sequence (the split rule: the first
    Nc mod P segments get one extra chunk).  Host-side helper for tests."""
    cu = _cu(cu_seqlens, None) if cu_seqlens is not None else None
    res = []
    for n in range(len(cu) - 1):
        nc = -(-(int(cu[n + 1]) - int(cu[n])) // C)
        base, extra = divmod(nc, P)
        for r in range(P):
            c0 = r * base + min(r, extra)
            res.append((c0, c0 + base + (1 if r < extra else 0)))
    return res
