"""Writes tests/golden/oracle_regression.json: the oracle's outputs on one small seeded problem
(two sequences, ragged tails, GQA, a nonzero initial state), so that any later change to the
oracle's arithmetic shows up as a diff of this file.  Calls only the oracle; run from the
repository root:  python tests/golden/make_regression.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def problem():
    rng = np.random.default_rng(2026)
    T, hk, hv, K, V = 70, 1, 2, 4, 4
    lengths = [29, 41]
    q = rng.standard_normal((T, hk, K))
    k = rng.standard_normal((T, hk, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, hv, V))
    g = -0.3 * rng.random((T, hv))
    beta = rng.random((T, hv))
    h0 = 0.5 * rng.standard_normal((len(lengths), hv, K, V))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu_seqlens=cu)


def main():
    p = problem()
    out, hf = oracle.token(**p)
    doc = {"source": "oracle.token (fp64 per-token recurrence) on problem() of this script",
           "generator": "tests/golden/make_regression.py",
           "out": out.tolist(), "h_final": hf.tolist()}
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(doc, f, indent=0)


if __name__ == "__main__":
    main()
