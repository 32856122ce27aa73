"""The oracle against the stored fixtures of tests/golden/.

* hand_worked_2x2.json: three tokens worked by hand from the recurrence (the pages print no
  worked example of their own); every form of the oracle (per token, chunked, segmented) must
  reproduce it to rounding.
  The decode step, fed the same three tokens one at a time from a slot of a state pool,
  must reproduce it too.
* oracle_regression.json: written by tests/golden/make_regression.py (which calls only the
  oracle); a later change to the oracle's arithmetic must show up here and be justified.
"""
import json
import os

import numpy as np

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_hand_worked_fixture():
    with open(os.path.join(HERE, "hand_worked_2x2.json")) as f:
        d = json.load(f)
    q, k, v = (np.array(d[n], float)[:, None] for n in ("q", "k", "v"))
    g = np.log(np.array(d["alpha"]))[:, None]
    beta = np.array(d["beta"])[:, None]
    for fn in (oracle.token, lambda *a: oracle.chunked(*a, C=2),
               lambda *a: oracle.segmented(*a, C=1, P=3)):
        o, hf = fn(q, k, v, g, beta)
        assert np.max(np.abs(o[:, 0] - np.array(d["out"]))) < 1e-14
        assert np.max(np.abs(hf[0, 0] - np.array(d["h_final"]))) < 1e-14


def test_hand_worked_fixture_through_decode_steps():
    with open(os.path.join(HERE, "hand_worked_2x2.json")) as f:
        d = json.load(f)
    q, k, v = (np.array(d[n], float) for n in ("q", "k", "v"))
    g = np.log(np.array(d["alpha"]))
    beta = np.array(d["beta"])
    state = np.zeros((2, 1, 2, 2))
    state[0, 0] = [[7.0, -1.0], [3.0, 5.0]]  # another request's slot: never touched
    for t in range(3):
        o, state = oracle.decode(q[t][None, None], k[t][None, None], v[t][None, None],
                                 g[t][None, None], beta[t][None, None], state, [1])
        assert np.max(np.abs(o[0, 0] - np.array(d["out"][t]))) < 1e-14
    assert np.max(np.abs(state[1, 0] - np.array(d["h_final"]))) < 1e-14
    assert np.array_equal(state[0, 0], [[7.0, -1.0], [3.0, 5.0]])


def test_regression_fixture():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_regression",
                                                  os.path.join(HERE, "make_regression.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(HERE, "oracle_regression.json")) as f:
        d = json.load(f)
    o, hf = oracle.token(**mod.problem())
    assert np.max(np.abs(o - np.array(d["out"]))) < 1e-12
    assert np.max(np.abs(hf - np.array(d["h_final"]))) < 1e-12
