"""GPU: the layer prologue (gdn_prologue) against the oracle's (oracle.prologue, fp64, pinned in
tests/test_oracle_prologue.py): the causal depthwise conv over the q | k | v channels with its
carried conv state, the optional SiLU, L2-normalised q and k, and the g, beta maps.

Tolerances: bf16 outputs (q, k, v) the bf16 rule of the forward (rms-relative <= 2e-2 and
elementwise within bf16 rounding + 2e-2 rms); fp32 I/O and the fp32 g, beta max |err| <= 2e-3;
the new conv state is a copy of inputs and must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from gdn_testutil import check_bf16_out, check_f32, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def case(hk, hv, K, V, W, lengths, dtype, seed, state=True):
    """Projection-like inputs: x ~ N(0, 1) over the channels, conv weights ~ N(0, 0.5^2), a, b ~
    N(0, 1), A_log ~ N(log 0.1, 0.3^2), dt_bias ~ N(0, 0.3^2), conv states ~ N(0, 1)."""
    gen = torch.Generator().manual_seed(seed)
    T = sum(lengths)
    Ch = 2 * hk * K + hv * V
    x = torch.randn(T, Ch, generator=gen).to(dtype)
    w = torch.randn(Ch, W, generator=gen) * 0.5
    a = torch.randn(T, hv, generator=gen).to(dtype)
    b = torch.randn(T, hv, generator=gen).to(dtype)
    A_log = np.log(0.1) + torch.randn(hv, generator=gen) * 0.3
    dt = torch.randn(hv, generator=gen) * 0.3
    st = torch.randn(len(lengths), Ch, W - 1, generator=gen).to(dtype) if state and W > 1 else None
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return x, w, a, b, A_log.float(), dt.float(), st, cu


def compare(gdn, args, hk, hv, K, V, act, name):
    x, w, a, b, A_log, dt, st, cu = args
    dev = lambda t: None if t is None else t.cuda().contiguous()
    got = gdn.prologue(dev(x), dev(w), dev(a), dev(b), dev(A_log), dev(dt), hk, hv, K, V,
                       dev(st), dev(cu), act, check_status=True)
    ref = oracle.prologue(x, w, a, b, A_log, dt, hk, hv, K, V, st, cu, act)
    for i, nm in enumerate(("q", "k", "v")):
        if x.dtype == torch.float32:
            check_f32(nm, to_np(got[i]), ref[i], case=name)
        else:
            check_bf16_out(to_np(got[i]), ref[i], case=f"{name} {nm}")
    check_f32("g", to_np(got[3]), ref[3], case=name)
    check_f32("beta", to_np(got[4]), ref[4], case=name)
    W = w.shape[1]
    if W > 1:  # the new state holds inputs (already in the I/O dtype): exact
        assert np.array_equal(to_np(got[5]), ref[5])
    return got


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("W,act", [(4, "none"), (4, "silu"), (2, "none"), (1, "silu")])
def test_prologue_matches_oracle(gdn, dtype, W, act):
    args = case(2, 4, 128, 64, W, (70, 1, 0, 130, 2), dtype, seed=W)
    compare(gdn, args, 2, 4, 128, 64, act, f"{dtype} W={W} {act}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_prologue_uneven_head_widths(gdn, dtype):
    """Head widths that do not fill a power of two of lanes (K = 96, V = 40: a thread's lanes
    are padded out to the next power of two per head, and the padding lanes neither load nor
    store), one key head, three value heads, sequences of 0, 1, 2, 3 and 77 tokens."""
    args = case(1, 3, 96, 40, 4, (3, 0, 77, 1, 2), dtype, seed=5)
    compare(gdn, args, 1, 3, 96, 40, "silu", f"uneven heads {dtype}")


def test_prologue_headline_geometry_bf16(gdn):
    """Hk = 16, Hv = 32, K = V = 128 (8192 channels), 8192 tokens in three sequences."""
    args = case(16, 32, 128, 128, 4, (3000, 64, 5128), torch.bfloat16, seed=9)
    compare(gdn, args, 16, 32, 128, 128, "silu", "headline bf16")


def test_prologue_continues_across_calls(gdn):
    """Two calls, the second from the first's new conv state, equal one call over the whole."""
    x, w, a, b, A_log, dt, st, _ = case(2, 4, 64, 64, 4, (150,), torch.bfloat16, seed=4)
    dev = lambda t: None if t is None else t.cuda().contiguous()
    one = gdn.prologue(dev(x), dev(w), dev(a), dev(b), dev(A_log), dev(dt), 2, 4, 64, 64, dev(st))
    for cut in (1, 2, 65):
        p1 = gdn.prologue(dev(x[:cut]), dev(w), dev(a[:cut]), dev(b[:cut]), dev(A_log), dev(dt),
                          2, 4, 64, 64, dev(st))
        p2 = gdn.prologue(dev(x[cut:]), dev(w), dev(a[cut:]), dev(b[cut:]), dev(A_log), dev(dt),
                          2, 4, 64, 64, p1[5])
        for i in range(5):
            assert torch.equal(torch.cat([p1[i], p2[i]]), one[i]), (cut, i)
        assert torch.equal(p2[5], one[5])
