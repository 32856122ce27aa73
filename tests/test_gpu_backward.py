"""GPU: the backward (gdn_backward) against the oracle's reverse mode (oracle.token_backward,
fp64, pinned by finite differences in tests/test_oracle_backward.py).

The page "Add context parallelism to the Gated Delta Net" holds the layer's backward to parity
with the single-device result (sections "Tests" and "Measured results": q/k/v/g/beta gradients
within 2.3e-7 to 4.3e-7 relative in f32 on TPU).  Here every gradient is compared element by
element with the fp64 oracle on the same inputs.  Tolerances, as for the forward: fp32 I/O
max |err| <= 2e-3 relative to the gradient's own scale (max(1, rms)); bf16 I/O: dq, dk, dv
(bf16) rms-relative <= 2e-2 and elementwise within bf16 rounding + 2e-2 rms; dg, dbeta, dh0
(fp32) max |err| / rms <= 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_07_gb300 import inputs
from gdn_testutil import check_bf16_out, record, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def cotangents(inp, seed, scale=1.0):
    gen = torch.Generator().manual_seed(seed)
    dout = (torch.randn(inp.v.shape, generator=gen) * scale).to(inp.v.dtype)
    N = inp.cu_seqlens.numel() - 1
    hv, K, V = inp.v.shape[1], inp.k.shape[2], inp.v.shape[2]
    dhf = torch.randn(N, hv, K, V, generator=gen) * 0.1
    return dout, dhf


def run(gdn, inp, dout, dhf, cu=True):
    d = {n: getattr(inp, n).cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    h0 = None if inp.h0 is None else inp.h0.cuda()
    cuq = inp.cu_seqlens.cuda() if cu else None
    r = gdn.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], dout.cuda(), h0, dhf.cuda(),
                     cuq, check_status=True)
    return dict(zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), (to_np(x) for x in r)))


def reference(inp, dout, dhf, cu=True):
    return oracle.token_backward(inp.q, inp.k, inp.v, inp.g, inp.beta, dout, inp.h0, dhf,
                                 inp.cu_seqlens if cu else None)


def check(got, ref, bf16, case):
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        g, r = got[name], ref[name]
        rms = float(np.sqrt(np.mean(r * r)))
        if bf16 and name in ("dq", "dk", "dv"):
            check_bf16_out(g, r, case=f"{case} {name}")
            continue
        err = float(np.max(np.abs(g - r)))
        if bf16:
            e = err / rms
            record(case, f"{name} max|err|/rms", e, 2e-2)
            assert e <= 2e-2, (name, e)
        else:
            e = err / max(1.0, rms)
            record(case, f"{name} max|err|/max(1,rms)", e, 2e-3)
            assert e <= 2e-3, (name, e)


@pytest.mark.parametrize("T,lengths", [(64, None), (64 * 3 + 21, None), (None, (120, 1, 257)),
                                       (None, (64, 128)), (None, (0, 70, 0, 5))])
def test_backward_fp32_small(gdn, T, lengths):
    if lengths is not None:
        T = sum(lengths)
    inp = inputs.custom(T, 2, 4, 64, 64, torch.float32, g_kind="log_uniform", h0_std=0.05,
                        seed=T, lengths=lengths)
    dout, dhf = cotangents(inp, seed=T + 1)
    check(run(gdn, inp, dout, dhf), reference(inp, dout, dhf), False, f"fp32 T={T}")


@pytest.mark.parametrize("K,V", [(128, 128), (128, 64), (64, 128)])
def test_backward_bf16_geometries(gdn, K, V):
    inp = inputs.custom(64 * 2 + 37, 2, 4, K, V, torch.bfloat16, h0_std=0.02, seed=K + V)
    dout, dhf = cotangents(inp, seed=7)
    check(run(gdn, inp, dout, dhf), reference(inp, dout, dhf), True, f"bf16 K={K} V={V}")


def test_backward_prefill_bf16_4096(gdn):
    """The prefill workload (T = 4096, Hk = 16, Hv = 32, K = V = 128), every head."""
    inp = inputs.make(inputs.prefill_bf16())
    dout, dhf = cotangents(inp, seed=11)
    check(run(gdn, inp, dout, dhf, cu=False), reference(inp, dout, dhf, cu=False), True,
          "prefill bf16 T=4096")


def test_backward_empty_sequences_bf16(gdn):
    """Empty sequences among packed ones: their dh0 is dh_final, and they take no chunk."""
    inp = inputs.custom(0, 2, 4, 128, 128, torch.bfloat16, h0_std=0.02, seed=41,
                        lengths=(0, 65, 0, 0, 130))
    dout, dhf = cotangents(inp, seed=42)
    check(run(gdn, inp, dout, dhf), reference(inp, dout, dhf), True, "empty sequences bf16")


def test_backward_varlen_bf16(gdn):
    """Packed sequences with chunk padding (g = 0, q = k = v = 0) and per-sequence h0."""
    inp = inputs.custom(0, 4, 8, 128, 128, torch.bfloat16, h0_std=0.02, seed=19,
                        lengths=(700, 64, 1300, 33))
    dout, dhf = cotangents(inp, seed=20)
    check(run(gdn, inp, dout, dhf), reference(inp, dout, dhf), True, "varlen bf16")


@pytest.mark.slow
def test_backward_long_bf16_65536(gdn):
    """The benchmark's workload, T = 65536 with 32 value heads: every gradient of every head."""
    inp = inputs.make(inputs.long_bf16())
    dout, dhf = cotangents(inp, seed=23)
    check(run(gdn, inp, dout, dhf, cu=False), reference(inp, dout, dhf, cu=False), True,
          "long bf16 T=65536")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_backward_strong_decay_blocks(gdn, dtype):
    """Stretches of strong decay (g = -3 and -8 per token) mixed with the usual recipe: the state
    recurrences carry a scaled state h = A h~ within each staged block and fall back to the plain
    recurrence where the block's summed decay leaves the range of the scale factors; this case
    takes both paths (and decays that underflow to zero within a chunk)."""
    lengths = (300, 150)
    inp = inputs.custom(sum(lengths), 2, 4, 128, 128, dtype, h0_std=0.05, seed=31, lengths=lengths)
    inp.g[40:90] = -3.0      # a block sum of -48: the plain recurrence
    inp.g[200:216, 1] = -8.0  # one value head only
    inp.g[330:345] = -0.5     # sums near the range's edge
    dout, dhf = cotangents(inp, seed=32)
    check(run(gdn, inp, dout, dhf), reference(inp, dout, dhf), dtype == torch.bfloat16,
          f"strong decay {dtype}")


def test_backward_empty_stream_passes_the_state_gradient(gdn):
    q = torch.zeros(0, 2, 64, device="cuda")
    v = torch.zeros(0, 4, 64, device="cuda")
    g = torch.zeros(0, 4, device="cuda")
    dhf = torch.randn(1, 4, 64, 64, device="cuda")
    r = gdn.backward(q, q, v, g, g, torch.zeros_like(v), None, dhf, None, check_status=True)
    assert torch.equal(r[5], dhf)
