"""GPU: failure detection by bounded device waits.

The layer raises instead of computing a wrong result (page "Add context parallelism to the Gated
Delta Net", section "Limitation").  On the device every wait of the tensor-core kernels is
bounded; this test makes one expire on purpose through gdn_forward_with_limits: a short limit
(1e5 SM cycles, about 50 microseconds) and an injected fault (the chain never signals its first
hand-off, so the wait for it runs out).  The call must report GDN_ERR_DEVICE_TIMEOUT through the
status word, and the context must stay usable: a normal call right after it on the same inputs
matches the oracle within the bf16 tolerance.  Nothing here faults, traps or hangs the GPU: the
expired wait makes every role of the kernel leave its loop, let its own copies and products
land, release its memory and exit.
"""
import pytest
import torch

import oracle
from gated_delta_rule_07_gb300 import inputs
from gdn_testutil import check_bf16, to_device, to_np

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # GDN_ERR_DEVICE_TIMEOUT


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


@pytest.mark.parametrize("P", [1, 3])
def test_expired_wait_is_reported_and_the_context_stays_usable(gdn, P):
    inp = inputs.custom(64 * 5 + 9, 1, 2, 128, 128, torch.bfloat16, h0_std=0.02, seed=41)
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], None, P=P)
    ws = gdn.workspace_for(p)
    out = torch.empty_like(d["v"])
    hf = torch.empty(1, 2, 128, 128, device="cuda")
    gdn.gdn_forward_with_limits(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], None, out,
                                hf, ws, wait_cycles=100000, fault=1)
    assert gdn.gdn_device_status(ws) == TIMEOUT
    # without the fault the same limit is ample, and the default limit works as before
    gdn.gdn_forward_with_limits(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], None, out,
                                hf, ws, wait_cycles=100000000, fault=0)
    assert gdn.gdn_device_status(ws) == 0
    o2, h2 = gdn.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], None, P=P,
                         check_status=True)
    ref_o, ref_h = oracle.token(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0)
    check_bf16(to_np(out), to_np(hf), ref_o, ref_h, case=f"after a timeout, limits P={P}")
    check_bf16(to_np(o2), to_np(h2), ref_o, ref_h, case=f"after a timeout P={P}")


def test_bad_limits_are_rejected_on_the_host(gdn):
    inp = inputs.custom(64, 1, 2, 128, 128, torch.bfloat16, seed=42)
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], None, P=1)
    ws = gdn.workspace_for(p)
    out = torch.empty_like(d["v"])
    for wc, fault in ((-1, 0), (0, 2), (0, -1)):
        with pytest.raises(gdn.GdnError) as ei:
            gdn.gdn_forward_with_limits(p, d["q"], d["k"], d["v"], d["g"], d["beta"], None, None,
                                        out, None, ws, wait_cycles=wc, fault=fault)
        assert ei.value.status == 1
