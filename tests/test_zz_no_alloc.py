"""gdn_forward_static_scratch: the forward pass for callers that cannot allocate device memory
(for example a plug-in whose host framework owns all device memory).  It keeps its scratch in
the library's own device array instead of a caller workspace; its results must equal those of
gdn_forward on the same inputs, on consecutive calls (the array keeps the previous call's
contents).  This file is collected last on purpose."""
import pytest
import torch

from gated_delta_rule_07_gb300 import inputs
from gdn_testutil import BF16_TOL, F32_TOL, check_bf16, max_abs, to_device, to_np


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    return mod


def test_rejects_problems_beyond_the_static_scratch(gdn):
    """64 MiB holds N*P*Hv <= 341 segment-heads of (M, U, h_in) at K = V = 128 (192 KiB each,
    after the 256-byte status word); beyond that the call fails before any device work (no GPU
    needed for this check)."""
    p = gdn.make_problem(65536, 1, 16, 32, 128, 128, P=64)
    assert gdn.gdn_workspace_size(p) > 64 << 20
    fake = 1 << 20
    rc = gdn._lib.gdn_forward_static_scratch(
        gdn.ctypes.byref(p), fake, fake, fake, fake, fake, None, None, fake, None, None)
    assert rc == 3  # GDN_ERR_WORKSPACE


def _both(gdn, inp, P):
    d = to_device(inp)
    cu = d["cu_seqlens"] if len(inp.lengths) > 1 else None
    ref_o, ref_h = gdn.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], cu, P=P,
                               check_status=True)
    p = gdn.problem_for(d["q"], d["v"], cu, P=P)
    out = torch.empty_like(d["v"])
    hf = torch.empty_like(ref_h)
    gdn.gdn_forward_static_scratch(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], cu,
                                   out, hf)
    torch.cuda.synchronize()
    return to_np(out), to_np(hf), to_np(ref_o), to_np(ref_h)


def test_static_scratch_limit_is_the_minimum_workspace(gdn):
    """342 segment-heads (3 x 342 x 64 KiB + the status word) exceed 64 MiB: rejected before any
    device work, whatever the optional factor tiles would add (no GPU needed)."""
    p342 = gdn.make_problem(64 * 400, 1, 1, 1, 128, 128, P=342)
    assert 256 + 3 * 342 * 65536 > 64 << 20 >= 256 + 3 * 341 * 65536
    fake = 1 << 20
    rc = gdn._lib.gdn_forward_static_scratch(
        gdn.ctypes.byref(p342), fake, fake, fake, fake, fake, None, None, fake, None, None)
    assert rc == 3  # GDN_ERR_WORKSPACE


@pytest.mark.gpu
def test_static_scratch_runs_when_only_the_minimum_fits(gdn):
    """A problem whose full workspace (with the factor tiles) exceeds 64 MiB while its minimum
    fits: the static-scratch call runs the kernels that compute their own factors and matches
    gdn_forward with a full workspace."""
    lengths = (64 * 600 + 17,)
    inp = inputs.custom(sum(lengths), 4, 8, 128, 128, torch.bfloat16, h0_std=0.02,
                        lengths=lengths, chunk=1, seed=25)
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], None, P=8)
    assert gdn.gdn_workspace_size(p) > 64 << 20
    o, h, ro, rh = _both(gdn, inp, 8)
    check_bf16(o, h, ro, rh, tol=BF16_TOL, case="static scratch, minimum only")


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_on_consecutive_calls(gdn):
    # bf16 on the tensor-core kernels, two segments per sequence, ragged varlen; then a second
    # call with other inputs and more segments, which reuses the same scratch
    for seed, P, lengths in ((21, 2, (300, 64, 129)), (22, 5, (700,))):
        inp = inputs.custom(sum(lengths), 2, 4, 128, 128, torch.bfloat16, h0_std=0.02,
                            lengths=lengths, chunk=1, seed=seed)
        o, h, ro, rh = _both(gdn, inp, P)
        check_bf16(o, h, ro, rh, tol=BF16_TOL)
    # fp32 on the SIMT kernels (materialised factors live in the scratch too), twice
    for seed in (23, 24):
        inp = inputs.custom(64 * 3 + 7, 1, 2, 64, 64, torch.float32, g_kind="log_uniform",
                            h0_std=0.02, seed=seed)
        o, h, ro, rh = _both(gdn, inp, 2)
        assert max_abs(o, ro) <= F32_TOL and max_abs(h, rh) <= F32_TOL
