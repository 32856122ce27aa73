"""GPU: the factor-record path of the tcgen05 forward against the path without records, and
the per-phase timing entry point.

With P > 1 and a workspace of gdn_workspace_size() bytes, the U summary stores each chunk's
factors (-w^T, fp16 K, u^T, decay) and the M summary and phase 3 read them; a workspace with
room for everything but the records makes every phase prepare its own factors.  Both must
match the fp64 oracle within the bf16 tolerances (2e-2 relative to RMS) and each other.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_07_gb300 import inputs
from gdn_testutil import BF16_TOL, check_bf16, rel_to_rms, rms_rel, to_device, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def forward_ws(gdn, d, cu, P, ws_bytes):
    p = gdn.problem_for(d["q"], d["v"], cu, P=P)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["v"])
    hf = torch.empty(p.num_seqs, d["v"].shape[1], d["k"].shape[2], d["v"].shape[2],
                     dtype=torch.float32, device="cuda")
    gdn.gdn_forward(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], cu, out, hf, ws)
    assert gdn.gdn_device_status(ws, True) == 0
    torch.cuda.synchronize()
    return to_np(out), to_np(hf)


@pytest.mark.parametrize("T,P,lengths", [(64 * 37 + 5, 3, None), (None, 4, (700, 64, 1, 1300))])
def test_records_and_recomputed_factors_agree(gdn, T, P, lengths):
    if lengths is not None:
        inp = inputs.custom(sum(lengths), 2, 4, 128, 128, torch.bfloat16, h0_std=0.02,
                            lengths=lengths, chunk=1, seed=5)
    else:
        inp = inputs.custom(T, 2, 4, 128, 128, torch.bfloat16, h0_std=0.02, seed=4)
    d = to_device(inp)
    cu = d["cu_seqlens"] if len(inp.lengths) > 1 else None
    p = gdn.problem_for(d["q"], d["v"], cu, P=P)
    full = gdn.gdn_workspace_size(p)
    o_rec, h_rec = forward_ws(gdn, d, cu, P, full)
    # one byte short of the records: the layout without them
    o_cmp, h_cmp = forward_ws(gdn, d, cu, P, full - 1)
    ref_o, ref_h = oracle.token(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, inp.cu_seqlens)
    check_bf16(o_rec, h_rec, ref_o, ref_h)
    check_bf16(o_cmp, h_cmp, ref_o, ref_h)
    assert rel_to_rms(h_rec, h_cmp) <= BF16_TOL and rms_rel(o_rec, o_cmp) <= BF16_TOL


def test_records_size_is_part_of_the_workspace(gdn):
    d = to_device(inputs.custom(64 * 8, 2, 4, 128, 128, torch.bfloat16, seed=2))
    p1 = gdn.problem_for(d["q"], d["v"], None, P=1)
    p4 = gdn.problem_for(d["q"], d["v"], None, P=4)
    # P = 4 adds M, U, h_in (3 x 4 segments x 4 heads x 64 KiB) and the records
    # (49,664 bytes per 64-token window and value head: (8 + 1 + 1) windows x 4 heads)
    extra = gdn.gdn_workspace_size(p4) - gdn.gdn_workspace_size(p1)
    assert extra >= 3 * 4 * 4 * 65536 + 10 * 4 * 49664


def test_forward_timed_matches_forward(gdn):
    inp = inputs.custom(64 * 20 + 9, 2, 4, 128, 128, torch.bfloat16, h0_std=0.02, seed=6)
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], None, P=3)
    ws = gdn.workspace_for(p)
    outs = []
    for timed in (False, True):
        out = torch.empty_like(d["v"])
        hf = torch.empty(1, 4, 128, 128, dtype=torch.float32, device="cuda")
        if timed:
            ms = gdn.gdn_forward_timed(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"],
                                       None, out, hf, ws)
        else:
            gdn.gdn_forward(p, d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], None, out,
                            hf, ws)
        torch.cuda.synchronize()
        outs.append((out.clone(), hf.clone()))
    # the same kernels on the same inputs: identical results
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    summary, scan, emit, first = ms
    assert summary > 0 and scan > 0 and emit > 0 and 0 < first <= summary
    # P = 1: no summary or scan
    p1 = gdn.problem_for(d["q"], d["v"], None, P=1)
    ms1 = gdn.gdn_forward_timed(p1, d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], None,
                                out, hf, gdn.workspace_for(p1))
    assert ms1[2] > 0 and ms1[0] < 0.05 and ms1[1] < 0.05
