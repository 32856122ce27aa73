"""GPU: each phase of the tensor-core path against the oracle's own stage functions.

Phase 1 (segment summaries M_r, U_r), phase 2 (the exclusive prefix scan) and phase 3 (the
re-emit) of the page "Add context parallelism to the Gated Delta Net", section
"Implementation", are run one at a time through the C ABI on bf16 inputs with K = V = 128
(the tensor-core kernels), a ragged packed stream and P = 3.  Each stage is fed the oracle's
exact result of the stage before it, so that its own error is measured alone.

Tolerances:
  * M_r, U_r and final states (fp32 results of bf16 inputs): max |err| / rms <= 2e-2;
  * outputs (bf16): the output reading of the tolerance (rms <= 2e-2 and no element beyond its
    own bf16 rounding plus 2e-2 rms);
  * the scan (fp32 inputs, fp32 arithmetic, a chain of P products of K = 128 terms): max |err| /
    rms <= 1e-4, far above fp32 rounding (~P * K * 2^-24 = 2e-5) and far below any real fault.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_07_gb300 import inputs
from gdn_testutil import BF16_TOL, check_bf16_out, check_state, to_device, to_np

pytestmark = pytest.mark.gpu

P = 3
SCAN_TOL = 1e-4


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


@pytest.fixture(scope="module")
def case():
    # three sequences: a ragged one, one shorter than P chunks (an empty segment), a long one.
    # Slow decay (alpha ~ U(0.99, 1)): with the workloads' decay a segment of a few chunks has
    # M_r ~ e^-20, below the fp16 operands' range, and its relative error means nothing.
    lengths = (64 * 11 + 37, 64 + 5, 64 * 23)
    inp = inputs.custom(sum(lengths), 4, 8, 128, 128, torch.bfloat16, g_kind="log_uniform_slow",
                        h0_std=0.02, lengths=lengths, chunk=1, seed=31)
    rM, rU = oracle.summary(inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, C=64, P=P)
    rh_in, rhf = oracle.scan(rM, rU, inp.h0, N=len(lengths), P=P)
    ro = oracle.emit(inp.q, inp.k, inp.v, inp.g, inp.beta, rh_in, inp.cu_seqlens, C=64, P=P)
    return inp, rM, rU, rh_in, rhf, ro


def test_segment_summaries_match_oracle(gdn, case):
    inp, rM, rU, _, _, _ = case
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], d["cu_seqlens"], P=P)
    S = p.num_seqs * P
    M = torch.full((S, p.hv, 128, 128), float("nan"), device="cuda")
    U = torch.full((S, p.hv, 128, 128), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_segment_summary_fused(p, d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], M, U,
                                  skip_last=False, dev_status=st)
    assert gdn.gdn_device_status(st) == 0
    M, U = to_np(M), to_np(U)
    for s in range(S):
        check_state(f"M[{s}]", M[s], rM[s], case=f"summary seg={s}")
        check_state(f"U[{s}]", U[s], rU[s], case=f"summary seg={s}")


def test_skip_last_leaves_last_segments_unwritten(gdn, case):
    inp, rM, rU, _, _, _ = case
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], d["cu_seqlens"], P=P)
    S = p.num_seqs * P
    M = torch.full((S, p.hv, 128, 128), 7.0, device="cuda")
    U = torch.full((S, p.hv, 128, 128), 7.0, device="cuda")
    gdn.gdn_segment_summary_fused(p, d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], M, U,
                                  skip_last=True)
    M, U = to_np(M), to_np(U)
    for s in range(S):
        if s % P == P - 1:
            assert np.all(M[s] == 7.0) and np.all(U[s] == 7.0)
        else:
            check_state(f"M[{s}]", M[s], rM[s], case=f"summary skip_last seg={s}")
            check_state(f"U[{s}]", U[s], rU[s], case=f"summary skip_last seg={s}")


def test_prefix_scan_matches_oracle(gdn, case):
    inp, rM, rU, rh_in, rhf, _ = case
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], d["cu_seqlens"], P=P)
    M = torch.tensor(rM, dtype=torch.float32, device="cuda")
    U = torch.tensor(rU, dtype=torch.float32, device="cuda")
    h_in = torch.empty_like(U)
    hf = torch.empty(p.num_seqs, p.hv, 128, 128, device="cuda")
    gdn.gdn_state_prefix_scan(p, M, U, d["h0"], h_in, hf)
    torch.cuda.synchronize()
    check_state("h_in", to_np(h_in), rh_in, tol=SCAN_TOL, case="scan")
    check_state("h_final", to_np(hf), rhf, tol=SCAN_TOL, case="scan")


def test_emit_matches_oracle(gdn, case):
    inp, _, _, rh_in, rhf, ro = case
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], d["cu_seqlens"], P=P)
    h_in = torch.tensor(rh_in, dtype=torch.float32, device="cuda")
    out = torch.empty_like(d["v"])
    hf = torch.empty(p.num_seqs, p.hv, 128, 128, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_chunk_emit_fused(p, d["q"], d["k"], d["v"], d["g"], d["beta"], h_in,
                             d["cu_seqlens"], out, hf, dev_status=st)
    assert gdn.gdn_device_status(st) == 0
    check_bf16_out(to_np(out), ro, BF16_TOL, case="emit")
    hf = to_np(hf)
    for n in range(p.num_seqs):
        check_state(f"h_final[{n}]", hf[n], rhf[n], case="emit")


def test_stages_chained_equal_forward(gdn, case):
    """The three stage calls chained on the GPU give the oracle's single-pass result."""
    inp, _, _, _, _, _ = case
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], d["cu_seqlens"], P=P)
    S = p.num_seqs * P
    M = torch.empty(S, p.hv, 128, 128, device="cuda")
    U = torch.empty_like(M)
    gdn.gdn_segment_summary_fused(p, d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], M, U,
                                  skip_last=True)
    h_in = torch.empty_like(M)
    gdn.gdn_state_prefix_scan(p, M, U, d["h0"], h_in, None)
    out = torch.empty_like(d["v"])
    hf = torch.empty(p.num_seqs, p.hv, 128, 128, device="cuda")
    gdn.gdn_chunk_emit_fused(p, d["q"], d["k"], d["v"], d["g"], d["beta"], h_in,
                             d["cu_seqlens"], out, hf)
    torch.cuda.synchronize()
    ref_o, ref_h = oracle.token(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, inp.cu_seqlens)
    check_bf16_out(to_np(out), ref_o, BF16_TOL, case="chained stages")
    hf = to_np(hf)
    for n in range(p.num_seqs):
        check_state(f"h_final[{n}]", hf[n], ref_h[n], case="chained stages")
