"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Tolerances (see gdn_testutil): fp32 I/O max |gpu - oracle| <= 2e-3; bf16 I/O: final states
max |gpu - oracle| / rms(oracle) <= 2e-2 per sequence, outputs rms-relative error <= 2e-2 and
no element off by more than its own bf16 rounding plus 2e-2 rms.  Both kernel families (SIMT
and tensor-core) are checked where they apply.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_07_gb300 import inputs
from gdn_testutil import (BF16_TOL, F32_TOL, check_bf16, check_bf16_out, check_f32,
                          check_state, key_group, max_abs, rel_to_rms, rms_rel, to_device,
                          to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def run_gpu(gdn, inp, P=1, check_status=True):
    d = to_device(inp)
    cu = d["cu_seqlens"] if len(inp.lengths) > 1 else None
    out, hf = gdn.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], cu, P=P,
                          check_status=check_status)
    torch.cuda.synchronize()
    return to_np(out), to_np(hf)


def run_oracle(inp, C=64, P=1):
    return oracle.token(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, inp.cu_seqlens)


# ------------------------------------------------------------------ tiny fp32 (SIMT)

def test_tiny_fp32_matches_oracle(gdn):
    inp = inputs.make(inputs.tiny_fp32())
    ref_o, ref_h = run_oracle(inp)
    for P in (1, 2, 3):
        o, h = run_gpu(gdn, inp, P=P)
        check_f32("out", o, ref_o, case=f"tiny fp32 P={P}")
        check_f32("h_final", h, ref_h, case=f"tiny fp32 P={P}")


# ------------------------------------------------------------------ small bf16, both paths

@pytest.mark.parametrize("T,P,lengths", [
    (64, 1, None), (64 * 5 + 17, 1, None), (64 * 5 + 17, 2, None), (64 * 7, 3, None),
    (64 * 3, 5, None), (None, 2, (100, 1, 0, 64, 257))])
def test_small_bf16_matches_oracle(gdn, T, P, lengths):
    if lengths is not None:
        inp = inputs.custom(sum(lengths), 2, 4, 128, 128, torch.bfloat16, h0_std=0.02,
                            lengths=lengths, chunk=1, seed=3)
    else:
        inp = inputs.custom(T, 2, 4, 128, 128, torch.bfloat16, h0_std=0.02, seed=1)
    ref_o, ref_h = run_oracle(inp)
    o, h = run_gpu(gdn, inp, P=P)
    check_bf16(o, h, ref_o, ref_h, case=f"T={inp.q.shape[0]} P={P}")


@pytest.mark.parametrize("KV", [(64, 64), (64, 128), (128, 64)])
def test_other_head_dims_simt(gdn, KV):
    K, V = KV
    inp = inputs.custom(64 * 3 + 5, 1, 2, K, V, torch.float32, g_kind="log_uniform",
                        h0_std=0.02, seed=4)
    ref_o, ref_h = run_oracle(inp)
    o, h = run_gpu(gdn, inp, P=2)
    assert max_abs(o, ref_o) <= F32_TOL and max_abs(h, ref_h) <= F32_TOL


# ------------------------------------------------------------------ stage entry points

@pytest.mark.parametrize("dtype,KV", [(torch.float32, 64), (torch.bfloat16, 128)],
                         ids=["fp32-K64", "bf16-K128"])
def test_stage_entry_points_match_oracle_stages(gdn, dtype, KV):
    """The materialising stage calls (prepare -> summary -> scan -> emit, fp32 factors in HBM)
    against the oracle's stages, for fp32 I/O and for the headline geometry's bf16 I/O with
    K = V = 128 (the same inputs, rounded to bf16, feed both sides)."""
    inp = inputs.custom(64 * 4 + 9, 1, 2, KV, KV, dtype, g_kind="log_uniform",
                        h0_std=0.05, seed=5, lengths=(120, 153))
    P = 2
    d = to_device(inp)
    p = gdn.problem_for(d["q"], d["v"], d["cu_seqlens"], P=P)
    T, hv = inp.v.shape[0], inp.v.shape[1]
    dev = "cuda"
    w = torch.empty(T, hv, KV, device=dev)  # fp32
    u = torch.empty(T, hv, KV, device=dev)
    gcum = torch.empty(T, hv, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gdn.gdn_chunk_prepare(p, d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], w, u, gcum, st)
    rw, ru, rg = oracle.prepare(inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, C=64)
    torch.cuda.synchronize()
    assert max_abs(to_np(w), rw) < 1e-4 and max_abs(to_np(u), ru) < 1e-4
    assert max_abs(to_np(gcum), rg) < 1e-5
    S = 2 * P
    M = torch.empty(S, hv, KV, KV, device=dev)
    U = torch.empty(S, hv, KV, KV, device=dev)
    gdn.gdn_segment_summary(p, d["k"], w, u, gcum, d["cu_seqlens"], M, U, st)
    rM, rU = oracle.summary(inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens, C=64, P=P)
    torch.cuda.synchronize()
    assert max_abs(to_np(M), rM) < 1e-4 and max_abs(to_np(U), rU) < 1e-4
    h_in = torch.empty(S, hv, KV, KV, device=dev)
    hf = torch.empty(2, hv, KV, KV, device=dev)
    gdn.gdn_state_prefix_scan(p, M, U, d["h0"], h_in, hf)
    rh_in, rhf = oracle.scan(rM, rU, inp.h0, N=2, P=P)
    torch.cuda.synchronize()
    assert max_abs(to_np(h_in), rh_in) < 1e-4 and max_abs(to_np(hf), rhf) < 1e-4
    out = torch.empty_like(d["v"])
    hf2 = torch.empty_like(hf)
    gdn.gdn_chunk_emit(p, d["q"], d["k"], w, u, gcum, h_in, d["cu_seqlens"], out, hf2, st)
    ro = oracle.emit(inp.q, inp.k, inp.v, inp.g, inp.beta, rh_in, inp.cu_seqlens, C=64, P=P)
    torch.cuda.synchronize()
    if dtype == torch.float32:
        check_f32("out", to_np(out), ro, case="stage calls fp32 K=64")
        check_f32("h_final", to_np(hf2), rhf, case="stage calls fp32 K=64")
    else:
        check_bf16(to_np(out), to_np(hf2), ro, rhf, case="stage calls bf16 K=128")
    assert gdn.gdn_device_status(st) == 0


# ------------------------------------------------------------------ workload configs

def test_prefill_bf16_4096(gdn):
    inp = inputs.make(inputs.prefill_bf16())
    ref_o, ref_h = run_oracle(inp)
    o, h = run_gpu(gdn, inp, P=1)
    check_bf16(o, h, ref_o, ref_h, case="prefill P=1")


def test_segment_bf16_16384_P8_equals_P1(gdn):
    inp = inputs.make(inputs.segment_bf16())
    ref_o, ref_h = run_oracle(inp)
    o8, h8 = run_gpu(gdn, inp, P=8)
    o1, h1 = run_gpu(gdn, inp, P=1)
    check_bf16(o8, h8, ref_o, ref_h, case="segment P=8")
    check_bf16(o1, h1, ref_o, ref_h, case="segment P=1")
    # the segment count changes only rounding: P=8 against P=1 on the GPU
    assert rel_to_rms(h8, h1) <= BF16_TOL and rms_rel(o8, o1) <= BF16_TOL


def oracle_by_key_group(inp):
    """The oracle's outputs and final states for every key-head group (grouped GQA order)."""
    grp = inp.v.shape[1] // inp.q.shape[1]
    return [oracle.token(**key_group(inp, kh, grp), cu_seqlens=inp.cu_seqlens)
            for kh in range(inp.q.shape[1])]


def check_all_groups(o, h, refs, case, valid=None):
    grp = o.shape[1] // len(refs)
    for kh, (ref_o, ref_h) in enumerate(refs):
        sl = slice(grp * kh, grp * kh + grp)
        check_bf16(o[:, sl], h[:, sl], ref_o, ref_h, valid=valid, case=f"{case} kh={kh}")


def test_varlen_bf16(gdn):
    """8 packed sequences: every key-head group and every sequence's final state against the
    oracle, for P = 1, 4 and 16 segments per sequence."""
    inp = inputs.make(inputs.varlen_bf16())
    valid = inp.valid.numpy()
    refs = oracle_by_key_group(inp)
    for P in (1, 4, 16):
        o, h = run_gpu(gdn, inp, P=P)
        # padded positions read zeros exactly (q = 0 there)
        assert np.all(o[~valid] == 0.0)
        check_all_groups(o, h, refs, f"varlen P={P}", valid=valid)


@pytest.mark.slow
def test_long_bf16_65536_all_heads(gdn):
    """The benchmark's workload (T = 65536, 32 value heads) at P = 1, 4, 16 and 64: every
    key-head group's outputs and final states against the oracle."""
    inp = inputs.make(inputs.long_bf16())
    refs = oracle_by_key_group(inp)
    for P in (1, 4, 16, 64):
        o, h = run_gpu(gdn, inp, P=P)
        check_all_groups(o, h, refs, f"T=65536 P={P}")


# ------------------------------------------------------------------ edge cases

def test_empty_stream_returns_h0(gdn):
    h0 = torch.randn(1, 4, 128, 128, device="cuda")
    q = torch.zeros(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(0, 4, 128, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(0, 4, device="cuda")
    out, hf = gdn.forward(q, q, v, g, g, h0, None, P=3, check_status=True)
    assert out.numel() == 0 and torch.equal(hf, h0)


def test_bad_cu_seqlens_is_reported_not_faulted(gdn):
    inp = inputs.custom(256, 2, 4, 128, 128, torch.bfloat16, lengths=(128, 128), seed=6)
    d = to_device(inp)
    bad = torch.tensor([0, 300, 256], dtype=torch.int32, device="cuda")
    with pytest.raises(gdn.GdnError) as ei:
        gdn.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], None, bad, P=2,
                    check_status=True)
    assert ei.value.status == 6


def test_split_call_resume(gdn):
    inp = inputs.custom(64 * 6 + 11, 2, 4, 128, 128, torch.bfloat16, h0_std=0.02, seed=7)
    d = to_device(inp)
    T1 = 64 * 2 + 30
    o_full, h_full = gdn.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], None, P=2)
    sl = lambda x, a, b: x[a:b].contiguous()
    oa, ha = gdn.forward(*(sl(d[n], 0, T1) for n in ("q", "k", "v", "g", "beta")), d["h0"], None)
    ob, hb = gdn.forward(*(sl(d[n], T1, None) for n in ("q", "k", "v", "g", "beta")), ha, None)
    o2 = torch.cat([oa, ob])
    assert rms_rel(to_np(o2), to_np(o_full)) <= BF16_TOL
    assert rel_to_rms(to_np(hb), to_np(h_full)) <= BF16_TOL


def test_negative_control_tiled_gqa_fails(gdn):
    """Feeding the key heads in tiled order must break parity (the check has teeth)."""
    inp = inputs.custom(192, 2, 4, 128, 128, torch.bfloat16, seed=8)
    ref_o, _ = run_oracle(inp)
    d = to_device(inp)
    k_tiled = d["k"][:, [1, 0]].contiguous()
    q_tiled = d["q"][:, [1, 0]].contiguous()
    out, _ = gdn.forward(q_tiled, k_tiled, d["v"], d["g"], d["beta"], None, None)
    assert rms_rel(to_np(out), ref_o) > BF16_TOL


def test_fp16_range_overflow_is_reported(gdn):
    """The tensor-core kernels keep fp16 operands: a value past 65504 is reported, not
    silently wrong; the same values through fp32 I/O (the CUDA-core kernels, no such limit)
    match the oracle."""
    inp = inputs.custom(128, 2, 4, 128, 128, torch.bfloat16, seed=9)
    d = to_device(inp)
    v = d["v"].clone()
    v[5, 1, 7] = 1.0e6
    with pytest.raises(gdn.GdnError) as ei:
        gdn.forward(d["q"], d["k"], v, d["g"], d["beta"], None, None, P=1, check_status=True)
    assert ei.value.status == 7
    f32 = {n: d[n].float() for n in ("q", "k")}
    out, hf = gdn.forward(f32["q"], f32["k"], v.float(), d["g"], d["beta"], None, None, P=1,
                          check_status=True)
    ref_o, ref_h = oracle.token(inp.q, inp.k, v.cpu(), inp.g, inp.beta)
    check_f32("out", to_np(out), ref_o, tol=2e-3 * 1e6, case="fp32 I/O past the fp16 range")
    check_state("h_final", to_np(hf), ref_h, case="fp32 I/O past the fp16 range")
