"""Shared helpers of the test suite: tolerance metrics and oracle/GPU runners.

Tolerances (written in the tests that use them):
  * fp32 I/O:  max |gpu - oracle| <= 2e-3;
  * bf16 I/O:  max |gpu - oracle| / rms(oracle) <= 2e-2, applied to `out` and to each
    sequence's final state separately.
"""
import numpy as np
import torch

BF16_TOL = 2e-2
F32_TOL = 2e-3


def rel_to_rms(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return err / rms if rms > 0 else err


def max_abs(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref))) if ref.size else 0.0


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def key_group(inp, kh, heads_per_key):
    """Sub-problem of one key head and the value heads that read it (grouped order)."""
    j0 = kh * heads_per_key
    j1 = j0 + heads_per_key
    return dict(q=inp.q[:, kh:kh + 1], k=inp.k[:, kh:kh + 1], v=inp.v[:, j0:j1],
                g=inp.g[:, j0:j1], beta=inp.beta[:, j0:j1],
                h0=None if inp.h0 is None else inp.h0[:, j0:j1])


def to_device(inp, device="cuda"):
    d = {n: getattr(inp, n).to(device).contiguous() for n in ("q", "k", "v", "g", "beta")}
    d["h0"] = None if inp.h0 is None else inp.h0.to(device).contiguous()
    d["cu_seqlens"] = inp.cu_seqlens.to(device)
    return d


def check_bf16(out_gpu, hf_gpu, out_ref, hf_ref, valid=None, tol=BF16_TOL):
    """Returns (out_err, [final-state err per sequence]) and asserts the tolerance."""
    og = np.asarray(out_gpu)
    orf = np.asarray(out_ref)
    if valid is not None:
        og, orf = og[valid], orf[valid]
    e_out = rel_to_rms(og, orf)
    e_h = [rel_to_rms(hf_gpu[n], hf_ref[n]) for n in range(len(hf_ref))]
    assert e_out <= tol, f"out rel-to-rms error {e_out:.3e} > {tol}"
    for n, e in enumerate(e_h):
        assert e <= tol, f"h_final[{n}] rel-to-rms error {e:.3e} > {tol}"
    return e_out, e_h


def gpu_available():
    return torch.cuda.is_available()
