"""Seeded synthetic inputs for the gated delta rule forward.

This module holds no arithmetic of the method itself: it only draws random tensors with
the shapes and value distributions of the workloads and rounds them to the I/O dtype.  The
same tensors feed the CUDA library and the fp64 oracle, so both see identical bytes.

Recipe (per workload; all draws on the CPU from one ``torch.Generator`` seeded as given):
  * q, k ~ N(0, 1), then L2-normalised over the key dimension per (token, key head), in fp32;
  * v ~ N(0, 1);
  * g (natural-log decay per token and value head):
      - ``"log_uniform"``: g = log(alpha), alpha ~ U(0.90, 1.00);
      - ``"softplus"``:    g = -softplus(N(0, 1)) * 0.1;
      - ``"log_uniform_slow"``: g = log(alpha), alpha ~ U(0.99, 1.00) (tests: slow decay keeps
        a segment's composed transition M_r well inside the fp32 and fp16 ranges);
  * beta = sigmoid(N(0, 1));
  * h0 = 0, or ~ N(0, std^2) per sequence in fp32;
  * packed variable-length streams: lengths ~ U[lmin, lmax] (integers, drawn first),
    each padded up to a multiple of the chunk with g = 0 and q = k = v = 0 (the padding
    no-op of "Add context parallelism to the Gated Delta Net", section "Implementation").
Draw order: lengths (varlen only), q, k, v, g, beta, h0.  q, k, v are rounded to the I/O
dtype after generation; g, beta and h0 stay fp32.

The workloads stand in for the 4096- to 65536-token contexts of the source pages with
the Qwen3-Next GDN geometry (16 key heads shared by 32 value heads, K = V = 128).
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass
class Workload:
    name: str
    T: int                      # total tokens of the packed stream (after padding)
    hk: int
    hv: int
    K: int
    V: int
    dtype: torch.dtype          # I/O dtype of q, k, v, out
    g_kind: str                 # "log_uniform" | "softplus"
    h0_std: float               # 0 -> h0 = 0
    P: int = 1                  # segments per sequence
    chunk: int = 64
    lengths: tuple | None = None  # per-sequence lengths for a packed stream (drawn if None)
    n_seqs: int = 1
    len_range: tuple | None = None
    seed: int = 0


def tiny_fp32(**kw) -> Workload:
    return Workload("tiny fp32 T=256 Hk=Hv=2 K=V=64", 256, 2, 2, 64, 64, torch.float32,
                    "log_uniform", 0.0, **kw)


def prefill_bf16(T=4096, **kw) -> Workload:
    return Workload(f"prefill bf16 T={T} Hk=16 Hv=32 K=V=128", T, 16, 32, 128, 128,
                    torch.bfloat16, "softplus", 0.0, **kw)


def segment_bf16(T=16384, P=8, **kw) -> Workload:
    return Workload(f"segment-composed bf16 T={T} P={P} Hk=16 Hv=32 K=V=128", T, 16, 32, 128,
                    128, torch.bfloat16, "softplus", 0.02, P=P, **kw)


def long_bf16(T=65536, P=16, **kw) -> Workload:
    return Workload(f"long-context bf16 T={T} P={P} Hk=16 Hv=32 K=V=128", T, 16, 32, 128, 128,
                    torch.bfloat16, "softplus", 0.0, P=P, **kw)


def varlen_bf16(n_seqs=8, len_range=(512, 16384), **kw) -> Workload:
    return Workload(f"packed varlen bf16 {n_seqs} seqs lengths U{list(len_range)} "
                    "Hk=16 Hv=32 K=V=128", 0, 16, 32, 128, 128, torch.bfloat16, "softplus",
                    0.02, n_seqs=n_seqs, len_range=len_range, **kw)


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: torch.Tensor | None
    cu_seqlens: torch.Tensor    # int32 [N+1], padded boundaries
    lengths: list               # true (unpadded) length of each sequence
    valid: torch.Tensor         # bool [T]: False at padding positions
    wl: Workload


def _l2norm(x):
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make(wl: Workload) -> Inputs:
    """Draws the inputs of a workload on the CPU (see the module docstring)."""
    gen = torch.Generator().manual_seed(wl.seed)
    C = wl.chunk
    if wl.len_range is not None or wl.lengths is not None:
        if wl.lengths is not None:
            lengths = [int(x) for x in wl.lengths]
        else:
            lo, hi = wl.len_range
            lengths = torch.randint(lo, hi + 1, (wl.n_seqs,), generator=gen).tolist()
        padded = [-(-L // C) * C for L in lengths]
    else:
        lengths = [wl.T]
        padded = [wl.T]
    T = sum(padded)
    cu = [0]
    for L in padded:
        cu.append(cu[-1] + L)
    valid = torch.zeros(T, dtype=torch.bool)
    for n, L in enumerate(lengths):
        valid[cu[n]:cu[n] + L] = True
    q = _l2norm(torch.randn(T, wl.hk, wl.K, generator=gen))
    k = _l2norm(torch.randn(T, wl.hk, wl.K, generator=gen))
    v = torch.randn(T, wl.hv, wl.V, generator=gen)
    if wl.g_kind == "log_uniform":
        g = torch.log(0.90 + 0.10 * torch.rand(T, wl.hv, generator=gen))
    elif wl.g_kind == "log_uniform_slow":
        g = torch.log(0.99 + 0.01 * torch.rand(T, wl.hv, generator=gen))
    elif wl.g_kind == "softplus":
        g = -torch.nn.functional.softplus(torch.randn(T, wl.hv, generator=gen)) * 0.1
    else:
        raise ValueError(wl.g_kind)
    beta = torch.sigmoid(torch.randn(T, wl.hv, generator=gen))
    h0 = None
    if wl.h0_std > 0:
        h0 = torch.randn(len(lengths), wl.hv, wl.K, wl.V, generator=gen) * wl.h0_std
    pad = ~valid
    q[pad] = 0
    k[pad] = 0
    v[pad] = 0
    g[pad] = 0
    return Inputs(q.to(wl.dtype), k.to(wl.dtype), v.to(wl.dtype), g.float().contiguous(),
                  beta.float().contiguous(), h0, torch.tensor(cu, dtype=torch.int32), lengths,
                  valid, wl)


def custom(T, hk, hv, K, V, dtype=torch.float32, g_kind="softplus", h0_std=0.0, seed=0,
           lengths=None, chunk=64) -> Inputs:
    """Inputs of an arbitrary geometry with the same recipe (for tests)."""
    wl = Workload("custom", T, hk, hv, K, V, dtype, g_kind, h0_std, chunk=chunk,
                  lengths=tuple(lengths) if lengths is not None else None,
                  n_seqs=len(lengths) if lengths is not None else 1, seed=seed)
    return make(wl)


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor       # [B, hk, K] io dtype
    k: torch.Tensor       # [B, hk, K]
    v: torch.Tensor       # [B, hv, V]
    g: torch.Tensor       # [B, hv] fp32
    beta: torch.Tensor    # [B, hv] fp32
    slot: torch.Tensor    # int32 [B]; -1 marks a padding row
    state: torch.Tensor   # fp32 [slots, hv, K, V]


def decode_batch(B, slots, hk=16, hv=32, K=128, V=128, dtype=torch.bfloat16, pad_rows=0,
                 state_std=0.12, seed=0) -> DecodeInputs:
    """One decode step's inputs.  Draw order: the rows' slots (distinct, a random subset of
    the pool; the last pad_rows rows are padding with slot -1 and q = k = v = 0), then q, k,
    v, g, beta with the forward recipe (g = -softplus(N(0, 1)) * 0.1), then the pool's states
    ~ N(0, state_std^2) in fp32 (0.12 is the rms of the state a 512-token prefill with this
    recipe leaves)."""
    if B - pad_rows > slots or pad_rows > B:
        raise ValueError("more live rows than slots")
    gen = torch.Generator().manual_seed(seed)
    live = torch.randperm(slots, generator=gen)[:B - pad_rows]
    slot = torch.cat([live, -torch.ones(pad_rows, dtype=torch.long)]).to(torch.int32)
    q = _l2norm(torch.randn(B, hk, K, generator=gen))
    k = _l2norm(torch.randn(B, hk, K, generator=gen))
    v = torch.randn(B, hv, V, generator=gen)
    g = -torch.nn.functional.softplus(torch.randn(B, hv, generator=gen)) * 0.1
    beta = torch.sigmoid(torch.randn(B, hv, generator=gen))
    state = torch.randn(slots, hv, K, V, generator=gen) * state_std
    if pad_rows:
        q[B - pad_rows:] = 0
        k[B - pad_rows:] = 0
        v[B - pad_rows:] = 0
    return DecodeInputs(q.to(dtype), k.to(dtype), v.to(dtype), g.float().contiguous(),
                        beta.float().contiguous(), slot, state.float().contiguous())
