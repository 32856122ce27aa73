"""Partitioning of the gated delta rule forward across GPUs (one process per GPU).

Two ways the computation splits, both from the sources:

* By key-head group ("RFC(qwen35): TP Phase2", section "Partition Contract": local heads,
  rank-local state): the Hk key heads and the Hv/Hk value heads that read each are fully
  independent, so rank r takes key heads [r Hk/W, (r+1) Hk/W) and the value heads grouped with
  them.  No collective touches the data path.

* By sequence ("Add context parallelism to the Gated Delta Net", sections "Why" and
  "Implementation"): rank r holds a contiguous, in-order range of one sequence's chunks (the
  section "Limitation: load balancing must be off" rules out any other order).  Each rank
  summarises its range as P_local segments (phase 1: the affine maps (M_s, U_s) from a zero
  state), one all_gather exchanges the fp32 summaries (W * P_local * Hv * K * (K + V) values:
  independent of the sequence length), every rank runs the exclusive prefix scan over all
  W * P_local segments in order (phase 2) and keeps the incoming states of its own segments,
  and re-emits its range from them (phase 3).  The rank holding the last range ends with the
  sequence's final state.

The arithmetic of each step is passed in (``summary``, ``scan``, ``emit``): on GPUs these are
the library's kernels through its C ABI (``gdn_segment_summary_fused``,
``gdn_state_prefix_scan``, ``gdn_chunk_emit_fused``, see ``gpu_steps``); this module only
partitions, exchanges and orders.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

CHUNK = 64


def head_partition(hk: int, hv: int, world: int, rank: int):
    """Key-head and value-head ranges of `rank` (grouped order: value head j reads key head
    j // (hv / hk), so a block of key heads owns a block of value heads)."""
    if hk % world != 0:
        raise ValueError(f"{hk} key heads do not split over {world} ranks")
    per = hk // world
    grp = hv // hk
    return slice(rank * per, (rank + 1) * per), slice(rank * per * grp, (rank + 1) * per * grp)


def sequence_partition(T: int, world: int, rank: int, chunk: int = CHUNK):
    """Token range [t0, t1) of `rank`: the ceil(T / chunk) chunks in `world` contiguous, in-order
    pieces, the first (Nc mod world) one chunk longer (the library's segment split, applied
    across ranks).  Boundaries fall on chunk boundaries, so every rank's range is a whole number
    of the sequence's chunks (the last one ragged)."""
    nc = -(-T // chunk)
    base, extra = divmod(nc, world)
    c0 = rank * base + min(rank, extra)
    c1 = c0 + base + (1 if rank < extra else 0)
    return min(c0 * chunk, T), min(c1 * chunk, T)


def head_sharded_forward(q, k, v, g, beta, h0, *, world: int, rank: int, forward):
    """This rank's share of a forward split by key-head group: `forward` (q, k, v, g, beta,
    h0) -> (out, h_final) runs on the rank's heads only.  Returns the rank's (out, h_final)
    slices ([T, hv/W, V] and [N, hv/W, K, V]); no collective is needed."""
    ks, vs = head_partition(q.shape[1], v.shape[1], world, rank)
    h0r = None if h0 is None else h0[:, vs].contiguous()
    return forward(q[:, ks].contiguous(), k[:, ks].contiguous(), v[:, vs].contiguous(),
                   g[:, vs].contiguous(), beta[:, vs].contiguous(), h0r)


def sequence_parallel_forward(q, k, v, g, beta, h0, *, summary, scan, emit, P_local: int = 1,
                              group=None):
    """The rank's slice of one sequence's forward, split by sequence across the process group.

    q, k, v, g, beta: this rank's contiguous token range (``sequence_partition``); h0: the
    sequence's initial state [1, hv, K, V] or None (read on every rank).
      summary(k, v, g, beta, P) -> (M [P, hv, K, K], U [P, hv, K, V]): phase 1 over P segments;
      scan(M_all, U_all, h0) -> h_in [S, hv, K, V]: phase 2 over S = W * P segments in order;
      emit(q, k, v, g, beta, h_in [P, hv, K, V], P) -> (out, h_final [1, hv, K, V]): phase 3.
    Returns (out, h_final): the final state of this rank's range (the sequence's on the last
    rank).  The only exchange is one all_gather of the fp32 summaries."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    M, U = summary(k, v, g, beta, P_local)
    payload = torch.cat([M.reshape(-1), U.reshape(-1)]).contiguous()
    gathered = [torch.empty_like(payload) for _ in range(world)]
    dist.all_gather(gathered, payload, group=group)
    nM = M.numel()
    M_all = torch.cat([x[:nM].view_as(M) for x in gathered])
    U_all = torch.cat([x[nM:].view_as(U) for x in gathered])
    h_in = scan(M_all, U_all, h0)
    mine = h_in[rank * P_local:(rank + 1) * P_local].contiguous()
    return emit(q, k, v, g, beta, mine, P_local)


def exchange_bytes(hv: int, K: int, V: int, P_local: int = 1) -> int:
    """fp32 bytes each rank contributes to the all_gather: independent of the sequence length."""
    return 4 * P_local * hv * K * (K + V)


def gpu_steps(gdn):
    """The summary / scan / emit steps of ``sequence_parallel_forward`` on the current GPU,
    through the library's C ABI (``gdn`` is the ``gated_delta_rule_07_gb300.gdn`` binding)."""

    def summary(k, v, g, beta, P):
        q_like = k
        p = gdn.problem_for(q_like, v, None, P=P)
        M = torch.empty(P, p.hv, p.k_dim, p.k_dim, dtype=torch.float32, device=k.device)
        U = torch.empty(P, p.hv, p.k_dim, p.v_dim, dtype=torch.float32, device=k.device)
        gdn.gdn_segment_summary_fused(p, k, v, g, beta, None, M, U, skip_last=False)
        return M, U

    def scan(M_all, U_all, h0):
        S, hv, K, _ = M_all.shape
        V = U_all.shape[-1]
        p = gdn.make_problem(S * CHUNK, 1, 1, hv, K, V, P=S)
        h_in = torch.empty_like(U_all)
        gdn.gdn_state_prefix_scan(p, M_all, U_all, h0, h_in, None)
        return h_in

    def emit(q, k, v, g, beta, h_in, P):
        p = gdn.problem_for(q, v, None, P=P)
        out = torch.empty_like(v)
        hf = torch.empty(1, p.hv, p.k_dim, p.v_dim, dtype=torch.float32, device=q.device)
        gdn.gdn_chunk_emit_fused(p, q, k, v, g, beta, h_in, None, out, hf)
        return out, hf

    return summary, scan, emit
