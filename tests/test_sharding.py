"""Partitioning across ranks (gated_delta_rule_07_gb300.sharding), on CPU with the gloo backend.

Two processes (world size 2) run the host-side partition, the all_gather exchange of the
segment summaries and the scan composition of the page "Add context parallelism to the Gated
Delta Net" (sections "Why", "Implementation"), with the fp64 oracle as each rank's arithmetic
(test infrastructure only: the sharding module takes the step functions as arguments and imports
no oracle).  The concatenated ranks must equal the single-rank oracle: sequence-sharded against
the plain recurrence and the segment form over all ranks' segments, head-sharded against the
full problem's head slices.  The exchanged payload must not depend on the sequence length
(section "Tests": the cross-rank payload is identical at every sequence length).
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from gated_delta_rule_07_gb300 import inputs, sharding

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(T, seed=3):
    return inputs.custom(T, 2, 4, 16, 16, torch.float32, g_kind="log_uniform", h0_std=0.05,
                         seed=seed)


def _oracle_steps():
    def summary(k, v, g, beta, P):
        M, U = oracle.summary(k, v, g, beta, None, C=64, P=P, nthreads=1)
        return torch.from_numpy(M), torch.from_numpy(U)

    def scan(M_all, U_all, h0):
        h_in, _ = oracle.scan(M_all.numpy(), U_all.numpy(), None if h0 is None else h0.numpy(),
                              N=1, P=M_all.shape[0])
        return torch.from_numpy(h_in)

    def emit(q, k, v, g, beta, h_in, P):
        out = oracle.emit(q, k, v, g, beta, h_in.numpy(), None, C=64, P=P, nthreads=1)
        _, hf = oracle.token(q, k, v, g, beta, h_in[0:1].numpy(), nthreads=1)
        return torch.from_numpy(out), torch.from_numpy(hf)

    return summary, scan, emit


def _worker(rank, port, T, P_local, outdir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        inp = _case(T)
        t0, t1 = sharding.sequence_partition(T, WORLD, rank)
        sl = {n: getattr(inp, n)[t0:t1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        summary, scan, emit = _oracle_steps()
        gathered_sizes = []
        orig_all_gather = dist.all_gather

        def counting_all_gather(lst, t, group=None):
            gathered_sizes.append(t.numel() * t.element_size())
            return orig_all_gather(lst, t, group=group)

        dist.all_gather = counting_all_gather
        out, hf = sharding.sequence_parallel_forward(
            sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], inp.h0.double(), summary=summary,
            scan=scan, emit=emit, P_local=P_local)
        dist.all_gather = orig_all_gather
        # head-sharded: each rank its key-head group, no collective
        ho, hh = sharding.head_sharded_forward(
            inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, world=WORLD, rank=rank,
            forward=lambda q, k, v, g, b, h0: tuple(
                torch.from_numpy(x) for x in oracle.token(q, k, v, g, b, h0, nthreads=1)))
        np.savez(os.path.join(outdir, f"rank{rank}.npz"), out=out.numpy(), hf=hf.numpy(),
                 t0=t0, t1=t1, sizes=np.array(gathered_sizes), ho=ho.numpy(), hh=hh.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("T,P_local", [(64 * 7 + 23, 2), (64 * 4, 1)])
def test_two_ranks_equal_single_rank_oracle(T, P_local):
    port = _free_port()
    with tempfile.TemporaryDirectory() as outdir:
        mp.start_processes(_worker, args=(port, T, P_local, outdir), nprocs=WORLD, join=True,
                           start_method="spawn")
        res = [np.load(os.path.join(outdir, f"rank{r}.npz")) for r in range(WORLD)]
    inp = _case(T)
    ref_o, ref_h = oracle.token(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0)
    # the ranks cover the sequence contiguously and in order
    assert res[0]["t0"] == 0 and res[-1]["t1"] == T
    assert all(res[r]["t1"] == res[r + 1]["t0"] for r in range(WORLD - 1))
    out = np.concatenate([r["out"] for r in res])
    assert np.max(np.abs(out - ref_o)) < 1e-10
    assert np.max(np.abs(res[-1]["hf"] - ref_h)) < 1e-10
    # the same as the segment form over all ranks' segments (W * P_local in order)
    seg_o, seg_h = oracle.segmented(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, C=64,
                                    P=WORLD * P_local)
    assert np.max(np.abs(out - seg_o)) < 1e-10
    # one all_gather per rank, of P_local * hv * K * (K + V) values (fp64 here)
    hv, K, V = inp.v.shape[1], inp.k.shape[2], inp.v.shape[2]
    for r in res:
        assert list(r["sizes"]) == [2 * sharding.exchange_bytes(hv, K, V, P_local)]
    # head-sharded ranks reassemble the full outputs and states
    ho = np.concatenate([r["ho"] for r in res], axis=1)
    hh = np.concatenate([r["hh"] for r in res], axis=1)
    assert np.max(np.abs(ho - ref_o)) < 1e-12 and np.max(np.abs(hh - ref_h)) < 1e-12


def test_partitions_cover_and_do_not_depend_on_length():
    for T in (1, 63, 64, 65, 64 * 9 + 5, 65536):
        for W in (1, 2, 3, 4, 8):
            rngs = [sharding.sequence_partition(T, W, r) for r in range(W)]
            assert rngs[0][0] == 0 and rngs[-1][1] == T
            assert all(rngs[r][1] == rngs[r + 1][0] for r in range(W - 1))
            # every non-empty range starts on a chunk boundary (empty ones sit at T)
            assert all(a % 64 == 0 or a == b == T for a, b in rngs)
    # the exchange does not grow with the sequence (fp32, Hv = 32, K = V = 128, 1 segment/rank)
    assert sharding.exchange_bytes(32, 128, 128) == 4 * 32 * 128 * 256
    ks, vs = sharding.head_partition(16, 32, 4, 3)
    assert (ks.start, ks.stop, vs.start, vs.stop) == (12, 16, 24, 32)
    with pytest.raises(ValueError):
        sharding.head_partition(16, 32, 3, 0)
