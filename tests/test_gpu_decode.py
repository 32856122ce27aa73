"""GPU: the decode step (gdn_decode_step) against the oracle's decode.

Page "RFC(qwen35): TP Phase2": decode kernels run against the head and state shapes and update
only request-local recurrent state ("Execution Contract"); the state is [Hv, K, V] f32 per
request ("Partition Contract"); requests live in reusable slots, and no slot exposes another
request's state ("Request-State Lifecycle").  Every row is compared with ``oracle.decode`` (the
fp64 token recurrence, one token per request, from the slot's state), and every slot of the pool
is checked: the ones no row names must come back bit-identical.

Tolerances: fp32 I/O max |err| <= 2e-3; bf16 I/O the forward's bf16 rule (out: rms-relative
<= 2e-2 and elementwise within bf16 rounding + 2e-2 rms; states: max |err| / rms <= 2e-2 per
slot).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_07_gb300 import inputs
from gdn_testutil import check_bf16, check_f32, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def run_decode(gdn, d, expect_status=0):
    q, k, v, g, beta = (getattr(d, n).cuda().contiguous() for n in ("q", "k", "v", "g", "beta"))
    slot = d.slot.cuda()
    state = d.state.cuda().clone()
    out = torch.full_like(v, 7.0)  # a sentinel: rows the step skips keep it
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_decode_step(gdn.decode_problem_for(q, v, state), q, k, v, g, beta, slot, state, out,
                        st)
    assert gdn.gdn_device_status(st) == expect_status
    return to_np(out), to_np(state)


def check(d, out, state, ref_out, ref_state, case):
    if d.q.dtype == torch.float32:
        check_f32("out", out, ref_out, case=case)
        check_f32("state", state, ref_state, case=case)
    else:
        check_bf16(out, state, ref_out, ref_state, case=case)
    named = set(d.slot[d.slot >= 0].tolist())
    for s in range(d.state.shape[0]):
        if s not in named:
            assert np.array_equal(state[s], d.state[s].numpy()), f"slot {s} was touched"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64), (64, 128)])
def test_decode_matches_oracle(gdn, dtype, K, V):
    d = inputs.decode_batch(37, 48, hk=2, hv=4, K=K, V=V, dtype=dtype, pad_rows=5, seed=K + V)
    out, state = run_decode(gdn, d)
    ref_out, ref_state = oracle.decode(d.q, d.k, d.v, d.g, d.beta, d.state, d.slot.numpy())
    check(d, out, state, ref_out, ref_state, f"{dtype} K={K} V={V}")
    assert np.all(out[-5:] == 0)  # padding rows


def test_decode_full_size_bf16(gdn):
    """The decode workload of the benchmark: 256 requests, a pool of 256 slots, Hk = 16,
    Hv = 32, K = V = 128 (every row and every slot against the oracle)."""
    d = inputs.decode_batch(256, 256, seed=3)
    out, state = run_decode(gdn, d)
    ref_out, ref_state = oracle.decode(d.q, d.k, d.v, d.g, d.beta, d.state, d.slot.numpy())
    check(d, out, state, ref_out, ref_state, "B=256 S=256")


def test_decode_continues_a_prefill(gdn):
    """A request prefilled by gdn_forward straight into its slot (h_final pointed at the slot),
    then decoded token by token in a batch with other requests, equals the recurrence over the
    whole sequence; the other slots keep their states."""
    T0, n_dec, hk, hv = 200, 24, 2, 4
    seq = inputs.custom(T0 + n_dec, hk, hv, 128, 128, torch.bfloat16, h0_std=0.02, seed=12)
    pool = inputs.decode_batch(6, 8, hk=hk, hv=hv, seed=13)  # other requests' rows and states
    state = pool.state.cuda().clone()
    home = 5
    assert home not in pool.slot.tolist()
    pre = {n: getattr(seq, n)[:T0].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")}
    gdn.forward(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], seq.h0.cuda(), None, P=1,
                h_final=state[home:home + 1], check_status=True)
    outs = []
    for t in range(T0, T0 + n_dec):
        rows = {n: torch.cat([getattr(seq, n)[t:t + 1], getattr(pool, n)])
                for n in ("q", "k", "v", "g", "beta")}
        slot = torch.cat([torch.tensor([home], dtype=torch.int32), pool.slot]).cuda()
        rows = {n: x.cuda().contiguous() for n, x in rows.items()}
        o = gdn.decode(rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], slot, state,
                       check_status=True)
        outs.append(to_np(o[0]))
    ref_o, ref_h = oracle.token(seq.q, seq.k, seq.v, seq.g, seq.beta, seq.h0)
    check_bf16(np.stack(outs), to_np(state[home:home + 1]), ref_o[T0:], ref_h,
               case="prefill 200 + 24 decode steps")


def test_bad_slots_are_reported_and_their_rows_skipped(gdn):
    """Two rows naming one slot, and a row naming a slot past the pool: those rows leave their
    state and output untouched and GDN_ERR_DEVICE_INPUT is recorded; the other rows run."""
    d = inputs.decode_batch(12, 16, hk=2, hv=4, seed=21)
    slot = d.slot.clone()
    slot[5] = slot[2]   # shared
    slot[7] = 16        # past the pool
    d.slot = slot
    out, state = run_decode(gdn, d, expect_status=6)
    good = [b for b in range(12) if b not in (2, 5, 7)]
    ref_out, ref_state = oracle.decode(d.q[good], d.k[good], d.v[good], d.g[good], d.beta[good],
                                       d.state, slot[good].numpy())
    check_bf16(out[good], state, ref_out, ref_state, case="bad slots, good rows")
    for b in (2, 5, 7):
        assert np.all(out[b] == 7.0), f"row {b} was written"
    assert np.array_equal(state[int(slot[2])], d.state[int(slot[2])].numpy())


def test_empty_batch_is_a_no_op(gdn):
    d = inputs.decode_batch(0, 4, hk=2, hv=4, seed=1)
    state = d.state.cuda().clone()
    p = gdn.make_decode_problem(0, 4, 2, 4, 128, 128)
    gdn.gdn_decode_step(p, None, None, None, None, None, None, state, None)
    assert torch.equal(state.cpu(), d.state)
