"""The mbarrier hand-off protocol of the tcgen05 chunk kernel, model-checked on the CPU.

Each role of the kernel (chain, the MMA issuers, prepare, transposer, loader, converter) is
written as the sequence of its waits and arrivals per chunk, in the kernel's order; tcgen05.mma
groups complete in order per issuing thread, and a commit arrives when everything its thread
issued before it has completed; TMA and bulk copies arrive at random later times.  Random
schedules then check the two properties every mbarrier wait of the kernel relies on:

* no deadlock: some role or copy can always make progress until every role has finished;
* no parity aliasing: a wait for completion k never finds the barrier two phases past k (a
  parity wait would then block until the next phase, which may never come).

The model mirrors gated_delta_rule_07_gb300/csrc/gdn_tc5.cu and must be kept in step with it.
A planted bug (phase 3's transposer handing over Q^T without waiting for the previous chunk's
Q K^T) must be found.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.arr, self.ph = count, 0, 0

    def arrive(self, w):
        self.arr += w
        assert self.arr <= self.count, "over-arrival"
        if self.arr == self.count:
            self.arr = 0
            self.ph += 1


def run(roles, counts, seed, max_steps=200000):
    rng = random.Random(seed)
    bars = {b: Bar(c) for b, c in counts.items()}
    gens = {name: g() for name, g in roles.items()}
    cur = {name: None for name in roles}
    done = set()
    queues = {}      # issuer -> list of pending ops (each op: list of bars to arrive at completion)
    pending_async = []  # (bar, w)
    steps = 0
    def fetch(name):
        try:
            cur[name] = next(gens[name])
        except StopIteration:
            cur[name] = None
            done.add(name)
    for n in roles:
        fetch(n)
    while len(done) < len(roles):
        steps += 1
        if steps > max_steps:
            return "too many steps"
        choices = []
        for n in roles:
            if n in done:
                continue
            a = cur[n]
            if a[0] == 'wait':
                b = bars[a[1]]
                k = a[2]
                if b.ph >= k + 2:
                    return f"ALIAS: {n} waits {a[1]} completion {k} but {b.ph} phases done"
                if b.ph == k + 1:
                    choices.append(('role', n))
            else:
                choices.append(('role', n))
        for iss, q in queues.items():
            if q:
                choices.append(('complete', iss))
        for i in range(len(pending_async)):
            choices.append(('async', i))
        if not choices:
            blocked = {n: cur[n] for n in roles if n not in done}
            return f"DEADLOCK: {blocked} phases {{{', '.join(f'{k}:{v.ph}' for k, v in bars.items())}}}"
        # a uniformly random next event: any role may fall far behind the others
        kind, x = rng.choice(choices)
        if kind == 'role':
            a = cur[x]
            if a[0] == 'arrive':
                bars[a[1]].arrive(a[2])
            elif a[0] == 'issue':
                queues.setdefault(a[1], []).append([])
            elif a[0] == 'commit':
                q = queues.setdefault(a[1], [])
                if q:
                    q[-1].append(a[2])
                else:
                    bars[a[2]].arrive(1)
            elif a[0] == 'async_arrive':
                pending_async.append((a[1], a[2]))
            fetch(x)
        elif kind == 'complete':
            op = queues[x].pop(0)
            for b in op:
                bars[b].arrive(1)
        else:
            b, w = pending_async.pop(x)
            bars[b].arrive(w)
    return None


# ----------------------------------------------------------------------------- phase 3 (kEmitR)
def emitR(n, transposer_waits_sq=True):
    """Phase 3 from factor records.  One MMA warp, per chunk c: [D | q h](c); attn_i delta and
    Dh (c); Q K^T (c + 1)."""
    W = lambda b, k: ('wait', b, k)
    A_ = lambda b, w=1: ('arrive', b, w)
    def chain():
        if n > 0:
            yield A_('HR', 256)
        for c in range(n):
            yield W('D', c)
            yield W(f'RL{c & 1}', c >> 1)
            yield A_('DR', 256)
            yield W('H', c)
            if c + 1 < n:
                yield A_('HR', 256)
    def mma():
        def sqr(c):
            yield W('CV', c)
            yield W(f'RL{c & 1}', c >> 1)
            yield ('issue', 'M'); yield ('commit', 'M', 'SQ')
        if n > 0:
            yield from sqr(0)
        for c in range(n):
            yield W('HR', c)
            yield ('issue', 'M'); yield ('commit', 'M', 'D')
            yield W('DR', c)
            yield W('E2', c)
            yield ('issue', 'M'); yield ('commit', 'M', 'H'); yield ('commit', 'M', f'RF{c & 1}')
            if c + 1 < n:
                yield from sqr(c + 1)
    def attn():  # prepare warps 8, 9
        for c in range(n):
            yield W('SQ', c)
            yield W('TB', c)
            yield A_('E2', 64)
    def transposer():  # prepare warps 10, 11
        for c in range(n):
            yield W(f'L{c & 1}', c >> 1)
            if c >= 1 and transposer_waits_sq:
                yield W('SQ', c - 1)
            yield A_('CV', 64)
            yield A_(f'QF{c & 1}', 64)
    def loader():
        for c in range(n):
            sg = c & 1
            if c >= 2:
                yield W(f'QF{sg}', (c >> 1) - 1)
            yield ('async_arrive', f'L{sg}', 33)
            if c >= 2:
                yield W(f'RF{sg}', (c >> 1) - 1)
            yield ('async_arrive', f'RL{sg}', 1)
    def converter():  # tables only
        for c in range(n):
            sg = c & 1
            yield W(f'L{sg}', c >> 1)
            if c >= 1:
                yield W('E2', c - 1)
            yield A_(f'QF{sg}', 64)
            yield A_('TB', 64)
    roles = dict(chain=chain, mma=mma, attn=attn, transposer=transposer, loader=loader,
                 converter=converter)
    counts = dict(HR=256, DR=256, D=1, H=1, RF0=1, RF1=1, SQ=1, E2=64, TB=64, CV=64,
                  QF0=128, QF1=128, L0=33, L1=33, RL0=1, RL1=1)
    return roles, counts


# ----------------------------------------------------------------------------- M summary (kSumML)
def sumML(n):
    """The M half of phase 1 from factor records: a three-stage record ring, D then Dh."""
    W = lambda b, k: ('wait', b, k)
    A_ = lambda b, w=1: ('arrive', b, w)
    def chain():
        if n > 0:
            yield A_('HR', 256)
        for c in range(n):
            yield W('D', c)
            yield A_('DR', 256)
            yield W('H', c)
            if c + 1 < n:
                yield A_('HR', 256)
    def mma():
        for c in range(n):
            st = c % 3
            yield W(f'L{st}', c // 3)
            yield W('HR', c)
            yield ('issue', 'M'); yield ('commit', 'M', 'D')
            yield W('DR', c)
            yield ('issue', 'M'); yield ('commit', 'M', 'H'); yield ('commit', 'M', f'F{st}')
    def loader():
        for c in range(n):
            st = c % 3
            if c >= 3:
                yield W(f'F{st}', c // 3 - 1)
            yield ('async_arrive', f'L{st}', 1)
    roles = dict(chain=chain, mma=mma, loader=loader)
    counts = dict(HR=256, DR=256, D=1, H=1, F0=1, F1=1, F2=1, L0=1, L1=1, L2=1)
    return roles, counts


# ----------------------------------------------------------------------------- U summary (kSumU)
def sumU(n):
    """The U half of phase 1 (preparing its own factors).  One MMA warp, per chunk c:
    w, u (c); D (c); Dh (c); [S ; QK] (c + 2), with [S](0) and [S](1) up front."""
    W = lambda b, k: ('wait', b, k)
    A_ = lambda b, w=1: ('arrive', b, w)
    def chain():
        if n > 0:
            yield A_('HR', 256)
        for c in range(n):
            yield W('D', c)
            yield A_('DR', 256)
            yield W('H', c)
            if c + 1 < n:
                yield A_('HR', 256)
    def mma():
        if n > 0:
            yield W('L0', 0)
            yield ('issue', 'M'); yield ('commit', 'M', 'SQ')
            if n > 1:
                yield W('E2', 0)
                yield W('L1', 0)
                yield ('issue', 'M'); yield ('commit', 'M', 'SQ')
        for c in range(n):
            yield W('T', c)
            yield W('CV', c)
            yield ('issue', 'M'); yield ('commit', 'M', 'WU'); yield ('commit', 'M', f'F{c & 1}')
            yield W('WR', c)
            yield W('HR', c)
            yield ('issue', 'M'); yield ('commit', 'M', 'D')
            yield W('DR', c)
            yield ('issue', 'M'); yield ('commit', 'M', 'H'); yield ('commit', 'M', f'KF{c & 1}')
            if c + 2 < n:
                yield W('E2', c + 1)
                yield W(f'L{c & 1}', (c + 2) >> 1)
                yield ('issue', 'M'); yield ('commit', 'M', 'SQ')
    def prep():  # 128 threads: gram one chunk ahead of the solve and -w
        def gram(c):
            yield W('SQ', c)
            yield W('TB', c)
            yield A_('E2', 128)
        if n > 0:
            yield from gram(0)
        for c in range(n):
            yield A_('T', 128)  # the solve
            if c + 1 < n:
                yield from gram(c + 1)
            yield W('WU', c)  # -w and u^T read out of TMEM
            yield A_('WR', 128)
    def loader():
        for c in range(n):
            sg = c & 1
            if c >= 2:
                yield W(f'F{sg}', (c >> 1) - 1)
            yield ('async_arrive', f'L{sg}', 33)
    def converter():  # tables, then fp16 V and K
        for c in range(n):
            sg = c & 1
            yield W(f'L{sg}', c >> 1)
            if c >= 1:
                yield W('E2', c - 1)
            yield A_('TB', 64)
            if c >= 2:
                yield W(f'KF{sg}', (c >> 1) - 1)
            if c >= 1:
                yield W('WU', c - 1)
            yield A_('CV', 64)
    roles = dict(chain=chain, mma=mma, prep=prep, loader=loader, converter=converter)
    counts = dict(HR=256, DR=256, D=1, H=1, SQ=1, E2=128, TB=64, T=128, CV=64, WU=1, WR=128,
                  F0=1, F1=1, KF0=1, KF1=1, L0=33, L1=33)
    return roles, counts


def _check(mk, trials, **kw):
    for seed in range(trials):
        n = 1 + seed % 12
        roles, counts = mk(n, **kw)
        r = run(roles, counts, seed)
        if r:
            return (seed, n, r)
    return None


@pytest.mark.parametrize("mk", [emitR, sumML, sumU], ids=["phase3_records", "M_summary_records",
                                                          "U_summary"])
def test_protocol_has_no_deadlock_or_aliasing(mk):
    assert _check(mk, 1500) is None


def test_checker_finds_the_planted_aliasing():
    """Without its wait for the previous Q K^T, phase 3's transposer could hand over Q^T two
    chunks ahead of the MMA warp's wait for it."""
    bad = _check(emitR, 1500, transposer_waits_sq=False)
    assert bad is not None and "ALIAS" in bad[2]
