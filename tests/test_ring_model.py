"""A CPU model of the prefill GEMM's A-tile ring protocol, checked over random
interleavings.  It shows why Q6_K needs at least three A stages (the host uses
four), while Q4_K may use any depth of two or more.

The model:
- The dequant writers put K step t into A slot t % SA. Before that they wait on
  done[t % SA] for the completion of step t - SA, with an mbarrier parity wait.
- The two UMMA issuers take alternate steps. Each waits for its step's A tile,
  then completes one phase of done[t % SA] (its commit).
- A packed-block producer refills one stage as soon as every writer has read
  the block.

An mbarrier parity wait for phase k passes while the barrier's current phase
index c has the other parity.  It is fooled when it passes with c <= k - 1,
i.e. before the awaited phase completed.  A writer that passes early would
overwrite an A tile the tensor core has not consumed yet.

Q4_K: every writer writes every K step, in order.
Q6_K: the two halves of a row write steps 4i, 4i+1 and 4i+2, 4i+3 of
super-block i respectively.

With SA = 2, each Q6_K half uses both slots.  Before writing step 4i+4 into
slot 0, half 0 waits for step 4i+2 (issuer 0).  Half 0 never waited for step
4i, the phase in between, so that phase may still be pending, and the parity
test then passes early.  With SA >= 3 the phase a half did not wait for always
belongs to an earlier step of the same issuer as the phase it does wait for.
That issuer's UMMAs complete in order, so the phase has completed before the
awaited one.

A second model checks Q4_K with an x ring and an A ring of different depths.
The two rings share one done ring of max(SX, SA) barriers, indexed by K step.
It covers gate/up, where both issuers take every step and a phase needs both
commits, and single-tensor problems, where the issuers alternate.  A third
adds the issuers' own parity waits on the x and A slots, x tiles that land
in any order, and the Q6_K halves on the done ring: it shows why a
single-tensor x ring is even.

A last model checks the GEMV's ring: a producer warp that refills a stage
after the compute warps release it and first adds their per-tile partial
sums, and compute warps that read stages and leave partials in them.  A
control drops the producer's wait and shows that the model then catches the
overwrite.
"""
import random

import pytest


def simulate(sa, q6k, blocks=6, seed=0, pstages=1):
    rng = random.Random(seed)
    steps = 4 * blocks
    done_c = [0] * sa  # completed phases of done[slot]
    a_ready = [False] * steps
    issued = [False] * steps
    # writers: (list of steps in order); Q6_K: part p writes 4i+2p, 4i+2p+1
    if q6k:
        writers = [[4 * i + 2 * p + j for i in range(blocks) for j in range(2)] for p in range(2)]
    else:
        writers = [list(range(steps))]
    pos = [0] * len(writers)  # next step index in each writer's list
    have_block = [0] * len(writers)  # blocks loaded into registers by each writer
    loaded = 0  # blocks whose packed copy has landed (producer)
    fooled = False

    def block_of(t):
        return t // 4

    while True:
        actions = []
        # packed producer: block b may land when all writers have read block b - pstages
        if loaded < blocks and all(h >= loaded - pstages + 1 for h in have_block):
            actions.append(("load", None))
        for w, lst in enumerate(writers):
            if pos[w] >= len(lst):
                continue
            t = lst[pos[w]]
            b = block_of(t)
            if have_block[w] <= b:  # needs this block in registers
                if loaded > b:
                    actions.append(("read", w))
                continue
            # wait on done[t % sa] for the completion of step t - sa (phase k of that slot)
            if t < sa:
                actions.append(("write", w))
                continue
            k = (t - sa) // sa
            c = done_c[t % sa]
            if (c & 1) != (k & 1):  # the parity test passes
                actions.append(("write", w))
        for e in range(2):  # issuer e takes steps e, e + 2, ...
            nxt = next((t for t in range(e, steps, 2) if not issued[t]), None)
            if nxt is not None and a_ready[nxt]:
                actions.append(("issue", nxt))
        if not actions:
            break
        kind, arg = rng.choice(actions)
        if kind == "load":
            loaded += 1
        elif kind == "read":
            have_block[arg] += 1
        elif kind == "write":
            t = writers[arg][pos[arg]]
            if t >= sa:
                k = (t - sa) // sa
                if done_c[t % sa] <= k:  # passed before step t - sa completed
                    fooled = True
            a_ready[t] = True  # Q6_K: one writer per step; Q4_K: the only writer
            pos[arg] += 1
        else:
            t = arg
            issued[t] = True
            done_c[t % sa] += 1
    return fooled


def fooled_in_any(sa, q6k, trials=3000):
    return any(simulate(sa, q6k, seed=s) for s in range(trials))


@pytest.mark.parametrize("sa", [2, 3, 4, 5, 6, 8])
def test_q4k_writers_never_pass_early(sa):
    """Every Q4_K writer writes every K step in order, so it observes every phase
    of each done barrier, at any ring depth."""
    assert not fooled_in_any(sa, q6k=False)


@pytest.mark.parametrize("sa", [3, 4, 5, 8])
def test_q6k_three_or_more_stages_never_pass_early(sa):
    assert not fooled_in_any(sa, q6k=True)


def test_q6k_two_stages_can_pass_early():
    """The failure seen on the GPU (wrong output and a wait timeout once the
    packed copies ran ahead) at SA = 2."""
    assert fooled_in_any(2, q6k=True)


def simulate_xa(sx, sa, gateup, blocks=5, seed=0):
    """x ring (SX) and A ring (SA) with done barriers indexed by K step modulo
    D = max(SX, SA), as the kernel runs Q4_K: the x producer loads step t after
    waiting for done(t - SX); the (Q4_K, in-order) dequant writes step t after
    waiting for done(t - SA); an issuer needs both tiles.  Gate/up: both
    issuers take every step and a done phase needs both commits; one tensor:
    the issuers alternate and one commit completes a phase.  Returns True if a
    wait passed before its phase completed."""
    rng = random.Random(seed)
    d = max(sx, sa)
    steps = 4 * blocks
    need = 2 if gateup else 1
    done_c = [0] * d   # completed phases of done[slot]
    done_n = [0] * d   # commits toward the current phase
    x_ready = [False] * steps
    a_ready = [False] * steps
    issued = [[False] * steps for _ in range(2)]
    xp = ap = 0        # next step of the x producer and of the dequant
    fooled = False

    def may_pass(t, lag):  # wait on done(t - lag): phase k of slot (t - lag) % d
        if t < lag:
            return True, False
        u = t - lag
        k, c = u // d, done_c[u % d]
        return (c & 1) != (k & 1), c <= k

    while True:
        acts = []
        if xp < steps and may_pass(xp, sx)[0]:
            acts.append(("x", None))
        if ap < steps and may_pass(ap, sa)[0]:
            acts.append(("a", None))
        for e in range(2):
            order = range(steps) if gateup else range(e, steps, 2)
            nxt = next((t for t in order if not issued[e][t]), None)
            if nxt is not None and x_ready[nxt] and a_ready[nxt]:
                acts.append(("issue", (e, nxt)))
        if not acts:
            break
        kind, arg = rng.choice(acts)
        if kind == "x":
            fooled |= may_pass(xp, sx)[1]
            x_ready[xp] = True
            xp += 1
        elif kind == "a":
            fooled |= may_pass(ap, sa)[1]
            a_ready[ap] = True
            ap += 1
        else:
            e, t = arg
            issued[e][t] = True
            done_n[t % d] += 1
            if done_n[t % d] == need:
                done_n[t % d] = 0
                done_c[t % d] += 1
    assert xp == steps and ap == steps  # no deadlock
    return fooled


@pytest.mark.parametrize("gateup", [True, False])
@pytest.mark.parametrize("sx,sa", [(2, 2), (2, 3), (3, 2), (4, 2), (3, 3), (4, 4), (4, 5)])
def test_q4k_x_and_a_rings_never_pass_early(sx, sa, gateup):
    """Separate x and A ring depths over one done ring of max(SX, SA): no wait
    passes early and nothing deadlocks (gate/up runs 3 x + 2 A stages)."""
    assert not any(simulate_xa(sx, sa, gateup, seed=s) for s in range(800))


def simulate_rings(sx, sa, gateup, q6k, blocks=5, seed=0):
    """The GEMM's three rings with parity waits everywhere, as the kernel runs
    them: x tiles (SX slots; the producer loads step t after waiting for
    done(t - SX), and loads in flight land in any order), A tiles (SA slots;
    the writers write step t after waiting for done(t - SA); Q4_K one writer
    of every step in order, Q6_K two halves, part p writing 4i+2p and
    4i+2p+1), and one done ring of D = max(SX, SA) barriers indexed by K step.
    An issuer waits on the x and A slots of its step by parity (gate/up: both
    issuers take every step and a done phase needs both commits; one tensor:
    the issuers alternate).  Returns "early" if a wait passed before the
    phase it waits for had completed, "stuck" if every party waits on a
    phase that has been overtaken (a deadlock), else None."""
    rng = random.Random(seed)
    d = max(sx, sa)
    steps = 4 * blocks
    need = 2 if gateup else 1
    done_c, done_n = [0] * d, [0] * d
    x_c, a_c = [0] * sx, [0] * sa  # completed phases of x_full / a_full per slot
    if q6k:
        writers = [[4 * i + 2 * p + j for i in range(blocks) for j in range(2)] for p in range(2)]
    else:
        writers = [list(range(steps))]
    wpos = [0] * len(writers)
    xp = 0
    in_flight = []
    issued = [[False] * steps for _ in range(2)]
    fooled = False

    def wait_done(t, lag):  # (parity passes, passed early) for done(t - lag)
        if t < lag:
            return True, False
        u = t - lag
        k, c = u // d, done_c[u % d]
        return (c & 1) != (k & 1), c <= k

    def wait_slot(cnt, n, t):  # the slot of step t in a ring of n, phase t // n
        k, c = t // n, cnt[t % n]
        return (c & 1) != (k & 1), c <= k

    while True:
        acts = []
        if xp < steps and wait_done(xp, sx)[0]:
            acts.append(("x", None))
        for i in range(len(in_flight)):
            acts.append(("land", i))
        for w, lst in enumerate(writers):
            if wpos[w] < len(lst) and wait_done(lst[wpos[w]], sa)[0]:
                acts.append(("a", w))
        for e in range(2):
            order = range(steps) if gateup else range(e, steps, 2)
            t = next((u for u in order if not issued[e][u]), None)
            if t is not None and wait_slot(x_c, sx, t)[0] and wait_slot(a_c, sa, t)[0]:
                acts.append(("issue", (e, t)))
        if not acts:
            break
        kind, arg = rng.choice(acts)
        if kind == "x":
            fooled |= wait_done(xp, sx)[1]
            in_flight.append(xp)
            xp += 1
        elif kind == "land":
            t = in_flight.pop(arg)
            x_c[t % sx] += 1
        elif kind == "a":
            t = writers[arg][wpos[arg]]
            fooled |= wait_done(t, sa)[1]
            a_c[t % sa] += 1
            wpos[arg] += 1
        else:
            e, t = arg
            fooled |= wait_slot(x_c, sx, t)[1] or wait_slot(a_c, sa, t)[1]
            issued[e][t] = True
            done_n[t % d] += 1
            if done_n[t % d] == need:
                done_n[t % d] = 0
                done_c[t % d] += 1
        if fooled:
            return "early"  # what follows a wrong pass is not the kernel's protocol
    if xp < steps or any(p < len(w) for p, w in zip(wpos, writers)):
        return "stuck"
    return None


# The plans the host picks (x stages, A stages): single-tensor Q4_K and Q6_K
# with even x rings up to 8, gate/up with up to 4 x stages and up to 5 A stages.
@pytest.mark.parametrize("sx,sa,gateup,q6k", [
    (4, 4, False, False), (4, 5, False, False), (6, 2, False, False), (6, 3, False, False),
    (8, 4, False, False), (8, 5, False, False), (2, 2, False, False),
    (4, 4, False, True), (6, 4, False, True), (8, 4, False, True),
    (2, 2, True, False), (3, 2, True, False), (4, 2, True, False), (3, 3, True, False),
    (4, 3, True, False), (3, 4, True, False), (3, 5, True, False), (4, 4, True, False), (4, 5, True, False)])
def test_rings_never_pass_early_nor_stall(sx, sa, gateup, q6k):
    assert all(simulate_rings(sx, sa, gateup, q6k, seed=s) is None for s in range(400))


def test_odd_x_ring_with_alternating_issuers_can_pass_early():
    """Why single-tensor x rings are even: with an odd ring an issuer skips
    the phases of the other issuer's steps, and an x tile landing out of
    order lets its parity wait pass on the slot's previous tile."""
    assert any(simulate_rings(3, 4, False, False, seed=s) == "early" for s in range(3000))


def test_odd_done_ring_can_stall_q6k():
    """Q6_K with an odd done ring (D = 5): a half waits on done(t - 4) in the
    slot that step t + 1 -- the other half's, already written and issued --
    completes next, so the barrier can run two phases past the wait, which
    then never passes."""
    assert any(simulate_rings(5, 4, False, True, seed=s) == "stuck" for s in range(3000))


class Bar:
    """An mbarrier: `count` arrivals complete a phase; a parity wait for phase k
    passes while the number of completed phases has the other parity than k."""

    def __init__(self, count):
        self.count, self.pending, self.done = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.done += 1

    def passes(self, k):
        return (self.done & 1) != (k & 1)

    def early(self, k):
        return self.done <= k  # passed although phase k has not completed


def simulate_decode_ring(warps, stages, steps, nchunks, seed, empty_wait=True):
    """The decode GEMV's producer/consumer ring.  The producer runs, in order,
    for every step st: (st >= S) wait for empty[s] phase st / S - 1 (every
    compute warp released step st - S), add the warps' partials of step st - S
    if that step ended a tile, then issue the copy of step st into stage
    st % S; at the end it waits for and adds the last S steps.  A copy lands
    later and completes full[s].  Each compute warp waits for full[s] phase
    st / S, reads the stage (start and end are separate events), writes its
    partial into the stage's slot at a tile's last chunk and arrives on
    empty[s].  Returns (fooled, overwritten): a wait that passed early, or a
    stage refilled while a warp read it, a warp reading stale bytes, or a
    partial missing or replaced when the producer adds it, or a hang (counted
    as overwritten).  empty_wait=False drops the producer's empty wait (a
    control)."""
    rng = random.Random(seed)
    full = [Bar(1) for _ in range(stages)]
    empty = [Bar(warps) for _ in range(stages)]
    ops = []
    for st in range(steps):
        if st >= stages:
            ops += [("wait", st - stages), ("finish", st - stages)]
        ops.append(("issue", st))
    for st in range(max(0, steps - stages), steps):
        ops += [("wait", st), ("finish", st)]
    pc = 0
    content = [None] * stages
    part = [[None] * warps for _ in range(stages)]
    inflight = []
    w_next = [0] * warps
    reading = [None] * warps
    fooled = overwritten = False
    while True:
        acts = []
        if pc < len(ops):
            kind, st = ops[pc]
            if kind != "wait" or not empty_wait or empty[st % stages].passes(st // stages):
                acts.append("p")
        if inflight:
            acts.append("land")
        for w in range(warps):
            st = w_next[w]
            if reading[w] is not None:
                acts.append(("end", w))
            elif st < steps and full[st % stages].passes(st // stages):
                acts.append(("start", w))
        if not acts:
            break
        a = rng.choice(acts)
        if a == "p":
            kind, st = ops[pc]
            s = st % stages
            if kind == "wait" and empty_wait:
                fooled |= empty[s].early(st // stages)
            elif kind == "finish" and st % nchunks == nchunks - 1:
                if any(p != st for p in part[s]):
                    overwritten = True
            elif kind == "issue":
                inflight.append((s, st))
            pc += 1
        elif a == "land":
            s, st = inflight.pop(rng.randrange(len(inflight)))
            if any(r is not None and r % stages == s for r in reading):
                overwritten = True  # bytes of a stage a warp is still reading
            content[s] = st
            full[s].arrive()
        elif a[0] == "start":
            w = a[1]
            st = w_next[w]
            fooled |= full[st % stages].early(st // stages)
            if content[st % stages] != st:
                overwritten = True
            reading[w] = st
        else:
            w = a[1]
            st = reading[w]
            s = st % stages
            if content[s] != st:
                overwritten = True
            if st % nchunks == nchunks - 1:
                part[s][w] = st
            reading[w] = None
            w_next[w] += 1
            empty[s].arrive()
    if pc < len(ops) or inflight or any(n != steps for n in w_next):
        overwritten = True  # stuck: a warp or the producer never finished
    return fooled, overwritten


@pytest.mark.parametrize("warps,stages,steps,nchunks", [(1, 2, 7, 1), (3, 3, 10, 1), (4, 3, 12, 4), (12, 6, 13, 2)])
def test_decode_ring(warps, stages, steps, nchunks):
    """The decode GEMV's ring: no wait passes early, no stage is refilled while
    a warp reads it, no partial is replaced before the producer adds it, and
    nothing deadlocks."""
    for seed in range(400):
        assert simulate_decode_ring(warps, stages, steps, nchunks, seed) == (False, False)


def test_decode_ring_without_the_empty_wait_can_race():
    """Control: a producer that refills without waiting for the warps' release
    overwrites a stage in use or adds partials not yet written, and the model
    sees it."""
    assert any(simulate_decode_ring(3, 2, 9, 1, seed, empty_wait=False)[1] for seed in range(400))
