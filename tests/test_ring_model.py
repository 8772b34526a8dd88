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
