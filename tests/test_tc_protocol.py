"""Exhaustive CPU model of the tcgen05 decode kernel's mbarrier protocol.

The warp-specialised kernel (csrc/pkv_decode_tc.cuh) runs three roles that
hand work on through mbarriers: a producer lane issuing TMA loads of K and V
tiles into a ring of SL slots (K one group ahead of V: K0 K1 V0 K2 V1 ...),
an MMA lane issuing S = K.Q^T and O += V^T.P^T as soon as either is ready,
and the softmax warps.  Every wait is a parity wait: waiting for completion
k of a barrier returns true when the barrier's completion count c has the
parity of k + 1.  That answer is right only while c is k or k + 1; at c =
k - 1 the wait passes a phase early (the tile a slot held before), at
c = k + 2 it misses the phase and would spin until its time limit.

This model explores every interleaving of the roles, the TMA landings (in any
order) and the tensor-core completions (in issue order) for small partitions,
and checks at every reachable state that each wait that is pending, or each
test the MMA lane makes, sees c in {k, k + 1}, and that no state is stuck
before the partition is done.  A variant without the MMA lane's bound (S at
most one group ahead of PV) must fail the check, which shows the model can
see the aliasing the bound prevents."""
from __future__ import annotations

import pytest


def tile_k(g, ng):
    return 0 if g == 0 else 2 * g - 1


def tile_v(g, ng):
    return 2 * g + 2 if g + 1 < ng else 2 * ng - 1


class Violation(AssertionError):
    pass


def explore(SL: int, ng: int, PBUF: int, ragged: bool, bound: bool = True) -> int:
    """Returns the number of reachable states; raises Violation on a wait
    that could alias or on a stuck state."""
    nt = 2 * ng
    tk = [tile_k(g, ng) for g in range(ng)]
    tv = [tile_v(g, ng) for g in range(ng)]
    group_of_tile = {}
    for g in range(ng):
        group_of_tile[tk[g]] = ("K", g)
        group_of_tile[tv[g]] = ("V", g)

    # state: (issued tiles, landed bitmask, drain index, gs, gp, MMA queue,
    #         S done, PV done, softmax group, softmax step, rescale flag)
    # softmax steps: 0 wait S(g) full; 1 choose rescale; 2 wait PV(g-1) for the
    # rescale; 3 wait the P buffer; 4 wait V(g) landed (ragged last group);
    # 5 publish P(g); past the last group: step 0 waits for the last PV, 7 is done.
    start = (0, 0, 0, 0, 0, (), 0, 0, 0, 0, False)
    seen = set()
    stack = [start]

    def check(c, k, what, st):
        if not (k <= c <= k + 1):
            raise Violation(f"{what}: completion {k} tested at count {c} "
                            f"(SL={SL} ng={ng} PBUF={PBUF} ragged={ragged}) state={st}")

    while stack:
        st = stack.pop()
        if st in seen:
            continue
        seen.add(st)
        npd, landed, drain, gs, gp, queue, sdone, pvdone, sg, step, resc = st

        # barrier completion counts
        def c_full(slot):
            return sum(1 for t in range(npd) if t % SL == slot and landed >> t & 1)

        def consumed(t):
            kind, g = group_of_tile[t]
            return g < sdone if kind == "K" else g < pvdone

        def c_empty(slot):
            return sum(1 for t in range(npd) if t % SL == slot and consumed(t))

        def c_sfull(b):
            return sum(1 for g in range(sdone) if g & 1 == b)

        reads = sg + (1 if step >= 1 and sg < ng else 0)       # S(g) read by the softmax
        pubs = sg                                               # P published

        def c_sfree(b):
            return sum(1 for g in range(reads) if g & 1 == b)

        def c_pfull(pb):
            return sum(1 for g in range(pubs) if g % PBUF == pb)

        def c_pvdone(pb):
            return sum(1 for j in range(pvdone) if j % PBUF == pb)

        def full_ok(t, what):
            check(c_full(t % SL), t // SL, what, st)
            return c_full(t % SL) >= t // SL + 1

        moves = []
        # producer: issue tile npd once the slot's previous tile was consumed
        if npd < nt:
            ok = True
            if npd >= SL:
                check(c_empty(npd % SL), npd // SL - 1, "producer empty wait", st)
                ok = c_empty(npd % SL) >= npd // SL
            if ok:
                moves.append((npd + 1, landed, drain, gs, gp, queue, sdone, pvdone, sg, step, resc))
        else:
            # drain: the last tile of each slot lands before exit
            first = max(0, nt - SL)
            d = max(drain, first)
            if d < nt and full_ok(d, "producer drain wait"):
                moves.append((npd, landed, d + 1, gs, gp, queue, sdone, pvdone, sg, step, resc))
        # TMA: any issued tile may land
        for t in range(npd):
            if not landed >> t & 1:
                moves.append((npd, landed | 1 << t, drain, gs, gp, queue, sdone, pvdone, sg, step,
                              resc))
        # MMA lane: S(gs) and PV(gp), whichever is ready
        if gp < ng:
            if gs < ng and (gs <= gp + 1 or not bound):
                ready = full_ok(tk[gs], "MMA test of K(%d)" % gs)
                if ready and gs >= 2:
                    check(c_sfree(gs & 1), (gs - 2) >> 1, "MMA test of S buffer free", st)
                    ready = c_sfree(gs & 1) >= ((gs - 2) >> 1) + 1
                if ready:
                    moves.append((npd, landed, drain, gs + 1, gp, queue + (("S", gs),), sdone,
                                  pvdone, sg, step, resc))
            if gp < gs:
                pb = gp % PBUF
                check(c_pfull(pb), gp // PBUF, "MMA test of P(%d)" % gp, st)
                if c_pfull(pb) >= gp // PBUF + 1 and full_ok(tv[gp], "MMA test of V(%d)" % gp):
                    moves.append((npd, landed, drain, gs, gp + 1, queue + (("P", gp),), sdone,
                                  pvdone, sg, step, resc))
        # tensor cores: the oldest issued MMA completes (commits arrive in order)
        if queue:
            kind, _ = queue[0]
            moves.append((npd, landed, drain, gs, gp, queue[1:],
                          sdone + (kind == "S"), pvdone + (kind == "P"), sg, step, resc))
        # softmax warps
        if sg < ng:
            g = sg
            nxt = None
            if step == 0:
                check(c_sfull(g & 1), g >> 1, "softmax S(%d) wait" % g, st)
                if c_sfull(g & 1) >= (g >> 1) + 1:
                    nxt = [(1, False)]
            elif step == 1:
                # a data-dependent rescale of O (needs PV(g-1) done) may or may not happen
                nxt = [(2, True), (3, False)] if g > 0 else [(3, False)]
            elif step == 2:
                pb = (g - 1) % PBUF
                check(c_pvdone(pb), (g - 1) // PBUF, "softmax rescale wait", st)
                if c_pvdone(pb) >= (g - 1) // PBUF + 1:
                    nxt = [(3, resc)]
            elif step == 3:
                if g >= PBUF:
                    pb = g % PBUF
                    check(c_pvdone(pb), (g - PBUF) // PBUF, "softmax P buffer wait", st)
                    if c_pvdone(pb) >= (g - PBUF) // PBUF + 1:
                        nxt = [(4, resc)]
                else:
                    nxt = [(4, resc)]
            elif step == 4:
                if ragged and g == ng - 1:
                    if full_ok(tv[g], "softmax V(%d) wait" % g):
                        nxt = [(5, resc)]
                else:
                    nxt = [(5, resc)]
            elif step == 5:
                moves.append((npd, landed, drain, gs, gp, queue, sdone, pvdone, sg + 1, 0, False))
            for s2, r2 in nxt or ():
                moves.append((npd, landed, drain, gs, gp, queue, sdone, pvdone, sg, s2, r2))
        elif step < 7:
            pb = (ng - 1) % PBUF
            check(c_pvdone(pb), (ng - 1) // PBUF, "softmax epilogue wait", st)
            if c_pvdone(pb) >= (ng - 1) // PBUF + 1:
                moves.append((npd, landed, drain, gs, gp, queue, sdone, pvdone, sg, 7, False))
        done = (npd == nt and drain >= nt and gp == ng and not queue and sg == ng and step == 7)
        if not moves and not done:
            raise Violation(f"stuck (SL={SL} ng={ng} PBUF={PBUF} ragged={ragged}) state={st}")
        stack.extend(moves)
    return len(seen)


# the kernel's two layouts: 3 slots with one P buffer (16 padded heads) and 5
# slots with two P buffers (32 padded heads); the other pairs for margin
@pytest.mark.parametrize("SL,PBUF", [(3, 1), (5, 2), (3, 2), (5, 1)])
@pytest.mark.parametrize("ng", [1, 2, 3, 4, 5, 6])
def test_no_wait_aliases_or_sticks(SL, PBUF, ng):
    for ragged in (False, True):
        assert explore(SL, ng, PBUF, ragged) > 0


def test_without_the_bound_a_wait_aliases():
    """Let S run ahead of PV without limit: some interleaving tests a K tile's
    barrier while the slot still holds an older tile."""
    found = False
    for SL, PBUF in ((3, 1), (5, 2)):
        for ng in (3, 4):
            try:
                explore(SL, ng, PBUF, False, bound=False)
            except Violation:
                found = True
    assert found
