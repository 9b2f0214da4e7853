"""Host-side model of the persistent (stream-K) decode schedule, CPU only.

The persistent kernel cuts the flattened (kv head, sequence, block) list into
ranges: W1 equal ranges over the first T1 = T * f entries (phase 1), then
chunks of C2 entries (phase 2); the merge kernel later finds the ranges that
touched a unit and the partial slot each of them wrote.  This test restates
both index formulas and checks, on random batches, that every KV block is
visited exactly once and that the merge reads exactly the partials that were
written for each cut unit (and no others)."""
import numpy as np
import pytest


class StreamK:
    """Restatement of the kernel's make_streamk / range_start / range_of."""

    def __init__(self, T, g1_warps, g2_warps, f_per_mille):
        if g2_warps == 0:
            f_per_mille = 1000
        self.T = T
        self.T1 = T * f_per_mille // 1000
        self.W1 = 0 if self.T1 == 0 else min(g1_warps, max(1, self.T1 // 4))
        if self.W1 == 0:
            self.T1 = 0
        rest = T - self.T1
        self.C2 = 1 if (rest == 0 or g2_warps == 0) else -(-rest // g2_warps)
        self.nranges = self.W1 + g2_warps

    def start(self, x):
        if x < self.W1:
            return x * self.T1 // self.W1
        return min(self.T1 + (x - self.W1) * self.C2, self.T)

    def range_of(self, n):
        if n < self.T1:
            return ((n + 1) * self.W1 - 1) // self.T1
        return self.W1 + (n - self.T1) // self.C2


def schedule(lens, bs, Hkv, g1, g2, f):
    nblk = [-(-L // bs) for L in lens]
    cum = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int64)
    return cum, StreamK(Hkv * int(cum[len(lens)]), g1, g2, f)


def range_parts(cum, sk, Hkv):
    """What each range visits and writes, following the decode kernel."""
    visits, written = [], {}   # written[unit] -> list of slots, or "final"
    for x in range(sk.nranges):
        r0, r1 = sk.start(x), sk.start(x + 1)
        cur, first_j, last_j, part = None, 0, 0, 0

        def finish(u, fj, lj, k):
            i = u // Hkv
            nbk = int(cum[i + 1] - cum[i])
            written.setdefault(u, []).append("final" if (fj == 0 and lj == nbk - 1) else 2 * x + k)

        Tseq = int(cum[-1])
        for n in range(r0, r1):
            h, m = n // Tseq, n % Tseq                       # head-major list
            i = int(np.searchsorted(cum, m, side="right") - 1)  # largest i: cum[i] <= m
            j = m - int(cum[i])
            u = i * Hkv + h
            visits.append((u, j))
            if u != cur:
                if cur is not None:
                    finish(cur, first_j, last_j, part)
                    part = 1
                cur, first_j = u, j
            last_j = j
        if cur is not None:
            finish(cur, first_j, last_j, part)
    return visits, written


def merge_slots(cum, sk, Hkv, i, h):
    """Slots the merge kernel reads for unit (i, h), or None if it skips."""
    nbk = int(cum[i + 1] - cum[i])
    if nbk == 0 or sk.T == 0:
        return None
    s = h * int(cum[-1]) + int(cum[i])
    e = s + nbk
    xs, xe = sk.range_of(s), sk.range_of(e - 1)
    if xs == xe:
        return None
    first_is_tail = s != sk.start(xs)
    return [2 * x + (1 if (x == xs and first_is_tail) else 0) for x in range(xs, xe + 1)]


@pytest.mark.parametrize("seed", range(60))
def test_every_block_once_and_merge_reads_what_was_written(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    bs = int(rng.choice([16, 32]))
    Hkv = int(rng.choice([1, 2, 8]))
    g1 = int(rng.choice([1, 3, 8, 64, 1216]))
    g2 = int(rng.choice([0, 1, 5, 64, 2432]))
    f = int(rng.choice([0, 1, 500, 750, 999, 1000]))
    hi = int(rng.choice([1, 20, 300, 3000]))
    lens = [int(x) for x in rng.integers(1, hi + 1, size=B)]
    cum, sk = schedule(lens, bs, Hkv, g1, g2, f)
    visits, written = range_parts(cum, sk, Hkv)
    expect = [(i * Hkv + h, j) for i in range(B) for h in range(Hkv)
              for j in range(-(-lens[i] // bs))]
    assert sorted(visits) == sorted(expect) and len(visits) == len(set(visits))
    slots_used = [sl for v in written.values() for sl in v if sl != "final"]
    assert len(slots_used) == len(set(slots_used))          # no slot written twice
    assert all(sl < 2 * (g1 + g2) for sl in slots_used)    # within the workspace
    for i in range(B):
        for h in range(Hkv):
            u = i * Hkv + h
            got = merge_slots(cum, sk, Hkv, i, h)
            if got is None:
                assert written[u] == ["final"]
            else:
                assert "final" not in written[u]
                assert sorted(got) == sorted(written[u])


def test_range_of_inverts_ranges():
    for T in (1, 5, 97, 4096, 10**6 + 7):
        for g1, g2, f in ((1, 0, 750), (1216, 0, 1000), (1216, 2432, 750), (3, 7, 0), (8, 1, 999)):
            sk = StreamK(T, g1, g2, f)
            assert sk.start(0) == 0 and sk.start(sk.nranges) == T
            for n in list(range(min(T, 300))) + [T - 1, T // 2]:
                x = sk.range_of(n)
                assert sk.start(x) <= n < sk.start(x + 1)
