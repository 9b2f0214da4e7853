"""The C block manager (pkv_bm_*) against a plain Python model of the same
bookkeeping (CPU only; the manager makes no GPU calls).

The model restates the block manager of the first page, section 4.2:
ceil(n / block_size) blocks per sequence from a free list (lowest id first),
reference-counted sharing after a fork, copy-on-write when a token lands in
a shared block, and swap of the blocks older than a GPU window to a CPU pool.
"""
import numpy as np
import pytest

from paged_kv_cache_268_gb300 import _binding as B
from paged_kv_cache_268_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.load_library()


class Model:
    def __init__(self, ng, nc, bs):
        self.bs = bs
        self.free = {"g": list(range(ng - 1, -1, -1)), "c": list(range(nc - 1, -1, -1))}
        self.ref = {"g": [0] * ng, "c": [0] * nc}
        self.seqs = {}

    def _pop(self, pool):
        i = self.free[pool].pop()
        self.ref[pool][i] = 1
        return i

    def _release(self, pool, i):
        self.ref[pool][i] -= 1
        if self.ref[pool][i] == 0:
            self.free[pool].append(i)

    def add(self, sid, n):
        need = -(-n // self.bs)
        if sid in self.seqs:
            return -2
        if need > len(self.free["g"]):
            return -8
        self.seqs[sid] = [n, [(self._pop("g"), "g") for _ in range(need)]]
        return 0

    def fork(self, p, c):
        if p not in self.seqs or c in self.seqs or any(pl == "c" for _, pl in self.seqs[p][1]):
            return -2
        for b, _ in self.seqs[p][1]:
            self.ref["g"][b] += 1
        self.seqs[c] = [self.seqs[p][0], list(self.seqs[p][1])]
        return 0

    def append(self, sid):
        if sid not in self.seqs:
            return -2, None
        n, blocks = self.seqs[sid]
        cs = cd = -1
        if n % self.bs == 0:
            if not self.free["g"]:
                return -8, None
            blocks.append((self._pop("g"), "g"))
        else:
            b, pl = blocks[-1]
            if pl == "c":
                return -2, None
            if self.ref["g"][b] > 1:
                if not self.free["g"]:
                    return -8, None
                f = self._pop("g")
                self.ref["g"][b] -= 1
                blocks[-1] = (f, "g")
                cs, cd = b, f
        self.seqs[sid][0] = n + 1
        return 0, (blocks[-1][0] * self.bs + n % self.bs, cs, cd)

    def free_seq(self, sid):
        if sid not in self.seqs:
            return -2
        for b, pl in self.seqs.pop(sid)[1]:
            self._release(pl, b)
        return 0

    def swap_out(self, sid, window):
        if sid not in self.seqs:
            return -2, None
        blocks = self.seqs[sid][1]
        cold = [j for j in range(len(blocks) - window)
                if blocks[j][1] == "g" and self.ref["g"][blocks[j][0]] == 1]
        if len(cold) > len(self.free["c"]):
            return -8, None
        pairs = []
        for j in cold:
            g = blocks[j][0]
            c = self._pop("c")
            self._release("g", g)
            blocks[j] = (c, "c")
            pairs.append((g, c))
        return 0, pairs

    def swap_in(self, sid):
        if sid not in self.seqs:
            return -2, None
        blocks = self.seqs[sid][1]
        warm = [j for j in range(len(blocks)) if blocks[j][1] == "c"]
        if len(warm) > len(self.free["g"]):
            return -8, None
        pairs = []
        for j in warm:
            c = blocks[j][0]
            g = self._pop("g")
            self._release("c", c)
            blocks[j] = (g, "g")
            pairs.append((c, g))
        return 0, pairs


def _code(fn, *a):
    try:
        return 0, fn(*a)
    except B.PkvError as e:
        return e.code, None


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_model(seed):
    rng = np.random.default_rng(seed)
    ng, nc, bs = int(rng.integers(8, 80)), int(rng.integers(0, 40)), int(rng.choice([1, 4, 16]))
    m = B.BlockManager(ng, nc, bs)
    ref = Model(ng, nc, bs)
    next_id = 0
    for _ in range(400):
        op = rng.choice(["add", "fork", "append", "append", "append", "free", "out", "in"])
        live = list(ref.seqs)
        sid = int(rng.choice(live)) if live and rng.random() < 0.9 else int(rng.integers(0, 1000))
        if op == "add":
            n = int(rng.integers(0, 5 * bs))
            rc, _ = _code(m.add_sequence, next_id, n)
            assert rc == ref.add(next_id, n)
            next_id += 1
        elif op == "fork":
            rc, _ = _code(m.fork, sid, next_id)
            assert rc == ref.fork(sid, next_id)
            next_id += 1
        elif op == "append":
            rc, got = _code(m.append_token, sid)
            erc, exp = ref.append(sid)
            assert rc == erc and (rc != 0 or got == exp)
        elif op == "free":
            rc, _ = _code(m.free_sequence, sid)
            assert rc == ref.free_seq(sid)
        elif op == "out":
            w = int(rng.integers(0, 4))
            rc, got = _code(m.swap_out, sid, w)
            erc, exp = ref.swap_out(sid, w)
            assert rc == erc and (rc != 0 or got.tolist() == [list(p) for p in exp])
        else:
            rc, got = _code(m.swap_in, sid)
            erc, exp = ref.swap_in(sid)
            assert rc == erc and (rc != 0 or got.tolist() == [list(p) for p in exp])
        assert m.num_free() == (len(ref.free["g"]), len(ref.free["c"]))
    # every live sequence's table and length agree with the model
    for sid, (n, blocks) in ref.seqs.items():
        nt, nb, ncpu = m.seq_info(sid)
        assert (nt, nb, ncpu) == (n, len(blocks), sum(pl == "c" for _, pl in blocks))
        if ncpu == 0 and nb <= 64:
            t, lens = m.block_tables([sid], 64)
            assert lens[0] == n and list(t[0, :nb]) == [b for b, _ in blocks]
            assert np.all(t[0, nb:] == -1)
    # reference counts are the number of sequences holding each block
    counts = {"g": [0] * ng, "c": [0] * nc}
    for _, blocks in ref.seqs.values():
        for b, pl in blocks:
            counts[pl][b] += 1
    assert counts == ref.ref
    m.close()


def test_allocation_follows_block_size_and_copy_on_write():
    m = B.BlockManager(10, 4, 16)
    m.add_sequence(1, 33)                         # ceil(33/16) = 3 blocks
    assert m.seq_info(1) == (33, 3, 0) and m.num_free() == (7, 4)
    m.fork(1, 2)                                  # shares the 3 blocks
    assert m.num_free() == (7, 4)
    slot, cs, cd = m.append_token(2)              # token 33 lands in shared block 2
    assert (cs, cd) == (2, 3) and slot == 3 * 16 + 1
    slot, cs, cd = m.append_token(1)              # block 2 is now private to seq 1
    assert (cs, cd) == (-1, -1) and slot == 2 * 16 + 1
    t, lens = m.block_tables([1, 2], 4)
    assert t.tolist() == [[0, 1, 2, -1], [0, 1, 3, -1]] and lens.tolist() == [34, 34]
    pairs = m.swap_out(1, 1)                      # block 2 private, 0 and 1 shared: nothing
    assert pairs.shape == (0, 2)
    m.free_sequence(2)
    pairs = m.swap_out(1, 1)                      # now 0 and 1 are private: to CPU 0 and 1
    assert pairs.tolist() == [[0, 0], [1, 1]]
    with pytest.raises(B.PkvError):
        m.block_tables([1], 4)                    # CPU-resident blocks cannot be decoded
    back = m.swap_in(1)
    assert back.tolist() == [[0, 1], [1, 0]]     # freed blocks are reused last-freed first
    with pytest.raises(B.PkvError) as e:
        m.add_sequence(9, 16 * 20)
    assert e.value.code == -8
    m.close()
