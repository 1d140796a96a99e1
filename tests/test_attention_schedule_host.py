"""The IKBO attention kernel's work schedule, checked on the CPU.

The kernel's roles each walk the same schedule (device code in
csrc/ikbo_attn_ws.cuh: AttnWalker maps an item index to its (user, head,
query tile); AttnSched deals whole items round-robin to the persistent CTAs
and spreads the last, partial wave's items over contiguous CTA groups, one
key-block fragment per CTA, publishers first).  This test restates that
schedule in Python, with C++ integer semantics, and checks the properties
the kernel relies on, for the bench shape and ragged ones: every (item, key
block) is covered exactly once; every fragment's item maps to the tile the
item denotes, whatever order the fragments come in (a fragment of a later
item can precede earlier ones); the CTA holding an item's first block merges
partials only from CTAs of higher index whose shares cover the rest."""
import itertools

import pytest

BM = 128


def cdiv(a, b):
    return (a + b - 1) // b


def trunc_div(a, b):  # C++ integer division
    q = abs(a) // abs(b)
    return q if (a >= 0) == (b > 0) else -q


class Walker:
    """AttnWalker: users in order, items (head, query tile) per user."""

    def __init__(self, offs, Lq, H):
        self.offs, self.Lq, self.H = offs, Lq, H
        self.users = len(offs) - 1
        self.init()

    def init(self):
        self.u, self.base = 0, 0
        self.load()

    def load(self):
        if self.u >= self.users:
            self.count = 0
            return
        a, b = self.offs[self.u], self.offs[self.u + 1]
        self.q0, self.nq = a * self.Lq, (b - a) * self.Lq
        self.tiles = cdiv(self.nq, BM)
        self.count = self.tiles * self.H

    def seek(self, t):
        if t < self.base:
            self.init()
        while self.u < self.users and t >= self.base + self.count:
            self.base += self.count
            self.u += 1
            self.load()
        return self.u < self.users

    def item(self, t):
        r = t - self.base
        h = trunc_div(r, self.tiles)
        qt = r - h * self.tiles
        return self.u, h, self.q0 + qt * BM, min(BM, self.nq - qt * BM)


def fragments(n_items, nblk, G, c, split=True):
    """AttnSched.next() sequence of CTA c: (item, jb, je, rank, k)."""
    tail = n_items % G
    n_full = n_items - tail if split and 2 * tail <= G else n_items
    R = n_items - n_full
    tl = None
    if R > 0:
        r = ((c + 1) * R - 1) // G
        c0, c1 = r * G // R, (r + 1) * G // R
        i, k = c - c0, c1 - c0
        jb, je = i * nblk // k, (i + 1) * nblk // k
        if je > jb:
            tl = (n_full + r, jb, je, i, k)
    out = []
    if tl and tl[1] > 0:
        out.append(tl)
    t = c
    while t < n_full:
        out.append((t, 0, nblk, 0, 1))
        t += G
    if tl and tl[1] == 0:
        out.append(tl)
    return out


@pytest.mark.parametrize("counts,Lq,H,Lkv,G", [
    ([256] * 32, 2, 4, 2048, 152),          # the bench shape
    ([256] * 32, 2, 4, 2048, 148),
    ([3, 60], 2, 2, 200, 152),              # fewer items than CTAs
    ([1024] * 16, 2, 4, 2048, 152),         # a last wave more than half full
    ([128] * 64, 1, 4, 8192, 152),          # long contexts
    ([0, 5, 0, 900, 1], 1, 3, 130, 152),    # empty users, ragged tiles
    ([20, 30], 1, 2, 150, 7),
    ([70, 9] * 40, 2, 2, 400, 152),
])
def test_schedule_covers_every_block_once(counts, Lq, H, Lkv, G):
    offs = list(itertools.accumulate([0] + counts))
    nq = offs[-1] * Lq
    n_items = sum(cdiv(c * Lq, BM) for c in counts) * H
    nblk = cdiv(Lkv, 128)
    w0 = Walker(offs, Lq, H)
    canon = []
    for t in range(n_items):
        assert w0.seek(t)
        canon.append(w0.item(t))
    owner = {}
    frags = {c: fragments(n_items, nblk, G, c) for c in range(G)}
    for c, fl in frags.items():
        w = Walker(offs, Lq, H)
        for (it, jb, je, rank, k) in fl:
            assert w.seek(it)
            u, h, row0, rows = w.item(it)
            assert (u, h, row0, rows) == canon[it]
            assert 0 <= h < H and 0 <= row0 and rows >= 1 and row0 + rows <= nq
            for j in range(jb, je):
                assert (it, j) not in owner
                owner[(it, j)] = c
        # a fragment with the item's first block but not its last (a merger)
        # comes last, and its partners are the CTAs after it
        for n, (it, jb, je, rank, k) in enumerate(fl):
            if jb == 0 and je != nblk:
                assert n == len(fl) - 1
                partners = [c + (i - rank) for i in range(rank + 1, k)
                            if (i + 1) * nblk // k > i * nblk // k]
                got = set(range(jb, je))
                for pc in partners:
                    assert pc > c
                    pf = [f for f in frags[pc] if f[0] == it]
                    assert len(pf) == 1 and pf[0][1] > 0
                    got |= set(range(pf[0][1], pf[0][2]))
                assert got == set(range(nblk))
    assert len(owner) == n_items * nblk
