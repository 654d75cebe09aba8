"""CPU model of the packed-batch work list of the forward kernel.

The kernel visits the non-empty (sequence, head, 256-row level) items of a
packed batch as one compact list, longest first: levels from the top down,
within a level every sequence longer than 256 * level in index order, each
with its H heads. CTA c of G takes list positions w*G + c in even waves w and
w*G + G-1-c in odd waves. One warp per CTA walks its positions with a cursor
(the current level, the level's first position and sequence count, and a scan
point), counting a level and locating the j-th sequence 32 sequences at a
time, as a warp ballot does, and hands the items to the other roles through a
ring (whose barrier protocol test_pipeline_protocol checks). This model
follows the cursor's steps and checks that
every non-empty item is visited by exactly one CTA, that no empty item is, that
malformed sequences are skipped, and that the causal work per CTA is balanced.
"""
import random

import pytest

ROWS = 256


def seq_len(cu, s, total, max_seqlen):
    a, b = cu[s], cu[s + 1]
    bad = a < 0 or b < a or b > total or b - a > max_seqlen
    return (0 if bad else b - a), bad


class Cursor:
    """The scheduler warp's walk over one CTA's positions of the compact list."""

    def __init__(self, cu, total, max_seqlen, H, G, cta):
        self.cu, self.total, self.N, self.H, self.G, self.cta = cu, total, max_seqlen, H, G, cta
        self.B = len(cu) - 1
        self.w = 0
        mx, self.any_bad = 0, False
        for s0 in range(0, self.B, 32):
            for s in range(s0, min(s0 + 32, self.B)):
                n, bad = seq_len(cu, s, total, max_seqlen)
                mx = max(mx, n)
                self.any_bad |= bad
        self.lvl = (mx - 1) // ROWS if mx > 0 else -1
        self.cnt = self.count_level(self.lvl) if self.lvl >= 0 else 0
        self.start = 0
        self.base_pos = self.base_rank = 0

    def qualifies(self, s, thr):
        return s < self.B and seq_len(self.cu, s, self.total, self.N)[0] > thr

    def count_level(self, lvl):
        thr = lvl * ROWS
        return sum(sum(self.qualifies(s, thr) for s in range(s0, s0 + 32)) for s0 in range(0, self.B, 32))

    def next(self):
        if self.lvl < 0:
            return None
        c = (self.G - 1 - self.cta) if (self.w & 1) else self.cta
        k = self.w * self.G + c
        self.w += 1
        while k >= self.start + self.cnt * self.H:
            self.start += self.cnt * self.H
            self.lvl -= 1
            if self.lvl < 0:
                return None
            self.cnt = self.count_level(self.lvl)
            self.base_pos = self.base_rank = 0
        r = k - self.start
        j, h = divmod(r, self.H)
        thr = self.lvl * ROWS
        while self.base_pos < self.B:
            bal = [self.qualifies(self.base_pos + i, thr) for i in range(32)]
            nb = sum(bal)
            if self.base_rank + nb > j:
                want = j - self.base_rank
                lanes = [i for i in range(32) if bal[i]]
                s = self.base_pos + lanes[want]
                return s, h, self.lvl
            self.base_rank += nb
            self.base_pos += 32
        self.lvl = -1
        return None


def walk(cu, total, max_seqlen, H, G):
    per_cta = []
    for cta in range(G):
        cur = Cursor(cu, total, max_seqlen, H, G, cta)
        items = []
        while (it := cur.next()) is not None:
            items.append(it)
        per_cta.append(items)
    return per_cta


def expected_items(cu, total, max_seqlen, H):
    out = set()
    for s in range(len(cu) - 1):
        n, _ = seq_len(cu, s, total, max_seqlen)
        for lvl in range((n + ROWS - 1) // ROWS):
            for h in range(H):
                out.add((s, h, lvl))
    return out


def cu_of(lengths):
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    return cu


def check_cover(cu, total, max_seqlen, H, G):
    per_cta = walk(cu, total, max_seqlen, H, G)
    seen = [it for items in per_cta for it in items]
    assert len(seen) == len(set(seen)), "an item visited twice"
    assert set(seen) == expected_items(cu, total, max_seqlen, H)
    return per_cta


@pytest.mark.parametrize("seed", range(6))
def test_every_nonempty_item_once(seed):
    rng = random.Random(seed)
    nseq = rng.choice([1, 3, 31, 32, 33, 70])
    lengths = [rng.choice([0, 1, 255, 256, 257, rng.randint(1, 3000)]) for _ in range(nseq)]
    cu = cu_of(lengths)
    H = rng.choice([1, 3, 8])
    G = rng.choice([1, 7, 152])
    check_cover(cu, cu[-1], max(max(lengths), 1), H, G)


def test_empty_batch_and_zero_lengths():
    assert walk(cu_of([0, 0, 0]), 0, 16, 4, 152) == [[] for _ in range(152)]
    check_cover(cu_of([0, 300, 0, 1]), 301, 300, 2, 5)


def test_malformed_sequences_are_skipped():
    # sequence 1 runs backwards, sequence 3 ends past total, sequence 4 is longer than max_seqlen
    cu = [0, 300, 200, 500, 900, 1600]
    per_cta = check_cover(cu, 800, 600, 2, 9)
    seqs = {s for items in per_cta for (s, _, _) in items}
    assert seqs == {0, 2}
    assert Cursor(cu, 800, 600, 2, 9, 0).any_bad


def test_order_is_longest_first_per_cta():
    lengths = [300, 5000, 700, 2048, 64]
    cu = cu_of(lengths)
    for items in walk(cu, cu[-1], 5000, 4, 13):
        lv = [lvl for (_, _, lvl) in items]
        assert lv == sorted(lv, reverse=True)


def test_balance_of_a_log_uniform_length_mix():
    """Causal work of an item = K/V blocks of its two 128-row tiles plus a fixed
    cost; the compact snake keeps the busiest CTA within 3 % of the mean on a
    65,536-token mix of 256..8192-token sequences over 152 CTAs."""
    rng = random.Random(7)
    lengths, acc = [], 0
    while acc < 65536:
        L = min(int(round(256 * (8192 / 256) ** rng.random())), 65536 - acc)
        lengths.append(L)
        acc += L
    cu = cu_of(lengths)
    H, G = 32, 152

    def cost(s, lvl):
        n = lengths[s]
        c = 0
        for t in range(2):
            r0 = lvl * ROWS + t * 128
            if r0 < n:
                c += (min(n, r0 + 128) - 1) // 64 + 1
        return c + 0.5

    per_cta = check_cover(cu, acc, max(lengths), H, G)
    loads = [sum(cost(s, lvl) for (s, _, lvl) in items) for items in per_cta]
    assert max(loads) <= 1.03 * (sum(loads) / G), max(loads) / (sum(loads) / G)
