"""A model of the ZipCCL encoder's two-level decoupled look-back, run under
random interleavings of the tickets' steps (no GPU).

The protocol (zc_codec.cu, common.cuh): every ticket publishes its aggregate
(its escape count) as soon as it is known, then later its inclusive prefix.
Tickets form blocks of `block`; each block has one word that only atomics
change: a count of the tickets whose aggregate is in, their sum, and an
inclusive flag that the block's first ticket adds together with the block's
exclusive prefix.  A word is trusted only once its count is full.  A
look-back reads its own block's tickets (one window of `window` states), then
the block words below it, and descends into a block's tickets while that
block is incomplete.  Each model step below is one read or one atomic of a
warp; windows are read entry by entry at one point in time, which the GPU's
relaxed reads of monotone states do not need but which changes nothing the
model checks: every ticket's exclusive prefix must be the true one.
"""
import random

import pytest

EMPTY, AGG, INC = 0, 1, 2


class Model:
    def __init__(self, aggs, block):
        self.aggs = aggs
        self.block = block
        n = len(aggs)
        self.state = [(EMPTY, 0)] * n
        nb = (n + block - 1) // block
        self.words = [[0, 0, 0] for _ in range(nb)]  # [inclusive flag, count, value]

    def ticket_entry(self, i):
        return self.state[i]

    def block_entry(self, b):
        inc, count, value = self.words[b]
        if count != self.block:
            return (EMPTY, 0)  # incomplete: whatever else is in the word
        return (INC if inc else AGG, value)

    def window(self, read, end, lo, width):
        """Entries end, end-1, ... (width of them) down to lo: (kind, sum, at).
        kind 'found': an inclusive entry (sum includes it); 'all': none in
        range (sum of all); 'empty': an empty entry first (at = its index, sum
        of the entries above it).  Below 0 reads as an inclusive zero when lo
        is 0."""
        total = 0
        for k in range(width):
            idx = end - k
            if idx < lo:
                if idx < 0 and lo == 0:
                    return "found", total, None
                continue
            kind, value = read(idx)
            if kind == EMPTY:
                return "empty", total, idx
            total += value
            if kind == INC:
                return "found", total, None
        return "all", total, None

    def lookback(self, t, width):
        """Generator: yields while it waits; returns the exclusive prefix."""
        if t == 0:
            return 0
        excl = 0
        blk, tend = t // self.block, t - 1
        while True:
            while True:
                kind, s, _ = self.window(self.ticket_entry, tend, blk * self.block, width)
                if kind != "empty":
                    break
                yield
            excl += s
            if kind == "found":
                return excl
            bend = blk - 1
            while True:
                if bend < 0:
                    return excl
                kind, s, at = self.window(self.block_entry, bend, 0, width)
                yield
                excl += s
                if kind == "found":
                    return excl
                if kind == "empty":
                    blk, tend = at, at * self.block + self.block - 1
                    break
                bend -= width

    def ticket(self, t, width, result):
        """Generator: one ticket's life, one model step per yield."""
        yield
        b = t // self.block
        self.words[b][1] += 1          # the count and the aggregate, one atomic
        self.words[b][2] += self.aggs[t]
        yield
        self.state[t] = (INC if t == 0 else AGG, self.aggs[t])
        yield
        excl = yield from self.lookback(t, width)
        result[t] = excl
        self.state[t] = (INC, excl + self.aggs[t])
        if t % self.block == 0:
            yield
            self.words[b][0] += 1       # the flag and the block's exclusive prefix
            self.words[b][2] += excl


@pytest.mark.parametrize("seed", range(100))
def test_two_level_lookback_prefixes(seed):
    rng = random.Random(seed)
    n = rng.choice([1, 2, 5, 31, 32, 33, 64, 65, 200, 700, 1500])
    block, width = rng.choice([(4, 4), (8, 8), (8, 32), (32, 32), (128, 128)])
    inflight = rng.choice([1, 4, 16, 64, 300])
    aggs = [rng.choice([0, 0, 1, 2, 7, 1000, 2 ** 40]) for _ in range(n)]
    model = Model(aggs, block)
    result = [None] * n
    live, nxt, done = [], 0, 0
    while done < n:
        while nxt < n and len(live) < inflight:  # tickets are taken in order
            live.append(model.ticket(nxt, width, result))
            nxt += 1
        g = rng.choice(live)
        try:
            next(g)
        except StopIteration:
            live.remove(g)
            done += 1
    prefix = 0
    for t in range(n):
        assert result[t] == prefix, (t, result[t], prefix)
        prefix += aggs[t]
    # every block word ends full, and with the flag its inclusive prefix
    for b, (inc, count, value) in enumerate(model.words):
        size = min(block, n - b * block)
        assert count == size
        assert inc == 1 and value == sum(aggs[: b * block + size])
