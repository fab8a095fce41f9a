"""Oracle of the adaptive runtime's policies (test infrastructure: only tests and the bench's reference
legs use it). Plain Python, written from "Magnitude: on-device AI-agent inference engine --
self-optimising scheduling and elastic memory pools":

* 3.1 load profile: a sliding window of the last `window` recorded inferences (default 64); one
  inference in `sample_every` is recorded (default 4, "sampling rate 1/4"); once the window is full,
  its P50 / P90 / P99 lengths drive the next decisions.
* 3.2 memory pool: the hot pool is slack (hot_pool_slack, default 1.2) times the KV need X of the
  window's P90 length.
* 3.3 fusion-plan switch: three preset plans; P90 below 128 selects the short plan, above 512 the long
  one (and between, the medium one).

Readings where the page is silent: the recorded inferences are the first and then every
sample_every-th (counts 0, r, 2r, ...); quantiles are nearest-rank (the ceil(q n)-th smallest value);
X counts whole 16-token blocks per open session and the hot size is rounded up to a whole block.
"""
from __future__ import annotations

import math
from collections import deque
from fractions import Fraction


class LoadWindow:
    """3.1: the profile's sliding window with its sampling."""

    def __init__(self, window: int = 64, sample_every: int = 4):
        assert window >= 1 and sample_every >= 1
        self.window, self.sample_every = window, sample_every
        self.seen = 0
        self.values: deque[int] = deque(maxlen=window)

    def observe(self, length: int) -> bool:
        take = self.seen % self.sample_every == 0
        self.seen += 1
        if take:
            self.values.append(int(length))
        return take

    def full(self) -> bool:
        return len(self.values) == self.window

    def quantile(self, q) -> int:
        """Nearest rank: the ceil(q n)-th smallest of the n values in the window; -1 when empty."""
        n = len(self.values)
        if n == 0:
            return -1
        rank = math.ceil(Fraction(str(q)) * n)
        rank = min(max(rank, 1), n)
        return sorted(self.values)[rank - 1]


def plan_for(p90: int, short_below: int = 128, long_above: int = 512) -> int:
    """3.3: 0 (short) when P90 < short_below, 2 (long) when P90 > long_above, else 1 (medium)."""
    if p90 < short_below:
        return 0
    if p90 > long_above:
        return 2
    return 1


def hot_pool_blocks(p90: int, n_sessions: int, slack="1.2", block_tokens: int = 16) -> int:
    """3.2: slack x X, X = the blocks of n_sessions sessions of the P90 length, rounded up."""
    if p90 <= 0 or n_sessions <= 0:
        return 0
    x = n_sessions * -(-p90 // block_tokens)
    return math.ceil(Fraction(str(slack)) * x)


class ElasticPoolModel:
    """3.2 (hot / cold pool) and 2.2 layer 1 (grow on demand, give idle memory back) on a block pool:
    groups of G blocks; the lowest `hot` groups stay mapped; another group is mapped when the free
    blocks run out (the lowest group not mapped) and unmapped once none of its blocks is in use; free
    blocks go out lowest id first. Reading: the group is the unit of mapping (whole pages per layer),
    the hot pool is at least one group."""

    def __init__(self, n_blocks: int, group_blocks: int):
        self.G = group_blocks
        self.n_groups = -(-n_blocks // group_blocks)
        self.P = self.n_groups * group_blocks
        self.hot = 1
        self.mapped: set[int] = set()
        self.free: set[int] = set()
        self.used = [0] * self.n_groups
        self._map(0)

    def _map(self, g):
        self.mapped.add(g)
        self.free.update(range(g * self.G, (g + 1) * self.G))

    def _unmap(self, g):
        self.mapped.discard(g)
        self.free.difference_update(range(g * self.G, (g + 1) * self.G))

    def available(self) -> int:
        return len(self.free) + self.G * (self.n_groups - len(self.mapped))

    def alloc(self, n: int):
        """n blocks, or None (and no change) when the pool can not hold them."""
        if n > self.available():
            return None
        g = 0
        while len(self.free) < n:
            if g not in self.mapped:
                self._map(g)
            g += 1
        out = []
        for _ in range(n):
            b = min(self.free)
            self.free.remove(b)
            self.used[b // self.G] += 1
            out.append(b)
        return out

    def release(self, blocks):
        for b in blocks:
            self.used[b // self.G] -= 1
            self.free.add(b)
        self.trim()

    def trim(self):
        for g in sorted(self.mapped):
            if g >= self.hot and self.used[g] == 0:
                self._unmap(g)

    def set_hot(self, blocks: int):
        self.hot = min(max(-(-blocks // self.G), 1), self.n_groups)
        for g in range(self.hot):
            if g not in self.mapped:
                self._map(g)
        self.trim()
