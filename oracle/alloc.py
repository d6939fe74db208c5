"""Page allocator mirror (oracle; test infrastructure).

[MTP] section "The Serving System": the INT2 mode stays compatible with paged
attention; [MTP] Visual Explainer step 5 / [MS] section "评估结果": prefix
caching and radix reuse keep working, i.e. prefix pages are shared.

Reading (the pages give no allocator): physical page ids 0..P-1 are handed out
from a stack whose initial pop order is a seeded permutation -- Fisher-Yates
from the identity, i = P-1 down to 1, j = next() mod (i+1), next() being
SplitMix64 -- or the identity when the seed is 0.  Freed pages go back on top
(last freed, first reused).  Pages carry reference counts; a page returns to
the stack when its count drops to zero.  Pinned by permutation / uniformity
tests (a Sattolo-style off-by-one would only make cyclic permutations).
"""
from __future__ import annotations

MASK64 = (1 << 64) - 1


class SplitMix64:
    """SplitMix64 generator (Steele, Lea, Flood 2014), 64-bit state."""

    def __init__(self, seed: int):
        self.state = seed & MASK64

    def next(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)


def seeded_order(n: int, seed: int) -> list[int]:
    """Pop order of a fresh allocator over n pages."""
    a = list(range(n))
    if seed:
        g = SplitMix64(seed)
        for i in range(n - 1, 0, -1):
            j = g.next() % (i + 1)
            a[i], a[j] = a[j], a[i]
    return a


class PagePool:
    def __init__(self, n: int, seed: int):
        self.n = n
        self.stack = list(reversed(seeded_order(n, seed)))
        self.refs = [0] * n

    def alloc(self) -> int:
        if not self.stack:
            raise MemoryError("out of pages")
        p = self.stack.pop()
        self.refs[p] = 1
        return p

    def share(self, p: int) -> None:
        assert self.refs[p] > 0
        self.refs[p] += 1

    def release(self, p: int) -> None:
        assert self.refs[p] > 0
        self.refs[p] -= 1
        if self.refs[p] == 0:
            self.stack.append(p)

    @property
    def free_count(self) -> int:
        return len(self.stack)
