"""A second, brute-force model of the swap-in policy for tiny inputs.

Written from the method's definition independently of the C++ oracle and with
different machinery: plain Python lists, linear scans instead of hash maps,
and repeated arg-min / arg-max selection instead of sorting.  It tracks only
the observable policy state per request (slot -> token, slot -> epoch,
position -> physical row, next epoch) and returns locations and counters.
Used only on tiny inputs, where its quadratic loops are cheap.

With an extra page of E rows (E > 0), a valid token on the same page as the
request's newest position (t // E == (limit - 1) // E) is served from row
R * (H + C) + q * E + t % E and touches nothing else.
"""
from __future__ import annotations

from typing import List


class ListCache:
    def __init__(self, H: int, C: int, E: int = 0, R: int = 0):
        self.H, self.C, self.E, self.R = H, C, E, R
        self.tok: List[int] = [-1] * H
        self.ep: List[int] = [-1] * H
        self.phys: List[int] = list(range(H + C))
        self.epoch = 0

    def slot_of(self, t: int) -> int:
        for v in range(self.H):
            if self.tok[v] == t:
                return v
        return -1

    def call(self, q: int, tokens_by_step: List[List[int]], limit: int):
        """One call for request q; returns (locations by step, counters)."""
        H, C = self.H, self.C
        base = q * (H + C)
        E = self.epoch
        misses: List[int] = []  # distinct missing tokens, first occurrence first
        last: List[int] = []  # last step of each miss
        hit_slots: List[int] = []
        locs = []
        hits = dups = invalid = extra = 0
        for s, row in enumerate(tokens_by_step):
            out = []
            for t in row:
                if t < 0 or t >= limit:
                    out.append(-1)
                    invalid += 1
                    continue
                if self.E and t // self.E == (limit - 1) // self.E:
                    out.append(self.R * (H + C) + q * self.E + t % self.E)
                    extra += 1
                    continue
                v = self.slot_of(t)
                if v >= 0:
                    hits += 1
                    if v not in hit_slots:
                        hit_slots.append(v)
                    out.append(base + self.phys[v])
                    continue
                if t in misses:
                    j = misses.index(t)
                    last[j] = s
                    dups += 1
                else:
                    misses.append(t)
                    last.append(s)
                    j = len(misses) - 1
                out.append(base + self.phys[H + j])
            locs.append(out)
        for v in hit_slots:
            self.ep[v] = E
        U = len(misses)
        m = min(U, H - len(hit_slots))
        # admission: repeatedly take the best remaining miss
        remaining = list(range(U))
        chosen = []
        for _ in range(m):
            best = remaining[0]
            for j in remaining[1:]:
                if last[j] > last[best]:
                    best = j
            remaining.remove(best)
            chosen.append(best)
        chosen.sort()
        # victims: repeatedly take the oldest remaining non-hit slot
        pool = [v for v in range(H) if v not in hit_slots]
        vict = []
        for _ in range(m):
            best = pool[0]
            for v in pool[1:]:
                if self.ep[v] < self.ep[best]:
                    best = v
            pool.remove(best)
            vict.append(best)
        vict.sort()
        evicted = 0
        for j, v in zip(chosen, vict):
            if self.tok[v] != -1:
                evicted += 1
            self.phys[v], self.phys[H + j] = self.phys[H + j], self.phys[v]
            self.tok[v] = misses[j]
            self.ep[v] = E
        self.epoch = E + 1
        stats = [hits, len(hit_slots), dups, U, m, evicted, U - m, invalid, extra]
        return locs, stats
