"""Shared helpers for the tests: host pools and oracle runs with checks."""
from __future__ import annotations

from typing import Dict

import numpy as np

import hs_workloads as W
from checker import check_call


def make_host_pool(R: int, L: int, width: int, layer: int) -> np.ndarray:
    pool = np.empty((R, L, width), dtype=np.uint8)
    W.fill_host_pool(pool, layer)
    return pool


def row_fn(layer: int, width: int):
    def host_row(q: int, toks: np.ndarray) -> np.ndarray:
        return W.host_rows(layer, np.full(toks.shape, q, dtype=np.int64), toks, width)
    return host_row


class OracleHarness:
    """Runs calls through the oracle and checks each one with the checker.

    Rows appended with `append` are remembered in a plain dict (the latest row
    of each (layer, q, t)), which the checks use as the expected host row in
    place of the generator's row."""

    def __init__(self, R, L, width, H, K, S_max, layers=1, lib=None, extra_page=0):
        from oracle import Oracle
        self.o = Oracle(R, L, width, H, K, S_max, layers, lib=lib, extra_page_size=extra_page)
        self.R, self.L, self.W, self.H, self.K, self.S_max = R, L, width, H, K, S_max
        self.C = S_max * K
        self.E = extra_page
        self.layers = layers
        self.pools = [make_host_pool(R, L, width, l) for l in range(layers)]
        self.dev = [np.zeros((R * (H + self.C + extra_page), width), dtype=np.uint8)
                    for _ in range(layers)]
        self.latest: Dict[tuple, np.ndarray] = {}

    def host_row(self, layer: int):
        gen = row_fn(layer, self.W)

        def rows(q: int, toks: np.ndarray) -> np.ndarray:
            out = gen(q, np.asarray(toks))
            for i, t in enumerate(np.asarray(toks).tolist()):
                r = self.latest.get((layer, q, int(t)))
                if r is not None:
                    out[i] = r
            return out
        return rows

    def append(self, req, tok, seq_lens, rows, layer=0) -> int:
        """Write-back through the oracle; returns the number of skipped entries."""
        skipped = self.o.append_rows(layer, self.pools[layer], self.dev[layer], req, tok,
                                     seq_lens, rows)
        for q, t, n, r in zip(np.asarray(req).tolist(), np.asarray(tok).tolist(),
                              np.asarray(seq_lens).tolist(), np.asarray(rows)):
            if 0 <= q < self.R and 0 <= t < min(n, self.L):
                self.latest[(layer, q, t)] = np.array(r, dtype=np.uint8)
        return skipped

    def states(self, layer: int) -> Dict[int, dict]:
        return {q: self.o.request_state(layer, q) for q in range(self.R)}

    def call(self, topk, rpi, seq_lens, layer=0, check=True, want_plan=False, threads=1):
        before = self.states(layer) if check else None
        out = self.o.swap_in(layer, self.pools[layer], self.dev[layer], rpi, seq_lens, topk,
                             want_plan=want_plan, num_threads=threads)
        if check:
            after = self.states(layer)
            dev = self.dev[layer]
            check_call(before, after, np.asarray(topk), np.asarray(rpi), np.asarray(seq_lens),
                       self.L, self.H, self.C, out["locs"], out["stats"],
                       rows_at=lambda locs: dev[locs], host_row=self.host_row(layer),
                       extra_page=self.E, R=self.R)
            out["before"], out["after"] = before, after
        return out
