"""Pins of the CPU oracle against facts that do not come from the oracle.

Each routine takes a loaded oracle library (so that the mutation test can
run the same pins against deliberately broken builds) and raises
AssertionError on a mismatch.

  pin_lru:            with one token per call, epoch-CLOCK with a lowest-slot
                      tie-break must equal textbook LRU (an OrderedDict);
  pin_first_call:     closed forms of the first call on an empty cache,
                      including its miss plan;
  pin_repeat_call:    repeating a call that fits is all hits, same locations;
  pin_invariants:     random tiny sweeps checked with the property checker;
  pin_simulator:      random tiny sweeps equal the brute-force list model;
  pin_overflow:       overflow cases checked with the property checker;
  pin_782:            the multi-step report's test shape: 782 cross-step
                      unique misses at batch 1 (section 实现拆解 item 4);
  pin_page_table:     sparse page table equals np.unique of the pages;
  pin_extra_simulator: with an extra page, random tiny sweeps equal the
                      brute-force list model (which finds the page by page
                      index, not by its first position);
  pin_extra_reduction: an extra-page cache behaves exactly like a cache
                      without one that is shown the same calls with the
                      extra-page entries blanked out;
  pin_reset:          random calls over two layers with requests reset in
                      between equal the brute-force list model, in which a
                      reset request simply starts a new empty cache in every
                      layer (other requests untouched);
  pin_append_decode:  a decode loop that appends every new token's row and
                      rewrites some older ones: every returned row and
                      every resident row equals the latest row written for
                      its (request, token) in a plain dict, and so does the
                      host pool.
"""
from __future__ import annotations

from collections import OrderedDict

import numpy as np

from common import OracleHarness
from simulator import ListCache

WIDTH = 32  # tiny rows for the CPU pins (the real rows are 656 bytes)


def pin_lru(lib, trials: int = 12, calls: int = 120) -> None:
    rng = np.random.default_rng(7)
    for trial in range(trials):
        H = int(rng.integers(1, 9))
        universe = int(rng.integers(H + 1, 3 * H + 4))
        h = OracleHarness(1, 64, WIDTH, H, 1, 1, lib=lib)
        lru = OrderedDict()
        for c in range(calls):
            t = int(rng.integers(0, universe))
            out = h.call(np.array([[[t]]], np.int32), np.array([0], np.int32),
                         np.array([64], np.int32))
            hit = t in lru
            st = out["stats"][0]
            assert st[0] == int(hit), "LRU hit/miss differs at call %d" % c
            if hit:
                lru.move_to_end(t)
            else:
                if len(lru) == H:
                    lru.popitem(last=False)
                lru[t] = None
            res = set(int(x) for x in out["after"][0]["tok"] if x != -1)
            assert res == set(lru), "resident set differs from LRU at call %d" % c


def pin_first_call(lib) -> None:
    rng = np.random.default_rng(11)
    for trial in range(20):
        R, H, K, S = 3, int(rng.integers(4, 40)), int(rng.integers(1, 9)), int(rng.integers(1, 5))
        C = S * K
        L = 50
        h = OracleHarness(R, L, WIDTH, H, K, S, lib=lib)
        topk = rng.integers(-3, L + 3, size=(2, S, K)).astype(np.int32)
        rpi = np.array([2, 0], np.int32)
        sl = np.array([L, 30], np.int32)
        out = h.call(topk, rpi, sl, want_plan=True)
        for b in range(2):
            q = int(rpi[b])
            flat = topk[b].reshape(-1)
            valid = [t for t in flat.tolist() if 0 <= t < sl[b]]
            distinct = list(dict.fromkeys(valid))
            assert out["stats"][b][3] == len(distinct)
            # the miss plan: host row (q, t_j) -> scratch row j, one per unique miss
            U = len(distinct)
            assert out["miss_count"][b] == U
            assert out["miss_src"][b][:U].tolist() == [q * L + t for t in distinct]
            assert out["miss_dst"][b][:U].tolist() == [q * (H + C) + H + j for j in range(U)]
            first = {t: j for j, t in enumerate(distinct)}
            for i, t in enumerate(flat.tolist()):
                want = q * (H + C) + H + first[t] if t in first else -1
                assert out["locs"][b].reshape(-1)[i] == want
            st = out["after"][q]
            m = min(len(distinct), H)
            # empty slots have the oldest mark, so the first m slots take misses 0..m-1
            assert st["tok"][:m].tolist() == distinct[:m] or len(distinct) > H
            if len(distinct) <= H:
                assert (st["tok"][m:] == -1).all()


def pin_repeat_call(lib) -> None:
    rng = np.random.default_rng(13)
    for trial in range(20):
        H, K, S = int(rng.integers(8, 40)), int(rng.integers(1, 9)), int(rng.integers(1, 5))
        h = OracleHarness(2, 64, WIDTH, H, K, S, lib=lib)
        topk = rng.integers(0, 64, size=(2, S, K)).astype(np.int32)
        rpi = np.array([1, 0], np.int32)
        sl = np.array([64, 64], np.int32)
        first = h.call(topk, rpi, sl)
        again = h.call(topk, rpi, sl)
        for b in range(2):
            if first["stats"][b][3] <= H:
                assert again["stats"][b][3] == 0
                assert (again["locs"][b] == first["locs"][b]).all()


def _random_call(rng, B, R, S, K, L):
    topk = rng.integers(-2, L + 2, size=(B, S, K)).astype(np.int32)
    # bias towards reuse so that hits, duplicates and evictions all occur
    small = rng.integers(0, max(2, L // 3), size=(B, S, K)).astype(np.int32)
    pick = rng.random((B, S, K)) < 0.5
    topk[pick] = small[pick]
    rpi = rng.permutation(R)[:B].astype(np.int32)
    sl = rng.integers(max(1, L // 2), L + 3, size=B).astype(np.int32)
    return topk, rpi, sl


def pin_invariants(lib, trials: int = 25, calls: int = 6) -> None:
    rng = np.random.default_rng(17)
    for trial in range(trials):
        H = int(rng.integers(1, 9))
        K = int(rng.integers(1, 9))
        S_max = int(rng.integers(1, 5))
        R = int(rng.integers(1, 4))
        L = 16
        h = OracleHarness(R, L, WIDTH, H, K, S_max, layers=2, lib=lib)
        for c in range(calls):
            B = int(rng.integers(1, R + 1))
            S = int(rng.integers(1, S_max + 1))
            layer = int(rng.integers(0, 2))
            topk, rpi, sl = _random_call(rng, B, R, S, K, L)
            h.call(topk, rpi, sl, layer=layer)


def pin_simulator(lib, trials: int = 25, calls: int = 8) -> None:
    rng = np.random.default_rng(19)
    for trial in range(trials):
        H = int(rng.integers(1, 9))
        K = int(rng.integers(1, 9))
        S_max = int(rng.integers(1, 5))
        R = int(rng.integers(1, 4))
        L = 16
        h = OracleHarness(R, L, WIDTH, H, K, S_max, lib=lib)
        sims = [ListCache(H, S_max * K) for _ in range(R)]
        for c in range(calls):
            B = int(rng.integers(1, R + 1))
            S = int(rng.integers(1, S_max + 1))
            topk, rpi, sl = _random_call(rng, B, R, S, K, L)
            out = h.call(topk, rpi, sl, check=False)
            for b in range(B):
                q = int(rpi[b])
                locs, stats = sims[q].call(q, topk[b].tolist(), min(int(sl[b]), L))
                assert out["locs"][b].tolist() == locs, "locations differ from the list model"
                assert out["stats"][b].tolist() == stats, "counters differ from the list model"
                st = h.o.request_state(0, q)
                assert st["tok"].tolist() == sims[q].tok
                assert st["ep"].tolist() == sims[q].ep
                assert st["phys"].tolist() == sims[q].phys
                assert st["epoch"] == sims[q].epoch


def pin_reset(lib, trials: int = 12, calls: int = 10) -> None:
    rng = np.random.default_rng(29)
    for trial in range(trials):
        H = int(rng.integers(1, 7))
        K = int(rng.integers(1, 7))
        S_max = int(rng.integers(1, 4))
        R = int(rng.integers(2, 5))
        L = 16
        h = OracleHarness(R, L, WIDTH, H, K, S_max, layers=2, lib=lib)
        sims = {(l, q): ListCache(H, S_max * K) for l in range(2) for q in range(R)}
        for c in range(calls):
            if c and rng.random() < 0.4:
                gone = rng.permutation(R)[:int(rng.integers(1, R))].astype(np.int32)
                h.o.reset_requests(gone)
                for q in gone.tolist():
                    for l in range(2):
                        sims[(l, q)] = ListCache(H, S_max * K)
            B = int(rng.integers(1, R + 1))
            S = int(rng.integers(1, S_max + 1))
            layer = int(rng.integers(0, 2))
            topk, rpi, sl = _random_call(rng, B, R, S, K, L)
            out = h.call(topk, rpi, sl, layer=layer, check=False)
            for b in range(B):
                q = int(rpi[b])
                locs, stats = sims[(layer, q)].call(q, topk[b].tolist(), min(int(sl[b]), L))
                assert out["locs"][b].tolist() == locs, "locations differ after a reset"
                assert out["stats"][b].tolist() == stats, "counters differ after a reset"
            for l in range(2):
                for q in range(R):
                    st = h.o.request_state(l, q)
                    assert st["tok"].tolist() == sims[(l, q)].tok
                    assert st["ep"].tolist() == sims[(l, q)].ep
                    assert st["phys"].tolist() == sims[(l, q)].phys
                    assert st["epoch"] == sims[(l, q)].epoch


def pin_overflow(lib) -> None:
    rng = np.random.default_rng(23)
    seen_overflow = 0
    for trial in range(30):
        H = int(rng.integers(1, 6))
        K = int(rng.integers(2, 9))
        S = int(rng.integers(2, 5))
        h = OracleHarness(2, 40, WIDTH, H, K, S, lib=lib)
        for c in range(5):
            topk = rng.integers(0, 40, size=(2, S, K)).astype(np.int32)
            out = h.call(topk, np.array([0, 1], np.int32), np.array([40, 40], np.int32))
            seen_overflow += int((out["stats"][:, 6] > 0).sum())
    assert seen_overflow > 20


def _steps_with_union(rng, S, K, union, universe):
    """S distinct-per-step rows of K tokens whose union has exactly `union` tokens."""
    assert K <= union <= S * K
    pool = rng.permutation(universe)[:union]
    steps = [pool[:K].copy()]
    used = K
    for s in range(1, S):
        left = S - s  # steps still to fill, including this one
        # spread the remaining new tokens evenly over the remaining steps
        new = min(K, -(-(union - used) // left))
        fresh = pool[used:used + new]
        used += new
        old = rng.choice(pool[:used - new], size=K - new, replace=False)
        row = np.concatenate([fresh, old])
        rng.shuffle(row)
        steps.append(row)
    assert used == union
    return np.stack(steps).astype(np.int32)


def pin_782(lib) -> None:
    rng = np.random.default_rng(782)
    S, K, H = 4, 256, 1024
    h = OracleHarness(1, 4096, WIDTH, H, K, S, lib=lib)
    topk = _steps_with_union(rng, S, K, 782, 4096)[None]
    out = h.call(topk, np.array([0], np.int32), np.array([4096], np.int32))
    st = out["stats"][0]
    assert st[3] == 782 and st[2] == S * K - 782 and st[0] == 0
    again = h.call(topk, np.array([0], np.int32), np.array([4096], np.int32))
    assert again["stats"][0][0] == S * K and again["stats"][0][3] == 0


def pin_page_table(lib) -> None:
    from oracle import page_table
    rng = np.random.default_rng(29)
    for trial in range(30):
        B, S, K = int(rng.integers(1, 4)), int(rng.integers(1, 5)), int(rng.integers(1, 40))
        P = int(rng.integers(1, 20))
        L = int(rng.integers(1, 300))
        topk = rng.integers(-3, L + 5, size=(B, S, K)).astype(np.int32)
        sl = rng.integers(1, L + 8, size=B).astype(np.int32)
        L_max = int(rng.integers(1, L + 1))
        pages, num, tp = page_table(topk, sl, P, max_seq_len=L_max, lib=lib)
        for b in range(B):
            flat = topk[b].reshape(-1)
            valid = (flat >= 0) & (flat < min(sl[b], L_max))
            want = np.unique(flat[valid] // P)
            assert num[b] == want.size
            assert (pages[b, :want.size] == want).all() and (pages[b, want.size:] == -1).all()
            idx = np.searchsorted(want, flat // P)
            exp = np.where(valid, idx * P + flat % P, -1)
            assert (tp[b].reshape(-1) == exp).all()


def pin_extra_simulator(lib, trials: int = 30, calls: int = 8) -> None:
    rng = np.random.default_rng(41)
    for trial in range(trials):
        H = int(rng.integers(1, 9))
        K = int(rng.integers(1, 9))
        S_max = int(rng.integers(1, 5))
        R = int(rng.integers(1, 4))
        E = int(rng.integers(1, 7))
        L = 16
        h = OracleHarness(R, L, WIDTH, H, K, S_max, lib=lib, extra_page=E)
        sims = [ListCache(H, S_max * K, E, R) for _ in range(R)]
        for c in range(calls):
            B = int(rng.integers(1, R + 1))
            S = int(rng.integers(1, S_max + 1))
            topk, rpi, sl = _random_call(rng, B, R, S, K, L)
            # lengths that end on, just after and inside a page all occur
            sl = rng.integers(1, L + 2, size=B).astype(np.int32)
            out = h.call(topk, rpi, sl, check=False)
            for b in range(B):
                q = int(rpi[b])
                locs, stats = sims[q].call(q, topk[b].tolist(), min(int(sl[b]), L))
                assert out["locs"][b].tolist() == locs, "extra page: locations differ"
                assert out["stats"][b].tolist() == stats, "extra page: counters differ"
                st = h.o.request_state(0, q)
                assert st["tok"].tolist() == sims[q].tok
                assert st["ep"].tolist() == sims[q].ep
                assert st["phys"].tolist() == sims[q].phys


def pin_extra_reduction(lib, trials: int = 12, calls: int = 6) -> None:
    rng = np.random.default_rng(43)
    for trial in range(trials):
        H, K, S_max, R = int(rng.integers(2, 12)), int(rng.integers(2, 9)), 3, 3
        E = int(rng.integers(1, 9))
        L = 24
        with_x = OracleHarness(R, L, WIDTH, H, K, S_max, lib=lib, extra_page=E)
        plain = OracleHarness(R, L, WIDTH, H, K, S_max, lib=lib)
        for c in range(calls):
            B = int(rng.integers(1, R + 1))
            S = int(rng.integers(1, S_max + 1))
            topk, rpi, sl = _random_call(rng, B, R, S, K, L)
            a = with_x.call(topk, rpi, sl, check=False)
            blank = topk.copy()
            for b in range(B):
                n = min(int(sl[b]), L)
                on_page = (topk[b] >= 0) & (topk[b] < n) & (topk[b] // E == (n - 1) // E)
                blank[b][on_page] = -1
            p = plain.call(blank, rpi, sl, check=False)
            kept = blank >= 0
            assert (a["locs"][kept] == p["locs"][kept]).all(), "non-extra locations differ"
            sa, sp = a["stats"], p["stats"]
            assert (sa[:, :7] == sp[:, :7]).all(), "policy counters differ"
            assert (sa[:, 7] + sa[:, 8] == sp[:, 7]).all(), "extra + invalid != blanked"
            for q in range(R):
                x, y = with_x.o.request_state(0, q), plain.o.request_state(0, q)
                for k in ("tok", "ep", "phys"):
                    assert (x[k] == y[k]).all(), "state %s differs" % k


def pin_append_decode(lib, trials: int = 6, steps: int = 24) -> None:
    rng = np.random.default_rng(47)
    for trial in range(trials):
        R, H, K, S_max = 3, int(rng.integers(2, 10)), int(rng.integers(2, 7)), 2
        E = int(rng.integers(1, 6))
        L = 64
        h = OracleHarness(R, L, WIDTH, H, K, S_max, lib=lib, extra_page=E)
        n = rng.integers(4, 20, size=R).astype(np.int32)
        # prefill: the still-filling page of each request is written once
        for q in range(R):
            toks = np.arange((n[q] - 1) // E * E, n[q], dtype=np.int32)
            rows = rng.integers(0, 256, size=(toks.size, WIDTH), dtype=np.uint8)
            assert h.append(np.full(toks.size, q, np.int32), toks, np.full(toks.size, n[q]),
                            rows) == 0
        for step in range(steps):
            # decode appends one token per request, plus a rewrite of an older one
            n = np.minimum(n + 1, L).astype(np.int32)
            req = np.arange(R, dtype=np.int32)
            tok = n - 1
            old = rng.integers(0, n).astype(np.int32)
            req2 = np.concatenate([req, req])
            tok2 = np.concatenate([tok, old])
            keep = np.ones(2 * R, bool)
            keep[R:] = old != tok  # one row per (request, token) per call
            rows = rng.integers(0, 256, size=(2 * R, WIDTH), dtype=np.uint8)
            assert h.append(req2[keep], tok2[keep], np.concatenate([n, n])[keep],
                            rows[keep]) == 0
            # an out-of-range entry is skipped
            assert h.append(np.array([0], np.int32), np.array([n[0]], np.int32),
                            np.array([n[0]], np.int32), rows[:1]) == 1
            S = int(rng.integers(1, S_max + 1))
            recent = (n[:, None, None] - 1 - rng.integers(0, 3 * E + 2, size=(R, S, K)))
            spread = rng.integers(0, n[:, None, None], size=(R, S, K))
            topk = np.where(rng.random((R, S, K)) < 0.5, recent, spread).astype(np.int32)
            h.call(topk, req, n)
        for (layer, q, t), r in h.latest.items():
            assert (h.pools[layer][q, t] == r).all(), "host pool row not written back"


ALL_PINS = (pin_lru, pin_first_call, pin_repeat_call, pin_invariants, pin_simulator,
            pin_overflow, pin_782, pin_page_table, pin_extra_simulator, pin_extra_reduction,
            pin_append_decode, pin_reset)
