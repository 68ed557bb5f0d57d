"""Property checks of one swap-in call, written from the method's definition.

These checks do not re-run the swap-in.  Given the policy state of every
request before and after a call, the call's inputs and its outputs, they
verify properties that any correct implementation must satisfy:

  I1  every returned location holds that token's host row;
  I2  within a request's call, equal tokens share a location and distinct
      tokens get distinct locations;
  I3  the unique-miss count equals the number of distinct valid tokens that
      were not resident before the call;
  I4  at most H tokens are resident per request;
  I5  every resident token's device row holds its host row (after the call);
  I6  the position -> physical-row table is a permutation of 0..H+C-1;
  I7  without overflow every valid token is resident after the call; with
      overflow every hit token stays resident;
and the policy the build fixes where the pages leave it open (the
multi-step swap report, sections 实现拆解 item 1 and 风险与影响):
  P1  hot slots referenced by the call take the call's epoch;
  P2  victims are the m non-hit slots with the smallest (epoch, slot) pairs,
      stated as: every victim's pair is below every surviving non-hit
      slot's pair;
  P3  with overflow, every admitted miss ranks above every non-admitted miss
      under (last occurrence step descending, first occurrence ascending);
  P4  admitted misses in first-occurrence order occupy ascending slots;
  P5  rotation: an admitted token's hot slot maps to the very row the call
      returned for it, so locations stay valid after the commit;
and, with an extra page of E rows per request (the newest, still-filling
page, looked up before the hot cache: same report, 实现拆解 item 1):
  X1  a valid token in [floor((n - 1) / E) * E, n), n = min(seq_len, L_max),
      gets row R * (H + C) + q * E + t mod E, and takes no part in hits,
      misses, admission or the state.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional

import numpy as np

STAT = {n: i for i, n in enumerate(("hits", "hit_slots", "dup_misses", "unique_misses",
                                    "admitted", "evicted", "overflow", "invalid", "extra"))}


class CheckError(AssertionError):
    pass


def _fail(msg: str):
    raise CheckError(msg)


def resident_map(tok: np.ndarray) -> Dict[int, int]:
    return {int(t): v for v, t in enumerate(tok.tolist()) if t != -1}


def check_state(st: dict, H: int, C: int, who: str = "") -> None:
    tok, ep, phys = st["tok"], st["ep"], st["phys"]
    if sorted(phys.tolist()) != list(range(H + C)):
        _fail("%s I6: phys is not a permutation" % who)
    live = tok[tok != -1]
    if live.size > H:
        _fail("%s I4: %d resident > H=%d" % (who, live.size, H))
    if np.unique(live).size != live.size:
        _fail("%s: a token is resident in two slots" % who)
    if ((tok == -1) != (ep == -1)).any():
        _fail("%s: empty slots and never-referenced slots disagree" % who)
    if (ep >= st["epoch"]).any():
        _fail("%s: an epoch is not older than the request's next epoch" % who)


def check_call(before: Dict[int, dict], after: Dict[int, dict], topk: np.ndarray,
               rpi: np.ndarray, seq_lens: np.ndarray, L_max: int, H: int, C: int,
               locs: np.ndarray, stats: Optional[np.ndarray] = None,
               rows_at: Optional[Callable[[np.ndarray], np.ndarray]] = None,
               host_row: Optional[Callable[[int, np.ndarray], np.ndarray]] = None,
               extra_page: int = 0, R: int = 0) -> None:
    """Check one call.  `before`/`after` map request q -> state dict.

    rows_at(locs) returns device rows uint8 [n, W] after the call;
    host_row(q, tokens) returns the expected host rows uint8 [n, W];
    extra_page is the extra page size (0: none), R the request-pool size.
    """
    B, S, K = topk.shape
    Ex = extra_page
    for b in range(B):
        q = int(rpi[b])
        pre, post = before[q], after[q]
        who = "request %d (q=%d)" % (b, q)
        check_state(post, H, C, who)
        base = q * (H + C)
        limit = min(int(seq_lens[b]), L_max)
        t_flat = topk[b].reshape(-1).astype(np.int64)
        l_flat = locs[b].reshape(-1).astype(np.int64)
        valid = (t_flat >= 0) & (t_flat < limit)
        if (l_flat[~valid] != -1).any():
            _fail("%s: invalid entry got a location" % who)
        # X1: entries on the extra page.
        extra = np.zeros_like(valid)
        if Ex > 0 and limit > 0:
            extra = valid & (t_flat >= (limit - 1) // Ex * Ex)
            want = R * (H + C) + q * Ex + t_flat[extra] % Ex
            if (l_flat[extra] != want).any():
                _fail("%s X1: an extra-page token is not at its extra row" % who)
        if rows_at is not None and host_row is not None and extra.any():
            xt = np.unique(t_flat[extra])
            got = rows_at(R * (H + C) + q * Ex + xt % Ex)
            if (got != host_row(q, xt)).any():
                _fail("%s I1: an extra-page row differs from the host row" % who)
        n_extra = int(extra.sum())
        valid = valid & ~extra
        res_pre = resident_map(pre["tok"])
        res_post = resident_map(post["tok"])
        vt = t_flat[valid]
        vl = l_flat[valid]
        # I2: the map token -> location is well defined and injective.
        tl = {}
        for t, l in zip(vt.tolist(), vl.tolist()):
            if tl.setdefault(t, l) != l:
                _fail("%s I2: token %d got two locations" % (who, t))
        if len(set(tl.values())) != len(tl):
            _fail("%s I2: two tokens share a location" % who)
        if any(not (base <= l < base + H + C) for l in tl.values()):
            _fail("%s: location outside the request's rows" % who)
        # Hits resolve to the hot slot's row; misses land in the scratch ring.
        scratch_rows = set((base + pre["phys"][H:]).tolist())
        hit_slots = set()
        for t, l in tl.items():
            if t in res_pre:
                v = res_pre[t]
                hit_slots.add(v)
                if l != base + pre["phys"][v]:
                    _fail("%s: hit token %d not at its hot row" % (who, t))
            elif l not in scratch_rows:
                _fail("%s: miss token %d not in the scratch ring" % (who, t))
        # I3: unique misses.
        order: List[int] = []
        last_step: Dict[int, int] = {}
        for i, t in enumerate(t_flat.tolist()):
            if valid[i] and t not in res_pre:
                if t not in last_step:
                    order.append(t)
                last_step[t] = i // K
        U = len(order)
        # Misses in first-occurrence order fill the scratch ring in order.
        for j, t in enumerate(order):
            if tl[t] != base + pre["phys"][H + j]:
                _fail("%s: miss %d (token %d) not at scratch position %d" % (who, j, t, j))
        # I1: rows.
        if rows_at is not None and host_row is not None and tl:
            toks = np.fromiter(tl.keys(), dtype=np.int64)
            got = rows_at(np.fromiter(tl.values(), dtype=np.int64))
            exp = host_row(q, toks)
            bad = np.nonzero((got != exp).any(axis=1))[0]
            if bad.size:
                _fail("%s I1: %d returned rows differ (first token %d)" % (who, bad.size,
                                                                          int(toks[bad[0]])))
        # P1: referenced hot slots take the call's epoch.
        E = pre["epoch"]
        if post["epoch"] != E + 1:
            _fail("%s: epoch did not advance by one" % who)
        for v in hit_slots:
            if post["ep"][v] != E or post["tok"][v] != pre["tok"][v]:
                _fail("%s P1: hit slot %d not marked or not kept" % (who, v))
        cap = H - len(hit_slots)
        m = min(U, cap)
        admitted = [t for t in order if t in res_post]
        if len(admitted) != m:
            _fail("%s: admitted %d misses, expected min(U=%d, cap=%d)" % (who, len(admitted), U,
                                                                          cap))
        # I7.
        if U <= cap:
            if any(t not in res_post for t in tl):
                _fail("%s I7: a token of the call is not resident after it" % who)
        elif any(t not in res_post for t in tl if t in res_pre):
            _fail("%s I7: a hit token was evicted" % who)
        # P3: admission ranking under overflow.
        if U > cap and m > 0:
            rank = {t: (-last_step[t], j) for j, t in enumerate(order)}
            adm_worst = max(rank[t] for t in admitted)
            rest = [rank[t] for t in order if t not in res_post]
            if rest and min(rest) < adm_worst:
                _fail("%s P3: a better-ranked miss was not admitted" % who)
        # P2: victim selection, and which slots changed.
        victims = [res_post[t] for t in admitted]
        vset = set(victims)
        if vset & hit_slots:
            _fail("%s: a hit slot was chosen as a victim" % who)
        if vset:
            worst = max((int(pre["ep"][v]), v) for v in vset)
            for v in range(H):
                if v not in vset and v not in hit_slots and (int(pre["ep"][v]), v) < worst:
                    _fail("%s P2: slot %d is older than a victim but survived" % (who, v))
        # P4: pairing order.
        if victims != sorted(victims):
            _fail("%s P4: admitted misses do not occupy ascending slots" % who)
        # P5: rotation keeps returned locations valid; untouched slots unchanged.
        for t in admitted:
            v = res_post[t]
            if base + post["phys"][v] != tl[t]:
                _fail("%s P5: admitted token %d's hot row is not its returned row" % (who, t))
            if post["ep"][v] != E:
                _fail("%s: admitted slot %d not stamped with the call's epoch" % (who, v))
        for v in range(H):
            if v in vset or v in hit_slots:
                continue
            if (post["tok"][v] != pre["tok"][v] or post["ep"][v] != pre["ep"][v]
                    or post["phys"][v] != pre["phys"][v]):
                _fail("%s: untouched slot %d changed" % (who, v))
        # I5 after the call, for every resident token.
        if rows_at is not None and host_row is not None and res_post:
            toks = np.fromiter(res_post.keys(), dtype=np.int64)
            slots = np.fromiter(res_post.values(), dtype=np.int64)
            got = rows_at(base + post["phys"][slots].astype(np.int64))
            exp = host_row(q, toks)
            bad = np.nonzero((got != exp).any(axis=1))[0]
            if bad.size:
                _fail("%s I5: %d resident rows corrupted" % (who, bad.size))
        # Counters.
        if stats is not None:
            st = stats[b]
            n_valid = int(valid.sum())
            hits = sum(1 for t in vt.tolist() if t in res_pre)
            evicted = sum(1 for v in vset if pre["tok"][v] != -1)
            exp = {"hits": hits, "hit_slots": len(hit_slots), "dup_misses": n_valid - hits - U,
                   "unique_misses": U, "admitted": m, "evicted": evicted, "overflow": U - m,
                   "invalid": int((~valid).sum()) - n_extra, "extra": n_extra}
            for name, val in exp.items():
                if int(st[STAT[name]]) != val:
                    _fail("%s: stat %s = %d, expected %d" % (who, name, int(st[STAT[name]]), val))
