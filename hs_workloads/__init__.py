"""Seeded synthetic inputs for the decode KV swap-in.

This module only draws inputs: top-k index streams, request-pool indices,
sequence lengths and the byte content of host KV rows.  It holds none of the
swap-in's own arithmetic (no lookup, dedup, eviction or location numbering),
so both the CPU oracle and the CUDA path can consume it without sharing any
of the method's code.

Workloads restate the test and benchmark shapes of the HiSparse write-ups:
  * "[HiSparse] Support hisparse multi-step swap io kernel" (PR #32162
    report), section 实现拆解 item 4: a CUDA-Graph benchmark of 4-step versus
    sequential swap at batch 64, and a test with cross-step duplicate misses;
  * the same report, section 风险与影响: 782 cross-step unique misses at
    batch 1, the 32768 hot-buffer bound, steps 2 and 3;
  * "SGLang HiSparse: 当稀疏注意力从算法变为系统组件", section 4.1: 256-token
    pages and clustered top-k selections.
The pages print no input data, so every stream here is synthetic.

KV rows are 656 bytes (the item size of the pages' MLA pool).  Row content is
counter-based: 8-byte word w of row (layer, q, t) is output number
``row_counter(layer, q, t) + w`` of SplitMix64 seeded with 0 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014), so any
row can be re-derived without a stored copy.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

ROW_BYTES = 656  # item_size_bytes of the pages' MLA KV rows (41 x 16 B)

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


def splitmix64_at(n: np.ndarray) -> np.ndarray:
    """Output number n (0-based) of SplitMix64 seeded with state 0.

    The generator adds the golden gamma to its state and then mixes the
    state; output n therefore mixes (n + 1) * gamma (mod 2**64).
    """
    with np.errstate(over="ignore"):
        z = (np.asarray(n, dtype=np.uint64) + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        return z ^ (z >> np.uint64(31))


def row_counter(layer, q, t) -> np.ndarray:
    """First SplitMix64 counter of row (layer, q, t): 256 counters per row."""
    layer = np.asarray(layer, dtype=np.uint64)
    q = np.asarray(q, dtype=np.uint64)
    t = np.asarray(t, dtype=np.uint64)
    return (layer << np.uint64(56)) | (q << np.uint64(36)) | (t << np.uint64(8))


def host_rows(layer: int, q, t, width: int = ROW_BYTES) -> np.ndarray:
    """Bytes of host KV rows (layer, q[i], t[i]) as uint8 [n, width]."""
    assert width % 8 == 0 and width // 8 <= 256
    q = np.atleast_1d(np.asarray(q, dtype=np.int64))
    t = np.atleast_1d(np.asarray(t, dtype=np.int64))
    q, t = np.broadcast_arrays(q, t)
    assert layer < 256 and (q < (1 << 20)).all() and (t < (1 << 28)).all()
    base = row_counter(layer, q, t)[:, None]
    words = splitmix64_at(base + np.arange(width // 8, dtype=np.uint64)[None, :])
    return words.view(np.uint8).reshape(q.shape[0], width)


def _mix_inplace(z: np.ndarray) -> None:
    """In-place SplitMix64 output function of counters z (uint64 array)."""
    tmp = np.empty_like(z)
    with np.errstate(over="ignore"):
        z += np.uint64(1)
        z *= _GAMMA
        np.right_shift(z, np.uint64(30), out=tmp)
        z ^= tmp
        z *= _MIX1
        np.right_shift(z, np.uint64(27), out=tmp)
        z ^= tmp
        z *= _MIX2
        np.right_shift(z, np.uint64(31), out=tmp)
        z ^= tmp


def fill_host_pool(pool: np.ndarray, layer: int, chunk_rows: int = 1 << 14,
                   threads: Optional[int] = None) -> None:
    """Fill a host pool view uint8 [R, L, W] with rows (layer, q, t).

    Same bytes as host_rows(); written in place, chunk by chunk, on a few
    threads (numpy releases the GIL inside its loops).
    """
    import concurrent.futures as cf
    import os

    R, L, Wd = pool.shape
    assert Wd % 8 == 0 and pool.flags["C_CONTIGUOUS"]
    nw = Wd // 8
    words = pool.reshape(R * L, Wd).view(np.uint64)
    offs = np.arange(nw, dtype=np.uint64)[None, :]

    def fill(start: int) -> None:
        stop = min(R * L, start + chunk_rows)
        idx = np.arange(start, stop, dtype=np.int64)
        base = row_counter(layer, idx // L, idx % L)[:, None]
        z = words[start:stop]
        np.add(base, offs, out=z)
        _mix_inplace(z)

    starts = range(0, R * L, chunk_rows)
    n = threads or min(16, os.cpu_count() or 1)
    if n <= 1 or len(starts) == 1:
        for st in starts:
            fill(st)
        return
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(fill, starts))


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic swap-in workload (shape, capacity and index recipe)."""

    cfg_id: int
    name: str
    batch: int
    steps: int
    top_k: int
    seq_len: int
    hot_buffer: int
    calls: int
    kind: str  # "uniform", "zipf", "cluster"
    reuse: float  # fraction of each step drawn from the previous step
    page_size: int = 0
    row_bytes: int = ROW_BYTES
    clusters: int = 16
    cluster_sigma: float = 128.0
    zipf_s: float = 1.1

    @property
    def num_requests(self) -> int:
        return self.batch

    @property
    def entries(self) -> int:
        return self.batch * self.steps * self.top_k


# The five workloads (tiny, DSA-like decode, 4-step MTP, capacity overflow,
# long-context paged).  Calls beyond `calls` continue the same stream.
WORKLOADS: Dict[str, Workload] = {
    "C1": Workload(1, "tiny_single_step", 1, 1, 64, 4096, 256, 8, "uniform", 0.5),
    "C2": Workload(2, "dsa_decode_b64_k2048", 64, 1, 2048, 32768, 4096, 32, "zipf", 0.8),
    "C3": Workload(3, "mtp4_b64_k2048", 64, 4, 2048, 32768, 8192, 32, "zipf", 0.7),
    "C4": Workload(4, "overflow_b8_s4_h2048", 8, 4, 2048, 65536, 2048, 32, "zipf", 0.2),
    "C5": Workload(5, "long_paged_b16_l131072", 16, 1, 2048, 131072, 8192, 32, "cluster", 0.0,
                   page_size=256),
}


def req_pool_indices(w: Workload) -> np.ndarray:
    """Seeded permutation of 0..B-1 (request-pool slot of each batch row)."""
    rng = np.random.Generator(np.random.PCG64(1000 * w.cfg_id + 999))
    return rng.permutation(w.batch).astype(np.int32)


def seq_lens(w: Workload) -> np.ndarray:
    return np.full(w.batch, w.seq_len, dtype=np.int32)


def _zipf_cdf(L: int, s: float) -> np.ndarray:
    r = np.arange(1, L + 1, dtype=np.float64)
    p = r ** (-s)
    c = np.cumsum(p)
    return c / c[-1]


def _draw_distinct(rng, need: int, sampler, exclude: np.ndarray) -> np.ndarray:
    """`need` distinct values from `sampler(n)`, none in `exclude`, in draw order."""
    out: List[np.ndarray] = []
    have = 0
    seen = set(int(x) for x in exclude)
    batch = max(64, 2 * need)
    while have < need:
        cand = sampler(batch)
        for x in cand.tolist():
            if x not in seen:
                seen.add(x)
                out.append(x)
                have += 1
                if have == need:
                    break
        batch = min(batch * 2, 1 << 20)
    return np.asarray(out, dtype=np.int64)


class TopkStream:
    """Seeded stream of top-k index tensors int32 [B, S, K], one per call.

    Each step's K indices are distinct and shuffled.  ``round(reuse * K)`` of
    them are a uniform random subset of the previous step's indices (the
    previous call's last step for step 0); the rest are fresh draws from the
    workload's distribution, distinct from the reused part:
      * uniform: without replacement from [0, L);
      * zipf: rank r ~ Zipf(s) truncated to [1, L], position L - r (rank 1 is
        the most recent token);
      * cluster: fixed per-request centres uniform in [0, L); each call draws
        K / clusters tokens per centre as round(Normal(c, sigma^2)) clipped to
        [0, L).
    Call c draws from numpy PCG64(1000 * cfg_id + c).
    """

    def __init__(self, w: Workload, batch: Optional[int] = None):
        self.w = w
        self.batch = w.batch if batch is None else batch
        self._prev: List[Optional[np.ndarray]] = [None] * self.batch
        self._next_call = 0
        self._cdf = _zipf_cdf(w.seq_len, w.zipf_s) if w.kind == "zipf" else None
        if w.kind == "cluster":
            crng = np.random.Generator(np.random.PCG64(1000 * w.cfg_id + 998))
            self._centres = crng.integers(0, w.seq_len, size=(self.batch, w.clusters))

    def _fresh(self, rng, b: int, need: int, exclude: np.ndarray) -> np.ndarray:
        w = self.w
        L = w.seq_len
        if need == 0:
            return np.zeros(0, dtype=np.int64)
        if w.kind == "uniform":
            return _draw_distinct(rng, need, lambda n: rng.integers(0, L, size=n), exclude)
        if w.kind == "zipf":
            cdf = self._cdf

            def zipf(n):
                r = np.searchsorted(cdf, rng.random(n), side="right") + 1
                r = np.minimum(r, L)
                return L - r

            return _draw_distinct(rng, need, zipf, exclude)
        if w.kind == "cluster":
            per = need // w.clusters
            extra = need - per * w.clusters
            parts: List[np.ndarray] = []
            taken = np.asarray(exclude, dtype=np.int64)
            for ci, c in enumerate(self._centres[b]):
                n_c = per + (1 if ci < extra else 0)

                def gauss(n, c=c):
                    x = np.rint(rng.normal(c, w.cluster_sigma, size=n))
                    return np.clip(x, 0, L - 1).astype(np.int64)

                got = _draw_distinct(rng, n_c, gauss, taken)
                parts.append(got)
                taken = np.concatenate([taken, got])
            return np.concatenate(parts)
        raise ValueError(w.kind)

    def next_call(self) -> np.ndarray:
        w = self.w
        c = self._next_call
        self._next_call += 1
        rng = np.random.Generator(np.random.PCG64(1000 * w.cfg_id + c))
        out = np.empty((self.batch, w.steps, w.top_k), dtype=np.int32)
        n_reuse = int(round(w.reuse * w.top_k))
        for b in range(self.batch):
            for s in range(w.steps):
                prev = self._prev[b]
                if prev is not None and n_reuse > 0:
                    reused = rng.choice(prev, size=n_reuse, replace=False).astype(np.int64)
                else:
                    reused = np.zeros(0, dtype=np.int64)
                fresh = self._fresh(rng, b, w.top_k - reused.size, reused)
                step = np.concatenate([reused, fresh])
                rng.shuffle(step)
                out[b, s] = step
                self._prev[b] = step
        return out

    def calls(self, n: int) -> List[np.ndarray]:
        return [self.next_call() for _ in range(n)]


def scaled(w: Workload, **changes) -> Workload:
    """A copy of workload `w` with some fields changed (smaller test cases)."""
    return dataclasses.replace(w, **changes)
