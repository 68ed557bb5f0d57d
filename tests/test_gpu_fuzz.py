"""Randomised parity sweep (needs a GB300): many small random configurations,
each a short decode loop with write-backs, checked call by call against the
oracle (locations, counters, policy state, index consistency, device rows,
host rows written).  Seeds are fixed, so a failure reproduces."""
import numpy as np
import pytest

import hs_workloads as W
from gpu_harness import ParityRun

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 9))
    L = int(rng.integers(40, 5000))
    H = int(rng.integers(1, 300))
    K = int(rng.integers(1, 600))
    S = int(rng.integers(1, 5))
    while S * K > 8192:
        K //= 2
    E = int(rng.choice([0, 0, 1, 3, 16, 64, 200]))
    dense = bool(rng.integers(0, 2))
    layers = int(rng.integers(1, 3))
    width = int(rng.choice([16, 64, W.ROW_BYTES]))
    return rng, R, L, H, K, S, E, dense, layers, width


@pytest.mark.parametrize("seed", range(120))
def test_random_configuration(seed):
    rng, R, L, H, K, S, E, dense, layers, width = _case(1000 + seed)
    run = ParityRun(R, L, width, H, K, S, layers=layers, dense=dense, extra_page=E,
                    own_pool=True)
    n = rng.integers(1, L + 1, size=R).astype(np.int32)
    for layer in range(layers):  # prefill of the still-filling page
        for q in range(R):
            lo = (n[q] - 1) // E * E if E else n[q] - 1
            toks = np.arange(lo, n[q], dtype=np.int32)
            run.append(np.full(toks.size, q, np.int32), toks, np.full(toks.size, n[q]),
                       rng.integers(0, 256, size=(toks.size, width), dtype=np.uint8),
                       layer=layer)
    for call in range(5):
        layer = int(rng.integers(0, layers))
        n = np.minimum(n + 1, L).astype(np.int32)
        every = np.arange(R, dtype=np.int32)
        for l in range(layers):  # decode writes every layer's new row
            run.append(every, n - 1, n, rng.integers(0, 256, size=(R, width), dtype=np.uint8),
                       layer=l)
        B = int(rng.integers(1, R + 1))
        rpi = rng.permutation(R)[:B].astype(np.int32)
        s = int(rng.integers(1, S + 1))
        recent = n[rpi][:, None, None] - 1 - rng.integers(0, 2 * max(E, 4), size=(B, s, K))
        wide = rng.integers(-3, L + 3, size=(B, s, K))
        topk = np.where(rng.random((B, s, K)) < 0.3, recent, wide).astype(np.int32)
        if s > 1:  # cross-step overlap
            m = K // 2
            topk[:, 1:, :m] = topk[:, :-1, K - m:]
        run.call(topk, rpi, n[rpi], layer=layer, properties=(call == 4), plan=(call % 2 == 1))
