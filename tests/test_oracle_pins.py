"""The CPU oracle against facts that do not come from the oracle itself."""
import os

import numpy as np
import pytest

import hs_workloads as W
import pins
from common import OracleHarness

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def lib():
    from oracle.oracle import load_library
    return load_library()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_splitmix64_known_answers():
    # Input generator pin: the published first outputs of SplitMix64(seed 0).
    with open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for n, hexval in rows:
        assert int(W.splitmix64_at(np.uint64(int(n)))) == int(hexval, 16)


def test_host_rows_are_distinct_and_deterministic():
    a = W.host_rows(0, [0, 0, 1], [5, 6, 5])
    b = W.host_rows(0, [0, 0, 1], [5, 6, 5])
    c = W.host_rows(1, [0], [5])
    assert (a == b).all() and a.shape == (3, W.ROW_BYTES)
    assert len({r.tobytes() for r in a} | {c[0].tobytes()}) == 4


def test_steps_two_and_three_and_multi_request(lib):
    rng = np.random.default_rng(31)
    for S in (2, 3):
        h = OracleHarness(6, 300, 32, 64, 40, 4, lib=lib)
        for c in range(6):
            topk = rng.integers(0, 300, size=(4, S, 40)).astype(np.int32)
            topk[:, 1:, :20] = topk[:, :-1, 20:]  # cross-step overlap
            rpi = rng.permutation(6)[:4].astype(np.int32)
            h.call(topk, rpi, np.full(4, 300, np.int32))


def test_hot_buffer_upper_bound(lib):
    # The multi-step report names 32768 as the hot-buffer bound.
    rng = np.random.default_rng(37)
    H, K, S = 32768, 2048, 4
    h = OracleHarness(1, 65536, 16, H, K, S, lib=lib)
    for c in range(3):
        topk = np.stack([rng.permutation(65536)[:K] for _ in range(S)])[None].astype(np.int32)
        h.call(topk, np.array([0], np.int32), np.array([65536], np.int32))


def test_layers_are_isolated(lib):
    rng = np.random.default_rng(41)
    h = OracleHarness(2, 64, 32, 8, 4, 2, layers=2, lib=lib)
    before = h.states(1)
    for c in range(4):
        topk = rng.integers(0, 64, size=(2, 2, 4)).astype(np.int32)
        h.call(topk, np.array([0, 1], np.int32), np.array([64, 64], np.int32), layer=0)
    after = h.states(1)
    for q in range(2):
        for k in ("tok", "ep", "phys"):
            assert (before[q][k] == after[q][k]).all()


def test_reset_requests(lib):
    rng = np.random.default_rng(43)
    h = OracleHarness(3, 64, 32, 8, 4, 2, layers=2, lib=lib)
    for c in range(3):
        for layer in range(2):
            topk = rng.integers(0, 64, size=(3, 2, 4)).astype(np.int32)
            h.call(topk, np.array([0, 1, 2], np.int32), np.full(3, 64, np.int32), layer=layer)
    h.o.reset_requests(np.array([1], np.int32))
    for layer in range(2):
        st = h.o.request_state(layer, 1)
        assert (st["tok"] == -1).all() and (st["ep"] == -1).all() and st["epoch"] == 0
        assert (st["phys"] == np.arange(8 + 8)).all()
        assert h.o.request_state(layer, 0)["epoch"] == 3


def test_seq_len_beyond_pool_is_invalid(lib):
    h = OracleHarness(1, 20, 32, 8, 4, 1, lib=lib)
    out = h.call(np.array([[[3, 19, 20, 25]]], np.int32), np.array([0], np.int32),
                 np.array([30], np.int32))
    assert out["locs"][0, 0, 2] == -1 and out["locs"][0, 0, 3] == -1
    assert out["stats"][0][7] == 2


def test_duplicate_request_rejected(lib):
    h = OracleHarness(2, 20, 32, 8, 4, 1, lib=lib)
    with pytest.raises(ValueError):
        h.call(np.zeros((2, 1, 4), np.int32), np.array([1, 1], np.int32),
               np.array([20, 20], np.int32), check=False)


def test_threads_match_single_thread(lib):
    w = W.scaled(W.WORKLOADS["C2"], batch=8, top_k=256, seq_len=2048, hot_buffer=512)
    stream = W.TopkStream(w)
    calls = stream.calls(4)
    rpi = W.req_pool_indices(w)
    sl = W.seq_lens(w)
    a = OracleHarness(8, 2048, 32, 512, 256, 1, lib=lib)
    b = OracleHarness(8, 2048, 32, 512, 256, 1, lib=lib)
    for topk in calls:
        oa = a.call(topk, rpi, sl, check=False, threads=1)
        ob = b.call(topk, rpi, sl, check=False, threads=4)
        assert (oa["locs"] == ob["locs"]).all() and (oa["stats"] == ob["stats"]).all()
    assert (a.dev[0] == b.dev[0]).all()


def test_miss_plan(lib):
    rng = np.random.default_rng(47)
    h = OracleHarness(3, 64, 32, 6, 5, 2, lib=lib)
    for c in range(4):
        topk = rng.integers(0, 64, size=(2, 2, 5)).astype(np.int32)
        rpi = np.array([2, 0], np.int32)
        out = h.call(topk, rpi, np.full(2, 64, np.int32), want_plan=True)
        for b in range(2):
            U = out["miss_count"][b]
            assert U == out["stats"][b][3]
            q = int(rpi[b])
            # every planned copy moves the token's host row to a returned location
            src, dst = out["miss_src"][b, :U], out["miss_dst"][b, :U]
            assert ((src // 64) == q).all()
            locs = out["locs"][b].reshape(-1)
            flat = topk[b].reshape(-1)
            for s, d in zip(src.tolist(), dst.tolist()):
                assert d in set(locs[flat == s % 64].tolist())
