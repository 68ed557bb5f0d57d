"""CUDA path against the CPU oracle, bit for bit (needs a GB300).

Small cases span several CTAs of a request (up to 1024 entries a pass), ragged
top-k widths, every step count, overflow and multiple layers; the workload
cases run the five configurations' index streams, scaled where marked and at
full size where the oracle still finishes in seconds.
"""
import numpy as np
import pytest

import hs_workloads as W
from gpu_harness import ParityRun

pytestmark = pytest.mark.gpu


def _rand_calls(rng, R, L, K, S_max, B, calls, reuse=0.5, invalid=0.05):
    prev = None
    for c in range(calls):
        S = int(rng.integers(1, S_max + 1))
        topk = rng.integers(0, L, size=(B, S, K)).astype(np.int32)
        if prev is not None:
            n = int(reuse * K)
            topk[:, 0, :n] = prev[:, -1, -n:]
        for s in range(1, S):
            n = int(reuse * K)
            topk[:, s, :n] = topk[:, s - 1, K - n:]
        mask = rng.random(topk.shape) < invalid
        topk[mask] = rng.choice([-1, L, L + 7, -5], size=int(mask.sum()))
        rpi = rng.permutation(R)[:B].astype(np.int32)
        sl = rng.integers(L // 2, L + 1, size=B).astype(np.int32)
        prev = topk
        yield topk, rpi, sl


SMALL = [
    # R, L, H, K, S_max, B, calls
    (1, 256, 16, 8, 1, 1, 12),
    (3, 500, 40, 37, 4, 3, 10),      # ragged K, all step counts
    (4, 2000, 300, 300, 4, 4, 8),    # several 1024-entry tiles per request
    (2, 9000, 1000, 2048, 4, 2, 6),  # 8192 entries per request (largest tile count)
    (5, 3000, 64, 600, 3, 5, 6),     # heavy overflow
    (2, 100, 1, 5, 2, 2, 10),        # a single hot slot
    (6, 70000, 512, 513, 2, 4, 5),   # long rows, ragged tile tail
]


@pytest.mark.parametrize("R,L,H,K,S_max,B,calls", SMALL)
def test_small_configs(R, L, H, K, S_max, B, calls):
    rng = np.random.default_rng(R * 1000 + K)
    run = ParityRun(R, L, W.ROW_BYTES, H, K, S_max)
    for topk, rpi, sl in _rand_calls(rng, R, L, K, S_max, B, calls):
        run.call(topk, rpi, sl, properties=True)


def test_two_layers_interleaved():
    rng = np.random.default_rng(5)
    run = ParityRun(3, 800, W.ROW_BYTES, 64, 48, 2, layers=2)
    gens = [_rand_calls(rng, 3, 800, 48, 2, 3, 6), _rand_calls(rng, 3, 800, 48, 2, 3, 6)]
    for c in range(6):
        for layer in (1, 0):
            topk, rpi, sl = next(gens[layer])
            run.call(topk, rpi, sl, layer=layer)


def test_miss_plan_matches():
    rng = np.random.default_rng(9)
    run = ParityRun(4, 1000, W.ROW_BYTES, 100, 64, 4)
    for topk, rpi, sl in _rand_calls(rng, 4, 1000, 64, 4, 4, 5):
        run.call(topk, rpi, sl, plan=True)


def test_deferred_copy_replays_plan_exactly():
    """Deferred mode: the call copies nothing; replaying its miss plan on
    another stream gives the same rows, locations and state as the oracle."""
    rng = np.random.default_rng(10)
    run = ParityRun(4, 3000, W.ROW_BYTES, 200, 300, 4, deferred=True)
    for topk, rpi, sl in _rand_calls(rng, 4, 3000, 300, 4, 4, 6):
        run.call(topk, rpi, sl)
    import pytest as _pt
    import torch
    import sparse_attention_kv_swap_gb300 as pkg
    with _pt.raises(pkg.HsError):  # deferred mode needs the plan outputs
        i32 = dict(dtype=torch.int32, device="cuda")
        pkg.hs_swap_in(run.cache.handle, torch.tensor([0], **i32), torch.tensor([5], **i32),
                       torch.zeros((1, 1, 300), **i32), 0, torch.empty((1, 1, 300), **i32))


def test_reset_requests_matches():
    import torch
    rng = np.random.default_rng(11)
    run = ParityRun(4, 600, W.ROW_BYTES, 50, 32, 2, layers=2)
    calls = list(_rand_calls(rng, 4, 600, 32, 2, 4, 6))
    for i, (topk, rpi, sl) in enumerate(calls):
        run.call(topk, rpi, sl, layer=i % 2)
        if i == 3:
            victims = np.array([1, 3], np.int32)
            run.cache.reset_requests(torch.from_numpy(victims).cuda())
            run.oracle.reset_requests(victims)
            for layer in range(2):
                for q in victims.tolist():
                    g = run.gpu_state(layer, q)
                    assert (g["tok"] == -1).all() and g["epoch"] == 0
                    assert (g["phys"] == np.arange(50 + 64)).all()


def test_batch_zero_and_all_invalid():
    import torch
    run = ParityRun(2, 100, W.ROW_BYTES, 8, 4, 1)
    empty = torch.empty((0, 1, 4), dtype=torch.int32, device="cuda")
    e32 = torch.empty(0, dtype=torch.int32, device="cuda")
    out = run.cache.swap_in(e32, e32, empty)
    assert out["device_locs"].numel() == 0
    topk = np.array([[[-1, 100, 200, -7]], [[5, 5, -1, 99]]], np.int32)
    g = run.call(topk, np.array([0, 1], np.int32), np.array([100, 50], np.int32))
    assert (g["device_locs"][0] == -1).all()


def test_hot_buffer_upper_bound():
    # 32768 hot slots (the multi-step report's stated bound), 8192 entries per call
    rng = np.random.default_rng(13)
    run = ParityRun(1, 70000, 64, 32768, 2048, 4)
    for c in range(4):
        topk = np.stack([rng.permutation(70000)[:2048] for _ in range(4)])[None]
        run.call(topk.astype(np.int32), np.array([0], np.int32), np.array([70000], np.int32))


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C5"])
def test_workload_scaled(name):
    w = W.WORKLOADS[name]
    if name != "C1":
        w = W.scaled(w, batch=4, seq_len=min(w.seq_len, 16384))
    stream = W.TopkStream(w)
    rpi = W.req_pool_indices(w)
    sl = W.seq_lens(w)
    run = ParityRun(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps)
    for c in range(w.calls if name == "C1" else 10):
        run.call(stream.next_call(), rpi, sl, properties=(name == "C4"))


@pytest.mark.parametrize("name", ["C2", "C3", "C4", "C5"])
def test_workload_full_size(name):
    """Full-size configuration, every output compared (8 calls of the stream)."""
    w = W.WORKLOADS[name]
    stream = W.TopkStream(w)
    rpi = W.req_pool_indices(w)
    sl = W.seq_lens(w)
    run = ParityRun(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps)
    for c in range(8):
        run.call(stream.next_call(), rpi, sl, compare_rows=(c % 4 == 3),
                 properties=(name == "C4" and c == 7))


# ---- dense token -> slot index (HS_INDEX_DENSE): identical observables --------

@pytest.mark.parametrize("R,L,H,K,S_max,B,calls", SMALL)
def test_small_configs_dense_index(R, L, H, K, S_max, B, calls):
    rng = np.random.default_rng(R * 1000 + K)
    run = ParityRun(R, L, W.ROW_BYTES, H, K, S_max, dense=True)
    for topk, rpi, sl in _rand_calls(rng, R, L, K, S_max, B, calls):
        run.call(topk, rpi, sl, properties=True)


def test_dense_index_reset_and_layers():
    import torch
    rng = np.random.default_rng(12)
    run = ParityRun(4, 600, W.ROW_BYTES, 50, 32, 2, layers=2, dense=True)
    calls = list(_rand_calls(rng, 4, 600, 32, 2, 4, 6))
    for i, (topk, rpi, sl) in enumerate(calls):
        run.call(topk, rpi, sl, layer=i % 2)
        if i == 3:
            victims = np.array([0, 2], np.int32)
            run.cache.reset_requests(torch.from_numpy(victims).cuda())
            run.oracle.reset_requests(victims)


@pytest.mark.parametrize("name", ["C2", "C3", "C4", "C5"])
def test_workload_full_size_dense_index(name):
    w = W.WORKLOADS[name]
    stream = W.TopkStream(w)
    rpi = W.req_pool_indices(w)
    sl = W.seq_lens(w)
    run = ParityRun(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps, dense=True)
    for c in range(6):
        run.call(stream.next_call(), rpi, sl, compare_rows=(c == 5),
                 properties=(name == "C4" and c == 5))


@pytest.mark.parametrize("name,dense", [("C2", True), ("C3", True), ("C2", False)])
def test_full_size_graph_replay_as_benchmarked(name, dense):
    """The benchmark's launch configuration at full size (dense index, and the
    hash banks as well): one swap-in captured in a CUDA graph on a side stream
    and replayed with each call's top-k staged into the graph's input buffer."""
    import torch
    import sparse_attention_kv_swap_gb300 as pkg
    w = W.WORKLOADS[name]
    stream = W.TopkStream(w)
    rpi, sl = W.req_pool_indices(w), W.seq_lens(w)
    run = ParityRun(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps, dense=dense)
    run.call(stream.next_call(), rpi, sl, compare_rows=False)  # also sets kernel attributes
    dev = torch.device("cuda")
    rpi_t, sl_t = torch.from_numpy(rpi).to(dev), torch.from_numpy(sl).to(dev)
    topk_buf = torch.empty((w.batch, w.steps, w.top_k), dtype=torch.int32, device=dev)
    out = {"device_locs": torch.empty_like(topk_buf),
           "stats": torch.empty((w.batch, pkg.binding.HS_NUM_STATS), dtype=torch.int32,
                                device=dev)}
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run.cache.swap_in(rpi_t, sl_t, topk_buf, 0, out=out, stream=side)
    for c in range(4):
        topk = stream.next_call()
        topk_buf.copy_(torch.from_numpy(topk))
        graph.replay()
        ref = run.oracle.swap_in(0, run.opools[0], run.mirror[0], rpi, sl, topk, num_threads=8)
        torch.cuda.synchronize()
        assert (out["device_locs"].cpu().numpy() == ref["locs"]).all(), "call %d: locations" % c
        assert (out["stats"].cpu().numpy() == ref["stats"]).all(), "call %d: counters" % c
        for q in rpi.tolist():
            g, o = run.gpu_state(0, q), run.oracle.request_state(0, q)
            for k in ("tok", "ep", "phys"):
                assert (g[k] == o[k]).all(), "call %d q=%d: %s" % (c, q, k)
    got = run.cache.device_kv[0].cpu().numpy()
    assert (got == run.mirror[0]).all(), "device rows differ after the replays"
    assert run.cache.status() == (0, 0)


@pytest.mark.parametrize("B,S,K", [(160, 1, 2048), (100, 4, 2048), (300, 2, 64)])
def test_batches_wider_than_the_gpu(B, S, K):
    """More requests than SMs: single-CTA gathers with 2 entries per thread
    (160 x 2048), 2-CTA clusters in more than one wave (100 x 4 x 2048), and
    many small requests (300 x 2 x 64)."""
    rng = np.random.default_rng(B + S)
    R, L, H = B + 7, 2500, 512
    run = ParityRun(R, L, W.ROW_BYTES, H, K, S, max_batch=B)
    for topk, rpi, sl in _rand_calls(rng, R, L, K, S, B, 4):
        run.call(topk, rpi, sl, properties=False)


def test_long_run_epochs_beyond_sixteen_bits():
    """65,600 calls on a 4-slot cache, both requests in every call: the epoch
    passes 2^8 and 2^16, so the commit's victim selection runs its radix
    select with two and then three digit passes.  Every call's locations and
    counters, and the final policy state and rows, equal the oracle's."""
    import torch
    import sparse_attention_kv_swap_gb300 as pkg
    R, L, Wd, H, K, N = 2, 64, 16, 4, 3, 65600
    run = ParityRun(R, L, Wd, H, K, 1)
    rng = np.random.default_rng(77)
    topk = rng.integers(0, 16, size=(N, R, 1, K)).astype(np.int32)
    topk[rng.random(topk.shape) < 0.02] = -1
    rpi = np.arange(R, dtype=np.int32)
    sl = np.full(R, L, dtype=np.int32)
    i32 = dict(dtype=torch.int32, device="cuda")
    topk_d = torch.from_numpy(topk).cuda()
    rpi_d, sl_d = torch.from_numpy(rpi).cuda(), torch.from_numpy(sl).cuda()
    locs_d = torch.empty((N, R, 1, K), **i32)
    stats_d = torch.empty((N, R, pkg.binding.HS_NUM_STATS), **i32)
    for i in range(N):
        run.cache.swap_in(rpi_d, sl_d, topk_d[i], 0,
                          out={"device_locs": locs_d[i], "stats": stats_d[i]})
    want_locs = np.empty((N, R, 1, K), dtype=np.int32)
    want_stats = np.empty((N, R, pkg.binding.HS_NUM_STATS), dtype=np.int32)
    for i in range(N):
        ref = run.oracle.swap_in(0, run.opools[0], run.mirror[0], rpi, sl, topk[i])
        want_locs[i], want_stats[i] = ref["locs"], ref["stats"]
    torch.cuda.synchronize()
    assert run.cache.status()[1] == 0
    got_locs, got_stats = locs_d.cpu().numpy(), stats_d.cpu().numpy()
    bad = np.argwhere((got_locs != want_locs).reshape(N, -1).any(axis=1))
    assert bad.size == 0, "locations differ from call %d on" % bad[0][0]
    bad = np.argwhere((got_stats != want_stats).reshape(N, -1).any(axis=1))
    assert bad.size == 0, "counters differ from call %d on" % bad[0][0]
    evicted = 5  # HS_STAT_EVICTED
    assert want_stats[:, :, evicted].sum() > N  # the cache kept evicting throughout
    for q in range(R):
        gs, os_ = run.gpu_state(0, q), run.oracle.request_state(0, q)
        assert gs["epoch"] == os_["epoch"] == N
        for k in ("tok", "ep", "phys"):
            assert (gs[k] == os_[k]).all(), (q, k)
    assert (run.cache.device_kv[0].cpu().numpy() == run.mirror[0]).all()


@pytest.mark.parametrize("dense", [False, True])
def test_hashed_dedup_for_sequences_beyond_the_position_table(dense):
    """max_seq_len past what a position-indexed de-duplication table can hold
    in 8 CTAs (5 bytes a position, 160 KiB a CTA): the table is hashed
    instead, with the same observables."""
    rng = np.random.default_rng(21 + dense)
    R, L, H, K, S = 3, 300000, 100, 700, 4
    run = ParityRun(R, L, 16, H, K, S, dense=dense)
    for topk, rpi, sl in _rand_calls(rng, R, L, K, S, R, 6):
        run.call(topk, rpi, sl, properties=True)


def test_timeline_stamps_are_ordered_and_change_nothing():
    """hs_set_timeline: every used CTA writes its phase stamps (words 0-8
    and 10) in order, the leader its commit stamp (word 9), word 15 the
    cluster size, nothing else; results stay exact."""
    import torch
    import sparse_attention_kv_swap_gb300 as pkg
    w = W.scaled(W.WORKLOADS["C3"], batch=4, seq_len=16384)
    stream = W.TopkStream(w)
    rpi, sl = W.req_pool_indices(w), W.seq_lens(w)
    run = ParityRun(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps, dense=True)
    tl = torch.zeros(w.batch * 128, dtype=torch.int64, device="cuda")
    pkg.hs_set_timeline(run.cache.handle, tl)
    for c in range(3):
        tl.zero_()
        run.call(stream.next_call(), rpi, sl)
        t = tl.view(w.batch, 8, 16).cpu().numpy()
        P = int(t[0, 0, 15])
        assert P in (1, 2, 4, 8) and (t[:, :P, 15] == P).all() and (t[:, P:] == 0).all()
        assert (t[:, :P, 11:15] == 0).all()
        for b in range(w.batch):
            for r in range(P):
                s = t[b, r]
                assert (s[:9] > 0).all() and (np.diff(s[:9]) >= 0).all(), (b, r, s)
                assert s[10] >= s[8], (b, r, s)
                if r == 0:
                    assert s[8] <= s[9] <= s[10], (b, s)
                else:
                    assert s[9] == 0, (b, r, s)
    pkg.hs_set_timeline(run.cache.handle, None)
    tl.zero_()
    run.call(stream.next_call(), rpi, sl)
    assert int(tl.abs().sum()) == 0


# (batch, steps, top_k, max_seq_len, expected cluster size P, entries a thread, table)
LAUNCH_SHAPES = [
    (1, 1, 300, 5000, 1, 1, "position"),
    # 49,104 bytes of dynamic shared memory: under 48 KB, but not with the
    # kernel's static arrays added, so the launch must raise the limit
    (1, 1, 300, 12250, 1, 1, "position"),
    (100, 1, 2048, 5000, 1, 2, "position"),
    (100, 2, 2048, 5000, 1, 4, "position"),
    (40, 1, 2048, 5000, 2, 1, "position"),
    (40, 2, 2048, 5000, 2, 2, "position"),
    (40, 4, 2048, 5000, 2, 4, "position"),
    (20, 1, 2048, 5000, 4, 1, "position"),
    (20, 4, 2048, 5000, 4, 2, "position"),
    (2, 4, 2048, 5000, 8, 1, "position"),
    (4, 1, 600, 300000, 8, 1, "position"),    # cluster raised until the table fits
    (40, 4, 2048, 300000, 2, 4, "hashed"),    # too long for a position table
    # 16 clusters of 8 one-per-SM CTAs do not fit the GPCs at once: the
    # launcher halves the cluster to keep the call in one wave
    (16, 4, 2048, 5000, 4, 2, "position"),
]


@pytest.mark.parametrize("Bn,S,K,L,P,rmax,table", LAUNCH_SHAPES)
def test_every_launch_shape(Bn, S, K, L, P, rmax, table):
    """Each cluster size and entries-a-thread combination the launch can pick
    (on a 152-SM GB300), with both kinds of de-duplication table and the
    fallback to a smaller cluster when the batch's clusters would not be
    co-resident: the timeline's cluster-size word shows the shape, and two
    calls match the oracle bit for bit."""
    import torch
    import sparse_attention_kv_swap_gb300 as pkg
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("launch shapes are stated for 152 SMs")
    rng = np.random.default_rng(Bn * 31 + S * 7 + L)
    run = ParityRun(Bn, L, 16, 512, K, S, dense=(table == "position"))
    tl = torch.zeros(Bn * 128, dtype=torch.int64, device="cuda")
    pkg.hs_set_timeline(run.cache.handle, tl)
    rpi = rng.permutation(Bn).astype(np.int32)
    sl = np.full(Bn, L, dtype=np.int32)
    prev = None
    for c in range(2):
        topk = rng.integers(0, L, size=(Bn, S, K)).astype(np.int32)
        if prev is not None:
            topk[:, 0, :K // 2] = prev[:, -1, K // 2:]
        for s in range(1, S):
            topk[:, s, :K // 3] = topk[:, s - 1, -(K // 3):]
        prev = topk
        run.call(topk, rpi, sl, compare_rows=(c == 1))
        t = tl.view(Bn, 8, 16).cpu().numpy()
        assert int(t[0, 0, 15]) == P, "cluster size %d, expected %d" % (t[0, 0, 15], P)
