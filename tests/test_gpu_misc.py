"""Page table, device status flags, argument errors and graph capture on the GPU."""
import numpy as np
import pytest
import torch

import hs_workloads as W
import sparse_attention_kv_swap_gb300 as pkg
from sparse_attention_kv_swap_gb300 import binding as B
from gpu_harness import ParityRun

pytestmark = pytest.mark.gpu


def _page_table_gpu(topk, sl, L_max, page):
    B_, S, K = topk.shape
    pages = torch.empty((B_, S * K), dtype=torch.int32, device="cuda")
    num = torch.empty(B_, dtype=torch.int32, device="cuda")
    tp = torch.empty((B_, S, K), dtype=torch.int32, device="cuda")
    B.hs_page_table(torch.from_numpy(topk).cuda(), torch.from_numpy(sl).cuda(), L_max, page,
                    pages, num, tp)
    torch.cuda.synchronize()
    return pages.cpu().numpy(), num.cpu().numpy(), tp.cpu().numpy()


@pytest.mark.parametrize("page", [1, 7, 64, 256])
def test_page_table_random(page):
    from oracle import page_table
    rng = np.random.default_rng(page)
    for trial in range(5):
        Bn, S, K = 3, int(rng.integers(1, 5)), int(rng.integers(1, 700))
        L = int(rng.integers(1, 20000))
        topk = rng.integers(-3, L + 40, size=(Bn, S, K)).astype(np.int32)
        sl = rng.integers(1, L + 20, size=Bn).astype(np.int32)
        got = _page_table_gpu(topk, sl, L, page)
        ref = page_table(topk, sl, page, max_seq_len=L)
        for g, r in zip(got, ref):
            assert (g == r).all()


def test_page_table_long_context_workload():
    from oracle import page_table
    w = W.WORKLOADS["C5"]
    stream = W.TopkStream(w)
    sl = W.seq_lens(w)
    for c in range(4):
        topk = stream.next_call()
        got = _page_table_gpu(topk, sl, w.seq_len, w.page_size)
        ref = page_table(topk, sl, w.page_size, max_seq_len=w.seq_len)
        for g, r in zip(got, ref):
            assert (g == r).all()
        assert got[1].max() < 200  # clustered selections touch few pages


def test_status_flags():
    run = ParityRun(3, 100, 32, 8, 4, 1)
    cache = run.cache
    topk = torch.zeros((2, 1, 4), dtype=torch.int32, device="cuda")
    sl = torch.full((2,), 100, dtype=torch.int32, device="cuda")
    cache.swap_in(torch.tensor([1, 1], dtype=torch.int32, device="cuda"), sl, topk)
    rc, flags = cache.status()
    assert rc == B.HS_ERR_DEVICE_STATUS and flags & B.HS_STATUS_DUPLICATE_REQUEST
    assert cache.status() == (0, 0)  # reading clears the flags
    cache.swap_in(torch.tensor([0, 7], dtype=torch.int32, device="cuda"), sl, topk)
    rc, flags = cache.status()
    assert flags & B.HS_STATUS_BAD_REQUEST
    out = cache.swap_in(torch.tensor([0, 2], dtype=torch.int32, device="cuda"),
                        torch.tensor([100, 500], dtype=torch.int32, device="cuda"), topk)
    rc, flags = cache.status()
    assert flags == B.HS_STATUS_SEQ_LEN_CLAMPED
    # locks were released: a normal call still works and raises nothing
    cache.swap_in(torch.tensor([1, 2], dtype=torch.int32, device="cuda"), sl, topk)
    assert cache.status() == (0, 0)


def test_argument_errors():
    run = ParityRun(2, 100, 32, 8, 4, 2, max_batch=2)
    c = run.cache
    i32 = dict(dtype=torch.int32, device="cuda")
    rpi = torch.tensor([0, 1], **i32)
    sl = torch.tensor([100, 100], **i32)
    with pytest.raises(pkg.HsError) as e:
        c.swap_in(rpi, sl, torch.zeros((2, 3, 4), **i32))  # 3 steps > max_steps
    assert e.value.code == B.HS_ERR_INVALID_ARG
    with pytest.raises(pkg.HsError):
        c.swap_in(rpi, sl, torch.zeros((2, 1, 4), **i32), layer_id=1)
    with pytest.raises(pkg.HsError):
        c.swap_in(torch.tensor([0, 1, 1], **i32), torch.tensor([1, 1, 1], **i32),
                  torch.zeros((3, 1, 4), **i32))  # batch > max_batch
    locs = torch.empty((2, 1, 4), **i32)
    src = torch.empty((2, 8), dtype=torch.int64, device="cuda")
    with pytest.raises(pkg.HsError):  # a partial miss plan
        B.hs_swap_in(c.handle, rpi, sl, torch.zeros((2, 1, 4), **i32), 0, locs, None, src)


def test_pageable_pool_rejected_or_served_exactly():
    """Pageable host memory is refused unless the device reads host page
    tables directly; where it is accepted, rows still arrive bit-exact."""
    cfg = pkg.make_config(1, 64, 32, 4, 2, 1)
    pool = torch.empty((1, 64, 32), dtype=torch.uint8)  # pageable
    W.fill_host_pool(pool.numpy(), 0)
    kv = torch.zeros((1 * 6, 32), dtype=torch.uint8, device="cuda")
    st = torch.empty(pkg.hs_state_bytes(cfg), dtype=torch.uint8, device="cuda")
    ws = torch.empty(pkg.hs_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    try:
        h = pkg.hs_create_state(cfg, [pool], [kv], st, ws)
    except pkg.HsError as e:
        assert e.code == B.HS_ERR_INVALID_ARG
        return
    i32 = dict(dtype=torch.int32, device="cuda")
    locs = torch.empty((1, 1, 2), **i32)
    B.hs_swap_in(h, torch.tensor([0], **i32), torch.tensor([64], **i32),
                 torch.tensor([[[7, 63]]], **i32), 0, locs)
    torch.cuda.synchronize()
    rows = kv[locs.view(-1).long()].cpu().numpy()
    assert (rows == W.host_rows(0, [0, 0], [7, 63], 32)).all()
    h.close()


def test_cuda_graph_replay_matches_direct():
    """A captured call replays to the same outputs and state as direct calls."""
    rng = np.random.default_rng(21)
    a = ParityRun(4, 4000, W.ROW_BYTES, 256, 256, 2)
    b = ParityRun(4, 4000, W.ROW_BYTES, 256, 256, 2, pools=a.pools)
    rpi = torch.tensor([3, 1, 0, 2], dtype=torch.int32, device="cuda")
    sl = torch.full((4,), 4000, dtype=torch.int32, device="cuda")
    topk_buf = torch.empty((4, 2, 256), dtype=torch.int32, device="cuda")
    out = {"device_locs": torch.empty((4, 2, 256), dtype=torch.int32, device="cuda"),
           "stats": torch.empty((4, B.HS_NUM_STATS), dtype=torch.int32, device="cuda")}
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b.cache.swap_in(rpi, sl, topk_buf.zero_(), stats=True, out=out, stream=s)  # warm-up
        b.cache.reset_requests(torch.arange(4, dtype=torch.int32, device="cuda"), stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.cache.swap_in(rpi, sl, topk_buf, stats=True, out=out, stream=s)
    b.cache.reset_requests(torch.arange(4, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    for c in range(5):
        topk = rng.integers(0, 4000, size=(4, 2, 256)).astype(np.int32)
        ga = a.call(topk, rpi.cpu().numpy(), sl.cpu().numpy())
        topk_buf.copy_(torch.from_numpy(topk))
        g.replay()
        torch.cuda.synchronize()
        assert (out["device_locs"].cpu().numpy() == ga["device_locs"]).all()
        assert (out["stats"].cpu().numpy() == ga["stats"]).all()
    for q in range(4):
        sa, sb = a.gpu_state(0, q), b.gpu_state(0, q)
        for k in ("tok", "ep", "phys"):
            assert (sa[k] == sb[k]).all()


def test_pinned_host_inputs_and_outputs_match_device_buffers():
    """Pinned host memory is device-addressable (mapped, unified addresses):
    the call given pinned host inputs and outputs, read and written by its
    kernels across the host link, gives what the same call on device buffers
    gives."""
    rng = np.random.default_rng(31)
    a = ParityRun(4, 3000, W.ROW_BYTES, 128, 256, 2, dense=True)
    b = ParityRun(4, 3000, W.ROW_BYTES, 128, 256, 2, dense=True, pools=a.pools)
    for c in range(4):
        topk = rng.integers(-3, 3000, size=(4, 2, 256)).astype(np.int32)
        rpi = rng.permutation(4).astype(np.int32)
        sl = rng.integers(2000, 3001, size=4).astype(np.int32)
        ga = a.call(topk, rpi, sl)
        pin = lambda x: torch.from_numpy(x).pin_memory()
        out = {"device_locs": torch.empty((4, 2, 256), dtype=torch.int32).pin_memory(),
               "stats": torch.empty((4, B.HS_NUM_STATS), dtype=torch.int32).pin_memory()}
        b.cache.swap_in(pin(rpi), pin(sl), pin(topk), 0, out=out)
        torch.cuda.synchronize()
        assert (out["device_locs"].numpy() == ga["device_locs"]).all()
        assert (out["stats"].numpy() == ga["stats"]).all()
        for q in range(4):
            sa, sb = a.gpu_state(0, q), b.gpu_state(0, q)
            for k in ("tok", "ep", "phys"):
                assert (sa[k] == sb[k]).all()
    assert (a.cache.device_kv[0].cpu() == b.cache.device_kv[0].cpu()).all()


def test_running_totals_are_the_sums_of_the_call_counters():
    """hs_get_stats: per layer, the sum of every call's per-request counters
    (summed on the oracle side), and reset clears them."""
    rng = np.random.default_rng(41)
    run = ParityRun(5, 2000, W.ROW_BYTES, 64, 256, 3, layers=2, extra_page=16, own_pool=True)
    want = [np.zeros(B.HS_NUM_STATS, np.int64) for _ in range(2)]
    for c in range(8):
        layer = c % 2
        S = int(rng.integers(1, 4))
        topk = rng.integers(-3, 2000, size=(4, S, 256)).astype(np.int32)
        rpi = rng.permutation(5)[:4].astype(np.int32)
        sl = rng.integers(1500, 2001, size=4).astype(np.int32)
        g = run.call(topk, rpi, sl, layer=layer)
        want[layer] += g["stats"].sum(axis=0)
    for layer in range(2):
        got = run.cache.totals(layer)
        assert (got == want[layer]).all(), (layer, got, want[layer])
    assert run.cache.totals(0, reset=True).sum() > 0
    assert (run.cache.totals(0) == 0).all() and (run.cache.totals(1) == want[1]).all()


def test_planned_copy_skips_out_of_range_plans():
    """hs_copy_planned takes the caller's plan: out-of-range rows are skipped
    and counts are clamped to [0, C], with HS_STATUS_BAD_PLAN set; the valid
    rows are still copied."""
    R, L, Wd, H, K, S = 3, 50, 32, 4, 4, 1
    C = S * K
    run = ParityRun(R, L, Wd, H, K, S)
    kv = run.cache.device_kv[0]
    rows_total = kv.shape[0]
    src = np.zeros((3, C), np.int64)
    dst = np.zeros((3, C), np.int64)
    cnt = np.array([3, C + 5, -2], np.int32)   # row 1 clamps to C, row 2 to 0
    src[0, :3] = [0 * L + 7, R * L, 2 * L + 9]   # the middle source is past the pool
    dst[0, :3] = [0, 1, -1]                      # the last destination is negative
    src[1, :] = 1 * L + np.arange(C)
    dst[1, :] = (H + C) + H + np.arange(C)
    d = lambda a: torch.from_numpy(a).cuda()
    kv.zero_()
    pkg.hs_copy_planned(run.cache.handle, 0, d(src), d(dst), d(cnt))
    torch.cuda.synchronize()
    rc, flags = run.cache.status()
    assert flags == B.HS_STATUS_BAD_PLAN
    got = kv.cpu().numpy()
    pool = run.pools[0].numpy()
    assert (got[0] == pool[0, 7]).all()                 # the one valid row of batch row 0
    assert (got[1] == 0).all()                          # its invalid rows wrote nothing
    for j in range(C):                                  # batch row 1: clamped to C rows
        assert (got[(H + C) + H + j] == pool[1, j]).all()
    untouched = np.ones(rows_total, bool)
    untouched[[0] + [(H + C) + H + j for j in range(C)]] = False
    assert (got[untouched] == 0).all()


def test_two_handles_concurrent_threads_and_streams():
    """Two independent handles (hash index; dense index with an extra page)
    driven at the same time from two host threads, each on its own stream with
    no ordering between the streams.  Every call's locations and counters, and
    each handle's final rows and policy state, equal the oracle's for that
    handle's own call sequence."""
    import threading
    rng = np.random.default_rng(41)
    specs = [dict(R=6, L=6000, H=400, K=300, S=3, B=6, n=10, dense=False, E=0),
             dict(R=5, L=3000, H=128, K=200, S=2, B=4, n=12, dense=True, E=64)]
    runs, calls, ins, outs = [], [], [], []
    for sp in specs:
        runs.append(ParityRun(sp["R"], sp["L"], W.ROW_BYTES, sp["H"], sp["K"], sp["S"],
                              dense=sp["dense"], extra_page=sp["E"]))
        seq = []
        for c in range(sp["n"]):
            S = int(rng.integers(1, sp["S"] + 1))
            topk = rng.integers(-2, sp["L"] + 2, size=(sp["B"], S, sp["K"])).astype(np.int32)
            if seq:  # half of the first step repeats the previous call's last step
                topk[:, 0, :sp["K"] // 2] = seq[-1][0][:, -1, :sp["K"] // 2]
            rpi = rng.permutation(sp["R"])[:sp["B"]].astype(np.int32)
            sl = rng.integers(sp["L"] // 2, sp["L"] + 1, size=sp["B"]).astype(np.int32)
            seq.append((topk, rpi, sl))
        calls.append(seq)
        ins.append([(torch.from_numpy(r).cuda(), torch.from_numpy(s).cuda(),
                     torch.from_numpy(t).cuda()) for t, r, s in seq])
        outs.append([{"device_locs": torch.empty(t.shape, dtype=torch.int32, device="cuda"),
                      "stats": torch.empty((t.shape[0], B.HS_NUM_STATS), dtype=torch.int32,
                                           device="cuda")} for t, _, _ in seq])
    torch.cuda.synchronize()
    start = threading.Barrier(2)
    errors = []

    def drive(i):
        try:
            s = torch.cuda.Stream()
            start.wait(timeout=60)
            for (rpi, sl, topk), o in zip(ins[i], outs[i]):
                runs[i].cache.swap_in(rpi, sl, topk, 0, out=o, stream=s)
            s.synchronize()
        except BaseException as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=drive, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    torch.cuda.synchronize()
    for i, run in enumerate(runs):
        for c, ((topk, rpi, sl), o) in enumerate(zip(calls[i], outs[i])):
            ref = run.oracle.swap_in(0, run.opools[0], run.mirror[0], rpi, sl, topk,
                                     want_plan=False, num_threads=8)
            assert (o["device_locs"].cpu().numpy() == ref["locs"]).all(), (i, c)
            assert (o["stats"].cpu().numpy() == ref["stats"]).all(), (i, c)
        got = run.cache.device_kv[0].cpu().numpy()
        assert (got == run.mirror[0]).all(), i
        for q in range(run.R):
            gs, os_ = run.gpu_state(0, q), run.oracle.request_state(0, q)
            for k in ("tok", "ep", "phys"):
                assert (gs[k] == os_[k]).all(), (i, q, k)
        assert run.cache.status()[1] == 0


def test_handle_is_bound_to_its_buffers_device():
    """The binding binds a handle to the device of its device buffers and runs
    each call with that device current."""
    cfg = pkg.make_config(2, 300, W.ROW_BYTES, 16, 8, 1, 1)
    from sparse_attention_kv_swap_gb300.cache import SwapInCache
    cache = SwapInCache(cfg, device=torch.device("cuda", 0))
    assert cache.handle.device == 0
    i32 = dict(dtype=torch.int32, device="cuda:0")
    out = cache.swap_in(torch.tensor([0, 1], **i32), torch.tensor([300, 300], **i32),
                        torch.arange(16, **i32).view(2, 1, 8), 0, stats=True)
    torch.cuda.synchronize()
    assert (out["device_locs"].cpu().numpy() >= 0).all()
    assert cache.status()[1] == 0
    cache.close()
