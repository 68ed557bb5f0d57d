"""Extra page and write-back on the GPU against the CPU oracle, bit for bit.

The extra page is the request's newest, still-filling page: the swap-in
serves a selected token on it from the page's device row before any
hot-cache lookup (the multi-step swap report, 实现拆解 item 1).  Decode
writes each new row back to the host pool (PR #20343 summary, 功能与动机)
and to every device copy of it.  The decode loops below append one new
token per request per step, rewrite older positions (a rolled-back
speculative token), and resolve a selection biased towards the newest
positions; every call compares locations, counters, policy state, the
whole device buffer and the host rows written.
"""
import numpy as np
import pytest

import hs_workloads as W
from gpu_harness import ParityRun

pytestmark = pytest.mark.gpu


def _decode_loop(run, rng, R, L, K, S_max, E, steps, layers=1, rewrites=True):
    n = rng.integers(L // 4, L // 2, size=R).astype(np.int32)
    for layer in range(layers):
        # prefill leaves the partial last page of every request on the device
        for q in range(R):
            toks = np.arange((n[q] - 1) // E * E if E else n[q] - 1, n[q], dtype=np.int32)
            rows = rng.integers(0, 256, size=(toks.size, run.W), dtype=np.uint8)
            run.append(np.full(toks.size, q, np.int32), toks, np.full(toks.size, n[q]), rows,
                       layer=layer)
    for step in range(steps):
        n = np.minimum(n + 1, L).astype(np.int32)
        B = int(rng.integers(1, R + 1))
        rpi = rng.permutation(R)[:B].astype(np.int32)
        for layer in range(layers):
            # every request decodes a token; the call then selects for B of them
            every = np.arange(R, dtype=np.int32)
            req, tok = every, n - 1
            if rewrites:
                old = rng.integers(0, n).astype(np.int32)
                keep = old != tok
                req = np.concatenate([req, every[keep]])
                tok = np.concatenate([tok, old[keep]])
            rows = rng.integers(0, 256, size=(req.size, run.W), dtype=np.uint8)
            run.append(req, tok, n[req], rows, layer=layer)
            S = int(rng.integers(1, S_max + 1))
            span = 3 * max(E, 1) + 8
            recent = n[rpi][:, None, None] - 1 - rng.integers(0, span, size=(B, S, K))
            spread = rng.integers(0, n[rpi][:, None, None], size=(B, S, K))
            topk = np.where(rng.random((B, S, K)) < 0.4, recent, spread).astype(np.int32)
            topk[rng.random(topk.shape) < 0.03] = -1
            run.call(topk, rpi, n[rpi], layer=layer, properties=(step % 5 == 4))


@pytest.mark.parametrize("dense", [False, True], ids=["hash", "dense"])
@pytest.mark.parametrize("E", [1, 7, 64, 256])
def test_decode_loop_extra_page(dense, E):
    rng = np.random.default_rng(100 + E + 1000 * dense)
    R, L, H, K, S_max = 6, 3000, 200, 300, 3
    run = ParityRun(R, L, W.ROW_BYTES, H, K, S_max, dense=dense, extra_page=E, own_pool=True)
    _decode_loop(run, rng, R, L, K, S_max, E, steps=14)


def test_decode_loop_two_layers_overflow():
    # small hot buffer: overflow every call; two layers keep separate rows
    rng = np.random.default_rng(7)
    R, L, H, K, S_max, E = 4, 1500, 40, 128, 4, 32
    run = ParityRun(R, L, W.ROW_BYTES, H, K, S_max, layers=2, extra_page=E, own_pool=True)
    _decode_loop(run, rng, R, L, K, S_max, E, steps=10, layers=2)


def test_write_back_without_extra_page():
    # E = 0: appended rows reach the host pool and the hot copies only
    rng = np.random.default_rng(8)
    R, L, H, K, S_max = 5, 2000, 150, 200, 2
    run = ParityRun(R, L, W.ROW_BYTES, H, K, S_max, extra_page=0, own_pool=True)
    _decode_loop(run, rng, R, L, K, S_max, 0, steps=10)


def test_append_skips_out_of_range_entries():
    rng = np.random.default_rng(9)
    R, L, H, K, E = 4, 500, 32, 16, 8
    run = ParityRun(R, L, W.ROW_BYTES, H, K, 1, extra_page=E, own_pool=True)
    req = np.array([0, 1, -1, 4, 2, 3, 3], np.int32)
    tok = np.array([10, 499, 5, 5, -2, 50, 60], np.int32)
    sl = np.array([11, 500, 10, 10, 10, 50, 61], np.int32)  # (3, 50): t == seq_len
    rows = rng.integers(0, 256, size=(7, W.ROW_BYTES), dtype=np.uint8)
    run.append(req, tok, sl, rows, expect_skipped=4)
    # the valid ones were applied: select them through the extra page
    # 10 is on the extra page [8, 11); 8 and 9, never appended, are not selected
    topk = np.array([[[10, 3, 1, 0, 2, 4, 5, 6, 7, -1, 11, 12, 13, 14, 15, 20]]], np.int32)
    run.call(topk, np.array([0], np.int32), np.array([11], np.int32), properties=True)


def test_extra_page_full_size_c2():
    """The 64-request, 32768-token workload with a 256-row extra page: the
    newest token of every request is appended before each call."""
    w = W.WORKLOADS["C2"]
    E = 256
    stream = W.TopkStream(w)
    rpi = W.req_pool_indices(w)
    sl = W.seq_lens(w)
    rng = np.random.default_rng(12)
    run = ParityRun(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps, dense=True,
                    extra_page=E, own_pool=True)
    q = np.arange(w.batch, dtype=np.int32)
    page = np.arange(w.seq_len - E, w.seq_len, dtype=np.int32)
    run.append(np.repeat(q, E), np.tile(page, w.batch), np.full(w.batch * E, w.seq_len),
               rng.integers(0, 256, size=(w.batch * E, w.row_bytes), dtype=np.uint8))
    for c in range(5):
        run.append(q, np.full(w.batch, w.seq_len - 1, np.int32), sl[q],
                   rng.integers(0, 256, size=(w.batch, w.row_bytes), dtype=np.uint8))
        g = run.call(stream.next_call(), rpi, sl, compare_rows=(c == 4), properties=(c == 4))
        assert g["stats"][:, 8].sum() > 0  # the Zipf draws favour the newest positions


def test_extra_page_covers_whole_sequence():
    """E >= L: every valid entry is on the extra page; no lookup, no miss, and
    the policy state changes only by its epoch."""
    rng = np.random.default_rng(13)
    R, L, H, K, E = 3, 200, 16, 64, 256
    run = ParityRun(R, L, W.ROW_BYTES, H, K, 2, extra_page=E, own_pool=True)
    n = np.array([200, 57, 1], np.int32)
    for q in range(R):
        toks = np.arange(n[q], dtype=np.int32)
        run.append(np.full(n[q], q, np.int32), toks, np.full(n[q], n[q]),
                   rng.integers(0, 256, size=(n[q], W.ROW_BYTES), dtype=np.uint8))
    for c in range(3):
        topk = rng.integers(-5, 210, size=(R, 2, K)).astype(np.int32)
        g = run.call(topk, np.arange(R, dtype=np.int32), n, properties=True)
        assert (g["stats"][:, [0, 2, 3]] == 0).all()


def test_extra_page_deferred_copy_plan():
    """Deferred copy: the recorded miss plan holds the misses only; the extra
    page needs no copy."""
    rng = np.random.default_rng(14)
    R, L, H, K, S_max, E = 4, 2000, 100, 200, 2, 64
    run = ParityRun(R, L, W.ROW_BYTES, H, K, S_max, deferred=True, extra_page=E, own_pool=True)
    _decode_loop(run, rng, R, L, K, S_max, E, steps=6, rewrites=False)


def test_largest_extra_page():
    """E = HS_MAX_EXTRA_PAGE (65536) on 70000-token requests: the extra page
    is [65536, n) once n passes 65536 and the whole sequence before that."""
    import sparse_attention_kv_swap_gb300 as pkg
    E = pkg.binding.HS_MAX_EXTRA_PAGE
    rng = np.random.default_rng(15)
    R, L, H, K = 2, 70000, 64, 512
    run = ParityRun(R, L, W.ROW_BYTES, H, K, 1, extra_page=E, own_pool=True)
    n = np.array([70000, 65536], np.int32)
    for q in range(R):
        toks = np.arange((n[q] - 1) // E * E, n[q], dtype=np.int32)
        run.append(np.full(toks.size, q, np.int32), toks, np.full(toks.size, n[q]),
                   rng.integers(0, 256, size=(toks.size, W.ROW_BYTES), dtype=np.uint8))
    for c in range(3):
        recent = n[:, None, None] - 1 - rng.integers(0, 6000, size=(R, 1, K))
        topk = np.where(rng.random((R, 1, K)) < 0.5, recent,
                        rng.integers(0, n[:, None, None], size=(R, 1, K))).astype(np.int32)
        g = run.call(topk, np.arange(R, dtype=np.int32), n, properties=True)
        assert g["stats"][1, 8] == int(((topk[1] >= 0) & (topk[1] < n[1])).sum())  # all extra


def test_noalloc_entry_with_extra_page_matches_swap_in():
    """hs_swap_in_noalloc serves the extra page exactly as hs_swap_in does."""
    import torch
    import sparse_attention_kv_swap_gb300 as pkg
    from sparse_attention_kv_swap_gb300 import binding as B
    from sparse_attention_kv_swap_gb300.cache import SwapInCache
    R, L, H, K, S, E = 4, 2000, 100, 200, 2, 32
    cfg = pkg.make_config(R, L, W.ROW_BYTES, H, K, S, extra_page_size=E)
    pool = torch.empty((R, L, W.ROW_BYTES), dtype=torch.uint8, pin_memory=True)
    W.fill_host_pool(pool.numpy(), 0)
    a, b = SwapInCache(cfg, host_pools=[pool]), SwapInCache(cfg, host_pools=[pool])
    for c in (a, b):
        c.device_kv[0].zero_()
    rng = np.random.default_rng(16)
    rpi = torch.tensor([2, 0, 3], dtype=torch.int32, device="cuda")
    sl = torch.tensor([2000, 1500, 777], dtype=torch.int32, device="cuda")
    for call in range(3):
        topk_np = rng.integers(-2, L, size=(3, S, K)).astype(np.int32)
        topk_np[:, :, :20] = (sl.cpu().numpy()[:, None, None] - 1
                              - rng.integers(0, 2 * E, size=(3, S, 20)))
        topk = torch.from_numpy(topk_np).cuda()
        outs = []
        for c, fn in ((a, B.hs_swap_in), (b, B.hs_swap_in_noalloc)):
            o = {"device_locs": torch.empty((3, S, K), dtype=torch.int32, device="cuda"),
                 "stats": torch.empty((3, B.HS_NUM_STATS), dtype=torch.int32, device="cuda")}
            fn(c.handle, rpi, sl, topk, 0, o["device_locs"], o["stats"])
            outs.append(o)
        torch.cuda.synchronize()
        assert torch.equal(outs[0]["device_locs"], outs[1]["device_locs"])
        assert torch.equal(outs[0]["stats"], outs[1]["stats"])
        assert int(outs[0]["stats"][:, B.HS_STAT_EXTRA].sum()) > 0
    for q in (0, 2, 3):
        sa, sb = a.export_request_state(0, q), b.export_request_state(0, q)
        for k in ("tok", "ep", "phys"):
            assert (sa[k] == sb[k]).all()
    assert torch.equal(a.device_kv[0][: R * (H + S * K)], b.device_kv[0][: R * (H + S * K)])
    assert a.status() == (0, 0) and b.status() == (0, 0)
