"""The multi-GPU path on the CPU: two gloo ranks.

The swap-in shards by request: each request's cache state, host rows and
device rows are independent, so N GPUs run N replicas with no collective on
the data path.  bench.py times each replica and reduces only the timing
(max over ranks).  Here two gloo ranks on CPU check:
  * the timing reduction gives every rank the slowest rank's time and the
    whole-job rate counts every replica;
  * serving the requests split over two ranks (rank r takes every other
    request, through the oracle) gives exactly the results of one process
    serving all of them: no exchange between ranks is needed.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist

    import bench
    import hs_workloads as W
    from oracle import Oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(torch, 1.0 + rank, world, torch.device("cpu"))
        rate = bench.whole_job_rate(1000, world, ms)
        # requests b with b % world == rank
        w = W.scaled(W.WORKLOADS["C3"], batch=6, top_k=128, seq_len=2048, hot_buffer=256)
        stream = W.TopkStream(w)
        rpi, sl = W.req_pool_indices(w), W.seq_lens(w)
        mine = np.arange(w.batch) % world == rank
        pool = np.empty((w.batch, w.seq_len, 32), np.uint8)
        W.fill_host_pool(pool, 0)
        C = w.steps * w.top_k
        o = Oracle(w.batch, w.seq_len, 32, w.hot_buffer, w.top_k, w.steps, 1)
        dev = np.zeros((w.batch * (w.hot_buffer + C), 32), np.uint8)
        locs = []
        for c in range(4):
            topk = stream.next_call()
            out = o.swap_in(0, pool, dev, rpi[mine], sl[mine], topk[mine])
            locs.append(out["locs"])
        np.savez(os.path.join(out_dir, "rank%d.npz" % rank), ms=ms, rate=rate, mine=mine,
                 locs=np.stack(locs), dev=dev)
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas(tmp_path):
    import socket

    import torch.multiprocessing as mp
    sys.path.insert(0, ROOT)
    import hs_workloads as W
    from oracle import Oracle

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [np.load(tmp_path / ("rank%d.npz" % r)) for r in range(2)]
    for r in res:
        assert float(r["ms"]) == 2.0  # every rank sees the slowest rank's time
        assert abs(float(r["rate"]) - 2 * 1000 / 2e-3) < 1e-6
    # one process serving all requests
    w = W.scaled(W.WORKLOADS["C3"], batch=6, top_k=128, seq_len=2048, hot_buffer=256)
    stream = W.TopkStream(w)
    rpi, sl = W.req_pool_indices(w), W.seq_lens(w)
    pool = np.empty((w.batch, w.seq_len, 32), np.uint8)
    W.fill_host_pool(pool, 0)
    C = w.steps * w.top_k
    o = Oracle(w.batch, w.seq_len, 32, w.hot_buffer, w.top_k, w.steps, 1)
    dev = np.zeros((w.batch * (w.hot_buffer + C), 32), np.uint8)
    for c in range(4):
        out = o.swap_in(0, pool, dev, rpi, sl, stream.next_call())
        for r in res:
            assert (out["locs"][r["mine"]] == r["locs"][c]).all()
    # each rank's device rows are exactly the single-process rows of its requests
    rows_per_q = w.hot_buffer + C
    for r in res:
        for b in np.nonzero(r["mine"])[0]:
            q = int(rpi[b])
            sl_q = slice(q * rows_per_q, (q + 1) * rows_per_q)
            assert (r["dev"][sl_q] == dev[sl_q]).all()
