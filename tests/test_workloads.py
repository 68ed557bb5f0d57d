"""The seeded input streams follow their stated recipe (CPU only).

Every top-k step is K distinct in-range indices; at least round(reuse * K)
of them repeat the previous step; the Zipf streams favour recent positions;
the clustered stream stays near its fixed centres; everything is
reproducible from the seeds; and a filled host pool holds exactly the rows
host_rows() defines.  Batches are cut to a few requests to keep this quick:
the recipe is per request."""
import numpy as np
import pytest

import hs_workloads as W


def _stream(name, batch=4, calls=3):
    w = W.scaled(W.WORKLOADS[name], batch=min(batch, W.WORKLOADS[name].batch))
    st = W.TopkStream(w)
    return w, st, st.calls(calls)


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_steps_are_distinct_in_range_and_reuse_the_previous_step(name):
    w, _, calls = _stream(name)
    K, L = w.top_k, w.seq_len
    n_reuse = int(round(w.reuse * K))
    for b in range(w.batch):
        prev = None
        for c in calls:
            assert c.shape == (w.batch, w.steps, K) and c.dtype == np.int32
            for s in range(w.steps):
                step = c[b, s]
                assert np.unique(step).size == K
                assert step.min() >= 0 and step.max() < L
                if prev is not None:
                    # fresh draws may also hit the previous step, never fewer
                    assert np.intersect1d(step, prev).size >= n_reuse
                prev = step


@pytest.mark.parametrize("name", ["C2", "C3", "C4"])
def test_zipf_streams_favour_recent_positions(name):
    w, _, calls = _stream(name)
    dist = np.concatenate([w.seq_len - 1 - c.reshape(-1).astype(np.int64) for c in calls])
    assert np.mean(dist < w.seq_len // 10) > 0.4  # uniform draws would give 0.1


def test_uniform_stream_is_not_recency_biased():
    w, _, calls = _stream("C1")
    dist = np.concatenate([w.seq_len - 1 - c.reshape(-1).astype(np.int64) for c in calls])
    assert np.mean(dist < w.seq_len // 10) < 0.25


def test_cluster_stream_stays_near_its_centres():
    w, st, calls = _stream("C5", batch=3)
    for c in calls:
        for b in range(w.batch):
            t = c[b, 0].astype(np.int64)
            near = np.min(np.abs(t[:, None] - st._centres[b][None, :]), axis=1)
            assert near.max() <= 8 * w.cluster_sigma
            # the selection touches few of the request's pages
            assert np.unique(t // w.page_size).size <= w.clusters * 8


def test_streams_and_request_slots_are_reproducible():
    for name in sorted(W.WORKLOADS):
        _, _, a = _stream(name, calls=2)
        _, _, b = _stream(name, calls=2)
        assert all((x == y).all() for x, y in zip(a, b))
        w = W.WORKLOADS[name]
        rpi = W.req_pool_indices(w)
        assert sorted(rpi.tolist()) == list(range(w.batch))
        assert (W.req_pool_indices(w) == rpi).all()


def test_filled_pool_equals_host_rows():
    pool = np.empty((3, 50, W.ROW_BYTES), dtype=np.uint8)
    W.fill_host_pool(pool, 2, chunk_rows=17, threads=2)
    q = np.repeat(np.arange(3), 50)
    t = np.tile(np.arange(50), 3)
    assert (pool.reshape(150, W.ROW_BYTES) == W.host_rows(2, q, t)).all()
    other = np.empty_like(pool)
    W.fill_host_pool(other, 3)
    assert (other != pool).any()  # a different layer gives different rows
