"""Runs the same call sequence through the CUDA library and the CPU oracle
and compares every observable output bit for bit."""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

import hs_workloads as W
from checker import check_call


def map_consistent(st: dict) -> Optional[str]:
    """The dense index maps exactly the resident tokens to their slots."""
    m = st["bank"]  # the dense map, widened to int64 [max_seq_len]
    got = {int(t): int(v) for t, v in enumerate(m.tolist()) if v != -1}
    want = {int(t): v for v, t in enumerate(st["tok"].tolist()) if t != -1}
    if got != want:
        return "dense map differs from the slot table"
    if int((st["tok"] != -1).sum()) != int(st["ctrl"][1]):
        return "resident counter is wrong"
    if int(st["ctrl"][3]) != 0:
        return "request lock still held"
    return None


def bank_consistent(st: dict, dense: bool = False) -> Optional[str]:
    """The hash bank holds exactly the resident (token, slot) pairs."""
    if dense:
        return map_consistent(st)
    bank = st["bank"]
    live = bank[bank >= 0]
    pairs = set(zip((live >> 32).astype(np.int64).tolist(),
                    (live & 0xFFFFFFFF).astype(np.int64).tolist()))
    if len(pairs) != live.size:
        return "duplicate hash entries"
    want = {(int(t), v) for v, t in enumerate(st["tok"].tolist()) if t != -1}
    if pairs != want:
        return "hash entries differ from the slot table"
    if int((bank != -1).sum()) != int(st["ctrl"][2]):
        return "used-entry counter is wrong"
    if int((st["tok"] != -1).sum()) != int(st["ctrl"][1]):
        return "resident counter is wrong"
    if int(st["ctrl"][3]) != 0:
        return "request lock still held"
    return None


class ParityRun:
    def __init__(self, R: int, L: int, width: int, H: int, K: int, S_max: int, layers: int = 1,
                 max_batch: Optional[int] = None, pools=None, deferred: bool = False,
                 dense: bool = False, extra_page: int = 0, own_pool: bool = False):
        """own_pool: the oracle works on its own copy of the host pools (needed
        once rows are appended, so that the library's write-back is compared
        with the oracle's instead of being overwritten by it)."""
        self.deferred = deferred
        self.dense = dense
        self.E = extra_page
        import sparse_attention_kv_swap_gb300 as pkg
        from oracle import Oracle
        from sparse_attention_kv_swap_gb300.cache import SwapInCache
        self.R, self.L, self.W, self.H, self.K, self.S_max = R, L, width, H, K, S_max
        self.C = S_max * K
        self.layers = layers
        cfg = pkg.make_config(R, L, width, H, K, S_max, layers, max_batch, index_kind=int(dense),
                              extra_page_size=extra_page)
        if pools is None:
            pools = []
            for l in range(layers):
                p = torch.empty((R, L, width), dtype=torch.uint8, pin_memory=True)
                W.fill_host_pool(p.numpy(), l)
                pools.append(p)
        self.pools = pools
        self.cache = SwapInCache(cfg, host_pools=pools)
        for t in self.cache.device_kv:
            t.zero_()
        if deferred:
            pkg.hs_set_defer_copy(self.cache.handle, True)
        self.oracle = Oracle(R, L, width, H, K, S_max, layers, extra_page_size=extra_page)
        self.mirror = [np.zeros((self.oracle.device_rows(), width), dtype=np.uint8)
                       for _ in range(layers)]
        self.opools = [p.numpy().copy() if own_pool else p.numpy() for p in pools]
        self.calls = 0

    def append(self, req: np.ndarray, tok: np.ndarray, seq_lens: np.ndarray, rows: np.ndarray,
               layer: int = 0, expect_skipped: int = 0) -> None:
        """Write-back through the library and the oracle; compares the host
        pool rows written and every device row."""
        req = np.ascontiguousarray(req, dtype=np.int32)
        tok = np.ascontiguousarray(tok, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        rows = np.ascontiguousarray(rows, dtype=np.uint8)
        dev = lambda a: torch.from_numpy(a).cuda()
        self.cache.append_rows(dev(req), dev(tok), dev(seq_lens), dev(rows), layer)
        skipped = self.oracle.append_rows(layer, self.opools[layer], self.mirror[layer], req, tok,
                                          seq_lens, rows)
        torch.cuda.synchronize()
        assert skipped == expect_skipped
        rc, flags = self.cache.status()
        import sparse_attention_kv_swap_gb300 as pkg
        want = pkg.binding.HS_STATUS_BAD_APPEND if skipped else 0
        assert flags == want, "append: device status flags %#x, expected %#x" % (flags, want)
        ok = (req >= 0) & (req < self.R) & (tok >= 0) & (tok < np.minimum(seq_lens, self.L))
        got = self.pools[layer].numpy()[req[ok], tok[ok]]
        assert (got == self.opools[layer][req[ok], tok[ok]]).all(), "appended host rows differ"
        diff = np.nonzero((self.cache.device_kv[layer].cpu().numpy() != self.mirror[layer])
                          .any(axis=1))[0]
        assert diff.size == 0, "append: %d device rows differ (first %d)" % (diff.size, diff[0])

    def gpu_state(self, layer: int, q: int) -> dict:
        return self.cache.export_request_state(layer, q)

    def call(self, topk: np.ndarray, rpi: np.ndarray, seq_lens: np.ndarray, layer: int = 0,
             compare_rows: bool = True, properties: bool = False, plan: bool = False,
             threads: int = 8) -> Dict[str, np.ndarray]:
        topk = np.ascontiguousarray(topk, dtype=np.int32)
        rpi = np.ascontiguousarray(rpi, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        before = {int(q): self.gpu_state(layer, int(q)) for q in rpi} if properties else None
        out = self.cache.swap_in(torch.from_numpy(rpi).cuda(), torch.from_numpy(seq_lens).cuda(),
                                 torch.from_numpy(topk).cuda(), layer, stats=True,
                                 plan=plan or self.deferred)
        if self.deferred:
            # the rows arrive only when the recorded plan is replayed, here on
            # a second stream ordered after the call
            import sparse_attention_kv_swap_gb300 as pkg
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            pkg.hs_copy_planned(self.cache.handle, layer, out["miss_src"], out["miss_dst"],
                                out["miss_count"], stream=side)
            torch.cuda.current_stream().wait_stream(side)
            plan = True
        ref = self.oracle.swap_in(layer, self.opools[layer], self.mirror[layer], rpi,
                                  seq_lens, topk, want_plan=plan, num_threads=threads)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in out.items()}
        self.calls += 1
        tag = "call %d layer %d" % (self.calls, layer)
        bad = np.argwhere(g["device_locs"] != ref["locs"])
        assert bad.size == 0, "%s: %d locations differ, first at %s" % (tag, len(bad),
                                                                       bad[0].tolist())
        assert (g["stats"] == ref["stats"]).all(), "%s: counters differ\n%s\n%s" % (
            tag, g["stats"], ref["stats"])
        if plan:
            for b in range(len(rpi)):
                U = int(ref["miss_count"][b])
                assert g["miss_count"][b] == U
                assert (g["miss_src"][b, :U] == ref["miss_src"][b, :U]).all()
                assert (g["miss_dst"][b, :U] == ref["miss_dst"][b, :U]).all()
        for q in rpi.tolist():
            gs = self.gpu_state(layer, q)
            os_ = self.oracle.request_state(layer, q)
            for k in ("tok", "ep", "phys"):
                assert (gs[k] == os_[k]).all(), "%s q=%d: state %s differs" % (tag, q, k)
            assert gs["epoch"] == os_["epoch"], "%s q=%d: epoch differs" % (tag, q)
            err = bank_consistent(gs, self.dense)
            assert err is None, "%s q=%d: %s" % (tag, q, err)
        dev = self.cache.device_kv[layer]
        if compare_rows:
            got = dev.cpu().numpy()
            diff = np.nonzero((got != self.mirror[layer]).any(axis=1))[0]
            assert diff.size == 0, "%s: %d device rows differ (first %d)" % (tag, diff.size,
                                                                             diff[0])
        if properties:
            after = {int(q): self.gpu_state(layer, int(q)) for q in rpi}

            def rows_at(locs):
                idx = torch.from_numpy(np.asarray(locs, dtype=np.int64)).cuda()
                return dev.index_select(0, idx).cpu().numpy()

            opool = self.opools[layer]
            check_call(before, after, topk, rpi, seq_lens, self.L, self.H, self.C,
                       g["device_locs"], g["stats"], rows_at=rows_at,
                       host_row=lambda q, toks: opool[q, np.asarray(toks)],
                       extra_page=self.E, R=self.R)
        rc, flags = self.cache.status()
        assert flags == 0, "%s: device status flags %#x" % (tag, flags)
        return g
