"""Memory plumbing around the C ABI: allocates the caller-owned buffers with
PyTorch (pinned host pools, device KV buffers, state, workspace) and forwards
each call to the library.  Nothing here computes any part of the swap-in."""
from __future__ import annotations

from typing import Dict, List, Optional

import torch

from . import binding as B


class SwapInCache:
    """One swap-in cache: pinned host pools + device hot buffers for all layers."""

    def __init__(self, cfg: B.HsConfig, host_pools: Optional[List[torch.Tensor]] = None,
                 device: Optional[torch.device] = None, stream=None):
        rc = B.hs_config_check(cfg)
        if rc != B.HS_OK:
            raise B.HsError(rc, "hs_config_check")
        self.cfg = cfg
        self.device = torch.device(device or "cuda")
        R, L, W = cfg.num_requests, cfg.max_seq_len, cfg.item_size_bytes
        self.H, self.C = cfg.hot_buffer_size, cfg.max_steps * cfg.top_k
        if host_pools is None:
            host_pools = [torch.empty((R, L, W), dtype=torch.uint8, pin_memory=True)
                          for _ in range(cfg.num_layers)]
        self.host_pools = host_pools
        self.E = cfg.extra_page_size
        rows = B.hs_device_kv_bytes(cfg) // W  # hot + scratch rows, then the extra pages
        self.device_kv = [torch.empty((rows, W), dtype=torch.uint8, device=self.device)
                          for _ in range(cfg.num_layers)]
        self.state = torch.empty(B.hs_state_bytes(cfg), dtype=torch.uint8, device=self.device)
        self.workspace = torch.empty(B.hs_workspace_bytes(cfg), dtype=torch.uint8,
                                     device=self.device)
        self.handle = B.hs_create_state(cfg, self.host_pools, self.device_kv, self.state,
                                        self.workspace, stream)

    def swap_in(self, req_pool_indices: torch.Tensor, seq_lens: torch.Tensor,
                topk: torch.Tensor, layer_id: int = 0, stats: bool = False, plan: bool = False,
                out: Optional[Dict[str, torch.Tensor]] = None, stream=None):
        Bn, S, K = topk.shape
        o = dict(out or {})
        if "device_locs" not in o:
            o["device_locs"] = torch.empty((Bn, S, K), dtype=torch.int32, device=self.device)
        if stats and "stats" not in o:
            o["stats"] = torch.empty((Bn, B.HS_NUM_STATS), dtype=torch.int32, device=self.device)
        if plan and "miss_src" not in o:
            o["miss_src"] = torch.full((Bn, self.C), -1, dtype=torch.int64, device=self.device)
            o["miss_dst"] = torch.full((Bn, self.C), -1, dtype=torch.int64, device=self.device)
            o["miss_count"] = torch.empty(Bn, dtype=torch.int32, device=self.device)
        B.hs_swap_in(self.handle, req_pool_indices, seq_lens, topk, layer_id, o["device_locs"],
                     o.get("stats"), o.get("miss_src"), o.get("miss_dst"), o.get("miss_count"),
                     stream)
        return o

    def page_table(self, topk: torch.Tensor, seq_lens: torch.Tensor, page_size: int,
                   out: Optional[Dict[str, torch.Tensor]] = None, stream=None):
        Bn, S, K = topk.shape
        o = dict(out or {})
        o.setdefault("pages", torch.empty((Bn, S * K), dtype=torch.int32, device=self.device))
        o.setdefault("num_pages", torch.empty(Bn, dtype=torch.int32, device=self.device))
        o.setdefault("token_page", torch.empty((Bn, S, K), dtype=torch.int32, device=self.device))
        B.hs_page_table(topk, seq_lens, self.cfg.max_seq_len, page_size, o["pages"],
                        o["num_pages"], o["token_page"], stream)
        return o

    def append_rows(self, req: torch.Tensor, tok: torch.Tensor, seq_lens: torch.Tensor,
                    rows: torch.Tensor, layer_id: int = 0, stream=None) -> None:
        """Write-back of newly decoded KV rows (host pool, extra page, hot copy)."""
        B.hs_append_rows(self.handle, layer_id, req, tok, seq_lens, rows, stream)

    def reset_requests(self, req_pool_indices: torch.Tensor, stream=None) -> None:
        B.hs_reset_requests(self.handle, req_pool_indices, stream)

    def totals(self, layer_id: int = 0, reset: bool = False, stream=None):
        """Running sums of the per-request counters of one layer (HS_STAT_* order)."""
        return B.hs_get_stats(self.handle, layer_id, reset, stream)

    def status(self, stream=None):
        return B.hs_get_status(self.handle, stream)

    def export_request_state(self, layer_id: int, request: int, stream=None):
        return B.hs_export_request_state(self.handle, layer_id, request, stream)

    def close(self) -> None:
        self.handle.close()
