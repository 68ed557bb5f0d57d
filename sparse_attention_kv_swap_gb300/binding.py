"""Thin ctypes binding of the C ABI in include/hisparse_swap.h.

Every function here only marshals arguments (tensor pointers, sizes, the
current CUDA stream) and calls the library of the same name; all work runs
in the library's CUDA kernels.  There is no fallback: if the library has not
been built for this machine, loading it raises.

Tensors: device tensors are torch CUDA tensors, host pools are pinned torch
CPU tensors (``pin_memory=True``); all must be contiguous.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Dict, List, Optional, Sequence

from . import build as _build

HS_OK = 0
HS_ERR_INVALID_ARG = -1
HS_ERR_UNSUPPORTED = -2
HS_ERR_CUDA = -3
HS_ERR_DEVICE_STATUS = -4
HS_ERR_TIMEOUT = -5

HS_STATUS_BAD_REQUEST = 0x1
HS_STATUS_DUPLICATE_REQUEST = 0x2
HS_STATUS_SEQ_LEN_CLAMPED = 0x4
HS_STATUS_PROBE_LIMIT = 0x8
HS_STATUS_TABLE_FULL = 0x10
HS_STATUS_BAD_APPEND = 0x20
HS_STATUS_BAD_PLAN = 0x40

HS_INDEX_HASH = 0
HS_INDEX_DENSE = 1

HS_STAT_EXTRA = 8
HS_NUM_STATS = 9
STAT_NAMES = ("hits", "hit_slots", "dup_misses", "unique_misses", "admitted", "evicted",
              "overflow", "invalid", "extra")
HS_MAX_EXTRA_PAGE = 65536
HS_MAX_ITEM_BYTES = 65536
HS_NOALLOC_SCRATCH_BYTES = 16 << 20
TIMELINE_WORDS_PER_ROW = 8 * 16  # hs_set_timeline: [batch][8 ranks][16 words]

HEADER = os.path.join(_build.INCLUDE, "hisparse_swap.h")


class HsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (where, status_string(code), code))


class HsConfig(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("item_size_bytes", ctypes.c_int32), ("hot_buffer_size", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("max_steps", ctypes.c_int32),
                ("num_layers", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("index_kind", ctypes.c_int32), ("extra_page_size", ctypes.c_int32)]

    def as_dict(self) -> Dict[str, int]:
        return {name: getattr(self, name) for name, _ in self._fields_}


def make_config(num_requests: int, max_seq_len: int, item_size_bytes: int,
                hot_buffer_size: int, top_k: int, max_steps: int, num_layers: int = 1,
                max_batch: Optional[int] = None, index_kind: int = 0,
                extra_page_size: int = 0) -> HsConfig:
    """index_kind: HS_INDEX_HASH (0, hash banks) or HS_INDEX_DENSE (1, dense map);
    extra_page_size: rows of each request's extra page (0 = none)."""
    return HsConfig(num_requests, max_seq_len, item_size_bytes, hot_buffer_size, top_k,
                    max_steps, num_layers, num_requests if max_batch is None else max_batch,
                    index_kind, extra_page_size)


_lib = None
_lock = threading.Lock()
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_cfgp = ctypes.POINTER(HsConfig)


def _declare(lib) -> None:
    sig = {
        "hs_config_check": (ctypes.c_int, [_cfgp]),
        "hs_state_bytes": (ctypes.c_size_t, [_cfgp]),
        "hs_workspace_bytes": (ctypes.c_size_t, [_cfgp]),
        "hs_device_kv_bytes": (ctypes.c_size_t, [_cfgp]),
        "hs_host_pool_bytes": (ctypes.c_size_t, [_cfgp]),
        "hs_hash_size": (_i32, [_cfgp]),
        "hs_create_state": (ctypes.c_int, [_cfgp, _vp, _vp, _vp, ctypes.c_size_t, _vp,
                                           ctypes.c_size_t, _vp, ctypes.POINTER(_vp)]),
        "hs_destroy_state": (None, [_vp]),
        "hs_swap_in": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                                      _vp, _vp]),
        "hs_page_table": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp,
                                         _vp]),
        "hs_reset_requests": (ctypes.c_int, [_vp, _vp, _i32, _vp]),
        "hs_get_status": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint32), _vp]),
        "hs_get_stats": (ctypes.c_int, [_vp, _i32, _vp, _i32, _vp]),
        "hs_export_request_state": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                                   _vp]),
        "hs_swap_in_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp,
                                              _vp, _vp, _vp, _vp]),
        "hs_append_rows": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp]),
        "hs_set_timeline": (ctypes.c_int, [_vp, _vp]),
        "hs_set_defer_copy": (ctypes.c_int, [_vp, _i32]),
        "hs_copy_planned": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _i32, _vp]),
        "hs_set_copy_ctas": (ctypes.c_int, [_vp, _i32]),
        "hs_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "hs_version": (_i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args


def load_library(path: Optional[str] = None, build_if_missing: bool = False):
    """Load the in-tree library (optionally building it first)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.lib_path()
        if not os.path.exists(p):
            if not build_if_missing:
                raise RuntimeError("CUDA library %s is not built; run __graft_entry__.build() or "
                                   "python -m sparse_attention_kv_swap_gb300.build" % p)
            p = _build.build()
        lib = ctypes.CDLL(p)
        _declare(lib)
        if path is None:
            _lib = lib
        return lib


def header_symbols(header: str = HEADER) -> List[str]:
    """Names of the functions the public header declares."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hs_[a-z_0-9]+)\s*\(", text)))


def status_string(code: int) -> str:
    try:
        return load_library().hs_status_string(code).decode()
    except Exception:
        return "status %d" % code


def _check(code: int, where: str) -> None:
    if code != HS_OK:
        raise HsError(code, where)


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    want = getattr(_call_device, "index", None)
    if want is not None and stream.device.index != want:
        raise ValueError("the stream is on cuda:%d, the call runs on cuda:%d"
                         % (stream.device.index, want))
    return int(stream.cuda_stream)


_call_device = threading.local()  # device of the handle whose call is being marshalled


class _on_device:
    """Makes device `index` current for one library call (a handle's calls
    must be made on its own device) and has _dptr and _stream_ptr reject
    device tensors and streams of another device.  `index` None checks and
    switches nothing."""

    def __init__(self, index: Optional[int]):
        self.index = index

    def __enter__(self):
        import torch
        self.outer = getattr(_call_device, "index", None)
        _call_device.index = self.index
        self.prev = None
        if self.index is not None and torch.cuda.is_available():
            prev = torch.cuda.current_device()
            if prev != self.index:
                torch.cuda.set_device(self.index)
                self.prev = prev
        return self

    def __exit__(self, *exc):
        _call_device.index = self.outer
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def _dptr(t, dtype=None, name="tensor") -> int:
    """Address of a tensor the kernels read or write: device memory, or pinned
    (mapped) host memory, which the device addresses directly.  Inside
    _on_device, a device tensor must be on that device."""
    if t is None:
        return 0
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must have dtype %s" % (name, dtype))
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("%s must be in device memory or pinned host memory" % name)
    want = getattr(_call_device, "index", None)
    if t.is_cuda and want is not None and t.device.index != want:
        raise ValueError("%s is on cuda:%d, the call runs on cuda:%d" % (name, t.device.index,
                                                                        want))
    return int(t.data_ptr())


def _hptr(t, name="tensor") -> int:
    """Address of a host pool: pinned, or pageable where the library accepts it
    (it checks the memory kind itself)."""
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return int(t.data_ptr())


def _shape(t, shape, name) -> None:
    """The kernels trust the sizes: check them before any launch."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _swap_in_shapes(handle, req_pool_indices, seq_lens, topk, device_locs, stats, miss_src,
                    miss_dst, miss_count):
    if topk.dim() != 3:
        raise ValueError("topk must be [batch, steps, top_k]")
    B, S, K = topk.shape
    cfg = handle.cfg
    if K != cfg.top_k:
        raise ValueError("topk's last dimension %d differs from the config's top_k %d"
                         % (K, cfg.top_k))
    C = cfg.max_steps * cfg.top_k
    _shape(req_pool_indices, (B,), "req_pool_indices")
    _shape(seq_lens, (B,), "seq_lens")
    _shape(device_locs, (B, S, K), "device_locs")
    _shape(stats, (B, HS_NUM_STATS), "stats")
    _shape(miss_src, (B, C), "miss_src")
    _shape(miss_dst, (B, C), "miss_dst")
    _shape(miss_count, (B,), "miss_count")
    return B, S, K


# ---- sizes -----------------------------------------------------------------

def hs_config_check(cfg: HsConfig) -> int:
    return load_library().hs_config_check(ctypes.byref(cfg))


def hs_state_bytes(cfg: HsConfig) -> int:
    return load_library().hs_state_bytes(ctypes.byref(cfg))


def hs_workspace_bytes(cfg: HsConfig) -> int:
    return load_library().hs_workspace_bytes(ctypes.byref(cfg))


def hs_device_kv_bytes(cfg: HsConfig) -> int:
    return load_library().hs_device_kv_bytes(ctypes.byref(cfg))


def hs_host_pool_bytes(cfg: HsConfig) -> int:
    return load_library().hs_host_pool_bytes(ctypes.byref(cfg))


def hs_hash_size(cfg: HsConfig) -> int:
    return load_library().hs_hash_size(ctypes.byref(cfg))


def hs_version() -> int:
    return load_library().hs_version()


def hs_status_string(code: int) -> str:
    return load_library().hs_status_string(code).decode()


# ---- state -------------------------------------------------------------------

class StateHandle:
    """Owns the library's host handle; keeps the caller's tensors alive."""

    def __init__(self, ptr: int, cfg: HsConfig, keep: Sequence, device: int):
        self.ptr = ctypes.c_void_p(ptr)
        self.cfg = cfg
        self.device = device  # the CUDA device the handle and its buffers are on
        self._keep = list(keep)

    def close(self) -> None:
        if self.ptr:
            load_library().hs_destroy_state(self.ptr)
            self.ptr = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def hs_create_state(cfg: HsConfig, host_pools: Sequence, device_kvs: Sequence, state, workspace,
                    stream=None) -> StateHandle:
    lib = load_library()
    L = cfg.num_layers
    if len(host_pools) != L or len(device_kvs) != L:
        raise ValueError("need one host pool and one device KV buffer per layer")
    # The handle belongs to the device that holds its device buffers.
    if not state.is_cuda:
        raise ValueError("state must be in device memory")
    device = state.device.index
    with _on_device(device):
        hp = (ctypes.c_void_p * L)(*[_hptr(t, name="host pool") for t in host_pools])
        dk = (ctypes.c_void_p * L)(*[_dptr(t, name="device kv") for t in device_kvs])
        out = ctypes.c_void_p()
        rc = lib.hs_create_state(ctypes.byref(cfg), ctypes.cast(hp, _vp), ctypes.cast(dk, _vp),
                                 _dptr(state, name="state"), state.numel() * state.element_size(),
                                 _dptr(workspace, name="workspace"),
                                 workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream), ctypes.byref(out))
    _check(rc, "hs_create_state")
    return StateHandle(out.value, cfg, list(host_pools) + list(device_kvs) + [state, workspace],
                       device)


def hs_destroy_state(handle: StateHandle) -> None:
    handle.close()


def hs_swap_in(handle: StateHandle, req_pool_indices, seq_lens, topk, layer_id: int,
               device_locs, stats=None, miss_src=None, miss_dst=None, miss_count=None,
               stream=None) -> None:
    import torch
    B, S, K = _swap_in_shapes(handle, req_pool_indices, seq_lens, topk, device_locs, stats,
                              miss_src, miss_dst, miss_count)
    with _on_device(handle.device):
        rc = load_library().hs_swap_in(
            handle.ptr, _dptr(req_pool_indices, torch.int32, "req_pool_indices"),
            _dptr(seq_lens, torch.int32, "seq_lens"), _dptr(topk, torch.int32, "topk"), B, S,
            layer_id, _dptr(device_locs, torch.int32, "device_locs"),
            _dptr(stats, torch.int32, "stats"), _dptr(miss_src, torch.int64, "miss_src"),
            _dptr(miss_dst, torch.int64, "miss_dst"),
            _dptr(miss_count, torch.int32, "miss_count"), _stream_ptr(stream))
        _check(rc, "hs_swap_in")


def hs_page_table(topk, seq_lens, max_seq_len: int, page_size: int, pages, num_pages,
                  token_page, stream=None) -> None:
    import torch
    if topk.dim() != 3:
        raise ValueError("topk must be [batch, steps, top_k]")
    B, S, K = topk.shape
    _shape(seq_lens, (B,), "seq_lens")
    _shape(pages, (B, S * K), "pages")
    _shape(num_pages, (B,), "num_pages")
    _shape(token_page, (B, S, K), "token_page")
    # runs on the device of its inputs (the current device for pinned host inputs)
    with _on_device(topk.device.index if topk.is_cuda else None):
        rc = load_library().hs_page_table(
            _dptr(topk, torch.int32, "topk"), _dptr(seq_lens, torch.int32, "seq_lens"), B, S, K,
            max_seq_len, page_size, _dptr(pages, torch.int32, "pages"),
            _dptr(num_pages, torch.int32, "num_pages"), _dptr(token_page, torch.int32, "token_page"),
            _stream_ptr(stream))
        _check(rc, "hs_page_table")


def hs_reset_requests(handle: StateHandle, req_pool_indices, stream=None) -> None:
    import torch
    if req_pool_indices.dim() != 1:
        raise ValueError("req_pool_indices must be 1-D")
    with _on_device(handle.device):
        rc = load_library().hs_reset_requests(
            handle.ptr, _dptr(req_pool_indices, torch.int32, "req_pool_indices"),
            req_pool_indices.numel(), _stream_ptr(stream))
        _check(rc, "hs_reset_requests")


def hs_get_status(handle: StateHandle, stream=None):
    """Returns (code, flags); synchronises the stream and clears the flags."""
    flags = ctypes.c_uint32(0)
    with _on_device(handle.device):
        rc = load_library().hs_get_status(handle.ptr, ctypes.byref(flags), _stream_ptr(stream))
        if rc not in (HS_OK, HS_ERR_DEVICE_STATUS):
            _check(rc, "hs_get_status")
    return rc, flags.value


def hs_export_request_state(handle: StateHandle, layer_id: int, request: int, stream=None):
    import numpy as np
    cfg = handle.cfg
    H = cfg.hot_buffer_size
    C = cfg.max_steps * cfg.top_k
    tok = np.empty(H, np.int32)
    ep = np.empty(H, np.int32)
    phys = np.empty(H + C, np.int32)
    ctrl = np.empty(8, np.int32)
    # hash entries, or the dense map widened to int64 [max_seq_len]
    bank = np.empty(cfg.max_seq_len if cfg.index_kind == HS_INDEX_DENSE else hs_hash_size(cfg),
                    np.int64)
    with _on_device(handle.device):
        rc = load_library().hs_export_request_state(
            handle.ptr, layer_id, request, tok.ctypes.data, ep.ctypes.data, phys.ctypes.data,
            ctrl.ctypes.data, bank.ctypes.data, _stream_ptr(stream))
        _check(rc, "hs_export_request_state")
    return {"tok": tok, "ep": ep, "phys": phys, "ctrl": ctrl, "bank": bank,
            "epoch": int(ctrl[0])}


def hs_append_rows(handle: StateHandle, layer_id: int, req, tok, seq_lens, rows,
                   stream=None) -> None:
    """Write-back of newly decoded rows: req/tok/seq_lens int32 [n], rows uint8
    [n, W] on the device (see the C header)."""
    import torch
    n = req.numel()
    _shape(req, (n,), "req")
    _shape(tok, (n,), "tok")
    _shape(seq_lens, (n,), "seq_lens")
    _shape(rows, (n, handle.cfg.item_size_bytes), "rows")
    with _on_device(handle.device):
        rc = load_library().hs_append_rows(
            handle.ptr, layer_id, _dptr(req, torch.int32, "req"), _dptr(tok, torch.int32, "tok"),
            _dptr(seq_lens, torch.int32, "seq_lens"), _dptr(rows, torch.uint8, "rows"), n,
            _stream_ptr(stream))
        _check(rc, "hs_append_rows")


def hs_get_stats(handle: StateHandle, layer_id: int, reset: bool = False, stream=None):
    """Running sums of the HS_STAT_* counters of one layer: int64 [HS_NUM_STATS]."""
    import numpy as np
    out = np.zeros(HS_NUM_STATS, dtype=np.int64)
    with _on_device(handle.device):
        rc = load_library().hs_get_stats(handle.ptr, layer_id, out.ctypes.data, 1 if reset else 0,
                                         _stream_ptr(stream))
        _check(rc, "hs_get_stats")
    return out


def hs_set_timeline(handle: StateHandle, timeline=None) -> None:
    """timeline: a uint64-sized CUDA tensor of at least max_batch * 128
    elements on the handle's device (the per-CTA phase stamps of later
    swap-ins, [batch][8][16]), or None to stop recording."""
    import torch
    ptr = 0
    with _on_device(handle.device):
        if timeline is not None:
            if not timeline.is_cuda:
                raise ValueError("timeline must be in device memory")
            if timeline.numel() < handle.cfg.max_batch * TIMELINE_WORDS_PER_ROW:
                raise ValueError("timeline: need %d elements, got %d"
                                 % (handle.cfg.max_batch * TIMELINE_WORDS_PER_ROW,
                                    timeline.numel()))
            ptr = _dptr(timeline, torch.int64, "timeline")
        _check(load_library().hs_set_timeline(handle.ptr, ptr), "hs_set_timeline")


def hs_set_copy_ctas(handle: StateHandle, copy_ctas: int) -> None:
    _check(load_library().hs_set_copy_ctas(handle.ptr, copy_ctas), "hs_set_copy_ctas")


def hs_set_defer_copy(handle: StateHandle, defer: bool) -> None:
    _check(load_library().hs_set_defer_copy(handle.ptr, 1 if defer else 0), "hs_set_defer_copy")


def hs_copy_planned(handle: StateHandle, layer_id: int, miss_src, miss_dst, miss_count,
                    stream=None) -> None:
    import torch
    B = miss_count.numel()
    C = handle.cfg.max_steps * handle.cfg.top_k
    _shape(miss_count, (B,), "miss_count")
    _shape(miss_src, (B, C), "miss_src")
    _shape(miss_dst, (B, C), "miss_dst")
    with _on_device(handle.device):
        rc = load_library().hs_copy_planned(
            handle.ptr, layer_id, _dptr(miss_src, torch.int64, "miss_src"),
            _dptr(miss_dst, torch.int64, "miss_dst"), _dptr(miss_count, torch.int32, "miss_count"),
            miss_count.numel(), _stream_ptr(stream))
        _check(rc, "hs_copy_planned")


def hs_swap_in_noalloc(handle: StateHandle, req_pool_indices, seq_lens, topk, layer_id: int,
                       device_locs, stats=None, miss_src=None, miss_dst=None, miss_count=None,
                       stream=None) -> None:
    """hs_swap_in whose per-call scratch is the library's fixed device array
    (for callers that cannot allocate device memory); see the C header."""
    import torch
    B, S, K = _swap_in_shapes(handle, req_pool_indices, seq_lens, topk, device_locs, stats,
                              miss_src, miss_dst, miss_count)
    with _on_device(handle.device):
        rc = load_library().hs_swap_in_noalloc(
            handle.ptr, _dptr(req_pool_indices, torch.int32, "req_pool_indices"),
            _dptr(seq_lens, torch.int32, "seq_lens"), _dptr(topk, torch.int32, "topk"), B, S,
            layer_id, _dptr(device_locs, torch.int32, "device_locs"),
            _dptr(stats, torch.int32, "stats"), _dptr(miss_src, torch.int64, "miss_src"),
            _dptr(miss_dst, torch.int64, "miss_dst"),
            _dptr(miss_count, torch.int32, "miss_count"), _stream_ptr(stream))
        _check(rc, "hs_swap_in_noalloc")
