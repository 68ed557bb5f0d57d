"""ctypes wrapper around the C++ oracle (test infrastructure only).

The oracle library is compiled from ``hs_oracle.cpp`` with the host g++ into
``oracle/_build/<machine>/libhs_oracle.so``; nothing else is linked in.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hs_oracle.cpp")
_HDR = os.path.join(_HERE, "hs_oracle.h")

NUM_STATS = 9
STAT_NAMES = ("hits", "hit_slots", "dup_misses", "unique_misses", "admitted", "evicted",
              "overflow", "invalid", "extra")

_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def _lib_path(out_dir: Optional[str] = None) -> str:
    d = out_dir or os.path.join(_HERE, "_build", platform.machine())
    return os.path.join(d, "libhs_oracle.so")


def build_oracle(src: str = _SRC, out_path: Optional[str] = None, force: bool = False) -> str:
    """Compile the oracle into a shared library and return its path."""
    out = out_path or _lib_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(src), os.path.getmtime(_HDR))):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread", "-I", _HERE, src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib) -> None:
    lib.hso_create.restype = ctypes.c_void_p
    lib.hso_create.argtypes = [ctypes.c_int32] * 8
    lib.hso_destroy.restype = None
    lib.hso_destroy.argtypes = [ctypes.c_void_p]
    lib.hso_swap_in.restype = ctypes.c_int
    lib.hso_swap_in.argtypes = [ctypes.c_void_p, ctypes.c_int32, _u8p, _u8p, _i32p, _i32p, _i32p,
                                ctypes.c_int32, ctypes.c_int32, _i32p, _i32p, _i64p, _i64p, _i32p,
                                ctypes.c_int32]
    lib.hso_append_rows.restype = ctypes.c_int
    lib.hso_append_rows.argtypes = [ctypes.c_void_p, ctypes.c_int32, _u8p, _u8p, _i32p, _i32p,
                                    _i32p, _u8p, ctypes.c_int32]
    lib.hso_get_request_state.restype = ctypes.c_int
    lib.hso_get_request_state.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, _i32p,
                                          _i32p, _i32p, _i32p]
    lib.hso_reset_requests.restype = ctypes.c_int
    lib.hso_reset_requests.argtypes = [ctypes.c_void_p, _i32p, ctypes.c_int32]
    lib.hso_page_table.restype = ctypes.c_int
    lib.hso_page_table.argtypes = [_i32p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int32, ctypes.c_int32, _i32p, _i32p, _i32p]


def load_library(path: Optional[str] = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            lib = ctypes.CDLL(path)
            _declare(lib)
            return lib
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            _declare(lib)
            _lib = lib
        return _lib


def _ptr(a: Optional[np.ndarray], typ):
    if a is None:
        return ctypes.cast(None, typ)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(typ)


class Oracle:
    """The CPU oracle's state for all layers and requests of one cache."""

    def __init__(self, num_requests: int, max_seq_len: int, item_size_bytes: int,
                 hot_buffer_size: int, top_k: int, max_steps: int, num_layers: int = 1,
                 lib=None, extra_page_size: int = 0):
        self.lib = lib if lib is not None else load_library()
        self.R, self.L, self.W = num_requests, max_seq_len, item_size_bytes
        self.H, self.K, self.S_max, self.layers = hot_buffer_size, top_k, max_steps, num_layers
        self.C = max_steps * top_k
        self.E = extra_page_size
        h = self.lib.hso_create(num_requests, max_seq_len, item_size_bytes, hot_buffer_size,
                                top_k, max_steps, num_layers, extra_page_size)
        if not h:
            raise ValueError("invalid oracle configuration")
        self._h = ctypes.c_void_p(h)

    def close(self) -> None:
        if getattr(self, "_h", None):
            self.lib.hso_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def swap_in(self, layer: int, host_pool: np.ndarray, device_kv: np.ndarray,
                req_pool_indices: np.ndarray, seq_lens: np.ndarray, topk: np.ndarray,
                want_plan: bool = False, num_threads: int = 1):
        """One call.  Returns dict(locs, stats, [miss_src, miss_dst, miss_count])."""
        topk = np.ascontiguousarray(topk, dtype=np.int32)
        B, S, K = topk.shape
        assert K == self.K
        rpi = np.ascontiguousarray(req_pool_indices, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        assert host_pool.dtype == np.uint8 and device_kv.dtype == np.uint8
        locs = np.empty((B, S, K), dtype=np.int32)
        stats = np.zeros((B, NUM_STATS), dtype=np.int32)
        src = dst = cnt = None
        if want_plan:
            src = np.full((B, self.C), -1, dtype=np.int64)
            dst = np.full((B, self.C), -1, dtype=np.int64)
            cnt = np.zeros(B, dtype=np.int32)
        rc = self.lib.hso_swap_in(self._h, layer, _ptr(host_pool, _u8p), _ptr(device_kv, _u8p),
                                  _ptr(rpi, _i32p), _ptr(sl, _i32p), _ptr(topk, _i32p), B, S,
                                  _ptr(locs, _i32p), _ptr(stats, _i32p), _ptr(src, _i64p),
                                  _ptr(dst, _i64p), _ptr(cnt, _i32p), num_threads)
        if rc != 0:
            raise ValueError("oracle swap_in failed with code %d" % rc)
        out = {"locs": locs, "stats": stats}
        if want_plan:
            out.update(miss_src=src, miss_dst=dst, miss_count=cnt)
        return out

    def device_rows(self) -> int:
        """Rows of one layer's device buffer: hot + scratch, then the extra pages."""
        return self.R * (self.H + self.C + self.E)

    def append_rows(self, layer: int, host_pool: np.ndarray, device_kv: np.ndarray,
                    req: np.ndarray, tok: np.ndarray, seq_lens: np.ndarray,
                    rows: np.ndarray) -> int:
        """Write-back of newly decoded rows; returns the number of skipped entries."""
        req = np.ascontiguousarray(req, dtype=np.int32)
        tok = np.ascontiguousarray(tok, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        rows = np.ascontiguousarray(rows, dtype=np.uint8)
        n = req.size
        assert tok.size == n and sl.size == n and rows.shape == (n, self.W)
        rc = self.lib.hso_append_rows(self._h, layer, _ptr(host_pool, _u8p),
                                      _ptr(device_kv, _u8p), _ptr(req, _i32p), _ptr(tok, _i32p),
                                      _ptr(sl, _i32p), _ptr(rows, _u8p), n)
        if rc < 0:
            raise ValueError("oracle append_rows failed with code %d" % rc)
        return rc

    def request_state(self, layer: int, q: int):
        tok = np.empty(self.H, dtype=np.int32)
        ep = np.empty(self.H, dtype=np.int32)
        phys = np.empty(self.H + self.C, dtype=np.int32)
        e = np.zeros(1, dtype=np.int32)
        rc = self.lib.hso_get_request_state(self._h, layer, q, _ptr(tok, _i32p), _ptr(ep, _i32p),
                                            _ptr(phys, _i32p), _ptr(e, _i32p))
        if rc != 0:
            raise ValueError("bad layer/request")
        return {"tok": tok, "ep": ep, "phys": phys, "epoch": int(e[0])}

    def reset_requests(self, req_pool_indices) -> None:
        rpi = np.ascontiguousarray(req_pool_indices, dtype=np.int32)
        rc = self.lib.hso_reset_requests(self._h, _ptr(rpi, _i32p), rpi.size)
        if rc != 0:
            raise ValueError("bad request index")


def page_table(topk: np.ndarray, seq_lens: np.ndarray, page_size: int,
               max_seq_len: int = 2**31 - 1, lib=None):
    """Oracle sparse page table: (pages [B, S*K], num_pages [B], token_page [B, S, K])."""
    lib = lib if lib is not None else load_library()
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    B, S, K = topk.shape
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    pages = np.empty((B, S * K), dtype=np.int32)
    num = np.empty(B, dtype=np.int32)
    tp = np.empty((B, S, K), dtype=np.int32)
    rc = lib.hso_page_table(_ptr(topk, _i32p), _ptr(sl, _i32p), B, S, K, max_seq_len, page_size,
                            _ptr(pages, _i32p), _ptr(num, _i32p), _ptr(tp, _i32p))
    if rc != 0:
        raise ValueError("oracle page_table failed")
    return pages, num, tp
