"""The C ABI library on the CPU: it builds, loads, exports every symbol that
include/hisparse_swap.h declares, and validates arguments before touching CUDA."""
import ctypes

import pytest

import sparse_attention_kv_swap_gb300 as pkg
from sparse_attention_kv_swap_gb300 import binding as B


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_kv_swap_gb300 import build
    build.build()
    return B.load_library()


def test_exports_every_declared_symbol(lib):
    names = B.header_symbols()
    assert len(names) >= 14
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_header_constants_match_binding():
    import re
    text = open(B.HEADER).read()
    consts = dict(re.findall(r"#define (HS_[A-Z_0-9]+) \(?(-?(?:0x)?[0-9a-fA-F]+)u?\)?", text))
    for name in ("HS_OK", "HS_ERR_INVALID_ARG", "HS_ERR_UNSUPPORTED", "HS_ERR_CUDA",
                 "HS_ERR_DEVICE_STATUS", "HS_ERR_TIMEOUT", "HS_STATUS_BAD_REQUEST",
                 "HS_STATUS_DUPLICATE_REQUEST", "HS_STATUS_SEQ_LEN_CLAMPED",
                 "HS_STATUS_PROBE_LIMIT", "HS_STATUS_TABLE_FULL", "HS_STATUS_BAD_APPEND",
                 "HS_NUM_STATS", "HS_MAX_EXTRA_PAGE", "HS_STAT_EXTRA", "HS_STATUS_BAD_PLAN",
                 "HS_MAX_ITEM_BYTES"):
        assert int(consts[name], 0) == getattr(B, name), name
    m = re.search(r"#define HS_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == B.HS_NOALLOC_SCRATCH_BYTES


def test_version_and_strings(lib):
    assert pkg.hs_version() == 20000
    assert pkg.hs_status_string(0) == "ok"
    assert "invalid" in pkg.hs_status_string(-1)
    assert pkg.hs_status_string(-99) == "unknown status"


def _cfg(**kw):
    base = dict(num_requests=64, max_seq_len=32768, item_size_bytes=656, hot_buffer_size=8192,
                top_k=2048, max_steps=4, num_layers=1, max_batch=64)
    base.update(kw)
    return B.HsConfig(**base)


def test_config_check(lib):
    assert pkg.hs_config_check(_cfg()) == B.HS_OK
    assert pkg.hs_config_check(_cfg(item_size_bytes=650)) == B.HS_ERR_INVALID_ARG
    assert pkg.hs_config_check(_cfg(hot_buffer_size=32769)) == B.HS_ERR_UNSUPPORTED
    assert pkg.hs_config_check(_cfg(hot_buffer_size=32768)) == B.HS_OK
    assert pkg.hs_config_check(_cfg(max_steps=5)) == B.HS_ERR_UNSUPPORTED
    assert pkg.hs_config_check(_cfg(top_k=4096)) == B.HS_ERR_UNSUPPORTED
    assert pkg.hs_config_check(_cfg(max_steps=2, top_k=4096)) == B.HS_OK
    assert pkg.hs_config_check(_cfg(max_batch=65)) == B.HS_ERR_INVALID_ARG
    assert pkg.hs_config_check(_cfg(num_layers=0)) == B.HS_ERR_INVALID_ARG
    assert lib.hs_config_check(None) == B.HS_ERR_INVALID_ARG


def test_sizes(lib):
    c = _cfg()
    H, C, R = 8192, 8192, 64
    assert pkg.hs_hash_size(c) == 16384
    assert pkg.hs_device_kv_bytes(c) == R * (H + C) * 656
    assert pkg.hs_host_pool_bytes(c) == R * 32768 * 656
    st = pkg.hs_state_bytes(c)
    assert st >= R * (16384 * 8 + H * 4 * 2 + (H + C) * 4 + 32)
    assert st % 256 == 0
    assert pkg.hs_workspace_bytes(c) >= 4 * 64 * C * 4
    assert pkg.hs_state_bytes(_cfg(max_steps=9)) == 0
    assert pkg.hs_hash_size(_cfg(hot_buffer_size=1)) == 32


def test_create_rejects_bad_arguments_without_cuda(lib):
    c = _cfg(num_requests=2, max_seq_len=16, hot_buffer_size=4, top_k=2, max_steps=1,
             max_batch=2)
    out = ctypes.c_void_p()
    arr = (ctypes.c_void_p * 1)(0x1000)
    rc = lib.hs_create_state(ctypes.byref(c), arr, arr, None, 0, None, 0, None, ctypes.byref(out))
    assert rc == B.HS_ERR_INVALID_ARG and not out.value
    big = 1 << 20
    rc = lib.hs_create_state(ctypes.byref(c), arr, arr, ctypes.c_void_p(0x100000), 8,
                             ctypes.c_void_p(0x200000), big, None, ctypes.byref(out))
    assert rc == B.HS_ERR_INVALID_ARG  # state smaller than hs_state_bytes
    rc = lib.hs_create_state(ctypes.byref(c), arr, arr, ctypes.c_void_p(0x100010), big,
                             ctypes.c_void_p(0x200000), big, None, ctypes.byref(out))
    assert rc == B.HS_ERR_INVALID_ARG  # state not 256-byte aligned
    bad = (ctypes.c_void_p * 1)(0x1001)
    rc = lib.hs_create_state(ctypes.byref(c), bad, arr, ctypes.c_void_p(0x100000), big,
                             ctypes.c_void_p(0x200000), big, None, ctypes.byref(out))
    assert rc == B.HS_ERR_INVALID_ARG  # host pool not 16-byte aligned
    assert lib.hs_create_state(ctypes.byref(c), arr, arr, None, 0, None, 0, None, None) == \
        B.HS_ERR_INVALID_ARG


def test_calls_reject_null_handle(lib):
    assert lib.hs_swap_in(None, None, None, None, 1, 1, 0, None, None, None, None, None,
                          None) == B.HS_ERR_INVALID_ARG
    assert lib.hs_reset_requests(None, None, 1, None) == B.HS_ERR_INVALID_ARG
    flags = ctypes.c_uint32()
    assert lib.hs_get_status(None, ctypes.byref(flags), None) == B.HS_ERR_INVALID_ARG
    assert lib.hs_export_request_state(None, 0, 0, None, None, None, None, None, None) == \
        B.HS_ERR_INVALID_ARG
    lib.hs_destroy_state(None)


def test_page_table_rejects_bad_arguments(lib):
    assert lib.hs_page_table(None, None, 1, 0, 4, 100, 16, None, None, None, None) == \
        B.HS_ERR_INVALID_ARG
    assert lib.hs_page_table(None, None, 1, 1, 4, 100, 0, None, None, None, None) == \
        B.HS_ERR_INVALID_ARG
    assert lib.hs_page_table(None, None, 1, 4, 4096, 100, 16, None, None, None, None) == \
        B.HS_ERR_UNSUPPORTED
    assert lib.hs_page_table(None, None, 1, 1, 4, 1 << 30, 1, None, None, None, None) == \
        B.HS_ERR_UNSUPPORTED
    assert lib.hs_page_table(None, None, 0, 1, 4, 100, 16, None, None, None, None) == B.HS_OK
    assert lib.hs_page_table(None, None, 2, 1, 4, 100, 16, None, None, None, None) == \
        B.HS_ERR_INVALID_ARG
    # int32 arrays must be 4-byte aligned: a misaligned address is refused on the
    # host (the addresses below are never dereferenced)
    ok, odd = 0x20000, 0x20002
    for bad in range(5):
        ptrs = [odd if i == bad else ok + 0x1000 * i for i in range(5)]
        assert lib.hs_page_table(ptrs[0], ptrs[1], 2, 1, 4, 100, 16, ptrs[2], ptrs[3],
                                 ptrs[4], None) == B.HS_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        B.load_library(str(tmp_path / "nope.so"))


def test_dense_index_config(lib):
    hashed, dense = _cfg(), _cfg(index_kind=B.HS_INDEX_DENSE)
    assert pkg.hs_config_check(dense) == B.HS_OK
    assert pkg.hs_config_check(_cfg(index_kind=2)) == B.HS_ERR_INVALID_ARG
    assert pkg.hs_hash_size(dense) == 0
    # the dense map replaces the 64 x 16384 x 8-byte hash banks by 64 x 32768 x 2 bytes
    diff = pkg.hs_state_bytes(hashed) - pkg.hs_state_bytes(dense)
    assert abs(diff - (64 * 16384 * 8 - 64 * 32768 * 2)) <= 512
    assert pkg.hs_workspace_bytes(dense) == pkg.hs_workspace_bytes(hashed)


def test_extra_page_config(lib):
    """The extra page adds R * E device rows and is bounded."""
    base = _cfg()
    x = _cfg(extra_page_size=256)
    assert pkg.hs_config_check(x) == B.HS_OK
    assert (pkg.hs_device_kv_bytes(x) - pkg.hs_device_kv_bytes(base)
            == base.num_requests * 256 * base.item_size_bytes)
    assert pkg.hs_state_bytes(x) == pkg.hs_state_bytes(base)  # no policy state of its own
    assert pkg.hs_config_check(_cfg(extra_page_size=-1)) == B.HS_ERR_INVALID_ARG
    assert pkg.hs_config_check(_cfg(extra_page_size=B.HS_MAX_EXTRA_PAGE)) == B.HS_OK
    assert pkg.hs_config_check(_cfg(extra_page_size=B.HS_MAX_EXTRA_PAGE + 1)) == \
        B.HS_ERR_UNSUPPORTED
    # rows up to 64 KiB (the copy counts 16-byte pieces of a call in 32 bits)
    assert pkg.hs_config_check(_cfg(item_size_bytes=B.HS_MAX_ITEM_BYTES)) == B.HS_OK
    assert pkg.hs_config_check(_cfg(item_size_bytes=B.HS_MAX_ITEM_BYTES + 16)) == \
        B.HS_ERR_UNSUPPORTED
    # device rows must stay addressable by int32 locations
    # (52428 requests of 32768 + 8192 rows are 32767 rows short of 2^31 - 1)
    assert pkg.hs_config_check(_cfg(num_requests=52428, hot_buffer_size=32768,
                                    extra_page_size=0)) == B.HS_OK
    assert pkg.hs_config_check(_cfg(num_requests=52428, hot_buffer_size=32768,
                                    extra_page_size=1)) == B.HS_ERR_UNSUPPORTED


def test_get_stats_argument_errors(lib):
    import numpy as np
    out = np.zeros(B.HS_NUM_STATS, np.int64)
    assert lib.hs_get_stats(None, 0, out.ctypes.data, 0, None) == B.HS_ERR_INVALID_ARG


def test_append_rows_argument_errors(lib):
    """hs_append_rows rejects bad handles, layers, counts and unaligned rows on the host."""
    assert lib.hs_append_rows(None, 0, None, None, None, None, 1, None) == B.HS_ERR_INVALID_ARG


def test_binding_checks_shapes_and_memory_before_any_launch():
    """The kernels trust the sizes they are given: the binding rejects wrong
    shapes, top-k widths and unpinned host tensors before calling the library."""
    import torch

    class Handle:  # never reaches the library: every call below fails first
        ptr = None
        device = 0
        cfg = _cfg(num_requests=8, max_seq_len=100, hot_buffer_size=16, top_k=4, max_steps=2,
                   max_batch=8)

    # plain host tensors: the shape checks come before the memory check, which
    # then rejects them (they are neither device nor pinned memory)
    i32 = dict(dtype=torch.int32)
    h = Handle()
    topk = torch.zeros((2, 1, 4), **i32)
    rpi = torch.zeros(2, **i32)
    locs = torch.zeros((2, 1, 4), **i32)
    with pytest.raises(ValueError, match="top_k"):
        B.hs_swap_in(h, rpi, rpi, torch.zeros((2, 1, 5), **i32), 0, locs)
    with pytest.raises(ValueError, match="seq_lens"):
        B.hs_swap_in(h, rpi, torch.zeros(3, **i32), topk, 0, locs)
    with pytest.raises(ValueError, match="device_locs"):
        B.hs_swap_in(h, rpi, rpi, topk, 0, torch.zeros((2, 2, 4), **i32))
    with pytest.raises(ValueError, match="stats"):
        B.hs_swap_in(h, rpi, rpi, topk, 0, locs, torch.zeros((2, 8), **i32))
    with pytest.raises(ValueError, match="miss_src"):
        B.hs_swap_in(h, rpi, rpi, topk, 0, locs, None, torch.zeros((2, 4), dtype=torch.int64),
                     torch.zeros((2, 8), dtype=torch.int64), rpi)
    with pytest.raises(ValueError, match="pinned"):
        B.hs_swap_in(h, rpi, rpi, topk, 0, locs)
    with pytest.raises(ValueError, match="rows"):
        B.hs_append_rows(h, 0, rpi, rpi, rpi, torch.zeros((2, 64), dtype=torch.uint8))
    with pytest.raises(ValueError, match="token_page"):
        B.hs_page_table(topk, rpi, 100, 16, torch.zeros((2, 4), **i32), rpi,
                        torch.zeros((2, 4), **i32))


def test_binding_rejects_tensors_and_streams_of_another_device():
    """A handle's calls run on its own device: inside a call for cuda:0 the
    binding refuses a device tensor or a stream that lives on cuda:1 (checked
    with stand-in objects, so no GPU is needed)."""
    import torch

    class OnCuda1:
        is_cuda = True
        dtype = torch.int32
        device = torch.device("cuda", 1)

        def is_contiguous(self):
            return True

        def is_pinned(self):
            return False

        def data_ptr(self):
            return 0x10000

    class Stream1:
        device = torch.device("cuda", 1)
        cuda_stream = 0

    with B._on_device(1):  # no switch without a GPU; checks only
        assert B._dptr(OnCuda1(), torch.int32, "x") == 0x10000
        assert B._stream_ptr(Stream1()) == 0
    with B._on_device(0):
        with pytest.raises(ValueError, match="cuda:1"):
            B._dptr(OnCuda1(), torch.int32, "topk")
        with pytest.raises(ValueError, match="stream"):
            B._stream_ptr(Stream1())
    assert B._dptr(OnCuda1(), torch.int32, "x") == 0x10000  # outside a call: no device rule


def test_product_path_never_reaches_the_oracle(lib):
    """The package (Python and CUDA sources) neither imports, links, loads nor
    names the CPU oracle, and the CUDA library exports none of its symbols:
    every step of a swap-in runs in the library's kernels."""
    import glob
    import os
    import re
    pkg_dir = os.path.dirname(B.__file__)
    files = (glob.glob(os.path.join(pkg_dir, "*.py"))
             + glob.glob(os.path.join(pkg_dir, "csrc", "*.cu"))
             + glob.glob(os.path.join(pkg_dir, "csrc", "*.cuh"))
             + glob.glob(os.path.join(os.path.dirname(B.HEADER), "*.h")))
    assert files
    for path in files:
        text = open(path).read()
        assert not re.search(r"\boracle\b|hso_|hs_oracle", text, re.IGNORECASE), path
    for sym in ("hso_create", "hso_swap_in", "hso_reset_requests"):
        assert not hasattr(lib, sym), sym
