"""hs_swap_in_noalloc against hs_swap_in, through the C ABI (needs a GPU).

hs_swap_in_noalloc serves callers that cannot allocate device memory (for
example a plugin that a serving runtime hands only its inputs and outputs):
its per-call scratch is a fixed device array inside the library instead of
the handle's workspace.  It must give exactly what hs_swap_in gives.  This
file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import hs_workloads as W
import sparse_attention_kv_swap_gb300 as pkg
from sparse_attention_kv_swap_gb300 import binding as B
from sparse_attention_kv_swap_gb300.cache import SwapInCache
from gpu_harness import bank_consistent

pytestmark = pytest.mark.gpu


def _outputs(Bn, S, K, C):
    dev = dict(device="cuda")
    return {"device_locs": torch.empty((Bn, S, K), dtype=torch.int32, **dev),
            "stats": torch.empty((Bn, B.HS_NUM_STATS), dtype=torch.int32, **dev),
            "miss_src": torch.full((Bn, C), -1, dtype=torch.int64, **dev),
            "miss_dst": torch.full((Bn, C), -1, dtype=torch.int64, **dev),
            "miss_count": torch.empty(Bn, dtype=torch.int32, **dev)}


def test_noalloc_matches_swap_in_on_two_calls():
    R, L, Wd, H, K, S = 5, 3000, W.ROW_BYTES, 200, 300, 3
    C = S * K
    cfg = pkg.make_config(R, L, Wd, H, K, S)
    pool = torch.empty((R, L, Wd), dtype=torch.uint8, pin_memory=True)
    W.fill_host_pool(pool.numpy(), 0)
    ref = SwapInCache(cfg, host_pools=[pool])
    new = SwapInCache(cfg, host_pools=[pool])
    for c in (ref, new):
        c.device_kv[0].zero_()
    rng = np.random.default_rng(77)
    rpi = torch.tensor([3, 0, 4, 1], dtype=torch.int32, device="cuda")
    sl = torch.tensor([3000, 2500, 3000, 1000], dtype=torch.int32, device="cuda")
    prev = None
    for call in range(2):
        topk_np = rng.integers(-2, L, size=(4, S, K)).astype(np.int32)
        if prev is not None:
            topk_np[:, 0, :K // 2] = prev[:, -1, K // 2:]  # reuse -> hits on the second call
        topk_np[:, 1:, :K // 3] = topk_np[:, :-1, -(K // 3):]  # cross-step duplicates
        prev = topk_np
        topk = torch.from_numpy(topk_np).cuda()
        a = _outputs(4, S, K, C)
        b = _outputs(4, S, K, C)
        B.hs_swap_in(ref.handle, rpi, sl, topk, 0, a["device_locs"], a["stats"], a["miss_src"],
                     a["miss_dst"], a["miss_count"])
        B.hs_swap_in_noalloc(new.handle, rpi, sl, topk, 0, b["device_locs"], b["stats"],
                             b["miss_src"], b["miss_dst"], b["miss_count"])
        torch.cuda.synchronize()
        for k in ("device_locs", "stats", "miss_count"):
            assert torch.equal(a[k], b[k]), "call %d: %s differs" % (call, k)
        cnt = a["miss_count"].cpu().numpy()
        for r in range(4):
            u = int(cnt[r])
            assert torch.equal(a["miss_src"][r, :u], b["miss_src"][r, :u])
            assert torch.equal(a["miss_dst"][r, :u], b["miss_dst"][r, :u])
        if call == 1:
            assert int(a["stats"][:, 0].sum()) > 0  # the second call has hits
        for q in range(R):
            sa = ref.export_request_state(0, q)
            sb = new.export_request_state(0, q)
            for k in ("tok", "ep", "phys"):
                assert (sa[k] == sb[k]).all(), "call %d q=%d: %s differs" % (call, q, k)
            # epoch and resident count; the hash layout (and its used-entry
            # count) depends on the order of concurrent inserts and is not
            # an observable, so each bank is only checked for consistency
            assert (sa["ctrl"][:2] == sb["ctrl"][:2]).all()
            for st in (sa, sb):
                assert bank_consistent(st) is None
        assert torch.equal(ref.device_kv[0], new.device_kv[0]), "call %d: rows differ" % call
    assert ref.status() == (0, 0) and new.status() == (0, 0)
    ref.close()
    new.close()


def test_noalloc_rejects_calls_beyond_its_scratch():
    # 128 rows x C = 8192 need 4 x 4 MiB + 8 KiB of scratch: more than the 16 MiB array
    cfg = pkg.make_config(128, 64, 16, 8, 2048, 4)
    pool = torch.empty((128, 64, 16), dtype=torch.uint8, pin_memory=True)
    cache = SwapInCache(cfg, host_pools=[pool])
    i32 = dict(dtype=torch.int32, device="cuda")
    topk = torch.zeros((128, 1, 2048), **i32)
    locs = torch.empty((128, 1, 2048), **i32)
    with pytest.raises(pkg.HsError) as e:
        B.hs_swap_in_noalloc(cache.handle, torch.arange(128, **i32), torch.full((128,), 64, **i32),
                             topk, 0, locs)
    assert e.value.code == B.HS_ERR_UNSUPPORTED
    cache.close()


def test_noalloc_scratch_limit_is_exact():
    """A call whose scratch is exactly HS_NOALLOC_SCRATCH_BYTES runs and
    matches hs_swap_in; one more entry of C is refused before any launch.
    batch 1024 and C = 1020: 4 * align256(4 * 1024 * 1020) + align256(64 * 1024)
    = 4 * 4177920 + 65536 = 16 MiB exactly; C = 1021 gives 16793600 bytes."""
    i32 = dict(dtype=torch.int32, device="cuda")
    Bn, L, Wd, H = 1024, 64, 16, 8
    for K, fits in ((1020, True), (1021, False)):
        need = 4 * ((4 * Bn * K + 255) // 256 * 256) + (64 * Bn + 255) // 256 * 256
        assert (need <= B.HS_NOALLOC_SCRATCH_BYTES) == fits
        if fits:
            assert need == B.HS_NOALLOC_SCRATCH_BYTES
        cfg = pkg.make_config(Bn, L, Wd, H, K, 1)
        pool = torch.empty((Bn, L, Wd), dtype=torch.uint8, pin_memory=True)
        W.fill_host_pool(pool.numpy(), 0)
        ref = SwapInCache(cfg, host_pools=[pool])
        new = SwapInCache(cfg, host_pools=[pool])
        for cache in (ref, new):
            cache.device_kv[0].zero_()
        rpi = torch.arange(Bn, **i32)
        sl = torch.full((Bn,), L, **i32)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(K)
        topk = torch.randint(-1, L, (Bn, 1, K), generator=gen, device="cuda", dtype=torch.int32)
        a = _outputs(Bn, 1, K, K)
        b = _outputs(Bn, 1, K, K)
        if not fits:
            with pytest.raises(pkg.HsError) as e:
                B.hs_swap_in_noalloc(new.handle, rpi, sl, topk, 0, b["device_locs"])
            assert e.value.code == B.HS_ERR_UNSUPPORTED
        else:
            B.hs_swap_in(ref.handle, rpi, sl, topk, 0, a["device_locs"], a["stats"],
                         a["miss_src"], a["miss_dst"], a["miss_count"])
            B.hs_swap_in_noalloc(new.handle, rpi, sl, topk, 0, b["device_locs"], b["stats"],
                                 b["miss_src"], b["miss_dst"], b["miss_count"])
            torch.cuda.synchronize()
            for k in ("device_locs", "stats", "miss_count"):
                assert torch.equal(a[k], b[k]), k
            assert torch.equal(ref.device_kv[0], new.device_kv[0])
            assert ref.status() == (0, 0) and new.status() == (0, 0)
        ref.close()
        new.close()


def test_noalloc_after_a_context_reset(tmp_path):
    """tests/c/noalloc_reset.c: no-alloc calls in a plain C program before and
    after cudaDeviceReset.  The scratch array's address is kept per device
    and context, so the calls after the reset look it up again in the new
    context and return exact rows."""
    import os
    import shutil
    import subprocess
    from sparse_attention_kv_swap_gb300 import build
    from test_c_abi import HERE, _cuda_include_dir, _cuda_lib_dirs
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include_dir()
    if cc is None or inc is None:
        pytest.skip("no C compiler or CUDA headers")
    lib = build.build()
    exe = str(tmp_path / "noalloc_reset")
    cuda_dirs = _cuda_lib_dirs()
    rpaths = [os.path.dirname(lib)] + cuda_dirs
    cmd = ([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
            "-I", os.path.dirname(B.HEADER), "-isystem", inc,
            os.path.join(HERE, "c", "noalloc_reset.c"), lib, "-o", exe]
           + ["-L" + d for d in cuda_dirs] + ["-lcudart"]
           + ["-Wl,-rpath," + d for d in rpaths])
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = ":".join(rpaths + [env.get("LD_LIBRARY_PATH", "")])
    res = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip() == "ok"
