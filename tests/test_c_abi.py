"""The public header compiles as strict C99 and C programs link against the
in-tree library: one calls its host-only entry points (no GPU needed), the
other runs swap-ins on the GPU with buffers from the CUDA runtime alone."""
import os
import shutil
import subprocess

import pytest

from sparse_attention_kv_swap_gb300 import binding as B
from sparse_attention_kv_swap_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))


def _cuda_lib_dirs():
    dirs = []
    for root in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if root:
            for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
                p = os.path.join(root, sub)
                if os.path.isdir(p):
                    dirs.append(p)
    return dirs


def test_header_compiles_as_c99_and_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = build.build()
    exe = str(tmp_path / "abi_smoke")
    rpaths = [os.path.dirname(lib)] + _cuda_lib_dirs()
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.dirname(B.HEADER), os.path.join(HERE, "c", "abi_smoke.c"), lib,
           "-o", exe] + ["-Wl,-rpath," + d for d in rpaths]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = ":".join(rpaths + [env.get("LD_LIBRARY_PATH", "")])
    res = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == "ok"


def _cuda_include_dir():
    for root in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if root and os.path.isfile(os.path.join(root, "include", "cuda_runtime_api.h")):
            return os.path.join(root, "include")
    return None


@pytest.mark.gpu
def test_c_program_runs_swap_ins_on_the_gpu(tmp_path):
    """tests/c/abi_gpu.c: a plain C99 program (no Python, no PyTorch) creates a
    state, runs a first call (all misses) and a repeat (all hits) and checks
    the counters and every returned row against the host pool it filled."""
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include_dir()
    if cc is None or inc is None:
        pytest.skip("no C compiler or CUDA headers")
    lib = build.build()
    exe = str(tmp_path / "abi_gpu")
    cuda_dirs = _cuda_lib_dirs()
    rpaths = [os.path.dirname(lib)] + cuda_dirs
    cmd = ([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
            "-I", os.path.dirname(B.HEADER), "-isystem", inc,
            os.path.join(HERE, "c", "abi_gpu.c"), lib, "-o", exe]
           + ["-L" + d for d in cuda_dirs] + ["-lcudart"]
           + ["-Wl,-rpath," + d for d in rpaths])
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = ":".join(rpaths + [env.get("LD_LIBRARY_PATH", "")])
    res = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip() == "ok"
