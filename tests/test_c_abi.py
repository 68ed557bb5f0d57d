"""The public header compiles as strict C99 and a C program links against the
in-tree library and calls its host-only entry points (no GPU needed)."""
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
