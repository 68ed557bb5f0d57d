"""Register and stack report of every kernel, compiled for sm_103a here (no GPU
needed).  No kernel may spill registers or keep a stack frame, and the
kernels whose launch bounds promise full occupancy (the swap-in kernel at
1024 threads per SM, the planned-copy kernel at 2 x 512) must
fit 64 registers a thread, so that the bounds hold without spilling.  A change
that breaks either shows up here before it costs time on the GPU.  The same
sources, and the CPU oracle, also compile with warnings as errors."""
import concurrent.futures as cf
import os
import re
import subprocess
import tempfile

import pytest

from sparse_attention_kv_swap_gb300 import build

FULL_OCCUPANCY = ("swapin_kernel", "planned_copy_kernel")
EXPECTED = FULL_OCCUPANCY + ("append_kernel", "page_table_kernel", "reset_kernel")


def _ptxas_report(src: str, out_dir: str) -> str:
    cmd = ([build._nvcc()] + build.ARCH_FLAGS + build.NVCC_FLAGS
           + ["-I", build.INCLUDE, "-I", build.CSRC, "-Xptxas", "-v", "-c", src,
              "-o", os.path.join(out_dir, os.path.basename(src) + ".o")])
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return res.stderr


def _parse(report: str):
    """{mangled entry name: (stack bytes, spill stores, spill loads, registers)}."""
    out, name, frame = {}, None, None
    for line in report.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            name, frame = m.group(1), None
            continue
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads",
                      line)
        if m and name:
            frame = tuple(int(x) for x in m.groups())
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and name and frame is not None:
            out[name] = frame + (int(m.group(1)),)
            name = None
    return out


def test_no_spills_and_full_occupancy_registers():
    try:
        build._nvcc()
    except Exception:
        pytest.skip("no nvcc")
    with tempfile.TemporaryDirectory() as d:
        srcs = build._sources()
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
            reports = list(ex.map(lambda s: _ptxas_report(s, d), srcs))
    kernels = {}
    for r in reports:
        kernels.update(_parse(r))
    for want in EXPECTED:
        assert any(want in k for k in kernels), "kernel %s not found in the ptxas report" % want
    for name, (stack, st, ld, regs) in kernels.items():
        assert stack == 0 and st == 0 and ld == 0, \
            "%s: %d B stack, %d B spill stores, %d B spill loads" % (name, stack, st, ld)
        if any(k in name for k in FULL_OCCUPANCY):
            assert regs <= 64, "%s uses %d registers a thread (at most 64)" % (name, regs)


def test_report_parser_reads_spills_and_registers():
    report = "\n".join([
        "ptxas info    : Compiling entry function '_Z3fooPi' for 'sm_103a'",
        "ptxas info    : Function properties for _Z3fooPi",
        "    16 bytes stack frame, 8 bytes spill stores, 4 bytes spill loads",
        "ptxas info    : Used 72 registers, used 1 barriers",
        "ptxas info    : Compiling entry function '_Z3barv' for 'sm_103a'",
        "ptxas info    : Function properties for _Z3barv",
        "    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads",
        "ptxas info    : Used 12 registers, used 0 barriers",
    ])
    assert _parse(report) == {"_Z3fooPi": (16, 8, 4, 72), "_Z3barv": (0, 0, 0, 12)}


def test_sources_compile_without_warnings(tmp_path):
    """The CUDA sources (device and host code) and the CPU oracle compile with
    every common warning turned into an error."""
    import shutil
    try:
        nvcc = build._nvcc()
    except Exception:
        pytest.skip("no nvcc")
    srcs = build._sources()

    def one(src):
        cmd = ([nvcc] + build.ARCH_FLAGS + build.NVCC_FLAGS
               + ["-Werror", "all-warnings", "-Xcompiler", "-Wall,-Wextra,-Werror",
                  "-I", build.INCLUDE, "-I", build.CSRC, "-c", src,
                  "-o", str(tmp_path / (os.path.basename(src) + ".o"))])
        return src, subprocess.run(cmd, capture_output=True, text=True)

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        for src, res in ex.map(one, srcs):
            assert res.returncode == 0, "%s:\n%s" % (src, res.stderr)
    gxx = shutil.which("g++")
    if gxx:
        oracle_src = os.path.join(os.path.dirname(build.CSRC), "..", "oracle", "hs_oracle.cpp")
        res = subprocess.run([gxx, "-std=c++17", "-O2", "-Wall", "-Wextra", "-Wpedantic",
                              "-Werror", "-fPIC", "-shared", "-pthread",
                              os.path.normpath(oracle_src), "-o", str(tmp_path / "o.so")],
                             capture_output=True, text=True)
        assert res.returncode == 0, res.stderr
