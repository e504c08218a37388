"""Every kernel compiles for sm_103a without register spills.

The kernels size their work per thread (registers for the GEMV activations,
the dequantised rows, the accumulator drains) so that nothing goes to local
memory; ptxas's resource report (`-Xptxas -v`) shows it.  A change that makes
any kernel spill fails here, on the CPU, before it costs GPU time.
"""
import concurrent.futures as cf
import os
import re
import shutil
import subprocess

import pytest

from mxfp4_mixture_experts_rms_gb300 import build


def _report(src):
    cmd = [build.nvcc(), *build.ARCH, *build.NVCC_FLAGS, "-Xptxas", "-v", "-c", src, "-o", os.devnull]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return src, r.stdout + r.stderr


def test_no_kernel_spills_registers():
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not available")
    srcs = build._sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        reports = list(ex.map(_report, srcs))
    n = 0
    for src, text in reports:
        for m in re.finditer(r"(\d+) bytes spill stores, (\d+) bytes spill loads", text):
            n += 1
            assert m.group(1) == "0" and m.group(2) == "0", (os.path.basename(src), m.group(0))
    assert n >= 40   # every kernel instance reported
