"""The kernels compile for sm_103a without register spills.

A spill in a GEMM's promotion or epilogue loop puts local-memory round trips on the path every K
block takes (the FP32-scale tile GEMM lost 5-11% that way), so the build's resource report is
checked here, on the CPU: ptxas prints one 'N bytes spill stores, M bytes spill loads' line per
kernel, and every one must read zero.
"""

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import tempfile

import pytest

from block_fp8_mixture_gb300 import build

NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
pytestmark = pytest.mark.skipif(not os.path.exists(NVCC), reason="nvcc not found")

# the translation units with kernels on the layer's path
KERNEL_SOURCES = ["moe_gemm.cu", "moe_gemm_bs.cu", "moe_gemm_small.cu", "moe_quant.cu",
                  "moe_align.cu"]

_ENTRY = re.compile(r"Compiling entry function '([^']+)'")
_SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")


def _resources(src: str, out_dir: str):
    cmd = [NVCC, *build.NVCC_FLAGS, "-Xptxas", "-v", "-c", os.path.join(build.CSRC, src), "-o",
           os.path.join(out_dir, src + ".o")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    kernels, current = {}, None
    for line in (res.stdout + res.stderr).splitlines():
        m = _ENTRY.search(line)
        if m:
            current = m.group(1)
            continue
        m = _SPILL.search(line)
        if m and current is not None:
            kernels[current] = (int(m.group(1)), int(m.group(2)))
            current = None
    return src, kernels


def test_no_register_spills():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(len(KERNEL_SOURCES)) as pool:
            reports = dict(pool.map(lambda s: _resources(s, tmp), KERNEL_SOURCES))
    assert all(reports.values()), reports   # every file reported its kernels
    spilled = {f"{src}:{k}": v for src, ks in reports.items() for k, v in ks.items() if any(v)}
    assert not spilled, spilled
