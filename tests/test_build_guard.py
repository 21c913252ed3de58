"""Compile-time guard for the GEMM kernels (CPU; nvcc cross-compiles for
sm_103a): the logits/LSE and the plain backward instantiations must not spill
registers, and every GEMM instantiation must stay within one 192-thread CTA
per SM (at most 255 registers a thread). A spill in the mainloop kernels
costs local-memory traffic in the hot path without changing any result, so
only a check on the compiler's report catches it."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ptxas_report(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path / "lce.o")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xptxas", "-v", "-c",
           os.path.join(ROOT, "chunked_vocab_cross_gb300", "csrc", "lce_api.cu"), "-I", os.path.join(ROOT, "include"),
           "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout + r.stderr


def _kernel_stats(report):
    """{mangled kernel name: (registers, spill store bytes, spill load bytes)}"""
    stats, name = {}, None
    for line in report.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            name = m.group(1)
            continue
        if name is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            stats.setdefault(name, [0, 0, 0])[1:] = [int(m.group(1)), int(m.group(2))]
        m = re.search(r"Used (\d+) registers", line)
        if m:
            stats.setdefault(name, [0, 0, 0])[0] = int(m.group(1))
    return {k: tuple(v) for k, v in stats.items()}


def test_gemm_kernels_do_not_spill(tmp_path):
    stats = _kernel_stats(_ptxas_report(tmp_path))
    gemm = {k: v for k, v in stats.items() if "k_gemm" in k}
    assert len(gemm) == 3, sorted(stats)            # LSE, backward, backward with a fused optimizer
    for name, (regs, st, ld) in gemm.items():
        assert regs <= 255, (name, regs)
        if "ILi0E" in name or "ILi1E" in name:      # the default path's instantiations
            assert st == 0 and ld == 0, (name, st, ld)
