"""The C ABI used from C: a small client (tests/c/lce_client.c, built with gcc
against include/lce.h, liblce.so and the CUDA runtime) runs
lce_forward_backward on seeded inputs; its outputs match the fp64 oracle
within the path's tolerances."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from lce_testutil import TOL_LOSS, TOL_REL, rel_fro
from synth_inputs import IGNORE_INDEX, bf16_bits_to_f32, make_inputs

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "chunked_vocab_cross_gb300")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_c_client_forward_backward(tmp_path):
    from chunked_vocab_cross_gb300.build import build
    build()
    cuda = _cuda_home()
    exe = str(tmp_path / "lce_client")
    libdirs = [os.path.join(cuda, d) for d in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib")
               if os.path.isdir(os.path.join(cuda, d))]
    cmd = ["gcc", "-O2", "-o", exe, os.path.join(ROOT, "tests", "c", "lce_client.c"), "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", PKG, "-llce"] + [f"-L{d}" for d in libdirs] + \
          ["-lcudart", f"-Wl,-rpath,{PKG}"] + [f"-Wl,-rpath,{d}" for d in libdirs]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    x = make_inputs("gpt1b", N=1200, d=256, V=3000, padding=("random_frac", 0.25), seqs=1)
    x.H.tofile(tmp_path / "H.bin")
    x.W.tofile(tmp_path / "W.bin")
    x.targets.astype(np.int64).tofile(tmp_path / "t.bin")
    r = subprocess.run([exe, str(tmp_path), "1200", "256", "3000", str(IGNORE_INDEX)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    loss = float(np.fromfile(tmp_path / "loss.bin", dtype=np.float32)[0])
    dH = bf16_bits_to_f32(np.fromfile(tmp_path / "dH.bin", dtype=np.uint16)).reshape(1200, 256)
    dW = np.fromfile(tmp_path / "dW.bin", dtype=np.float32).reshape(3000, 256)
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss - ref["loss"]) <= TOL_LOSS
    assert rel_fro(dH, ref["dH"]) <= TOL_REL and rel_fro(dW, ref["dW"]) <= TOL_REL
    assert np.all(dH[x.targets == IGNORE_INDEX] == 0)
