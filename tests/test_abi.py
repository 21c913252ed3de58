"""The C-ABI library without a GPU: it builds, loads, exports every function
include/lce.h declares, its host-side argument checks answer synchronously,
and the ctypes mirror of lce_args_t has the C layout."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from chunked_vocab_cross_gb300 import _abi
from chunked_vocab_cross_gb300.build import INCLUDE, build

HEADER = os.path.join(INCLUDE, "lce.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _abi.lib()


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:lce_status_t|size_t|const char \*|int64_t|int)\s*\*?(lce_\w+)\(", src, re.M)))


def test_header_declares_expected_entry_points():
    names = _declared()
    for n in ("lce_forward", "lce_forward_backward", "lce_backward", "lce_run", "lce_workspace_size", "lce_compact",
              "lce_get_device_status", "lce_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(lce_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    assert set(names) == set(_abi.SIGNATURES), set(names) ^ set(_abi.SIGNATURES)
    for n in names:
        assert getattr(lib, n) is not None


def test_host_checks_without_gpu(lib):
    a = _abi.LceArgs()
    assert lib.lce_run(None) == 1                      # NULL args
    assert lib.lce_run(ctypes.byref(a)) == 1           # NULL tensors
    a.H = a.W = a.targets = a.loss = 4096
    a.N, a.d, a.V = 0, 64, 10
    assert lib.lce_run(ctypes.byref(a)) == 2           # N < 1
    a.N, a.d = 10, 12
    assert lib.lce_run(ctypes.byref(a)) == 3           # d*2 not a multiple of 16
    a.d, a.H = 64, 4100
    assert lib.lce_run(ctypes.byref(a)) == 3           # misaligned H
    a.H, a.dtype = 4096, 7
    assert lib.lce_run(ctypes.byref(a)) == 4           # dtype
    a.dtype, a.vocab_chunk = 0, 100
    assert lib.lce_run(ctypes.byref(a)) == 2           # chunk not a multiple of 256
    a.vocab_chunk, a.dH = 0, 4096
    assert lib.lce_run(ctypes.byref(a)) == 1           # dH without dW
    assert lib.lce_status_string(0) == b"ok"
    assert lib.lce_version() >= 100


def test_workspace_size_is_linear_in_N_not_N_times_V(lib):
    ws = lib.lce_workspace_size(16384, 4096, 128256, 0, 0)
    logits = 16384 * 128256 * 4
    assert 0 < ws < logits / 8
    assert lib.lce_workspace_size(16384, 4096, 262144, 0, 0) == ws         # independent of V (fixed chunk)
    assert lib.lce_workspace_size(0, 4096, 100, 0, 0) == 0
    assert lib.lce_workspace_size(100, 4096, 100, 0, 300) == 0


def test_args_struct_layout_matches_c():
    src = f"""
#include <stdio.h>
#include <stddef.h>
#include "lce.h"
int main(void) {{
  printf("%zu", sizeof(lce_args_t));
#define F(x) printf(" %zu", offsetof(lce_args_t, x));
  F(dtype) F(H) F(W) F(targets) F(ignore_index) F(N) F(d) F(V) F(loss) F(dH) F(dW)
  F(accumulate_dW) F(grad_scale) F(lse) F(workspace) F(workspace_bytes) F(vocab_chunk) F(stream)
  F(lse_in) F(grad_loss) F(token_chunk)
  printf("\\n"); return 0; }}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", INCLUDE, "-o", exe, c], check=True)
        vals = [int(v) for v in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    names = [f[0] for f in _abi.LceArgs._fields_]
    assert vals[0] == ctypes.sizeof(_abi.LceArgs)
    assert vals[1:] == [getattr(_abi.LceArgs, n).offset for n in names]
