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
    a.dH, a.dW, a.dW_bf16 = 4096, 4096, 1
    a.dtype = 1
    assert lib.lce_run(ctypes.byref(a)) == 10          # bf16 dW of fp32 inputs
    a.dtype, a.accumulate_dW = 0, 1
    assert lib.lce_run(ctypes.byref(a)) == 10          # bf16 dW accumulated into
    a.accumulate_dW, a.token_chunk = 0, 4
    assert lib.lce_run(ctypes.byref(a)) == 10          # bf16 dW over token chunks
    assert lib.lce_status_string(0) == b"ok"
    assert lib.lce_version() == 600          # 0.6.0: bf16 embedding gradient


def test_workspace_size_is_linear_in_N_not_N_times_V(lib):
    ws = lib.lce_workspace_size(16384, 4096, 128256, 0, 0)
    logits = 16384 * 128256 * 4
    assert 0 < ws < logits / 8
    assert lib.lce_workspace_size(16384, 4096, 262144, 0, 0) == ws         # independent of V (fixed chunk)
    assert lib.lce_workspace_size(0, 4096, 100, 0, 0) == 0
    assert lib.lce_workspace_size(100, 4096, 100, 0, 300) == 0


def test_default_vocab_chunk_is_evened_out_over_V(lib):
    """The default backward chunk is 6144 rows spread evenly over the chunks V
    needs (256-row tiles), visible in the G buffers of the workspace."""
    for V, vc in ((32000, 5376), (50304, 5632), (128256, 6144), (262144, 6144), (1000, 1024), (6145, 3328)):
        assert lib.lce_workspace_size(4096, 512, V, 0, 0) == lib.lce_workspace_size(4096, 512, V, 0, vc), V


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
  F(lse_in) F(grad_loss) F(token_chunk) F(optim) F(row_gather) F(dW_bf16)
  printf(" %zu", sizeof(lce_optim_t));
#define G(x) printf(" %zu", offsetof(lce_optim_t, x));
  G(kind) G(lr) G(weight_decay) G(momentum) G(beta1) G(beta2) G(eps) G(step) G(master_W) G(exp_avg)
  G(exp_avg_sq) G(state_bf16)
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
    n = len(names)
    assert vals[1:1 + n] == [getattr(_abi.LceArgs, k).offset for k in names]
    onames = [f[0] for f in _abi.LceOptim._fields_]
    assert vals[1 + n] == ctypes.sizeof(_abi.LceOptim)
    assert vals[2 + n:] == [getattr(_abi.LceOptim, k).offset for k in onames]


def test_fused_optimizer_option_checks_without_gpu(lib):
    """Option combinations the fused optimizer step refuses on the host."""
    def args(**kw):
        a = _abi.LceArgs()
        a.H = a.W = a.targets = a.loss = a.dH = 4096
        a.N, a.d, a.V = 10, 64, 100
        o = _abi.LceOptim()
        o.kind, o.lr, o.step = _abi.LCE_OPT_ADAMW, 1e-3, 1
        o.beta1, o.beta2, o.eps = 0.9, 0.999, 1e-8
        o.exp_avg = o.exp_avg_sq = 8192
        for k, v in kw.items():
            setattr(o if hasattr(o, k) and k not in ("dW",) and not hasattr(a, k) else a, k, v)
        a.optim = ctypes.addressof(o)
        return a, o

    def run(**kw):
        a, o = args(**kw)
        return lib.lce_run(ctypes.byref(a))

    ok_codes = (5, 9)   # the host checks pass; there is no sm_103 device here
    assert run() in ok_codes
    assert run(dW=4096) == 10                       # a gradient output is never written
    assert run(accumulate_dW=1) == 10
    assert run(token_chunk=5) == 10                 # one token chunk only
    assert run(token_chunk=10) in ok_codes          # a cap >= N is one chunk
    assert run(exp_avg_sq=None) == 1                # AdamW needs both moments
    assert run(step=0) == 10
    assert run(beta1=1.0) == 10
    assert run(eps=0.0) == 10
    assert run(lr=-1.0) == 10
    assert run(kind=7) == 10
    assert run(kind=_abi.LCE_OPT_SGD, exp_avg=None, exp_avg_sq=None) in ok_codes
    assert run(kind=_abi.LCE_OPT_SGD, momentum=0.9, exp_avg=None) == 1
    assert run(master_W=8200) == 3                  # misaligned state
    assert run(dtype=1, master_W=12288) == 10       # master weights are for bf16 W
    assert run(dH=None) == 1                        # the update runs in the backward
    a, _ = args()
    a.optim = None
    assert lib.lce_run(ctypes.byref(a)) == 1        # without an optimizer dH needs dW



def test_row_gather_option_checks_without_gpu(lib):
    a = _abi.LceArgs()
    a.H = a.W = a.targets = a.loss = 4096
    a.N, a.d, a.V = 10, 512, 100
    a.row_gather = 1
    assert lib.lce_run(ctypes.byref(a)) in (5, 9)     # accepted (no sm_103 device here)
    a.d = 320
    assert lib.lce_run(ctypes.byref(a)) == 10         # d not a multiple of 256
    a.d, a.dtype = 512, 1
    assert lib.lce_run(ctypes.byref(a)) == 10         # fp32 inputs are split, not gathered
    # the gathered operand needs no compacted copy: N_pad * d * 2 bytes less workspace
    b = _abi.LceArgs()
    b.N, b.d, b.V, b.dH = 1000, 512, 5000, 4096
    full = lib.lce_workspace_size_args(ctypes.byref(b))
    b.row_gather = 1
    assert full - lib.lce_workspace_size_args(ctypes.byref(b)) == 1024 * 512 * 2


def test_embedding_entry_points_host_checks_without_gpu(lib):
    f, b = lib.lce_embedding_forward, lib.lce_embedding_backward
    assert f(0, None, 4096, 0, 10, 64, 100, 4096, None) == 1             # NULL W
    assert f(0, 4096, 4096, 0, 0, 64, 100, 4096, None) == 2              # N < 1
    assert f(0, 4096, 4096, 0, 10, 12, 100, 4096, None) == 3             # d % 8
    assert f(0, 4100, 4096, 0, 10, 64, 100, 4096, None) == 3             # misaligned W
    assert f(7, 4096, 4096, 0, 10, 64, 100, 4096, None) == 4             # dtype
    assert b(0, 4096, 4096, 0, 10, 64, 0, 4096, 0, None, 0, None) == 2   # V < 1
    assert b(0, 4096, None, 0, 10, 64, 100, 4096, 0, None, 0, None) == 1
    ws = lib.lce_embedding_workspace_size(10, 64)
    assert ws > 0 and lib.lce_embedding_workspace_size(0, 64) == 0
    assert b(0, 4096, 4096, 0, 10, 64, 100, 4096, 0, 8192, ws - 1, None) == 6   # workspace too small
    # scratch grows with N (grouping the positions) and two partial rows of d per
    # 32 sorted positions, never with V
    assert lib.lce_embedding_workspace_size(16384, 4096) < 16384 * 64 + 2 * (16384 // 32 + 1) * 4096 * 4


def test_workspace_relations_across_options(lib):
    """The workspace of lce_run for each option, against what the layout
    needs: a fused optimizer holds a fourth G chunk buffer (N_pad * Vc bf16),
    a token cap bounds scratch by the cap instead of N, fp32 inputs hold
    split (hi, lo) copies."""
    def ws(**kw):
        a = _abi.LceArgs()
        a.dtype = kw.pop("dtype", 0)
        a.N, a.d, a.V = kw.pop("N", 5000), kw.pop("d", 1024), kw.pop("V", 50000)
        a.dH = 4096
        o = _abi.LceOptim()
        if kw.pop("optim", False):
            o.kind = _abi.LCE_OPT_SGD
            a.optim = ctypes.addressof(o)
        for k, v in kw.items():
            setattr(a, k, v)
        return lib.lce_workspace_size_args(ctypes.byref(a))

    n_pad = (5000 + 255) // 256 * 256
    vc = 5632                                                           # V = 50000: 9 chunks of 5632
    assert ws(optim=True) - ws() == n_pad * vc * 2                      # one more G buffer, default chunk
    assert ws(optim=True, vocab_chunk=2048) - ws(vocab_chunk=2048) == n_pad * 2048 * 2
    capped = ws(N=100000, token_chunk=4096)
    assert abs(capped - ws(N=200000, token_chunk=4096)) < 4096         # only the per-chunk loss sums grow
    assert capped < ws(N=100000) / 10
    assert ws(dtype=1) > ws() + 2 * 50000 * 1024 * 2                   # split copy of W (hi + lo)


def test_binding_arity_matches_header():
    """Each function's parameter count in include/lce.h equals the length of
    its ctypes argtypes (a mismatch would shift every later argument)."""
    import re
    text = open(os.path.join(INCLUDE, "lce.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = re.findall(r"\b(?:lce_status_t|size_t|int|int64_t|const char \*)\s*(lce_\w+)\s*\(([^)]*)\)\s*;", text)
    assert decls
    for name, params in decls:
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert name in _abi.SIGNATURES, name
        assert len(_abi.SIGNATURES[name][1]) == n, (name, n, len(_abi.SIGNATURES[name][1]))
    assert {d[0] for d in decls} == set(_abi.SIGNATURES)
