"""ctypes front end of the plain fp64 C++ oracle (oracle/lce_oracle.cpp).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module:
only the tests, the package's smoke check and the benchmark's CPU-baseline
leg do. It shares no code with the CUDA library; the two meet only through the
seeded arrays of ``synth_inputs``.

The functions mirror ``oracle.lce_oracle`` (same arguments, same result keys),
so the same pins run against both. Inputs may be float64, float32 or bf16 bit
patterns (uint16): each value is widened exactly inside the C++ code, so a
full-size bf16 workload needs no float64 copy. ``threads`` defaults to the
cores this process may run on (``os.sched_getaffinity``); the results do not
depend on it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

__all__ = ["build", "lib", "default_threads", "valid_rows", "forward", "forward_backward",
           "sampled_reference"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lce_oracle.cpp")
_LIB = os.path.join(_HERE, "liblce_oracle.so")
_lib = None

_F64, _F32, _BF16 = 0, 1, 2
_ERRORS = {1: "invalid arguments", 2: "a target outside [0, V) that is not ignore_index"}


def build(force: bool = False) -> str:
    """Compile liblce_oracle.so with the host C++ compiler (portable flags:
    no -march, so the same source builds on x86-64 and aarch64)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cmd = ["g++", "-O3", "-std=c++17", "-fPIC", "-shared", "-pthread", "-o", _LIB + ".tmp", _SRC]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"g++ failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        p, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.lceo_valid_rows.argtypes = [p, i64, i64, i64, p, p]
        L.lceo_forward_backward.argtypes = [p, p, c_int, p, i64, i64, i64, i64, c_int, p, p, p, p, p]
        L.lceo_sampled.argtypes = [p, p, c_int, p, i64, i64, i64, i64, c_int, p, i64, p, i64, p, p, p, p]
        for f in (L.lceo_valid_rows, L.lceo_forward_backward, L.lceo_sampled):
            f.restype = c_int
        _lib = L
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _input(a):
    """(contiguous array, dtype code) without copying float32 / bf16 bits."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), _BF16
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), _F32
    return np.ascontiguousarray(a, dtype=np.float64), _F64


def _operands(H, W, targets, bf16):
    H, W = np.asarray(H), np.asarray(W)
    if bf16:
        H, W = H.view(np.uint16), W.view(np.uint16)
    H, dh = _input(H)
    W, dw = _input(W)
    if dh != dw:                       # mixed input types: widen both to float64
        H, W, dh = _as_f64(H, dh), _as_f64(W, dw), _F64
    t = np.ascontiguousarray(targets, dtype=np.int64)
    if H.ndim != 2 or W.ndim != 2 or t.ndim != 1 or H.shape[0] != t.shape[0] or H.shape[1] != W.shape[1]:
        raise ValueError("H must be [N,d], W [V,d], targets [N]")
    return H, W, dh, t


def _as_f64(a, code):
    if code == _BF16:
        a = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.ascontiguousarray(a, dtype=np.float64)


def _raise(rc):
    if rc:
        raise ValueError(f"C++ oracle: {_ERRORS.get(rc, rc)}")


def valid_rows(targets, ignore_index: int, V: int | None = None) -> np.ndarray:
    t = np.ascontiguousarray(targets, dtype=np.int64)
    idx = np.empty(t.shape[0], dtype=np.int64)
    nv = ctypes.c_int64(0)
    _raise(lib().lceo_valid_rows(_ptr(t), ignore_index, t.shape[0], V if V is not None else 0, _ptr(idx),
                                 ctypes.byref(nv)))
    return idx[:nv.value]


def forward_backward(H, W, targets, ignore_index: int = -100, threads: int | None = None, bf16: bool = False,
                     grads: bool = True) -> dict:
    """Loss, per-row lse and loss terms, dH [N,d] and dW [V,d] (float64).
    bf16=True reads uint16 / int16 arrays as bf16 bit patterns."""
    H, W, dt, t = _operands(H, W, targets, bf16)
    N, d = H.shape
    V = W.shape[0]
    loss = ctypes.c_double(0.0)
    lse = np.empty(N)
    terms = np.empty(N)
    dH = np.empty((N, d)) if grads else None
    dW = np.empty((V, d)) if grads else None
    _raise(lib().lceo_forward_backward(_ptr(H), _ptr(W), dt, _ptr(t), ignore_index, N, d, V,
                                       threads or default_threads(), ctypes.byref(loss), _ptr(lse), _ptr(terms),
                                       _ptr(dH), _ptr(dW)))
    idx = np.nonzero(t != ignore_index)[0]
    out = {"loss": loss.value, "lse": lse[idx], "loss_rows": terms[idx], "idx": idx, "n_valid": int(idx.shape[0])}
    if grads:
        out.update(dH=dH, dW=dW)
    return out


def forward(H, W, targets, ignore_index: int = -100, threads: int | None = None, bf16: bool = False) -> dict:
    return forward_backward(H, W, targets, ignore_index, threads, bf16, grads=False)


def sampled_reference(H, W, targets, ignore_index, token_rows, vocab_rows, threads: int | None = None,
                      bf16: bool = False) -> dict:
    """The loss and every valid row's lse, dH on the sampled token rows and dW
    on the sampled vocab rows (same keys as oracle.sampled_reference)."""
    H, W, dt, t = _operands(H, W, targets, bf16)
    N, d = H.shape
    V = W.shape[0]
    rows = np.ascontiguousarray(token_rows, dtype=np.int64)
    vocab = np.ascontiguousarray(vocab_rows, dtype=np.int64)
    loss = ctypes.c_double(0.0)
    lse = np.empty(N)
    dH_rows = np.empty((rows.shape[0], d))
    dW_rows = np.empty((vocab.shape[0], d))
    _raise(lib().lceo_sampled(_ptr(H), _ptr(W), dt, _ptr(t), ignore_index, N, d, V, threads or default_threads(),
                              _ptr(rows), rows.shape[0], _ptr(vocab), vocab.shape[0], ctypes.byref(loss), _ptr(lse),
                              _ptr(dH_rows), _ptr(dW_rows)))
    idx = np.nonzero(t != ignore_index)[0]
    return {"loss": loss.value, "lse": lse[idx], "idx": idx, "n_valid": int(idx.shape[0]),
            "token_rows": rows, "dH_rows": dH_rows, "vocab_rows": vocab, "dW_rows": dW_rows}
