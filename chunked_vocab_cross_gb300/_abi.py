"""ctypes binding of liblce.so (include/lce.h). Argument marshalling only: every
step of the computation runs in the library's CUDA kernels. There is no CPU
path: if the library is missing or cannot load, every call raises."""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblce.so")

LCE_BF16, LCE_FP32 = 0, 1
LCE_DEV_TARGET_RANGE, LCE_DEV_TIMEOUT = 0x1, 0x2
PROFILE_PHASES = 5
PHASE_NAMES = ("compact_gather", "logits_lse", "lse_merge_loss", "backward", "dH_scatter")

STATUS = {
    0: "LCE_OK", 1: "LCE_ERR_NULL", 2: "LCE_ERR_SHAPE", 3: "LCE_ERR_ALIGN", 4: "LCE_ERR_DTYPE",
    5: "LCE_ERR_CUDA", 6: "LCE_ERR_WORKSPACE", 7: "LCE_ERR_TARGET_RANGE", 8: "LCE_ERR_TIMEOUT",
    9: "LCE_ERR_DEVICE", 10: "LCE_ERR_ARG",
}
LCE_OPT_NONE, LCE_OPT_SGD, LCE_OPT_ADAMW = 0, 1, 2

# Every function include/lce.h declares: name -> (restype, argtypes)
SIGNATURES = {
    "lce_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_void_p, c_void_p]),
    "lce_forward_backward": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_void_p,
                                     c_void_p, c_void_p, c_void_p]),
    "lce_forward_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_void_p,
                                    c_void_p]),
    "lce_compact": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p, c_void_p, c_void_p]),
    "lce_run": (c_int, [c_void_p]),
    "lce_backward": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_void_p]),
    "lce_workspace_size": (c_size_t, [c_int64, c_int64, c_int64, c_int, c_int64]),
    "lce_workspace_size_args": (c_size_t, [c_void_p]),
    "lce_get_device_status": (c_int, [c_void_p, ctypes.POINTER(c_int32)]),
    "lce_status_string": (ctypes.c_char_p, [c_int]),
    "lce_last_cuda_error": (c_int, []),
    "lce_launch_count": (c_int64, []),
    "lce_profile_begin": (c_int, []),
    "lce_profile_end": (c_int, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_int64), c_int]),
    "lce_version": (c_int, []),
    "lce_selftest_wait_timeout": (c_int, [c_int64, c_void_p, c_void_p]),
    "lce_embedding_forward": (c_int, [c_int, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_void_p,
                                      c_void_p]),
    "lce_embedding_workspace_size": (c_size_t, [c_int64, c_int64]),
    "lce_embedding_backward": (c_int, [c_int, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_void_p, c_int,
                                       c_void_p, c_size_t, c_void_p]),
    "lce_embedding_backward_bf16": (c_int, [c_int, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_void_p,
                                            c_void_p, c_size_t, c_void_p]),
}


class LceOptim(ctypes.Structure):
    """Mirror of lce_optim_t."""
    _fields_ = [
        ("kind", c_int),
        ("lr", c_float), ("weight_decay", c_float), ("momentum", c_float),
        ("beta1", c_float), ("beta2", c_float), ("eps", c_float),
        ("step", c_int64),
        ("master_W", c_void_p), ("exp_avg", c_void_p), ("exp_avg_sq", c_void_p),
        ("state_bf16", c_int),
    ]


class LceArgs(ctypes.Structure):
    """Mirror of lce_args_t."""
    _fields_ = [
        ("dtype", c_int),
        ("H", c_void_p), ("W", c_void_p), ("targets", c_void_p),
        ("ignore_index", c_int64), ("N", c_int64), ("d", c_int64), ("V", c_int64),
        ("loss", c_void_p), ("dH", c_void_p), ("dW", c_void_p),
        ("accumulate_dW", c_int), ("grad_scale", c_float),
        ("lse", c_void_p),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("vocab_chunk", c_int64),
        ("stream", c_void_p),
        ("lse_in", c_void_p),
        ("grad_loss", c_void_p),
        ("token_chunk", c_int64),
        ("optim", c_void_p),
        ("row_gather", c_int),
        ("dW_bf16", c_int),
    ]


class LceError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        name = STATUS.get(code, str(code))
        msg = f"{what}: {name}" if what else name
        if code == 5:
            msg += f" (cudaError {lib().lce_last_cuda_error()})"
        super().__init__(msg)


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded library; raises if liblce.so has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise ImportError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc 13, sm_103a)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def check(code: int, what: str = "") -> None:
    if code != 0:
        raise LceError(code, what)
