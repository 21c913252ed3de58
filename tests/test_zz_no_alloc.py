"""lce_forward_noalloc: the forward loss for callers that must not allocate
device memory (fixed memory budgets, hosts that forbid allocation after
start-up). Called through the C ABI and compared with the fp64 C++ oracle and
with lce_forward, which allocates its scratch, on calls in a row: each reuses
the library's fixed scratch array left over from the one before, including a
small call with another N and V right after one at the size limits, and a call
with no valid token (NaN loss). This file is collected last so a failure here
never hides another test's result."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from chunked_vocab_cross_gb300 import _abi  # noqa: E402
from lce_testutil import TOL_LOSS, to_device  # noqa: E402
from oracle import cpp_oracle  # noqa: E402
from synth_inputs import IGNORE_INDEX, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from chunked_vocab_cross_gb300.build import build
    build()
    yield


def _call(fn, H, W, t, loss):
    lib = _abi.lib()
    N, d = H.shape
    V = W.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    return getattr(lib, fn)(ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                            ctypes.c_void_p(t.data_ptr()), IGNORE_INDEX, N, d, V,
                            ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(stream))


def test_noalloc_forward_matches_oracle_and_lce_forward_in_a_row():
    cases = [make_inputs("gpt1b", N=4096, d=2048, V=5000, seqs=1),                         # at the limits
             make_inputs("gpt1b", N=777, d=512, V=3001, padding=("random_frac", 0.4), seqs=1),
             make_inputs("gpt1b", N=4096, d=2048, V=5000, seqs=1, seed=3),
             make_inputs("gpt1b", N=33, d=64, V=257, padding=("random_frac", 0.5), seqs=1, seed=5)]
    for x in cases:
        H, W, t = to_device(x)
        ref = cpp_oracle.forward(x.H, x.W, x.targets, IGNORE_INDEX, bf16=True)["loss"]
        lf = torch.empty((), dtype=torch.float32, device="cuda")
        assert _call("lce_forward", H, W, t, lf) == 0
        for _ in range(2):
            out = torch.full((), float("nan"), dtype=torch.float32, device="cuda")
            assert _call("lce_forward_noalloc", H, W, t, out) == 0
            torch.cuda.synchronize()
            assert np.isfinite(out.item())
            assert abs(out.item() - ref) <= TOL_LOSS, (x.workload, out.item(), ref)
            assert abs(out.item() - lf.item()) <= TOL_LOSS, (out.item(), lf.item())


def test_noalloc_without_valid_tokens_gives_nan():
    x = make_inputs("gpt1b", N=1000, d=256, V=999, padding=("all",), seqs=1)
    assert cpp_oracle.forward(x.H, x.W, x.targets, IGNORE_INDEX, bf16=True)["n_valid"] == 0
    H, W, t = to_device(x)
    out = torch.zeros((), dtype=torch.float32, device="cuda")
    assert _call("lce_forward_noalloc", H, W, t, out) == 0
    torch.cuda.synchronize()
    assert np.isnan(out.item())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    x = make_inputs("gpt1b", N=64, d=64, V=500, seqs=1)
    H, W, t = to_device(x)
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    big = torch.zeros((4097, 64), dtype=torch.bfloat16, device="cuda")
    tb = torch.zeros(4097, dtype=torch.int64, device="cuda")
    assert _call("lce_forward_noalloc", big, W, tb, loss) == 2          # N > 4096: LCE_ERR_SHAPE
    wide = torch.zeros((64, 2056), dtype=torch.bfloat16, device="cuda")
    wW = torch.zeros((500, 2056), dtype=torch.bfloat16, device="cuda")
    assert _call("lce_forward_noalloc", wide, wW, t, loss) == 2         # d > 2048: LCE_ERR_SHAPE
