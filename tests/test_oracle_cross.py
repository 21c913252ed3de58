"""The two implementations of the oracle agree: the plain C++ one (loops over
rows, std::thread) and the numpy one (library matmuls). They share nothing but
the definition, so agreement to rounding on random shapes — tails of the
eight-way dot product, a single class, no valid row, bf16 and fp32 inputs
widened exactly, the tiny workload in full — says that neither has a slip the
pins could both miss. Also: the C++ results do not depend on the thread count
(each output is produced by one thread in a fixed order)."""
import numpy as np
import pytest

import oracle
from oracle import cpp_oracle
from synth_inputs import IGNORE_INDEX, make_inputs


def _case(N, d, V, seed, pad=0.3, scale=2.0):
    g = np.random.default_rng(seed)
    H = g.standard_normal((N, d))
    W = g.standard_normal((V, d)) * scale
    t = g.integers(0, V, N)
    t[g.random(N) < pad] = IGNORE_INDEX
    return H, W, t


def _agree(a, b, rtol=1e-12):
    if np.isnan(a["loss"]):
        assert np.isnan(b["loss"])
    else:
        assert b["loss"] == pytest.approx(a["loss"], rel=rtol, abs=1e-14)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=rtol, atol=1e-13)
    for k in ("dH", "dW"):
        scale = max(np.abs(a[k]).max(), 1e-300)
        assert np.abs(b[k] - a[k]).max() <= rtol * scale, k


@pytest.mark.parametrize("N,d,V,seed", [(1, 1, 2, 0), (5, 7, 3, 1), (40, 9, 1, 2), (64, 17, 130, 3),
                                         (123, 33, 257, 4), (300, 40, 517, 5)])
def test_cpp_and_numpy_agree_float64(N, d, V, seed):
    H, W, t = _case(N, d, V, seed)
    _agree(oracle.forward_backward(H, W, t), cpp_oracle.forward_backward(H, W, t))


def test_cpp_and_numpy_agree_without_valid_rows():
    H, W, t = _case(20, 8, 11, 6)
    t[:] = IGNORE_INDEX
    _agree(oracle.forward_backward(H, W, t), cpp_oracle.forward_backward(H, W, t))


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("gpt1b", dict(N=200, d=72, V=701))])
def test_cpp_reads_the_workload_inputs_exactly(name, kw):
    """fp32 and bf16 inputs are handed to the C++ oracle as stored (bf16 as bit
    patterns) and widened there; the numpy oracle gets the float64 values."""
    x = make_inputs(name, **kw)
    a = oracle.forward_backward(x.H_f32().astype(np.float64), x.W_f32().astype(np.float64), x.targets)
    b = cpp_oracle.forward_backward(x.H, x.W, x.targets, bf16=x.bf16)
    _agree(a, b)


def test_cpp_sampled_reference_matches_numpy():
    H, W, t = _case(300, 24, 170, 7)
    rows = np.array([0, 5, 17, 299, 123, 5])
    vocab = np.array([0, 169, 33, 1, t[3] if t[3] >= 0 else 2])
    a = oracle.sampled_reference(H, W, t, IGNORE_INDEX, rows, vocab)
    b = cpp_oracle.sampled_reference(H, W, t, IGNORE_INDEX, rows, vocab)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-12)
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=1e-12)
    np.testing.assert_allclose(b["dH_rows"], a["dH_rows"], rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(b["dW_rows"], a["dW_rows"], rtol=1e-11, atol=1e-15)


def test_cpp_results_do_not_depend_on_thread_count():
    H, W, t = _case(97, 19, 61, 8)
    one = cpp_oracle.forward_backward(H, W, t, threads=1)
    for th in (2, 3, 7):
        r = cpp_oracle.forward_backward(H, W, t, threads=th)
        assert r["loss"] == one["loss"]
        assert np.array_equal(r["dH"], one["dH"]) and np.array_equal(r["dW"], one["dW"])


def test_cpp_refuses_out_of_range_targets():
    H, W, t = _case(6, 3, 4, 9, pad=0.0)
    t[2] = 4
    with pytest.raises(ValueError):
        cpp_oracle.forward_backward(H, W, t)
    t[2] = -1
    with pytest.raises(ValueError):
        cpp_oracle.forward(H, W, t)
