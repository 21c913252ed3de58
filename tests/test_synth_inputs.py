"""The seeded generator: determinism, the padding recipes and the bf16 rounding."""
import numpy as np
import pytest

import synth_inputs as si


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, -2.5, 0.0], dtype=np.float32)
    assert si.f32_to_bf16_bits(x).tolist() == [0x3F80, 0xC020, 0x0000]
    bits = np.array([0x3F808000, 0x3F818000, 0x3F808001, 0x3F807FFF], dtype=np.uint32)
    # tie rounds to even (down, then up), above the tie rounds up, below rounds down
    assert si.f32_to_bf16_bits(bits.view(np.float32)).tolist() == [0x3F80, 0x3F82, 0x3F81, 0x3F80]
    back = si.bf16_bits_to_f32(np.array([0x3F80, 0xC020], dtype=np.uint16))
    assert back.tolist() == [1.0, -2.5]


@pytest.mark.parametrize("name,nv", [("tiny", 230), ("gpt1b", 3482), ("vocab256k", 9832)])
def test_valid_counts_follow_the_recipe(name, nv):
    t = si.make_targets(si.WORKLOADS[name])
    assert int((t != si.IGNORE_INDEX).sum()) == nv


def test_targets_in_range_and_padding_layout():
    w = si.WORKLOADS["llama8b"]
    t = si.make_targets(w)
    v = t != si.IGNORE_INDEX
    assert t[v].min() >= 0 and t[v].max() < w.V
    L = w.N // w.seqs
    for b in range(w.seqs):
        seg = v[b * L:(b + 1) * L]
        n = seg.sum()
        assert 64 <= n <= 2048
        assert seg[:n].all() and not seg[n:].any()      # first L_b positions valid


def test_deterministic_and_thread_independent():
    a = si.make_inputs("tiny")
    b = si.make_inputs("tiny")
    np.testing.assert_array_equal(a.H, b.H)
    np.testing.assert_array_equal(a.W, b.W)
    np.testing.assert_array_equal(a.targets, b.targets)
    m1 = si._normal_matrix(0, 2, 3000, 16, 1.0, True, threads=1)
    m4 = si._normal_matrix(0, 2, 3000, 16, 1.0, True, threads=4)
    np.testing.assert_array_equal(m1, m4)


def test_weight_scale():
    x = si.make_inputs("gpt1b", N=64, V=4096)
    W = x.W_f32().astype(np.float64)
    assert W.std() * np.sqrt(x.workload.d) == pytest.approx(3.0, rel=0.02)
