"""Input-embedding lookup that skips padding and its gradient, through the C
ABI, against the fp64 oracle: the forward is an exact copy (bit for bit), the
backward a sum of each token's gradient rows in fp32 (relative Frobenius error
within 1e-6: the rows of the bf16/fp32 inputs are added exactly in fp64 by the
oracle, in fp32 here; a row of k terms is off by at most about k * 2^-24 of its
absolute sum, and the segments here have at most a few hundred rows), and
bit-for-bit reproducible."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import chunked_vocab_cross_gb300 as lce  # noqa: E402
import oracle  # noqa: E402
from lce_testutil import TOL_LOSS, TOL_REL, np64, rel_fro, to_device  # noqa: E402
from synth_inputs import (IGNORE_INDEX, WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_inputs,  # noqa: E402
                          make_targets)

pytestmark = pytest.mark.gpu
TOL_EMB = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from chunked_vocab_cross_gb300.build import build
    build()
    lce.device_status()
    yield


def _case(N, d, V, pad, dtype, seed=0, frac=0.3):
    g = np.random.default_rng(seed)
    W = g.standard_normal((V, d)).astype(np.float32)
    dE = g.standard_normal((N, d)).astype(np.float32)
    # Zipf-like token ids (a few very frequent ones), a fraction of padding
    t = np.minimum((g.pareto(1.1, N) * 3).astype(np.int64), V - 1)
    t[g.random(N) < frac] = pad
    if dtype == torch.bfloat16:
        W = bf16_bits_to_f32(f32_to_bf16_bits(W))
        dE = bf16_bits_to_f32(f32_to_bf16_bits(dE))
    dev = lambda a: torch.from_numpy(a).to("cuda").to(dtype)  # noqa: E731
    return W, dE, t, dev(W), dev(dE), torch.from_numpy(t).cuda()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("shape", [(1, 8, 3, 0), (777, 200, 5000, 0), (4100, 256, 300, 2), (2048, 1024, 70000, 0)],
                         ids=lambda s: f"N{s[0]}_d{s[1]}_V{s[2]}_pad{s[3]}")
def test_embedding_forward_backward_vs_oracle(shape, dtype):
    N, d, V, pad = shape
    W, dE, t, Wd, dEd, td = _case(N, d, V, pad, dtype)
    E = lce.embedding_forward(Wd, td, pad)
    dW = lce.embedding_backward(dEd, td, pad, V)
    dW2 = lce.embedding_backward(dEd, td, pad, V)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    np.testing.assert_array_equal(np64(E), oracle.embedding_forward(W, t, pad))
    ref = oracle.embedding_backward(dE, t, pad, V)
    err = rel_fro(np64(dW), ref) if np.any(ref) else float(np.abs(np64(dW)).max())
    assert err <= TOL_EMB, err
    assert torch.equal(dW, dW2)                        # reproducible bit for bit
    untouched = np.setdiff1d(np.arange(V), t[t != pad])
    assert torch.count_nonzero(dW[torch.from_numpy(untouched).cuda()]).item() == 0


def test_embedding_accumulate_and_all_padding():
    W, dE, t, Wd, dEd, td = _case(500, 64, 900, 0, torch.float32, seed=1)
    base = torch.randn(900, 64, device="cuda")
    dW = lce.embedding_backward(dEd, td, 0, 900, dW=base.clone(), accumulate=True)
    ref = oracle.embedding_backward(dE, t, 0, 900) + np64(base)
    assert rel_fro(np64(dW), ref) <= TOL_EMB
    tp = torch.zeros_like(td)                           # every position is padding
    E = lce.embedding_forward(Wd, tp, 0)
    dW = lce.embedding_backward(dEd, tp, 0, 900, dW=base.clone(), accumulate=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(E).item() == 0 and torch.equal(dW, base)


def test_embedding_out_of_range_token_is_flagged_and_skipped():
    W, dE, t, Wd, dEd, td = _case(300, 64, 500, 0, torch.bfloat16, seed=2)
    td = td.clone()
    td[7] = 500
    td[9] = -5
    E = lce.embedding_forward(Wd, td, 0)
    torch.cuda.synchronize()
    assert lce.device_status() & 1
    assert torch.count_nonzero(E[7]).item() == 0 and torch.count_nonzero(E[9]).item() == 0
    dW = lce.embedding_backward(dEd, td, 0, 500)
    torch.cuda.synchronize()
    assert lce.device_status() & 1
    t2 = t.copy()
    t2[[7, 9]] = 0                                      # the oracle's reading: skipped like padding
    assert rel_fro(np64(dW), oracle.embedding_backward(dE, t2, 0, 500)) <= TOL_EMB


def test_tied_W_gradients_add_into_one_buffer():
    """A tied W: the output projection's dW (lce_run) and the input
    embedding's gradient accumulate into one fp32 buffer; equals the oracle's
    two gradients added."""
    x = make_inputs("gpt1b", N=900, d=256, V=3000, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    tokens = torch.from_numpy(np.where(x.targets == IGNORE_INDEX, 0, (x.targets + 1) % 3000)).cuda()
    dE = torch.randn(900, 256, device="cuda").to(torch.bfloat16)
    loss, dH, dW = lce.lce_forward_backward(H, W, t, IGNORE_INDEX)
    lce.embedding_backward(dE, tokens, 0, 3000, dW=dW, accumulate=True)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    ref_dW = ref["dW"] + oracle.embedding_backward(np64(dE), tokens.cpu().numpy(), 0, 3000)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
    assert rel_fro(np64(dW), ref_dW) <= TOL_REL


def test_embedding_autograd_function():
    W, dE, t, Wd, dEd, td = _case(400, 128, 1000, 0, torch.float32, seed=4)
    Wp = Wd.clone().requires_grad_(True)
    E = lce.embedding(Wp, td, 0)
    E.backward(dEd)
    assert rel_fro(np64(Wp.grad), oracle.embedding_backward(dE, t, 0, 1000)) <= TOL_EMB
    np.testing.assert_array_equal(np64(E.detach()), oracle.embedding_forward(W, t, 0))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["dE_bf16", "dE_fp32"])
@pytest.mark.parametrize("shape", [(1, 8, 3, 0), (777, 200, 5000, 0), (4100, 256, 300, 2), (3000, 64, 40, 1)],
                         ids=lambda s: f"N{s[0]}_d{s[1]}_V{s[2]}_pad{s[3]}")
def test_embedding_backward_bf16_output_is_the_fp32_output_rounded(shape, dtype):
    """bf16 dW: every row sum taken in fp32 as for the fp32 output and rounded
    once (tokens whose rows span several 32-element chunks included: V = 40
    and 300 with thousands of positions), bit for bit."""
    N, d, V, pad = shape
    _, _, _, _, dEd, td = _case(N, d, V, pad, dtype, seed=7)
    dW32 = lce.embedding_backward(dEd, td, pad, V)
    dW16 = torch.full((V, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lce.embedding_backward(dEd, td, pad, V, dW=dW16)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    assert torch.equal(dW16.view(torch.int16), dW32.to(torch.bfloat16).view(torch.int16))
    with pytest.raises(ValueError):
        lce.embedding_backward(dEd, td, pad, V, dW=dW16, accumulate=True)


def test_embedding_autograd_bf16_W_grad_in_bf16():
    W, dE, t, Wd, dEd, td = _case(900, 96, 700, 0, torch.bfloat16, seed=5)
    Wp = Wd.clone().requires_grad_(True)
    E = lce.embedding(Wp, td, 0)
    E.backward(dEd)
    torch.cuda.synchronize()
    assert Wp.grad.dtype == torch.bfloat16
    ref32 = lce.embedding_backward(dEd, td, 0, 700)
    assert torch.equal(Wp.grad.view(torch.int16), ref32.to(torch.bfloat16).view(torch.int16))
    assert rel_fro(np64(Wp.grad), oracle.embedding_backward(dE, t, 0, 700)) <= 2 ** -8


def test_embedding_llama8b_shape_sampled_rows():
    """Full llama8b shape (N=16384, d=4096, V=128256): Zipf token ids with the
    workload's padding; the gradient checked on 256 sampled vocab rows (the
    oracle run on the positions of those tokens, ids remapped to 0..255), the
    forward on 256 sampled positions."""
    tg = make_targets(WORKLOADS["llama8b"])
    pad = 0
    t = np.where(tg == IGNORE_INDEX, pad, tg)
    g = np.random.default_rng(9)
    W32 = bf16_bits_to_f32(f32_to_bf16_bits(g.standard_normal((128256, 4096), dtype=np.float32) * 0.05))
    dE32 = bf16_bits_to_f32(f32_to_bf16_bits(g.standard_normal((16384, 4096), dtype=np.float32) * 1e-3))
    Wd = torch.from_numpy(W32).cuda().to(torch.bfloat16)
    dEd = torch.from_numpy(dE32).cuda().to(torch.bfloat16)
    td = torch.from_numpy(t).cuda()
    E = lce.embedding_forward(Wd, td, pad)
    dW = lce.embedding_backward(dEd, td, pad, 128256)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    pos = np.sort(g.choice(16384, 256, replace=False))
    np.testing.assert_array_equal(np64(E[torch.from_numpy(pos).cuda()]), oracle.embedding_forward(W32, t[pos], pad))
    valid_ids = np.unique(t[t != pad])
    rows = np.sort(np.concatenate([valid_ids[:128], g.choice(128256, 128, replace=False)]))
    rows = np.unique(rows[rows != pad])
    remap = np.full(128256, -1, dtype=np.int64)
    remap[rows] = np.arange(len(rows))
    sel = (t != pad) & (remap[t] >= 0)
    ref = oracle.embedding_backward(dE32[sel], remap[t[sel]], -1, len(rows))
    got = np64(dW[torch.from_numpy(rows).cuda()])
    assert rel_fro(got, ref) <= TOL_EMB
