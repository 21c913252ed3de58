"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on seeded
inputs: element by element at sizes the oracle finishes in seconds (several
tiles plus ragged tails), and edge cases. Tolerances: |loss| <= 1e-3 and
relative Frobenius error <= 5e-3 for dH and dW on bf16 inputs."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import chunked_vocab_cross_gb300 as lce  # noqa: E402
import oracle  # noqa: E402
from lce_testutil import TOL_LOSS, TOL_LSE, TOL_REL, np64, rel_fro, to_device  # noqa: E402
from synth_inputs import IGNORE_INDEX, WORKLOADS, make_inputs, make_targets  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from chunked_vocab_cross_gb300.build import build
    build()
    lce.device_status()   # clear the status word
    yield


def _run_and_compare(x, vocab_chunk=0, tol_loss=TOL_LOSS, tol_rel=TOL_REL, tol_lse=TOL_LSE):
    H, W, t = to_device(x)
    loss, dH, dW, lse = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, vocab_chunk=vocab_chunk, return_lse=True)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    valid = x.targets != IGNORE_INDEX
    lse_g = np64(lse)
    errs = {
        "loss": abs(loss.item() - ref["loss"]),
        "lse": float(np.max(np.abs(lse_g[valid] - ref["lse"]))) if valid.any() else 0.0,
        "dH": rel_fro(np64(dH), ref["dH"]),
        "dW": rel_fro(np64(dW), ref["dW"]),
    }
    print(x.workload, errs)
    assert np.all(np.isnan(lse_g[~valid]))
    assert np.all(np64(dH)[~valid] == 0.0)
    assert errs["loss"] <= tol_loss, errs
    assert errs["lse"] <= tol_lse, errs
    assert errs["dH"] <= tol_rel, errs
    assert errs["dW"] <= tol_rel, errs
    return errs


# ------------------------------------------------------------------ compaction

def _compaction_cases():
    g = np.random.default_rng(0)
    cases = []
    for name, w in WORKLOADS.items():
        cases.append((name, make_targets(w), w.V))
    for n in (1, 31, 32, 33, 1023, 1024, 1025, 5000):
        t = g.integers(0, 100, n)
        t[g.random(n) < 0.37] = IGNORE_INDEX
        cases.append((f"rand{n}", t, 100))
    cases.append(("all_ignored", np.full(77, IGNORE_INDEX), 10))
    cases.append(("none_ignored", np.arange(2049) % 10, 10))
    t = np.array([5, IGNORE_INDEX, 10, -1, 9, 12, IGNORE_INDEX, 0])
    cases.append(("out_of_range", t, 10))
    return cases


@pytest.mark.parametrize("case", _compaction_cases(), ids=lambda c: c[0])
def test_compaction_bit_exact(case):
    _, t, V = case
    idx, inv, nv, bad = lce.lce_compact(torch.from_numpy(t).cuda(), IGNORE_INDEX, V)
    expect = oracle.valid_rows(t, IGNORE_INDEX)
    assert nv == len(expect)
    np.testing.assert_array_equal(idx.cpu().numpy(), expect)
    inv_expect = np.full(len(t), -1)
    inv_expect[expect] = np.arange(len(expect))
    np.testing.assert_array_equal(inv.cpu().numpy(), inv_expect)
    assert bad == oracle.out_of_range_targets(t, IGNORE_INDEX, V)
    lce.device_status()


# ------------------------------------------------------------- small parity

SMALL = [
    # (N, d, V, padding)   chosen to span several 128x256 tiles and ragged tails
    (1, 64, 1000, ("none",)),
    (127, 64, 1000, ("random_frac", 0.0)),
    (129, 128, 513, ("random_frac", 0.2)),
    (300, 128, 1000, ("random_frac", 0.1)),
    (256, 64, 1000, ("random_frac", 0.1)),
    (700, 200, 4099, ("random_frac", 0.3)),
    (1000, 256, 3000, ("random_frac", 0.5)),
    (640, 512, 8192, ("trailing_frac", 0.25)),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: f"N{s[0]}_d{s[1]}_V{s[2]}")
def test_small_bf16_parity(shape):
    N, d, V, pad = shape
    x = make_inputs("gpt1b", N=N, d=d, V=V, padding=pad, seqs=1)
    _run_and_compare(x)


FP32 = [(1, 64, 1000), (300, 128, 1000), (700, 200, 4099), (333, 64, 300)]


@pytest.mark.parametrize("shape", FP32, ids=lambda s: f"N{s[0]}_d{s[1]}_V{s[2]}")
def test_small_fp32_split_parity(shape):
    """fp32 inputs through the split-precision (bf16 hi/lo) tensor-core path,
    including several vocab chunks."""
    N, d, V = shape
    x = make_inputs("tiny", N=N, d=d, V=V, padding=("random_frac", 0.1))
    errs = _run_and_compare(x, vocab_chunk=1024)
    assert errs["loss"] <= 1e-4 and errs["dH"] <= 1e-3 and errs["dW"] <= 1e-3, errs


@pytest.mark.parametrize("vocab_chunk", [256, 768, 1024])
def test_vocab_chunk_sizes(vocab_chunk):
    x = make_inputs("gpt1b", N=500, d=256, V=2900, padding=("random_frac", 0.2), seqs=1)
    _run_and_compare(x, vocab_chunk=vocab_chunk)


def test_tiny_workload_bf16_rounded():
    """The tiny workload's shapes with bf16 inputs (the fp32 path has its own test)."""
    w = WORKLOADS["tiny"].with_(dtype="bf16")
    _run_and_compare(make_inputs(w))


def test_all_ignored_gives_nan_and_zero_grads():
    x = make_inputs("gpt1b", N=200, d=64, V=700, padding=("all",), seqs=1)
    H, W, t = to_device(x)
    loss, dH, dW = lce.lce_forward_backward(H, W, t, IGNORE_INDEX)
    torch.cuda.synchronize()
    assert math.isnan(loss.item())
    assert torch.count_nonzero(dH).item() == 0
    assert torch.count_nonzero(dW).item() == 0
    assert lce.device_status() == 0


def test_forward_only_matches_oracle():
    x = make_inputs("gpt1b", N=400, d=128, V=2000, padding=("random_frac", 0.15), seqs=1)
    H, W, t = to_device(x)
    loss = lce.lce_forward(H, W, t, IGNORE_INDEX)
    ref = oracle.forward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS


def test_out_of_range_target_sets_status_and_nan():
    x = make_inputs("gpt1b", N=64, d=64, V=500, padding=("none",), seqs=1)
    x.targets[7] = 500
    H, W, t = to_device(x)
    loss, dH, dW = lce.lce_forward_backward(H, W, t, IGNORE_INDEX)
    bits = lce.device_status()
    assert bits & 0x1
    assert math.isnan(loss.item())


def test_deterministic_bitwise():
    x = make_inputs("gpt1b", N=1500, d=512, V=6000, padding=("random_frac", 0.3), seqs=1)
    H, W, t = to_device(x)
    a = lce.lce_forward_backward(H, W, t, IGNORE_INDEX)
    b = lce.lce_forward_backward(H, W, t, IGNORE_INDEX)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int8) if u.dim() else u, v.view(torch.int8) if v.dim() else v)


def test_accumulate_dW_and_grad_scale():
    x = make_inputs("gpt1b", N=300, d=128, V=1500, padding=("random_frac", 0.1), seqs=1)
    H, W, t = to_device(x)
    base = torch.randn(W.shape, device="cuda", dtype=torch.float32)
    dW = base.clone()
    loss, dH, dW = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, dW=dW, accumulate_dW=True, grad_scale=0.5)
    torch.cuda.synchronize()
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert rel_fro(np64(dW - base), 0.5 * ref["dW"]) <= TOL_REL
    assert rel_fro(np64(dH), 0.5 * ref["dH"]) <= TOL_REL


def test_autograd_function_input_grad_only():
    x = make_inputs("gpt1b", N=200, d=64, V=900, padding=("random_frac", 0.1), seqs=1)
    H, W, t = to_device(x)
    H.requires_grad_(True)
    loss = lce.linear_cross_entropy(H, W, t, IGNORE_INDEX)
    (2.0 * loss).backward()
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
    assert rel_fro(np64(H.grad), 2 * ref["dH"]) <= 1e-2      # grads rounded to bf16 on return
    assert W.grad is None


def test_canaries_untouched():
    """Outputs sit inside larger buffers filled with a sentinel; nothing outside
    the output ranges may change (bounds check without compute-sanitizer)."""
    x = make_inputs("gpt1b", N=333, d=136, V=1234, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    N, d, V = 333, 136, 1234
    pad = 4096
    dh_buf = torch.full((N * d + 2 * pad,), 7.0, device="cuda", dtype=torch.bfloat16)
    dw_buf = torch.full((V * d + 2 * pad,), 7.0, device="cuda", dtype=torch.float32)
    loss_buf = torch.full((2 * pad + 1,), 7.0, device="cuda", dtype=torch.float32)
    lse_buf = torch.full((N + 2 * pad,), 7.0, device="cuda", dtype=torch.float32)
    dH = dh_buf[pad:pad + N * d].view(N, d)
    dW = dw_buf[pad:pad + V * d].view(V, d)
    loss = loss_buf[pad]
    lse = lse_buf[pad:pad + N]
    lce.lce_run(H, W, t, IGNORE_INDEX, loss=loss, dH=dH, dW=dW, lse=lse)
    torch.cuda.synchronize()
    for buf, n in ((dh_buf, N * d), (dw_buf, V * d), (loss_buf, 1), (lse_buf, N)):
        assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + n:] == 7.0)
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
    assert rel_fro(np64(dW), ref["dW"]) <= TOL_REL


def test_caller_workspace_and_size():
    x = make_inputs("gpt1b", N=400, d=128, V=1500, padding=("random_frac", 0.1), seqs=1)
    H, W, t = to_device(x)
    n = lce.workspace_size(400, 128, 1500)
    assert n > 0      # the O(N*(d + chunk)) bound at scale is checked in test_abi.py
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    loss, dH, dW = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, workspace=ws)
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
    small = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lce.LceError):
        lce.lce_forward_backward(H, W, t, IGNORE_INDEX, workspace=small)


# ------------------------------------------------ backward from a stored lse

@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_backward_from_stored_lse(dtype):
    """Forward keeps the per-row lse; a separate backward call recomputes the
    logits and produces dH and dW, scaled by a device-side upstream gradient."""
    base = "gpt1b" if dtype == "bf16" else "tiny"
    x = make_inputs(base, N=900, d=256, V=5000, padding=("random_frac", 0.25), seqs=1)
    H, W, t = to_device(x)
    loss, lse = lce.lce_forward(H, W, t, IGNORE_INDEX, return_lse=True)
    g = torch.tensor(2.5, device="cuda")
    dH, dW = lce.lce_backward(H, W, t, lse, IGNORE_INDEX, grad_loss=g)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
    assert rel_fro(np64(dH), 2.5 * ref["dH"]) <= TOL_REL
    assert rel_fro(np64(dW), 2.5 * ref["dW"]) <= TOL_REL
    # same as the fused call up to the rounding of the stored lse
    _, dH2, dW2 = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, grad_scale=2.5)
    assert rel_fro(np64(dW), np64(dW2)) <= 1e-4
    assert rel_fro(np64(dH), np64(dH2)) <= 1e-2      # dH is rounded to bf16 / exact fp32


def test_autograd_split_form():
    x = make_inputs("gpt1b", N=300, d=128, V=2100, padding=("random_frac", 0.1), seqs=1)
    H, W, t = to_device(x)
    H.requires_grad_(True)
    W.requires_grad_(True)
    loss = lce.linear_cross_entropy(H, W, t, IGNORE_INDEX)
    (3.0 * loss).backward()
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
    assert rel_fro(np64(H.grad), 3 * ref["dH"]) <= 1e-2
    assert rel_fro(np64(W.grad), 3 * ref["dW"]) <= 1e-2
    assert W.grad.dtype == torch.bfloat16


def test_autograd_bf16_W_grad_is_the_fp32_gradient_rounded_once():
    """W.grad of a bf16 W is written in bf16 by the library: each element the
    fp32 accumulator of the fp32-dW path rounded to nearest, bit for bit."""
    x = make_inputs("gpt1b", N=300, d=128, V=2100, padding=("random_frac", 0.1), seqs=1)
    H, W, t = to_device(x)
    W.requires_grad_(True)
    loss = lce.linear_cross_entropy(H, W, t, IGNORE_INDEX)
    loss.backward()
    _, lse = lce.lce_forward(H, W.detach(), t, IGNORE_INDEX, return_lse=True)
    _, dW32 = lce.lce_backward(H, W.detach(), t, lse, IGNORE_INDEX, grad_loss=torch.ones((), device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(W.grad.view(torch.int16), dW32.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("shape", [(1500, 512, 6000), (333, 72, 1000), (300, 64, 50257)],
                         ids=["gpt1b_small", "d72_ragged", "V50257"])
def test_bf16_dW_output_is_fp32_dW_rounded(shape):
    """dW_bf16: the dW tiles are staged and stored as bf16; every element equals
    the fp32 output rounded to nearest, loss and dH are bitwise those of the
    fp32-dW call, and the result is within the bf16 tolerance of the oracle."""
    N, d, V = shape
    x = make_inputs("gpt1b", N=N, d=d, V=V, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    l32, dH32, dW32 = lce.lce_forward_backward(H, W, t, IGNORE_INDEX)
    dW16 = torch.full(W.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    l16, dH16, dW16 = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, dW=dW16)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    assert dW16.dtype == torch.bfloat16
    assert torch.equal(l16, l32) and torch.equal(dH16.view(torch.int16), dH32.view(torch.int16))
    assert torch.equal(dW16.view(torch.int16), dW32.to(torch.bfloat16).view(torch.int16))
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert rel_fro(np64(dW16), ref["dW"]) <= TOL_REL


@pytest.mark.parametrize("kw", [dict(row_gather=True), dict(vocab_chunk=768), dict(vocab_chunk=256, row_gather=True)],
                         ids=["row_gather", "chunk768", "chunk256_gather"])
def test_bf16_dW_output_with_other_options(kw):
    """The bf16 dW output under row gather and other vocab chunks (a ragged
    last chunk): still the fp32 output of the same options rounded once."""
    x = make_inputs("gpt1b", N=700, d=256, V=2000, padding=("random_frac", 0.25), seqs=1)
    H, W, t = to_device(x)
    outs = []
    for dt in (torch.float32, torch.bfloat16):
        loss = torch.empty((), dtype=torch.float32, device="cuda")
        dH = torch.empty_like(H)
        dW = torch.full(W.shape, float("nan"), dtype=dt, device="cuda")
        lce.lce_run(H, W, t, IGNORE_INDEX, loss=loss, dH=dH, dW=dW, **kw)
        outs.append((loss, dH, dW))
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    (l32, dH32, dW32), (l16, dH16, dW16) = outs
    assert torch.equal(l16, l32) and torch.equal(dH16.view(torch.int16), dH32.view(torch.int16))
    assert torch.equal(dW16.view(torch.int16), dW32.to(torch.bfloat16).view(torch.int16))
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert rel_fro(np64(dW16), ref["dW"]) <= TOL_REL


def test_bf16_dW_refused_where_it_would_be_rounded_twice():
    x = make_inputs("gpt1b", N=200, d=64, V=900, padding=("random_frac", 0.1), seqs=1)
    H, W, t = to_device(x)
    dW16 = torch.zeros(W.shape, dtype=torch.bfloat16, device="cuda")
    for kw in (dict(accumulate_dW=True), dict(token_chunk=100)):
        with pytest.raises(RuntimeError) as e:
            lce.lce_forward_backward(H, W, t, IGNORE_INDEX, dW=dW16, **kw)
        assert e.value.code == 10                     # LCE_ERR_ARG
    with pytest.raises(RuntimeError) as e:
        lce.lce_forward_backward(H.float(), W.float(), t, IGNORE_INDEX, dW=dW16)
    assert e.value.code == 10


# ---------------------------------------------------------- token chunk cap

@pytest.mark.parametrize("token_chunk", [512, 1000])
def test_token_chunk_cap(token_chunk):
    """Rows processed token_chunk positions at a time: same loss and dH, dW
    summed across chunks in a fixed order, and scratch bounded by the cap."""
    x = make_inputs("gpt1b", N=2600, d=256, V=5000, padding=("random_frac", 0.3), seqs=1)
    H, W, t = to_device(x)
    loss_c, dH_c, dW_c, lse_c = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, token_chunk=token_chunk,
                                                         return_lse=True)
    loss, dH, dW, lse = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, return_lse=True)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss_c.item() - ref["loss"]) <= TOL_LOSS
    assert rel_fro(np64(dH_c), ref["dH"]) <= TOL_REL
    assert rel_fro(np64(dW_c), ref["dW"]) <= TOL_REL
    assert abs(loss_c.item() - loss.item()) <= 1e-6
    # the log-sum-exp merge order follows the number of row blocks per chunk,
    # so the chunked call agrees with the whole-batch one to rounding only
    valid = x.targets != IGNORE_INDEX
    np.testing.assert_allclose(np64(lse_c)[valid], np64(lse)[valid], rtol=0, atol=1e-5)
    assert rel_fro(np64(dH_c), np64(dH)) <= 1e-3
    assert rel_fro(np64(dW_c), np64(dW)) <= 1e-4
    assert lce.workspace_size(2600, 256, 5000, token_chunk=token_chunk) < lce.workspace_size(2600, 256, 5000)


def test_token_chunk_backward_from_stored_lse():
    x = make_inputs("gpt1b", N=1500, d=128, V=3000, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    loss, lse = lce.lce_forward(H, W, t, IGNORE_INDEX, return_lse=True)
    dH = torch.empty_like(H)
    dW = torch.empty(W.shape, dtype=torch.float32, device="cuda")
    lce.lce_run(H, W, t, IGNORE_INDEX, dH=dH, dW=dW, lse_in=lse, token_chunk=400)
    torch.cuda.synchronize()
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert rel_fro(np64(dH), ref["dH"]) <= TOL_REL
    assert rel_fro(np64(dW), ref["dW"]) <= TOL_REL


# ---------------------------------------------------------------- edge cases

def _oracle_check(H, W, t, x_H, x_W, targets, ignore_index=IGNORE_INDEX, **kw):
    loss, dH, dW = lce.lce_forward_backward(H, W, t, ignore_index, **kw)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    ref = oracle.forward_backward(x_H, x_W, targets, ignore_index)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS, (loss.item(), ref["loss"])
    assert rel_fro(np64(dH), ref["dH"]) <= TOL_REL
    assert rel_fro(np64(dW), ref["dW"]) <= TOL_REL
    return loss, dH, dW


def test_single_class_vocab():
    x = make_inputs("gpt1b", N=300, d=64, V=1, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    loss, dH, dW = lce.lce_forward_backward(H, W, t, IGNORE_INDEX)
    torch.cuda.synchronize()
    # exactly 0 in the definition; the kernel's log2-domain lse rounds to ~1 ulp
    assert abs(loss.item()) <= 1e-6
    assert dH.float().abs().max().item() <= 1e-6 and dW.abs().max().item() <= 1e-6


@pytest.mark.parametrize("d", [8, 24, 72])
def test_small_and_ragged_hidden_sizes(d):
    x = make_inputs("gpt1b", N=500, d=d, V=1300, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    _oracle_check(H, W, t, x.H_f32(), x.W_f32(), x.targets)


def test_single_token():
    for pad in (("none",), ("all",)):
        x = make_inputs("gpt1b", N=1, d=64, V=700, padding=pad, seqs=1)
        H, W, t = to_device(x)
        loss, dH, dW = lce.lce_forward_backward(H, W, t, IGNORE_INDEX)
        torch.cuda.synchronize()
        ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
        if pad[0] == "all":
            assert math.isnan(loss.item()) and torch.count_nonzero(dW).item() == 0
        else:
            assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
            assert rel_fro(np64(dW), ref["dW"]) <= TOL_REL


def test_extreme_logits_and_last_vocab_target():
    """Logit std ~30 (exp far outside fp32 without the running max) and
    targets on the last vocabulary row (the ragged last tile)."""
    x = make_inputs("gpt1b", N=400, d=128, V=2049, padding=("random_frac", 0.1), seqs=1, w_scale=30.0)
    x.targets[::7] = 2048
    H, W, t = to_device(x)
    loss, dH, dW = _oracle_check(H, W, t, x.H_f32(), x.W_f32(), x.targets)
    assert math.isfinite(loss.item())


def test_other_ignore_index():
    x = make_inputs("gpt1b", N=600, d=64, V=900, padding=("none",), seqs=1)
    x.targets[::3] = 0           # class 0 doubles as the padding marker here
    H, W, t = to_device(x)
    _oracle_check(H, W, t, x.H_f32(), x.W_f32(), x.targets, ignore_index=0)


def test_cuda_graph_capture_and_replay():
    """lce_run with a caller workspace enqueues kernels only (no host sync, no
    allocation), so a training step can capture it in a CUDA graph; replays
    reproduce the eager results bit for bit."""
    x = make_inputs("gpt1b", N=1024, d=256, V=5000, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    N, d = H.shape
    V = W.shape[0]
    ws = torch.empty(lce.workspace_size(N, d, V), dtype=torch.uint8, device="cuda")
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    dH = torch.empty_like(H)
    dW = torch.empty(W.shape, dtype=torch.float32, device="cuda")
    lce.lce_run(H, W, t, IGNORE_INDEX, loss=loss, dH=dH, dW=dW, workspace=ws)   # warm-up (device set-up)
    torch.cuda.synchronize()
    ref = (loss.clone(), dH.clone(), dW.clone())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lce.lce_run(H, W, t, IGNORE_INDEX, loss=loss, dH=dH, dW=dW, workspace=ws)
    for _ in range(2):
        loss.zero_()
        dH.zero_()
        dW.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(loss, ref[0])
        assert torch.equal(dH.view(torch.int16), ref[1].view(torch.int16))
        assert torch.equal(dW, ref[2])


def test_bounded_wait_times_out_into_the_status_word():
    """A pipeline wait that nothing completes gives up after its limit, raises
    LCE_DEV_TIMEOUT and returns; the context stays usable (a full call after
    it still matches the oracle)."""
    import ctypes
    from chunked_vocab_cross_gb300 import _abi
    lce.device_status()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = _abi.lib().lce_selftest_wait_timeout(2_000_000, ctypes.c_void_p(flag.data_ptr()),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert r == 0
    bits = lce.device_status()
    assert flag.item() == 1
    assert bits & 0x2
    assert lce.device_status() == 0      # reading clears the word
    x = make_inputs("gpt1b", N=300, d=128, V=1000, padding=("random_frac", 0.1), seqs=1)
    _run_and_compare(x)


@pytest.mark.parametrize("nv", [0, 1, 255, 256, 257, 511])
def test_row_gather_ragged_valid_counts(nv):
    """row_gather: the GEMMs gather H's valid rows by TMA gather4 through the
    compaction index (no compacted copy). Valid counts around the 256-row pair
    blocks, valid rows scattered over the batch; results equal to the oracle
    and bitwise equal to the default (copy) path."""
    import dataclasses
    x = make_inputs("gpt1b", N=700, d=256, V=1500, padding=("none",), seqs=1)
    g = np.random.default_rng(nv)
    t = np.full(700, IGNORE_INDEX, dtype=np.int64)
    pos = np.sort(g.choice(700, nv, replace=False))
    t[pos] = g.integers(0, 1500, nv)
    x = dataclasses.replace(x, targets=t)
    H, W, tt = to_device(x)
    outs = []
    for rg in (True, False):
        loss = torch.empty((), dtype=torch.float32, device="cuda")
        dH, dW = torch.empty_like(H), torch.empty(W.shape, dtype=torch.float32, device="cuda")
        lse = torch.empty(700, dtype=torch.float32, device="cuda")
        lce.lce_run(H, W, tt, IGNORE_INDEX, loss=loss, dH=dH, dW=dW, lse=lse, vocab_chunk=768, row_gather=rg)
        torch.cuda.synchronize()
        assert lce.device_status() == 0
        outs.append((loss, dH, dW))
    (loss, dH, dW), (loss_c, dH_c, dW_c) = outs
    assert torch.equal(dH, dH_c) and torch.equal(dW, dW_c)
    if nv == 0:
        assert math.isnan(loss.item()) and torch.count_nonzero(dH).item() == 0 and torch.count_nonzero(dW).item() == 0
        return
    assert torch.equal(loss, loss_c)
    ref = oracle.forward_backward(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
    assert rel_fro(np64(dH), ref["dH"]) <= TOL_REL and rel_fro(np64(dW), ref["dW"]) <= TOL_REL


def test_row_gather_gpt1b_shape_bitwise_equal_to_copy_path():
    """Full gpt1b shape: the gathered-row call gives the copy path's loss, dH
    and dW bit for bit (the same bf16 values reach the same MMAs)."""
    x = make_inputs("gpt1b")
    H, W, t = to_device(x)
    outs = []
    for rg in (True, False):
        loss = torch.empty((), dtype=torch.float32, device="cuda")
        dH, dW = torch.empty_like(H), torch.empty(W.shape, dtype=torch.float32, device="cuda")
        lce.lce_run(H, W, t, IGNORE_INDEX, loss=loss, dH=dH, dW=dW, row_gather=rg)
        torch.cuda.synchronize()
        assert lce.device_status() == 0
        outs.append((loss, dH, dW))
    for a_, b_ in zip(*outs):
        assert torch.equal(a_, b_)


@pytest.mark.parametrize("shape", [(300, 16384, 700), (3, 64, 300001), (131072, 64, 500)],
                         ids=["large_d", "large_V_tiny_N", "large_N"])
def test_extreme_shapes(shape):
    """Shapes at the edges of what the tiles handle: d = 16384 (256 k-blocks
    per logits tile, 64 d tiles in dW/dH), V = 300001 with 3 tokens (one row
    block against 1172 vocab tiles, a ragged last tile), and N = 131072 (512
    row blocks; 128 compaction rounds)."""
    N, d, V = shape
    x = make_inputs("gpt1b", N=N, d=d, V=V, padding=("random_frac", 0.2), seqs=1)
    _run_and_compare(x, vocab_chunk=4096 if V > 4096 else 0)


@pytest.mark.parametrize("shape", [(300, 64, 50257, ("random_frac", 0.2)), (200, 64, 262144 - 57, ("random_frac", 0.1)),
                                   (129, 64, 1000, ("none",))],
                         ids=["V50257", "V262087", "Nv129"])
def test_tail_shapes(shape):
    """Vocabulary sizes that are not multiples of the 256-wide tiles (GPT-2's
    50257 and 2^18 - 57) and a valid count one past a 128-row boundary."""
    N, d, V, pad = shape
    x = make_inputs("gpt1b", N=N, d=d, V=V, padding=pad, seqs=1)
    if pad == ("none",):
        assert int((x.targets != IGNORE_INDEX).sum()) == N
    _run_and_compare(x, vocab_chunk=4096)


@pytest.mark.parametrize("shape", [(100, 64, 50257), (300, 72, 1000)], ids=["V50257", "d72"])
def test_fp32_tail_shapes(shape):
    """The split-precision path on a GPT-2-sized ragged vocabulary and on a d
    that is not a multiple of 64 (per-block MN-major boxes)."""
    N, d, V = shape
    x = make_inputs("tiny", N=N, d=d, V=V, padding=("random_frac", 0.1))
    errs = _run_and_compare(x, vocab_chunk=4096)
    assert errs["loss"] <= 1e-4 and errs["dH"] <= 1e-3 and errs["dW"] <= 1e-3, errs
