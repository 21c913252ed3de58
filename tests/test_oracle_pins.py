"""Pins for the fp64 oracles against facts fixed by the definition and by
mathematics, not by the oracles themselves: closed forms, a hand-derived worked
example, central finite differences, an independent library autograd, and
invariants. Each is chosen so that a plausible slip in an oracle (a dropped
-onehot term, the wrong normaliser, a transposed operand, a wrong index or sign)
fails at least one of them.

The loss-path pins run against both implementations of the definition: the
plain C++ one (oracle/lce_oracle.cpp, loops and std::thread) and the numpy one
(oracle/lce_oracle.py, library matmuls), through the ``lo`` fixture."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import cpp_oracle
from synth_inputs import IGNORE_INDEX

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(params=["cpp", "numpy"])
def lo(request):
    """The loss-path oracle under test: the C++ one or the numpy one."""
    return cpp_oracle if request.param == "cpp" else oracle


def _rand(N, d, V, seed=0, pad=0.25, scale=1.0):
    g = np.random.default_rng(seed)
    H = g.standard_normal((N, d))
    W = g.standard_normal((V, d)) * scale
    t = g.integers(0, V, N)
    t[g.random(N) < pad] = IGNORE_INDEX
    return H, W, t


# ---------------------------------------------------------------- closed forms

def test_zero_W_gives_ln_V_and_closed_form_dW(lo):
    H, _, t = _rand(37, 5, 11, seed=1)
    W = np.zeros((11, 5))
    r = lo.forward_backward(H, W, t)
    valid = t != IGNORE_INDEX
    nv = valid.sum()
    assert r["loss"] == pytest.approx(math.log(11), abs=1e-14)
    # every logit is 0, p = 1/V: dW_v = (1/(V Nv)) sum_i H_i - (1/Nv) sum_{i: t_i = v} H_i
    expect = np.tile(H[valid].sum(0) / (11 * nv), (11, 1))
    for i in np.nonzero(valid)[0]:
        expect[t[i]] -= H[i] / nv
    np.testing.assert_allclose(r["dW"], expect, atol=1e-14)
    np.testing.assert_array_equal(r["dH"], 0.0)


def test_zero_H_gives_ln_V_and_closed_form_dH(lo):
    _, W, t = _rand(29, 4, 7, seed=2)
    H = np.zeros((29, 4))
    r = lo.forward_backward(H, W, t)
    valid = t != IGNORE_INDEX
    nv = valid.sum()
    assert r["loss"] == pytest.approx(math.log(7), abs=1e-14)
    expect = np.zeros_like(H)
    for i in np.nonzero(valid)[0]:
        expect[i] = (W.mean(0) - W[t[i]]) / nv
    np.testing.assert_allclose(r["dH"], expect, atol=1e-14)
    np.testing.assert_array_equal(r["dW"], 0.0)


def test_single_class_gives_zero(lo):
    H, W, _ = _rand(9, 3, 1, seed=3)
    t = np.array([0, 0, IGNORE_INDEX, 0, 0, 0, IGNORE_INDEX, 0, 0])
    r = lo.forward_backward(H, W, t)
    assert r["loss"] == 0.0
    np.testing.assert_array_equal(r["dH"], 0.0)
    np.testing.assert_array_equal(r["dW"], 0.0)


def test_two_class_softplus_closed_form(lo):
    # d = 1, V = 2: loss_i = softplus(s_other - s_target), a logistic loss
    g = np.random.default_rng(4)
    N = 13
    H = g.standard_normal((N, 1))
    W = np.array([[0.7], [-1.3]])
    t = g.integers(0, 2, N)
    t[[2, 5]] = IGNORE_INDEX
    r = lo.forward_backward(H, W, t)
    valid = np.nonzero(t != IGNORE_INDEX)[0]
    nv = len(valid)
    loss = 0.0
    dH = np.zeros((N, 1))
    dW = np.zeros((2, 1))
    for i in valid:
        h = H[i, 0]
        o = 1 - t[i]
        delta = h * (W[o, 0] - W[t[i], 0])
        loss += math.log1p(math.exp(delta))
        sig = 1.0 / (1.0 + math.exp(-delta))          # d softplus / d delta
        dH[i, 0] = sig * (W[o, 0] - W[t[i], 0]) / nv
        dW[o, 0] += sig * h / nv
        dW[t[i], 0] -= sig * h / nv
    assert r["loss"] == pytest.approx(loss / nv, rel=1e-14)
    np.testing.assert_allclose(r["dH"], dH, rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(r["dW"], dW, rtol=1e-13, atol=1e-16)


def test_hand_derived_worked_example(lo):
    with open(os.path.join(GOLDEN, "worked_example_3x3.json")) as f:
        ex = json.load(f)
    ln2, ln3 = math.log(2), math.log(3)
    H = np.array(ex["H"], dtype=float)
    W = np.array([[0, 0], [ln2, 0], [0, ln3]])
    t = np.array(ex["targets"])
    r = lo.forward_backward(H, W, t, ex["ignore_index"])
    assert r["loss"] == pytest.approx(math.log(20) / 3, rel=1e-15)
    np.testing.assert_allclose(np.exp(r["lse"]), [4, 5, 6], rtol=1e-15)
    dH = np.array([[-ln2 / 2, ln3 / 4], [ln2 / 5, 3 * ln3 / 5], [ln2 / 3, -ln3 / 2], [0, 0]]) / 3
    np.testing.assert_allclose(r["dH"], dH, rtol=1e-14, atol=1e-16)
    dW = np.array([[1 / 4 + 1 / 6, -4 / 5 + 1 / 6],
                   [-1 / 2 + 1 / 3, 1 / 5 + 1 / 3],
                   [1 / 4 - 1 / 2, 3 / 5 - 1 / 2]]) / 3
    np.testing.assert_allclose(r["dW"], dW, rtol=1e-14, atol=1e-16)
    assert np.all(r["dH"][3] == 0.0)


def test_no_valid_rows_gives_nan_loss_and_zero_grads(lo):
    H, W, _ = _rand(6, 3, 4, seed=5)
    t = np.full(6, IGNORE_INDEX)
    r = lo.forward_backward(H, W, t)
    assert math.isnan(r["loss"])
    np.testing.assert_array_equal(r["dH"], 0.0)
    np.testing.assert_array_equal(r["dW"], 0.0)
    assert r["n_valid"] == 0


# ---------------------------------------------------------- finite differences

def _loss_only(lo, H, W, t):
    return lo.forward(H, W, t)["loss"]


def test_central_finite_differences(lo):
    H, W, t = _rand(4, 3, 5, seed=6, pad=0.0)
    t[1] = IGNORE_INDEX
    r = lo.forward_backward(H, W, t)
    eps = 1e-6
    for A, grad in ((H, r["dH"]), (W, r["dW"])):
        num = np.zeros_like(A)
        for idx in np.ndindex(A.shape):
            old = A[idx]
            A[idx] = old + eps
            lp = _loss_only(lo, H, W, t)
            A[idx] = old - eps
            lm = _loss_only(lo, H, W, t)
            A[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, atol=2e-9)


# --------------------------------------------------- independent library check

@pytest.mark.parametrize("shape", [(1, 1, 2), (7, 3, 5), (64, 16, 33), (200, 24, 300)])
def test_torch_float64_autograd(lo, shape):
    torch = pytest.importorskip("torch")
    N, d, V = shape
    H, W, t = _rand(N, d, V, seed=N + d + V, scale=2.0)
    if N > 1:
        t[0] = IGNORE_INDEX
    r = lo.forward_backward(H, W, t)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(t), ignore_index=IGNORE_INDEX)
    loss.backward()
    assert r["loss"] == pytest.approx(loss.item(), rel=1e-12)
    np.testing.assert_allclose(r["dH"], Ht.grad.numpy(), rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(r["dW"], Wt.grad.numpy(), rtol=1e-10, atol=1e-15)


def test_torch_float64_autograd_tiny_workload(lo):
    torch = pytest.importorskip("torch")
    from synth_inputs import make_inputs
    x = make_inputs("tiny")
    H, W = x.H.astype(np.float64), x.W.astype(np.float64)
    r = lo.forward_backward(H, W, x.targets)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(x.targets), ignore_index=IGNORE_INDEX)
    loss.backward()
    assert r["n_valid"] == 230
    assert r["loss"] == pytest.approx(loss.item(), rel=1e-12)
    np.testing.assert_allclose(r["dH"], Ht.grad.numpy(), rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(r["dW"], Wt.grad.numpy(), rtol=1e-9, atol=1e-15)


# ------------------------------------------------------------------ invariants

def test_columns_of_dW_sum_to_zero(lo):
    H, W, t = _rand(50, 6, 17, seed=7, scale=3.0)
    r = lo.forward_backward(H, W, t)
    np.testing.assert_allclose(r["dW"].sum(0), 0.0, atol=1e-15)


def test_common_shift_of_vocab_rows_changes_nothing(lo):
    H, W, t = _rand(40, 5, 9, seed=8)
    c = np.random.default_rng(9).standard_normal(5)
    a = lo.forward_backward(H, W, t)
    b = lo.forward_backward(H, W + c[None, :], t)
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-12)
    np.testing.assert_allclose(a["dH"], b["dH"], atol=1e-14)
    np.testing.assert_allclose(a["dW"], b["dW"], atol=1e-14)


def test_token_permutation(lo):
    H, W, t = _rand(31, 4, 10, seed=10)
    p = np.random.default_rng(11).permutation(31)
    a = lo.forward_backward(H, W, t)
    b = lo.forward_backward(H[p], W, t[p])
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-13)
    np.testing.assert_allclose(a["dH"][p], b["dH"], atol=1e-15)
    np.testing.assert_allclose(a["dW"], b["dW"], atol=1e-15)


def test_padded_rows_are_exact_zero_and_removable(lo):
    H, W, t = _rand(30, 4, 8, seed=12, pad=0.4)
    a = lo.forward_backward(H, W, t)
    pad = t == IGNORE_INDEX
    assert pad.any()
    assert np.all(a["dH"][pad] == 0.0)
    b = lo.forward_backward(H[~pad], W, t[~pad])
    assert a["loss"] == pytest.approx(b["loss"], rel=1e-14)
    np.testing.assert_allclose(a["dH"][~pad], b["dH"], atol=1e-16)
    np.testing.assert_allclose(a["dW"], b["dW"], atol=1e-16)
    # padded rows' H values must not matter at all
    H2 = H.copy()
    H2[pad] = 1e6
    c = lo.forward_backward(H2, W, t)
    np.testing.assert_array_equal(a["dW"], c["dW"])


def test_normaliser_is_valid_count_not_N(lo):
    H, W, t = _rand(20, 3, 6, seed=13, pad=0.0)
    t[:10] = IGNORE_INDEX
    r = lo.forward_backward(H, W, t)
    assert r["loss"] == pytest.approx(r["loss_rows"].mean(), rel=1e-14)
    assert r["n_valid"] == 10


# --------------------------------------------------------------- compaction

def test_compaction_golden_cases(lo):
    with open(os.path.join(GOLDEN, "compaction_small.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        t = np.array(c["targets"], dtype=np.int64)
        assert lo.valid_rows(t, c["ignore_index"]).tolist() == c["valid"]
        # the numpy oracle counts out-of-range targets; the C++ one refuses them
        assert oracle.out_of_range_targets(t, c["ignore_index"], c["V"]) == c["out_of_range"]
        if c["out_of_range"]:
            with pytest.raises(ValueError):
                cpp_oracle.valid_rows(t, c["ignore_index"], c["V"])
        else:
            assert cpp_oracle.valid_rows(t, c["ignore_index"], c["V"]).tolist() == c["valid"]


def test_compaction_brute_force(lo):
    g = np.random.default_rng(14)
    for n in (0, 1, 31, 32, 33, 1000, 4097):
        t = g.integers(-3, 5, n)
        t[g.random(n) < 0.3] = IGNORE_INDEX
        expect = [i for i in range(n) if t[i] != IGNORE_INDEX]
        assert lo.valid_rows(t, IGNORE_INDEX).tolist() == expect


def test_out_of_range_target_is_refused(lo):
    H, W, t = _rand(5, 2, 3, seed=15, pad=0.0)
    t[2] = 3
    with pytest.raises(ValueError):
        lo.forward_backward(H, W, t)


# ------------------------------------------------------- sampled reference

def test_sampled_reference_matches_full(lo):
    H, W, t = _rand(300, 8, 70, seed=16, scale=2.0)
    full = lo.forward_backward(H, W, t)
    rows = np.array([0, 5, 17, 299, 123])
    vocab = np.array([0, 69, 33, 1])
    s = lo.sampled_reference(H, W, t, IGNORE_INDEX, rows, vocab)
    assert s["loss"] == pytest.approx(full["loss"], rel=1e-13)
    np.testing.assert_allclose(s["dH_rows"], full["dH"][rows], atol=1e-15)
    np.testing.assert_allclose(s["dW_rows"], full["dW"][vocab], atol=1e-15)


# ------------------------------------------------ fused optimizer step (oracle)

def _torch_steps(kind, w0, grads, **hp):
    torch = pytest.importorskip("torch")
    p = torch.nn.Parameter(torch.tensor(w0, dtype=torch.float64))
    if kind == "sgd":
        opt = torch.optim.SGD([p], lr=hp["lr"], momentum=hp.get("momentum", 0.0),
                              weight_decay=hp.get("weight_decay", 0.0))
    else:
        opt = torch.optim.AdamW([p], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                                weight_decay=hp.get("weight_decay", 0.0))
    for g in grads:
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
    st = opt.state[p]
    m = st.get("momentum_buffer", st.get("exp_avg"))
    v = st.get("exp_avg_sq")
    return (p.detach().numpy(), None if m is None else m.numpy(), None if v is None else v.numpy())


def _oracle_steps(kind, w0, grads, **hp):
    w, m, v = np.array(w0), None, None
    for t, g in enumerate(grads, start=1):
        r = oracle.optimizer_step(kind, w, g, step=t, exp_avg=m, exp_avg_sq=v, **hp)
        w, m, v = r["w"], r["exp_avg"], r["exp_avg_sq"]
    return w, m, v


@pytest.mark.parametrize("kind,hp", [
    ("sgd", dict(lr=0.1)),
    ("sgd", dict(lr=0.05, momentum=0.9, weight_decay=0.01)),
    ("adamw", dict(lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8)),
    ("adamw", dict(lr=1e-2, beta1=0.8, beta2=0.95, eps=1e-6, weight_decay=0.1)),
])
def test_optimizer_step_matches_torch_optim(kind, hp):
    g = np.random.default_rng(7)
    w0 = g.standard_normal((6, 5))
    grads = [g.standard_normal((6, 5)) * s for s in (1.0, 0.3, 2.0, 0.01)]
    ow, om, ov = _oracle_steps(kind, w0, grads, **hp)
    tw, tm, tv = _torch_steps(kind, w0, grads, **hp)
    np.testing.assert_allclose(ow, tw, rtol=1e-13, atol=1e-15)
    if tm is not None:
        np.testing.assert_allclose(om, tm, rtol=1e-13, atol=1e-15)
    if tv is not None:
        np.testing.assert_allclose(ov, tv, rtol=1e-13, atol=1e-18)


def test_adamw_first_step_closed_form():
    # t = 1: m_hat = g, v_hat = g^2, so w moves by lr * g / (|g| + eps)
    g = np.array([[3.0, -0.5, 1e-9, 0.0]])
    w = np.array([[1.0, 2.0, -3.0, 4.0]])
    r = oracle.optimizer_step("adamw", w, g, lr=0.01, step=1, beta1=0.9, beta2=0.99, eps=1e-8)
    np.testing.assert_allclose(r["w"], w - 0.01 * g / (np.abs(g) + 1e-8), rtol=1e-14, atol=0)


def test_bf16_state_rounding_matches_torch_and_leaves_w_unchanged():
    """State kept in bf16: the returned state is the fp32-state step's state
    rounded to the nearest bf16 as torch converts it, and w is the fp32-state
    step's w (the update uses the unrounded values)."""
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(21)
    w0 = g.standard_normal((5, 7))
    grads = g.standard_normal((5, 7)) * 0.3
    for kind, hp in (("adamw", dict(lr=1e-2, beta1=0.9, beta2=0.99, eps=1e-6, weight_decay=0.1)),
                     ("sgd", dict(lr=0.05, momentum=0.9, weight_decay=0.01))):
        m0 = torch.tensor(g.standard_normal((5, 7))).to(torch.bfloat16).double().numpy()
        v0 = torch.tensor(g.uniform(0.1, 1.0, (5, 7))).to(torch.bfloat16).double().numpy()
        a = oracle.optimizer_step(kind, w0, grads, step=3, exp_avg=m0, exp_avg_sq=v0 if kind == "adamw" else None,
                                  **hp)
        b = oracle.optimizer_step(kind, w0, grads, step=3, exp_avg=m0, exp_avg_sq=v0 if kind == "adamw" else None,
                                  state_bf16=True, **hp)
        np.testing.assert_array_equal(a["w"], b["w"])
        for k in ("exp_avg", "exp_avg_sq"):
            if a[k] is None:
                continue
            ref = torch.tensor(a[k]).float().to(torch.bfloat16).double().numpy()
            np.testing.assert_array_equal(b[k], ref)


def test_zero_gradient_without_decay_only_decays_the_moments():
    g0 = np.zeros((3, 4))
    w = np.arange(12.0).reshape(3, 4)
    m = np.full((3, 4), 2.0)
    v = np.full((3, 4), 4.0)
    r = oracle.optimizer_step("adamw", w, g0, lr=0.1, step=5, beta1=0.9, beta2=0.99, eps=1e-8,
                              exp_avg=m, exp_avg_sq=v)
    np.testing.assert_allclose(r["exp_avg"], 0.9 * m)
    np.testing.assert_allclose(r["exp_avg_sq"], 0.99 * v)
    s = oracle.optimizer_step("sgd", w, g0, lr=0.1, step=3)
    np.testing.assert_array_equal(s["w"], w)


# ------------------------------------ input-embedding lookup skipping padding

def _emb_case(seed=3, N=57, d=6, V=13, pad=0):
    g = np.random.default_rng(seed)
    W = g.standard_normal((V, d))
    t = g.integers(0, V, N)
    t[g.random(N) < 0.3] = pad
    dE = g.standard_normal((N, d))
    return W, t, dE


def test_embedding_matches_torch_autograd_of_masked_lookup():
    torch = pytest.importorskip("torch")
    W, t, dE = _emb_case()
    pad = 0
    Wt = torch.tensor(W, requires_grad=True)
    mask = torch.tensor(t != pad, dtype=torch.float64)[:, None]
    E = torch.nn.functional.embedding(torch.tensor(t), Wt) * mask
    (E * torch.tensor(dE)).sum().backward()
    np.testing.assert_allclose(oracle.embedding_forward(W, t, pad), E.detach().numpy(), rtol=0, atol=0)
    np.testing.assert_allclose(oracle.embedding_backward(dE, t, pad, W.shape[0]), Wt.grad.numpy(),
                               rtol=1e-14, atol=1e-14)


def test_embedding_invariants():
    W, t, dE = _emb_case(seed=5, pad=2)
    pad, V = 2, W.shape[0]
    valid = t != pad
    E = oracle.embedding_forward(W, t, pad)
    assert np.all(E[~valid] == 0.0) and np.array_equal(E[valid], W[t[valid]])
    dW = oracle.embedding_backward(dE, t, pad, V)
    np.testing.assert_allclose(dW.sum(0), dE[valid].sum(0), rtol=1e-12, atol=1e-12)
    untouched = np.setdiff1d(np.arange(V), t[valid])
    assert np.all(dW[untouched] == 0.0)
    assert np.all(dW[pad] == 0.0)          # the padding id never receives a gradient
    perm = np.random.default_rng(0).permutation(len(t))
    np.testing.assert_allclose(oracle.embedding_backward(dE[perm], t[perm], pad, V), dW, rtol=1e-13, atol=1e-13)


def test_embedding_refuses_out_of_range_tokens():
    W, t, dE = _emb_case()
    t = t.copy()
    t[4] = W.shape[0]
    with pytest.raises(ValueError):
        oracle.embedding_forward(W, t, 0)
    with pytest.raises(ValueError):
        oracle.embedding_backward(dE, t, 0, W.shape[0])
