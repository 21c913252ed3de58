"""Parity of the fused optimizer step (SGD / AdamW applied to W inside the
backward, no dW buffer) with the fp64 oracle: the oracle's gradient of W fed
to the oracle's optimizer step, both computed from the same seeded inputs.

Tolerances. The update is compared as a step (W_new - W_old) by relative
Frobenius error. The gradient it is built from carries the bf16 path's
5e-3 bound (3e-3 for the fp32 path's dW, plus its rounding), and the cases
are chosen so that the step is a smooth function of the gradient, which then
passes that bound through: AdamW with eps well above |g| (so the step is
nearly linear in g) or with beta1 = 0 and seeded second moments; SGD is linear
in g. A bf16 W updated in place is rounded to nearest once more, at most
2^-8 |w| per element, which is added to the bound."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import chunked_vocab_cross_gb300 as lce  # noqa: E402
import oracle  # noqa: E402
from lce_testutil import TOL_LOSS, TOL_REL, np64, rel_fro, to_device  # noqa: E402
from synth_inputs import IGNORE_INDEX, bf16_bits_to_f32, f32_to_bf16_bits, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from chunked_vocab_cross_gb300.build import build
    build()
    lce.device_status()
    yield


def _bf16_round(a):
    """Nearest bf16 of each value (through fp32, as the library rounds its fp32 master)."""
    return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(a, dtype=np.float32))).astype(np.float64)


def _f32(x):
    """A hyperparameter as the library receives it (fp32 in the C ABI)."""
    return float(np.float32(x))


def _step(kind, w, g, **hp):
    """The oracle's optimizer step on the fp32 values of the hyperparameters."""
    for k in ("lr", "weight_decay", "momentum", "beta1", "beta2", "eps"):
        if k in hp:
            hp[k] = _f32(hp[k])
    if kind == "adamw":
        hp.setdefault("beta1", _f32(0.9))
        hp.setdefault("beta2", _f32(0.999))
        hp.setdefault("eps", _f32(1e-8))
    return oracle.optimizer_step(kind, w, g, **hp)


def _oracle_grad(H, W, t):
    return oracle.forward_backward(H, W, t, IGNORE_INDEX)


def test_adamw_master_weights_three_steps_bf16():
    """AdamW on a bf16 W with fp32 master weights, three steps with fresh H
    each step; ragged V (several vocab chunks) and d not a multiple of 64."""
    x = make_inputs("gpt1b", N=1100, d=200, V=5000, padding=("random_frac", 0.3), seqs=1)
    H0, W, t = to_device(x)
    opt = lce.FusedOptimizer(W, "adamw", lr=1e-2, betas=(0.9, 0.99), weight_decay=0.1, master_weights=True)
    w_or = x.W_f32().astype(np.float64)             # the oracle's own master trajectory
    m_or = v_or = None
    rng = np.random.default_rng(3)
    for step in (1, 2, 3):
        Hs = x.H_f32() if step == 1 else _bf16_round(rng.standard_normal(x.H_f32().shape))
        Hd = H0 if step == 1 else torch.from_numpy(Hs.astype(np.float32)).to("cuda").to(torch.bfloat16)
        ref = _oracle_grad(Hs, _bf16_round(w_or), x.targets)   # forward on the bf16 copy of the master
        eps = 10.0 * float(np.max(np.abs(ref["dW"])))          # step nearly linear in g
        opt.eps = eps
        master_old = np64(opt.master)
        loss, dH = opt.step(Hd, t, IGNORE_INDEX, vocab_chunk=1024)
        torch.cuda.synchronize()
        assert lce.device_status() == 0
        o = _step("adamw", w_or, ref["dW"], lr=1e-2, step=step, weight_decay=0.1, beta1=0.9,
                                  beta2=0.99, eps=eps, exp_avg=m_or, exp_avg_sq=v_or)
        errs = {"loss": abs(loss.item() - ref["loss"]), "dH": rel_fro(np64(dH), ref["dH"]),
                "step": rel_fro(np64(opt.master) - master_old, o["w"] - w_or),
                "m": rel_fro(np64(opt.exp_avg), o["exp_avg"]), "v": rel_fro(np64(opt.exp_avg_sq), o["exp_avg_sq"])}
        print(step, errs)
        assert errs["loss"] <= TOL_LOSS and errs["dH"] <= TOL_REL, errs
        assert errs["step"] <= TOL_REL and errs["m"] <= TOL_REL and errs["v"] <= 2 * TOL_REL, errs
        # W is the bf16 rounding of the master, bit for bit
        assert torch.equal(W, opt.master.to(torch.bfloat16))
        w_or, m_or, v_or = o["w"], o["exp_avg"], o["exp_avg_sq"]


def test_adamw_in_place_bf16_seeded_moments():
    """AdamW on a bf16 W in place (no master), beta1 = 0 and seeded moments at
    step 5, so the step is linear in the gradient and the bias corrections of
    both moments matter."""
    x = make_inputs("gpt1b", N=900, d=256, V=3000, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    ref = _oracle_grad(x.H_f32(), x.W_f32(), x.targets)
    g_rms = float(np.sqrt(np.mean(ref["dW"] ** 2)))
    rng = np.random.default_rng(11)
    m0 = (rng.standard_normal(ref["dW"].shape) * g_rms).astype(np.float32)
    v0 = (g_rms ** 2 * rng.uniform(0.5, 2.0, ref["dW"].shape)).astype(np.float32)
    opt = lce.FusedOptimizer(W, "adamw", lr=0.05, betas=(0.0, 0.9), eps=1e-12)
    opt.exp_avg.copy_(torch.from_numpy(m0))
    opt.exp_avg_sq.copy_(torch.from_numpy(v0))
    opt.step_count = 4
    w_old = np64(W)
    loss, dH = opt.step(H, t, IGNORE_INDEX, vocab_chunk=1024)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    o = _step("adamw", x.W_f32(), ref["dW"], lr=0.05, step=5, beta1=0.0, beta2=0.9, eps=1e-12,
                              exp_avg=m0, exp_avg_sq=v0)
    w_new = np64(W)
    tol = TOL_REL + 2.0 ** -8 * np.linalg.norm(w_new) / np.linalg.norm(o["w"] - w_old)
    errs = {"step": rel_fro(w_new - w_old, o["w"] - w_old), "tol": tol,
            "m": rel_fro(np64(opt.exp_avg), o["exp_avg"]), "v": rel_fro(np64(opt.exp_avg_sq), o["exp_avg_sq"])}
    print(errs)
    assert abs(loss.item() - ref["loss"]) <= TOL_LOSS
    assert errs["step"] <= tol and errs["m"] <= TOL_REL and errs["v"] <= TOL_REL, errs


def test_sgd_momentum_fp32_two_steps():
    """SGD with momentum and weight decay on an fp32 W (split-precision path),
    updated in place: step 1 starts the momentum buffer, step 2 runs the
    recurrence on the oracle's own updated weights."""
    x = make_inputs("tiny", N=700, d=96, V=2100, seqs=1)
    assert not x.bf16
    H, W, t = to_device(x)
    opt = lce.FusedOptimizer(W, "sgd", lr=2.0, momentum=0.9, weight_decay=0.01)
    w_or, m_or = x.W_f32().astype(np.float64), None
    for step in (1, 2):
        ref = _oracle_grad(x.H_f32(), w_or, x.targets)
        w_old = np64(W)
        loss, dH = opt.step(H, t, IGNORE_INDEX, vocab_chunk=512)
        torch.cuda.synchronize()
        assert lce.device_status() == 0
        o = _step("sgd", w_or, ref["dW"], lr=2.0, step=step, momentum=0.9, weight_decay=0.01,
                                  exp_avg=m_or)
        errs = {"loss": abs(loss.item() - ref["loss"]), "step": rel_fro(np64(W) - w_old, o["w"] - w_or),
                "buf": rel_fro(np64(opt.exp_avg), o["exp_avg"])}
        print(step, errs)
        assert errs["loss"] <= 1e-4 and errs["step"] <= 3e-3 and errs["buf"] <= 3e-3, errs
        w_or, m_or = o["w"], o["exp_avg"]


def test_optimizer_leaves_loss_and_dH_bitwise_unchanged():
    """loss and dH are those of the old W, bit for bit the same as a call
    without the optimizer (the update of a W row follows its last read)."""
    x = make_inputs("gpt1b", N=1500, d=512, V=7000, padding=("random_frac", 0.25), seqs=1)
    H, W, t = to_device(x)
    loss0, dH0, _ = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, vocab_chunk=1536)
    for algo, kw in (("sgd", dict(lr=0.5)), ("adamw", dict(lr=1e-3))):
        Wc = W.clone()
        opt = lce.FusedOptimizer(Wc, algo, **kw)
        loss1, dH1 = opt.step(H, t, IGNORE_INDEX, vocab_chunk=1536)
        torch.cuda.synchronize()
        assert lce.device_status() == 0
        assert torch.equal(loss0, loss1) and torch.equal(dH0, dH1), algo
        assert not torch.equal(Wc, W), algo


def test_sgd_matches_the_unfused_gradient_step():
    """Plain SGD fused into the backward equals W - lr * dW formed from the
    library's own dW output, computed in fp32 and rounded once (the same
    tiles produce the same gradient values in both calls)."""
    x = make_inputs("gpt1b", N=1000, d=320, V=4500, padding=("random_frac", 0.3), seqs=1)
    H, W, t = to_device(x)
    _, _, dW = lce.lce_forward_backward(H, W, t, IGNORE_INDEX, vocab_chunk=1024)
    expect = (W.float() - 0.25 * dW).to(torch.bfloat16)
    opt = lce.FusedOptimizer(W, "sgd", lr=0.25)
    opt.step(H, t, IGNORE_INDEX, vocab_chunk=1024)
    torch.cuda.synchronize()
    assert torch.equal(W, expect)


def test_backward_from_stored_lse_with_optimizer():
    """The backward-only call (stored lse) with a fused AdamW step agrees with
    the oracle."""
    x = make_inputs("gpt1b", N=800, d=256, V=4000, padding=("random_frac", 0.3), seqs=1)
    H, W, t = to_device(x)
    _, lse = lce.lce_forward(H, W, t, IGNORE_INDEX, return_lse=True)
    ref = _oracle_grad(x.H_f32(), x.W_f32(), x.targets)
    eps = 10.0 * float(np.max(np.abs(ref["dW"])))
    opt = lce.FusedOptimizer(W, "adamw", lr=1e-2, eps=eps, master_weights=True)
    master_old = np64(opt.master)
    loss, dH = opt.step(H, t, IGNORE_INDEX, lse_in=lse)
    torch.cuda.synchronize()
    assert loss is None and lce.device_status() == 0
    o = _step("adamw", x.W_f32(), ref["dW"], lr=1e-2, step=1, eps=eps)
    assert rel_fro(np64(dH), ref["dH"]) <= TOL_REL
    assert rel_fro(np64(opt.master) - master_old, o["w"] - x.W_f32()) <= TOL_REL


def test_all_ignored_tokens_apply_a_zero_gradient():
    """Nv = 0: the gradient is zero, so AdamW only decays the moments and the
    weights (decoupled weight decay); loss is NaN and dH zero."""
    x = make_inputs("gpt1b", N=300, d=128, V=1000, seqs=1)
    H, W, _ = to_device(x)
    t = torch.full((300,), IGNORE_INDEX, dtype=torch.int64, device="cuda")
    opt = lce.FusedOptimizer(W, "adamw", lr=0.1, weight_decay=0.5, master_weights=True)
    opt.exp_avg.fill_(1e-3)
    opt.exp_avg_sq.fill_(4e-6)
    opt.step_count = 9
    master_old = np64(opt.master)
    loss, dH = opt.step(H, t, IGNORE_INDEX)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    assert np.isnan(loss.item()) and torch.count_nonzero(dH).item() == 0
    o = _step("adamw", master_old, np.zeros_like(master_old), lr=0.1, step=10, weight_decay=0.5,
                              exp_avg=np.full(master_old.shape, 1e-3, np.float32),
                              exp_avg_sq=np.full(master_old.shape, 4e-6, np.float32))
    np.testing.assert_allclose(np64(opt.master), o["w"], rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(np64(opt.exp_avg), o["exp_avg"], rtol=1e-6)
    np.testing.assert_allclose(np64(opt.exp_avg_sq), o["exp_avg_sq"], rtol=1e-6)


def test_fused_optimizer_sampled_rows_gpt1b():
    """Full gpt1b shape (N=4096, d=2048, V=50304) with the default vocab chunk:
    one AdamW step (eps well above |g|), checked on 256 seeded vocab rows
    against the oracle's gradient of those rows."""
    x = make_inputs("gpt1b")
    H, W, t = to_device(x)
    rows = np.sort(np.random.default_rng(5).choice(x.W.shape[0], 256, replace=False))
    ref = oracle.sampled_reference(x.H_f32(), x.W_f32(), x.targets, IGNORE_INDEX,
                                   token_rows=np.array([], dtype=np.int64), vocab_rows=rows)
    gW = ref["dW_rows"]
    eps = 10.0 * float(np.max(np.abs(gW)))
    opt = lce.FusedOptimizer(W, "adamw", lr=1e-2, eps=eps, weight_decay=0.1, master_weights=True)
    master_old = np64(opt.master[torch.from_numpy(rows).cuda()])
    loss, _ = opt.step(H, t, IGNORE_INDEX)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    o = _step("adamw", x.W_f32()[rows], gW, lr=1e-2, step=1, weight_decay=0.1, eps=eps)
    got = np64(opt.master[torch.from_numpy(rows).cuda()])
    err = rel_fro(got - master_old, o["w"] - x.W_f32()[rows])
    print("sampled step err", err)
    assert err <= TOL_REL


@pytest.mark.parametrize("case", [
    ("adamw", "fp32", False, 0.0),   # fp32 W in place: 8 KB ring buffers, fp32 weight boxes
    ("sgd", "fp32", False, 0.0),     # fp32 W, no state: weight boxes only
    ("sgd", "bf16", False, 0.9),     # bf16 W in place with a momentum buffer
    ("sgd", "bf16", True, 0.5),      # fp32 master weights with a momentum buffer
], ids=lambda c: f"{c[0]}_{c[1]}_{'master' if c[2] else 'inplace'}_m{c[3]}")
def test_optimizer_state_layouts(case):
    """Every combination of weights and state the optimizer ring moves (boxes
    of m, v, fp32 or bf16 weights, bf16 rounding of a master copy), on a
    ragged V, two steps, against the oracle's own trajectory."""
    kind, dt, master, momentum = case
    base = "tiny" if dt == "fp32" else "gpt1b"
    x = make_inputs(base, N=640, d=136, V=2333, padding=("random_frac", 0.2), seqs=1)
    assert x.bf16 == (dt == "bf16")
    H, W, t = to_device(x)
    # a bf16 W updated in place keeps the update above its rounding (2^-8 |w|)
    lr = (50.0 if (dt == "bf16" and not master) else 0.5) if kind == "sgd" else 1e-2
    hp = dict(lr=lr, weight_decay=0.01)
    if kind == "sgd":
        opt = lce.FusedOptimizer(W, "sgd", momentum=momentum, master_weights=master, **hp)
    else:
        opt = lce.FusedOptimizer(W, "adamw", master_weights=master, **hp)
    w_or = x.W_f32().astype(np.float64)
    m_or = v_or = None
    tol = 3e-3 if dt == "fp32" else TOL_REL
    for step in (1, 2):
        w_in = w_or if (dt == "fp32" or master) else _bf16_round(w_or)
        ref = _oracle_grad(x.H_f32(), _bf16_round(w_or) if dt == "bf16" else w_or, x.targets)
        kw = dict(hp)
        if kind == "adamw":
            kw["eps"] = 10.0 * float(np.max(np.abs(ref["dW"])))
            opt.eps = kw["eps"]
        else:
            kw["momentum"] = momentum
        old = np64(opt.master if master else W)
        loss, dH = opt.step(H, t, IGNORE_INDEX, vocab_chunk=768)
        torch.cuda.synchronize()
        assert lce.device_status() == 0
        o = _step(kind, w_in, ref["dW"], step=step, exp_avg=m_or, exp_avg_sq=v_or, **kw)
        new = np64(opt.master if master else W)
        bound = tol
        if dt == "bf16" and not master:   # the in-place bf16 rounding of W
            bound += 2.0 ** -8 * np.linalg.norm(new) / np.linalg.norm(o["w"] - w_in)
        errs = {"loss": abs(loss.item() - ref["loss"]), "step": rel_fro(new - old, o["w"] - w_in)}
        if o["exp_avg"] is not None:
            errs["m"] = rel_fro(np64(opt.exp_avg), o["exp_avg"])
        if o["exp_avg_sq"] is not None:
            errs["v"] = rel_fro(np64(opt.exp_avg_sq), o["exp_avg_sq"])
        print(case, step, errs, bound)
        assert errs["loss"] <= (1e-4 if dt == "fp32" else TOL_LOSS), errs
        assert errs["step"] <= bound, errs
        assert errs.get("m", 0.0) <= tol and errs.get("v", 0.0) <= 2 * tol, errs
        if master:
            assert torch.equal(W, opt.master.to(torch.bfloat16))
        w_or, m_or, v_or = o["w"], o["exp_avg"], o["exp_avg_sq"]
        if dt == "bf16" and not master:
            w_or = _bf16_round(w_or)   # W is stored as the bf16 rounding of the update (the contract)


@pytest.mark.parametrize("kind,hp", [("adamw", dict(lr=1e-2, betas=(0.9, 0.99), weight_decay=0.1)),
                                     ("sgd", dict(lr=0.05, momentum=0.9, weight_decay=0.01))])
def test_bf16_state_first_step_equals_fp32_state_rounded(kind, hp):
    """Optimizer state kept in bf16: on a first step (zero state, exact in
    both) the update of W is bit for bit the fp32-state update (both run in
    fp32 from the same values), and the stored state is the fp32 state
    rounded to the nearest bf16, bit for bit."""
    x = make_inputs("gpt1b", N=700, d=192, V=2500, padding=("random_frac", 0.2), seqs=1)
    H, W0, t = to_device(x)
    outs = {}
    for sd in (torch.float32, torch.bfloat16):
        W = W0.clone()
        opt = lce.FusedOptimizer(W, kind, master_weights=True, state_dtype=sd, **hp)
        assert opt.exp_avg.dtype == sd
        opt.step(H, t, IGNORE_INDEX, vocab_chunk=1024)
        torch.cuda.synchronize()
        assert lce.device_status() == 0
        outs[sd] = (W, opt.master, opt.exp_avg, opt.exp_avg_sq)
    W32, M32, m32, v32 = outs[torch.float32]
    W16, M16, m16, v16 = outs[torch.bfloat16]
    assert torch.equal(W32, W16) and torch.equal(M32, M16)
    assert torch.equal(m32.to(torch.bfloat16), m16)
    if kind == "adamw":
        assert torch.equal(v32.to(torch.bfloat16), v16)


def test_adamw_bf16_state_three_steps_against_oracle():
    """AdamW with bf16 moments on a bf16 W with fp32 master weights, three
    steps, against the oracle's step with bf16-rounded state: the step within
    the gradient's bound, the moments within it plus one bf16 rounding
    (2^-8 relative)."""
    x = make_inputs("gpt1b", N=1100, d=200, V=5000, padding=("random_frac", 0.3), seqs=1)
    H0, W, t = to_device(x)
    opt = lce.FusedOptimizer(W, "adamw", lr=1e-2, betas=(0.9, 0.99), weight_decay=0.1, master_weights=True,
                             state_dtype=torch.bfloat16)
    w_or = x.W_f32().astype(np.float64)
    m_or = v_or = None
    rng = np.random.default_rng(5)
    for step in (1, 2, 3):
        Hs = x.H_f32() if step == 1 else _bf16_round(rng.standard_normal(x.H_f32().shape))
        Hd = H0 if step == 1 else torch.from_numpy(Hs.astype(np.float32)).to("cuda").to(torch.bfloat16)
        ref = _oracle_grad(Hs, _bf16_round(w_or), x.targets)
        eps = 10.0 * float(np.max(np.abs(ref["dW"])))          # step nearly linear in g
        opt.eps = eps
        master_old = np64(opt.master)
        loss, dH = opt.step(Hd, t, IGNORE_INDEX, vocab_chunk=1024)
        torch.cuda.synchronize()
        assert lce.device_status() == 0
        o = _step("adamw", w_or, ref["dW"], lr=1e-2, step=step, weight_decay=0.1, beta1=0.9, beta2=0.99, eps=eps,
                  exp_avg=m_or, exp_avg_sq=v_or, state_bf16=True)
        errs = {"loss": abs(loss.item() - ref["loss"]), "step": rel_fro(np64(opt.master) - master_old, o["w"] - w_or),
                "m": rel_fro(np64(opt.exp_avg), o["exp_avg"]), "v": rel_fro(np64(opt.exp_avg_sq), o["exp_avg_sq"])}
        print(step, errs)
        assert errs["loss"] <= TOL_LOSS and errs["step"] <= TOL_REL, errs
        assert errs["m"] <= TOL_REL + 2.0 ** -8 and errs["v"] <= 2 * TOL_REL + 2.0 ** -8, errs
        assert torch.equal(W, opt.master.to(torch.bfloat16))
        w_or, m_or, v_or = o["w"], o["exp_avg"], o["exp_avg_sq"]
