"""Options of lce_run used together. Each pair below changes how the same
arithmetic is scheduled or where an operand comes from, not the arithmetic
itself, so the results must agree bit for bit with the call without the
second option (the oracle comparisons of each option alone are in
test_gpu_parity.py and test_gpu_optim.py)."""
import pytest

torch = pytest.importorskip("torch")

import chunked_vocab_cross_gb300 as lce  # noqa: E402
from chunked_vocab_cross_gb300 import _abi  # noqa: E402
from lce_testutil import to_device  # noqa: E402
from synth_inputs import IGNORE_INDEX, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from chunked_vocab_cross_gb300.build import build
    build()
    lce.device_status()
    yield


def _outs(H, W, t, **kw):
    N = H.shape[0]
    loss = torch.full((), float("nan"), dtype=torch.float32, device="cuda")
    dH = torch.empty_like(H)
    dW = torch.empty(W.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(N, dtype=torch.float32, device="cuda")
    lse_in = kw.pop("lse_in", None)
    if lse_in is not None:
        lce.lce_run(H, W, t, IGNORE_INDEX, dH=dH, dW=dW, lse_in=lse_in, **kw)
        lse = None
    else:
        lce.lce_run(H, W, t, IGNORE_INDEX, loss=loss, dH=dH, dW=dW, lse=lse, **kw)
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    return loss, dH, dW, lse


def _bits(x):
    return x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32)


def _same(a, b):
    """Bit-for-bit equality (NaN rows, e.g. lse of ignored tokens, included)."""
    for x, y in zip(a, b):
        if x is None or y is None:
            assert x is None and y is None
            continue
        assert torch.equal(_bits(x.reshape(-1)), _bits(y.reshape(-1)))


def test_row_gather_with_token_chunks():
    x = make_inputs("gpt1b", N=2600, d=256, V=5000, padding=("random_frac", 0.3), seqs=1)
    H, W, t = to_device(x)
    _same(_outs(H, W, t, token_chunk=1000, vocab_chunk=1024, row_gather=True),
          _outs(H, W, t, token_chunk=1000, vocab_chunk=1024))


def test_row_gather_with_backward_from_stored_lse():
    x = make_inputs("gpt1b", N=1300, d=512, V=4100, padding=("random_frac", 0.25), seqs=1)
    H, W, t = to_device(x)
    _, _, _, lse = _outs(H, W, t)
    _same(_outs(H, W, t, lse_in=lse, row_gather=True), _outs(H, W, t, lse_in=lse))


def _adamw_run(H, W, t, row_gather, master):
    Wc = W.clone()
    opt = lce.FusedOptimizer(Wc, "adamw", lr=1e-2, weight_decay=0.05, master_weights=master)
    outs = []
    for _ in range(2):
        loss = torch.empty((), dtype=torch.float32, device="cuda")
        dH = torch.empty_like(H)
        opt.step_count += 1
        lce.lce_run(H, Wc, t, IGNORE_INDEX, loss=loss, dH=dH, vocab_chunk=1024, optim=opt.optim_args(),
                    row_gather=row_gather)
        outs += [loss, dH]
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    return outs + [Wc, opt.exp_avg, opt.exp_avg_sq] + ([opt.master] if master else [])


@pytest.mark.parametrize("master", [False, True], ids=["in_place", "master"])
def test_row_gather_with_fused_optimizer(master):
    x = make_inputs("gpt1b", N=1500, d=256, V=4500, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    _same(_adamw_run(H, W, t, True, master), _adamw_run(H, W, t, False, master))


def test_fused_optimizer_captured_in_a_cuda_graph():
    """The fused-optimizer call with a caller workspace enqueues kernels only,
    so it can be captured; a replay applies the same update as an eager call
    (the optimizer arguments, step included, are fixed at capture)."""
    x = make_inputs("gpt1b", N=1024, d=256, V=3000, padding=("random_frac", 0.2), seqs=1)
    H, W, t = to_device(x)
    N, d = H.shape
    V = W.shape[0]
    ws = torch.empty(lce.workspace_size(N, d, V, fused_optimizer=True), dtype=torch.uint8, device="cuda")

    def state():
        g = torch.Generator(device="cuda").manual_seed(1)
        return (W.clone(), torch.randn(W.shape, device="cuda", generator=g) * 1e-4,
                torch.rand(W.shape, device="cuda", generator=g) * 1e-8)

    def optim(Wc, m, v):
        o = _abi.LceOptim()
        o.kind, o.lr, o.weight_decay, o.step = _abi.LCE_OPT_ADAMW, 1e-2, 0.1, 3
        o.beta1, o.beta2, o.eps = 0.9, 0.999, 1e-8
        o.exp_avg, o.exp_avg_sq = m.data_ptr(), v.data_ptr()
        return o

    loss_e, dH_e = torch.empty((), dtype=torch.float32, device="cuda"), torch.empty_like(H)
    We, me, ve = state()
    lce.lce_run(H, We, t, IGNORE_INDEX, loss=loss_e, dH=dH_e, workspace=ws, optim=optim(We, me, ve))
    torch.cuda.synchronize()

    Wg, mg, vg = state()
    o = optim(Wg, mg, vg)
    loss_g, dH_g = torch.empty((), dtype=torch.float32, device="cuda"), torch.empty_like(H)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        lce.lce_run(H, Wg, t, IGNORE_INDEX, loss=loss_g, dH=dH_g, workspace=ws, optim=o)
    W0, m0, v0 = state()                  # capture runs nothing: restore the state, then replay once
    Wg.copy_(W0), mg.copy_(m0), vg.copy_(v0)
    graph.replay()
    torch.cuda.synchronize()
    assert lce.device_status() == 0
    _same([loss_g, dH_g, Wg, mg, vg], [loss_e, dH_e, We, me, ve])
