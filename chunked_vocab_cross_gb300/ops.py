"""Python entry points with the C ABI's names. PyTorch provides device memory
and the current stream; the arithmetic is all in liblce.so."""
from __future__ import annotations

import ctypes

import torch

from . import _abi

_DT = {torch.bfloat16: _abi.LCE_BF16, torch.float32: _abi.LCE_FP32}


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check_inputs(H: torch.Tensor, W: torch.Tensor, targets: torch.Tensor):
    if not (H.is_cuda and W.is_cuda and targets.is_cuda):
        raise ValueError("H, W and targets must be CUDA tensors (there is no CPU path)")
    if H.dtype not in _DT or W.dtype != H.dtype:
        raise ValueError("H and W must both be bfloat16 or both float32")
    if targets.dtype != torch.int64:
        raise ValueError("targets must be int64")
    if H.dim() != 2 or W.dim() != 2 or targets.dim() != 1:
        raise ValueError("H must be [N,d], W [V,d], targets [N]")
    if H.shape[1] != W.shape[1] or H.shape[0] != targets.shape[0]:
        raise ValueError("shape mismatch between H, W and targets")
    if not (H.is_contiguous() and W.is_contiguous() and targets.is_contiguous()):
        raise ValueError("H, W and targets must be contiguous")


def workspace_size(N: int, d: int, V: int, dtype=torch.bfloat16, vocab_chunk: int = 0, token_chunk: int = 0,
                   backward: bool = True, fused_optimizer: bool = False, row_gather: bool = False) -> int:
    a = _abi.LceArgs()
    a.dtype = _DT[dtype]
    a.N, a.d, a.V = N, d, V
    a.vocab_chunk, a.token_chunk = vocab_chunk, token_chunk
    a.dH = 1 if backward else None      # only whether gradients are wanted matters
    a.row_gather = 1 if row_gather else 0
    o = _abi.LceOptim()
    if fused_optimizer:
        o.kind = _abi.LCE_OPT_SGD
        a.optim = ctypes.addressof(o)
    return int(_abi.lib().lce_workspace_size_args(ctypes.byref(a)))


def lce_run(H, W, targets, ignore_index: int = -100, *, loss=None, dH=None, dW=None, accumulate_dW: bool = False,
            grad_scale: float = 1.0, lse=None, workspace=None, vocab_chunk: int = 0, lse_in=None, grad_loss=None,
            token_chunk: int = 0, optim=None, row_gather: bool = False, stream=None) -> None:
    """Raw lce_run over caller-provided output tensors. `optim` is an
    _abi.LceOptim (a fused optimizer step on W) or None. dW may be fp32 or,
    for bf16 inputs without accumulation, bf16."""
    _check_inputs(H, W, targets)
    a = _abi.LceArgs()
    a.dtype = _DT[H.dtype]
    a.H, a.W, a.targets = H.data_ptr(), W.data_ptr(), targets.data_ptr()
    a.ignore_index = int(ignore_index)
    a.N, a.d = H.shape
    a.V = W.shape[0]
    a.loss = loss.data_ptr() if loss is not None else None
    a.lse_in = lse_in.data_ptr() if lse_in is not None else None
    a.grad_loss = grad_loss.data_ptr() if grad_loss is not None else None
    a.dH = dH.data_ptr() if dH is not None else None
    a.dW = dW.data_ptr() if dW is not None else None
    a.dW_bf16 = 1 if (dW is not None and dW.dtype == torch.bfloat16) else 0
    a.accumulate_dW = 1 if accumulate_dW else 0
    a.grad_scale = float(grad_scale)
    a.lse = lse.data_ptr() if lse is not None else None
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    a.vocab_chunk = int(vocab_chunk)
    a.token_chunk = int(token_chunk)
    a.optim = ctypes.addressof(optim) if optim is not None else None
    a.row_gather = 1 if row_gather else 0
    a.stream = _stream(stream)
    _abi.check(_abi.lib().lce_run(ctypes.byref(a)), "lce_run")


def lce_forward(H, W, targets, ignore_index: int = -100, *, return_lse: bool = False, stream=None):
    """Mean cross-entropy over valid tokens of (H @ W^T, targets); fp32 0-d tensor."""
    _check_inputs(H, W, targets)
    loss = torch.empty((), dtype=torch.float32, device=H.device)
    lse = torch.empty(H.shape[0], dtype=torch.float32, device=H.device) if return_lse else None
    if H.dtype == torch.bfloat16 and not return_lse:
        _abi.check(_abi.lib().lce_forward(H.data_ptr(), W.data_ptr(), targets.data_ptr(), int(ignore_index),
                                          H.shape[0], H.shape[1], W.shape[0], loss.data_ptr(), _stream(stream)),
                   "lce_forward")
    else:
        lce_run(H, W, targets, ignore_index, loss=loss, lse=lse, stream=stream)
    return (loss, lse) if return_lse else loss


def lce_forward_backward(H, W, targets, ignore_index: int = -100, *, dW=None, accumulate_dW: bool = False,
                         grad_scale: float = 1.0, vocab_chunk: int = 0, return_lse: bool = False,
                         workspace=None, token_chunk: int = 0, stream=None):
    """Loss, dH (H's dtype, zero on ignored rows) and dW (fp32, or the given
    dW's dtype: bf16 for bf16 inputs without accumulation) in one pass."""
    _check_inputs(H, W, targets)
    loss = torch.empty((), dtype=torch.float32, device=H.device)
    dH = torch.empty_like(H)
    if dW is None:
        dW = torch.empty(W.shape, dtype=torch.float32, device=W.device)
        accumulate_dW = False
    elif dW.dtype not in (torch.float32, torch.bfloat16) or dW.shape != W.shape or not dW.is_contiguous():
        raise ValueError("dW must be a contiguous fp32 (or bf16) tensor shaped like W")
    lse = torch.empty(H.shape[0], dtype=torch.float32, device=H.device) if return_lse else None
    simple = (H.dtype == torch.bfloat16 and dW.dtype == torch.float32 and not accumulate_dW and grad_scale == 1.0
              and vocab_chunk == 0 and not return_lse and workspace is None and token_chunk == 0)
    if simple:
        _abi.check(_abi.lib().lce_forward_backward(H.data_ptr(), W.data_ptr(), targets.data_ptr(),
                                                   int(ignore_index), H.shape[0], H.shape[1], W.shape[0],
                                                   loss.data_ptr(), dH.data_ptr(), dW.data_ptr(),
                                                   _stream(stream)),
                   "lce_forward_backward")
    else:
        lce_run(H, W, targets, ignore_index, loss=loss, dH=dH, dW=dW, accumulate_dW=accumulate_dW,
                grad_scale=grad_scale, lse=lse, workspace=workspace, vocab_chunk=vocab_chunk,
                token_chunk=token_chunk, stream=stream)
    out = (loss, dH, dW)
    return out + (lse,) if return_lse else out


def lce_backward(H, W, targets, lse, ignore_index: int = -100, *, grad_loss=None, dW=None,
                 accumulate_dW: bool = False, vocab_chunk: int = 0, workspace=None, stream=None):
    """dH and dW from a stored per-row lse (lce_forward(..., return_lse=True)),
    times the device scalar grad_loss (None = 1). Logits are recomputed."""
    _check_inputs(H, W, targets)
    if lse.dtype != torch.float32 or lse.shape != (H.shape[0],) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [N] tensor")
    if grad_loss is not None:
        grad_loss = grad_loss.detach().to(device=H.device, dtype=torch.float32).contiguous()
    dH = torch.empty_like(H)
    if dW is None:
        dW = torch.empty(W.shape, dtype=torch.float32, device=W.device)
        accumulate_dW = False
    if dW.dtype not in (torch.float32, torch.bfloat16) or dW.shape != W.shape or not dW.is_contiguous():
        raise ValueError("dW must be a contiguous fp32 (or bf16) tensor shaped like W")
    if (H.dtype == torch.bfloat16 and dW.dtype == torch.float32 and not accumulate_dW and vocab_chunk == 0
            and workspace is None):
        _abi.check(_abi.lib().lce_backward(H.data_ptr(), W.data_ptr(), targets.data_ptr(), int(ignore_index),
                                           H.shape[0], H.shape[1], W.shape[0], lse.data_ptr(),
                                           grad_loss.data_ptr() if grad_loss is not None else None,
                                           dH.data_ptr(), dW.data_ptr(), _stream(stream)),
                   "lce_backward")
    else:
        lce_run(H, W, targets, ignore_index, dH=dH, dW=dW, accumulate_dW=accumulate_dW, lse_in=lse,
                grad_loss=grad_loss, vocab_chunk=vocab_chunk, workspace=workspace, stream=stream)
    return dH, dW


def lce_compact(targets, ignore_index: int = -100, V: int | None = None, *, stream=None):
    """(idx[:Nv] int32, inv int32, Nv, out_of_range) from the compaction kernel."""
    if not targets.is_cuda or targets.dtype != torch.int64 or targets.dim() != 1:
        raise ValueError("targets must be a 1-D int64 CUDA tensor")
    targets = targets.contiguous()
    N = targets.shape[0]
    idx = torch.empty(N, dtype=torch.int32, device=targets.device)
    inv = torch.empty(N, dtype=torch.int32, device=targets.device)
    counts = torch.empty(2, dtype=torch.int32, device=targets.device)
    _abi.check(_abi.lib().lce_compact(targets.data_ptr(), N, int(ignore_index), int(V if V else 2**31 - 1),
                                      idx.data_ptr(), inv.data_ptr(), counts.data_ptr(), _stream(stream)),
               "lce_compact")
    nv, bad = counts.tolist()
    return idx[:nv], inv, nv, bad


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status bits."""
    bits = ctypes.c_int32(0)
    _abi.lib().lce_get_device_status(_stream(stream), ctypes.byref(bits))
    return int(bits.value)


def launch_count() -> int:
    return int(_abi.lib().lce_launch_count())


def profile_begin() -> None:
    _abi.check(_abi.lib().lce_profile_begin(), "lce_profile_begin")


def profile_end() -> dict:
    n = _abi.PROFILE_PHASES
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _abi.check(_abi.lib().lce_profile_end(ms, cnt, n), "lce_profile_end")
    return {name: {"ms": ms[i], "launches": int(cnt[i])} for i, name in enumerate(_abi.PHASE_NAMES)}


class _LinearCrossEntropySplit(torch.autograd.Function):
    """Two-call form: the forward computes the loss and keeps only the per-row
    lse [N]; the backward recomputes the logits and applies the incoming
    gradient on the device."""

    @staticmethod
    def forward(ctx, H, W, targets, ignore_index):
        H, W, targets = H.contiguous(), W.contiguous(), targets.contiguous()
        loss, lse = lce_forward(H, W, targets, ignore_index, return_lse=True)
        ctx.save_for_backward(H, W, targets, lse)
        ctx.ignore_index = ignore_index
        return loss

    @staticmethod
    def backward(ctx, g):
        H, W, targets, lse = ctx.saved_tensors
        # the gradient of W in W's dtype, written by the library (a bf16 W
        # gets a bf16 dW: each fp32 accumulator rounded once)
        dW = torch.empty(W.shape, dtype=W.dtype, device=W.device)
        dH, dW = lce_backward(H, W, targets, lse, ctx.ignore_index, grad_loss=g, dW=dW)
        return (dH if ctx.needs_input_grad[0] else None,
                dW if ctx.needs_input_grad[1] else None, None, None)


def linear_cross_entropy(H, W, targets, ignore_index: int = -100):
    """loss = cross_entropy(H @ W^T, targets, ignore_index) without materialising logits.

    The forward keeps only the per-row lse [N]; the backward recomputes the
    logits and runs the gradient passes with the incoming gradient applied
    inside the kernels (a device scalar read in the G epilogue, no host sync)
    and dW written in W's dtype by the library."""
    return _LinearCrossEntropySplit.apply(H, W, targets, ignore_index)


class FusedOptimizer:
    """SGD or AdamW on the vocabulary matrix W, applied inside the backward
    pass of lce_run (the optimizer item of include/lce.h): each call of step()
    returns the loss and dH for the current W and leaves W updated, without a
    gradient buffer for W ever existing. Holds the state (moments or momentum
    buffer, fp32 by default or bf16 with state_dtype=torch.bfloat16, as
    torch.optim keeps them for a bf16 parameter; optional fp32 master weights
    of a bf16 W) on W's device.

    The pages' training loop attaches an optimizer with algorithm "adamw" or
    "sgd" that updates weights in place during backward ("OjasX 0.6.1:
    Training a 1B-Parameter LLM in 6.35GB of RAM", usage listing)."""

    def __init__(self, W: torch.Tensor, algorithm: str = "adamw", lr: float = 3e-4, betas=(0.9, 0.999),
                 eps: float = 1e-8, weight_decay: float = 0.0, momentum: float = 0.0, master_weights: bool = False,
                 state_dtype=torch.float32):
        if algorithm not in ("adamw", "sgd"):
            raise ValueError("algorithm must be 'adamw' or 'sgd'")
        if not W.is_cuda or not W.is_contiguous() or W.dtype not in _DT:
            raise ValueError("W must be a contiguous bf16 or fp32 CUDA tensor")
        if master_weights and W.dtype != torch.bfloat16:
            raise ValueError("master weights are kept for a bf16 W only")
        if state_dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("state_dtype must be torch.float32 or torch.bfloat16")
        self.state_dtype = state_dtype
        self.W = W
        self.algorithm = algorithm
        self.lr, self.betas, self.eps = float(lr), (float(betas[0]), float(betas[1])), float(eps)
        self.weight_decay, self.momentum = float(weight_decay), float(momentum)
        self.step_count = 0
        z = lambda: torch.zeros(W.shape, dtype=state_dtype, device=W.device)  # noqa: E731
        self.exp_avg = z() if (algorithm == "adamw" or momentum != 0.0) else None
        self.exp_avg_sq = z() if algorithm == "adamw" else None
        self.master = W.float() if master_weights else None

    def optim_args(self) -> "_abi.LceOptim":
        """The lce_optim_t of the next update (the step count as it stands),
        for a direct lce_run(..., optim=...) call."""
        o = _abi.LceOptim()
        o.kind = _abi.LCE_OPT_ADAMW if self.algorithm == "adamw" else _abi.LCE_OPT_SGD
        o.lr, o.weight_decay, o.momentum = self.lr, self.weight_decay, self.momentum
        o.beta1, o.beta2 = self.betas
        o.eps = self.eps
        o.step = self.step_count
        o.master_W = self.master.data_ptr() if self.master is not None else None
        o.exp_avg = self.exp_avg.data_ptr() if self.exp_avg is not None else None
        o.exp_avg_sq = self.exp_avg_sq.data_ptr() if self.exp_avg_sq is not None else None
        o.state_bf16 = 1 if self.state_dtype == torch.bfloat16 else 0
        return o

    def step(self, H, targets, ignore_index: int = -100, *, grad_scale: float = 1.0, grad_loss=None,
             lse_in=None, vocab_chunk: int = 0, workspace=None, stream=None):
        """One forward + backward + update of W. Returns (loss, dH); with
        lse_in (a stored per-row lse of the current W) the forward is skipped
        and loss is None."""
        self.step_count += 1
        loss = None if lse_in is not None else torch.empty((), dtype=torch.float32, device=H.device)
        dH = torch.empty_like(H)
        try:
            lce_run(H, self.W, targets, ignore_index, loss=loss, dH=dH, grad_scale=grad_scale, grad_loss=grad_loss,
                    lse_in=lse_in, vocab_chunk=vocab_chunk, workspace=workspace, optim=self.optim_args(),
                    stream=stream)
        except Exception:
            self.step_count -= 1
            raise
        return loss, dH


def embedding_forward(W, tokens, pad_id: int = 0, *, out=None, stream=None):
    """E [N, d] (W's dtype): rows of W for the tokens, zero rows where the token
    is pad_id; non-padding ids outside [0, V) give zero rows and set the
    target-range bit of the device status word. `out` receives E if given."""
    if not (W.is_cuda and tokens.is_cuda) or W.dtype not in _DT or tokens.dtype != torch.int64:
        raise ValueError("W must be a bf16/fp32 CUDA tensor and tokens int64 on the same device")
    if W.dim() != 2 or tokens.dim() != 1 or not W.is_contiguous():
        raise ValueError("W must be a contiguous [V, d] tensor and tokens [N]")
    tokens = tokens.contiguous()
    if out is None:
        out = torch.empty((tokens.shape[0], W.shape[1]), dtype=W.dtype, device=W.device)
    elif out.dtype != W.dtype or out.shape != (tokens.shape[0], W.shape[1]) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [N, d] tensor of W's dtype")
    _abi.check(_abi.lib().lce_embedding_forward(_DT[W.dtype], W.data_ptr(), tokens.data_ptr(), int(pad_id),
                                                tokens.shape[0], W.shape[1], W.shape[0], out.data_ptr(),
                                                _stream(stream)), "lce_embedding_forward")
    return out


def embedding_workspace_size(N: int, d: int) -> int:
    """Bytes of scratch lce_embedding_backward needs for N positions of width d."""
    return int(_abi.lib().lce_embedding_workspace_size(int(N), int(d)))


def embedding_backward(dE, tokens, pad_id: int, V: int, *, dW=None, accumulate: bool = False, workspace=None,
                       stream=None):
    """dW [V, d] with each token's gradient rows summed in fp32 in a fixed
    order: fp32 (overwritten, or added into a given dW with accumulate), or a
    given bf16 dW (each row sum rounded once; overwritten). `workspace`: a
    uint8 CUDA tensor of at least embedding_workspace_size(N, d) bytes; without
    it the library allocates its scratch on the stream."""
    if not (dE.is_cuda and tokens.is_cuda) or dE.dtype not in _DT or tokens.dtype != torch.int64:
        raise ValueError("dE must be a bf16/fp32 CUDA tensor and tokens int64 on the same device")
    if dE.dim() != 2 or tokens.dim() != 1 or dE.shape[0] != tokens.shape[0]:
        raise ValueError("dE must be [N, d] and tokens [N]")
    dE, tokens = dE.contiguous(), tokens.contiguous()
    if dW is None:
        dW = torch.empty((V, dE.shape[1]), dtype=torch.float32, device=dE.device)
        accumulate = False
    elif dW.dtype not in (torch.float32, torch.bfloat16) or dW.shape != (V, dE.shape[1]) or not dW.is_contiguous():
        raise ValueError("dW must be a contiguous fp32 (or bf16) [V, d] tensor")
    if dW.dtype == torch.bfloat16 and accumulate:
        raise ValueError("a bf16 dW is overwritten, not accumulated into")
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    if dW.dtype == torch.bfloat16:
        _abi.check(_abi.lib().lce_embedding_backward_bf16(_DT[dE.dtype], dE.data_ptr(), tokens.data_ptr(),
                                                          int(pad_id), tokens.shape[0], dE.shape[1], V,
                                                          dW.data_ptr(), ws_ptr, ws_bytes, _stream(stream)),
                   "lce_embedding_backward_bf16")
    else:
        _abi.check(_abi.lib().lce_embedding_backward(_DT[dE.dtype], dE.data_ptr(), tokens.data_ptr(), int(pad_id),
                                                     tokens.shape[0], dE.shape[1], V, dW.data_ptr(),
                                                     1 if accumulate else 0, ws_ptr, ws_bytes, _stream(stream)),
                   "lce_embedding_backward")
    return dW


class _Embedding(torch.autograd.Function):
    @staticmethod
    def forward(ctx, W, tokens, pad_id):
        ctx.save_for_backward(tokens)
        ctx.pad_id, ctx.V, ctx.w_dtype = pad_id, W.shape[0], W.dtype
        return embedding_forward(W, tokens, pad_id)

    @staticmethod
    def backward(ctx, dE):
        (tokens,) = ctx.saved_tensors
        # the gradient of W in W's dtype, written by the library from dE as it
        # arrives (bf16 or fp32)
        dW = torch.empty((ctx.V, dE.shape[1]), dtype=ctx.w_dtype, device=dE.device)
        return embedding_backward(dE, tokens, ctx.pad_id, ctx.V, dW=dW), None, None


def embedding(W, tokens, pad_id: int = 0):
    """Autograd input-embedding lookup that skips padding (zero rows, no
    gradient); with a W tied to the output projection its gradient adds to
    linear_cross_entropy's through autograd."""
    return _Embedding.apply(W, tokens, pad_id)
