"""fp64 CPU oracle for the optimizer step that the library can fuse into the
backward pass (the weights W updated where their gradient is produced, so no
persistent gradient buffer exists).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
this module: only the tests do. It shares no code with the CUDA library.

Source: "OjasX 0.6.1: Training a 1B-Parameter LLM in 6.35GB of RAM", section
"Core Technology" (the zero-byte persistent .grad buffers item: weights are
updated and the gradient released as soon as a layer's backward is done), and
its usage listing, which attaches that optimizer with algorithm "adamw" or
"sgd" and lr=3e-4. The pages name the two algorithms without defining them;
the reading taken here is PyTorch's definitions, since the pages' code is
PyTorch: SGD with optional momentum (no dampening, no Nesterov) and L2 weight
decay added to the gradient; AdamW with the weight decay decoupled from the
gradient (Loshchilov & Hutter, "Decoupled Weight Decay Regularization") and
Adam's bias-corrected moments (Kingma & Ba, "Adam"), epsilon added to the
bias-corrected root of the second moment, no amsgrad.

One step, elementwise, in float64 (w the weights, g their gradient, t the
1-based step number):

    SGD     g' = g + wd * w
            momentum != 0:  b = g' if t == 1 else momentum * b + g';  g' = b
            w  = w - lr * g'
    AdamW   w  = w * (1 - lr * wd)
            m  = beta1 * m + (1 - beta1) * g
            v  = beta2 * v + (1 - beta2) * g^2
            w  = w - lr * (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)

State kept in bf16 (state_bf16=True, the layout torch.optim uses for a bf16
parameter): the step itself is the same; the state it returns is rounded to
the nearest bf16 (ties to even), while the update of w uses the unrounded
values, so w is the fp32-state step's w and the state is that step's state
rounded.

Pins (tests/test_oracle_pins.py): torch.optim.SGD and torch.optim.AdamW in
float64 over several steps (independent implementations of the same rules),
the closed form of AdamW's first step (m_hat = g and v_hat = g^2, so the step
is lr * g / (|g| + eps)), and invariants (a zero gradient with no decay leaves
w unchanged and scales m by beta1 and v by beta2).
"""
from __future__ import annotations

import numpy as np

__all__ = ["optimizer_step"]


def optimizer_step(kind: str, w, g, *, lr: float, step: int, weight_decay: float = 0.0,
                   momentum: float = 0.0, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                   exp_avg=None, exp_avg_sq=None, state_bf16: bool = False) -> dict:
    """One optimizer step on weights w with gradient g (any shapes, equal).

    Returns float64 arrays {"w", "exp_avg", "exp_avg_sq"} (state entries None
    when the rule keeps none); the inputs are not modified. exp_avg is the SGD
    momentum buffer or AdamW's first moment, exp_avg_sq AdamW's second moment;
    None means zeros (the state before the first step). With state_bf16
    the returned state is rounded to bf16 (as float64 values)."""
    if step < 1:
        raise ValueError("step is 1-based")
    w = np.array(w, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    if w.shape != g.shape:
        raise ValueError("w and g differ in shape")
    m = np.zeros_like(w) if exp_avg is None else np.array(exp_avg, dtype=np.float64)
    v = np.zeros_like(w) if exp_avg_sq is None else np.array(exp_avg_sq, dtype=np.float64)
    if kind == "sgd":
        d = g + weight_decay * w
        if momentum != 0.0:
            m = d.copy() if step == 1 else momentum * m + d
            d = m
            out_m = m
        else:
            out_m = None
        return {"w": w - lr * d, "exp_avg": _store(out_m, state_bf16), "exp_avg_sq": None}
    if kind == "adamw":
        w = w * (1.0 - lr * weight_decay)
        m = beta1 * m + (1.0 - beta1) * g
        v = beta2 * v + (1.0 - beta2) * g * g
        m_hat = m / (1.0 - beta1 ** step)
        v_hat = v / (1.0 - beta2 ** step)
        return {"w": w - lr * m_hat / (np.sqrt(v_hat) + eps), "exp_avg": _store(m, state_bf16),
                "exp_avg_sq": _store(v, state_bf16)}
    raise ValueError(f"unknown optimizer {kind!r}")


def _store(x, bf16: bool):
    """State as stored: unchanged, or rounded to the nearest bf16 (ties to
    even) by way of its float32 value."""
    if x is None or not bf16:
        return x
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF))) & np.uint32(0xFFFF0000)
    return r.view(np.float32).astype(np.float64)
