"""fp64 CPU oracle for the input-embedding lookup that skips padding, and its
gradient (the input side of a tied vocabulary matrix W).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
this module: only the tests do. It shares no code with the CUDA library.

Source: "为什么26万词表会卡死16GB显卡" (the 260K-vocabulary embedding page),
section 2.3 稀疏索引引擎: a valid mask is built from the input token ids and
only masked-in positions look up their embedding row; padding positions
return a zero vector. Section 2.2 梯度延迟聚合: the per-token gradient rows
of a batch are aggregated into the embedding rows after the batch's backward.
The tied use (one W for the input lookup and the output layer) is from
"6GB显卡预训练11亿参数模型", section "关键参数说明" (--tie-embeddings).
Readings: the padding id is a parameter; a non-padding token id outside
[0, V) is an input error (the oracle refuses it); the aggregation is the
plain sum over positions, taken in float64 (the page's time-dependent
"temporal gradient calibration" changes the gradient and is not part of it).

    E[i, :]  = W[t_i, :]  if t_i != pad_id, else 0
    dW[v, :] = sum over positions i with t_i == v (t_i != pad_id) of dE[i, :]

Pins (tests/test_oracle_pins.py): float64 torch autograd of a masked
F.embedding, exact row copies in the forward, and invariants (the rows of dW
sum to the sum of dE over valid positions; vocab rows no token hits are
exactly zero; reordering positions together with dE leaves dW unchanged).
"""
from __future__ import annotations

import numpy as np

__all__ = ["embedding_forward", "embedding_backward"]


def _valid(tokens, pad_id: int, V: int) -> np.ndarray:
    t = np.asarray(tokens, dtype=np.int64)
    valid = t != pad_id
    if np.any((t[valid] < 0) | (t[valid] >= V)):
        raise ValueError("a non-padding token id is outside [0, V)")
    return valid


def embedding_forward(W, tokens, pad_id: int) -> np.ndarray:
    """E [N, d] float64: the rows of W for valid positions, zeros for padding."""
    W = np.asarray(W)
    t = np.asarray(tokens, dtype=np.int64)
    valid = _valid(t, pad_id, W.shape[0])
    E = np.zeros((t.shape[0], W.shape[1]), dtype=np.float64)
    E[valid] = W[t[valid]].astype(np.float64)
    return E


def embedding_backward(dE, tokens, pad_id: int, V: int) -> np.ndarray:
    """dW [V, d] float64: each valid position's gradient row added to its token's row."""
    dE = np.asarray(dE, dtype=np.float64)
    t = np.asarray(tokens, dtype=np.int64)
    valid = _valid(t, pad_id, V)
    dW = np.zeros((V, dE.shape[1]), dtype=np.float64)
    np.add.at(dW, t[valid], dE[valid])
    return dW
