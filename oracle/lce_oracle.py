"""fp64 CPU oracle for the fused output-projection + cross-entropy path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
this module: only the tests, the package's smoke check and the benchmark's
CPU-baseline leg do. It shares no code with the CUDA library; the two meet only
through the seeded arrays of ``synth_inputs``.

What it computes is the plain definition, written out in float64 on the exact
input values (bf16 or fp32 widened to float64, which is exact):

    valid rows    I = { i : t_i != ignore_index }, ascending, Nv = |I|
    logits        s_iv = sum_k H[i,k] W[v,k]                       (all v)
    log-sum-exp   lse_i = M_i + log sum_v exp(s_iv - M_i), M_i = max_v s_iv
    loss          loss = (1/Nv) sum_{i in I} (lse_i - s_{i,t_i})
    softmax grad  g_iv = (exp(s_iv - lse_i) - [v == t_i]) / Nv
    dH[i,:]       = sum_v g_iv W[v,:]   for i in I, 0 on ignored rows
    dW[v,:]       = sum_{i in I} g_iv H[i,:]

Sources: the projection-plus-loss computed in streamed chunks with padding
tokens skipped ("OjasX 0.6.1: Training a 1B-Parameter LLM in 6.35GB of RAM",
section "Core Technology", the zero-byte vocabulary logits item); logits
recomputed in backward rather than stored, which leaves the gradients unchanged
("6GB显卡预训练11亿参数模型", sections "内存实际花在哪里" and "关键参数说明",
--chunked-loss 512); online softmax reaching the same result as the two-pass
one (same OjasX page, "Online Softmax" note). The normaliser is the number of
valid tokens and Nv = 0 gives a NaN loss with zero gradients (the mean over an
empty set). A target outside [0, V) that is not ignore_index is an input error;
the oracle reports it and refuses the input.

Every step is a whole-row numpy operation; the matrix products are library
matmuls computed for a batch of rows at a time (a batch of rows of one matmul,
not a reordering of the arithmetic). Each row's max and log-sum-exp are taken
over the complete row of V logits, never by the streaming recurrence the fast
path uses.

The same definition is written a second time as plain C++ loops
(oracle/lce_oracle.cpp, loaded through oracle/cpp_oracle.py); the two share
nothing but the definition, and tests/test_oracle_cross.py checks that they
agree to rounding.

Pins (tests/test_oracle_pins.py, run against both): closed forms at W=0, H=0, V=1 and V=2,
central finite differences on tiny inputs, float64 torch autograd of
cross_entropy(H @ W.T), and invariants (rows of G sum to zero so the columns of
dW sum to zero; shifting every vocab row by the same vector changes nothing;
permuting tokens permutes dH; padded rows get exact zeros).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "valid_rows", "out_of_range_targets", "forward", "forward_backward",
    "sampled_reference",
]

_ROW_BATCH = 256      # rows of H per matmul call
_VOCAB_BLOCK = 16384  # vocab rows widened to float64 at a time


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def valid_rows(targets: np.ndarray, ignore_index: int) -> np.ndarray:
    """Ascending positions whose target is not ignore_index (the dense index
    list of the padding-aware valid mask: "为什么26万词表会卡死16GB显卡",
    section 2.3 稀疏索引引擎)."""
    return np.nonzero(np.asarray(targets) != ignore_index)[0].astype(np.int64)


def out_of_range_targets(targets: np.ndarray, ignore_index: int, V: int) -> int:
    """Count of non-ignored targets outside [0, V)."""
    t = np.asarray(targets, dtype=np.int64)
    keep = t != ignore_index
    return int(np.count_nonzero(keep & ((t < 0) | (t >= V))))


def _logits(Hrows: np.ndarray, W: np.ndarray) -> np.ndarray:
    """s = Hrows @ W^T in float64; W is widened block by block so a bf16/fp32 W
    never needs a full float64 copy."""
    V = W.shape[0]
    S = np.empty((Hrows.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, _VOCAB_BLOCK):
        v1 = min(V, v0 + _VOCAB_BLOCK)
        S[:, v0:v1] = Hrows @ _f64(W[v0:v1]).T
    return S


def _lse(S: np.ndarray) -> np.ndarray:
    M = S.max(axis=1)
    return M + np.log(np.exp(S - M[:, None]).sum(axis=1))


def _check(H, W, targets, ignore_index):
    H = np.asarray(H)
    W = np.asarray(W)
    t = np.asarray(targets, dtype=np.int64)
    if H.ndim != 2 or W.ndim != 2 or t.ndim != 1:
        raise ValueError("H must be [N,d], W [V,d], targets [N]")
    if H.shape[0] != t.shape[0] or H.shape[1] != W.shape[1]:
        raise ValueError("shape mismatch")
    bad = out_of_range_targets(t, ignore_index, W.shape[0])
    if bad:
        raise ValueError(f"{bad} targets outside [0, V) that are not ignore_index")
    return H, W, t


def forward(H, W, targets, ignore_index: int = -100) -> dict:
    """Loss only. Returns loss, per-valid-row lse and loss_i, and the valid rows."""
    H, W, t = _check(H, W, targets, ignore_index)
    idx = valid_rows(t, ignore_index)
    nv = idx.shape[0]
    lse = np.empty(nv)
    z = np.empty(nv)
    for b0 in range(0, nv, _ROW_BATCH):
        r = idx[b0:b0 + _ROW_BATCH]
        S = _logits(_f64(H[r]), W)
        lse[b0:b0 + r.shape[0]] = _lse(S)
        z[b0:b0 + r.shape[0]] = S[np.arange(r.shape[0]), t[r]]
    loss_rows = lse - z
    loss = loss_rows.sum() / nv if nv else float("nan")
    return {"loss": float(loss), "lse": lse, "loss_rows": loss_rows, "idx": idx, "n_valid": nv}


def forward_backward(H, W, targets, ignore_index: int = -100) -> dict:
    """Loss, dH [N,d] and dW [V,d], all float64, by the definition above."""
    H, W, t = _check(H, W, targets, ignore_index)
    N, d = H.shape
    V = W.shape[0]
    idx = valid_rows(t, ignore_index)
    nv = idx.shape[0]
    dH = np.zeros((N, d))
    dW = np.zeros((V, d))
    lse_all = np.empty(nv)
    loss_rows = np.empty(nv)
    W64 = _f64(W)
    for b0 in range(0, nv, _ROW_BATCH):
        r = idx[b0:b0 + _ROW_BATCH]
        nb = r.shape[0]
        Hb = _f64(H[r])
        S = Hb @ W64.T                                   # s_iv
        lse = _lse(S)                                    # lse_i
        z = S[np.arange(nb), t[r]]                       # s_{i,t_i}
        G = np.exp(S - lse[:, None])                     # p_iv
        G[np.arange(nb), t[r]] -= 1.0                    # p_iv - [v == t_i]
        G /= nv                                          # g_iv
        dH[r] = G @ W64                                  # sum_v g_iv W_v
        dW += G.T @ Hb                                   # sum_i g_iv H_i
        lse_all[b0:b0 + nb] = lse
        loss_rows[b0:b0 + nb] = lse - z
    loss = loss_rows.sum() / nv if nv else float("nan")
    return {"loss": float(loss), "lse": lse_all, "loss_rows": loss_rows,
            "dH": dH, "dW": dW, "idx": idx, "n_valid": nv}


def sampled_reference(H, W, targets, ignore_index, token_rows, vocab_rows) -> dict:
    """For shapes too large for forward_backward: the full loss and every valid
    row's lse, plus dH on the sampled token rows and dW on the sampled vocab rows.

    dW[v] needs g_iv for every valid i, hence every valid row's lse; dH[i]
    needs all V logits of row i only.
    """
    H, W, t = _check(H, W, targets, ignore_index)
    idx = valid_rows(t, ignore_index)
    nv = idx.shape[0]
    fw = forward(H, W, t, ignore_index)
    lse_of = np.full(H.shape[0], np.nan)
    lse_of[idx] = fw["lse"]

    token_rows = np.asarray(token_rows, dtype=np.int64)
    dH_rows = np.zeros((token_rows.shape[0], H.shape[1]))
    for j, i in enumerate(token_rows):
        if t[i] == ignore_index:
            continue
        S = _logits(_f64(H[i:i + 1]), W)[0]
        g = np.exp(S - lse_of[i])
        g[t[i]] -= 1.0
        g /= nv
        dH_rows[j] = _gemv_T(W, g)

    vocab_rows = np.asarray(vocab_rows, dtype=np.int64)
    dW_rows = np.zeros((vocab_rows.shape[0], H.shape[1]))
    if nv:
        Wv = _f64(W[vocab_rows])
        for b0 in range(0, nv, _ROW_BATCH):
            r = idx[b0:b0 + _ROW_BATCH]
            Hb = _f64(H[r])
            Sv = Hb @ Wv.T                                # s_iv for sampled v
            G = np.exp(Sv - lse_of[r][:, None])
            G -= (t[r][:, None] == vocab_rows[None, :])
            G /= nv
            dW_rows += G.T @ Hb
    return {**fw, "token_rows": token_rows, "dH_rows": dH_rows,
            "vocab_rows": vocab_rows, "dW_rows": dW_rows}


def _gemv_T(W, g) -> np.ndarray:
    """sum_v g_v W[v,:] in float64, W widened block by block."""
    out = np.zeros(W.shape[1])
    for v0 in range(0, W.shape[0], _VOCAB_BLOCK):
        v1 = min(W.shape[0], v0 + _VOCAB_BLOCK)
        out += g[v0:v1] @ _f64(W[v0:v1])
    return out
