"""Plain CPU oracle of the tied 4-bit head (and the tied embedding).

TEST INFRASTRUCTURE ONLY, like moe_oracle (whose number-format and
dequantisation functions it uses): nothing in the product package imports or
runs this file.  float64 throughout.

Sources (page "TurboFieldfare - System design"):
  * Section "Why the runtime has this shape": the embedding and the language-
    model head share the same quantised weights (4-bit MLX affine, groups of
    64 with a BF16 scale and bias); the model ends with a final logit softcap
    of 30.0.
  * Section "Decode" (after the layer stack): the tied head either returns the
    argmax token directly (pure-greedy configuration) or writes the full
    logits vector for the sampler.

Readings where the pages are silent:
  * the softcap is cap * tanh(z / cap) with cap = 30 (the usual form of a
    logit softcap);
  * the head takes its input rows as given (any final norm is the caller's);
  * the greedy token is the argmax of the softcapped logits, ties to the
    lower token id;
  * the tied embedding of token v is row v of the dequantised matrix, rounded
    to bf16, with no scale (any embedding scale is the caller's);
  * the head's rows are independent, so head_logits works through them in
    blocks of rows to bound memory; each row's value is the same as with the
    whole matrix at once.
"""
from __future__ import annotations

import numpy as np

from oracle.moe_oracle import bf16_to_f64, dequantize, f64_to_bf16

SOFTCAP = 30.0
ROW_BLOCK = 4096


def softcap(z, cap: float = SOFTCAP) -> np.ndarray:
    """cap * tanh(z / cap), float64."""
    return cap * np.tanh(np.asarray(z, dtype=np.float64) / cap)


def head_logits(x_bits, head: dict, cap: float = SOFTCAP, rows=None) -> np.ndarray:
    """logits[t, v] = softcap((W x_t)[v]) for the head W (4-bit affine [V, H],
    dict q/s/b); float64 [T, V], or [T, len(rows)] for the given rows only."""
    x = bf16_to_f64(x_bits)
    idx = np.arange(head["q"].shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((x.shape[0], idx.size), dtype=np.float64)
    for b0 in range(0, idx.size, ROW_BLOCK):
        sel = idx[b0:b0 + ROW_BLOCK]
        w = dequantize(head["q"][sel], head["s"][sel], head["b"][sel], 4)
        out[:, b0:b0 + sel.size] = softcap(x @ w.T, cap)
    return out


def dense(x_bits, w: dict) -> np.ndarray:
    """y[t, n] = (W x_t)[n] for a dense 4-bit affine matrix W [N, K] (dict
    q/s/b, the format of the head and of the attention projections: page
    "TurboFieldfare - System design", section ".gturbo directory", stores the
    attention weights 4-bit affine, group 64, like the embedding); float64
    [T, N]."""
    x = bf16_to_f64(x_bits)
    out = np.full((x.shape[0], w["q"].shape[0]), np.nan)  # a row block left out stays visible
    for b0 in range(0, out.shape[1], ROW_BLOCK):
        sel = slice(b0, min(out.shape[1], b0 + ROW_BLOCK))
        out[:, sel] = x @ dequantize(w["q"][sel], w["s"][sel], w["b"][sel], 4).T
    return out


def greedy_token(logits) -> np.ndarray:
    """Index of the largest logit per row, the lowest index among equal
    maxima; int64 [T]."""
    lg = np.asarray(logits)
    out = np.empty(lg.shape[0], dtype=np.int64)
    for t in range(lg.shape[0]):
        m = lg[t].max()
        out[t] = int(np.flatnonzero(lg[t] == m)[0])
    return out


def embed(ids, head: dict) -> np.ndarray:
    """bf16 bits [n, H]: row ids[i] of the dequantised head, rounded to bf16."""
    ids = np.asarray(ids, dtype=np.int64)
    w = dequantize(head["q"][ids], head["s"][ids], head["b"][ids], 4)
    return f64_to_bf16(w)
