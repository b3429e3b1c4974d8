"""Pure-Python brute force of the MoE block for tiny layers.

Written independently of the numpy oracle: scalar loops over Python ints and
floats, codes pulled out of each packed word one at a time, the top-k found
by sorting all experts.  Only for tiny shapes (hidden <= 256); it is a pin
for the oracle, not a second oracle.
"""
from __future__ import annotations

import math
import struct


def bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def weight(words_row, s_row, b_row, bits: int, col: int) -> float:
    per_word = 32 // bits
    word = int(words_row[col // per_word])
    code = (word >> (bits * (col % per_word))) & ((1 << bits) - 1)
    g = col // 64
    return code * bf16(s_row[g]) + bf16(b_row[g])


def matvec(mat: dict, bits: int, vec) -> list:
    q, s, b = mat["q"], mat["s"], mat["b"]
    rows = len(q)
    cols = len(vec)
    out = []
    for r in range(rows):
        acc = 0.0
        for c in range(cols):
            acc += weight(q[r], s[r], b[r], bits, c) * vec[c]
        out.append(acc)
    return out


def gelu_tanh(z: float) -> float:
    return 0.5 * z * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z * z * z)))


def ffn(expert: dict, vec) -> list:
    g = matvec(expert["gate"], 4, vec)
    u = matvec(expert["up"], 4, vec)
    h = [gelu_tanh(a) * c for a, c in zip(g, u)]
    return matvec(expert["down"], 4, h)


def block(x_rows_bits, router: dict, experts: list, shared: dict, k: int, logit_bias=None):
    """Returns per token: (logits, ids, weights, y) as Python lists."""
    out = []
    for row in x_rows_bits:
        x = [bf16(v) for v in row]
        logits = matvec(router, 8, x)
        if logit_bias is not None:
            logits = [a + float(bb) for a, bb in zip(logits, logit_bias)]
        order = sorted(range(len(logits)), key=lambda e: (-logits[e], e))
        ids = order[:k]
        m = max(logits[e] for e in ids)
        ex = [math.exp(logits[e] - m) for e in ids]
        tot = sum(ex)
        w = [v / tot for v in ex]
        y = [0.0] * len(x)
        for j, e in enumerate(ids):
            o = ffn(experts[e], x)
            y = [a + w[j] * c for a, c in zip(y, o)]
        o_sh = ffn(shared, x)
        y = [a + c for a, c in zip(y, o_sh)]
        out.append((logits, ids, w, y))
    return out
