"""Seeded synthetic inputs shared by the oracle tests and the CUDA path.

This module draws random numbers and lays them out; it computes nothing of the
MoE block itself.  Everything is a pure function of integer seeds, so the host
(numpy) and the device (``synth/gpu_fill.cu``) produce identical bits.

Counter-based generator
-----------------------
SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; finaliser constants of Stafford's "Mix13"):

    mix64(z):  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9
               z ^= z >> 27; z *= 0x94D049BB133111EB
               z ^= z >> 31
    draw(k, i) = mix64(k + (i + 1) * 0x9E3779B97F4A7C15)     (mod 2**64)

A stream key is folded from a tuple of small integers:
    k = 0x243F6A8885A308D3; for c in tuple: k = mix64(k ^ ((c + 1) * golden))

Derived draws
-------------
* 32-bit words: word 2i is the low half of draw(k, i), word 2i+1 the high half.
  Uniform words give uniform nibbles (4-bit codes) and uniform bytes (8-bit
  codes) in every position.
* U[0,1): (draw >> 11) * 2**-53.
* N(0,1): Box-Muller on consecutive draws (2j, 2j+1), host libm, float64.
* bf16: round to float32 (nearest even), then to bf16 (nearest even).

Synthetic weight recipe (the five workload descriptions of the MoE block)
-------------------------------------------------------------------------
* router [E, H], 8-bit: codes uniform 0..255; scale = bf16(U(0.5,1.5) /
  (128*sqrt(H))) per group of 64; bias = bf16(-128 * scale).
* expert matrices (gate/up [I, H], down [H, I]), 4-bit: codes uniform 0..15;
  scale = bf16(U(0.5,1.5) / (8*sqrt(K))) with K the input width;
  bias = bf16(-8*scale + 0.01*scale*N(0,1)), from the bf16-rounded scale.
* Zipf logit offsets: offset_e = 2 * r_e**-1.1, r_e = 1 + pi(e), pi a
  Fisher-Yates permutation of 0..E-1 keyed by the layer.
* hidden states: N(0,1) rows, optionally scaled to unit root-mean-square
  before the bf16 rounding (an input distribution, not a model step).
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
KEY0 = 0x243F6A8885A308D3
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB

# stream tags
STREAM_WEIGHTS = 1
STREAM_INPUT = 2
STREAM_ZIPF = 3
STREAM_ROUTER_SCALES = 4  # learned router scales of the optional-scale tests
STREAM_LAYER_TAIL = 5     # post-FFN norm weight and layer scalar of the layer-tail tests
# weight tuple fields
ROUTER_ID = 2000          # "expert" slot of the router projection
SHARED_ID = 1000          # "expert" slot of the dense shared expert
HEAD_ID = 3000            # "expert" slot of the tied head / embedding
MAT_GATE, MAT_UP, MAT_DOWN, MAT_ROUTER, MAT_HEAD = 0, 1, 2, 3, 4
FIELD_Q, FIELD_S, FIELD_B = 0, 1, 2

GROUP = 64


# ---------------------------------------------------------------- SplitMix64
def mix64_int(z: int) -> int:
    z &= MASK64
    z ^= z >> 30
    z = (z * M1) & MASK64
    z ^= z >> 27
    z = (z * M2) & MASK64
    z ^= z >> 31
    return z


def stream_key(*components: int) -> int:
    k = KEY0
    for c in components:
        k = mix64_int(k ^ (((int(c) + 1) * GOLDEN) & MASK64))
    return k


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(M1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(M2)
    z ^= z >> np.uint64(31)
    return z


def draws(key: int, n: int, start: int = 0) -> np.ndarray:
    """draw(key, i) for i in [start, start+n) as uint64."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + i * np.uint64(GOLDEN)
        return _mix64_np(z)


def words(key: int, n: int) -> np.ndarray:
    """n uint32 words; word 2i / 2i+1 = low / high half of draw(key, i)."""
    d = draws(key, (n + 1) // 2)
    w = np.empty(2 * d.size, dtype=np.uint32)
    w[0::2] = (d & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    w[1::2] = (d >> np.uint64(32)).astype(np.uint32)
    return w[:n]


def uniform(key: int, n: int) -> np.ndarray:
    return (draws(key, n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def normal(key: int, n: int) -> np.ndarray:
    m = (n + 1) // 2
    d = draws(key, 2 * m)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n]


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bf16 (RNE); returns uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- weights
def weight_key(layer_seed: int, expert: int, matrix: int, field: int) -> int:
    return stream_key(STREAM_WEIGHTS, layer_seed, expert, matrix, field)


def qmat_words(n_rows: int, k: int, bits: int) -> int:
    return n_rows * k * bits // 32


def expert_scale_bias(layer_seed: int, expert: int, matrix: int, n_rows: int, k: int):
    """bf16 scale and bias bit arrays [n_rows, k/64] of one 4-bit matrix."""
    ng = k // GROUP
    u = uniform(weight_key(layer_seed, expert, matrix, FIELD_S), n_rows * ng)
    s_bits = to_bf16_bits((0.5 + u) / (8.0 * np.sqrt(float(k))))
    s = bf16_bits_to_f64(s_bits)
    z = normal(weight_key(layer_seed, expert, matrix, FIELD_B), n_rows * ng)
    b_bits = to_bf16_bits(-8.0 * s + (0.01 * s) * z)
    return s_bits.reshape(n_rows, ng), b_bits.reshape(n_rows, ng)


def expert_matrix(layer_seed: int, expert: int, matrix: int, hidden: int, inter: int):
    """(q_words uint32 [N, K/8], scale bits, bias bits) of gate/up/down."""
    n_rows, k = (inter, hidden) if matrix in (MAT_GATE, MAT_UP) else (hidden, inter)
    q = words(weight_key(layer_seed, expert, matrix, FIELD_Q), qmat_words(n_rows, k, 4))
    s, b = expert_scale_bias(layer_seed, expert, matrix, n_rows, k)
    return q.reshape(n_rows, k // 8), s, b


def expert_weights(layer_seed: int, expert: int, hidden: int, inter: int) -> dict:
    """All three matrices of routed expert `expert` (or SHARED_ID)."""
    out = {}
    for name, m in (("gate", MAT_GATE), ("up", MAT_UP), ("down", MAT_DOWN)):
        q, s, b = expert_matrix(layer_seed, expert, m, hidden, inter)
        out[name] = {"q": q, "s": s, "b": b}
    return out


def router_weights(layer_seed: int, n_experts: int, hidden: int) -> dict:
    ng = hidden // GROUP
    q = words(weight_key(layer_seed, ROUTER_ID, MAT_ROUTER, FIELD_Q), qmat_words(n_experts, hidden, 8))
    u = uniform(weight_key(layer_seed, ROUTER_ID, MAT_ROUTER, FIELD_S), n_experts * ng)
    s_bits = to_bf16_bits((0.5 + u) / (128.0 * np.sqrt(float(hidden))))
    b_bits = to_bf16_bits(-128.0 * bf16_bits_to_f64(s_bits))
    return {"q": q.reshape(n_experts, hidden // 4), "s": s_bits.reshape(n_experts, ng),
            "b": b_bits.reshape(n_experts, ng)}


def head_weights(seed: int, vocab: int, hidden: int, rows=None) -> dict:
    """The tied 4-bit head [vocab, hidden] (the embedding shares it): codes
    uniform 0..15, scale bf16(U(0.5, 1.5) / (8 sqrt(H))), bias
    bf16(-8 scale + 0.01 scale N(0, 1)), like the experts.  With `rows`, only
    those rows (the same values as in the whole matrix)."""
    ng, nw = hidden // GROUP, hidden // 8
    idx = np.arange(vocab) if rows is None else np.asarray(rows, dtype=np.int64)
    kq, ks, kb = (weight_key(seed, HEAD_ID, MAT_HEAD, f) for f in (FIELD_Q, FIELD_S, FIELD_B))
    q = np.empty((idx.size, nw), dtype=np.uint32)
    u = np.empty((idx.size, ng), dtype=np.float64)
    z = np.empty((idx.size, ng), dtype=np.float64)
    if rows is None:
        q[:] = words(kq, vocab * nw).reshape(vocab, nw)
        u[:] = uniform(ks, vocab * ng).reshape(vocab, ng)
        z[:] = normal(kb, vocab * ng).reshape(vocab, ng)
    else:
        for i, r in enumerate(idx):
            d = draws(kq, nw // 2, int(r) * (nw // 2))      # word 2j/2j+1 = halves of draw j
            q[i, 0::2] = (d & np.uint64(0xFFFFFFFF)).astype(np.uint32)
            q[i, 1::2] = (d >> np.uint64(32)).astype(np.uint32)
            u[i] = (draws(ks, ng, int(r) * ng) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
            z[i] = _normal_at(kb, ng, int(r) * ng)
    s_bits = to_bf16_bits((0.5 + u) / (8.0 * np.sqrt(float(hidden))))
    b_bits = to_bf16_bits(-8.0 * bf16_bits_to_f64(s_bits) + (0.01 * bf16_bits_to_f64(s_bits)) * z)
    return {"q": q, "s": s_bits, "b": b_bits}


def _normal_at(key: int, n: int, start: int) -> np.ndarray:
    """normal(key, start + n)[start:] for even start and n (whole Box-Muller pairs)."""
    d = draws(key, n, start)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(n, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z


def zipf_logit_bias(layer_seed: int, n_experts: int, s: float = 1.1, top: float = 2.0) -> np.ndarray:
    """float32 [E] per-expert offsets top * rank**-s, ranks a keyed permutation."""
    d = draws(stream_key(STREAM_ZIPF, layer_seed), n_experts)
    perm = list(range(n_experts))
    for step, i in enumerate(range(n_experts - 1, 0, -1)):
        j = int(d[step] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    rank = 1.0 + np.asarray(perm, dtype=np.float64)
    return (top * rank ** (-s)).astype(np.float32)


def router_scales(layer_seed: int, n_experts: int, hidden: int):
    """Learned router scales for the tests of that option: router_scale bf16
    bits [H] = bf16(sqrt(H) * U(0.5, 1.5)) (so x * scale / sqrt(H) stays near
    x) and per_expert_scale float32 [E] = U(0.5, 1.5)."""
    u = uniform(stream_key(STREAM_ROUTER_SCALES, layer_seed, 0), hidden)
    v = uniform(stream_key(STREAM_ROUTER_SCALES, layer_seed, 1), n_experts)
    return to_bf16_bits(np.sqrt(hidden) * (0.5 + u)), (0.5 + v).astype(np.float32)


def layer_tail(layer_seed: int, hidden: int):
    """Layer-tail weights for the tests of that option: post-FFN norm weight
    bf16 bits [H] = bf16(U(0.5, 1.5)) and the layer scalar float32 U(0.5, 1.5)."""
    u = uniform(stream_key(STREAM_LAYER_TAIL, layer_seed, 0), hidden)
    v = uniform(stream_key(STREAM_LAYER_TAIL, layer_seed, 1), 1)
    return to_bf16_bits(0.5 + u), np.float32(0.5 + v[0])


# ---------------------------------------------------------------- inputs
def hidden_states(input_seed: int, chunk: int, n_tokens: int, hidden: int, rms_normalize: bool) -> np.ndarray:
    """bf16 bits [T, H]: N(0,1) rows, optionally scaled to unit RMS first."""
    z = normal(stream_key(STREAM_INPUT, input_seed, chunk), n_tokens * hidden).reshape(n_tokens, hidden)
    if rms_normalize:
        z = z / np.sqrt(np.mean(z * z, axis=1, keepdims=True))
    return to_bf16_bits(z)


# ---------------------------------------------------------------- layout
def align_up(v: int, a: int) -> int:
    return (v + a - 1) // a * a


def blob_layout(hidden: int, inter: int, page: int = 16384) -> dict:
    """Byte offsets of the nine sub-tensors of one expert blob.

    Order gate(q,s,b), up(q,s,b), down(q,s,b); each sub-tensor starts on a
    256-byte boundary and the blob stride is rounded up to `page` bytes
    (fixed-stride, page-aligned expert blobs)."""
    off = 0
    out = {}
    for name, (n, k) in (("gate", (inter, hidden)), ("up", (inter, hidden)), ("down", (hidden, inter))):
        for field, size in (("q", n * k // 2), ("s", n * (k // GROUP) * 2), ("b", n * (k // GROUP) * 2)):
            out[f"{name}_{field}"] = off
            off = align_up(off + size, 256)
    out["bytes"] = off
    out["stride"] = align_up(off, page)
    return out


def router_layout(n_experts: int, hidden: int) -> dict:
    q = n_experts * hidden
    s = n_experts * (hidden // GROUP) * 2
    out = {"q": 0, "s": align_up(q, 256)}
    out["b"] = align_up(out["s"] + s, 256)
    out["bytes"] = align_up(out["b"] + s, 256)
    return out
