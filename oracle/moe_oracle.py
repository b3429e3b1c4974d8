"""Plain CPU oracle of the 4-bit/8-bit affine mixture-of-experts FFN block.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, links or
runs this file; only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may call it.  It shares no code with the CUDA
path and is written for checking by eye, not for speed: every value is
float64, every quantised weight is expanded to a dense float64 matrix first,
and sums are taken in the order the definition states (a library matmul is
used for plain dot products).

Sources (page "TurboFieldfare - System design", by section):
  * Quantisation format, section "Why the runtime has this shape": MLX affine
    quantisation, groups of 64 weights along the input axis, one BF16 scale
    and one BF16 bias per group, w = q * scale + bias.  Router projections
    use 8-bit codes, shared and routed experts use 4-bit codes.  The pages do
    not give the bit order of the packed codes; this oracle reads code i of a
    row from bits 4*(i % 8) of little-endian uint32 word i // 8 (4-bit) or
    bits 8*(i % 4) of word i // 4 (8-bit).
  * Same section: 128 routed experts, 8 selected per token; a dense shared
    expert is a separate branch whose output is added with no routing weight;
    the router logits have no softcap; shared and routed FFNs run in parallel
    on the same input.
  * Section "Decode", router description: normalise, scale, project with the
    8-bit affine weights, take the 8 highest logits, softmax over those 8,
    times the selected experts' learned scales.  The block here receives an
    already normalised input x; the router projects x * router_scale /
    sqrt(H) when a learned router scale (one value per input feature) is
    given, else x; the routing weights are softmax(selected logits) *
    per_expert_scale[id] when per-expert scales are given, else the softmax
    alone (+ an optional per-expert logit offset used by the skewed
    workloads).
  * Section "Metal execution": the routed kernels fuse affine decode, GeGLU
    and the weighted reduction over the selected experts.  GeGLU here is
    h = gelu_tanh(W_gate x) * (W_up x), out = W_down h (Gemma's gated FFN;
    gelu_tanh from Hendrycks & Gimpel 2016, tanh form).
  * Section "Prefill": token/expert pairs of a chunk (at most 128 rows) are
    grouped per expert; the grouping is a stable counting sort of the pair
    index t*k + j by expert id.

Readings where the pages are silent:
  * top-k ties go to the lower expert id, and the k ids are returned in
    order of descending logit (ties: ascending id);
  * the softmax weights are computed in float64 (the pages return FP16);
  * y = sum_j w_j * o_j (j in selection order) + o_shared, float64; the
    block's bf16 output is the round-to-nearest-even of that value;
  * stacked layers: x_l = bf16(rmsnorm_no_scale(h_l)), eps = 1e-6,
    h_{l+1} = bf16(h_l + bf16(y_l));
  * the layer tail (section "Decode", cb2 phase: after the combine, the
    post-FFN norms, the residual and a learned layer scalar), when a layer
    has one: one RMS norm with a learned per-feature weight g on the combined
    output y (eps 1e-6), then the residual add, then the scalar lambda:
    h_{l+1} = bf16(lambda * bf16(h_l + bf16(g * y / rms(y)))).
"""
from __future__ import annotations

import numpy as np

GROUP = 64
RMS_EPS = 1e-6


# ------------------------------------------------------------- number format
def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(v) -> np.ndarray:
    """float64 -> bf16 bit patterns, one rounding to nearest (ties to even).

    Done exactly: the float64 is split at bf16 precision with integer
    arithmetic on its bit pattern (finite inputs, normal range)."""
    v = np.asarray(v, dtype=np.float64)
    bits = v.view(np.uint64)
    sign = (bits >> np.uint64(63)).astype(np.uint64)
    mag = bits & np.uint64(0x7FFFFFFFFFFFFFFF)
    # float64 has 52 fraction bits, bf16 has 7: drop 45 bits with RNE.
    drop = np.uint64(45)
    keep = mag >> drop
    rem = mag & np.uint64((1 << 45) - 1)
    half = np.uint64(1 << 44)
    up = (rem > half) | ((rem == half) & ((keep & np.uint64(1)) == np.uint64(1)))
    keep = keep + up.astype(np.uint64)
    # keep = float64 exponent (11 bits) + 7 fraction bits; rebias 1023 -> 127
    exp64 = (keep >> np.uint64(7)).astype(np.int64)
    frac = (keep & np.uint64(0x7F)).astype(np.int64)
    exp16 = exp64 - 1023 + 127
    zero = mag == 0
    if np.any(~zero & ((exp16 <= 0) | (exp16 >= 255))):
        raise ValueError("value outside the normal bf16 range")
    out = (sign.astype(np.int64) << 15) | (np.clip(exp16, 0, 255) << 7) | frac
    out = np.where(zero, sign.astype(np.int64) << 15, out)
    return out.astype(np.uint16)


# ------------------------------------------------------------- dequantisation
def unpack_codes(words, bits: int) -> np.ndarray:
    """Packed little-endian uint32 words [N, K*bits/32] -> integer codes [N, K].

    Code i of a row sits at bits (bits * (i % (32/bits))) of word
    i // (32/bits): lowest code in the lowest bits."""
    w = np.asarray(words, dtype=np.uint32)
    per = 32 // bits
    mask = (1 << bits) - 1
    n, nw = w.shape
    codes = np.empty((n, nw * per), dtype=np.int64)
    for pos in range(per):
        codes[:, pos::per] = (w >> np.uint32(bits * pos)) & np.uint32(mask)
    return codes


def dequantize(words, scale_bits, bias_bits, bits: int) -> np.ndarray:
    """w[n, k] = q[n, k] * scale[n, k // 64] + bias[n, k // 64] in float64."""
    q = unpack_codes(words, bits).astype(np.float64)
    s = bf16_to_f64(scale_bits)
    b = bf16_to_f64(bias_bits)
    n, k = q.shape
    if s.shape != (n, k // GROUP) or b.shape != (n, k // GROUP):
        raise ValueError("scale/bias shape does not match [N, K/64]")
    s_full = np.repeat(s, GROUP, axis=1)
    b_full = np.repeat(b, GROUP, axis=1)
    return q * s_full + b_full


# ------------------------------------------------------------- router
def router_logits(x_bits, router: dict, logit_bias=None, router_scale=None) -> np.ndarray:
    """logits[t, e] = sum_k W_r[e, k] x'[t, k] (+ offset[e]); float64 [T, E].

    x' = x, or x * router_scale / sqrt(H) with router_scale bf16 bits [H]."""
    x = bf16_to_f64(x_bits)
    if router_scale is not None:
        x = x * bf16_to_f64(router_scale)[None, :] / np.sqrt(x.shape[1])
    w_r = dequantize(router["q"], router["s"], router["b"], 8)
    logits = x @ w_r.T
    if logit_bias is not None:
        logits = logits + np.asarray(logit_bias, dtype=np.float64)[None, :]
    return logits


def select_top_k(logits, k: int) -> np.ndarray:
    """Indices of the k largest entries per row: descending value, ties to the
    lower index.  Works on whatever precision `logits` is given in."""
    lg = np.asarray(logits)
    t, e = lg.shape
    if not 1 <= k <= e:
        raise ValueError("k out of range")
    if not np.all(np.isfinite(lg)):
        raise ValueError("non-finite logits")
    ids = np.empty((t, k), dtype=np.int64)
    order_ids = np.arange(e)
    for row in range(t):
        # lexsort: last key is primary -> (-value, id)
        order = np.lexsort((order_ids, -lg[row].astype(np.float64)))
        ids[row] = order[:k]
    return ids


def routing_weights(logits, ids, per_expert_scale=None) -> np.ndarray:
    """softmax over the selected logits of each token, float64 [T, k], times
    per_expert_scale[id] of each selected expert when given."""
    lg = np.take_along_axis(np.asarray(logits, dtype=np.float64), np.asarray(ids), axis=1)
    m = lg.max(axis=1, keepdims=True)
    e = np.exp(lg - m)
    w = e / e.sum(axis=1, keepdims=True)
    if per_expert_scale is not None:
        w = w * np.asarray(per_expert_scale, dtype=np.float64)[np.asarray(ids)]
    return w


# ------------------------------------------------------------- experts
def gelu_tanh(z):
    """0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))."""
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (z + 0.044715 * z ** 3)))


def dense_expert(expert: dict) -> dict:
    """Dequantised float64 gate [I,H], up [I,H], down [H,I] of one expert."""
    return {m: dequantize(expert[m]["q"], expert[m]["s"], expert[m]["b"], 4) for m in ("gate", "up", "down")}


def expert_hidden(x, dense: dict) -> np.ndarray:
    """h = gelu_tanh(W_gate x) * (W_up x) for rows x [n, H] (float64)."""
    g = x @ dense["gate"].T
    u = x @ dense["up"].T
    return gelu_tanh(g) * u


def expert_ffn(x, dense: dict) -> np.ndarray:
    """out = W_down (gelu_tanh(W_gate x) * W_up x) for rows x [n, H]."""
    return expert_hidden(x, dense) @ dense["down"].T


# ------------------------------------------------------------- grouping
def route_sort(ids, n_experts: int):
    """Stable counting sort of the pairs p = t*k + j by expert id.

    Returns counts [E], offsets [E+1] (exclusive prefix sums of counts),
    perm [T*k] (pair index at each sorted position) and pos [T*k] (sorted
    position of each pair; the inverse of perm)."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= n_experts):
        raise ValueError("expert id out of range")
    counts = np.zeros(n_experts, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    for e in range(n_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    perm = np.empty(flat.size, dtype=np.int64)
    pos = np.empty(flat.size, dtype=np.int64)
    for p, e in enumerate(flat):
        perm[fill[e]] = p
        pos[p] = fill[e]
        fill[e] += 1
    return counts, offsets, perm, pos


# ------------------------------------------------------------- block
def moe_block(x_bits, router: dict, get_expert, shared: dict, k: int, logit_bias=None, ids=None,
              router_scale=None, per_expert_scale=None):
    """One MoE FFN block on bf16 hidden rows x [T, H].

    get_expert(e) -> expert dict (q/s/b of gate, up, down); shared likewise.
    If `ids` is given (teacher forcing), the selection is taken from it and
    only the weights/outputs are computed here.

    Returns dict: logits [T,E], ids [T,k], weights [T,k], y [T,H] float64,
    y_bf16 bits [T,H]."""
    logits = router_logits(x_bits, router, logit_bias, router_scale)
    if ids is None:
        ids = select_top_k(logits, k)
    ids = np.asarray(ids, dtype=np.int64)
    weights = routing_weights(logits, ids, per_expert_scale)
    y = expert_mix(x_bits, ids, weights, get_expert, shared)
    return {"logits": logits, "ids": ids, "weights": weights, "y": y, "y_bf16": f64_to_bf16(y)}


def expert_mix(x_bits, ids, weights, get_expert, shared=None) -> np.ndarray:
    """y[t] = sum_j weights[t, j] * FFN_{ids[t, j]}(x_t)  (+ FFN_shared(x_t)).

    Sum in selection order j, then the shared term (omitted if shared is
    None).  Each distinct expert is expanded once.  float64 [T, H]."""
    x = bf16_to_f64(x_bits)
    ids = np.asarray(ids, dtype=np.int64)
    weights = np.asarray(weights, dtype=np.float64)
    t_count, k = ids.shape
    h_dim = x.shape[1]
    outs = np.zeros((t_count, k, h_dim), dtype=np.float64)
    for e in np.unique(ids):
        rows, cols = np.nonzero(ids == e)
        dense = dense_expert(get_expert(int(e)))
        outs[rows, cols] = expert_ffn(x[rows], dense)
    y = np.zeros((t_count, h_dim), dtype=np.float64)
    for j in range(k):
        y += weights[:, j:j + 1] * outs[:, j]
    if shared is not None:
        shared_out = expert_ffn(x, dense_expert(shared))
        y += shared_out
    return y


def rmsnorm_no_scale(h_bits, eps: float = RMS_EPS) -> np.ndarray:
    """bf16(h / sqrt(mean(h^2) + eps)) per row; returns bf16 bits."""
    h = bf16_to_f64(h_bits)
    r = np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps)
    return f64_to_bf16(h / r)


def residual_add(h_bits, y_bf16_bits) -> np.ndarray:
    """bf16(h + y) with y the block's bf16 output."""
    return f64_to_bf16(bf16_to_f64(h_bits) + bf16_to_f64(y_bf16_bits))


def post_ffn_norm(y_bits, post_norm_bits, eps: float = RMS_EPS) -> np.ndarray:
    """z = y / sqrt(mean(y^2) + eps) * g per row, float64 [T, H]; y the block's
    bf16 output, g the learned norm weight (bf16 bits [H])."""
    y = bf16_to_f64(y_bits)
    r = np.sqrt(np.mean(y * y, axis=1, keepdims=True) + eps)
    return y / r * bf16_to_f64(post_norm_bits)[None, :]


def layer_tail(h_bits, y_bits, post_norm_bits=None, layer_scalar=None) -> np.ndarray:
    """The layer tail after the combine (section "Decode", cb2 phase): post-FFN
    norm, residual, layer scalar.  Each step's result is a bf16 tensor:
    z = bf16(post_ffn_norm(y)) (z = y without a norm weight),
    s = bf16(h + z), h' = bf16(layer_scalar * s) (h' = s without a scalar).
    Returns bf16 bits [T, H]."""
    z = y_bits if post_norm_bits is None else f64_to_bf16(post_ffn_norm(y_bits, post_norm_bits))
    s = f64_to_bf16(bf16_to_f64(h_bits) + bf16_to_f64(z))
    if layer_scalar is None:
        return s
    return f64_to_bf16(float(np.float32(layer_scalar)) * bf16_to_f64(s))


def stack_layer(h_bits, router, get_expert, shared, k: int, logit_bias=None, ids=None):
    """One layer of a stack: x = rmsnorm_no_scale(h); y = block(x); h' = h + y."""
    x_bits = rmsnorm_no_scale(h_bits)
    out = moe_block(x_bits, router, get_expert, shared, k, logit_bias, ids)
    out["x_bits"] = x_bits
    out["h_next"] = residual_add(h_bits, out["y_bf16"])
    return out
