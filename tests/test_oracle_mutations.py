"""Plant plausible mistakes in a copy of the oracle; some pin must fail.

Each mutation is a textual edit of the oracle's source, executed as a fresh
module on the CPU.  The real oracle is never modified.
"""
import importlib.util
import os
import types

import pytest

import oracle_pins

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
ORACLE_SRC = os.path.join(ORACLE_DIR, "moe_oracle.py")
HEAD_SRC = os.path.join(ORACLE_DIR, "head_oracle.py")

MUTATIONS = {
    "reversed_code_order": ("(w >> np.uint32(bits * pos))", "(w >> np.uint32(bits * (per - 1 - pos)))"),
    "dropped_bias": ("return q * s_full + b_full", "return q * s_full"),
    "wrong_group_map": ("s_full = np.repeat(s, GROUP, axis=1)", "s_full = np.tile(s, (1, GROUP))"),
    "tie_to_higher_id": ("np.lexsort((order_ids, -lg", "np.lexsort((-order_ids, -lg"),
    "ascending_topk": ("np.lexsort((order_ids, -lg[row]", "np.lexsort((order_ids, lg[row]"),
    "gelu_cubic_term": ("0.044715 * z ** 3", "0.044715 * z ** 2"),
    "gelu_sign": ("(1.0 + np.tanh(", "(1.0 - np.tanh("),
    "dropped_shared": ("    y += shared_out\n", "    pass\n"),
    "unweighted_routes": ("y += weights[:, j:j + 1] * outs[:, j]", "y += outs[:, j]"),
    "softmax_perturbed": ("e = np.exp(lg - m)", "e = np.exp(lg - m) + 0.0 * m + 1e-3"),
    "gate_up_swapped_in_geglu": ("return gelu_tanh(g) * u", "return gelu_tanh(u) * g"),
    "unstable_sort": ("for p, e in enumerate(flat):", "for p, e in reversed(list(enumerate(flat))):"),
    "rms_without_eps": ("np.mean(h * h, axis=1, keepdims=True) + eps", "np.mean(h * h, axis=1, keepdims=True)"),
    "bf16_truncation": ("keep = keep + up.astype(np.uint64)", "keep = keep"),
    "router_scale_not_normalised": ("bf16_to_f64(router_scale)[None, :] / np.sqrt(x.shape[1])", "bf16_to_f64(router_scale)[None, :]"),
    "router_scale_transposed": ("bf16_to_f64(router_scale)[None, :]", "bf16_to_f64(router_scale)[::-1][None, :]"),
    "per_expert_scale_dropped": ("w = w * np.asarray(per_expert_scale, dtype=np.float64)[np.asarray(ids)]", "w = w"),
    "tail_scalar_dropped": ("return f64_to_bf16(float(np.float32(layer_scalar)) * bf16_to_f64(s))", "return s"),
    "tail_norm_weight_dropped": ("return y / r * bf16_to_f64(post_norm_bits)[None, :]", "return y / r"),
    "tail_norm_sum_not_mean": ("np.sqrt(np.mean(y * y, axis=1, keepdims=True) + eps)", "np.sqrt(np.sum(y * y, axis=1, keepdims=True) + eps)"),
    "tail_eps_dropped": ("np.sqrt(np.mean(y * y, axis=1, keepdims=True) + eps)", "np.sqrt(np.mean(y * y, axis=1, keepdims=True))"),
    "tail_residual_dropped": ("s = f64_to_bf16(bf16_to_f64(h_bits) + bf16_to_f64(z))", "s = f64_to_bf16(bf16_to_f64(z))"),
    "router_bias_dropped": ("logits = logits + np.asarray(logit_bias", "logits = logits + 0 * np.asarray(logit_bias"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    with open(ORACLE_SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    src = src.replace(old, new, 1)
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


# a planted mistake may divide by zero on the pins' all-zero rows (numpy warns; the pins still fail it)
@pytest.mark.filterwarnings("ignore:invalid value encountered:RuntimeWarning")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name):
    mod = _mutant(name)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, ZeroDivisionError, FloatingPointError, IndexError) as exc:
            caught.append((pin.__name__, type(exc).__name__))
    assert caught, f"no pin caught mutation {name}"


HEAD_MUTATIONS = {
    "softcap_outer_cap_dropped": ("return cap * np.tanh(np.asarray(z, dtype=np.float64) / cap)",
                                  "return np.tanh(np.asarray(z, dtype=np.float64) / cap)"),
    "softcap_inner_unscaled": ("return cap * np.tanh(np.asarray(z, dtype=np.float64) / cap)",
                               "return cap * np.tanh(np.asarray(z, dtype=np.float64))"),
    "softcap_dropped": ("out[:, b0:b0 + sel.size] = softcap(x @ w.T, cap)", "out[:, b0:b0 + sel.size] = x @ w.T"),
    "greedy_ties_to_higher": ("out[t] = int(np.flatnonzero(lg[t] == m)[0])", "out[t] = int(np.flatnonzero(lg[t] == m)[-1])"),
    "greedy_argmin": ("m = lg[t].max()", "m = lg[t].min()"),
    "row_block_short": ("sel = idx[b0:b0 + ROW_BLOCK]", "sel = idx[b0:b0 + ROW_BLOCK - 1]"),
    "dense_block_short": ("sel = slice(b0, min(out.shape[1], b0 + ROW_BLOCK))",
                          "sel = slice(b0, min(out.shape[1], b0 + ROW_BLOCK - 1))"),
    "dense_scale_for_bias": ("w[\"s\"][sel], w[\"b\"][sel], 4).T", "w[\"s\"][sel], w[\"s\"][sel], 4).T"),
    "dense_rows_reversed": ("out[:, sel] = x @ dequantize", "out[:, sel][:, ::-1] = x @ dequantize"),
    "embed_unrounded_rows_shifted": ("w = dequantize(head[\"q\"][ids], head[\"s\"][ids], head[\"b\"][ids], 4)",
                                     "w = dequantize(head[\"q\"][ids], head[\"s\"][ids[::-1]], head[\"b\"][ids], 4)"),
}


@pytest.mark.parametrize("name", sorted(HEAD_MUTATIONS))
def test_head_mutation_is_caught(name):
    import head_pins
    old, new = HEAD_MUTATIONS[name]
    with open(HEAD_SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mod = types.ModuleType(f"head_mutant_{name}")
    exec(compile(src.replace(old, new, 1), f"<mutant {name}>", "exec"), mod.__dict__)
    caught = []
    for pin in head_pins.ALL_HEAD_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, ZeroDivisionError, FloatingPointError, IndexError) as exc:
            caught.append((pin.__name__, type(exc).__name__))
    assert caught, f"no pin caught mutation {name}"
