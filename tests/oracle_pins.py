"""Pins that tie the oracle to facts outside itself.

Each pin takes the oracle module as an argument so that the mutation test can
run the same pins against a copy of the oracle with a planted mistake.  A pin
raises AssertionError (or the oracle's own ValueError) when it fails.

What pins what:
  pin_layout_sizes     byte sizes printed on the pages (expert slot and the
                       routed-expert file total) <- code width, scale/bias
                       type, group size, matrix shapes
  pin_dequant_golden   hand-worked dequantisation examples (fixtures)
  pin_bf16_rounding    bf16 rounding against torch's float32->bf16 and
                       hand-picked ties
  pin_gelu             closed forms + torch's tanh-GELU
  pin_topk             brute-force sort, exact ties, k = E
  pin_softmax_full     k = E reduces to the textbook softmax (scipy)
  pin_integer_layer    unit scale / zero bias -> exact integer arithmetic
  pin_brute_force      whole block vs a pure-Python scalar brute force
  pin_invariants       sum of weights, zero expert, expert relabelling,
                       batch invariance, exact doubling of W_down
  pin_route_sort       stable counting sort vs numpy's stable argsort
  pin_rmsnorm          closed-form rows
  pin_router_scales    scaled router vs brute force on exactly scaled rows,
                       per-expert scales on the softmax, zero / doubled scales
  pin_layer_tail       closed forms, eps on small rows, a plain-Python brute force
                       with hand rounding, zero rows and weights
"""
from __future__ import annotations

import math
import os

import numpy as np

import _brute
from synth import gen

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- format
def pin_layout_sizes(o):
    sizes = {k: int(v) for k, v in _read_table("layout_sizes.txt")}
    hidden, inter = 2816, 704
    total = 0
    for n, k in ((inter, hidden), (inter, hidden), (hidden, inter)):
        q = np.zeros((n, k // 8), dtype=np.uint32)
        s = np.zeros((n, k // 64), dtype=np.uint16)
        b = np.zeros((n, k // 64), dtype=np.uint16)
        w = o.dequantize(q, s, b, 4)        # the oracle accepts exactly these shapes
        assert w.shape == (n, k)
        total += q.nbytes + s.nbytes + b.nbytes
    page = sizes["page_bytes"]
    slot = (total + page - 1) // page * page
    assert slot == sizes["slot_bytes"], (total, slot)
    assert slot * sizes["layers"] * sizes["experts_per_layer"] == sizes["expert_files_bytes"]
    assert gen.blob_layout(hidden, inter)["stride"] == sizes["slot_bytes"]
    # a group of 32 must be rejected (scale shape mismatch)
    try:
        o.dequantize(np.zeros((4, 16), np.uint32), np.zeros((4, 4), np.uint16), np.zeros((4, 4), np.uint16), 4)
    except ValueError:
        pass
    else:
        raise AssertionError("group-32 scale shape accepted")


def _bf16_bits_exact(v: float) -> int:
    f = np.array([v], dtype=np.float32)
    bits = int(f.view(np.uint32)[0])
    assert bits & 0xFFFF == 0, f"{v} is not a bf16 value"
    return bits >> 16


def pin_dequant_golden(o):
    for row in _read_table("dequant_examples.txt"):
        bits, word, scale, bias = int(row[0]), int(row[1], 16), float(row[2]), float(row[3])
        codes = [int(c) for c in row[4].split(",")]
        want = [float(c) for c in row[5].split(",")]
        per = 32 // bits
        n_words = 64 // per                       # one group of 64 weights
        words = np.full((1, n_words), word, dtype=np.uint32)
        s = np.array([[_bf16_bits_exact(scale)]], dtype=np.uint16)
        b = np.array([[_bf16_bits_exact(bias)]], dtype=np.uint16)
        got_codes = o.unpack_codes(words, bits)[0, :per].tolist()
        assert got_codes == codes, (row, got_codes)
        got = o.dequantize(words, s, b, bits)[0]
        assert got[:per].tolist() == want, (row, got[:per])
        assert got.tolist() == want * n_words


def pin_bf16_rounding(o):
    import torch
    # hand ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert int(o.f64_to_bf16(np.array([1.0 + 2.0 ** -8]))[0]) == 0x3F80
    assert int(o.f64_to_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0]) == 0x3F82
    assert int(o.f64_to_bf16(np.array([-(1.0 + 2.0 ** -8 + 2.0 ** -40)]))[0]) == 0xBF81
    assert int(o.f64_to_bf16(np.array([0.0]))[0]) == 0
    # float32-exact values: a single rounding equals torch's conversion
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = o.f64_to_bf16(v.astype(np.float64))
    assert np.array_equal(got, ref)
    # round trip
    assert np.array_equal(o.f64_to_bf16(o.bf16_to_f64(got)), got)


def pin_gelu(o):
    import torch
    assert o.gelu_tanh(np.array([0.0]))[0] == 0.0
    z = np.linspace(-8, 8, 2001)
    odd = o.gelu_tanh(z) - o.gelu_tanh(-z)          # = z exactly in real arithmetic
    assert np.max(np.abs(odd - z)) < 1e-14 * 8
    ref = torch.nn.functional.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    assert np.max(np.abs(o.gelu_tanh(z) - ref)) < 1e-14
    # limits: ~z for large z, ~0 for very negative z
    assert abs(o.gelu_tanh(np.array([30.0]))[0] - 30.0) < 1e-12
    assert abs(o.gelu_tanh(np.array([-30.0]))[0]) < 1e-12


def pin_topk(o):
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((50, 16)).astype(np.float32)
    for k in (1, 2, 5, 16):
        ids = o.select_top_k(lg, k)
        for t in range(lg.shape[0]):
            brute = sorted(range(16), key=lambda e: (-float(lg[t, e]), e))[:k]
            assert ids[t].tolist() == brute
    # exact ties go to the lower id, output order by descending value
    tie = np.array([[0.5, 2.0, 2.0, -1.0, 2.0, 0.5]], dtype=np.float32)
    assert o.select_top_k(tie, 4)[0].tolist() == [1, 2, 4, 0]
    assert o.select_top_k(tie, 2)[0].tolist() == [1, 2]


def pin_softmax_full(o):
    from scipy.special import softmax
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((7, 12)) * 3
    ids = o.select_top_k(lg, 12)
    w = o.routing_weights(lg, ids)
    ref = np.take_along_axis(softmax(lg, axis=1), ids, axis=1)
    assert np.max(np.abs(w - ref)) < 1e-15


def _tiny_layer(seed, hidden, inter, n_experts):
    router = gen.router_weights(seed, n_experts, hidden)
    experts = [gen.expert_weights(seed, e, hidden, inter) for e in range(n_experts)]
    shared = gen.expert_weights(seed, gen.SHARED_ID, hidden, inter)
    return router, experts, shared


def pin_integer_layer(o):
    """Unit scale, zero bias: weights are the integer codes, x small integers,
    so gate/up outputs are exact integers computable in int64."""
    hidden, inter = 128, 64
    rng = np.random.default_rng(5)
    one = _bf16_bits_exact(1.0)
    mats = {}
    for m, (n, k) in (("gate", (inter, hidden)), ("up", (inter, hidden)), ("down", (hidden, inter))):
        q = rng.integers(0, 2 ** 32, size=(n, k // 8), dtype=np.uint64).astype(np.uint32)
        mats[m] = {"q": q, "s": np.full((n, k // 64), one, np.uint16), "b": np.zeros((n, k // 64), np.uint16)}
    xi = rng.integers(-3, 4, size=(4, hidden))
    x = xi.astype(np.float64)
    dense = o.dense_expert(mats)
    # integer reference: unpack codes with explicit shifts
    def codes(q):
        n, nw = q.shape
        out = np.zeros((n, nw * 8), dtype=np.int64)
        for r in range(n):
            for c in range(nw * 8):
                out[r, c] = (int(q[r, c // 8]) >> (4 * (c % 8))) & 15
        return out
    g_int = xi @ codes(mats["gate"]["q"]).T
    u_int = xi @ codes(mats["up"]["q"]).T
    assert np.array_equal(x @ dense["gate"].T, g_int.astype(np.float64))
    assert np.array_equal(x @ dense["up"].T, u_int.astype(np.float64))
    h = o.expert_hidden(x, dense)
    ref_h = np.array([[_brute.gelu_tanh(float(a)) * float(b) for a, b in zip(ga, ua)] for ga, ua in zip(g_int, u_int)])
    assert np.max(np.abs(h - ref_h)) <= 1e-12 * max(1.0, np.max(np.abs(ref_h)))


def pin_brute_force(o):
    hidden, inter, n_experts, k, t = 128, 128, 8, 2, 3
    router, experts, shared = _tiny_layer(11, hidden, inter, n_experts)
    x = gen.hidden_states(11, 0, t, hidden, rms_normalize=True)
    bias = (np.arange(n_experts, dtype=np.float32) * np.float32(0.05))
    for lb in (None, bias):
        got = o.moe_block(x, router, lambda e: experts[e], shared, k, logit_bias=lb)
        ref = _brute.block(x.tolist(), router_rows(router), [expert_rows(e) for e in experts], expert_rows(shared), k,
                           None if lb is None else lb.tolist())
        for ti, (lg, ids, w, y) in enumerate(ref):
            assert got["ids"][ti].tolist() == ids
            assert np.max(np.abs(got["logits"][ti] - np.array(lg))) <= 1e-12 * max(1.0, np.max(np.abs(lg)))
            assert np.max(np.abs(got["weights"][ti] - np.array(w))) <= 1e-12
            scale = max(1e-30, float(np.max(np.abs(y))))
            assert np.max(np.abs(got["y"][ti] - np.array(y))) <= 1e-11 * scale


def router_rows(router):
    return {"q": router["q"].tolist(), "s": router["s"].tolist(), "b": router["b"].tolist()}


def expert_rows(expert):
    return {m: {f: expert[m][f].tolist() for f in ("q", "s", "b")} for m in ("gate", "up", "down")}


def pin_invariants(o):
    hidden, inter, n_experts, k, t = 128, 64, 8, 3, 5
    router, experts, shared = _tiny_layer(21, hidden, inter, n_experts)
    x = gen.hidden_states(21, 1, t, hidden, rms_normalize=True)
    base = o.moe_block(x, router, lambda e: experts[e], shared, k)
    # routing weights sum to 1, ids unique and in range
    assert np.max(np.abs(base["weights"].sum(axis=1) - 1.0)) < 1e-14
    for row in base["ids"]:
        assert len(set(row.tolist())) == k and min(row) >= 0 and max(row) < n_experts
    # a zeroed expert (scale = bias = 0) contributes exactly 0
    e0 = int(base["ids"][0, 0])
    zeroed = {m: {"q": experts[e0][m]["q"], "s": np.zeros_like(experts[e0][m]["s"]),
                  "b": np.zeros_like(experts[e0][m]["b"])} for m in ("gate", "up", "down")}
    exps = list(experts)
    exps[e0] = zeroed
    z = o.moe_block(x, router, lambda e: exps[e], shared, k)
    assert np.array_equal(z["ids"], base["ids"])
    manual = np.zeros_like(base["y"])
    outs = {}
    for ti in range(t):
        for j, e in enumerate(base["ids"][ti]):
            if int(e) == e0:
                continue
            if int(e) not in outs:
                outs[int(e)] = o.dense_expert(experts[int(e)])
            manual[ti] += base["weights"][ti, j] * o.expert_ffn(o.bf16_to_f64(x[ti:ti + 1]), outs[int(e)])[0]
    manual += o.expert_ffn(o.bf16_to_f64(x), o.dense_expert(shared))
    assert np.max(np.abs(z["y"] - manual)) <= 1e-12 * np.max(np.abs(manual))
    # relabelling experts together with their router rows leaves y unchanged
    perm = np.random.default_rng(0).permutation(n_experts)
    inv = np.argsort(perm)
    r2 = {f: router[f][perm] for f in ("q", "s", "b")}
    p = o.moe_block(x, r2, lambda e: experts[int(perm[e])], shared, k)
    assert np.array_equal(perm[p["ids"]], base["ids"])
    assert np.max(np.abs(p["y"] - base["y"])) <= 1e-13 * np.max(np.abs(base["y"]))
    del inv
    # batch invariance: each token alone gives the same output
    for ti in range(t):
        one = o.moe_block(x[ti:ti + 1], router, lambda e: experts[e], shared, k)
        assert np.array_equal(one["ids"][0], base["ids"][ti])
        assert np.max(np.abs(one["y"][0] - base["y"][ti])) <= 1e-13 * np.max(np.abs(base["y"][ti]))
    # scaling W_down's scale and bias by 2 doubles the expert output exactly
    ex = experts[1]
    two = dict(ex)
    two["down"] = {"q": ex["down"]["q"],
                   "s": o.f64_to_bf16(2.0 * o.bf16_to_f64(ex["down"]["s"])),
                   "b": o.f64_to_bf16(2.0 * o.bf16_to_f64(ex["down"]["b"]))}
    xf = o.bf16_to_f64(x)
    assert np.array_equal(o.expert_ffn(xf, o.dense_expert(two)), 2.0 * o.expert_ffn(xf, o.dense_expert(ex)))


def pin_route_sort(o):
    rng = np.random.default_rng(9)
    for t, k, e_count in ((1, 8, 128), (13, 8, 128), (128, 8, 128), (7, 3, 5), (0, 8, 128)):
        ids = np.stack([rng.permutation(e_count)[:k] for _ in range(t)]) if t else np.zeros((0, k), np.int64)
        counts, offsets, perm, pos = o.route_sort(ids, e_count)
        flat = ids.reshape(-1)
        assert np.array_equal(counts, np.bincount(flat, minlength=e_count))
        assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        assert np.array_equal(np.sort(perm), np.arange(flat.size))
        assert np.array_equal(pos[perm], np.arange(flat.size))
        for e in range(e_count):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def pin_rmsnorm(o):
    two = _bf16_bits_exact(2.0)
    h = np.full((1, 64), two, dtype=np.uint16)
    assert np.all(o.rmsnorm_no_scale(h) == _bf16_bits_exact(1.0))
    row = np.zeros((1, 4), dtype=np.float64)
    row[0, :2] = [3.0, 4.0]                       # rms = 2.5
    got = o.bf16_to_f64(o.rmsnorm_no_scale(o.f64_to_bf16(row)))
    want = o.bf16_to_f64(o.f64_to_bf16(np.array([[3.0, 4.0, 0, 0]]) / math.sqrt(6.25 + 1e-6)))
    assert np.array_equal(got, want)
    assert abs(got[0, 0] - 1.2) < 1e-2 and abs(got[0, 1] - 1.6) < 1e-2
    zero = np.zeros((1, 64), dtype=np.uint16)
    assert np.all(o.rmsnorm_no_scale(zero) == 0)


def pin_router_scales(o):
    """The learned router scale and per-expert scales (page "TurboFieldfare -
    System design", section "Decode", router description)."""
    hidden, inter, n_experts, k, t = 256, 64, 8, 3, 4      # sqrt(hidden) = 16 exactly
    router, experts, shared = _tiny_layer(31, hidden, inter, n_experts)
    x = gen.hidden_states(31, 0, t, hidden, rms_normalize=True)
    # router_scale = 16 * 2^j per feature: x * scale / 16 is x * 2^j, an exact
    # bf16 value, so the scaled router equals the brute-force router on that row
    j = np.random.default_rng(3).integers(-2, 3, size=hidden)
    rs = np.array([_bf16_bits_exact(16.0 * 2.0 ** int(v)) for v in j], dtype=np.uint16)
    got = o.router_logits(x, router, router_scale=rs)
    rr = router_rows(router)
    for ti in range(t):
        xs = [_brute.bf16(v) * 2.0 ** int(e) for v, e in zip(x[ti].tolist(), j)]
        ref = _brute.matvec(rr, 8, xs)
        assert np.max(np.abs(got[ti] - np.array(ref))) <= 1e-12 * max(1.0, max(abs(a) for a in ref))
    # a constant scale of 16 is the identity
    same = np.full(hidden, _bf16_bits_exact(16.0), dtype=np.uint16)
    assert np.array_equal(o.router_logits(x, router, router_scale=same), o.router_logits(x, router))
    # per-expert scales multiply the softmax weight of each selected expert
    pes = (0.5 + np.random.default_rng(4).random(n_experts)).astype(np.float32)
    base = o.moe_block(x, router, lambda e: experts[e], shared, k)
    sc = o.moe_block(x, router, lambda e: experts[e], shared, k, per_expert_scale=pes)
    assert np.array_equal(sc["ids"], base["ids"])
    for ti in range(t):
        lg = [float(base["logits"][ti, e]) for e in base["ids"][ti]]
        ex = [math.exp(v - max(lg)) for v in lg]
        want = [a / sum(ex) * float(pes[e]) for a, e in zip(ex, base["ids"][ti])]
        assert np.max(np.abs(sc["weights"][ti] - np.array(want))) <= 1e-14
    # zero scales leave the shared expert alone; doubling them doubles the routed part
    zero = o.moe_block(x, router, lambda e: experts[e], shared, k, per_expert_scale=np.zeros(n_experts, np.float32))
    sh = o.expert_ffn(o.bf16_to_f64(x), o.dense_expert(shared))
    assert np.max(np.abs(zero["y"] - sh)) <= 1e-13 * np.max(np.abs(sh))
    two = o.moe_block(x, router, lambda e: experts[e], shared, k, per_expert_scale=np.full(n_experts, 2.0, np.float32))
    assert np.max(np.abs((two["y"] - sh) - 2.0 * (base["y"] - sh))) <= 1e-12 * np.max(np.abs(base["y"]))


def _rne_bf16(v: float) -> float:
    """Round a float to the nearest bf16 value (ties to even), in plain Python:
    v / 2^(e-7) is exact, and round() on a float rounds half to even."""
    if v == 0.0 or not math.isfinite(v):
        return v
    e = math.frexp(v)[1] - 1
    step = 2.0 ** (e - 7)
    return round(v / step) * step


def pin_layer_tail(o):
    """Post-FFN norm, residual and layer scalar (page "TurboFieldfare - System
    design", section "Decode", cb2 phase)."""
    f = o.f64_to_bf16
    # closed form: y = 2 everywhere -> y / rms(y) rounds to 1; 0.5 + 1 = 1.5; 2 * 1.5 = 3
    y, h, g = f(np.full((1, 64), 2.0)), f(np.full((1, 64), 0.5)), f(np.ones(64))
    assert np.all(o.bf16_to_f64(o.layer_tail(h, y, g, 2.0)) == 3.0)
    # eps matters for small rows: c / sqrt(c^2 + 1e-6)
    c = float(o.bf16_to_f64(f(np.array([1e-3])))[0])
    want = _rne_bf16(c / math.sqrt(c * c + 1e-6))
    got = o.bf16_to_f64(o.layer_tail(f(np.zeros((1, 64))), f(np.full((1, 64), c)), g))
    assert np.all(got == want) and abs(want - 0.7071) < 0.01
    # brute force on random rows: plain-Python sums, hand rounding
    rng = np.random.default_rng(17)
    hb, yb = f(rng.normal(size=(3, 64))), f(rng.normal(size=(3, 64)) * 0.3)
    gb = f(0.5 + rng.random(64))
    lam = float(np.float32(0.5 + rng.random()))
    got = o.bf16_to_f64(o.layer_tail(hb, yb, gb, lam))
    for t in range(3):
        yr = [_brute.bf16(v) for v in yb[t].tolist()]
        rms = math.sqrt(math.fsum(v * v for v in yr) / 64 + 1e-6)
        for j in range(64):
            z = _rne_bf16(yr[j] / rms * _brute.bf16(int(gb[j])))
            sj = _rne_bf16(_brute.bf16(int(hb[t, j])) + z)
            assert got[t, j] == _rne_bf16(lam * sj), (t, j)
    # y = 0 leaves lambda * h; a zero norm weight leaves lambda * h on that feature
    zero = o.layer_tail(hb, f(np.zeros((3, 64))), gb, lam)
    assert np.array_equal(o.bf16_to_f64(zero), np.vectorize(_rne_bf16)(lam * o.bf16_to_f64(hb)))
    g0 = gb.copy()
    g0[5] = 0
    one = o.bf16_to_f64(o.layer_tail(hb, yb, g0, lam))
    assert np.array_equal(one[:, 5], np.vectorize(_rne_bf16)(lam * o.bf16_to_f64(hb[:, 5])))
    # no norm weight and no scalar: the plain residual add
    assert np.array_equal(o.layer_tail(hb, yb), o.residual_add(hb, yb))


ALL_PINS = [pin_layout_sizes, pin_dequant_golden, pin_bf16_rounding, pin_gelu, pin_topk, pin_softmax_full,
            pin_integer_layer, pin_brute_force, pin_invariants, pin_route_sort, pin_rmsnorm,
            pin_router_scales, pin_layer_tail]
