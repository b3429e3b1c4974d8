"""Pins of the tied-head oracle (oracle/head_oracle.py) to facts outside it.

Each pin takes the head-oracle module, so the mutation test can run the pins
against a copy with a planted mistake.

  pin_softcap        closed forms of cap * tanh(z / cap): 0, oddness, the
                     bound, the half-cap point, slope 1 at 0
  pin_head_brute     a tiny head against a plain-Python scalar brute force
                     (codes pulled out one at a time, math.tanh)
  pin_head_rows      row subsets and row blocking change no value
  pin_head_onehot    a one-hot input reads one column of hand-worked weights
                     (the dequantisation fixtures)
  pin_greedy         argmax with ties to the lower id, -inf entries
  pin_embed          tied embedding = dequantised row (hand-worked fixtures)
  pin_dense_exact    the dense projection on unit scales, zero biases and
                     small integer inputs equals the exact int64 product
  pin_dense_brute    the dense projection of a tiny matrix against the
                     plain-Python scalar brute force, row blocking included
"""
from __future__ import annotations

import math
import os

import numpy as np

import _brute
from synth import gen

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _fixture_rows():
    """4-bit rows of the dequantisation fixtures: (word, scale, bias, weights)."""
    out = []
    with open(os.path.join(GOLDEN_DIR, "dequant_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            p = line.split()
            if p[0] == "4":
                out.append((int(p[1], 16), float(p[2]), float(p[3]), [float(v) for v in p[5].split(",")]))
    return out


def _bf16(v: float) -> int:
    bits = int(np.array([v], dtype=np.float32).view(np.uint32)[0])
    assert bits & 0xFFFF == 0, v
    return bits >> 16


def _fixture_head(hidden=64):
    """One head row per fixture: the fixture word repeated over the row's 8
    words, the fixture's scale and bias for its one group."""
    rows = _fixture_rows()
    q = np.array([[w] * (hidden // 8) for w, _, _, _ in rows], dtype=np.uint32)
    s = np.array([[_bf16(sc)] * (hidden // 64) for _, sc, _, _ in rows], dtype=np.uint16)
    b = np.array([[_bf16(bi)] * (hidden // 64) for _, _, bi, _ in rows], dtype=np.uint16)
    return {"q": q, "s": s, "b": b}, [wts * (hidden // 8) for _, _, _, wts in rows]


def pin_softcap(h):
    assert h.softcap(np.array([0.0]))[0] == 0.0
    z = np.array([-1e3, -45.0, -3.0, 0.5, 7.0, 29.0, 1e3])
    assert np.array_equal(h.softcap(-z), -h.softcap(z))
    assert np.all(np.abs(h.softcap(z)) <= 30.0) and np.all(np.abs(h.softcap(z[1:-1])) < 30.0)
    assert abs(h.softcap(np.array([1e3]))[0] - 30.0) < 1e-12
    half = 30.0 * math.atanh(0.5)
    assert abs(h.softcap(np.array([half]))[0] - 15.0) < 1e-12
    assert abs(h.softcap(np.array([1e-6]))[0] - 1e-6) < 1e-18


def pin_head_brute(h):
    vocab, hidden, t = 40, 128, 3
    head = gen.head_weights(2, vocab, hidden)
    x = gen.hidden_states(2, 0, t, hidden, rms_normalize=True)
    # inputs at two magnitudes: the softcap is near-linear at unit rms, active at 60x
    xs = [x, (gen.bf16_bits_to_f64(x) * 60.0)]
    xs[1] = gen.to_bf16_bits(xs[1])
    rows = {"q": head["q"].tolist(), "s": head["s"].tolist(), "b": head["b"].tolist()}
    active = False
    for xb in xs:
        got = h.head_logits(xb, head)
        for ti in range(t):
            z = _brute.matvec(rows, 4, [_brute.bf16(v) for v in xb[ti].tolist()])
            want = [30.0 * math.tanh(v / 30.0) for v in z]
            active |= max(abs(v) for v in z) > 20.0
            assert np.max(np.abs(got[ti] - np.array(want))) <= 1e-12 * max(1.0, max(abs(v) for v in want))
    assert active, "the inputs never reach the softcap's curved part"


def pin_head_rows(h):
    vocab, hidden = 50, 128
    head = gen.head_weights(3, vocab, hidden)
    x = gen.hidden_states(3, 0, 2, hidden, rms_normalize=True)
    full = h.head_logits(x, head)
    rows = [49, 0, 17, 17, 3]
    sub = h.head_logits(x, head, rows=rows)
    assert np.max(np.abs(sub - full[:, rows])) <= 1e-13 * np.max(np.abs(full))
    old = h.ROW_BLOCK
    try:
        h.ROW_BLOCK = 7
        blocked = h.head_logits(x, head)
    finally:
        h.ROW_BLOCK = old
    assert np.max(np.abs(blocked - full)) <= 1e-13 * np.max(np.abs(full))


def pin_head_onehot(h):
    head, weights = _fixture_head()
    hidden = 64
    for k in (0, 5, 7, 63):
        x = np.zeros((1, hidden), dtype=np.uint16)
        x[0, k] = _bf16(1.0)
        got = h.head_logits(x, head)[0]
        want = [30.0 * math.tanh(w[k] / 30.0) for w in weights]
        assert np.max(np.abs(got - np.array(want))) <= 1e-14


def pin_greedy(h):
    lg = np.array([[1.0, 3.0, 3.0, 2.0], [0.0, 0.0, 0.0, 0.0], [-5.0, -1.0, -np.inf, -1.0],
                   [-np.inf, -np.inf, 4.0, -np.inf], [2.0, 1.0, 0.0, -1.0], [-1.0, 0.0, 1.0, 2.0]])
    assert h.greedy_token(lg).tolist() == [1, 0, 1, 2, 0, 3]
    rng = np.random.default_rng(4)
    r = rng.normal(size=(20, 300))
    assert np.array_equal(h.greedy_token(r), np.argmax(r, axis=1))


def pin_embed(h):
    head, weights = _fixture_head()
    got = h.embed([3, 0, 2, 1, 0], head)
    for i, r in enumerate([3, 0, 2, 1, 0]):
        want = np.array([_bf16(v) for v in weights[r]], dtype=np.uint16)
        assert np.array_equal(got[i], want)


def pin_dense_exact(h):
    rng = np.random.default_rng(7)
    n, k, t = 48, 192, 3
    codes = rng.integers(0, 16, size=(n, k))
    q = np.zeros((n, k // 8), dtype=np.uint32)
    for i in range(8):
        q |= (codes[:, i::8].astype(np.uint32) << np.uint32(4 * i))
    one = _bf16(1.0)
    w = {"q": q, "s": np.full((n, k // 64), one, dtype=np.uint16), "b": np.zeros((n, k // 64), dtype=np.uint16)}
    xi = rng.integers(-8, 9, size=(t, k))
    x = gen.to_bf16_bits(xi.astype(np.float64))
    want = xi.astype(np.int64) @ codes.astype(np.int64).T
    assert np.array_equal(h.dense(x, w), want.astype(np.float64))


def pin_dense_brute(h):
    n, k, t = 24, 128, 2
    w = gen.head_weights(4, n, k)
    x = gen.hidden_states(4, 0, t, k, rms_normalize=True)
    rows = {"q": w["q"].tolist(), "s": w["s"].tolist(), "b": w["b"].tolist()}
    old = h.ROW_BLOCK
    try:
        for block in (old, 5):
            h.ROW_BLOCK = block
            got = h.dense(x, w)
            for ti in range(t):
                want = np.array(_brute.matvec(rows, 4, [_brute.bf16(v) for v in x[ti].tolist()]))
                assert np.max(np.abs(got[ti] - want)) <= 1e-13 * max(1.0, np.max(np.abs(want)))
    finally:
        h.ROW_BLOCK = old


ALL_HEAD_PINS = [pin_softcap, pin_head_brute, pin_head_rows, pin_head_onehot, pin_greedy, pin_embed,
                 pin_dense_exact, pin_dense_brute]
