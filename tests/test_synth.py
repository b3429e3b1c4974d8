"""The seeded input generators (shared by the oracle tests and the device
fillers): row subsets reproduce the whole matrix, and the host-side parts of
the device generators equal the host generator."""
import numpy as np

from synth import gen


def test_head_rows_match_whole_matrix():
    whole = gen.head_weights(5, 96, 256)
    rows = [95, 0, 31, 32, 64, 7]
    sub = gen.head_weights(5, 96, 256, rows=rows)
    for f in ("q", "s", "b"):
        assert np.array_equal(sub[f], whole[f][rows]), f


def test_head_words_follow_the_word_stream():
    # the device filler writes words(key, n) over the whole matrix: the host
    # generator must read the same stream in row-major order
    V, H = 32, 128
    whole = gen.head_weights(2, V, H)
    key = gen.weight_key(2, gen.HEAD_ID, gen.MAT_HEAD, gen.FIELD_Q)
    assert np.array_equal(whole["q"].reshape(-1), gen.words(key, V * H // 8))


def test_head_value_ranges():
    w = gen.head_weights(1, 64, 2816)
    s = gen.bf16_bits_to_f64(w["s"])
    lo, hi = 0.5 / (8 * np.sqrt(2816.0)), 1.5 / (8 * np.sqrt(2816.0))
    assert np.all(s >= lo * (1 - 2 ** -8)) and np.all(s <= hi * (1 + 2 ** -8))
    codes = [(int(x) >> (4 * i)) & 15 for x in w["q"].reshape(-1)[:512] for i in range(8)]
    assert min(codes) == 0 and max(codes) == 15


def test_tail_and_router_scale_generators_are_deterministic():
    a = gen.layer_tail(3, 256)
    b = gen.layer_tail(3, 256)
    assert np.array_equal(a[0], b[0]) and a[1] == b[1] and 0.5 <= a[1] <= 1.5
    rs, pes = gen.router_scales(3, 16, 256)
    assert rs.shape == (256,) and pes.shape == (16,) and np.all((pes >= 0.5) & (pes <= 1.5))
