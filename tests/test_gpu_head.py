"""The tied 4-bit head and embedding on a GB300, through the C ABI, against
the float64 oracle (page "TurboFieldfare - System design": the embedding and
the head share one 4-bit affine matrix; a final logit softcap of 30; the head
returns the argmax token or the full logits).

Logits are compared with the oracle at the block's tolerance; the greedy
token, a decision taken in floating point, must equal the argmax (ties to the
lower id) of the GPU's own fp32 logits; the embedding is bit-exact."""
import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import from_dev_bf16, to_dev_bf16
from numerics import assert_close
from oracle import head_oracle as HO
from synth import gen
from synth.device import DeviceHead

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def moe():
    bq.build_library()
    m = bq.Moe()
    yield m
    m.close()


def _hw(head):
    q, s, b = head.addresses()
    return bq.make_head_weights(head.vocab, head.hidden, q, s, b)


def _x(seed, T, H, scale):
    x = gen.hidden_states(seed, 0, T, H, rms_normalize=True)
    return x if scale == 1.0 else gen.to_bf16_bits(gen.bf16_bits_to_f64(x) * scale)


def _run(moe, head, x_bits, want_logits=True, want_tokens=True, cap=30.0):
    T = x_bits.shape[0]
    logits = torch.empty((T, head.vocab), dtype=torch.float32, device="cuda") if want_logits else None
    tokens = torch.empty(T, dtype=torch.int32, device="cuda") if want_tokens else None
    moe.head_forward(to_dev_bf16(x_bits), T, _hw(head), cap, logits=logits, tokens=tokens)
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK
    return (None if logits is None else logits.cpu().numpy().astype(np.float64),
            None if tokens is None else tokens.cpu().numpy())


@pytest.mark.parametrize("scale", [1.0, 60.0], ids=["unit-rms", "softcap-active"])
@pytest.mark.parametrize("V,H,T", [(256, 128, 1), (1024, 256, 3), (4096, 2816, 8), (4112, 2816, 5), (16, 64, 2)])
def test_head_small(moe, V, H, T, scale):
    head = DeviceHead(5, V, H)
    x = _x(7, T, H, scale)
    logits, tokens = _run(moe, head, x)
    ref = HO.head_logits(x, head.host_rows())
    assert_close(logits, ref, f"head logits V={V} H={H} T={T}")
    assert np.array_equal(tokens, HO.greedy_token(logits))
    # each output alone: the same values
    lg_only, _ = _run(moe, head, x, want_tokens=False)
    _, tk_only = _run(moe, head, x, want_logits=False)
    assert np.array_equal(lg_only, logits) and np.array_equal(tk_only, tokens)
    if scale > 1.0:
        assert np.max(np.abs(ref)) > 20.0, "the inputs never reach the softcap's curved part"


def test_head_without_softcap(moe):
    head = DeviceHead(6, 512, 256)
    x = _x(8, 2, 256, 60.0)
    logits, tokens = _run(moe, head, x, cap=0.0)
    w = head.host_rows()
    from oracle.moe_oracle import bf16_to_f64, dequantize
    ref = bf16_to_f64(x) @ dequantize(w["q"], w["s"], w["b"], 4).T
    assert_close(logits, ref, "head logits without softcap")
    assert np.array_equal(tokens, HO.greedy_token(logits))


@pytest.mark.parametrize("T", [1, 8])
def test_head_full_vocab(moe, T):
    """V = 262,144, H = 2816: logits on sampled rows against the oracle, the
    token against the argmax of the GPU's logits, and the oracle's logit of
    that token against the oracle's best sampled logit."""
    V, H = 262144, 2816
    head = DeviceHead(1, V, H)
    x = _x(9, T, H, 30.0)
    logits, tokens = _run(moe, head, x)
    assert np.array_equal(tokens, HO.greedy_token(logits))
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.integers(0, V, 3000), [0, V - 1], tokens]))
    ref = HO.head_logits(x, head.host_rows(rows), rows=None)
    assert_close(logits[:, rows], ref, "sampled head logits")
    scale = np.sqrt(np.mean(ref * ref))
    for t in range(T):
        j = int(np.flatnonzero(rows == tokens[t])[0])
        assert ref[t, j] >= ref[t].max() - 4e-2 * scale


def test_embed(moe):
    V, H = 4112, 2816
    head = DeviceHead(5, V, H)
    ids = np.array([0, V - 1, 17, 17, 4095, 2048], dtype=np.int32)
    out = torch.empty((ids.size, H), dtype=torch.int16, device="cuda")
    moe.embed(torch.from_numpy(ids).cuda(), ids.size, _hw(head), out)
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK
    want = HO.embed(np.arange(ids.size), head.host_rows(ids))
    assert np.array_equal(from_dev_bf16(out), want)


def test_embed_bad_ids(moe):
    V, H = 256, 128
    head = DeviceHead(5, V, H)
    ids = np.array([3, -1, V, 5], dtype=np.int32)
    out = torch.full((ids.size, H), 7, dtype=torch.int16, device="cuda")
    moe.embed(torch.from_numpy(ids).cuda(), ids.size, _hw(head), out)
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_ERR_BAD_EXPERT_ID
    got = from_dev_bf16(out)
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    assert np.array_equal(got[[0, 3]], HO.embed(np.arange(2), head.host_rows([3, 5])))


def test_head_then_embed_chained(moe):
    """head -> embed of its greedy tokens on one stream (programmatic
    dependent launch between them), captured in a graph and replayed twice:
    the embedding must be that of the head's tokens."""
    V, H, T = 4096, 2816, 4
    head = DeviceHead(11, V, H)
    x = to_dev_bf16(_x(12, T, H, 10.0))
    tokens = torch.empty(T, dtype=torch.int32, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            moe.head_forward(x, T, _hw(head), 30.0, tokens=tokens, stream=st)
            moe.embed(tokens, T, _hw(head), out, stream=st)
        for _ in range(2):
            out.zero_()
            g.replay()
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK
    tk = tokens.cpu().numpy()
    assert np.array_equal(from_dev_bf16(out), HO.embed(np.arange(T), head.host_rows(tk)))


@pytest.mark.parametrize("N,K,T", [(4096, 2816, 1), (2816, 4096, 4), (1024, 256, 8), (16, 64, 3)])
def test_dense_projection(moe, N, K, T):
    """The dense 4-bit projection (Q/K/V- and O-like shapes; the pages give the
    format, not the attention's sizes): fp32 and bf16 outputs against the
    float64 oracle, and each output alone gives the same values."""
    w = DeviceHead(21, N, K)
    x = _x(22, T, K, 1.0)
    y32 = torch.empty((T, N), dtype=torch.float32, device="cuda")
    y16 = torch.empty((T, N), dtype=torch.int16, device="cuda")
    moe.dense_forward(to_dev_bf16(x), T, _hw(w), y=y16, y32=y32)
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK
    ref = HO.dense(x, w.host_rows())
    got32 = y32.cpu().numpy().astype(np.float64)
    assert_close(got32, ref, "dense fp32")
    got16 = from_dev_bf16(y16)
    assert np.array_equal(got16, gen.to_bf16_bits(got32.astype(np.float32).astype(np.float64)))
    only16 = torch.empty_like(y16)
    moe.dense_forward(to_dev_bf16(x), T, _hw(w), y=only16)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_bf16(only16), got16)


def test_dense_projection_leaves_greedy_state(moe):
    """A projection between two head calls must not disturb the head's argmax state."""
    head = DeviceHead(23, 1024, 256)
    x = _x(24, 2, 256, 30.0)
    _, t0 = _run(moe, head, x)
    w = DeviceHead(25, 512, 256)
    y = torch.empty((2, 512), dtype=torch.float32, device="cuda")
    moe.dense_forward(to_dev_bf16(_x(26, 2, 256, 1.0)), 2, _hw(w), y32=y)
    _, t1 = _run(moe, head, x)
    assert np.array_equal(t0, t1)
