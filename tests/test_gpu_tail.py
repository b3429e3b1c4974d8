"""The layer tail on a GB300: post-FFN norm, residual and layer scalar after
the combine (page "TurboFieldfare - System design", section "Decode", cb2
phase), through moe_layer_forward_residual and moe_layer_forward_stack.

The block itself is checked as elsewhere (ids bit-exact on the GPU's logits,
outputs against the oracle on the GPU's ids).  The tail is checked on the
GPU's own block output y (teacher forcing on y): the new residual stream must
equal the oracle's layer_tail(h, y) bit for bit (at least 99% of the
elements) except where an fp32-vs-fp64 difference moves one of the three
bf16 roundings across a tie, and there by at most one bf16 step of each
rounded term."""
import os

import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import E, H, I, K, from_dev_bf16, hidden, oracle_layer, to_dev_bf16, workspace
from numerics import assert_close, bf16_bits_to_f64
from oracle import moe_oracle as O
from synth.device import DeviceLayer

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def layer_tail():
    bq.build_library()
    return DeviceLayer(3, H, I, E, zipf=True, tail=True)


def _handle(var, fused):
    old = os.environ.get(var)
    os.environ[var] = fused
    try:
        return bq.Moe()
    finally:
        if old is None:
            del os.environ[var]
        else:
            os.environ[var] = old


def _weights(layer, k=K, drop=()):
    addr = dict(layer.addresses())
    for name in drop:
        addr[name] = None
    return bq.layer_weights_from(bq.make_dims(layer.hidden, layer.inter, layer.n_experts, k), addr)


def check_tail(h0_bits, y_bits, h_bits, g_bits, lam):
    """h_bits (GPU) against layer_tail(h0, y) of the oracle."""
    ref = O.layer_tail(h0_bits, y_bits, g_bits, lam)
    got_f, ref_f = bf16_bits_to_f64(h_bits), bf16_bits_to_f64(ref)
    exact = np.mean(h_bits == ref)
    assert exact >= 0.99, f"only {exact:.4f} of the tail outputs are bit-exact"
    # a flipped rounding moves its result by one bf16 step, at most 2^-7 of
    # its magnitude: z by 2^-7 |z|, s = h + z by 2^-7 (|h| + |z|) more, and
    # the scaled result by 2^-7 |h'|
    z = bf16_bits_to_f64(y_bits) if g_bits is None else O.post_ffn_norm(y_bits, g_bits)
    h0 = bf16_bits_to_f64(h0_bits)
    lam_f = 1.0 if lam is None else float(lam)
    bound = 2.0 ** -7 * (abs(lam_f) * (np.abs(h0) + 2.0 * np.abs(z)) + np.abs(ref_f)) * 1.01
    err = np.abs(got_f - ref_f)
    i = np.unravel_index(np.argmax(err - bound), err.shape)
    assert not (err > bound).any(), (f"{(err > bound).sum()} tail outputs beyond one bf16 step of each rounding; "
                                     f"worst at {i}: h {h0[i]}, z {z[i]}, got {got_f[i]}, want {ref_f[i]}")


def _run_residual(m, layer, h0, k=K, drop=()):
    n = h0.shape[0]
    w = _weights(layer, k, drop)
    h = to_dev_bf16(h0)
    y = torch.empty_like(h)
    xo = torch.empty_like(h)
    ids = torch.empty((n, k), dtype=torch.int32, device="cuda")
    logits = torch.empty((n, layer.n_experts), dtype=torch.float32, device="cuda")
    ws = workspace(m, w, n)
    m.layer_forward_residual(h, n, w, ws, y_out=y, x_out=xo, ids_out=ids, logits_out=logits)
    torch.cuda.synchronize()
    assert m.get_error() == bq.MOE_OK
    return {"h": from_dev_bf16(h), "y": from_dev_bf16(y), "x": from_dev_bf16(xo), "ids": ids.cpu().numpy(),
            "logits": logits.cpu().numpy()}


@pytest.mark.parametrize("fused", ["1", "0"])
@pytest.mark.parametrize("n_tokens", [1, 37, 128])
def test_layer_tail(layer_tail, n_tokens, fused):
    m = _handle("MOE_DECODE_FUSED" if n_tokens == 1 else "MOE_PREFILL_FUSED", fused)
    try:
        h0 = hidden(41, n_tokens, n_tokens, rms=False)
        out = _run_residual(m, layer_tail, h0)
    finally:
        m.close()
    # the block input is the normalised residual stream, the block as usual
    xr = bf16_bits_to_f64(O.rmsnorm_no_scale(h0))
    assert np.all(np.abs(bf16_bits_to_f64(out["x"]) - xr) <= 2.0 ** -7 * np.abs(xr))
    assert np.array_equal(out["ids"], O.select_top_k(out["logits"], K))
    ref = oracle_layer(layer_tail, out["x"], K, out["ids"])
    assert_close(bf16_bits_to_f64(out["y"]), ref["y"], f"y (T={n_tokens}, fused={fused})")
    g, lam = layer_tail.host_layer_tail()
    check_tail(h0, out["y"], out["h"], g, lam)


@pytest.mark.parametrize("drop", [(), ("post_norm",), ("layer_scalar",)], ids=["both", "scalar-only", "norm-only"])
@pytest.mark.parametrize("n_tokens", [1, 5])
def test_partial_tails_small(drop, n_tokens):
    layer = DeviceLayer(8, 256, 128, 16, tail=True)
    m = bq.Moe()
    try:
        h0 = hidden(8, n_tokens, n_tokens, 256, rms=False)
        out = _run_residual(m, layer, h0, k=4, drop=drop)
    finally:
        m.close()
    ref = oracle_layer(layer, out["x"], 4, out["ids"])
    assert_close(bf16_bits_to_f64(out["y"]), ref["y"], "small-shape y")
    g, lam = layer.host_layer_tail()
    check_tail(h0, out["y"], out["h"], None if "post_norm" in drop else g, None if "layer_scalar" in drop else lam)


def test_tail_without_y_out(layer_tail):
    """The block output goes to the workspace when the caller gives no y_out;
    the residual stream must be the same as with y_out."""
    m = bq.Moe()
    try:
        h0 = hidden(43, 0, 4, rms=False)
        with_y = _run_residual(m, layer_tail, h0)
        w = _weights(layer_tail)
        h = to_dev_bf16(h0)
        m.layer_forward_residual(h, 4, w, workspace(m, w, 4))
        torch.cuda.synchronize()
        assert m.get_error() == bq.MOE_OK
        assert np.array_equal(from_dev_bf16(h), with_y["h"])
    finally:
        m.close()


def test_stack_with_tails_matches_layer_calls():
    """moe_layer_forward_stack over layers with tails, captured in a graph,
    equals the same layers called one by one."""
    layers = [DeviceLayer(20 + l, 256, 128, 16, zipf=True, tail=True) for l in range(4)]
    ws_list = [_weights(L, 4) for L in layers]
    m = bq.Moe()
    try:
        ws = workspace(m, ws_list[0], 1)
        h0 = hidden(44, 0, 1, 256, rms=False)
        a = to_dev_bf16(h0)
        for w in ws_list:
            m.layer_forward_residual(a, 1, w, ws)
        b = to_dev_bf16(h0)
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                m.layer_forward_stack(b, ws_list, ws, stream=st)
            b.copy_(to_dev_bf16(h0))
            g.replay()
        torch.cuda.synchronize()
        assert m.get_error() == bq.MOE_OK
        assert np.array_equal(from_dev_bf16(a), from_dev_bf16(b))
    finally:
        m.close()
