"""The allocation-free single-token entry point (moe_layer_forward_static).

It serves hosts that cannot allocate device memory (their own pool owns the
device, or an allocation would stall a per-token loop), so it keeps its
scratch in static device arrays instead of a caller workspace.  Two calls in
a row, through the C ABI, must match the regular entry point
(moe_layer_forward, T = 1) and the float64 oracle within the block's
tolerance: the second call shows that what the first left in the shared
arrays does not leak into it.  Its device-side errors go to a static error
word of their own, read back by moe_static_get_error.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one; it builds everything it needs itself, so it
also passes alone in a fresh process."""
import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import E, H, I, K, from_dev_bf16, hidden, oracle_layer, to_dev_bf16, weights_of, workspace
from numerics import assert_close, bf16_bits_to_f64
from oracle import moe_oracle as O
from synth import gen
from synth.device import DeviceLayer

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def layer5():
    bq.build_library()
    return DeviceLayer(5, H, I, E)


def _static_call(x, w):
    y = torch.empty_like(x)
    ids = torch.full((1, K), -1, dtype=torch.int32, device="cuda")
    lg = torch.empty((1, E), dtype=torch.float32, device="cuda")
    wts = torch.empty((1, K), dtype=torch.float32, device="cuda")
    bq.layer_forward_static(x, w, y, ids_out=ids, logits_out=lg, weights_out=wts)
    torch.cuda.synchronize()
    return y, ids, lg, wts


def test_static_entry_matches_layer_forward_twice(layer5):
    w = weights_of(layer5)
    moe = bq.Moe()
    ws = workspace(moe, w, 1)
    for call, seed in enumerate((31, 32)):
        x_bits = hidden(seed, 0, 1)
        x = to_dev_bf16(x_bits)
        y_ref = torch.empty_like(x)
        ids_ref = torch.empty((1, K), dtype=torch.int32, device="cuda")
        lg_ref = torch.empty((1, E), dtype=torch.float32, device="cuda")
        moe.layer_forward(x, 1, w, y_ref, ws, ids_out=ids_ref, logits_out=lg_ref)
        y, ids, lg, wts = _static_call(x, w)
        assert bq.static_get_error() == bq.MOE_OK
        assert moe.get_error() == bq.MOE_OK
        ids_np = ids.cpu().numpy()
        assert np.array_equal(ids_np, ids_ref.cpu().numpy()), f"call {call}: ids differ"
        assert np.array_equal(ids_np, O.select_top_k(lg.cpu().numpy(), K)), f"call {call}: ids vs oracle top-k"
        assert_close(lg.cpu().numpy(), lg_ref.cpu().numpy(), f"call {call}: logits")
        assert_close(lg.cpu().numpy(), O.router_logits(x_bits, layer5.host_router()), f"call {call}: logits vs oracle")
        got = bf16_bits_to_f64(from_dev_bf16(y))
        assert_close(got, bf16_bits_to_f64(from_dev_bf16(y_ref)), f"call {call}: y vs moe_layer_forward")
        assert_close(got, oracle_layer(layer5, x_bits, K, ids_np)["y"], f"call {call}: y vs oracle")
        assert abs(float(wts.sum()) - 1.0) < 1e-5
    moe.close()


def test_static_entry_reports_device_errors(layer5):
    """Expert activations pushed out of fp16 range (input at rms 1000) are
    flagged in the static error word; the read clears it and the next call
    is clean and correct."""
    w = weights_of(layer5)
    big = gen.to_bf16_bits(bf16_bits_to_f64(hidden(40, 0, 1)) * 1000.0)
    _static_call(to_dev_bf16(big), w)
    assert bq.static_get_error() == bq.MOE_ERR_NONFINITE
    assert bq.static_get_error() == bq.MOE_OK
    x_bits = hidden(41, 0, 1)
    y, ids, lg, _ = _static_call(to_dev_bf16(x_bits), w)
    assert bq.static_get_error() == bq.MOE_OK
    ids_np = ids.cpu().numpy()
    assert np.array_equal(ids_np, O.select_top_k(lg.cpu().numpy(), K))
    assert_close(bf16_bits_to_f64(from_dev_bf16(y)), oracle_layer(layer5, x_bits, K, ids_np)["y"], "y after error")


def test_static_entry_rejects_oversized_shapes():
    """top-8 of inter 1024 needs (8+1)*1024*2 B of h, beyond the static array:
    refused before anything is launched (the weight addresses are never read)."""
    bq.build_library()
    dims = bq.make_dims(256, 1024, 8, 8)
    bl = gen.blob_layout(256, 1024)
    layout = {k: v for k, v in bl.items() if k not in ("bytes", "stride")}
    big = bq.make_layer_weights(dims, 1 << 40, (1 << 40) + 4096, (1 << 40) + 8192, 1 << 41, bl["stride"], layout,
                                1 << 42)
    x = torch.zeros(256, dtype=torch.int16, device="cuda")
    with pytest.raises(bq.MoeError) as ei:
        bq.layer_forward_static(x, big, torch.empty_like(x))
    assert ei.value.status == bq.MOE_ERR_UNSUPPORTED
