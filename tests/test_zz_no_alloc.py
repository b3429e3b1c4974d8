"""The allocation-free single-token entry point (moe_layer_forward_static).

It serves hosts that cannot allocate device memory (their own pool owns the
device, or an allocation would stall a per-token loop), so it keeps its
scratch in a static device array instead of a caller workspace.  Two calls in
a row, through the C ABI, must match the regular entry point
(moe_layer_forward, T = 1) within the block's tolerance: the second call shows
that what the first left in the shared array does not leak into it.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one; it builds everything it needs itself, so it
also passes alone in a fresh process."""
import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import E, H, I, K, from_dev_bf16, hidden, to_dev_bf16, weights_of, workspace
from numerics import assert_close, bf16_bits_to_f64
from synth.device import DeviceLayer

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_static_entry_matches_layer_forward_twice():
    bq.build_library()
    layer = DeviceLayer(5, H, I, E)
    w = weights_of(layer)
    moe = bq.Moe()
    ws = workspace(moe, w, 1)
    for call, seed in enumerate((31, 32)):
        x = to_dev_bf16(hidden(seed, 0, 1))
        y_ref = torch.empty_like(x)
        ids_ref = torch.empty((1, K), dtype=torch.int32, device="cuda")
        lg_ref = torch.empty((1, E), dtype=torch.float32, device="cuda")
        moe.layer_forward(x, 1, w, y_ref, ws, ids_out=ids_ref, logits_out=lg_ref)
        y = torch.empty_like(x)
        ids = torch.full((1, K), -1, dtype=torch.int32, device="cuda")
        lg = torch.empty((1, E), dtype=torch.float32, device="cuda")
        wts = torch.empty((1, K), dtype=torch.float32, device="cuda")
        bq.layer_forward_static(x, w, y, ids_out=ids, logits_out=lg, weights_out=wts)
        torch.cuda.synchronize()
        assert moe.get_error() == bq.MOE_OK
        assert np.array_equal(ids.cpu().numpy(), ids_ref.cpu().numpy()), f"call {call}: ids differ"
        assert_close(lg.cpu().numpy(), lg_ref.cpu().numpy(), f"call {call}: logits")
        assert_close(bf16_bits_to_f64(from_dev_bf16(y)), bf16_bits_to_f64(from_dev_bf16(y_ref)), f"call {call}: y")
        assert abs(float(wts.sum()) - 1.0) < 1e-5
    moe.close()


def test_static_entry_rejects_oversized_shapes():
    """top-8 of inter 1024 needs (8+1)*1024*2 B of h, beyond the static array:
    refused before anything is launched (the weight addresses are never read)."""
    from synth import gen
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
