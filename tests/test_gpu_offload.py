"""Expert offload on a GB300 (moe_layer_forward_offload): each layer's routed
experts in pinned host memory, its 16 device slots filled through the LFU
cache.  Every layer call must match the resident layer call (chained
launches: the same router, sort and expert kernels) on the same input within
the block's tolerance with identical ids, the slots must hold exact copies of
the experts the cache says they hold, and the cache's hits and misses must
add up to the selections."""
import os

import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import E, H, I, K, from_dev_bf16, hidden, to_dev_bf16
from numerics import assert_close, bf16_bits_to_f64
from synth.device import DeviceLayer

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N_LAYERS, N_SLOTS, STEPS = 3, 16, 10


@pytest.fixture(scope="module")
def stack():
    bq.build_library()
    return [DeviceLayer(l, H, I, E, zipf=True) for l in range(N_LAYERS)]


def _dims():
    return bq.make_dims(H, I, E, K)


def _offload_weights(layer):
    """The layer with its routed experts copied to pinned host memory."""
    n = layer.n_experts * layer.stride
    host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    host.copy_(layer.buf[layer.experts_off:layer.experts_off + n])
    addr = dict(layer.addresses())
    addr["experts"] = host.data_ptr()
    return host, bq.layer_weights_from(_dims(), addr)


def test_offload_matches_resident(stack):
    os.environ["MOE_DECODE_FUSED"] = "0"
    try:
        ref = bq.Moe()
    finally:
        del os.environ["MOE_DECODE_FUSED"]
    moe = bq.Moe()
    cache = bq.ExpertCache(N_LAYERS, N_SLOTS)
    hosts, w_off, slots = [], [], []
    for L in stack:
        h, w = _offload_weights(L)
        hosts.append(h)
        w_off.append(w)
        slots.append(torch.empty(N_SLOTS * L.stride, dtype=torch.uint8, device="cuda"))
    w_res = [bq.layer_weights_from(_dims(), L.addresses()) for L in stack]
    ws = torch.empty(moe.workspace_bytes(_dims(), 1), dtype=torch.uint8, device="cuda")
    ws_ref = torch.empty_like(ws)
    ids = torch.empty((1, K), dtype=torch.int32, device="cuda")
    for s in range(STEPS):
        h = to_dev_bf16(hidden(1000, s, 1, rms=False))
        for l in range(N_LAYERS):
            h_in = from_dev_bf16(h)
            h_off = h.clone()
            moe.layer_forward_offload(h_off, cache, l, w_off[l], slots[l], ws)
            ref.layer_forward_residual(h, 1, w_res[l], ws_ref, ids_out=ids)
            torch.cuda.synchronize()
            assert moe.get_error() == bq.MOE_OK and ref.get_error() == bq.MOE_OK
            y_off = bf16_bits_to_f64(from_dev_bf16(h_off)) - bf16_bits_to_f64(h_in)
            y_ref = bf16_bits_to_f64(from_dev_bf16(h)) - bf16_bits_to_f64(h_in)
            assert_close(y_off, y_ref, f"step {s} layer {l}: offload against resident")
            # the slots hold what the cache says: exact copies of those experts
            sel = ids.cpu().numpy()[0]
            held = [cache.slot_expert(l, q) for q in range(N_SLOTS)]
            assert set(sel.tolist()) <= set(held), f"step {s} layer {l}: a selected expert is not in a slot"
            stride = stack[l].stride
            for e in sel[:2].tolist():
                q = held.index(e)
                assert torch.equal(slots[l][q * stride:(q + 1) * stride].cpu(),
                                   hosts[l][e * stride:(e + 1) * stride]), f"slot {q} is not expert {e}"
    for l in range(N_LAYERS):
        hits, misses = cache.stats(l)
        assert hits + misses == STEPS * K
        assert misses >= K  # the first step fills 8 slots
    cache.close()
    moe.close()
    ref.close()


def test_offload_rejects_bad_calls(stack):
    moe = bq.Moe()
    cache = bq.ExpertCache(1, N_SLOTS)
    host, w = _offload_weights(stack[0])
    slots = torch.empty(N_SLOTS * stack[0].stride, dtype=torch.uint8, device="cuda")
    ws = torch.empty(moe.workspace_bytes(_dims(), 1), dtype=torch.uint8, device="cuda")
    h = to_dev_bf16(hidden(1000, 0, 1, rms=False))
    with pytest.raises(bq.MoeError) as e:  # layer outside the cache
        moe.layer_forward_offload(h, cache, 1, w, slots, ws)
    assert e.value.status == bq.MOE_ERR_INVALID_ARG
    small = bq.ExpertCache(1, K - 1)  # fewer slots than one token selects
    with pytest.raises(bq.MoeError) as e:
        moe.layer_forward_offload(h, small, 0, w, slots, ws)
    assert e.value.status == bq.MOE_ERR_UNSUPPORTED
    small.close()
    cache.close()
    moe.close()
