"""Full-size stacks, in the configuration the benchmark runs them: 30
independent layers (seeds 0..29, all 30 x 129 experts resident in HBM), the
residual stream carried through moe_layer_forward_residual, every layer call
one launch of the fused kernel, the layer calls of a step captured in one CUDA
graph (programmatic dependent launch between them).

Each layer writes its normalised input, logits, ids and output to buffers of
its own, so the checks need no extra launches inside the step:
- the residual stream is the exact bf16 chain h_{l+1} = bf16(h_l + y_l) of the
  outputs, and each normalised input is rmsnorm_no_scale of its h_l;
- ids are the top-k of the layer's own fp32 logits (bit-exact);
- sampled layers match the oracle run on the GPU's input and ids (teacher
  forcing), within the block's tolerance.
"""
import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import E, H, I, K, HostExperts, from_dev_bf16, hidden, to_dev_bf16
from numerics import assert_close, bf16_bits_to_f64
from oracle import moe_oracle as O
from synth.device import DeviceLayer

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N_LAYERS = 30


@pytest.fixture(scope="module")
def stack():
    bq.build_library()
    # Zipf offsets on every layer (the prefill stack); the decode stack runs the
    # same weights without them
    return [DeviceLayer(l, H, I, E, zipf=True) for l in range(N_LAYERS)]


def _weights(layer, with_bias: bool):
    addr = dict(layer.addresses())
    if not with_bias:
        addr["logit_bias"] = None
    return bq.layer_weights_from(bq.make_dims(H, I, E, K), addr)


def _run_stack(stack, n_tokens: int, steps: int, zipf: bool):
    moe = bq.Moe()
    ws_list = [_weights(L, zipf) for L in stack]
    ws = torch.empty(moe.workspace_bytes(ws_list[0].dims, n_tokens), dtype=torch.uint8, device="cuda")
    h = torch.empty((n_tokens, H), dtype=torch.int16, device="cuda")
    xo = torch.empty((N_LAYERS, n_tokens, H), dtype=torch.int16, device="cuda")
    yo = torch.empty_like(xo)
    ids = torch.empty((N_LAYERS, n_tokens, K), dtype=torch.int32, device="cuda")
    logits = torch.empty((N_LAYERS, n_tokens, E), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def body():
        for l, w in enumerate(ws_list):
            moe.layer_forward_residual(h, n_tokens, w, ws, y_out=yo[l], x_out=xo[l], ids_out=ids[l],
                                       logits_out=logits[l], stream=stream)

    with torch.cuda.stream(stream):
        h.copy_(to_dev_bf16(hidden(1000, 0, n_tokens, rms=False)))
        body()  # warm the path outside the capture
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            body()
    torch.cuda.synchronize()
    results = []
    for s in range(steps):
        h0 = hidden(1000, s, n_tokens, rms=False)
        with torch.cuda.stream(stream):
            h.copy_(to_dev_bf16(h0))
            graph.replay()
        torch.cuda.synchronize()
        assert moe.get_error() == bq.MOE_OK
        results.append({"h0": h0, "h": from_dev_bf16(h), "x": from_dev_bf16(xo).reshape(N_LAYERS, n_tokens, H),
                        "y": from_dev_bf16(yo).reshape(N_LAYERS, n_tokens, H), "ids": ids.cpu().numpy(),
                        "logits": logits.cpu().numpy()})
    moe.close()
    return results


def _check_step(stack, r, n_tokens: int, zipf: bool, sampled):
    h = r["h0"]
    for l in range(N_LAYERS):
        xr = bf16_bits_to_f64(O.rmsnorm_no_scale(h))
        # fp32 on the device against fp64: at most one bf16 rounding step apart
        assert np.all(np.abs(bf16_bits_to_f64(r["x"][l]) - xr) <= 2.0 ** -7 * np.abs(xr)), f"layer {l}: rmsnorm"
        assert np.array_equal(r["ids"][l], O.select_top_k(r["logits"][l], K)), f"layer {l}: ids"
        if l in sampled:
            L = stack[l]
            ref = O.moe_block(r["x"][l], L.host_router(), HostExperts(L), L.host_shared(), K,
                              L.host_logit_bias() if zipf else None, ids=r["ids"][l])
            assert_close(r["logits"][l], ref["logits"], f"layer {l}: logits")
            assert_close(bf16_bits_to_f64(r["y"][l]), ref["y"], f"layer {l}: y")
        h = O.residual_add(h, r["y"][l])
    assert np.array_equal(r["h"], h), "residual stream differs from the chain of the layer outputs"


def test_decode_stack_30_layers(stack):
    """The bench workload: one token per step through 30 layers, 3 steps."""
    results = _run_stack(stack, 1, 3, zipf=False)
    for s, r in enumerate(results):
        _check_step(stack, r, 1, False, sampled={0, 14, 29} if s == 0 else {29})


def test_prefill_stack_30_layers(stack):
    """A 128-token chunk through the 30 layers with per-layer Zipf offsets
    (one chunk of the 32-chunk prefill workload); first and last layer
    against the oracle."""
    results = _run_stack(stack, 128, 1, zipf=True)
    _check_step(stack, results[0], 128, True, sampled={0, 29})


def _stack_vs_layers(stack, n_layers: int, steps: int):
    moe = bq.Moe()
    ws_list = [_weights(L, False) for L in stack[:n_layers]]
    ws = torch.empty(moe.workspace_bytes(ws_list[0].dims, 1), dtype=torch.uint8, device="cuda")
    h_ref = torch.empty((1, H), dtype=torch.int16, device="cuda")
    h_st = torch.empty_like(h_ref)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        h_st.copy_(to_dev_bf16(hidden(1000, 0, 1, rms=False)))
        moe.layer_forward_stack(h_st, ws_list, ws, stream=stream)  # warm the path outside the capture
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            moe.layer_forward_stack(h_st, ws_list, ws, stream=stream)
    torch.cuda.synchronize()
    for s in range(steps):
        h0 = to_dev_bf16(hidden(1000, s, 1, rms=False))
        with torch.cuda.stream(stream):
            h_ref.copy_(h0)
            for w in ws_list:
                moe.layer_forward_residual(h_ref, 1, w, ws, stream=stream)
            h_st.copy_(h0)
            graph.replay()
        torch.cuda.synchronize()
        assert moe.get_error() == bq.MOE_OK
        assert torch.equal(h_ref, h_st), f"step {s}: the stack call differs from the layer calls"
    moe.close()


def test_stack_call_30_layers_matches_layer_calls(stack):
    """moe_layer_forward_stack (one call for the decode step, captured in a
    graph) against 30 moe_layer_forward_residual calls: bit-identical
    residual streams over 3 replays."""
    _stack_vs_layers(stack, N_LAYERS, 3)


@pytest.mark.parametrize("n_layers", [1, 2, 5])
def test_stack_call_short_stacks(stack, n_layers):
    _stack_vs_layers(stack, n_layers, 2)
