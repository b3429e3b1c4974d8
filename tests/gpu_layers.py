"""Shared helpers of the GPU tests: device layers, calls through the C ABI,
oracle references (regenerated on the host from the same seeds)."""
from __future__ import annotations

import numpy as np

import bit_affine_quantized_gb300 as bq
from oracle import moe_oracle as O
from synth import gen
from synth.device import DeviceLayer

H, I, E, K = 2816, 704, 128, 8


def torch():
    import torch as _t
    return _t


def weights_of(layer: DeviceLayer, k: int = K) -> bq.LayerWeights:
    dims = bq.make_dims(layer.hidden, layer.inter, layer.n_experts, k)
    return bq.layer_weights_from(dims, layer.addresses())


def to_dev_bf16(bits: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def from_dev_bf16(x) -> np.ndarray:
    return x.cpu().numpy().view(np.uint16)


def workspace(moe: bq.Moe, w: bq.LayerWeights, n_tokens: int):
    t = torch()
    return t.empty(moe.workspace_bytes(w.dims, n_tokens), dtype=t.uint8, device="cuda")


def run_layer(moe: bq.Moe, layer: DeviceLayer, x_bits: np.ndarray, k: int = K):
    """moe_layer_forward; returns host copies (y bits, ids, logits, weights)."""
    t = torch()
    n = x_bits.shape[0]
    w = weights_of(layer, k)
    x = to_dev_bf16(x_bits)
    y = t.empty_like(x)
    ids = t.empty((n, k), dtype=t.int32, device="cuda")
    logits = t.empty((n, layer.n_experts), dtype=t.float32, device="cuda")
    wts = t.empty((n, k), dtype=t.float32, device="cuda")
    ws = workspace(moe, w, n)
    moe.layer_forward(x, n, w, y, ws, ids_out=ids, logits_out=logits, weights_out=wts)
    t.cuda.synchronize()
    status = moe.get_error()
    return {"y": from_dev_bf16(y), "ids": ids.cpu().numpy(), "logits": logits.cpu().numpy(),
            "weights": wts.cpu().numpy(), "status": status}


class HostExperts:
    """Lazily regenerated host copies of a layer's experts for the oracle."""

    def __init__(self, layer: DeviceLayer):
        self.layer = layer
        self.cache = {}

    def __call__(self, e: int):
        if e not in self.cache:
            self.cache[e] = self.layer.host_expert(e)
        return self.cache[e]


def oracle_layer(layer: DeviceLayer, x_bits, k, ids, experts: HostExperts | None = None):
    experts = experts or HostExperts(layer)
    rs, pes = layer.host_router_scales()
    return O.moe_block(x_bits, layer.host_router(), experts, layer.host_shared(), k,
                       layer.host_logit_bias(), ids=ids, router_scale=rs, per_expert_scale=pes)


def hidden(seed: int, chunk: int, n_tokens: int, hidden_dim: int = H, rms: bool = True) -> np.ndarray:
    return gen.hidden_states(seed, chunk, n_tokens, hidden_dim, rms_normalize=rms)
