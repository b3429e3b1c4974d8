"""Python binding of libmoe_gb300 (include/moe.h): argument marshalling only.

Every step of the MoE block runs in the CUDA library; this module turns
torch tensors into device pointers and status codes into exceptions.  It
fails loudly when the compiled library is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import LIB_PATH, build as build_library

__all__ = [
    "MoeError", "Dims", "QMat", "BlobLayout", "LayerWeights", "Moe", "load_library", "header_symbols",
    "MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_CUDA", "MOE_ERR_BAD_EXPERT_ID",
    "MOE_ERR_TIMEOUT", "MOE_ERR_NONFINITE", "MOE_ERR_WORKSPACE", "build_library", "static_get_error",
    "layer_forward_static", "ExpertCache",
]

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_BAD_EXPERT_ID = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_NONFINITE = 6
MOE_ERR_WORKSPACE = 7
MOE_PROMPT_MAX_ROWS = 4096

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("group", ctypes.c_int)]


class QMat(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


_BLOB_FIELDS = ("gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q", "down_s", "down_b")


class BlobLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in _BLOB_FIELDS]


class LayerWeights(ctypes.Structure):
    _fields_ = [("dims", Dims), ("router", QMat), ("experts", ctypes.c_void_p), ("expert_stride", ctypes.c_size_t),
                ("layout", BlobLayout), ("shared", ctypes.c_void_p), ("logit_bias", ctypes.c_void_p),
                ("router_scale", ctypes.c_void_p), ("per_expert_scale", ctypes.c_void_p),
                ("post_norm", ctypes.c_void_p), ("layer_scalar", ctypes.c_void_p)]


class HeadWeights(ctypes.Structure):
    _fields_ = [("vocab", ctypes.c_int), ("hidden", ctypes.c_int), ("w", QMat)]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)} ({status})")


_lib = None


def load_library(path: str = LIB_PATH):
    """dlopen the in-tree library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (bit_affine_quantized_gb300.build_library())")
    lib = ctypes.CDLL(path)
    P, I, Z, V = ctypes.POINTER, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    proto = {
        "moe_status_string": (ctypes.c_char_p, [I]),
        "moe_create": (I, [P(V)]),
        "moe_destroy": (I, [V]),
        "moe_check_weights": (I, [P(LayerWeights)]),
        "moe_workspace_bytes": (Z, [P(Dims), I]),
        "moe_router_topk": (I, [V, V, I, P(LayerWeights), V, V, V, V, Z, V]),
        "moe_route_sort": (I, [V, V, I, P(Dims), V, V, V, V, V]),
        "moe_expert_ffn": (I, [V, V, I, V, V, P(LayerWeights), I, V, V, Z, V]),
        "moe_layer_forward": (I, [V, V, I, P(LayerWeights), V, V, V, V, V, Z, V]),
        "moe_layer_forward_residual": (I, [V, V, I, P(LayerWeights), V, V, V, V, V, Z, V]),
        "moe_selftest_wait_timeout": (I, [V, ctypes.c_ulonglong, V]),
        "moe_set_trace": (I, [V, V, I]),
        "moe_layer_forward_static": (I, [V, P(LayerWeights), V, V, V, V, V]),
        "moe_static_get_error": (I, [P(I)]),
        "moe_selftest_skip_arrival": (I, [V, I, ctypes.c_ulonglong]),
        "moe_layer_forward_stack": (I, [V, V, I, P(LayerWeights), V, Z, V]),
        "moe_get_error": (I, [V, P(I)]),
        "moe_head_forward": (I, [V, V, I, P(HeadWeights), ctypes.c_float, V, V, V]),
        "moe_embed": (I, [V, V, I, P(HeadWeights), V, V]),
        "moe_dense_forward": (I, [V, V, I, P(HeadWeights), V, V, V]),
        "moe_cache_create": (I, [I, I, P(V)]),
        "moe_cache_destroy": (None, [V]),
        "moe_cache_lookup": (I, [V, I, V, I, V, V, V, P(I)]),
        "moe_cache_stats": (I, [V, I, P(ctypes.c_longlong), P(ctypes.c_longlong)]),
        "moe_cache_slot_expert": (I, [V, I, I]),
        "moe_cache_slots": (I, [V]),
        "moe_layer_forward_offload": (I, [V, V, I, V, P(LayerWeights), V, V, Z, V]),
        "moe_prompt_workspace_bytes": (Z, [P(Dims), I]),
        "moe_layer_forward_prompt": (I, [V, V, I, P(LayerWeights), V, V, V, V, V, Z, V]),
    }
    for name, (res, args) in proto.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _status_string(status: int) -> str:
    try:
        return load_library().moe_status_string(status).decode()
    except Exception:  # library not loadable: still report the number
        return "status"


def header_symbols(path: str = HEADER) -> list[str]:
    """Names of the functions include/moe.h declares."""
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def _ptr(t):
    """Device (or host) address of a tensor, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_dims(hidden: int, inter: int, n_experts: int, top_k: int, group: int = 64) -> Dims:
    return Dims(hidden, inter, n_experts, top_k, group)


def make_layer_weights(dims: Dims, router_q: int, router_s: int, router_b: int, experts: int, expert_stride: int,
                       layout: dict, shared: int, logit_bias=None, router_scale=None,
                       per_expert_scale=None, post_norm=None, layer_scalar=None) -> LayerWeights:
    """LayerWeights from device addresses; `layout` maps gate_q .. down_b to byte offsets.

    Optional entries (device address, CUDA tensor or None): logit_bias fp32
    [E]; router_scale bf16 [H] and per_expert_scale fp32 [E], the router's
    learned scales; post_norm bf16 [H] and layer_scalar fp32 [1], the layer
    tail, which only the residual calls apply."""
    return LayerWeights(dims, QMat(router_q, router_s, router_b), experts, expert_stride,
                        BlobLayout(*[layout[n] for n in _BLOB_FIELDS]), shared, _ptr(logit_bias),
                        _ptr(router_scale), _ptr(per_expert_scale), _ptr(post_norm), _ptr(layer_scalar))


def make_head_weights(vocab: int, hidden: int, q: int, scales: int, biases: int) -> HeadWeights:
    """HeadWeights from device addresses (or CUDA tensors) of the tied head."""
    return HeadWeights(vocab, hidden, QMat(_ptr(q), _ptr(scales), _ptr(biases)))


def layer_forward_static(x, w: LayerWeights, y, ids_out=None, logits_out=None, weights_out=None, stream=None):
    """moe_layer_forward_static: one token, no handle, no workspace.

    For hosts that cannot allocate device memory; the library's scratch for
    this call is a fixed static device array (see include/moe.h)."""
    st = load_library().moe_layer_forward_static(_ptr(x), ctypes.byref(w), _ptr(y), _ptr(ids_out), _ptr(logits_out),
                                                 _ptr(weights_out), _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_layer_forward_static")


def static_get_error() -> int:
    """moe_static_get_error: the device-side status of the static calls on the
    current device since the last read (waits for the device; clears it)."""
    st = ctypes.c_int(0)
    rc = load_library().moe_static_get_error(ctypes.byref(st))
    if rc != MOE_OK:
        raise MoeError(rc, "moe_static_get_error")
    return st.value


class ExpertCache:
    """Host-side slot policy of the expert offload (moe_cache_*): n_layers
    layers of n_slots slots, least frequently used eviction, recency breaking
    ties."""

    def __init__(self, n_layers: int, n_slots: int = 16):
        self.lib = load_library()
        self.c = ctypes.c_void_p()
        st = self.lib.moe_cache_create(n_layers, n_slots, ctypes.byref(self.c))
        if st:
            raise MoeError(st, "moe_cache_create")
        self.n_layers, self.n_slots = n_layers, n_slots

    def lookup(self, layer: int, ids):
        """One step for a sequence of selected expert ids: (slots, [(slot,
        expert) loads])."""
        n = len(ids)
        a = (ctypes.c_int32 * n)(*ids)
        sl, ls, li = (ctypes.c_int32 * n)(), (ctypes.c_int32 * n)(), (ctypes.c_int32 * n)()
        nl = ctypes.c_int()
        st = self.lib.moe_cache_lookup(self.c, layer, a, n, sl, ls, li, ctypes.byref(nl))
        if st:
            raise MoeError(st, "moe_cache_lookup")
        return list(sl), [(ls[i], li[i]) for i in range(nl.value)]

    def stats(self, layer: int):
        h, m = ctypes.c_longlong(), ctypes.c_longlong()
        st = self.lib.moe_cache_stats(self.c, layer, ctypes.byref(h), ctypes.byref(m))
        if st:
            raise MoeError(st, "moe_cache_stats")
        return h.value, m.value

    def slot_expert(self, layer: int, slot: int) -> int:
        return self.lib.moe_cache_slot_expert(self.c, layer, slot)

    def close(self):
        if self.c:
            self.lib.moe_cache_destroy(self.c)
            self.c = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Moe:
    """One library handle (device error word + router counter) on the current device."""

    def __init__(self):
        self.lib = load_library()
        h = ctypes.c_void_p()
        st = self.lib.moe_create(ctypes.byref(h))
        if st != MOE_OK:
            raise MoeError(st, "moe_create")
        self.h = h

    def close(self):
        if self.h:
            self.lib.moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st, what):
        if st != MOE_OK:
            raise MoeError(st, what)

    def workspace_bytes(self, dims: Dims, n_tokens: int) -> int:
        return int(self.lib.moe_workspace_bytes(ctypes.byref(dims), n_tokens))

    def router_topk(self, x, n_tokens, w: LayerWeights, ids, weights, ws, logits=None, stream=None):
        self._check(self.lib.moe_router_topk(self.h, _ptr(x), n_tokens, ctypes.byref(w), _ptr(logits), _ptr(ids),
                                             _ptr(weights), _ptr(ws), ws.numel() * ws.element_size(),
                                             _stream(stream)), "moe_router_topk")

    def route_sort(self, ids, n_tokens, dims: Dims, counts, offsets, perm, pos, stream=None):
        self._check(self.lib.moe_route_sort(self.h, _ptr(ids), n_tokens, ctypes.byref(dims), _ptr(counts),
                                            _ptr(offsets), _ptr(perm), _ptr(pos), _stream(stream)), "moe_route_sort")

    def expert_ffn(self, x, n_tokens, ids, weights, w: LayerWeights, y, ws, include_shared=True, stream=None):
        self._check(self.lib.moe_expert_ffn(self.h, _ptr(x), n_tokens, _ptr(ids), _ptr(weights), ctypes.byref(w),
                                            1 if include_shared else 0, _ptr(y), _ptr(ws),
                                            ws.numel() * ws.element_size(), _stream(stream)), "moe_expert_ffn")

    def layer_forward(self, x, n_tokens, w: LayerWeights, y, ws, ids_out=None, logits_out=None, weights_out=None,
                      stream=None):
        self._check(self.lib.moe_layer_forward(self.h, _ptr(x), n_tokens, ctypes.byref(w), _ptr(y), _ptr(ids_out),
                                               _ptr(logits_out), _ptr(weights_out), _ptr(ws),
                                               ws.numel() * ws.element_size(), _stream(stream)), "moe_layer_forward")

    def layer_forward_residual(self, hidden, n_tokens, w: LayerWeights, ws, y_out=None, x_out=None, ids_out=None,
                               logits_out=None, stream=None):
        """One layer of a residual stack: hidden <- hidden + MoE(rmsnorm(hidden))
        in place, or with the layer's tail hidden <- lambda * (hidden +
        post_norm * y / rms(y)); y_out / x_out receive the block output and
        its normalised input."""
        self._check(self.lib.moe_layer_forward_residual(self.h, _ptr(hidden), n_tokens, ctypes.byref(w), _ptr(y_out),
                                                        _ptr(x_out), _ptr(ids_out), _ptr(logits_out), _ptr(ws),
                                                        ws.numel() * ws.element_size(), _stream(stream)),
                    "moe_layer_forward_residual")

    def prompt_workspace_bytes(self, dims: Dims, n_rows: int) -> int:
        return int(self.lib.moe_prompt_workspace_bytes(ctypes.byref(dims), n_rows))

    def layer_forward_prompt(self, hidden, n_rows, w: LayerWeights, ws, y_out=None, x_out=None, ids_out=None,
                             logits_out=None, stream=None):
        """One residual layer on a whole prompt of up to 4096 rows
        (moe_layer_forward_prompt): the same function as
        layer_forward_residual, row by row, with the expert work grouped over
        all rows; ws of prompt_workspace_bytes(dims, n_rows) bytes."""
        self._check(self.lib.moe_layer_forward_prompt(self.h, _ptr(hidden), n_rows, ctypes.byref(w), _ptr(y_out),
                                                      _ptr(x_out), _ptr(ids_out), _ptr(logits_out), _ptr(ws),
                                                      ws.numel() * ws.element_size(), _stream(stream)),
                    "moe_layer_forward_prompt")

    def layer_forward_stack(self, hidden, layers, ws, stream=None):
        """Single-token layers of a residual stack in one call (hidden bf16 [H]
        updated in place); `layers` is a sequence of LayerWeights."""
        arr = (LayerWeights * len(layers))(*layers)
        self._check(self.lib.moe_layer_forward_stack(self.h, _ptr(hidden), len(layers), arr, _ptr(ws),
                                                     ws.numel() * ws.element_size(), _stream(stream)),
                    "moe_layer_forward_stack")

    def layer_forward_offload(self, hidden, cache: "ExpertCache", layer: int, w: LayerWeights, slots, ws,
                              stream=None):
        """One single-token residual layer with its routed experts in host
        memory (w.experts: pinned host memory), filling the layer's device
        `slots` through `cache` (moe_layer_forward_offload)."""
        self._check(self.lib.moe_layer_forward_offload(self.h, cache.c, layer, _ptr(hidden), ctypes.byref(w),
                                                       _ptr(slots), _ptr(ws), ws.numel() * ws.element_size(),
                                                       _stream(stream)), "moe_layer_forward_offload")

    def head_forward(self, x, n_tokens, hw: HeadWeights, softcap: float = 30.0, logits=None, tokens=None,
                     stream=None):
        """The tied head on n_tokens (<= 8) rows of x: logits (fp32 [T, V])
        and/or greedy tokens (int32 [T])."""
        self._check(self.lib.moe_head_forward(self.h, _ptr(x), n_tokens, ctypes.byref(hw), ctypes.c_float(softcap),
                                              _ptr(logits), _ptr(tokens), _stream(stream)), "moe_head_forward")

    def dense_forward(self, x, n_tokens, w: HeadWeights, y=None, y32=None, stream=None):
        """A dense 4-bit affine projection y = W x on n_tokens (<= 8) rows:
        bf16 [T, N] and/or fp32 [T, N] outputs."""
        self._check(self.lib.moe_dense_forward(self.h, _ptr(x), n_tokens, ctypes.byref(w), _ptr(y), _ptr(y32),
                                               _stream(stream)), "moe_dense_forward")

    def embed(self, ids, n, hw: HeadWeights, out, stream=None):
        """Tied embedding rows (bf16 [n, H]) of int32 token ids on the device."""
        self._check(self.lib.moe_embed(self.h, _ptr(ids), n, ctypes.byref(hw), _ptr(out), _stream(stream)),
                    "moe_embed")

    def set_trace(self, buffer=None, n_launches: int = 0):
        """Record per-launch device timestamps into `buffer` (u64 x 4 x n)."""
        self._check(self.lib.moe_set_trace(self.h, _ptr(buffer), n_launches), "moe_set_trace")

    def selftest_wait_timeout(self, limit_ns: int, stream=None):
        self._check(self.lib.moe_selftest_wait_timeout(self.h, limit_ns, _stream(stream)), "moe_selftest_wait_timeout")

    def selftest_skip_arrival(self, block: int, limit_ns: int):
        """Arms the next fused single-token launch: `block` withholds its
        barrier arrival, every wait gives up after limit_ns (failure test)."""
        self._check(self.lib.moe_selftest_skip_arrival(self.h, block, limit_ns), "moe_selftest_skip_arrival")

    def get_error(self) -> int:
        st = ctypes.c_int(0)
        self._check(self.lib.moe_get_error(self.h, ctypes.byref(st)), "moe_get_error")
        return st.value


def layer_weights_from(dims: Dims, addr: dict) -> LayerWeights:
    """LayerWeights from a dict with router_q/router_s/router_b/experts/stride/
    shared/layout entries and optional logit_bias/router_scale/per_expert_scale/
    post_norm/layer_scalar entries (device addresses and byte offsets)."""
    return make_layer_weights(dims, addr["router_q"], addr["router_s"], addr["router_b"], addr["experts"],
                              addr["stride"], addr["layout"], addr["shared"], addr.get("logit_bias"),
                              addr.get("router_scale"), addr.get("per_expert_scale"), addr.get("post_norm"),
                              addr.get("layer_scalar"))
