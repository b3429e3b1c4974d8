"""Synthetic MoE layers materialised in device memory.

The packed codes (the bulk of the bytes) are written by the device word
filler (``gpu_fill.cu``), the scales/biases and router come from the host
generator in ``gen.py``; both use the same counter-based streams, so a host
copy of any tensor can be regenerated bit-exactly for the oracle.

Layout of one layer's buffer (byte offsets, all 256-aligned):
  [router q | router scales | router biases] [E routed blobs, fixed stride]
  [shared blob]
with the blob layout of ``gen.blob_layout``.
"""
from __future__ import annotations

import concurrent.futures
import ctypes
import os
import subprocess

import numpy as np

from . import gen

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libsynth_gpu.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

_lib = None


def build(force: bool = False) -> str:
    src = os.path.join(HERE, "gpu_fill.cu")
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(src):
        return LIB_PATH
    os.makedirs(os.path.dirname(LIB_PATH), exist_ok=True)
    tmp = LIB_PATH + ".tmp"
    cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", src, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"synth build failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            build()
        lib = ctypes.CDLL(LIB_PATH)
        lib.synth_fill_words.restype = ctypes.c_int
        lib.synth_fill_words.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_ulonglong, ctypes.c_void_p]
        _lib = lib
    return _lib


def fill_words(addr: int, n_words: int, key: int, stream: int = 0) -> None:
    st = _load().synth_fill_words(ctypes.c_void_p(addr), n_words, key, ctypes.c_void_p(stream))
    if st != 0:
        raise RuntimeError(f"synth_fill_words failed ({st})")


class DeviceHead:
    """The synthetic tied 4-bit head [vocab, hidden] on the device: codes from
    the device filler, scales and biases generated on the host (the same
    values as gen.head_weights)."""

    def __init__(self, seed: int, vocab: int, hidden: int, device="cuda"):
        import torch
        self.seed, self.vocab, self.hidden = seed, vocab, hidden
        ng = hidden // gen.GROUP
        self.q = torch.empty(vocab * hidden // 8, dtype=torch.int32, device=device)
        stream = torch.cuda.current_stream(self.q.device).cuda_stream
        fill_words(self.q.data_ptr(), vocab * hidden // 8,
                   gen.weight_key(seed, gen.HEAD_ID, gen.MAT_HEAD, gen.FIELD_Q), stream)
        s, b = self._scale_bias()
        self.s = torch.from_numpy(s.reshape(-1).view(np.int16).copy()).to(device)
        self.b = torch.from_numpy(b.reshape(-1).view(np.int16).copy()).to(device)
        assert self.s.numel() == vocab * ng
        torch.cuda.synchronize(self.q.device)

    def _scale_bias(self):
        # the generator's scales and biases without its codes (those come from the device filler)
        ng = self.hidden // gen.GROUP
        u = gen.uniform(gen.weight_key(self.seed, gen.HEAD_ID, gen.MAT_HEAD, gen.FIELD_S), self.vocab * ng)
        z = gen.normal(gen.weight_key(self.seed, gen.HEAD_ID, gen.MAT_HEAD, gen.FIELD_B), self.vocab * ng)
        s_bits = gen.to_bf16_bits((0.5 + u) / (8.0 * np.sqrt(float(self.hidden))))
        s = gen.bf16_bits_to_f64(s_bits)
        b_bits = gen.to_bf16_bits(-8.0 * s + (0.01 * s) * z)
        return s_bits, b_bits

    def addresses(self):
        return self.q.data_ptr(), self.s.data_ptr(), self.b.data_ptr()

    def host_rows(self, rows=None) -> dict:
        """Host copy of the given rows (all rows if None), regenerated from the seed."""
        return gen.head_weights(self.seed, self.vocab, self.hidden, rows)


class DeviceLayer:
    """All weights of one synthetic MoE layer in one device buffer."""

    def __init__(self, layer_seed: int, hidden: int, inter: int, n_experts: int, device="cuda",
                 zipf: bool = False, threads: int = 8, router_scales: bool = False, tail: bool = False):
        import torch
        self.seed = layer_seed
        self.hidden, self.inter, self.n_experts = hidden, inter, n_experts
        self.rl = gen.router_layout(n_experts, hidden)
        self.bl = gen.blob_layout(hidden, inter)
        self.stride = self.bl["stride"]
        self.router_off = 0
        self.experts_off = gen.align_up(self.rl["bytes"], 256)
        self.shared_off = self.experts_off + n_experts * self.stride
        total = self.shared_off + self.stride
        self.buf = torch.empty(total, dtype=torch.uint8, device=device)
        base = self.buf.data_ptr()
        stream = torch.cuda.current_stream(self.buf.device).cuda_stream

        # router (small): host generated
        r = gen.router_weights(layer_seed, n_experts, hidden)
        self._h2d(self.router_off + self.rl["q"], r["q"])
        self._h2d(self.router_off + self.rl["s"], r["s"])
        self._h2d(self.router_off + self.rl["b"], r["b"])

        # packed 4-bit codes: device filler, same stream keys as gen.expert_matrix
        blobs = list(range(n_experts)) + [gen.SHARED_ID]
        for idx, e in enumerate(blobs):
            blob = self.experts_off + idx * self.stride
            for name, m, (n, k) in self._mats():
                key = gen.weight_key(layer_seed, e, m, gen.FIELD_Q)
                fill_words(base + blob + self.bl[f"{name}_q"], gen.qmat_words(n, k, 4), key, stream)

        # scales/biases: host generated per matrix, staged as one tensor per
        # sub-tensor kind and scattered with one strided copy each
        mats = self._mats()
        per = inter * (hidden // gen.GROUP)
        def one(e):
            out = []
            for name, m, (n, k) in mats:
                s, b = gen.expert_scale_bias(layer_seed, e, m, n, k)
                out.append((s.reshape(-1), b.reshape(-1)))
            return out
        with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
            results = list(ex.map(one, blobs))
        nb = len(blobs)
        view = self.buf[self.experts_off:self.experts_off + nb * self.stride].view(nb, self.stride)
        for mi, (name, m, (n, k)) in enumerate(mats):
            for fi, field in enumerate(("s", "b")):
                host = np.stack([results[i][mi][fi] for i in range(nb)]).view(np.uint8)
                off = self.bl[f"{name}_{field}"]
                view[:, off:off + 2 * per].copy_(torch.from_numpy(host).to(self.buf.device))
        self.logit_bias = None
        if zipf:
            self.logit_bias = torch.from_numpy(gen.zipf_logit_bias(layer_seed, n_experts)).to(self.buf.device)
        self.router_scale = self.per_expert_scale = None
        if router_scales:
            rs, pes = gen.router_scales(layer_seed, n_experts, hidden)
            self.router_scale = torch.from_numpy(rs.view(np.int16).copy()).to(self.buf.device)
            self.per_expert_scale = torch.from_numpy(pes).to(self.buf.device)
        self.post_norm = self.layer_scalar = None
        if tail:
            g, lam = gen.layer_tail(layer_seed, hidden)
            self.post_norm = torch.from_numpy(g.view(np.int16).copy()).to(self.buf.device)
            self.layer_scalar = torch.tensor([lam], dtype=torch.float32, device=self.buf.device)
        torch.cuda.synchronize(self.buf.device)

    def _mats(self):
        H, I = self.hidden, self.inter
        return (("gate", gen.MAT_GATE, (I, H)), ("up", gen.MAT_UP, (I, H)), ("down", gen.MAT_DOWN, (H, I)))

    def _h2d(self, off: int, arr: np.ndarray) -> None:
        import torch
        raw = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
        self.buf[off:off + raw.size].copy_(torch.from_numpy(raw).to(self.buf.device))

    # addresses for the C ABI
    def addresses(self) -> dict:
        base = self.buf.data_ptr()
        return {
            "router_q": base + self.router_off + self.rl["q"],
            "router_s": base + self.router_off + self.rl["s"],
            "router_b": base + self.router_off + self.rl["b"],
            "experts": base + self.experts_off,
            "stride": self.stride,
            "shared": base + self.shared_off,
            "layout": {k: v for k, v in self.bl.items() if k not in ("bytes", "stride")},
            "logit_bias": None if self.logit_bias is None else self.logit_bias.data_ptr(),
            "router_scale": None if self.router_scale is None else self.router_scale.data_ptr(),
            "per_expert_scale": None if self.per_expert_scale is None else self.per_expert_scale.data_ptr(),
            "post_norm": None if self.post_norm is None else self.post_norm.data_ptr(),
            "layer_scalar": None if self.layer_scalar is None else self.layer_scalar.data_ptr(),
        }

    # host copies for the oracle (regenerated, never read back from the device)
    def host_router(self) -> dict:
        return gen.router_weights(self.seed, self.n_experts, self.hidden)

    def host_expert(self, e: int) -> dict:
        return gen.expert_weights(self.seed, e, self.hidden, self.inter)

    def host_shared(self) -> dict:
        return gen.expert_weights(self.seed, gen.SHARED_ID, self.hidden, self.inter)

    def host_router_scales(self):
        """(router_scale bf16 bits [H], per_expert_scale float32 [E]), or (None, None)."""
        if self.router_scale is None:
            return None, None
        return gen.router_scales(self.seed, self.n_experts, self.hidden)

    def host_layer_tail(self):
        """(post_norm bf16 bits [H], layer_scalar float32), or (None, None)."""
        if self.post_norm is None:
            return None, None
        return gen.layer_tail(self.seed, self.hidden)

    def host_logit_bias(self):
        return None if self.logit_bias is None else gen.zipf_logit_bias(self.seed, self.n_experts)
