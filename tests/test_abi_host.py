"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host-side checks answer before anything is launched."""
import ctypes

import pytest

import bit_affine_quantized_gb300 as bq
from synth import gen


@pytest.fixture(scope="module")
def lib():
    bq.build_library()
    return bq.load_library()


def _weights(dims, base=1 << 40, layout=None, stride=None, align=256):
    bl = gen.blob_layout(dims.hidden, dims.inter)
    layout = layout or {k: v for k, v in bl.items() if k not in ("bytes", "stride")}
    return bq.make_layer_weights(dims, base, base + 4096 * align, base + 8192 * align, base + (1 << 30),
                                 stride or bl["stride"], layout, base + (1 << 33))


def test_every_header_symbol_is_exported(lib):
    names = bq.header_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(8):
        s = lib.moe_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.moe_status_string(99).decode() == "unknown status"


def test_workspace_bytes(lib):
    d = bq.make_dims(2816, 704, 128, 8)
    sizes = [lib.moe_workspace_bytes(ctypes.byref(d), t) for t in (1, 2, 64, 128)]
    assert all(s > 0 and s % 256 == 0 for s in sizes)
    assert sizes == sorted(sizes)
    # h buffer alone: (T*k + T) * I fp16
    assert sizes[0] >= (8 + 1) * 704 * 2
    # the grouped path also holds fp32 expert outputs (T*k + T) * H
    assert sizes[3] >= (128 * 9) * 2816 * 4
    for t in (0, -1, 129):
        assert lib.moe_workspace_bytes(ctypes.byref(d), t) == 0
    for bad in (bq.make_dims(2816, 704, 128, 8, group=32), bq.make_dims(2800, 704, 128, 8),
                bq.make_dims(2816, 704, 4, 8), bq.make_dims(2816, 704, 129, 8), bq.make_dims(2816, 704, 128, 9),
                bq.make_dims(8192, 704, 128, 8)):
        assert lib.moe_workspace_bytes(ctypes.byref(bad), 1) == 0


def test_prompt_workspace_bytes(lib):
    """The whole-prompt layer's workspace: every sorted position's operand row
    (fp16 [T*k + T, H]), h row (fp16 [.., I]) and fp32 expert output row, the
    normalised rows and the routing; zero outside 1 <= n_rows <= 4096."""
    d = bq.make_dims(2816, 704, 128, 8)
    sizes = [lib.moe_prompt_workspace_bytes(ctypes.byref(d), t) for t in (1, 129, 1000, 4096)]
    assert all(s > 0 and s % 256 == 0 for s in sizes)
    assert sizes == sorted(sizes)
    npos = 4096 * 9
    assert sizes[3] >= npos * (2816 * 2 + 704 * 2 + 2816 * 4) + 4096 * 2816 * 2
    assert sizes[3] < 1 << 30
    for t in (0, -1, bq.MOE_PROMPT_MAX_ROWS + 1):
        assert lib.moe_prompt_workspace_bytes(ctypes.byref(d), t) == 0
    for bad in (bq.make_dims(2816, 704, 128, 8, group=32), bq.make_dims(2816, 704, 129, 8),
                bq.make_dims(8192, 704, 128, 8)):
        assert lib.moe_prompt_workspace_bytes(ctypes.byref(bad), 16) == 0
    # every supported small shape has a plan
    for dims in ((64, 64, 1, 1), (128, 64, 8, 2), (192, 128, 16, 8), (4096, 2048, 128, 8)):
        assert lib.moe_prompt_workspace_bytes(ctypes.byref(bq.make_dims(*dims)), 33) > 0, dims


def test_check_weights(lib):
    d = bq.make_dims(2816, 704, 128, 8)
    w = _weights(d)
    assert lib.moe_check_weights(ctypes.byref(w)) == bq.MOE_OK
    bad = _weights(d)
    bad.router.q = (1 << 40) + 8
    assert lib.moe_check_weights(ctypes.byref(bad)) == bq.MOE_ERR_INVALID_ARG
    bad = _weights(d)
    bad.layout.down_s += 16
    assert lib.moe_check_weights(ctypes.byref(bad)) == bq.MOE_ERR_INVALID_ARG
    bad = _weights(d, stride=3345408 - 256)
    assert lib.moe_check_weights(ctypes.byref(bad)) == bq.MOE_ERR_INVALID_ARG
    bad = _weights(d)
    bad.shared = None
    assert lib.moe_check_weights(ctypes.byref(bad)) == bq.MOE_ERR_INVALID_ARG
    bad = _weights(bq.make_dims(2816, 704, 128, 8, group=128))
    assert lib.moe_check_weights(ctypes.byref(bad)) == bq.MOE_ERR_UNSUPPORTED
    # optional vectors: null is fine, set they must be aligned
    for field, ok, misaligned in (("router_scale", 1 << 40, (1 << 40) + 8), ("per_expert_scale", 1 << 40, (1 << 40) + 2),
                                  ("post_norm", 1 << 40, (1 << 40) + 8), ("layer_scalar", 1 << 40, (1 << 40) + 2)):
        good = _weights(d)
        setattr(good, field, ok)
        assert lib.moe_check_weights(ctypes.byref(good)) == bq.MOE_OK, field
        bad = _weights(d)
        setattr(bad, field, misaligned)
        assert lib.moe_check_weights(ctypes.byref(bad)) == bq.MOE_ERR_INVALID_ARG, field
    assert lib.moe_check_weights(None) == bq.MOE_ERR_INVALID_ARG


def test_calls_without_handle_are_rejected(lib):
    d = bq.make_dims(2816, 704, 128, 8)
    w = _weights(d)
    V = ctypes.c_void_p
    assert lib.moe_layer_forward(None, V(1 << 40), 1, ctypes.byref(w), V(1 << 40), None, None, None, V(1 << 40),
                                 1 << 30, None) == bq.MOE_ERR_INVALID_ARG
    assert lib.moe_route_sort(None, V(1 << 40), 1, ctypes.byref(d), V(16), V(16), V(16), V(16),
                              None) == bq.MOE_ERR_INVALID_ARG
    layers = (bq.LayerWeights * 2)(w, w)
    assert lib.moe_layer_forward_stack(None, V(1 << 40), 2, layers, V(1 << 40), 1 << 30,
                                       None) == bq.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_prompt(None, V(1 << 40), 300, ctypes.byref(w), None, None, None, None, V(1 << 40),
                                        1 << 30, None) == bq.MOE_ERR_INVALID_ARG
    assert lib.moe_get_error(None, None) == bq.MOE_ERR_INVALID_ARG
    assert lib.moe_destroy(None) == bq.MOE_ERR_INVALID_ARG
    hw = bq.make_head_weights(262144, 2816, 1 << 40, 1 << 41, 1 << 42)
    assert lib.moe_head_forward(None, V(1 << 40), 1, ctypes.byref(hw), 30.0, V(1 << 40), None,
                                None) == bq.MOE_ERR_INVALID_ARG
    assert lib.moe_embed(None, V(1 << 40), 1, ctypes.byref(hw), V(1 << 40), None) == bq.MOE_ERR_INVALID_ARG


def test_create_without_gpu_fails_cleanly(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib.moe_create(ctypes.byref(h))
    assert st == bq.MOE_ERR_CUDA and not h.value
