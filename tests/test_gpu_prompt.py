"""The whole-prompt layer (moe_layer_forward_prompt) on a GB300 against the
float64 oracle, through the C ABI.

As elsewhere: the normalised input within one bf16 step of the oracle's
rmsnorm, ids equal to the oracle's top-k of the GPU's own fp32 logits, the
logits against the oracle's router at the block's tolerance, the block
output against the oracle run on the GPU's ids (teacher forcing), and the new
residual stream equal to bf16(h + y) bit for bit.  At the full prompt size
(4096 rows) the routing is checked on every row, the output on sampled rows
against the oracle and on every row against the chunked layer calls (the
fused multi-token kernel, itself checked against the oracle)."""
import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import E, H, I, K, from_dev_bf16, hidden, oracle_layer, to_dev_bf16, weights_of, workspace
from numerics import MAX_ABS_VS_RMS, MEAN_REL, assert_close, bf16_bits_to_f64, errors
from oracle import moe_oracle as O
from synth.device import DeviceLayer

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def moe():
    bq.build_library()
    m = bq.Moe()
    yield m
    m.close()


@pytest.fixture(scope="module")
def layer0():
    return DeviceLayer(0, H, I, E)


@pytest.fixture(scope="module")
def layer0_zipf():
    return DeviceLayer(0, H, I, E, zipf=True)


def _prompt_ws(moe, w, n):
    return torch.empty(moe.prompt_workspace_bytes(w.dims, n), dtype=torch.uint8, device="cuda")


def run_prompt(moe, layer, h_bits, k=K, w=None, ws=None):
    n = h_bits.shape[0]
    w = w or weights_of(layer, k)
    h = to_dev_bf16(h_bits)
    y = torch.empty_like(h)
    xo = torch.empty_like(h)
    ids = torch.empty((n, k), dtype=torch.int32, device="cuda")
    logits = torch.empty((n, layer.n_experts), dtype=torch.float32, device="cuda")
    ws = ws if ws is not None else _prompt_ws(moe, w, n)
    moe.layer_forward_prompt(h, n, w, ws, y_out=y, x_out=xo, ids_out=ids, logits_out=logits)
    torch.cuda.synchronize()
    return {"h": from_dev_bf16(h), "y": from_dev_bf16(y), "x": from_dev_bf16(xo), "ids": ids.cpu().numpy(),
            "logits": logits.cpu().numpy(), "status": moe.get_error()}


def check_block(out, layer, h_bits, k, rows=None):
    """Routing on every row; y on `rows` (all if None) against the oracle."""
    assert out["status"] == bq.MOE_OK
    x_ref = O.rmsnorm_no_scale(h_bits)
    diff = np.abs(out["x"].astype(np.int32) - x_ref.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3, "rmsnorm differs by more than rounding"
    assert np.array_equal(out["ids"], O.select_top_k(out["logits"], k)), "ids differ from the top-k of the GPU's logits"
    rs, pes = layer.host_router_scales()
    assert_close(out["logits"], O.router_logits(out["x"], layer.host_router(), layer.host_logit_bias(), rs), "logits")
    sel = np.arange(h_bits.shape[0]) if rows is None else np.asarray(rows)
    ref = oracle_layer(layer, out["x"][sel], k, out["ids"][sel])
    assert_close(bf16_bits_to_f64(out["y"][sel]), ref["y"], f"y ({len(sel)} rows)")
    assert np.array_equal(out["h"], O.residual_add(h_bits, out["y"])), "residual stream is not bf16(h + y)"


@pytest.mark.parametrize("n_rows,zipf", [(300, True), (200, False), (1, False), (129, True)],
                         ids=["ragged300-zipf", "200-uniform", "one-row", "129-zipf"])
def test_prompt_matches_oracle(moe, layer0, layer0_zipf, n_rows, zipf):
    layer = layer0_zipf if zipf else layer0
    h0 = hidden(500 + n_rows, 0, n_rows, rms=False)
    out = run_prompt(moe, layer, h0)
    check_block(out, layer, h0, K)


def test_prompt_full_size(moe, layer0_zipf):
    """4096 rows (32 chunks of 128) with Zipf-skewed routing: the head experts
    get several hundred rows, i.e. several bounded units of up to 256 rows each."""
    n = bq.MOE_PROMPT_MAX_ROWS
    h0 = hidden(4242, 0, n, rms=False)
    out = run_prompt(moe, layer0_zipf, h0)
    counts = np.bincount(out["ids"].ravel(), minlength=E)
    assert counts.max() > 2 * 256, "the skew should give some expert more than two bounded units of 256 rows"
    rng = np.random.default_rng(11)
    rows = np.sort(np.concatenate([[0, 127, 128, n - 1], rng.choice(n, 28, replace=False)]))
    check_block(out, layer0_zipf, h0, K, rows=rows)
    # every row against the chunked residual calls (same function, 128 rows
    # per call), on the rows where both computed the same normalised input
    # and ids.  Each path is within the block's bar of the oracle, so their
    # difference is within twice the bar for the largest error; the mean
    # error of the difference stays within the bar itself.
    w = weights_of(layer0_zipf)
    h = to_dev_bf16(h0)
    y = torch.empty_like(h)
    xo = torch.empty_like(h)
    ids = torch.empty((n, K), dtype=torch.int32, device="cuda")
    ws = workspace(moe, w, 128)
    for c0 in range(0, n, 128):
        sl = slice(c0, c0 + 128)
        moe.layer_forward_residual(h[sl], 128, w, ws, y_out=y[sl], x_out=xo[sl], ids_out=ids[sl])
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK
    same = np.all(ids.cpu().numpy() == out["ids"], axis=1) & np.all(from_dev_bf16(xo) == out["x"], axis=1)
    assert same.mean() > 0.95, "the two paths disagree on the routing beyond near-ties and rmsnorm roundings"
    got, ref = bf16_bits_to_f64(out["y"][same]), bf16_bits_to_f64(from_dev_bf16(y))[same]
    max_rel_rms, mean_rel = errors(got, ref)
    assert max_rel_rms <= 2 * MAX_ABS_VS_RMS and mean_rel <= MEAN_REL, (
        f"prompt layer against the chunked layer calls: max|err|/rms = {max_rel_rms:.3e}, mean rel = {mean_rel:.3e}")


def test_prompt_repeated_calls_bit_identical(moe, layer0_zipf):
    """No atomics on the path: eight calls on the same input are identical."""
    h0 = hidden(77, 0, 300, rms=False)
    w = weights_of(layer0_zipf)
    ws = _prompt_ws(moe, w, 300)
    first = run_prompt(moe, layer0_zipf, h0, w=w, ws=ws)
    assert first["status"] == bq.MOE_OK
    for rep in range(7):
        out = run_prompt(moe, layer0_zipf, h0, w=w, ws=ws)
        for key in ("y", "h", "ids"):
            assert np.array_equal(out[key], first[key]), f"call {rep + 1}: {key} differs"


@pytest.mark.parametrize("hidden_dim,inter,n_experts,k,n_rows", [
    (128, 64, 8, 2, 33), (192, 128, 16, 8, 170), (256, 128, 4, 4, 5), (64, 64, 1, 1, 3), (320, 192, 32, 8, 260),
])
def test_prompt_small_shapes(moe, hidden_dim, inter, n_experts, k, n_rows):
    """Ragged weight tiles (inter or hidden not a multiple of 128), few experts,
    k = 1, every expert taking more than one chunk."""
    layer = DeviceLayer(13, hidden_dim, inter, n_experts, zipf=n_experts >= 8)
    h0 = hidden(13, n_rows, n_rows, hidden_dim, rms=False)
    out = run_prompt(moe, layer, h0, k)
    check_block(out, layer, h0, k)


def test_prompt_router_scales(moe):
    layer = DeviceLayer(0, H, I, E, zipf=True, router_scales=True)
    h0 = hidden(31, 0, 200, rms=False)
    out = run_prompt(moe, layer, h0)
    check_block(out, layer, h0, K)
    plain = O.select_top_k(O.router_logits(out["x"], layer.host_router(), layer.host_logit_bias()), K)
    assert not np.array_equal(plain, out["ids"]), "the router scales should change the routing"


def test_prompt_layer_tail(moe):
    """With the layer's tail the combine writes y and the tail updates the
    stream: the same bits as the oracle's layer_tail(h, y) (one bf16 step at
    flipped roundings, as for the other layer calls)."""
    from test_gpu_tail import check_tail
    layer = DeviceLayer(3, H, I, E, zipf=True, tail=True)
    h0 = hidden(41, 0, 150, rms=False)
    out = run_prompt(moe, layer, h0)
    assert out["status"] == bq.MOE_OK
    assert np.array_equal(out["ids"], O.select_top_k(out["logits"], K))
    ref = oracle_layer(layer, out["x"], K, out["ids"])
    assert_close(bf16_bits_to_f64(out["y"]), ref["y"], "y with a tail")
    g, lam = layer.host_layer_tail()
    check_tail(h0, out["y"], out["h"], g, lam)


def test_prompt_argument_errors(moe, layer0):
    w = weights_of(layer0)
    h = to_dev_bf16(hidden(0, 0, 4, rms=False))
    ws = _prompt_ws(moe, w, 4)
    for n in (0, bq.MOE_PROMPT_MAX_ROWS + 1):
        with pytest.raises(bq.MoeError) as ei:
            moe.layer_forward_prompt(h, n, w, ws)
        assert ei.value.status == bq.MOE_ERR_INVALID_ARG
    with pytest.raises(bq.MoeError) as ei:
        moe.layer_forward_prompt(h, 4, w, ws[:4096])
    assert ei.value.status == bq.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK
