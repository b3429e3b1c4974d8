"""Edge cases of the routing and of the device-side failure paths, on a
GB300 through the C ABI.

Exact logit ties.  The selection rule (page "TurboFieldfare - System
design", section "Decode": eight experts per token; ties go to the lower
expert id) only matters when two logits are equal to the last bit, which
random weights never produce.  Here the router rows come in triplets of
identical rows (experts j, j + 42 and j + 84 share one row), so every token
has exact ties between their logits: the top-8 then usually holds two whole
triplets and two members of a third, and which two is decided by the tie
rule alone.  Each kernel that selects experts (the single-token kernel, the
multi-token kernel at two chunk sizes, the stand-alone router of the
chained launches) must return exactly the oracle's top-k of its own fp32
logits, and the test checks that boundary ties really occurred.

Failure detection without a GPU fault.  A test hook makes one block of the
next single-token launch withhold its grid-barrier arrival with a 5 ms wait
limit: every block gives up, MOE_ERR_TIMEOUT is reported, and the call after
it must be correct again (the timeout left the barrier counter short of a
whole grid; moe_get_error restores it).  An input large enough to push the
expert activations out of fp16 range must be reported as MOE_ERR_NONFINITE,
and the next call must be clean."""
import os

import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import E, H, I, K, HostExperts, from_dev_bf16, hidden, oracle_layer, run_layer, to_dev_bf16, \
    weights_of, workspace
from numerics import assert_close, bf16_bits_to_f64
from oracle import moe_oracle as O
from synth import gen
from synth.device import DeviceLayer

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TRIPLE = 42  # experts j, j + 42, j + 84 (j < 42) share one router row; 126 and 127 keep their own


def tie_groups(n_experts: int = E):
    return [[j, j + TRIPLE, j + 2 * TRIPLE] for j in range(TRIPLE) if j + 2 * TRIPLE < n_experts]


def make_tied(layer: DeviceLayer) -> DeviceLayer:
    """Rewrites the layer's router so that every tie group shares the row of
    its last member (codes, scales and biases), on the device and in the host
    copy the oracle reads."""
    r = layer.host_router()
    q, s, b = r["q"].copy(), r["s"].copy(), r["b"].copy()
    for grp in tie_groups(layer.n_experts):
        src = grp[-1]
        for e in grp[:-1]:
            q[e], s[e], b[e] = q[src], s[src], b[src]
    layer._h2d(layer.router_off + layer.rl["q"], q)
    layer._h2d(layer.router_off + layer.rl["s"], s)
    layer._h2d(layer.router_off + layer.rl["b"], b)
    torch.cuda.synchronize()
    tied = {"q": q, "s": s, "b": b}
    layer.host_router = lambda: tied
    return layer


@pytest.fixture(scope="module")
def tied_layer():
    return make_tied(DeviceLayer(3, H, I, E))


@pytest.fixture(scope="module")
def moe():
    bq.build_library()
    m = bq.Moe()
    yield m
    m.close()


def _handle(var, value):
    old = os.environ.get(var)
    os.environ[var] = value
    try:
        return bq.Moe()
    finally:
        if old is None:
            del os.environ[var]
        else:
            os.environ[var] = old


def boundary_ties(logits: np.ndarray, ids: np.ndarray) -> int:
    """Tokens whose k-th selected logit equals the logit of an expert left out."""
    n = 0
    for t in range(logits.shape[0]):
        last = logits[t, ids[t, -1]]
        left_out = np.setdiff1d(np.arange(logits.shape[1]), ids[t])
        n += int(np.any(logits[t, left_out] == last))
    return n


def check_tied_routing(out, layer, x_bits, what):
    ids, logits = out["ids"], out["logits"]
    # triplet members' logits are bit-identical on the GPU
    for grp in tie_groups():
        col = logits[:, grp]
        assert np.array_equal(col.view(np.uint32), np.repeat(col[:, :1], 3, axis=1).view(np.uint32)), \
            f"{what}: experts {grp} have identical router rows but different logits"
    assert np.array_equal(ids, O.select_top_k(logits, K)), f"{what}: ids differ from the oracle's top-k"
    # where the boundary is a tie, the selected member is the lowest id among the tied experts left
    for t in range(ids.shape[0]):
        last = logits[t, ids[t, -1]]
        tied = np.flatnonzero(logits[t] == last)
        chosen = [e for e in ids[t] if logits[t, e] == last]
        assert sorted(chosen) == sorted(tied[:len(chosen)].tolist()), f"{what}: token {t} tie not to lower ids"
    ref_logits = O.router_logits(x_bits, layer.host_router(), layer.host_logit_bias())
    assert_close(logits, ref_logits, f"{what}: logits")
    assert_close(out["weights"], O.routing_weights(logits.astype(np.float64), ids), f"{what}: routing weights")
    return boundary_ties(logits, ids)


def test_ties_single_token_fused(moe, tied_layer):
    n_ties = 0
    for seed in range(6):
        x = hidden(400 + seed, 0, 1)
        out = run_layer(moe, tied_layer, x)
        assert out["status"] == bq.MOE_OK
        n_ties += check_tied_routing(out, tied_layer, x, f"decode seed {seed}")
        if seed == 0:
            ref = oracle_layer(tied_layer, x, K, out["ids"])
            assert_close(bf16_bits_to_f64(out["y"]), ref["y"], "decode y with tied router")
    assert n_ties >= 3, f"only {n_ties} of 6 tokens had a tie at the top-k boundary"


@pytest.mark.parametrize("n_tokens", [37, 128])
def test_ties_multi_token_fused(moe, tied_layer, n_tokens):
    x = hidden(500, n_tokens, n_tokens)
    out = run_layer(moe, tied_layer, x)
    assert out["status"] == bq.MOE_OK
    n_ties = check_tied_routing(out, tied_layer, x, f"T={n_tokens}")
    assert n_ties >= n_tokens // 2, f"only {n_ties} of {n_tokens} tokens had a boundary tie"
    ref = oracle_layer(tied_layer, x, K, out["ids"])
    assert_close(bf16_bits_to_f64(out["y"]), ref["y"], f"y with tied router (T={n_tokens})")


@pytest.mark.parametrize("n_tokens", [1, 37])
def test_ties_chained_launches(tied_layer, n_tokens):
    var = "MOE_DECODE_FUSED" if n_tokens == 1 else "MOE_PREFILL_FUSED"
    m = _handle(var, "0")
    try:
        n_ties = 0
        for seed in range(4 if n_tokens == 1 else 1):
            x = hidden(600 + seed, n_tokens, n_tokens)
            out = run_layer(m, tied_layer, x)
            assert out["status"] == bq.MOE_OK
            n_ties += check_tied_routing(out, tied_layer, x, f"chained T={n_tokens} seed {seed}")
        assert n_ties >= 1
        ref = oracle_layer(tied_layer, x, K, out["ids"])
        assert_close(bf16_bits_to_f64(out["y"]), ref["y"], f"chained y with tied router (T={n_tokens})")
    finally:
        m.close()


def test_ties_router_entry(moe, tied_layer):
    n_tokens = 33
    x_bits = hidden(700, 0, n_tokens)
    w = weights_of(tied_layer)
    ids = torch.empty((n_tokens, K), dtype=torch.int32, device="cuda")
    wts = torch.empty((n_tokens, K), dtype=torch.float32, device="cuda")
    logits = torch.empty((n_tokens, E), dtype=torch.float32, device="cuda")
    moe.router_topk(to_dev_bf16(x_bits), n_tokens, w, ids, wts, workspace(moe, w, n_tokens), logits=logits)
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK
    out = {"ids": ids.cpu().numpy(), "logits": logits.cpu().numpy(), "weights": wts.cpu().numpy()}
    assert check_tied_routing(out, tied_layer, x_bits, "router entry") >= 1


@pytest.fixture(scope="module")
def plain_layer():
    return DeviceLayer(4, H, I, E)


def _check_layer(moe, layer, x_bits, what):
    out = run_layer(moe, layer, x_bits)
    assert out["status"] == bq.MOE_OK, f"{what}: status {out['status']}"
    assert np.array_equal(out["ids"], O.select_top_k(out["logits"], K)), f"{what}: ids"
    ref = oracle_layer(layer, x_bits, K, out["ids"])
    assert_close(bf16_bits_to_f64(out["y"]), ref["y"], f"{what}: y")
    # the logits themselves, not only the selection (stale mailboxes would pass the ids check)
    assert_close(out["logits"], O.router_logits(x_bits, layer.host_router()), f"{what}: logits")


def test_withheld_arrival_times_out_then_recovers(plain_layer):
    m = bq.Moe()
    try:
        w = weights_of(plain_layer)
        ws = workspace(m, w, 1)
        _check_layer(m, plain_layer, hidden(800, 0, 1), "before")
        for block in (0, 97):
            x = to_dev_bf16(hidden(801 + block, 0, 1))
            y = torch.empty_like(x)
            m.selftest_skip_arrival(block, 5_000_000)
            m.layer_forward(x, 1, w, y, ws)
            assert m.get_error() == bq.MOE_ERR_TIMEOUT
            assert m.get_error() == bq.MOE_OK  # cleared by the read
            # the next calls are correct again (two, so two epochs pass)
            _check_layer(m, plain_layer, hidden(900 + block, 0, 1), f"after withheld arrival of block {block}, 1")
            _check_layer(m, plain_layer, hidden(950 + block, 0, 1), f"after withheld arrival of block {block}, 2")
    finally:
        m.close()


def test_skip_arrival_hook_rejects_bad_arguments(moe):
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    for block, limit in ((-1, 1000), (n_sm, 1000), (0, 0), (0, 3_000_000_000)):
        with pytest.raises(bq.MoeError) as ei:
            moe.selftest_skip_arrival(block, limit)
        assert ei.value.status == bq.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("n_tokens", [1, 16])
def test_activations_out_of_fp16_range_are_flagged(moe, plain_layer, n_tokens):
    """x scaled to rms 1000 (still finite in fp16) gives gate and up values near
    500 and h = gelu(g) * u far beyond fp16's 65504: recorded as non-finite."""
    big = gen.to_bf16_bits(bf16_bits_to_f64(hidden(1100, 0, n_tokens)) * 1000.0)
    out = run_layer(moe, plain_layer, big)
    assert out["status"] == bq.MOE_ERR_NONFINITE
    assert moe.get_error() == bq.MOE_OK
    _check_layer(moe, plain_layer, hidden(1101, 0, n_tokens), f"after a non-finite call (T={n_tokens})")
