"""CUDA path vs the float64 oracle, through the C ABI, on a GB300.

Decisions taken in floating point (the top-k) are checked on the GPU's own
fp32 logits: ids must equal the oracle's top-k of those logits bit for bit.
Values (logits, routing weights, outputs) are checked against the oracle at
the block's tolerance (numerics.py).  Outputs are compared with the oracle
run on the GPU's ids (teacher forcing), so a near-tie that flips the
selection cannot hide an arithmetic error or fake one."""
import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from gpu_layers import (E, H, I, K, HostExperts, hidden, oracle_layer, run_layer, to_dev_bf16, from_dev_bf16,
                        weights_of, workspace)
from numerics import assert_close, bf16_bits_to_f64
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


def _check_routing(out, layer, x_bits, k):
    ids, logits = out["ids"], out["logits"]
    assert np.array_equal(ids, O.select_top_k(logits, k)), "ids differ from the top-k of the GPU's own logits"
    rs, pes = layer.host_router_scales()
    ref_logits = O.router_logits(x_bits, layer.host_router(), layer.host_logit_bias(), rs)
    assert_close(logits, ref_logits, "logits")
    assert_close(out["weights"], O.routing_weights(logits.astype(np.float64), ids, pes), "routing weights")


@pytest.mark.parametrize("n_tokens,zipf", [(1, False), (13, False), (64, False), (100, True), (128, True)],
                         ids=["decode", "ragged13", "batch64-uniform", "ragged100-zipf", "prefill128-zipf"])
def test_layer_forward(moe, layer0, layer0_zipf, n_tokens, zipf):
    layer = layer0_zipf if zipf else layer0
    x = hidden(0, n_tokens, n_tokens)
    out = run_layer(moe, layer, x)
    assert out["status"] == bq.MOE_OK
    _check_routing(out, layer, x, K)
    ref = oracle_layer(layer, x, K, out["ids"])
    assert_close(bf16_bits_to_f64(out["y"]), ref["y"], f"y (T={n_tokens})")


def test_zipf_skews_routing(moe, layer0_zipf):
    out = run_layer(moe, layer0_zipf, hidden(0, 7, 128))
    counts = np.bincount(out["ids"].reshape(-1), minlength=E)
    assert counts.max() >= 30 and (counts == 0).sum() >= 1


def test_route_sort_bit_exact(moe, layer0):
    rng = np.random.default_rng(5)
    for n_tokens in (1, 7, 64, 128):
        ids_np = np.stack([rng.permutation(E)[:K] for _ in range(n_tokens)]).astype(np.int32)
        ids = torch.from_numpy(ids_np).cuda()
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        perm = torch.empty(n_tokens * K, dtype=torch.int32, device="cuda")
        pos = torch.empty(n_tokens * K, dtype=torch.int32, device="cuda")
        moe.route_sort(ids, n_tokens, weights_of(layer0).dims, counts, offsets, perm, pos)
        torch.cuda.synchronize()
        rc, ro, rp, rq = O.route_sort(ids_np, E)
        assert np.array_equal(counts.cpu().numpy(), rc)
        assert np.array_equal(offsets.cpu().numpy(), ro)
        assert np.array_equal(perm.cpu().numpy(), rp)
        assert np.array_equal(pos.cpu().numpy(), rq)
        assert moe.get_error() == bq.MOE_OK


def test_route_sort_drops_bad_ids(moe, layer0):
    ids_np = np.array([[3, 200, 5, -1, 3, 9, 127, 0]], dtype=np.int32).repeat(3, axis=0)
    ids = torch.from_numpy(ids_np).cuda()
    n = ids_np.size
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    pos = torch.empty(n, dtype=torch.int32, device="cuda")
    moe.route_sort(ids, 3, weights_of(layer0).dims, counts, offsets, perm, pos)
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_ERR_BAD_EXPERT_ID
    # reference: out-of-range ids as one extra expert sorted last
    flat = ids_np.reshape(-1).astype(np.int64)
    mapped = np.where((flat < 0) | (flat >= E), E, flat).reshape(ids_np.shape)
    rc, ro, rp, rq = O.route_sort(mapped, E + 1)
    kept = int(ro[E])
    assert np.array_equal(counts.cpu().numpy(), rc[:E])
    assert np.array_equal(offsets.cpu().numpy(), ro[:E + 1])
    assert np.array_equal(perm.cpu().numpy()[:kept], rp[:kept])
    want_pos = np.where(mapped.reshape(-1) == E, -1, rq)
    assert np.array_equal(pos.cpu().numpy(), want_pos)


@pytest.mark.parametrize("include_shared", [True, False])
@pytest.mark.parametrize("n_tokens", [1, 5, 40])
def test_expert_ffn_forced_routing(moe, layer0, n_tokens, include_shared):
    rng = np.random.default_rng(n_tokens)
    ids_np = np.stack([rng.permutation(E)[:K] for _ in range(n_tokens)]).astype(np.int32)
    if n_tokens > 1:
        ids_np[1, 3] = ids_np[1, 0]            # a token that picks one expert twice
    w_np = rng.uniform(0.0, 1.0, size=(n_tokens, K)).astype(np.float32)
    x_bits = hidden(3, n_tokens, n_tokens)
    w = weights_of(layer0)
    x = to_dev_bf16(x_bits)
    y = torch.empty_like(x)
    ws = workspace(moe, w, n_tokens)
    moe.expert_ffn(x, n_tokens, torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda(), w, y, ws,
                   include_shared=include_shared)
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK
    ref = O.expert_mix(x_bits, ids_np, w_np.astype(np.float64), HostExperts(layer0),
                       layer0.host_shared() if include_shared else None)
    assert_close(bf16_bits_to_f64(from_dev_bf16(y)), ref, "expert_ffn y")


def test_expert_ffn_skips_bad_ids(moe, layer0):
    n_tokens = 4
    rng = np.random.default_rng(11)
    ids_np = np.stack([rng.permutation(E)[:K] for _ in range(n_tokens)]).astype(np.int32)
    ids_np[0, 2] = 128
    ids_np[2, 7] = -3
    w_np = rng.uniform(0.1, 1.0, size=(n_tokens, K)).astype(np.float32)
    x_bits = hidden(4, 0, n_tokens)
    w = weights_of(layer0)
    x = to_dev_bf16(x_bits)
    y = torch.empty_like(x)
    ws = workspace(moe, w, n_tokens)
    moe.expert_ffn(x, n_tokens, torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda(), w, y, ws)
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_ERR_BAD_EXPERT_ID
    bad = (ids_np < 0) | (ids_np >= E)
    ref = O.expert_mix(x_bits, np.where(bad, 0, ids_np), np.where(bad, 0.0, w_np.astype(np.float64)),
                       HostExperts(layer0), layer0.host_shared())
    assert_close(bf16_bits_to_f64(from_dev_bf16(y)), ref, "y with dropped pairs")


def test_router_topk_entry(moe, layer0_zipf):
    n_tokens = 33
    x_bits = hidden(5, 0, n_tokens)
    w = weights_of(layer0_zipf)
    ids = torch.empty((n_tokens, K), dtype=torch.int32, device="cuda")
    wts = torch.empty((n_tokens, K), dtype=torch.float32, device="cuda")
    logits = torch.empty((n_tokens, E), dtype=torch.float32, device="cuda")
    moe.router_topk(to_dev_bf16(x_bits), n_tokens, w, ids, wts, workspace(moe, w, n_tokens), logits=logits)
    torch.cuda.synchronize()
    out = {"ids": ids.cpu().numpy(), "logits": logits.cpu().numpy(), "weights": wts.cpu().numpy()}
    _check_routing(out, layer0_zipf, x_bits, K)


def test_residual_stack_teacher_forced(moe):
    layers = [DeviceLayer(s, H, I, E) for s in (0, 1, 2)]
    for n_tokens in (1, 8):
        h_bits = hidden(1000, 0, n_tokens, rms=False)
        h = to_dev_bf16(h_bits)
        ws = workspace(moe, weights_of(layers[0]), n_tokens)
        for layer in layers:
            w = weights_of(layer)
            h_in = from_dev_bf16(h)
            y = torch.empty_like(h)
            xo = torch.empty_like(h)
            ids = torch.empty((n_tokens, K), dtype=torch.int32, device="cuda")
            logits = torch.empty((n_tokens, E), dtype=torch.float32, device="cuda")
            moe.layer_forward_residual(h, n_tokens, w, ws, y_out=y, x_out=xo, ids_out=ids, logits_out=logits)
            torch.cuda.synchronize()
            assert moe.get_error() == bq.MOE_OK
            x_gpu = from_dev_bf16(xo)
            x_ref = O.rmsnorm_no_scale(h_in)
            diff = np.abs(x_gpu.astype(np.int32) - x_ref.astype(np.int32))
            assert diff.max() <= 1 and (diff > 0).mean() < 1e-3, "rmsnorm differs by more than rounding"
            ids_np = ids.cpu().numpy()
            assert np.array_equal(ids_np, O.select_top_k(logits.cpu().numpy(), K))
            ref = oracle_layer(layer, x_gpu, K, ids_np)
            y_gpu = from_dev_bf16(y)
            assert_close(bf16_bits_to_f64(y_gpu), ref["y"], "stack layer y")
            assert np.array_equal(from_dev_bf16(h), O.residual_add(h_in, y_gpu))


@pytest.mark.parametrize("n_tokens", [1, 128])
def test_deterministic(moe, layer0_zipf, n_tokens):
    x = hidden(9, 0, n_tokens)
    a = run_layer(moe, layer0_zipf, x)
    b = run_layer(moe, layer0_zipf, x)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["ids"], b["ids"])
    assert np.array_equal(a["logits"].view(np.uint32), b["logits"].view(np.uint32))


@pytest.mark.parametrize("n_tokens", [37, 100])
def test_repeated_calls_bit_identical(moe, layer0, n_tokens):
    """Sixteen residual calls of the multi-token kernel on the same input all
    bit-identical (fixed-order reductions): a ring or buffer race in the
    kernel (a consumer group reading a slot before its copy landed, a buffer
    released while still read) shows up here as a call that differs."""
    w = weights_of(layer0)
    x_bits = hidden(2024, 0, n_tokens, rms=False)
    ws = workspace(moe, w, n_tokens)
    first = None
    for rep in range(16):
        h = to_dev_bf16(x_bits)
        y = torch.empty_like(h)
        ids = torch.empty((n_tokens, K), dtype=torch.int32, device="cuda")
        moe.layer_forward_residual(h, n_tokens, w, ws, y_out=y, ids_out=ids)
        torch.cuda.synchronize()
        assert moe.get_error() == bq.MOE_OK
        out = (from_dev_bf16(y), from_dev_bf16(h), ids.cpu().numpy())
        if first is None:
            first = out
            continue
        for got, want, what in zip(out, first, ("y", "residual stream", "ids")):
            assert np.array_equal(got, want), f"call {rep}: {what} differs from the first call"


@pytest.mark.parametrize("hidden_dim,inter,n_experts,k,n_tokens", [
    (128, 64, 8, 2, 1), (128, 64, 8, 2, 33), (256, 128, 4, 4, 5), (192, 128, 16, 8, 17), (64, 64, 1, 1, 3),
])
def test_small_shapes(moe, hidden_dim, inter, n_experts, k, n_tokens):
    layer = DeviceLayer(7, hidden_dim, inter, n_experts, zipf=n_experts >= 8)
    x = hidden(7, n_tokens, n_tokens, hidden_dim)
    out = run_layer(moe, layer, x, k)
    assert out["status"] == bq.MOE_OK
    _check_routing(out, layer, x, k)
    ref = oracle_layer(layer, x, k, out["ids"])
    assert_close(bf16_bits_to_f64(out["y"]), ref["y"], "small-shape y")


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("n_tokens", [1, 2, 4, 37, 128])
def test_fused_and_chained_paths_agree(layer0, layer0_zipf, residual, n_tokens):
    """Layer calls run a fused one-launch kernel by default (the single-token
    kernel for T == 1, the prefill kernel for 2 <= T <= 128); a handle created
    with MOE_DECODE_FUSED=0 / MOE_PREFILL_FUSED=0 runs the router, gate/up and
    down launches instead.  Both must match the oracle; ids must be identical."""
    import os
    var = "MOE_DECODE_FUSED" if n_tokens == 1 else "MOE_PREFILL_FUSED"
    layer = layer0_zipf if n_tokens == 128 else layer0
    outs = {}
    for fused in ("1", "0"):
        old = os.environ.get(var)
        os.environ[var] = fused
        try:
            m = bq.Moe()
        finally:
            if old is None:
                del os.environ[var]
            else:
                os.environ[var] = old
        w = weights_of(layer)
        x_bits = hidden(2024, 0, n_tokens, rms=not residual)
        h = to_dev_bf16(x_bits)
        y = torch.empty_like(h)
        xo = torch.empty_like(h)
        ids = torch.empty((n_tokens, K), dtype=torch.int32, device="cuda")
        logits = torch.empty((n_tokens, E), dtype=torch.float32, device="cuda")
        ws = workspace(m, w, n_tokens)
        trace = torch.zeros(4 * 4, dtype=torch.int64, device="cuda")
        m.set_trace(trace, 4)
        if residual:
            m.layer_forward_residual(h, n_tokens, w, ws, y_out=y, x_out=xo, ids_out=ids, logits_out=logits)
        else:
            m.layer_forward(h, n_tokens, w, y, ws, ids_out=ids, logits_out=logits)
        torch.cuda.synchronize()
        m.set_trace(None, 0)
        assert m.get_error() == bq.MOE_OK
        # which path ran: the fused kernel traces one launch, the chain one per launch
        launches = int((trace.view(4, 4) != 0).any(dim=1).sum())
        assert launches == (1 if fused == "1" else (3 if n_tokens == 1 else 4)), f"fused={fused}: {launches} launches"
        x_used = from_dev_bf16(xo) if residual else x_bits
        out = {"ids": ids.cpu().numpy(), "logits": logits.cpu().numpy(), "y": from_dev_bf16(y), "x": x_used,
               "h": from_dev_bf16(h)}
        assert np.array_equal(out["ids"], O.select_top_k(out["logits"], K))
        ref = oracle_layer(layer, x_used, K, out["ids"])
        assert_close(bf16_bits_to_f64(out["y"]), ref["y"], f"y fused={fused}")
        if residual:
            assert np.array_equal(out["h"], O.residual_add(x_bits, out["y"]))
            xr = bf16_bits_to_f64(O.rmsnorm_no_scale(x_bits))
            # fp32 on the device against fp64: at most one bf16 rounding step apart
            assert np.all(np.abs(bf16_bits_to_f64(out["x"]) - xr) <= 2.0 ** -7 * np.abs(xr))
        outs[fused] = out
        m.close()
    assert np.array_equal(outs["1"]["ids"], outs["0"]["ids"])


@pytest.fixture(scope="module")
def layer0_scaled():
    return DeviceLayer(0, H, I, E, zipf=True, router_scales=True)


@pytest.mark.parametrize("fused", ["1", "0"])
@pytest.mark.parametrize("n_tokens", [1, 37, 128])
def test_router_scales(layer0_scaled, n_tokens, fused):
    """The learned router scale (x * router_scale / sqrt(H) into the router) and
    the per-expert scales (softmax weight times the selected expert's scale),
    on the fused kernels and on the chained launches."""
    import os
    var = "MOE_DECODE_FUSED" if n_tokens == 1 else "MOE_PREFILL_FUSED"
    old = os.environ.get(var)
    os.environ[var] = fused
    try:
        m = bq.Moe()
    finally:
        if old is None:
            del os.environ[var]
        else:
            os.environ[var] = old
    try:
        x = hidden(31, n_tokens, n_tokens)
        out = run_layer(m, layer0_scaled, x)
        assert out["status"] == bq.MOE_OK
        _check_routing(out, layer0_scaled, x, K)
        # the scales change the routing: compare with the same layer unscaled
        plain = O.select_top_k(O.router_logits(x, layer0_scaled.host_router(), layer0_scaled.host_logit_bias()), K)
        assert not np.array_equal(plain, out["ids"])
        ref = oracle_layer(layer0_scaled, x, K, out["ids"])
        assert_close(bf16_bits_to_f64(out["y"]), ref["y"], f"y with router scales (T={n_tokens}, fused={fused})")
    finally:
        m.close()


@pytest.mark.parametrize("hidden_dim,inter,n_experts,k,n_tokens", [(128, 64, 8, 2, 1), (192, 128, 16, 8, 17)])
def test_router_scales_small_shapes(moe, hidden_dim, inter, n_experts, k, n_tokens):
    layer = DeviceLayer(9, hidden_dim, inter, n_experts, router_scales=True)
    x = hidden(9, n_tokens, n_tokens, hidden_dim)
    out = run_layer(moe, layer, x, k)
    assert out["status"] == bq.MOE_OK
    _check_routing(out, layer, x, k)
    ref = oracle_layer(layer, x, k, out["ids"])
    assert_close(bf16_bits_to_f64(out["y"]), ref["y"], "small-shape y with router scales")


def test_argument_errors(moe, layer0):
    w = weights_of(layer0)
    x = to_dev_bf16(hidden(0, 0, 2))
    y = torch.empty_like(x)
    ws = workspace(moe, w, 2)
    for n in (0, 129):
        with pytest.raises(bq.MoeError) as ei:
            moe.layer_forward(x, n, w, y, ws)
        assert ei.value.status == bq.MOE_ERR_INVALID_ARG
    with pytest.raises(bq.MoeError) as ei:
        moe.layer_forward(x, 2, w, y, ws[:1024])
    assert ei.value.status == bq.MOE_ERR_WORKSPACE
    with pytest.raises(bq.MoeError) as ei:
        moe.layer_forward(x.view(-1)[1:], 1, w, y, ws)
    assert ei.value.status == bq.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert moe.get_error() == bq.MOE_OK


def test_bounded_wait_reports_timeout(moe):
    moe.selftest_wait_timeout(5_000_000)
    assert moe.get_error() == bq.MOE_ERR_TIMEOUT
    assert moe.get_error() == bq.MOE_OK     # cleared by the read


@pytest.mark.parametrize("n_tokens,zipf", [(100, False), (100, True), (128, False), (128, True)],
                         ids=["T100-uniform", "ragged100-zipf", "prefill128-uniform", "prefill128-zipf"])
def test_prefill_dense_slots(layer0, layer0_zipf, n_tokens, zipf):
    """Slots with at least 96 rows in the chunk (the shared expert; the heaviest
    experts of a Zipf-skewed chunk) run on the tcgen05 path: weight tiles
    dequantised once to fp16 in shared memory, tcgen05.mma into tensor memory.
    Both paths must meet the oracle; their outputs differ in some bits (the
    tcgen05 path rounds each weight to fp16), which shows the path ran.  The
    routing is computed before the experts, so the ids are identical."""
    import os
    layer = layer0_zipf if zipf else layer0
    x = hidden(77, n_tokens, n_tokens)
    outs = {}
    for dense in ("1", "0"):
        old = os.environ.get("MOE_PREFILL_DENSE")
        os.environ["MOE_PREFILL_DENSE"] = dense
        try:
            m = bq.Moe()
        finally:
            if old is None:
                del os.environ["MOE_PREFILL_DENSE"]
            else:
                os.environ["MOE_PREFILL_DENSE"] = old
        try:
            out = run_layer(m, layer, x)
        finally:
            m.close()
        assert out["status"] == bq.MOE_OK
        _check_routing(out, layer, x, K)
        ref = oracle_layer(layer, x, K, out["ids"])
        assert_close(bf16_bits_to_f64(out["y"]), ref["y"], f"y (T={n_tokens}, dense={dense})")
        outs[dense] = out
    assert np.array_equal(outs["1"]["ids"], outs["0"]["ids"])
    assert not np.array_equal(outs["1"]["y"], outs["0"]["y"]), "the tcgen05 path did not run"
