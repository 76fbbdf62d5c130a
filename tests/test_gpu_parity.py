"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Routing (ids, slot, row_of, src_token, counts, offsets) must match bit-exactly;
floats must satisfy max|gpu - ref| <= tol * max|ref| per tensor with tol 2e-2
for bf16 layers and 1e-4 for fp32 layers.  Sizes here let the oracle finish in
seconds while spanning several tiles per expert and a ragged tail.
"""
import numpy as np
import pytest
import torch

import routing_permute_grouped_router_gb300 as pkg
from _util import TOL, assert_close, assert_routing_equal, check_no_device_error
from oracle import moe_oracle as O
from routing_permute_grouped_router_gb300 import layer
from routing_permute_grouped_router_gb300 import workload as W

pytestmark = pytest.mark.gpu

LS = W.LayerShape
SMALL = {
    "switch_tiny_f32": W.WORKLOADS["switch_tiny_f32"],
    "top2_e8_small": LS("top2_e8_small", 1000, 256, 512, 8, 2, 1.25, W.BF16),
    "zipf_e64_small": LS("zipf_e64_small", 2000, 256, 256, 64, 2, 1.0, W.BF16, zipf_s=1.1),
    "dropless_e32_small": LS("dropless_e32_small", 1500, 512, 256, 32, 4, 0.0, W.BF16, zipf_s=1.3),
    "train_e16_small": LS("train_e16_small", 700, 256, 512, 16, 2, 1.25, W.BF16, micro_batches=4, backward=True),
    "train_f32_small": LS("train_f32_small", 333, 64, 96, 5, 2, 1.0, W.F32, micro_batches=2, backward=True),
    # d = 4096 (any d >= 2048) selects the long-K dgrad h shape (three 64 KB stages, one a|b buffer a warp)
    "wide_d4096": LS("wide_d4096", 400, 4096, 256, 4, 2, 1.25, W.BF16),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    from routing_permute_grouped_router_gb300 import build

    build.build()
    pkg.lib()
    torch.cuda.set_device(0)
    pkg.moe_get_device_error(clear=True)


def _cap(s):
    return O.capacity(s.T, s.k, s.E, s.capacity_factor, s.capacity)


def _oracle_fwd(wl, m=0):
    s = wl.shape
    return O.forward(wl.x[m].f64(), wl.W_r, wl.bias, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), s.k, _cap(s))


def _check_forward(L, ref, s, x_exact=True):
    tol = TOL[s.dtype]
    assert_routing_equal(L.saved, ref, s.T)
    rows = int(ref["offsets"][-1])
    assert_close("gates", L.saved["gates"], ref["gates"], 1e-5)
    assert_close("probs", L.saved["probs"], ref["probs"], 1e-5)
    if x_exact:
        np.testing.assert_array_equal(L.saved["x_perm"][:rows].float().cpu().numpy(), ref["x_perm"])
    assert_close("h", L.saved["h"][:rows], ref["h"], tol)
    assert_close("y_perm", L.saved["y_perm"][:rows], ref["Y_perm"], tol)
    assert_close("y", L.y[: s.T], ref["y"], tol)


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_forward(name):
    s = SMALL[name]
    wl = W.make(s, with_dy=False, micro_batches=1)
    L = layer.from_workload(wl)
    L.forward(wl.x[0].torch("cuda"))
    torch.cuda.synchronize()
    check_no_device_error()
    _check_forward(L, _oracle_fwd(wl), s)


@pytest.mark.parametrize("name", ["train_e16_small", "train_f32_small", "top2_e8_small", "zipf_e64_small",
                                  "dropless_e32_small", "wide_d4096"])
def test_layer_backward_with_accumulation(name):
    """The dropless layer runs the long-K wgrad shape and the d = 4096 layer (d >= 2048) the
    long-K dgrad h shape; the others the short-K shapes."""
    s = SMALL[name]
    nmb = max(s.micro_batches, 2)
    wl = W.make(s, micro_batches=nmb, with_dy=True)
    L = layer.from_workload(wl)
    tol = TOL[s.dtype]
    ref = O.train_step([x.f64() for x in wl.x], [dy.f64() for dy in wl.dy], wl.W_r, wl.bias, wl.W1.f64(),
                       wl.W3.f64(), wl.W2.f64(), s.k, _cap(s))
    for m in range(nmb):
        x = wl.x[m].torch("cuda")
        L.forward(x)
        L.backward(x, wl.dy[m].torch("cuda"), accumulate=m > 0)
        torch.cuda.synchronize()
        check_no_device_error()
        st, gr = ref["micro_batches"][m]
        assert_routing_equal(L.saved, st, s.T)
        assert_close(f"y[{m}]", L.y[: s.T], st["y"], tol)
        assert_close(f"dx[{m}]", L.dx[: s.T], gr["dx"], tol)
    for n in ("dW_r", "dW1", "dW3", "dW2"):
        assert_close(n, L.grads[n], ref["grads"][n], tol)


def test_backward_stage_outputs():
    """Intermediate tensors of the backward against the oracle (one micro-batch)."""
    s = SMALL["train_e16_small"]
    wl = W.make(s, micro_batches=1, with_dy=True)
    cfg = pkg.config_of(s)
    L = layer.from_workload(wl)
    x = wl.x[0].torch("cuda")
    L.forward(x)
    st = _oracle_fwd(wl)
    gr = O.backward(wl.dy[0].f64(), wl.x[0].f64(), wl.W_r, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), st)
    sv = L.saved
    R = L.max_rows
    rows = int(st["offsets"][-1])
    dev = dict(device="cuda")
    dy_perm = torch.empty(R, s.d_model, dtype=torch.bfloat16, **dev)
    dg = torch.empty(s.T, s.k, dtype=torch.float32, **dev)
    dl = torch.empty(s.T, s.E, dtype=torch.float32, **dev)
    pkg.moe_combine_bwd(cfg, wl.dy[0].torch("cuda"), sv["y_perm"], sv["ids"], sv["row_of"], sv["gates"],
                        sv["probs"], sv["counts"], sv["offsets"], dy_perm, dg, dl)
    da = torch.empty(R, s.d_ff, dtype=torch.bfloat16, **dev)
    db = torch.empty_like(da)
    dx_perm = torch.empty(R, s.d_model, dtype=torch.bfloat16, **dev)
    g = pkg.allocate_grads(cfg)
    pkg.moe_grouped_ffn_bwd(cfg, sv["x_perm"], sv["a"], sv["b"], sv["h"], dy_perm, sv["counts"], sv["offsets"],
                            L.weights["W1"], L.weights["W3"], L.weights["W2"], da, db, dx_perm, g["dW1"], g["dW3"],
                            g["dW2"], 0)
    dx = torch.empty(s.T, s.d_model, dtype=torch.bfloat16, **dev)
    pkg.moe_unpermute_dx_router_bwd(cfg, x, dx_perm, sv["row_of"], dl, L.weights["W_r"], dx, g["dW_r"], 0, L.ws)
    torch.cuda.synchronize()
    check_no_device_error()
    tol = 2e-2
    assert_close("a", sv["a"][:rows], st["a"], tol)
    assert_close("b", sv["b"][:rows], st["b"], tol)
    assert_close("dy_perm", dy_perm[:rows], gr["dY_perm"], tol)
    assert_close("dg", dg, gr["dg"], tol)
    assert_close("dl", dl, gr["dl"], tol)
    assert_close("da", da[:rows], gr["da"], tol)
    assert_close("db", db[:rows], gr["db"], tol)
    assert_close("dx_perm", dx_perm[:rows], gr["dX_perm"], tol)
    for n in ("dW1", "dW3", "dW2", "dW_r"):
        assert_close(n, g[n], gr[n], tol)
    assert_close("dx", dx, gr["dx"], tol)
    # pad rows of the per-expert buffers are zero
    counts = st["counts"]
    offs = st["offsets"]
    for e in range(s.E):
        pad = slice(int(offs[e] + counts[e]), int(offs[e + 1]))
        for t in (sv["x_perm"], sv["h"], sv["y_perm"], dy_perm, da, db, dx_perm):
            assert not t[pad].float().abs().sum().item()


# ------------------------------ edge cases -------------------------------- #
def _edge(shape, seed=3):
    wl = W.make(shape, seed=seed, micro_batches=1, with_dy=True)
    L = layer.from_workload(wl)
    x = wl.x[0].torch("cuda")
    L.forward(x)
    L.backward(x, wl.dy[0].torch("cuda"), accumulate=False)
    torch.cuda.synchronize()
    check_no_device_error()
    st = _oracle_fwd(wl)
    gr = O.backward(wl.dy[0].f64(), wl.x[0].f64(), wl.W_r, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), st)
    return wl, L, st, gr


@pytest.mark.parametrize("shape", [
    LS("cap0", 200, 256, 256, 4, 2, 1.0, W.BF16, capacity=0, backward=True),
    LS("cap1", 200, 256, 256, 4, 2, 1.0, W.BF16, capacity=1, backward=True),
    LS("e1k1", 130, 256, 256, 1, 1, 0.0, W.BF16, backward=True),
    LS("k_eq_E", 150, 256, 256, 4, 4, 0.0, W.BF16, backward=True),
    LS("one_token", 1, 256, 256, 8, 2, 1.25, W.BF16, backward=True),
    LS("ragged_T", 65, 256, 512, 3, 2, 2.0, W.BF16, backward=True),
    LS("e128_k8", 300, 256, 256, 128, 8, 1.0, W.BF16, backward=True),
    LS("f32_k1_cap", 97, 32, 48, 3, 1, 0.7, W.F32, backward=True),
])
def test_edge_cases(shape):
    wl, L, st, gr = _edge(shape)
    tol = TOL[shape.dtype]
    assert_routing_equal(L.saved, st, shape.T)
    assert_close("y", L.y[: shape.T], st["y"], tol)
    assert_close("dx", L.dx[: shape.T], gr["dx"], tol)
    for n in ("dW_r", "dW1", "dW3", "dW2"):
        assert_close(n, L.grads[n], gr[n], tol)
    if shape.capacity == 0:
        assert not L.y[: shape.T].float().abs().sum().item()
        assert (L.saved["slot"].cpu() == -1).all()
    if shape.E == 1:
        assert (L.saved["gates"].cpu() == 1.0).all()


@pytest.mark.parametrize("cf", [1.25, 0.0])
def test_zero_tokens(cf):
    """T = 0: no work, zero gradients when overwriting, untouched when accumulating."""
    s = LS("empty", 0, 256, 256, 4, 2, cf, W.BF16, backward=True)
    wl = W.make(s.replace(T=8), micro_batches=1, with_dy=True)
    L = layer.from_workload(wl, T=0)
    x = torch.zeros(1, s.d_model, dtype=torch.bfloat16, device="cuda")  # a valid pointer; no row is read
    for n in L.grads:
        L.grads[n].fill_(3.0)
    L.forward(x)
    L.backward(x, x, accumulate=True)
    torch.cuda.synchronize()
    check_no_device_error()
    weight_grads = ("dW_r", "dW1", "dW3", "dW2")
    for n in weight_grads:
        assert (L.grads[n] == 3.0).all(), n
    L.backward(x, x, accumulate=False)
    torch.cuda.synchronize()
    for n in weight_grads:
        assert not L.grads[n].any(), n
    assert not L.saved["counts"].any() and not L.saved["offsets"].any()


def test_huge_capacity_equals_dropless_bitwise():
    a = LS("huge", 500, 256, 256, 6, 2, 0.0, W.BF16, capacity=10 ** 6)
    b = a.replace(capacity=-1, capacity_factor=0.0)
    outs = []
    for s in (a, b):
        wl = W.make(s, seed=5, micro_batches=1, with_dy=False)
        L = layer.from_workload(wl, training=False)
        outs.append(L.forward(wl.x[0].torch("cuda")).clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("shape", [SMALL["top2_e8_small"], SMALL["zipf_e64_small"],
                                   LS("inf_k1_drop", 900, 256, 512, 6, 1, 0.8, W.BF16)])
def test_inference_forward_is_bit_identical_run_to_run(shape):
    """The inference forward of a bf16 layer with k <= 2 adds each kept row into
    y from the down product's epilogue; with at most two additions onto a zeroed
    element the order in which they land cannot change y, so repeated runs are
    bit for bit equal, and y matches the oracle."""
    wl = W.make(shape, seed=13, micro_batches=1, with_dy=False)
    L = layer.from_workload(wl, training=False)
    x = wl.x[0].torch("cuda")
    outs = []
    for _ in range(3):
        L.y.fill_(7.0)  # anything the forward leaves unwritten would show
        outs.append(L.forward(x)[: shape.T].clone())
    torch.cuda.synchronize()
    check_no_device_error()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert_close("y", outs[0], _oracle_fwd(wl)["y"], TOL[shape.dtype])


def test_nvtx_ranges_change_nothing():
    """With NVTX ranges on around every launch and layer call the step runs as
    without them, bit for bit."""
    s = SMALL["top2_e8_small"]
    wl = W.make(s, seed=3, micro_batches=1, with_dy=True)
    res = []
    for on in (False, True):
        pkg.moe_nvtx_enable(on)
        try:
            L = layer.from_workload(wl)
            x = wl.x[0].torch("cuda")
            L.forward(x)
            L.backward(x, wl.dy[0].torch("cuda"), accumulate=False)
            torch.cuda.synchronize()
        finally:
            pkg.moe_nvtx_enable(False)
        check_no_device_error()
        res.append([L.y.clone(), L.dx.clone(), L.grads["dW1"].clone(), L.grads["dW_r"].clone()])
    for u, v in zip(*res):
        assert torch.equal(u, v)


def test_runs_are_bit_identical():
    s = SMALL["train_e16_small"]
    wl = W.make(s, micro_batches=1, with_dy=True)
    res = []
    for _ in range(2):
        L = layer.from_workload(wl)
        x = wl.x[0].torch("cuda")
        L.forward(x)
        L.backward(x, wl.dy[0].torch("cuda"), accumulate=False)
        torch.cuda.synchronize()
        res.append([L.y.clone(), L.dx.clone()] + [L.grads[n].clone() for n in ("dW_r", "dW1", "dW3", "dW2")] +
                   [L.saved[n].clone() for n in ("ids", "slot", "row_of", "gates")])
    for u, v in zip(*res):
        assert torch.equal(u, v)


def test_corrupt_routing_state_is_reported_not_followed():
    s = SMALL["top2_e8_small"]
    wl = W.make(s, micro_batches=1, with_dy=False)
    cfg = pkg.config_of(s)
    L = layer.from_workload(wl, training=True)
    x = wl.x[0].torch("cuda")
    L.forward(x)
    torch.cuda.synchronize()
    check_no_device_error()
    bad = L.saved["row_of"].clone()
    bad[3, 0] = 10 ** 8  # far beyond max_rows
    bad[7, 1] = -5       # negative but not the -1 marker: treated as dropped
    x_perm = torch.zeros_like(L.saved["x_perm"])
    pkg.moe_permute(cfg, x, bad, L.saved["counts"], L.saved["offsets"], x_perm)
    code, detail = pkg.moe_get_device_error(clear=True)
    assert pkg.STATUS[code] == "MOE_ERR_DEVICE_CHECK"
    # every other row was still moved
    good = L.saved["row_of"][10].tolist()
    for j, r in enumerate(good):
        if r >= 0:
            assert torch.equal(x_perm[r], x[10])
    # a corrupt offsets table stops the grouped GEMM before any tile is read
    offs = L.saved["offsets"].clone()
    offs[2] = offs[1] + 5  # not a multiple of 128
    pkg.moe_grouped_ffn(cfg, L.saved["x_perm"], L.saved["counts"], offs, L.weights["W1"], L.weights["W3"],
                        L.weights["W2"], L.saved["h"], L.saved["y_perm"])
    code, _ = pkg.moe_get_device_error(clear=True)
    assert pkg.STATUS[code] == "MOE_ERR_DEVICE_CHECK"


# ------------------------------ failure detection ------------------------- #
def test_bounded_wait_reports_timeout_and_gpu_stays_usable():
    """A pipeline wait that nothing satisfies gives up after its limit and
    reports MOE_ERR_TIMEOUT; the control (a warp arrives) reports nothing, and
    a full layer step runs correctly afterwards."""
    import time

    pkg.moe_get_device_error(clear=True)
    pkg.moe_selftest_bounded_wait(50_000_000, arrive=True)
    code, _ = pkg.moe_get_device_error(clear=True)
    assert code == 0
    t0 = time.perf_counter()
    pkg.moe_selftest_bounded_wait(50_000_000, arrive=False)
    code, detail = pkg.moe_get_device_error(clear=True)
    waited = time.perf_counter() - t0
    assert pkg.STATUS[code] == "MOE_ERR_TIMEOUT"
    assert (detail & 0xFFFFFF) == 700
    assert 0.04 < waited < 5.0
    test_layer_forward("top2_e8_small")


@pytest.mark.parametrize("k", [1, 2])
def test_permute_then_unpermute_is_identity_on_gpu(k):
    """moe_permute followed by moe_unpermute_combine with gates summing to 1 in
    powers of two (1, or 0.5 + 0.5) gives x back bit for bit: every token is kept
    (dropless), each of its rows is an exact copy, and the fp32 sum of the
    halves of a bf16 value is that value."""
    s = LS(f"ident_k{k}", 777, 256, 256, 8, k, 0.0, W.BF16)
    wl = W.make(s, seed=11, micro_batches=1, with_dy=False)
    cfg = pkg.config_of(s)
    L = layer.from_workload(wl, training=True)
    x = wl.x[0].torch("cuda")
    L.forward(x)
    sv = L.saved
    x_perm = torch.zeros(L.max_rows, s.d_model, dtype=torch.bfloat16, device="cuda")
    pkg.moe_permute(cfg, x, sv["row_of"], sv["counts"], sv["offsets"], x_perm)
    gates = torch.full((s.T, k), 1.0 / k, dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    pkg.moe_unpermute_combine(cfg, x_perm, sv["row_of"], gates, y)
    torch.cuda.synchronize()
    check_no_device_error()
    assert (sv["slot"] >= 0).all()
    assert torch.equal(y, x)


@pytest.mark.parametrize("shape", [SMALL["top2_e8_small"], SMALL["zipf_e64_small"], SMALL["dropless_e32_small"],
                                   SMALL["train_f32_small"],
                                   LS("inf_ragged", 65, 256, 512, 3, 2, 2.0, W.BF16),
                                   LS("inf_one", 1, 256, 256, 8, 2, 1.25, W.BF16),
                                   LS("inf_cap0", 200, 256, 256, 4, 2, 1.0, W.BF16, capacity=0),
                                   LS("inf_e128_k8", 300, 256, 256, 128, 8, 1.0, W.BF16)])
def test_inference_forward(shape):
    """Forward without saved state (permuted rows and products in the workspace,
    nothing kept for a backward); y must match the oracle."""
    wl = W.make(shape, seed=12, micro_batches=1, with_dy=False)
    L = layer.from_workload(wl, training=False)
    y = L.forward(wl.x[0].torch("cuda"))
    torch.cuda.synchronize()
    check_no_device_error()
    st = _oracle_fwd(wl)
    assert_close("y", y[: shape.T], st["y"], 1e-4 if shape.dtype == W.F32 else 2e-2)


@pytest.mark.parametrize("name", ["train_e16_small", "top2_e8_small", "train_f32_small"])
def test_recompute_variant_matches_oracle_and_the_saving_path(name):
    """Keeping neither a, b nor h (the backward recomputes them with the same up
    product): y, dx and every gradient over two accumulated micro-batches match
    the oracle's training step at the layer's tolerance, and bit for bit the
    layer that keeps them."""
    s = SMALL[name]
    tol = TOL[s.dtype]
    wl = W.make(s, seed=21, micro_batches=2, with_dy=True)
    ref = O.train_step([x.f64() for x in wl.x], [dy.f64() for dy in wl.dy], wl.W_r, wl.bias, wl.W1.f64(),
                       wl.W3.f64(), wl.W2.f64(), s.k, _cap(s))
    res = []
    for recompute in (False, True):
        L = layer.from_workload(wl, recompute=recompute)
        assert (L.saved["a"] is None) == recompute
        out = []
        for m in range(2):
            x, dy = wl.x[m].torch("cuda"), wl.dy[m].torch("cuda")
            L.forward(x)
            L.backward(x, dy, accumulate=m > 0)
            torch.cuda.synchronize()
            check_no_device_error()
            st, gr = ref["micro_batches"][m]
            assert_routing_equal(L.saved, st, s.T)
            assert_close(f"y[{m}] recompute={recompute}", L.y[: s.T], st["y"], tol)
            assert_close(f"dx[{m}] recompute={recompute}", L.dx[: s.T], gr["dx"], tol)
            out += [L.y[: s.T].clone(), L.dx[: s.T].clone()]
        for n in ("dW_r", "dW1", "dW3", "dW2"):
            assert_close(f"{n} recompute={recompute}", L.grads[n], ref["grads"][n], tol)
        out += [L.grads[n].clone() for n in ("dW_r", "dW1", "dW3", "dW2")]
        res.append(out)
    for u, v in zip(*res):
        assert torch.equal(u, v)


@pytest.mark.parametrize("E,k,extra", [(8, 2, 3), (32, 4, 3), (64, 2, 3), (32, 2, 2), (5, 1, 2), (128, 8, 3)])
def test_router_more_tiles_than_sms_matches_oracle(E, k, extra):
    """More 128-token tiles than SMs (the router runs without a K split, two CTAs
    an SM up to 32 experts, each tile starting its K loop at its own k-block;
    even and odd tile counts, expert padding with E = 5, and E = 128 with k = 8):
    routing must match the oracle bit for bit and the probabilities and gates
    to fp32 rounding."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = 128 * (sms + extra) + 44  # sms + extra + 1 tiles, the last one partial
    s = LS(f"two_tiles_e{E}", T, 256, 256, E, k, 1.25, W.BF16)
    wl = W.make(s, seed=14, micro_batches=1, with_dy=False)
    L = layer.from_workload(wl)
    L.forward(wl.x[0].torch("cuda"))
    torch.cuda.synchronize()
    check_no_device_error()
    st = O.route(wl.x[0].f64(), wl.W_r, wl.bias, k, _cap(s))
    assert_routing_equal(L.saved, st, T)
    assert_close("probs", L.saved["probs"], st["probs"], 1e-5)
    assert_close("gates", L.saved["gates"], st["gates"], 1e-5)
