"""GPU parity at the full layer sizes, in the launch configuration bench.py times.

Routing state is compared whole and bit-exactly.  Floats are compared whole
where the float64 oracle can run the full layer in seconds (the top-2 E=8 and
the Zipf E=64 layers), and otherwise on sampled tokens (y, dx) and sampled
weight columns (dW1, dW3, dW2), which the oracle computes exactly one at a
time.  Tolerance: max|gpu - ref| <= 2e-2 * max|ref| per tensor.
"""
import numpy as np
import pytest
import torch

import routing_permute_grouped_router_gb300 as pkg
from _util import assert_close, assert_routing_equal, check_no_device_error
from oracle import moe_oracle as O
from routing_permute_grouped_router_gb300 import layer
from routing_permute_grouped_router_gb300 import workload as W

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from routing_permute_grouped_router_gb300 import build

    build.build()
    pkg.lib()
    torch.cuda.set_device(0)
    pkg.moe_get_device_error(clear=True)


def _cap(s):
    return O.capacity(s.T, s.k, s.E, s.capacity_factor, s.capacity)


def _sample(T, n, seed):
    return np.sort(np.random.default_rng(seed).choice(T, size=min(n, T), replace=False))


def test_top2_e8_full_forward_backward_and_repeat_accumulation():
    s = W.WORKLOADS["top2_e8_bf16"]
    wl = W.make(s, micro_batches=1, with_dy=True)
    L = layer.from_workload(wl)
    x, dy = wl.x[0].torch("cuda"), wl.dy[0].torch("cuda")
    L.forward(x)
    L.backward(x, dy, accumulate=False)
    torch.cuda.synchronize()
    check_no_device_error()
    g1 = {n: L.grads[n].clone() for n in L.grads}
    st = O.forward(wl.x[0].f64(), wl.W_r, wl.bias, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), s.k, _cap(s))
    gr = O.backward(wl.dy[0].f64(), wl.x[0].f64(), wl.W_r, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), st)
    assert_routing_equal(L.saved, st, s.T)
    rows = int(st["offsets"][-1])
    assert_close("h", L.saved["h"][:rows], st["h"], TOL)
    assert_close("y", L.y, st["y"], TOL)
    assert_close("dx", L.dx, gr["dx"], TOL)
    for n in ("dW_r", "dW1", "dW3", "dW2"):
        assert_close(n, L.grads[n], gr[n], TOL)
    # the bench repeats the step with accumulate=1: same input twice doubles the
    # fp32 gradients exactly, because every step is deterministic
    L.forward(x)
    L.backward(x, dy, accumulate=True)
    torch.cuda.synchronize()
    for n in g1:
        assert torch.equal(L.grads[n], 2 * g1[n]), n


def test_zipf_e64_full_forward_counts_and_drop_rate():
    s = W.WORKLOADS["zipf_e64_bf16"]
    wl = W.make(s, micro_batches=1, with_dy=False)
    L = layer.from_workload(wl)
    L.forward(wl.x[0].torch("cuda"))
    torch.cuda.synchronize()
    check_no_device_error()
    st = O.forward(wl.x[0].f64(), wl.W_r, wl.bias, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), s.k, _cap(s))
    assert_routing_equal(L.saved, st, s.T)
    counts = L.saved["counts"].cpu().numpy()
    assert counts.max() == _cap(s)  # the hottest experts overflow
    drop = 1.0 - counts.sum() / (s.T * s.k)
    assert 0.5 < drop < 0.95, drop
    assert_close("y", L.y, st["y"], TOL)


def test_dropless_e32_routing_full_and_sampled_outputs():
    s = W.WORKLOADS["dropless_e32_bf16"]
    wl = W.make(s, micro_batches=1, with_dy=False)
    L = layer.from_workload(wl, training=True)
    L.forward(wl.x[0].torch("cuda"))
    torch.cuda.synchronize()
    check_no_device_error()
    st = O.route(wl.x[0].f64(), wl.W_r, wl.bias, s.k, None)
    assert_routing_equal(L.saved, st, s.T)
    counts = st["counts"]
    assert counts.sum() == s.T * s.k  # dropless keeps everything
    share = counts / counts.sum()
    assert share.max() > 0.15 and share.min() < 0.01  # ragged groups
    W1, W3, W2 = wl.W1.f32, wl.W3.f32, wl.W2.f32
    toks = _sample(s.T, 256, 1)
    ref = np.stack([O.token_outputs(t, wl.x[0].f32, None, wl.W_r, wl.bias, W1, W3, W2, st, want_dx=False)["y"]
                    for t in toks])
    assert_close("y[sampled]", L.y[torch.from_numpy(toks).cuda()], ref, TOL)


def test_dropless_e32_full_backward_sampled():
    """The largest layer's backward at full size, twice accumulated: dx on sampled
    tokens and dW1, dW3, dW2 on sampled columns against the oracle (the long-K
    wgrad and dgrad h shapes run here)."""
    s = W.WORKLOADS["dropless_e32_bf16"]
    wl = W.make(s, micro_batches=1, with_dy=True)
    L = layer.from_workload(wl)
    x, dy = wl.x[0].torch("cuda"), wl.dy[0].torch("cuda")
    L.forward(x)
    L.backward(x, dy, accumulate=False)
    L.backward(x, dy, accumulate=True)
    torch.cuda.synchronize()
    check_no_device_error()
    xs, dys = wl.x[0].f32, wl.dy[0].f32
    W1, W3, W2 = wl.W1.f32, wl.W3.f32, wl.W2.f32
    st = O.route(xs, wl.W_r, wl.bias, s.k, None)
    assert_routing_equal(L.saved, st, s.T)
    toks = _sample(s.T, 96, 3)
    outs = [O.token_outputs(t, xs, dys, wl.W_r, wl.bias, W1, W3, W2, st) for t in toks]
    assert_close("dx[sampled]", L.dx[torch.from_numpy(toks).cuda()], np.stack([o["dx"] for o in outs]), TOL)
    cols = _sample(s.d_ff, 24, 4)
    c = O.weight_grad_columns(xs, dys, W1, W3, W2, st, cols)
    ci = torch.from_numpy(cols).cuda()
    assert_close("dW1[:, :, cols]", L.grads["dW1"][:, :, ci], 2 * c["dW1"], TOL)
    assert_close("dW3[:, :, cols]", L.grads["dW3"][:, :, ci], 2 * c["dW3"], TOL)
    assert_close("dW2[:, cols, :]", L.grads["dW2"][:, ci, :], 2 * c["dW2"], TOL)


def test_large_layer_logit_gradient_from_the_dgrad_h_product():
    """A bf16 layer whose Y_perm would be at least 256 MB (T k d = 2^27) takes each kept
    row's g * dg from the dgrad h epilogue instead of reading Y_perm back: the logit
    gradient reaches dx (router term) and dW_r, compared whole with the oracle."""
    s = W.LayerShape("fused_dg", 16384, 2048, 256, 8, 4, 0.0, W.BF16)
    assert s.T * s.k * s.d_model * 2 >= 256 << 20
    wl = W.make(s, micro_batches=1, with_dy=True)
    L = layer.from_workload(wl)
    x, dy = wl.x[0].torch("cuda"), wl.dy[0].torch("cuda")
    L.forward(x)
    L.backward(x, dy, accumulate=False)
    torch.cuda.synchronize()
    check_no_device_error()
    st = O.forward(wl.x[0].f64(), wl.W_r, wl.bias, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), s.k, _cap(s))
    gr = O.backward(wl.dy[0].f64(), wl.x[0].f64(), wl.W_r, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), st)
    assert_routing_equal(L.saved, st, s.T)
    assert_close("y", L.y, st["y"], TOL)
    assert_close("dx", L.dx, gr["dx"], TOL)
    for n in ("dW_r", "dW1", "dW3", "dW2"):
        assert_close(n, L.grads[n], gr[n], TOL)


def test_dropless_skewed_wgrad_host_and_guest_tiles_sampled():
    """wgrad with interleaved host and guest tiles away from the benchmark shape.

    Dropless top-4 over 32 log-Zipf(1.3) experts, T = 8192, d = 2048, f = 1024:
    the busiest expert gets about 7,700 rows (60 stages of 128) and the idlest
    a few dozen, so the tiles are listed by expert size and each of the 96
    pair tiles per expert may host guests; the first rounds' hosts lie in the
    two busiest experts and carry two to four guests each, and later rounds
    straddle experts of different sizes.  dW on sampled columns of every expert
    and dx on sampled tokens against the oracle, after two accumulated passes.
    """
    s = W.LayerShape("dropless_skewed", 8192, 2048, 1024, 32, 4, 0.0, W.BF16, zipf_s=1.3)
    wl = W.make(s, micro_batches=1, with_dy=True)
    L = layer.from_workload(wl)
    x, dy = wl.x[0].torch("cuda"), wl.dy[0].torch("cuda")
    L.forward(x)
    L.backward(x, dy, accumulate=False)
    L.backward(x, dy, accumulate=True)
    torch.cuda.synchronize()
    check_no_device_error()
    xs, dys = wl.x[0].f32, wl.dy[0].f32
    W1, W3, W2 = wl.W1.f32, wl.W3.f32, wl.W2.f32
    st = O.route(xs, wl.W_r, wl.bias, s.k, None)
    assert_routing_equal(L.saved, st, s.T)
    counts = np.bincount(st["ids"].ravel(), minlength=s.E)
    assert counts.max() >= 60 * 128 - 128 and counts.max() >= 8 * counts.min()
    toks = _sample(s.T, 48, 5)
    outs = [O.token_outputs(t, xs, dys, wl.W_r, wl.bias, W1, W3, W2, st) for t in toks]
    assert_close("dx[sampled]", L.dx[torch.from_numpy(toks).cuda()], np.stack([o["dx"] for o in outs]), TOL)
    cols = np.concatenate([_sample(s.d_ff, 12, 6), [0, 255, 256, s.d_ff - 1]])
    cols = np.unique(cols)
    c = O.weight_grad_columns(xs, dys, W1, W3, W2, st, cols)
    ci = torch.from_numpy(cols).cuda()
    assert_close("dW1[:, :, cols]", L.grads["dW1"][:, :, ci], 2 * c["dW1"], TOL)
    assert_close("dW3[:, :, cols]", L.grads["dW3"][:, :, ci], 2 * c["dW3"], TOL)
    assert_close("dW2[:, cols, :]", L.grads["dW2"][:, ci, :], 2 * c["dW2"], TOL)


def test_train_e16_four_micro_batches_sampled():
    s = W.WORKLOADS["train_e16_bf16"]
    wl = W.make(s)
    L = layer.from_workload(wl)
    W1, W3, W2 = wl.W1.f32, wl.W3.f32, wl.W2.f32
    cols = _sample(s.d_ff, 48, 2)
    acc = None
    dWr = np.zeros((s.d_model, s.E))
    for m in range(s.micro_batches):
        x, dy = wl.x[m].torch("cuda"), wl.dy[m].torch("cuda")
        L.forward(x)
        L.backward(x, dy, accumulate=m > 0)
        torch.cuda.synchronize()
        check_no_device_error()
        xs, dys = wl.x[m].f64(), wl.dy[m].f64()
        st = O.forward(xs, wl.W_r, wl.bias, W1, W3, W2, s.k, _cap(s))
        assert_routing_equal(L.saved, st, s.T)
        assert_close(f"y[{m}]", L.y, st["y"], TOL)
        _, dg = O.combine_backward(dys, st)
        dWr += xs.T @ O.router_logit_grad(dg, st)
        toks = _sample(s.T, 128, 10 + m)
        outs = [O.token_outputs(t, xs, dys, wl.W_r, wl.bias, W1, W3, W2, st) for t in toks]
        idx = torch.from_numpy(toks).cuda()
        assert_close(f"dx[{m}]", L.dx[idx], np.stack([o["dx"] for o in outs]), TOL)
        c = O.weight_grad_columns(xs, dys, W1, W3, W2, st, cols)
        acc = c if acc is None else {n: acc[n] + c[n] for n in acc}
    ci = torch.from_numpy(cols).cuda()
    assert_close("dW1[:, :, cols]", L.grads["dW1"][:, :, ci], acc["dW1"], TOL)
    assert_close("dW3[:, :, cols]", L.grads["dW3"][:, :, ci], acc["dW3"], TOL)
    assert_close("dW2[:, cols, :]", L.grads["dW2"][:, ci, :], acc["dW2"], TOL)
    assert_close("dW_r", L.grads["dW_r"], dWr, TOL)
