"""GPU parity of the auxiliary load-balancing loss (oracle reading 8) through the C ABI.

The loss value and its logit gradient come out of fp32 kernels and are compared
with the float64 oracle at the fp32 tolerance (max|gpu - ref| <= 1e-4 * max|ref|);
a whole layer backward with the loss switched on is compared at the bf16
tolerance of its layer.
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
LS = W.LayerShape


@pytest.fixture(scope="module", autouse=True)
def built():
    from routing_permute_grouped_router_gb300 import build

    build.build()
    pkg.lib()
    torch.cuda.set_device(0)
    pkg.moe_get_device_error(clear=True)


@pytest.mark.parametrize("shape,coeff", [
    (LS("aux_e8", 1000, 256, 256, 8, 2, 1.25, W.BF16), 0.01),
    (LS("aux_e128_k8", 300, 256, 256, 128, 8, 1.0, W.BF16), 0.3),
    (LS("aux_e5_k1", 513, 64, 64, 5, 1, 0.0, W.F32), 1.0),
])
def test_aux_loss_stage_matches_oracle(shape, coeff):
    wl = W.make(shape, seed=4, micro_batches=1, with_dy=False)
    L = layer.from_workload(wl, aux_loss_coeff=coeff)
    L.forward(wl.x[0].torch("cuda"))
    torch.cuda.synchronize()
    st = O.route(wl.x[0].f64(), wl.W_r, wl.bias, shape.k,
                 O.capacity(shape.T, shape.k, shape.E, shape.capacity_factor, shape.capacity))
    assert_routing_equal(L.saved, st, shape.T)
    sv = L.saved
    loss = torch.full((1,), -1.0, device="cuda")
    dl = torch.zeros(shape.T, shape.E, device="cuda")
    pkg.moe_aux_loss(L.cfg, sv["probs"], sv["ids"], loss, dl, L.ws)
    torch.cuda.synchronize()
    check_no_device_error()
    # expected values from the oracle's own routing state: its fp64 probabilities and ids
    ref_loss, ref_dl = O.aux_loss(st["probs"], st["ids"], coeff)
    assert abs(loss.item() - ref_loss) <= 1e-4 * abs(ref_loss), (loss.item(), ref_loss)
    assert_close("dl_aux", dl, ref_dl, 1e-4)
    # a second call adds the same gradient again and rewrites the same loss, bit for bit
    loss2 = torch.empty_like(loss)
    dl2 = dl.clone()
    pkg.moe_aux_loss(L.cfg, sv["probs"], sv["ids"], loss2, dl2, L.ws)
    torch.cuda.synchronize()
    assert torch.equal(loss2, loss)
    assert torch.equal(dl2, dl + dl)


@pytest.mark.parametrize("coeff", [0.01, 200.0])
def test_layer_backward_with_aux_loss_matches_oracle(coeff):
    """With the loss on, moe_layer_bwd's dW_r, dx and loss match the oracle; with a
    coefficient large enough for the term to stand out, the change it makes to dW_r
    on the GPU (with minus without) matches x^T dl_aux of the oracle."""
    s = LS("aux_train", 700, 256, 512, 16, 2, 1.25, W.BF16)
    wl = W.make(s, seed=6, micro_batches=1, with_dy=True)
    x, dy = wl.x[0].torch("cuda"), wl.dy[0].torch("cuda")
    res = {}
    for c in (coeff, 0.0):
        L = layer.from_workload(wl, aux_loss_coeff=c)
        L.forward(x)
        L.backward(x, dy, accumulate=False)
        torch.cuda.synchronize()
        check_no_device_error()
        res[c] = (L.grads["dW_r"].double().cpu().numpy(), L.dx.clone(), L.grads["aux_loss"].item())
    C = O.capacity(s.T, s.k, s.E, s.capacity_factor, s.capacity)
    st = O.forward(wl.x[0].f64(), wl.W_r, wl.bias, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), s.k, C)
    gr = O.backward(wl.dy[0].f64(), wl.x[0].f64(), wl.W_r, wl.W1.f64(), wl.W3.f64(), wl.W2.f64(), st,
                    aux_coeff=coeff)
    dWr, dx, loss = res[coeff]
    assert abs(loss - gr["aux_loss"]) <= 1e-4 * abs(gr["aux_loss"]), (loss, gr["aux_loss"])
    assert_close("dW_r", dWr, gr["dW_r"], 2e-2)
    assert_close("dx", dx, gr["dx"], 2e-2)
    if coeff >= 1.0:
        _, dl_aux = O.aux_loss(st["probs"], st["ids"], coeff)
        assert_close("dW_r(aux) - dW_r(no aux)", dWr - res[0.0][0], wl.x[0].f64().T @ dl_aux, 1e-2)


def test_zero_coefficient_leaves_the_backward_unchanged_bitwise():
    s = LS("aux_off", 400, 256, 256, 8, 2, 1.25, W.BF16)
    wl = W.make(s, seed=8, micro_batches=1, with_dy=True)
    x, dy = wl.x[0].torch("cuda"), wl.dy[0].torch("cuda")
    outs = []
    for coeff in (0.0, 0.0):
        L = layer.from_workload(wl, aux_loss_coeff=coeff)
        L.forward(x)
        L.backward(x, dy, accumulate=False)
        torch.cuda.synchronize()
        outs.append([L.dx.clone()] + [L.grads[n].clone() for n in ("dW_r", "dW1", "dW3", "dW2", "aux_loss")])
    for u, v in zip(*outs):
        assert torch.equal(u, v)
    assert outs[0][-1].item() == 0.0  # not written: the loss is off
