"""Pins of the CPU oracle to things other than itself.

Each test checks the oracle against what the pages or the mathematics fix:
hand-derived routing fixtures, brute force on tiny inputs, special cases that
reduce to a dense library computation, invariants, and central finite
differences for the backward.  The last block plants mistakes in the oracle and
checks that a pin catches each one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from routing_permute_grouped_router_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


# --------------------------------------------------------------------------- #
# Routing
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("name", ["routing_top2_capacity.json", "routing_top1_switch.json"])
def test_golden_routing(name):
    g = _load(name)
    C = O.capacity(g["T"], g["k"], g["E"], g["capacity_factor"])
    assert C == g["capacity"]
    st = O.route(np.array(g["x"], float), np.array(g["W_r"], float), None, g["k"], C)
    assert st["ids"].tolist() == g["ids"]
    assert st["slot"].tolist() == g["slot"]
    assert st["counts"].tolist() == g["counts"]
    assert st["offsets"].tolist() == g["offsets"]
    assert st["row_of"].tolist() == g["row_of"]
    np.testing.assert_allclose(st["gates"], np.array(g["gates"]), rtol=0, atol=1e-15)
    if "probs" in g:
        np.testing.assert_allclose(st["probs"], np.array(g["probs"]), rtol=0, atol=1e-15)


def test_capacity_of_the_five_layer_configs():
    # Tiny Switch layer: ceil(1.25 * 256 / 4) = 80, as its configuration states.
    expect = {"switch_tiny_f32": 80, "top2_e8_bf16": 1280, "zipf_e64_bf16": 512,
              "dropless_e32_bf16": None, "train_e16_bf16": 1280}
    for name, s in W.WORKLOADS.items():
        assert O.capacity(s.T, s.k, s.E, s.capacity_factor) == expect[name]
    assert O.capacity(10, 2, 4, 1.25, override=0) == 0


def _brute_topk(l32, k):
    """All ordered k-tuples of distinct experts; keep the lexicographically best
    sequence of (logit desc, index asc) pairs."""
    E = len(l32)
    best = None
    for tup in itertools.permutations(range(E), k):
        key = tuple((-float(l32[e]), e) for e in tup)
        if best is None or key < best[0]:
            best = (key, tup)
    return list(best[1])


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    T, E = 12, 5
    l = rng.integers(-3, 4, size=(T, E)).astype(np.float64)  # many exact ties
    for k in (1, 2, 3, 5):
        ids = O.topk(l, k)
        for t in range(T):
            assert ids[t].tolist() == _brute_topk(l[t].astype(np.float32), k)


def _brute_slots(ids, E, C):
    """slot = number of earlier assignments (choice-major, then token order) to the
    same expert, kept iff that number is below C.  Quadratic on purpose."""
    T, k = ids.shape
    order = [(j, t) for j in range(k) for t in range(T)]
    slot = np.full((T, k), -1)
    for n, (j, t) in enumerate(order):
        pos = sum(1 for (jj, tt) in order[:n] if ids[tt, jj] == ids[t, j])
        if C is None or pos < C:
            slot[t, j] = pos
    return slot


@pytest.mark.parametrize("C", [None, 0, 1, 3, 7, 100])
def test_slots_brute_force(C):
    rng = np.random.default_rng(11)
    T, E, k = 17, 4, 3
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    slot, counts = O.assign_slots(ids, E, C)
    assert slot.tolist() == _brute_slots(ids, E, C).tolist()
    for e in range(E):
        total = int((ids == e).sum())
        assert counts[e] == (total if C is None else min(total, C))


def test_permutation_map_is_a_bijection_onto_kept_rows():
    rng = np.random.default_rng(3)
    T, E, k, d = 50, 6, 2, 4
    x = rng.standard_normal((T, d))
    W_r = rng.standard_normal((d, E))
    st = O.route(x, W_r, None, k, 9)
    offs, cnt, rof, src = st["offsets"], st["counts"], st["row_of"], st["src_token"]
    assert offs[0] == 0 and all(o % 128 == 0 for o in offs)
    kept_rows = sorted(int(r) for r in rof.ravel() if r >= 0)
    expect = sorted(r for e in range(E) for r in range(offs[e], offs[e] + cnt[e]))
    assert kept_rows == expect
    for t in range(T):
        for j in range(k):
            if rof[t, j] >= 0:
                assert src[rof[t, j]] == t
                assert offs[st["ids"][t, j]] <= rof[t, j] < offs[st["ids"][t, j] + 1]
    assert (src >= 0).sum() == len(kept_rows)


def test_invariants_on_generated_workload():
    s = W.WORKLOADS["switch_tiny_f32"]
    wl = W.make(s)
    C = O.capacity(s.T, s.k, s.E, s.capacity_factor)
    st = O.route(wl.x[0].f64(), wl.W_r, wl.bias, s.k, C)
    assert (st["counts"] <= C).all()
    assert st["counts"].sum() == (st["slot"] >= 0).sum()
    s2 = s.replace(k=3, E=8, name="k3")
    wl2 = W.make(s2)
    st2 = O.route(wl2.x[0].f64(), wl2.W_r, None, 3, None)
    assert all(len(set(r)) == 3 for r in st2["ids"].tolist())
    np.testing.assert_allclose(st2["gates"].sum(axis=1), 1.0, rtol=0, atol=1e-12)
    # k = 1: the gate is the softmax probability of the chosen expert.
    g1 = np.take_along_axis(st["probs"], st["ids"].astype(np.int64), axis=1)
    np.testing.assert_array_equal(st["gates"], g1)
    assert np.all(st["probs"].argmax(axis=1) == st["ids"][:, 0])


def test_generated_margin_holds():
    s = W.WORKLOADS["top2_e8_bf16"].replace(T=512, d_model=128, d_ff=128)
    wl = W.make(s)
    l = O.router_logits(wl.x[0].f64(), wl.W_r, wl.bias)
    top = -np.sort(-l, axis=1)[:, :3]
    assert (top[:, :-1] - top[:, 1:]).min() >= 1e-3


# --------------------------------------------------------------------------- #
# Forward: special cases with a dense library computation
# --------------------------------------------------------------------------- #
def _rand_layer(rng, T, d, f, E):
    x = rng.standard_normal((T, d))
    W_r = rng.standard_normal((d, E)) / math.sqrt(d)
    W1 = rng.standard_normal((E, d, f)) / math.sqrt(d)
    W3 = rng.standard_normal((E, d, f)) / math.sqrt(d)
    W2 = rng.standard_normal((E, f, d)) / math.sqrt(f)
    return x, W_r, W1, W3, W2


def _torch_swiglu(x, W1, W3, W2):
    x, W1, W3, W2 = (torch.from_numpy(np.asarray(a, np.float64)) for a in (x, W1, W3, W2))
    return (torch.nn.functional.silu(x @ W1) * (x @ W3)) @ W2


def test_single_expert_is_dense_swiglu():
    rng = np.random.default_rng(0)
    x, W_r, W1, W3, W2 = _rand_layer(rng, 40, 8, 12, 1)
    st = O.forward(x, W_r, None, W1, W3, W2, k=1, C=40)
    np.testing.assert_allclose(st["gates"], 1.0, rtol=0, atol=0)
    ref = _torch_swiglu(x, W1[0], W3[0], W2[0]).numpy()
    np.testing.assert_allclose(st["y"], ref, rtol=1e-12, atol=1e-12)


def test_all_experts_dropless_is_soft_mixture():
    rng = np.random.default_rng(1)
    T, d, f, E = 30, 6, 10, 4
    x, W_r, W1, W3, W2 = _rand_layer(rng, T, d, f, E)
    b = rng.standard_normal(E)
    st = O.forward(x, W_r, b, W1, W3, W2, k=E, C=None)
    p = torch.softmax(torch.from_numpy(x @ W_r + b), dim=1).numpy()
    ref = sum(p[:, e:e + 1] * _torch_swiglu(x, W1[e], W3[e], W2[e]).numpy() for e in range(E))
    np.testing.assert_allclose(st["y"], ref, rtol=1e-12, atol=1e-12)


def test_capacity_zero_gives_zero_output_and_gradients():
    rng = np.random.default_rng(2)
    x, W_r, W1, W3, W2 = _rand_layer(rng, 16, 6, 8, 3)
    st = O.forward(x, W_r, None, W1, W3, W2, k=2, C=0)
    assert (st["slot"] == -1).all() and st["counts"].sum() == 0
    assert not st["y"].any()
    gr = O.backward(rng.standard_normal((16, 6)), x, W_r, W1, W3, W2, st)
    for n in ("dx", "dW_r", "dW1", "dW3", "dW2"):
        assert not gr[n].any(), n


def test_huge_capacity_equals_dropless():
    rng = np.random.default_rng(4)
    x, W_r, W1, W3, W2 = _rand_layer(rng, 25, 6, 8, 5)
    a = O.forward(x, W_r, None, W1, W3, W2, k=2, C=None)
    b = O.forward(x, W_r, None, W1, W3, W2, k=2, C=10 ** 9)
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["row_of"], b["row_of"])


def test_permute_then_unpermute_is_identity():
    rng = np.random.default_rng(5)
    T, d, E = 33, 5, 4
    x = rng.standard_normal((T, d))
    W_r = rng.standard_normal((d, E))
    for k in (1, 2, 3):
        st = O.route(x, W_r, None, k, None)
        xp = O.permute(x, st["row_of"], int(st["offsets"][-1]))
        back = O.unpermute_combine(xp, st["row_of"], st["gates"] if k > 1 else np.ones((T, 1)))
        np.testing.assert_allclose(back, x, rtol=1e-14, atol=1e-14)
    # With a capacity, dropped tokens come back as zero and kept ones unchanged.
    st = O.route(x, W_r, None, 1, 4)
    xp = O.permute(x, st["row_of"], int(st["offsets"][-1]))
    back = O.unpermute_combine(xp, st["row_of"], np.ones((T, 1)))
    kept = st["slot"][:, 0] >= 0
    np.testing.assert_array_equal(back[kept], x[kept])
    assert not back[~kept].any()


def test_partially_dropped_token_keeps_pre_drop_gate():
    # Token 1's second pick (expert 0) finds expert 0 full; its output is the first
    # pick's FFN scaled by the gate computed over both picks.
    x = np.array([[2.0, 0.0], [0.5, 1.5]])
    W_r = np.eye(2)
    rng = np.random.default_rng(6)
    W1 = rng.standard_normal((2, 2, 3))
    W3 = rng.standard_normal((2, 2, 3))
    W2 = rng.standard_normal((2, 3, 2))
    st = O.forward(x, W_r, None, W1, W3, W2, k=2, C=1)
    assert st["slot"].tolist() == [[0, -1], [0, -1]]
    g1 = 1.0 / (1.0 + math.exp(-1.0))  # picks differ by 1 logit
    ref = g1 * _torch_swiglu(x[1:2], W1[1], W3[1], W2[1]).numpy()[0]
    np.testing.assert_allclose(st["y"][1], ref, rtol=1e-13)


# --------------------------------------------------------------------------- #
# Backward: central finite differences in float64
# --------------------------------------------------------------------------- #
def _loss(x, W_r, b, W1, W3, W2, k, C, dy):
    return float((O.forward(x, W_r, b, W1, W3, W2, k, C)["y"] * dy).sum())


@pytest.mark.parametrize("k,C", [(1, 4), (2, 5), (2, None), (3, 3)])
def test_backward_matches_finite_differences(k, C):
    rng = np.random.default_rng(100 + k)
    T, d, f, E = 12, 6, 7, 4
    x, W_r, W1, W3, W2 = _rand_layer(rng, T, d, f, E)
    b = 0.3 * rng.standard_normal(E)
    l = x @ W_r + b
    srt = -np.sort(-l, axis=1)
    assert (srt[:, :-1] - srt[:, 1:]).min() > 1e-4  # no routing flip within h
    dy = rng.standard_normal((T, d))
    st = O.forward(x, W_r, b, W1, W3, W2, k, C)
    assert (st["slot"] < 0).any() or C is None  # the capacity cases drop something
    gr = O.backward(dy, x, W_r, W1, W3, W2, st)
    params = dict(x=x, W_r=W_r, W1=W1, W3=W3, W2=W2)
    grads = dict(x=gr["dx"], W_r=gr["dW_r"], W1=gr["dW1"], W3=gr["dW3"], W2=gr["dW2"])
    h = 1e-6
    for name in params:
        for _ in range(3):
            v = rng.standard_normal(params[name].shape)
            plus = dict(params)
            minus = dict(params)
            plus[name] = params[name] + h * v
            minus[name] = params[name] - h * v
            fd = (_loss(plus["x"], plus["W_r"], b, plus["W1"], plus["W3"], plus["W2"], k, C, dy)
                  - _loss(minus["x"], minus["W_r"], b, minus["W1"], minus["W3"], minus["W2"], k, C, dy)) / (2 * h)
            an = float((grads[name] * v).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_gradient_accumulation_sums_micro_batches():
    rng = np.random.default_rng(9)
    T, d, f, E, k = 10, 4, 6, 3, 2
    _, W_r, W1, W3, W2 = _rand_layer(rng, T, d, f, E)
    xs = [rng.standard_normal((T, d)) for _ in range(3)]
    dys = [rng.standard_normal((T, d)) for _ in range(3)]
    res = O.train_step(xs, dys, W_r, None, W1, W3, W2, k, 6)
    for n in ("dW_r", "dW1", "dW3", "dW2"):
        sep = sum(O.backward(dy, x, W_r, W1, W3, W2, O.forward(x, W_r, None, W1, W3, W2, k, 6))[n]
                  for x, dy in zip(xs, dys))
        np.testing.assert_allclose(res["grads"][n], sep, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------- #
# Auxiliary load-balancing loss (reading 8: coeff * E * sum_e f_e P_e)
# --------------------------------------------------------------------------- #
def test_aux_loss_balanced_routing_is_the_coefficient_with_zero_gradient():
    # uniform probabilities and an equal share of assignments per expert: f = P = 1/E,
    # so L = coeff * E * E * (1/E)^2 = coeff, and no logit can lower it to first order
    T, E, k, coeff = 12, 4, 2, 0.37
    probs = np.full((T, E), 1.0 / E)
    ids = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)])
    loss, dl = O.aux_loss(probs, ids, coeff)
    assert abs(loss - coeff) < 1e-15
    assert np.abs(dl).max() < 1e-15


def test_aux_loss_collapsed_routing_is_coefficient_times_experts():
    # every assignment and all probability on expert 0: f_0 = P_0 = 1, L = coeff * E
    T, E, coeff = 5, 6, 0.01
    probs = np.zeros((T, E))
    probs[:, 0] = 1.0
    loss, _ = O.aux_loss(probs, np.zeros((T, 1), dtype=np.int64), coeff)
    assert abs(loss - coeff * E) < 1e-15


def test_aux_loss_hand_computed_example():
    # T = 2, E = 2, k = 1, both tokens pick expert 0: f = (1, 0);
    # P = ((0.75 + 0.5) / 2, (0.25 + 0.5) / 2) = (0.625, 0.375); L = c * 2 * 0.625 = 1.25 c
    probs = np.array([[0.75, 0.25], [0.5, 0.5]])
    loss, dl = O.aux_loss(probs, np.array([[0], [0]]), 0.2)
    assert abs(loss - 0.25) < 1e-15
    # dl[t, e'] = c E / T p[t, e'] (f_e' - sum_e f_e p[t, e]): token 0: s = 0.75
    np.testing.assert_allclose(dl[0], [0.2 * 0.75 * 0.25, 0.2 * 0.25 * -0.75], rtol=0, atol=1e-15)


def test_aux_loss_gradient_matches_finite_differences():
    rng = np.random.default_rng(77)
    T, E, k, coeff = 9, 5, 2, 0.3
    l = rng.standard_normal((T, E))
    ids = np.argsort(-l, axis=1, kind="stable")[:, :k]

    def L(logits):
        return O.aux_loss(O.softmax(logits), ids, coeff)[0]

    _, dl = O.aux_loss(O.softmax(l), ids, coeff)
    h = 1e-6
    for _ in range(5):
        v = rng.standard_normal(l.shape)
        fd = (L(l + h * v) - L(l - h * v)) / (2 * h)
        assert abs(fd - float((dl * v).sum())) <= 1e-8, fd


def test_backward_with_aux_loss_matches_finite_differences():
    # total loss <dy, y> + L_aux as a function of W_r and x (routing fixed within h)
    rng = np.random.default_rng(31)
    T, d, f, E, k, C, coeff = 12, 6, 7, 4, 2, 5, 0.5
    x, W_r, W1, W3, W2 = _rand_layer(rng, T, d, f, E)
    l = x @ W_r
    srt = -np.sort(-l, axis=1)
    assert (srt[:, :-1] - srt[:, 1:]).min() > 1e-4
    dy = rng.standard_normal((T, d))
    st = O.forward(x, W_r, None, W1, W3, W2, k, C)
    gr = O.backward(dy, x, W_r, W1, W3, W2, st, aux_coeff=coeff)
    assert abs(gr["aux_loss"] - O.aux_loss(st["probs"], st["ids"], coeff)[0]) < 1e-15

    def total(xx, wr):
        s2 = O.forward(xx, wr, None, W1, W3, W2, k, C)
        return float((s2["y"] * dy).sum()) + O.aux_loss(s2["probs"], s2["ids"], coeff)[0]

    h = 1e-6
    for name, base, g in (("W_r", W_r, gr["dW_r"]), ("x", x, gr["dx"])):
        for _ in range(3):
            v = rng.standard_normal(base.shape)
            if name == "W_r":
                fd = (total(x, W_r + h * v) - total(x, W_r - h * v)) / (2 * h)
            else:
                fd = (total(x + h * v, W_r) - total(x - h * v, W_r)) / (2 * h)
            an = float((g * v).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


# --------------------------------------------------------------------------- #
# Planted mistakes: each must be caught by one of the pins above
# --------------------------------------------------------------------------- #
def _pins_pass():
    try:
        test_single_expert_is_dense_swiglu()
        test_all_experts_dropless_is_soft_mixture()
        test_golden_routing("routing_top2_capacity.json")
        test_golden_routing("routing_top1_switch.json")
        for k, C in [(1, 4), (2, 5)]:
            test_backward_matches_finite_differences(k, C)
        test_slots_brute_force(3)
        test_aux_loss_balanced_routing_is_the_coefficient_with_zero_gradient()
        test_aux_loss_hand_computed_example()
        test_aux_loss_gradient_matches_finite_differences()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("mutation", [
    "silu_is_sigmoid", "transposed_w2", "gate_not_renormalised", "second_choice_first",
    "router_grad_sign", "missing_router_dx", "slot_off_by_one", "aux_share_per_token", "aux_grad_sign",
])
def test_planted_mistake_is_caught(monkeypatch, mutation):
    if mutation == "silu_is_sigmoid":
        monkeypatch.setattr(O, "silu", O.sigmoid)
    elif mutation == "transposed_w2":
        orig = O.expert_ffn

        def bad(X, W1e, W3e, W2e):
            a, b, h, Y = orig(X, W1e, W3e, W2e)
            return a, b, h, h @ W2e[::-1]
        monkeypatch.setattr(O, "expert_ffn", bad)
    elif mutation == "gate_not_renormalised":
        monkeypatch.setattr(O, "gates_of", lambda p, ids: np.take_along_axis(p, ids.astype(np.int64), axis=1))
    elif mutation == "second_choice_first":
        orig = O.assign_slots

        def bad(ids, E, C):
            s, c = orig(ids[:, ::-1].copy(), E, C)
            return s[:, ::-1].copy(), c
        monkeypatch.setattr(O, "assign_slots", bad)
    elif mutation == "router_grad_sign":
        orig = O.router_logit_grad
        monkeypatch.setattr(O, "router_logit_grad", lambda dg, st: -orig(dg, st))
    elif mutation == "missing_router_dx":
        orig = O.router_logit_grad

        def bad(dg, st):
            return np.zeros_like(orig(dg, st))
        monkeypatch.setattr(O, "router_logit_grad", bad)
    elif mutation == "slot_off_by_one":
        orig = O.assign_slots

        def bad(ids, E, C):
            s, c = orig(ids, E, None if C is None else C + 1)
            return s, c
        monkeypatch.setattr(O, "assign_slots", bad)
    elif mutation == "aux_grad_sign":
        orig = O.aux_loss

        def bad(probs, ids, coeff):
            loss, dl = orig(probs, ids, coeff)
            return loss, -dl
        monkeypatch.setattr(O, "aux_loss", bad)
    elif mutation == "aux_share_per_token":
        orig = O.aux_loss

        def bad(probs, ids, coeff):  # f_e divided by T instead of T k
            k = ids.shape[1]
            loss, dl = orig(probs, ids, coeff * k)
            return loss, dl
        monkeypatch.setattr(O, "aux_loss", bad)
    assert not _pins_pass(), mutation


def test_token_and_column_helpers_agree_with_the_whole_layer():
    rng = np.random.default_rng(21)
    T, d, f, E, k = 40, 6, 9, 5, 2
    x, W_r, W1, W3, W2 = _rand_layer(rng, T, d, f, E)
    dy = rng.standard_normal((T, d))
    st = O.forward(x, W_r, None, W1, W3, W2, k, 9)
    gr = O.backward(dy, x, W_r, W1, W3, W2, st)
    assert (st["slot"] < 0).any()
    for t in (0, 7, 39):
        o = O.token_outputs(t, x, dy, W_r, None, W1, W3, W2, st)
        np.testing.assert_allclose(o["y"], st["y"][t], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(o["dx"], gr["dx"][t], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(o["dl"], gr["dl"][t], rtol=1e-12, atol=1e-12)
    cols = [0, 4, 8]
    c = O.weight_grad_columns(x, dy, W1, W3, W2, st, cols)
    np.testing.assert_allclose(c["dW1"], gr["dW1"][:, :, cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(c["dW3"], gr["dW3"][:, :, cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(c["dW2"], gr["dW2"][:, cols, :], rtol=1e-12, atol=1e-12)
