"""CPU oracle for the mixture-of-experts layer step (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call this
module: only the tests, the package smoke check and the CPU-baseline leg of the
benchmark use it.  It shares no code with the CUDA library and imports nothing
from it.

It is a plain, slow statement of what the layer computes, in float64, with one
numpy matmul per expert as the only library primitive.  The steps and their
order follow the pages:

* "The step timeline: dispatch, expert GEMM, combine" (gpu_expert_parallel
  page): the router scores every token, tokens are permuted into contiguous
  per-destination buffers, the local experts run over whatever arrived, and the
  inverse permutation restores the original token order; backward walks the
  same path in reverse.
* "The Capacity Factor: A Dial Between Imbalance and Dropping" (distributed
  training tutorial, Expert Parallelism section): each expert reserves room for
  a fixed number of tokens; the excess is dropped.
* "Recomputation re-runs the dispatch unless you save the permutation"
  (gpu_expert_parallel page): backward reuses the saved assignment indices and
  permutation map instead of re-routing.
* "Sharded by expert, replicated everywhere else" (gpu_expert_parallel page):
  the router's gradient is that of an ordinary shared parameter.

Readings where the pages leave a step open (each is also listed in the
design notes):

1. capacity C = ceil(cf * T * k / E); cf <= 0 means no capacity (dropless);
2. slots are filled first choices first, then second choices, each in token
   order;
3. gates are computed before the drop and are not renormalised after it;
   a dropped assignment contributes zero and receives zero gate gradient;
4. k = 1: the gate is the softmax probability of the chosen expert; k > 1:
   the softmax probabilities of the picks renormalised over the picks;
5. top-k is taken on the logits (monotone with the probabilities), in fp32 --
   the router precision the layer configurations fix -- with ties going to the
   lower expert index;
6. expert FFN is SwiGLU without biases: (silu(x W1) * (x W3)) W2,
   silu(z) = z / (1 + exp(-z));
7. the router bias is a fixed term (no gradient); gradients are summed (not
   averaged) over micro-batches;
8. the auxiliary load-balancing loss, which the tutorial's MoE configuration
   example only names ("aux_loss coeff"), is taken in its usual expert-balance
   form L = coeff * E * sum_e f_e * P_e, where f_e is the share of the T*k
   assignments that chose expert e before the capacity drop (a count: no
   gradient flows through it) and P_e the mean router probability of e; it is
   off (coeff = 0) unless asked for.

Data layout of the permutation map (the library's convention, adopted here so
that row numbers compare exactly): each expert's rows start at a multiple of
128; rows of expert e are [offsets[e], offsets[e] + counts[e]) followed by
zero pad rows up to offsets[e+1].
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np

ROW_ALIGN = 128


# --------------------------------------------------------------------------- #
# Routing: router scoring, top-k, gates, capacity, slots, permutation map
# --------------------------------------------------------------------------- #
def capacity(T: int, k: int, E: int, capacity_factor: float, override: int = -1) -> Optional[int]:
    """Tokens each expert can hold; None when there is no capacity (dropless).

    The capacity-factor passage of the Expert Parallelism section: each expert
    reserves capacity for a fixed number of tokens, and the tokens actually
    exchanged are token count x experts routed to; hence C = ceil(cf*T*k/E).
    The factor is taken at float32 precision, as the library receives it.
    """
    if override >= 0:
        return int(override)
    if capacity_factor <= 0:
        return None
    cf = float(np.float32(capacity_factor))
    return int(math.ceil(cf * T * k / E))


def router_logits(x: np.ndarray, W_r: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    """l = x W_r + b in float64 (the router scores every token against every expert)."""
    l = np.asarray(x, np.float64) @ np.asarray(W_r, np.float64)
    if bias is not None:
        l = l + np.asarray(bias, np.float64)[None, :]
    return l


def softmax(l: np.ndarray) -> np.ndarray:
    z = l - l.max(axis=1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=1, keepdims=True)


def topk(l: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest fp32 logits per token, descending, ties to the lower index."""
    l32 = np.asarray(l, np.float64).astype(np.float32)
    order = np.argsort(-l32, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def gates_of(p: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """k=1: g = p[e1].  k>1: g_j = p[e_j] / sum_i p[e_i] (renormalised over the picks)."""
    picked = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    if ids.shape[1] == 1:
        return picked
    return picked / picked.sum(axis=1, keepdims=True)


def assign_slots(ids: np.ndarray, E: int, C: Optional[int]):
    """Capacity slotting with overflow drop.

    Assignments are visited choice-major (all first choices in token order, then
    all second choices, ...).  Each expert hands out slots 0, 1, 2, ... in that
    visiting order; an assignment that finds its expert full is dropped
    (slot -1).  Returns (slot [T,k], counts [E] of kept assignments).
    """
    T, k = ids.shape
    filled = [0] * E
    slot = np.full((T, k), -1, dtype=np.int32)
    for j in range(k):
        for t in range(T):
            e = int(ids[t, j])
            if C is None or filled[e] < C:
                slot[t, j] = filled[e]
                filled[e] += 1
    return slot, np.array(filled, dtype=np.int32)


def permutation_map(ids: np.ndarray, slot: np.ndarray, counts: np.ndarray):
    """Row layout of the per-expert buffers: (offsets [E+1], row_of [T,k], src_token [rows])."""
    E = counts.shape[0]
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + ROW_ALIGN * ((int(counts[e]) + ROW_ALIGN - 1) // ROW_ALIGN)
    T, k = ids.shape
    row_of = np.full((T, k), -1, dtype=np.int32)
    src_token = np.full(int(offsets[E]), -1, dtype=np.int32)
    for t in range(T):
        for j in range(k):
            if slot[t, j] >= 0:
                r = int(offsets[ids[t, j]]) + int(slot[t, j])
                row_of[t, j] = r
                src_token[r] = t
    return offsets.astype(np.int32), row_of, src_token


def route(x, W_r, bias, k: int, C: Optional[int]) -> Dict[str, np.ndarray]:
    """Router scoring, top-k, gates, capacity slotting and the permutation map."""
    E = W_r.shape[1]
    l = router_logits(x, W_r, bias)
    p = softmax(l)
    ids = topk(l, k)
    g = gates_of(p, ids)
    slot, counts = assign_slots(ids, E, C)
    offsets, row_of, src_token = permutation_map(ids, slot, counts)
    return dict(logits=l, probs=p, ids=ids, gates=g, slot=slot, counts=counts,
                offsets=offsets, row_of=row_of, src_token=src_token)


# --------------------------------------------------------------------------- #
# Permute, expert FFN, unpermute + combine
# --------------------------------------------------------------------------- #
def permute(x: np.ndarray, row_of: np.ndarray, rows: int) -> np.ndarray:
    """x_perm[row_of[t,j]] = x[t] for kept assignments; every other row is zero."""
    xp = np.zeros((rows, x.shape[1]), dtype=np.float64)
    T, k = row_of.shape
    for t in range(T):
        for j in range(k):
            r = row_of[t, j]
            if r >= 0:
                xp[r] = x[t]
    return xp


def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def sigmoid(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def expert_ffn(X: np.ndarray, W1e: np.ndarray, W3e: np.ndarray, W2e: np.ndarray):
    """SwiGLU expert: a = X W1, b = X W3, h = silu(a) * b, Y = h W2 (float64)."""
    a = X @ W1e
    b = X @ W3e
    h = silu(a) * b
    return a, b, h, h @ W2e


def grouped_ffn(x_perm, offsets, counts, W1, W3, W2):
    """Each expert's FFN over its contiguous row segment; pad rows stay zero."""
    rows = x_perm.shape[0]
    f = W1.shape[2]
    d = W2.shape[2]
    a = np.zeros((rows, f))
    b = np.zeros((rows, f))
    h = np.zeros((rows, f))
    Y = np.zeros((rows, d))
    for e in range(W1.shape[0]):
        r0, n = int(offsets[e]), int(counts[e])
        if n == 0:
            continue
        sl = slice(r0, r0 + n)
        a[sl], b[sl], h[sl], Y[sl] = expert_ffn(x_perm[sl], W1[e], W3[e], W2[e])
    return a, b, h, Y


def unpermute_combine(Y_perm: np.ndarray, row_of: np.ndarray, gates: np.ndarray) -> np.ndarray:
    """y[t] = sum over kept j of g[t,j] * Y_perm[row_of[t,j]]; all dropped -> 0."""
    T, k = row_of.shape
    y = np.zeros((T, Y_perm.shape[1]))
    for t in range(T):
        for j in range(k):
            r = row_of[t, j]
            if r >= 0:
                y[t] += gates[t, j] * Y_perm[r]
    return y


def forward(x, W_r, bias, W1, W3, W2, k: int, C: Optional[int]) -> Dict[str, np.ndarray]:
    """One layer forward; returns every intermediate the backward needs."""
    x = np.asarray(x, np.float64)
    W1, W3, W2 = (np.asarray(w, np.float64) for w in (W1, W3, W2))
    st = route(x, W_r, bias, k, C)
    rows = int(st["offsets"][-1])
    st["x_perm"] = permute(x, st["row_of"], rows)
    st["a"], st["b"], st["h"], st["Y_perm"] = grouped_ffn(st["x_perm"], st["offsets"], st["counts"], W1, W3, W2)
    st["y"] = unpermute_combine(st["Y_perm"], st["row_of"], st["gates"])
    return st


# --------------------------------------------------------------------------- #
# Backward
# --------------------------------------------------------------------------- #
def combine_backward(dy: np.ndarray, st) -> tuple:
    """Token-gradient routing: dY_perm[row] = g * dy[t];  dg[t,j] = <dy[t], Y_perm[row]> (0 if dropped)."""
    row_of, g, Yp = st["row_of"], st["gates"], st["Y_perm"]
    T, k = row_of.shape
    dYp = np.zeros_like(Yp)
    dg = np.zeros((T, k))
    for t in range(T):
        for j in range(k):
            r = row_of[t, j]
            if r >= 0:
                dYp[r] = g[t, j] * dy[t]
                dg[t, j] = float(np.dot(dy[t], Yp[r]))
    return dYp, dg


def ffn_backward(dYp, st, W1, W3, W2):
    """Per expert: dH = dY W2^T; SwiGLU backward; dX = da W1^T + db W3^T; weight gradients."""
    W1, W3, W2 = (np.asarray(w, np.float64) for w in (W1, W3, W2))
    E, d, f = W1.shape
    dXp = np.zeros_like(st["x_perm"])
    dW1 = np.zeros((E, d, f))
    dW3 = np.zeros((E, d, f))
    dW2 = np.zeros((E, f, d))
    da_all = np.zeros_like(st["a"])
    db_all = np.zeros_like(st["b"])
    for e in range(E):
        r0, n = int(st["offsets"][e]), int(st["counts"][e])
        if n == 0:
            continue
        sl = slice(r0, r0 + n)
        a, b, h, X, dY = st["a"][sl], st["b"][sl], st["h"][sl], st["x_perm"][sl], dYp[sl]
        dH = dY @ W2[e].T
        s = sigmoid(a)
        da = dH * b * s * (1.0 + a * (1.0 - s))
        db = dH * silu(a)
        dXp[sl] = da @ W1[e].T + db @ W3[e].T
        dW2[e] = h.T @ dY
        dW1[e] = X.T @ da
        dW3[e] = X.T @ db
        da_all[sl], db_all[sl] = da, db
    return dict(dX_perm=dXp, dW1=dW1, dW3=dW3, dW2=dW2, da=da_all, db=db_all)


def router_logit_grad(dg: np.ndarray, st) -> np.ndarray:
    """dL/dl from the gate gradients.

    k > 1: g is a softmax over the picked logits, so dl[e_j] = g_j (dg_j - sum_i g_i dg_i)
    and zero on unpicked experts.  k = 1: g = p[e1], so dl = g dg (onehot(e1) - p).
    """
    ids, g, p = st["ids"], st["gates"], st["probs"]
    T, k = ids.shape
    dl = np.zeros_like(p)
    for t in range(T):
        if k == 1:
            e1 = int(ids[t, 0])
            dl[t] = -g[t, 0] * dg[t, 0] * p[t]
            dl[t, e1] += g[t, 0] * dg[t, 0]
        else:
            s = float(np.dot(g[t], dg[t]))
            for j in range(k):
                dl[t, int(ids[t, j])] += g[t, j] * (dg[t, j] - s)
    return dl


def aux_loss(probs: np.ndarray, ids: np.ndarray, coeff: float):
    """Auxiliary load-balancing loss and its logit gradient (reading 8).

    f_e = #{(t, j): ids[t, j] = e} / (T k)      assignment share before the drop
    P_e = (1/T) sum_t probs[t, e]              mean router probability
    L   = coeff * E * sum_e f_e P_e
    With p = softmax(l) per token, dP_e / dl[t, e'] = p[t, e] (delta_ee' - p[t, e']) / T, so
    dL/dl[t, e'] = coeff * E / T * p[t, e'] * (f_e' - sum_e f_e p[t, e]).
    Returns (L, dL/dl [T, E]).
    """
    p = np.asarray(probs, np.float64)
    T, E = p.shape
    k = ids.shape[1]
    f = np.zeros(E)
    for t in range(T):
        for j in range(k):
            f[int(ids[t, j])] += 1.0
    f /= T * k
    P = p.mean(axis=0)
    loss = coeff * E * float(np.dot(f, P))
    dl = np.zeros_like(p)
    for t in range(T):
        s = float(np.dot(f, p[t]))
        dl[t] = coeff * E / T * p[t] * (f - s)
    return loss, dl


def backward(dy, x, W_r, W1, W3, W2, st, aux_coeff: float = 0.0) -> Dict[str, np.ndarray]:
    """Layer backward from the saved routing state (no re-routing).  With
    aux_coeff > 0 the auxiliary loss's logit gradient joins dl (reading 8)."""
    dy = np.asarray(dy, np.float64)
    x = np.asarray(x, np.float64)
    dYp, dg = combine_backward(dy, st)
    fb = ffn_backward(dYp, st, W1, W3, W2)
    dl = router_logit_grad(dg, st)
    aux = None
    if aux_coeff > 0:
        aux, dl_aux = aux_loss(st["probs"], st["ids"], aux_coeff)
        dl = dl + dl_aux
    row_of = st["row_of"]
    T, k = row_of.shape
    dx = dl @ np.asarray(W_r, np.float64).T
    for t in range(T):
        for j in range(k):
            r = row_of[t, j]
            if r >= 0:
                dx[t] += fb["dX_perm"][r]
    out = dict(dx=dx, dW_r=x.T @ dl, dl=dl, dg=dg, dY_perm=dYp)
    if aux is not None:
        out["aux_loss"] = aux
    out.update(fb)
    return out


def train_step(xs, dys, W_r, bias, W1, W3, W2, k: int, C: Optional[int]) -> Dict[str, np.ndarray]:
    """Forward + backward over micro-batches, summing the weight gradients (no 1/n)."""
    acc = None
    outs = []
    for x, dy in zip(xs, dys):
        st = forward(x, W_r, bias, W1, W3, W2, k, C)
        gr = backward(dy, x, W_r, W1, W3, W2, st)
        outs.append((st, gr))
        if acc is None:
            acc = {n: gr[n].copy() for n in ("dW_r", "dW1", "dW3", "dW2")}
        else:
            for n in acc:
                acc[n] += gr[n]
    return dict(grads=acc, micro_batches=outs)


# --------------------------------------------------------------------------- #
# Exact outputs at full size, one token or a few weight columns at a time.
# The same formulas as above restricted to a subset, for layers too large to
# run whole on the CPU.
# --------------------------------------------------------------------------- #
def token_outputs(t: int, x, dy, W_r, bias, W1, W3, W2, st, want_dx: bool = True) -> Dict[str, np.ndarray]:
    """y[t] and (optionally) dx[t] of token t from the routing state ``st`` of its batch.

    ``st`` needs ids, gates, probs and slot (from ``route`` on the full batch);
    a token's output depends only on its own row, its picks and whether each
    pick was kept.
    """
    xt = np.asarray(x[t], np.float64)
    k = st["ids"].shape[1]
    Ys, dX = [], np.zeros_like(xt)
    y = np.zeros_like(xt)
    for j in range(k):
        e = int(st["ids"][t, j])
        if st["slot"][t, j] < 0:
            Ys.append(None)
            continue
        a, b, h, Y = expert_ffn(xt[None, :], np.asarray(W1[e], np.float64), np.asarray(W3[e], np.float64),
                                np.asarray(W2[e], np.float64))
        Ys.append((a[0], b[0], Y[0]))
        y += st["gates"][t, j] * Y[0]
    out = dict(y=y)
    if not want_dx:
        return out
    dyt = np.asarray(dy[t], np.float64)
    dg = np.array([[0.0 if Ys[j] is None else float(np.dot(dyt, Ys[j][2])) for j in range(k)]])
    one = {n: st[n][t:t + 1] for n in ("ids", "gates", "probs")}
    dl = router_logit_grad(dg, one)[0]
    for j in range(k):
        if Ys[j] is None:
            continue
        e = int(st["ids"][t, j])
        a, b, _ = Ys[j]
        dY = st["gates"][t, j] * dyt
        dH = np.asarray(W2[e], np.float64) @ dY
        s = sigmoid(a)
        da = dH * b * s * (1.0 + a * (1.0 - s))
        db = dH * silu(a)
        dX += np.asarray(W1[e], np.float64) @ da + np.asarray(W3[e], np.float64) @ db
    out["dx"] = dX + np.asarray(W_r, np.float64) @ dl
    out["dl"] = dl
    out["dg"] = dg[0]
    return out


def weight_grad_columns(x, dy, W1, W3, W2, st, cols) -> Dict[str, np.ndarray]:
    """dW1[:, :, cols], dW3[:, :, cols] and dW2[:, cols, :] of one micro-batch.

    Column j of a, b, h, dH, da, db depends only on column j of W1, W3 and row j
    of W2, so the expert backward restricted to ``cols`` is exact.
    """
    cols = np.asarray(cols)
    E = W1.shape[0]
    d = W1.shape[1]
    out = dict(dW1=np.zeros((E, d, cols.size)), dW3=np.zeros((E, d, cols.size)),
               dW2=np.zeros((E, cols.size, W2.shape[2])))
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    T, k = st["ids"].shape
    for e in range(E):
        toks, gs = [], []
        for j in range(k):
            for t in range(T):
                if st["ids"][t, j] == e and st["slot"][t, j] >= 0:
                    toks.append(t)
                    gs.append(st["gates"][t, j])
        if not toks:
            continue
        X = x[toks]
        dY = np.asarray(gs)[:, None] * dy[toks]
        W1c = np.asarray(W1[e][:, cols], np.float64)
        W3c = np.asarray(W3[e][:, cols], np.float64)
        W2r = np.asarray(W2[e][cols, :], np.float64)
        a = X @ W1c
        b = X @ W3c
        h = silu(a) * b
        dH = dY @ W2r.T
        s = sigmoid(a)
        da = dH * b * s * (1.0 + a * (1.0 - s))
        db = dH * silu(a)
        out["dW1"][e] = X.T @ da
        out["dW3"][e] = X.T @ db
        out["dW2"][e] = h.T @ dY
    return out
