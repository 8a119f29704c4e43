"""CPU oracle for the DeepSeekMoE layer's backward pass -- TEST INFRASTRUCTURE ONLY.

The gradient, for an upstream gradient dy [T, d], of the layer output of
moe_oracle.moe_forward with respect to the tokens x and every parameter
(W_g, W_noise, W1, W3, W2). It is the derivative of the forward the pages
define: [DSMoE] section 3.2, eqs (9)-(11) (softmax gate over the routed
experts, top-k, shared experts at gate 1, y = sum of gated expert outputs),
the noisy top-k gate of [MoE-notes] section 2 (H = x W_g + eps *
Softplus(x W_noise), G = Softmax(KeepTopK(H, k))), GShard's ReLU expert of
[MoE-notes] section 3, and the expert capacity of [MoE-notes] sections 3-4.
Like moe_oracle it is the plain fp64 statement of the mathematics, for
checking a GPU implementation; nothing here is shared with the CUDA code.

Reading taken (the pages define no backward): the selection is held fixed.
The top-k set, and an expert capacity's keep/drop decisions, are piecewise
constant in the inputs. Away from ties they do not move under a small
perturbation, and the gradient flows through the selected gates and the
kept experts only. The per-expert selection bias of the auxiliary-loss-free
strategy ([DS-article]) steers the selection only, so it receives no
gradient.

Pinned in tests/test_oracle_backward.py against central finite differences
of the forward oracle, by linearity in dy, by token independence, by the
k = E reduction and by the fine-grained segmentation identity; planted
mistakes in each helper below must be caught there.
"""

from __future__ import annotations

import numpy as np

from oracle import moe_oracle as O

F64 = np.float64


def sigmoid(z) -> np.ndarray:
    z = np.asarray(z, dtype=F64)
    return 1.0 / (1.0 + np.exp(-z))


def silu_grad(a) -> np.ndarray:
    """d/da [a * sigmoid(a)] = sigmoid(a) (1 + a (1 - sigmoid(a)))."""
    sa = sigmoid(a)
    return sa * (1.0 + np.asarray(a, dtype=F64) * (1.0 - sa))


def softplus_grad(z) -> np.ndarray:
    """d/dz log(1 + e^z) = sigmoid(z)."""
    return sigmoid(z)


def softmax_backward(p, dp) -> np.ndarray:
    """For p = Softmax(z) row-wise: dz = p * (dp - <dp, p>)."""
    p = np.asarray(p, dtype=F64)
    dp = np.asarray(dp, dtype=F64)
    return p * (dp - (dp * p).sum(axis=-1, keepdims=True))


def expert_backward(X, W1, W3, W2, dO, act: str = "swiglu"):
    """One expert FFN over rows X [n, d] (moe_oracle.ffn), given dO [n, d]:
    SwiGLU O = (silu(X W1^T) * (X W3^T)) W2^T, or ReLU O = relu(X W1^T) W2^T.
    Returns (dX [n, d], dW1 [I, d], dW3 [I, d] or None, dW2 [d, I])."""
    X = np.asarray(X, dtype=F64)
    dO = np.asarray(dO, dtype=F64)
    W1 = np.asarray(W1, dtype=F64)
    W2 = np.asarray(W2, dtype=F64)
    a = X @ W1.T
    if act == "relu":
        h = np.maximum(a, 0.0)
        dh = dO @ W2
        da = dh * (a > 0.0)
        return da @ W1, da.T @ X, None, dO.T @ h
    W3 = np.asarray(W3, dtype=F64)
    b = X @ W3.T
    h = O.silu(a) * b
    dh = dO @ W2
    da = dh * b * silu_grad(a)
    db = dh * O.silu(a)
    return da @ W1 + db @ W3, da.T @ X, db.T @ X, dO.T @ h


def gates_backward_to_scores(dg, gates, s_sel, renormalize: bool) -> np.ndarray:
    """Gradient with respect to the selected scores s_sel [T, k] of the gates:
    g = s_sel (eq (10)), or g = s_sel / S with S = sum of s_sel (renormalised):
    ds_j = (dg_j - <dg, g>) / S."""
    dg = np.asarray(dg, dtype=F64)
    if not renormalize:
        return dg
    S = np.asarray(s_sel, dtype=F64).sum(axis=1, keepdims=True)
    return (dg - (dg * gates).sum(axis=1, keepdims=True)) / S


def moe_backward(x, W_g, W1, W3, W2, n_shared: int, top_k: int, dy, *, renormalize: bool = False,
                 noisy: bool = False, W_noise=None, eps=None, bias=None, capacity: int = 0,
                 act: str = "swiglu") -> dict:
    """Gradients of <dy, y> for y = moe_oracle.moe_forward of the same layer
    (routing by moe_oracle.route, drops by moe_oracle.capacity_keep).

    Returns a dict: dx [T, d], dW_g [d, E], dW_noise [d, E] (noisy, else
    None), dW1 / dW3 [G, I, d] (dW3 None for ReLU experts), dW2 [G, d, I],
    and the intermediate dg [T, k] (gradient of each selected gate) and
    dlogits [T, E] (of x W_g)."""
    x = O._f64(x)
    dy = O._f64(dy)
    W_g = O._f64(W_g)
    W1 = O._f64(W1)
    W2 = O._f64(W2)
    W3 = None if act == "relu" else O._f64(W3)
    T = x.shape[0]
    G = W1.shape[0]
    E = G - n_shared
    r = O.route(x, W_g, top_k, renormalize=renormalize, noisy=noisy, W_noise=W_noise, eps=eps,
                bias=bias)
    ids, gates = r["ids"], r["gates"]
    keep = (O.capacity_keep(ids, E, capacity) if capacity else np.ones(ids.shape, dtype=bool))

    dx = np.zeros_like(x)
    dW1 = np.zeros_like(W1)
    dW3 = None if W3 is None else np.zeros_like(W3)
    dW2 = np.zeros_like(W2)
    dg = np.zeros(ids.shape, dtype=F64)

    def add(e, rows, dX, dw1, dw3, dw2):
        np.add.at(dx, rows, dX)
        dW1[e] += dw1
        dW2[e] += dw2
        if dW3 is not None:
            dW3[e] += dw3

    # shared experts: every token, gate 1 (eq (9))
    for i in range(n_shared):
        add(i, np.arange(T), *expert_backward(x, W1[i], None if W3 is None else W3[i], W2[i], dy, act))
    # routed experts: the kept assignments of each, scaled by their gates
    for e in range(E):
        rows, slot = np.nonzero((ids == e) & keep)
        if rows.size == 0:
            continue
        ge = n_shared + e
        Xe = x[rows]
        out = O.ffn(Xe, W1[ge], None if W3 is None else W3[ge], W2[ge], act)
        dg[rows, slot] = (dy[rows] * out).sum(axis=1)              # d<dy, g*FFN>/dg
        g = gates[rows, slot][:, None]
        add(ge, rows, *expert_backward(Xe, W1[ge], None if W3 is None else W3[ge], W2[ge], g * dy[rows], act))

    # gates -> router logits
    dW_noise = None
    if noisy:
        # g = Softmax over the kept H: dH_sel = g * (dg - <dg, g>)
        dH = np.zeros((T, E), dtype=F64)
        np.put_along_axis(dH, ids, softmax_backward(gates, dg), axis=1)
        dlogits = dH
        n = O.gate_logits(x, W_noise)
        dn = dH * O._f64(eps) * softplus_grad(n)
        dW_noise = x.T @ dn
        dx += dn @ O._f64(W_noise).T
    else:
        s = r["s"]
        s_sel = np.take_along_axis(s, ids, axis=1)
        ds = np.zeros((T, E), dtype=F64)
        np.put_along_axis(ds, ids, gates_backward_to_scores(dg, gates, s_sel, renormalize), axis=1)
        dlogits = softmax_backward(s, ds)
    dW_g = x.T @ dlogits
    dx += dlogits @ W_g.T
    return {"dx": dx, "dW_g": dW_g, "dW_noise": dW_noise, "dW1": dW1, "dW3": dW3, "dW2": dW2,
            "dg": dg, "dlogits": dlogits}
