"""CPU oracle for the DeepSeekMoE layer forward -- TEST INFRASTRUCTURE ONLY.

This module is the plain, slow, fp64 statement of what the layer computes. It
exists to check the CUDA library. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does, and
nothing here is shared with the CUDA kernels (no helpers, tables or
constants flow either way).

Sources (each function cites the passage it follows):
  [DSMoE]     "DeepSeekMoE: Towards Ultimate Expert Specialization in
              Mixture-of-Experts Language Models", Chinese translation
              (gitcode.csdn.net): section 2 eqs (3)-(5), section 3.1 eqs
              (6)-(8), section 3.2 eqs (9)-(11), section 3.3 eqs (12)-(17).
  [MoE-notes] "Mixture of Experts" study notes (blog.carolineworld.cn):
              section 2 "Outrageously Large Neural Networks" (MoE layer
              output, softmax gating, noisy top-k gating, importance loss),
              section 3 "GShard" (expert FFN, running counter c_e),
              section 4 "Switch Transformers" (load-balancing loss),
              section 5 "ST-MoE" (router z-loss, float32 router).
  [DS-article] "DeepSeek MoE: innovation and breakthrough of the mixture of
              experts architecture" (cloud.tencent.com), section on the
              auxiliary-loss-free load-balancing strategy (per-expert bias).

Readings taken where the pages are silent (all listed in the design notes):
  * the softmax of eq (11) runs over the routed experts only;
  * ties in top-k go to the lowest expert index, and the k outputs are listed
    by descending key;
  * the expert FFN is SwiGLU, W2 (silu(W1 x) * (W3 x)), silu(z) = z*sigmoid(z);
  * the per-expert bias of the auxiliary-loss-free strategy is added to the
    selection key only (key = s + b); the gate stays s;
  * noise draws of the noisy gate are an input (eps), not drawn here;
  * CV is the population coefficient of variation.

Everything is computed in float64 from the stored input values (bf16 inputs
are widened exactly).

Parity pins: every function here is pinned by the not-gpu tests in
tests/test_oracle_pins.py (closed forms, brute force on tiny inputs,
structural reductions between the equations, and the combinatorics the
DeepSeekMoE translation prints in section 3.1). The choice of SwiGLU as the
expert FFN, the bias scale and the noise values are fixed by the workload
definition, not by the pages: "parity unpinned" for the choice of activation.
"""

from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    """Widen an array (numpy, or a CPU torch tensor in any float dtype) to fp64."""
    if hasattr(a, "detach"):  # torch tensor: widen through fp32, exact for bf16
        a = a.detach().float().numpy()
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------------
# Gate: affinities, softmax and top-k
# --------------------------------------------------------------------------

def gate_logits(x, W_g) -> np.ndarray:
    """Token-to-centroid affinities u_t^T e_i for every routed expert.

    [DSMoE] section 3.2, eq (11): s_{i,t} = Softmax_i(u_t^T e_i); the centroids
    e_i are the columns of W_g ([MoE-notes] section 2, softmax gating x . W_g).
    x: [T, d]; W_g: [d, E]. Returns [T, E] fp64.
    """
    return _f64(x) @ _f64(W_g)


def softmax(z: np.ndarray) -> np.ndarray:
    """Row softmax, exp(z_i - max) / sum_j exp(z_j - max).  [DSMoE] eq (11)."""
    z = np.asarray(z, dtype=F64)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def softplus(z: np.ndarray) -> np.ndarray:
    """log(1 + e^z), written out stably.  [MoE-notes] section 2, noisy top-k."""
    z = np.asarray(z, dtype=F64)
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + e^-z); the SwiGLU activation."""
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def topk_order(key: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k of each row of `key`, by descending key, ties to the lower index.

    [DSMoE] eq (10): Topk({s_j}, K) is the set of the K largest affinities.
    The pages leave ties open; the reading is lowest index first. A stable
    sort of -key keeps equal keys in index order, which is that rule.
    Returns (ids [T, k] int64, margin [T]) where margin = key of the k-th
    pick minus the key of the (k+1)-th (inf when k equals the row length).
    """
    key = np.asarray(key, dtype=F64)
    order = np.argsort(-key, axis=1, kind="stable")
    ids = order[:, :k]
    kth = np.take_along_axis(key, order[:, k - 1:k], axis=1)[:, 0]
    if k < key.shape[1]:
        nxt = np.take_along_axis(key, order[:, k:k + 1], axis=1)[:, 0]
        margin = kth - nxt
    else:
        margin = np.full(key.shape[0], np.inf)
    return ids, margin


def route(x, W_g, top_k: int, *, renormalize: bool = False,
          noisy: bool = False, W_noise=None, eps=None, bias=None) -> dict:
    """Gate of one MoE layer: selection of top_k routed experts and their gates.

    softmax gate ([DSMoE] eqs (10)-(11)):
        s = Softmax(x W_g); selected = Topk(s, k); g_i = s_i on the selected
        set, 0 elsewhere. With renormalize, g_i = s_i / sum_selected s_j
        (the KeepTopK-then-Softmax form of [MoE-notes] section 2 gives the
        same renormalised gates when the noise is zero).
    bias (auxiliary-loss-free balancing, [DS-article]): selection key s_i + b_i,
        gate s_i (the bias steers selection only).
    noisy ([MoE-notes] section 2, Noisy Top-K Gating):
        H_i = (x W_g)_i + eps_i * Softplus((x W_noise)_i),
        G = Softmax(KeepTopK(H, k)), i.e. the softmax of H over the kept
        entries (the others are -inf and get gate 0).

    Returns a dict with ids [T,k] (descending key, ties to lower index),
    gates [T,k], s [T,E] (softmax of the plain logits), logits [T,E],
    key [T,E] (what was sorted), margin [T] (k-th minus (k+1)-th of the
    comparison key: the plain logits in softmax mode, s + b with a bias,
    H when noisy) and, when noisy, H [T,E].
    """
    logits = gate_logits(x, W_g)
    s = softmax(logits)
    out = {"logits": logits, "s": s}
    if noisy:
        if bias is not None:
            raise ValueError("noisy gating and a selection bias are not combined")
        noise_logits = gate_logits(x, W_noise)
        H = logits + _f64(eps) * softplus(noise_logits)
        ids, margin = topk_order(H, top_k)
        kept = np.take_along_axis(H, ids, axis=1)
        gates = softmax(kept)          # softmax over KeepTopK: -inf entries add 0
        out.update(H=H, key=H)
    else:
        if bias is not None:
            key = s + _f64(bias)[None, :]
            ids, margin = topk_order(key, top_k)
        else:
            key = s
            ids, _ = topk_order(key, top_k)
            # margin on the logits: Softmax is strictly increasing, so the
            # order of s is the order of the logits
            _, margin = topk_order(logits, top_k)
        gates = np.take_along_axis(s, ids, axis=1)
        if renormalize:
            gates = gates / gates.sum(axis=1, keepdims=True)
        out.update(key=key)
    out.update(ids=ids, gates=gates, margin=margin)
    return out


def dense_gates(ids: np.ndarray, gates: np.ndarray, n_experts: int) -> np.ndarray:
    """The sparse gate vector G(x) of [MoE-notes] section 2 / g_{i,t} of [DSMoE]
    eq (10) as a dense [T, E] matrix: the gate on the selected experts, 0 elsewhere."""
    T = ids.shape[0]
    G = np.zeros((T, n_experts), dtype=F64)
    np.put_along_axis(G, ids, gates, axis=1)
    return G


# --------------------------------------------------------------------------
# Dispatch: per-expert counts and token groups
# --------------------------------------------------------------------------

def capacity_keep(ids: np.ndarray, n_experts: int, capacity: int) -> np.ndarray:
    """Which assignments an expert with a capacity accepts.

    [MoE-notes] section 3 (GShard, expert capacity): the gate keeps a running
    counter c_e of the tokens sent to expert e; once c_e reaches the capacity
    the expert takes no more, and the overflowing token's assignment is
    dropped (its gate for that expert becomes zero; the token still reaches
    the output through the residual). Section 4 (Switch) sets the capacity to
    tokens/experts x capacity factor. Reading: tokens arrive in ascending
    order, and a token's k picks in its listed order, i.e. ascending flat
    assignment index t*k + j. capacity = 0 means no limit (the DeepSeekMoE
    layer is dropless). Returns keep [T, k] bool.
    """
    ids = np.asarray(ids)
    keep = np.ones(ids.shape, dtype=bool)
    if capacity <= 0:
        return keep
    c = np.zeros(n_experts, dtype=np.int64)   # the running counters c_e
    for t in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            if c[e] < capacity:
                c[e] += 1
            else:
                keep[t, j] = False
    return keep


def dispatch(ids: np.ndarray, n_experts: int, capacity: int = 0) -> dict:
    """Group the T*k assignments by expert.

    The pages state only that each token is assigned to its selected experts
    ([DSMoE] section 2) and that a running counter c_e tracks how many tokens
    an expert has received ([MoE-notes] section 3, expert capacity). The
    reading: counts[e] = c_e after all tokens; rows of expert e are laid out
    contiguously after those of experts < e (offsets = exclusive prefix sum
    of counts), in ascending flat assignment index t*k + j (so ascending
    token within an expert).

    With a capacity (capacity_keep), dropped assignments take no row: counts
    are the accepted counts, and their dest is -1.

    Returns counts [E], offsets [E+1], perm_src [sum(counts)] (flat assignment
    index of each grouped row) and dest [T, k] (grouped row of each
    assignment, -1 if dropped).
    """
    ids = np.asarray(ids)
    flat = ids.reshape(-1)
    kept = capacity_keep(ids, n_experts, capacity).reshape(-1)
    counts = np.bincount(flat[kept], minlength=n_experts).astype(np.int64)
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")
    perm_src = order[kept[order]]
    dest = np.full(flat.size, -1, dtype=np.int64)
    dest[perm_src] = np.arange(perm_src.size)
    return {"counts": counts, "offsets": offsets, "perm_src": perm_src,
            "dest": dest.reshape(ids.shape)}


# --------------------------------------------------------------------------
# Experts and the layer output
# --------------------------------------------------------------------------

def expert_ffn(X, W1, W3, W2) -> np.ndarray:
    """One expert FFN over a batch of rows: W2 (silu(W1 x) * (W3 x)).

    Each expert is a standard FFN ([DSMoE] section 2); GShard's form is
    wo . ReLU(wi . x) ([MoE-notes] section 3). The gated SwiGLU variant is
    the workload's choice. W1, W3: [I, d]; W2: [d, I]; X: [n, d].
    """
    X = _f64(X)
    a = X @ _f64(W1).T
    b = X @ _f64(W3).T
    return (silu(a) * b) @ _f64(W2).T


def expert_ffn_relu(X, wi, wo) -> np.ndarray:
    """GShard's expert FFN_e(x) = wo . ReLU(wi . x) ([MoE-notes] section 3).
    wi: [I, d]; wo: [d, I]."""
    h = np.maximum(_f64(X) @ _f64(wi).T, 0.0)
    return h @ _f64(wo).T


def ffn(X, W1, W3, W2, act: str = "swiglu") -> np.ndarray:
    """The expert FFN of the layer: SwiGLU W2 (silu(W1 x) * (W3 x)), or GShard's
    W2 . ReLU(W1 x) (act = "relu", W3 unused)."""
    if act == "relu":
        return expert_ffn_relu(X, W1, W2)
    return expert_ffn(X, W1, W3, W2)


def moe_forward(x, W1, W3, W2, n_shared: int, ids, gates,
                tokens=None, act: str = "swiglu", keep=None) -> np.ndarray:
    """Layer output without the residual:
        y_t = sum_{i<K_s} FFN_i(u_t) + sum_{j<k} g_{t,j} FFN_{K_s+ids[t,j]}(u_t).

    [DSMoE] section 3.2, eq (9) (minus the +u_t term, which the caller adds).
    Expert weights are stacked shared first, then routed, as in eq (9)'s
    numbering. Sparse evaluation ([MoE-notes] section 2: E_i is not computed
    where G(x)_i = 0): each expert runs only on the tokens that select it.

    `tokens` (optional) restricts the output to a subset of token indices;
    tokens are independent, so the rows of that subset are exact. `act`
    selects the expert FFN (see ffn). `keep` [T, k] (optional, from
    capacity_keep) drops the assignments an expert's capacity refused.
    Returns y [len(tokens) or T, d] fp64.
    """
    x = _f64(x)
    ids = np.asarray(ids)
    gates = _f64(gates)
    if keep is not None:
        gates = np.where(np.asarray(keep), gates, 0.0)
        ids = np.where(np.asarray(keep), ids, -1)
    if tokens is None:
        tokens = np.arange(x.shape[0])
    tokens = np.asarray(tokens)
    xs = x[tokens]
    ids_s = ids[tokens]
    g_s = gates[tokens]
    W3i = (lambda i: None) if act == "relu" else (lambda i: W3[i])
    y = np.zeros((tokens.size, x.shape[1]), dtype=F64)
    for i in range(n_shared):
        y += ffn(xs, W1[i], W3i(i), W2[i], act)
    n_routed = W1.shape[0] - n_shared
    for e in range(n_routed):
        rows, slot = np.nonzero(ids_s == e)
        if rows.size == 0:
            continue
        o = ffn(xs[rows], W1[n_shared + e], W3i(n_shared + e), W2[n_shared + e], act)
        np.add.at(y, rows, g_s[rows, slot][:, None] * o)
    return y


def moe_forward_dense(x, W1, W3, W2, n_shared: int, G) -> np.ndarray:
    """Dense form y = sum_shared FFN_i(x) + sum_i G_i E_i(x) over all routed
    experts ([MoE-notes] section 2, y = sum_i G(x)_i E_i(x)); every expert is
    evaluated and multiplied by its (possibly zero) gate. Used to pin the
    sparse evaluation of moe_forward."""
    x = _f64(x)
    G = _f64(G)
    y = np.zeros_like(x)
    for i in range(n_shared):
        y += expert_ffn(x, W1[i], W3[i], W2[i])
    for e in range(G.shape[1]):
        y += G[:, e:e + 1] * expert_ffn(x, W1[n_shared + e], W3[n_shared + e], W2[n_shared + e])
    return y


def expert_rows(x, W1, W3, W2, n_shared: int, perm_src, offsets, top_k: int,
                act: str = "swiglu") -> np.ndarray:
    """Per-row expert outputs, unweighted, in the grouped layout.

    Rows [0, K_s*T): shared expert i on token t at row i*T + t.
    Rows K_s*T + r: routed expert e on grouped row r in [offsets[e], offsets[e+1]),
    whose token is perm_src[r] // top_k. Returns [K_s*T + T*k, d] fp64.
    """
    x = _f64(x)
    T = x.shape[0]
    W3i = (lambda i: None) if act == "relu" else (lambda i: W3[i])
    out = np.zeros((n_shared * T + perm_src.size, x.shape[1]), dtype=F64)
    for i in range(n_shared):
        out[i * T:(i + 1) * T] = ffn(x, W1[i], W3i(i), W2[i], act)
    n_routed = offsets.size - 1
    for e in range(n_routed):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            toks = np.asarray(perm_src[a:b]) // top_k
            out[n_shared * T + a:n_shared * T + b] = ffn(
                x[toks], W1[n_shared + e], W3i(n_shared + e), W2[n_shared + e], act)
    return out


def combine(rows, dest, gates, n_shared: int, T: int) -> np.ndarray:
    """Gate-weighted combine of per-row expert outputs back to token order:
    y_t = sum_i rows[i*T + t] + sum_j g_{t,j} rows[K_s*T + dest[t,j]]
    ([DSMoE] eq (9); [MoE-notes] section 3, y_s = sum_e G_{s,e} FFN_e(x_s))."""
    rows = _f64(rows)
    gates = _f64(gates)
    y = np.zeros((T, rows.shape[1]), dtype=F64)
    for i in range(n_shared):
        y += rows[i * T:(i + 1) * T]
    dest = np.asarray(dest)
    kept = dest >= 0   # assignments an expert's capacity dropped add nothing
    y += np.einsum("tk,tkd->td", np.where(kept, gates, 0.0),
                   rows[n_shared * T + np.where(kept, dest, 0)])
    return y


# --------------------------------------------------------------------------
# Balance statistics (forward by-products; not on the layer's output path)
# --------------------------------------------------------------------------

def cv_squared(v) -> float:
    """Squared coefficient of variation, population variance / mean^2
    ([MoE-notes] section 2, L_importance = w * CV(Importance)^2)."""
    v = _f64(v)
    m = v.mean()
    return float(((v - m) ** 2).mean() / (m * m))


def importance(G) -> np.ndarray:
    """Importance(X) = sum over the batch of the gate vectors G(x)
    ([MoE-notes] section 2, Balancing Expert Utilization)."""
    return _f64(G).sum(axis=0)


def expert_balance_loss(ids, s, n_routed: int, top_k: int, alpha1: float) -> float:
    """L_ExpBal = alpha1 * sum_i f_i P_i with f_i = N'/(K'T) * #{t selects i},
    P_i = (1/T) sum_t s_{i,t}. [DSMoE] section 3.3, eqs (12)-(14)."""
    ids = np.asarray(ids)
    T = ids.shape[0]
    cnt = np.bincount(ids.reshape(-1), minlength=n_routed)
    f = n_routed / (top_k * T) * cnt
    P = _f64(s).mean(axis=0)
    return float(alpha1 * np.sum(f * P))


def device_balance_loss(ids, s, n_routed: int, top_k: int, groups, alpha2: float) -> float:
    """L_DevBal = alpha2 * sum_d f'_d P'_d, f'_d = mean of f_j over group d,
    P'_d = sum of P_j over group d. [DSMoE] section 3.3, eqs (15)-(17)."""
    ids = np.asarray(ids)
    T = ids.shape[0]
    cnt = np.bincount(ids.reshape(-1), minlength=n_routed)
    f = n_routed / (top_k * T) * cnt
    P = _f64(s).mean(axis=0)
    tot = 0.0
    for g in groups:
        g = np.asarray(g)
        tot += f[g].mean() * P[g].sum()
    return float(alpha2 * tot)


def switch_balance_loss(p, alpha: float) -> float:
    """Switch Transformer loss = alpha * N * sum_i f_i P_i, f_i the fraction of
    tokens whose argmax is i, P_i the mean router probability
    ([MoE-notes] section 4, A Differentiable Load Balancing Loss)."""
    p = _f64(p)
    T, N = p.shape
    top1, _ = topk_order(p, 1)
    f = np.bincount(top1[:, 0], minlength=N) / T
    P = p.mean(axis=0)
    return float(alpha * N * np.sum(f * P))


def logsumexp(logits) -> np.ndarray:
    """Per-token log sum_j exp(x_j), with max subtraction: the term the router
    z-loss squares ([MoE-notes] section 5, ST-MoE). [T]."""
    z = _f64(logits)
    m = z.max(axis=1, keepdims=True)
    return m[:, 0] + np.log(np.exp(z - m).sum(axis=1))


def prob_column_sums(logits) -> np.ndarray:
    """sum_t s_{i,t}: the softmax router probabilities summed over tokens, so
    that P_i = (1/T) of it ([DSMoE] section 3.3, eq (14); the Switch loss's
    P_i, [MoE-notes] section 4). [E]."""
    return softmax(logits).sum(axis=0)


def router_z_loss(logits) -> float:
    """L_z = (1/B) sum_b (log sum_j exp(x_j^(b)))^2 ([MoE-notes] section 5, ST-MoE)."""
    z = _f64(logits)
    m = z.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(z - m).sum(axis=1))
    return float(np.mean(lse ** 2))
