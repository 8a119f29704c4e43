"""Pins of the CPU oracle to facts the pages and mathematics fix (no GPU).

Every check here is independent of the oracle's own code: closed forms,
brute force in plain Python loops on tiny inputs, structural reductions
between the DeepSeekMoE equations, and the combinatorics the DeepSeekMoE
translation prints. tests/test_oracle_mutants.py plants plausible mistakes
in the oracle and checks that these pins catch them.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def py_silu(z: float) -> float:
    return z / (1.0 + math.exp(-z))


def py_ffn(xv, W1, W3, W2):
    """Plain-loop SwiGLU expert on one token: W2 (silu(W1 x) * (W3 x))."""
    I, d = len(W1), len(W1[0])
    h = []
    for i in range(I):
        a = sum(W1[i][c] * xv[c] for c in range(d))
        b = sum(W3[i][c] * xv[c] for c in range(d))
        h.append(py_silu(a) * b)
    return [sum(W2[r][i] * h[i] for i in range(I)) for r in range(len(W2))]


def py_forward(x, W_g, W1, W3, W2, n_shared, k, renorm=False):
    """Eq (9)-(11) of the DeepSeekMoE translation, token by token, in Python
    floats: softmax over routed affinities, brute-force top-k over all
    k-subsets (largest sum, then lexicographically smallest index tuple),
    gates s_i (optionally renormalised), shared experts at gate 1."""
    T, d = x.shape
    E = W_g.shape[1]
    ys, all_ids = [], []
    for t in range(T):
        xv = [float(v) for v in x[t]]
        logit = [sum(xv[c] * float(W_g[c, i]) for c in range(d)) for i in range(E)]
        m = max(logit)
        ex = [math.exp(v - m) for v in logit]
        Z = sum(ex)
        s = [v / Z for v in ex]
        best = None
        for sub in itertools.combinations(range(E), k):
            key = (sum(s[i] for i in sub), tuple(-i for i in sub))
            if best is None or key > best[0]:
                best = (key, sub)
        sel = sorted(best[1], key=lambda i: (-s[i], i))
        g = [s[i] for i in sel]
        if renorm:
            tot = sum(g)
            g = [v / tot for v in g]
        y = [0.0] * d
        for i in range(n_shared):
            o = py_ffn(xv, W1[i].tolist(), W3[i].tolist(), W2[i].tolist())
            y = [a + b for a, b in zip(y, o)]
        for gi, e in zip(g, sel):
            o = py_ffn(xv, W1[n_shared + e].tolist(), W3[n_shared + e].tolist(),
                       W2[n_shared + e].tolist())
            y = [a + gi * b for a, b in zip(y, o)]
        ys.append(y)
        all_ids.append(sel)
    return np.array(ys), np.array(all_ids)


def tiny_layer(seed, T=5, d=6, E=5, K_s=1, I=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    W_g = rng.standard_normal((d, E)) * 0.5
    W1 = rng.standard_normal((K_s + E, I, d)) * 0.4
    W3 = rng.standard_normal((K_s + E, I, d)) * 0.4
    W2 = rng.standard_normal((K_s + E, d, I)) * 0.4
    return x, W_g, W1, W3, W2


# ---------------------------------------------------------------- top-k

@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 4), (7, 7)])
def test_topk_matches_subset_brute_force(seed, E, k):
    rng = np.random.default_rng(seed)
    key = rng.integers(-3, 3, size=(12, E)).astype(float)   # integer keys: many exact ties
    ids, margin = O.topk_order(key, k)
    for t in range(key.shape[0]):
        row = [int(v) for v in key[t]]
        best = max(itertools.combinations(range(E), k),
                   key=lambda sub: (sum(row[i] for i in sub), tuple(-i for i in sub)))
        want = sorted(best, key=lambda i: (-row[i], i))
        assert list(ids[t]) == want
        if k < E:
            rest = sorted((row[i] for i in range(E) if i not in best), reverse=True)
            assert margin[t] == min(row[i] for i in best) - rest[0]


def test_all_equal_logits_pick_lowest_indices():
    """W_g = 0: every affinity ties, so the tie rule alone decides."""
    x = np.ones((3, 4))
    r = O.route(x, np.zeros((4, 8)), 3)
    assert (r["ids"] == [0, 1, 2]).all()
    np.testing.assert_allclose(r["gates"], 1.0 / 8, rtol=0, atol=1e-15)
    r = O.route(x, np.zeros((4, 8)), 3, renormalize=True)
    np.testing.assert_allclose(r["gates"], 1.0 / 3, rtol=0, atol=1e-15)


# ---------------------------------------------------------------- gate values

def test_softmax_closed_form():
    p = np.array([1.0, 2.0, 3.0, 4.0]) / 10.0
    for shift in (0.0, 37.5, -800.0):
        np.testing.assert_allclose(O.softmax((np.log(p) + shift)[None])[0], p, rtol=1e-13)
    s = O.softmax(np.random.default_rng(0).standard_normal((50, 9)) * 4)
    assert (s >= 0).all()
    np.testing.assert_allclose(s.sum(1), 1.0, rtol=1e-14)


def test_softplus_and_silu_closed_forms():
    np.testing.assert_allclose(O.softplus(np.array([0.0])), [math.log(2.0)], rtol=1e-15)
    np.testing.assert_allclose(O.softplus(np.array([math.log(3.0)])), [math.log(4.0)], rtol=1e-15)
    np.testing.assert_allclose(O.softplus(np.array([-800.0, 800.0])), [0.0, 800.0], atol=1e-300)
    z = np.linspace(-6, 6, 25)
    np.testing.assert_allclose(O.silu(z) - O.silu(-z), z, atol=1e-14)
    np.testing.assert_allclose(O.silu(np.array([math.log(3.0)])), [0.75 * math.log(3.0)], rtol=1e-15)


def test_gates_sum_to_one():
    """Softmax gates are >= 0 and sum to 1 over all routed experts before top-k;
    after renormalisation they sum to 1 over the selected set."""
    x, W_g, *_ = tiny_layer(1, T=40, d=8, E=12)
    r = O.route(x, W_g, 4)
    np.testing.assert_allclose(r["s"].sum(1), 1.0, rtol=1e-14)
    assert (r["gates"] > 0).all() and (r["gates"].sum(1) < 1).all()
    rn = O.route(x, W_g, 4, renormalize=True)
    np.testing.assert_allclose(rn["gates"].sum(1), 1.0, rtol=1e-14)
    assert (rn["ids"] == r["ids"]).all()


def test_worked_example_closed_form():
    """Hand-derived layer with d = 2, I = 1, 4 routed + 1 shared expert.

    x = (1, 0); routed logits ln1..ln4 so s = (1,2,3,4)/10; top-2 = experts
    3, 2 with gates 0.4, 0.3 (renormalised: 4/7, 3/7). Expert e has W1 x = a_e,
    W3 x = 1 and W2 = (c_e, -c_e), so FFN_e(x) = c_e silu(a_e) (1, -1).
    """
    x = np.array([[1.0, 0.0]])
    W_g = np.array([[0.0, math.log(2), math.log(3), math.log(4)], [5.0, -1.0, 2.0, 7.0]])
    a = [math.log(3), 0.0, 1.0, -math.log(3), math.log(3)]   # shared, routed 0..3
    c = [1.0, 9.0, 9.0, 2.0, 0.5]
    W1 = np.array([[[ai, 3.0]] for ai in a])
    W3 = np.array([[[1.0, -4.0]] for _ in a])
    W2 = np.array([[[ci], [-ci]] for ci in c])
    r = O.route(x, W_g, 2)
    assert list(r["ids"][0]) == [3, 2]
    np.testing.assert_allclose(r["gates"][0], [0.4, 0.3], rtol=1e-14)
    y = O.moe_forward(x, W1, W3, W2, 1, r["ids"], r["gates"])[0]
    ln3 = math.log(3)
    want = 1.0 * 0.75 * ln3 + 0.4 * 0.5 * 0.75 * ln3 + 0.3 * 2.0 * (-ln3 * 0.25)
    np.testing.assert_allclose(y, [want, -want], rtol=1e-14)
    rn = O.route(x, W_g, 2, renormalize=True)
    yn = O.moe_forward(x, W1, W3, W2, 1, rn["ids"], rn["gates"])[0]
    want_n = 0.75 * ln3 + (4 / 7) * 0.5 * 0.75 * ln3 + (3 / 7) * 2.0 * (-ln3 * 0.25)
    np.testing.assert_allclose(yn, [want_n, -want_n], rtol=1e-14)


def test_noisy_gate_reductions():
    """Noisy top-k: with zero noise it is the renormalised softmax top-k; with
    x.W_noise = 0 the noise scale is softplus(0) = ln 2; with k = E it is the
    dense softmax of H."""
    x, W_g, *_ = tiny_layer(2, T=30, d=7, E=9)
    rng = np.random.default_rng(3)
    W_noise = rng.standard_normal((7, 9))
    eps0 = np.zeros((30, 9))
    rz = O.route(x, W_g, 3, noisy=True, W_noise=W_noise, eps=eps0)
    rr = O.route(x, W_g, 3, renormalize=True)
    assert (rz["ids"] == rr["ids"]).all()
    np.testing.assert_allclose(rz["gates"], rr["gates"], rtol=1e-13)
    eps = rng.standard_normal((30, 9))
    r0 = O.route(x, W_g, 9, noisy=True, W_noise=np.zeros((7, 9)), eps=eps)
    H = x @ W_g + eps * math.log(2.0)
    np.testing.assert_allclose(r0["H"], H, rtol=1e-13)
    dense = np.exp(H - H.max(1, keepdims=True))
    dense /= dense.sum(1, keepdims=True)
    np.testing.assert_allclose(O.dense_gates(r0["ids"], r0["gates"], 9), dense, rtol=1e-13)


def test_bias_steers_selection_not_gates():
    """Aux-loss-free bias: a large bias on an expert forces its selection,
    but its gate stays the plain softmax score."""
    x, W_g, *_ = tiny_layer(4, T=25, d=6, E=8)
    bias = np.zeros(8)
    bias[5] = 10.0
    r = O.route(x, W_g, 2, bias=bias)
    assert (r["ids"][:, 0] == 5).all()
    np.testing.assert_allclose(r["gates"][:, 0], r["s"][:, 5], rtol=1e-15)
    r0 = O.route(x, W_g, 2, bias=np.full(8, 0.3))   # a uniform bias changes nothing
    rp = O.route(x, W_g, 2)
    assert (r0["ids"] == rp["ids"]).all()
    np.testing.assert_allclose(r0["gates"], rp["gates"], rtol=1e-15)


def test_bias_key_is_score_plus_bias_hand_values():
    """The biased selection key is s_i + b_i, the softmax score plus the bias.
    The page on the auxiliary-loss-free strategy says only that a per-expert
    bias steers the assignment; adding it to the score (not the logit) is the
    reading taken, and this pins it. One token with logits (2, 0, -1) and
    b = (0, 0.9, 0):
    s = (e^2, 1, e^-1) / (e^2 + 1 + e^-1) = (0.8438, 0.1142, 0.0420), so
    s + b = (0.8438, 1.0142, 0.0420) ranks expert 1 first and expert 0 second,
    where logit + b = (2, 0.9, -1) would rank 0 first. Gates are s of the picks."""
    x = np.array([[1.0]])
    W_g = np.array([[2.0, 0.0, -1.0]])
    r = O.route(x, W_g, 2, bias=np.array([0.0, 0.9, 0.0]))
    z = math.exp(2.0) + 1.0 + math.exp(-1.0)
    assert r["ids"].tolist() == [[1, 0]]
    np.testing.assert_allclose(r["gates"], [[1.0 / z, math.exp(2.0) / z]], rtol=1e-14)
    np.testing.assert_allclose(r["margin"], [math.exp(2.0) / z - math.exp(-1.0) / z], rtol=1e-13)


# ---------------------------------------------------------------- layer output

@pytest.mark.parametrize("renorm", [False, True])
@pytest.mark.parametrize("K_s,E,k", [(0, 5, 2), (1, 5, 2), (2, 6, 3)])
def test_forward_matches_plain_loop_brute_force(renorm, K_s, E, k):
    x, W_g, W1, W3, W2 = tiny_layer(10 + K_s + E, T=6, d=5, E=E, K_s=K_s, I=3)
    r = O.route(x, W_g, k, renormalize=renorm)
    y = O.moe_forward(x, W1, W3, W2, K_s, r["ids"], r["gates"])
    y_bf, ids_bf = py_forward(x, W_g, W1, W3, W2, K_s, k, renorm)
    assert (r["ids"] == ids_bf).all()
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-14)


def test_sparse_equals_dense():
    """Skipping experts whose gate is zero changes nothing."""
    x, W_g, W1, W3, W2 = tiny_layer(5, T=40, d=8, E=10, K_s=2, I=4)
    r = O.route(x, W_g, 3)
    y = O.moe_forward(x, W1, W3, W2, 2, r["ids"], r["gates"])
    yd = O.moe_forward_dense(x, W1, W3, W2, 2, O.dense_gates(r["ids"], r["gates"], 10))
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-14)
    sub = np.array([3, 17, 0, 39])
    np.testing.assert_allclose(O.moe_forward(x, W1, W3, W2, 2, r["ids"], r["gates"], tokens=sub),
                               y[sub], rtol=1e-13, atol=1e-15)


def test_dense_gate_k_equals_E_is_softmax_mixture():
    """With K = E every expert is kept, so the layer is the dense softmax mixture."""
    x, W_g, W1, W3, W2 = tiny_layer(6, T=9, d=5, E=4, K_s=0, I=3)
    r = O.route(x, W_g, 4)
    y = O.moe_forward(x, W1, W3, W2, 0, r["ids"], r["gates"])
    yd = O.moe_forward_dense(x, W1, W3, W2, 0, r["s"])
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("m", [2, 4])
def test_fine_grained_segmentation_identity(m):
    """Splitting the intermediate dim into m segments, all active at gate 1,
    reproduces the unsplit FFN (section 3.1 of the DeepSeekMoE translation)."""
    rng = np.random.default_rng(7)
    T, d, I = 11, 6, 8
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((I, d))
    W3 = rng.standard_normal((I, d))
    W2 = rng.standard_normal((d, I))
    full = O.moe_forward(x, W1[None], W3[None], W2[None], 1,
                         np.zeros((T, 0), int), np.zeros((T, 0)))
    seg = I // m
    W1s = np.stack([W1[j * seg:(j + 1) * seg] for j in range(m)])
    W3s = np.stack([W3[j * seg:(j + 1) * seg] for j in range(m)])
    W2s = np.stack([W2[:, j * seg:(j + 1) * seg] for j in range(m)])
    split = O.moe_forward(x, W1s, W3s, W2s, m, np.zeros((T, 0), int), np.zeros((T, 0)))
    np.testing.assert_allclose(split, full, rtol=1e-12, atol=1e-13)


def test_relu_expert_closed_form():
    x = np.array([[1.0, -2.0]])
    wi = np.array([[1.0, 1.0], [2.0, 0.5]])     # wi x = (-1, 1) -> ReLU (0, 1)
    wo = np.array([[3.0, 4.0], [5.0, 6.0]])
    np.testing.assert_allclose(O.expert_ffn_relu(x, wi, wo), [[4.0, 6.0]])


# ---------------------------------------------------------------- dispatch / combine

@pytest.mark.parametrize("seed", range(4))
def test_dispatch_brute_force(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 37, 7, 3
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    dsp = O.dispatch(ids, E)
    want_rows = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    want_rows.append(t * k + j)
    assert list(dsp["perm_src"]) == want_rows
    for e in range(E):
        assert dsp["counts"][e] == sum(1 for v in ids.flat if v == e)
        assert dsp["offsets"][e + 1] - dsp["offsets"][e] == dsp["counts"][e]
    for t in range(T):
        for j in range(k):
            assert want_rows[dsp["dest"][t, j]] == t * k + j


def test_expert_rows_and_combine_equal_forward():
    x, W_g, W1, W3, W2 = tiny_layer(8, T=20, d=6, E=7, K_s=2, I=3)
    r = O.route(x, W_g, 3)
    dsp = O.dispatch(r["ids"], 7)
    rows = O.expert_rows(x, W1, W3, W2, 2, dsp["perm_src"], dsp["offsets"], 3)
    for t in (0, 13):   # one row by plain loops
        for i in range(2):
            np.testing.assert_allclose(rows[i * 20 + t],
                                       py_ffn(x[t].tolist(), W1[i].tolist(), W3[i].tolist(), W2[i].tolist()),
                                       rtol=1e-12)
    y = O.combine(rows, dsp["dest"], r["gates"], 2, 20)
    np.testing.assert_allclose(y, O.moe_forward(x, W1, W3, W2, 2, r["ids"], r["gates"]),
                               rtol=1e-12, atol=1e-14)


def test_combine_plain_loop():
    rng = np.random.default_rng(9)
    T, k, K_s, d = 6, 2, 1, 3
    rows = rng.standard_normal((K_s * T + T * k, d))
    dest = rng.permutation(T * k).reshape(T, k)
    g = rng.random((T, k))
    y = O.combine(rows, dest, g, K_s, T)
    for t in range(T):
        want = [rows[t][c] + sum(g[t, j] * rows[K_s * T + dest[t, j]][c] for j in range(k))
                for c in range(d)]
        np.testing.assert_allclose(y[t], want, rtol=1e-14)


# ---------------------------------------------------------------- expert capacity (GShard / Switch)

def py_capacity_keep(ids, capacity):
    """An assignment is accepted iff fewer than `capacity` earlier assignments
    (ascending t*k + j) chose the same expert -- the running counter c_e of
    the GShard passage, counted afresh for every assignment."""
    T, k = len(ids), len(ids[0])
    flat = [int(v) for row in ids for v in row]
    keep = []
    for a, e in enumerate(flat):
        earlier = sum(1 for b in range(a) if flat[b] == e)
        keep.append(earlier < capacity)
    return np.array(keep).reshape(T, k)


@pytest.mark.parametrize("seed,capacity", [(0, 1), (1, 3), (2, 5), (3, 9)])
def test_capacity_keep_matches_counting(seed, capacity):
    rng = np.random.default_rng(seed)
    T, E, k = 23, 5, 2
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    ids[:9, 0] = 0   # a hot expert that overflows
    np.testing.assert_array_equal(O.capacity_keep(ids, E, capacity), py_capacity_keep(ids.tolist(), capacity))


def test_capacity_hot_expert_keeps_first_tokens():
    T, E, C = 12, 4, 5
    ids = np.zeros((T, 1), dtype=int)            # every token picks expert 0
    keep = O.capacity_keep(ids, E, C)
    assert keep[:C, 0].all() and not keep[C:, 0].any()
    dsp = O.dispatch(ids, E, capacity=C)
    assert list(dsp["counts"]) == [C, 0, 0, 0]
    assert list(dsp["perm_src"]) == list(range(C))
    assert list(dsp["dest"][:, 0]) == list(range(C)) + [-1] * (T - C)


def test_capacity_at_or_above_max_count_is_dropless():
    rng = np.random.default_rng(4)
    T, E, k = 40, 6, 3
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    cmax = int(np.bincount(ids.reshape(-1)).max())
    a, b = O.dispatch(ids, E), O.dispatch(ids, E, capacity=cmax)
    for key in ("counts", "offsets", "perm_src", "dest"):
        np.testing.assert_array_equal(a[key], b[key])
    assert (O.dispatch(ids, E, capacity=cmax - 1)["counts"] == np.minimum(np.bincount(ids.reshape(-1)), cmax - 1)).all()


def test_capacity_forward_drops_only_refused_assignments():
    """y with a capacity = shared experts + the accepted routed terms, by loops;
    a token all of whose picks were refused gets the shared experts alone."""
    x, W_g, W1, W3, W2 = tiny_layer(11, T=9, d=4, E=4, K_s=1, I=2)
    ids = np.array([[0, 1]] * 6 + [[2, 3], [0, 1], [1, 2]])
    g = np.full(ids.shape, 0.5)
    keep = O.capacity_keep(ids, 4, 5)            # expert 0 and 1 take tokens 0..4 only
    y = O.moe_forward(x, W1, W3, W2, 1, ids, g, keep=keep)
    for t in range(9):
        want = py_ffn(x[t].tolist(), W1[0].tolist(), W3[0].tolist(), W2[0].tolist())
        for j in range(2):
            if keep[t, j]:
                e = 1 + ids[t, j]
                o = py_ffn(x[t].tolist(), W1[e].tolist(), W3[e].tolist(), W2[e].tolist())
                want = [a + 0.5 * b for a, b in zip(want, o)]
        np.testing.assert_allclose(y[t], want, rtol=1e-12, atol=1e-14)
    assert not keep[5].any() and not keep[7].any()
    # the grouped path (dispatch -> expert_rows -> combine) gives the same y
    dsp = O.dispatch(ids, 4, capacity=5)
    rows = O.expert_rows(x, W1, W3, W2, 1, dsp["perm_src"], dsp["offsets"], 2)
    np.testing.assert_allclose(O.combine(rows, dsp["dest"], g, 1, 9), y, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- GShard ReLU experts

def test_relu_layer_matches_plain_loops():
    """wo . ReLU(wi . x) experts ([MoE-notes] section 3) through the whole layer."""
    x, W_g, W1, W3, W2 = tiny_layer(12, T=6, d=5, E=5, K_s=1, I=3)
    r = O.route(x, W_g, 2)
    y = O.moe_forward(x, W1, None, W2, 1, r["ids"], r["gates"], act="relu")
    for t in range(6):
        def relu_ffn(e):
            h = [max(0.0, sum(W1[e][i][c] * x[t][c] for c in range(5))) for i in range(3)]
            return [sum(W2[e][o][i] * h[i] for i in range(3)) for o in range(5)]
        want = relu_ffn(0)
        for gj, e in zip(r["gates"][t], r["ids"][t]):
            want = [a + gj * b for a, b in zip(want, relu_ffn(1 + e))]
        np.testing.assert_allclose(y[t], want, rtol=1e-12, atol=1e-14)
    dsp = O.dispatch(r["ids"], 5)
    rows = O.expert_rows(x, W1, None, W2, 1, dsp["perm_src"], dsp["offsets"], 2, act="relu")
    np.testing.assert_allclose(O.combine(rows, dsp["dest"], r["gates"], 1, 6), y, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- statistics

def test_logsumexp_and_probability_sums_closed_forms():
    z = np.full((3, 8), 1.5)
    np.testing.assert_allclose(O.logsumexp(z), 1.5 + math.log(8), rtol=1e-15)
    np.testing.assert_allclose(O.prob_column_sums(z), np.full(8, 3 / 8), rtol=1e-15)
    z = np.array([[0.0, math.log(3.0)], [math.log(2.0), math.log(2.0)]])
    np.testing.assert_allclose(O.logsumexp(z), [math.log(4.0), math.log(4.0)], rtol=1e-15)
    np.testing.assert_allclose(O.prob_column_sums(z), [0.25 + 0.5, 0.75 + 0.5], rtol=1e-15)
    rng = np.random.default_rng(3)
    z = rng.standard_normal((50, 7)) * 3
    assert O.prob_column_sums(z).sum() == pytest.approx(50.0, rel=1e-13)   # each row of s sums to 1
    assert np.mean(O.logsumexp(z) ** 2) == pytest.approx(O.router_z_loss(z), rel=1e-13)


def test_cv_squared_hand_values():
    assert O.cv_squared([1, 1, 1, 1]) == 0.0
    assert O.cv_squared([4, 0, 0, 0]) == pytest.approx(3.0, rel=1e-15)
    assert O.cv_squared([2, 0]) == pytest.approx(1.0, rel=1e-15)
    G = np.array([[0.5, 0.5, 0.0], [0.0, 0.5, 0.5]])
    np.testing.assert_allclose(O.importance(G), [0.5, 1.0, 0.5])
    assert O.cv_squared(O.importance(G)) == pytest.approx(0.125, rel=1e-14)


def test_balance_losses_uniform_routing():
    """Uniform routing: f_i = 1 under eq (13)'s normalisation, so
    L_ExpBal = alpha1 * sum_i P_i = alpha1; the Switch loss is alpha;
    the device loss with equal groups is alpha2."""
    T, N, k = 8, 4, 2
    ids = np.array([[t % N, (t + 1) % N] for t in range(T)])
    s = np.full((T, N), 1.0 / N)
    assert O.expert_balance_loss(ids, s, N, k, 0.01) == pytest.approx(0.01, rel=1e-14)
    assert O.device_balance_loss(ids, s, N, k, [[0, 1], [2, 3]], 0.05) == pytest.approx(0.05, rel=1e-14)
    p = np.eye(N)[np.arange(T) % N] * 0.7 + 0.3 / N
    assert O.switch_balance_loss(p, 0.01) == pytest.approx(0.01, rel=1e-14)
    # collapse onto one expert: f = (4, 0, 0, 0) * N/(kT) ... with P = (1,0,0,0)
    ids_c = np.array([[0, 1]] * T)
    s_c = np.tile([1.0, 0.0, 0.0, 0.0], (T, 1))
    assert O.expert_balance_loss(ids_c, s_c, N, k, 1.0) == pytest.approx(N / k, rel=1e-14)


def test_router_z_loss_closed_form():
    assert O.router_z_loss(np.zeros((5, 8))) == pytest.approx(math.log(8) ** 2, rel=1e-14)
    z = np.array([[math.log(1), math.log(2), math.log(5)]])    # logsumexp = ln 8
    assert O.router_z_loss(z) == pytest.approx(math.log(8) ** 2, rel=1e-14)


def test_combinatorics_golden():
    with open(os.path.join(GOLDEN, "combinatorics.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        assert math.comb(c["n"], c["k"]) == c["combinations"]
