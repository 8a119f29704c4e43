"""Pins of the backward oracle (oracle/moe_backward.py), on the CPU.

The backward is the derivative of the forward oracle, which is itself pinned
to the pages (test_oracle_pins.py). Each case compares every gradient with
central finite differences of <dy, y(theta)> computed through the forward
oracle alone, at inputs whose routing margins keep the selection fixed under
the perturbation (checked). Structural pins: linearity in dy, token
independence, the k = E reduction (renormalising over all experts changes
nothing), and the fine-grained segmentation identity ([DSMoE] section 3.1:
an expert split into m segments, all at gate 1, is the unsplit expert).
Planted mistakes in each helper must fail at least one pin.
"""

import numpy as np
import pytest

from oracle import moe_backward as B
from oracle import moe_oracle as O

H_STEP = 1e-6


def layer(seed, T=5, d=4, E=5, K_s=1, I=3, scale=0.6, noisy=False):
    rng = np.random.default_rng(seed)
    G = E + K_s
    p = {"x": rng.normal(size=(T, d)), "W_g": rng.normal(size=(d, E)),
         "W1": scale * rng.normal(size=(G, I, d)), "W3": scale * rng.normal(size=(G, I, d)),
         "W2": scale * rng.normal(size=(G, d, I))}
    if noisy:
        p["W_noise"] = 0.5 * rng.normal(size=(d, E))
        p["eps"] = rng.normal(size=(T, E))
    return p, rng.normal(size=(T, d))


def forward(p, K_s, k, opts):
    """y, and the routing it took, through the forward oracle only."""
    r = O.route(p["x"], p["W_g"], k, renormalize=opts.get("renormalize", False), noisy=opts.get("noisy", False),
                W_noise=p.get("W_noise"), eps=p.get("eps"), bias=opts.get("bias"))
    E = p["W1"].shape[0] - K_s
    cap = opts.get("capacity", 0)
    keep = O.capacity_keep(r["ids"], E, cap) if cap else None
    act = opts.get("act", "swiglu")
    y = O.moe_forward(p["x"], p["W1"], None if act == "relu" else p["W3"], p["W2"], K_s, r["ids"], r["gates"],
                      act=act, keep=keep)
    return y, r, keep


def numeric_grads(p, dy, K_s, k, opts, names):
    _, r0, keep0 = forward(p, K_s, k, opts)
    out = {}
    for name in names:
        g = np.zeros_like(p[name])
        it = np.nditer(p[name], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            vals = []
            for sgn in (1.0, -1.0):
                q = {kk: (v.copy() if kk == name else v) for kk, v in p.items()}
                q[name][idx] += sgn * H_STEP
                y, r, keep = forward(q, K_s, k, opts)
                assert (r["ids"] == r0["ids"]).all(), "routing moved under the perturbation"
                if keep0 is not None:
                    assert (keep == keep0).all()
                vals.append((dy * y).sum())
            g[idx] = (vals[0] - vals[1]) / (2 * H_STEP)
        out[name] = g
    return out


def analytic(p, dy, K_s, k, opts):
    act = opts.get("act", "swiglu")
    return B.moe_backward(p["x"], p["W_g"], p["W1"], None if act == "relu" else p["W3"], p["W2"], K_s, k, dy,
                          renormalize=opts.get("renormalize", False), noisy=opts.get("noisy", False),
                          W_noise=p.get("W_noise"), eps=p.get("eps"), bias=opts.get("bias"),
                          capacity=opts.get("capacity", 0), act=act)


GRAD_OF = {"x": "dx", "W_g": "dW_g", "W_noise": "dW_noise", "W1": "dW1", "W3": "dW3", "W2": "dW2"}

CASES = {
    "softmax": (dict(seed=1, K_s=1), 2, {}),
    "renormalised": (dict(seed=2, K_s=2), 2, {"renormalize": True}),
    "bias": (dict(seed=3, K_s=1), 2, {"bias": np.array([0.0, 0.3, 0.0, 0.2, 0.0])}),
    "noisy": (dict(seed=4, K_s=0, noisy=True), 2, {"noisy": True, "renormalize": True}),
    "capacity": (dict(seed=5, T=8, E=4, K_s=1), 2, {"capacity": 3}),
    "relu": (dict(seed=6, K_s=1), 2, {"act": "relu"}),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_gradients_match_finite_differences(case):
    kw, k, opts = CASES[case]
    p, dy = layer(**kw)
    K_s = kw.get("K_s", 1)
    _, r, keep = forward(p, K_s, k, opts)
    assert r["margin"].min() > 1e-3            # the selection is well inside its region
    if case == "capacity":
        assert not keep.all()                  # some assignments dropped
    if case == "relu":                         # no pre-activation at the ReLU kink
        for e in range(p["W1"].shape[0]):
            assert np.abs(p["x"] @ p["W1"][e].T).min() > 1e-3
    names = [n for n in ("x", "W_g", "W_noise", "W1", "W3", "W2") if n in p]
    if opts.get("act") == "relu":
        names.remove("W3")
    num = numeric_grads(p, dy, K_s, k, opts, names)
    got = analytic(p, dy, K_s, k, opts)
    for n in names:
        np.testing.assert_allclose(got[GRAD_OF[n]], num[n], rtol=1e-6, atol=1e-8, err_msg=f"{case} d{n}")
    if opts.get("act") == "relu":
        assert got["dW3"] is None


def test_linear_in_dy():
    p, dy = layer(7, K_s=2)
    a = analytic(p, dy, 2, 2, {"renormalize": True})
    b = analytic(p, -2.5 * dy, 2, 2, {"renormalize": True})
    for n in ("dx", "dW_g", "dW1", "dW3", "dW2"):
        np.testing.assert_allclose(b[n], -2.5 * a[n], rtol=1e-12, atol=1e-14)


def test_tokens_are_independent():
    """An upstream gradient on one token moves only that token's dx, and the
    parameter gradients equal those of that token alone."""
    p, dy = layer(8, T=6, K_s=1)
    t = 3
    one = np.zeros_like(dy)
    one[t] = dy[t]
    g = analytic(p, one, 1, 2, {})
    assert np.abs(np.delete(g["dx"], t, axis=0)).max() == 0.0
    q = dict(p, x=p["x"][t:t + 1])
    g1 = analytic(q, dy[t:t + 1], 1, 2, {})
    for n in ("dW_g", "dW1", "dW3", "dW2"):
        np.testing.assert_allclose(g[n], g1[n], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(g["dx"][t], g1["dx"][0], rtol=1e-12, atol=1e-15)


def test_k_equals_E_renormalisation_changes_nothing():
    """With k = E the selected scores sum to 1, so renormalising is the
    identity on the forward and must be on every gradient too."""
    p, dy = layer(9, E=4, K_s=1)
    a = analytic(p, dy, 1, 4, {})
    b = analytic(p, dy, 1, 4, {"renormalize": True})
    for n in ("dx", "dW_g", "dW1", "dW3", "dW2"):
        np.testing.assert_allclose(b[n], a[n], rtol=1e-10, atol=1e-13)


@pytest.mark.parametrize("m", [2, 3])
def test_segmentation_identity_for_gradients(m):
    """[DSMoE] section 3.1: a shared expert of width I split into m segments of
    width I/m, all always active, gives the same layer; so each segment's
    weight gradients are the matching slices of the unsplit expert's."""
    I = 6
    p, dy = layer(10, K_s=1, I=I)
    seg = I // m
    # only the shared expert is split; the routed experts (width I/m) are the
    # same in both layers, zero-padded to width I in the unsplit one
    rng = np.random.default_rng(11)
    E = p["W1"].shape[0] - 1
    r1 = 0.6 * rng.normal(size=(E, seg, p["x"].shape[1]))
    r3 = 0.6 * rng.normal(size=(E, seg, p["x"].shape[1]))
    r2 = 0.6 * rng.normal(size=(E, p["x"].shape[1], seg))
    split = {"x": p["x"], "W_g": p["W_g"],
             "W1": np.concatenate([p["W1"][0, j * seg:(j + 1) * seg][None] for j in range(m)] + [r1], axis=0),
             "W3": np.concatenate([p["W3"][0, j * seg:(j + 1) * seg][None] for j in range(m)] + [r3], axis=0),
             "W2": np.concatenate([p["W2"][0, :, j * seg:(j + 1) * seg][None] for j in range(m)] + [r2], axis=0)}
    # the unsplit layer: routed experts padded with zero rows up to width I
    pad = np.zeros((E, I - seg, p["x"].shape[1]))
    whole = {"x": p["x"], "W_g": p["W_g"],
             "W1": np.concatenate([p["W1"][:1], np.concatenate([r1, pad], axis=1)], axis=0),
             "W3": np.concatenate([p["W3"][:1], np.concatenate([r3, pad], axis=1)], axis=0),
             "W2": np.concatenate([p["W2"][:1], np.concatenate([r2, pad.transpose(0, 2, 1)], axis=2)], axis=0)}
    ys = forward(split, m, 2, {})[0]
    yw = forward(whole, 1, 2, {})[0]
    np.testing.assert_allclose(ys, yw, rtol=1e-12, atol=1e-14)
    gs = analytic(split, dy, m, 2, {})
    gw = analytic(whole, dy, 1, 2, {})
    np.testing.assert_allclose(gs["dx"], gw["dx"], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(gs["dW_g"], gw["dW_g"], rtol=1e-11, atol=1e-14)
    for j in range(m):
        np.testing.assert_allclose(gs["dW1"][j], gw["dW1"][0, j * seg:(j + 1) * seg], rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(gs["dW3"][j], gw["dW3"][0, j * seg:(j + 1) * seg], rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(gs["dW2"][j], gw["dW2"][0, :, j * seg:(j + 1) * seg], rtol=1e-11, atol=1e-14)


# ---------------------------------------------------------------- planted mistakes

def _silu_grad_no_product_term(a):
    return B.sigmoid(a)


def _softplus_grad_as_softplus(z):
    return O.softplus(z)


def _softmax_backward_no_projection(p, dp):
    return np.asarray(p) * np.asarray(dp)


def _renorm_without_sum_term(dg, gates, s_sel, renormalize):
    if not renormalize:
        return dg
    return dg / np.asarray(s_sel).sum(axis=1, keepdims=True)


_expert_backward = B.expert_backward


def _expert_backward_w2_reinterpreted(X, W1, W3, W2, dO, act="swiglu"):
    dX, dW1, dW3, dW2 = _expert_backward(X, W1, W3, W2, dO, act)
    return dX, dW1, dW3, dW2.T.reshape(dW2.shape)


def _expert_backward_gate_up_swapped(X, W1, W3, W2, dO, act="swiglu"):
    if act == "relu":
        return _expert_backward(X, W1, W3, W2, dO, act)
    dX, dW1, dW3, dW2 = _expert_backward(X, W1, W3, W2, dO, act)
    return dX, dW3, dW1, dW2


BACKWARD_MUTANTS = {
    "silu_grad_no_product_term": ("silu_grad", _silu_grad_no_product_term),
    "softplus_grad_as_softplus": ("softplus_grad", _softplus_grad_as_softplus),
    "softmax_backward_no_projection": ("softmax_backward", _softmax_backward_no_projection),
    "renorm_without_sum_term": ("gates_backward_to_scores", _renorm_without_sum_term),
    "dW2_reinterpreted": ("expert_backward", _expert_backward_w2_reinterpreted),
    "dW1_dW3_swapped": ("expert_backward", _expert_backward_gate_up_swapped),
}


def _pins_failing() -> int:
    failed = 0
    for case in sorted(CASES):
        try:
            test_gradients_match_finite_differences(case)
        except AssertionError:
            failed += 1
    for pin in (test_k_equals_E_renormalisation_changes_nothing,
                lambda: test_segmentation_identity_for_gradients(2)):
        try:
            pin()
        except AssertionError:
            failed += 1
    return failed


@pytest.mark.parametrize("name", sorted(BACKWARD_MUTANTS))
def test_backward_mutant_is_caught(name, monkeypatch):
    attr, fn = BACKWARD_MUTANTS[name]
    monkeypatch.setattr(B, attr, fn)
    assert _pins_failing() > 0, f"planted mistake {name} went unnoticed"
