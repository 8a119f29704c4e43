"""Planted mistakes in the oracle (on the CPU) must be caught by the pins.

Each mutant replaces one oracle function with a plausible wrong version
(a dropped term, a wrong sign or index, a swapped operand) and runs the pins
that should notice; at least one of them must fail.
"""

import numpy as np
import pytest

from oracle import moe_oracle as O
from tests import test_oracle_pins as P

_orig = {name: getattr(O, name) for name in
         ("silu", "topk_order", "softmax", "expert_ffn", "moe_forward", "route",
          "dispatch", "combine", "softplus", "cv_squared", "expert_balance_loss",
          "capacity_keep", "expert_ffn_relu", "logsumexp")}


def _silu_relu(z):
    z = np.asarray(z, dtype=float)
    return np.maximum(z, 0.0)


def _topk_high_index_ties(key, k):
    key = np.asarray(key, dtype=float)
    order = np.argsort(key, axis=1, kind="stable")[:, ::-1]   # ties -> highest index
    ids = order[:, :k]
    kth = np.take_along_axis(key, order[:, k - 1:k], axis=1)[:, 0]
    nxt = (np.take_along_axis(key, order[:, k:k + 1], axis=1)[:, 0]
           if k < key.shape[1] else np.full(key.shape[0], -np.inf))
    return ids, kth - nxt


def _topk_ascending_within_k(key, k):
    ids, margin = _orig["topk_order"](key, k)
    return ids[:, ::-1].copy(), margin          # the right set, listed by ascending key


def _topk_margin_negated(key, k):
    ids, margin = _orig["topk_order"](key, k)
    return ids, -margin                          # (k+1)-th minus k-th


def _softmax_wrong_axis(z):
    z = np.asarray(z, dtype=float)
    e = np.exp(z - z.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def _ffn_swapped(X, W1, W3, W2):
    return _orig["expert_ffn"](X, W3, W1, W2)


def _ffn_w2_transposed(X, W1, W3, W2):
    X = np.asarray(X, float)
    h = _orig["silu"](X @ np.asarray(W1, float).T) * (X @ np.asarray(W3, float).T)
    W2 = np.asarray(W2, float)
    return h @ W2.reshape(W2.shape[1], W2.shape[0])     # reinterpreted, not transposed


def _forward_no_shared(x, W1, W3, W2, n_shared, ids, gates, tokens=None, **kw):
    if kw.get("act", "swiglu") != "swiglu":
        return _orig["moe_forward"](x, W1, W3, W2, n_shared, ids, gates, tokens, **kw)
    y = _orig["moe_forward"](x, W1, W3, W2, n_shared, ids, gates, tokens, **kw)
    xs = np.asarray(x, float) if tokens is None else np.asarray(x, float)[tokens]
    for i in range(n_shared):
        y = y - _orig["expert_ffn"](xs, W1[i], W3[i], W2[i])
    return y


def _route_no_renorm(x, W_g, top_k, **kw):
    if not kw.get("noisy"):
        kw["renormalize"] = False
    return _orig["route"](x, W_g, top_k, **kw)


def _route_bias_in_gate(x, W_g, top_k, **kw):
    r = _orig["route"](x, W_g, top_k, **kw)
    if kw.get("bias") is not None:
        r["gates"] = r["gates"] + np.asarray(kw["bias"])[r["ids"]]
    return r


def _route_bias_on_logits(x, W_g, top_k, **kw):
    # selection key logit + b instead of the score s + b
    r = _orig["route"](x, W_g, top_k, **kw)
    bias = kw.get("bias")
    if bias is None:
        return r
    key = r["logits"] + np.asarray(bias, float)[None, :]
    ids, margin = O.topk_order(key, top_k)
    gates = np.take_along_axis(r["s"], ids, axis=1)
    if kw.get("renormalize"):
        gates = gates / gates.sum(axis=1, keepdims=True)
    r.update(ids=ids, gates=gates, key=key, margin=margin)
    return r


def _dispatch_descending(ids, n_experts, capacity=0):
    d = _orig["dispatch"](ids, n_experts, capacity)
    if capacity:
        return d
    flat = np.asarray(ids).reshape(-1)
    order = np.lexsort((-np.arange(flat.size), flat))     # within expert: descending index
    dest = np.empty_like(order)
    dest[order] = np.arange(flat.size)
    d.update(perm_src=order, dest=dest.reshape(np.asarray(ids).shape))
    return d


def _combine_flipped_gates(rows, dest, gates, n_shared, T):
    return _orig["combine"](rows, dest, np.asarray(gates)[:, ::-1], n_shared, T)


def _softplus_exp(z):
    return np.exp(np.asarray(z, dtype=float))


def _cv_sample(v):
    v = np.asarray(v, float)
    return float(v.var(ddof=1) / v.mean() ** 2)


def _expbal_no_norm(ids, s, n_routed, top_k, alpha1):
    return _orig["expert_balance_loss"](ids, s, n_routed, top_k, alpha1) * top_k


def _capacity_keeps_latest(ids, n_experts, capacity):
    # counts from the last token backwards: keeps the latest arrivals instead
    ids = np.asarray(ids)
    return _orig["capacity_keep"](ids[::-1, ::-1], n_experts, capacity)[::-1, ::-1]


def _relu_without_max(X, wi, wo):
    return (np.asarray(X, float) @ np.asarray(wi, float).T) @ np.asarray(wo, float).T


def _logsumexp_no_max(logits):
    z = np.asarray(logits, float)
    m = z.max(axis=1, keepdims=True)
    return np.log(np.exp(z - m).sum(axis=1))      # the max term dropped


def _run_pins():
    pins = [
        lambda: P.test_softplus_and_silu_closed_forms(),
        lambda: P.test_softmax_closed_form(),
        lambda: P.test_all_equal_logits_pick_lowest_indices(),
        lambda: [P.test_topk_matches_subset_brute_force(s, 6, 3) for s in range(3)],
        lambda: P.test_gates_sum_to_one(),
        lambda: P.test_worked_example_closed_form(),
        lambda: P.test_noisy_gate_reductions(),
        lambda: P.test_bias_steers_selection_not_gates(),
        lambda: P.test_bias_key_is_score_plus_bias_hand_values(),
        lambda: P.test_forward_matches_plain_loop_brute_force(False, 1, 5, 2),
        lambda: P.test_forward_matches_plain_loop_brute_force(True, 2, 6, 3),
        lambda: P.test_sparse_equals_dense(),
        lambda: [P.test_dispatch_brute_force(s) for s in range(2)],
        lambda: P.test_expert_rows_and_combine_equal_forward(),
        lambda: P.test_combine_plain_loop(),
        lambda: P.test_cv_squared_hand_values(),
        lambda: P.test_balance_losses_uniform_routing(),
        lambda: P.test_capacity_keep_matches_counting(0, 1),
        lambda: P.test_capacity_hot_expert_keeps_first_tokens(),
        lambda: P.test_capacity_forward_drops_only_refused_assignments(),
        lambda: P.test_relu_expert_closed_form(),
        lambda: P.test_relu_layer_matches_plain_loops(),
        lambda: P.test_logsumexp_and_probability_sums_closed_forms(),
    ]
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    return failed


MUTANTS = {
    "silu_as_relu": ("silu", _silu_relu),
    "topk_ties_high_index": ("topk_order", _topk_high_index_ties),
    "topk_ascending_within_k": ("topk_order", _topk_ascending_within_k),
    "topk_margin_negated": ("topk_order", _topk_margin_negated),
    "softmax_wrong_axis": ("softmax", _softmax_wrong_axis),
    "ffn_gate_up_swapped": ("expert_ffn", _ffn_swapped),
    "ffn_w2_reinterpreted": ("expert_ffn", _ffn_w2_transposed),
    "forward_drops_shared": ("moe_forward", _forward_no_shared),
    "route_ignores_renorm": ("route", _route_no_renorm),
    "route_bias_in_gate": ("route", _route_bias_in_gate),
    "route_bias_on_logits": ("route", _route_bias_on_logits),
    "dispatch_unstable": ("dispatch", _dispatch_descending),
    "combine_gates_flipped": ("combine", _combine_flipped_gates),
    "softplus_as_exp": ("softplus", _softplus_exp),
    "cv_sample_variance": ("cv_squared", _cv_sample),
    "expbal_missing_k": ("expert_balance_loss", _expbal_no_norm),
    "capacity_keeps_latest": ("capacity_keep", _capacity_keeps_latest),
    "relu_without_max": ("expert_ffn_relu", _relu_without_max),
    "logsumexp_drops_max": ("logsumexp", _logsumexp_no_max),
}


def test_unmutated_oracle_passes_pins():
    assert _run_pins() == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    assert _run_pins() > 0, f"mutant {name} passed every pin"
