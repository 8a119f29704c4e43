"""Seeded synthetic inputs for a layer workload (no arithmetic of the method).

Recipe (the same for the CUDA path, its tests and the oracle):
  * one torch CPU generator seeded with the workload's seed;
  * x ~ N(0, 1), drawn in fp32 and stored as bf16 (fp32 for fp32 workloads);
  * W_g ~ N(0, 0.02^2) fp32 [d, N_r]; W_noise likewise for the noisy gate;
  * expert weights ~ N(0, 0.02^2): W1, W3 [K_s+N_r, I, d], W2 [K_s+N_r, d, I],
    stored bf16 (fp32 for fp32 workloads), shared experts first (ReLU
    experts have no W3: that draw is skipped);
  * noisy gate: eps ~ N(0, 1) fp32 [T, N_r], the StandardNormal() draws;
  * selection bias: b_i = 0.05 * r_i^(-1.1), r a seeded permutation of
    1..N_r (a Zipf(1.1) skew over the experts).
Draw order is fixed: x, W_g, W_noise, eps, bias, W1, W3, W2.

Everything is returned as CPU torch tensors; callers move them to a device.
"""

from __future__ import annotations

import torch

from .workloads import Workload

WEIGHT_STD = 0.02
BIAS_SCALE = 0.05
BIAS_ZIPF_S = 1.1


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def make_inputs(w: Workload, *, with_experts: bool = True) -> dict:
    """All inputs of one forward of workload `w` (CPU tensors)."""
    g = _gen(w.seed)
    act = torch.float32 if w.fp32 else torch.bfloat16
    out = {}
    out["x"] = torch.randn(w.T, w.d, generator=g).to(act)
    out["W_g"] = torch.randn(w.d, w.n_routed, generator=g) * WEIGHT_STD
    out["W_noise"] = None
    out["eps"] = None
    out["bias"] = None
    if w.noisy:
        out["W_noise"] = torch.randn(w.d, w.n_routed, generator=g) * WEIGHT_STD
        out["eps"] = torch.randn(w.T, w.n_routed, generator=g)
    if w.bias:
        r = torch.randperm(w.n_routed, generator=g).to(torch.float64) + 1.0
        out["bias"] = (BIAS_SCALE * r.pow(-BIAS_ZIPF_S)).to(torch.float32)
    if with_experts:
        E, I, d = w.n_experts, w.d_ff, w.d
        out["W1"] = _randn_chunked((E, I, d), g, act)
        out["W3"] = _randn_chunked((E, I, d), g, act) if w.act != "relu" else None
        out["W2"] = _randn_chunked((E, d, I), g, act)
    return out


def make_tokens(w: Workload, replica: int) -> dict:
    """The token-side inputs (x, and eps for the noisy gate) of another batch
    of the same layer: replica r > 0 of a data-parallel run draws its own
    batch from generator seed + 1000 r (replica 0 uses make_inputs' x)."""
    g = _gen(w.seed + 1000 * replica)
    act = torch.float32 if w.fp32 else torch.bfloat16
    out = {"x": torch.randn(w.T, w.d, generator=g).to(act), "eps": None}
    if w.noisy:
        out["eps"] = torch.randn(w.T, w.n_routed, generator=g)
    return out


def _randn_chunked(shape, g, dtype) -> torch.Tensor:
    """N(0, WEIGHT_STD^2) drawn expert by expert (bounded fp32 temporaries)."""
    out = torch.empty(shape, dtype=dtype)
    for e in range(shape[0]):
        out[e] = (torch.randn(shape[1:], generator=g) * WEIGHT_STD).to(dtype)
    return out


def make_upstream_grad(w: Workload, seed: int) -> torch.Tensor:
    """dy ~ N(0, 1) [T, d] for a backward pass, stored like x (bf16, or fp32
    for fp32 workloads), from its own generator."""
    act = torch.float32 if w.fp32 else torch.bfloat16
    return torch.randn(w.T, w.d, generator=_gen(seed)).to(act)


def random_topk_ids(T: int, n_routed: int, top_k: int, seed: int,
                    skew: str = "uniform") -> torch.Tensor:
    """Valid routing decisions for dispatch tests: k distinct experts per token.

    skew = "uniform": a random k-subset per token, in random order.
    skew = "hot":     expert 0 is picked by every token; experts n_routed-1
                      and n_routed-2 are never picked (empty groups).
    """
    g = _gen(seed)
    if skew == "uniform":
        return torch.rand(T, n_routed, generator=g).argsort(dim=1)[:, :top_k].to(torch.int32)
    if skew == "hot":
        assert n_routed - 2 > top_k
        rest = torch.rand(T, n_routed - 3, generator=g).argsort(dim=1)[:, :top_k - 1] + 1
        ids = torch.cat([torch.zeros(T, 1, dtype=rest.dtype), rest], dim=1)
        perm = torch.rand(T, top_k, generator=g).argsort(dim=1)
        return torch.gather(ids, 1, perm).to(torch.int32)
    raise ValueError(skew)


def random_rows(n: int, d: int, seed: int) -> torch.Tensor:
    """fp32 N(0,1) rows (stand-in per-row expert outputs for combine tests)."""
    return torch.randn(n, d, generator=_gen(seed))


def random_gates(T: int, top_k: int, seed: int) -> torch.Tensor:
    """fp32 U(0,1) gate values for combine tests."""
    return torch.rand(T, top_k, generator=_gen(seed))
