"""CUDA path vs the CPU oracle, through the C ABI (needs a B300).

Criteria:
  * routing ids bit-exact on every token whose oracle key margin (k-th minus
    (k+1)-th of the sorted key) is >= 1e-5; on the other tokens every GPU pick
    must be a valid top-k member within that margin;
  * counts equal a host recount of the GPU's ids, and the oracle's counts up
    to the near-tie tokens;
  * dispatch (counts, offsets, dest, perm_src, x_perm) bit-exact;
  * bf16 outputs: relative Frobenius error <= 1e-2 and max |err| <= 3e-2 * max |ref|;
    fp32 outputs: relative Frobenius error <= 1e-5.
Large layers compare a seeded sample of tokens (tokens are independent: the
layer has no capacity limit).
"""

import numpy as np
import pytest
import torch

from mixture_experts_layer_91_b300 import binding, inputs, workloads
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

MARGIN = 1e-5
DEV = "cuda"

# bf16 tokens with more than 128 router columns take the CUDA-core router
WIDE_ROUTER = workloads.Workload("wide_router_bf16_T777", T=777, d=512, n_routed=160, n_shared=1,
                                 top_k=8, d_ff=128, seed=17)
# GShard ReLU experts under an expert capacity (mean load 37.5 per expert): some overflow
GSHARD_RELU_SMALL = workloads.Workload("gshard_relu_cap40_T300", T=300, d=512, n_routed=16, n_shared=0,
                                       top_k=2, d_ff=320, renormalize=True, noisy=True, seed=21,
                                       capacity=40, act="relu")
# shared + routed SwiGLU experts under a capacity below the mean load (333*6/64 = 31.2)
DSMOE_16B_CAP = workloads.DSMOE_16B.with_tokens(333, "dsmoe16b_cap28_T333")
DSMOE_16B_CAP = workloads.replace(DSMOE_16B_CAP, capacity=28)
TINY_RELU = workloads.replace(workloads.TINY_FP32, name="tiny_fp32_relu_T256", act="relu", seed=23)
# ragged in every dimension: T not a multiple of 128 (or 32), d and I not
# multiples of 64 (partial k-blocks, partial n-tiles, clipped H stores), E odd
RAGGED = workloads.Workload("ragged_T129_d520_I200_E23", T=129, d=520, n_routed=23, n_shared=1, top_k=5,
                            d_ff=200, seed=31)
RAGGED_BIG = workloads.replace(RAGGED, name="ragged_T4999_d520_I200_E23", T=4999, seed=32)
SMALL = [
    workloads.TINY_FP32,
    TINY_RELU,
    WIDE_ROUTER,
    GSHARD_RELU_SMALL,
    DSMOE_16B_CAP,
    RAGGED,
    RAGGED_BIG,
    workloads.DSMOE_2B.with_tokens(700),
    workloads.DSMOE_16B.with_tokens(333),
    workloads.GSHARD_NOISY.with_tokens(300),
    workloads.DSMOE_145B.with_tokens(150),
    workloads.DSMOE_145B_DECODE,
]
FULL = [workloads.DSMOE_2B, workloads.DSMOE_16B, workloads.GSHARD_NOISY, workloads.DSMOE_145B,
        workloads.GSHARD_RELU_CAP]

_cache = {}


def get_inputs(w, with_experts=True):
    key = (w.name, w.T, with_experts)
    if key not in _cache:
        if len(_cache) > 3:
            _cache.clear()
        _cache[key] = inputs.make_inputs(w, with_experts=with_experts)
    return _cache[key]


def dev(t):
    return None if t is None else t.to(DEV)


def oracle_route(w, inp):
    return O.route(inp["x"], inp["W_g"], w.top_k, renormalize=w.renormalize, noisy=w.noisy,
                   W_noise=inp["W_noise"], eps=inp["eps"], bias=inp["bias"])


def check_close(got, ref, fp32, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    if fp32:
        assert rel <= 1e-5, f"{what}: relative Frobenius error {rel:.3e} > 1e-5"
    else:
        mx = np.abs(got - ref).max()
        assert rel <= 1e-2, f"{what}: relative Frobenius error {rel:.3e} > 1e-2"
        assert mx <= 3e-2 * np.abs(ref).max(), f"{what}: max error {mx:.3e} > 3e-2 max|ref|"
    return rel


def check_routing(w, r, ids, gates):
    """Selected sets bit-exact where the k/(k+1) margin clears MARGIN; the
    order inside the top-k (descending key) exact where every gap between
    consecutive picks clears MARGIN too; gates matched by expert id."""
    ids = ids.cpu().numpy()
    gates = gates.cpu().numpy()
    T, k = ids.shape
    assert ((ids >= 0) & (ids < w.n_routed)).all()
    assert all(len(set(row)) == k for row in ids), "duplicate expert in a token's picks"
    ok = r["margin"] >= MARGIN
    ref_ids = r["ids"]
    set_eq = (np.sort(ids, axis=1) == np.sort(ref_ids, axis=1)).all(axis=1)
    assert set_eq[ok].all(), f"{int((~set_eq[ok]).sum())} margin tokens select a different set"
    key = r["key"] if w.noisy or w.bias else r["logits"]   # what the GPU sorts on
    ref_keys = np.take_along_axis(key, ref_ids, axis=1)
    gaps = (ref_keys[:, :-1] - ref_keys[:, 1:]).min(axis=1) if k > 1 else np.full(T, np.inf)
    ordered = ok & (gaps >= MARGIN)
    assert (ids[ordered] == ref_ids[ordered]).all(), "order inside the top-k differs"
    gi = np.take_along_axis(gates, np.argsort(ids, axis=1), axis=1)
    gr = np.take_along_axis(r["gates"], np.argsort(ref_ids, axis=1), axis=1)
    np.testing.assert_allclose(gi[ok], gr[ok], rtol=2e-5, atol=1e-7)
    # near-tie tokens: each pick must rank within MARGIN of the oracle's k-th key
    kth = np.sort(key, axis=1)[:, ::-1][:, k - 1]
    for t in np.nonzero(~ok)[0]:
        assert (key[t, ids[t]] >= kth[t] - MARGIN).all()
    return ok


# ------------------------------------------------------------------ stages

@pytest.mark.parametrize("w", SMALL + FULL, ids=lambda w: w.name)
def test_route(w, cuda_lib):
    inp = get_inputs(w, with_experts=False)
    cfg = binding.config(w)
    ids, g, logits, stats = binding.route(cfg, dev(inp["x"]), dev(inp["W_g"]), dev(inp["W_noise"]),
                                          dev(inp["eps"]), dev(inp["bias"]), want_logits=True,
                                          want_stats=True)
    r = oracle_route(w, inp)
    ok = check_routing(w, r, ids, g)
    np.testing.assert_allclose(logits.cpu().numpy(), r["logits"], rtol=0, atol=2e-5)
    # router statistics: per-token logsumexp, per-expert sums of s and of the gates
    np.testing.assert_allclose(stats["lse"].cpu().numpy(), O.logsumexp(r["logits"]), rtol=0, atol=4e-5)
    psum = O.prob_column_sums(r["logits"])
    np.testing.assert_allclose(stats["prob_sum"].cpu().numpy(), psum, rtol=2e-4, atol=1e-3)
    imp = O.importance(O.dense_gates(r["ids"], r["gates"], w.n_routed))
    near = r["gates"][~ok].sum()    # tokens under the margin may pick a different (near-equal) expert
    gsum = stats["gate_sum"].cpu().numpy()
    assert np.abs(gsum - imp).max() <= 2e-4 * np.abs(imp).max() + 1e-3 + 2 * near
    assert O.router_z_loss(r["logits"]) == pytest.approx(float(np.mean(stats["lse"].cpu().numpy().astype(np.float64) ** 2)), rel=2e-5)
    ids2, g2 = binding.route(cfg, dev(inp["x"]), dev(inp["W_g"]), dev(inp["W_noise"]),
                             dev(inp["eps"]), dev(inp["bias"]))
    assert torch.equal(ids, ids2) and torch.equal(g, g2), "routing is not deterministic"


# Router-only cases for the tensor-core router (bf16, T >= 4096): expert counts
# that are not a multiple of 8 and a reduction width with a partial last
# k-block and an odd number of tensor-memory drains.
TC_ROUTE_NOISY_ODD = workloads.Workload("tc_route_noisy_e63_T4100", T=4100, d=520, n_routed=63, n_shared=0,
                                        top_k=7, d_ff=64, renormalize=True, noisy=True, seed=31)
TC_ROUTE_BIAS_ODD = workloads.Workload("tc_route_bias_e20_T4133", T=4133, d=1000, n_routed=20, n_shared=0,
                                       top_k=3, d_ff=64, bias=True, seed=32)


@pytest.mark.parametrize("w", [TC_ROUTE_NOISY_ODD, TC_ROUTE_BIAS_ODD], ids=lambda w: w.name)
def test_route_tensor_core_odd_shapes(w, cuda_lib):
    test_route(w, cuda_lib)


# The router's three forms at their boundaries: split-K partial + finish for
# T <= 512, one CTA or cluster per 32 tokens above, the tensor-core router for
# bf16 at T >= 4096 (<= 128 router columns); 256 router columns (EPAD 256) on the
# CUDA-core forms; an fp32 layer with many splits of a long d; noisy at T = 64.
ROUTE_EDGES = [
    workloads.Workload("route_T512_bf16", T=512, d=1024, n_routed=64, n_shared=0, top_k=6, d_ff=64, seed=61),
    workloads.Workload("route_T513_bf16", T=513, d=1024, n_routed=64, n_shared=0, top_k=6, d_ff=64, seed=62),
    workloads.Workload("route_T4095_bf16", T=4095, d=512, n_routed=64, n_shared=0, top_k=6, d_ff=64, seed=63),
    workloads.Workload("route_T4096_bf16", T=4096, d=512, n_routed=64, n_shared=0, top_k=6, d_ff=64, seed=64),
    workloads.Workload("route_T64_E256_bf16", T=64, d=2048, n_routed=256, n_shared=0, top_k=8, d_ff=64,
                       bias=True, seed=65),
    workloads.Workload("route_T700_E256_bf16", T=700, d=512, n_routed=256, n_shared=0, top_k=8, d_ff=64, seed=66),
    workloads.Workload("route_T300_d4096_fp32", T=300, d=4096, n_routed=40, n_shared=0, top_k=4, d_ff=64,
                       fp32=True, seed=67),
    workloads.Workload("route_T64_noisy_bf16", T=64, d=1024, n_routed=32, n_shared=0, top_k=2, d_ff=64,
                       renormalize=True, noisy=True, seed=68),
]


@pytest.mark.parametrize("w", ROUTE_EDGES, ids=lambda w: w.name)
def test_route_forms_at_their_boundaries(w, cuda_lib):
    test_route(w, cuda_lib)


@pytest.mark.parametrize("w", [workloads.DSMOE_145B_DECODE, RAGGED], ids=lambda w: w.name)
def test_route_split_k_on_a_dirty_workspace(w, cuda_lib):
    """Few tokens: the router's split-K partial tiles meet in the route
    workspace. A workspace full of 0xFF bytes gives the same bits as a fresh
    one, and so does a second call on it (every tile is written before it is
    read, and the splits are summed in a fixed order)."""
    inp = get_inputs(w, with_experts=False)
    cfg = binding.config(w)
    assert binding.route_workspace_size(cfg) > 0
    args = (cfg, dev(inp["x"]), dev(inp["W_g"]), dev(inp["W_noise"]), dev(inp["eps"]), dev(inp["bias"]))
    ids, g, lg = binding.route(*args, want_logits=True)
    ws = torch.full((binding.route_workspace_size(cfg),), 0xFF, dtype=torch.uint8, device=DEV)
    for _ in range(2):
        ids2, g2, lg2 = binding.route(*args, want_logits=True, workspace=ws)
        assert torch.equal(ids, ids2) and torch.equal(g, g2) and torch.equal(lg, lg2)
    assert binding.device_status()[0] == 0
    check_routing(w, oracle_route(w, inp), ids, g)


@pytest.mark.parametrize("T,E,k", [(70, 64, 6), (4101, 64, 6), (4101, 63, 7), (4101, 20, 3), (4101, 128, 12)])
def test_route_ties_pick_lowest_index(T, E, k, cuda_lib):
    """All logits equal (W_g = 0): the picks are experts 0..k-1 in order with
    gates 1/E, on the CUDA-core router (T < 4096) and the tensor-core one."""
    w = workloads.Workload("ties", T=T, d=256, n_routed=E, n_shared=0, top_k=k, d_ff=64)
    cfg = binding.config(w)
    x = torch.randn(w.T, w.d, device=DEV).to(torch.bfloat16)
    ids, g = binding.route(cfg, x, torch.zeros(w.d, w.n_routed, device=DEV))
    assert (ids.cpu() == torch.arange(w.top_k, dtype=torch.int32)).all()
    torch.testing.assert_close(g.cpu(), torch.full((w.T, w.top_k), 1.0 / w.n_routed), rtol=1e-6, atol=0)


@pytest.mark.parametrize("T,E,k,skew", [
    (1, 64, 6, "uniform"), (333, 64, 6, "uniform"), (1000, 63, 7, "hot"), (4097, 128, 12, "hot"),
    (16384, 64, 6, "uniform"), (2000, 256, 32, "uniform"), (257, 16, 16, "uniform"),
])
def test_permute_bit_exact(T, E, k, skew, cuda_lib):
    d = 256
    w = workloads.Workload("perm", T=T, d=d, n_routed=E, n_shared=0, top_k=k, d_ff=64, seed=7)
    cfg = binding.config(w)
    ids = inputs.random_topk_ids(T, E, k, seed=T + E, skew=skew)
    x = torch.randn(T, d).to(torch.bfloat16)
    out = binding.permute(cfg, x.to(DEV), ids.to(DEV))
    ref = O.dispatch(ids.numpy(), E)
    assert (out["counts"].cpu().numpy() == ref["counts"]).all()
    assert (out["offsets"].cpu().numpy() == ref["offsets"]).all()
    assert (out["dest"].cpu().numpy() == ref["dest"]).all()
    assert (out["perm_src"].cpu().numpy() == ref["perm_src"]).all()
    want = x[torch.from_numpy(ref["perm_src"] // k)]
    assert torch.equal(out["x_perm"].cpu(), want)
    st, _ = binding.device_status()
    assert st == 0


@pytest.mark.parametrize("T,E,k,cap", [(1000, 63, 7, 60), (4097, 128, 12, 300), (300, 16, 2, 1), (2000, 64, 6, 5000)])
def test_permute_capacity_bit_exact(T, E, k, cap, cuda_lib):
    """Expert capacity: the first `cap` assignments of each expert (ascending
    t*k + j) are grouped, the rest get dest = -1 and no row."""
    d = 128
    w = workloads.Workload("perm_cap", T=T, d=d, n_routed=E, n_shared=0, top_k=k, d_ff=64, capacity=cap)
    cfg = binding.config(w)
    ids = inputs.random_topk_ids(T, E, k, seed=T + cap, skew="hot")
    x = torch.randn(T, d).to(torch.bfloat16)
    out = binding.permute(cfg, x.to(DEV), ids.to(DEV))
    ref = O.dispatch(ids.numpy(), E, capacity=cap)
    n = int(ref["offsets"][-1])
    assert (out["counts"].cpu().numpy() == ref["counts"]).all()
    assert (out["offsets"].cpu().numpy() == ref["offsets"]).all()
    assert (out["dest"].cpu().numpy() == ref["dest"]).all()
    assert (out["perm_src"].cpu().numpy()[:n] == ref["perm_src"]).all()
    assert torch.equal(out["x_perm"].cpu()[:n], x[torch.from_numpy(ref["perm_src"] // k)])
    st, _ = binding.device_status()
    assert st == 0


def test_stages_with_capacity_match_oracle(cuda_lib):
    """permute (with capacity) -> expert_ffn -> combine against the oracle's
    dispatch -> expert_rows -> combine on the same routing."""
    w = DSMOE_16B_CAP
    inp = get_inputs(w)
    cfg = binding.config(w)
    ids = inputs.random_topk_ids(w.T, w.n_routed, w.top_k, seed=29, skew="hot")
    gates = inputs.random_gates(w.T, w.top_k, seed=30)
    g = {k: dev(v) for k, v in inp.items()}
    p = binding.permute(cfg, g["x"], ids.to(DEV))
    rows = binding.expert_ffn(cfg, g["x"], p["x_perm"], p["offsets"], g["W1"], g["W3"], g["W2"])
    y = binding.combine(cfg, rows, p["dest"], gates.to(DEV))
    dsp = O.dispatch(ids.numpy(), w.n_routed, capacity=w.capacity)
    assert (dsp["dest"] < 0).any(), "the capacity should drop assignments in this case"
    ref_rows = O.expert_rows(inp["x"], inp["W1"], inp["W3"], inp["W2"], w.n_shared, dsp["perm_src"],
                             dsp["offsets"], w.top_k)
    ref = O.combine(ref_rows, dsp["dest"], gates.numpy(), w.n_shared, w.T)
    check_close(y.float().cpu().numpy(), ref, False, "capacity stages")


def test_permute_flags_out_of_range_ids(cuda_lib):
    w = workloads.Workload("perm_bad", T=64, d=64, n_routed=8, n_shared=0, top_k=2, d_ff=64)
    cfg = binding.config(w)
    ids = inputs.random_topk_ids(64, 8, 2, seed=1)
    ids[5, 1] = 8      # out of range: skipped by the kernels and reported
    ids[9, 0] = -3
    out = binding.permute(cfg, torch.randn(64, 64).to(torch.bfloat16).to(DEV), ids.to(DEV))
    st, raw = binding.device_status()
    assert st == 6 and raw & 2
    assert int(out["offsets"][-1]) == 64 * 2 - 2
    assert int(out["dest"][5, 1]) == -1 and int(out["dest"][9, 0]) == -1
    assert binding.device_status()[0] == 0   # the flag was cleared


def expert_case(w, seed):
    """Seeded dispatch inputs for moe_expert_ffn: oracle routing of random ids."""
    inp = get_inputs(w)
    ids = inputs.random_topk_ids(w.T, w.n_routed, w.top_k, seed=seed,
                                 skew="hot" if w.n_routed > w.top_k + 3 else "uniform")
    dsp = O.dispatch(ids.numpy(), w.n_routed)
    x_perm = inp["x"][torch.from_numpy(dsp["perm_src"] // w.top_k)]
    return inp, ids, dsp, x_perm


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_expert_ffn(w, cuda_lib):
    inp, ids, dsp, x_perm = expert_case(w, seed=11)
    cfg = binding.config(w)
    out = binding.expert_ffn(cfg, dev(inp["x"]), x_perm.to(DEV),
                             torch.from_numpy(dsp["offsets"].astype(np.int32)).to(DEV),
                             dev(inp["W1"]), dev(inp["W3"]), dev(inp["W2"]))
    ref = O.expert_rows(inp["x"], inp["W1"], inp["W3"], inp["W2"], w.n_shared, dsp["perm_src"],
                        dsp["offsets"], w.top_k, act=w.act)
    check_close(out.cpu().numpy(), ref, w.fp32, "expert rows")
    assert binding.device_status()[0] == 0


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_combine(w, cuda_lib):
    T, k, K_s, d = w.T, w.top_k, w.n_shared, w.d
    rows = inputs.random_rows(K_s * T + T * k, d, seed=3)
    gates = inputs.random_gates(T, k, seed=4)
    ids = inputs.random_topk_ids(T, w.n_routed, k, seed=5)
    dest = O.dispatch(ids.numpy(), w.n_routed)["dest"].astype(np.int32)
    y = binding.combine(binding.config(w), rows.to(DEV), torch.from_numpy(dest).to(DEV), gates.to(DEV))
    ref = O.combine(rows, dest, gates, K_s, T)
    check_close(y.float().cpu().numpy(), ref, w.fp32, "combine")


def test_stages_compose_to_forward(cuda_lib):
    """route -> permute -> expert_ffn -> combine equals moe_forward."""
    w = workloads.DSMOE_16B.with_tokens(257)
    inp = get_inputs(w)
    cfg = binding.config(w)
    g = {k: dev(v) for k, v in inp.items()}
    ids, gw = binding.route(cfg, g["x"], g["W_g"], None, None, None)
    p = binding.permute(cfg, g["x"], ids)
    rows = binding.expert_ffn(cfg, g["x"], p["x_perm"], p["offsets"], g["W1"], g["W3"], g["W2"])
    y_st = binding.combine(cfg, rows, p["dest"], gw)
    y_fw, ids_fw, gw_fw, counts = binding.forward(cfg, g["x"], g["W_g"], None, None, None, g["W1"],
                                                  g["W3"], g["W2"], routing=True)
    assert torch.equal(ids, ids_fw) and torch.equal(gw, gw_fw)   # same kernels, same inputs
    assert torch.equal(counts, p["counts"])
    check_close(y_fw.float().cpu().numpy(), y_st.float().cpu().numpy(), False, "stages vs forward")


# ------------------------------------------------------------------ whole layer

def forward_case(w, sample):
    inp = get_inputs(w)
    cfg = binding.config(w)
    g = {k: dev(v) for k, v in inp.items()}
    y, ids, gw, counts = binding.forward(cfg, g["x"], g["W_g"], g["W_noise"], g["eps"], g["bias"],
                                         g["W1"], g["W3"], g["W2"], routing=True)
    st, raw = binding.device_status()
    assert st == 0, f"device fault flag {raw}"
    r = oracle_route(w, inp)
    ok = check_routing(w, r, ids, gw)
    ids_h = ids.cpu().numpy()
    recount = np.bincount(ids_h.reshape(-1), minlength=w.n_routed)
    if w.capacity:
        recount = np.minimum(recount, w.capacity)
    assert (counts.cpu().numpy() == recount).all()
    ref_counts = np.bincount(r["ids"].reshape(-1), minlength=w.n_routed)
    if w.capacity:
        ref_counts = np.minimum(ref_counts, w.capacity)
    assert np.abs(recount - ref_counts).sum() <= 2 * w.top_k * int((~ok).sum())
    rng = np.random.default_rng(w.seed)
    toks = np.arange(w.T) if sample is None or sample >= w.T else np.sort(rng.choice(w.T, sample, replace=False))
    toks = toks[ok[toks]]
    keep = None
    if w.capacity:
        # a token's capacity decisions depend on the routing of the tokens before
        # it: compare only tokens before the first one under the margin
        first_near = int(np.argmin(ok)) if not ok.all() else w.T
        toks = toks[toks < first_near]
        keep = O.capacity_keep(r["ids"], w.n_routed, w.capacity)
        assert toks.size > 0
    ref = O.moe_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], w.n_shared, r["ids"], r["gates"],
                        tokens=toks, act=w.act, keep=keep)
    got = y.float().cpu().numpy()[toks]
    return check_close(got, ref, w.fp32, f"{w.name} y")


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_forward_small(w, cuda_lib):
    forward_case(w, None)


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_forward_full_size_sampled(w, cuda_lib):
    forward_case(w, 512 if w.d >= 4096 else 1024)


def test_forward_is_repeatable(cuda_lib):
    w = workloads.DSMOE_2B.with_tokens(999)
    inp = get_inputs(w)
    layer = binding.MoELayer(w, inp)
    x = inp["x"].to(DEV)
    y1 = layer(x).clone()
    y2 = layer(x).clone()
    check_close(y2.float().cpu().numpy(), y1.float().cpu().numpy(), False, "repeat")
    assert (y1 - y2).abs().max().item() <= 1e-2 * y1.abs().max().item()


@pytest.mark.parametrize("depth", [2, 3])
def test_host_stream_matches_device_forward(depth, cuda_lib):
    """Overlapped host-batch pipeline: each y equals the device forward of its x."""
    w = workloads.GSHARD_NOISY.with_tokens(512)
    inp = get_inputs(w)
    layer = binding.MoELayer(w, inp)
    g = torch.Generator().manual_seed(5)
    xs = [torch.randn(w.T, w.d, generator=g).to(torch.bfloat16).pin_memory() for _ in range(5)]
    es = [torch.randn(w.T, w.n_routed, generator=g).pin_memory() for _ in range(5)]
    ys = [torch.empty(w.T, w.d, dtype=torch.bfloat16, pin_memory=True) for _ in range(5)]
    layer.forward_host_stream(xs, ys, es, depth=depth)
    torch.cuda.synchronize()
    for i in range(5):
        ref = layer(xs[i].to(DEV), es[i].to(DEV)).float().cpu().numpy()
        check_close(ys[i].float().numpy(), ref, False, f"host batch {i}")


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    binding.debug_wait_timeout(100000)           # 0.1 s wait that nothing satisfies
    st, raw = binding.device_status()
    assert st == 5 and raw & 1
    assert binding.device_status()[0] == 0
    test_forward_small(workloads.TINY_FP32, cuda_lib)   # the context is still usable


# ------------------------------------------------------------------ combine modes
# The layers above run the default MOE_COMBINE_ROWS (bf16 expert rows summed per
# token by the combine kernel); these run the down GEMM's gate-weighted
# scatter-add into an fp32 accumulator (MOE_COMBINE_SCATTER_ADD). Same names and
# inputs as their row-combine twins.
SCATTER = [workloads.replace(w, combine="scatter") for w in
           (workloads.DSMOE_16B.with_tokens(333), GSHARD_RELU_SMALL, RAGGED, DSMOE_16B_CAP,
            workloads.DSMOE_145B_DECODE)]


@pytest.mark.parametrize("w", SCATTER, ids=lambda w: w.name + "_scatter")
def test_forward_scatter_add_combine(w, cuda_lib):
    forward_case(w, None)


def test_forward_scatter_add_combine_full_size(cuda_lib):
    forward_case(workloads.DSMOE_16B_SCATTER, 1024)


def test_combine_modes_agree_and_rows_are_bitwise_repeatable(cuda_lib):
    w = workloads.DSMOE_16B.with_tokens(333)
    inp = get_inputs(w)
    g = {k: dev(v) for k, v in inp.items()}

    def run(wl):
        return binding.forward(binding.config(wl), g["x"], g["W_g"], g["W_noise"], g["eps"], g["bias"],
                               g["W1"], g["W3"], g["W2"]).float().cpu().numpy()

    y_rows, y_rows2 = run(w), run(w)
    y_scatter = run(workloads.replace(w, combine="scatter"))
    assert np.array_equal(y_rows, y_rows2), "the row combine is not deterministic"
    check_close(y_rows, y_scatter, False, "rows vs scatter-add")
