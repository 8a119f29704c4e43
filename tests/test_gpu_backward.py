"""Backward pass on the GPU (moe_backward through the C ABI) vs the fp64
oracle of the layer's gradients (oracle/moe_backward.py).

The upstream gradient dy is seeded N(0, 1). Tokens whose oracle routing
margin (k-th minus (k+1)-th key) is below 1e-5 get dy = 0: the GPU may pick a
different (equally valid) expert for them, and with dy = 0 such a token
contributes nothing to any gradient on either side. Under an expert capacity,
where a token's keep/drop decisions depend on every earlier token's routing,
dy is zeroed from the first near-tie token on.

Criteria per gradient tensor (dx, dW_g, dW_noise, dW1, dW3, dW2), the same
as the forward's: bf16 layers relative Frobenius error <= 1e-2 and max |err|
<= 3e-2 max |ref|; the fp32 layer relative Frobenius error <= 1e-5.
"""

import numpy as np
import pytest
import torch

from mixture_experts_layer_91_b300 import binding, inputs, workloads
from oracle import moe_backward as B
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"
MARGIN = 1e-5

RAGGED = workloads.Workload("ragged_T129_d520_I200_E23", T=129, d=520, n_routed=23, n_shared=1, top_k=5,
                            d_ff=200, seed=31)
RAGGED_BIG = workloads.replace(RAGGED, name="ragged_T1999_d520_I200_E23", T=1999, seed=32)
TINY_RELU = workloads.replace(workloads.TINY_FP32, name="tiny_fp32_relu_T256", act="relu", seed=23)
TINY_NOISY = workloads.Workload("tiny_fp32_noisy_T200", T=200, d=64, n_routed=8, n_shared=0, top_k=2,
                                d_ff=32, renormalize=True, noisy=True, fp32=True, seed=41)
TINY_RENORM_CAP = workloads.Workload("tiny_fp32_renorm_cap_T160", T=160, d=96, n_routed=10, n_shared=2,
                                     top_k=3, d_ff=48, renormalize=True, fp32=True, seed=42, capacity=40)
GSHARD_RELU_SMALL = workloads.Workload("gshard_relu_cap40_T300", T=300, d=512, n_routed=16, n_shared=0,
                                       top_k=2, d_ff=320, renormalize=True, noisy=True, seed=21,
                                       capacity=40, act="relu")
DSMOE_16B_CAP = workloads.replace(workloads.DSMOE_16B.with_tokens(333, "dsmoe16b_cap28_T333"), capacity=28)
# the tensor-core router path (bf16 tokens, T >= 4096) feeding the backward
ROUTER_TC = workloads.Workload("bwd_tc_router_T4100_d256", T=4100, d=256, n_routed=20, n_shared=1, top_k=4,
                               d_ff=128, renormalize=True, seed=43)

FP32 = [workloads.TINY_FP32, TINY_RELU, TINY_NOISY, TINY_RENORM_CAP]
BF16 = [RAGGED, RAGGED_BIG, workloads.DSMOE_16B.with_tokens(333), workloads.DSMOE_2B.with_tokens(300),
        workloads.GSHARD_NOISY.with_tokens(300), GSHARD_RELU_SMALL, DSMOE_16B_CAP,
        workloads.DSMOE_145B.with_tokens(100), workloads.DSMOE_145B_DECODE, ROUTER_TC]


def check_close(got, ref, fp32, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nref = np.linalg.norm(ref)
    assert nref > 0, f"{what}: reference gradient is zero"
    rel = np.linalg.norm(got - ref) / nref
    if fp32:
        assert rel <= 1e-5, f"{what}: relative Frobenius error {rel:.3e} > 1e-5"
    else:
        mx = np.abs(got - ref).max()
        assert rel <= 1e-2, f"{what}: relative Frobenius error {rel:.3e} > 1e-2"
        assert mx <= 3e-2 * np.abs(ref).max(), f"{what}: max error {mx:.3e} > 3e-2 max|ref|"
    return rel


def upstream(w, inp):
    """Seeded dy with the rows of near-tie tokens zeroed (see the module doc)."""
    r = O.route(inp["x"], inp["W_g"], w.top_k, renormalize=w.renormalize, noisy=w.noisy,
                W_noise=inp["W_noise"], eps=inp["eps"], bias=inp["bias"])
    ok = r["margin"] >= MARGIN
    if w.capacity and not ok.all():
        ok[int(np.argmin(ok)):] = False
    dy = inputs.make_upstream_grad(w, seed=w.seed + 500)
    dy[torch.from_numpy(~ok)] = 0
    return dy, ok


def run_case(w):
    inp = inputs.make_inputs(w)
    dy, ok = upstream(w, inp)
    assert ok.sum() > 0
    cfg = binding.config(w)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    got = binding.backward(cfg, g["x"], g["W_g"], g["W_noise"], g["eps"], g["bias"], g["W1"], g["W3"],
                           g["W2"], dy.to(DEV))
    st, raw = binding.device_status()
    assert st == 0, f"device fault flag {raw}"
    ref = B.moe_backward(inp["x"], inp["W_g"], inp["W1"], inp["W3"], inp["W2"], w.n_shared, w.top_k, dy,
                         renormalize=w.renormalize, noisy=w.noisy, W_noise=inp["W_noise"], eps=inp["eps"],
                         bias=inp["bias"], capacity=w.capacity, act=w.act)
    names = ["dx", "dW_g", "dW1", "dW2"]
    if w.noisy:
        names.append("dW_noise")
    if w.act != "relu":
        names.append("dW3")
    errs = {}
    for n in names:
        errs[n] = check_close(got[n].float().cpu().numpy(), ref[n], w.fp32, f"{w.name} {n}")
    return errs


@pytest.mark.parametrize("w", FP32, ids=lambda w: w.name)
def test_backward_fp32(w, cuda_lib):
    run_case(w)


@pytest.mark.parametrize("w", BF16, ids=lambda w: w.name)
def test_backward_bf16(w, cuda_lib):
    run_case(w)


def test_backward_repeatable_and_independent_of_workspace_contents(cuda_lib):
    """Two calls, the second on a workspace filled with garbage, agree (up to
    the router-weight gradient's atomics order)."""
    w = RAGGED
    inp = inputs.make_inputs(w)
    dy, _ = upstream(w, inp)
    cfg = binding.config(w)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    ws = torch.empty(binding.backward_workspace_size(cfg), dtype=torch.uint8, device=DEV)
    args = (cfg, g["x"], g["W_g"], g["W_noise"], g["eps"], g["bias"], g["W1"], g["W3"], g["W2"], dy.to(DEV))
    a = binding.backward(*args, workspace=ws)
    ws.fill_(0xFF)   # NaN bit patterns everywhere
    b = binding.backward(*args, workspace=ws)
    for n in ("dx", "dW1", "dW3", "dW2"):
        assert torch.equal(a[n], b[n]), n
    torch.testing.assert_close(a["dW_g"], b["dW_g"], rtol=1e-5, atol=1e-6)


def test_backward_no_tokens_gives_zero_weight_gradients(cuda_lib):
    w = RAGGED.with_tokens(0)
    cfg = binding.config(w)
    inp = inputs.make_inputs(workloads.replace(RAGGED, T=1))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    x = torch.empty(0, w.d, dtype=torch.bfloat16, device=DEV)
    out = binding.backward(cfg, x, g["W_g"], None, None, None, g["W1"], g["W3"], g["W2"], x)
    for n in ("dW_g", "dW1", "dW3", "dW2"):
        assert torch.count_nonzero(out[n]).item() == 0, n


TRAIN = [workloads.TINY_FP32, TINY_NOISY, RAGGED, workloads.DSMOE_16B.with_tokens(333), GSHARD_RELU_SMALL,
         DSMOE_16B_CAP]


@pytest.mark.parametrize("w", TRAIN, ids=lambda w: w.name)
def test_forward_train_then_backward_from_forward(w, cuda_lib):
    """moe_forward_train's y matches the oracle forward and moe_forward;
    moe_backward_from_forward on its state gives moe_backward's gradients
    (bitwise for bf16 layers: the same kernels on the same inputs)."""
    inp = inputs.make_inputs(w)
    dy, ok = upstream(w, inp)
    cfg = binding.config(w)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    ws = torch.empty(binding.backward_workspace_size(cfg), dtype=torch.uint8, device=DEV)
    ws.fill_(0xFF)
    fw = (cfg, g["x"], g["W_g"], g["W_noise"], g["eps"], g["bias"], g["W1"], g["W3"], g["W2"])
    y = binding.forward_train(*fw, workspace=ws)
    assert binding.device_status()[0] == 0
    # y against the oracle on the tokens whose routing is unambiguous
    r = O.route(inp["x"], inp["W_g"], w.top_k, renormalize=w.renormalize, noisy=w.noisy,
                W_noise=inp["W_noise"], eps=inp["eps"], bias=inp["bias"])
    toks = np.nonzero(ok)[0]
    keep = O.capacity_keep(r["ids"], w.n_routed, w.capacity) if w.capacity else None
    ref_y = O.moe_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], w.n_shared, r["ids"], r["gates"],
                          tokens=toks, act=w.act, keep=keep)
    check_close(y.float().cpu().numpy()[toks], ref_y, w.fp32, f"{w.name} forward_train y")
    y_ref = binding.forward(*fw)
    check_close(y.float().cpu().numpy()[toks], y_ref.float().cpu().numpy()[toks], w.fp32, "vs moe_forward")
    ref = binding.backward(*fw, dy.to(DEV))
    got = binding.backward(*fw, dy.to(DEV), workspace=ws, from_forward=True)
    assert binding.device_status()[0] == 0
    for n in ("dx", "dW_g", "dW_noise", "dW1", "dW3", "dW2"):
        if got[n] is None:
            continue
        if w.fp32:   # the fp32 router-weight gradient sums chunks with atomics
            torch.testing.assert_close(got[n], ref[n], rtol=1e-5, atol=1e-7)
        else:
            assert torch.equal(got[n], ref[n]), n
