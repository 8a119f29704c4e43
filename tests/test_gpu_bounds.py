"""Output bounds: no entry point writes outside the buffers it is given.

Every output of the stage calls and of moe_forward, and the workspace, is
placed inside a larger device buffer whose margins (4 KiB on each side) hold
a sentinel byte pattern. After the call the margins must be untouched, and the
outputs must equal those of a plain (unguarded) call. The shapes are the ones
where an off-by-one would show: ragged in every dimension (partial k-blocks,
n-tiles and 128-row tiles, clipped TMA stores), an expert capacity that drops
assignments, and the 64-token decode layer (mostly empty tiles).
This stands in for a memory sanitizer, which this GPU pool does not offer.
"""

import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_91_b300 import binding, inputs, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"
MARGIN = 4096          # bytes of sentinel on each side of every buffer
SENTINEL = 0xA5

RAGGED = workloads.Workload("ragged_T129_d520_I200_E23", T=129, d=520, n_routed=23, n_shared=1, top_k=5,
                            d_ff=200, seed=31)
CAP = workloads.replace(workloads.DSMOE_16B.with_tokens(333, "dsmoe16b_cap28_T333"), capacity=28)
CASES = [RAGGED, CAP, workloads.DSMOE_145B_DECODE, workloads.TINY_FP32,
         workloads.replace(RAGGED, name="ragged_scatter", combine="scatter")]


class Guarded:
    """A tensor of `shape`/`dtype` in the middle of a sentinel-filled buffer."""

    def __init__(self, shape, dtype, fill=None):
        esize = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) if len(shape) else 1
        self.raw = torch.full((2 * MARGIN + max(n, 1) * esize,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.t = self.raw[MARGIN:MARGIN + n * esize].view(dtype).view(*shape)
        if fill is not None:
            self.t.copy_(fill)

    @property
    def ptr(self):
        return self.t.data_ptr()

    def margins_intact(self):
        head = self.raw[:MARGIN]
        tail = self.raw[self.raw.numel() - MARGIN:]
        return bool((head == SENTINEL).all().item()) and bool((tail == SENTINEL).all().item())


def _cfg(w):
    return binding.config(w)


def _p(t):
    return None if t is None else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _all_intact(bufs):
    bad = [name for name, b in bufs.items() if not b.margins_intact()]
    assert not bad, f"writes outside the buffer: {bad}"


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_outputs_stay_in_bounds(w, cuda_lib):
    lib = cuda_lib
    inp = inputs.make_inputs(w)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    cfg = _cfg(w)
    T, k, E, d, K_s = w.T, w.top_k, w.n_routed, w.d, w.n_shared
    act = torch.float32 if w.fp32 else torch.bfloat16

    # ---- moe_route: ids, gates, logits, statistics and the workspace
    b = {"ids": Guarded((T, k), torch.int32), "w": Guarded((T, k), torch.float32),
         "logits": Guarded((T, E), torch.float32), "lse": Guarded((T,), torch.float32),
         "prob_sum": Guarded((E,), torch.float32), "gate_sum": Guarded((E,), torch.float32),
         "ws": Guarded((max(binding.route_workspace_size(cfg), 16),), torch.uint8)}
    stats = binding.RouterStats(b["lse"].ptr, b["prob_sum"].ptr, b["gate_sum"].ptr)
    st = lib.moe_route(ctypes.byref(cfg), _p(g["x"]), _p(g["W_g"]), _p(g["W_noise"]), _p(g["eps"]),
                       _p(g["bias"]), b["ids"].ptr, b["w"].ptr, b["logits"].ptr, ctypes.byref(stats),
                       b["ws"].ptr, b["ws"].t.numel(), _stream())
    assert st == 0
    torch.cuda.synchronize()
    _all_intact(b)
    ids_ref, w_ref = binding.route(cfg, g["x"], g["W_g"], g["W_noise"], g["eps"], g["bias"])
    assert torch.equal(b["ids"].t, ids_ref) and torch.equal(b["w"].t, w_ref)
    ids = ids_ref

    # ---- moe_permute
    p = {"counts": Guarded((E,), torch.int32), "offsets": Guarded((E + 1,), torch.int32),
         "dest": Guarded((T, k), torch.int32), "perm_src": Guarded((T * k,), torch.int32),
         "x_perm": Guarded((T * k, d), act),
         "ws": Guarded((max(binding.permute_workspace_size(cfg), 16),), torch.uint8)}
    st = lib.moe_permute(ctypes.byref(cfg), _p(g["x"]), _p(ids), p["ws"].ptr, p["ws"].t.numel(),
                         p["counts"].ptr, p["offsets"].ptr, p["dest"].ptr, p["perm_src"].ptr,
                         p["x_perm"].ptr, _stream())
    assert st == 0
    torch.cuda.synchronize()
    _all_intact(p)
    ref = binding.permute(cfg, g["x"], ids)
    n = int(ref["offsets"][-1])
    for name in ("counts", "offsets", "dest"):
        assert torch.equal(p[name].t, ref[name]), name
    assert torch.equal(p["perm_src"].t[:n], ref["perm_src"][:n])
    assert torch.equal(p["x_perm"].t[:n], ref["x_perm"][:n])

    # ---- moe_expert_ffn: per-row outputs and its workspace (group plan and H)
    f = {"rows": Guarded((K_s * T + T * k, d), torch.float32),
         "ws": Guarded((binding.expert_ffn_workspace_size(cfg),), torch.uint8)}
    st = lib.moe_expert_ffn(ctypes.byref(cfg), _p(g["x"]), _p(ref["x_perm"]), _p(ref["offsets"]),
                            _p(g["W1"]), _p(g["W3"]), _p(g["W2"]), f["ws"].ptr, f["ws"].t.numel(),
                            f["rows"].ptr, _stream())
    assert st == 0
    torch.cuda.synchronize()
    _all_intact(f)

    # ---- moe_combine
    c = {"y": Guarded((T, d), act)}
    st = lib.moe_combine(ctypes.byref(cfg), f["rows"].ptr, _p(ref["dest"]), _p(w_ref), c["y"].ptr, _stream())
    assert st == 0
    torch.cuda.synchronize()
    _all_intact(c)

    # ---- moe_forward: y, routing outputs, counts and the whole workspace
    fw = {"y": Guarded((T, d), act), "ids": Guarded((T, k), torch.int32), "w": Guarded((T, k), torch.float32),
          "counts": Guarded((E,), torch.int32), "ws": Guarded((binding.workspace_size(cfg),), torch.uint8)}
    st = lib.moe_forward(ctypes.byref(cfg), _p(g["x"]), _p(g["W_g"]), _p(g["W_noise"]), _p(g["eps"]),
                         _p(g["bias"]), _p(g["W1"]), _p(g["W3"]), _p(g["W2"]), fw["ws"].ptr,
                         fw["ws"].t.numel(), fw["y"].ptr, fw["ids"].ptr, fw["w"].ptr, fw["counts"].ptr,
                         _stream())
    assert st == 0
    torch.cuda.synchronize()
    _all_intact(fw)
    assert torch.equal(fw["ids"].t, ids_ref)
    assert torch.equal(fw["counts"].t, ref["counts"])
    y_ref = binding.forward(cfg, g["x"], g["W_g"], g["W_noise"], g["eps"], g["bias"], g["W1"], g["W3"], g["W2"])
    if w.fp32 or w.combine == "scatter":   # fp32 atomics: the summation order may differ
        torch.testing.assert_close(fw["y"].t.float(), y_ref.float(), rtol=1e-2, atol=1e-2)
    else:
        assert torch.equal(fw["y"].t, y_ref)
    st, raw = binding.device_status()
    assert st == 0, raw
