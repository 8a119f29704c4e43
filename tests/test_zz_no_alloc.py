"""moe_permute_static: dispatch with no caller workspace and no allocation.

Some callers cannot allocate device memory for scratch (a framework that owns
the whole device-memory budget, a serving loop that must never enter an
allocator). For them the library keeps the dispatch scratch in a fixed device
array of its own. These tests check, through the C ABI, that this entry point
gives exactly what moe_permute (caller workspace) gives, on two calls in a
row (the array keeps the previous call's contents), and that problems larger
than the array are refused on the host.

This file is named to be collected last.
"""

import ctypes

import pytest
import torch

from mixture_experts_layer_91_b300 import binding, build, inputs, workloads


def _cfg(T, E, k, d):
    return binding.config(workloads.Workload("static", T=T, d=d, n_routed=E, n_shared=0,
                                             top_k=k, d_ff=64))


def test_static_limit_refused_on_host():
    build.build()
    lib = binding.load()
    too_big = _cfg(binding.PERMUTE_STATIC_MAX_ASSIGN // 8 + 1, 64, 8, 128)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    st = lib.moe_permute_static(ctypes.byref(too_big), fake, fake, fake, fake, fake, fake, fake, None)
    assert st == 7   # MOE_ERR_STATIC_LIMIT
    assert b"moe_permute_static" in lib.moe_status_string(7)


@pytest.mark.gpu
def test_permute_static_matches_permute_on_two_calls(cuda_lib):
    dev = "cuda"
    # two different problems back to back: the second call must not see the first's scratch
    cases = [(4097, 128, 12, "hot", 1024), (16384, 64, 6, "uniform", 256)]
    for T, E, k, skew, d in cases:
        cfg = _cfg(T, E, k, d)
        ids = inputs.random_topk_ids(T, E, k, seed=T, skew=skew).to(dev)
        x = torch.randn(T, d, device=dev).to(torch.bfloat16)
        ref = binding.permute(cfg, x, ids)
        got = binding.permute_static(cfg, x, ids)
        for name in ("counts", "offsets", "dest", "perm_src", "x_perm"):
            assert torch.equal(got[name], ref[name]), name
        st, raw = binding.device_status()
        assert st == 0, raw
    # the largest problem the fixed scratch admits
    T, E, k = binding.PERMUTE_STATIC_MAX_ASSIGN // 16, 256, 16
    cfg = _cfg(T, E, k, 64)
    ids = inputs.random_topk_ids(T, E, k, seed=3).to(dev)
    x = torch.randn(T, 64, device=dev).to(torch.bfloat16)
    ref = binding.permute(cfg, x, ids)
    got = binding.permute_static(cfg, x, ids)
    for name in ("counts", "offsets", "dest", "perm_src", "x_perm"):
        assert torch.equal(got[name], ref[name]), name
