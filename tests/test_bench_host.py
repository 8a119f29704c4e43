"""Host-side arithmetic of bench.py's JSON line (no GPU): the dominant
kernel's roofline object and the FLOP / byte counts behind it."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mixture_experts_layer_91_b300 import workloads  # noqa: E402

PK = {"hbm_gbs": 6500.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def test_prefill_gate_up_is_tensor_bound():
    w = workloads.DSMOE_16B
    kept = w.T * w.top_k
    flops = 4.0 * w.d * w.d_ff * (kept + w.n_shared * w.T)   # W1 and W3 products of every row
    ms = flops / 1500e12 * 1e3                                # as if it ran at 1500 TFLOP/s
    r = bench.gate_up_roofline(w, w.n_experts, kept, ms, PK, "measured", None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1500.0)
    assert r["frac"] == pytest.approx(1500.0 / 1800.0)
    assert r["frac_of_sustained"] == pytest.approx(1500.0 / 1400.0)
    assert r["algorithmic_flops_per_launch"] == pytest.approx(flops)


def test_decode_gate_up_is_hbm_bound():
    w = workloads.DSMOE_145B_DECODE
    kept = w.T * w.top_k
    touched = 120 + w.n_shared
    nbytes = touched * 2 * w.d * w.d_ff * 2 + w.T * w.d * 2   # touched W1 + W3 in bf16, x once
    ms = nbytes / 5200e9 * 1e3                                 # as if it moved them at 5.2 TB/s
    r = bench.gate_up_roofline(w, touched, kept, ms, PK, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(5200.0)
    assert r["frac"] == pytest.approx(5200.0 / 6500.0)
    assert r["algorithmic_bytes_per_launch"] == pytest.approx(nbytes)


def test_relu_experts_count_one_gate_up_matrix():
    w = workloads.GSHARD_RELU_CAP
    kept = 5000
    r = bench.gate_up_roofline(w, w.n_experts, kept, 1.0, PK, "measured", None)
    assert r["algorithmic_flops_per_launch"] == pytest.approx(2.0 * w.d * w.d_ff * kept)


def test_traffic_record_applies_only_to_its_workload():
    rec = bench.ncu_traffic(workloads.DSMOE_16B)
    if rec is not None:   # present while the gate-up sources match the capture
        assert rec["workload"] == workloads.DSMOE_16B.name
    for w in (workloads.DSMOE_145B_DECODE, workloads.GSHARD_NOISY, workloads.DSMOE_2B):
        assert bench.ncu_traffic(w) is None


def test_kernel_key_ignores_comments_but_not_code():
    a = 'int f(int x) { // doubles\n  return 2 * x;  /* fast */ }\nconst char* s = "a // b";\n'
    b = 'int f(int x) {   // returns twice x\n  return 2 * x; }\nconst char* s = "a // b";\n'
    c = 'int f(int x) { return 3 * x; }\nconst char* s = "a // b";\n'
    assert bench.code_tokens(a) == bench.code_tokens(b)
    assert bench.code_tokens(a) != bench.code_tokens(c)
    assert '"a // b"' in bench.code_tokens(a)        # a // inside a string literal is code


def test_reference_arm_reports_what_it_ran(capsys):
    """--impl reference times the oracle on the fixed sample, step by step:
    ms_per_step is the measured step time (steps x ms_per_step is the run),
    value is the sample's tokens over the median step, and its config equals
    the main arm's."""
    import argparse
    import json
    import time

    w = workloads.TINY_FP32
    args = argparse.Namespace(steps=2, warmup=1)
    t0 = time.perf_counter()
    assert bench.run_reference(args, w) == 0
    wall = time.perf_counter() - t0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2
    assert line["ms_per_step"] * line["steps"] / 1e3 <= wall
    assert line["value"] == pytest.approx(bench.oracle_sample(w).size / (line["ms_per_step"] / 1e3), rel=0.5)
    assert line["config"] == bench.workload_config(w, 1)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_oracle_sample_is_fixed_and_bounded():
    w = workloads.DSMOE_16B
    a, b = bench.oracle_sample(w), bench.oracle_sample(w)
    assert (a == b).all() and a.size == bench.ORACLE_SAMPLE_TOKENS and len(set(a.tolist())) == a.size
    assert bench.oracle_sample(workloads.TINY_FP32).size == workloads.TINY_FP32.T


def test_backward_flops_count_each_weight_product_twice():
    """The derivative's own FLOPs are twice the forward's expert FLOPs (dgrad +
    wgrad) plus the router's two products; the recomputed gate-up is counted
    per stage but not in the algorithmic total."""
    for w in (workloads.DSMOE_16B, workloads.GSHARD_RELU_CAP):
        kept = w.T * w.top_k
        fl = bench.backward_flops(w, kept)
        fwd = bench.kernel_flops(w, kept)
        assert fl["save"] == pytest.approx(fwd["gate_up"])
        assert fl["dh"] + fl["dx"] + fl["wgrad"] == pytest.approx(2 * (fwd["gate_up"] + fwd["down"]))
        assert fl["algorithmic"] == pytest.approx(2 * (fwd["gate_up"] + fwd["down"]) + 2 * fwd["router"])


def test_launch_counts_follow_the_router_choice():
    """Kernels per forward / backward, as the launch lists of a B300 (148 SMs)
    show them: the 16B layer routes through split + tensor-core router + finish
    (9 forward kernels, 18 backward), the 145B decode (T = 64) through split-K
    partial + finish (8), the tiny fp32 layer through split-K too but with no
    combine kernel (7), and a 1000-token bf16 layer through the cluster router +
    finish (8)."""
    import bench
    from mixture_experts_layer_91_b300 import workloads as W
    assert bench.forward_launches(W.DSMOE_16B, 148) == 9
    assert bench.backward_launches(W.DSMOE_16B, 148) == 18
    assert bench.forward_launches(W.DSMOE_2B, 148) == 9
    assert bench.forward_launches(W.DSMOE_145B_DECODE, 148) == 8
    assert bench.forward_launches(W.TINY_FP32, 148) == 7
    assert bench.forward_launches(W.DSMOE_16B.with_tokens(1000), 148) == 8
    # noisy with 2 x 64 router columns still fits the tensor-core router
    assert bench.route_launches(W.replace(W.GSHARD_NOISY, n_routed=64), 148) == 3
    assert bench.route_launches(W.replace(W.GSHARD_NOISY, n_routed=65), 148) == 2
