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
