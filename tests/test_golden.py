"""Stored fixtures: the pages' printed figures and the oracle's tiny outputs."""
import json
import math
import os

import numpy as np

from tests.golden import make_golden

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_pages_teacher_tensor_size():
    # the dense teacher-probability tensor the method avoids: ~50 GB in bf16
    t = _load("pages_figures.json")["teacher_tensor"]
    gb = t["batch"] * t["vocab"] * t["seq"] * t["dtype_bytes"] / 1e9
    assert abs(gb - t["approx_GB"]) / t["approx_GB"] < 0.06


def test_pages_ratios_are_self_consistent():
    f = _load("pages_figures.json")
    r = f["isolated_32k"]
    assert abs(r["dense_GiB"] / r["fused_GiB"] - r["reduction"]) < 0.05
    g = f["gptoss20b_32k"]
    # step-time ratio and per-GPU throughput ratio are equal (both ~4.66)
    assert math.isclose(g["step_s_before"] / g["step_s_after"],
                        g["tflops_per_gpu_after"] / g["tflops_per_gpu_before"],
                        rel_tol=1e-3)


def test_oracle_matches_its_stored_tiny_outputs():
    want = _load("tiny_oracle.json")
    got = make_golden.summary()
    for key in ("loss", "grad_hidden_fro", "grad_W_fro", "grad_hidden_00", "grad_W_00"):
        assert math.isclose(got[key], want[key], rel_tol=1e-10, abs_tol=1e-16), key
    np.testing.assert_allclose(got["lse_first4"], want["lse_first4"], rtol=1e-12)
