"""The oracle against facts outside itself (CPU only).

The pins are described in ``oracle_pins``.  Besides them: chunk-size
independence of the oracle's row blocking, the per-row and per-vocab-row
helpers against the full computation, and the input generators' contract.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import oracle_pins as pins


def impl(h, W, idx, lg, T):
    return oracle.fused_topk_kl(h, W, idx, lg, T)


@pytest.mark.parametrize("T", [1.0, 2.0])
@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, T):
    pin(impl, T)


def test_finite_differences_with_repeated_id():
    # a repeated id in a row adds up its teacher mass in dZ (scatter-add)
    pins.pin_finite_differences(impl, 1.5, dup=True)


@pytest.mark.parametrize("T", [0.7, 3.0])
def test_chunk_rows_do_not_change_the_result(T):
    h, W, idx, lg = pins.small_case(11, N=64, H=12, V=50, K=7)
    ref = oracle.fused_topk_kl(h, W, idx, lg, T, chunk_rows=64)
    for c in (1, 7, 13):
        out = oracle.fused_topk_kl(h, W, idx, lg, T, chunk_rows=c)
        assert abs(out["loss"] - ref["loss"]) <= 1e-12
        for key in ("grad_hidden", "grad_W", "lse", "zg", "loss_rows"):
            np.testing.assert_allclose(out[key], ref[key], rtol=0, atol=1e-12)


def test_rows_forward_matches_full():
    h, W, idx, lg = pins.small_case(12, N=20, H=9, V=33, K=5)
    full = oracle.fused_topk_kl(h, W, idx, lg, 1.3)
    rows = np.array([0, 3, 19, 7])
    part = oracle.rows_forward(h[rows], W, idx[rows], lg[rows], 1.3, N_total=20)
    for key in ("lse", "zg", "loss_rows", "grad_hidden"):
        np.testing.assert_allclose(part[key], full[key][rows], rtol=0, atol=1e-13)


def test_rows_forward_vocab_rows_add_up_to_full_grad_W():
    # per-block shares of grad_W rows, summed over disjoint token blocks,
    # equal the full problem's rows; grad_hidden=False leaves the rest alone
    h, W, idx, lg = pins.small_case(14, N=23, H=7, V=37, K=5)
    T = 1.7
    full = oracle.fused_topk_kl(h, W, idx, lg, T)
    vrows = np.array([36, 0, int(idx[5, 1]), 11, int(idx[5, 1])])
    acc = np.zeros((len(vrows), 7))
    for r0, r1 in ((0, 9), (9, 10), (10, 23)):
        part = oracle.rows_forward(h[r0:r1], W, idx[r0:r1], lg[r0:r1], T, N_total=23,
                                   vrows=vrows, grad_hidden=False)
        assert "grad_hidden" not in part
        np.testing.assert_allclose(part["lse"], full["lse"][r0:r1], rtol=0, atol=1e-13)
        np.testing.assert_allclose(part["loss_rows"], full["loss_rows"][r0:r1], rtol=0,
                                   atol=1e-13)
        acc += part["grad_W_rows"]
    np.testing.assert_allclose(acc, full["grad_W"][vrows], rtol=0, atol=1e-14)


def test_grad_W_rows_matches_full():
    h, W, idx, lg = pins.small_case(13, N=25, H=6, V=40, K=6)
    full = oracle.fused_topk_kl(h, W, idx, lg, 0.9)
    vrows = np.array([0, 39, int(idx[3, 2]), 17])
    got = oracle.grad_W_rows(h, W, idx, lg, 0.9, vrows, chunk_rows=6)
    np.testing.assert_allclose(got, full["grad_W"][vrows], rtol=0, atol=1e-14)


def test_oracle_reads_torch_tensors_exactly():
    inp = workloads.make_inputs(workloads.custom(N=16, H=32, V=64, K=4), seed=3)
    out_t = oracle.fused_topk_kl(inp["hidden"], inp["W"], inp["topk_idx"],
                                 inp["topk_logit"], 1.0)
    h = inp["hidden"].to(torch.float64).numpy()
    W = inp["W"].to(torch.float64).numpy()
    out_n = oracle.fused_topk_kl(h, W, inp["topk_idx"].numpy().astype(np.int64),
                                 inp["topk_logit"].double().numpy(), 1.0)
    assert out_t["loss"] == out_n["loss"]


@pytest.mark.parametrize("name", ["tiny"])
def test_tiny_config_loss_is_sane(name):
    cfg = workloads.CONFIGS[name]
    inp = workloads.make_inputs(cfg, seed=0)
    out = oracle.fused_topk_kl(inp["hidden"], inp["W"], inp["topk_idx"],
                               inp["topk_logit"], cfg.T)
    # the student is near uniform (|z| ~ 0.3), so the loss is close to
    # log V minus the teacher's mean entropy
    assert 0 < out["loss"] < np.log(cfg.V) + 1
    assert np.isfinite(out["grad_hidden"]).all() and np.isfinite(out["grad_W"]).all()
    assert np.abs(out["grad_W"].sum(axis=0)).max() < 1e-12


def impl_m(h, W, idx, lg, T, mask):
    return oracle.fused_topk_kl(h, W, idx, lg, T, mask=mask)


@pytest.mark.parametrize("T", [1.0, 2.5])
@pytest.mark.parametrize("pin", pins.MASK_PINS, ids=lambda f: f.__name__)
def test_mask_pin(pin, T):
    pin(impl_m, T)
