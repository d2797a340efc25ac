"""Helpers shared by the GPU tests: build/load the library, run the CUDA
path with its debug exports, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import chunked_top_kl_gemm_b300 as kd
from chunked_top_kl_gemm_b300 import _build

# Tolerances of the GPU path against the float64 oracle (bf16 inputs, fp32
# tensor-core accumulation, bf16 dZ scratch).
LOSS_RTOL = 1e-3
GRAD_REL_L2 = 2e-2
LSE_ATOL = 2e-4          # lse ~ log V ~ 8..13, fp32 accumulation over H
ZG_RTOL = 1e-3           # z at the cached ids, relative to max |z| of the row set


def ensure_lib():
    _build.build()
    return kd.lib()


def rel_l2(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def to_device(inp: dict, dev="cuda") -> dict:
    return {k: v.to(dev).contiguous() for k, v in inp.items()}


def run_debug(inp: dict, T: float, chunk: int, timeout_ns: int = 0, inject: int = 0):
    """Run the CUDA path with every debug export; returns numpy results."""
    h, W, idx, lg = inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"]
    N, H = h.shape
    V = W.shape[0]
    K = idx.shape[1]
    dev = h.device
    gh = torch.full((N, H), float("nan"), dtype=torch.float32, device=dev)
    gW = torch.full((V, H), float("nan"), dtype=torch.float32, device=dev)
    ws = kd.alloc_workspace(N, H, V, K, chunk, device=dev)
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    zg = torch.full((N, K), float("nan"), dtype=torch.float32, device=dev)
    found = torch.full((N, K), -1, dtype=torch.int32, device=dev)
    loss = kd.kd_topk_kl_debug(h, W, idx, lg, T, chunk, gh, gW, ws, lse=lse, zg=zg,
                               found_idx=found, timeout_ns=timeout_ns, inject_timeout=inject)
    torch.cuda.synchronize()
    return {"loss": loss, "grad_hidden": gh.cpu().numpy(), "grad_W": gW.cpu().numpy(),
            "lse": lse.cpu().numpy(), "zg": zg.cpu().numpy(), "found": found.cpu().numpy()}


def assert_parity(got: dict, want: dict, idx: np.ndarray, check_grads=True):
    assert np.array_equal(got["found"], idx), "gathered ids differ from the cached ids"
    assert abs(got["loss"] - want["loss"]) <= LOSS_RTOL * abs(want["loss"]) + 1e-6, \
        (got["loss"], want["loss"])
    np.testing.assert_allclose(got["lse"], want["lse"], rtol=0, atol=LSE_ATOL)
    zscale = max(np.abs(want["zg"]).max(), 1e-6)
    assert np.abs(got["zg"] - want["zg"]).max() <= ZG_RTOL * zscale
    if check_grads:
        for key in ("grad_hidden", "grad_W"):
            assert np.isfinite(got[key]).all(), key
            err = rel_l2(got[key], want[key])
            assert err <= GRAD_REL_L2, (key, err)
