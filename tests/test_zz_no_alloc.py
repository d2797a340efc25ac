"""The allocation-free entry point against the ordinary one (GPU).

``kd_topk_kl_fwd_bwd_noalloc`` serves callers that may not allocate device
memory themselves (a host framework that owns all allocations, or a runtime
whose memory is already fully reserved by its own pool): it runs the same
loss with the library's built-in 64 MiB scratch buffer instead of a caller
workspace.  These tests call it through the C ABI twice in a row, on two
different inputs, and compare each result with ``kd_topk_kl_fwd_bwd_ex`` on
the same inputs, within the tolerances the parity tests use.  The file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import workloads
from tests.gpu_util import GRAD_REL_L2, LOSS_RTOL, ensure_lib, rel_l2, to_device

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    L = ensure_lib()
    f = L.kd_topk_kl_fwd_bwd_noalloc
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, f32, i32, vp, vp, vp, vp]
    f.restype = i32
    return f


def _call_noalloc(f, inp, T, chunk):
    h, W, idx, lg = inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"]
    N, H = h.shape
    V, K = W.shape[0], idx.shape[1]
    gh = torch.full((N, H), float("nan"), dtype=torch.float32, device="cuda")
    gW = torch.full((V, H), float("nan"), dtype=torch.float32, device="cuda")
    loss = ctypes.c_float(float("nan"))
    torch.cuda.synchronize()
    st = f(h.data_ptr(), W.data_ptr(), idx.data_ptr(), lg.data_ptr(), N, H, V, K, T, chunk,
           ctypes.addressof(loss), gh.data_ptr(), gW.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    return st, loss.value, gh.cpu().numpy(), gW.cpu().numpy()


def _reference(inp, T, chunk):
    loss, gh, gW = kd.fwd_bwd(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                              T, chunk)
    torch.cuda.synchronize()
    return loss, gh.cpu().numpy(), gW.cpu().numpy()


CASES = [
    workloads.custom("na_ragged", N=300, H=200, V=1000, K=7, T=0.7, chunk=128),
    workloads.custom("na_mid", N=640, H=576, V=8192, K=100, T=1.0, chunk=256,
                     hidden_rms_norm=True, teacher="zipf"),
]


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    f = _noalloc_fn()
    for seed, cfg in enumerate(CASES):
        inp = to_device(workloads.make_inputs(cfg, seed=11 + seed))
        st, loss, gh, gW = _call_noalloc(f, inp, cfg.T, cfg.chunk)
        assert st == 0, kd.kd_status_string(st)
        ref_loss, ref_gh, ref_gW = _reference(inp, cfg.T, cfg.chunk)
        assert abs(loss - ref_loss) <= LOSS_RTOL * abs(ref_loss), (loss, ref_loss)
        assert rel_l2(gh, ref_gh) <= GRAD_REL_L2
        assert rel_l2(gW, ref_gW) <= GRAD_REL_L2
        assert np.isfinite(gh).all() and np.isfinite(gW).all()


def test_repeated_call_on_same_inputs_is_unchanged():
    f = _noalloc_fn()
    cfg = CASES[0]
    inp = to_device(workloads.make_inputs(cfg, seed=3))
    a = _call_noalloc(f, inp, cfg.T, cfg.chunk)
    b = _call_noalloc(f, inp, cfg.T, cfg.chunk)
    assert a[0] == 0 and b[0] == 0
    assert abs(a[1] - b[1]) <= LOSS_RTOL * abs(a[1])
    assert rel_l2(b[2], a[2]) <= GRAD_REL_L2 and rel_l2(b[3], a[3]) <= GRAD_REL_L2


def test_oversized_problem_is_rejected_before_any_launch():
    f = _noalloc_fn()
    N, H, V, K, chunk = 4096, 2880, 201088, 100, 128
    assert kd.kd_topk_kl_workspace_size(N, H, V, K, chunk) > 64 << 20
    inp = {"hidden": torch.zeros((N, H), dtype=torch.bfloat16, device="cuda"),
           "W": torch.zeros((V, H), dtype=torch.bfloat16, device="cuda"),
           "topk_idx": torch.zeros((N, K), dtype=torch.int32, device="cuda"),
           "topk_logit": torch.zeros((N, K), dtype=torch.float32, device="cuda")}
    st, *_ = _call_noalloc(f, inp, 1.0, chunk)
    assert kd.STATUS_NAMES[st] == "KD_ERR_TOO_LARGE"
