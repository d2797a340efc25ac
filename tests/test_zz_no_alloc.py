"""The allocation-free entry point against the ordinary one (GPU).

``kd_topk_kl_fwd_bwd_noalloc`` serves callers that may not allocate device
memory themselves (a host framework that owns all allocations, or a runtime
whose memory is already fully reserved by its own pool): it runs the same
loss with the library's built-in 64 MiB scratch buffer instead of a caller
workspace.  It runs the same plan and kernels as ``kd_topk_kl_fwd_bwd_ex``,
whose results are deterministic, so the two must agree bit for bit.  These
tests call it through the C ABI several times in a row, on inputs of
different sizes (a larger problem first, so a smaller one runs over the
scratch contents a larger layout left behind), and compare every result
with ``kd_topk_kl_fwd_bwd_ex`` on the same inputs.  They also check that a
call allocates no device memory.  The file is named so that pytest
collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import workloads
from tests.gpu_util import ensure_lib, to_device

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    L = ensure_lib()
    f = L.kd_topk_kl_fwd_bwd_noalloc
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, f32, i32, vp, vp, vp, vp]
    f.restype = i32
    return f


def _outputs(inp):
    N, H = inp["hidden"].shape
    V = inp["W"].shape[0]
    gh = torch.full((N, H), float("nan"), dtype=torch.float32, device="cuda")
    gW = torch.full((V, H), float("nan"), dtype=torch.float32, device="cuda")
    return gh, gW


def _raw_call(f, inp, T, chunk, gh, gW):
    h, W, idx, lg = inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"]
    N, H = h.shape
    V, K = W.shape[0], idx.shape[1]
    loss = ctypes.c_float(float("nan"))
    st = f(h.data_ptr(), W.data_ptr(), idx.data_ptr(), lg.data_ptr(), N, H, V, K, T, chunk,
           ctypes.addressof(loss), gh.data_ptr(), gW.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    return st, loss.value


def _call_noalloc(f, inp, T, chunk):
    gh, gW = _outputs(inp)
    torch.cuda.synchronize()
    st, loss = _raw_call(f, inp, T, chunk, gh, gW)
    return st, loss, gh.cpu().numpy(), gW.cpu().numpy()


def _reference(inp, T, chunk):
    loss, gh, gW = kd.fwd_bwd(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                              T, chunk)
    torch.cuda.synchronize()
    return loss, gh.cpu().numpy(), gW.cpu().numpy()


def _assert_same_bits(got, ref):
    st, loss, gh, gW = got
    ref_loss, ref_gh, ref_gW = ref
    assert st == 0, kd.kd_status_string(st)
    assert np.float32(loss).tobytes() == np.float32(ref_loss).tobytes(), (loss, ref_loss)
    assert np.array_equal(gh, ref_gh), float(np.abs(gh - ref_gh).max())
    assert np.array_equal(gW, ref_gW), float(np.abs(gW - ref_gW).max())


# the larger layout first: the ragged problem's last chunk then runs over
# scratch that the larger problem's dZ and partials filled
CASES = [
    workloads.custom("na_mid", N=640, H=576, V=8192, K=100, T=1.0, chunk=256,
                     hidden_rms_norm=True, teacher="zipf"),
    workloads.custom("na_ragged", N=300, H=200, V=1000, K=7, T=0.7, chunk=128),
]


def test_calls_in_a_row_match_the_workspace_entry_point_bitwise():
    f = _noalloc_fn()
    for seed, cfg in enumerate(CASES):
        inp = to_device(workloads.make_inputs(cfg, seed=11 + seed))
        got = _call_noalloc(f, inp, cfg.T, cfg.chunk)
        _assert_same_bits(got, _reference(inp, cfg.T, cfg.chunk))
        assert np.isfinite(got[2]).all() and np.isfinite(got[3]).all()


def test_after_a_larger_problem_the_result_is_unchanged():
    # the same small problem before and after a larger one that leaves other
    # contents in the shared scratch: both results equal the workspace entry
    # point's bit for bit
    f = _noalloc_fn()
    small, large = CASES[1], CASES[0]
    inp = to_device(workloads.make_inputs(small, seed=3))
    ref = _reference(inp, small.T, small.chunk)
    _assert_same_bits(_call_noalloc(f, inp, small.T, small.chunk), ref)
    big = to_device(workloads.make_inputs(large, seed=4))
    assert _call_noalloc(f, big, large.T, large.chunk)[0] == 0
    _assert_same_bits(_call_noalloc(f, inp, small.T, small.chunk), ref)
    _assert_same_bits(_call_noalloc(f, inp, small.T, small.chunk), ref)


def test_a_call_allocates_no_device_memory():
    f = _noalloc_fn()
    cfg = CASES[0]
    inp = to_device(workloads.make_inputs(cfg, seed=5))
    gh, gW = _outputs(inp)
    assert _raw_call(f, inp, cfg.T, cfg.chunk, gh, gW)[0] == 0   # warm: code and buffer loaded
    torch.cuda.synchronize()
    stats0 = torch.cuda.memory_stats()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert _raw_call(f, inp, cfg.T, cfg.chunk, gh, gW)[0] == 0
    torch.cuda.synchronize()
    stats1 = torch.cuda.memory_stats()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    for key in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key


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
