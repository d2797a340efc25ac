"""Error paths on the GPU, none of which faults or hangs the device.

Bad ids are only ever compared by the kernels, never used as addresses,
so an id outside [0, V) is safe to pass and must come back as
KD_ERR_INDEX.  The timeout path uses the library's own hook: one GEMM's
epilogue waits, with a 50 ms limit, on a barrier that nothing completes;
the bounded wait gives up, the CTA drains and frees TMEM, and the call
returns KD_ERR_TIMEOUT.  A normal call afterwards checks that the context
is still usable.
"""
import time

import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import workloads
from tests.gpu_util import ensure_lib, run_debug, to_device

pytestmark = pytest.mark.gpu

CFG = workloads.custom("err", N=200, H=64, V=512, K=8, T=1.0, chunk=128)


def _inputs(seed=0):
    ensure_lib()
    return to_device(workloads.make_inputs(CFG, seed=seed))


@pytest.mark.parametrize("bad", [-1, 512, 1 << 30])
def test_out_of_range_id_is_reported(bad):
    inp = _inputs()
    inp["topk_idx"][17, 3] = bad
    with pytest.raises(kd.KdError) as ei:
        run_debug(inp, CFG.T, CFG.chunk)
    assert ei.value.name == "KD_ERR_INDEX"


@pytest.mark.parametrize("bad", [-1, 512, 1 << 30])
def test_out_of_range_id_is_reported_with_stored_logits(bad):
    # the stored-logits backward rewrites dZ at the cached ids; it skips an
    # id outside [0, V) instead of addressing the logits with it
    inp = _inputs()
    inp["topk_idx"][150, 0] = bad
    N, H = inp["hidden"].shape
    V, K = inp["W"].shape[0], inp["topk_idx"].shape[1]
    flags = kd.KD_FLAG_STORE_LOGITS
    ws = torch.empty(kd.kd_topk_kl_workspace_size_flags(N, H, V, K, CFG.chunk, flags),
                     dtype=torch.uint8, device="cuda")
    gh = torch.empty((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    with pytest.raises(kd.KdError) as ei:
        kd.kd_topk_kl_fwd_bwd_flags(inp["hidden"], inp["W"], inp["topk_idx"],
                                    inp["topk_logit"], None, CFG.T, CFG.chunk, flags, gh, gW, ws)
    assert ei.value.name == "KD_ERR_INDEX"
    torch.cuda.synchronize()


@pytest.mark.parametrize("site", [1, 2, 3, 4], ids=["fwd", "recompute", "grad_hidden", "grad_W"])
def test_injected_wait_times_out_and_context_survives(site):
    # each GEMM kind (its epilogue, staging and stores) takes the abort and
    # drain path of a CTA pair once
    inp = _inputs()
    t0 = time.time()
    with pytest.raises(kd.KdError) as ei:
        run_debug(inp, CFG.T, CFG.chunk, timeout_ns=50_000_000, inject=site)
    assert ei.value.name == "KD_ERR_TIMEOUT"
    assert time.time() - t0 < 30
    ok = run_debug(inp, CFG.T, CFG.chunk)
    assert np.isfinite(ok["loss"])
    assert np.array_equal(ok["found"], inp["topk_idx"].cpu().numpy())


def test_host_pointer_is_rejected():
    ensure_lib()
    inp = _inputs()
    host_hidden = inp["hidden"].cpu()
    gh = torch.empty((CFG.N, CFG.H), dtype=torch.float32, device="cuda")
    gW = torch.empty((CFG.V, CFG.H), dtype=torch.float32, device="cuda")
    ws = kd.alloc_workspace(CFG.N, CFG.H, CFG.V, CFG.K, CFG.chunk, device="cuda")
    L = kd.lib()
    import ctypes
    loss = ctypes.c_float()
    st = L.kd_topk_kl_fwd_bwd_ex(host_hidden.data_ptr(), inp["W"].data_ptr(),
                                 inp["topk_idx"].data_ptr(), inp["topk_logit"].data_ptr(),
                                 CFG.N, CFG.H, CFG.V, CFG.K, CFG.T, CFG.chunk,
                                 ctypes.addressof(loss), gh.data_ptr(), gW.data_ptr(),
                                 ws.data_ptr(), ws.numel(), None)
    assert st == 1


def test_small_workspace_is_oom_status():
    inp = _inputs()
    gh = torch.empty((CFG.N, CFG.H), dtype=torch.float32, device="cuda")
    gW = torch.empty((CFG.V, CFG.H), dtype=torch.float32, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(kd.KdError) as ei:
        kd.kd_topk_kl_fwd_bwd_ex(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                                 CFG.T, CFG.chunk, gh, gW, ws)
    assert ei.value.name == "KD_ERR_OOM"


def test_binding_checks_the_buffers_the_library_writes():
    # the library sees only addresses: a gradient buffer of the wrong dtype,
    # shape or layout, or on the host, is refused before anything is launched
    inp = _inputs()
    N, H = inp["hidden"].shape
    V = inp["W"].shape[0]
    ws = kd.alloc_workspace(CFG.N, CFG.H, CFG.V, CFG.K, CFG.chunk, device="cuda")
    gh = torch.empty((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    args = (inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"], CFG.T, CFG.chunk)
    with pytest.raises(TypeError):
        kd.kd_topk_kl_fwd_bwd_ex(*args, gh.to(torch.bfloat16), gW, ws)
    with pytest.raises(ValueError):
        kd.kd_topk_kl_fwd_bwd_ex(*args, gh, gW[:-8], ws)
    with pytest.raises(ValueError):
        kd.kd_topk_kl_fwd_bwd_ex(*args, torch.empty((H, N), device="cuda").t(), gW, ws)
    with pytest.raises(ValueError):
        kd.kd_topk_kl_fwd_bwd_ex(*args, gh, gW.cpu(), ws)
    with pytest.raises(ValueError):
        kd.kd_topk_kl_fwd_bwd_flags(*args[:4], None, CFG.T, CFG.chunk, 0, gh, gW, ws.cpu())
    loss = kd.kd_topk_kl_fwd_bwd_ex(*args, gh, gW, ws)   # the same call with good buffers
    assert np.isfinite(loss)
