"""The C ABI library loads and exports what its header declares (CPU only).

No compute call is made here: only symbol lookup, status strings, the
workspace planner and argument checks that fail before any CUDA call.
"""
import ctypes

import pytest

import chunked_top_kl_gemm_b300 as kd
from chunked_top_kl_gemm_b300 import _build


@pytest.fixture(scope="module")
def L():
    _build.build()
    return kd.lib()


def test_every_declared_function_is_exported(L):
    names = kd.header_functions()
    assert "kd_topk_kl_fwd_bwd" in names and "kd_topk_kl_fwd_bwd_ex" in names
    for name in names:
        assert hasattr(L, name), name


def test_library_is_built_from_the_sources_in_the_tree(L):
    # the build id compiled into the library is the hash of the sources now
    assert kd.build_id() == _build.source_hash()
    assert not _build.stale()


def test_status_strings(L):
    for code in range(8):
        assert kd.kd_status_string(code)
    assert kd.kd_status_string(0) == "ok"
    assert kd.abi_version() >= 1


def test_workspace_size_scales_with_chunk_not_tokens(L):
    # scratch is chunk x V (bf16) plus O(N K) teacher tables: doubling N at a
    # fixed chunk adds only the per-token tables
    V, H, K = 201088, 2880, 100
    a = kd.kd_topk_kl_workspace_size(32768, H, V, K, 2048)
    b = kd.kd_topk_kl_workspace_size(65536, H, V, K, 2048)
    assert a > 2 * 2048 * V
    assert b - a < 32768 * (K * 12 + 8 * 3) + 4096
    c = kd.kd_topk_kl_workspace_size(32768, H, V, K, 4096)
    assert c - a >= 2 * 2048 * V


@pytest.mark.parametrize("args", [
    (0, 256, 4096, 16, 64),      # N = 0
    (16, 250, 4096, 16, 64),     # H % 8
    (16, 256, 4090, 16, 64),     # V % 8
    (16, 256, 4096, 0, 64),      # K = 0
    (16, 256, 64, 65, 64),       # K > V
    (16, 256, 4096, 16, 0),      # chunk = 0
])
def test_workspace_size_rejects_bad_sizes(L, args):
    assert kd.kd_topk_kl_workspace_size(*args) == 0


def _call(L, ptrs, N=16, H=64, V=128, K=4, T=1.0, chunk=128, loss=True):
    out = ctypes.c_float(0)
    h, w, i, l, gh, gw = ptrs
    return L.kd_topk_kl_fwd_bwd(h, w, i, l, N, H, V, K, T, chunk,
                                ctypes.addressof(out) if loss else None, gh, gw)


GOOD = (0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000)


@pytest.mark.parametrize("which", range(6))
def test_null_pointer_is_invalid_arg(L, which):
    ptrs = list(GOOD)
    ptrs[which] = None
    assert _call(L, ptrs) == 1


def test_null_loss_is_invalid_arg(L):
    assert _call(L, GOOD, loss=False) == 1


@pytest.mark.parametrize("kw", [dict(N=0), dict(H=12), dict(V=100), dict(K=0), dict(K=129),
                                dict(chunk=0), dict(T=0.0), dict(T=-1.0),
                                dict(T=float("inf")), dict(T=float("nan"))])
def test_bad_sizes_are_invalid_arg(L, kw):
    assert _call(L, GOOD, **kw) == 1


@pytest.mark.parametrize("which", [0, 1, 4, 5])
def test_misaligned_tma_pointer_is_alignment_error(L, which):
    ptrs = list(GOOD)
    ptrs[which] += 8
    assert _call(L, ptrs) == 2


def _call_async(L, ptrs, loss_dev=0x70000, status_dev=0x80000, N=16, H=64, V=128, K=4):
    h, w, i, l, gh, gw = ptrs
    return L.kd_topk_kl_fwd_bwd_async(h, w, i, l, None, N, H, V, K, 1.0, 128, 0, loss_dev,
                                      status_dev, gh, gw, 0x90000, 1 << 30, None)


def test_async_entry_checks_arguments_before_enqueueing(L):
    assert _call_async(L, GOOD, loss_dev=None) == 1
    ptrs = list(GOOD)
    ptrs[0] = None
    assert _call_async(L, ptrs) == 1
    ptrs = list(GOOD)
    ptrs[4] += 8
    assert _call_async(L, ptrs) == 2
    assert _call_async(L, GOOD, N=0) == 1


def test_sharded_entry_checks_its_normaliser_and_arguments(L):
    h, w, i, l, gh, gw = GOOD
    out = ctypes.c_float(0)

    def call(n_norm, hidden=h, N=16):
        return L.kd_topk_kl_fwd_bwd_sharded(hidden, w, i, l, None, N, 64, 128, 4, 1.0, 128, 0,
                                            n_norm, ctypes.addressof(out), gh, gw, 0x90000,
                                            1 << 30, None)
    assert call(0) == 1 and call(-5) == 1
    assert call(32, hidden=None) == 1
    assert call(32, N=0) == 1


def test_flags_outside_the_defined_set_are_rejected(L):
    for bad in (8, 16, 1 << 31):
        assert L.kd_topk_kl_workspace_size_flags(16, 64, 128, 4, 128, bad) == 0
    assert L.kd_topk_kl_workspace_size_flags(16, 64, 128, 4, 128, kd.KD_FLAG_MIN_SCRATCH) > 0
