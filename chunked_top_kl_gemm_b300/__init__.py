"""Python binding of ``libkdtopk.so``: the fused chunked top-K KL loss on B300.

Argument marshalling only.  Every step of the loss runs in the library's
CUDA kernels; PyTorch provides device memory and the current stream.  If
the library is missing this module raises on first use -- there is no CPU
fallback.

The C entry points are exposed under the same names
(``kd_topk_kl_fwd_bwd``, ``kd_topk_kl_fwd_bwd_ex``,
``kd_topk_kl_workspace_size``, ``kd_topk_kl_debug``, ``kd_gemm_bf16_test``,
``kd_status_string``); ``fwd_bwd`` is the convenience wrapper that
allocates outputs and the workspace with torch.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkdtopk.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "kd_topk_kl.h")

KD_OK = 0
KD_ERR_INDEX = 3
KD_ERR_TIMEOUT = 6
KD_FLAG_ACCUMULATE = 1
KD_FLAG_STORE_LOGITS = 2
KD_FLAG_MIN_SCRATCH = 4
STATUS_NAMES = {
    0: "KD_OK", 1: "KD_ERR_INVALID_ARG", 2: "KD_ERR_ALIGNMENT", 3: "KD_ERR_INDEX",
    4: "KD_ERR_OOM", 5: "KD_ERR_CUDA", 6: "KD_ERR_TIMEOUT", 7: "KD_ERR_NOT_IMPLEMENTED",
    8: "KD_ERR_TOO_LARGE",
}


class KdError(RuntimeError):
    """A non-KD_OK status from the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{what}: {self.name} ({kd_status_string(status)})"
                         + (f" [{last_cuda_error()}]" if status == 5 else ""))


class _DebugOpts(ctypes.Structure):
    _fields_ = [("lse", ctypes.c_void_p), ("zg", ctypes.c_void_p),
                ("found_idx", ctypes.c_void_p), ("timeout_ns", ctypes.c_uint64),
                ("inject_timeout", ctypes.c_int), ("loss_rows", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load ``libkdtopk.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m chunked_top_kl_gemm_b300._build` (there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                             ctypes.c_float, ctypes.c_size_t)
    common = [vp, vp, vp, vp, i64, i32, i32, i32, f32, i32, vp, vp, vp]
    L.kd_topk_kl_fwd_bwd.argtypes = common
    L.kd_topk_kl_fwd_bwd.restype = i32
    L.kd_topk_kl_fwd_bwd_ex.argtypes = common + [vp, sz, vp]
    L.kd_topk_kl_fwd_bwd_ex.restype = i32
    L.kd_topk_kl_fwd_bwd_masked.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, i32,
                                             i32, vp, vp, vp, vp, sz, vp]
    L.kd_topk_kl_fwd_bwd_masked.restype = i32
    L.kd_topk_kl_fwd_bwd_flags.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, i32,
                                            ctypes.c_uint, vp, vp, vp, vp, sz, vp]
    L.kd_topk_kl_fwd_bwd_flags.restype = i32
    L.kd_topk_kl_fwd_bwd_sharded.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, i32,
                                              ctypes.c_uint, i64, vp, vp, vp, vp, sz, vp]
    L.kd_topk_kl_fwd_bwd_sharded.restype = i32
    L.kd_topk_kl_fwd_bwd_async.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, i32,
                                            ctypes.c_uint, vp, vp, vp, vp, vp, sz, vp]
    L.kd_topk_kl_fwd_bwd_async.restype = i32
    L.kd_topk_kl_workspace_size_flags.argtypes = [i64, i32, i32, i32, i32, ctypes.c_uint]
    L.kd_topk_kl_workspace_size_flags.restype = sz
    L.kd_topk_cache_workspace_size.argtypes = [i64, i32, i32, i32, i32]
    L.kd_topk_cache_workspace_size.restype = sz
    L.kd_topk_cache_build.argtypes = [vp, vp, i64, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    L.kd_topk_cache_build.restype = i32
    L.kd_topk_kl_debug.argtypes = common + [vp, sz, vp, ctypes.POINTER(_DebugOpts)]
    L.kd_topk_kl_debug.restype = i32
    L.kd_topk_kl_workspace_size.argtypes = [i64, i32, i32, i32, i32]
    L.kd_topk_kl_workspace_size.restype = sz
    L.kd_gemm_bf16_test.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp]
    L.kd_gemm_bf16_test.restype = i32
    L.kd_status_string.argtypes = [i32]
    L.kd_status_string.restype = ctypes.c_char_p
    L.kd_last_cuda_error.argtypes = []
    L.kd_last_cuda_error.restype = ctypes.c_char_p
    L.kd_abi_version.argtypes = []
    L.kd_abi_version.restype = i32
    L.kd_build_id.argtypes = []
    L.kd_build_id.restype = ctypes.c_char_p
    L.kd_profile_enable.argtypes = [i32]
    L.kd_profile_enable.restype = None
    L.kd_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_longlong), i32]
    L.kd_profile_read.restype = i32
    L.kd_profile_kind_name.argtypes = [i32]
    L.kd_profile_kind_name.restype = ctypes.c_char_p
    _check_build_id(L)
    _lib = L
    return L


def _check_build_id(L) -> None:
    """Refuse a library built from other sources than the ones beside it
    (it would run code that is not in the tree)."""
    from . import _build
    if not os.path.isdir(_build.CSRC):
        return                      # installed without sources: nothing to compare
    built = L.kd_build_id().decode()
    want = _build.source_hash()
    if built != want:
        raise RuntimeError(
            f"{LIB_PATH} was built from other sources (build id {built}, sources {want}): "
            "rebuild it with `python -m chunked_top_kl_gemm_b300._build`")


def build_id() -> str:
    """The source hash compiled into the loaded library."""
    return lib().kd_build_id().decode()


def header_functions() -> list:
    """Names of the functions ``include/kd_topk_kl.h`` declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kd_[a-z0-9_]+)\s*\(", text)))


def kd_status_string(status: int) -> str:
    return lib().kd_status_string(int(status)).decode()


def last_cuda_error() -> str:
    return lib().kd_last_cuda_error().decode()


def abi_version() -> int:
    return lib().kd_abi_version()


def _check(status: int, what: str):
    if status != KD_OK:
        raise KdError(status, what)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _on_device(t):
    """Make t's device current for the library call (it checks pointers and
    sizes its work against the current device)."""
    import contextlib
    import torch
    if t is None or not t.is_cuda:
        return contextlib.nullcontext()
    return torch.cuda.device(t.device)


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_inputs(hidden, W, topk_idx, topk_logit):
    import torch
    if hidden.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("hidden and W must be bfloat16")
    if topk_idx.dtype != torch.int32:
        raise TypeError("topk_idx must be int32 (convert torch.topk's int64 ids with .int())")
    if topk_logit.dtype != torch.float32:
        raise TypeError("topk_logit must be float32")
    for name, t in (("hidden", hidden), ("W", W), ("topk_idx", topk_idx),
                    ("topk_logit", topk_logit)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != hidden.device:
            raise ValueError(f"{name} must be on {hidden.device}")
    N, H = hidden.shape
    V, H2 = W.shape
    if H2 != H or topk_idx.shape != topk_logit.shape or topk_idx.shape[0] != N:
        raise ValueError("shape mismatch: hidden [N,H], W [V,H], topk_* [N,K]")
    return N, H, V, topk_idx.shape[1]


def _check_out(name, t, shape, dtype, device):
    """A buffer the library writes: the library sees only its address, so its
    dtype, shape, layout and device are checked here (a smaller buffer would
    be written past its end)."""
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor of shape {tuple(shape)}")


def _check_grads(grad_hidden, grad_W, hidden, V):
    import torch
    N, H = hidden.shape
    _check_out("grad_hidden", grad_hidden, (N, H), torch.float32, hidden.device)
    _check_out("grad_W", grad_W, (V, H), torch.float32, hidden.device)


def _check_workspace(workspace, hidden):
    if workspace is None or not workspace.is_cuda or workspace.device != hidden.device \
            or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous CUDA tensor on {hidden.device}")


def kd_topk_kl_workspace_size(N: int, H: int, V: int, K: int, chunk: int) -> int:
    return int(lib().kd_topk_kl_workspace_size(N, H, V, K, chunk))


def kd_topk_kl_fwd_bwd(hidden, W, topk_idx, topk_logit, T: float, chunk: int,
                       grad_hidden, grad_W) -> float:
    """The spec entry point: default stream, self-allocated workspace.

    Writes grad_hidden / grad_W in place and returns the loss.
    """
    N, H, V, K = _check_inputs(hidden, W, topk_idx, topk_logit)
    _check_grads(grad_hidden, grad_W, hidden, V)
    loss = ctypes.c_float(0.0)
    with _on_device(hidden):
        st = lib().kd_topk_kl_fwd_bwd(_ptr(hidden), _ptr(W), _ptr(topk_idx), _ptr(topk_logit),
                                      N, H, V, K, float(T), int(chunk), ctypes.addressof(loss),
                                      _ptr(grad_hidden), _ptr(grad_W))
    _check(st, "kd_topk_kl_fwd_bwd")
    return float(loss.value)


def kd_topk_kl_fwd_bwd_ex(hidden, W, topk_idx, topk_logit, T: float, chunk: int,
                          grad_hidden, grad_W, workspace, stream=None) -> float:
    """Caller stream (default: torch's current stream) and workspace tensor."""
    N, H, V, K = _check_inputs(hidden, W, topk_idx, topk_logit)
    _check_grads(grad_hidden, grad_W, hidden, V)
    _check_workspace(workspace, hidden)
    loss = ctypes.c_float(0.0)
    with _on_device(hidden):
        st = lib().kd_topk_kl_fwd_bwd_ex(
            _ptr(hidden), _ptr(W), _ptr(topk_idx), _ptr(topk_logit), N, H, V, K, float(T),
            int(chunk), ctypes.addressof(loss), _ptr(grad_hidden), _ptr(grad_W),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_bwd_ex")
    return float(loss.value)


def _check_mask(token_mask, N):
    import torch
    if token_mask is None:
        return None
    if token_mask.dtype == torch.bool:
        token_mask = token_mask.view(torch.uint8)
    if token_mask.dtype != torch.uint8 or token_mask.shape != (N,) or not token_mask.is_cuda \
            or not token_mask.is_contiguous():
        raise ValueError("token_mask must be a contiguous uint8/bool CUDA tensor of shape [N]")
    return token_mask


def kd_topk_kl_fwd_bwd_masked(hidden, W, topk_idx, topk_logit, token_mask, T: float,
                              chunk: int, grad_hidden, grad_W, workspace, accumulate=False,
                              stream=None) -> float:
    """Per-token mask (uint8/bool [N] CUDA tensor or None) and accumulate flag."""
    import torch
    N, H, V, K = _check_inputs(hidden, W, topk_idx, topk_logit)
    token_mask = _check_mask(token_mask, N)
    _check_grads(grad_hidden, grad_W, hidden, V)
    _check_workspace(workspace, hidden)
    if token_mask is not None and token_mask.device != hidden.device:
        raise ValueError(f"token_mask must be on {hidden.device}")
    loss = ctypes.c_float(0.0)
    with _on_device(hidden):
        st = lib().kd_topk_kl_fwd_bwd_masked(
            _ptr(hidden), _ptr(W), _ptr(topk_idx), _ptr(topk_logit), _ptr(token_mask), N, H, V, K,
            float(T), int(chunk), 1 if accumulate else 0, ctypes.addressof(loss), _ptr(grad_hidden),
            _ptr(grad_W), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_bwd_masked")
    return float(loss.value)


def kd_topk_kl_workspace_size_flags(N: int, H: int, V: int, K: int, chunk: int,
                                    flags: int) -> int:
    return int(lib().kd_topk_kl_workspace_size_flags(N, H, V, K, chunk, int(flags)))


def kd_topk_kl_fwd_bwd_flags(hidden, W, topk_idx, topk_logit, token_mask, T: float, chunk: int,
                             flags: int, grad_hidden, grad_W, workspace, stream=None) -> float:
    """Mask (or None) and KD_FLAG_* flags (accumulate, store logits)."""
    N, H, V, K = _check_inputs(hidden, W, topk_idx, topk_logit)
    token_mask = _check_mask(token_mask, N)
    _check_grads(grad_hidden, grad_W, hidden, V)
    _check_workspace(workspace, hidden)
    if token_mask is not None and token_mask.device != hidden.device:
        raise ValueError(f"token_mask must be on {hidden.device}")
    loss = ctypes.c_float(0.0)
    with _on_device(hidden):
        st = lib().kd_topk_kl_fwd_bwd_flags(
            _ptr(hidden), _ptr(W), _ptr(topk_idx), _ptr(topk_logit), _ptr(token_mask), N, H, V, K,
            float(T), int(chunk), int(flags), ctypes.addressof(loss), _ptr(grad_hidden),
            _ptr(grad_W), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_bwd_flags")
    return float(loss.value)


def kd_topk_kl_fwd_bwd_sharded(hidden, W, topk_idx, topk_logit, token_mask, T: float,
                               chunk: int, flags: int, n_norm: int, grad_hidden, grad_W,
                               workspace, stream=None) -> float:
    """One shard of a batch whose mean runs over ``n_norm`` tokens: the
    returned loss and the gradients are normalised by the whole batch, so
    shards' losses and grad_W add up to the batch's (``KD_FLAG_ACCUMULATE``
    adds into grad_W on one device)."""
    N, H, V, K = _check_inputs(hidden, W, topk_idx, topk_logit)
    token_mask = _check_mask(token_mask, N)
    _check_grads(grad_hidden, grad_W, hidden, V)
    _check_workspace(workspace, hidden)
    if token_mask is not None and token_mask.device != hidden.device:
        raise ValueError(f"token_mask must be on {hidden.device}")
    loss = ctypes.c_float(0.0)
    with _on_device(hidden):
        st = lib().kd_topk_kl_fwd_bwd_sharded(
            _ptr(hidden), _ptr(W), _ptr(topk_idx), _ptr(topk_logit), _ptr(token_mask), N, H, V, K,
            float(T), int(chunk), int(flags), int(n_norm), ctypes.addressof(loss),
            _ptr(grad_hidden), _ptr(grad_W), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_bwd_sharded")
    return float(loss.value)


def kd_topk_kl_fwd_bwd_async(hidden, W, topk_idx, topk_logit, token_mask, T: float, chunk: int,
                             flags: int, loss_out, status_out, grad_hidden, grad_W, workspace,
                             stream=None) -> None:
    """Enqueue the call on ``stream`` (default: the current stream) and return
    at once; capturable in a CUDA graph.  ``loss_out`` (float32 [1]) and
    ``status_out`` (int32 [1]) are CUDA tensors the last kernel writes; read
    them after the stream has passed the call (see ``check_status``)."""
    import torch
    N, H, V, K = _check_inputs(hidden, W, topk_idx, topk_logit)
    token_mask = _check_mask(token_mask, N)
    _check_grads(grad_hidden, grad_W, hidden, V)
    _check_workspace(workspace, hidden)
    if token_mask is not None and token_mask.device != hidden.device:
        raise ValueError(f"token_mask must be on {hidden.device}")
    for name, t, dt in (("loss_out", loss_out, torch.float32), ("status_out", status_out, torch.int32)):
        if t.dtype != dt or t.numel() < 1 or not t.is_cuda or t.device != hidden.device:
            raise ValueError(f"{name} must be a {dt} CUDA tensor on {hidden.device} with at "
                             "least one element")
    with _on_device(hidden):
        st = lib().kd_topk_kl_fwd_bwd_async(
            _ptr(hidden), _ptr(W), _ptr(topk_idx), _ptr(topk_logit), _ptr(token_mask), N, H, V, K,
            float(T), int(chunk), int(flags), _ptr(loss_out), _ptr(status_out), _ptr(grad_hidden),
            _ptr(grad_W), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream))
    _check(st, "kd_topk_kl_fwd_bwd_async")


def check_status(status_out) -> None:
    """Raise KdError if an asynchronous call's device status word is not KD_OK
    (reads it: synchronises with the stream that wrote it)."""
    _check(int(status_out.reshape(-1)[0].item()), "kd_topk_kl_fwd_bwd_async (device status)")


def kd_topk_cache_workspace_size(N: int, H: int, V: int, K: int, chunk: int) -> int:
    return int(lib().kd_topk_cache_workspace_size(N, H, V, K, chunk))


def kd_topk_cache_build(hidden, W, K: int, chunk: int = 2048, *, topk_idx=None,
                        topk_logit=None, workspace=None, stream=None):
    """The offline teacher cache: (int32 ids [N,K], fp32 logits [N,K]) of the
    K largest logits of ``hidden @ W.T`` per token, decreasing, ties by id."""
    import torch
    if hidden.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("hidden and W must be bfloat16")
    if not (hidden.is_cuda and W.is_cuda and hidden.is_contiguous() and W.is_contiguous()):
        raise ValueError("hidden and W must be contiguous CUDA tensors")
    N, H = hidden.shape
    V = W.shape[0]
    dev = hidden.device
    if W.shape[1] != H or W.device != dev:
        raise ValueError("W must be [V, H] on hidden's device")
    if topk_idx is None:
        topk_idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    if topk_logit is None:
        topk_logit = torch.empty((N, K), dtype=torch.float32, device=dev)
    _check_out("topk_idx", topk_idx, (N, K), torch.int32, dev)
    _check_out("topk_logit", topk_logit, (N, K), torch.float32, dev)
    if workspace is None:
        nbytes = kd_topk_cache_workspace_size(N, H, V, K, chunk)
        if nbytes == 0:
            raise KdError(1, "kd_topk_cache_workspace_size")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _check_workspace(workspace, hidden)
    with _on_device(hidden):
        st = lib().kd_topk_cache_build(_ptr(hidden), _ptr(W), N, H, V, int(K), int(chunk),
                                       _ptr(topk_idx), _ptr(topk_logit), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream_handle(stream))
    _check(st, "kd_topk_cache_build")
    return topk_idx, topk_logit


def kd_topk_kl_debug(hidden, W, topk_idx, topk_logit, T: float, chunk: int, grad_hidden,
                     grad_W, workspace, *, lse=None, zg=None, found_idx=None, loss_rows=None,
                     timeout_ns: int = 0, inject_timeout: bool = False, stream=None) -> float:
    """``kd_topk_kl_fwd_bwd_ex`` plus the debug exports (fp32 ``lse`` [N], fp32 ``zg``
    [N,K], int32 ``found_idx`` [N,K] pre-filled by the caller, float64 ``loss_rows`` [N])
    and the bounded-wait test hook."""
    import torch
    N, H, V, K = _check_inputs(hidden, W, topk_idx, topk_logit)
    _check_grads(grad_hidden, grad_W, hidden, V)
    _check_workspace(workspace, hidden)
    for name, t, shape, dt in (("lse", lse, (N,), torch.float32), ("zg", zg, (N, K), torch.float32),
                               ("found_idx", found_idx, (N, K), torch.int32),
                               ("loss_rows", loss_rows, (N,), torch.float64)):
        if t is not None:
            _check_out(name, t, shape, dt, hidden.device)
    # inject_timeout: False / True (= 1, the forward GEMM) or 1..4 (forward,
    # recompute, grad_hidden, grad_W GEMM of the first chunk)
    opts = _DebugOpts(_ptr(lse) or None, _ptr(zg) or None, _ptr(found_idx) or None,
                      int(timeout_ns), int(inject_timeout), _ptr(loss_rows) or None)
    loss = ctypes.c_float(0.0)
    with _on_device(hidden):
        st = lib().kd_topk_kl_debug(
            _ptr(hidden), _ptr(W), _ptr(topk_idx), _ptr(topk_logit), N, H, V, K, float(T),
            int(chunk), ctypes.addressof(loss), _ptr(grad_hidden), _ptr(grad_W),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream),
            ctypes.byref(opts))
    _check(st, "kd_topk_kl_debug")
    return float(loss.value)


def kd_gemm_bf16_test(A, B, a_mn: bool, b_mn: bool, bn: int = 0, pair: bool = False,
                      stream=None):
    """C = A_op * B_op^T in fp32 (test entry of the tensor-core core); ``pair``
    selects the CTA-pair (2-CTA MMA) form the loss uses."""
    import torch
    if a_mn:
        K, M = A.shape
    else:
        M, K = A.shape
    if b_mn:
        K2, N = B.shape
    else:
        N, K2 = B.shape
    if K2 != K:
        raise ValueError("K mismatch")
    C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    with _on_device(A):
        st = lib().kd_gemm_bf16_test(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(bool(a_mn)),
                                     int(bool(b_mn)), int(bn), int(pair),
                                     _stream_handle(stream))
    _check(st, "kd_gemm_bf16_test")
    return C


def alloc_workspace(N: int, H: int, V: int, K: int, chunk: int, device=None):
    import torch
    dev = torch.device(device) if device is not None else None
    if dev is not None and dev.type == "cuda":
        with torch.cuda.device(dev):
            nbytes = kd_topk_kl_workspace_size(N, H, V, K, chunk)
    else:
        nbytes = kd_topk_kl_workspace_size(N, H, V, K, chunk)
    if nbytes == 0:
        raise KdError(1, "kd_topk_kl_workspace_size")
    # torch allocations are at least 512-byte aligned
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def fwd_bwd(hidden, W, topk_idx, topk_logit, T: float = 1.0, chunk: int = 2048, *,
            workspace=None, grad_hidden=None, grad_W=None, stream=None, token_mask=None,
            accumulate: bool = False):
    """Loss (float) and fp32 grad_hidden [N,H], grad_W [V,H] of the top-K KL.

    Outputs and the workspace are allocated with torch on hidden's device
    unless given.  ``token_mask`` restricts the mean to the valid tokens;
    ``accumulate`` adds into the given gradient tensors.
    """
    import torch
    N, H, V, K = _check_inputs(hidden, W, topk_idx, topk_logit)
    dev = hidden.device
    if accumulate and (grad_hidden is None or grad_W is None):
        raise ValueError("accumulate=True needs grad_hidden and grad_W to add into")
    if grad_hidden is None:
        grad_hidden = torch.empty((N, H), dtype=torch.float32, device=dev)
    if grad_W is None:
        grad_W = torch.empty((V, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(N, H, V, K, chunk, device=dev)
    if token_mask is None and not accumulate:
        loss = kd_topk_kl_fwd_bwd_ex(hidden, W, topk_idx, topk_logit, T, chunk, grad_hidden,
                                     grad_W, workspace, stream=stream)
    else:
        loss = kd_topk_kl_fwd_bwd_masked(hidden, W, topk_idx, topk_logit, token_mask, T, chunk,
                                         grad_hidden, grad_W, workspace, accumulate=accumulate,
                                         stream=stream)
    return loss, grad_hidden, grad_W


def kd_profile_enable(on: bool) -> None:
    """Start (and reset) or stop the library's per-kernel event timing."""
    lib().kd_profile_enable(1 if on else 0)


def kd_profile_read() -> dict:
    """{kernel kind: (total_ms, launches)} accumulated while profiling was on."""
    L = lib()
    n = L.kd_profile_read(None, None, 0)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_longlong * n)()
    L.kd_profile_read(ms, cnt, n)
    return {L.kd_profile_kind_name(i).decode(): (float(ms[i]), int(cnt[i])) for i in range(n)}
