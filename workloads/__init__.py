"""Seeded synthetic inputs for the fused top-K KL loss.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It draws inputs only: student hidden states, the LM-head
weight and an offline top-K teacher cache. It contains none of the loss's
arithmetic (no softmax, no logsumexp, no KL, no gradient).

The pages (Multiverse Computing, "Efficient Knowledge Distillation for LLMs:
Offline Top-K Logits and a Fused Chunked KL Loss", news coverage) give no
shapes for their isolated output-projection benchmark (glonce.com, body) and
no dataset is available, so each configuration stands in for one of the
pages' workloads with synthetic values of the stated shape:

* ``tiny``      -- small case the oracle finishes in well under a second.
* ``llama3b``   -- a Llama-3-like head (H=3072, V=128,256) at 8K context,
                   standing in for the pages' 8K Llama comparison.
* ``gptoss32k`` -- a GPT-OSS-like head (H=2880, V=201,088) at 32,768 tokens,
                   the context of the pages' GPT-OSS 20B run and of the
                   32K row of the isolated benchmark.
* ``long64k``   -- 65,536 tokens at T=2 with 10% near-one-hot teachers.
* ``ext256k``   -- 262,144 tokens, the longest row of the isolated benchmark.

The cache format follows the pages' description of top-K caching (epoka.news,
"The two proposed changes"; ainewsbank.com, "Two changes remove different
bottlenecks"): per token, K teacher token ids and their K logits.  Here ids
are int32 and distinct within a row, logits are fp32 and sorted in
descending order, paired with the ids in order.

Hidden states and W are drawn in fp32 and rounded to bf16 (round to nearest
even, by ``Tensor.to(torch.bfloat16)``); every consumer reads the rounded
values.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    N: int          # tokens
    H: int          # hidden size
    V: int          # vocabulary size
    K: int          # cached teacher entries per token
    T: float        # temperature
    chunk: int      # token rows per chunk
    hidden_rms_norm: bool   # divide each hidden row by its RMS after drawing
    teacher: str    # "exp_gaps" or "zipf"
    gap_scale: float = 1.0  # mean of the exponential gaps (exp_gaps only)
    spike_frac: float = 0.0  # fraction of tokens whose top logit gets +spike
    spike: float = 20.0
    w_std: float = 0.02

    @property
    def flops(self) -> float:
        """Tensor-core work of one forward+backward: four GEMMs of 2*N*H*V."""
        return 8.0 * self.N * self.H * self.V


CONFIGS = {
    "tiny": Config("tiny", N=256, H=256, V=4096, K=16, T=1.0, chunk=64,
                   hidden_rms_norm=False, teacher="exp_gaps", gap_scale=1.0),
    # "Exp(0.5)" gaps are read as rate 0.5 (mean gap 2).
    "llama3b": Config("llama3b", N=8192, H=3072, V=128256, K=100, T=1.0,
                      chunk=1024, hidden_rms_norm=False, teacher="exp_gaps",
                      gap_scale=2.0),
    # "Zipf-like" teacher logits are read as l_k = 10 - ln k (Zipf, s=1).
    "gptoss32k": Config("gptoss32k", N=32768, H=2880, V=201088, K=100, T=1.0,
                        chunk=2048, hidden_rms_norm=True, teacher="zipf"),
    "long64k": Config("long64k", N=65536, H=2880, V=201088, K=100, T=2.0,
                      chunk=2048, hidden_rms_norm=True, teacher="zipf",
                      spike_frac=0.1, spike=20.0),
    "ext256k": Config("ext256k", N=262144, H=2880, V=201088, K=100, T=1.0,
                      chunk=4096, hidden_rms_norm=True, teacher="zipf"),
}


def custom(name: str = "custom", **kw) -> Config:
    """A config with explicit sizes (tests use these for ragged shapes)."""
    base = dict(N=256, H=256, V=4096, K=16, T=1.0, chunk=128,
                hidden_rms_norm=False, teacher="exp_gaps", gap_scale=1.0)
    base.update(kw)
    return Config(name, **base)


def distinct_ids(gen: torch.Generator, n: int, k: int, v: int,
                 device="cpu") -> torch.Tensor:
    """[n, k] int32 ids, distinct within each row, uniform over [0, v).

    Draws uniformly, then redraws the later copy of every repeated id in a
    row until no row holds a repeat.  The rows are left unsorted.
    """
    if k > v:
        raise ValueError("cannot draw k > v distinct ids")
    if k == v:
        # every row is a permutation of the whole vocabulary
        keys = torch.rand((n, v), generator=gen, device=device)
        return keys.argsort(dim=1).to(torch.int32)
    ids = torch.randint(0, v, (n, k), generator=gen, device=device,
                        dtype=torch.int64)
    for _ in range(10000):
        srt, order = ids.sort(dim=1)
        dup_sorted = torch.zeros_like(srt, dtype=torch.bool)
        dup_sorted[:, 1:] = srt[:, 1:] == srt[:, :-1]
        if not bool(dup_sorted.any()):
            return ids.to(torch.int32)
        dup = torch.zeros_like(dup_sorted)
        dup.scatter_(1, order, dup_sorted)
        redraw = torch.randint(0, v, (int(dup.sum()),), generator=gen,
                               device=device, dtype=torch.int64)
        ids[dup] = redraw
    raise RuntimeError("distinct id redraw did not converge")


def teacher_logits(cfg: Config, gen: torch.Generator, n: int,
                   device="cpu") -> torch.Tensor:
    """[n, K] fp32 teacher logits, sorted in descending order per row."""
    K = cfg.K
    if cfg.teacher == "exp_gaps":
        # l_1 = 10, l_k = l_{k-1} - g_k with g_k exponential of mean gap_scale
        u = torch.rand((n, K - 1), generator=gen, device=device,
                       dtype=torch.float64)
        gaps = -torch.log1p(-u) * cfg.gap_scale
        lg = torch.empty((n, K), dtype=torch.float64, device=device)
        lg[:, 0] = 10.0
        lg[:, 1:] = 10.0 - torch.cumsum(gaps, dim=1)
    elif cfg.teacher == "zipf":
        k = torch.arange(1, K + 1, dtype=torch.float64, device=device)
        lg = (10.0 - torch.log(k)).expand(n, K).clone()
    else:
        raise ValueError(cfg.teacher)
    if cfg.spike_frac > 0:
        spike = torch.rand((n,), generator=gen, device=device) < cfg.spike_frac
        lg[:, 0] += spike.to(torch.float64) * cfg.spike
    return lg.to(torch.float32)


def make_inputs(cfg: Config, seed: int = 0, device="cpu",
                n_rows: Optional[int] = None) -> dict:
    """Draw (hidden, W, topk_idx, topk_logit) for ``cfg``.

    Streams are drawn in a fixed order from one torch generator on
    ``device``: hidden, W, ids, teacher logits.  The CPU and CUDA generators
    are different streams, so a given seed gives different (identically
    distributed) values on the two devices.

    Returns a dict of tensors on ``device``:
      hidden      bf16 [N, H] row-major
      W           bf16 [V, H] row-major
      topk_idx    int32 [N, K]
      topk_logit  fp32 [N, K]
    """
    N = cfg.N if n_rows is None else n_rows
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    hidden = torch.randn((N, cfg.H), generator=gen, device=device,
                         dtype=torch.float32)
    if cfg.hidden_rms_norm:
        rms = hidden.pow(2).mean(dim=1, keepdim=True).sqrt()
        hidden = hidden / rms
    hidden = hidden.to(torch.bfloat16)
    W = (torch.randn((cfg.V, cfg.H), generator=gen, device=device,
                     dtype=torch.float32) * cfg.w_std).to(torch.bfloat16)
    idx = distinct_ids(gen, N, cfg.K, cfg.V, device=device)
    logit = teacher_logits(cfg, gen, N, device=device)
    return {"hidden": hidden, "W": W, "topk_idx": idx, "topk_logit": logit}


def make_inputs_host(cfg: Config, seed: int = 0,
                     n_rows: Optional[int] = None) -> dict:
    """Draw (hidden, W, topk_idx, topk_logit) for ``cfg`` on the host with
    numpy's PCG64 generator.

    The recipe is that of ``make_inputs`` (same distributions, same stream
    order: hidden, W, ids, teacher logits, spikes), but every value comes
    from numpy's bit generator and IEEE-exact arithmetic (multiplies,
    divides, square roots, fp32 -> bf16 rounding to nearest even), so the
    same seed gives the same bytes on any host with this numpy.  Values
    that a committed script computed from these inputs on one machine can
    therefore be compared with a GPU run on another (``input_digest``
    checks that the bytes agree).

    Returns CPU tensors with the dtypes and layouts of ``make_inputs``.
    """
    N = cfg.N if n_rows is None else n_rows
    H, V, K = cfg.H, cfg.V, cfg.K
    rng = np.random.Generator(np.random.PCG64(seed))
    # normal draws in float64 (numpy's fast path), rounded to fp32, in row
    # blocks to bound the temporaries; consecutive blocks continue the stream
    # (block buffers reused across blocks: the same draws and operations as
    # whole-array temporaries, without fresh allocations; each block is
    # rounded fp32 -> bf16 into the output)
    B = min(_HOST_BLOCK, max(N, V))
    buf = np.empty((B, H))
    tmp = np.empty_like(buf)
    b32 = np.empty((B, H), dtype=np.float32)
    hidden_t = torch.empty((N, H), dtype=torch.bfloat16)
    for r0 in range(0, N, _HOST_BLOCK):
        rows = min(N, r0 + _HOST_BLOCK) - r0
        blk, h32 = buf[:rows], b32[:rows]
        rng.standard_normal(out=blk)
        h32[...] = blk                                    # rounded to fp32
        if cfg.hidden_rms_norm:
            # each row divided by its RMS (computed from the fp32 values)
            blk[...] = h32
            np.multiply(blk, blk, out=tmp[:rows])
            rms = np.sqrt(tmp[:rows].sum(axis=1, keepdims=True) / H)
            np.divide(blk, rms, out=tmp[:rows])
            h32[...] = tmp[:rows]
        hidden_t[r0:r0 + rows] = torch.from_numpy(h32).to(torch.bfloat16)
    W_t = torch.empty((V, H), dtype=torch.bfloat16)
    for r0 in range(0, V, _HOST_BLOCK):
        rows = min(V, r0 + _HOST_BLOCK) - r0
        w32 = b32[:rows]
        rng.standard_normal(out=buf[:rows])
        w32[...] = buf[:rows]                             # rounded to fp32
        np.multiply(w32, np.float32(cfg.w_std), out=w32)
        W_t[r0:r0 + rows] = torch.from_numpy(w32).to(torch.bfloat16)
    del buf, tmp, b32
    idx = _distinct_ids_host(rng, N, K, V)
    if cfg.teacher == "exp_gaps":
        gaps = rng.exponential(scale=cfg.gap_scale, size=(N, K - 1))
        lg = np.empty((N, K), dtype=np.float64)
        lg[:, 0] = 10.0
        lg[:, 1:] = 10.0 - np.cumsum(gaps, axis=1)
    elif cfg.teacher == "zipf":
        # scalar libm logs of 1..K (no vectorised math in the recipe)
        row = np.array([10.0 - math.log(k) for k in range(1, K + 1)], dtype=np.float64)
        lg = np.repeat(row[None, :], N, axis=0)
    else:
        raise ValueError(cfg.teacher)
    if cfg.spike_frac > 0:
        spike = rng.random(N) < cfg.spike_frac
        lg[:, 0] += np.where(spike, cfg.spike, 0.0)
    return {"hidden": hidden_t, "W": W_t, "topk_idx": torch.from_numpy(idx),
            "topk_logit": torch.from_numpy(lg.astype(np.float32))}


_HOST_BLOCK = 8192


def _distinct_ids_host(rng: np.random.Generator, n: int, k: int, v: int) -> np.ndarray:
    """[n, k] int32 ids, distinct within each row, uniform over [0, v):
    uniform draws, then the later copy of every repeated id in a row is
    redrawn until no row holds a repeat (rows left unsorted)."""
    if k > v:
        raise ValueError("cannot draw k > v distinct ids")
    if k == v:
        return rng.permuted(np.tile(np.arange(v, dtype=np.int32), (n, 1)), axis=1)
    ids = rng.integers(0, v, size=(n, k), dtype=np.int64)
    for _ in range(10000):
        order = np.argsort(ids, axis=1, kind="stable")
        srt = np.take_along_axis(ids, order, axis=1)
        dup_sorted = np.zeros(srt.shape, dtype=bool)
        dup_sorted[:, 1:] = srt[:, 1:] == srt[:, :-1]
        if not dup_sorted.any():
            return ids.astype(np.int32)
        dup = np.zeros_like(dup_sorted)
        np.put_along_axis(dup, order, dup_sorted, axis=1)
        ids[dup] = rng.integers(0, v, size=int(dup.sum()), dtype=np.int64)
    raise RuntimeError("distinct id redraw did not converge")


def input_digest(inp: dict) -> str:
    """SHA-256 of the raw bytes of (hidden, W, topk_idx, topk_logit), in
    that order: equal digests mean bit-identical inputs."""
    h = hashlib.sha256()
    for key in ("hidden", "W", "topk_idx", "topk_logit"):
        t = inp[key].detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        h.update(key.encode())
        h.update(t.numpy())            # the array's bytes, without a copy
    return h.hexdigest()


def bytes_of_inputs(cfg: Config) -> dict:
    """Device bytes of each input of ``cfg`` (bf16 hidden/W, int32+fp32 cache)."""
    return {
        "hidden": 2 * cfg.N * cfg.H,
        "W": 2 * cfg.V * cfg.H,
        "topk_idx": 4 * cfg.N * cfg.K,
        "topk_logit": 4 * cfg.N * cfg.K,
    }


def n_chunks(cfg: Config) -> int:
    return math.ceil(cfg.N / cfg.chunk)
