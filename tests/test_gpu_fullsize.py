"""The CUDA path at the workloads' full sizes, in the benchmark's launch configuration.

Each workload (llama3b, gptoss32k, long64k, ext256k) runs whole on the GPU
with its own N, H, V, K, T and chunk, exactly as ``bench.py`` times it.
Its inputs come from ``workloads.make_inputs_host`` (numpy's PCG64, the
same bytes on every host), so the float64 oracle's values for the whole
problem, computed once on the host by ``tests/golden/make_fullsize.py``
(which calls only ``oracle/`` and ``workloads/``), apply to this run; the
stored input digest proves the inputs are the same.  Checked against the
oracle:

* the mean loss over all N tokens (relative 1e-3);
* every token's logsumexp and KL term;
* grad_W on the stored vocabulary rows (teacher-hit ids, the last vocabulary
  tile's boundary and end, random ids), each summing over all N tokens and
  so over every chunk's reduce-add (relative L2 2e-2);
* gathered z and grad_hidden of sampled tokens (``oracle.rows_forward``,
  computed here);
* at llama3b, all of grad_hidden and grad_W against the dense oracle run
  here on the host cores.

At gptoss32k the token mask and the sharded entry point are checked too:
the masked loss against the oracle's per-token terms over the valid
tokens, grad_hidden of sampled valid tokens against the oracle, masked rows
zero; two token shards normalised by the batch add up to the oracle's loss
and grad_W rows.

Also: every gathered id on every row equals the cached id (bit-exact), the
loss is the mean of the per-token terms, and grad_W satisfies two
identities that hold at any size (its vocabulary rows sum to zero;
<grad_W, W> = <grad_hidden, hidden>).
"""
import os

import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import oracle
import workloads
from tests.gpu_util import (GRAD_REL_L2, LOSS_RTOL, LSE_ATOL, ZG_RTOL, assert_parity,
                            ensure_lib, rel_l2, run_debug, to_device)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FULL_SIZE = ["llama3b", "gptoss32k", "long64k", "ext256k"]
N_SAMPLES = 40


def load_fixture(name):
    path = os.path.join(GOLDEN, f"fullsize_{name}.npz")
    assert os.path.exists(path), f"{path} missing: run tests/golden/make_fullsize.py {name}"
    return dict(np.load(path))


def _sample_rows(cfg, lg):
    """Evenly spaced tokens, both ends, both sides of every chunk boundary,
    and (when the workload has them) near-one-hot teacher rows."""
    N, c = cfg.N, cfg.chunk
    rows = set(np.linspace(0, N - 1, N_SAMPLES // 2).astype(np.int64).tolist())
    for b in (c, (N // c // 2) * c, N - c):
        rows.update({b - 1, b})
    rows.update({0, N - 1})
    if cfg.spike_frac > 0:
        spiky = torch.nonzero(lg[:, 0] > lg[:, 1] + 10).flatten()[:8].cpu().numpy()
        rows.update(int(r) for r in spiky)
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)


def _run_full(name):
    """The workload's host-drawn inputs (digest-checked against the
    fixture) through the debug entry point on the GPU."""
    ensure_lib()
    cfg = workloads.CONFIGS[name]
    fx = load_fixture(name)
    for key in ("N", "H", "V", "K", "chunk"):
        assert int(fx[key]) == getattr(cfg, key), (key, int(fx[key]), getattr(cfg, key))
    assert float(fx["T"]) == cfg.T
    inp_cpu = workloads.make_inputs_host(cfg, seed=int(fx["seed"]))
    assert workloads.input_digest(inp_cpu) == str(fx["digest"]), \
        "host-drawn inputs differ from the ones the fixture was computed on"
    N, H, V, K, T = cfg.N, cfg.H, cfg.V, cfg.K, cfg.T
    dev = torch.device("cuda")
    inp = to_device(inp_cpu, dev)
    gh = torch.empty((N, H), dtype=torch.float32, device=dev)
    gW = torch.empty((V, H), dtype=torch.float32, device=dev)
    ws = kd.alloc_workspace(N, H, V, K, cfg.chunk, device=dev)
    lse = torch.empty((N,), dtype=torch.float32, device=dev)
    zg = torch.empty((N, K), dtype=torch.float32, device=dev)
    found = torch.full((N, K), -1, dtype=torch.int32, device=dev)
    loss_rows = torch.empty((N,), dtype=torch.float64, device=dev)
    loss = kd.kd_topk_kl_debug(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"], T,
                               cfg.chunk, gh, gW, ws, lse=lse, zg=zg, found_idx=found,
                               loss_rows=loss_rows)
    torch.cuda.synchronize()
    del ws
    return cfg, fx, inp_cpu, inp, loss, dict(gh=gh, gW=gW, lse=lse, zg=zg, found=found,
                                             loss_rows=loss_rows)


@pytest.mark.parametrize("name", FULL_SIZE)
def test_full_size_against_oracle(name):
    cfg, fx, inp_cpu, inp, loss, out = _run_full(name)
    N, T = cfg.N, cfg.T
    gh, gW, found, loss_rows = out["gh"], out["gW"], out["found"], out["loss_rows"]

    # gathered ids: bit-exact on every row
    assert torch.equal(found, inp["topk_idx"]), "a cached id was gathered from the wrong column"

    # the whole-N loss against the oracle's
    want_loss = float(fx["loss"])
    assert abs(loss - want_loss) <= LOSS_RTOL * abs(want_loss), (loss, want_loss)
    # ... and it is the mean of the per-token terms (double sum, fp32 result)
    mean_rows = float(loss_rows.sum().item()) / N
    assert abs(loss - mean_rows) <= 1e-6 * abs(mean_rows), (loss, mean_rows)

    # every token's normaliser and KL term against the oracle's
    lse_err = np.abs(out["lse"].cpu().numpy() - fx["lse"].astype(np.float64)).max()
    assert lse_err <= LSE_ATOL, lse_err
    np.testing.assert_allclose(loss_rows.cpu().numpy(), fx["loss_rows"].astype(np.float64),
                               rtol=LOSS_RTOL, atol=1e-5)

    # grad_W rows (each a sum over all N tokens, i.e. over every chunk)
    assert torch.isfinite(gh).all() and torch.isfinite(gW).all()
    vrows = torch.from_numpy(fx["vrows"]).to(gW.device)
    got_rows = gW[vrows].cpu().numpy()
    want_rows = fx["grad_W_rows"].astype(np.float64)
    err = rel_l2(got_rows, want_rows)
    assert err <= GRAD_REL_L2, err
    # no single row is far off either (rows of non-hit ids are small)
    row_err = np.linalg.norm(got_rows - want_rows, axis=1) / np.linalg.norm(want_rows, axis=1)
    assert row_err.max() <= 5 * GRAD_REL_L2, (fx["vrows"][row_err.argmax()], row_err.max())

    # sampled tokens: gathered z and grad_hidden rows against the oracle
    rows = _sample_rows(cfg, inp_cpu["topk_logit"])
    want = oracle.rows_forward(inp_cpu["hidden"][rows], inp_cpu["W"], inp_cpu["topk_idx"][rows],
                               inp_cpu["topk_logit"][rows], T, N_total=N)
    rt = torch.from_numpy(rows).to(gh.device)
    zscale = max(np.abs(want["zg"]).max(), 1e-6)
    assert np.abs(out["zg"][rt].cpu().numpy() - want["zg"]).max() <= ZG_RTOL * zscale
    np.testing.assert_allclose(out["lse"][rt].cpu().numpy(), want["lse"], rtol=0, atol=LSE_ATOL)
    err = rel_l2(gh[rt].cpu().numpy(), want["grad_hidden"])
    assert err <= GRAD_REL_L2, err

    # grad_W: its vocabulary rows sum to zero, relative to the size of one
    # row-sum's terms (|dZ| summed over v is at most 2/(T N) per token)
    h = inp["hidden"]
    col = gW.double().sum(dim=0)
    scale = (h.double().abs().sum(dim=0) * (2.0 / (T * N)))
    assert float((col.abs() / scale).max()) <= 1e-3
    # grad_W: <grad_W, W> = <grad_hidden, hidden> (both sum_{n,v} dZ_nv z_nv)
    a = float((gW.double() * inp["W"].double()).sum())
    b = float((gh.double() * h.double()).sum())
    mag = float((gh.double() * h.double()).abs().sum())
    assert abs(a - b) <= 1e-3 * mag, (a, b, mag)
    assert abs(b) >= 1e-2 * mag


def test_llama3b_dense_gradients():
    """llama3b (8,192 tokens, H=3072, V=128,256, chunk 1024) against the
    dense float64 oracle run here on the host: all of grad_hidden and
    grad_W, every lse and gathered z, and the loss."""
    cfg, fx, inp_cpu, inp, loss, out = _run_full("llama3b")
    want = oracle.fused_topk_kl(inp_cpu["hidden"], inp_cpu["W"], inp_cpu["topk_idx"],
                                inp_cpu["topk_logit"], cfg.T)
    assert abs(want["loss"] - float(fx["loss"])) <= 1e-9 * abs(want["loss"])
    got = {"loss": loss, "found": out["found"].cpu().numpy(), "lse": out["lse"].cpu().numpy(),
           "zg": out["zg"].cpu().numpy(), "grad_hidden": out["gh"].cpu().numpy(),
           "grad_W": out["gW"].cpu().numpy()}
    assert_parity(got, want, inp_cpu["topk_idx"].numpy())


def test_full_vocab_head_single_chunk():
    """256 tokens of the GPT-OSS-like head (H=2880, V=201,088) in one
    2048-row chunk: every output against the dense oracle, grad_W on
    sampled vocabulary rows (teacher-hit rows, the last rows of the ragged
    last vocab tile, random rows) and in full."""
    ensure_lib()
    base = workloads.CONFIGS["gptoss32k"]
    inp = workloads.make_inputs(base, seed=4, n_rows=256)
    got = run_debug(to_device(inp), base.T, base.chunk)
    want = oracle.fused_topk_kl(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                                base.T)
    assert_parity(got, want, inp["topk_idx"].numpy(), check_grads=False)
    assert rel_l2(got["grad_hidden"], want["grad_hidden"]) <= GRAD_REL_L2
    idx = inp["topk_idx"].numpy()
    rng = np.random.default_rng(0)
    V = base.V
    vrows = np.unique(np.concatenate([idx[:8, 0], idx[100:104, 3], np.arange(V - 4, V),
                                      np.arange(V - 260, V - 256),
                                      rng.integers(0, V, size=24)]))
    err = rel_l2(got["grad_W"][vrows], want["grad_W"][vrows])
    assert err <= GRAD_REL_L2, err
    assert rel_l2(got["grad_W"], want["grad_W"]) <= GRAD_REL_L2


@pytest.mark.parametrize("flag", ["min_scratch", "store_logits"])
def test_gptoss32k_other_plans_against_oracle(flag):
    """gptoss32k with grad_W per chunk (KD_FLAG_MIN_SCRATCH) and with the
    stored-logits backward: the same stored oracle values hold for every
    plan (loss, every token's KL term, the grad_W rows)."""
    ensure_lib()
    cfg = workloads.CONFIGS["gptoss32k"]
    fx = load_fixture("gptoss32k")
    inp_cpu = workloads.make_inputs_host(cfg, seed=int(fx["seed"]))
    assert workloads.input_digest(inp_cpu) == str(fx["digest"])
    inp = to_device(inp_cpu)
    flags = {"min_scratch": kd.KD_FLAG_MIN_SCRATCH, "store_logits": kd.KD_FLAG_STORE_LOGITS}[flag]
    N, H, V, K = cfg.N, cfg.H, cfg.V, cfg.K
    gh = torch.empty((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(kd.kd_topk_kl_workspace_size_flags(N, H, V, K, cfg.chunk, flags),
                     dtype=torch.uint8, device="cuda")
    loss = kd.kd_topk_kl_fwd_bwd_flags(inp["hidden"], inp["W"], inp["topk_idx"],
                                       inp["topk_logit"], None, cfg.T, cfg.chunk, flags, gh, gW,
                                       ws)
    torch.cuda.synchronize()
    del ws
    want_loss = float(fx["loss"])
    assert abs(loss - want_loss) <= LOSS_RTOL * abs(want_loss), (loss, want_loss)
    vrows = torch.from_numpy(fx["vrows"]).to(gW.device)
    err = rel_l2(gW[vrows].cpu().numpy(), fx["grad_W_rows"].astype(np.float64))
    assert err <= GRAD_REL_L2, err
    assert torch.isfinite(gh).all()


def test_gptoss32k_masked_against_oracle():
    """The token mask at the headline size.  A mask leaves every token's KL
    term unchanged and takes the mean over the valid tokens, so the stored
    oracle terms give the masked loss; grad_hidden of sampled valid tokens
    against the oracle normalised by the valid count, masked rows zero, and
    grad_W's two identities."""
    ensure_lib()
    cfg = workloads.CONFIGS["gptoss32k"]
    fx = load_fixture("gptoss32k")
    inp_cpu = workloads.make_inputs_host(cfg, seed=int(fx["seed"]))
    assert workloads.input_digest(inp_cpu) == str(fx["digest"])
    N, H, V, K, T = cfg.N, cfg.H, cfg.V, cfg.K, cfg.T
    g = torch.Generator().manual_seed(11)
    mask_cpu = (torch.rand(N, generator=g) < 0.6).to(torch.uint8)
    mask_cpu[0] = 1
    n_valid = int(mask_cpu.sum())
    inp = to_device(inp_cpu)
    gh = torch.empty((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(kd.kd_topk_kl_workspace_size_flags(N, H, V, K, cfg.chunk, 0),
                     dtype=torch.uint8, device="cuda")
    loss = kd.kd_topk_kl_fwd_bwd_flags(inp["hidden"], inp["W"], inp["topk_idx"],
                                       inp["topk_logit"], mask_cpu.cuda(), T, cfg.chunk, 0, gh,
                                       gW, ws)
    torch.cuda.synchronize()
    del ws
    valid = mask_cpu.numpy().astype(bool)
    want_loss = float(fx["loss_rows"].astype(np.float64)[valid].sum() / n_valid)
    assert abs(loss - want_loss) <= LOSS_RTOL * abs(want_loss), (loss, want_loss)

    masked_rows = torch.from_numpy(np.flatnonzero(~valid)).cuda()
    assert int(torch.count_nonzero(gh[masked_rows])) == 0
    rows = _sample_rows(cfg, inp_cpu["topk_logit"])
    rows = rows[valid[rows]]
    want = oracle.rows_forward(inp_cpu["hidden"][rows], inp_cpu["W"], inp_cpu["topk_idx"][rows],
                               inp_cpu["topk_logit"][rows], T, N_total=n_valid)
    rt = torch.from_numpy(rows).cuda()
    assert rel_l2(gh[rt].cpu().numpy(), want["grad_hidden"]) <= GRAD_REL_L2

    h = inp["hidden"]
    assert torch.isfinite(gW).all()
    col = gW.double().sum(dim=0)
    scale = h.double().abs().sum(dim=0) * (2.0 / (T * n_valid))
    assert float((col.abs() / scale).max()) <= 1e-3
    a = float((gW.double() * inp["W"].double()).sum())
    b = float((gh.double() * h.double()).sum())
    mag = float((gh.double() * h.double()).abs().sum())
    assert abs(a - b) <= 1e-3 * mag, (a, b, mag)


def test_gptoss32k_two_shards_against_oracle():
    """The batch as two token shards, each normalised by the whole batch's
    N and adding into one grad_W: the shards' losses add up to the oracle's
    loss and the accumulated grad_W matches the oracle's stored rows."""
    ensure_lib()
    cfg = workloads.CONFIGS["gptoss32k"]
    fx = load_fixture("gptoss32k")
    inp_cpu = workloads.make_inputs_host(cfg, seed=int(fx["seed"]))
    assert workloads.input_digest(inp_cpu) == str(fx["digest"])
    N, H, V, K, T = cfg.N, cfg.H, cfg.V, cfg.K, cfg.T
    inp = to_device(inp_cpu)
    # KD_FLAG_ACCUMULATE adds into grad_hidden as well as grad_W: the second
    # shard's rows must start from zero
    gh = torch.zeros((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    cut = 3 * cfg.chunk + 517                      # unequal shards; a ragged last chunk in each
    total = 0.0
    for k, (r0, r1) in enumerate(((0, cut), (cut, N))):
        n = r1 - r0
        ws = torch.empty(kd.kd_topk_kl_workspace_size_flags(n, H, V, K, cfg.chunk, 0),
                         dtype=torch.uint8, device="cuda")
        flags = kd.KD_FLAG_ACCUMULATE if k else 0
        total += kd.kd_topk_kl_fwd_bwd_sharded(inp["hidden"][r0:r1], inp["W"],
                                               inp["topk_idx"][r0:r1], inp["topk_logit"][r0:r1],
                                               None, T, cfg.chunk, flags, N, gh[r0:r1], gW, ws)
        del ws
    torch.cuda.synchronize()
    want_loss = float(fx["loss"])
    assert abs(total - want_loss) <= LOSS_RTOL * abs(want_loss), (total, want_loss)
    vrows = torch.from_numpy(fx["vrows"]).cuda()
    assert rel_l2(gW[vrows].cpu().numpy(), fx["grad_W_rows"].astype(np.float64)) <= GRAD_REL_L2
    rows = _sample_rows(cfg, inp_cpu["topk_logit"])
    want = oracle.rows_forward(inp_cpu["hidden"][rows], inp_cpu["W"], inp_cpu["topk_idx"][rows],
                               inp_cpu["topk_logit"][rows], T, N_total=N)
    rt = torch.from_numpy(rows).cuda()
    assert rel_l2(gh[rt].cpu().numpy(), want["grad_hidden"]) <= GRAD_REL_L2
