"""Oracle values of the four full-size workloads for ``tests/test_gpu_fullsize.py``.

Writes ``tests/golden/fullsize_<name>.npz`` for llama3b, gptoss32k, long64k
and ext256k.  Each file holds, for the inputs that
``workloads.make_inputs_host(cfg, seed=0)`` draws:

  digest       SHA-256 of those inputs (``workloads.input_digest``)
  N, H, V, K, T, chunk, seed
  loss         the oracle's mean loss over all N tokens (float64)
  lse          [N] float32: every token's logsumexp_v(z / T)
  loss_rows    [N] float32: every token's KL term
  vrows        [R] vocabulary ids: teacher-hit ids, ids at and past the
               last 256-wide vocabulary tile boundary, seeded random ids
  grad_W_rows  [R, H] float32: those rows of grad_W, over all N tokens

Only ``oracle/`` and ``workloads/`` are called.  Full logits of all N
tokens are needed (every grad_W row depends on every token's
full-vocabulary normaliser), so the oracle runs on row blocks in worker
processes: ``oracle.rows_forward`` with ``vrows`` and without the
grad_hidden product.  The blocks' grad_W shares are added in block order.
ext256k alone is about 3e14 float64 flop (tens of minutes on 8 cores).

    python tests/golden/make_fullsize.py [--workers 4] [--block 512] [name ...]
"""
from __future__ import annotations

import argparse
import ctypes
import multiprocessing as mp
import os
import shutil
import sys
import tempfile
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

NAMES = ("llama3b", "gptoss32k", "long64k", "ext256k")
SEED = 0
N_VROWS = 64


def fixture_path(name: str) -> str:
    return os.path.join(HERE, f"fullsize_{name}.npz")


def _keep_freed_memory():
    """Serve every allocation from the heap and never hand freed memory
    back to the kernel: the oracle allocates and frees block-sized
    temporaries, and on hosts where touching fresh pages is slow that
    costs more than the arithmetic."""
    try:
        libc = ctypes.CDLL("libc.so.6")
        libc.mallopt(-4, 0)            # M_MMAP_MAX: no mmap-backed chunks
        libc.mallopt(-1, 1 << 30)      # M_TRIM_THRESHOLD: keep up to 1 GiB of free top
    except OSError:
        pass


def choose_vrows(idx: np.ndarray, V: int, count: int = N_VROWS) -> np.ndarray:
    """Vocabulary rows to check: ids the teacher cache hits, the ids around
    the last 256-wide tile boundary and at the end of the vocabulary, and
    seeded random ids, sorted and distinct."""
    N = idx.shape[0]
    fixed = set(int(v) for v in idx[0, :4])
    fixed.update(int(v) for v in idx[N // 2, :2])
    fixed.add(int(idx[N - 1, 0]))
    last_tile = (V - 1) // 256 * 256
    fixed.update({0, 255, 256, last_tile - 1, last_tile, V - 4, V - 3, V - 2, V - 1})
    fixed = sorted(v for v in fixed if 0 <= v < V)
    rng = np.random.Generator(np.random.PCG64(1))
    pool = np.setdiff1d(np.arange(V), np.array(fixed))
    extra = rng.choice(pool, size=count - len(fixed), replace=False)
    return np.unique(np.concatenate([np.array(fixed, dtype=np.int64), extra]))


# ------------------------------------------------------------------ workers
_W = {}


def _init_worker(tmpdir: str, T: float, N: int, vrows: np.ndarray):
    _keep_freed_memory()
    _W["h"] = np.load(os.path.join(tmpdir, "hidden.npy"), mmap_mode="r")
    _W["W"] = np.load(os.path.join(tmpdir, "W.npy"), mmap_mode="r")
    _W["idx"] = np.load(os.path.join(tmpdir, "idx.npy"), mmap_mode="r")
    _W["lg"] = np.load(os.path.join(tmpdir, "lg.npy"), mmap_mode="r")
    _W["T"], _W["N"], _W["vrows"] = T, N, vrows


def _block(rng_):
    import oracle
    r0, r1 = rng_
    out = oracle.rows_forward(np.asarray(_W["h"][r0:r1]), _W["W"], np.asarray(_W["idx"][r0:r1]),
                              np.asarray(_W["lg"][r0:r1]), _W["T"], N_total=_W["N"],
                              vrows=_W["vrows"], grad_hidden=False)
    return r0, out["lse"], out["loss_rows"], out["grad_W_rows"]


# ------------------------------------------------------------------ per workload
def make(name: str, workers: int, block: int, tmp_root: str) -> None:
    import oracle
    import workloads

    cfg = workloads.CONFIGS[name]
    t0 = time.time()
    inp = workloads.make_inputs_host(cfg, seed=SEED)
    digest = workloads.input_digest(inp)
    N, H, V, K, T = cfg.N, cfg.H, cfg.V, cfg.K, cfg.T
    tmpdir = tempfile.mkdtemp(prefix=f"kd_{name}_", dir=tmp_root)
    try:
        # float64 copies of the inputs, shared with the workers through files
        shapes = {"hidden": ((N, H), np.float64), "W": ((V, H), np.float64),
                  "idx": ((N, K), np.int64), "lg": ((N, K), np.float64)}
        src = {"hidden": inp["hidden"], "W": inp["W"], "idx": inp["topk_idx"],
               "lg": inp["topk_logit"]}
        for key, (shape, dt) in shapes.items():
            mm = np.lib.format.open_memmap(os.path.join(tmpdir, f"{key}.npy"), mode="w+",
                                           dtype=dt, shape=shape)
            for r0 in range(0, shape[0], 16384):
                mm[r0:r0 + 16384] = oracle.to_f64(src[key][r0:r0 + 16384])
            mm.flush()
            del mm
        idx_np = inp["topk_idx"].numpy()
        vrows = choose_vrows(idx_np, V)
        del inp, src
        print(f"[{name}] inputs ready in {time.time() - t0:.0f} s, digest {digest[:16]}",
              flush=True)

        lse = np.empty(N, dtype=np.float64)
        loss_rows = np.empty(N, dtype=np.float64)
        gW = np.zeros((len(vrows), H), dtype=np.float64)
        tasks = [(r0, min(N, r0 + block)) for r0 in range(0, N, block)]
        ctx = mp.get_context("spawn")
        done = 0
        with ctx.Pool(workers, initializer=_init_worker, initargs=(tmpdir, T, N, vrows)) as pool:
            for r0, l, lr, g in pool.imap(_block, tasks, chunksize=1):
                r1 = r0 + l.shape[0]
                lse[r0:r1] = l
                loss_rows[r0:r1] = lr
                gW += g                      # block order: a fixed summation order
                done += 1
                if done % max(1, len(tasks) // 10) == 0:
                    print(f"[{name}] {done}/{len(tasks)} blocks, {time.time() - t0:.0f} s",
                          flush=True)
        loss = float(loss_rows.sum() / N)
        np.savez_compressed(fixture_path(name), digest=np.array(digest), seed=SEED, N=N, H=H,
                            V=V, K=K, T=T, chunk=cfg.chunk, loss=loss,
                            lse=lse.astype(np.float32), loss_rows=loss_rows.astype(np.float32),
                            vrows=vrows, grad_W_rows=gW.astype(np.float32))
        print(f"[{name}] loss {loss:.9f}; wrote {fixture_path(name)} in {time.time() - t0:.0f} s",
              flush=True)
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("names", nargs="*", default=list(NAMES))
    ap.add_argument("--workers", type=int, default=4)
    ap.add_argument("--block", type=int, default=512)
    args = ap.parse_args(argv)
    threads = max(1, (os.cpu_count() or 1) // args.workers)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = str(threads)        # inherited by the spawned workers
    _keep_freed_memory()
    tmp_root = "/dev/shm" if os.path.isdir("/dev/shm") else None
    for name in args.names:
        make(name, args.workers, args.block, tmp_root)


if __name__ == "__main__":
    main()
