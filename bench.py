#!/usr/bin/env python
"""Benchmark of the fused chunked top-K KL loss (forward + backward) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config gptoss32k]
    python bench.py --impl reference ...      # the float64 CPU oracle arm

A step is one call of ``kd_topk_kl_fwd_bwd_ex`` over one batch of synthetic
tokens: the whole hot path (teacher prep, per-chunk forward GEMM with the
logsumexp/gather epilogue, loss fold, recompute GEMM with the dZ epilogue,
grad_hidden and grad_W GEMMs, final loss).  The default workload is the
GPT-OSS-like head at 32,768 tokens (H=2880, V=201,088, K=100, chunk 2048),
the configuration the pages' 32K figures and GPT-OSS 20B run refer to.

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs an
independent replica of the workload (the library has no cross-GPU exchange),
the timed region is bracketed by barriers and the time is the maximum over
ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tokens/s fused top-K KL fwd+bwd (N×H×V), % bf16 tensor peak, peak GiB"
GEMM_KINDS = ("gemm_fwd_lse_gather", "gemm_bwd_dz", "gemm_dz_and_next_fwd", "gemm_grad_hidden",
              "gemm_grad_W")


def gemm_flops_per_step(kind: str, N: int, H: int, V: int, chunk: int, store_logits: bool) -> float:
    """Flops one step spends in the GEMM launches of a profiler kind: 2 H V
    per token row multiplied.  The forward of the first chunk runs alone and
    every later chunk's forward shares a launch with the previous chunk's
    recompute; the last chunk's recompute runs alone.  With stored logits
    every chunk's forward runs alone and nothing is recomputed."""
    c = min(-(-chunk // 128) * 128, -(-N // 128) * 128)
    n = -(-N // c)
    first = min(c, N)
    last = N - (n - 1) * c
    rows = {"gemm_fwd_lse_gather": N if store_logits else first,
            "gemm_bwd_dz": 0 if store_logits else last,
            "gemm_dz_and_next_fwd": 0 if store_logits else (N - last) + (N - first),
            "gemm_grad_hidden": N, "gemm_grad_W": N}[kind]
    return 2.0 * rows * H * V
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ------------------------------------------------------------------ helpers
def load_peaks() -> tuple:
    """The measured peaks of this machine's B300, else the fallback figures;
    a measured file without a figure takes the fallback for it (and says so)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"
    missing = [k for k in FALLBACK_PEAKS if not isinstance(p.get(k), (int, float))]
    for k in missing:
        p[k] = FALLBACK_PEAKS[k]
    return p, "measured" if not missing else "measured, fallback for " + ", ".join(missing)


GEMM_SOURCES = ("kd_args.h", "kd_gemm.cuh", "kd_ptx.cuh")
GEMM_SECTION_END = b"// ------------------------------------------------------------------ prep"


def kernel_source_hash() -> str:
    """Hash of the sources that define the GEMM kernels: their template, PTX
    helpers and arguments, and the part of kd_kernels.cu that instantiates
    and launches them (up to the first SIMT kernel).  Stored DRAM counters
    are reported only while this hash is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunked_top_kl_gemm_b300", "csrc")
    for name in GEMM_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    with open(os.path.join(csrc, "kd_kernels.cu"), "rb") as f:
        text = f.read()
    h.update(b"kd_kernels.cu")
    h.update(text.split(GEMM_SECTION_END)[0])
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/ncu_traffic.txt if the counters were
    taken on the current kernel sources, else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
            if (kv.get("kernel") == kernel and kv.get("workload") == workload
                    and kv.get("src") == src):
                return float(kv["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (200 ms)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="kd_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", self.gpu_id],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            rows = [[c.strip() for c in ln.split(",")] for ln in f if ln.strip()]
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, power, reasons = [], [], [], set()
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _gpu_id(local: int) -> str:
    """nvidia-smi's id of the GPU behind CUDA device `local`."""
    if "CUDA_VISIBLE_DEVICES" in os.environ:
        return os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]
    return str(local)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_max(value: float, device=None) -> float:
    """Maximum of `value` over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def throughput(tokens_per_rank: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job tokens/s: the tokens every rank processed over the slowest rank's time."""
    return tokens_per_rank * steps * world / seconds


# ------------------------------------------------------------------ oracle legs
def host_info() -> dict:
    """CPU model and BLAS library of the host the oracle runs on."""
    info = {"cpu_model": None, "blas": None}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    info["cpu_model"] = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        import numpy
        blas = numpy.show_config(mode="dicts").get("Build Dependencies", {}).get("blas", {})
        info["blas"] = f"{blas.get('name')} {blas.get('version')}"
    except Exception:  # pragma: no cover
        pass
    return info


def nvml_used_bytes(dev):
    """Device memory in use per NVML on the GPU behind torch device `dev`, in
    bytes (None when it cannot be read).  Through pynvml when it is
    installed, else through nvidia-smi (NVML's command-line front end, MiB
    resolution).  The device is matched by its UUID: NVML's numbering need
    not follow CUDA_VISIBLE_DEVICES."""
    import torch
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    if uuid is None:
        return None
    try:
        import pynvml
    except ImportError:
        pynvml = None
    if pynvml is not None:
        try:
            pynvml.nvmlInit()
            try:
                h = pynvml.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}")
                return int(pynvml.nvmlDeviceGetMemoryInfo(h).used)
            finally:
                pynvml.nvmlShutdown()
        except Exception:
            pass
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=memory.used", "--format=csv,noheader,nounits",
                              "-i", f"GPU-{uuid}"], capture_output=True, text=True, timeout=20)
        if out.returncode == 0 and out.stdout.strip():
            return int(float(out.stdout.strip().splitlines()[0])) * 2**20
    except (OSError, ValueError, subprocess.TimeoutExpired):
        pass
    return None


def oracle_sample_rate(inp_cpu: dict, T: float, sample: int) -> dict:
    """Time the float64 oracle on the first `sample` tokens (tokens/s)."""
    import oracle
    try:
        from threadpoolctl import threadpool_info
        threads = max((d.get("num_threads", 0) for d in threadpool_info()), default=0)
    except Exception:  # pragma: no cover
        threads = 0
    threads = threads or os.cpu_count()
    t0 = time.perf_counter()
    oracle.fused_topk_kl(inp_cpu["hidden"][:sample], inp_cpu["W"], inp_cpu["topk_idx"][:sample],
                         inp_cpu["topk_logit"][:sample], T)
    dt = time.perf_counter() - t0
    return {"value": sample / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "seconds": dt, "tokens": sample}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import workloads
    cfg = workloads.CONFIGS[args.config]
    sample = args.ref_sample
    inp = workloads.make_inputs(cfg, seed=0, n_rows=sample)
    for _ in range(args.warmup):
        oracle_sample_rate(inp, cfg.T, sample)
    t0 = time.perf_counter()
    last = None
    for _ in range(args.steps):
        last = oracle_sample_rate(inp, cfg.T, sample)
    dt = time.perf_counter() - t0
    value = sample * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "N": cfg.N, "H": cfg.H, "V": cfg.V, "K": cfg.K,
                   "T": cfg.T, "chunk": cfg.chunk,
                   "step": f"oracle over {sample} of the workload's tokens (full V, full W)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": last["cores"],
                         "kind": "oracle", **host_info(),
                         "sample": f"{sample} tokens of {cfg.name} per step, float64 numpy"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main arm
def run_gpu(args):
    import torch
    import torch.distributed as dist

    import chunked_top_kl_gemm_b300 as kd
    import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    kd.lib()  # fail loudly if the library is missing

    cfg = workloads.CONFIGS[args.config]
    if args.tokens:
        import dataclasses
        cfg = dataclasses.replace(cfg, N=args.tokens, name=f"{cfg.name}_n{args.tokens}")
    chunk = args.chunk or cfg.chunk
    N, H, V, K, T = cfg.N, cfg.H, cfg.V, cfg.K, cfg.T

    mem0 = torch.cuda.memory_allocated(dev)
    torch.cuda.synchronize(dev)
    nvml0 = nvml_used_bytes(dev)
    inp = workloads.make_inputs(cfg, seed=rank, device=dev)
    h, W, idx, lg = inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"]
    # the peak counts the resident inputs, outputs, workspace and whatever the
    # calls allocate, not the temporaries of drawing the inputs on the device
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    gh = torch.empty((N, H), dtype=torch.float32, device=dev)
    gW = torch.empty((V, H), dtype=torch.float32, device=dev)
    flags = (kd.KD_FLAG_STORE_LOGITS if args.store_logits else 0) | \
        (kd.KD_FLAG_MIN_SCRATCH if args.min_scratch else 0)
    ws = torch.empty(kd.kd_topk_kl_workspace_size_flags(N, H, V, K, chunk, flags),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    del inp

    if flags:
        def step():
            return kd.kd_topk_kl_fwd_bwd_flags(h, W, idx, lg, None, T, chunk, flags, gh, gW, ws,
                                               stream=stream)
    else:
        def step():
            return kd.kd_topk_kl_fwd_bwd_ex(h, W, idx, lg, T, chunk, gh, gW, ws, stream=stream)

    for _ in range(max(args.warmup, 3) if not args.allow_short_warmup else args.warmup):
        loss = step()
    peak_gib = (torch.cuda.max_memory_allocated(dev) - mem0) / 2**30
    nvml1 = nvml_used_bytes(dev)
    # cross-check: device memory NVML sees in use grew by (torch's reserved pool)
    nvml_delta_gib = (nvml1 - nvml0) / 2**30 if nvml0 is not None and nvml1 is not None else None

    gpu_id = _gpu_id(local)
    # the headline: K steps with the library's per-kernel profiler off
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.5)
    dist_barrier(dev)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        loss = step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    dist_barrier(dev)
    clk = clocks.stop()
    t_dev = e0.elapsed_time(e1) / 1e3

    # a second, labelled pass with the profiler on: every launch bracketed by
    # two CUDA events on the launch stream (per-kernel times, the roofline of
    # the dominant kernel and the launch count)
    prof_steps = max(1, args.profile_steps or args.steps)
    pclocks = ClockSampler(gpu_id)
    pclocks.start()
    time.sleep(0.2)
    kd.kd_profile_enable(True)
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(prof_steps):
        step()
    p1.record(stream)
    torch.cuda.synchronize(dev)
    kd.kd_profile_enable(False)
    pclk = pclocks.stop()
    prof = kd.kd_profile_read()
    t_prof = p0.elapsed_time(p1) / 1e3
    t_max = dist_max(t_dev, dev)
    value = throughput(N, args.steps, world, t_max)
    # the recompute path does four GEMMs of 2NHV; storing the logits skips one
    flops_step = cfg.flops * (0.75 if args.store_logits else 1.0)
    tflops = flops_step * args.steps / t_max / 1e12

    # end to end: every step's inputs are copied from pinned host memory and
    # its loss (and status word) is read back into pinned host memory, as a
    # training loop feeding the loss would do it, through the library's
    # asynchronous entry point (no host synchronisation per step).  The next
    # step's inputs are copied on a second stream into a second set of
    # device buffers while the current step computes; a buffer set is
    # refilled only after the step that read it has passed on the GPU.
    h_host = h.cpu().pin_memory()
    idx_host = idx.cpu().pin_memory()
    lg_host = lg.cpu().pin_memory()
    h2d = h_host.numel() * 2 + idx_host.numel() * 4 + lg_host.numel() * 4
    bufs = [(h, idx, lg), (torch.empty_like(h), torch.empty_like(idx), torch.empty_like(lg))]
    copy_stream = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    loss_dev = torch.zeros(1, dtype=torch.float32, device=dev)
    status_dev = torch.zeros(1, dtype=torch.int32, device=dev)
    n_read = max(args.steps, 2)
    loss_host = torch.zeros(n_read, dtype=torch.float32).pin_memory()
    status_host = torch.zeros(n_read, dtype=torch.int32).pin_memory()

    def copy_in(slot, first):
        with torch.cuda.stream(copy_stream):
            if not first:
                copy_stream.wait_event(done[slot])     # the step that read this set passed
            for dst, src in zip(bufs[slot], (h_host, idx_host, lg_host)):
                dst.copy_(src, non_blocking=True)
            ready[slot].record(copy_stream)

    def e2e_steps(n):
        copy_in(0, True)
        for i in range(n):
            slot = i % 2
            stream.wait_event(ready[slot])
            if i + 1 < n:
                copy_in(1 - slot, i == 0)
            hb, ib, lb = bufs[slot]
            kd.kd_topk_kl_fwd_bwd_async(hb, W, ib, lb, None, T, chunk, flags, loss_dev,
                                        status_dev, gh, gW, ws, stream=stream)
            done[slot].record(stream)
            with torch.cuda.stream(stream):
                loss_host[i].copy_(loss_dev[0], non_blocking=True)
                status_host[i].copy_(status_dev[0], non_blocking=True)

    e2e_steps(2)
    dist_barrier(dev)
    torch.cuda.synchronize(dev)
    w0 = time.perf_counter()
    e2e_steps(args.steps)
    torch.cuda.synchronize(dev)
    t_e2e = dist_max(time.perf_counter() - w0, dev)
    dist_barrier(dev)
    if int(status_host[:args.steps].abs().sum()) != 0:
        raise RuntimeError(f"end-to-end steps reported device status {status_host.tolist()}")
    if not bool(torch.isfinite(loss_host[:args.steps]).all()):
        raise RuntimeError("end-to-end steps returned a non-finite loss")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    gemm = {k: prof[k] for k in GEMM_KINDS if k in prof and prof[k][1] > 0}
    dom = max(gemm, key=lambda k: gemm[k][0])
    dom_ms, dom_launches = gemm[dom]
    dom_flops = gemm_flops_per_step(dom, N, H, V, chunk, args.store_logits)
    flops_per_launch = dom_flops / (dom_launches / prof_steps)
    achieved = flops_per_launch / (dom_ms / dom_launches / 1e3) / 1e12
    peak_sust = float(peaks["bf16_tflops_sustained"])
    traffic = stored_traffic(dom, cfg.name)
    # the library's launches per step are fixed by the plan: the profiled
    # pass counts them
    launches_per_step = sum(c for _, c in prof.values()) / prof_steps

    cpu = None
    if world == 1 and not args.skip_cpu_baseline:
        inp_cpu = workloads.make_inputs(cfg, seed=0, n_rows=args.cpu_sample)
        cpu = oracle_sample_rate(inp_cpu, T, args.cpu_sample)
        cpu = {"value": cpu["value"], "unit": "tokens/s", "cores": cpu["cores"],
               "kind": "oracle", **host_info(),
               "sample": f"first {args.cpu_sample} tokens of {cfg.name} (full V and W), "
                         f"float64 numpy, {cpu['seconds']:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name, "N": N, "H": H, "V": V, "K": K, "T": T,
                   "chunk": chunk, "parallelism": f"replicas{world}" if world > 1 else "single",
                   "backward": "stored fp32 logits (6NHV)" if args.store_logits
                               else "recompute (8NHV)",
                   "grad_W_depth": "one chunk (minimal scratch)" if args.min_scratch
                                   else "two chunks",
                   "l2": "inputs larger than L2 (W is 1.16 GB and is streamed every GEMM)"},
        "tflops": tflops,
        "frac_bf16_peak_burst": tflops / float(peaks["bf16_tflops"]),
        "frac_bf16_peak_sustained": tflops / peak_sust,
        "peak_gib": peak_gib,
        "peak_gib_nvml_delta": nvml_delta_gib,
        "loss": loss,
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_sust,
                     "peak_kind": f"bf16_tflops_sustained ({peak_src})", "unit": "TFLOP/s",
                     "frac": achieved / peak_sust, "traffic": traffic,
                     "flops_per_launch": flops_per_launch,
                     "avg_launch_ms": dom_ms / dom_launches,
                     "source": f"separate pass of {prof_steps} steps with the per-launch "
                               "event profiler on (not the headline loop)"},
        "kernels": {k: {"ms_per_step": v[0] / prof_steps, "launches_per_step": v[1] / prof_steps}
                    for k, v in prof.items() if v[1] > 0},
        # every GEMM kind against the same sustained peak (its share of the
        # 8NHV flops over its event time)
        "gemm_rooflines": {k: {"tflops": gemm_flops_per_step(k, N, H, V, chunk, args.store_logits)
                                         / (v[0] / prof_steps / 1e3) / 1e12,
                               "frac": gemm_flops_per_step(k, N, H, V, chunk, args.store_logits)
                                       / (v[0] / prof_steps / 1e3) / 1e12 / peak_sust}
                           for k, v in gemm.items()},
        "profile_pass": {"steps": prof_steps, "ms_per_step": t_prof / prof_steps * 1e3,
                         "clocks": pclk},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clk,
        "e2e": {"value": throughput(N, args.steps, world, t_e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 8,
                "api": "kd_topk_kl_fwd_bwd_async, loss and status read back every step"},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ sweep
# The shape of the pages' isolated output-projection benchmark (glonce.com,
# body; ainewsbank.com, "What the long-context measurements show"): peak
# memory should stay flat in N x V and grow only with the per-token tensors,
# and the chunk size trades workspace for speed.  One JSON line per point.
SWEEP_POINTS = (
    [("tiny", None, None), ("llama3b", None, None)]
    + [("gptoss32k", n, 2048) for n in (8192, 32768, 65536, 131072, 262144)]
    + [("long64k", None, None)]
    + [("ext256k", None, c) for c in (1024, 2048, 4096, 8192)]
)


def _sweep_point(kd, cfg, chunk, flags, dev, peaks):
    """Peak memory and power-capped throughput of one call plan on one
    workload: the inputs drawn on the device, one cold call for the peak,
    then enough timed steps for about 1.5 s of clock samples.  Returns the
    JSON fields, or a `skipped` reason when the plan's buffers would not fit
    in 85 % of the device memory that is free."""
    import torch

    import workloads

    N, H, V, K, T = cfg.N, cfg.H, cfg.V, cfg.K, cfg.T
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    ws_bytes = kd.kd_topk_kl_workspace_size_flags(N, H, V, K, chunk, flags)
    need = ws_bytes + sum(workloads.bytes_of_inputs(cfg).values()) + 4 * (N * H + V * H)
    free, _ = torch.cuda.mem_get_info(dev)
    if need > 0.85 * free:
        return {"skipped": f"needs {need / 2**30:.1f} GiB, {free / 2**30:.1f} GiB free",
                "needs_gib": need / 2**30}
    mem0 = torch.cuda.memory_allocated(dev)
    inp = workloads.make_inputs(cfg, seed=0, device=dev)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)     # not the input draw's temporaries
    gh = torch.empty((N, H), dtype=torch.float32, device=dev)
    gW = torch.empty((V, H), dtype=torch.float32, device=dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    h_, W_, i_, l_ = inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"]

    def call():
        return kd.kd_topk_kl_fwd_bwd_flags(h_, W_, i_, l_, None, T, chunk, flags, gh, gW, ws)
    loss = call()
    torch.cuda.synchronize(dev)
    peak = (torch.cuda.max_memory_allocated(dev) - mem0) / 2**30
    # time one more warm call, then enough steps for ~1.5 s of samples
    w0 = time.perf_counter()
    call()
    steps = max(3, min(200, int(1.5 / max(time.perf_counter() - w0, 1e-4)) + 1))
    clocks = ClockSampler(_gpu_id(0))
    clocks.start()
    time.sleep(0.2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        loss = call()
    e1.record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    t = e0.elapsed_time(e1) / 1e3 / steps
    flops = cfg.flops * (0.75 if flags & kd.KD_FLAG_STORE_LOGITS else 1.0)
    tflops = flops / t / 1e12
    out = {"N": N, "H": H, "V": V, "K": K, "T": T, "chunk": chunk, "steps": steps,
           "tokens_per_s": N / t, "ms_per_step": t * 1e3, "tflops": tflops,
           "frac_bf16_peak_burst": tflops / float(peaks["bf16_tflops"]),
           "peak_gib": peak,
           "inputs_gib": sum(workloads.bytes_of_inputs(cfg).values()) / 2**30,
           "grads_gib": 4 * (N * H + V * H) / 2**30,
           "workspace_gib": ws_bytes / 2**30,
           "dense_fp32_logits_gib": 4 * N * V / 2**30, "loss": loss, "clocks": clk}
    del inp, gh, gW, ws, h_, W_, i_, l_
    return out


def run_sweep(args):
    import dataclasses

    import torch

    import chunked_top_kl_gemm_b300 as kd
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kd.lib()
    peaks, _ = load_peaks()
    oracle_rate = {}   # per workload: the float64 oracle on its first tokens (host cores)
    flags = kd.KD_FLAG_MIN_SCRATCH if args.min_scratch else 0
    for name, n_tokens, chunk in SWEEP_POINTS:
        cfg = workloads.CONFIGS[name]
        if name not in oracle_rate and not args.skip_cpu_baseline:
            sample = min(cfg.N, args.cpu_sample)
            r = oracle_sample_rate(workloads.make_inputs(cfg, seed=0, n_rows=sample), cfg.T, sample)
            oracle_rate[name] = {"value": r["value"], "unit": "tokens/s", "cores": r["cores"],
                                 "kind": "oracle",
                                 "sample": f"first {sample} tokens of {name} (full V and W), "
                                           f"float64 numpy, {r['seconds']:.1f} s"}
        if n_tokens:
            cfg = dataclasses.replace(cfg, N=n_tokens, name=f"{name}_n{n_tokens}")
        chunk = chunk or cfg.chunk
        point = _sweep_point(kd, cfg, chunk, flags, dev, peaks)
        print(json.dumps({
            "sweep": "memory_and_throughput", "workload": cfg.name,
            "grad_W_depth": "one chunk (minimal scratch)" if args.min_scratch else "two chunks",
            **point, "cpu_baseline": oracle_rate.get(name)}), flush=True)


# The full logits grid against the chunked plan.  The pages' "forward-chunked"
# comparison variant uses the sparse teacher cache but holds every student
# logit of the batch for its backward pass (glonce.com, body).  The same
# library holds exactly that grid when the stored-logits backward runs as one
# chunk of all N tokens: fp32 z [N, V] and bf16 dZ [N, V].  Both plans on the
# gptoss32k head at growing N; a point that would not fit is reported as
# skipped with what it needed.
GRID_TOKENS = (8192, 16384, 32768, 65536, 131072, 262144)


def run_sweep_grid(args):
    import dataclasses

    import torch

    import chunked_top_kl_gemm_b300 as kd
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kd.lib()
    peaks, _ = load_peaks()
    base = workloads.CONFIGS["gptoss32k"]
    for n in GRID_TOKENS:
        cfg = dataclasses.replace(base, N=n, name=f"gptoss32k_n{n}")
        for plan, chunk, flags in (("chunked (recompute, chunk 2048)", base.chunk, 0),
                                   ("full logits grid (stored logits, one chunk of N)", n,
                                    kd.KD_FLAG_STORE_LOGITS)):
            point = _sweep_point(kd, cfg, chunk, flags, dev, peaks)
            print(json.dumps({"sweep": "full_grid_vs_chunked", "workload": cfg.name,
                              "plan": plan, **point}), flush=True)


# ------------------------------------------------------------------ cache builder
def run_cache_build(args):
    """Throughput of the offline top-K cache builder on the workload's head
    (the teacher side: hidden [N,H] through W [V,H], K per token)."""
    import torch

    import chunked_top_kl_gemm_b300 as kd
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kd.lib()
    cfg = workloads.CONFIGS[args.config]
    chunk = args.chunk or cfg.chunk
    N, H, V, K = cfg.N, cfg.H, cfg.V, cfg.K
    inp = workloads.make_inputs(cfg, seed=0, device=dev)
    h, W = inp["hidden"], inp["W"]
    idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    val = torch.empty((N, K), dtype=torch.float32, device=dev)
    ws = torch.empty(kd.kd_topk_cache_workspace_size(N, H, V, K, chunk), dtype=torch.uint8,
                     device=dev)

    def step():
        kd.kd_topk_cache_build(h, W, K, chunk, topk_idx=idx, topk_logit=val, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(_gpu_id(0))
    clocks.start()
    time.sleep(0.2)
    torch.cuda.synchronize(dev)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    t = e0.elapsed_time(e1) / 1e3 / args.steps
    # per-kernel split from a separate pass with the event profiler on
    kd.kd_profile_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    kd.kd_profile_enable(False)
    prof = kd.kd_profile_read()
    peaks, _ = load_peaks()
    gemm_ms = prof["cache_gemm_logits"][0] / args.steps
    sel_ms = prof["cache_topk_select"][0] / args.steps
    # the select reads every stored logit once (4 N V bytes) on its fast path
    print(json.dumps({
        "metric": "tokens/s offline top-K cache build (N x H x V GEMM + top-K select)",
        "value": N / t, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "ms_per_step": t * 1e3, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name, "N": N, "H": H, "V": V, "K": K, "chunk": chunk},
        "gemm_tflops": 2.0 * N * H * V / (gemm_ms / 1e3) / 1e12,
        "gemm_frac_bf16_peak_burst": 2.0 * N * H * V / (gemm_ms / 1e3) / 1e12
                                     / float(peaks["bf16_tflops"]),
        "select_gbs": 4.0 * N * V / (sel_ms / 1e3) / 1e9,
        "select_frac_hbm": 4.0 * N * V / (sel_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
        "kernels": {k: {"ms_per_step": v[0] / args.steps} for k, v in prof.items() if v[1]},
        "kernels_source": "separate pass with the per-launch event profiler on",
        "clocks": clk,
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["kd", "reference"], default="kd")
    ap.add_argument("--config", default="gptoss32k")
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (profiling captures)")
    ap.add_argument("--cpu-sample", type=int, default=512)
    ap.add_argument("--ref-sample", type=int, default=64)
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--store-logits", action="store_true",
                    help="ablation: keep each chunk's logits instead of recomputing them")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="steps of the separate per-kernel profiling pass (default: --steps)")
    ap.add_argument("--min-scratch", action="store_true",
                    help="one chunk's dZ in the workspace: grad_W formed per chunk")
    ap.add_argument("--allow-short-warmup", action="store_true",
                    help="profiling runs only: honour --warmup below 3")
    ap.add_argument("--sweep-grid", action="store_true",
                    help="peak memory and throughput of the full logits grid (stored logits, one "
                         "chunk of all tokens) against the chunked plan, gptoss32k head, 8K-256K")
    ap.add_argument("--sweep", action="store_true",
                    help="peak memory and throughput over token counts and chunk sizes "
                         "(one JSON line per point)")
    ap.add_argument("--cache-build", action="store_true",
                    help="time the offline top-K cache builder on the workload's head")
    args = ap.parse_args(argv)
    if args.sweep:
        return run_sweep(args)
    if args.sweep_grid:
        return run_sweep_grid(args)
    if args.cache_build:
        return run_cache_build(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
