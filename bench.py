#!/usr/bin/env python3
"""Benchmark of the persistent decode megakernel: batch-1 decode of the Llama-3.2-1B-shaped
decoder (16 layers, hidden 2048, 32/8 heads, FFN 8192, vocab 128256, tied, bf16 weights),
KV cache prefilled to 512 positions.

One "step" = one decode step of the whole model = one launch of the resident grid.
Prints one JSON line.

  value     device time per token (us/token) from CUDA events around each launch on the
            launching stream, inputs resident in HBM (weights 2.47 GB >> 129 MB L2, so every
            step streams its weights from HBM; no L2 flush is needed)
  e2e       the same metric through the synchronous C-ABI call mk_decode_step: host token and
            position in, greedy next token (and the device error word) copied back each step
  e2e_chained  the same through mk_decode_steps: all timed steps in one call, each step's greedy
            token feeding the next on the device, tokens copied back once at the end
  persistent   ONE launch running the same number of steps (mk_decode_persistent_*): device
            time per token from an event pair around the launch, its end-to-end time, and the
            HBM fraction of the per-token bytes at that time
  roofline  algorithmic bytes per step (weights + KV read + KV written) / median step time,
            against the measured HBM copy bandwidth
  cpu_baseline  the CPU oracle on the host cores, on a bounded sample (whole decode steps)

--impl reference runs the CPU oracle (the reference arm of this build) on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llama1b_ctx512"
METRIC = "batch-1 decode us/token (Llama-3.2-1B shape, bf16 weights/KV); achieved HBM GB/s vs GB300 peak"
KERNEL_SRC = os.path.join(ROOT, "persistent_megakernel_decode_sm_gb300", "csrc", "mk_kernel.cu")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _code_only(text: str) -> str:
    """C++ source without comments and blank space: edits to comments do not change the code."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':   # string literal, kept whole
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_hash() -> str:
    """Hash of the kernel's code (mk_kernel.cu + mk_internal.h, comments and spacing ignored)."""
    h = hashlib.sha256()
    for name in ("mk_kernel.cu", "mk_internal.h"):
        with open(os.path.join(os.path.dirname(KERNEL_SRC), name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_record(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this very kernel
    source (its hash is recorded beside the figure); None otherwise."""
    p = os.path.join(ROOT, "profiles", f"megakernel_{workload}_traffic.txt")
    if not os.path.exists(p):
        return None
    rec = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("kernel_hash") != kernel_hash():
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def job_time_ms(total_ms: float, world: int) -> float:
    """The job's timed region: the maximum over ranks of each rank's timed region (ms).  Every rank
    calls it (a collective when world > 1; the tensor lives where the process group's backend
    wants it)."""
    if world <= 1:
        return float(total_ms)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value_us_per_token(job_ms: float, steps: int, batch: int, world: int) -> float:
    """Whole-job figure of N independent replicas: the job's time over every token all ranks
    decoded (each rank decodes `batch` tokens per step)."""
    return job_ms * 1000.0 / steps / (batch * world)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def oracle_step_timer(cfg, kv_len, seed, threads, steps, warmup):
    """Times whole oracle decode steps of the workload on the host; returns (us per token list, cores)."""
    import numpy as np  # noqa: F401
    import oracle
    from oracle import HostWeights, Oracle, kv_to_host
    from workload import make_weights, prefilled_kv, token_ids
    cores = oracle.set_threads(threads)
    w = make_weights(cfg, seed=seed, device="cpu")
    hw = HostWeights(w)
    kh, vh = kv_to_host(prefilled_kv(cfg, [kv_len], seed=seed))
    del w
    orc = Oracle("f32")
    toks = token_ids(cfg, warmup + steps, seed=seed, tag="bench")
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        orc.decode_step(cfg, hw, kh, vh, [toks[i]], [kv_len + (i % (cfg.max_seq - kv_len))])
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt * 1e6 / cfg.batch)
    return times, cores


def run_reference(args, rank, world):
    from workload import get_workload
    wl = get_workload(WORKLOAD)
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    steps, warm = max(1, args.steps), max(0, args.warmup)
    # bounded sample: whole decode steps of the workload, capped so the run stays within minutes
    cap = int(os.environ.get("MK_REF_MAX_STEPS", "20"))
    steps = min(steps, cap)
    warm = min(warm, 1)
    times, cores = oracle_step_timer(wl.cfg, wl.kv_len[0], 0, threads, steps, warm)
    v = statistics.mean(times)
    sample = f"{len(times)} whole decode steps (+{warm} warm-up) of {WORKLOAD} at pos 512+"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/token", "n_gpus": args.gpus,
            "steps": len(times), "warmup": warm, "ms_per_step": v * wl.cfg.batch / 1000.0,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": WORKLOAD, "batch": 1, "kv_len": 512,
                                            "weights": "bf16", "kv": "bf16"},
            "cpu_baseline": {"value": v, "unit": "us/token", "cores": cores, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model()},
            "e2e": {"value": v, "unit": "us/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-steps", type=int, default=3)
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--attn-chunk", type=int, default=0,
                    help="KV positions per split-K attention tile (0: the scheduler's rule)")
    ap.add_argument("--sync", default="tags", choices=["tags", "counters"],
                    help="how consumers learn their inputs are ready (mk_set_sync)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    W = max(3, args.warmup)
    K = max(1, args.steps)

    import persistent_megakernel_decode_sm_gb300 as mk
    from workload import get_workload, make_weights, prefilled_kv, token_ids

    wl = get_workload(args.workload)
    cfg = wl.cfg
    w = make_weights(cfg, seed=0, device="cuda")
    kv = prefilled_kv(cfg, wl.kv_len, seed=0, device="cuda")
    S = mk.device_sm_count()
    stream = torch.cuda.Stream()
    # a batch of uneven lengths is planned for the positions this run reaches: attention chunks
    # past each sequence's window get no tile (variable-length re-planning)
    span = cfg.max_seq - max(wl.kv_len)
    windows = [min(cfg.max_seq, l + min(W + K, span) + 1) for l in wl.kv_len] if cfg.batch > 1 else None
    sched = mk.Schedule(cfg, S, attn_chunk=args.attn_chunk, kv_limit=windows)
    dec = mk.Decoder(sched, w, kv, stream=stream)
    dec.set_sync(args.sync)
    toks = token_ids(cfg, (W + K) * cfg.batch, seed=1, tag="bench")

    def args_for(i):
        t = toks[i * cfg.batch:(i + 1) * cfg.batch]
        p = [l + (i % span) for l in wl.kv_len]
        return t, p

    # ---- device-timed region: K launches, an event pair around each, on the launching stream
    for i in range(W):
        dec.launch(*args_for(i))
    dec.status()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            dec.launch(*args_for(W + i))
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    dec.status()
    total_ms = t_start.elapsed_time(t_end)
    per = [a.elapsed_time(b) * 1000.0 for a, b in ev]   # us per launch
    total_ms = job_time_ms(total_ms, world)   # max over ranks
    if world > 1:
        dist.barrier()
    med = statistics.median(per)
    p10 = sorted(per)[max(0, int(0.1 * K) - 1)]
    p90 = sorted(per)[min(K - 1, int(0.9 * K))]

    # ---- end-to-end through mk_decode_step (host token in, greedy token out)
    tok = toks[:cfg.batch]
    torch.cuda.synchronize()
    e2e_times = []
    for i in range(W + K):
        p = [l + (i % span) for l in wl.kv_len]
        t0 = time.perf_counter()
        tok = dec.step(tok, p)
        dt = time.perf_counter() - t0
        if i >= W:
            e2e_times.append(dt * 1e6)
    e2e_us = statistics.mean(e2e_times) / cfg.batch

    # ---- end-to-end through mk_decode_steps: n chained steps per call (each step's greedy token
    # feeds the next on the device), one host synchronisation per call
    n_chain = min(K, span)
    tokens_dev = torch.empty(n_chain * cfg.batch, dtype=torch.int32, device=dec.logits.device)
    dec.steps(toks[:cfg.batch], list(wl.kv_len), min(W, n_chain), tokens_dev=tokens_dev)   # warm-up call
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dec.steps(toks[:cfg.batch], list(wl.kv_len), n_chain, tokens_dev=tokens_dev)
    chained_us = (time.perf_counter() - t0) * 1e6 / n_chain / cfg.batch

    # ---- one persistent launch of n_chain steps (mk_decode_persistent_*): the resident grid runs
    # every step, each step's greedy token feeding the next on the device; device time from an
    # event pair around the launch, end-to-end time around start + wait (tokens read back once)
    dec.persistent(toks[:cfg.batch], list(wl.kv_len), min(W, n_chain), tokens_dev=tokens_dev)   # warm-up
    torch.cuda.synchronize()
    pe0 = torch.cuda.Event(enable_timing=True)
    pe1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    pe0.record(stream)
    dec.persistent_start(toks[:cfg.batch], list(wl.kv_len), n_chain, tokens_dev=tokens_dev)
    pe1.record(stream)
    ran = len(dec.persistent_wait())
    persistent_e2e_us = (time.perf_counter() - t0) * 1e6 / ran / cfg.batch
    persistent_dev_us = pe0.elapsed_time(pe1) * 1000.0 / ran / cfg.batch

    pos_mid = [l + 0 for l in wl.kv_len]
    step_bytes = cfg.step_bytes(pos_mid)
    peak, peak_kind = peaks()
    mean_us = statistics.mean(per)
    achieved = step_bytes / (mean_us * 1e-6) / 1e9   # per launch: algorithmic bytes / mean launch time
    value = job_value_us_per_token(total_ms, K, cfg.batch, world)

    line = {
        "metric": METRIC, "value": value, "unit": "us/token", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": total_ms / K, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "batch": cfg.batch, "kv_len": wl.kv_len[0] if cfg.batch == 1 else wl.kv_len,
                   "weights": "bf16", "kv": "bf16", "sm_count": S, "parallelism": "replicas" if world > 1 else "single",
                   "sync": args.sync, "attn_chunk": sched.attn_chunk, "kv_windows": windows,
                   "l2": f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB of weights and KV streamed per step)",
                   "step_us_mean": mean_us, "step_us_median": med, "step_us_p10": p10, "step_us_p90": p90},
        "e2e": {"value": e2e_us, "unit": "us/token", "h2d_bytes_per_step": 8 * cfg.batch,
                "d2h_bytes_per_step": 96},
        "e2e_chained": {"value": chained_us, "unit": "us/token", "steps_per_call": n_chain,
                        "h2d_bytes_per_step": 8 * cfg.batch / n_chain,
                        "d2h_bytes_per_step": (4 * cfg.batch * n_chain + 96) / n_chain},
        "persistent": {"value": persistent_dev_us, "unit": "us/token", "steps_per_launch": ran,
                       "e2e": persistent_e2e_us, "h2d_bytes_per_step": 8 * cfg.batch / ran,
                       "d2h_bytes_per_step": (4 * cfg.batch * ran + 96) / ran,
                       "frac": step_bytes / (persistent_dev_us * cfg.batch * 1e-6) / 1e9 / peak},
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic_record(args.workload), "peak_kind": peak_kind,
                     "algorithmic_bytes_per_step": step_bytes, "vs_nominal_8000": achieved / 8000.0},
        "clocks": clk.summary(),
    }
    dec.close()
    del w, kv
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle as it stands: OpenMP over matvec rows on every host core (per-row sums in the
        # same order), and single-threaded (one step)
        times, cores = oracle_step_timer(cfg, wl.kv_len[0], 0, os.cpu_count() or 1, args.cpu_steps, 1)
        single, _ = oracle_step_timer(cfg, wl.kv_len[0], 0, 1, 1, 0)
        line["cpu_baseline"] = {"value": statistics.mean(times), "unit": "us/token", "cores": cores,
                                "kind": "oracle", "cpu_model": cpu_model(),
                                "single_thread": {"value": statistics.mean(single), "unit": "us/token", "cores": 1,
                                                  "sample": f"{len(single)} whole decode step of {args.workload}"},
                                "sample": f"{len(times)} whole decode steps (+1 warm-up) of {args.workload}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
