#!/usr/bin/env python
"""Benchmark of the fused top-K KL distillation head (forward + backward).

One step = forward (kd_topk_kl_fwd), the mean-loss gradient on the device
(kd_topk_kl_mean_grad) and backward (kd_topk_kl_bwd) over one batch of
synthetic inputs of the named workload, all in the CUDA library, driven by the
product's token-sharded step (top_kl_loss_lm_b300.sharded.TokenShardedHead).
Default workload: the long-context gpt-oss-shaped head, N = 32,768 tokens
(batch 1 x seq 32,768), D = 2,880, V = 201,088, K = 64, T = 1, 2% of rows masked.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU fp64 oracle, timed on host cores
  python bench.py --sweep                # peak memory and rate for N = 4K ... 256K

Prints one JSON line (rank 0). With N > 1 (torchrun, one rank per GPU) the
ranks run data parallelism over a global batch of N x 32,768 tokens: each rank
its own 32,768 (weak scaling), the count of counted rows all-reduced before
the backward and dW (V x D fp32) and the loss sum all-reduced after it, inside
the timed step (NCCL). The barrier-bracketed time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused top-K KL head fwd+bwd tokens/s & TFLOP/s (% bf16 peak); peak GB vs N"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
GEMM_CATS = ("fwd_gemm", "dz_gemm", "dh_gemm", "dw_gemm")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gptoss_32k")
    ap.add_argument("--chunk", type=int, default=4096)
    ap.add_argument("--K", type=int, default=None, help="override the workload's teacher top-K")
    ap.add_argument("--T", type=float, default=None, help="override the workload's temperature")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--logits", action="store_true",
                    help="measure the loss from materialised logits (kd_topk_kl_logits) instead")
    ap.add_argument("--logits-rows", type=int, default=32768)
    ap.add_argument("--teacher-topk", action="store_true",
                    help="measure the teacher top-K cache producer (kd_teacher_topk) instead")
    ap.add_argument("--traffic-from", default=None,
                    help="write the per-launch DRAM traffic record of --workload (the small "
                         "profiling case) from these comma-separated ncu --csv logs and exit")
    return ap.parse_args()


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "dram_traffic_profile_medium.json")
# the sources of the loss step's kernels (the logits and teacher-cache kernels
# are not launched by the step, so their files do not invalidate its record)
KERNEL_SOURCES = ("kd_lib.cu", "kd_gemm.cuh", "kd_aux.cuh", "kd_ptx.cuh", "kd_sched.h")
# template argument of kd_gemm_kernel -> category of the library's launch timing
GEMM_EPI = {"0": "fwd_gemm", "1": "dz_gemm", "2": "dh_gemm", "3": "dw_gemm", "4": "topk_gemm",
            "5": "topk_gemm"}


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: comments and runs of whitespace are
    dropped first, so a record stays valid across comment-only edits."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "top_kl_loss_lm_b300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def kernel_category(name: str):
    import re
    m = re.search(r"kd_gemm_kernel<(\d)", name)
    if m:
        return GEMM_EPI[m.group(1)]
    for key, cat in (("kd_logits_kernel", "logits"), ("kd_topk_select_kernel", "topk_select"),
                     ("kd_cand_select_kernel", "topk_select"), ("kd_row_threshold_kernel", "topk_select"),
                     ("kd_transpose_kernel", "transpose"), ("kd_gather_rows_kernel", "transpose")):
        if key in name:
            return cat
    return None


def traffic_from_ncu_csv(csv_paths, workload: str, chunk: int) -> dict:
    """DRAM bytes of every captured launch (dram__bytes_read.sum + dram__bytes_write.sum),
    in capture order, from ncu csv exports of the small profiling case: either the long
    form (--csv --metrics ..., one row per metric) or the wide form of
    `ncu -i report --page raw --csv` (one row per launch, a units row under the header)."""
    import csv
    scale_of = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9}
    launches = []
    for path in csv_paths:
        with open(path) as f:
            rows = [r for r in csv.reader(f) if r]
        start = next(i for i, r in enumerate(rows) if r[0] == "ID")
        hdr = rows[start]
        body = rows[start + 1:]
        if "dram__bytes_read.sum" in hdr:      # wide
            units = dict(zip(hdr, body[0]))
            for r in body[1:]:
                d = dict(zip(hdr, r))
                cat = kernel_category(d["Kernel Name"])
                if cat is None:
                    continue
                b = sum(float(d[m].replace(",", "")) * scale_of.get(units[m].lower(), 1)
                        for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"))
                launches.append({"cat": cat, "bytes": b})
            continue
        per = {}
        for r in body:                          # long
            d = dict(zip(hdr, r))
            cat = kernel_category(d.get("Kernel Name", ""))
            if cat is None or d.get("Metric Name") not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                continue
            e = per.setdefault(int(d["ID"]), {"cat": cat, "bytes": 0.0})
            e["bytes"] += float(d["Metric Value"].replace(",", "")) * scale_of.get(
                d.get("Metric Unit", "byte").lower(), 1)
        launches += [per[k] for k in sorted(per)]
    from workloads import CONFIGS
    case = dict(CONFIGS[workload], chunk_tokens=chunk)
    return {"source_hash": kernel_source_hash(), "workload": workload, "case": case,
            "launches": launches}


def recorded_traffic(kernel: str, p, chunk: int):
    """DRAM bytes per launch of `kernel` at the bench's workload, scaled from the
    small-case record, or None when the record is missing, was taken from other
    kernel sources, or its case does not have the bench's D, K and launch sizes.

    The small case runs the same launches (4,096 rows per forward / dZ / dH
    launch, 8,192 tokens per dW launch) over a smaller vocabulary, so a launch's
    traffic scales with V. dW's first launch of a step stores and the later ones
    add: the per-launch figure weights the captured store and add launches as
    the bench's step does."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    case = rec.get("case", {})
    if (rec.get("source_hash") != kernel_source_hash() or case.get("D") != p.D
            or case.get("K") != p.K or case.get("chunk_tokens") != chunk):
        return None
    got = [x["bytes"] for x in rec.get("launches", []) if x["cat"] == kernel]
    if not got:
        return None
    if kernel == "dw_gemm" and len(got) >= 2:
        groups = -(-p.N // (2 * chunk))
        per = (got[0] + (groups - 1) * (sum(got[1:]) / len(got[1:]))) / groups
    else:
        per = sum(got) / len(got)
    return per * p.V / case["V"]


def issued_width_factor(kernel: str, D: int, V: int) -> float:
    """Tensor-core work a GEMM issues per useful FLOP. Every tile is one MMA
    instruction wide in its output columns, and an instruction narrower than 256
    columns takes as long as a 256-wide one (240 and 256 measured equal; 11 x 256
    tiles take 11/12 of the time of 12), so a launch costs ceil(n / 256) x 256
    columns for n useful ones: the hidden size D for dH and dW (2,880 -> 3,072),
    the vocabulary V for the forward and dZ."""
    n = D if kernel in ("dh_gemm", "dw_gemm") else V
    return (-(-n // 256) * 256) / n


def dense_grid_bytes(n_tokens: int, vocab: int, bytes_per_elem: int) -> int:
    """Bytes of one dense tokens x vocabulary grid: what the fused head never allocates."""
    return int(n_tokens) * int(vocab) * int(bytes_per_elem)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def per_clock_fraction(achieved: float, peak: float, clocks, peaks) -> float | None:
    """achieved / peak with both taken per MHz of SM clock: the kernel's rate at
    the median SM clock sampled during the timed region against the sustained
    peak at the median clock under load recorded with it. Under the power cap
    the clock differs from box to box, while the work done per clock does not.
    None when the timed region was too short for five clock samples."""
    try:
        if int(clocks.get("samples", 0)) < 5:
            return None
        mhz = float(clocks["sm_mhz"])
        peak_mhz = float(peaks["clocks_under_load"]["sm_mhz_median"])
    except (AttributeError, KeyError, TypeError, ValueError):
        return None
    if mhz <= 0 or peak_mhz <= 0:
        return None
    return (achieved / mhz) / (peak / peak_mhz)


def workload_desc(p, chunk):
    return {
        "workload": f"{p.name}: N={p.N} tokens, D={p.D}, V={p.V}, K={p.K}, T={p.T}",
        "N": p.N, "D": p.D, "V": p.V, "K": p.K, "T": p.T,
        "masked_rows": int(p.N - int(p.mask.sum().item())),
        "chunk_tokens": chunk,
        "l2": "inputs larger than L2 (W alone is %.2f GB; every pass streams it)" % (p.V * p.D * 2 / 1e9),
        "inputs": "H ~ N(0,1), W ~ N(0,1/D) in bf16; teacher ids distinct uniform, logits N(0,4)+Gumbel sorted",
    }


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader",
                                          "-lms", "200"] + sel, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def mhz(x):
            try:
                return float(x.split()[0])
            except Exception:
                return None

        sm = [mhz(r[1]) for r in rows if mhz(r[1])]
        mx = [mhz(r[2]) for r in rows if mhz(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s in sm if mx and s > 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Largest elapsed time over the ranks (one float64 all-reduce; identity at world 1)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_rate(units_per_rank: int, world: int, steps: int, ms: float) -> float:
    """Whole-job rate: units every rank processed over the slowest rank's time."""
    return world * units_per_rank * steps / (ms / 1000.0)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------------- CPU oracle

ORACLE_ROWS_PER_CALL = 64   # the same batch for the in-line cpu_baseline and --impl reference


def oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        return max(int(d.get("num_threads", 1)) for d in threadpool_info()) or os.cpu_count()
    except Exception:
        return os.cpu_count()


class OracleSample:
    """The CPU oracle (fwd + bwd over the full vocabulary) on seeded samples of a
    workload's rows, ORACLE_ROWS_PER_CALL rows a call. The oracle is row-additive,
    so rows per second is its tokens per second."""

    def __init__(self, p, seed: int = 0):
        import numpy as np
        self.np = np
        self.p = p
        self.W64 = p.W.double().cpu().numpy()      # input conversion, outside the timed part
        self.H = p.H.cpu()
        self.m = p.mask.cpu().numpy()
        self.idx = p.idx.cpu().numpy()
        self.t = p.t.double().cpu().numpy()
        self.nv = max(int(self.m.sum()), 1)
        self.rng = np.random.default_rng(seed)

    def call(self) -> float:
        """One oracle call on a fresh sample; returns its seconds."""
        import oracle
        np, p = self.np, self.p
        rows = np.sort(self.rng.choice(p.N, size=min(ORACLE_ROWS_PER_CALL, p.N), replace=False))
        Hs = self.H[rows].double().numpy()
        t0 = time.perf_counter()
        oracle.kd_forward(Hs, self.W64, self.idx[rows], self.t[rows], self.m[rows], p.T)
        oracle.kd_backward(Hs, self.W64, self.idx[rows], self.t[rows], self.m[rows], p.T,
                           self.m[rows] / self.nv)
        return time.perf_counter() - t0


def oracle_rate(p, seconds: float, seed: int = 0, max_calls: int = 16):
    """Oracle fwd+bwd on seeded row samples for about `seconds`; (tokens/s, rows, secs, threads)."""
    o = OracleSample(p, seed)
    o.call()                     # first call pays BLAS start-up; not timed
    calls, secs = 0, 0.0
    while secs < seconds and calls < max_calls:
        secs += o.call()
        calls += 1
    rows = calls * min(ORACLE_ROWS_PER_CALL, p.N)
    return rows / secs, rows, secs, oracle_threads()


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from workloads import config_problem
    p = config_problem(args.workload, seed=args.seed, device="cpu", K=args.K, T=args.T)
    o = OracleSample(p, args.seed)
    times = []
    for i in range(args.warmup + args.steps):
        dt = o.call()
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    rows = min(ORACLE_ROWS_PER_CALL, p.N)
    rate = rows * args.steps / total
    sample = (f"{rows} seeded rows of {p.N} per step (fwd+bwd over the full V={p.V}); "
              f"the oracle is row-additive so rows/s is its tokens/s")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_desc(p, args.chunk),
        "parallelism": "none (CPU oracle, rank 0 only)",
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": f"CPU fp64 oracle (numpy/OpenBLAS) on host cores; one step = {rows} rows",
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- CUDA path

class Head:
    """One rank's device buffers and its step, through the product's
    TokenShardedHead (all collectives are no-ops at world size 1)."""

    def __init__(self, p, chunk, group=None):
        from top_kl_loss_lm_b300.sharded import TokenShardedHead
        self.p = p
        self.chunk = chunk
        self.h = TokenShardedHead(p.N, p.D, p.V, p.K, p.T, p.H.device, chunk_tokens=chunk, group=group)
        self.ws = self.h.ws

    def step(self, H=None, idx=None, t=None, mask=None):
        p = self.p
        return self.h.step(p.H if H is None else H, p.W, p.idx if idx is None else idx,
                           p.t if t is None else t, p.mask if mask is None else mask)


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist

    from top_kl_loss_lm_b300 import binding
    from workloads import config_problem

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # weak scaling: each rank holds its own N-token slice of the global batch
    p = config_problem(args.workload, seed=args.seed + rank, device=dev, K=args.K, T=args.T)
    head = Head(p, args.chunk)
    N, D, V = p.N, p.D, p.V
    flops_step = 8.0 * N * D * V
    stream = torch.cuda.current_stream()

    def timed(steps, fn):
        """Device time (ms) of `steps` calls of fn on this stream, max over ranks."""
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return max_over_ranks(e0.elapsed_time(e1), world, dev)

    for _ in range(max(args.warmup, 3)):
        head.step()
    st = binding.kd_get_status()
    if st != 0:
        raise RuntimeError(f"device status {binding.STATUS.get(st, st)} after warm-up")

    # ------------------------------------------------ device-timed region (no per-kernel events)
    sampler = ClockSampler(local)
    torch.cuda.reset_peak_memory_stats()
    sampler.start()
    ms = timed(args.steps, head.step)
    # per-kernel times: a second pass of the same length with an event pair around every
    # launch, started right after the first (a pause lets the power-capped clock recover,
    # which would flatter the kernels timed after it)
    prof_steps = args.steps
    binding.kd_debug_profile(True)
    prof_ms = timed(prof_steps, head.step)
    prof = binding.kd_debug_profile_read()
    binding.kd_debug_profile(False)
    clocks = sampler.stop()
    st = binding.kd_get_status()
    if st != 0:
        raise RuntimeError(f"device status {binding.STATUS.get(st, st)} in the timed region")
    peak_mem = torch.cuda.max_memory_allocated()
    value = job_rate(N, world, args.steps, ms)
    tflops = job_rate(flops_step, world, args.steps, ms) / 1e12

    # ------------------------------------------------ end to end from host buffers
    # Every step copies its own inputs from pinned host memory and reads its results
    # back. The copies run on a second stream into two alternating input buffers, so
    # the inputs of step i + 1 travel while step i computes, as a training loop
    # prefetches its next batch; step i waits for its own copies only.
    e2e = None
    if not args.no_e2e:
        hH = p.H.cpu().pin_memory()
        hidx = p.idx.cpu().pin_memory()
        ht = p.t.cpu().pin_memory()
        hm = p.mask.cpu().pin_memory()
        hloss = torch.empty(N, dtype=torch.float32).pin_memory()
        hsum = torch.empty(1, dtype=torch.float64).pin_memory()
        hnv = torch.empty(1, dtype=torch.int64).pin_memory()
        bufs = [(torch.empty_like(p.H), torch.empty_like(p.idx), torch.empty_like(p.t),
                 torch.empty_like(p.mask)) for _ in range(2)]
        copy_stream = torch.cuda.Stream(device=dev)
        ready = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        for ev in free:
            ev.record(stream)

        def copy_in(i):
            b = bufs[i % 2]
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(free[i % 2])   # the step that last read this buffer is done
                for dst, src in zip(b, (hH, hidx, ht, hm)):
                    dst.copy_(src, non_blocking=True)
                ready[i % 2].record(copy_stream)

        def e2e_run(steps):
            start = torch.cuda.Event()
            start.record(stream)
            copy_stream.wait_event(start)   # no copy of this run starts before the timed region
            copy_in(0)
            for i in range(steps):
                if i + 1 < steps:
                    copy_in(i + 1)
                stream.wait_event(ready[i % 2])
                Hb, ib, tb, mb = bufs[i % 2]
                loss_sum, nv = head.step(H=Hb, idx=ib, t=tb, mask=mb)
                free[i % 2].record(stream)
                hloss.copy_(head.h.loss, non_blocking=True)
                hsum.copy_(loss_sum, non_blocking=True)
                hnv.copy_(nv, non_blocking=True)

        e2e_run(2)
        ems = timed(1, lambda: e2e_run(args.steps))
        h2d = sum(x.numel() * x.element_size() for x in (hH, hidx, ht, hm))
        d2h = hloss.numel() * 4 + 8 + 8
        e2e = {"value": job_rate(N, world, args.steps, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "every step copies H, teacher ids/logits and mask from pinned host memory "
                       "(on a second stream, into alternating buffers, overlapping the previous "
                       "step) and reads back the per-row loss, loss sum and n_valid; W, dH, dW "
                       "stay resident"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    # ------------------------------------------------ roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    kernels = {}
    for c, (tot, n) in prof.items():
        if n == 0:
            continue
        entry = {"ms_per_step": tot / prof_steps, "launches_per_step": n / prof_steps, "share": None}
        if c in GEMM_CATS:
            entry["tflops"] = 2.0 * N * D * V * prof_steps / (tot / 1000.0) / 1e12
            entry["issued_per_useful"] = issued_width_factor(c, D, V)
        kernels[c] = entry
    total_k = sum(prof[c][0] for c in prof)
    for c in kernels:
        kernels[c]["share"] = prof[c][0] / total_k if total_k else None
    dom = max((c for c in kernels if c in GEMM_CATS), key=lambda c: prof[c][0])
    tot, n = prof[dom]
    flops_per_launch = 2.0 * N * D * V * prof_steps / n
    achieved = flops_per_launch / (tot / n / 1000.0) / 1e12
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    traffic = recorded_traffic(dom, p, args.chunk)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_sus,
                "unit": "TFLOP/s", "frac": achieved / peak_sus, "traffic": traffic,
                "traffic_unit": "bytes per launch (dram read + write, ncu, scaled from the small "
                                "capture in profiles/)",
                "peak_kind": f"sustained bf16 dense ({peak_src}); kernel timed inside a long step",
                "frac_of_burst": achieved / peak_burst,
                "flops_per_launch": flops_per_launch,
                "issued_per_useful": issued_width_factor(dom, D, V),
                "frac_issued": achieved * issued_width_factor(dom, D, V) / peak_sus,
                "frac_per_clock": per_clock_fraction(achieved, peak_sus, clocks, peaks),
                "timing": f"per-launch CUDA events over a second {prof_steps}-step pass right after "
                          f"the timed one ({prof_ms / prof_steps:.2f} ms/step with the events)"}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, nrows, secs, threads = oracle_rate(p, args.cpu_seconds, seed=args.seed)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{nrows} seeded rows of {N} in {ORACLE_ROWS_PER_CALL}-row calls "
                         f"(fwd+bwd over the full V={V}), {secs:.1f} s; W converted to fp64 "
                         f"outside the timed part"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_desc(p, args.chunk),
        "parallelism": (f"dp{world}: token-sharded, {N} tokens per rank, dW / n_valid / loss sum "
                        f"all-reduced (NCCL) inside the step") if world > 1 else "single GPU",
        "tflops": tflops, "frac_of_bf16_peak": {"burst": tflops / world / peak_burst,
                                                "sustained": tflops / world / peak_sus},
        "peak_mem_gb": peak_mem / 1e9,
        "roofline": roofline, "kernels": kernels,
        "gpu_launches": int(round(sum(n for _, n in prof.values()) * args.steps / prof_steps)),
        "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


LOGITS_METRIC = "top-K KL + logit gradient from materialised logits: tokens/s; HBM GB/s"


def run_logits(args):
    """The forward-chunked form: loss and dZ from bf16 logits already in HBM.

    One step = one kd_topk_kl_logits call over N rows of V logits (the
    gpt-oss head's vocabulary) with the gradient written to a separate buffer.
    """
    import torch

    from top_kl_loss_lm_b300 import binding
    from workloads import make_problem, mean_upstream_grad

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    N, V = args.logits_rows, 201088
    K = args.K or 64
    T = args.T or 1.0
    p = make_problem(N, 8, V, K, T, seed=args.seed, mask="frac", mask_frac=0.02, device=dev,
                     name="gptoss_logits")
    g = torch.Generator(device=dev).manual_seed(args.seed + 7)
    Z = torch.empty(N, V, dtype=torch.bfloat16, device=dev)
    for r0 in range(0, N, 4096):
        r1 = min(N, r0 + 4096)
        Z[r0:r1] = (3.0 * torch.randn(r1 - r0, V, device=dev, generator=g)).to(torch.bfloat16)
    dZ = torch.empty_like(Z)
    ws = torch.empty(binding.kd_topk_kl_logits_workspace_size(N, K), dtype=torch.uint8, device=dev)
    loss = torch.empty(N, device=dev)
    lse = torch.empty(N, device=dev)
    nv = torch.empty(1, dtype=torch.int64, device=dev)
    dl = mean_upstream_grad(p.mask).to(dev)

    def step():
        binding.kd_topk_kl_logits(Z, p.idx, p.t, p.mask, T, loss, lse, nv, ws, dloss=dl, dZ=dZ)

    for _ in range(max(args.warmup, 3)):
        step()
    if binding.kd_get_status() != 0:
        raise RuntimeError("device status after warm-up")
    sampler = ClockSampler(0)
    torch.cuda.synchronize()
    sampler.start()
    binding.kd_debug_profile(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    prof = binding.kd_debug_profile_read()
    binding.kd_debug_profile(False)
    if binding.kd_get_status() != 0:
        raise RuntimeError("device status in the timed region")
    ms = e0.elapsed_time(e1)
    tot, n = prof["logits"]
    # algorithmic bytes of one launch: logits read once, dZ written once, the sorted
    # teacher pairs read, and per row: mask, dloss, entropy read, loss and lse written
    per_launch = N * V * 2 * 2 + N * K * 8 + N * (1 + 4 + 4 + 4 + 4)
    achieved = per_launch / (tot / n / 1000.0) / 1e9
    peaks, src = load_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    cpu = None
    if not args.no_cpu_baseline:
        import numpy as np

        import oracle
        rng = np.random.default_rng(args.seed)
        idx, t, m = p.idx.cpu().numpy(), p.t.double().cpu().numpy(), p.mask.cpu().numpy()
        done, secs = 0, 0.0
        while secs < args.cpu_seconds and done < 4096:
            rows = np.sort(rng.choice(N, size=64, replace=False))
            Zs = Z[torch.as_tensor(rows, device=dev)].double().cpu().numpy()
            t0 = time.perf_counter()
            oracle.kd_from_logits(Zs, idx[rows], t[rows], m[rows], T, m[rows] / max(int(m.sum()), 1))
            secs += time.perf_counter() - t0
            done += len(rows)
        try:
            from threadpoolctl import threadpool_info
            threads = max(int(d.get("num_threads", 1)) for d in threadpool_info())
        except Exception:
            threads = os.cpu_count()
        cpu = {"value": done / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{done} seeded rows of {N} in 64-row calls ({secs:.1f} s); the oracle is "
                         f"row-additive, so rows/s is its tokens/s"}
    line = {
        "metric": LOGITS_METRIC, "value": args.steps * N / (ms / 1000.0), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"gptoss_logits: N={N} rows of V={V} bf16 logits, K={K}, T={T}",
                   "N": N, "V": V, "K": K, "T": T, "masked_rows": int(N - int(p.mask.sum().item())),
                   "l2": "inputs larger than L2 (the logits are %.1f GB)" % (N * V * 2 / 1e9),
                   "inputs": "logits 3*N(0,1) in bf16; teacher ids distinct uniform, logits "
                             "N(0,4)+Gumbel sorted"},
        "roofline": {"bound": "hbm", "kernel": "kd_logits_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None,
                     "traffic_unit": "bytes per launch (dram read + write, ncu)",
                     "peak_kind": f"HBM copy bandwidth ({src})",
                     "bytes_per_launch": per_launch},
        "kernels": {c: {"ms_per_step": prof[c][0] / args.steps,
                        "launches_per_step": prof[c][1] / args.steps}
                    for c in prof if prof[c][1]},
        "gpu_launches": int(sum(c[1] for c in prof.values())),
        "clocks": clocks, "e2e": None, "cpu_baseline": cpu,
        "note": "secondary line (the next row after the fused head); e2e omitted: the logits "
                "would be copied from host memory every step",
    }
    print(json.dumps(line), flush=True)
    return 0


TOPK_METRIC = "teacher top-K cache (logit GEMM + exact per-row top-K): rows/s; GEMM TFLOP/s"


def run_teacher_topk(args):
    """The offline step: the teacher's top-K ids and logits of H W^T for N rows."""
    import torch

    from top_kl_loss_lm_b300 import binding
    from workloads import make_problem

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    N, D, V = args.logits_rows, 2880, 201088
    K = args.K or 100
    p = make_problem(N, D, V, 1, 1.0, seed=args.seed, device=dev, name="gptoss_teacher")
    ws = torch.empty(binding.kd_teacher_topk_workspace_size(N, D, V, K), dtype=torch.uint8,
                     device=dev)
    ids = torch.empty(N, K, dtype=torch.int32, device=dev)
    vals = torch.empty(N, K, device=dev)

    def step():
        binding.kd_teacher_topk(p.H, p.W, ids, vals, ws)

    for _ in range(max(args.warmup, 3)):
        step()
    if binding.kd_get_status() != 0:
        raise RuntimeError("device status after warm-up")
    sampler = ClockSampler(0)
    torch.cuda.synchronize()
    sampler.start()
    binding.kd_debug_profile(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    prof = binding.kd_debug_profile_read()
    binding.kd_debug_profile(False)
    if binding.kd_get_status() != 0:
        raise RuntimeError("device status in the timed region")
    ms = e0.elapsed_time(e1)
    gemm_ms = prof["topk_gemm"][0] / args.steps
    sel_ms = prof["topk_select"][0] / args.steps
    flops = 2.0 * N * D * V
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = flops / (gemm_ms / 1000.0) / 1e12
    cpu = None
    if not args.no_cpu_baseline:
        import numpy as np

        import oracle
        W64 = p.W.double().cpu().numpy()
        rng = np.random.default_rng(args.seed)
        done, secs = 0, 0.0
        while secs < args.cpu_seconds and done < 4096:
            rows = np.sort(rng.choice(N, size=64, replace=False))
            Hs = p.H[torch.as_tensor(rows, device=dev)].double().cpu().numpy()
            t0 = time.perf_counter()
            oracle.teacher_topk(Hs, W64, K)
            secs += time.perf_counter() - t0
            done += len(rows)
        try:
            from threadpoolctl import threadpool_info
            threads = max(int(d.get("num_threads", 1)) for d in threadpool_info())
        except Exception:
            threads = os.cpu_count()
        cpu = {"value": done / secs, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "sample": f"{done} seeded rows of {N} in 64-row calls ({secs:.1f} s)"}
    line = {
        "metric": TOPK_METRIC, "value": args.steps * N / (ms / 1000.0), "unit": "rows/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"gptoss_teacher: N={N} rows, D={D}, V={V}, K={K}",
                   "N": N, "D": D, "V": V, "K": K,
                   "l2": "inputs larger than L2 (W alone is 1.16 GB)",
                   "inputs": "H ~ N(0,1), W ~ N(0,1/D) in bf16"},
        "roofline": {"bound": "tensor", "kernel": "topk_gemm", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "frac_per_clock": per_clock_fraction(achieved, peak, clocks, peaks),
                     "traffic": None,
                     "peak_kind": f"sustained bf16 dense ({src})", "flops_per_step": flops},
        "kernels": {"topk_gemm": {"ms_per_step": gemm_ms}, "topk_select": {"ms_per_step": sel_ms}},
        "gpu_launches": int(sum(c[1] for c in prof.values())),
        "clocks": clocks, "e2e": None, "cpu_baseline": cpu,
        "note": "secondary line (the upstream caching step); e2e omitted",
    }
    print(json.dumps(line), flush=True)
    return 0


def run_sweep(args):
    """Peak device memory and rate vs N (D, V, K of the gpt-oss head)."""
    import torch

    from workloads import make_problem
    for N in (4096, 16384, 65536, 131072, 262144):
        torch.cuda.empty_cache()
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        p = make_problem(N, 2880, 201088, 64, 1.0, seed=args.seed, mask="frac", mask_frac=0.02,
                         device="cuda", name=f"sweep_{N}")
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        head = Head(p, args.chunk)
        for _ in range(2):
            head.step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        steps = 3
        e0.record()
        for _ in range(steps):
            head.step()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        # cross-check on the device: the drop in free memory since before the problem
        # was drawn (the caching allocator keeps its peak reservation) against torch's
        # own peak; the library allocates nothing outside the caller's tensors
        device_used = free0 - torch.cuda.mem_get_info()[0]
        print(json.dumps({"sweep": True, "N": N, "ms_per_step": ms, "tokens_per_s": N / (ms / 1e3),
                          "tflops": 8.0 * N * 2880 * 201088 / (ms / 1e3) / 1e12,
                          "peak_mem_gb": torch.cuda.max_memory_allocated() / 1e9,
                          "peak_reserved_gb": torch.cuda.max_memory_reserved() / 1e9,
                          "device_free_drop_gb": device_used / 1e9,
                          "workspace_gb": head.ws.numel() / 1e9,
                          "dense_grid_bf16_gb": dense_grid_bytes(N, 201088, 2) / 1e9}), flush=True)
        del head, p
        torch.cuda.empty_cache()


def main():
    args = parse()
    if args.traffic_from:
        rec = traffic_from_ncu_csv(args.traffic_from.split(","), args.workload, args.chunk)
        with open(TRAFFIC_RECORD, "w") as f:
            json.dump(rec, f, indent=1)
        print(json.dumps(rec))
        return 0
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.sweep:
        return run_sweep(args)
    if args.logits:
        return run_logits(args)
    if args.teacher_topk:
        return run_teacher_topk(args)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
