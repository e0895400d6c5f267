"""Benchmark: top-k sparse decode attention with GQA on GB300.

One step = one pass of the whole hot path over one batch: indexer score of every cached
token -> per-KV-head top-k -> gather of the selected K/V rows + exact attention (split-K
with log-sum-exp merge).  The workload is the Llama-3-8B-shaped GQA layer (batch 8, 32/8
heads, d = 128, bf16, T = 32768, top-1024), seeded synthetic inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Timing: W untimed warm-up steps, then K timed steps bracketed by a barrier and a device
synchronize; each step is timed with CUDA events on the launching stream, and a buffer
larger than L2 is written between timed steps (outside the events).  Rank 0 prints one
JSON line; under torchrun every rank runs its own full workload (weak scaling) and the
time is the maximum over ranks.

``--impl reference`` times the plain CPU oracle (the slow fp64 reference the kernels are
checked against) on this machine's host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-decode queries/s and achieved HBM GB/s (% of GB300 peak), T=32K–128K"
DEFAULT_WORKLOAD = "c2_llama3_8b_gqa"
PROFILES = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------------------- helpers


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of `value` over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / max_seconds


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.interval}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sm, mx, reasons = [], None, set()
        for ts, line in self.lines:
            if self.t0 is not None and not (self.t0 - 0.06 <= ts <= (self.t1 or ts) + 0.06):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
            for name, flag in zip(names, f[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_digest(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "top_sparse_decode_gqa_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str, digest: str):
    """Per-launch DRAM bytes from the committed ncu summary of this kernel and workload,
    or None when the summary is missing or the kernel source changed since it was taken."""
    path = os.path.join(PROFILES, f"{kernel}_{workload}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_digest") != digest:
            return None
        return int(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- the step


class SparseDecodeStep:
    """Device buffers and the launch sequence of one decode step (all inputs resident)."""

    def __init__(self, w, x, device):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        self.sd, self.w, self.dev = sd, w, device
        g = {k: v.to(device) for k, v in x.items() if isinstance(v, torch.Tensor)}
        self.q_idx, self.k_idx, self.q = g["q_idx"], g["k_idx"], g["q"]
        self.k, self.v = g["k"], g["v"]
        self.scores = torch.empty(w.B, w.Hkv, w.N, dtype=torch.float32, device=device)
        self.idx = torch.empty(w.B, w.Hkv, w.k, dtype=torch.int32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.args, self.out, self.lse, _ = sd.make_attend_args(
            self.q, self.k, self.v, self.idx, block=w.block, T=w.T, err_word=self.err)
        need = sd.sd_gather_attend_workspace_bytes(self.args)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        self.splits_merge = need > 0
        self.keys = self.k_idx
        if w.block > 1:
            self.keys = sd.sd_block_pool(self.k_idx, w.block)

    @property
    def launches_per_step(self) -> int:
        return 3 + (1 if self.splits_merge else 0)

    def run(self, ev=None):
        sd = self.sd
        if ev is not None:
            ev[0].record()
        sd.sd_index_score(self.q_idx, self.keys, self.scores, self.err)
        if ev is not None:
            ev[1].record()
        sd.sd_topk(self.scores, self.w.k, self.idx)
        if ev is not None:
            ev[2].record()
        sd.sd_gather_attend(self.args, self.ws)
        if ev is not None:
            ev[3].record()

    def algorithmic_bytes(self):
        """(index_score bytes per launch, whole-step bytes): what the method must move."""
        w = self.w
        e = w.elem_bytes
        key_bytes = w.B * w.Hkv * w.N * w.dI * (4 if w.block > 1 else e)
        q_idx_bytes = w.B * w.Hkv * w.V * w.dI * e
        score_bytes = w.B * w.Hkv * w.N * 4
        kv_bytes = w.B * w.Hkv * w.n_rows * w.d * e * 2
        q_bytes = w.B * w.V * w.Hq * w.d * e
        out_bytes = w.B * w.V * w.Hq * (w.d + 1) * 4 + w.B * w.Hkv * w.k * 4
        return key_bytes + q_idx_bytes + score_bytes, key_bytes + q_idx_bytes + kv_bytes + q_bytes + out_bytes


# ----------------------------------------------------------------------------- arms


def run_ours(args):
    import torch
    from top_sparse_decode_gqa_gb300 import build as cuda_build
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    if rank == 0:
        cuda_build.build()
    if world > 1:
        dist.barrier()
    w = WORKLOADS[args.workload]
    x = generate(w)
    step = SparseDecodeStep(w, x, device)
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(device)
    flush = torch.empty(2 * max(int(getattr(props, "L2_cache_size", 0)), 128 << 20), dtype=torch.uint8,
                        device=device)

    for _ in range(args.warmup):
        flush.zero_()
        step.run()
    torch.cuda.synchronize()
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error word {int(step.err.item())}")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    for i in range(K):
        flush.zero_()
        step.run(evs[i])
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()

    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    idx_ms = [e[0].elapsed_time(e[1]) for e in evs]
    topk_ms = [e[1].elapsed_time(e[2]) for e in evs]
    att_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_s = reduce_max(sum(step_ms) / 1e3, world, device)
    queries = w.queries_per_step * K
    value = aggregate(queries, world, total_s)
    ms_per_step = total_s * 1e3 / K

    # ---- end to end through the public API: host query in, host result out
    e2e = measure_e2e(step, w, x, flush, K=min(K, 200))

    peak, peak_kind = load_peaks()
    idx_bytes, step_bytes = step.algorithmic_bytes()
    idx_avg_s = statistics.mean(idx_ms) / 1e3
    achieved = idx_bytes / idx_avg_s / 1e9
    digest = source_digest("index_score.cu", "sd_common.cuh")
    traffic = profiled_traffic(args.workload, "index_score", digest)
    step_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "queries/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; integer indexer keys in [-8,8], N(0,1) q/K/V, 2% planted heavy hitters)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "T": w.T,
                   "k": w.k, "block": w.block, "V": w.V, "queries_per_step": w.queries_per_step,
                   "l2": "flushed between timed steps (write of 2x L2 outside the events)",
                   "parallelism": f"replica x{world} (each rank its own batch)"},
        "roofline": {"bound": "hbm", "kernel": "sd_index_score", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs", "traffic": traffic,
                     "algorithmic_bytes_per_launch": idx_bytes,
                     "avg_launch_us": round(idx_avg_s * 1e6, 2)},
        "step_roofline": {"bound": "hbm", "algorithmic_bytes": step_bytes,
                          "achieved": round(step_gbs, 1), "unit": "GB/s",
                          "frac": round(step_gbs / peak, 4),
                          "kernel_us": {"index_score": round(statistics.mean(idx_ms) * 1e3, 2),
                                        "topk": round(statistics.mean(topk_ms) * 1e3, 2),
                                        "gather_attend": round(statistics.mean(att_ms) * 1e3, 2)}},
        "e2e": e2e,
        "gpu_launches": step.launches_per_step * K,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_e2e(step, w, x, flush, K):
    """The same metric through the public calls with host buffers: every step copies the
    step's query tensors from pinned host memory, runs the three calls, and reads the
    result (out, lse, selected indices) back into pinned host memory."""
    import torch
    q_h = x["q"].pin_memory()
    qi_h = x["q_idx"].pin_memory()
    out_h = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    lse_h = torch.empty(step.lse.shape, dtype=step.lse.dtype).pin_memory()
    idx_h = torch.empty(step.idx.shape, dtype=step.idx.dtype).pin_memory()
    times = []
    for i in range(K + 3):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step.q.copy_(q_h, non_blocking=True)
        step.q_idx.copy_(qi_h, non_blocking=True)
        step.run()
        out_h.copy_(step.out, non_blocking=True)
        lse_h.copy_(step.lse, non_blocking=True)
        idx_h.copy_(step.idx, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if i >= 3:
            times.append(time.perf_counter() - t0)
    bi = q_h.numel() * q_h.element_size() + qi_h.numel() * qi_h.element_size()
    bo = sum(t.numel() * t.element_size() for t in (out_h, lse_h, idx_h))
    return {"value": round(w.queries_per_step * len(times) / sum(times), 1), "unit": "queries/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "timing": "host wall clock per step incl. copies and sync"}


def oracle_step(w, x, b0, b1):
    """The whole step on the CPU oracle for sequences [b0, b1)."""
    import oracle
    nb = b1 - b0
    q_idx = x["q_idx"][b0:b1].contiguous()
    keys = x["k_idx"][b0:b1].contiguous()
    if w.block > 1:
        keys = oracle.block_pool(keys, nb, w.Hkv, w.T, w.dI, w.block).astype("float32")
    s = oracle.index_score(q_idx, keys, nb, w.Hkv, w.V, w.N, w.dI)
    idx = oracle.topk(s, w.k)
    return oracle.gather_attend(x["q"][b0:b1].contiguous(), x["k"][b0:b1].contiguous(),
                                x["v"][b0:b1].contiguous(), idx, nb, w.V, w.Hq, w.Hkv, w.d, w.T,
                                w.k, w.block, 1.0 / math.sqrt(w.d))


def cpu_baseline(w, x, budget_s: float = 10.0, nseq: int = 1):
    """The oracle as it stands on the host cores, on a bounded sample of the workload:
    whole steps over `nseq` sequence(s) of the batch, repeated for about `budget_s`."""
    import oracle
    t0 = time.perf_counter()
    reps = 0
    while True:
        b0 = reps % w.B
        oracle_step(w, x, b0, min(w.B, b0 + nseq))
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(reps * nseq * w.V / el, 3), "unit": "queries/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} whole steps over {nseq} of {w.B} sequences of {w.name} ({el:.1f} s)"}


def run_reference(args):
    """The base contract's reference arm: the CPU oracle, timed on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    import oracle
    w = WORKLOADS[args.workload]
    x = generate(w)
    nseq = 1
    for _ in range(args.warmup):
        oracle_step(w, x, 0, nseq)
    times = []
    for i in range(args.steps):
        b0 = i % w.B
        t0 = time.perf_counter()
        oracle_step(w, x, b0, b0 + nseq)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = nseq * w.V * len(times) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "queries/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total * 1e3 / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "T": w.T,
                   "k": w.k, "sample": f"each step covers {nseq} of {w.B} sequences"},
        "cpu_baseline": {"value": round(value, 3), "unit": "queries/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": f"{nseq} of {w.B} sequences per step"},
        "e2e": {"value": round(value, 3), "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
