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
time is the maximum over ranks.  ``--gpus N`` (N > 1) run outside torchrun launches the N
local ranks itself (torch.distributed.run on 127.0.0.1), or fails when fewer than N GPUs
are visible.

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


class StepMarks:
    """CUDA events of one timed step: start/end of the step and a (before, after) pair
    around every launch of the step's dominant kernel, plus named phase boundaries."""

    def __init__(self, n_dominant: int, phases=()):
        import torch
        ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        self.start, self.end = ev(), ev()
        self.dom = [(ev(), ev()) for _ in range(n_dominant)]
        self.phase = {name: ev() for name in phases}

    def before(self, i):
        if i < len(self.dom):
            self.dom[i][0].record()

    def after(self, i):
        if i < len(self.dom):
            self.dom[i][1].record()

    def at(self, name):
        if name in self.phase:
            self.phase[name].record()

    def step_ms(self):
        return self.start.elapsed_time(self.end)

    def dominant_ms(self):
        return [a.elapsed_time(b) for a, b in self.dom]


def step_supported(w) -> bool:
    """Whether sd_decode_step (the whole step in one launch) takes this workload."""
    return (w.resident_frac >= 1.0 and w.dtype == "bf16" and w.d == 128 and w.dI == 128 and w.V <= 8
            and w.G * w.V <= 16 and w.N <= 32768 and w.N % 4 == 0)


def cluster_step_supported(w) -> bool:
    """Whether sd_decode_step runs this workload as one thread-block cluster per KV group:
    block selection (whole 16- or 32-row runs of a block) over at most 8192 blocks."""
    runs = w.block % 16 == 0 and (32 % w.block == 0 if w.block <= 32 else w.block % 32 == 0)
    return step_supported(w) and runs and w.N <= 8192


class SparseDecodeStep:
    """One sparse decode step, inputs resident.  Paths: "step" runs the indexer, the top-k and
    the gather-attend in one persistent launch (sd_decode_step; the default where it applies:
    bf16, K/V in HBM); "select_attend" runs the indexer, then the fused select + attend launch
    (token-level selection); "separate" runs the indexer, the top-k and the gather-attend as
    three launches.  For a tiered workload the full K/V cache stays in pinned host memory and
    only the resident share sits in the HBM pool; there the default path copies the selected
    host rows into an HBM stage with one copy kernel spread over every SM
    (sd_stage_host_rows) between the top-k and the attention."""

    def __init__(self, w, x, device, path="auto", tiered_path="staged"):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        self.sd, self.w, self.dev = sd, w, device
        self.tiered = w.resident_frac < 1.0
        if path == "auto":
            # block selection over short score rows: the whole step in one cluster launch;
            # token selection: indexer + fused select/attend; tiered: the separate calls
            path = ("step" if cluster_step_supported(w) else
                    "select_attend" if w.dtype == "bf16" and w.block == 1 and not self.tiered else "separate")
        if path == "step" and not step_supported(w):
            raise ValueError(f"sd_decode_step does not take {w.name}")
        self.path = path
        self.step_kernel = path == "step"
        self.staged = self.tiered and tiered_path == "staged" and path == "separate"
        # block selection picks few entries but many rows per group: the separate top-k and
        # gather-attend spread the rows over the whole GPU, the fused kernel over one cluster
        self.fused = path == "select_attend" or (self.tiered and tiered_path == "fused")
        self.dominant = "sd_decode_step" if self.step_kernel else "sd_index_score"
        self.phases = (() if self.fused or self.step_kernel else ("after_topk", "after_stage") if self.staged
                       else ("after_topk",))
        self.launches_per_step = 1 if self.step_kernel else 2 if self.fused else 4 if self.staged else 3
        self.q_idx, self.k_idx, self.q = (x[k].to(device) for k in ("q_idx", "k_idx", "q"))
        self.scores = torch.empty(w.B, w.Hkv, w.N, dtype=torch.float32, device=device)
        self.idx = torch.empty(w.B, w.Hkv, w.k, dtype=torch.int32, device=device)
        self.key_hist = sd.key_hist_buffer(w.B * w.Hkv, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        if self.tiered:
            self.k_cache, self.v_cache = x["k_pool"].to(device), x["v_pool"].to(device)
            self.slot_map = x["slot_map"].to(device)
            self.k_host, self.v_host = x["k"].pin_memory(), x["v"].pin_memory()
            kw = dict(k_host=self.k_host, v_host=self.v_host, slot_map=self.slot_map)
        else:
            self.k_cache, self.v_cache = x["k"].to(device), x["v"].to(device)
            kw = {}
        self.args, self.out, self.lse, _ = sd.make_attend_args(
            self.q, self.k_cache, self.v_cache, None if self.fused else self.idx, n_idx=w.k,
            block=w.block, T=w.T, err_word=self.err, **kw)
        need = 0 if self.fused else sd.sd_gather_attend_workspace_bytes(self.args)
        self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)
        if need > 0 and not self.step_kernel:
            self.launches_per_step += 1  # the split-K merge kernel
        if self.staged:
            self.stage = sd.stage_buffers(self.args, self.q.dtype, device)
            self.counter = sd.stage_counter(device)
        self.keys = self.k_idx
        if w.block > 1:  # pooled block keys, built once (cache fill): fp16 to meet an fp16 query
            self.keys = sd.sd_block_pool(self.k_idx, w.block, dtype=self.q_idx.dtype
                                         if self.q_idx.dtype == torch.float16 else torch.float32)
        if self.step_kernel:
            self.step_args, _, _, self.out, self.lse = sd.make_decode_step_args(
                self.q_idx, self.keys, self.q, self.k_cache, self.v_cache, w.k, block=w.block, scores=self.scores,
                idx=self.idx, err_word=self.err)
            self.step_ws = sd.decode_step_workspace(self.step_args, device)
        self.host_rows = None

    dominant_per_step = 1

    def run(self, m: "StepMarks" = None):
        sd = self.sd
        if m is not None:
            m.start.record()
            m.before(0)
        if self.step_kernel:
            sd.sd_decode_step(self.step_args)
            if m is not None:
                m.after(0)
                m.end.record()
            return
        sd.sd_index_score(self.q_idx, self.keys, self.scores, self.err, key_hist=self.key_hist)
        if m is not None:
            m.after(0)
        if self.fused:
            sd.sd_select_attend(self.scores, self.args, self.idx, key_hist=self.key_hist)
        else:
            sd.sd_topk(self.scores, self.w.k, self.idx, key_hist=self.key_hist)
            if m is not None:
                m.at("after_topk")
            if self.staged:
                sd.sd_stage_host_rows(self.args, self.counter)
                if m is not None:
                    m.at("after_stage")
            sd.sd_gather_attend(self.args, self.ws)
        if m is not None:
            m.end.record()

    def rotation(self, n):
        """n input sets in distinct device memory (set 0 is the step's own tensors; the others
        are copies of q, q_idx, the keys and the K/V cache), each as the list of the step's
        C-ABI calls with their arguments marshalled once.  Steps run back to back over the sets
        in turn meet none of their own bytes in L2 when n sets hold a few times L2.  K/V
        resident in HBM only."""
        import torch
        sd = self.sd
        assert not self.tiered
        sets = []
        for i in range(n):
            if i == 0:
                q, q_idx, keys, kc, vc = self.q, self.q_idx, self.keys, self.k_cache, self.v_cache
            else:
                q, q_idx, keys, kc, vc = (t.clone() for t in (self.q, self.q_idx, self.keys, self.k_cache,
                                                              self.v_cache))
            keep = [q, q_idx, keys, kc, vc]
            if self.step_kernel:
                a, _, _, _, _ = sd.make_decode_step_args(q_idx, keys, q, kc, vc, self.w.k, block=self.w.block,
                                                         scores=self.scores, idx=self.idx, out=self.out,
                                                         lse=self.lse, err_word=self.err)
                ws = sd.decode_step_workspace(a, self.dev)
                keep += [a, ws]
                calls = [sd.prepare_decode_step(a)]
            else:
                a, _, _, _ = sd.make_attend_args(q, kc, vc, None if self.fused else self.idx, n_idx=self.w.k,
                                                 block=self.w.block, T=self.w.T, err_word=self.err, out=self.out,
                                                 lse=self.lse)
                keep.append(a)
                calls = [sd.prepare_index_score(q_idx, keys, self.scores, self.err, key_hist=self.key_hist)]
                if self.fused:
                    calls.append(sd.prepare_select_attend(self.scores, a, self.idx, key_hist=self.key_hist))
                else:
                    calls += [sd.prepare_topk(self.scores, self.w.k, self.idx, key_hist=self.key_hist),
                              sd.prepare_gather_attend(a, self.ws)]
            sets.append((calls, keep))
        torch.cuda.synchronize()
        return sets

    def io_set(self, stream):
        """A second, independent set of the step's per-step buffers for a pipelined run: its own
        packed inputs (q, q_idx) and results (out, lse, idx) and its own intermediates (scores,
        key histogram, workspaces), sharing the resident keys and K/V; the step's C-ABI calls
        on `stream`, prebound.  Returns (d_in, d_out, calls, keep)."""
        import torch
        sd = self.sd
        assert not self.tiered
        w = self.w

        def pack(tensors):
            sizes = [t.numel() * t.element_size() for t in tensors]
            offs = [sum((n + 255) // 256 * 256 for n in sizes[:i]) for i in range(len(sizes))]
            buf = torch.empty(offs[-1] + (sizes[-1] + 255) // 256 * 256, dtype=torch.uint8, device=self.dev)
            views = []
            for t, o, n in zip(tensors, offs, sizes):
                v = buf[o:o + n].view(t.dtype).view(t.shape)
                v.copy_(t)
                views.append(v)
            return buf, views

        d_in, (q, q_idx) = pack([self.q, self.q_idx])
        d_out, (out, lse, idx) = pack([self.out, self.lse, self.idx])
        scores = torch.empty_like(self.scores)
        err = self.err
        keep = [q, q_idx, out, lse, idx, scores]
        if self.step_kernel:
            a, _, _, _, _ = sd.make_decode_step_args(q_idx, self.keys, q, self.k_cache, self.v_cache, w.k,
                                                     block=w.block, scores=scores, idx=idx, out=out, lse=lse,
                                                     err_word=err)
            keep += [a, sd.decode_step_workspace(a, self.dev)]
            calls = [sd.prepare_decode_step(a, stream=stream)]
        else:
            hist = sd.key_hist_buffer(w.B * w.Hkv, self.dev)
            a, _, _, _ = sd.make_attend_args(q, self.k_cache, self.v_cache, None if self.fused else idx, n_idx=w.k,
                                             block=w.block, T=w.T, err_word=err, out=out, lse=lse)
            ws = torch.zeros_like(self.ws)
            keep += [hist, a, ws]
            calls = [sd.prepare_index_score(q_idx, self.keys, scores, err, key_hist=hist, stream=stream)]
            if self.fused:
                calls.append(sd.prepare_select_attend(scores, a, idx, key_hist=hist, stream=stream))
            else:
                calls += [sd.prepare_topk(scores, w.k, idx, key_hist=hist, stream=stream),
                          sd.prepare_gather_attend(a, ws, stream=stream)]
        torch.cuda.synchronize()
        return d_in, d_out, calls, keep

    def packed_io(self):
        """Moves the step's per-step inputs (q, q_idx) into one device buffer and its results
        (out, lse, idx) into another, re-points the calls at them, and returns (d_in, d_out,
        calls): one copy brings a step's inputs, one copy returns its results, and `calls` are
        the step's C-ABI calls with their arguments marshalled once (one ctypes call per kernel).
        K/V resident in HBM only."""
        import torch
        sd = self.sd
        assert not self.tiered

        def pack(tensors):
            sizes = [t.numel() * t.element_size() for t in tensors]
            offs = [sum((n + 255) // 256 * 256 for n in sizes[:i]) for i in range(len(sizes))]
            buf = torch.empty(offs[-1] + (sizes[-1] + 255) // 256 * 256, dtype=torch.uint8, device=self.dev)
            views = []
            for t, o, n in zip(tensors, offs, sizes):
                v = buf[o:o + n].view(t.dtype).view(t.shape)
                v.copy_(t)
                views.append(v)
            return buf, views

        d_in, (self.q, self.q_idx) = pack([self.q, self.q_idx])
        d_out, (self.out, self.lse, self.idx) = pack([self.out, self.lse, self.idx])
        if self.step_kernel:
            a = self.step_args
            a.q, a.q_idx = self.q.data_ptr(), self.q_idx.data_ptr()
            a.out, a.lse, a.idx = self.out.data_ptr(), self.lse.data_ptr(), self.idx.data_ptr()
            calls = [sd.prepare_decode_step(a)]
        else:
            a = self.args
            a.q, a.out, a.lse = self.q.data_ptr(), self.out.data_ptr(), self.lse.data_ptr()
            calls = [sd.prepare_index_score(self.q_idx, self.keys, self.scores, self.err, key_hist=self.key_hist)]
            if self.fused:
                calls.append(sd.prepare_select_attend(self.scores, a, self.idx, key_hist=self.key_hist))
            else:
                a.idx = self.idx.data_ptr()
                calls += [sd.prepare_topk(self.scores, self.w.k, self.idx, key_hist=self.key_hist),
                          sd.prepare_gather_attend(a, self.ws)]
        return d_in, d_out, calls

    def after_warmup(self):
        """Counts the selected rows that live in host memory (fixed by the inputs)."""
        if self.tiered:
            import torch
            rows = self.idx.long() * self.w.block
            b = torch.arange(self.w.B, device=self.dev)[:, None, None]
            self.host_rows = int((self.slot_map[b, rows] < 0).sum().item())

    def bytes(self):
        """Algorithmic bytes: per launch of the dominant kernel; per step from HBM and from
        host memory (what the method must move: keys, selected K/V rows, queries, outputs)."""
        w = self.w
        e = w.elem_bytes
        key_bytes = w.B * w.Hkv * w.N * w.dI * (self.keys.element_size() if w.block > 1 else e)
        q_idx_bytes = w.B * w.Hkv * w.V * w.dI * self.q_idx.element_size()
        score_bytes = w.B * w.Hkv * w.N * 4
        row_bytes = w.d * e * 2
        kv_rows = w.B * w.Hkv * w.n_rows
        host_rows = self.host_rows or 0
        q_bytes = w.B * w.V * w.Hq * w.d * e
        out_bytes = w.B * w.V * w.Hq * (w.d + 1) * 4 + w.B * w.Hkv * w.k * 4
        hbm = key_bytes + q_idx_bytes + (kv_rows - host_rows) * row_bytes + q_bytes + out_bytes
        if self.step_kernel:  # the one launch moves the whole step, the scores written included
            return {"dominant": hbm + score_bytes, "hbm": hbm, "host": 0}
        return {"dominant": key_bytes + q_idx_bytes + score_bytes, "hbm": hbm,
                "host": host_rows * row_bytes}


class WindowStep:
    """One sparse decode step on the overlapping compression-window grid: the indexer, the
    windows' max-pooled scores (with the key histogram), the top-k windows, the union of
    their segments, and the attention over it (segments of `stride` tokens, empty slots
    skipped)."""

    dominant = "sd_index_score"
    phases = ()
    launches_per_step = 5
    dominant_per_step = 1

    def __init__(self, w, x, device):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        self.sd, self.w, self.dev = sd, w, device
        self.q_idx, self.k_idx, self.q = (x[k].to(device) for k in ("q_idx", "k_idx", "q"))
        self.k_cache, self.v_cache = x["k"].to(device), x["v"].to(device)
        self.kern, self.strd = w.window_kernel, w.window_stride
        self.NW = sd.sd_window_count(w.T, self.kern, self.strd)
        self.max_segs = w.k * (self.kern // self.strd)
        self.scores = torch.empty(w.B, w.Hkv, w.T, dtype=torch.float32, device=device)
        self.wscores = torch.empty(w.B, w.Hkv, self.NW, dtype=torch.float32, device=device)
        self.widx = torch.empty(w.B, w.Hkv, w.k, dtype=torch.int32, device=device)
        self.segs = torch.empty(w.B, w.Hkv, self.max_segs, dtype=torch.int32, device=device)
        self.key_hist = sd.key_hist_buffer(w.B * w.Hkv, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.args, self.out, self.lse, _ = sd.make_attend_args(
            self.q, self.k_cache, self.v_cache, self.segs, block=self.strd, T=w.T, err_word=self.err)
        need = sd.sd_gather_attend_workspace_bytes(self.args)
        self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)
        self.idx = self.segs
        self.rows_used = None

    def run(self, m: "StepMarks" = None):
        sd = self.sd
        if m is not None:
            m.start.record()
            m.before(0)
        sd.sd_index_score(self.q_idx, self.k_idx, self.scores, self.err)
        if m is not None:
            m.after(0)
        sd.sd_window_max(self.scores, self.kern, self.strd, self.wscores, key_hist=self.key_hist)
        sd.sd_topk(self.wscores, self.w.k, self.widx, key_hist=self.key_hist)
        sd.sd_window_union(self.widx, self.w.T, self.kern, self.strd, self.segs, err_word=self.err)
        sd.sd_gather_attend(self.args, self.ws)
        if m is not None:
            m.end.record()

    def after_warmup(self):
        """Counts the K/V rows the union selects (fixed by the inputs)."""
        self.rows_used = int((self.segs >= 0).sum().item()) * self.strd

    def bytes(self):
        w = self.w
        e = w.elem_bytes
        key_bytes = w.B * w.Hkv * w.T * w.dI * e
        q_idx_bytes = w.B * w.Hkv * w.V * w.dI * e
        score_bytes = w.B * w.Hkv * w.T * 4
        kv = (self.rows_used or 0) * w.d * e * 2
        q_bytes = w.B * w.V * w.Hq * w.d * e
        out_bytes = w.B * w.V * w.Hq * (w.d + 1) * 4 + w.B * w.Hkv * self.max_segs * 4
        return {"dominant": key_bytes + q_idx_bytes + score_bytes,
                "hbm": key_bytes + q_idx_bytes + kv + q_bytes + out_bytes, "host": 0}


class HeadsStep:
    """One sparse decode step with selection per query head: every head's unscaled
    attention logits against its KV head's keys (with the key histogram, one row per head),
    each head's top-k, and the attention of each head over its own selected rows."""

    dominant = "sd_index_score_heads"
    phases = ("after_topk",)
    launches_per_step = 3
    dominant_per_step = 1

    def __init__(self, w, x, device):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        assert w.V == 1, "per-head selection scores the decode query of every head"
        self.sd, self.w, self.dev = sd, w, device
        self.q = x["q"].to(device)                              # [B,1,Hq,d]
        self.q_heads = self.q.view(w.B, w.Hkv, w.G, w.d)        # the same bytes, [B,Hkv,G,d]
        self.k_cache, self.v_cache = x["k"].to(device), x["v"].to(device)
        self.scores = torch.empty(w.B, w.Hkv, w.G, w.T, dtype=torch.float32, device=device)
        self.idx = torch.empty(w.B, w.Hq, w.k, dtype=torch.int32, device=device)
        self.key_hist = sd.key_hist_buffer(w.B * w.Hq, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.args, self.out, self.lse, _ = sd.make_attend_args(
            self.q, self.k_cache, self.v_cache, self.idx, T=w.T, err_word=self.err, per_head=True)
        need = sd.sd_gather_attend_workspace_bytes(self.args)
        self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)

    def run(self, m: "StepMarks" = None):
        sd = self.sd
        if m is not None:
            m.start.record()
            m.before(0)
        sd.sd_index_score_heads(self.q_heads, self.k_cache, self.scores, self.err, key_hist=self.key_hist)
        if m is not None:
            m.after(0)
        sd.sd_topk(self.scores, self.w.k, self.idx, key_hist=self.key_hist)
        if m is not None:
            m.at("after_topk")
        sd.sd_gather_attend(self.args, self.ws)
        if m is not None:
            m.end.record()

    def after_warmup(self):
        pass

    def bytes(self):
        w = self.w
        e = w.elem_bytes
        key_bytes = w.B * w.Hkv * w.T * w.d * e
        q_bytes = w.B * w.Hq * w.d * e
        score_bytes = w.B * w.Hq * w.T * 4
        kv = w.B * w.Hq * w.k * w.d * e * 2
        out_bytes = w.B * w.Hq * (w.d + 1) * 4 + w.B * w.Hq * w.k * 4
        return {"dominant": key_bytes + q_bytes + score_bytes,
                "hbm": key_bytes + q_bytes + kv + out_bytes, "host": 0}


class VerifyGroupStep:
    """One speculative-verify step over a group of layers that share one selection: the
    indexer and the top-k once, then for every layer the V draft tokens' K/V appended to the
    layer's window-bounded ring and the attention over the selected rows plus the ring
    (causal among the drafts)."""

    dominant = "sd_index_score"
    phases = ("after_topk",)
    dominant_per_step = 1

    def __init__(self, w, x, device):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        self.sd, self.w, self.dev = sd, w, device
        self.launches_per_step = 2 + 2 * w.layers
        self.q_idx, self.k_idx = x["q_idx"].to(device), x["k_idx"].to(device)
        self.q = x["q"][0].to(device)                       # [layers,B,V,Hq,d]
        self.ks = [k.to(device) for k in x["k"]]
        self.vs = [v.to(device) for v in x["v"]]
        self.ring_k, self.ring_v = x["ring_k"].to(device), x["ring_v"].to(device)
        self.ring_pos = [x["ring_pos"].to(device) for _ in range(w.layers)]
        self.draft_k, self.draft_v = x["draft_k"].to(device), x["draft_v"].to(device)
        self.qpos = x["qpos"].to(device)
        self.pos0 = torch.full((w.B,), w.T, dtype=torch.int32, device=device)
        self.scores = torch.empty(w.B, w.Hkv, w.N, dtype=torch.float32, device=device)
        self.idx = torch.empty(w.B, w.Hkv, w.k, dtype=torch.int32, device=device)
        self.key_hist = sd.key_hist_buffer(w.B * w.Hkv, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.args = []
        for layer in range(w.layers):
            a, out, lse, _ = sd.make_attend_args(self.q[layer], self.ks[layer], self.vs[layer], self.idx, T=w.T,
                                                 err_word=self.err, ring_k=self.ring_k[layer],
                                                 ring_v=self.ring_v[layer], ring_pos=self.ring_pos[layer],
                                                 qpos=self.qpos)
            self.args.append((a, out, lse))
        need = sd.sd_gather_attend_workspace_bytes(self.args[0][0])
        self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)
        self.out, self.lse = self.args[-1][1], self.args[-1][2]

    def run(self, m: "StepMarks" = None):
        sd, w = self.sd, self.w
        if m is not None:
            m.start.record()
            m.before(0)
        sd.sd_index_score(self.q_idx, self.k_idx, self.scores, self.err, key_hist=self.key_hist)
        if m is not None:
            m.after(0)
        sd.sd_topk(self.scores, w.k, self.idx, key_hist=self.key_hist)
        if m is not None:
            m.at("after_topk")
        for layer in range(w.layers):
            sd.sd_ring_append(self.draft_k[layer], self.draft_v[layer], self.ring_k[layer], self.ring_v[layer],
                              self.ring_pos[layer], self.pos0)
            sd.sd_gather_attend(self.args[layer][0], self.ws)
        if m is not None:
            m.end.record()

    def after_warmup(self):
        pass

    def bytes(self):
        w = self.w
        e = w.elem_bytes
        key_bytes = w.B * w.Hkv * w.T * w.dI * e
        q_idx_bytes = w.B * w.Hkv * w.V * w.dI * e
        score_bytes = w.B * w.Hkv * w.T * 4
        row = w.d * e * 2
        per_layer = (w.B * w.Hkv * (w.k + w.ring_w) * row            # selected rows + ring read
                     + w.B * w.Hkv * w.V * row * 2                     # drafts read and written into the ring
                     + w.B * w.V * w.Hq * w.d * e                      # queries
                     + w.B * w.V * w.Hq * (w.d + 1) * 4)               # out, lse
        return {"dominant": key_bytes + q_idx_bytes + score_bytes,
                "hbm": key_bytes + q_idx_bytes + w.B * w.Hkv * w.k * 4 + w.layers * per_layer, "host": 0}


class CachedTieredStep:
    """One decode step of a tiered layer whose pool is kept as a cache: the indexer (this
    step's window of the sliding verify queries), the top-k, the staging of the selected
    rows the pool does not hold, the attention, and the promotion of the staged rows into
    the pool (evicting rows not selected).  Steps cycle over the query windows; the pool
    carries over from step to step.

    With residency per (sequence, KV head) the promotion copies the rows from the stage
    (sd_promote_staged_rows) after the attention, and step s+1 runs step s's promotion on a
    side stream beside its own indexer and top-k (two selection buffers alternate), joining
    it before its staging; `concurrent = False` runs the same calls in order on one stream.
    With one slot map per sequence the promotion reads the host cache before the staging
    (sd_promote_rows)."""

    dominant = "sd_index_score"
    launches_per_step = 8  # indexer, top-k, promotion (3), staging, attention, merge
    dominant_per_step = 1

    def __init__(self, w, x, device, concurrent=True):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        self.sd, self.w, self.dev = sd, w, device
        self.staged_promotion = bool(w.slot_per_head)
        self.concurrent = concurrent
        self.phases = (("after_topk", "promote_start", "promote_end") if self.staged_promotion
                       else ("after_topk", "after_promote"))
        seq = x["q_idx_seq"]
        self.q_idx_win = [seq[:, :, s:s + w.V].contiguous().to(device) for s in range(w.drift_steps)]
        self.q_idx = self.q_idx_win[0]
        self.k_idx = x["k_idx"].to(device)
        self.q = x["q"].to(device)
        self.k_cache, self.v_cache = x["k_pool"].to(device), x["v_pool"].to(device)  # the pool, written
        sm = x["slot_map"]
        if w.slot_per_head:  # every KV head starts from the generated residency
            sm = sm[:, None, :].expand(w.B, w.Hkv, w.T).contiguous()
        self.slot_map = sm.to(device)
        self.k_host, self.v_host = x["k"].pin_memory(), x["v"].pin_memory()
        self.static_map = sm.to(device)  # the residency as generated (for comparison)
        self.pool_pos, self.hand = sd.pool_state(self.slot_map, w.pool_rows)
        self.scores = torch.empty(w.B, w.Hkv, w.T, dtype=torch.float32, device=device)
        self.idx_buf = [torch.empty(w.B, w.Hkv, w.k, dtype=torch.int32, device=device) for _ in range(2)]
        self.idx = self.idx_buf[0]
        self.key_hist = sd.key_hist_buffer(w.B * w.Hkv, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.args, self.out, self.lse, _ = sd.make_attend_args(
            self.q, self.k_cache, self.v_cache, self.idx, T=w.T, k_host=self.k_host, v_host=self.v_host,
            slot_map=self.slot_map, err_word=self.err)
        self.stage = sd.stage_buffers(self.args, self.q.dtype, device)
        args1 = type(self.args).from_buffer_copy(self.args)  # the same call on the other selection buffer
        args1.idx = self.idx_buf[1].data_ptr()
        self.args_buf = [self.args, args1]
        self.counter = sd.stage_counter(device)
        ws_bytes = (sd.sd_promote_staged_rows_workspace_bytes(self.args) if self.staged_promotion
                    else sd.sd_promote_rows_workspace_bytes(self.args))
        self.ws_promote = torch.zeros(max(16, ws_bytes), dtype=torch.uint8, device=device)
        need = sd.sd_gather_attend_workspace_bytes(self.args)
        self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)
        self.side = torch.cuda.Stream(device=device)
        self.pending = None  # the args of the step whose staged rows are still to be promoted
        self.step_no = 0
        self.host_bytes = None

    def run(self, m: "StepMarks" = None):
        import contextlib
        import torch
        sd, w = self.sd, self.w
        q_idx = self.q_idx_win[self.step_no % w.drift_steps]
        args = self.args_buf[self.step_no % 2]
        self.step_no += 1
        if m is not None:
            m.start.record()
        if self.pending is not None:  # the previous step's promotion, beside this step's selection
            main = torch.cuda.current_stream()
            if self.concurrent:
                self.side.wait_stream(main)
            with torch.cuda.stream(self.side) if self.concurrent else contextlib.nullcontext():
                if m is not None:
                    m.at("promote_start")
                sd.sd_promote_staged_rows(self.pending, self.pool_pos, self.hand, self.ws_promote)
                if m is not None:
                    m.at("promote_end")
        if m is not None:
            m.before(0)
        sd.sd_index_score(q_idx, self.k_idx, self.scores, self.err, key_hist=self.key_hist)
        if m is not None:
            m.after(0)
        self.idx = self.idx_buf[(self.step_no - 1) % 2]
        sd.sd_topk(self.scores, w.k, self.idx, key_hist=self.key_hist)
        if m is not None:
            m.at("after_topk")
        if self.staged_promotion:
            if self.pending is not None and self.concurrent:
                torch.cuda.current_stream().wait_stream(self.side)
            sd.sd_stage_host_rows(args, self.counter)
            sd.sd_gather_attend(args, self.ws)
            self.pending = args
        else:
            sd.sd_promote_rows(args, self.pool_pos, self.hand, self.ws_promote)
            if m is not None:
                m.at("after_promote")
            sd.sd_stage_host_rows(args, self.counter)
            sd.sd_gather_attend(args, self.ws)
        if m is not None:
            m.end.record()

    def host_misses(self, slot_map):
        """(distinct host units, host rows over the KV heads) of the current selection: a
        unit is a (sequence, position), or a (sequence, KV head, position) with residency
        per KV head."""
        import torch
        B, T = self.w.B, self.w.T
        if slot_map.dim() == 3:
            miss = slot_map.gather(2, self.idx.long()) < 0
            n = int(miss.sum().item())
            return n, n
        sel = self.idx.view(B, -1).long()
        b = torch.arange(B, device=sel.device)[:, None].expand_as(sel)
        miss = slot_map[b, sel] < 0
        return int(torch.unique((b * T + sel)[miss]).numel()), int(miss.sum().item())

    def after_warmup(self):
        """Host bytes per step in the steady state, averaged over one cycle of the query
        windows: the rows promoted from host memory (K and V of every KV head of a promoted
        position; none with staged promotion) plus the selected rows left in host memory
        (staged); and, for comparison, the host rows the same selections would read with
        the pool kept as it was generated."""
        import torch
        w, row = self.w, self.w.d * self.w.elem_bytes * 2
        with_cache = without = 0
        for _ in range(w.drift_steps):
            if self.staged_promotion:
                # after the step, the slot map is the one its staging saw (its own promotion
                # runs with the next step)
                self.run()
                torch.cuda.synchronize()
                without += self.host_misses(self.static_map)[1] * row
                with_cache += self.host_misses(self.slot_map)[1] * row
                continue
            q_idx = self.q_idx_win[self.step_no % w.drift_steps]
            args, self.idx = self.args_buf[self.step_no % 2], self.idx_buf[self.step_no % 2]
            self.step_no += 1
            self.sd.sd_index_score(q_idx, self.k_idx, self.scores, self.err, key_hist=self.key_hist)
            self.sd.sd_topk(self.scores, w.k, self.idx, key_hist=self.key_hist)
            without += self.host_misses(self.static_map)[1] * row
            before, _ = self.host_misses(self.slot_map)
            self.sd.sd_promote_rows(args, self.pool_pos, self.hand, self.ws_promote)
            left_pos, left_rows = self.host_misses(self.slot_map)
            with_cache += (before - left_pos) * w.Hkv * row + left_rows * row
            self.sd.sd_stage_host_rows(args, self.counter)
            self.sd.sd_gather_attend(args, self.ws)
        torch.cuda.synchronize()
        self.host_bytes = with_cache // w.drift_steps
        self.host_bytes_static = without // w.drift_steps

    def bytes(self):
        w = self.w
        e = w.elem_bytes
        key_bytes = w.B * w.Hkv * w.T * w.dI * e
        q_idx_bytes = w.B * w.Hkv * w.V * w.dI * e
        score_bytes = w.B * w.Hkv * w.T * 4
        q_bytes = w.B * w.V * w.Hq * w.d * e
        out_bytes = w.B * w.V * w.Hq * (w.d + 1) * 4 + w.B * w.Hkv * w.k * 4
        rows = w.B * w.Hkv * w.k * w.d * e * 2
        return {"dominant": key_bytes + q_idx_bytes + score_bytes,
                "hbm": key_bytes + q_idx_bytes + rows + q_bytes + out_bytes, "host": self.host_bytes or 0}


class LookaheadStep:
    """One decode step over L tiered layers, each with its own selection: per layer the
    indexer, the top-k, the copy of the selected host-resident rows into an HBM stage, and
    the attention.  With lookahead (default) layer l+1's indexer and top-k are issued once
    layer l has started, before layer l's attention, and the staging copies (host link) run
    on their own stream beside the selection and attention kernels (HBM), which stay in
    order on the main stream so that no two of them share the SMs.  Two stage buffers
    alternate between layers.  Without lookahead every call runs in order on one stream."""

    dominant = "sd_index_score"
    phases = ()

    def __init__(self, w, x, device, lookahead=True):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        self.sd, self.w, self.dev, self.lookahead = sd, w, device, lookahead
        L = w.layers
        self.launches_per_step = 5 * L  # indexer, top-k, staging, attention, merge
        self.dominant_per_step = L
        self.q_idx = x["q_idx"].to(device)                          # [L,B,Hkv,V,dI]
        self.k_idx = [k.to(device) for k in x["k_idx"]]
        self.q = x["q"][0].to(device)                               # [L,B,V,Hq,d]
        self.k_pool = [k.to(device) for k in x["k_pool"]]
        self.v_pool = [v.to(device) for v in x["v_pool"]]
        self.k_host = [k.pin_memory() for k in x["k"]]
        self.v_host = [v.pin_memory() for v in x["v"]]
        self.slot_map = x["slot_map"].to(device)
        self.scores = [torch.empty(w.B, w.Hkv, w.T, dtype=torch.float32, device=device) for _ in range(L)]
        self.idx = [torch.empty(w.B, w.Hkv, w.k, dtype=torch.int32, device=device) for _ in range(L)]
        self.key_hist = [sd.key_hist_buffer(w.B * w.Hkv, device) for _ in range(L)]
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.args = []
        for layer in range(L):
            a, out, lse, _ = sd.make_attend_args(self.q[layer], self.k_pool[layer], self.v_pool[layer],
                                                 self.idx[layer], T=w.T, k_host=self.k_host[layer],
                                                 v_host=self.v_host[layer], slot_map=self.slot_map, err_word=self.err)
            self.args.append((a, out, lse))
        self.stages = [sd.stage_buffers(self.args[0][0], self.q.dtype, device) for _ in range(2)]
        self.counters = [sd.stage_counter(device) for _ in range(2)]
        for layer in range(L):
            ks, vs = self.stages[layer % 2]
            self.args[layer][0].k_stage, self.args[layer][0].v_stage = ks.data_ptr(), vs.data_ptr()
        need = sd.sd_gather_attend_workspace_bytes(self.args[0][0])
        self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)
        self.out, self.lse = self.args[-1][1], self.args[-1][2]
        self.s_stage = torch.cuda.Stream(device)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        self.ev_sel = [ev() for _ in range(L)]
        self.ev_stage = [ev() for _ in range(L)]
        self.ev_att = [ev() for _ in range(L)]
        self.ev_start = ev()
        self.host_rows = None

    def _select(self, layer, m):
        sd, w = self.sd, self.w
        if m is not None:
            m.before(layer)
        sd.sd_index_score(self.q_idx[layer], self.k_idx[layer], self.scores[layer], self.err,
                          key_hist=self.key_hist[layer])
        if m is not None:
            m.after(layer)
        sd.sd_topk(self.scores[layer], w.k, self.idx[layer], key_hist=self.key_hist[layer])

    def run(self, m: "StepMarks" = None):
        import torch
        sd, L = self.sd, self.w.layers
        main = torch.cuda.current_stream()
        if m is not None:
            m.start.record()
        if not self.lookahead:
            for layer in range(L):
                self._select(layer, m)
                sd.sd_stage_host_rows(self.args[layer][0], self.counters[layer % 2])
                sd.sd_gather_attend(self.args[layer][0], self.ws)
            if m is not None:
                m.end.record()
            return
        # the selection of layer l+1 is issued on the main stream before layer l's attention
        # (layer l has started, so its forecast is available); only the staging copies run
        # on their own stream, beside the selection and attention kernels
        self.ev_start.record(main)
        self.s_stage.wait_event(self.ev_start)

        def select_and_stage(layer):
            self._select(layer, m)
            self.ev_sel[layer].record(main)
            with torch.cuda.stream(self.s_stage):
                self.s_stage.wait_event(self.ev_sel[layer])
                if layer >= 2:  # stage buffer layer % 2 was read by layer - 2's attention
                    self.s_stage.wait_event(self.ev_att[layer - 2])
                sd.sd_stage_host_rows(self.args[layer][0], self.counters[layer % 2], stream=self.s_stage)
                self.ev_stage[layer].record(self.s_stage)

        select_and_stage(0)
        for layer in range(L):
            if layer + 1 < L:
                select_and_stage(layer + 1)
            main.wait_event(self.ev_stage[layer])
            sd.sd_gather_attend(self.args[layer][0], self.ws, stream=main)
            self.ev_att[layer].record(main)
        if m is not None:
            m.end.record()

    def after_warmup(self):
        """Counts the selected rows that live in host memory (fixed by the inputs)."""
        import torch
        rows = 0
        b = torch.arange(self.w.B, device=self.dev)[:, None, None]
        for layer in range(self.w.layers):
            rows += int((self.slot_map[b, self.idx[layer].long()] < 0).sum().item())
        self.host_rows = rows

    def bytes(self):
        w = self.w
        e = w.elem_bytes
        key_bytes = w.B * w.Hkv * w.T * w.dI * e
        q_idx_bytes = w.B * w.Hkv * w.V * w.dI * e
        score_bytes = w.B * w.Hkv * w.T * 4
        row = w.d * e * 2
        host_rows = self.host_rows or 0
        dev_rows = w.layers * w.B * w.Hkv * w.k - host_rows
        q_bytes = w.B * w.V * w.Hq * w.d * e
        out_bytes = w.B * w.V * w.Hq * (w.d + 1) * 4 + w.B * w.Hkv * w.k * 4
        hbm = w.layers * (key_bytes + q_idx_bytes + q_bytes + out_bytes) + dev_rows * row
        return {"dominant": key_bytes + q_idx_bytes + score_bytes, "hbm": hbm, "host": host_rows * row}


class DenseScoringStep:
    """One decode step of the importance-scoring workload: for every layer, dense attention
    over all cached rows (logits kept) and that layer's term of the importance score."""

    dominant = "sd_gather_attend"
    phases = ()

    def __init__(self, w, x, device):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        self.sd, self.w, self.dev = sd, w, device
        self.ks = [k.to(device) for k in x["k"]]
        self.vs = [v.to(device) for v in x["v"]]
        self.qall = x["q"].to(device)              # [steps, layers, B, V, Hq, d]
        self.s = torch.zeros(w.B, w.T, dtype=torch.float64, device=device)
        self.logits = torch.empty(w.B, w.V, w.Hq, w.T, dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.q = torch.empty_like(self.qall[0, 0])
        self.args = []
        for layer in range(w.layers):
            a, out, lse, _ = sd.make_attend_args(self.q, self.ks[layer], self.vs[layer], None, T=w.T,
                                                 logits=self.logits, err_word=self.err)
            self.args.append((a, out, lse))
        need = sd.sd_gather_attend_workspace_bytes(self.args[0][0])
        self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)
        self.step_no = 0
        self.weight = 1.0 / (w.layers * w.Hq)
        self.out, self.lse = self.args[-1][1], self.args[-1][2]

    @property
    def launches_per_step(self):
        return 2 * self.w.layers

    @property
    def dominant_per_step(self):
        return self.w.layers

    def run(self, m: "StepMarks" = None):
        sd, w = self.sd, self.w
        if m is not None:
            m.start.record()
        qs = self.qall[self.step_no % w.steps]
        self.step_no += 1
        for layer in range(w.layers):
            a, out, lse = self.args[layer]
            a.q = qs[layer].data_ptr()
            if m is not None:
                m.before(layer)
            sd.sd_gather_attend(a, self.ws)
            if m is not None:
                m.after(layer)
            sd.sd_score_accumulate(self.logits, lse, None, self.s, w.Hkv, 1, self.weight, err_word=self.err)
        if m is not None:
            m.end.record()

    def after_warmup(self):
        pass

    def bytes(self):
        w = self.w
        kv = w.B * w.Hkv * w.T * w.d * w.elem_bytes * 2
        q = w.B * w.V * w.Hq * w.d * w.elem_bytes
        logits = w.B * w.V * w.Hq * w.T * 4
        out = w.B * w.V * w.Hq * (w.d + 1) * 4
        # dominant kernel per launch: one layer's K and V, its query, logits and outputs out
        return {"dominant": kv + q + logits + out, "hbm": w.layers * (kv + q + out) + w.B * w.T * 8 * 2,
                "host": 0}


class TieredAttendStep:
    """One decode step over a tiered cache: for every layer, dense attention over all
    positions with the four tiers of a seeded importance score driving the rows' sources --
    T0 and T1 at bf16 from HBM, T2 as int8 codes times their per-row scale, T3 left out.
    The tiers and the int8 codes (of every layer's K and V) are built once, untimed."""

    dominant = "sd_gather_attend"
    phases = ()
    tier_seed = 2011

    def __init__(self, w, x, device):
        import torch
        from top_sparse_decode_gqa_gb300 import binding as sd
        from top_sparse_decode_gqa_gb300.workloads import importance_scores
        self.sd, self.w, self.dev = sd, w, device
        self.ks = [k.to(device) for k in x["k"]]
        self.vs = [v.to(device) for v in x["v"]]
        self.q = x["q"][0].to(device)              # [layers, B, V, Hq, d]
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        s = importance_scores(w.B, w.T, self.tier_seed).to(device)
        self.tier, counts = sd.sd_tier_classify(s, w.cum_frac)
        self.counts = counts.cpu()
        self.codes = [sd.sd_quantize_rows_int8(k, self.tier) + sd.sd_quantize_rows_int8(v, self.tier)
                      for k, v in zip(self.ks, self.vs)]  # (k codes, k scales, v codes, v scales)
        self.args = []
        for layer in range(w.layers):
            kc, ksc, vc, vsc = self.codes[layer]
            a, out, lse, _ = sd.make_attend_args(self.q[layer], self.ks[layer], self.vs[layer], None, T=w.T,
                                                 err_word=self.err, tier=self.tier, k_int8=kc, v_int8=vc,
                                                 k_scale=ksc, v_scale=vsc)
            self.args.append((a, out, lse))
        need = sd.sd_gather_attend_workspace_bytes(self.args[0][0])
        self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)
        self.out, self.lse = self.args[-1][1], self.args[-1][2]

    @property
    def launches_per_step(self):
        return 2 * self.w.layers  # attention + split merge per layer

    @property
    def dominant_per_step(self):
        return self.w.layers

    def run(self, m: "StepMarks" = None):
        sd = self.sd
        if m is not None:
            m.start.record()
        for layer in range(self.w.layers):
            if m is not None:
                m.before(layer)
            sd.sd_gather_attend(self.args[layer][0], self.ws)
            if m is not None:
                m.after(layer)
        if m is not None:
            m.end.record()

    def after_warmup(self):
        pass

    def bytes(self):
        w = self.w
        c = [int(v) for v in self.counts[0]]  # per sequence (all equal: exact fractions)
        heads = w.B * w.Hkv
        rows_bf16 = (c[0] + c[1]) * heads   # T0 + T1 rows, K and V at bf16
        rows_i8 = c[2] * heads              # T2 rows: K and V codes + scales
        per_layer = rows_bf16 * 2 * w.d * 2 + rows_i8 * 2 * (w.d + 4) + w.B * w.T  # + the tier map
        q = w.B * w.V * w.Hq * w.d * 2
        out = w.B * w.V * w.Hq * (w.d + 1) * 4
        return {"dominant": per_layer + q + out, "hbm": w.layers * (per_layer + q + out), "host": 0}


def make_step(w, x, device, path="auto", tiered_path="staged", lookahead=True):
    if w.tiered_attention:
        return TieredAttendStep(w, x, device)
    if w.drift_steps > 0:
        return CachedTieredStep(w, x, device, concurrent=lookahead)
    if w.layer_indexers:
        return LookaheadStep(w, x, device, lookahead)
    if w.ring_w > 0:
        return VerifyGroupStep(w, x, device)
    if w.layers > 1:
        return DenseScoringStep(w, x, device)
    if w.window_kernel > 0:
        return WindowStep(w, x, device)
    if w.per_head:
        return HeadsStep(w, x, device)
    return SparseDecodeStep(w, x, device, path, tiered_path)


def host_link_gbs(device, nbytes=256 << 20, reps=5):
    """Host->device bandwidth of a pinned copy (CUDA events): the best of `reps` copies after
    two untimed ones, the host-row roofline term."""
    import torch
    h = torch.ones(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    for _ in range(2):
        d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        d.copy_(h, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
    return best


# ----------------------------------------------------------------------------- arms


def step_report(step, w, workload, kmarks, dom_ms, ms_per_step, peak, device, K, clean_l2):
    """The step's roofline record (bytes, t_roof, fraction, per-kernel times) from its timed
    steps, and the committed ncu traffic of its dominant kernel (None when stale)."""
    import torch
    by = step.bytes()
    if isinstance(step, SparseDecodeStep) and step.step_kernel:
        kernel_file, kernel_tag = (("block_step.cu", "step_tiles.cuh", "tc_common.cuh", "sd_common.cuh")
                                   if cluster_step_supported(w) else
                                   ("decode_step.cu", "step_tiles.cuh", "tc_common.cuh", "sd_common.cuh")), "decode_step"
    elif isinstance(step, (SparseDecodeStep, WindowStep, HeadsStep, VerifyGroupStep, LookaheadStep, CachedTieredStep)):
        kernel_file, kernel_tag = ("index_score.cu", "index_score_tc.cu", "tc_common.cuh", "sd_common.cuh"), "index_score"
    elif isinstance(step, DenseScoringStep):  # dense over the cache: the tiled path
        kernel_file, kernel_tag = ("dense_attend.cu", "step_tiles.cuh", "tc_common.cuh", "sd_common.cuh"), "dense_attend"
    else:
        kernel_file, kernel_tag = ("gather_attend.cu", "attend_mma.cuh", "sd_common.cuh"), "gather_attend"
    traffic = profiled_traffic(workload, kernel_tag, source_digest(*kernel_file))
    step_s = ms_per_step / 1e3
    step_roof = {"bound": "hbm", "hbm_bytes": by["hbm"], "unit": "GB/s",
                 "achieved": round(by["hbm"] / step_s / 1e9, 1)}
    t_roof = by["hbm"] / (peak * 1e9)
    if by["host"]:
        host_gbs = host_link_gbs(device)
        t_host = by["host"] / (host_gbs * 1e9)
        step_roof.update({"host_bytes": by["host"], "host_link_gbs_measured": round(host_gbs, 1),
                          "bound": "hbm+host"})
        if isinstance(step, LookaheadStep) and step.lookahead:
            # the host copies of one layer run beside another layer's HBM work: the bound is
            # the larger of the two streams of bytes, not their sum
            step_roof.update({"bound": "max(hbm, host)", "t_roof_serial_us": round((t_roof + t_host) * 1e6, 2)})
            t_roof = max(t_roof, t_host)
        else:
            t_roof += t_host
    step_roof["t_roof_us"] = round(t_roof * 1e6, 2)
    step_roof["frac"] = round(t_roof / step_s, 4)
    if isinstance(step, SparseDecodeStep) and step.step_kernel:
        step_roof["kernel_us"] = {"decode_step": round(statistics.mean(dom_ms) * 1e3, 2)}
    elif isinstance(step, SparseDecodeStep) and step.fused:
        tail = [m.dom[0][1].elapsed_time(m.end) for m in kmarks]
        step_roof["kernel_us"] = {"index_score": round(statistics.mean(dom_ms) * 1e3, 2),
                                  "select_attend": round(statistics.mean(tail) * 1e3, 2)}
    elif isinstance(step, WindowStep):
        tail = [m.dom[0][1].elapsed_time(m.end) for m in kmarks]
        step_roof["kernel_us"] = {"index_score": round(statistics.mean(dom_ms) * 1e3, 2),
                                  "window_max+topk+union+gather_attend": round(statistics.mean(tail) * 1e3, 2)}
        step_roof["kv_rows_selected"] = step.rows_used
    elif isinstance(step, SparseDecodeStep) and step.staged:
        k_us = lambda a, b: round(statistics.mean(a(m).elapsed_time(b(m)) for m in kmarks) * 1e3, 2)
        step_roof["kernel_us"] = {
            "index_score": round(statistics.mean(dom_ms) * 1e3, 2),
            "topk": k_us(lambda m: m.dom[0][1], lambda m: m.phase["after_topk"]),
            "stage_host_rows": k_us(lambda m: m.phase["after_topk"], lambda m: m.phase["after_stage"]),
            "gather_attend": k_us(lambda m: m.phase["after_stage"], lambda m: m.end)}
    elif isinstance(step, CachedTieredStep):
        k_us = lambda a, b: round(statistics.mean(a(m).elapsed_time(b(m)) for m in kmarks) * 1e3, 2)  # noqa: E731
        if step.staged_promotion:
            # the promotion (of the previous step's staged rows) runs on the side stream beside
            # the indexer and top-k; the staging waits for it
            step_roof["kernel_us"] = {
                "index_score": round(statistics.mean(dom_ms) * 1e3, 2),
                "topk": k_us(lambda m: m.dom[0][1], lambda m: m.phase["after_topk"]),
                "promote_staged_rows (side stream)": k_us(lambda m: m.phase["promote_start"],
                                                          lambda m: m.phase["promote_end"]),
                "stage_host_rows+gather_attend": k_us(lambda m: m.phase["after_topk"], lambda m: m.end)}
            if step.concurrent:  # the same steps with every call in order on one stream
                step.concurrent = False
                serial = []
                for i in range(3 + min(K, 20)):  # 3 untimed, then the median
                    clean_l2()
                    sm_ = StepMarks(0)
                    step.run(sm_)
                    torch.cuda.synchronize()
                    if i >= 3:
                        serial.append(sm_.step_ms())
                step.concurrent = True
                step_roof["serial_ms_per_step_median"] = round(statistics.median(serial), 5)
        else:
            step_roof["kernel_us"] = {
                "index_score": round(statistics.mean(dom_ms) * 1e3, 2),
                "topk": k_us(lambda m: m.dom[0][1], lambda m: m.phase["after_topk"]),
                "promote": k_us(lambda m: m.phase["after_topk"], lambda m: m.phase["after_promote"]),
                "stage_host_rows+gather_attend": k_us(lambda m: m.phase["after_promote"], lambda m: m.end)}
        step_roof["host_bytes_per_step_without_cache"] = step.host_bytes_static
    elif isinstance(step, LookaheadStep):
        step_roof["kernel_us"] = {"index_score": round(statistics.mean(dom_ms) * 1e3, 2), "layers": w.layers}
        if step.lookahead:  # the same steps with every call in order on one stream, for comparison
            step.lookahead = False
            serial = []
            for i in range(3 + min(K, 20)):  # 3 untimed, then the median
                clean_l2()
                sm_ = StepMarks(0)
                step.run(sm_)
                torch.cuda.synchronize()
                if i >= 3:
                    serial.append(sm_.step_ms())
            step.lookahead = True
            step_roof["serial_ms_per_step_median"] = round(statistics.median(serial), 5)
    elif isinstance(step, VerifyGroupStep):
        after_topk = [m.dom[0][1].elapsed_time(m.phase["after_topk"]) for m in kmarks]
        tail = [m.phase["after_topk"].elapsed_time(m.end) for m in kmarks]
        step_roof["kernel_us"] = {"index_score": round(statistics.mean(dom_ms) * 1e3, 2),
                                  "topk": round(statistics.mean(after_topk) * 1e3, 2),
                                  "ring_append+gather_attend_all_layers": round(statistics.mean(tail) * 1e3, 2),
                                  "layers": w.layers}
    elif isinstance(step, (SparseDecodeStep, HeadsStep)):
        after_topk = [m.dom[0][1].elapsed_time(m.phase["after_topk"]) for m in kmarks]
        tail = [m.phase["after_topk"].elapsed_time(m.end) for m in kmarks]
        step_roof["kernel_us"] = {"index_score": round(statistics.mean(dom_ms) * 1e3, 2),
                                  "topk": round(statistics.mean(after_topk) * 1e3, 2),
                                  "gather_attend": round(statistics.mean(tail) * 1e3, 2)}
    else:
        step_roof["kernel_us"] = {"gather_attend_per_layer": round(statistics.mean(dom_ms) * 1e3, 2),
                                  "layers": w.layers}
    return traffic, step_roof


def path_description(step, w) -> str:
    """What one timed step of `step` runs, for the JSON line's config."""
    if isinstance(step, SparseDecodeStep):
        if step.step_kernel:
            return ("indexer + top-k + gather-attend in one launch (sd_decode_step, one thread-block cluster "
                    "per KV group)" if cluster_step_supported(w)
                    else "indexer + top-k + gather-attend in one persistent launch (sd_decode_step)")
        if step.fused:
            return "indexer + fused select/attend"
        if step.staged:
            return "indexer + top-k + host-row staging + gather-attend"
        return "indexer + top-k + gather-attend"
    if isinstance(step, WindowStep):
        return "indexer + window max + top-k windows + union + gather-attend"
    if isinstance(step, HeadsStep):
        return "per-head logits + per-head top-k + per-head gather-attend"
    if isinstance(step, VerifyGroupStep):
        return (f"indexer + top-k once, then per layer ({w.layers}) ring append + gather-attend over the "
                "selected rows and the draft ring")
    if isinstance(step, CachedTieredStep):
        if step.staged_promotion:
            head = ("indexer + top-k + staging of the rows the pool lacks + gather-attend, then their promotion "
                    "from the stage into the pool (cache) "
                    + ("beside the next step's indexer and top-k" if step.concurrent else "in order on one stream"))
        else:
            head = "indexer + top-k + promotion into the pool (cache) + staging of the rest + gather-attend"
        return head + ", the query window sliding step by step"
    if isinstance(step, TieredAttendStep):
        return (f"per layer ({w.layers}): dense attention over the tiered cache (T0 and T1 rows at bf16, T2 rows as "
                "int8 codes and per-row scales, T3 rows left out) + split merge")
    if isinstance(step, LookaheadStep):
        return (f"per layer ({w.layers}): indexer + top-k + host-row staging + gather-attend, "
                + ("next layer's selection before this layer's attention, staging on its own stream"
                   if step.lookahead else "in order on one stream"))
    return "dense attention + score accumulate per layer"


def capture_graph(step):
    """One step's C-ABI calls captured into a CUDA graph (its launches and the events that
    order its streams), for steps whose time is mostly launches; None (with the reason on
    stderr) when the capture fails, and the steps then run eagerly."""
    import torch
    g = torch.cuda.CUDAGraph()
    try:
        torch.cuda.synchronize()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            step.run()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
    except RuntimeError as e:
        print(f"bench: CUDA graph capture failed, steps run eagerly: {e}", file=sys.stderr)
        torch.cuda.synchronize()
        return None
    return g


def rotation_count(step, l2_bytes) -> int:
    """Input sets a back-to-back run rotates through: enough that at least three times L2 of
    other steps' traffic passes between two uses of one set (at least two sets)."""
    fp = max(1, step.bytes()["hbm"])
    return max(2, -(-3 * l2_bytes // fp) + 1)


def time_rotated(sets, K) -> float:
    """ms for K steps run back to back over the input sets in turn (prebound C-ABI calls, the
    kernels of consecutive launches overlapping programmatically), one event pair around them."""
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = len(sets)
    start.record()
    for i in range(K):
        for c in sets[i % n][0]:
            c()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def rotated_l2_note(n, step, l2_bytes) -> str:
    fp = step.bytes()["hbm"]
    return (f"inputs larger than L2: steps back to back over {n} copies of the step's inputs in distinct "
            f"memory ({(n - 1) * fp / 1e6:.0f} MB = {(n - 1) * fp / l2_bytes:.1f}x L2 of other steps' traffic "
            f"between two uses of one copy), no flush; one event pair around the timed steps")


def measure_extra(name, args, device, local, clean_l2, peak, steps=100, warmup=3):
    """A compact measurement of another workload in the same run (the T = 131072 configurations
    beside the headline): the default path, `warmup` untimed steps, then `steps` steps timed as
    the headline's are (back to back over copies of the inputs for a sparse step with K/V in
    HBM, else one event pair per flushed step), and `steps` more, flushed, with events around
    every kernel; clocks sampled meanwhile.  Returns the record attached to the JSON line."""
    import torch
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS[name]
    x = generate(w)
    step = make_step(w, x, device, "auto", "staged", True)
    for _ in range(warmup):
        clean_l2()
        step.run()
    torch.cuda.synchronize()
    if int(step.err.item()) != 0:
        raise RuntimeError(f"{name}: device error word {int(step.err.item())}")
    step.after_warmup()
    l2_bytes = max(int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0)), 1)
    rot = None
    if isinstance(step, SparseDecodeStep) and not step.tiered:
        rot = step.rotation(rotation_count(step, l2_bytes))
        for calls, _ in rot:
            for c in calls:
                c()
        torch.cuda.synchronize()
    marks = [StepMarks(0) for _ in range(steps)]
    kmarks = [StepMarks(step.dominant_per_step, step.phases) for _ in range(steps)]
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    clocks.mark(True)
    if rot is not None:
        rot_ms = time_rotated(rot, steps)
    else:
        for i in range(steps):
            clean_l2()
            step.run(marks[i])
    torch.cuda.synchronize()
    for i in range(steps):
        clean_l2()
        step.run(kmarks[i])
    torch.cuda.synchronize()
    clocks.mark(False)
    clk = clocks.stop()
    if int(step.err.item()) != 0:
        raise RuntimeError(f"{name}: device error word {int(step.err.item())} after the timed steps")
    if rot is not None:
        ms_per_step = rot_ms / steps
        l2_note = rotated_l2_note(len(rot), step, l2_bytes)
        del rot
    else:
        ms_per_step = sum(m.step_ms() for m in marks) / steps
        l2_note = "flushed between timed steps: 2x L2 written then read, outside the events"
    dom_ms = [t for m in kmarks for t in m.dominant_ms()]
    _, step_roof = step_report(step, w, name, kmarks, dom_ms, ms_per_step, peak, device, steps, clean_l2)
    rec = {"value": round(w.queries_per_step / (ms_per_step / 1e3), 1), "unit": "queries/s",
           "ms_per_step": round(ms_per_step, 5), "steps": steps, "warmup": warmup,
           "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "T": w.T, "k": w.k,
                      "block": w.block, "V": w.V, "resident_frac": w.resident_frac,
                      "path": path_description(step, w), "l2": l2_note},
           "step_roofline": step_roof, "clocks": clk,
           "gpu_launches": step.launches_per_step * steps}
    del step, x
    torch.cuda.empty_cache()
    return rec


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
    step = make_step(w, x, device, "separate" if args.separate else args.path, args.tiered_path,
                     not args.no_lookahead)
    props = torch.cuda.get_device_properties(device)
    flush = torch.empty(2 * max(int(getattr(props, "L2_cache_size", 0)), 128 << 20), dtype=torch.uint8,
                        device=device)

    def clean_l2():
        # write a buffer of 2x L2, then read it back so the step starts on a cold, clean L2
        flush.fill_(1)
        flush.view(torch.int32).sum()

    for _ in range(args.warmup):
        clean_l2()
        step.run()
    torch.cuda.synchronize()
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error word {int(step.err.item())}")
    step.after_warmup()

    # Timed region 1 (the headline).  A sparse step with K/V in HBM runs its K steps back to
    # back over copies of its inputs that together hold several times L2 (inputs larger than
    # L2, no flush; one event pair around the K steps).  Other steps: K steps with one event
    # pair per step and L2 flushed before each, so nothing between the step's kernels breaks
    # their programmatic overlap.  Timed region 2: the same steps (flushed) with events around
    # every kernel, for the per-kernel roofline.
    K = args.steps
    K2 = min(K, 500)
    l2_bytes = max(int(getattr(props, "L2_cache_size", 0)), 1)
    rot = None
    if isinstance(step, SparseDecodeStep) and not step.tiered and not args.no_rotate:
        rot = step.rotation(rotation_count(step, l2_bytes))
        for calls, _ in rot:  # every copy once, untimed
            for c in calls:
                c()
        torch.cuda.synchronize()
    graph = capture_graph(step) if args.graph and rot is None else None
    if graph is not None and int(step.err.item()) != 0:
        raise RuntimeError(f"device error word {int(step.err.item())} after the graph's first replay")
    marks = [StepMarks(0) for _ in range(K)]
    kmarks = [StepMarks(step.dominant_per_step, step.phases) for _ in range(K2)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    if rot is not None:
        rot_ms = time_rotated(rot, K)
    else:
        for i in range(K):
            clean_l2()
            if graph is not None:
                marks[i].start.record()
                graph.replay()
                marks[i].end.record()
            else:
                step.run(marks[i])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    for i in range(K2):
        clean_l2()
        step.run(kmarks[i])
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error word {int(step.err.item())} after the timed steps")

    if rot is not None:
        l2_note = rotated_l2_note(len(rot), step, l2_bytes)
        total_ms = rot_ms
        del rot
        torch.cuda.empty_cache()
    else:
        l2_note = "flushed between timed steps: 2x L2 written then read, outside the events"
        total_ms = sum(m.step_ms() for m in marks)
    dom_ms = [t for m in kmarks for t in m.dominant_ms()]
    total_s = reduce_max(total_ms / 1e3, world, device)
    value = aggregate(w.queries_per_step * K, world, total_s)
    ms_per_step = total_s * 1e3 / K

    if isinstance(step, SparseDecodeStep) and not step.tiered:
        serial = measure_e2e_packed(step, w, clean_l2, K=min(K, 200))
        e2e = measure_e2e_pipelined(step, w, K=min(K, 200))
        e2e["serial"] = {k: serial[k] for k in ("value", "timing")}
    else:
        e2e = measure_e2e(step, w, x, clean_l2, K=min(K, 200))

    peak, peak_kind = load_peaks()
    by = step.bytes()
    dom_s = statistics.mean(dom_ms) / 1e3
    achieved = by["dominant"] / dom_s / 1e9
    traffic, step_roof = step_report(step, w, args.workload, kmarks, dom_ms, ms_per_step, peak, device, K, clean_l2)
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
        "dtype": "f32" if w.dtype == "f32" else "bf16",
        "data": "synthetic (seeded; integer indexer keys in [-8,8], N(0,1) q/K/V)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "T": w.T,
                   "k": w.k, "block": w.block, "V": w.V, "layers": w.layers,
                   "queries_per_step": w.queries_per_step,
                   "path": path_description(step, w),
                   "l2": l2_note,
                   "launch": ("each timed step one replay of a CUDA graph of the step's C-ABI calls (the per-kernel "
                              "pass runs them eagerly)" if graph is not None else "C-ABI calls from Python"),
                   "parallelism": f"replica x{world} (each rank its own batch)"},
        "roofline": {"bound": "hbm", "kernel": step.dominant, "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)", "traffic": traffic,
                     "algorithmic_bytes_per_launch": by["dominant"],
                     "avg_launch_us": round(dom_s * 1e6, 2)},
        "step_roofline": step_roof,
        "e2e": e2e,
        "gpu_launches": step.launches_per_step * K,
        "clocks": clk,
    }
    if not args.no_extra and args.workload == DEFAULT_WORKLOAD:
        # the T = 131072 configurations (block-sparse; tiered verify) measured in the same run
        line["t131072"] = {name: measure_extra(name, args, device, local, clean_l2, peak)
                           for name in ("c3_block_sparse", "c4_tiered_verify")}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cuda_runtime():
    """ctypes handle on the CUDA runtime the library uses (already loaded with it)."""
    import ctypes
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
        except OSError:
            continue
        rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
        rt.cudaStreamSynchronize.argtypes = [ctypes.c_void_p]
        return rt
    raise RuntimeError("the CUDA runtime library was not found")


def measure_e2e_pipelined(step, w, K, n_sets=2):
    """End to end through the C ABI with host buffers, with `n_sets` batches in flight: every
    step copies its queries in from pinned host memory (one packed copy, on an input stream)
    and its results (out, lse, idx) back to pinned host memory (one packed copy, on an output
    stream), while the kernels of the step before run on the compute stream; events order each
    set's copy in, kernels and copy out: a set's inputs are refilled once its previous kernels
    are done, and its kernels run once its previous results left.  Host wall clock over K
    steps, ending with a synchronize."""
    import ctypes
    import torch
    rt = cuda_runtime()
    rt.cudaStreamWaitEvent.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    rt.cudaEventRecord.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    s_c, s_x, s_o = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sets = [step.io_set(s_c) for _ in range(n_sets)]
    h_in = []
    for d_in, _, _, _ in sets:
        h = torch.empty(d_in.numel(), dtype=torch.uint8).pin_memory()
        h.copy_(d_in)  # the step's queries in the packed layout
        h_in.append(h)
    h_out = [torch.empty(d_out.numel(), dtype=torch.uint8).pin_memory() for _, d_out, _, _ in sets]
    rt.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint]
    rt.cudaEventDestroy.argtypes = [ctypes.c_void_p]

    def ev():
        h = ctypes.c_void_p()
        if rt.cudaEventCreateWithFlags(ctypes.byref(h), 2) != 0:  # cudaEventDisableTiming
            raise RuntimeError("cudaEventCreateWithFlags failed")
        return h
    ev_in = [ev() for _ in sets]
    ev_done = [ev() for _ in sets]
    ev_out = [ev() for _ in sets]
    cx, cc, co = ctypes.c_void_p(s_x.cuda_stream), ctypes.c_void_p(s_c.cuda_stream), ctypes.c_void_p(s_o.cuda_stream)

    def one(i):
        j = i % n_sets
        d_in, d_out, calls, _ = sets[j]
        if i >= n_sets:  # the set's previous kernels have read its inputs
            rt.cudaStreamWaitEvent(cx, ev_done[j], 0)
        if rt.cudaMemcpyAsync(ctypes.c_void_p(d_in.data_ptr()), ctypes.c_void_p(h_in[j].data_ptr()), d_in.numel(), 1,
                              cx) != 0:
            raise RuntimeError("cudaMemcpyAsync (inputs) failed")
        rt.cudaEventRecord(ev_in[j], cx)
        rt.cudaStreamWaitEvent(cc, ev_in[j], 0)
        if i >= n_sets:  # the set's previous results have left
            rt.cudaStreamWaitEvent(cc, ev_out[j], 0)
        for c in calls:
            c()
        rt.cudaEventRecord(ev_done[j], cc)
        rt.cudaStreamWaitEvent(co, ev_done[j], 0)
        if rt.cudaMemcpyAsync(ctypes.c_void_p(h_out[j].data_ptr()), ctypes.c_void_p(d_out.data_ptr()), d_out.numel(), 2,
                              co) != 0:
            raise RuntimeError("cudaMemcpyAsync (results) failed")
        rt.cudaEventRecord(ev_out[j], co)

    for i in range(2 * n_sets):  # warm-up, untimed
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        one(i)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    for e in ev_in + ev_done + ev_out:
        rt.cudaEventDestroy(e)
    # every set ran the same inputs: the same result bytes, as the step's own buffers hold
    ref = torch.cat([step.out.reshape(-1).view(torch.uint8), step.lse.reshape(-1).view(torch.uint8),
                     step.idx.reshape(-1).view(torch.uint8)]).cpu()
    for (_, d_out, _, keep), h in zip(sets, h_out):
        out, lse, idx = keep[2], keep[3], keep[4]
        got = torch.cat([out.reshape(-1).view(torch.uint8), lse.reshape(-1).view(torch.uint8),
                         idx.reshape(-1).view(torch.uint8)]).cpu()
        if not torch.equal(got, ref) or not torch.equal(h, d_out.cpu()):
            raise RuntimeError("pipelined end-to-end results differ from the step's own")
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error word {int(step.err.item())} after the end-to-end steps")
    return {"value": round(w.queries_per_step * K / dt, 1), "unit": "queries/s",
            "h2d_bytes_per_step": int(sets[0][0].numel()), "d2h_bytes_per_step": int(sets[0][1].numel()),
            "timing": (f"host wall clock over {K} steps with {n_sets} batches in flight: per step one packed copy "
                       "of the queries in from pinned memory and one of out, lse and idx back, on input and output "
                       "copy streams beside the compute stream; prebound C-ABI calls"),
            "ctypes_calls_per_step": len(sets[0][2]) + 9}


def measure_e2e_packed(step, w, clean_l2, K):
    """End to end through the C ABI with host buffers, for a step whose inputs and results
    are packed (SparseDecodeStep.packed_io): per step one host->device copy of the step's
    queries from pinned memory, the step's C-ABI calls (one ctypes call per kernel), one
    device->host copy of out, lse and idx into pinned memory, and a stream synchronize; host
    wall clock per step."""
    import ctypes
    import torch
    d_in, d_out, calls = step.packed_io()
    h_in = torch.empty(d_in.numel(), dtype=torch.uint8).pin_memory()
    h_in.copy_(d_in)  # this step's queries, in the packed layout
    h_out = torch.empty(d_out.numel(), dtype=torch.uint8).pin_memory()
    rt = cuda_runtime()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cin = (ctypes.c_void_p(d_in.data_ptr()), ctypes.c_void_p(h_in.data_ptr()), d_in.numel(), 1, st)
    cout = (ctypes.c_void_p(h_out.data_ptr()), ctypes.c_void_p(d_out.data_ptr()), d_out.numel(), 2, st)
    times = []
    for i in range(K + 3):
        clean_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if rt.cudaMemcpyAsync(*cin) != 0:
            raise RuntimeError("cudaMemcpyAsync (inputs) failed")
        for c in calls:
            c()
        if rt.cudaMemcpyAsync(*cout) != 0:
            raise RuntimeError("cudaMemcpyAsync (results) failed")
        if rt.cudaStreamSynchronize(st) != 0:
            raise RuntimeError("cudaStreamSynchronize failed")
        if i >= 3:
            times.append(time.perf_counter() - t0)
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error word {int(step.err.item())} after the end-to-end steps")
    return {"value": round(w.queries_per_step * len(times) / sum(times), 1), "unit": "queries/s",
            "h2d_bytes_per_step": int(d_in.numel()), "d2h_bytes_per_step": int(d_out.numel()),
            "timing": "host wall clock per step incl. one packed copy each way and the stream sync",
            "ctypes_calls_per_step": len(calls) + 3}


def measure_e2e(step, w, x, clean_l2, K):
    """The same metric through the public calls with host buffers: every step copies the
    step's query tensors from pinned host memory, runs the calls, and reads the result
    (attention output, lse and, for sparse steps, the selected indices) back into pinned
    host memory; host wall clock per step, including the copies and the final sync."""
    import torch
    verify = isinstance(step, VerifyGroupStep)
    multi = isinstance(step, (VerifyGroupStep, LookaheadStep, TieredAttendStep))
    ins = [(step.q, x["q"][0] if multi else x["q"][0, 0] if w.layers > 1 else x["q"])]
    if isinstance(step, (SparseDecodeStep, WindowStep, VerifyGroupStep, LookaheadStep)):
        ins.append((step.q_idx, x["q_idx"]))
    if isinstance(step, CachedTieredStep):  # every window of indexer queries comes from the host
        ins += [(dst, x["q_idx_seq"][:, :, s:s + w.V]) for s, dst in enumerate(step.q_idx_win)]
    if verify:  # the drafts' K/V come from the host with the queries
        ins += [(step.draft_k, x["draft_k"]), (step.draft_v, x["draft_v"])]
    ins = [(dst, src.contiguous().pin_memory()) for dst, src in ins]
    sparse = isinstance(step, (SparseDecodeStep, WindowStep, HeadsStep, VerifyGroupStep, LookaheadStep,
                               CachedTieredStep))
    # the result tensors, looked up after every step (a step may alternate its buffers)
    results = lambda: [step.out, step.lse] + (  # noqa: E731
        [] if isinstance(step, TieredAttendStep) else
        [step.idx[-1] if isinstance(step.idx, list) else step.idx] if sparse else [step.s])
    outs = [torch.empty(src.shape, dtype=src.dtype).pin_memory() for src in results()]
    times = []
    for i in range(K + 3):
        clean_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for dst, src in ins:
            dst.copy_(src, non_blocking=True)
        step.run()
        for src, dst in zip(results(), outs):
            dst.copy_(src, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if i >= 3:
            times.append(time.perf_counter() - t0)
    err = getattr(step, "err", None)
    if err is not None and int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} after the end-to-end steps")
    bi = sum(src.numel() * src.element_size() for _, src in ins)
    bo = sum(dst.numel() * dst.element_size() for dst in outs)
    return {"value": round(w.queries_per_step * len(times) / sum(times), 1), "unit": "queries/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "timing": "host wall clock per step incl. copies and sync"}


def oracle_step(w, x, b0, b1):
    """The whole step on the CPU oracle for sequences [b0, b1)."""
    import numpy as np
    import oracle
    nb = b1 - b0
    scale = 1.0 / math.sqrt(w.d)
    if w.layer_indexers:  # every layer: its own selection, then attention over its rows
        res = []
        for layer in range(w.layers):
            sc = oracle.index_score(x["q_idx"][layer, b0:b1].contiguous(), x["k_idx"][layer][b0:b1].contiguous(), nb,
                                    w.Hkv, w.V, w.N, w.dI)
            idx = oracle.topk(sc, w.k)
            res.append((idx, oracle.gather_attend(x["q"][0, layer, b0:b1].contiguous(),
                                                  x["k"][layer][b0:b1].contiguous(),
                                                  x["v"][layer][b0:b1].contiguous(), idx, nb, w.V, w.Hq, w.Hkv, w.d,
                                                  w.T, w.k, 1, scale)))
        return res
    if w.ring_w > 0:  # one selection for the layer group, then per layer: ring append + attention
        sc = oracle.index_score(x["q_idx"][b0:b1].contiguous(), x["k_idx"][b0:b1].contiguous(), nb, w.Hkv, w.V,
                                w.N, w.dI)
        idx = oracle.topk(sc, w.k)
        res = []
        for layer in range(w.layers):
            rk = x["ring_k"][layer, b0:b1].float().numpy().copy()
            rv = x["ring_v"][layer, b0:b1].float().numpy().copy()
            rp = x["ring_pos"][b0:b1].numpy().copy()
            oracle.ring_append(x["draft_k"][layer, b0:b1].float().numpy(), x["draft_v"][layer, b0:b1].float().numpy(),
                               rk, rv, rp, [w.T] * nb)
            res.append(oracle.gather_attend_ring(x["q"][0, layer, b0:b1].contiguous(), x["k"][layer][b0:b1].contiguous(),
                                                 x["v"][layer][b0:b1].contiguous(), idx, nb, w.V, w.Hq, w.Hkv, w.d, w.T,
                                                 w.k, 1, scale, torch_bf16(rk), torch_bf16(rv), rp,
                                                 x["qpos"][b0:b1].numpy()))
        return idx, res
    if w.tiered_attention:  # the tiers of the seeded score drive every layer's dense attention
        from top_sparse_decode_gqa_gb300.workloads import importance_scores
        tier, _ = oracle.tier_classify(importance_scores(w.B, w.T, TieredAttendStep.tier_seed).numpy()[b0:b1],
                                       np.array(w.cum_frac))
        idx = np.broadcast_to(np.arange(w.T, dtype=np.int32), (nb, w.Hkv, w.T)).copy()
        for b in range(nb):
            idx[b][:, tier[b] == 3] = -1
        t2 = np.broadcast_to((tier == 2)[:, None, :, None], (nb, w.Hkv, w.T, w.d))
        res = []
        for layer in range(w.layers):
            kv = []
            for t in (x["k"][layer][b0:b1].contiguous(), x["v"][layer][b0:b1].contiguous()):
                codes, scales = oracle.quantize_rows_int8(t, tier, nb, w.Hkv, w.T, w.d)
                kv.append(np.where(t2, codes.astype(np.float32) * scales[..., None], t.float().numpy()))
            res.append(oracle.gather_attend(x["q"][0, layer, b0:b1].float(), kv[0], kv[1], idx, nb, w.V, w.Hq,
                                            w.Hkv, w.d, w.T, w.T, 1, scale)[:2])
        return res
    if w.layers > 1:  # dense attention per layer and the layer's importance-score term
        s = np.zeros((nb, w.T))
        for layer in range(w.layers):
            _, lse, z = oracle.gather_attend(x["q"][0, layer, b0:b1].contiguous(),
                                             x["k"][layer][b0:b1].contiguous(),
                                             x["v"][layer][b0:b1].contiguous(), None, nb, w.V, w.Hq,
                                             w.Hkv, w.d, w.T, w.T, 1, scale, True)
            oracle.score_accumulate(z, lse, None, s, nb, w.V, w.Hq, w.Hkv, w.T, 1, w.T,
                                    1.0 / (w.layers * w.Hq))
        return s
    if w.per_head:  # every head's own logits, its own top-k, attention over its own rows
        q = x["q"][b0:b1].contiguous()
        sc = oracle.index_score_heads(q.view(nb, w.Hkv, w.G, w.d), x["k"][b0:b1].contiguous(), nb, w.Hkv, w.G,
                                      w.T, w.d)
        idx = oracle.topk(sc.reshape(nb, w.Hq, w.T), w.k)
        return oracle.gather_attend(q, x["k"][b0:b1].contiguous(), x["v"][b0:b1].contiguous(), idx, nb, w.V,
                                    w.Hq, w.Hkv, w.d, w.T, w.k, 1, scale, per_head=True)
    q_idx = x["q_idx"][b0:b1].contiguous()
    if w.drift_steps > 0:  # the first query window
        q_idx = x["q_idx_seq"][b0:b1, :, :w.V].contiguous()
    keys = x["k_idx"][b0:b1].contiguous()
    if w.block > 1:
        keys = oracle.block_pool(keys, nb, w.Hkv, w.T, w.dI, w.block).astype("float32")
    sc = oracle.index_score(q_idx, keys, nb, w.Hkv, w.V, w.N, w.dI)
    if w.window_kernel > 0:  # windows: max-pooled scores, top-k windows, their union
        widx = oracle.topk(oracle.window_max(sc, w.window_kernel, w.window_stride), w.k)
        segs = oracle.window_union(widx, w.T, w.window_kernel, w.window_stride)
        return oracle.gather_attend(x["q"][b0:b1].contiguous(), x["k"][b0:b1].contiguous(),
                                    x["v"][b0:b1].contiguous(), segs, nb, w.V, w.Hq, w.Hkv, w.d, w.T,
                                    segs.shape[-1], w.window_stride, scale)
    idx = oracle.topk(sc, w.k)
    return oracle.gather_attend(x["q"][b0:b1].contiguous(), x["k"][b0:b1].contiguous(),
                                x["v"][b0:b1].contiguous(), idx, nb, w.V, w.Hq, w.Hkv, w.d, w.T,
                                w.k, w.block, scale)


def torch_bf16(a):
    """A float array of bf16-representable values back as a bf16 tensor (exact)."""
    import torch
    return torch.from_numpy(a).to(torch.bfloat16)


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


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_command(gpus: int, argv, port: int):
    """The command that runs this benchmark as `gpus` local ranks, one per GPU."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", str(gpus),
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)


def self_spawn(args, argv):
    """--gpus N > 1 without a torchrun environment: run N local ranks under
    torch.distributed.run and return their exit status (an error, not a silent one-GPU run,
    when fewer GPUs are visible).  None when this process is already a rank or N == 1."""
    if args.gpus <= 1 or "WORLD_SIZE" in os.environ:
        return None
    if args.impl == "ours":
        import torch
        have = torch.cuda.device_count()
        if have < args.gpus:
            print(f"bench.py: --gpus {args.gpus} needs {args.gpus} visible GPUs, found {have}", file=sys.stderr)
            return 2
    return subprocess.call(spawn_command(args.gpus, argv, free_port()))


def main(argv=None):
    raw_argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rotate", action="store_true",
                    help="time the sparse step like the others (one flushed step per event pair) instead of back "
                         "to back over copies of its inputs (keeps the device footprint at one copy, e.g. for ncu)")
    ap.add_argument("--no-extra", action="store_true",
                    help="with the default workload, skip the T = 131072 configurations measured beside it")
    ap.add_argument("--separate", action="store_true",
                    help="run the indexer, top-k and gather-attend as three launches (same as --path separate)")
    ap.add_argument("--path", choices=("auto", "step", "select_attend", "separate"), default="auto",
                    help="sparse decode workloads: one persistent launch (step), indexer + fused select/attend, "
                         "or three launches; auto takes indexer + fused select/attend for token-level bf16 "
                         "selection and three launches otherwise")
    ap.add_argument("--graph", action="store_true",
                    help="time each flushed step as one replay of a CUDA graph of its calls")
    ap.add_argument("--no-lookahead", action="store_true",
                    help="lookahead and cached tiered workloads: run every call in order on one stream "
                         "(no selection of the next layer, or promotion of the previous step, beside others)")
    ap.add_argument("--tiered-path", choices=("staged", "fused"), default="staged",
                    help="tiered workloads: stage the selected host rows into HBM with one copy kernel "
                         "before the attention (staged), or read them inside the fused select/attend")
    args = ap.parse_args(raw_argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rc = self_spawn(args, raw_argv)
    if rc is not None:
        if rc != 0:
            raise SystemExit(rc)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
