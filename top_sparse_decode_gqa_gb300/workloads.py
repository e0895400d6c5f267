"""Seeded synthetic workloads for top-k sparse decode attention with GQA.

This module only draws inputs.  It holds none of the method's arithmetic (no scoring,
selection, softmax or tiering), so both the CUDA path and the CPU oracle can be fed from
it.  Every tensor is drawn on the host from one CPU ``torch.Generator`` seeded with
``1000 + cfg_id``, in a fixed order (indexer query, indexer keys, attention query, K, V,
planted positions and values, residency), so any two consumers see the same bytes.

The workloads are the shapes the source pages benchmark on, with synthetic values in
place of trained models and datasets (which the pages evaluate on and which are not
available here):

* ``c1_tiny``: one decode step, 4 query heads over 1 KV head, d = 64, T = 1024, fp32,
  top-64 tokens, 8 planted high-score tokens.
* ``c2_llama3_8b_gqa``: Llama-3-8B-shaped GQA layer, batch 8, 32/8 heads, d = 128, bf16,
  T = 32768, top-1024 tokens, 2 % planted heavy hitters.
* ``c3_block_sparse``: batch 4, 32/8 heads, d = 128, bf16, T = 131072 in 64-token blocks,
  top-64 blocks by the mean-pooled block key, exact attention over the 4096 rows.  Its
  indexer query is stored in fp16 (the same integers), to meet the fp16 pooled keys.
* ``c4_tiered_verify``: batch 4, 8 speculative-verify query tokens, 32/8 heads, d = 128,
  bf16, T = 131072, one top-2048 union per KV head, 10 % of positions resident in an HBM
  pool and the full cache in pinned host memory.
* ``c5_importance_tiering``: Qwen2.5-7B-shaped, 28 layers of 28/4 heads, d = 128, bf16,
  T = 65536, batch 2, dense decode for 64 steps accumulating the importance score, then
  a 20/40/30/10 % four-tier split.
* ``c6_window_blocks``: the Llama-3-8B-shaped layer of ``c2`` on the overlapping
  compression-window grid (windows of 32 tokens every 16): token scores max-pooled onto
  2047 windows, top-64 windows per KV head, attention over their union (at most 2048
  tokens, as 16-token segments).
* ``c7_head_topk``: the layer of ``c2`` with selection per query head: each head's own
  unscaled attention logits against its KV head's keys score the tokens, each head keeps
  its own top-1024 and attends over those rows only (the indexer tensors are drawn, to keep
  the draw order, but not used).
* ``c8_verify_layer_group``: a speculative-verify step over a group of 4 Llama-shaped layers
  that share one selection: batch 2, 8 draft tokens, 32/8 heads, d = 128, bf16, T = 32768;
  one indexer pass and one union top-1024 per KV head serve all 4 layers; every layer
  appends the 8 drafts' K/V to its own 64-slot window-bounded ring (which already holds the
  56 most recent accepted tokens) and attends the selected rows plus the ring, causally
  among the drafts.
* ``c9_lookahead_tiered``: 4 layers of the tiered verify layer of ``c4`` at batch 2, each
  with its own indexer query and keys (a selection per layer), its own K/V cache in pinned
  host memory and its own HBM pool of the same resident 10 % of positions; the step runs
  layer l+1's indexer, top-k and host-row staging ahead, beside layer l's attention.
* ``c10_cached_tiered``: the tiered verify layer of ``c4`` (10 % pool), over 16 decode
  steps whose 8 verify queries slide along a sequence of 23 indexer queries (each step
  drops the oldest and adds one), so consecutive selections overlap; residency is kept per
  (sequence, KV head) -- every head starts from the generated resident positions -- and the
  pool is a cache: each step stages the selected rows the pool lacks, attends, and then
  promotes those rows from the stage into the pool (beside the next step's selection).
* ``c11_tiered_attention``: the shape of ``c5`` (28 layers of 28/4 heads, T = 65536, batch
  2) one decode step after tiering: the four tiers of a seeded importance score
  (``importance_scores``, seed 2011; 20/40/30/10 %) drive every layer's dense attention --
  T0 and T1 rows read at bf16 from HBM, T2 rows as int8 codes and per-row scales (the
  int8 encode of each layer's K and V), T3 rows left out.

Value recipe: indexer query and keys are integers drawn uniformly from [-8, 8] (exact in
bf16 and fp32); attention q, K, V are standard normal, rounded to bf16 (nearest even)
where the workload is bf16.  Planted tokens (c1, c2) get indexer keys aligned with the
indexer query's signs (c1: 8 * sign, c2: sign * U{5..8}); in c2 their attention keys also
get + 0.5 x the mean of the group's query heads so they are heavy hitters in the softmax
too.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int
    B: int            # sequences in the batch
    V: int            # query tokens per sequence (speculative-verify batch; 1 = plain decode)
    Hq: int           # attention query heads
    Hkv: int          # KV heads (= indexer heads, one per GQA group)
    d: int            # head dim
    T: int            # cached tokens per sequence
    dtype: str        # "f32" or "bf16": storage type of q, K, V and the indexer tensors
    dI: int           # indexer head dim
    k: int            # selected tokens (block == 1) or blocks per (b, kvh); k*block == T: dense
    block: int = 1    # selection granularity in tokens
    planted: int = 0  # planted high-score tokens per (b, kvh)
    planted_values: str = "none"  # "eight" (c1) or "five_to_eight" (c2)
    planted_attn_boost: float = 0.0
    resident_frac: float = 1.0    # fraction of positions resident in the HBM pool
    layers: int = 1
    steps: int = 1
    window_kernel: int = 0  # > 0: select compression windows of this many tokens ...
    window_stride: int = 0  # ... moved by this many (k counts windows)
    per_head: bool = False  # select per query head from the attention logits (k per head)
    ring_w: int = 0         # > 0: draft-token ring of this many slots per layer (verify loop)
    q_idx_dtype: str = ""   # storage type of the indexer query if not `dtype` ("f16": with fp16 pooled keys)
    layer_indexers: bool = False  # one indexer query and key set per layer (selection per layer)
    drift_steps: int = 0    # > 0: decode steps whose V verify queries slide along a query sequence
    slot_per_head: bool = False  # residency (slot map) per (sequence, KV head) instead of per sequence
    tiered_attention: bool = False  # the attention reads the four tiers of a seeded importance score
    cum_frac: tuple = (0.2, 0.6, 0.9)
    n_sink: int = 0
    n_recent: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def dense(self) -> bool:
        return self.k * self.block == self.T

    @property
    def n_rows(self) -> int:
        """Selected K/V row slots per (b, kvh) after block expansion (windows: the segment
        slots of their union, some of them empty)."""
        if self.window_kernel > 0:
            return self.k * self.window_kernel
        return self.k * self.block

    @property
    def N(self) -> int:
        """Entries the indexer scores per (b, kvh): tokens, or blocks in block mode."""
        return self.T // self.block

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def pool_rows(self) -> int:
        return int(math.floor(self.resident_frac * self.T))

    @property
    def queries_per_step(self) -> int:
        return self.B * self.V

    def scaled(self, **overrides) -> "Workload":
        """Same structure at other sizes (parity cases the oracle finishes quickly).
        The planted count keeps its 2 % share when T changes, unless given."""
        if "T" in overrides and "planted" not in overrides and self.planted_values == "five_to_eight":
            overrides["planted"] = int(math.floor(0.02 * overrides["T"]))
        if "name" not in overrides:
            overrides["name"] = self.name + "_scaled"
        return dataclasses.replace(self, **overrides)


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("c1_tiny", 0, B=1, V=1, Hq=4, Hkv=1, d=64, T=1024, dtype="f32", dI=64, k=64,
                 planted=8, planted_values="eight"),
        Workload("c2_llama3_8b_gqa", 1, B=8, V=1, Hq=32, Hkv=8, d=128, T=32768, dtype="bf16",
                 dI=128, k=1024, planted=655, planted_values="five_to_eight",
                 planted_attn_boost=0.5),
        Workload("c3_block_sparse", 2, B=4, V=1, Hq=32, Hkv=8, d=128, T=131072, dtype="bf16",
                 dI=128, k=64, block=64, q_idx_dtype="f16"),
        Workload("c4_tiered_verify", 3, B=4, V=8, Hq=32, Hkv=8, d=128, T=131072, dtype="bf16",
                 dI=128, k=2048, resident_frac=0.1),
        Workload("c5_importance_tiering", 4, B=2, V=1, Hq=28, Hkv=4, d=128, T=65536,
                 dtype="bf16", dI=128, k=65536, layers=28, steps=64),
        Workload("c6_window_blocks", 5, B=8, V=1, Hq=32, Hkv=8, d=128, T=32768, dtype="bf16",
                 dI=128, k=64, planted=655, planted_values="five_to_eight", planted_attn_boost=0.5,
                 window_kernel=32, window_stride=16),
        Workload("c7_head_topk", 6, B=8, V=1, Hq=32, Hkv=8, d=128, T=32768, dtype="bf16",
                 dI=128, k=1024, planted=655, planted_values="five_to_eight", planted_attn_boost=0.5,
                 per_head=True),
        Workload("c8_verify_layer_group", 7, B=2, V=8, Hq=32, Hkv=8, d=128, T=32768, dtype="bf16",
                 dI=128, k=1024, layers=4, ring_w=64),
        Workload("c9_lookahead_tiered", 8, B=2, V=8, Hq=32, Hkv=8, d=128, T=131072, dtype="bf16",
                 dI=128, k=2048, resident_frac=0.1, layers=4, layer_indexers=True),
        Workload("c11_tiered_attention", 10, B=2, V=1, Hq=28, Hkv=4, d=128, T=65536, dtype="bf16", dI=128,
                 k=65536, layers=28, steps=1, tiered_attention=True),
        Workload("c10_cached_tiered", 9, B=4, V=8, Hq=32, Hkv=8, d=128, T=131072, dtype="bf16",
                 dI=128, k=2048, resident_frac=0.1, drift_steps=16, slot_per_head=True),
    )
}


def _store(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to({"f32": torch.float32, "f16": torch.float16}.get(dtype, torch.bfloat16))


def _randint(g, shape, dtype):
    return _store(torch.randint(-8, 9, shape, generator=g, dtype=torch.int16), dtype)


def _randn(g, shape, dtype, chunk_rows: int = 1 << 22):
    """Standard normal, drawn in row chunks along dim 0 to bound the fp32 temporary."""
    out = torch.empty(shape, dtype=torch.float32 if dtype == "f32" else torch.bfloat16)
    flat = out.view(-1, shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, shape[-1]), generator=g, dtype=torch.float32)
    return out


def generate(w: Workload, seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw every input of workload ``w`` on the host (CPU tensors).

    Keys: ``q_idx`` [B,Hkv,V,dI], ``k_idx`` [B,Hkv,T,dI] (indexer); ``q`` [B,V,Hq,d] (or
    [steps,layers,B,V,Hq,d] when layers*steps > 1); ``k``, ``v`` [B,Hkv,T,d] (or a list of
    per-layer tensors); ``planted`` int64 [B,Hkv,planted] positions (sorted); and, when
    resident_frac < 1, ``resident`` int64 [B,P] sorted resident positions, ``slot_map``
    int32 [B,T] (slot or -1) and ``k_pool``, ``v_pool`` [B,Hkv,P,d].  With a draft ring
    (ring_w > 0): ``ring_k``, ``ring_v`` [layers,B,Hkv,W,d] (slots of the recent accepted
    tokens T-(W-V) .. T-1 filled, at slot position mod W), ``ring_pos`` int32 [B,W] (-1 where
    empty), ``draft_k``, ``draft_v`` [layers,B,Hkv,V,d] (the V draft tokens, positions
    T .. T+V-1, appended by the step) and ``qpos`` int32 [B,V] = T + v.
    """
    g = torch.Generator().manual_seed(1000 + w.cfg_id if seed is None else seed)
    B, Hkv, V, T = w.B, w.Hkv, w.V, w.T
    out: Dict[str, torch.Tensor] = {}
    # 1. indexer query, 2. indexer keys (per layer: all layers' queries, then all layers' keys)
    if w.layer_indexers:
        out["q_idx"] = _randint(g, (w.layers, B, Hkv, V, w.dI), w.q_idx_dtype or w.dtype)
        out["k_idx"] = [_randint(g, (B, Hkv, T, w.dI), w.dtype) for _ in range(w.layers)]
    else:
        out["q_idx"] = _randint(g, (B, Hkv, V, w.dI), w.q_idx_dtype or w.dtype)
        out["k_idx"] = _randint(g, (B, Hkv, T, w.dI), w.dtype)
    # 3. attention query
    if w.layers * w.steps > 1:
        out["q"] = _randn(g, (w.steps, w.layers, B, V, w.Hq, w.d), w.dtype)
    else:
        out["q"] = _randn(g, (B, V, w.Hq, w.d), w.dtype)
    # 4. K, 5. V
    if w.layers > 1:
        ks, vs = [], []
        for _ in range(w.layers):
            ks.append(_randn(g, (B, Hkv, T, w.d), w.dtype))
            vs.append(_randn(g, (B, Hkv, T, w.d), w.dtype))
        out["k"], out["v"] = ks, vs
    else:
        out["k"] = _randn(g, (B, Hkv, T, w.d), w.dtype)
        out["v"] = _randn(g, (B, Hkv, T, w.d), w.dtype)
    # 6. planted positions and values
    if w.planted > 0:
        pos = torch.empty((B, Hkv, w.planted), dtype=torch.int64)
        for b in range(B):
            for h in range(Hkv):
                pos[b, h] = torch.sort(torch.randperm(T, generator=g)[: w.planted]).values
        sign = torch.where(out["q_idx"][:, :, 0, :].float() >= 0, 1.0, -1.0)  # [B,Hkv,dI]
        for b in range(B):
            for h in range(Hkv):
                p = pos[b, h]
                if w.planted_values == "eight":
                    vals = 8.0 * sign[b, h].expand(len(p), w.dI)
                else:
                    mag = torch.randint(5, 9, (len(p), w.dI), generator=g).float()
                    vals = sign[b, h] * mag
                out["k_idx"][b, h, p] = _store(vals, w.dtype)
                if w.planted_attn_boost != 0.0:
                    qbar = out["q"][b, 0, h * w.G:(h + 1) * w.G, :].float().mean(0)
                    kp = out["k"][b, h, p].float() + w.planted_attn_boost * qbar
                    out["k"][b, h, p] = _store(kp, w.dtype)
        out["planted"] = pos
    # 7. residency: a uniform share of positions per sequence lives in the HBM pool
    if w.resident_frac < 1.0:
        P = w.pool_rows
        res = torch.empty((B, P), dtype=torch.int64)
        slot_map = torch.full((B, T), -1, dtype=torch.int32)
        for b in range(B):
            res[b] = torch.sort(torch.randperm(T, generator=g)[:P]).values
            slot_map[b, res[b]] = torch.arange(P, dtype=torch.int32)
        out["resident"] = res
        out["slot_map"] = slot_map
        idx = res[:, None, :, None].expand(B, Hkv, P, w.d)
        if isinstance(out["k"], list):  # every layer's pool holds the same resident positions
            out["k_pool"] = [torch.gather(k, 2, idx).contiguous() for k in out["k"]]
            out["v_pool"] = [torch.gather(v, 2, idx).contiguous() for v in out["v"]]
        else:
            out["k_pool"] = torch.gather(out["k"], 2, idx).contiguous()
            out["v_pool"] = torch.gather(out["v"], 2, idx).contiguous()
    # 8. sliding indexer queries: a sequence of V + drift_steps - 1 queries per (b, kvh);
    # step s uses queries s .. s + V - 1
    if w.drift_steps > 0:
        out["q_idx_seq"] = _randint(g, (B, Hkv, V + w.drift_steps - 1, w.dI), w.q_idx_dtype or w.dtype)
    # 9. draft ring: its K/V, then the drafts' K/V
    if w.ring_w > 0:
        W, L = w.ring_w, max(1, w.layers)
        out["ring_k"] = _randn(g, (L, B, Hkv, W, w.d), w.dtype)
        out["ring_v"] = _randn(g, (L, B, Hkv, W, w.d), w.dtype)
        out["draft_k"] = _randn(g, (L, B, Hkv, V, w.d), w.dtype)
        out["draft_v"] = _randn(g, (L, B, Hkv, V, w.d), w.dtype)
        ring_pos = torch.full((B, W), -1, dtype=torch.int32)
        for t in range(max(0, T - (W - V)), T):
            ring_pos[:, t % W] = t
        out["ring_pos"] = ring_pos
        out["qpos"] = (T + torch.arange(V, dtype=torch.int32)).expand(B, V).contiguous()
    return out


def residency_map(B: int, T: int, P: int, seed: int):
    """A seeded uniform choice of P resident positions per sequence (sorted) and the
    matching slot map (slot s holds the s-th smallest resident position; -1 = host)."""
    g = torch.Generator().manual_seed(seed)
    res = torch.empty((B, P), dtype=torch.int64)
    slot_map = torch.full((B, T), -1, dtype=torch.int32)
    for b in range(B):
        res[b] = torch.sort(torch.randperm(T, generator=g)[:P]).values
        slot_map[b, res[b]] = torch.arange(P, dtype=torch.int32)
    return res, slot_map


def importance_scores(B: int, T: int, seed: int, ties: bool = False) -> torch.Tensor:
    """Seeded synthetic importance scores s [B,T] (fp64) for tier tests: positive values
    with a heavy tail, or coarse values with many exact ties when ``ties``."""
    g = torch.Generator().manual_seed(seed)
    if ties:
        return torch.randint(0, 16, (B, T), generator=g).to(torch.float64) / 8.0
    return torch.rand((B, T), generator=g, dtype=torch.float64) ** 4 * 3.0
