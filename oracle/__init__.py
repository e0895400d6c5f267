"""CPU oracle for top-k sparse decode attention with GQA -- TEST INFRASTRUCTURE ONLY.

This package wraps ``oracle.c`` (plain fp64 loops, one function per step of the method)
with numpy in / numpy out.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the CUDA library never does, and the two
share no code.  Each wrapper restates which passage of the source pages its step
follows (see the C source for the full citations).

Arrays: fp32 data is a float32 array; bfloat16 data is a uint16 array of raw bits (or a
CPU torch tensor of dtype bfloat16, which is viewed as such without copying).
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_num_threads.restype = I
        lib.oracle_index_score.argtypes = [P, I, P, I, I, I, I, I, I, P]
        lib.oracle_block_pool.argtypes = [P, I, I, I, I, I, I, P]
        lib.oracle_topk.argtypes = [P, I, I, I, P]
        lib.oracle_gather_attend.argtypes = [P, P, P, I, P, I, I, I, I, I, I, I, I, D, P, P, P, I]
        lib.oracle_index_score_heads.argtypes = [P, I, P, I, I, I, I, I, I, P]
        lib.oracle_score_accumulate.argtypes = [P, P, P, I, I, I, I, I, I, I, D, P]
        lib.oracle_tier_classify.argtypes = [P, I, I, P, I, I, P, P]
        lib.oracle_quantize_rows_int8.argtypes = [P, I, P, I, I, I, I, P, P]
        lib.oracle_window_count.argtypes = [I, I, I]
        lib.oracle_window_max.argtypes = [P, I, I, I, I, P]
        lib.oracle_window_union.argtypes = [P, I, I, I, I, I, P, I]
        lib.oracle_gather_attend_ring.argtypes = [P, P, P, I, P, I, I, I, I, I, I, I, I, D, P, P, P, P, I, P, P,
                                                  P]
        for name in ("oracle_index_score", "oracle_block_pool", "oracle_topk",
                     "oracle_gather_attend", "oracle_gather_attend_ring", "oracle_score_accumulate", "oracle_tier_classify",
                     "oracle_quantize_rows_int8", "oracle_window_count", "oracle_window_max",
                     "oracle_window_union", "oracle_index_score_heads"):
            getattr(lib, name).restype = I
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc == -1:
        raise OracleError(f"{what}: invalid argument")
    if rc == -2:
        raise OracleError(f"{what}: selected row index out of range")
    if rc != 0:
        raise OracleError(f"{what}: error {rc}")


def _as_data(x):
    """Return (contiguous numpy array, dtype code) for fp32, bfloat16 or float16 data (float16
    passed on as the equal fp32 values)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            if x.dtype == torch.float16:  # every binary16 value is a binary32 value: exact
                return x.to(torch.float32).numpy(), F32
            raise TypeError(f"unsupported tensor dtype {x.dtype}")
    except ImportError:
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"unsupported array dtype {x.dtype} (float32, or uint16 bfloat16 bits)")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def num_threads() -> int:
    """OpenMP threads the oracle runs on (all host cores unless OMP_NUM_THREADS says)."""
    return _load().oracle_num_threads()


def index_score(q_idx, k_idx, B, Hkv, V, N, dI):
    """Compact indexer score, max over the V verify queries (SparDA, "Indexador de
    Previsao Compacto").  Returns fp64 [B,Hkv,N]."""
    q, qd = _as_data(q_idx)
    k, kd = _as_data(k_idx)
    assert q.size == B * Hkv * V * dI and k.size == B * Hkv * N * dI
    out = np.empty((B, Hkv, N), dtype=np.float64)
    _check(_load().oracle_index_score(_ptr(q), qd, _ptr(k), kd, B, Hkv, V, N, dI, _ptr(out)),
           "index_score")
    return out


def index_score_heads(q, k, B, Hkv, V, N, dI):
    """Per-query scores (Illusion sec. 2, Oracle Top-K per query head): fp64 [B,Hkv,V,N],
    scores[b,h,v,t] = sum_j q[b,h,v,j] k[b,h,t,j] (no max over v)."""
    qa, qd = _as_data(q)
    ka, kd = _as_data(k)
    assert qa.size == B * Hkv * V * dI and ka.size == B * Hkv * N * dI
    out = np.empty((B, Hkv, V, N), dtype=np.float64)
    _check(_load().oracle_index_score_heads(_ptr(qa), qd, _ptr(ka), kd, B, Hkv, V, N, dI, _ptr(out)),
           "index_score_heads")
    return out


def block_pool(k_idx, B, Hkv, T, dI, block):
    """Mean of each disjoint block of `block` indexer keys (SparDA, block grid).
    Returns fp64 [B,Hkv,T/block,dI]."""
    k, kd = _as_data(k_idx)
    assert k.size == B * Hkv * T * dI
    out = np.empty((B, Hkv, T // block, dI), dtype=np.float64)
    _check(_load().oracle_block_pool(_ptr(k), kd, B, Hkv, T, dI, block, _ptr(out)), "block_pool")
    return out


def topk(scores, k):
    """Exact top-k per row, ties to the lower index, ascending output (Illusion,
    "Oracle Top-K").  scores [..., N] (any float type, compared as fp64) -> int32 [..., k]."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    N = s.shape[-1]
    rows = s.size // N if N > 0 else int(np.prod(s.shape[:-1]))
    out = np.empty(s.shape[:-1] + (k,), dtype=np.int32)
    _check(_load().oracle_topk(_ptr(s), rows, N, k, _ptr(out)), "topk")
    return out


def window_count(N, kernel, stride):
    """Compression windows of `kernel` scores every `stride` over N scores (SparDA,
    "Estrategia de Treinamento": the (32, 16) inference grid)."""
    return _load().oracle_window_count(N, kernel, stride)


def window_max(scores, kernel, stride):
    """Window score = max of the token scores the window covers.  scores [..., N] (compared
    as fp64) -> fp64 [..., NW]."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    N = s.shape[-1]
    rows = s.size // N if N > 0 else int(np.prod(s.shape[:-1]))
    NW = window_count(N, kernel, stride)
    out = np.empty(s.shape[:-1] + (NW,), dtype=np.float64)
    _check(_load().oracle_window_max(_ptr(s), rows, N, kernel, stride, _ptr(out)), "window_max")
    return out


def window_union(widx, N, kernel, stride, max_segs=None):
    """Union of the selected windows' segments of `stride` tokens, ascending, padded with -1
    (empty slots).  widx [..., k] int -> int32 [..., max_segs] (default k * kernel/stride)."""
    w = np.ascontiguousarray(widx, dtype=np.int32)
    k = w.shape[-1]
    rows = w.size // k if k > 0 else int(np.prod(w.shape[:-1]))
    if max_segs is None:
        max_segs = k * (kernel // stride)
    out = np.empty(w.shape[:-1] + (max_segs,), dtype=np.int32)
    _check(_load().oracle_window_union(_ptr(w), rows, k, N, kernel, stride, _ptr(out), max_segs),
           "window_union")
    return out


def gather_attend(q, K, Vv, idx, B, V, Hq, Hkv, d, T, n_idx, block, scale, want_logits=False, per_head=False):
    """Exact softmax attention of every query row over the selected rows only
    (Illusion sec. 2 / 3C).  idx None means dense (all T rows).
    Returns (out fp64 [B,V,Hq,d], lse fp64 [B,V,Hq], logits fp64 [B,V,Hq,n_idx*block] or None)."""
    qa, qd = _as_data(q)
    ka, kd = _as_data(K)
    va, vd = _as_data(Vv)
    assert qd == kd == vd, "q, K and V must share one dtype"
    assert qa.size == B * V * Hq * d and ka.size == B * Hkv * T * d and va.size == ka.size
    ia = None
    if idx is not None:
        ia = np.ascontiguousarray(idx, dtype=np.int32)
        assert ia.size == B * (Hq if per_head else Hkv) * n_idx
    out = np.empty((B, V, Hq, d), dtype=np.float64)
    lse = np.empty((B, V, Hq), dtype=np.float64)
    logits = np.empty((B, V, Hq, n_idx * block), dtype=np.float64) if want_logits else None
    _check(_load().oracle_gather_attend(_ptr(qa), _ptr(ka), _ptr(va), qd, _ptr(ia), B, V, Hq, Hkv,
                                        d, T, n_idx, block, float(scale), _ptr(out), _ptr(lse),
                                        _ptr(logits), 1 if per_head else 0), "gather_attend")
    return out, lse, logits


def gather_attend_ring(q, K, Vv, idx, B, V, Hq, Hkv, d, T, n_idx, block, scale, ring_k, ring_v, ring_pos, qpos,
                       want_logits=False):
    """Verify attention with the draft tokens' window-bounded ring (Adaptive DHiSparse,
    "Metodologia"): the selected history rows as gather_attend, plus every ring slot s of
    the KV head with 0 <= ring_pos[b,s] <= qpos[b,v].  ring_k/ring_v [B,Hkv,W,d] (dtype of
    q), ring_pos int [B,W] (-1 = empty), qpos int [B,V].  Returns (out, lse, logits
    [B,V,Hq,n_idx*block + W] or None), fp64."""
    qa, qd = _as_data(q)
    ka, kd = _as_data(K)
    va, vd = _as_data(Vv)
    rka, rkd = _as_data(ring_k)
    rva, rvd = _as_data(ring_v)
    assert qd == kd == vd == rkd == rvd, "q, K, V and the ring must share one dtype"
    W = ring_pos.shape[-1]
    assert qa.size == B * V * Hq * d and ka.size == B * Hkv * T * d and va.size == ka.size
    assert rka.size == B * Hkv * W * d and rva.size == rka.size
    rp = np.ascontiguousarray(ring_pos, dtype=np.int32)
    qp = np.ascontiguousarray(qpos, dtype=np.int32)
    assert rp.size == B * W and qp.size == B * V
    ia = None
    if idx is not None:
        ia = np.ascontiguousarray(idx, dtype=np.int32)
        assert ia.size == B * Hkv * n_idx
    out = np.empty((B, V, Hq, d), dtype=np.float64)
    lse = np.empty((B, V, Hq), dtype=np.float64)
    logits = np.empty((B, V, Hq, n_idx * block + W), dtype=np.float64) if want_logits else None
    _check(_load().oracle_gather_attend_ring(_ptr(qa), _ptr(ka), _ptr(va), qd, _ptr(ia), B, V, Hq, Hkv, d, T, n_idx,
                                             block, float(scale), _ptr(rka), _ptr(rva), _ptr(rp), _ptr(qp), W,
                                             _ptr(out), _ptr(lse), _ptr(logits)), "gather_attend_ring")
    return out, lse, logits


def ring_append(k_new, v_new, ring_k, ring_v, ring_pos, pos0):
    """Appends n new tokens to the window-bounded ring (Adaptive DHiSparse, "Metodologia"):
    token i of sequence b (position pos0[b] + i) goes to slot (pos0[b] + i) mod W.
    k_new/v_new [B,Hkv,n,d]; ring_k/ring_v [B,Hkv,W,d] and ring_pos [B,W] (numpy arrays or
    CPU tensors) are updated in place, token by token in order."""
    B, Hkv, n, _ = k_new.shape
    W = ring_pos.shape[-1]
    for b in range(B):
        for i in range(n):
            pos = int(pos0[b]) + i
            slot = pos % W
            for h in range(Hkv):
                ring_k[b, h, slot] = k_new[b, h, i]
                ring_v[b, h, slot] = v_new[b, h, i]
            ring_pos[b, slot] = pos


def score_accumulate(logits, lse, idx, s, B, V, Hq, Hkv, n_idx, block, T, weight):
    """One layer's term of the cumulative importance score (Not All Thoughts Need HBM,
    Metodologia 2), added in place to the fp64 array s [B,T]."""
    la = np.ascontiguousarray(logits, dtype=np.float64)
    ea = np.ascontiguousarray(lse, dtype=np.float64)
    assert s.dtype == np.float64 and s.flags.c_contiguous and s.size == B * T
    ia = None if idx is None else np.ascontiguousarray(idx, dtype=np.int32)
    _check(_load().oracle_score_accumulate(_ptr(la), _ptr(ea), _ptr(ia), B, V, Hq, Hkv, n_idx,
                                           block, T, float(weight), _ptr(s)), "score_accumulate")
    return s


def tier_classify(s, cum_frac, n_sink=0, n_recent=0):
    """Four-tier split by importance rank (Not All Thoughts Need HBM, Metodologia 1).
    s [B,T] -> (tier uint8 [B,T], counts int32 [B,4])."""
    sa = np.ascontiguousarray(s, dtype=np.float64)
    B, T = sa.shape
    fr = np.ascontiguousarray(cum_frac, dtype=np.float64)
    assert fr.size == 3
    tier = np.empty((B, T), dtype=np.uint8)
    counts = np.empty((B, 4), dtype=np.int32)
    _check(_load().oracle_tier_classify(_ptr(sa), B, T, _ptr(fr), n_sink, n_recent, _ptr(tier),
                                        _ptr(counts)), "tier_classify")
    return tier, counts


def quantize_rows_int8(x, tier, B, Hkv, T, d, codes=None, scales=None):
    """Symmetric per-row int8 codes of the rows whose tier is 2 (Not All Thoughts Need
    HBM, Metodologia 1, T2).  Rows of other tiers keep what `codes`/`scales` held (zeros
    if they are created here).  Returns (codes int8 [B,Hkv,T,d], scales fp32 [B,Hkv,T])."""
    xa, xd = _as_data(x)
    ta = np.ascontiguousarray(tier, dtype=np.uint8)
    assert xa.size == B * Hkv * T * d and ta.size == B * T
    if codes is None:
        codes = np.zeros((B, Hkv, T, d), dtype=np.int8)
    if scales is None:
        scales = np.zeros((B, Hkv, T), dtype=np.float32)
    _check(_load().oracle_quantize_rows_int8(_ptr(xa), xd, _ptr(ta), B, Hkv, T, d, _ptr(codes),
                                             _ptr(scales)), "quantize_rows_int8")
    return codes, scales


def promote_rows(idx, block, slot_map, pool_pos, hand, k_host, v_host, k_pool, v_pool):
    """Keeps the HBM pool as a cache of host rows (Adaptive DHiSparse "Metodologia": the
    pool holds extra history while memory allows; SparDA sec. 2 item 3: needed rows are
    fetched ahead).  Reading taken, per sequence b:
      1. the step's selected positions are the union over the KV heads of the rows of
         idx[b, h, :] (block-expanded; -1 entries empty);
      2. the misses are the selected positions whose slot_map is -1, in ascending order;
      3. a slot is pinned when it holds a selected position; the victims are the first
         unpinned slots in ring order starting at hand[b], one per miss while they last;
      4. miss m goes to victim m: the victim's old position (if any) leaves the pool
         (slot_map = -1), the miss's host K/V rows of every KV head are copied into the
         slot, slot_map[b, miss] = slot, pool_pos[b, slot] = miss;
      5. hand[b] moves past the last victim taken (unchanged when there is none).
    All arrays are numpy (modified in place): idx [B,Hkv,n_idx], slot_map [B,T],
    pool_pos [B,P], hand [B], k/v_host [B,Hkv,T,d], k/v_pool [B,Hkv,P,d].
    Returns the number of rows promoted per sequence."""
    B, Hkv, n_idx = idx.shape
    T, P = slot_map.shape[1], pool_pos.shape[1]
    promoted = []
    for b in range(B):
        sel = set()
        for h in range(Hkv):
            for e in idx[b, h]:
                if e >= 0:
                    sel.update(range(int(e) * block, int(e) * block + block))
        misses = sorted(t for t in sel if slot_map[b, t] == -1)
        victims = []
        for i in range(P):
            if len(victims) == len(misses):
                break
            s = (int(hand[b]) + i) % P
            if pool_pos[b, s] < 0 or int(pool_pos[b, s]) not in sel:
                victims.append(s)
        for t, s in zip(misses, victims):
            old = int(pool_pos[b, s])
            if old >= 0:
                slot_map[b, old] = -1
            k_pool[b, :, s] = k_host[b, :, t]
            v_pool[b, :, s] = v_host[b, :, t]
            slot_map[b, t] = s
            pool_pos[b, s] = t
        taken = min(len(misses), len(victims))
        if taken:
            hand[b] = (victims[taken - 1] + 1) % P
        promoted.append(taken)
    return promoted
