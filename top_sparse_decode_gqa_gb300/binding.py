"""Thin Python binding over libsdgqa's C ABI (include/sd.h), with the same call names.

Argument marshalling only: shapes are read off torch tensors, pointers and the current
CUDA stream are passed through, and a non-OK status raises ``SdError``.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback of any kind, and
a missing library is an error.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdgqa.so")

SD_OK, SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED, SD_ERR_CUDA = 0, 1, 2, 3
SD_F32, SD_BF16, SD_F16 = 0, 1, 2
SD_DEVERR_INDEX, SD_DEVERR_SLOT, SD_DEVERR_TIMEOUT = 0x1, 0x2, 0x4

# Every symbol include/sd.h declares (checked by the tests against the built library).
EXPORTS = (
    "sd_version", "sd_status_string", "sd_last_error_message", "sd_index_score", "sd_block_pool",
    "sd_topk_workspace_bytes", "sd_topk", "sd_gather_attend_workspace_bytes", "sd_gather_attend",
    "sd_score_accumulate", "sd_tier_classify_workspace_bytes", "sd_tier_classify",
    "sd_quantize_rows_int8", "sd_gather_attend_noalloc", "sd_select_attend", "sd_window_count",
    "sd_window_max", "sd_window_union", "sd_index_score_heads", "sd_stage_host_rows", "sd_ring_append",
    "sd_promote_rows_workspace_bytes", "sd_promote_rows", "sd_promote_staged_rows_workspace_bytes",
    "sd_promote_staged_rows", "sd_decode_step_workspace_bytes", "sd_decode_step",
)


class SdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class sd_attend_args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("k_host", ctypes.c_void_p), ("v_host", ctypes.c_void_p), ("slot_map", ctypes.c_void_p),
        ("idx", ctypes.c_void_p), ("dtype", ctypes.c_int),
        ("B", ctypes.c_int), ("V", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("d", ctypes.c_int), ("T", ctypes.c_int), ("pool_rows", ctypes.c_int),
        ("n_idx", ctypes.c_int), ("block", ctypes.c_int), ("scale", ctypes.c_float),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("logits", ctypes.c_void_p),
        ("err_word", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t), ("splits", ctypes.c_int), ("per_head", ctypes.c_int),
        ("k_stage", ctypes.c_void_p), ("v_stage", ctypes.c_void_p),
        ("ring_k", ctypes.c_void_p), ("ring_v", ctypes.c_void_p), ("ring_pos", ctypes.c_void_p),
        ("qpos", ctypes.c_void_p), ("ring_w", ctypes.c_int), ("slot_per_head", ctypes.c_int),
        ("tier", ctypes.c_void_p), ("k_int8", ctypes.c_void_p), ("v_int8", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("row_loop", ctypes.c_int),
    ]


class sd_decode_step_args(ctypes.Structure):
    _fields_ = [
        ("q_idx", ctypes.c_void_p), ("keys", ctypes.c_void_p), ("key_dtype", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("B", ctypes.c_int), ("V", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("d", ctypes.c_int), ("d_idx", ctypes.c_int), ("T", ctypes.c_int), ("block", ctypes.c_int),
        ("n_idx", ctypes.c_int), ("scale", ctypes.c_float),
        ("scores", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("err_word", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("lag", ctypes.c_int), ("wait_limit_ns", ctypes.c_longlong),
    ]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded libsdgqa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with top_sparse_decode_gqa_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_double
        L.sd_version.restype = I
        L.sd_status_string.restype = ctypes.c_char_p
        L.sd_status_string.argtypes = [I]
        L.sd_last_error_message.restype = ctypes.c_char_p
        L.sd_index_score.argtypes = [P, I, P, I, I, I, I, I, I, P, P, P, P]
        L.sd_block_pool.argtypes = [P, I, I, I, I, I, I, P, I, P]
        L.sd_topk_workspace_bytes.argtypes = [I, I, I]
        L.sd_topk_workspace_bytes.restype = Z
        L.sd_topk.argtypes = [P, I, I, I, P, P, P, Z, P]
        L.sd_gather_attend_workspace_bytes.argtypes = [ctypes.POINTER(sd_attend_args)]
        L.sd_gather_attend_workspace_bytes.restype = Z
        L.sd_gather_attend.argtypes = [ctypes.POINTER(sd_attend_args), P]
        L.sd_gather_attend_noalloc.argtypes = [ctypes.POINTER(sd_attend_args), P]
        L.sd_select_attend.argtypes = [P, I, P, P, ctypes.POINTER(sd_attend_args), P]
        L.sd_index_score_heads.argtypes = [P, I, P, I, I, I, I, I, I, P, P, P, P]
        L.sd_stage_host_rows.argtypes = [ctypes.POINTER(sd_attend_args), P, P]
        L.sd_ring_append.argtypes = [P, P, I, I, I, I, I, P, P, P, P, I, P]
        L.sd_promote_rows_workspace_bytes.argtypes = [ctypes.POINTER(sd_attend_args)]
        L.sd_promote_rows_workspace_bytes.restype = Z
        L.sd_promote_rows.argtypes = [ctypes.POINTER(sd_attend_args), P, P, P, Z, P]
        L.sd_promote_staged_rows_workspace_bytes.argtypes = [ctypes.POINTER(sd_attend_args)]
        L.sd_promote_staged_rows_workspace_bytes.restype = Z
        L.sd_promote_staged_rows.argtypes = [ctypes.POINTER(sd_attend_args), P, P, P, Z, P]
        L.sd_window_count.argtypes = [I, I, I]
        L.sd_window_count.restype = I
        L.sd_window_max.argtypes = [P, I, I, I, I, P, P, P]
        L.sd_window_union.argtypes = [P, I, I, I, I, I, P, I, P, P]
        L.sd_score_accumulate.argtypes = [P, P, P, I, I, I, I, I, I, I, D, P, P, P]
        L.sd_tier_classify_workspace_bytes.argtypes = [I, I]
        L.sd_tier_classify_workspace_bytes.restype = Z
        L.sd_tier_classify.argtypes = [P, I, I, P, I, I, P, P, P, Z, P]
        L.sd_quantize_rows_int8.argtypes = [P, I, P, I, I, I, I, P, P, P]
        L.sd_decode_step_workspace_bytes.argtypes = [ctypes.POINTER(sd_decode_step_args)]
        L.sd_decode_step_workspace_bytes.restype = Z
        L.sd_decode_step.argtypes = [ctypes.POINTER(sd_decode_step_args), P]
        L.sd_stage_host_rows.restype = I
        L.sd_select_attend.restype = I
        for name in ("sd_index_score", "sd_block_pool", "sd_topk", "sd_gather_attend",
                     "sd_score_accumulate", "sd_tier_classify", "sd_quantize_rows_int8",
                     "sd_gather_attend_noalloc", "sd_decode_step"):
            getattr(L, name).restype = I
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != SD_OK:
        msg = lib().sd_last_error_message().decode() or lib().sd_status_string(status).decode()
        raise SdError(status, f"{what}: {msg}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SD_F32
    if t.dtype == torch.bfloat16:
        return SD_BF16
    if t.dtype == torch.float16:
        return SD_F16
    raise TypeError(f"unsupported dtype {t.dtype} (float32, bfloat16 or float16)")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def sd_version() -> int:
    return lib().sd_version()


KEY_HIST_BINS = 2048


def key_hist_buffer(rows: int, device="cuda") -> torch.Tensor:
    """A zero-filled [rows, 2048] uint32 (held as int32) order-key histogram for
    sd_index_score / sd_topk."""
    return torch.zeros((rows, KEY_HIST_BINS), dtype=torch.int32, device=device)


def sd_index_score(q_idx: torch.Tensor, k_idx: torch.Tensor, scores: Optional[torch.Tensor] = None,
                   err_word: Optional[torch.Tensor] = None, stream=None,
                   key_hist: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Indexer scores [B,Hkv,N] fp32 from q_idx [B,Hkv,V,dI] and k_idx [B,Hkv,N,dI]
    (optionally accumulating their order-key histogram into key_hist)."""
    _dev(q_idx, "q_idx")
    _dev(k_idx, "k_idx")
    B, Hkv, V, dI = q_idx.shape
    N = k_idx.shape[2]
    if tuple(k_idx.shape) != (B, Hkv, N, dI):
        raise ValueError("k_idx shape must be [B,Hkv,N,dI] matching q_idx")
    if scores is None:
        scores = torch.empty((B, Hkv, N), dtype=torch.float32, device=k_idx.device)
    _check(lib().sd_index_score(_ptr(q_idx), _dtype_code(q_idx), _ptr(k_idx), _dtype_code(k_idx), B,
                                Hkv, V, N, dI, _ptr(scores), _ptr(key_hist), _ptr(err_word),
                                _stream(stream)),
           "sd_index_score")
    return scores


def sd_index_score_heads(q: torch.Tensor, k: torch.Tensor, scores: Optional[torch.Tensor] = None,
                         err_word: Optional[torch.Tensor] = None, stream=None,
                         key_hist: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One score row per query row: scores [B,Hkv,V,N] from q [B,Hkv,V,d] and k [B,Hkv,N,d],
    no max over V.  With the attention query [B,1,Hq,d] viewed as [B,Hkv,G,d] and the
    attention keys, every query head's unscaled logits ([B,Hq,N] in memory)."""
    _dev(q, "q")
    _dev(k, "k")
    B, Hkv, V, d = q.shape
    N = k.shape[2]
    if tuple(k.shape) != (B, Hkv, N, d):
        raise ValueError("k shape must be [B,Hkv,N,d] matching q")
    if scores is None:
        scores = torch.empty((B, Hkv, V, N), dtype=torch.float32, device=k.device)
    _check(lib().sd_index_score_heads(_ptr(q), _dtype_code(q), _ptr(k), _dtype_code(k), B, Hkv, V, N, d,
                                      _ptr(scores), _ptr(key_hist), _ptr(err_word), _stream(stream)),
           "sd_index_score_heads")
    return scores


def sd_block_pool(k_idx: torch.Tensor, block: int, pooled: Optional[torch.Tensor] = None,
                  stream=None, dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """Mean-pooled block keys [B,Hkv,T/block,dI] of k_idx [B,Hkv,T,dI], as float32 or
    float16 (`dtype`, or the dtype of a given `pooled`)."""
    _dev(k_idx, "k_idx")
    B, Hkv, T, dI = k_idx.shape
    if pooled is None:
        pooled = torch.empty((B, Hkv, T // block, dI), dtype=dtype, device=k_idx.device)
    _check(lib().sd_block_pool(_ptr(k_idx), _dtype_code(k_idx), B, Hkv, T, dI, block, _ptr(pooled),
                               _dtype_code(pooled), _stream(stream)), "sd_block_pool")
    return pooled


def sd_topk(scores: torch.Tensor, k: int, idx: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, stream=None,
            key_hist: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Top-k indices (ascending, ties to the lower index) of each row of scores [..., N];
    key_hist: the histogram sd_index_score accumulated for these scores (zeroed again)."""
    _dev(scores, "scores")
    if scores.dtype != torch.float32:
        raise TypeError("scores must be float32")
    N = scores.shape[-1]
    rows = scores.numel() // N if N > 0 else math.prod(scores.shape[:-1])
    if idx is None:
        idx = torch.empty(scores.shape[:-1] + (k,), dtype=torch.int32, device=scores.device)
    ws_bytes = lib().sd_topk_workspace_bytes(rows, N, k)
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=scores.device)
    _check(lib().sd_topk(_ptr(scores), rows, N, k, _ptr(idx), _ptr(key_hist), _ptr(workspace),
                         ws_bytes, _stream(stream)), "sd_topk")
    return idx


def make_attend_args(q, k_cache, v_cache, idx=None, *, n_idx=None, block=1, T=None, scale=None,
                     k_host=None, v_host=None, slot_map=None, out=None, lse=None, logits=None,
                     want_logits=False, err_word=None, splits=0, per_head=False, k_stage=None,
                     v_stage=None, ring_k=None, ring_v=None, ring_pos=None, qpos=None, tier=None,
                     k_int8=None, v_int8=None, k_scale=None, v_scale=None, row_loop=False) -> tuple:
    """Fill an sd_attend_args from tensors; returns (args, out, lse, logits).  slot_map is
    [B,T] (residency per sequence) or [B,Hkv,T] (per KV head).  tier [B,T] uint8 with
    k_int8/v_int8 [B,Hkv,T,d] int8 and k_scale/v_scale [B,Hkv,T] fp32: the tiered rows.
    row_loop: a dense or tiled block-sparse call runs the general row loop (the one tiered
    calls take)."""
    _dev(q, "q")
    B, V, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    pool_rows = k_cache.shape[2]
    if T is None:
        T = k_host.shape[2] if k_host is not None else pool_rows
    if idx is not None:
        _dev(idx, "idx")
        n_idx = idx.shape[-1]
    elif n_idx is None:
        n_idx = T // block
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.device
    if out is None:
        out = torch.empty((B, V, Hq, d), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, V, Hq), dtype=torch.float32, device=dev)
    ring_w = ring_pos.shape[-1] if ring_pos is not None else 0
    if logits is None and want_logits:
        logits = torch.empty((B, V, Hq, n_idx * block + ring_w), dtype=torch.float32, device=dev)
    for name, t in (("k_host", k_host), ("v_host", v_host)):
        if t is not None and (t.is_cuda or not t.is_pinned() or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous pinned host tensor")
    a = sd_attend_args()
    a.q, a.k_cache, a.v_cache = q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr()
    a.k_host = k_host.data_ptr() if k_host is not None else None
    a.v_host = v_host.data_ptr() if v_host is not None else None
    a.slot_map = slot_map.data_ptr() if slot_map is not None else None
    a.idx = idx.data_ptr() if idx is not None else None
    a.dtype = _dtype_code(q)
    a.B, a.V, a.Hq, a.Hkv, a.d, a.T = B, V, Hq, Hkv, d, T
    a.pool_rows, a.n_idx, a.block = pool_rows, n_idx, block
    a.scale = scale
    a.out, a.lse = out.data_ptr(), lse.data_ptr()
    a.logits = logits.data_ptr() if logits is not None else None
    a.err_word = err_word.data_ptr() if err_word is not None else None
    a.splits = splits
    a.per_head = 1 if per_head else 0
    for name, t in (("k_stage", k_stage), ("v_stage", v_stage), ("ring_k", ring_k), ("ring_v", ring_v),
                    ("ring_pos", ring_pos), ("qpos", qpos), ("tier", tier), ("k_int8", k_int8),
                    ("v_int8", v_int8), ("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None:
            _dev(t, name)
            setattr(a, name, t.data_ptr())
    a.ring_w = ring_w
    a.slot_per_head = 1 if slot_map is not None and slot_map.dim() == 3 else 0
    a.row_loop = 1 if row_loop else 0
    return a, out, lse, logits


def sd_gather_attend_workspace_bytes(args: sd_attend_args) -> int:
    return lib().sd_gather_attend_workspace_bytes(ctypes.byref(args))


def sd_gather_attend(args: sd_attend_args, workspace: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    """Runs one sd_gather_attend call described by `args` (see make_attend_args).  The
    workspace must be zero-filled before its first use (torch.zeros); calls leave it so."""
    need = sd_gather_attend_workspace_bytes(args)
    if need:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"sd_gather_attend needs a workspace of {need} bytes")
        args.workspace = workspace.data_ptr()
        args.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().sd_gather_attend(ctypes.byref(args), _stream(stream)), "sd_gather_attend")


def sd_gather_attend_noalloc(args: sd_attend_args, stream=None) -> None:
    """Runs one sd_gather_attend_noalloc call: the same computation as sd_gather_attend,
    with the split-K scratch taken from the library's own static device array (for callers
    that cannot allocate); args.workspace is ignored."""
    _check(lib().sd_gather_attend_noalloc(ctypes.byref(args), _stream(stream)),
           "sd_gather_attend_noalloc")


def stage_buffers(args: sd_attend_args, dtype: torch.dtype, device="cuda") -> tuple:
    """HBM stage tensors (k_stage, v_stage) [groups, n_idx*block, d] for `args` (groups =
    B*Hkv, or B*Hq per head), set into args; returns them."""
    groups = args.B * (args.Hq if args.per_head else args.Hkv)
    shape = (groups, args.n_idx * args.block, args.d)
    ks = torch.empty(shape, dtype=dtype, device=device)
    vs = torch.empty(shape, dtype=dtype, device=device)
    args.k_stage, args.v_stage = ks.data_ptr(), vs.data_ptr()
    return ks, vs


def stage_counter(device="cuda") -> torch.Tensor:
    """A zero-filled device uint32[2] (held as int32) for sd_stage_host_rows."""
    return torch.zeros(2, dtype=torch.int32, device=device)


def sd_stage_host_rows(args: sd_attend_args, counter: torch.Tensor, stream=None) -> None:
    """Copies the selected host-resident rows `args` describes into args.k_stage/v_stage
    (see stage_buffers); counter from stage_counter, left at zero."""
    _dev(counter, "counter")
    _check(lib().sd_stage_host_rows(ctypes.byref(args), _ptr(counter), _stream(stream)), "sd_stage_host_rows")


def pool_state(slot_map: torch.Tensor, pool_rows: int) -> tuple:
    """(pool_pos [U, pool_rows], hand [U]) consistent with slot_map [B, T] (U = B) or
    [B, Hkv, T] (U = B*Hkv), device int32."""
    slot_map = slot_map.reshape(-1, slot_map.shape[-1])
    B, T = slot_map.shape
    pool_pos = torch.full((B, pool_rows), -1, dtype=torch.int32, device=slot_map.device)
    res = slot_map >= 0
    b, t = res.nonzero(as_tuple=True)
    pool_pos[b, slot_map[b, t].long()] = t.to(torch.int32)
    return pool_pos, torch.zeros(B, dtype=torch.int32, device=slot_map.device)


def sd_promote_rows_workspace_bytes(args: sd_attend_args) -> int:
    return lib().sd_promote_rows_workspace_bytes(ctypes.byref(args))


def sd_promote_rows(args: sd_attend_args, pool_pos: torch.Tensor, hand: torch.Tensor,
                    workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Promotes the selected host rows `args` describes into its pool (see include/sd.h);
    returns the workspace (zero-filled when created here), to pass to the next call."""
    _dev(pool_pos, "pool_pos")
    _dev(hand, "hand")
    need = lib().sd_promote_rows_workspace_bytes(ctypes.byref(args))
    if workspace is None:
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=pool_pos.device)
    _check(lib().sd_promote_rows(ctypes.byref(args), _ptr(pool_pos), _ptr(hand), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)), "sd_promote_rows")
    return workspace


def sd_promote_staged_rows_workspace_bytes(args: sd_attend_args) -> int:
    return lib().sd_promote_staged_rows_workspace_bytes(ctypes.byref(args))


def sd_promote_staged_rows(args: sd_attend_args, pool_pos: torch.Tensor, hand: torch.Tensor,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Promotes the step's misses from the stage `args` names into its pool, after the
    staging and the attention (see include/sd.h); returns the workspace (zero-filled when
    created here), to pass to the next call."""
    _dev(pool_pos, "pool_pos")
    _dev(hand, "hand")
    need = lib().sd_promote_staged_rows_workspace_bytes(ctypes.byref(args))
    if workspace is None:
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=pool_pos.device)
    _check(lib().sd_promote_staged_rows(ctypes.byref(args), _ptr(pool_pos), _ptr(hand), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)),
           "sd_promote_staged_rows")
    return workspace


def ring_buffers(B: int, Hkv: int, W: int, d: int, dtype: torch.dtype, device="cuda") -> tuple:
    """An empty draft ring: (ring_k, ring_v) [B,Hkv,W,d] zeros and ring_pos [B,W] = -1."""
    rk = torch.zeros((B, Hkv, W, d), dtype=dtype, device=device)
    return rk, torch.zeros_like(rk), torch.full((B, W), -1, dtype=torch.int32, device=device)


def sd_ring_append(k_new: torch.Tensor, v_new: torch.Tensor, ring_k: torch.Tensor, ring_v: torch.Tensor,
                   ring_pos: torch.Tensor, pos0: torch.Tensor, stream=None) -> None:
    """Writes k_new/v_new [B,Hkv,n,d] into the ring at slots (pos0[b] + i) mod W and records
    the positions in ring_pos [B,W]."""
    for name, t in (("k_new", k_new), ("v_new", v_new), ("ring_k", ring_k), ("ring_v", ring_v),
                    ("ring_pos", ring_pos), ("pos0", pos0)):
        _dev(t, name)
    B, Hkv, n, d = k_new.shape
    W = ring_k.shape[2]
    _check(lib().sd_ring_append(_ptr(k_new), _ptr(v_new), _dtype_code(k_new), B, Hkv, n, d, _ptr(ring_k),
                                _ptr(ring_v), _ptr(ring_pos), _ptr(pos0), W, _stream(stream)), "sd_ring_append")


def sd_select_attend(scores: torch.Tensor, args: sd_attend_args, idx: torch.Tensor,
                     key_hist: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Runs one sd_select_attend call: the top-args.n_idx selection of every row of scores
    [B, Hkv, N] written to idx [B, Hkv, n_idx], and the attention `args` describes over it
    (args.idx and the workspace are ignored)."""
    _dev(scores, "scores")
    _dev(idx, "idx")
    if scores.dtype != torch.float32 or idx.dtype != torch.int32:
        raise TypeError("scores must be float32 and idx int32")
    _check(lib().sd_select_attend(_ptr(scores), scores.shape[-1], _ptr(key_hist), _ptr(idx),
                                  ctypes.byref(args), _stream(stream)), "sd_select_attend")
    return idx


def sd_window_count(N: int, kernel: int, stride: int) -> int:
    return lib().sd_window_count(N, kernel, stride)


def sd_window_max(scores: torch.Tensor, kernel: int, stride: int, wscores: Optional[torch.Tensor] = None,
                  key_hist: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Max-pooled scores of overlapping windows (kernel, stride) of each row of scores [..., N];
    key_hist (zero-filled) receives the histogram sd_topk takes for the window scores."""
    _dev(scores, "scores")
    N = scores.shape[-1]
    rows = scores.numel() // N if N > 0 else math.prod(scores.shape[:-1])
    NW = sd_window_count(N, kernel, stride)
    if wscores is None:
        wscores = torch.empty(scores.shape[:-1] + (NW,), dtype=torch.float32, device=scores.device)
    _check(lib().sd_window_max(_ptr(scores), rows, N, kernel, stride, _ptr(wscores), _ptr(key_hist),
                               _stream(stream)), "sd_window_max")
    return wscores


def sd_window_union(widx: torch.Tensor, N: int, kernel: int, stride: int, segs: Optional[torch.Tensor] = None,
                    max_segs: Optional[int] = None, err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Segments of `stride` tokens covered by the selected windows widx [..., k], ascending,
    padded with -1 to max_segs (default k * kernel/stride)."""
    _dev(widx, "widx")
    k = widx.shape[-1]
    rows = widx.numel() // k if k > 0 else math.prod(widx.shape[:-1])
    if max_segs is None:
        max_segs = k * (kernel // stride)
    if segs is None:
        segs = torch.empty(widx.shape[:-1] + (max_segs,), dtype=torch.int32, device=widx.device)
    _check(lib().sd_window_union(_ptr(widx), rows, k, N, kernel, stride, _ptr(segs), max_segs, _ptr(err_word),
                                 _stream(stream)), "sd_window_union")
    return segs


def select_attend(scores, k, q, k_cache, v_cache, key_hist=None, stream=None, **kw):
    """Convenience wrapper: top-k selection fused with the attention over it; returns
    (idx, out, lse, logits)."""
    idx = torch.empty(scores.shape[:-1] + (k,), dtype=torch.int32, device=scores.device)
    a, out, lse, logits = make_attend_args(q, k_cache, v_cache, None, n_idx=k, **kw)
    sd_select_attend(scores, a, idx, key_hist, stream)
    return idx, out, lse, logits


def gather_attend(q, k_cache, v_cache, idx=None, workspace=None, stream=None, **kw):
    """Convenience wrapper: builds the args, sizes a workspace if none is given, runs the
    call and returns (out, lse, logits)."""
    a, out, lse, logits = make_attend_args(q, k_cache, v_cache, idx, **kw)
    need = sd_gather_attend_workspace_bytes(a)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    sd_gather_attend(a, workspace, stream)
    return out, lse, logits


def sd_score_accumulate(logits: torch.Tensor, lse: torch.Tensor, idx: Optional[torch.Tensor],
                        s: torch.Tensor, Hkv: int, block: int, weight: float,
                        err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """s [B,T] fp64 += weight * sum over query rows of the softmax weight of each selected row."""
    _dev(logits, "logits")
    _dev(lse, "lse")
    _dev(s, "s")
    if s.dtype != torch.float64:
        raise TypeError("s must be float64")
    B, V, Hq, n_rows = logits.shape
    T = s.shape[1]
    n_idx = idx.shape[-1] if idx is not None else n_rows // block
    _check(lib().sd_score_accumulate(_ptr(logits), _ptr(lse), _ptr(idx), B, V, Hq, Hkv, n_idx, block,
                                     T, float(weight), _ptr(s), _ptr(err_word), _stream(stream)),
           "sd_score_accumulate")
    return s


def sd_tier_classify(s: torch.Tensor, cum_frac: Sequence[float] = (0.2, 0.6, 0.9), n_sink: int = 0,
                     n_recent: int = 0, tier: Optional[torch.Tensor] = None,
                     counts: Optional[torch.Tensor] = None, stream=None):
    """(tier uint8 [B,T], counts int32 [B,4]) from the importance score s [B,T] fp64."""
    _dev(s, "s")
    B, T = s.shape
    if tier is None:
        tier = torch.empty((B, T), dtype=torch.uint8, device=s.device)
    if counts is None:
        counts = torch.empty((B, 4), dtype=torch.int32, device=s.device)
    fr = (ctypes.c_double * 3)(*[float(f) for f in cum_frac])
    ws_bytes = lib().sd_tier_classify_workspace_bytes(B, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=s.device) if ws_bytes else None
    _check(lib().sd_tier_classify(_ptr(s), B, T, fr, n_sink, n_recent, _ptr(tier), _ptr(counts),
                                  _ptr(ws), ws_bytes, _stream(stream)), "sd_tier_classify")
    return tier, counts


def sd_quantize_rows_int8(x: torch.Tensor, tier: torch.Tensor, codes: Optional[torch.Tensor] = None,
                          scales: Optional[torch.Tensor] = None, stream=None):
    """int8 codes [B,Hkv,T,d] and fp32 scales [B,Hkv,T] of the rows whose tier is 2."""
    _dev(x, "x")
    _dev(tier, "tier")
    B, Hkv, T, d = x.shape
    if codes is None:
        codes = torch.zeros((B, Hkv, T, d), dtype=torch.int8, device=x.device)
    if scales is None:
        scales = torch.zeros((B, Hkv, T), dtype=torch.float32, device=x.device)
    _check(lib().sd_quantize_rows_int8(_ptr(x), _dtype_code(x), _ptr(tier), B, Hkv, T, d, _ptr(codes),
                                       _ptr(scales), _stream(stream)), "sd_quantize_rows_int8")
    return codes, scales


def make_decode_step_args(q_idx, keys, q, k_cache, v_cache, k, *, block=1, scale=None, scores=None, idx=None,
                          out=None, lse=None, err_word=None, lag=0, wait_limit_ns=0) -> tuple:
    """Fill an sd_decode_step_args from tensors: q_idx [B,Hkv,V,dI] and keys [B,Hkv,T/block,dI]
    (bf16 or fp16 alike), q [B,V,Hq,d], k_cache/v_cache [B,Hkv,T,d] bf16; returns (args, scores,
    idx, out, lse) with the outputs allocated where not given (the workspace is set separately)."""
    for name, t in (("q_idx", q_idx), ("keys", keys), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, name)
    B, Hkv, V, dI = q_idx.shape
    N = keys.shape[2]
    _, Vq, Hq, d = q.shape
    T = k_cache.shape[2]
    if Vq != V or tuple(keys.shape) != (B, Hkv, N, dI) or k_cache.shape[:2] != (B, Hkv):
        raise ValueError("inconsistent shapes for sd_decode_step")
    dev = q.device
    if scores is None:
        scores = torch.empty((B, Hkv, N), dtype=torch.float32, device=dev)
    if idx is None:
        idx = torch.empty((B, Hkv, k), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty((B, V, Hq, d), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, V, Hq), dtype=torch.float32, device=dev)
    a = sd_decode_step_args()
    a.q_idx, a.keys, a.key_dtype = q_idx.data_ptr(), keys.data_ptr(), _dtype_code(keys)
    a.q, a.k_cache, a.v_cache = q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr()
    a.B, a.V, a.Hq, a.Hkv, a.d, a.d_idx, a.T, a.block, a.n_idx = B, V, Hq, Hkv, d, dI, T, block, k
    a.scale = 1.0 / math.sqrt(d) if scale is None else scale
    a.scores, a.idx, a.out, a.lse = scores.data_ptr(), idx.data_ptr(), out.data_ptr(), lse.data_ptr()
    a.err_word = err_word.data_ptr() if err_word is not None else None
    a.lag, a.wait_limit_ns = lag, wait_limit_ns
    return a, scores, idx, out, lse


def sd_decode_step_workspace_bytes(args: sd_decode_step_args) -> int:
    return lib().sd_decode_step_workspace_bytes(ctypes.byref(args))


def decode_step_workspace(args: sd_decode_step_args, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for sd_decode_step calls shaped like `args`, set into args."""
    n = max(256, sd_decode_step_workspace_bytes(args))
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    args.workspace, args.workspace_bytes = ws.data_ptr(), n
    return ws


def sd_decode_step(args: sd_decode_step_args, stream=None) -> None:
    """Runs one sd_decode_step call described by `args` (see make_decode_step_args; the
    workspace must be set, e.g. by decode_step_workspace)."""
    _check(lib().sd_decode_step(ctypes.byref(args), _stream(stream)), "sd_decode_step")


def decode_step(q_idx, keys, q, k_cache, v_cache, k, workspace=None, stream=None, **kw):
    """Convenience wrapper: one fused decode step; returns (scores, idx, out, lse)."""
    a, scores, idx, out, lse = make_decode_step_args(q_idx, keys, q, k_cache, v_cache, k, **kw)
    need = sd_decode_step_workspace_bytes(a)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=q.device)
    a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    sd_decode_step(a, stream)
    return scores, idx, out, lse


class PreparedCall:
    """One C-ABI call with its arguments marshalled once: calling the object invokes the
    library function directly, with no per-call shape checks, pointer lookups or Python
    object creation (a step loop then costs one ctypes call per kernel).  The tensors whose
    pointers it holds must stay alive and in place."""

    def __init__(self, name: str, *args):
        self.name = name
        self.fn = getattr(lib(), name)
        self.args = args

    def __call__(self) -> None:
        st = self.fn(*self.args)
        if st != SD_OK:
            _check(st, self.name)


def prepare_index_score(q_idx, k_idx, scores, err_word=None, key_hist=None, stream=None) -> PreparedCall:
    B, Hkv, V, dI = q_idx.shape
    return PreparedCall("sd_index_score", _ptr(q_idx), _dtype_code(q_idx), _ptr(k_idx), _dtype_code(k_idx), B, Hkv,
                        V, k_idx.shape[2], dI, _ptr(scores), _ptr(key_hist), _ptr(err_word), _stream(stream))


def prepare_topk(scores, k, idx, key_hist=None, stream=None) -> PreparedCall:
    N = scores.shape[-1]
    rows = scores.numel() // N
    ws_bytes = lib().sd_topk_workspace_bytes(rows, N, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=scores.device) if ws_bytes else None
    call = PreparedCall("sd_topk", _ptr(scores), rows, N, k, _ptr(idx), _ptr(key_hist), _ptr(ws), ws_bytes,
                        _stream(stream))
    call.keep = ws   # the workspace lives as long as the call
    return call


def prepare_select_attend(scores, args: sd_attend_args, idx, key_hist=None, stream=None) -> PreparedCall:
    return PreparedCall("sd_select_attend", _ptr(scores), scores.shape[-1], _ptr(key_hist), _ptr(idx),
                        ctypes.byref(args), _stream(stream))


def prepare_gather_attend(args: sd_attend_args, workspace=None, stream=None) -> PreparedCall:
    if workspace is not None:
        args.workspace, args.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    return PreparedCall("sd_gather_attend", ctypes.byref(args), _stream(stream))


def prepare_stage_host_rows(args: sd_attend_args, counter, stream=None) -> PreparedCall:
    return PreparedCall("sd_stage_host_rows", ctypes.byref(args), _ptr(counter), _stream(stream))


def prepare_decode_step(args: sd_decode_step_args, stream=None) -> PreparedCall:
    return PreparedCall("sd_decode_step", ctypes.byref(args), _stream(stream))
