"""The C-ABI library builds, loads and exports every symbol include/sd.h declares; host-side
argument validation rejects bad calls before anything is launched.  No GPU needed: no
call here reaches a kernel."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from top_sparse_decode_gqa_gb300 import build, binding
    build.build()
    return binding.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "sd.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sd_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    from top_sparse_decode_gqa_gb300 import binding
    decl = declared_functions()
    assert decl == sorted(binding.EXPORTS)
    for name in decl:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.sd_version() == 100
    assert lib.sd_status_string(0) == b"ok"
    assert lib.sd_status_string(1) == b"invalid argument"
    assert lib.sd_status_string(99) == b"unknown status"


def test_host_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    dummy = P(16)
    # k > N
    assert lib.sd_topk(dummy, 1, 10, 11, dummy, None, None, 0, None) == 1
    assert b"k (11)" in lib.sd_last_error_message()
    # unsupported indexer dim
    assert lib.sd_index_score(dummy, 1, dummy, 1, 1, 1, 1, 10, 96, dummy, None, None, None) == 2
    # V out of range
    assert lib.sd_index_score(dummy, 1, dummy, 1, 1, 1, 9, 10, 128, dummy, None, None, None) == 1
    # ragged block pooling
    assert lib.sd_block_pool(dummy, 1, 1, 1, 100, 128, 64, dummy, 0, None) == 1
    # pooled keys are F32 or F16 only; F16 indexer operands go together
    assert lib.sd_block_pool(dummy, 1, 1, 1, 128, 128, 64, dummy, 1, None) == 1
    assert lib.sd_index_score(dummy, 2, dummy, 1, 1, 1, 1, 10, 128, dummy, None, None, None) == 1
    # non-monotone tier fractions
    fr = (ctypes.c_double * 3)(0.5, 0.2, 0.9)
    assert lib.sd_tier_classify(dummy, 1, 10, fr, 0, 0, dummy, dummy, None, 0, None) == 1
    # empty work is a successful no-op
    assert lib.sd_topk(None, 0, 10, 3, None, None, None, 0, None) == 0
    assert lib.sd_index_score(None, 1, None, 1, 0, 8, 1, 100, 128, None, None, None, None) == 0


def test_attend_validation_and_workspace_query(lib):
    from top_sparse_decode_gqa_gb300.binding import sd_attend_args
    a = sd_attend_args()
    a.q = a.k_cache = a.v_cache = a.out = a.lse = 16
    a.dtype, a.B, a.V, a.Hq, a.Hkv, a.d, a.T = 1, 2, 1, 32, 8, 128, 4096
    a.pool_rows, a.n_idx, a.block, a.scale = 4096, 4096, 1, 0.1
    # dense without idx is fine; workspace is a pure host computation
    assert lib.sd_gather_attend_workspace_bytes(ctypes.byref(a)) >= 0
    a.d = 96
    assert lib.sd_gather_attend(ctypes.byref(a), None) == 2
    a.d, a.V = 128, 9  # G*V = 36 > 32
    assert lib.sd_gather_attend(ctypes.byref(a), None) == 2
    a.V, a.n_idx = 1, 100  # dense mode with n_idx*block != T
    assert lib.sd_gather_attend(ctypes.byref(a), None) == 1


def test_select_attend_validation(lib):
    from top_sparse_decode_gqa_gb300.binding import sd_attend_args
    P = ctypes.c_void_p
    dummy = P(16)
    a = sd_attend_args()
    a.q = a.k_cache = a.v_cache = a.out = a.lse = 16
    a.dtype, a.B, a.V, a.Hq, a.Hkv, a.d, a.T = 1, 2, 1, 32, 8, 128, 4096
    a.pool_rows, a.n_idx, a.block, a.scale = 4096, 64, 1, 0.1
    # one score per token: N must equal T / block
    assert lib.sd_select_attend(dummy, 4000, None, dummy, ctypes.byref(a), None) == 1
    assert b"must equal T" in lib.sd_last_error_message()
    # k beyond N
    a.n_idx = 5000
    assert lib.sd_select_attend(dummy, 4096, None, dummy, ctypes.byref(a), None) == 1
    a.n_idx = 64
    # the cluster holds at most 8 CTAs
    a.splits = 9
    assert lib.sd_select_attend(dummy, 4096, None, dummy, ctypes.byref(a), None) == 1
    a.splits = 0
    # fp32 inputs and G*V > 32 go through the separate calls
    a.dtype = 0
    assert lib.sd_select_attend(dummy, 4096, None, dummy, ctypes.byref(a), None) == 2
    a.dtype, a.V = 1, 9
    assert lib.sd_select_attend(dummy, 4096, None, dummy, ctypes.byref(a), None) == 2
    # block selection: N blocks of `block` tokens
    a.V, a.block, a.n_idx = 1, 64, 8
    a.B = 0  # nothing to do: accepted without touching the pointers
    assert lib.sd_select_attend(None, 64, None, None, ctypes.byref(a), None) == 0


def test_stage_host_rows_validation(lib):
    from top_sparse_decode_gqa_gb300.binding import sd_attend_args
    dummy = ctypes.c_void_p(16)
    a = sd_attend_args()
    a.q = a.k_cache = a.v_cache = a.out = a.lse = a.idx = 16
    a.dtype, a.B, a.V, a.Hq, a.Hkv, a.d, a.T = 1, 2, 1, 32, 8, 128, 4096
    a.pool_rows, a.n_idx, a.block, a.scale = 409, 64, 1, 0.1
    # the staged copy needs a slot map, host K/V, both stage buffers and a counter
    assert lib.sd_stage_host_rows(ctypes.byref(a), dummy, None) == 1
    assert b"slot_map" in lib.sd_last_error_message()
    a.slot_map = 16
    assert lib.sd_stage_host_rows(ctypes.byref(a), dummy, None) == 1
    assert b"k_host" in lib.sd_last_error_message()
    a.k_host = a.v_host = 16
    assert lib.sd_stage_host_rows(ctypes.byref(a), dummy, None) == 1
    assert b"k_stage" in lib.sd_last_error_message()
    a.k_stage = 16
    assert lib.sd_stage_host_rows(ctypes.byref(a), dummy, None) == 1
    a.v_stage = 24  # misaligned
    assert lib.sd_stage_host_rows(ctypes.byref(a), dummy, None) == 1
    assert b"aligned" in lib.sd_last_error_message()
    a.v_stage = 32
    assert lib.sd_stage_host_rows(ctypes.byref(a), None, None) == 1
    assert b"counter" in lib.sd_last_error_message()
    # the shared attention checks apply, named for this call
    a.d = 96
    assert lib.sd_stage_host_rows(ctypes.byref(a), dummy, None) == 2
    assert lib.sd_last_error_message().startswith(b"sd_stage_host_rows:")
    # sd_gather_attend: a stage needs both buffers
    a.d, a.v_stage = 128, None
    a.workspace, a.workspace_bytes = 16, 1 << 30
    assert lib.sd_gather_attend(ctypes.byref(a), None) == 1
    assert b"go together" in lib.sd_last_error_message()


def test_ring_validation(lib):
    from top_sparse_decode_gqa_gb300.binding import sd_attend_args
    dummy = ctypes.c_void_p(16)
    # sd_ring_append: n must be in [1, W]; d 64 or 128
    assert lib.sd_ring_append(dummy, dummy, 1, 2, 8, 9, 128, dummy, dummy, dummy, dummy, 8, None) == 1
    assert lib.sd_ring_append(dummy, dummy, 1, 2, 8, 0, 128, dummy, dummy, dummy, dummy, 8, None) == 1
    assert lib.sd_ring_append(dummy, dummy, 1, 2, 8, 4, 96, dummy, dummy, dummy, dummy, 8, None) == 2
    assert lib.sd_ring_append(None, None, 1, 0, 8, 4, 128, None, None, None, None, 8, None) == 0
    a = sd_attend_args()
    a.q = a.k_cache = a.v_cache = a.out = a.lse = a.idx = 16
    a.dtype, a.B, a.V, a.Hq, a.Hkv, a.d, a.T = 1, 2, 8, 32, 8, 128, 4096
    a.pool_rows, a.n_idx, a.block, a.scale = 4096, 64, 1, 0.1
    # a ring needs its four arrays
    a.ring_w = 64
    assert lib.sd_gather_attend(ctypes.byref(a), None) == 1
    assert b"ring" in lib.sd_last_error_message()
    a.ring_k = a.ring_v = a.ring_pos = a.qpos = 16
    # the fused select/attend has no ring
    assert lib.sd_select_attend(dummy, 4096, None, dummy, ctypes.byref(a), None) == 2


def test_promote_validation(lib):
    from top_sparse_decode_gqa_gb300.binding import sd_attend_args
    dummy = ctypes.c_void_p(16)
    a = sd_attend_args()
    a.q = a.k_cache = a.v_cache = a.out = a.lse = 16
    a.dtype, a.B, a.V, a.Hq, a.Hkv, a.d, a.T = 1, 2, 8, 32, 8, 128, 4096
    a.pool_rows, a.n_idx, a.block, a.scale = 409, 64, 1, 0.1
    # needs a selection and a slot map
    a.idx = 16
    assert lib.sd_promote_rows(ctypes.byref(a), dummy, dummy, dummy, 1 << 20, None) == 1
    assert b"idx and slot_map" in lib.sd_last_error_message()
    a.slot_map = 16
    # needs the host cache and the caller's pool state
    assert lib.sd_promote_rows(ctypes.byref(a), dummy, dummy, dummy, 1 << 20, None) == 1
    assert b"k_host" in lib.sd_last_error_message()
    a.k_host = a.v_host = 16
    assert lib.sd_promote_rows(ctypes.byref(a), None, dummy, dummy, 1 << 20, None) == 1
    # and a workspace of the queried size
    need = lib.sd_promote_rows_workspace_bytes(ctypes.byref(a))
    assert need > 4096 * 2 // 8  # at least the bitmap of 2 x 4096 positions
    assert lib.sd_promote_rows(ctypes.byref(a), dummy, dummy, dummy, need - 16, None) == 1
    assert b"workspace" in lib.sd_last_error_message()
    a.pool_rows = 0
    assert lib.sd_promote_rows_workspace_bytes(ctypes.byref(a)) == 0


def test_promote_staged_validation(lib):
    from top_sparse_decode_gqa_gb300.binding import sd_attend_args
    dummy = ctypes.c_void_p(16)
    a = sd_attend_args()
    a.q = a.k_cache = a.v_cache = a.out = a.lse = a.idx = a.slot_map = 16
    a.dtype, a.B, a.V, a.Hq, a.Hkv, a.d, a.T = 1, 2, 8, 32, 8, 128, 4096
    a.pool_rows, a.n_idx, a.block, a.scale = 409, 64, 1, 0.1
    # the staged promotion works on (sequence, KV head) units only
    assert lib.sd_promote_staged_rows(ctypes.byref(a), dummy, dummy, dummy, 1 << 24, None) == 1
    assert b"(sequence, KV head)" in lib.sd_last_error_message()
    a.slot_per_head = 1
    # it reads the stage, not the host cache
    assert lib.sd_promote_staged_rows(ctypes.byref(a), dummy, dummy, dummy, 1 << 24, None) == 1
    assert b"k_stage" in lib.sd_last_error_message()
    a.k_stage = a.v_stage = 24  # not 16-byte aligned
    assert lib.sd_promote_staged_rows(ctypes.byref(a), dummy, dummy, dummy, 1 << 24, None) == 1
    a.k_stage = a.v_stage = 32
    # its workspace adds a [B*Hkv, T] int32 map to the host-mode layout
    need = lib.sd_promote_staged_rows_workspace_bytes(ctypes.byref(a))
    assert need >= lib.sd_promote_rows_workspace_bytes(ctypes.byref(a)) + 2 * 8 * 4096 * 4
    assert lib.sd_promote_staged_rows(ctypes.byref(a), dummy, dummy, dummy, need - 16, None) == 1
    assert b"workspace" in lib.sd_last_error_message()
    a.pool_rows = 0
    assert lib.sd_promote_staged_rows_workspace_bytes(ctypes.byref(a)) == 0


def test_index_score_heads_validation(lib):
    dummy = ctypes.c_void_p(16)
    # negative sizes, mixed f16/bf16 operands, too many query columns, unsupported d
    assert lib.sd_index_score_heads(dummy, 1, dummy, 1, -1, 8, 4, 4096, 128, dummy, None, None, None) == 1
    assert lib.sd_index_score_heads(dummy, 2, dummy, 1, 2, 8, 4, 4096, 128, dummy, None, None, None) == 1
    assert b"F16" in lib.sd_last_error_message()
    assert lib.sd_index_score_heads(dummy, 1, dummy, 1, 2, 8, 17, 4096, 128, dummy, None, None, None) == 1
    assert lib.sd_index_score_heads(dummy, 1, dummy, 1, 2, 8, 4, 4096, 96, dummy, None, None, None) == 2
    # nothing to do
    assert lib.sd_index_score_heads(None, 1, None, 1, 0, 8, 4, 4096, 128, None, None, None, None) == 0


def test_window_calls_validation(lib):
    # the window count is host arithmetic: ceil((N - kernel) / stride) + 1 windows, 0 below one
    assert lib.sd_window_count(32768, 32, 16) == 2047
    assert lib.sd_window_count(64, 32, 16) == 3
    assert lib.sd_window_count(-1, 32, 16) == 0
    dummy = ctypes.c_void_p(16)
    assert lib.sd_window_max(dummy, 4, 1024, 16, 32, dummy, None, None) == 1  # stride > kernel
    assert lib.sd_window_max(dummy, 4, 1 << 16, 2048, 16, dummy, None, None) == 1  # kernel > 1024
    assert lib.sd_window_max(None, 0, 1024, 32, 16, None, None, None) == 0
    assert lib.sd_window_union(dummy, 4, 8, 1024, 24, 16, dummy, 16, None, None) == 1  # kernel % stride
    assert lib.sd_window_union(dummy, 4, 8, 1000, 32, 16, dummy, 16, None, None) == 1  # N % stride
    assert lib.sd_window_union(dummy, 4, 8, 1024, 32, 16, dummy, 15, None, None) == 1  # max_segs < k*2
    assert b"max_segs" in lib.sd_last_error_message()
    assert lib.sd_window_union(None, 0, 8, 1024, 32, 16, None, 16, None, None) == 0


def test_importance_and_tier_validation(lib):
    dummy = ctypes.c_void_p(16)
    f64 = ctypes.c_double
    # Hq not a multiple of Hkv; dense mode needs n_idx * block == T; null outputs
    assert lib.sd_score_accumulate(dummy, dummy, None, 2, 1, 28, 3, 64, 1, 64, f64(0.1), dummy, None, None) == 1
    assert lib.sd_score_accumulate(dummy, dummy, None, 2, 1, 28, 4, 64, 1, 65, f64(0.1), dummy, None, None) == 1
    assert b"dense" in lib.sd_last_error_message()
    assert lib.sd_score_accumulate(None, dummy, dummy, 2, 1, 28, 4, 64, 1, 4096, f64(0.1), dummy, None, None) == 1
    assert lib.sd_score_accumulate(None, None, None, 0, 1, 28, 4, 64, 1, 64, f64(0.1), None, None, None) == 0
    frac = (f64 * 3)
    assert lib.sd_tier_classify_workspace_bytes(2, 65536) == 0
    assert lib.sd_tier_classify(dummy, 2, 64, frac(0.2, 0.6, 1.5), 0, 0, dummy, dummy, None, 0, None) == 1
    assert lib.sd_tier_classify(dummy, 2, 64, frac(0.6, 0.2, 0.9), 0, 0, dummy, dummy, None, 0, None) == 1
    assert b"nondecreasing" in lib.sd_last_error_message()
    assert lib.sd_tier_classify(dummy, 2, 64, None, 0, 0, dummy, dummy, None, 0, None) == 1
    assert lib.sd_tier_classify(dummy, 2, 64, frac(0.2, 0.6, 0.9), -1, 0, dummy, dummy, None, 0, None) == 1
    assert lib.sd_tier_classify(None, 0, 64, frac(0.2, 0.6, 0.9), 0, 0, None, None, None, 0, None) == 0
    # int8 rows: bad dtype, unsupported d, null outputs, nothing to do
    assert lib.sd_quantize_rows_int8(dummy, 7, dummy, 2, 4, 64, 128, dummy, dummy, None) == 1
    assert lib.sd_quantize_rows_int8(dummy, 1, dummy, 2, 4, 64, 96, dummy, dummy, None) == 2
    assert lib.sd_quantize_rows_int8(dummy, 1, dummy, 2, 4, 64, 128, None, dummy, None) == 1
    assert lib.sd_quantize_rows_int8(None, 1, None, 0, 4, 64, 128, None, None, None) == 0


def test_noalloc_validation(lib):
    from top_sparse_decode_gqa_gb300.binding import sd_attend_args
    assert lib.sd_gather_attend_noalloc(None, None) == 1
    a = sd_attend_args()
    a.q = a.k_cache = a.v_cache = a.out = a.lse = a.idx = 16
    a.dtype, a.B, a.V, a.Hq, a.Hkv, a.d, a.T = 1, 64, 8, 32, 8, 128, 1 << 16
    a.pool_rows, a.n_idx, a.block, a.scale, a.splits = 1 << 16, 4096, 1, 0.1, 64
    # 512 groups x 64 splits x 32 query rows of (d + 2) floats: far beyond the 16 MiB scratch
    assert lib.sd_gather_attend_workspace_bytes(ctypes.byref(a)) > 16 << 20
    assert lib.sd_gather_attend_noalloc(ctypes.byref(a), None) == 1
    assert b"static scratch" in lib.sd_last_error_message()
    # an invalid request reports the gather-attend's own error
    a.d = 96
    assert lib.sd_gather_attend_noalloc(ctypes.byref(a), None) in (1, 2)
