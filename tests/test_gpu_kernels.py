"""Per-call parity of the CUDA library against the CPU oracle on seeded inputs: index
sets, scores, tiers and int8 codes bit-exact; attention within 2e-3 max-abs and 1e-3
relative L2 of the fp64 oracle.  Sizes span several tiles with ragged tails, plus the
empty and degenerate cases.  All calls go through the C ABI (via the ctypes binding)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attend_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_decode_gqa_gb300 import build
    build.build()


def sd():
    from top_sparse_decode_gqa_gb300 import binding
    return binding


def rint(g, shape, dtype):
    x = torch.randint(-8, 9, shape, generator=g).float()
    return x.to(dtype)


def err_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# --------------------------------------------------------------------------- indexer


@pytest.mark.parametrize("B,Hkv,V,N,dI,qdt,kdt", [
    (2, 3, 1, 1000, 128, torch.bfloat16, torch.bfloat16),
    (1, 2, 1, 4099, 64, torch.bfloat16, torch.bfloat16),
    (2, 2, 3, 777, 128, torch.bfloat16, torch.bfloat16),
    (1, 4, 8, 2500, 128, torch.bfloat16, torch.bfloat16),
    (1, 2, 1, 513, 64, torch.float32, torch.float32),
    (1, 1, 2, 300, 128, torch.bfloat16, torch.float32),
    (3, 1, 5, 65, 64, torch.float32, torch.bfloat16),
    (1, 1, 1, 1, 128, torch.bfloat16, torch.bfloat16),
    (2, 8, 1, 20000, 128, torch.bfloat16, torch.bfloat16),
])
def test_index_score_bit_exact(B, Hkv, V, N, dI, qdt, kdt):
    g = torch.Generator().manual_seed(B * 1000 + N + V)
    q, k = rint(g, (B, Hkv, V, dI), qdt), rint(g, (B, Hkv, N, dI), kdt)
    e = err_word()
    s = sd().sd_index_score(q.cuda(), k.cuda(), err_word=e)
    ref = oracle.index_score(q, k, B, Hkv, V, N, dI)
    assert int(e.item()) == 0
    np.testing.assert_array_equal(s.cpu().numpy().astype(np.float64), ref)


def test_index_score_empty():
    q = torch.zeros(2, 2, 1, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(2, 2, 0, 128, dtype=torch.bfloat16, device="cuda")
    assert sd().sd_index_score(q, k).shape == (2, 2, 0)


@pytest.mark.parametrize("T,dI,block,dt", [(1024, 128, 64, torch.bfloat16), (256, 64, 16, torch.float32),
                                           (4096, 128, 128, torch.bfloat16)])
def test_block_pool_bit_exact(T, dI, block, dt):
    g = torch.Generator().manual_seed(T + block)
    k = rint(g, (2, 3, T, dI), dt)
    p = sd().sd_block_pool(k.cuda(), block)
    ref = oracle.block_pool(k, 2, 3, T, dI, block)
    np.testing.assert_array_equal(p.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("T,dI,block,V", [(2048 * 64, 128, 64, 1), (64 * 300 + 0, 64, 64, 4), (16 * 777, 128, 16, 8),
                                          (64 * 5, 128, 64, 2)])
def test_fp16_pooled_keys_on_the_tensor_cores(T, dI, block, V):
    # fp16 pooled keys of integer keys are exact (multiples of 1/block below 8); with an fp16
    # query of the same integers the block scores run on the tensor cores, bit-exact
    g = torch.Generator().manual_seed(T + V)
    B, Hkv = 2, 2
    k = rint(g, (B, Hkv, T, dI), torch.bfloat16)
    q = rint(g, (B, Hkv, V, dI), torch.float16)
    p = sd().sd_block_pool(k.cuda(), block, dtype=torch.float16)
    ref = oracle.block_pool(k, B, Hkv, T, dI, block)
    np.testing.assert_array_equal(p.cpu().numpy().astype(np.float64), ref)
    hist = sd().key_hist_buffer(B * Hkv)
    s = sd().sd_index_score(q.cuda(), p, key_hist=hist)
    rs = oracle.index_score(q, ref.astype(np.float32), B, Hkv, V, T // block, dI)
    np.testing.assert_array_equal(s.cpu().numpy().astype(np.float64), rs)
    kk = min(64, T // block)
    idx = sd().sd_topk(s, kk, key_hist=hist)
    np.testing.assert_array_equal(idx.cpu().numpy(), oracle.topk(rs, kk))
    # mixed 16-bit types are rejected
    with pytest.raises(sd().SdError):
        sd().sd_index_score(q.to(torch.bfloat16).cuda(), p)


# --------------------------------------------------------------------------- top-k


@pytest.mark.parametrize("N", [1, 7, 100, 1000, 2048, 4096, 5000, 12000, 32768, 65536, 131072])
def test_topk_bit_exact_with_ties(N):
    # N <= 4096: the short-row kernel; 4096 < N < 16384: one CTA per row with three digit
    # passes; longer rows: thread-block clusters
    rng = np.random.default_rng(N)
    rows = 5
    # heavy ties: integer scores in a narrow range, one row all equal
    s = rng.integers(-40, 40, size=(rows, N)).astype(np.float32)
    s[2] = 3.0
    st = torch.from_numpy(s).cuda()
    for k in sorted({0, 1, N // 3, max(N - 1, 0), N}):
        idx = sd().sd_topk(st, k)
        ref = oracle.topk(s.astype(np.float64), k)
        np.testing.assert_array_equal(idx.cpu().numpy(), ref, err_msg=f"N={N} k={k}")


def test_topk_float_scores_and_signed_zero():
    rng = np.random.default_rng(3)
    s = (rng.standard_normal((4, 3000)) * 100).astype(np.float32)
    s[1, ::2] = 0.0
    s[1, 1::2] = -0.0       # -0.0 and +0.0 tie: the lower index must win
    s[3, :] = -np.abs(s[3, :])
    st = torch.from_numpy(s).cuda()
    for k in (1, 17, 1499, 1500, 1501, 2999):
        idx = sd().sd_topk(st, k)
        np.testing.assert_array_equal(idx.cpu().numpy(), oracle.topk(s.astype(np.float64), k))


@pytest.mark.parametrize("B,Hkv,V,N,k,flat", [
    (2, 4, 1, 32768, 1024, False),
    (1, 2, 8, 131072, 2048, False),
    (1, 2, 1, 20000, 100, True),      # every score equal: one bin beyond the candidate capacity
    (2, 2, 1, 5000, 4999, False),
    (1, 1, 1, 3000, 0, False),
    (1, 1, 1, 3000, 3000, False),
    (3, 1, 3, 777, 13, False),
    (2, 3, 1, 2048, 64, False),       # block-selection shape (the short-row kernel)
    (1, 2, 1, 12000, 50, False),      # N between the cached and uncached sizes
    (1, 2, 1, 9000, 100, True),       # every score equal, one 1024-thread CTA per row: its full-pass fallback
    (8, 32, 1, 4096 + 5, 300, False),  # more rows than SMs: the 512-thread variant
    (10, 16, 1, 3000, 100, True),     # every score equal, short rows: the short-row kernel
    (10, 16, 1, 5000, 100, True),     # ... longer rows: the 512-thread variant's full-pass fallback
    (4, 40, 2, 2048, 2047, False),
])
def test_index_topk_with_key_histogram(B, Hkv, V, N, k, flat):
    g = torch.Generator().manual_seed(N + k)
    q = rint(g, (B, Hkv, V, 128), torch.bfloat16)
    if flat:
        q.zero_()
    kk = rint(g, (B, Hkv, N, 128), torch.bfloat16)
    hist = sd().key_hist_buffer(B * Hkv)
    s = sd().sd_index_score(q.cuda(), kk.cuda(), key_hist=hist)
    assert torch.equal(hist.sum(1).cpu(), torch.full((B * Hkv,), N, dtype=torch.int64))
    idx = sd().sd_topk(s, k, key_hist=hist)
    torch.cuda.synchronize()
    assert int(hist.abs().sum().item()) == 0, "the histogram must be left zeroed"
    ref = oracle.topk(oracle.index_score(q, kk, B, Hkv, V, N, 128), k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
    # a second step with the same buffers gives the same result
    s = sd().sd_index_score(q.cuda(), kk.cuda(), key_hist=hist)
    idx2 = sd().sd_topk(s, k, key_hist=hist)
    assert torch.equal(idx2, idx)


# --------------------------------------------------------------------------- gather + attend


def _attend_case(g, B, V, Hq, Hkv, d, T, n_idx, block, dt):
    q = torch.randn(B, V, Hq, d, generator=g).to(dt)
    K = torch.randn(B, Hkv, T, d, generator=g).to(dt)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(dt)
    nb = T // block
    idx = None
    if n_idx is not None:
        idx = torch.stack([torch.stack([torch.sort(torch.randperm(nb, generator=g)[:n_idx]).values
                                        for _ in range(Hkv)]) for _ in range(B)]).int()
    return q, K, Vv, idx


@pytest.mark.parametrize("B,V,Hq,Hkv,d,T,n_idx,block,dt,splits", [
    (2, 1, 32, 8, 128, 3000, 300, 1, torch.bfloat16, 0),       # C2-like group of 4
    (1, 2, 16, 2, 64, 2048, 500, 1, torch.bfloat16, 0),         # R = 16
    (1, 8, 8, 2, 128, 5000, 777, 1, torch.bfloat16, 0),         # R = 32 (verify batch)
    (1, 1, 4, 1, 64, 1024, 64, 1, torch.float32, 0),            # C1 shape
    (2, 3, 4, 2, 128, 900, 111, 1, torch.float32, 0),           # R = 6, fp32, d = 128
    (1, 1, 8, 2, 128, 4096, 7, 64, torch.bfloat16, 0),          # block mode
    (1, 1, 28, 4, 128, 1000, None, 1, torch.bfloat16, 0),       # dense, R = 7
    (1, 1, 8, 8, 128, 700, 300, 1, torch.bfloat16, 0),          # MHA (G = 1)
    (2, 1, 8, 2, 128, 3000, 1000, 1, torch.bfloat16, 1),        # forced one split
    (2, 1, 8, 2, 128, 3000, 1000, 1, torch.bfloat16, 3),        # forced three splits
    (1, 1, 8, 2, 128, 3000, 1000, 1, torch.bfloat16, 500),      # more splits than chunks
    (1, 1, 8, 2, 128, 100, 1, 1, torch.bfloat16, 0),            # one selected row
])
def test_gather_attend_matches_oracle(B, V, Hq, Hkv, d, T, n_idx, block, dt, splits):
    g = torch.Generator().manual_seed(T + Hq + V * 7 + (n_idx or 0))
    q, K, Vv, idx = _attend_case(g, B, V, Hq, Hkv, d, T, n_idx, block, dt)
    scale = 1.0 / math.sqrt(d)
    e = err_word()
    out, lse, logits = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(),
                                          idx.cuda() if idx is not None else None, block=block,
                                          T=T, scale=scale, want_logits=True, err_word=e,
                                          splits=splits)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    n_sel = n_idx if idx is not None else T // block
    ro, rl, rz = oracle.gather_attend(q, K, Vv, idx.numpy() if idx is not None else None, B, V, Hq,
                                      Hkv, d, T, n_sel, block, scale, True)
    assert_attend_close(out, ro, "out")
    assert_attend_close(lse, rl, "lse")
    np.testing.assert_allclose(logits.cpu().numpy(), rz, atol=1e-4, rtol=1e-5)
    # the softmax weights implied by logits and lse sum to one per query row
    w = torch.exp(logits.double() - lse.double()[..., None]).sum(-1)
    assert torch.allclose(w, torch.ones_like(w), atol=1e-5)


def test_gather_attend_empty_selection():
    g = torch.Generator().manual_seed(5)
    q, K, Vv, _ = _attend_case(g, 1, 1, 8, 2, 128, 64, None, 1, torch.bfloat16)
    idx = torch.zeros(1, 2, 0, dtype=torch.int32, device="cuda")
    out, lse, _ = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), idx, T=64)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def _residency_inputs(seed, B=2, V=4, Hq=8, Hkv=2, d=128, T=4000, k=300):
    g = torch.Generator().manual_seed(seed)
    q, K, Vv, idx = _attend_case(g, B, V, Hq, Hkv, d, T, k, 1, torch.bfloat16)
    return q, K, Vv, idx


def _run_tiered(q, K, Vv, idx, P, seed):
    from top_sparse_decode_gqa_gb300.workloads import residency_map
    B, Hkv, T, d = K.shape
    res, slot_map = residency_map(B, T, P, seed)
    gi = res[:, None, :, None].expand(B, Hkv, P, d)
    k_pool = torch.gather(K, 2, gi).contiguous().cuda()
    v_pool = torch.gather(Vv, 2, gi).contiguous().cuda()
    if P == 0:  # keep a valid (unused) device pointer
        k_pool = torch.zeros(B, Hkv, 1, d, dtype=K.dtype, device="cuda")
        v_pool = torch.zeros_like(k_pool)
    e = err_word()
    out, lse, _ = sd().gather_attend(q.cuda(), k_pool, v_pool, idx.cuda(), T=T,
                                     k_host=K.pin_memory(), v_host=Vv.pin_memory(),
                                     slot_map=slot_map.cuda(), err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    return out.cpu(), lse.cpu()


def test_residency_does_not_change_the_result_bit_for_bit():
    # Zero-approximation-error offload: the output must be the same bits whether each
    # selected row came from the HBM pool or from pinned host memory.
    q, K, Vv, idx = _residency_inputs(41)
    T = K.shape[2]
    runs = [_run_tiered(q, K, Vv, idx, P, seed=7) for P in (0, T // 10, T)]
    out_dev, lse_dev, _ = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), idx.cuda(), T=T)
    for out, lse in runs[1:] + [(out_dev.cpu(), lse_dev.cpu())]:
        assert torch.equal(out, runs[0][0]) and torch.equal(lse, runs[0][1])
    B, V, Hq, d = q.shape
    ro, rl, _ = oracle.gather_attend(q, K, Vv, idx.numpy(), B, V, Hq, K.shape[1], d, T,
                                     idx.shape[-1], 1, 1.0 / math.sqrt(d))
    assert_attend_close(runs[0][0], ro)


def test_bad_index_and_slot_are_skipped_and_reported():
    q, K, Vv, idx = _residency_inputs(43, B=1, T=500, k=20)
    T = K.shape[2]
    bad = idx.clone()
    bad[0, 0, 3] = T + 5
    e = err_word()
    sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), bad.cuda(), T=T, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) & sd().SD_DEVERR_INDEX
    from top_sparse_decode_gqa_gb300.workloads import residency_map
    _, slot_map = residency_map(1, T, 10, 3)
    slot_map[0, idx[0, 1, 0]] = 12345          # beyond the pool
    e.zero_()
    k_pool = torch.zeros(1, 2, 10, 128, dtype=torch.bfloat16, device="cuda")
    sd().gather_attend(q.cuda(), k_pool, k_pool.clone(), idx.cuda(), T=T, k_host=K.pin_memory(),
                       v_host=Vv.pin_memory(), slot_map=slot_map.cuda(), err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) & sd().SD_DEVERR_SLOT


def test_host_pointer_must_be_pinned():
    q, K, Vv, idx = _residency_inputs(44, B=1, T=200, k=10)
    from top_sparse_decode_gqa_gb300.workloads import residency_map
    _, slot_map = residency_map(1, 200, 10, 3)
    a, *_ = sd().make_attend_args(q.cuda(), K.cuda(), Vv.cuda(), idx.cuda(), T=200,
                                  slot_map=slot_map.cuda())
    a.k_host = K.data_ptr()   # pageable host memory
    a.v_host = Vv.data_ptr()
    with pytest.raises(sd().SdError):
        sd().sd_gather_attend(a, torch.zeros(1 << 20, dtype=torch.uint8, device="cuda"))


# --------------------------------------------------------------------------- importance


@pytest.mark.parametrize("dense,block,V,Hq,T", [(True, 1, 2, 8, 1024), (False, 1, 2, 8, 1024), (False, 16, 2, 8, 1024),
                                                 (True, 1, 1, 28, 2048), (True, 1, 3, 12, 1022)])
def test_score_accumulate_matches_oracle(dense, block, V, Hq, T):
    g = torch.Generator().manual_seed(51 + block + T)
    B, Hkv, d = 2, 2 if Hq % 2 == 0 else 1, 64
    n_idx = T // block if dense else (40 if block > 1 else 300)
    q, K, Vv, idx = _attend_case(g, B, V, Hq, Hkv, d, T, None if dense else n_idx, block, torch.float32)
    _, lse, logits = oracle.gather_attend(q, K, Vv, None if dense else idx.numpy(), B, V, Hq, Hkv, d, T,
                                          n_idx, block, 0.125, True)
    # both sides get the same fp32 logits / lse
    lg32, ls32 = logits.astype(np.float32), lse.astype(np.float32)
    s0 = torch.rand(B, T, generator=g, dtype=torch.float64)
    w = 1.0 / (3 * Hq)
    s_gpu = sd().sd_score_accumulate(torch.from_numpy(lg32).cuda(), torch.from_numpy(ls32).cuda(),
                                     None if dense else idx.cuda(), s0.clone().cuda(), Hkv, block, w)
    s_ref = s0.numpy().copy()
    oracle.score_accumulate(lg32.astype(np.float64), ls32.astype(np.float64),
                            None if dense else idx.numpy(), s_ref, B, V, Hq, Hkv, n_idx, block, T, w)
    delta_gpu = s_gpu.cpu().numpy() - s0.numpy()
    delta_ref = s_ref - s0.numpy()
    np.testing.assert_allclose(delta_gpu, delta_ref, rtol=2e-6, atol=1e-12)
    # each layer's term adds weight * (number of query rows) per sequence
    np.testing.assert_allclose(delta_gpu.sum(1), w * V * Hq, rtol=1e-5)


@pytest.mark.parametrize("T,ties,n_sink,n_recent,fr", [
    (10, False, 0, 0, (0.2, 0.6, 0.9)),
    (1000, True, 0, 0, (0.2, 0.6, 0.9)),
    (65536, False, 0, 0, (0.2, 0.6, 0.9)),
    (65536, True, 4, 64, (0.2, 0.6, 0.9)),
    (5000, False, 100, 100, (0.01, 0.5, 0.9)),    # protection beyond the T0 budget
    (777, False, 0, 0, (0.0, 0.0, 0.0)),
    (777, False, 0, 0, (1.0, 1.0, 1.0)),
    (777, True, 3, 0, (0.0, 0.5, 1.0)),
])
def test_tier_classify_bit_exact(T, ties, n_sink, n_recent, fr):
    from top_sparse_decode_gqa_gb300.workloads import importance_scores
    s = importance_scores(2, T, seed=T + n_sink, ties=ties)
    tier, counts = sd().sd_tier_classify(s.cuda(), fr, n_sink, n_recent)
    rt, rc = oracle.tier_classify(s.numpy(), fr, n_sink, n_recent)
    np.testing.assert_array_equal(tier.cpu().numpy(), rt)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)


@pytest.mark.parametrize("d,dt", [(128, torch.bfloat16), (64, torch.bfloat16), (128, torch.float32),
                                  (64, torch.float32)])
def test_quantize_rows_int8_bit_exact(d, dt):
    g = torch.Generator().manual_seed(d + (dt == torch.float32))
    B, Hkv, T = 2, 3, 1000
    x = (torch.randn(B, Hkv, T, d, generator=g) * 3).to(dt)
    x[0, 1, 5] = 0          # all-zero row
    x[1, 2, 7, 3] = 1e-30   # tiny row
    tier = torch.randint(0, 4, (B, T), generator=g).to(torch.uint8)
    tier[0, 5] = tier[1, 7] = 2
    codes0 = torch.full((B, Hkv, T, d), 99, dtype=torch.int8)
    scales0 = torch.full((B, Hkv, T), -1.0)
    c, s = sd().sd_quantize_rows_int8(x.cuda(), tier.cuda(), codes0.clone().cuda(), scales0.clone().cuda())
    rc, rs = oracle.quantize_rows_int8(x, tier.numpy(), B, Hkv, T, d, codes0.numpy().copy(),
                                       scales0.numpy().copy())
    np.testing.assert_array_equal(c.cpu().numpy(), rc)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
