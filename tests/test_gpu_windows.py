"""Parity of the overlapping-window path with the CPU oracle: window scores (max-pooled token
scores) and the union of the selected windows' segments bit-exact, the key histogram checked
through the top-k it seeds, empty slots (-1) in gather-attend and score accumulate within the
attention tolerance, and the whole chain (indexer -> window max -> top-k -> union ->
gather-attend over 16-token segments).  All calls go through the C ABI."""
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


@pytest.mark.parametrize("rows,N,kernel,stride", [(4, 32768, 32, 16), (3, 1000, 32, 16), (2, 20, 32, 16),
                                                  (5, 4096, 64, 64), (2, 777, 2, 1), (1, 1, 32, 16),
                                                  (2, 5000, 1024, 512)])
def test_window_max_bit_exact(rows, N, kernel, stride):
    rng = np.random.default_rng(N + kernel)
    s = (rng.standard_normal((rows, N)) * 50).astype(np.float32)
    w = sd().sd_window_max(torch.from_numpy(s).cuda(), kernel, stride)
    ref = oracle.window_max(s.astype(np.float64), kernel, stride)
    np.testing.assert_array_equal(w.cpu().numpy().astype(np.float64), ref)


def test_window_histogram_seeds_the_topk():
    # the histogram the window kernel adds is the one sd_topk needs: top-k through it equals
    # the oracle's top-k of the window scores, and the histogram is left zeroed
    rng = np.random.default_rng(3)
    rows, N, k = 6, 32768, 64
    s = rng.integers(-300, 300, size=(rows, N)).astype(np.float32)  # integer scores: many ties
    hist = sd().key_hist_buffer(rows)
    w = sd().sd_window_max(torch.from_numpy(s).cuda(), 32, 16, key_hist=hist)
    assert torch.equal(hist.sum(1).cpu(), torch.full((rows,), w.shape[-1], dtype=torch.int64))
    idx = sd().sd_topk(w, k, key_hist=hist)
    torch.cuda.synchronize()
    assert int(hist.abs().sum().item()) == 0
    ref = oracle.topk(oracle.window_max(s.astype(np.float64), 32, 16), k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)


@pytest.mark.parametrize("rows,N,kernel,stride,k", [(64, 32768, 32, 16, 64), (3, 512, 32, 16, 31),
                                                    (2, 96, 48, 16, 3), (4, 4096, 16, 16, 100),
                                                    (2, 64, 32, 16, 0), (1, 1048576, 32, 16, 500)])
def test_window_union_bit_exact(rows, N, kernel, stride, k):
    rng = np.random.default_rng(N + k)
    NW = oracle.window_count(N, kernel, stride)
    widx = np.stack([np.sort(rng.permutation(NW)[:k]) for _ in range(rows)]).astype(np.int32)
    widx_t = torch.from_numpy(widx).reshape(rows, k).cuda()
    segs = sd().sd_window_union(widx_t, N, kernel, stride, max_segs=k * (kernel // stride) + 3)
    ref = oracle.window_union(widx.reshape(rows, k), N, kernel, stride, max_segs=k * (kernel // stride) + 3)
    np.testing.assert_array_equal(segs.cpu().numpy(), ref)


def test_window_union_flags_a_bad_window():
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    widx = torch.tensor([[0, 5]], dtype=torch.int32, device="cuda")  # 64 tokens: windows 0..2
    segs = sd().sd_window_union(widx, 64, 32, 16, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) & sd().SD_DEVERR_INDEX
    np.testing.assert_array_equal(segs.cpu().numpy()[0], [0, 1, -1, -1])


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_gather_attend_skips_empty_slots(dt):
    g = torch.Generator().manual_seed(21)
    B, V, Hq, Hkv, d, T, blk, n = 2, 2, 8, 2, 128, 1024, 16, 9
    q = torch.randn(B, V, Hq, d, generator=g).to(dt)
    K = torch.randn(B, Hkv, T, d, generator=g).to(dt)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(dt)
    sidx = torch.full((B, Hkv, n), -1, dtype=torch.int32)
    for b in range(B):
        for h in range(Hkv):
            m = 3 + 2 * b + h  # varying counts, the rest empty
            sidx[b, h, :m] = torch.sort(torch.randperm(T // blk, generator=g)[:m]).values
    sidx[1, 1, :] = -1  # one group with nothing selected
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, logits = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), sidx.cuda(), block=blk, T=T,
                                          scale=1 / math.sqrt(d), want_logits=True, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0, "empty slots are not errors"
    ro, rl, rz = oracle.gather_attend(q, K, Vv, sidx.numpy(), B, V, Hq, Hkv, d, T, n, blk, 1 / math.sqrt(d), True)
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")
    lz = logits.cpu().numpy()
    assert np.array_equal(np.isneginf(lz), np.isneginf(rz))
    fin = np.isfinite(rz)
    np.testing.assert_allclose(lz[fin], rz[fin], atol=1e-4, rtol=1e-5)
    # the sparse score accumulate skips them too
    s0 = torch.zeros(B, T, dtype=torch.float64)
    s_gpu = sd().sd_score_accumulate(logits, lse, sidx.cuda(), s0.clone().cuda(), Hkv, blk, 0.5)
    s_ref = s0.numpy().copy()
    oracle.score_accumulate(lz.astype(np.float64), lse.cpu().numpy().astype(np.float64), sidx.numpy(), s_ref, B, V,
                            Hq, Hkv, n, blk, T, 0.5)
    np.testing.assert_allclose(s_gpu.cpu().numpy(), s_ref, rtol=2e-6, atol=1e-12)


def test_window_pipeline_end_to_end():
    # indexer -> window max (with the histogram) -> top-k windows -> union -> attention over
    # 16-token segments, against the oracle chain on the same inputs
    g = torch.Generator().manual_seed(22)
    B, Hq, Hkv, d, T, k, kern, strd = 2, 16, 4, 128, 8192, 48, 32, 16
    qi = torch.randint(-8, 9, (B, Hkv, 1, 128), generator=g).float().to(torch.bfloat16)
    ki = torch.randint(-8, 9, (B, Hkv, T, 128), generator=g).float().to(torch.bfloat16)
    q = torch.randn(B, 1, Hq, d, generator=g).to(torch.bfloat16)
    K = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    hist = sd().key_hist_buffer(B * Hkv)
    s = sd().sd_index_score(qi.cuda(), ki.cuda())
    w = sd().sd_window_max(s, kern, strd, key_hist=hist)
    widx = sd().sd_topk(w, k, key_hist=hist)
    segs = sd().sd_window_union(widx, T, kern, strd)
    out, lse, _ = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), segs, block=strd, T=T)
    rs = oracle.index_score(qi, ki, B, Hkv, 1, T, 128)
    rw = oracle.window_max(rs, kern, strd)
    np.testing.assert_array_equal(w.cpu().numpy().astype(np.float64), rw)
    ri = oracle.topk(rw, k)
    np.testing.assert_array_equal(widx.cpu().numpy(), ri)
    rseg = oracle.window_union(ri, T, kern, strd)
    np.testing.assert_array_equal(segs.cpu().numpy(), rseg)
    ro, rl, _ = oracle.gather_attend(q, K, Vv, rseg, B, 1, Hq, Hkv, d, T, rseg.shape[-1], strd, 1 / math.sqrt(d))
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")


def test_c6_window_blocks_full():
    # the benchmark's window workload at full size, in its launch configuration
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c6_window_blocks"]
    x = generate(w)
    g = {k: x[k].cuda() for k in ("q_idx", "k_idx", "q", "k", "v")}
    kern, strd = w.window_kernel, w.window_stride
    hist = sd().key_hist_buffer(w.B * w.Hkv)
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = sd().sd_index_score(g["q_idx"], g["k_idx"], err_word=e)
    ws = sd().sd_window_max(s, kern, strd, key_hist=hist)
    widx = sd().sd_topk(ws, w.k, key_hist=hist)
    segs = sd().sd_window_union(widx, w.T, kern, strd, err_word=e)
    out, lse, _ = sd().gather_attend(g["q"], g["k"], g["v"], segs, block=strd, T=w.T, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    rs = oracle.index_score(x["q_idx"], x["k_idx"], w.B, w.Hkv, w.V, w.T, w.dI)
    rw = oracle.window_max(rs, kern, strd)
    ri = oracle.topk(rw, w.k)
    np.testing.assert_array_equal(widx.cpu().numpy(), ri)
    rseg = oracle.window_union(ri, w.T, kern, strd)
    np.testing.assert_array_equal(segs.cpu().numpy(), rseg)
    # planted heavy hitters outscore every other token, so every selected window holds one
    for b in range(w.B):
        for h in range(w.Hkv):
            planted = set(int(t) for t in x["planted"][b, h])
            for n in ri[b, h]:
                assert planted & set(range(n * strd, n * strd + kern))
    ro, rl, _ = oracle.gather_attend(x["q"], x["k"], x["v"], rseg, w.B, w.V, w.Hq, w.Hkv, w.d, w.T,
                                     rseg.shape[-1], strd, 1 / math.sqrt(w.d))
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")
