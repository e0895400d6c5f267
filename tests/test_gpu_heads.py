"""Parity of per-query-head selection with the CPU oracle: one score row per query head
(sd_index_score_heads: bit-exact on integer inputs, within the fp32 summation bound on real
ones), the per-row key histogram checked through the top-k it seeds, the per-head mode of
gather-attend (each head over its own rows, from the pool or pinned host memory), and the
whole chain at a small size and at the benchmark's full size.  All calls go through the C
ABI."""
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


def _ints(g, shape, dt):
    return torch.randint(-8, 9, shape, generator=g).float().to(dt)


@pytest.mark.parametrize("qdt,kdt", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32),
                                     (torch.float32, torch.bfloat16)])
@pytest.mark.parametrize("B,Hkv,V,N,d", [(2, 3, 4, 4096 + 37, 128), (1, 2, 1, 1000, 64), (2, 1, 8, 300, 128),
                                         (1, 1, 3, 5, 64)])
def test_index_score_heads_exact_on_integers(qdt, kdt, B, Hkv, V, N, d):
    g = torch.Generator().manual_seed(B * 1000 + N + V)
    q, k = _ints(g, (B, Hkv, V, d), qdt), _ints(g, (B, Hkv, N, d), kdt)
    s = sd().sd_index_score_heads(q.cuda(), k.cuda())
    ref = oracle.index_score_heads(q, k, B, Hkv, V, N, d)
    np.testing.assert_array_equal(s.cpu().numpy().astype(np.float64), ref)


def test_index_score_heads_sixteen_queries_on_the_tensor_cores():
    g = torch.Generator().manual_seed(5)
    B, Hkv, V, N, d = 2, 2, 16, 3000, 128
    q, k = _ints(g, (B, Hkv, V, d), torch.bfloat16), _ints(g, (B, Hkv, N, d), torch.bfloat16)
    s = sd().sd_index_score_heads(q.cuda(), k.cuda())
    np.testing.assert_array_equal(s.cpu().numpy().astype(np.float64), oracle.index_score_heads(q, k, B, Hkv, V, N, d))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_index_score_heads_real_values_within_the_fp32_bound(dt):
    # |fl(sum) - sum| <= gamma_d * sum |q_j k_j| for any summation order; 2x for margin
    g = torch.Generator().manual_seed(6)
    B, Hkv, V, N, d = 2, 4, 4, 5000, 128
    q = torch.randn(B, Hkv, V, d, generator=g).to(dt)
    k = torch.randn(B, Hkv, N, d, generator=g).to(dt)
    s = sd().sd_index_score_heads(q.cuda(), k.cuda()).cpu().numpy().astype(np.float64)
    ref = oracle.index_score_heads(q, k, B, Hkv, V, N, d)
    mag = oracle.index_score_heads(q.abs(), k.abs(), B, Hkv, V, N, d)
    bound = 2 * d * 2.0 ** -24 * mag + 1e-30
    assert np.all(np.abs(s - ref) <= bound)


def test_heads_histogram_seeds_the_topk():
    # the histogram holds one row per query row, and top-k through it equals the oracle's
    # top-k of the same fp32 scores (the comparison the kernel makes, in the kernel's type)
    g = torch.Generator().manual_seed(7)
    B, Hkv, G, N, d, k = 2, 2, 4, 32768, 128, 1024
    q = torch.randn(B, Hkv, G, d, generator=g).to(torch.bfloat16)
    K = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16)
    hist = sd().key_hist_buffer(B * Hkv * G)
    s = sd().sd_index_score_heads(q.cuda(), K.cuda(), key_hist=hist)
    assert torch.equal(hist.sum(1).cpu(), torch.full((B * Hkv * G,), N, dtype=torch.int64))
    idx = sd().sd_topk(s, k, key_hist=hist)
    torch.cuda.synchronize()
    assert int(hist.abs().sum().item()) == 0
    ref = oracle.topk(s.cpu().numpy().astype(np.float64), k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)


def _per_head_idx(g, B, Hq, T, n, block=1, empty=0):
    idx = torch.full((B, Hq, n), -1, dtype=torch.int32)
    for b in range(B):
        for h in range(Hq):
            m = n - (empty if (b + h) % 3 == 0 else 0)
            idx[b, h, :m] = torch.sort(torch.randperm(T // block, generator=g)[:m]).values
    return idx


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,block,n,T", [(1, 1, 1024, 8192), (1, 1, 700, 3001), (2, 16, 40, 4096), (4, 1, 5, 64)])
def test_gather_attend_per_head_matches_the_oracle(dt, V, block, n, T):
    g = torch.Generator().manual_seed(V * 100 + n)
    B, Hq, Hkv, d = 2, 16, 4, 128
    q = torch.randn(B, V, Hq, d, generator=g).to(dt)
    K = torch.randn(B, Hkv, T, d, generator=g).to(dt)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(dt)
    idx = _per_head_idx(g, B, Hq, T, n, block, empty=min(3, n - 1))
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, logits = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), idx.cuda(), block=block, T=T,
                                          want_logits=True, err_word=e, per_head=True)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    ro, rl, rz = oracle.gather_attend(q, K, Vv, idx.numpy(), B, V, Hq, Hkv, d, T, n, block, 1 / math.sqrt(d), True,
                                      per_head=True)
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")
    lz = logits.cpu().numpy()
    assert np.array_equal(np.isneginf(lz), np.isneginf(rz))
    fin = np.isfinite(rz)
    np.testing.assert_allclose(lz[fin], rz[fin], atol=1e-4, rtol=1e-5)


def test_per_head_equals_shared_when_the_heads_agree():
    # every head of a group given its group's rows: the per-head mode returns the shared
    # selection's result (within the attention tolerance: the two modes tile the query rows
    # differently, so the summation order may differ)
    g = torch.Generator().manual_seed(8)
    B, Hq, Hkv, d, T, n = 2, 32, 8, 128, 4096, 512
    q = torch.randn(B, 1, Hq, d, generator=g).to(torch.bfloat16).cuda()
    K = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16).cuda()
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16).cuda()
    shared = _per_head_idx(g, B, Hkv, T, n).cuda()
    o1, l1, _ = sd().gather_attend(q, K, Vv, shared, T=T)
    o2, l2, _ = sd().gather_attend(q, K, Vv, shared.repeat_interleave(Hq // Hkv, dim=1).contiguous(), T=T,
                                   per_head=True)
    ro, rl, _ = oracle.gather_attend(q.cpu(), K.cpu(), Vv.cpu(), shared.cpu().numpy(), B, 1, Hq, Hkv, d, T, n, 1,
                                     1 / math.sqrt(d))
    assert_attend_close(o1, ro)
    assert_attend_close(o2, ro)
    assert_attend_close(l2, rl, "lse")


def test_per_head_rows_from_the_pool_and_host_memory_are_the_same_bits():
    from top_sparse_decode_gqa_gb300.workloads import residency_map
    g = torch.Generator().manual_seed(9)
    B, Hq, Hkv, d, T, n = 2, 8, 2, 128, 4000, 300
    q = torch.randn(B, 1, Hq, d, generator=g).to(torch.bfloat16)
    K = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    idx = _per_head_idx(g, B, Hq, T, n).cuda()
    base_o, base_l, _ = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), idx, T=T, per_head=True)
    P = T // 10
    res, slot_map = residency_map(B, T, P, 3)
    gi = res[:, None, :, None].expand(B, Hkv, P, d)
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse, _ = sd().gather_attend(q.cuda(), torch.gather(K, 2, gi).contiguous().cuda(),
                                   torch.gather(Vv, 2, gi).contiguous().cuda(), idx, T=T, k_host=K.pin_memory(),
                                   v_host=Vv.pin_memory(), slot_map=slot_map.cuda(), err_word=e, per_head=True)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    assert torch.equal(o, base_o) and torch.equal(lse, base_l)
    ro, rl, _ = oracle.gather_attend(q, K, Vv, idx.cpu().numpy(), B, 1, Hq, Hkv, d, T, n, 1, 1 / math.sqrt(d),
                                     per_head=True)
    assert_attend_close(o, ro)


def _chain(w, x):
    """Per-head logits -> per-head top-k -> per-head attention on the device."""
    dev = {k: x[k].cuda() for k in ("q", "k", "v")}
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = sd().key_hist_buffer(w.B * w.Hq)
    s = sd().sd_index_score_heads(dev["q"].view(w.B, w.Hkv, w.G, w.d), dev["k"], err_word=e, key_hist=hist)
    idx = sd().sd_topk(s.view(w.B, w.Hq, w.T), w.k, key_hist=hist)
    out, lse, _ = sd().gather_attend(dev["q"], dev["k"], dev["v"], idx, T=w.T, err_word=e, per_head=True)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    return s, idx, out, lse


def _check_chain(w, x, s, idx, out, lse, seqs):
    scale = 1 / math.sqrt(w.d)
    for b in seqs:
        q = x["q"][b:b + 1].contiguous()
        k, v = x["k"][b:b + 1].contiguous(), x["v"][b:b + 1].contiguous()
        rs = oracle.index_score_heads(q.view(1, w.Hkv, w.G, w.d), k, 1, w.Hkv, w.G, w.T, w.d)
        sg = s[b].cpu().numpy().astype(np.float64)
        mag = oracle.index_score_heads(q.abs().view(1, w.Hkv, w.G, w.d), k.abs(), 1, w.Hkv, w.G, w.T, w.d)
        assert np.all(np.abs(sg - rs[0]) <= 2 * w.d * 2.0 ** -24 * mag[0] + 1e-30)
        # the selection is decided on the kernel's fp32 scores, compared exactly
        ri = oracle.topk(sg.reshape(w.Hq, w.T), w.k)
        np.testing.assert_array_equal(idx[b].cpu().numpy(), ri)
        ro, rl, _ = oracle.gather_attend(q, k, v, ri[None], 1, w.V, w.Hq, w.Hkv, w.d, w.T, w.k, 1, scale,
                                         per_head=True)
        assert_attend_close(out[b:b + 1], ro)
        assert_attend_close(lse[b:b + 1], rl, "lse")


def test_head_topk_chain_small():
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c7_head_topk"].scaled(B=2, T=4096 + 96, k=200)
    x = generate(w)
    _check_chain(w, x, *_chain(w, x), seqs=range(w.B))


def test_c7_head_topk_full():
    # the benchmark's per-head workload at full size, in its launch configuration; the oracle
    # checks two of the eight sequences whole
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c7_head_topk"]
    x = generate(w)
    s, idx, out, lse = _chain(w, x)
    _check_chain(w, x, s, idx, out, lse, seqs=(0, w.B - 1))
    # planted heavy hitters are boosted toward every head of their group: each head keeps
    # them far above the uniform share k/T (about a third of them at these sizes)
    kept = 0
    for b in (0, w.B - 1):
        for h in range(w.Hq):
            kept += len(set(x["planted"][b, h // w.G].tolist()) & set(idx[b, h].cpu().tolist()))
    assert kept > 5 * (w.k / w.T) * 2 * w.Hq * w.planted
