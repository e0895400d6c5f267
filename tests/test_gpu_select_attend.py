"""Parity of the fused select + attend call (sd_select_attend) with the CPU oracle: the
index sets bit-exact with the oracle's top-k (and with sd_topk), attention outputs within
2e-3 max-abs and 1e-3 relative L2 of the fp64 oracle over the oracle's selection.  The
cases cover several parts per row with ragged tails, scores read from shared memory and
from global memory, the indexer's histogram given or not, heavy ties (the candidate
buffer overflows and the cluster falls back to passes over the keys), k = 0 / 1 / N,
block selection, the verify batch (32 query rows), every cluster size and the host-memory
residency path.  All calls go through the C ABI."""
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


def err_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def make_scores(kind, B, Hkv, N, seed):
    """(device scores, host fp64 scores, key_hist or None) of one kind."""
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    if kind in ("index", "flat"):
        q = torch.randint(-8, 9, (B, Hkv, 1, 128), generator=g).float().to(torch.bfloat16)
        if kind == "flat":
            q.zero_()   # every score 0: one bin, all ties
        k = torch.randint(-8, 9, (B, Hkv, N, 128), generator=g).float().to(torch.bfloat16)
        hist = sd().key_hist_buffer(B * Hkv)
        s = sd().sd_index_score(q.cuda(), k.cuda(), key_hist=hist)
        return s, oracle.index_score(q, k, B, Hkv, 1, N, 128), hist
    if kind == "normal":
        s = (rng.standard_normal((B, Hkv, N)) * 10).astype(np.float32)
    elif kind == "few":       # three distinct values: the boundary bin overflows
        s = rng.integers(0, 3, size=(B, Hkv, N)).astype(np.float32)
    elif kind == "zeros":     # +0 and -0 tie; the lower index wins
        s = (rng.standard_normal((B, Hkv, N)) * 3).astype(np.float32)
        s[..., ::3] = 0.0
        s[..., 1::3] = -0.0
    elif kind == "denorm":    # boundary among negative denormals, just below the zeros' bin
        s = np.empty((B, Hkv, N), dtype=np.float32)
        for r in np.ndindex(B, Hkv):
            q4 = N // 4
            vals = np.concatenate([rng.uniform(1, 2, q4).astype(np.float32),            # positives
                                   np.where(rng.random(q4) < 0.5, 0.0, -0.0).astype(np.float32),
                                   -(rng.permutation(N - 2 * q4) + 1).astype(np.float32) * np.float32(1e-42)])
            s[r] = vals[rng.permutation(N)]
    else:
        raise ValueError(kind)
    return torch.from_numpy(s).cuda(), s.astype(np.float64), None


def run_case(B, V, Hq, Hkv, d, N, block, k, kind, splits, seed, want_logits=True):
    T = N * block
    s_dev, s_ref, hist = make_scores(kind, B, Hkv, N, seed)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, V, Hq, d, generator=g).to(torch.bfloat16)
    K = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    e = err_word()
    scale = 1.0 / math.sqrt(d)
    idx, out, lse, logits = sd().select_attend(s_dev, k, q.cuda(), K.cuda(), Vv.cuda(), key_hist=hist,
                                               block=block, T=T, scale=scale, want_logits=want_logits,
                                               err_word=e, splits=splits)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    if hist is not None:
        assert int(hist.abs().sum().item()) == 0, "the histogram must be left zeroed"
    ri = oracle.topk(s_ref, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ri)
    ro, rl, rz = oracle.gather_attend(q, K, Vv, ri, B, V, Hq, Hkv, d, T, k, block, scale, want_logits)
    assert_attend_close(out, ro, "out")
    assert_attend_close(lse, rl, "lse")
    if want_logits:
        np.testing.assert_allclose(logits.cpu().numpy(), rz, atol=1e-4, rtol=1e-5)
    return idx, out, lse


@pytest.mark.parametrize("B,V,Hq,Hkv,d,N,block,k,kind,splits", [
    (2, 1, 32, 8, 128, 32768, 1, 1024, "index", 0),   # Llama-3-8B-shaped rows, 2 sequences
    (1, 8, 8, 2, 128, 20000, 1, 700, "index", 0),     # 32 query rows, ragged last part
    (1, 1, 8, 2, 128, 4099, 1, 300, "normal", 0),     # N % 4 != 0: scores read from global
    (1, 2, 16, 2, 64, 3000, 1, 100, "normal", 0),     # d = 64, R = 16
    (1, 1, 8, 2, 128, 20000, 1, 100, "few", 0),       # candidate overflow -> key passes
    (1, 1, 8, 2, 128, 20000, 1, 100, "flat", 0),      # every score equal, histogram given
    (1, 1, 8, 2, 128, 3001, 1, 1500, "zeros", 0),     # signed zeros in the boundary
    (1, 1, 8, 2, 128, 4000, 1, 2300, "denorm", 0),    # boundary bin just below zero
    (1, 1, 8, 8, 128, 5000, 1, 333, "normal", 0),     # MHA (G = 1)
    (1, 1, 8, 2, 128, 64, 64, 7, "normal", 0),        # 7 blocks of 64 tokens
    (1, 1, 8, 2, 128, 2048, 64, 64, "index", 0),      # block-selection shape: 2048 blocks
    (1, 1, 8, 2, 128, 200000, 1, 2048, "index", 0),   # long rows: parts beyond shared memory
])
def test_select_attend_matches_oracle(B, V, Hq, Hkv, d, N, block, k, kind, splits):
    run_case(B, V, Hq, Hkv, d, N, block, k, kind, splits, seed=N + k + V)


@pytest.mark.parametrize("k", [0, 1, 4095, 4096])
def test_select_attend_degenerate_k(k):
    idx, out, lse = run_case(1, 1, 8, 2, 128, 4096, 1, k, "normal", 0, seed=17 + k)
    if k == 0:
        assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
def test_select_attend_every_cluster_size(splits):
    idx, _, _ = run_case(1, 1, 8, 2, 128, 12000, 1, 500, "index", splits, seed=23)
    # the index set does not depend on the cluster size
    s_dev, s_ref, _ = make_scores("index", 1, 2, 12000, 23)
    np.testing.assert_array_equal(idx.cpu().numpy(), sd().sd_topk(s_dev, 500).cpu().numpy())


def test_select_attend_agrees_with_the_separate_calls():
    # same index set as sd_topk; attention equal to sd_gather_attend within tolerance
    B, V, Hq, Hkv, d, N, k = 2, 1, 32, 8, 128, 32768, 1024
    s_dev, s_ref, hist = make_scores("index", B, Hkv, N, 5)
    g = torch.Generator().manual_seed(6)
    q = torch.randn(B, V, Hq, d, generator=g).to(torch.bfloat16).cuda()
    K = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16).cuda()
    Vv = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16).cuda()
    idx_f, out_f, lse_f, _ = sd().select_attend(s_dev, k, q, K, Vv, key_hist=hist, T=N)
    idx_s = sd().sd_topk(s_dev, k)   # the fused call leaves the scores as they were
    out_s, lse_s, _ = sd().gather_attend(q, K, Vv, idx_s, T=N)
    assert torch.equal(idx_f, idx_s)
    assert_attend_close(out_f, out_s.double().cpu().numpy(), "out")
    assert_attend_close(lse_f, lse_s.double().cpu().numpy(), "lse")


def test_select_attend_residency_is_bit_identical():
    # rows read from pinned host memory give the same bits as rows read from HBM
    from top_sparse_decode_gqa_gb300.workloads import residency_map
    B, V, Hq, Hkv, d, N, k = 2, 4, 8, 2, 128, 8000, 400
    s_dev, s_ref, _ = make_scores("normal", B, Hkv, N, 31)
    g = torch.Generator().manual_seed(32)
    q = torch.randn(B, V, Hq, d, generator=g).to(torch.bfloat16)
    K = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16)
    Vv = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16)
    kh, vh = K.pin_memory(), Vv.pin_memory()
    results = []
    for P in (0, N // 10, N):
        res, slot_map = residency_map(B, N, P, seed=7)
        gi = res[:, None, :, None].expand(B, Hkv, P, d)
        k_pool = torch.gather(K, 2, gi).contiguous().cuda()
        v_pool = torch.gather(Vv, 2, gi).contiguous().cuda()
        if P == 0:
            k_pool = torch.zeros(B, Hkv, 1, d, dtype=K.dtype, device="cuda")
            v_pool = torch.zeros_like(k_pool)
        e = err_word()
        idx, out, lse, _ = sd().select_attend(s_dev, k, q.cuda(), k_pool, v_pool, T=N, k_host=kh, v_host=vh,
                                              slot_map=slot_map.cuda(), err_word=e)
        torch.cuda.synchronize()
        assert int(e.item()) == 0
        results.append((idx.cpu(), out.cpu(), lse.cpu()))
    idx_d, out_d, lse_d, _ = sd().select_attend(s_dev, k, q.cuda(), K.cuda(), Vv.cuda(), T=N)
    for idx, out, lse in results[1:] + [(idx_d.cpu(), out_d.cpu(), lse_d.cpu())]:
        assert torch.equal(idx, results[0][0])
        assert torch.equal(out, results[0][1]) and torch.equal(lse, results[0][2])
    ri = oracle.topk(s_ref, k)
    ro, rl, _ = oracle.gather_attend(q, K, Vv, ri, B, V, Hq, Hkv, d, N, k, 1, 1.0 / math.sqrt(d))
    assert_attend_close(results[0][1], ro)


def test_select_attend_repeated_calls_reuse_the_histogram():
    B, Hkv, N, k = 2, 4, 16384, 512
    g = torch.Generator().manual_seed(71)
    qi = torch.randint(-8, 9, (B, Hkv, 1, 128), generator=g).float().to(torch.bfloat16).cuda()
    ki = torch.randint(-8, 9, (B, Hkv, N, 128), generator=g).float().to(torch.bfloat16).cuda()
    q = torch.randn(B, 1, Hkv * 4, 128, generator=g).to(torch.bfloat16).cuda()
    K = torch.randn(B, Hkv, N, 128, generator=g).to(torch.bfloat16).cuda()
    hist = sd().key_hist_buffer(B * Hkv)
    first = None
    for _ in range(3):
        s = sd().sd_index_score(qi, ki, key_hist=hist)
        idx, out, lse, _ = sd().select_attend(s, k, q, K, K, key_hist=hist, T=N)
        torch.cuda.synchronize()
        assert int(hist.abs().sum().item()) == 0
        if first is None:
            first = (idx.clone(), out.clone(), lse.clone())
        else:
            assert torch.equal(idx, first[0]) and torch.equal(out, first[1]) and torch.equal(lse, first[2])
