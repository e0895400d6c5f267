"""Pins for the CPU oracle: each step checked against something other than itself --
hand-derived worked examples (tests/golden, each citing the passage it follows), closed
forms, invariants the mathematics fixes, brute force, and library routines (torch's fp64
scaled-dot-product attention, numpy's lexsort) where a special case reduces to one.

No GPU is needed.  The pins are chosen so that a dropped term, a wrong sign or index, or
a transposed operand in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import load_golden

# ----------------------------------------------------------------------------- helpers


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def rand_int(g, shape):
    return torch.randint(-8, 9, shape, generator=g).to(torch.float32)


# ----------------------------------------------------------------------------- step 1


def test_index_score_golden_bf16():
    gd = load_golden("index_score_bf16_small.json")
    q = np.array(gd["q_bits"], dtype=np.uint16)
    k = np.array(gd["k_bits"], dtype=np.uint16)
    s = oracle.index_score(q, k, 1, 1, 1, 3, 3)
    assert s.reshape(-1).tolist() == gd["scores"]
    q2 = np.array(gd["q_bits_two_queries"], dtype=np.uint16)
    s2 = oracle.index_score(q2, k, 1, 1, 2, 3, 3)
    assert s2.reshape(-1).tolist() == gd["scores_union"]


def test_index_score_unit_vectors_pin_every_coordinate_and_head():
    # A unit query e_j (times a per-(b,h) factor) must return column j of that head's keys:
    # this pins operand order (no transpose), the (b, h) indexing and each coordinate.
    g = torch.Generator().manual_seed(1)
    B, Hkv, N, dI = 2, 3, 37, 5
    k = rand_int(g, (B, Hkv, N, dI))
    for j in range(dI):
        q = torch.zeros(B, Hkv, 1, dI)
        for b in range(B):
            for h in range(Hkv):
                q[b, h, 0, j] = float(b * Hkv + h + 1)
        s = oracle.index_score(q.numpy(), k.numpy(), B, Hkv, 1, N, dI)
        for b in range(B):
            for h in range(Hkv):
                np.testing.assert_array_equal(s[b, h], (b * Hkv + h + 1) * k[b, h, :, j].numpy())


def test_index_score_linear_in_query():
    # Linearity plus the unit-vector pin fixes the map completely (a missing term, an
    # absolute value or a square would break one or the other).
    g = torch.Generator().manual_seed(2)
    B, Hkv, N, dI = 1, 2, 50, 16
    k = rand_int(g, (B, Hkv, N, dI))
    q1, q2 = rand_int(g, (B, Hkv, 1, dI)), rand_int(g, (B, Hkv, 1, dI))
    s1 = oracle.index_score(q1.numpy(), k.numpy(), B, Hkv, 1, N, dI)
    s2 = oracle.index_score(q2.numpy(), k.numpy(), B, Hkv, 1, N, dI)
    s12 = oracle.index_score((q1 + q2).numpy(), k.numpy(), B, Hkv, 1, N, dI)
    np.testing.assert_array_equal(s1 + s2, s12)
    sneg = oracle.index_score((-q1).numpy(), k.numpy(), B, Hkv, 1, N, dI)
    np.testing.assert_array_equal(sneg, -s1)


def test_index_score_union_is_max_over_verify_queries():
    # Queries c_v * e_0: the union score of token t is max_v c_v * k[t, 0].
    g = torch.Generator().manual_seed(3)
    B, Hkv, N, dI, V = 1, 1, 40, 4, 3
    k = rand_int(g, (B, Hkv, N, dI))
    c = [2.0, -3.0, 0.5]
    q = torch.zeros(B, Hkv, V, dI)
    for v in range(V):
        q[0, 0, v, 0] = c[v]
    s = oracle.index_score(q.numpy(), k.numpy(), B, Hkv, V, N, dI)
    expect = np.max(np.stack([cv * k[0, 0, :, 0].numpy() for cv in c]), axis=0)
    np.testing.assert_array_equal(s[0, 0], expect)


def test_index_score_bf16_matches_fp32_for_integers():
    g = torch.Generator().manual_seed(4)
    B, Hkv, N, dI = 2, 2, 33, 128
    q, k = rand_int(g, (B, Hkv, 1, dI)), rand_int(g, (B, Hkv, N, dI))
    a = oracle.index_score(q.numpy(), k.numpy(), B, Hkv, 1, N, dI)
    b = oracle.index_score(bf16_bits(q), bf16_bits(k), B, Hkv, 1, N, dI)
    np.testing.assert_array_equal(a, b)
    # |score| <= 128 * 64 = 8192: integers, so exactly representable in fp32.
    assert np.all(np.abs(a) <= 8192) and np.all(a == np.round(a))


# ----------------------------------------------------------------------------- step 1'


def test_block_pool_closed_forms():
    B, Hkv, T, dI, blk = 1, 2, 256, 3, 64
    # Ramp keys k[t, j] = t + j: the mean over block n is n*blk + (blk-1)/2 + j.
    k = np.zeros((B, Hkv, T, dI), dtype=np.float32)
    for t in range(T):
        for j in range(dI):
            k[:, :, t, j] = t + j
    p = oracle.block_pool(k, B, Hkv, T, dI, blk)
    for n in range(T // blk):
        for j in range(dI):
            assert p[0, 1, n, j] == n * blk + (blk - 1) / 2 + j
    # Constant blocks pool to their constant; a single outlier moves the mean by 1/blk.
    k2 = np.zeros((B, Hkv, T, dI), dtype=np.float32)
    k2[0, 0, 64:128, :] = 5.0
    k2[0, 0, 130, 1] = 64.0
    p2 = oracle.block_pool(k2, B, Hkv, T, dI, blk)
    assert p2[0, 0, 1].tolist() == [5.0, 5.0, 5.0]
    assert p2[0, 0, 2].tolist() == [0.0, 1.0, 0.0]
    assert p2[0, 0, 0].tolist() == [0.0, 0.0, 0.0]


def test_block_score_is_mean_of_token_scores():
    # q . mean(K_block) = mean over the block of q . K_t (linearity of the mean).
    g = torch.Generator().manual_seed(5)
    B, Hkv, T, dI, blk = 2, 2, 512, 8, 64
    k = rand_int(g, (B, Hkv, T, dI))
    q = rand_int(g, (B, Hkv, 1, dI))
    tok = oracle.index_score(q.numpy(), k.numpy(), B, Hkv, 1, T, dI)
    pooled = oracle.block_pool(k.numpy(), B, Hkv, T, dI, blk).astype(np.float32)
    blk_s = oracle.index_score(q.numpy(), pooled, B, Hkv, 1, T // blk, dI)
    np.testing.assert_allclose(blk_s, tok.reshape(B, Hkv, T // blk, blk).mean(-1), rtol=0, atol=1e-9)
    # The pooled keys are multiples of 1/64 with |x| <= 8: exact in fp32.
    p64 = oracle.block_pool(k.numpy(), B, Hkv, T, dI, blk)
    np.testing.assert_array_equal(p64, p64.astype(np.float32).astype(np.float64))


def test_block_pool_rejects_ragged_blocks():
    with pytest.raises(oracle.OracleError):
        oracle.block_pool(np.zeros((1, 1, 100, 4), np.float32), 1, 1, 100, 4, 64)


# ----------------------------------------------------------------------------- step 2


def test_topk_golden_ties():
    gd = load_golden("topk_ties.json")
    s = np.array([gd["scores"]], dtype=np.float64)
    for k, expect in gd["cases"].items():
        assert oracle.topk(s, int(k))[0].tolist() == expect


def _check_topk_valid(s_row, idx_row, k):
    # Defining property: size k, ascending, unique, and every chosen index precedes every
    # other index in the order (score desc, index asc).
    assert len(idx_row) == k
    assert np.all(np.diff(idx_row) > 0)
    chosen = np.zeros(len(s_row), bool)
    chosen[idx_row] = True
    if k == 0 or k == len(s_row):
        return
    cs, ci = s_row[chosen], np.nonzero(chosen)[0]
    us, ui = s_row[~chosen], np.nonzero(~chosen)[0]
    worst_chosen = np.lexsort((-ci, cs))[0]        # lowest score, highest index among chosen
    best_other = np.lexsort((ui, -us))[0]          # highest score, lowest index among others
    a_s, a_i = cs[worst_chosen], ci[worst_chosen]
    b_s, b_i = us[best_other], ui[best_other]
    assert a_s > b_s or (a_s == b_s and a_i < b_i)


@pytest.mark.parametrize("N,k,levels", [(1, 1, 3), (17, 5, 3), (300, 64, 7), (1000, 999, 2),
                                        (4096, 1024, 50), (257, 0, 4)])
def test_topk_brute_force_validity(N, k, levels):
    rng = np.random.default_rng(N * 31 + k)
    s = rng.integers(0, levels, size=(3, N)).astype(np.float64)
    idx = oracle.topk(s, k)
    for r in range(3):
        _check_topk_valid(s[r], idx[r], k)


def test_topk_exhaustive_tiny():
    # Against the definition by enumeration: the chosen set is the lexicographically best
    # k-subset of (score desc, index asc) keys, found here by trying all subsets.
    from itertools import combinations
    rng = np.random.default_rng(7)
    for trial in range(30):
        N = 7
        k = int(rng.integers(0, N + 1))
        s = rng.integers(0, 3, size=N).astype(np.float64)
        best = None
        for comb in combinations(range(N), k):
            key = sorted([(-s[i], i) for i in comb])
            if best is None or key < best[0]:
                best = (key, comb)
        assert oracle.topk(s[None], k)[0].tolist() == list(best[1])


def test_topk_full_and_negative_scores():
    s = -np.arange(10, dtype=np.float64)[None] * 0.5
    assert oracle.topk(s, 10)[0].tolist() == list(range(10))
    assert oracle.topk(s, 3)[0].tolist() == [0, 1, 2]
    assert oracle.topk(s[:, ::-1].copy(), 3)[0].tolist() == [7, 8, 9]


# ----------------------------------------------------------------------------- step 3


def test_attend_golden_three_keys():
    gd = load_golden("attend_three_keys.json")
    q = np.array(gd["q"], np.float32).reshape(1, 1, 1, 2)
    K = np.array(gd["K"], np.float32).reshape(1, 1, 4, 2)
    V = np.array(gd["V"], np.float32).reshape(1, 1, 4, 2)
    idx = np.array(gd["idx"], np.int32).reshape(1, 1, 3)
    out, lse, logits = oracle.gather_attend(q, K, V, idx, 1, 1, 1, 1, 2, 4, 3, 1, 1.0, True)
    tol = gd["tol_from_fp32_inputs"]
    np.testing.assert_allclose(out.reshape(-1), gd["out"], atol=tol)
    assert abs(lse.item() - gd["lse"]) < tol
    alpha = np.exp(logits.reshape(-1) - lse.item())
    np.testing.assert_allclose(alpha, gd["alpha"], atol=tol)


def _sdpa_reference(q, K, V, scale):
    """torch fp64 SDPA on q [B,V,Hq,d], K/V [B,Hkv,n,d] (GQA: query head h uses KV head
    h // G) -> out [B,V,Hq,d], lse [B,V,Hq]."""
    B, Vq, Hq, d = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    qt = q.permute(0, 2, 1, 3).to(torch.float64)                   # [B,Hq,V,d]
    Kt = K.to(torch.float64).repeat_interleave(G, dim=1)           # [B,Hq,n,d]
    Vt = V.to(torch.float64).repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    lse = torch.logsumexp(scale * qt @ Kt.transpose(-1, -2), dim=-1)  # [B,Hq,V]
    return out.permute(0, 2, 1, 3).numpy(), lse.permute(0, 2, 1).numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_attend_dense_equals_sdpa(dtype):
    # With every row selected (k = T) sparse attention is dense softmax attention.
    g = torch.Generator().manual_seed(11)
    B, Vq, Hq, Hkv, d, T = 2, 2, 8, 2, 16, 70
    q, K, V = torch.randn(B, Vq, Hq, d, generator=g), torch.randn(B, Hkv, T, d, generator=g), \
        torch.randn(B, Hkv, T, d, generator=g)
    if dtype == "bf16":
        q, K, V = q.bfloat16(), K.bfloat16(), V.bfloat16()
    scale = 1 / math.sqrt(d)
    out, lse, _ = oracle.gather_attend(q, K, V, None, B, Vq, Hq, Hkv, d, T, T, 1, scale)
    ro, rl = _sdpa_reference(q, K, V, scale)
    np.testing.assert_allclose(out, ro, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(lse, rl, atol=1e-12, rtol=1e-12)
    # identity idx == NULL idx
    idx = np.tile(np.arange(T, dtype=np.int32), (B, Hkv, 1))
    out2, lse2, _ = oracle.gather_attend(q, K, V, idx, B, Vq, Hq, Hkv, d, T, T, 1, scale)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_attend_selection_equals_sdpa_on_gathered_rows():
    # Attention over idx equals dense attention over the rows K[idx], V[idx]; every head
    # group selects different rows, so a wrong (b, kvh) or GQA mapping fails.
    g = torch.Generator().manual_seed(12)
    B, Vq, Hq, Hkv, d, T, k = 2, 1, 8, 4, 32, 200, 23
    q = torch.randn(B, Vq, Hq, d, generator=g)
    K, V = torch.randn(B, Hkv, T, d, generator=g), torch.randn(B, Hkv, T, d, generator=g)
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(T, generator=g)[:k]).values
                                    for _ in range(Hkv)]) for _ in range(B)]).to(torch.int32)
    scale = 0.3
    out, lse, logits = oracle.gather_attend(q, K, V, idx.numpy(), B, Vq, Hq, Hkv, d, T, k, 1,
                                            scale, True)
    Kg = torch.gather(K, 2, idx.long()[..., None].expand(B, Hkv, k, d))
    Vg = torch.gather(V, 2, idx.long()[..., None].expand(B, Hkv, k, d))
    ro, rl = _sdpa_reference(q, Kg, Vg, scale)
    np.testing.assert_allclose(out, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)
    # softmax weights sum to one for every query row
    np.testing.assert_allclose(np.exp(logits - lse[..., None]).sum(-1), 1.0, atol=1e-12)


def test_attend_block_mode_expands_blocks():
    g = torch.Generator().manual_seed(13)
    B, Vq, Hq, Hkv, d, T, blk, k = 1, 1, 4, 2, 16, 256, 16, 3
    q = torch.randn(B, Vq, Hq, d, generator=g)
    K, V = torch.randn(B, Hkv, T, d, generator=g), torch.randn(B, Hkv, T, d, generator=g)
    bidx = np.array([[[1, 4, 15], [0, 7, 8]]], dtype=np.int32)
    out, lse, _ = oracle.gather_attend(q, K, V, bidx, B, Vq, Hq, Hkv, d, T, k, blk, 0.25)
    rows = torch.tensor(bidx).long()[..., None] * blk + torch.arange(blk)  # [B,Hkv,k,blk]
    rows = rows.reshape(B, Hkv, k * blk)
    Kg = torch.gather(K, 2, rows[..., None].expand(B, Hkv, k * blk, d))
    Vg = torch.gather(V, 2, rows[..., None].expand(B, Hkv, k * blk, d))
    ro, rl = _sdpa_reference(q, Kg, Vg, 0.25)
    np.testing.assert_allclose(out, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)


def test_attend_identical_keys_give_mean_of_values():
    g = torch.Generator().manual_seed(14)
    B, Vq, Hq, Hkv, d, T = 1, 1, 2, 1, 8, 50
    q = torch.randn(B, Vq, Hq, d, generator=g)
    K = torch.randn(1, 1, 1, d, generator=g).expand(B, Hkv, T, d).contiguous()
    V = torch.randn(B, Hkv, T, d, generator=g)
    idx = np.array([[[3, 9, 10, 44]]], np.int32)
    out, lse, _ = oracle.gather_attend(q, K, V, idx, B, Vq, Hq, Hkv, d, T, 4, 1, 1.0)
    vmean = V[0, 0, [3, 9, 10, 44]].double().mean(0).numpy()
    np.testing.assert_allclose(out[0, 0, 0], vmean, atol=1e-12)
    np.testing.assert_allclose(out[0, 0, 1], vmean, atol=1e-12)
    z = (q[0, 0].double() @ K[0, 0, 0].double()).numpy()
    np.testing.assert_allclose(lse[0, 0], z + math.log(4), atol=1e-12)


def test_attend_empty_selection_and_bad_index():
    q = np.ones((1, 1, 2, 4), np.float32)
    K = np.ones((1, 1, 8, 4), np.float32)
    out, lse, _ = oracle.gather_attend(q, K, K, np.zeros((1, 1, 0), np.int32), 1, 1, 2, 1, 4, 8,
                                       0, 1, 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    with pytest.raises(oracle.OracleError):
        oracle.gather_attend(q, K, K, np.array([[[8]]], np.int32), 1, 1, 2, 1, 4, 8, 1, 1, 1.0)


# ----------------------------------------------------------------------------- step 4


def test_score_recurrence_golden():
    gd = load_golden("score_recurrence_small.json")
    logits = np.array(gd["logits"]).reshape(1, 1, 2, 3)
    lse = np.array(gd["lse"]).reshape(1, 1, 2)
    s = np.array([gd["s_before"]], dtype=np.float64)
    oracle.score_accumulate(logits, lse, None, s, 1, 1, 2, 1, 3, 1, 3, gd["weight"])
    np.testing.assert_allclose(s[0], gd["s_after"], atol=1e-15)


def test_score_recurrence_against_softmax_weights():
    # The page's equation over |L| layers and H heads, with alpha from torch.softmax of
    # the layer's logits, for a sparse selection (rows not selected get nothing).
    g = torch.Generator().manual_seed(21)
    B, Vq, Hq, Hkv, d, T, k, L = 2, 1, 6, 2, 16, 90, 20, 3
    s = np.zeros((B, T))
    expect = torch.zeros(B, T, dtype=torch.float64)
    for layer in range(L):
        q = torch.randn(B, Vq, Hq, d, generator=g)
        K, V = torch.randn(B, Hkv, T, d, generator=g), torch.randn(B, Hkv, T, d, generator=g)
        idx = torch.stack([torch.stack([torch.sort(torch.randperm(T, generator=g)[:k]).values
                                        for _ in range(Hkv)]) for _ in range(B)]).int()
        out, lse, logits = oracle.gather_attend(q, K, V, idx.numpy(), B, Vq, Hq, Hkv, d, T, k, 1,
                                                0.25, True)
        oracle.score_accumulate(logits, lse, idx.numpy(), s, B, Vq, Hq, Hkv, k, 1, T,
                                1.0 / (L * Hq))
        for b in range(B):
            for h in range(Hq):
                kvh = h // (Hq // Hkv)
                rows = idx[b, kvh].long()
                z = 0.25 * (K[b, kvh, rows].double() @ q[b, 0, h].double())
                expect[b, rows] += torch.softmax(z, 0) / (L * Hq)
    np.testing.assert_allclose(s, expect.numpy(), atol=1e-14)
    # every layer adds (1/|L|) * sum_h (1/H) * 1 = 1/|L| per sequence: total mass 1
    np.testing.assert_allclose(s.sum(1), 1.0, atol=1e-12)


def test_score_uniform_keys_give_t_over_T():
    # All keys equal: every softmax is uniform, so after t dense steps s_i = t / T.
    B, Vq, Hq, Hkv, d, T = 1, 1, 4, 2, 8, 64
    q = np.random.default_rng(0).standard_normal((B, Vq, Hq, d)).astype(np.float32)
    K = np.ones((B, Hkv, T, d), np.float32)
    s = np.zeros((B, T))
    for t in range(3):
        _, lse, logits = oracle.gather_attend(q, K, K, None, B, Vq, Hq, Hkv, d, T, T, 1, 1.0, True)
        oracle.score_accumulate(logits, lse, None, s, B, Vq, Hq, Hkv, T, 1, T, 1.0 / Hq)
        np.testing.assert_allclose(s, (t + 1) / T, atol=1e-14)


# ----------------------------------------------------------------------------- step 5


def test_tiers_golden():
    gd = load_golden("tiers_small.json")
    s = np.array([gd["s"]])
    tier, counts = oracle.tier_classify(s, gd["cum_frac"])
    assert tier[0].tolist() == gd["tier"] and counts[0].tolist() == gd["counts"]
    tier, counts = oracle.tier_classify(s, gd["cum_frac"], 1, 1)
    assert tier[0].tolist() == gd["tier_protected_1_1"]
    assert counts[0].tolist() == gd["counts_protected_1_1"]


@pytest.mark.parametrize("ties", [False, True])
def test_tiers_against_lexsort_and_counts(ties):
    B, T = 2, 65536 if not ties else 5000
    from top_sparse_decode_gqa_gb300.workloads import importance_scores
    s = importance_scores(B, T, seed=5, ties=ties).numpy()
    fr = (0.2, 0.6, 0.9)
    tier, counts = oracle.tier_classify(s, fr)
    c = [math.floor(f * T) for f in fr]
    for b in range(B):
        order = np.lexsort((np.arange(T), -s[b]))       # s desc, index asc
        rank = np.empty(T, np.int64)
        rank[order] = np.arange(T)
        expect = np.select([rank < c[0], rank < c[1], rank < c[2]], [0, 1, 2], 3)
        np.testing.assert_array_equal(tier[b], expect)
        assert counts[b].tolist() == [c[0], c[1] - c[0], c[2] - c[1], T - c[2]]
        # monotone: a lower tier never holds a smaller score than a higher tier
        for m in range(3):
            if np.any(tier[b] == m) and np.any(tier[b] == m + 1):
                assert s[b][tier[b] == m].min() >= s[b][tier[b] == m + 1].max()
    if not ties:
        assert counts[0].tolist() == [13107, 26214, 19661, 6554]


def test_tiers_protected_positions():
    B, T = 1, 1000
    s = np.linspace(1.0, 0.0, T)[None].copy()   # position 0 most important
    tier, counts = oracle.tier_classify(s, (0.2, 0.6, 0.9), 4, 64)
    assert np.all(tier[0, :4] == 0) and np.all(tier[0, -64:] == 0)
    # 68 protected take ranks 0..67, so T0 also holds the next 132 by score: 4..135
    assert np.all(tier[0, 4:136] == 0) and tier[0, 136] == 1
    assert counts[0].tolist() == [200, 400, 300, 100]
    # protection beyond the T0 budget keeps every protected position in T0
    tier, counts = oracle.tier_classify(s, (0.05, 0.6, 0.9), 40, 40)
    assert np.all(tier[0, :40] == 0) and np.all(tier[0, -40:] == 0) and counts[0, 0] == 80


# ----------------------------------------------------------------------------- step 6


def test_int8_golden():
    gd = load_golden("int8_rows.json")
    rows = np.array(gd["rows"], np.float32)
    n, d = rows.shape
    x = rows.reshape(1, 1, n, d)
    tier = np.full((1, n), 2, np.uint8)
    codes, scales = oracle.quantize_rows_int8(x, tier, 1, 1, n, d)
    assert codes.reshape(n, d).tolist() == gd["codes"]
    expect = [np.float32(a) / np.float32(gd["scales_den"]) for a in gd["scales_num"]]
    assert scales.reshape(-1).tolist() == [float(e) for e in expect]


def test_int8_error_bound_and_untouched_rows():
    g = torch.Generator().manual_seed(31)
    B, Hkv, T, d = 2, 2, 300, 128
    x = torch.randn(B, Hkv, T, d, generator=g).bfloat16()
    tier = torch.randint(0, 4, (B, T), generator=g).to(torch.uint8).numpy()
    codes0 = np.full((B, Hkv, T, d), 99, np.int8)
    scales0 = np.full((B, Hkv, T), -1.0, np.float32)
    codes, scales = oracle.quantize_rows_int8(x, tier, B, Hkv, T, d, codes0, scales0)
    xf = x.float().numpy()
    t2 = np.broadcast_to((tier == 2)[:, None, :], (B, Hkv, T))
    assert np.all(codes[~t2] == 99) and np.all(scales[~t2] == -1.0)
    rec = codes.astype(np.float64) * scales[..., None]
    err = np.abs(rec - xf)[t2]
    bound = (scales[..., None] * np.ones_like(xf))[t2] * (0.5 + 1e-5)
    assert np.all(err <= bound)
    amax = np.abs(xf).max(-1)
    # the largest-magnitude element of each row maps to +-127
    assert np.all(np.abs(codes).max(-1)[t2] == 127)
    np.testing.assert_allclose(scales[t2], (amax / np.float32(127))[t2], rtol=1e-7)


# ----------------------------------------------------------------------------- windows


@pytest.mark.parametrize("N,kernel,stride", [(64, 32, 16), (70, 32, 16), (20, 32, 16), (48, 16, 16),
                                             (33, 2, 1), (1, 32, 16), (0, 32, 16)])
def test_window_max_brute_force(N, kernel, stride):
    # every window's score is the maximum of the scores it covers (numpy over explicit slices)
    rng = np.random.default_rng(N + kernel)
    s = rng.integers(-50, 50, size=(3, N)).astype(np.float64)
    w = oracle.window_max(s, kernel, stride)
    starts = list(range(0, max(N - kernel, 0) + stride, stride)) if N > 0 else []
    starts = [t for t in starts if t < N and (t == 0 or t + kernel - stride < N)]
    assert w.shape == (3, len(starts)) == (3, oracle.window_count(N, kernel, stride))
    for r in range(3):
        for n, t0 in enumerate(starts):
            assert w[r, n] == s[r, t0:min(t0 + kernel, N)].max()


def test_window_count_closed_form():
    assert oracle.window_count(32768, 32, 16) == 2047        # (32768 - 32) / 16 + 1
    assert oracle.window_count(32769, 32, 16) == 2048        # one clipped window more
    assert oracle.window_count(32, 32, 16) == 1
    assert oracle.window_count(10, 32, 16) == 1
    assert oracle.window_count(0, 32, 16) == 0
    assert oracle.window_count(100, 1, 1) == 100             # token grid


def test_window_max_of_a_ramp():
    # increasing scores: window n's maximum is its last score
    s = np.arange(160, dtype=np.float64)[None]
    w = oracle.window_max(s, 32, 16)
    np.testing.assert_array_equal(w[0], [min(16 * n + 31, 159) for n in range(w.shape[1])])


@pytest.mark.parametrize("N,kernel,stride,k", [(64, 32, 16, 2), (512, 32, 16, 7), (512, 32, 16, 31),
                                               (96, 48, 16, 3), (64, 16, 16, 4)])
def test_window_union_is_the_set_of_covered_tokens(N, kernel, stride, k):
    # brute force: the union of the selected windows' token ranges, as segments of `stride`
    rng = np.random.default_rng(N + k)
    NW = oracle.window_count(N, kernel, stride)
    widx = np.stack([np.sort(rng.permutation(NW)[:k]) for _ in range(4)]).astype(np.int32)
    segs = oracle.window_union(widx, N, kernel, stride)
    assert segs.shape == (4, k * (kernel // stride))
    for r in range(4):
        tokens = set()
        for n in widx[r]:
            tokens |= set(range(n * stride, min(n * stride + kernel, N)))
        want = sorted({t // stride for t in tokens})
        got = segs[r]
        np.testing.assert_array_equal(got[:len(want)], want)
        assert np.all(got[len(want):] == -1)
        # segments cover exactly the tokens
        covered = {g * stride + i for g in got[got >= 0] for i in range(stride)}
        assert covered == tokens


def test_window_union_padding_and_bad_window():
    segs = oracle.window_union(np.array([[0, 1]], np.int32), 64, 32, 16, max_segs=8)
    np.testing.assert_array_equal(segs[0], [0, 1, 2, -1, -1, -1, -1, -1])  # windows 0, 1 share segment 1
    with pytest.raises(oracle.OracleError):
        oracle.window_union(np.array([[3]], np.int32), 64, 32, 16)          # only windows 0..2 exist
    with pytest.raises(oracle.OracleError):
        oracle.window_union(np.array([[0]], np.int32), 64, 24, 16)          # kernel not a multiple


def test_attend_empty_slots_take_no_part():
    # a selection padded with -1 equals SDPA over the non-empty rows only
    g = torch.Generator().manual_seed(15)
    B, Vq, Hq, Hkv, d, T, blk = 1, 2, 4, 2, 16, 128, 16
    q = torch.randn(B, Vq, Hq, d, generator=g)
    K, V = torch.randn(B, Hkv, T, d, generator=g), torch.randn(B, Hkv, T, d, generator=g)
    sidx = np.array([[[1, 2, 5, -1, -1], [0, 7, -1, -1, -1]]], np.int32)
    out, lse, logits = oracle.gather_attend(q, K, V, sidx, B, Vq, Hq, Hkv, d, T, 5, blk, 0.25, True)
    for kvh, segs in enumerate(([1, 2, 5], [0, 7])):
        rows = torch.tensor([g_ * blk + i for g_ in segs for i in range(blk)])
        ro, rl = _sdpa_reference(q[:, :, kvh * 2:kvh * 2 + 2], K[:, kvh:kvh + 1, rows], V[:, kvh:kvh + 1, rows], 0.25)
        np.testing.assert_allclose(out[:, :, kvh * 2:kvh * 2 + 2], ro, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, kvh * 2:kvh * 2 + 2], rl, atol=1e-12)
    # the empty slots' logits are -inf; the rest of each query row's weights sum to one
    assert np.all(np.isneginf(logits[0, :, 0:2, 3 * blk:]))
    np.testing.assert_allclose(np.exp(logits - lse[..., None]).sum(-1), 1.0, atol=1e-12)
    # all slots empty: nothing is attended
    out0, lse0, _ = oracle.gather_attend(q, K, V, np.full((1, 2, 3), -1, np.int32), B, Vq, Hq, Hkv, d, T, 3, blk, 0.25)
    assert np.all(out0 == 0) and np.all(np.isneginf(lse0))
    # any other negative entry is still an error
    with pytest.raises(oracle.OracleError):
        oracle.gather_attend(q, K, V, np.array([[[-2], [0]]], np.int32), B, Vq, Hq, Hkv, d, T, 1, blk, 0.25)


def test_score_accumulate_skips_empty_slots():
    g = torch.Generator().manual_seed(16)
    B, Vq, Hq, Hkv, d, T, blk = 1, 1, 4, 2, 8, 64, 16
    q = torch.randn(B, Vq, Hq, d, generator=g)
    K, V = torch.randn(B, Hkv, T, d, generator=g), torch.randn(B, Hkv, T, d, generator=g)
    sidx = np.array([[[1, -1], [3, 0]]], np.int32)
    _, lse, logits = oracle.gather_attend(q, K, V, sidx, B, Vq, Hq, Hkv, d, T, 2, blk, 0.5, True)
    s = np.zeros((B, T))
    oracle.score_accumulate(logits, lse, sidx, s, B, Vq, Hq, Hkv, 2, blk, T, 1.0)
    # KV head 0's two query heads put all their mass on segment 1 (its other slot is empty);
    # KV head 1's on segments 3 and 0
    assert np.all(s[0, 32:48] == 0)                              # segment 2: never selected
    np.testing.assert_allclose(s.sum(), Vq * Hq, atol=1e-12)       # every head's weights sum to 1
    np.testing.assert_allclose(s[0, 16:32].sum(), 2.0, atol=1e-12)  # heads 0, 1 -> segment 1 only


# ----------------------------------------------------------------------------- per-head selection


def test_index_score_heads_are_each_heads_logits():
    # with the attention query viewed as [B,Hkv,G,d], the per-query scores are every query
    # head's unscaled logits against its KV head's keys (fp64 einsum)
    g = torch.Generator().manual_seed(31)
    B, Hkv, G, N, d = 2, 3, 4, 50, 16
    q = torch.randn(B, 1, Hkv * G, d, generator=g)
    K = torch.randn(B, Hkv, N, d, generator=g)
    s = oracle.index_score_heads(q.reshape(B, Hkv, G, d), K, B, Hkv, G, N, d)
    ref = torch.einsum("bhd,bhtd->bht", q[:, 0].double(), K.double().repeat_interleave(G, dim=1))
    np.testing.assert_allclose(s.reshape(B, Hkv * G, N), ref.numpy(), atol=1e-12)
    # the union score of the shared indexer is their max over the group
    u = oracle.index_score(q.reshape(B, Hkv, G, d), K, B, Hkv, G, N, d)
    np.testing.assert_array_equal(u, s.max(axis=2))


def test_attend_per_head_uses_each_heads_own_rows():
    g = torch.Generator().manual_seed(32)
    B, Vq, Hq, Hkv, d, T, k = 2, 2, 8, 2, 16, 120, 11
    G = Hq // Hkv
    q = torch.randn(B, Vq, Hq, d, generator=g)
    K, V = torch.randn(B, Hkv, T, d, generator=g), torch.randn(B, Hkv, T, d, generator=g)
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(T, generator=g)[:k]).values
                                    for _ in range(Hq)]) for _ in range(B)]).to(torch.int32)  # [B,Hq,k]
    out, lse, logits = oracle.gather_attend(q, K, V, idx.numpy(), B, Vq, Hq, Hkv, d, T, k, 1, 0.3, True,
                                            per_head=True)
    for h in range(Hq):
        kvh = h // G
        rows = idx[:, h].long()  # [B,k]
        Kg = torch.gather(K[:, kvh], 1, rows[..., None].expand(B, k, d))[:, None]
        Vg = torch.gather(V[:, kvh], 1, rows[..., None].expand(B, k, d))[:, None]
        ro, rl = _sdpa_reference(q[:, :, h:h + 1], Kg, Vg, 0.3)
        np.testing.assert_allclose(out[:, :, h:h + 1], ro, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, h:h + 1], rl, atol=1e-12)
    np.testing.assert_allclose(np.exp(logits - lse[..., None]).sum(-1), 1.0, atol=1e-12)
    # when every head of a group picks the group's rows, per-head equals the shared selection
    shared = idx[:, ::G].contiguous()                        # [B,Hkv,k]
    per = shared.repeat_interleave(G, dim=1).contiguous()    # [B,Hq,k]
    o1, l1, _ = oracle.gather_attend(q, K, V, shared.numpy(), B, Vq, Hq, Hkv, d, T, k, 1, 0.3)
    o2, l2, _ = oracle.gather_attend(q, K, V, per.numpy(), B, Vq, Hq, Hkv, d, T, k, 1, 0.3, per_head=True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ----------------------------------------------------------------------------- draft ring (verify)


def _ring_case(seed, B=2, Vq=3, Hq=8, Hkv=2, d=16, T=90, k=7, W=6):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Vq, Hq, d, generator=g)
    K, V = torch.randn(B, Hkv, T, d, generator=g), torch.randn(B, Hkv, T, d, generator=g)
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(T, generator=g)[:k]).values
                                    for _ in range(Hkv)]) for _ in range(B)]).to(torch.int32)
    rk, rv = torch.randn(B, Hkv, W, d, generator=g), torch.randn(B, Hkv, W, d, generator=g)
    # ring positions: some empty, the rest a window of recent positions in ring order
    rpos = torch.full((B, W), -1, dtype=torch.int32)
    for b in range(B):
        n = W - b  # sequence 1 has one empty slot
        first = T - 2
        for i in range(n):
            rpos[b, (first + i) % W] = first + i
    qpos = torch.stack([torch.arange(T - 1, T - 1 + Vq) for _ in range(B)]).to(torch.int32)
    return q, K, V, idx, rk, rv, rpos, qpos


def test_ring_attend_equals_sdpa_over_each_querys_visible_rows():
    q, K, V, idx, rk, rv, rpos, qpos = _ring_case(41)
    B, Vq, Hq, d = q.shape
    Hkv, T, W = K.shape[1], K.shape[2], rpos.shape[1]
    G, k = Hq // Hkv, idx.shape[-1]
    out, lse, z = oracle.gather_attend_ring(q, K, V, idx.numpy(), B, Vq, Hq, Hkv, d, T, k, 1, 0.4, rk, rv,
                                            rpos.numpy(), qpos.numpy(), want_logits=True)
    for b in range(B):
        for v in range(Vq):
            vis = [s for s in range(W) if 0 <= int(rpos[b, s]) <= int(qpos[b, v])]
            for h in range(Hq):
                kvh = h // G
                Kr = torch.cat([K[b, kvh, idx[b, kvh].long()], rk[b, kvh, vis]])[None, None]
                Vr = torch.cat([V[b, kvh, idx[b, kvh].long()], rv[b, kvh, vis]])[None, None]
                ro, rl = _sdpa_reference(q[b:b + 1, v:v + 1, h:h + 1], Kr, Vr, 0.4)
                np.testing.assert_allclose(out[b, v, h], ro[0, 0, 0], atol=1e-12)
                np.testing.assert_allclose(lse[b, v, h], rl[0, 0, 0], atol=1e-12)
                hidden = [s for s in range(W) if s not in vis]
                assert np.all(np.isneginf(z[b, v, h, k + np.array(hidden, dtype=int)]))
                assert np.all(np.isfinite(z[b, v, h, k + np.array(vis, dtype=int)]))


def test_ring_causal_among_drafts_and_reductions():
    q, K, V, idx, rk, rv, rpos, qpos = _ring_case(42, W=8)
    B, Vq, Hq, d = q.shape
    Hkv, T, W = K.shape[1], K.shape[2], rpos.shape[1]
    k = idx.shape[-1]
    args = (q, K, V, idx.numpy(), B, Vq, Hq, Hkv, d, T, k, 1, 0.3, rk, rv)
    # an empty ring is plain gather-attend, bit for bit
    empty = np.full((B, W), -1, dtype=np.int32)
    o0, l0, _ = oracle.gather_attend_ring(*args, empty, qpos.numpy())
    o1, l1, _ = oracle.gather_attend(q, K, V, idx.numpy(), B, Vq, Hq, Hkv, d, T, k, 1, 0.3)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)
    # a ring entirely in every query's past: plain gather-attend over the history rows
    # followed by the ring rows as extra cache rows selected after them
    past = np.tile(np.arange(W, dtype=np.int32), (B, 1))
    Kx, Vx = torch.cat([K, rk], dim=2), torch.cat([V, rv], dim=2)
    idx_x = torch.cat([idx, torch.arange(T, T + W, dtype=torch.int32).expand(B, Hkv, W)], dim=2)
    o2, l2, _ = oracle.gather_attend_ring(*args, past, np.full((B, Vq), T, dtype=np.int32))
    o3, l3, _ = oracle.gather_attend(q, Kx, Vx, idx_x.numpy(), B, Vq, Hq, Hkv, d, T + W, k + W, 1, 0.3)
    np.testing.assert_array_equal(o2, o3)
    np.testing.assert_array_equal(l2, l3)
    # the V draft tokens in the ring: draft v sees drafts 0..v only; slot order is irrelevant
    drafts = np.full((B, W), -1, dtype=np.int32)
    for b in range(B):
        for v in range(Vq):
            drafts[b, (5 + v) % W] = 100 + v
    qp = np.tile(np.arange(100, 100 + Vq, dtype=np.int32), (B, 1))
    _, _, z = oracle.gather_attend_ring(*args, drafts, qp, want_logits=True)
    for b in range(B):
        for v in range(Vq):
            for u in range(Vq):
                col = k + (5 + u) % W
                assert np.isfinite(z[b, v, 0, col]) == (u <= v)
    perm = np.random.default_rng(0).permutation(W)
    o4, l4, _ = oracle.gather_attend_ring(*args, drafts, qp)
    o5, l5, _ = oracle.gather_attend_ring(q, K, V, idx.numpy(), B, Vq, Hq, Hkv, d, T, k, 1, 0.3, rk[:, :, perm],
                                          rv[:, :, perm], drafts[:, perm], qp)
    np.testing.assert_allclose(o4, o5, atol=1e-13)
    np.testing.assert_allclose(l4, l5, atol=1e-13)


def test_ring_append_keeps_the_last_window():
    g = torch.Generator().manual_seed(43)
    B, Hkv, d, W = 2, 3, 4, 5
    ring_k, ring_v = np.zeros((B, Hkv, W, d)), np.zeros((B, Hkv, W, d))
    ring_pos = np.full((B, W), -1, dtype=np.int32)
    toks_k = torch.randn(B, Hkv, 23, d, generator=g).numpy()
    toks_v = torch.randn(B, Hkv, 23, d, generator=g).numpy()
    pos0 = np.array([0, 0])
    for n in (3, 1, 8, 4, 7):  # appends of varying size, wrapping the ring several times
        oracle.ring_append(toks_k[:, :, pos0[0]:pos0[0] + n], toks_v[:, :, pos0[0]:pos0[0] + n], ring_k, ring_v,
                           ring_pos, pos0)
        pos0 = pos0 + n
        held = np.sort(ring_pos, axis=1)
        want = np.arange(max(0, pos0[0] - W), pos0[0])
        assert np.array_equal(held[0][held[0] >= 0], want)
        for b in range(B):
            for s in range(W):
                if ring_pos[b, s] >= 0:
                    assert s == ring_pos[b, s] % W
                    np.testing.assert_array_equal(ring_k[b, :, s], toks_k[b, :, ring_pos[b, s]])
                    np.testing.assert_array_equal(ring_v[b, :, s], toks_v[b, :, ring_pos[b, s]])


# ----------------------------------------------------------------------------- pool as a cache


def _pool_state(pool_pos, T):
    slot_map = np.full((pool_pos.shape[0], T), -1, dtype=np.int32)
    for b in range(pool_pos.shape[0]):
        for s, t in enumerate(pool_pos[b]):
            if t >= 0:
                slot_map[b, t] = s
    return slot_map


def test_promote_hand_worked_example():
    gd = load_golden("promote_small.json")
    T, P = gd["T"], gd["P"]
    idx = np.array(gd["idx"], dtype=np.int32)
    pool_pos = np.array(gd["pool_pos_before"], dtype=np.int32)
    slot_map = _pool_state(pool_pos, T)
    hand = np.array(gd["hand_before"], dtype=np.int32)
    kh = np.arange(1 * 2 * T * 4, dtype=np.float64).reshape(1, 2, T, 4)
    vh = -kh
    kp, vp = np.zeros((1, 2, P, 4)), np.zeros((1, 2, P, 4))
    n = oracle.promote_rows(idx, gd["block"], slot_map, pool_pos, hand, kh, vh, kp, vp)
    assert n == gd["promoted"]
    np.testing.assert_array_equal(pool_pos, gd["pool_pos_after"])
    np.testing.assert_array_equal(slot_map, gd["slot_map_after"])
    np.testing.assert_array_equal(hand, gd["hand_after"])
    for s, t in enumerate(pool_pos[0]):
        if t in (1, 5, 10):
            np.testing.assert_array_equal(kp[0, :, s], kh[0, :, t])
            np.testing.assert_array_equal(vp[0, :, s], vh[0, :, t])
    assert oracle.promote_rows(idx, gd["block"], slot_map, pool_pos, hand, kh, vh, kp, vp) == [0]


def test_promote_invariants_under_random_drifting_selections():
    rng = np.random.default_rng(7)
    B, Hkv, T, P, n, blk, d = 3, 2, 400, 60, 9, 4, 2
    kh = rng.standard_normal((B, Hkv, T, d))
    vh = rng.standard_normal((B, Hkv, T, d))
    kp, vp = np.zeros((B, Hkv, P, d)), np.zeros((B, Hkv, P, d))
    pool_pos = np.full((B, P), -1, dtype=np.int32)
    slot_map = np.full((B, T), -1, dtype=np.int32)
    hand = np.zeros(B, dtype=np.int32)
    base = rng.permutation(T // blk)[:n]
    for step in range(12):
        idx = np.empty((B, Hkv, n), dtype=np.int32)
        for b in range(B):
            for h in range(Hkv):
                cur = base.copy()
                cur[rng.integers(0, n, 2)] = rng.integers(0, T // blk, 2)  # drift
                idx[b, h] = np.sort(cur)
        before = slot_map.copy()
        oracle.promote_rows(idx, blk, slot_map, pool_pos, hand, kh, vh, kp, vp)
        for b in range(B):
            sel = {int(e) * blk + o for h in range(Hkv) for e in idx[b, h] for o in range(blk)}
            # slot_map and pool_pos are inverse maps of the occupied slots
            assert all(slot_map[b, t] == s for s, t in enumerate(pool_pos[b]) if t >= 0)
            assert all(pool_pos[b, s] == t for t, s in enumerate(slot_map[b]) if s >= 0)
            # pool rows hold the host rows of their positions
            for s, t in enumerate(pool_pos[b]):
                if t >= 0:
                    np.testing.assert_array_equal(kp[b, :, s], kh[b, :, t])
                    np.testing.assert_array_equal(vp[b, :, s], vh[b, :, t])
            # a selected row resident before the step stays resident
            assert all(slot_map[b, t] >= 0 for t in sel if before[b, t] >= 0)
            # every selected row is resident unless every slot holds a selected row
            if len(sel) <= P:
                assert all(slot_map[b, t] >= 0 for t in sel)
            else:
                assert sum(slot_map[b, t] >= 0 for t in sel) == P
