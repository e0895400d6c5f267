"""Dense attention over a cache in HBM ("Nem Todos os Pensamentos Necessitam de HBM",
gist.science summary, Metodologia 2: every layer attends to every cached row and keeps its
logits for the importance score).  sd_gather_attend moves such calls' rows as whole 64-row
tiles through a ring of shared-memory stages, and the rows of selected blocks of 16 or more
rows (SparDA, gist.science summary: sec. 2 item 1, top-k blocks; "Estrategia de
Treinamento", the union of compression windows as 16-token segments) as 16-row boxes of
the same tiles; out and lse within 2e-3 max-abs and 1e-3
relative L2 of the fp64 oracle, the logits within 1e-4, and the row loop (row_loop = 1)
within the same tolerance of the tiled path.  Every call goes through the C ABI."""
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


def case(seed, B, V, Hq, Hkv, T):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, V, Hq, 128, generator=g).bfloat16()
    K = torch.randn(B, Hkv, T, 128, generator=g).bfloat16()
    Vv = torch.randn(B, Hkv, T, 128, generator=g).bfloat16()
    return q, K, Vv


@pytest.mark.parametrize("B,V,Hq,Hkv,T,splits,logits", [
    (1, 1, 8, 2, 1000, 0, True),      # ragged tail (1000 = 15 tiles + 40 rows), R = 4
    (2, 1, 28, 4, 4096, 0, True),     # R = 7, several splits per group
    (1, 4, 16, 4, 777, 0, True),      # R = 16: two query tiles of 8
    (1, 1, 4, 4, 64, 0, False),       # one tile, one query row per group
    (1, 1, 8, 2, 3000, 1, True),      # one split: out and lse written directly
    (2, 1, 8, 2, 3000, 5, False),     # five splits requested (ranges of whole tiles)
    (1, 2, 8, 1, 33, 0, True),        # fewer rows than one tile half
])
def test_dense_tiles_match_oracle(B, V, Hq, Hkv, T, splits, logits):
    q, K, Vv = case(B * 131 + V * 17 + Hq + T, B, V, Hq, Hkv, T)
    scale = 1.0 / math.sqrt(128)
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, lz = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), None, T=T, scale=scale, want_logits=logits,
                                      err_word=e, splits=splits)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    ro, rl, rz = oracle.gather_attend(q, K, Vv, None, B, V, Hq, Hkv, 128, T, T, 1, scale, True)
    assert_attend_close(out, ro, "out")
    assert_attend_close(lse, rl, "lse")
    if logits:
        np.testing.assert_allclose(lz.cpu().numpy(), rz, atol=1e-4, rtol=1e-5)


def test_dense_tiles_agree_with_the_row_loop():
    # the same call through the general row loop: the same values within rounding
    B, V, Hq, Hkv, T = 2, 1, 28, 4, 5000
    q, K, Vv = case(77, B, V, Hq, Hkv, T)
    dev = [q.cuda(), K.cuda(), Vv.cuda()]
    o0, l0, z0 = sd().gather_attend(*dev, None, T=T, want_logits=True)
    o1, l1, z1 = sd().gather_attend(*dev, None, T=T, want_logits=True, row_loop=True)
    torch.cuda.synchronize()
    assert_attend_close(o0, o1.cpu().double().numpy(), "out")
    assert_attend_close(l0, l1.cpu().double().numpy(), "lse")
    np.testing.assert_allclose(z0.cpu().numpy(), z1.cpu().numpy(), atol=1e-4, rtol=1e-5)


def test_dense_tiles_at_the_importance_scoring_size():
    # one layer of the importance-scoring workload (B 2, 28 query heads over 4 KV heads,
    # T 65536): sampled query rows against the oracle, every logit row's softmax sums to one
    B, V, Hq, Hkv, T = 2, 1, 28, 4, 65536
    q, K, Vv = case(2024, B, V, Hq, Hkv, T)
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, lz = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), None, T=T, want_logits=True, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    w = torch.exp(lz.double() - lse.double()[..., None]).sum(-1)
    assert torch.allclose(w, torch.ones_like(w), atol=1e-5)
    for b, h in ((0, 0), (1, 27), (1, 13)):
        kvh = h // (Hq // Hkv)
        ro, rl, rz = oracle.gather_attend(q[b:b + 1, :, h:h + 1].contiguous(), K[b:b + 1, kvh:kvh + 1].contiguous(),
                                          Vv[b:b + 1, kvh:kvh + 1].contiguous(), None, 1, V, 1, 1, 128, T, T, 1,
                                          1.0 / math.sqrt(128), True)
        assert_attend_close(out[b:b + 1, :, h:h + 1], ro, "out")
        assert_attend_close(lse[b:b + 1, :, h:h + 1], rl, "lse")
        np.testing.assert_allclose(lz[b:b + 1, :, h:h + 1].cpu().numpy(), rz, atol=1e-4, rtol=1e-5)


# --------------------------------------------------------------------------- block-sparse tiles
# Calls with an index list whose blocks hold whole 16-row sub-tiles (block a multiple of 16,
# T a multiple of block, no logits) take the same tiles: each stage is four 16-row boxes at
# the selected blocks' rows.  Same tolerance against the oracle and against the row loop.

def block_idx(seed, B, Hkv, nb, n, empty):
    """Sorted distinct blocks per (b, kvh); empty slots (-1) at the list's end ("tail", the
    window union's padding), in its middle ("mid"), or one group's whole list ("group")."""
    g = torch.Generator().manual_seed(seed)
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(nb, generator=g)[:n]).values for _ in range(Hkv)])
                       for _ in range(B)]).int()
    if empty == "tail":
        idx[..., n - n // 4:] = -1
    elif empty == "mid":
        idx[..., 1::3] = -1
    elif empty == "group":
        idx[0, 1] = -1
    return idx


@pytest.mark.parametrize("B,V,Hq,Hkv,T,n,block,splits,empty", [
    (2, 1, 32, 8, 4096, 40, 16, 0, "tail"),   # 16-row segments padded with -1 (window union layout)
    (1, 2, 8, 2, 8192, 64, 64, 0, "mid"),     # blocks of 64, R = 8, empty slots between blocks
    (1, 1, 28, 4, 2048, 7, 32, 1, "none"),    # one split: out and lse written directly, R = 7
    (2, 4, 16, 4, 1024, 9, 16, 3, "mid"),     # R = 16 (two query tiles), three splits, 144-row lists
    (1, 1, 8, 2, 512, 32, 16, 0, "none"),     # every block selected
    (1, 1, 8, 2, 1024, 8, 16, 0, "group"),    # one group without rows: out 0, lse -inf
])
def test_block_tiles_match_oracle(B, V, Hq, Hkv, T, n, block, splits, empty):
    q, K, Vv = case(T + n * 7 + block + B, B, V, Hq, Hkv, T)
    idx = block_idx(T + n, B, Hkv, T // block, n, empty)
    scale = 1.0 / math.sqrt(128)
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = [q.cuda(), K.cuda(), Vv.cuda(), idx.cuda()]
    out, lse, _ = sd().gather_attend(*dev, n_idx=n, block=block, T=T, scale=scale, err_word=e, splits=splits)
    o1, l1, _ = sd().gather_attend(*dev, n_idx=n, block=block, T=T, scale=scale, splits=splits, row_loop=True)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    ro, rl, _ = oracle.gather_attend(q, K, Vv, idx.numpy(), B, V, Hq, Hkv, 128, T, n, block, scale)
    assert_attend_close(out, ro, "out")
    assert_attend_close(lse, rl, "lse")
    assert_attend_close(out, o1.cpu().double().numpy(), "out vs row loop")
    assert_attend_close(lse, l1.cpu().double().numpy(), "lse vs row loop")
    if empty == "group":
        assert torch.all(out[0, :, 4:8] == 0) and torch.all(torch.isneginf(lse[0, :, 4:8]))


def test_block_tiles_report_bad_indices():
    # an index past the cache or below -1 is reported and its rows left out, as in the row loop
    B, V, Hq, Hkv, T, n, block = 1, 1, 8, 2, 2048, 16, 32
    q, K, Vv = case(5, B, V, Hq, Hkv, T)
    idx = block_idx(6, B, Hkv, T // block, n, "none")
    bad = idx.clone()
    bad[0, 0, 3] = T // block
    bad[0, 1, 9] = -7
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), bad.cuda(), n_idx=n, block=block, T=T, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) & sd().SD_DEVERR_INDEX
    ref_idx = idx.clone()
    ref_idx[0, 0, 3] = -1
    ref_idx[0, 1, 9] = -1
    ro, rl, _ = oracle.gather_attend(q, K, Vv, ref_idx.numpy(), B, V, Hq, Hkv, 128, T, n, block, 1.0 / math.sqrt(128))
    assert_attend_close(out, ro, "out")
    assert_attend_close(lse, rl, "lse")


def test_block_tiles_at_the_window_size():
    # the compression-window layer's attention: 64 groups of 4 query rows over up to 128
    # segments of 16 tokens (T 32768), the union's padding at the end; sampled groups
    B, V, Hq, Hkv, T, n, block = 8, 1, 32, 8, 32768, 128, 16
    q, K, Vv = case(606, B, V, Hq, Hkv, T)
    g = torch.Generator().manual_seed(607)
    idx = torch.full((B, Hkv, n), -1, dtype=torch.int32)
    for b in range(B):
        for h in range(Hkv):
            m = int(torch.randint(60, n + 1, (1,), generator=g))
            idx[b, h, :m] = torch.sort(torch.randperm(T // block, generator=g)[:m]).values.int()
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), idx.cuda(), n_idx=n, block=block, T=T, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    for b, h in ((0, 0), (3, 5), (7, 7)):
        sl = slice(h * 4, h * 4 + 4)
        ro, rl, _ = oracle.gather_attend(q[b:b + 1, :, sl].contiguous(), K[b:b + 1, h:h + 1].contiguous(),
                                          Vv[b:b + 1, h:h + 1].contiguous(), idx[b:b + 1, h:h + 1].numpy(), 1, V, 4,
                                          1, 128, T, n, block, 1.0 / math.sqrt(128))
        assert_attend_close(out[b:b + 1, :, sl], ro, "out")
        assert_attend_close(lse[b:b + 1, :, sl], rl, "lse")
