"""Parity of sd_decode_step (indexer, top-k and gather-attend in one persistent launch) with
the CPU oracle: scores and index sets bit-exact, attention within 2e-3 max-abs and 1e-3
relative L2 of the fp64 oracle.  Cases span many scoring tiles and attention tasks with
ragged tails, token and block selection (whole 64-row blocks moved by tiled TMA, and
16-row blocks moved row by row), verify batches, heavy ties (the selection's overflow
path), the empty and the full selection, repeated calls on one workspace, and a bounded
wait that is made to run out.  Every call goes through the C ABI."""
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


def rint(g, shape, dtype, lo=-8, hi=8):
    return torch.randint(lo, hi + 1, shape, generator=g).float().to(dtype)


def make_inputs(B, Hkv, G, V, T, block, seed, kdt=torch.bfloat16, key_lo=-8, key_hi=8):
    g = torch.Generator().manual_seed(seed)
    N = T // block
    Hq = Hkv * G
    q_idx = rint(g, (B, Hkv, V, 128), kdt)
    keys = rint(g, (B, Hkv, N, 128), kdt, key_lo, key_hi)
    q = torch.randn(B, V, Hq, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, T, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, T, 128, generator=g).to(torch.bfloat16)
    return q_idx, keys, q, k, v


def check_against_oracle(inp, B, Hkv, G, V, T, block, kk, scores, idx, out, lse):
    q_idx, keys, q, k, v = inp
    N = T // block
    Hq = Hkv * G
    rs = oracle.index_score(q_idx, keys, B, Hkv, V, N, 128)
    np.testing.assert_array_equal(scores.cpu().numpy().astype(np.float64), rs)
    ri = oracle.topk(rs, kk)
    np.testing.assert_array_equal(idx.cpu().numpy(), ri)
    ro, rl, _ = oracle.gather_attend(q, k, v, ri, B, V, Hq, Hkv, 128, T, kk, block, 1 / math.sqrt(128))
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")


@pytest.mark.parametrize("B,Hkv,G,V,T,block,kk,kdt,lag", [
    (2, 2, 4, 1, 1000, 1, 100, torch.bfloat16, 0),     # ragged tiles, a tail stage of 36 rows
    (1, 3, 4, 1, 1004, 1, 257, torch.bfloat16, 0),     # a 1-row attention task tail
    (2, 2, 4, 4, 3000, 1, 300, torch.bfloat16, 0),     # verify batch: 16 query rows per group
    (1, 2, 2, 8, 700, 1, 64, torch.bfloat16, 1),       # V = 8, lag 1
    (2, 4, 4, 1, 64 * 300, 64, 20, torch.float16, 0),  # whole 64-row blocks (tiled TMA), fp16 keys
    (1, 2, 4, 2, 64 * 76, 64, 76, torch.float16, 2),   # every block selected
    (2, 2, 4, 1, 16 * 900, 16, 70, torch.bfloat16, 0),  # 16-row blocks, row by row
    (1, 1, 8, 1, 128 * 40, 128, 9, torch.bfloat16, 0),  # 128-row blocks: two TMA runs each
    (3, 8, 4, 1, 9000, 1, 1024, torch.bfloat16, 0),    # many groups and tasks in flight
    (1, 1, 1, 1, 4, 1, 1, torch.bfloat16, 0),          # four tokens, one selected
    # block selection over short score rows: one thread-block cluster per KV group
    (2, 8, 4, 1, 32 * 2048, 32, 64, torch.float16, 0),  # 16 groups: clusters of 8, one CTA per SM
    (5, 8, 4, 1, 32 * 1000, 32, 40, torch.bfloat16, 0),  # 40 groups: clusters of 4, two CTAs per SM
    (40, 8, 4, 1, 16 * 64, 16, 12, torch.bfloat16, 0),  # 320 groups: single CTAs, several waves
    (1, 2, 4, 4, 32 * 516, 32, 33, torch.bfloat16, 0),  # 16 query rows, ragged shares and list
    (1, 1, 4, 1, 16 * 8196, 16, 50, torch.bfloat16, 0),  # N > 8192: the persistent kernel's block path
])
def test_decode_step_matches_oracle(B, Hkv, G, V, T, block, kk, kdt, lag):
    inp = make_inputs(B, Hkv, G, V, T, block, seed=B * 7919 + T + kk, kdt=kdt)
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = [t.cuda() for t in inp]
    scores, idx, out, lse = sd().decode_step(*dev, kk, block=block, err_word=e, lag=lag)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    check_against_oracle(inp, B, Hkv, G, V, T, block, kk, scores, idx, out, lse)


@pytest.mark.parametrize("key_lo,key_hi,T,kk", [
    (0, 0, 5000, 300),     # every score 0: one bin holds all (candidate overflow), ties by index
    (-1, 1, 6000, 1500),   # few distinct values: heavy ties at the threshold
    (0, 0, 700, 10),       # all equal, few entries: ties resolved among candidates
])
def test_decode_step_ties(key_lo, key_hi, T, kk):
    B, Hkv, G, V = 2, 2, 4, 1
    inp = make_inputs(B, Hkv, G, V, T, 1, seed=T + kk, key_lo=key_lo, key_hi=key_hi)
    dev = [t.cuda() for t in inp]
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    scores, idx, out, lse = sd().decode_step(*dev, kk, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    check_against_oracle(inp, B, Hkv, G, V, T, 1, kk, scores, idx, out, lse)


@pytest.mark.parametrize("key_lo,key_hi,N,kk", [
    (0, 0, 600, 37),     # every block score equal: the lowest 37 indices
    (-1, 1, 2000, 300),  # few distinct values: heavy ties at the threshold
])
def test_decode_step_block_ties(key_lo, key_hi, N, kk):
    B, Hkv, G, V, block = 2, 4, 4, 1, 32
    inp = make_inputs(B, Hkv, G, V, N * block, block, seed=N + kk, key_lo=key_lo, key_hi=key_hi)
    dev = [t.cuda() for t in inp]
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    scores, idx, out, lse = sd().decode_step(*dev, kk, block=block, err_word=e)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    check_against_oracle(inp, B, Hkv, G, V, N * block, block, kk, scores, idx, out, lse)


def test_decode_step_block_empty_and_full_selection():
    B, Hkv, G, V, block, N = 1, 2, 4, 2, 64, 40
    inp = make_inputs(B, Hkv, G, V, N * block, block, seed=8)
    dev = [t.cuda() for t in inp]
    scores, idx, out, lse = sd().decode_step(*dev, 0, block=block)
    torch.cuda.synchronize()
    assert idx.numel() == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    np.testing.assert_array_equal(scores.cpu().numpy().astype(np.float64),
                                  oracle.index_score(inp[0], inp[1], B, Hkv, V, N, 128))
    scores, idx, out, lse = sd().decode_step(*dev, N, block=block)
    torch.cuda.synchronize()
    check_against_oracle(inp, B, Hkv, G, V, N * block, block, N, scores, idx, out, lse)


def test_decode_step_empty_and_full_selection():
    B, Hkv, G, V, T = 1, 2, 4, 1, 600
    inp = make_inputs(B, Hkv, G, V, T, 1, seed=3)
    dev = [t.cuda() for t in inp]
    # k = 0: no rows, out = 0 and lse = -inf
    scores, idx, out, lse = sd().decode_step(*dev, 0)
    torch.cuda.synchronize()
    assert idx.numel() == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    np.testing.assert_array_equal(scores.cpu().numpy().astype(np.float64),
                                  oracle.index_score(inp[0], inp[1], B, Hkv, V, T, 128))
    # k = N: every token, i.e. dense attention
    scores, idx, out, lse = sd().decode_step(*dev, T)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), np.broadcast_to(np.arange(T, dtype=np.int32), (B, Hkv, T)))
    check_against_oracle(inp, B, Hkv, G, V, T, 1, T, scores, idx, out, lse)


def test_decode_step_repeated_calls_share_one_workspace():
    # every call leaves the workspace ready for the next: calls of one shape, then of another,
    # reuse it without clearing
    B, Hkv, G, V = 2, 2, 4, 1
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    for r, (T, kk) in enumerate([(3000, 200), (3000, 200), (5000, 999), (1000, 64)]):
        inp = make_inputs(B, Hkv, G, V, T, 1, seed=100 + r)
        dev = [t.cuda() for t in inp]
        scores, idx, out, lse = sd().decode_step(*dev, kk, workspace=ws, err_word=e)
        torch.cuda.synchronize()
        assert int(e.item()) == 0
        check_against_oracle(inp, B, Hkv, G, V, T, 1, kk, scores, idx, out, lse)
    # the task counter, the per-group counters and the histograms (the workspace's first 256 +
    # 256 + B*Hkv*8192 bytes) are back at zero; the attention partials after them are scratch
    assert int(torch.count_nonzero(ws[:512 + B * Hkv * 8192]).item()) == 0


def test_decode_step_lag_does_not_change_the_result():
    B, Hkv, G, V, T, kk = 2, 4, 4, 1, 4000, 300
    inp = make_inputs(B, Hkv, G, V, T, 1, seed=11)
    dev = [t.cuda() for t in inp]
    res = [sd().decode_step(*dev, kk, lag=lag) for lag in (1, 3, B * Hkv)]
    torch.cuda.synchronize()
    for r in res[1:]:
        for a, b in zip(res[0], r):
            assert torch.equal(a, b)
    check_against_oracle(inp, B, Hkv, G, V, T, 1, kk, *res[0])


def test_decode_step_bounded_wait_runs_out():
    # A group's scoring counter is preset so that its last scoring task is never recognised:
    # its selection never runs, and every attention task of the group waits on a flag nothing
    # sets.  With a 2 ms wait limit the kernel reports SD_DEVERR_TIMEOUT and returns; the
    # stream stays usable, and with the workspace zero-filled again the next call is correct.
    B, Hkv, G, V, T, kk = 1, 2, 4, 1, 2000, 100
    inp = make_inputs(B, Hkv, G, V, T, 1, seed=5)
    dev = [t.cuda() for t in inp]
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, scores, idx, out, lse = sd().make_decode_step_args(*dev, kk, err_word=e, wait_limit_ns=2_000_000)
    ws = sd().decode_step_workspace(a)
    gstate = ws[256:256 + 16].view(torch.int32)   # group 0: scoring tasks done, attention done, ready
    gstate[0] = 1 << 20
    sd().sd_decode_step(a)
    torch.cuda.synchronize()
    assert int(e.item()) & sd().SD_DEVERR_TIMEOUT
    # the context is intact: the same call on a clean workspace matches the oracle
    ws.zero_()
    e.zero_()
    sd().sd_decode_step(a)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    check_against_oracle(inp, B, Hkv, G, V, T, 1, kk, scores, idx, out, lse)


def test_decode_step_rejects_unsupported():
    inp = make_inputs(1, 1, 4, 1, 100, 1, seed=1)
    dev = [t.cuda() for t in inp]
    with pytest.raises(sd().SdError):
        sd().decode_step(*dev, 101)  # k > N
    q_idx, keys, q, k, v = dev
    with pytest.raises(sd().SdError):  # 32 query rows per group
        sd().decode_step(q_idx, keys, torch.zeros(1, 1, 32, 128, dtype=torch.bfloat16, device="cuda"), k, v, 10)
    inp = make_inputs(1, 1, 4, 1, 102, 1, seed=2)  # T / block not a multiple of 4
    with pytest.raises(sd().SdError):
        sd().decode_step(*[t.cuda() for t in inp], 10)
