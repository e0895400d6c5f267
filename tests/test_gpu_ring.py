"""The draft tokens' window-bounded ring: sd_ring_append bit-exact against the oracle's
append (wrapping the ring), and sd_gather_attend with a ring -- the selected history rows
plus the ring slots at or before each query token's position -- against the oracle within
the attention tolerance, with the masked logits exactly -inf.  Also with per-head
selections, host-resident history rows (direct and staged) and every attention path."""
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


@pytest.mark.parametrize("dt,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_ring_append_matches_the_oracle(dt, d):
    g = torch.Generator().manual_seed(3)
    B, Hkv, W = 3, 2, 10
    rk, rv, rpos = sd().ring_buffers(B, Hkv, W, d, dt)
    ok, ov = np.zeros((B, Hkv, W, d), np.float32), np.zeros((B, Hkv, W, d), np.float32)
    opos = np.full((B, W), -1, np.int32)
    pos0 = np.array([0, 5, 17], np.int32)
    for n in (4, 10, 1, 7, 9):
        kn = torch.randn(B, Hkv, n, d, generator=g).to(dt)
        vn = torch.randn(B, Hkv, n, d, generator=g).to(dt)
        sd().sd_ring_append(kn.cuda(), vn.cuda(), rk, rv, rpos, torch.from_numpy(pos0).cuda())
        oracle.ring_append(kn.float().numpy(), vn.float().numpy(), ok, ov, opos, pos0)
        pos0 = pos0 + n
        torch.cuda.synchronize()
        np.testing.assert_array_equal(rpos.cpu().numpy(), opos)
        np.testing.assert_array_equal(rk.float().cpu().numpy(), ok)
        np.testing.assert_array_equal(rv.float().cpu().numpy(), ov)


def _verify_case(seed, B, V, Hq, Hkv, d, T, n, block, W, dt, per_head=False, empty=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, V, Hq, d, generator=g).to(dt)
    K = torch.randn(B, Hkv, T, d, generator=g).to(dt)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(dt)
    groups = Hq if per_head else Hkv
    idx = torch.full((B, groups, n), -1, dtype=torch.int32)
    for b in range(B):
        for h in range(groups):
            m = n - (empty if (b + h) % 2 == 0 else 0)
            idx[b, h, :m] = torch.sort(torch.randperm(T // block, generator=g)[:m]).values
    rk = torch.randn(B, Hkv, W, d, generator=g).to(dt)
    rv = torch.randn(B, Hkv, W, d, generator=g).to(dt)
    # the ring: recent accepted tokens before T, then the V draft tokens at T..T+V-1, in
    # ring order (slot = position mod W); sequence 1 leaves two slots empty
    rpos = torch.full((B, W), -1, dtype=torch.int32)
    for b in range(B):
        first = T + V - W + (2 if b == 1 else 0)
        for t in range(first, T + V):
            rpos[b, t % W] = t
    qpos = torch.stack([torch.arange(T, T + V) for _ in range(B)]).to(torch.int32)
    return q, K, Vv, idx, rk, rv, rpos, qpos


@pytest.mark.parametrize("dt,d,V,block,W,per_head,dense", [
    (torch.bfloat16, 128, 8, 1, 64, False, False), (torch.bfloat16, 128, 1, 1, 16, False, False),
    (torch.bfloat16, 64, 4, 16, 24, False, False), (torch.float32, 128, 8, 1, 40, False, False),
    (torch.float32, 64, 2, 1, 8, False, True), (torch.bfloat16, 128, 4, 1, 32, True, False),
    (torch.bfloat16, 128, 8, 1, 700, False, False),
])
def test_gather_attend_with_a_draft_ring(dt, d, V, block, W, per_head, dense):
    B, Hq, Hkv, T = 2, 16, 4, 2048
    n = T // block if dense else 300 // block
    q, K, Vv, idx, rk, rv, rpos, qpos = _verify_case(V * 31 + W, B, V, Hq, Hkv, d, T, n, block, W, dt, per_head,
                                                     empty=0 if dense else 3)
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, z = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), None if dense else idx.cuda(), n_idx=n,
                                     block=block, T=T, want_logits=True, err_word=e, per_head=per_head,
                                     ring_k=rk.cuda(), ring_v=rv.cuda(), ring_pos=rpos.cuda(), qpos=qpos.cuda())
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    if per_head:  # the oracle takes one shared selection per KV head: compare head by head
        G = Hq // Hkv
        for h in range(Hq):
            kvh = h // G
            ro, rl, rz = oracle.gather_attend_ring(q[:, :, h:h + 1].contiguous(), K[:, kvh:kvh + 1].contiguous(),
                                                   Vv[:, kvh:kvh + 1].contiguous(), idx[:, h:h + 1].numpy(), B, V, 1,
                                                   1, d, T, n, block, 1 / math.sqrt(d), rk[:, kvh:kvh + 1],
                                                   rv[:, kvh:kvh + 1], rpos.numpy(), qpos.numpy(), True)
            assert_attend_close(out[:, :, h:h + 1], ro)
            assert_attend_close(lse[:, :, h:h + 1], rl, "lse")
            _check_logits(z[:, :, h:h + 1], rz)
        return
    ro, rl, rz = oracle.gather_attend_ring(q, K, Vv, None if dense else idx.numpy(), B, V, Hq, Hkv, d, T, n, block,
                                           1 / math.sqrt(d), rk, rv, rpos.numpy(), qpos.numpy(), True)
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")
    _check_logits(z, rz)


def _check_logits(z, rz):
    lz = z.cpu().numpy()
    assert np.array_equal(np.isneginf(lz), np.isneginf(rz)), "masked rows must be exactly -inf"
    fin = np.isfinite(rz)
    np.testing.assert_allclose(lz[fin], rz[fin], atol=1e-4, rtol=1e-5)


def test_ring_with_host_rows_direct_and_staged():
    from top_sparse_decode_gqa_gb300.workloads import residency_map
    B, V, Hq, Hkv, d, T, n, W = 2, 8, 32, 8, 128, 4096, 512, 64
    q, K, Vv, idx, rk, rv, rpos, qpos = _verify_case(77, B, V, Hq, Hkv, d, T, n, 1, W, torch.bfloat16)
    P = T // 10
    res, slot_map = residency_map(B, T, P, 5)
    gi = res[:, None, :, None].expand(B, Hkv, P, d)
    keep = [q.cuda(), torch.gather(K, 2, gi).contiguous().cuda(), torch.gather(Vv, 2, gi).contiguous().cuda(),
            idx.cuda(), K.pin_memory(), Vv.pin_memory(), slot_map.cuda(), rk.cuda(), rv.cuda(), rpos.cuda(),
            qpos.cuda()]
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, out, lse, _ = sd().make_attend_args(keep[0], keep[1], keep[2], keep[3], T=T, k_host=keep[4], v_host=keep[5],
                                           slot_map=keep[6], err_word=e, ring_k=keep[7], ring_v=keep[8],
                                           ring_pos=keep[9], qpos=keep[10])
    ws = torch.zeros(max(16, sd().sd_gather_attend_workspace_bytes(a)), dtype=torch.uint8, device="cuda")
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    o_direct, l_direct = out.clone(), lse.clone()
    stage = sd().stage_buffers(a, torch.bfloat16)
    sd().sd_stage_host_rows(a, sd().stage_counter())
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    assert torch.equal(out, o_direct) and torch.equal(lse, l_direct)
    # and all rows in HBM: the same bits again
    o2, l2, _ = sd().gather_attend(keep[0], K.cuda(), Vv.cuda(), keep[3], T=T, ring_k=keep[7], ring_v=keep[8],
                                   ring_pos=keep[9], qpos=keep[10])
    assert torch.equal(o2, o_direct) and torch.equal(l2, l_direct)
    ro, rl, _ = oracle.gather_attend_ring(q, K, Vv, idx.numpy(), B, V, Hq, Hkv, d, T, n, 1, 1 / math.sqrt(d), rk, rv,
                                          rpos.numpy(), qpos.numpy())
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")
    del stage


def test_empty_ring_is_plain_attention():
    B, V, Hq, Hkv, d, T, n, W = 2, 4, 16, 4, 128, 2048, 256, 32
    q, K, Vv, idx, rk, rv, rpos, qpos = _verify_case(9, B, V, Hq, Hkv, d, T, n, 1, W, torch.bfloat16)
    rpos.fill_(-1)
    o1, l1, _ = sd().gather_attend(q.cuda(), K.cuda(), Vv.cuda(), idx.cuda(), T=T, ring_k=rk.cuda(), ring_v=rv.cuda(),
                                   ring_pos=rpos.cuda(), qpos=qpos.cuda())
    ro, rl, _ = oracle.gather_attend(q, K, Vv, idx.numpy(), B, V, Hq, Hkv, d, T, n, 1, 1 / math.sqrt(d))
    assert_attend_close(o1, ro)
    assert_attend_close(l1, rl, "lse")


def test_c8_verify_layer_group_full():
    # the benchmark's verify workload at full size, in its launch sequence: one indexer pass
    # and one top-k for the layer group, then per layer the drafts appended to the layer's
    # ring and the attention over the selected rows plus the ring
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c8_verify_layer_group"]
    x = generate(w)
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = sd().key_hist_buffer(w.B * w.Hkv)
    s = sd().sd_index_score(x["q_idx"].cuda(), x["k_idx"].cuda(), err_word=e, key_hist=hist)
    idx = sd().sd_topk(s, w.k, key_hist=hist)
    qpos, pos0 = x["qpos"].cuda(), torch.full((w.B,), w.T, dtype=torch.int32, device="cuda")
    outs = []
    for layer in range(w.layers):
        rk, rv = x["ring_k"][layer].cuda(), x["ring_v"][layer].cuda()
        rp = x["ring_pos"].cuda()
        sd().sd_ring_append(x["draft_k"][layer].cuda(), x["draft_v"][layer].cuda(), rk, rv, rp, pos0)
        out, lse, _ = sd().gather_attend(x["q"][0, layer].cuda(), x["k"][layer].cuda(), x["v"][layer].cuda(), idx,
                                         T=w.T, err_word=e, ring_k=rk, ring_v=rv, ring_pos=rp, qpos=qpos)
        outs.append((out.cpu(), lse.cpu(), rp.cpu()))
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    ri = oracle.topk(oracle.index_score(x["q_idx"], x["k_idx"], w.B, w.Hkv, w.V, w.T, w.dI), w.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ri)
    for layer in range(w.layers):
        rk = x["ring_k"][layer].float().numpy().copy()
        rv = x["ring_v"][layer].float().numpy().copy()
        rp = x["ring_pos"].numpy().copy()
        oracle.ring_append(x["draft_k"][layer].float().numpy(), x["draft_v"][layer].float().numpy(), rk, rv, rp,
                           [w.T] * w.B)
        np.testing.assert_array_equal(outs[layer][2].numpy(), rp)
        ro, rl, _ = oracle.gather_attend_ring(x["q"][0, layer], x["k"][layer], x["v"][layer], ri, w.B, w.V, w.Hq,
                                              w.Hkv, w.d, w.T, w.k, 1, 1 / math.sqrt(w.d),
                                              torch.from_numpy(rk).to(torch.bfloat16),
                                              torch.from_numpy(rv).to(torch.bfloat16), rp, x["qpos"].numpy())
        assert_attend_close(outs[layer][0], ro)
        assert_attend_close(outs[layer][1], rl, "lse")
