"""The HBM pool kept as a cache (sd_promote_rows): over several steps of drifting
selections the device's slot map, reverse map, hand and pool rows equal the oracle's
after every step, bit for bit; the attention over promoted rows gives the same bits as over
the same rows read from host memory; and the full-size tiered verify workload promotes
its selection.  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import oracle

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


def _drift(rng, base, n, n_blocks, groups, B):
    idx = np.empty((B, groups, n), dtype=np.int32)
    for b in range(B):
        for h in range(groups):
            cur = base.copy()
            k = rng.integers(1, 4)
            cur[rng.integers(0, n, k)] = rng.integers(0, n_blocks, k)
            cur = np.unique(cur)
            row = np.full(n, -1, dtype=np.int32)  # duplicates removed: the tail stays empty
            row[:len(cur)] = cur
            idx[b, h] = row
    return idx


@pytest.mark.parametrize("T,P,n,block,per_head", [(2000, 60, 9, 4, False), (4096, 300, 64, 1, False),
                                                  (1000, 50, 12, 1, True), (640, 8, 5, 2, False)])
def test_promotion_matches_the_oracle_over_drifting_steps(T, P, n, block, per_head):
    rng = np.random.default_rng(T + P)
    B, Hq, Hkv, d = 3, 8, 2, 128
    groups = Hq if per_head else Hkv
    kh = torch.randn(B, Hkv, T, d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    vh = torch.randn(B, Hkv, T, d, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    k_host, v_host = kh.pin_memory(), vh.pin_memory()
    k_pool = torch.zeros(B, Hkv, P, d, dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    slot_map = torch.full((B, T), -1, dtype=torch.int32, device="cuda")
    pool_pos, hand = sd().pool_state(slot_map, P)
    q = torch.zeros(B, 1, Hq, d, dtype=torch.bfloat16, device="cuda")
    # the oracle's copy of the state
    o_slot = np.full((B, T), -1, dtype=np.int32)
    o_pos = np.full((B, P), -1, dtype=np.int32)
    o_hand = np.zeros(B, dtype=np.int32)
    o_kp = np.zeros((B, Hkv, P, d), dtype=np.float32)
    o_vp = np.zeros((B, Hkv, P, d), dtype=np.float32)
    khf, vhf = kh.float().numpy(), vh.float().numpy()
    base = rng.permutation(T // block)[:n].astype(np.int32)
    ws = None
    for step in range(6):
        idx_np = _drift(rng, base, n, T // block, groups, B)
        idx = torch.from_numpy(idx_np).cuda()
        a, _, _, _ = sd().make_attend_args(q, k_pool, v_pool, idx, block=block, T=T, k_host=k_host, v_host=v_host,
                                           slot_map=slot_map, per_head=per_head)
        ws = sd().sd_promote_rows(a, pool_pos, hand, ws)
        torch.cuda.synchronize()
        # (with per-head selections the union over the query heads is what is promoted)
        oracle.promote_rows(idx_np, block, o_slot, o_pos, o_hand, khf, vhf, o_kp, o_vp)
        np.testing.assert_array_equal(slot_map.cpu().numpy(), o_slot, err_msg=f"step {step}")
        np.testing.assert_array_equal(pool_pos.cpu().numpy(), o_pos)
        np.testing.assert_array_equal(hand.cpu().numpy(), o_hand)
        occ = o_pos >= 0
        kp, vp = k_pool.float().cpu().numpy(), v_pool.float().cpu().numpy()
        for b in range(B):
            np.testing.assert_array_equal(kp[b][:, occ[b]], o_kp[b][:, occ[b]])
            np.testing.assert_array_equal(vp[b][:, occ[b]], o_vp[b][:, occ[b]])


@pytest.mark.parametrize("T,P,n,block,per_head", [(2000, 60, 9, 4, False), (4096, 300, 64, 1, False),
                                                  (1000, 50, 12, 1, True)])
def test_staged_promotion_matches_the_oracle(T, P, n, block, per_head):
    # per (b, KV head) units: each step stages the misses, attends, then promotes them from
    # the stage; the state and the pool rows equal the oracle's promotion of the same
    # selections, and the attention equals the one over the host rows
    import math
    rng = np.random.default_rng(T + P + 1)
    B, Hq, Hkv, d, V = 3, 8, 2, 128, 1
    G = Hq // Hkv
    groups = Hq if per_head else Hkv
    kh = torch.randn(B, Hkv, T, d, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    vh = torch.randn(B, Hkv, T, d, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    k_host, v_host = kh.pin_memory(), vh.pin_memory()
    k_pool = torch.zeros(B, Hkv, P, d, dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    slot_map = torch.full((B, Hkv, T), -1, dtype=torch.int32, device="cuda")
    pool_pos, hand = sd().pool_state(slot_map, P)
    q = torch.randn(B, V, Hq, d, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    U = B * Hkv
    o_slot = np.full((U, T), -1, dtype=np.int32)
    o_pos = np.full((U, P), -1, dtype=np.int32)
    o_hand = np.zeros(U, dtype=np.int32)
    o_kp = np.zeros((U, 1, P, d), dtype=np.float32)
    o_vp = np.zeros((U, 1, P, d), dtype=np.float32)
    khf, vhf = kh.float().numpy().reshape(U, 1, T, d), vh.float().numpy().reshape(U, 1, T, d)
    base = rng.permutation(T // block)[:n].astype(np.int32)
    ws = None
    counter = sd().stage_counter()
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(6):
        idx_np = _drift(rng, base, n, T // block, groups, B)
        idx = torch.from_numpy(idx_np).cuda()
        a, out, lse, _ = sd().make_attend_args(q, k_pool, v_pool, idx, block=block, T=T, k_host=k_host,
                                               v_host=v_host, slot_map=slot_map, per_head=per_head, err_word=e)
        assert a.slot_per_head == 1
        stage = sd().stage_buffers(a, torch.bfloat16)
        sd().sd_stage_host_rows(a, counter)
        gws = torch.zeros(max(16, sd().sd_gather_attend_workspace_bytes(a)), dtype=torch.uint8, device="cuda")
        sd().sd_gather_attend(a, gws)
        ws = sd().sd_promote_staged_rows(a, pool_pos, hand, ws)
        torch.cuda.synchronize()
        assert int(e.item()) == 0
        oracle.promote_rows(idx_np.reshape(U, groups // Hkv, n), block, o_slot, o_pos, o_hand, khf, vhf, o_kp, o_vp)
        np.testing.assert_array_equal(slot_map.cpu().numpy().reshape(U, T), o_slot, err_msg=f"step {step}")
        np.testing.assert_array_equal(pool_pos.cpu().numpy(), o_pos)
        np.testing.assert_array_equal(hand.cpu().numpy(), o_hand)
        occ = o_pos >= 0
        kp = k_pool.float().cpu().numpy().reshape(U, 1, P, d)
        vp = v_pool.float().cpu().numpy().reshape(U, 1, P, d)
        for u in range(U):
            np.testing.assert_array_equal(kp[u][:, occ[u]], o_kp[u][:, occ[u]])
            np.testing.assert_array_equal(vp[u][:, occ[u]], o_vp[u][:, occ[u]])
        if step == 5 and not per_head:  # the attention of the last step against the oracle
            from gpu_util import assert_attend_close
            ro, rl, _ = oracle.gather_attend(q.cpu(), kh, vh, idx_np, B, V, Hq, Hkv, d, T, n, block,
                                             1 / math.sqrt(d))
            assert_attend_close(out, ro)
            assert_attend_close(lse, rl, "lse")
        del stage


def test_attention_over_promoted_rows_is_the_same():
    from top_sparse_decode_gqa_gb300.workloads import residency_map
    g = torch.Generator().manual_seed(5)
    B, Hq, Hkv, d, T, n, V = 2, 16, 4, 128, 4096, 200, 2
    q = torch.randn(B, V, Hq, d, generator=g).to(torch.bfloat16).cuda()
    K = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(T, generator=g)[:n]).values for _ in range(Hkv)])
                       for _ in range(B)]).int().cuda()
    P = T // 4
    res, slot_map = residency_map(B, T, P, 7)
    gi = res[:, None, :, None].expand(B, Hkv, P, d)
    k_pool = torch.gather(K, 2, gi).contiguous().cuda()
    v_pool = torch.gather(Vv, 2, gi).contiguous().cuda()
    slot_map = slot_map.cuda()
    k_host, v_host = K.pin_memory(), Vv.pin_memory()
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, out, lse, _ = sd().make_attend_args(q, k_pool, v_pool, idx, T=T, k_host=k_host, v_host=v_host,
                                           slot_map=slot_map, err_word=e)
    ws = torch.zeros(max(16, sd().sd_gather_attend_workspace_bytes(a)), dtype=torch.uint8, device="cuda")
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    o0, l0 = out.clone(), lse.clone()
    host_before = int((slot_map.gather(1, idx.view(B, -1).long()) < 0).sum().item())
    pool_pos, hand = sd().pool_state(slot_map, P)
    sd().sd_promote_rows(a, pool_pos, hand)
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    assert torch.equal(out, o0) and torch.equal(lse, l0)
    host_after = int((slot_map.gather(1, idx.view(B, -1).long()) < 0).sum().item())
    assert host_before > 0 and host_after == 0  # the pool had room for the whole selection


def test_c4_promotion_full():
    # the tiered verify workload: its selection promoted into the 10 % pool (more misses
    # than free slots), then the attention over pool and host rows; the same bits as before
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c4_tiered_verify"]
    x = generate(w)
    dev = {k: x[k].cuda() for k in ("q_idx", "k_idx", "q", "slot_map", "k_pool", "v_pool")}
    k_host, v_host = x["k"].pin_memory(), x["v"].pin_memory()
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = sd().key_hist_buffer(w.B * w.Hkv)
    scores = sd().sd_index_score(dev["q_idx"], dev["k_idx"], key_hist=hist)
    idx = sd().sd_topk(scores, w.k, key_hist=hist)
    a, out, lse, _ = sd().make_attend_args(dev["q"], dev["k_pool"], dev["v_pool"], idx, T=w.T, k_host=k_host,
                                           v_host=v_host, slot_map=dev["slot_map"], err_word=e)
    ws = torch.zeros(max(16, sd().sd_gather_attend_workspace_bytes(a)), dtype=torch.uint8, device="cuda")
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    o0, l0 = out.clone(), lse.clone()
    sm0 = dev["slot_map"].cpu().numpy().copy()
    pool_pos, hand = sd().pool_state(dev["slot_map"], w.pool_rows)
    pp0, h0 = pool_pos.cpu().numpy().copy(), hand.cpu().numpy().copy()
    sd().sd_promote_rows(a, pool_pos, hand)
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    assert torch.equal(out, o0) and torch.equal(lse, l0)
    # the device state equals the oracle's promotion of the same selection
    o_slot, o_pos, o_hand = sm0.copy(), pp0.copy(), h0.copy()
    P = w.pool_rows
    dummy = np.zeros((w.B, 1, w.T, 1)), np.zeros((w.B, 1, w.T, 1))
    oracle.promote_rows(idx.cpu().numpy(), 1, o_slot, o_pos, o_hand, dummy[0], dummy[1],
                        np.zeros((w.B, 1, P, 1)), np.zeros((w.B, 1, P, 1)))
    np.testing.assert_array_equal(dev["slot_map"].cpu().numpy(), o_slot)
    np.testing.assert_array_equal(pool_pos.cpu().numpy(), o_pos)
    np.testing.assert_array_equal(hand.cpu().numpy(), o_hand)
    # the promoted rows are the host rows of their positions (a sample of slots)
    kp = dev["k_pool"].cpu()
    for b in range(w.B):
        for s in range(0, P, 997):
            t = int(o_pos[b, s])
            if t >= 0:
                assert torch.equal(kp[b, :, s], x["k"][b, :, t])


def test_c10_cached_tiered_steps():
    # the benchmark's cached workload over a whole cycle of query windows: every step's
    # attention equals (bit for bit) the same selection read with the pool as generated, and
    # the oracle on a sampled group; the cache ends up serving most of the selected rows
    import math
    import bench
    from gpu_util import assert_attend_close
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c10_cached_tiered"]
    x = generate(w)
    step = bench.make_step(w, x, torch.device("cuda"))
    static_pool = (x["k_pool"].cuda(), x["v_pool"].cuda(), x["slot_map"].cuda())
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    a0, out0, lse0, _ = sd().make_attend_args(step.q, static_pool[0], static_pool[1], step.idx, T=w.T,
                                              k_host=step.k_host, v_host=step.v_host, slot_map=static_pool[2],
                                              err_word=e)
    ws0 = torch.zeros(max(16, sd().sd_gather_attend_workspace_bytes(a0)), dtype=torch.uint8, device="cuda")
    assert step.staged_promotion and step.concurrent
    # the oracle's promotion state, from the generated residency (one unit per (b, KV head))
    U = w.B * w.Hkv
    sm0 = x["slot_map"].numpy()
    o_slot = np.repeat(sm0, w.Hkv, axis=0).astype(np.int32)
    o_pos = np.full((U, w.pool_rows), -1, dtype=np.int32)
    for u in range(U):
        t = np.nonzero(sm0[u // w.Hkv] >= 0)[0]
        o_pos[u, sm0[u // w.Hkv, t]] = t
    o_hand = np.zeros(U, dtype=np.int32)
    dummy_h = np.zeros((U, 1, w.T, 1), dtype=np.float32)  # rows checked below, against the host cache
    dummy_p = np.zeros((U, 1, w.pool_rows, 1), dtype=np.float32)
    host_rows, sel = [], []
    for s in range(w.drift_steps):
        step.run()
        a0.idx = step.idx.data_ptr()  # the step alternates two selection buffers
        sd().sd_gather_attend(a0, ws0)
        torch.cuda.synchronize()
        assert int(step.err.item()) == 0 and int(e.item()) == 0
        assert torch.equal(step.out, out0) and torch.equal(step.lse, lse0)
        host_rows.append(step.host_misses(step.slot_map)[1])
        sel.append(step.idx.cpu().numpy().reshape(U, 1, w.k))
        if s in (0, w.drift_steps - 1):
            b, h = s % w.B, 3
            qw = x["q_idx_seq"][b:b + 1, h:h + 1, s:s + w.V]
            rs = oracle.index_score(qw, x["k_idx"][b:b + 1, h:h + 1], 1, 1, w.V, w.T, w.dI)
            ri = oracle.topk(rs, w.k)
            np.testing.assert_array_equal(step.idx[b:b + 1, h:h + 1].cpu().numpy(), ri)
            qh = x["q"][b:b + 1, :, h * w.G:(h + 1) * w.G].contiguous()
            ro, rl, _ = oracle.gather_attend(qh, x["k"][b:b + 1, h:h + 1].contiguous(),
                                             x["v"][b:b + 1, h:h + 1].contiguous(), ri, 1, w.V, w.G, 1, w.d, w.T,
                                             w.k, 1, 1 / math.sqrt(w.d))
            assert_attend_close(step.out[b:b + 1, :, h * w.G:(h + 1) * w.G], ro)
            assert_attend_close(step.lse[b:b + 1, :, h * w.G:(h + 1) * w.G], rl, "lse")
    # after the first steps most selected rows are in the pool
    total_rows = w.B * w.Hkv * w.k
    assert host_rows[-1] < 0.5 * total_rows
    # every step's promotion ran with the next step, beside its selection: the state equals
    # the oracle's promotions of the same selections in order; then the last one
    for s in range(w.drift_steps - 1):
        oracle.promote_rows(sel[s], 1, o_slot, o_pos, o_hand, dummy_h, dummy_h, dummy_p, dummy_p)
    np.testing.assert_array_equal(step.slot_map.cpu().numpy().reshape(U, w.T), o_slot)
    np.testing.assert_array_equal(step.pool_pos.cpu().numpy(), o_pos)
    np.testing.assert_array_equal(step.hand.cpu().numpy(), o_hand)
    sd().sd_promote_staged_rows(step.pending, step.pool_pos, step.hand, step.ws_promote)
    torch.cuda.synchronize()
    oracle.promote_rows(sel[-1], 1, o_slot, o_pos, o_hand, dummy_h, dummy_h, dummy_p, dummy_p)
    np.testing.assert_array_equal(step.slot_map.cpu().numpy().reshape(U, w.T), o_slot)
    np.testing.assert_array_equal(step.pool_pos.cpu().numpy(), o_pos)
    np.testing.assert_array_equal(step.hand.cpu().numpy(), o_hand)
    # every occupied slot holds its position's K and V rows of its own KV head
    pos = torch.from_numpy(o_pos.astype(np.int64))
    occ = pos >= 0
    unit = torch.arange(U)[:, None].expand_as(pos)
    for pool, host in ((step.k_cache, x["k"]), (step.v_cache, x["v"])):
        got = pool.view(U, w.pool_rows, w.d).cpu()[occ]
        want = host.view(U, w.T, w.d)[unit[occ], pos[occ]]
        assert torch.equal(got, want)


def test_residency_per_kv_head():
    # per-head slot maps: the same residency copied to every head gives the same bits as the
    # shared map; promoting per head moves one row per miss and matches the oracle run on
    # the (b, KV head) units; the attention bits do not change
    from top_sparse_decode_gqa_gb300.workloads import residency_map
    g = torch.Generator().manual_seed(11)
    B, Hq, Hkv, d, T, n, V, P = 2, 16, 4, 128, 4096, 300, 2, 512
    q = torch.randn(B, V, Hq, d, generator=g).to(torch.bfloat16).cuda()
    K = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    Vv = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(T, generator=g)[:n]).values for _ in range(Hkv)])
                       for _ in range(B)]).int().cuda()
    res, slot_map = residency_map(B, T, P, 3)
    gi = res[:, None, :, None].expand(B, Hkv, P, d)
    k_pool = torch.gather(K, 2, gi).contiguous().cuda()
    v_pool = torch.gather(Vv, 2, gi).contiguous().cuda()
    k_host, v_host = K.pin_memory(), Vv.pin_memory()
    o_shared, l_shared, _ = sd().gather_attend(q, k_pool, v_pool, idx, T=T, k_host=k_host, v_host=v_host,
                                               slot_map=slot_map.cuda())
    per_head = slot_map[:, None, :].expand(B, Hkv, T).contiguous().cuda()
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, out, lse, _ = sd().make_attend_args(q, k_pool, v_pool, idx, T=T, k_host=k_host, v_host=v_host,
                                           slot_map=per_head, err_word=e)
    assert a.slot_per_head == 1
    ws = torch.zeros(max(16, sd().sd_gather_attend_workspace_bytes(a)), dtype=torch.uint8, device="cuda")
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, o_shared) and torch.equal(lse, l_shared)
    # promotion per (b, KV head)
    pool_pos, hand = sd().pool_state(per_head, P)
    assert pool_pos.shape == (B * Hkv, P)
    o_slot = per_head.cpu().numpy().reshape(B * Hkv, T).copy()
    o_pos, o_hand = pool_pos.cpu().numpy().copy(), hand.cpu().numpy().copy()
    sd().sd_promote_rows(a, pool_pos, hand)
    sd().sd_gather_attend(a, ws)
    # the staged path over per-head maps as well
    stage = sd().stage_buffers(a, torch.bfloat16)
    sd().sd_stage_host_rows(a, sd().stage_counter())
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    assert int(e.item()) == 0
    assert torch.equal(out, o_shared) and torch.equal(lse, l_shared)
    kh = K.float().numpy().reshape(B * Hkv, 1, T, d)
    vh = Vv.float().numpy().reshape(B * Hkv, 1, T, d)
    kp = np.zeros((B * Hkv, 1, P, d), dtype=np.float32)
    vp = np.zeros_like(kp)
    for u in range(B * Hkv):  # the oracle's pool starts with the generated rows
        for s_, t in enumerate(o_pos[u]):
            if t >= 0:
                kp[u, 0, s_], vp[u, 0, s_] = kh[u, 0, t], vh[u, 0, t]
    oracle.promote_rows(idx.cpu().numpy().reshape(B * Hkv, 1, n), 1, o_slot, o_pos, o_hand, kh, vh, kp, vp)
    np.testing.assert_array_equal(per_head.cpu().numpy().reshape(B * Hkv, T), o_slot)
    np.testing.assert_array_equal(pool_pos.cpu().numpy(), o_pos)
    np.testing.assert_array_equal(hand.cpu().numpy(), o_hand)
    got = k_pool.float().cpu().numpy().reshape(B * Hkv, 1, P, d)
    np.testing.assert_array_equal(got, kp)
    del stage
