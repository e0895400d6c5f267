"""Staged host rows (sd_stage_host_rows): the selected rows whose slot is -1 are copied from
pinned host memory into an HBM stage at their list position, nothing else is written, and
sd_gather_attend reading them from the stage gives the same bits as reading them from host
memory (and the oracle's values within the attention tolerance).  The full-size tiered
verify workload runs the staged pipeline in the benchmark's launch configuration."""
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


def _case(seed, B, V, Hq, Hkv, d, T, n, block, dt, per_head=False, P=None, empty=0):
    from top_sparse_decode_gqa_gb300.workloads import residency_map
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
    P = T // 10 if P is None else P
    res, slot_map = residency_map(B, T, P, seed + 1)
    gi = res[:, None, :, None].expand(B, Hkv, P, d)
    k_pool = torch.gather(K, 2, gi).contiguous() if P else torch.zeros(B, Hkv, 1, d, dtype=dt)
    v_pool = torch.gather(Vv, 2, gi).contiguous() if P else torch.zeros(B, Hkv, 1, d, dtype=dt)
    return q, K, Vv, idx, slot_map, k_pool, v_pool


def _run(q, K, Vv, idx, slot_map, k_pool, v_pool, block, per_head, staged, counter=None, sentinel=None):
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    T = K.shape[2]
    # every tensor the args point to stays referenced here until the kernels have finished
    keep = [q.cuda(), k_pool.cuda(), v_pool.cuda(), idx.cuda(), K.pin_memory(), Vv.pin_memory(), slot_map.cuda()]
    a, out, lse, _ = sd().make_attend_args(keep[0], keep[1], keep[2], keep[3], block=block, T=T, k_host=keep[4],
                                           v_host=keep[5], slot_map=keep[6], err_word=e, per_head=per_head)
    stage = None
    if staged:
        stage = sd().stage_buffers(a, q.dtype)
        if sentinel is not None:
            stage[0].fill_(sentinel)
            stage[1].fill_(sentinel)
        counter = sd().stage_counter() if counter is None else counter
        sd().sd_stage_host_rows(a, counter)
    ws = torch.zeros(max(16, sd().sd_gather_attend_workspace_bytes(a)), dtype=torch.uint8, device="cuda")
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    del keep
    return out.cpu(), lse.cpu(), int(e.item()), stage, counter


@pytest.mark.parametrize("dt,d,block,per_head,V", [(torch.bfloat16, 128, 1, False, 1), (torch.bfloat16, 64, 1, False, 4),
                                                   (torch.float32, 128, 1, False, 2), (torch.bfloat16, 128, 16, False, 1),
                                                   (torch.bfloat16, 128, 1, True, 1), (torch.float32, 64, 4, True, 1)])
def test_staged_attention_is_bit_identical_to_host_reads(dt, d, block, per_head, V):
    B, Hq, Hkv, T = 2, 8, 2, 4096
    n = 300 // block
    q, K, Vv, idx, slot_map, kp, vp = _case(11 + d + block, B, V, Hq, Hkv, d, T, n, block, dt, per_head, empty=3)
    o0, l0, e0, _, _ = _run(q, K, Vv, idx, slot_map, kp, vp, block, per_head, staged=False)
    o1, l1, e1, stage, counter = _run(q, K, Vv, idx, slot_map, kp, vp, block, per_head, staged=True)
    assert e0 == 0 and e1 == 0
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert int(counter.abs().sum().item()) == 0, "the counter is left at zero"
    ro, rl, _ = oracle.gather_attend(q, K, Vv, idx.numpy(), B, V, Hq, Hkv, d, T, n, block, 1 / math.sqrt(d),
                                     per_head=per_head)
    assert_attend_close(o1, ro)
    assert_attend_close(l1, rl, "lse")


def test_stage_holds_exactly_the_host_rows():
    B, Hq, Hkv, d, T, n = 2, 8, 2, 128, 3000, 257
    dt = torch.bfloat16
    q, K, Vv, idx, slot_map, kp, vp = _case(5, B, 1, Hq, Hkv, d, T, n, 1, dt, empty=5)
    _, _, e, (ks, vs), _ = _run(q, K, Vv, idx, slot_map, kp, vp, 1, False, staged=True, sentinel=7.0)
    assert e == 0
    ks, vs = ks.cpu().view(B, Hkv, n, d), vs.cpu().view(B, Hkv, n, d)
    copied = 0
    for b in range(B):
        for h in range(Hkv):
            for j in range(n):
                t = int(idx[b, h, j])
                if t >= 0 and int(slot_map[b, t]) == -1:
                    assert torch.equal(ks[b, h, j], K[b, h, t]) and torch.equal(vs[b, h, j], Vv[b, h, t])
                    copied += 1
                else:  # pool rows and empty slots are not written
                    assert torch.all(ks[b, h, j] == 7.0) and torch.all(vs[b, h, j] == 7.0)
    assert copied > 0.8 * B * Hkv * (n - 5)


def test_counter_is_reused_across_calls():
    counter = sd().stage_counter()
    for seed in (21, 22, 23):
        q, K, Vv, idx, slot_map, kp, vp = _case(seed, 1, 1, 8, 2, 128, 2048, 200, 1, torch.bfloat16)
        o0, l0, _, _, _ = _run(q, K, Vv, idx, slot_map, kp, vp, 1, False, staged=False)
        o1, l1, e, _, counter = _run(q, K, Vv, idx, slot_map, kp, vp, 1, False, staged=True, counter=counter)
        assert e == 0 and torch.equal(o0, o1) and torch.equal(l0, l1)
        assert int(counter.abs().sum().item()) == 0


def test_all_host_and_no_host_rows():
    for P in (0, 2048):
        q, K, Vv, idx, slot_map, kp, vp = _case(31, 2, 1, 8, 2, 128, 2048, 128, 1, torch.bfloat16, P=P)
        o0, l0, _, _, _ = _run(q, K, Vv, idx, slot_map, kp, vp, 1, False, staged=False)
        o1, l1, e, _, _ = _run(q, K, Vv, idx, slot_map, kp, vp, 1, False, staged=True)
        assert e == 0 and torch.equal(o0, o1) and torch.equal(l0, l1)


def test_stage_reports_bad_index_and_slot():
    q, K, Vv, idx, slot_map, kp, vp = _case(41, 1, 1, 8, 2, 128, 1000, 20, 1, torch.bfloat16)
    bad = idx.clone()
    bad[0, 0, 3] = 1000 + 5
    _, _, e, _, _ = _run(q, K, Vv, bad, slot_map, kp, vp, 1, False, staged=True)
    assert e & sd().SD_DEVERR_INDEX
    sm2 = slot_map.clone()
    sm2[0, int(idx[0, 1, 0])] = 12345  # beyond the pool
    _, _, e, _, _ = _run(q, K, Vv, idx, sm2, kp, vp, 1, False, staged=True)
    assert e & sd().SD_DEVERR_SLOT


def test_c4_staged_pipeline_full():
    # indexer -> top-k -> staged host rows -> attention from HBM, at the full tiered-verify
    # size: the same bits as the attention reading host memory directly
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c4_tiered_verify"]
    x = generate(w)
    dev = {k: x[k].cuda() for k in ("q_idx", "k_idx", "q", "slot_map", "k_pool", "v_pool")}
    k_host, v_host = x["k"].pin_memory(), x["v"].pin_memory()
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = sd().key_hist_buffer(w.B * w.Hkv)
    scores = sd().sd_index_score(dev["q_idx"], dev["k_idx"], err_word=e, key_hist=hist)
    idx = sd().sd_topk(scores, w.k, key_hist=hist)
    a, out, lse, _ = sd().make_attend_args(dev["q"], dev["k_pool"], dev["v_pool"], idx, T=w.T, k_host=k_host,
                                           v_host=v_host, slot_map=dev["slot_map"], err_word=e)
    ws = torch.zeros(max(16, sd().sd_gather_attend_workspace_bytes(a)), dtype=torch.uint8, device="cuda")
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    o_host, l_host = out.clone(), lse.clone()
    stage = sd().stage_buffers(a, torch.bfloat16)
    counter = sd().stage_counter()
    sd().sd_stage_host_rows(a, counter)
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()
    assert int(e.item()) == 0 and int(counter.abs().sum().item()) == 0
    assert torch.equal(out, o_host) and torch.equal(lse, l_host)
    i_gpu = idx.cpu().numpy()
    for b, h in ((0, 0), (w.B - 1, w.Hkv - 1)):
        rs = oracle.index_score(x["q_idx"][b:b + 1, h:h + 1], x["k_idx"][b:b + 1, h:h + 1], 1, 1, w.V, w.T, w.dI)
        ri = oracle.topk(rs, w.k)
        np.testing.assert_array_equal(i_gpu[b:b + 1, h:h + 1], ri)
        qh = x["q"][b:b + 1, :, h * w.G:(h + 1) * w.G].contiguous()
        ro, rl, _ = oracle.gather_attend(qh, x["k"][b:b + 1, h:h + 1].contiguous(),
                                         x["v"][b:b + 1, h:h + 1].contiguous(), ri, 1, w.V, w.G, 1,
                                         w.d, w.T, w.k, 1, 1 / math.sqrt(w.d))
        assert_attend_close(out[b:b + 1, :, h * w.G:(h + 1) * w.G], ro)
        assert_attend_close(lse[b:b + 1, :, h * w.G:(h + 1) * w.G], rl, "lse")
    del stage


def test_c9_lookahead_full():
    # the benchmark's multi-layer tiered workload in its launch configuration: every layer's
    # selection and staging run on their own streams ahead of the attention, and the results
    # are the same bits as the same calls in order on one stream, and the oracle's values
    import bench
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c9_lookahead_tiered"]
    x = generate(w)
    step = bench.make_step(w, x, torch.device("cuda"), lookahead=True)
    step.run()
    torch.cuda.synchronize()
    assert int(step.err.item()) == 0
    got = [(step.idx[l].clone(), step.args[l][1].clone(), step.args[l][2].clone()) for l in range(w.layers)]
    step.lookahead = False
    step.run()
    torch.cuda.synchronize()
    for l in range(w.layers):
        assert torch.equal(step.idx[l], got[l][0])
        assert torch.equal(step.args[l][1], got[l][1]) and torch.equal(step.args[l][2], got[l][2])
    ref = bench.oracle_step(w, x, 0, 1)  # sequence 0, every layer
    for l, (ri, (ro, rl, _)) in enumerate(ref):
        np.testing.assert_array_equal(got[l][0][:1].cpu().numpy(), ri)
        assert_attend_close(got[l][1][:1], ro)
        assert_attend_close(got[l][2][:1], rl, "lse")
