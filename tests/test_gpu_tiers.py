"""Attention over a tiered cache ("Nem Todos os Pensamentos Necessitam de HBM", gist.science
summary, Metodologia 1: T0 in HBM, T1 in host memory, T2 at 8 bits, T3 evicted; Metodologia
3: a row contributes the same terms wherever it is stored).  sd_gather_attend with `tier`
reads T2 rows as int8 codes times their per-row scale and leaves T3 rows out; it is compared
with the oracle's attention over the same selection at the values the tiers give the rows
(T2: code x scale, T3: an empty slot), within 2e-3 max-abs and 1e-3 relative L2.  Tiers,
codes and scales are the oracle's own (they are inputs here; their GPU versions are pinned
bit-exact elsewhere).  Every call goes through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attend_close

pytestmark = pytest.mark.gpu

FRAC = np.array([0.2, 0.6, 0.9])


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_decode_gqa_gb300 import build
    build.build()


def sd():
    from top_sparse_decode_gqa_gb300 import binding
    return binding


def make(seed, B=2, Hkv=2, G=4, V=1, T=3000):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, V, Hkv * G, 128, generator=g).bfloat16()
    K = torch.randn(B, Hkv, T, 128, generator=g).bfloat16()
    Vv = torch.randn(B, Hkv, T, 128, generator=g).bfloat16()
    s = torch.rand(B, T, generator=g, dtype=torch.float64).numpy()
    tier, _ = oracle.tier_classify(s, FRAC)
    kc, ks = oracle.quantize_rows_int8(K, tier, B, Hkv, T, 128)
    vc, vs = oracle.quantize_rows_int8(Vv, tier, B, Hkv, T, 128)
    return q, K, Vv, tier, kc, ks, vc, vs


def tiered_values(x, tier, codes, scales):
    """The rows as the tiers give them: T2 rows code x scale (fp32), the others unchanged."""
    xf = x.float().numpy().copy()
    deq = codes.astype(np.float32) * scales[..., None]
    t2 = np.broadcast_to((tier == 2)[:, None, :, None], xf.shape)
    return torch.from_numpy(np.where(t2, deq, xf))


def reference(q, K, Vv, tier, kc, ks, vc, vs, idx):
    """The oracle's attention over idx [B,Hkv,n] (T3 positions as empty slots)."""
    B, V, Hq, _ = q.shape
    Hkv, T = K.shape[1], K.shape[2]
    ii = idx.copy()
    for b in range(B):
        ii[b][tier[b][idx[b]] == 3] = -1
    return oracle.gather_attend(q.float(), tiered_values(K, tier, kc, ks), tiered_values(Vv, tier, vc, vs), ii, B,
                                V, Hq, Hkv, 128, T, ii.shape[-1], 1, 1 / math.sqrt(128))[:2]


def tier_kwargs(tier, kc, ks, vc, vs):
    return dict(tier=torch.from_numpy(tier).cuda(), k_int8=torch.from_numpy(kc).cuda(),
                v_int8=torch.from_numpy(vc).cuda(), k_scale=torch.from_numpy(ks).cuda(),
                v_scale=torch.from_numpy(vs).cuda())


def run(a, *alive):
    """Runs the call `a` describes; `alive` holds the device tensors whose addresses the
    args carry (the args keep no references of their own)."""
    need = sd().sd_gather_attend_workspace_bytes(a)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    sd().sd_gather_attend(a, ws)
    torch.cuda.synchronize()


def test_tiers_dense_over_the_cache():
    q, K, Vv, tier, kc, ks, vc, vs = make(1)
    B, Hkv, T = K.shape[0], K.shape[1], K.shape[2]
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = [q.cuda(), K.cuda(), Vv.cuda()]
    tk = tier_kwargs(tier, kc, ks, vc, vs)
    a, out, lse, _ = sd().make_attend_args(*dev, None, T=T, err_word=e, **tk)
    run(a, dev, tk)
    assert int(e.item()) == 0
    idx = np.broadcast_to(np.arange(T, dtype=np.int32), (B, Hkv, T)).copy()
    ro, rl = reference(q, K, Vv, tier, kc, ks, vc, vs, idx)
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")


def test_tiers_with_pool_and_host_rows():
    # T0 rows in the HBM pool, T1 rows read from pinned host memory (slot -1), T2 from the
    # int8 rows, T3 left out; a sparse selection with entries of every tier
    q, K, Vv, tier, kc, ks, vc, vs = make(2, B=2, Hkv=2, G=4, V=2, T=4000)
    B, Hkv, T = K.shape[0], K.shape[1], K.shape[2]
    g = torch.Generator().manual_seed(7)
    k = 700
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(T, generator=g)[:k]).values for _ in range(Hkv)])
                       for _ in range(B)]).int()
    n0 = int((tier[0] == 0).sum())
    assert all(int((tier[b] == 0).sum()) == n0 for b in range(B))
    slot_map = np.full((B, T), -1, dtype=np.int32)
    kp = torch.zeros(B, Hkv, n0, 128, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    for b in range(B):
        pos = np.nonzero(tier[b] == 0)[0]
        slot_map[b, pos] = np.arange(n0)
        kp[b] = K[b][:, torch.from_numpy(pos)]
        vp[b] = Vv[b][:, torch.from_numpy(pos)]
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = [q.cuda(), kp.cuda(), vp.cuda(), idx.cuda(), torch.from_numpy(slot_map).cuda()]
    host = [K.pin_memory(), Vv.pin_memory()]
    tk = tier_kwargs(tier, kc, ks, vc, vs)
    a, out, lse, _ = sd().make_attend_args(*dev[:4], T=T, k_host=host[0], v_host=host[1], slot_map=dev[4], err_word=e,
                                          **tk)
    run(a, dev, host, tk)
    assert int(e.item()) == 0
    ro, rl = reference(q, K, Vv, tier, kc, ks, vc, vs, idx.numpy())
    assert_attend_close(out, ro)
    assert_attend_close(lse, rl, "lse")


def test_tiers_without_t2_or_t3_give_the_untiered_bits():
    # every position in T0 or T1: the tiered call reads the same rows at the same values, so
    # it gives the bits of the untiered call through the same row loop
    q, K, Vv, _, kc, ks, vc, vs = make(3, T=2500)
    B, T = K.shape[0], K.shape[2]
    tier = np.zeros((B, T), dtype=np.uint8)
    tier[:, 1::2] = 1
    qd, Kd, Vd = q.cuda(), K.cuda(), Vv.cuda()
    a0, out0, lse0, _ = sd().make_attend_args(qd, Kd, Vd, None, T=T, row_loop=True)
    run(a0)
    tk = tier_kwargs(tier, kc, ks, vc, vs)
    a1, out1, lse1, _ = sd().make_attend_args(qd, Kd, Vd, None, T=T, **tk)
    run(a1, tk)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_tiers_all_evicted_is_the_empty_selection():
    q, K, Vv, _, kc, ks, vc, vs = make(4, T=600)
    B, T = K.shape[0], K.shape[2]
    tier = np.full((B, T), 3, dtype=np.uint8)
    dev = [q.cuda(), K.cuda(), Vv.cuda()]
    tk = tier_kwargs(tier, kc, ks, vc, vs)
    a, out, lse, _ = sd().make_attend_args(*dev, None, T=T, **tk)
    run(a, dev, tk)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_tiers_unsupported_combinations_are_rejected():
    q, K, Vv, tier, kc, ks, vc, vs = make(5, T=256)
    T = K.shape[2]
    tk = tier_kwargs(tier, kc, ks, vc, vs)
    qd, Kd, Vd = q.cuda(), K.cuda(), Vv.cuda()
    # fp32 rows
    a, _, _, _ = sd().make_attend_args(qd.float(), Kd.float(), Vd.float(), None, T=T, **tk)
    with pytest.raises(sd().SdError):
        run(a)
    # the fused select + attend
    a, _, _, _ = sd().make_attend_args(qd, Kd, Vd, None, n_idx=16, T=T, **tk)
    scores = torch.zeros(K.shape[0], K.shape[1], T, dtype=torch.float32, device="cuda")
    idx = torch.empty(K.shape[0], K.shape[1], 16, dtype=torch.int32, device="cuda")
    with pytest.raises(sd().SdError):
        sd().sd_select_attend(scores, a, idx)
    # missing codes
    bad = dict(tk)
    bad["v_scale"] = None
    a, _, _, _ = sd().make_attend_args(qd, Kd, Vd, None, T=T, **bad)
    with pytest.raises(sd().SdError):
        run(a)
