"""Host-side checks of the seeded input generators (no GPU)."""
import math

import torch

from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate, residency_map


def test_configs_match_the_workload_table():
    c1, c2, c3, c4, c5 = (WORKLOADS[n] for n in ("c1_tiny", "c2_llama3_8b_gqa", "c3_block_sparse",
                                                 "c4_tiered_verify", "c5_importance_tiering"))
    assert (c1.B, c1.Hq, c1.Hkv, c1.d, c1.T, c1.k, c1.planted, c1.dtype) == (1, 4, 1, 64, 1024, 64, 8, "f32")
    assert (c2.B, c2.Hq, c2.Hkv, c2.d, c2.T, c2.k, c2.planted) == (8, 32, 8, 128, 32768, 1024, 655)
    assert (c3.T, c3.block, c3.k, c3.N, c3.n_rows) == (131072, 64, 64, 2048, 4096)
    assert (c4.V, c4.k, c4.pool_rows, c4.queries_per_step) == (8, 2048, 13107, 32)
    assert (c5.layers, c5.Hq, c5.Hkv, c5.T, c5.B, c5.steps, c5.dense) == (28, 28, 4, 65536, 2, 64, True)


def test_generation_is_deterministic_and_structured():
    w = WORKLOADS["c2_llama3_8b_gqa"].scaled(B=2, Hq=8, Hkv=2, T=2048)
    a, b = generate(w), generate(w)
    for key in ("q_idx", "k_idx", "q", "k", "v", "planted"):
        assert torch.equal(a[key], b[key]), key
    assert a["planted"].shape == (2, 2, math.floor(0.02 * 2048))
    ki = a["k_idx"].float()
    assert ki.abs().max() <= 8 and torch.equal(ki, ki.round())
    # planted keys carry the sign of the indexer query and magnitude 5..8
    sign = torch.where(a["q_idx"][:, :, 0].float() >= 0, 1.0, -1.0)
    for bb in range(2):
        for h in range(2):
            rows = ki[bb, h, a["planted"][bb, h]]
            assert torch.all(rows * sign[bb, h] >= 5) and torch.all(rows * sign[bb, h] <= 8)
    c = generate(w, seed=7)
    assert not torch.equal(a["k"], c["k"])


def test_c1_planted_keys_are_eight_times_sign():
    w = WORKLOADS["c1_tiny"]
    x = generate(w)
    assert x["k"].dtype == torch.float32 and x["q_idx"].dtype == torch.float32
    sign = torch.where(x["q_idx"][0, 0, 0] >= 0, 1.0, -1.0)
    for p in x["planted"][0, 0]:
        assert torch.equal(x["k_idx"][0, 0, p], 8 * sign)


def test_residency_pool_holds_copies_of_resident_rows():
    w = WORKLOADS["c4_tiered_verify"].scaled(B=2, Hq=8, Hkv=2, T=1000, k=64)
    x = generate(w)
    P = w.pool_rows
    assert P == 100 and x["k_pool"].shape == (2, 2, P, w.d)
    for b in range(2):
        sm = x["slot_map"][b]
        assert int((sm >= 0).sum()) == P
        pos = torch.nonzero(sm >= 0).flatten()
        assert torch.equal(pos, x["resident"][b])
        assert torch.equal(x["k_pool"][b, :, sm[pos].long()], x["k"][b, :, pos])
        assert torch.equal(x["v_pool"][b, :, sm[pos].long()], x["v"][b, :, pos])
    res, sm = residency_map(3, 50, 0, seed=1)
    assert res.shape == (3, 0) and torch.all(sm == -1)


def test_later_workloads_match_their_descriptions():
    c3, c6, c7, c8, c9, c10 = (WORKLOADS[n] for n in ("c3_block_sparse", "c6_window_blocks", "c7_head_topk",
                                                      "c8_verify_layer_group", "c9_lookahead_tiered",
                                                      "c10_cached_tiered"))
    assert c3.q_idx_dtype == "f16"
    assert (c6.window_kernel, c6.window_stride, c6.k, c6.n_rows) == (32, 16, 64, 2048)
    assert (c7.per_head, c7.k, c7.Hq, c7.Hkv, c7.T) == (True, 1024, 32, 8, 32768)
    assert (c8.layers, c8.ring_w, c8.V, c8.k, c8.B) == (4, 64, 8, 1024, 2)
    assert (c9.layers, c9.layer_indexers, c9.resident_frac, c9.B, c9.T) == (4, True, 0.1, 2, 131072)
    assert (c10.drift_steps, c10.resident_frac, c10.pool_rows, c10.slot_per_head) == (16, 0.1, 13107, True)


def test_sliding_query_windows_and_rings_are_drawn():
    w = WORKLOADS["c10_cached_tiered"].scaled(B=1, T=2048, k=64)
    x = generate(w)
    assert x["q_idx_seq"].shape == (1, w.Hkv, w.V + w.drift_steps - 1, w.dI)
    w8 = WORKLOADS["c8_verify_layer_group"].scaled(T=1024, k=32)
    x8 = generate(w8)
    W, T, V = w8.ring_w, w8.T, w8.V
    held = x8["ring_pos"][0]
    # the ring holds the W - V tokens before T at slot position mod W; the drafts' slots are empty
    assert sorted(int(t) for t in held if t >= 0) == list(range(T - (W - V), T))
    assert all(int(held[t % W]) == t for t in range(T - (W - V), T))
    assert x8["qpos"].tolist() == [[T + v for v in range(V)]] * w8.B
