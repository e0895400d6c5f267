"""sd_gather_attend_noalloc: the gather-attend call for callers that cannot allocate
device memory (for example a plugin that receives only input and output pointers from a
framework that owns all device memory).  It must give what sd_gather_attend gives, using
the library's own static scratch array instead of a caller workspace, call after call.

This file is collected last on purpose, and it also passes when run alone in a fresh
process: it builds and loads the library itself.
"""
import pytest
import torch

from gpu_util import assert_attend_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_decode_gqa_gb300 import binding, build
    build.build()
    return binding


def _case(seed, B=2, Hq=32, Hkv=8, d=128, T=8192, k=512):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, 1, Hq, d, generator=g).bfloat16().cuda()
    K = torch.randn(B, Hkv, T, d, generator=g).bfloat16().cuda()
    V = torch.randn(B, Hkv, T, d, generator=g).bfloat16().cuda()
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(T, generator=g)[:k]).values
                                    for _ in range(Hkv)]) for _ in range(B)]).int().cuda()
    return q, K, V, idx


def _oracle(q, K, V, idx):
    import math

    import oracle
    B, _, Hq, d = q.shape
    Hkv, T, k = K.shape[1], K.shape[2], idx.shape[-1]
    return oracle.gather_attend(q.cpu(), K.cpu(), V.cpu(), idx.cpu().numpy(), B, 1, Hq, Hkv, d, T, k, 1,
                                1 / math.sqrt(d))[:2]


def test_noalloc_matches_the_workspace_call_twice_in_a_row(sd):
    for seed in (1, 2):   # two calls in a row share (and reuse) the static scratch
        q, K, V, idx = _case(seed)
        a_ref, out_ref, lse_ref, _ = sd.make_attend_args(q, K, V, idx, T=K.shape[2])
        need = sd.sd_gather_attend_workspace_bytes(a_ref)
        assert need > 0, "the case must use split-K scratch"
        sd.sd_gather_attend(a_ref, torch.zeros(need, dtype=torch.uint8, device="cuda"))
        a, out, lse, _ = sd.make_attend_args(q, K, V, idx, T=K.shape[2])
        a.workspace, a.workspace_bytes = None, 0      # no caller scratch at all
        sd.sd_gather_attend_noalloc(a)
        torch.cuda.synchronize()
        # the same split plan and kernels as the workspace call: the same bits
        assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
        ro, rl = _oracle(q, K, V, idx)
        assert_attend_close(out, ro)
        assert_attend_close(lse, rl, "lse")


def test_noalloc_partials_of_a_larger_split_do_not_leak_into_a_smaller_one(sd):
    # more splits first, then fewer, with nothing cleared in between: the second call reads
    # only the partials it wrote itself
    q, K, V, idx = _case(4)
    ro, rl = _oracle(q, K, V, idx)
    for splits in (16, 3):
        a_ref, out_ref, lse_ref, _ = sd.make_attend_args(q, K, V, idx, T=K.shape[2], splits=splits)
        need = sd.sd_gather_attend_workspace_bytes(a_ref)
        sd.sd_gather_attend(a_ref, torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda"))
        a, out, lse, _ = sd.make_attend_args(q, K, V, idx, T=K.shape[2], splits=splits)
        sd.sd_gather_attend_noalloc(a)
        torch.cuda.synchronize()
        assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref), splits
        assert_attend_close(out, ro)
        assert_attend_close(lse, rl, "lse")


def test_noalloc_rejects_requests_beyond_its_scratch(sd):
    # 32 query heads on one KV head (32 query rows per group), dense over 8192 rows in 128
    # splits: 8 * 128 * 32 * (128 + 2) * 4 bytes of partials > 16 MiB.
    g = torch.Generator().manual_seed(3)
    B, Hq, Hkv, d, T = 8, 32, 1, 128, 8192
    q = torch.randn(B, 1, Hq, d, generator=g).bfloat16().cuda()
    K = torch.randn(B, Hkv, T, d, generator=g).bfloat16().cuda()
    V = torch.randn(B, Hkv, T, d, generator=g).bfloat16().cuda()
    a, out, lse, _ = sd.make_attend_args(q, K, V, None, T=T, splits=128)
    assert sd.sd_gather_attend_workspace_bytes(a) > (16 << 20)
    out.fill_(7.0)
    with pytest.raises(sd.SdError) as ei:
        sd.sd_gather_attend_noalloc(a)
    assert "static scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)   # nothing was launched
