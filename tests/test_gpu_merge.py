"""det_gemm_merge: partial products over equal contiguous leaf ranges,
merged with the tree's top levels, give the full product bit for bit
(RL-Kernel, "Batch-Invariant Deterministic GEMM (det_gemm)", section
"Ascend NPU backend": a contiguous half-K GEMM is one child of the tree; the
same holds for quarters and eighths when the leaf count divides evenly)."""
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import workloads as W
from gpu_util import check, dev

pytestmark = pytest.mark.gpu


def bits(t):
    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("n", [2, 4, 8])
@pytest.mark.parametrize("K", [4096, 1000])        # 128 leaves; 32 leaves with a partial last one
def test_sharded_contraction_merges_to_the_full_product(n, K):
    M, N = 300, 520
    L = (K + 31) // 32
    if L % n:
        pytest.skip("leaf count not divisible by the shard count")
    A = dev(W.randn_bf16((M, K), 1.0, 8100 + K))
    B = dev(W.randn_bf16((K, N), 0.02, 8200 + K))
    step = L // n * 32                               # contraction elements per shard
    cuts = [min(K, i * step) for i in range(n + 1)]
    for f32 in (False, True):
        f = dg.det_gemm_fwd_fp32 if f32 else dg.det_gemm_fwd
        full = f(A, B)
        parts = [f(A[:, cuts[i]:cuts[i + 1]], B[cuts[i]:cuts[i + 1]]) for i in range(n)]
        merged = (dg.det_gemm_merge_fp32 if f32 else dg.det_gemm_merge)(parts)
        check()
        assert torch.equal(bits(merged), bits(full)), (n, K, f32)


def test_merge_of_da_shards_and_a_wrong_order_differs():
    # dA = dC . B^T contracts over N: shard N in two halves.
    M, K, N = 256, 384, 2048
    dC = W.randn_bf16((M, N), 1.0, 8301).cuda()
    B = W.randn_bf16((K, N), 1.0, 8302).cuda()
    full = dg.det_gemm_da(dC, B)
    h = N // 2
    lo = dg.det_gemm_da(dC[:, :h], B[:, :h])
    hi = dg.det_gemm_da(dC[:, h:], B[:, h:])
    assert torch.equal(bits(dg.det_gemm_merge([lo, hi])), bits(full))
    check()
