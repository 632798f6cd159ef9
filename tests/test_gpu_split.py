"""Skinny launches split every tile's contraction into 2, 4 or 8 subtrees of
the merge tree and merge them afterwards. The result must be the unsplit
launch's bits (RL-Kernel, "Batch-Invariant Deterministic GEMM (det_gemm)",
section "Ascend NPU backend": a contiguous half-K GEMM is one child of the
tree, and so on level by level). These cases take the split (few output
tiles) and compare with the same rows inside a launch that does not (many
tiles), bit for bit, and with the oracle on exact inputs."""
import numpy as np
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W
from gpu_util import check, dev, exact_equal

pytestmark = pytest.mark.gpu


def bits_equal(x, y):
    a = x.contiguous().view(torch.int32 if x.dtype == torch.float32 else torch.int16)
    b = y.contiguous().view(torch.int32 if y.dtype == torch.float32 else torch.int16)
    return torch.equal(a, b)


@pytest.mark.parametrize("K", [4096, 768, 750])       # 128 leaves; 24 leaves (3 per eighth); partial last leaf
@pytest.mark.parametrize("fn", ["fwd", "fwd_fp32"])
def test_split_forward_rows_equal_the_unsplit_launch(K, fn):
    N = 1024
    A = dev(W.randn_bf16((4096, K), 1.0, 7100 + K))     # row pitch padded to 16 bytes
    B = dev(W.randn_bf16((K, N), 0.02, 7200 + K))
    f = getattr(dg, "det_gemm_" + fn)
    full = f(A, B)                       # 32 x 8 tiles: not split
    for M in (1, 5, 100, 256):           # 8 or 16 tiles: split
        assert bits_equal(f(A[:M], B), full[:M]), (K, fn, M)
    check()


def test_split_rhs_transposed_and_da_rows_equal_the_unsplit_launch():
    K, N = 2048, 1024
    A = W.randn_bf16((4096, K), 1.0, 7301).cuda()
    Wt = W.randn_bf16((N, K), 0.02, 7302).cuda()        # [N, K]
    full = dg.det_gemm_fwd_rhs_transposed(A, Wt)
    full32 = dg.det_gemm_fwd_fp32_rhs_transposed(A, Wt)
    dC = W.randn_bf16((4096, N), 1e-3, 7303).cuda()
    Bw = W.randn_bf16((K, N), 0.02, 7304).cuda()
    full_da = dg.det_gemm_da(dC, Bw)                     # [4096, K], contraction N = 1024
    for M in (3, 130):
        assert bits_equal(dg.det_gemm_fwd_rhs_transposed(A[:M], Wt), full[:M]), M
        assert bits_equal(dg.det_gemm_fwd_fp32_rhs_transposed(A[:M], Wt), full32[:M]), M
        assert bits_equal(dg.det_gemm_da(dC[:M], Bw), full_da[:M]), M
    check()


def test_split_weight_gradient_is_exact_on_integer_inputs():
    # dB of a small weight over many tokens: 2 x 2 or 2 x 16 output tiles
    # and a 4096-long contraction, so the launch splits.
    M = 4096
    for kout, n in ((256, 256), (256, 2048)):
        A = W.randint_bf16((M, kout), -3, 4, 7401 + n)
        dC = W.randint_bf16((M, n), -3, 4, 7402 + n)
        got = dg.det_gemm_db(A.cuda(), dC.cuda())
        got_t = dg.det_gemm_db_transposed(A.cuda(), dC.cuda())
        check()
        want = oracle.db(W.bits(A), W.bits(dC))
        assert exact_equal(W.bits(got), want), (kout, n)
        assert exact_equal(W.bits(got_t), np.ascontiguousarray(want.T)), (kout, n)


def test_tail_split_equals_one_launch():
    """A launch whose tiles fill whole rounds of one CTA per SM but a few
    (the QKV projection at 1024 rows: 8 x 96 = 768 = 5 x 152 + 8 tiles)
    runs its last column panel as a second launch whose tiles split their
    contraction over the idle SMs. The result must be one launch's bits: a
    one-group grouped launch never splits, and exact inputs must give the
    oracle's bits."""
    M, K, N = 1024, 4096, 12288
    A = dev(W.randn_bf16((M, K), 1.0, 7600))
    B = dev(W.randn_bf16((K, N), 0.02, 7601))
    C = dg.det_gemm_fwd(A, B)
    (G,) = dg.det_gemm_fwd_grouped([A], [B])
    check()
    assert bits_equal(C, G)
    # the same through the other operand layouts that take the tail split
    Wt = dev(W.randn_bf16((N, K), 0.02, 7602))
    Ct = dg.det_gemm_fwd_rhs_transposed(A, Wt)
    check()
    Ai = W.randint_bf16((M, K), -3, 4, 7603)
    Bi = W.randint_bf16((K, N), -3, 4, 7604)
    Ci = dg.det_gemm_fwd(dev(Ai), dev(Bi))
    check()
    rows = np.array([0, 1, 511, 1023])
    want = oracle.fwd(W.bits(Ai)[rows], W.bits(Bi))
    assert exact_equal(W.bits(Ci.cpu())[rows], want)
    # rhs-transposed against the forward with the weight transposed
    Cf = dg.det_gemm_fwd(A, Wt.t().contiguous())
    check()
    assert bits_equal(Ct, Cf)
