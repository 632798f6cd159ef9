"""Every block shape of both block schedules, on exact inputs.

The plain tiles merge blocks of up to four leaves in registers, the
transposed tile (at most 64 output rows) blocks of up to eight, each as a
left and a right half. A tree of L <= 8 leaves is one block of L leaves and
a tree of 9 to 16 leaves two blocks of 4 to 8, so contractions of 1 to 40
leaves reach every block shape of both schedules, with and without pending
partials above them; a few larger odd counts add deeper slots. With integer
inputs in [-3, 3] every leaf sum is exact, so the GPU's bits must equal the
oracle's for every row count (RL-Kernel, "Batch-Invariant Deterministic GEMM
(det_gemm)", sections "Guarantees" and "Ascend NPU backend"), and the rows
computed by the transposed tile must equal the same rows of a plain-tile
launch."""
import pytest

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W
from gpu_util import check, dev, exact_equal

pytestmark = pytest.mark.gpu

LEAF_COUNTS = list(range(1, 41)) + [67, 100, 129, 257]


@pytest.mark.parametrize("L", LEAF_COUNTS)
def test_both_tiles_match_the_oracle_for_every_block_shape(L):
    K = 32 * L - (L % 3) * 5          # a partial last leaf for two L in three
    N = 136                           # two column tiles (weight tiles), the second ragged
    seed = 52000 + L
    A = W.randint_bf16((65, K), -3, 4, seed)
    B = W.randint_bf16((K, N), -3, 4, seed + 1)
    Wt = W.randint_bf16((N, K), -3, 4, seed + 2)
    a, b, wt = W.bits(A), W.bits(B), W.bits(Wt)
    Ad, Bd, Wd = dev(A), dev(B), dev(Wt)
    want = oracle.fwd(a, b)
    want_t = oracle.fwd_rhs_transposed(a, wt)
    plain = dg.det_gemm_fwd(Ad, Bd)                       # 65 rows: the plain tile
    plain_t = dg.det_gemm_fwd_rhs_transposed(Ad, Wd)
    check()
    assert exact_equal(W.bits(plain.cpu()), want), ("plain", L)
    assert exact_equal(W.bits(plain_t.cpu()), want_t), ("plain rhs_transposed", L)
    for M in (1, 8, 16, 17, 64):                          # the transposed tile (narrow up to 8 and 16 rows)
        got = dg.det_gemm_fwd(Ad[:M], Bd)
        got_t = dg.det_gemm_fwd_rhs_transposed(Ad[:M], Wd)
        check()
        assert exact_equal(W.bits(got.cpu()), want[:M]), ("transposed", L, M)
        assert exact_equal(W.bits(got_t.cpu()), want_t[:M]), ("transposed rhs_transposed", L, M)
