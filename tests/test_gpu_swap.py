"""Launches with at most 64 output rows take the transposed tile: the MMA's
128 lanes carry output columns and its N side the few rows, so the
epilogue's work follows the rows that exist. The page promises that a row's
bits do not depend on how many rows are computed with it (RL-Kernel,
"Batch-Invariant Deterministic GEMM (det_gemm)", sections "Why" and
"Guarantees"), so every case here checks the transposed launch against the
same rows computed by the plain tile (more than 64 rows), bit for bit, and
against the oracle on exact inputs and within the derived tolerance on
normal ones.

Why the bits can be equal: with the operands' roles swapped the tensor core
still forms, for each output element, the same 32 products of the same
BF16 pairs (a product of two BF16 values is exact and commutative) into a
fresh FP32 accumulator, in the same two K = 16 steps; what could differ is
only how the hardware orders and aligns those products inside a step if
that depended on the operand roles. The stress cases below are built to
expose such a dependence: products spread over 60 binades, so that the
alignment of a hardware FP32 sum decides which low bits survive, and sums
of signed powers of two that land exactly on BF16 rounding midpoints with
residues far below them, over contractions from one leaf to 1024 leaves,
at row counts on both sides of 64."""
import numpy as np
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W
from gpu_util import assert_bf16_close, check, dev, exact_equal

pytestmark = pytest.mark.gpu

ROWS = (1, 2, 7, 8, 9, 16, 17, 33, 63, 64)


def bits_equal(x, y):
    return torch.equal(x.contiguous().view(torch.int16), y.contiguous().view(torch.int16))


@pytest.mark.parametrize("K,N", [(4096, 1024), (100, 200), (14336, 256), (32, 8)])
def test_forward_rows_equal_the_plain_tile(K, N):
    A = dev(W.randn_bf16((256, K), 1.0, 8100 + K))
    B = dev(W.randn_bf16((K, N), 0.02, 8200 + K))
    full = dg.det_gemm_fwd(A, B)                    # 256 rows: plain tile
    for M in ROWS:
        assert bits_equal(dg.det_gemm_fwd(A[:M], B), full[:M]), (K, N, M)
    # rows taken from the middle of the batch
    assert bits_equal(dg.det_gemm_fwd(A[100:137], B), full[100:137])
    check()


@pytest.mark.parametrize("K,N", [(4096, 1024), (744, 136)])   # 744: a partial last leaf
def test_rhs_transposed_and_da_rows_equal_the_plain_tile(K, N):
    A = dev(W.randn_bf16((256, K), 1.0, 8301 + K))
    Wt = dev(W.randn_bf16((N, K), 0.02, 8302 + K))          # [N, K]
    dC = dev(W.randn_bf16((256, N), 1e-3, 8303 + K))
    Bw = dev(W.randn_bf16((K, N), 0.02, 8304 + K))          # [K, N]
    full = dg.det_gemm_fwd_rhs_transposed(A, Wt)
    full_da = dg.det_gemm_da(dC, Bw)                         # [256, K], contraction N
    for M in ROWS:
        assert bits_equal(dg.det_gemm_fwd_rhs_transposed(A[:M], Wt), full[:M]), (K, N, M)
        assert bits_equal(dg.det_gemm_da(dC[:M], Bw), full_da[:M]), (K, N, M)
    check()


def test_split_contraction_rows_equal_the_plain_tile():
    # Few column tiles and a long contraction: the transposed launch also
    # splits its contraction into subtrees (MLP down-projection of 4 tokens).
    K, N = 14336, 512
    A = dev(W.randn_bf16((128, K), 1.0, 8401))
    B = dev(W.randn_bf16((K, N), 0.02, 8402))
    full = dg.det_gemm_fwd(A, B)
    for M in (1, 4, 64):
        assert bits_equal(dg.det_gemm_fwd(A[:M], B), full[:M]), M
    check()


def test_padded_pitches_and_the_allocation_free_entry_point():
    K, N = 512, 384
    A = W.randn_bf16((128, K), 1.0, 8501)
    B = W.randn_bf16((K, N), 0.02, 8502)
    Ab = torch.zeros((128, K + 24), dtype=torch.bfloat16, device="cuda")
    Ab[:, :K] = A.cuda()
    Bb = torch.zeros((K, N + 40), dtype=torch.bfloat16, device="cuda")
    Bb[:, :N] = B.cuda()
    full = dg.det_gemm_fwd(Ab[:, :K], Bb[:, :N])
    for M in (5, 64):
        Cb = torch.full((M, N + 56), 7.0, dtype=torch.bfloat16, device="cuda")   # padded output pitch
        dg.det_gemm_fwd(Ab[:M, :K], Bb[:, :N], out=Cb[:, :N])
        assert bits_equal(Cb[:, :N], full[:M]), M
        assert bool((Cb[:, N:] == 7.0).all()), "columns past N were written"
        C2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        dg.det_gemm_fwd_noalloc(Ab[:M, :K], Bb[:, :N], C2)
        assert bits_equal(C2, full[:M]), M
    check()


@pytest.mark.parametrize("M,K,N", [(1, 96, 136), (13, 4096, 256), (64, 2000, 128)])
def test_integer_inputs_match_oracle_bit_for_bit(M, K, N):
    A = W.randint_bf16((M, K), -8, 9, 8600 + M)
    B = W.randint_bf16((K, N), -8, 9, 8700 + M)
    got = W.bits(dg.det_gemm_fwd(dev(A), dev(B)))
    check()
    want = oracle.gemm(W.bits(A), W.bits(B))
    assert exact_equal(got, want)


def test_normal_inputs_within_tolerance_of_oracle():
    M, K, N = 3, 4096, 640
    A = W.randn_bf16((M, K), 1.0, 8801)
    B = W.randn_bf16((K, N), 0.02, 8802)
    got = W.bits(dg.det_gemm_fwd(dev(A), dev(B)))
    Wt = W.randn_bf16((N, K), 0.02, 8803)
    got_t = W.bits(dg.det_gemm_fwd_rhs_transposed(dev(A), dev(Wt)))
    check()
    want, nodemax = oracle.gemm(W.bits(A), W.bits(B), with_node_max=True)
    assert_bf16_close(got, want, nodemax, K // 32, "fwd, 3 rows")
    want_t, nodemax_t = oracle.gemm(W.bits(A), np.ascontiguousarray(W.bits(Wt).T), with_node_max=True)
    assert_bf16_close(got_t, want_t, nodemax_t, K // 32, "rhs_transposed, 3 rows")


def test_transposed_tile_with_several_units_per_cta():
    """More output columns than 152 tiles of 128 hold: each CTA of a
    transposed launch walks two or three tiles, with its copy warp's stage
    and prefetch cursors crossing from one tile to the next (and a ragged
    last tile). Rows 1, 9 and 64 (all three epilogue widths) must equal the
    same rows of a 256-row plain-tile launch, through both transposed
    instances."""
    K, N = 256, 2 * 152 * 128 + 200
    A = dev(W.randn_bf16((256, K), 1.0, 30101))
    B = dev(W.randn_bf16((K, N), 0.05, 30102))
    Wt = dev(W.randn_bf16((N, K), 0.05, 30103))
    full = dg.det_gemm_fwd(A, B)
    full_t = dg.det_gemm_fwd_rhs_transposed(A, Wt)
    for M in (1, 9, 64):
        assert bits_equal(dg.det_gemm_fwd(A[:M], B), full[:M]), (M, "fwd")
        assert bits_equal(dg.det_gemm_fwd_rhs_transposed(A[:M], Wt), full_t[:M]), (M, "rhs_t")
    check()


ADV_KC = [32, 96, 4096, 14336, 32768]


def _adversarial(kind, shape, seed):
    if kind == "normal":
        return W.randn_bf16(shape, 1.0, seed)
    if kind == "wide":
        return W.wide_exponent_bf16(shape, -15, 15, seed)
    # "ties": signed powers of two; products 1, 2^-8, 2^-9 sum onto BF16
    # midpoints, products near 2^-24 .. 2^-34 are residues an FP32 sum may
    # keep or drop depending on its alignment
    return W.power_of_two_bf16(shape, [0, 0, 0, -8, -9, -12, -17], seed)


@pytest.mark.parametrize("kind", ["normal", "wide", "ties"])
@pytest.mark.parametrize("Kc", ADV_KC)
def test_transposed_tile_equals_the_plain_tile_on_stress_inputs(kind, Kc):
    """Five seeds per case. Rows 1, 8, 9, 16, 17, 64 take the transposed tile
    (both of its instances: B stored [K, N] for the forward, and K-major
    operands for the rhs-transposed forward and dA; at most 8 and at most 16
    rows with its narrow epilogues); rows 65 and 128 take the plain tile;
    all are compared with the same rows of a 256-row launch."""
    N = 192                                            # two column tiles, the second ragged
    for seed in range(5):
        base = 20000 + 100 * seed + Kc
        A = dev(_adversarial(kind, (256, Kc), base))
        B = dev(_adversarial(kind, (Kc, N), base + 1))
        Wt = dev(_adversarial(kind, (N, Kc), base + 2))
        dC = dev(_adversarial(kind, (256, Kc), base + 3))    # dA with contraction Kc
        Bd = dev(_adversarial(kind, (N, Kc), base + 4))      # dA = dC Bd^T: [256, N]
        full = dg.det_gemm_fwd(A, B)
        full_t = dg.det_gemm_fwd_rhs_transposed(A, Wt)
        full_da = dg.det_gemm_da(dC, Bd)
        for M in (1, 8, 9, 16, 17, 64, 65, 128):
            assert bits_equal(dg.det_gemm_fwd(A[:M], B), full[:M]), (kind, Kc, seed, M, "fwd")
            assert bits_equal(dg.det_gemm_fwd_rhs_transposed(A[:M], Wt), full_t[:M]), (kind, Kc, seed, M, "rhs_t")
            assert bits_equal(dg.det_gemm_da(dC[:M], Bd), full_da[:M]), (kind, Kc, seed, M, "da")
        check()
