"""GPU parity: every C-ABI entry point against the CPU oracle, element by
element, on seeded inputs that span several tiles and ragged tails.

Exact-arithmetic inputs (small integers) must match the oracle bit for bit:
every product and every partial sum inside a leaf is then exact in FP32, so
the tensor core's summation order cannot matter. Normal inputs must match
within one BF16 ulp (FP32 output: 2^-20 relative to |A||B|), the
spec tolerance; the only difference is the FP32 summation order
inside a leaf ("Ascend NPU backend", last bullet). The leaf-decomposition
test then pins the tree and the epilogue exactly: the GPU result equals the
oracle's tree applied to the GPU's own rounded leaves."""
import numpy as np
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W
from gpu_util import assert_bf16_close, assert_f32_close, check, dev, exact_equal, f32

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed, kind="randn"):
    if kind == "int":
        A = W.randint_bf16((M, K), -8, 8, seed)
        B = W.randint_bf16((K, N), -8, 8, seed + 1)
        dC = W.randint_bf16((M, N), -8, 8, seed + 2)
    else:
        A = W.randn_bf16((M, K), 1.0, seed)
        B = W.randn_bf16((K, N), 1.0, seed + 1)
        dC = W.randn_bf16((M, N), 1.0, seed + 2)
    return A, B, dC


def _run_all(A, B, dC):
    """Every entry point on the GPU; returns {name: numpy result}."""
    Ag, Bg, dCg = dev(A), dev(B), dev(dC)
    Wg = dev(B.t().contiguous())      # the weight stored [N, K]
    out = {
        "fwd": dg.det_gemm_fwd(Ag, Bg),
        "fwd_rhs_transposed": dg.det_gemm_fwd_rhs_transposed(Ag, Wg),
        "fwd_fp32": dg.det_gemm_fwd_fp32(Ag, Bg),
        "fwd_fp32_rhs_transposed": dg.det_gemm_fwd_fp32_rhs_transposed(Ag, Wg),
        "da": dg.det_gemm_da(dCg, Bg),
        "db": dg.det_gemm_db(Ag, dCg),
        "db_transposed": dg.det_gemm_db_transposed(Ag, dCg),
    }
    check()
    res = {}
    for k, v in out.items():
        res[k] = v.cpu().numpy() if v.dtype == torch.float32 else W.bits(v)
    return res


def _oracle_all(A, B, dC):
    a, b, g = W.bits(A), W.bits(B), W.bits(dC)
    w = np.ascontiguousarray(b.T)
    af, bf, gf = (np.abs(f32(x).astype(np.float64)) for x in (a, b, g))
    return {
        "fwd": oracle.fwd(a, b, with_node_max=True),
        "fwd_rhs_transposed": oracle.fwd_rhs_transposed(a, w, with_node_max=True),
        "fwd_fp32": (oracle.fwd_fp32(a, b), af @ bf),
        "fwd_fp32_rhs_transposed": (oracle.fwd_fp32_rhs_transposed(a, w), af @ bf),
        "da": oracle.da(g, b, with_node_max=True),
        "db": oracle.db(a, g, with_node_max=True),
        "db_transposed": oracle.db_transposed(a, g, with_node_max=True),
    }


SHAPES = [
    (1, 64, 256), (7, 64, 256), (64, 64, 256),      # the tiny workload
    (300, 200, 1000),                              # several tiles, ragged M, N and last leaf
    (129, 65, 33),                                 # one row / one column past a tile, Kc = 33
    (5, 24, 7),                                    # everything smaller than a tile and a leaf
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_integer_inputs_match_oracle_bit_for_bit(M, N, K):
    A, B, dC = _operands(M, N, K, 2000 + M + N + K, "int")
    got = _run_all(A, B, dC)
    want = _oracle_all(A, B, dC)
    for name, g in got.items():
        w = want[name][0]
        if g.dtype == np.float32:
            assert np.array_equal(g, w), name
        else:
            assert exact_equal(g, w), name


@pytest.mark.parametrize("M,N,K", SHAPES + [(130, 136, 14336)])
def test_normal_inputs_within_one_ulp_of_oracle(M, N, K):
    A, B, dC = _operands(M, N, K, 3000 + M + N + K)
    got = _run_all(A, B, dC)
    want = _oracle_all(A, B, dC)
    kc = {"da": N, "db": M, "db_transposed": M}
    for name, g in got.items():
        if g.dtype == np.float32:
            assert_f32_close(g, want[name][0], want[name][1], name)
        else:
            L = (kc.get(name, K) + 31) // 32
            assert_bf16_close(g, want[name][0], want[name][1], L, "%s %dx%dx%d" % (name, M, N, K))


@pytest.mark.parametrize("M,N,K", [(150, 140, 224), (40, 130, 1000), (17, 33, 4096), (9, 20, 14336)])
def test_result_is_the_oracle_tree_over_the_gpu_leaves(M, N, K):
    """C_gpu == tree(leaves_gpu) exactly, where leaves_gpu[l] is the GPU's
    BF16 result on the single leaf l alone (a one-leaf product is its own
    root); and every GPU leaf is within one leaf-ulp of the oracle's.
    K = 14336 is 448 leaves: the tree's ranges of 7 leaves split 3 + 4."""
    A, B, _ = _operands(M, N, K, 4000 + K)
    Ag, Bg = dev(A), dev(B)
    C = W.bits(dg.det_gemm_fwd(Ag, Bg))
    L = (K + 31) // 32
    leaves = np.stack([W.bits(dg.det_gemm_fwd(Ag[:, 32 * l:min(32 * l + 32, K)],
                                              Bg[32 * l:min(32 * l + 32, K)])) for l in range(L)], axis=-1)
    check()
    for i in range(M):
        for j in range(N):
            assert oracle.tree_bf16(leaves[i, j]) == C[i, j], (i, j)
    a, b = W.bits(A), W.bits(B)
    rng = np.random.default_rng(K)
    for _ in range(64):
        i, j = int(rng.integers(M)), int(rng.integers(N))
        lo = oracle.round_bf16(oracle.leaves_f32(a, b, i, j))
        d = np.abs(f32(leaves[i, j]).astype(np.float64) - f32(lo))
        from gpu_util import ulp_bf16
        assert np.all(d <= ulp_bf16(np.abs(f32(lo)))), (i, j)


def test_half_k_merge_equals_full_k_bitwise():
    M, N, K = 200, 136, 2048
    A, B, _ = _operands(M, N, K, 5000)
    Ag, Bg = dev(A), dev(B)
    full = W.bits(dg.det_gemm_fwd(Ag, Bg))
    h = K // 2
    a = W.bits(dg.det_gemm_fwd(Ag[:, :h], Bg[:h]))
    b = W.bits(dg.det_gemm_fwd(Ag[:, h:], Bg[h:]))
    check()
    assert np.array_equal(oracle.add_bf16(a, b), full)


def test_transposition_identities_bitwise():
    M, N, K = 160, 144, 320
    A, B, dC = _operands(M, N, K, 6000)
    Ag, Bg, dCg = dev(A), dev(B), dev(dC)
    Wg = Bg.t().contiguous()
    fwd = dg.det_gemm_fwd
    assert torch.equal(dg.det_gemm_fwd_rhs_transposed(Ag, Wg).view(torch.int16), fwd(Ag, Bg).view(torch.int16))
    assert torch.equal(dg.det_gemm_da(dCg, Bg).view(torch.int16),
                       fwd(dCg, Bg.t().contiguous()).view(torch.int16))
    db = dg.det_gemm_db(Ag, dCg)
    assert torch.equal(db.view(torch.int16), fwd(Ag.t().contiguous(), dCg).view(torch.int16))
    assert torch.equal(dg.det_gemm_db_transposed(Ag, dCg).view(torch.int16), db.t().contiguous().view(torch.int16))
    f1 = dg.det_gemm_fwd_fp32(Ag, Bg)
    assert torch.equal(dg.det_gemm_fwd_fp32_rhs_transposed(Ag, Wg), f1)
    check()


def test_repeated_runs_are_bitwise_identical():
    M, N, K = 256, 256, 2000
    A, B, dC = _operands(M, N, K, 7000)
    first = _run_all(A, B, dC)
    for _ in range(2):
        again = _run_all(A, B, dC)
        for k in first:
            assert np.array_equal(first[k].view(np.uint8), again[k].view(np.uint8)), k


def test_kc_zero_writes_positive_zero():
    A = dev(torch.zeros(5, 0, dtype=torch.bfloat16))
    B = dev(torch.zeros(0, 9, dtype=torch.bfloat16))
    C = dev(torch.full((5, 9), 3.0, dtype=torch.bfloat16))
    dg.det_gemm_fwd(A, B, out=C)
    C32 = dg.det_gemm_fwd_fp32(A, B)
    check()
    assert torch.all(C.view(torch.int16) == 0) and torch.all(C32.view(torch.int32) == 0)
