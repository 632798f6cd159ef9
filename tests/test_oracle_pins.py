"""Pins of the CPU oracle against things other than itself.

Each test ties one part of the oracle (the BF16 rounding, the BF16 add, the
FP32 leaves, the mid-split tree, the strided GEMM and its entry-point
mappings) to exact rational arithmetic, closed forms, the page's stated
invariants, or hand-derived roots (tests/golden/). Definitions: RL-Kernel,
"Batch-Invariant Deterministic GEMM (det_gemm)", sections "Guarantees",
"Ascend NPU backend" and "Dtypes".
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact
import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_split_cases.txt")
LEAF_ORDER = os.path.join(os.path.dirname(__file__), "golden", "leaf_order_cases.txt")


def f32_bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


# ------------------------------------------------------------ rounding ----

def _special_f32():
    vals = [0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 3.4028235e38, 1e-40, -1e-40,
            1.1754944e-38, 2.0 ** -133, 2.0 ** -134, 2.0 ** -149]
    out = [np.float32(v) for v in vals]
    # exact ties: low 16 bits == 0x8000 with even and odd kept LSB
    for hi in (0x3F80, 0x3F81, 0x4049, 0xC049, 0x0001, 0x7F7F, 0x0080):
        out.append(np.uint32((hi << 16) | 0x8000).view(np.float32))
        out.append(np.uint32((hi << 16) | 0x7FFF).view(np.float32))
        out.append(np.uint32((hi << 16) | 0x8001).view(np.float32))
    return np.array(out, dtype=np.float32)


def test_round_bf16_matches_exact_rational_rounding():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        _special_f32(),
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-36).astype(np.float32),
        rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x = x[np.isfinite(x)]
    got = oracle.round_bf16(x)
    for xi, gi in zip(x, got):
        want = exact.rne_bf16_bits(exact.f32_to_value(xi))
        if xi == 0 and np.signbit(xi):
            want = 0x8000
        if exact.rne(exact.f32_to_value(xi)) == 0 and np.signbit(xi):
            want = 0x8000
        assert int(gi) == want, (float(xi), hex(int(gi)), hex(want))


def test_round_bf16_matches_torch_cast_and_keeps_nonfinite():
    rng = np.random.default_rng(2)
    x = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    got = oracle.round_bf16(x)
    ref = W.bits(torch.from_numpy(x.copy()).to(torch.bfloat16))
    fin = np.isfinite(x)
    assert np.array_equal(got[fin], ref[fin])
    nan = np.isnan(x)
    assert np.all(np.isnan(oracle.bf16_bits_to_f32(got[nan])))
    inf = np.isinf(x)
    assert np.array_equal(got[inf], ref[inf])


def test_add_bf16_matches_exact_rational_rounding():
    rng = np.random.default_rng(3)
    n = 6000
    a = rng.integers(0, 2 ** 16, n, dtype=np.uint32).astype(np.uint16)
    # b near a in exponent half the time, so that ties and cancellation occur
    b = np.where(rng.random(n) < 0.5,
                 rng.integers(0, 2 ** 16, n, dtype=np.uint32).astype(np.uint16),
                 (a.astype(np.int32) + rng.integers(-400, 400, n)).astype(np.uint16) ^
                 (rng.integers(0, 2, n).astype(np.uint16) << 15))
    a = np.concatenate([a, np.array([0x3F80, 0x3F80, 0x3F81, 0x7F7F, 0x0001], np.uint16)])
    b = np.concatenate([b, np.array([0x3B80, 0xBB80, 0x3B80, 0x7F7F, 0x8001], np.uint16)])
    got = oracle.add_bf16(a, b)
    checked = 0
    for ai, bi, gi in zip(a, b, got):
        va, vb = exact.bits_to_value(ai), exact.bits_to_value(bi)
        if isinstance(va, float) or isinstance(vb, float):
            continue  # inf/nan handled by IEEE float addition itself
        q = va + vb
        r = exact.rne(q)
        want = exact.value_to_bf16_bits(r)
        if r == 0:
            # exact zero sum: IEEE gives +0 except (-0) + (-0)
            want = 0x8000 if (ai == 0x8000 and bi == 0x8000) else 0x0000
            if q != 0:  # underflow to zero keeps the sign of the sum
                want = 0x8000 if q < 0 else 0x0000
        assert int(gi) == want, (hex(int(ai)), hex(int(bi)), hex(int(gi)), hex(want))
        checked += 1
    assert checked > 5000


# ------------------------------------------------------------- leaves -----

def test_leaves_within_sequential_error_bound_of_exact_sum():
    """|fl(sum) - sum| <= gamma_n * sum|x y| for recursive summation of n terms."""
    u = 2.0 ** -24
    for Kc in (1, 5, 31, 32, 33, 64, 95, 1000):
        X = W.bits(W.randn_bf16((3, Kc), 1.0, 10 + Kc))
        Y = W.bits(W.randn_bf16((Kc, 4), 1.0, 20 + Kc))
        xf = oracle.bf16_bits_to_f32(X).astype(np.float64)
        yf = oracle.bf16_bits_to_f32(Y).astype(np.float64)
        for i in range(3):
            for j in range(4):
                lv = oracle.leaves_f32(X, Y, i, j)
                assert lv.size == (Kc + 31) // 32
                for l in range(lv.size):
                    k0, k1 = 32 * l, min(32 * l + 32, Kc)
                    prods = xf[i, k0:k1] * yf[k0:k1, j]      # exact in double
                    s = math.fsum(prods)
                    n = k1 - k0
                    gamma = n * u / (1 - n * u)
                    bound = gamma * float(np.sum(np.abs(prods)))
                    assert abs(float(lv[l]) - s) <= bound * 1.0000001 + 1e-45, (Kc, i, j, l)


def test_single_leaf_gemm_is_rounded_dot_product():
    """Kc <= 32: one leaf, so C = RNE_bf16(FP32 dot). Where the exact dot is
    farther than the FP32 error bound from a BF16 rounding midpoint, that is
    RNE of the exact value; elsewhere C is one of the two neighbours."""
    u = 2.0 ** -24
    for Kc in (1, 7, 16, 32):
        X = W.bits(W.randn_bf16((16, Kc), 1.0, 100 + Kc))
        Y = W.bits(W.randn_bf16((Kc, 16), 1.0, 200 + Kc))
        C = oracle.fwd(X, Y)
        xf = [[exact.bits_to_value(v) for v in row] for row in X]
        yf = [[exact.bits_to_value(v) for v in row] for row in Y]
        for i in range(16):
            for j in range(16):
                prods = [xf[i][k] * yf[k][j] for k in range(Kc)]
                q = sum(prods, Fraction(0))
                bound = Fraction(Kc * u / (1 - Kc * u)) * sum(abs(p) for p in prods)
                lo, hi = exact.rne(q - bound), exact.rne(q + bound)
                got = exact.bits_to_value(int(C[i, j]))
                if lo == hi:
                    assert got == exact.rne(q), (Kc, i, j)
                else:
                    assert got in (lo, hi), (Kc, i, j)


def _leaf_order_rows():
    rows = []
    with open(LEAF_ORDER) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, x, y, leaf32, leaf16, _ = [p.strip() for p in line.split("|", 5)]
            rows.append((name, np.array([int(h, 16) for h in x.split()], np.uint16),
                         np.array([int(h, 16) for h in y.split()], np.uint16), int(leaf32, 16), int(leaf16, 16)))
    return rows


@pytest.mark.parametrize("case", _leaf_order_rows(), ids=lambda c: c[0])
def test_leaf_sums_its_products_in_ascending_k(case):
    """The FP32 leaf and the single-leaf products of every entry point match
    hand-derived sums in ascending k order (tests/golden/leaf_order_cases.txt,
    where a descending or pairwise loop gives other bits). dA and dB reach
    the same contraction through their own operand layouts."""
    _, x, y, leaf32, leaf16 = case
    Kc = x.size
    assert x.size == y.size <= 32
    X, Y = x[None, :], y[:, None]
    assert int(oracle.leaves_f32(X, Y, 0, 0)[0].view(np.uint32)) == leaf32
    assert int(f32_bits(oracle.fwd_fp32(X, Y))[0, 0]) == leaf32
    assert int(oracle.fwd(X, Y)[0, 0]) == leaf16
    assert int(oracle.fwd_rhs_transposed(X, y[None, :])[0, 0]) == leaf16
    # dA[0, 0] = sum_n dC[0, n] B[0, n]: dC = x as a row, B = y as a row
    assert int(oracle.da(X, y[None, :])[0, 0]) == leaf16
    # dB[0, 0] = sum_m A[m, 0] dC[m, 0]: the contraction runs down the rows
    A = np.ascontiguousarray(np.stack([x, np.zeros(Kc, np.uint16)], axis=1))
    dC = np.ascontiguousarray(np.stack([y, np.zeros(Kc, np.uint16)], axis=1))
    assert int(oracle.db(A, dC)[0, 0]) == leaf16
    assert int(oracle.db_transposed(A, dC)[0, 0]) == leaf16


# -------------------------------------------------------------- trees -----

def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, leaves, root, why = [p.strip() for p in line.split("|", 3)]
            rows.append((kind, [int(h, 16) for h in leaves.split()], int(root, 16), why))
    return rows


@pytest.mark.parametrize("case", _golden_rows(), ids=lambda c: c[0] + ":" + "-".join("%X" % v for v in c[1]))
def test_tree_hand_derived_roots(case):
    kind, leaves, root, _ = case
    if kind == "bf16":
        assert oracle.tree_bf16(np.array(leaves, np.uint16)) == root
    else:
        got = oracle.tree_f32(np.array(leaves, np.uint32).view(np.float32))
        assert int(np.float32(got).view(np.uint32)) == root


@pytest.mark.parametrize("case", [c for c in _golden_rows() if c[0] == "bf16"],
                         ids=lambda c: "-".join("%X" % v for v in c[1]))
def test_hand_derived_roots_through_the_whole_gemm(case):
    """The same roots through oracle.gemm: one row whose leaf l holds a single
    nonzero product equal to leaf value l (times 1.0)."""
    _, leaves, root, _ = case
    L = len(leaves)
    X = np.zeros((1, 32 * L), np.uint16)
    for l, h in enumerate(leaves):
        X[0, 32 * l + (l % 32)] = h
    Y = np.full((32 * L, 2), 0x3F80, np.uint16)
    C = oracle.fwd(X, Y)
    assert C[0, 0] == root and C[0, 1] == root


def _pairwise_levels_exact(leaves_bits):
    vals = [exact.bits_to_value(h) for h in leaves_bits]
    while len(vals) > 1:
        vals = [exact.rne(vals[2 * t] + vals[2 * t + 1]) for t in range(len(vals) // 2)]
    return exact.value_to_bf16_bits(vals[0])


def test_power_of_two_tree_is_level_by_level_pairwise_sum():
    """For L = 2^t every mid-split reading is the plain pairwise tree; compare
    with level-by-level pairwise sums rounded by exact rational RNE."""
    rng = np.random.default_rng(5)
    for t in range(0, 11):
        n = 2 ** t
        for rep in range(3):
            leaves = oracle.round_bf16(rng.standard_normal(n).astype(np.float32) * (rep + 1))
            want = _pairwise_levels_exact(leaves)
            got = oracle.tree_bf16(leaves)
            if want == 0:
                assert got in (0, 0x8000)
            else:
                assert got == want, (n, rep)


def test_half_k_gemm_is_a_child_of_the_tree():
    """A contiguous half-K GEMM is one child of the root (page: simulated TP=2
    a+b equals TP=1 bitwise), for every even L; quarters when L % 4 == 0."""
    for Kc in (64, 128, 192, 2048, 14336):
        M, N = 3, 5
        X = W.bits(W.randn_bf16((M, Kc), 1.0, 300 + Kc))
        Y = W.bits(W.randn_bf16((Kc, N), 0.02, 400 + Kc))
        full = oracle.fwd(X, Y)
        h = Kc // 2
        a = oracle.fwd(X[:, :h], Y[:h])
        b = oracle.fwd(X[:, h:], Y[h:])
        assert np.array_equal(oracle.add_bf16(a, b), full), Kc
        f32 = oracle.fwd_fp32(X, Y)
        a32 = oracle.fwd_fp32(X[:, :h], Y[:h])
        b32 = oracle.fwd_fp32(X[:, h:], Y[h:])
        assert np.array_equal(f32_bits(a32 + b32), f32_bits(f32)), Kc
        if (Kc // 32) % 4 == 0:
            q = Kc // 4
            parts = [oracle.fwd(X[:, i * q:(i + 1) * q], Y[i * q:(i + 1) * q]) for i in range(4)]
            merged = oracle.add_bf16(oracle.add_bf16(parts[0], parts[1]),
                                     oracle.add_bf16(parts[2], parts[3]))
            assert np.array_equal(merged, full), Kc


def test_half_k_is_not_a_child_when_leaf_count_is_odd_split():
    """Guard against a tree over a fixed power-of-two slot count: for L = 7
    (Kc = 224) the root splits 3 + 4 leaves, so the 96 / 128 split is a child
    and the 112 / 112 split is not (it cuts a leaf)."""
    X = W.bits(W.randn_bf16((8, 224), 1.0, 501))
    Y = W.bits(W.randn_bf16((224, 8), 1.0, 502))
    full = oracle.fwd(X, Y)
    a = oracle.fwd(X[:, :96], Y[:96])
    b = oracle.fwd(X[:, 96:], Y[96:])
    assert np.array_equal(oracle.add_bf16(a, b), full)


# ---------------------------------------------------- closed-form GEMMs ---

def test_all_ones_gives_kc_exactly():
    for Kc in (1, 31, 32, 256, 1000, 4096, 8192, 12288, 14336, 16384, 32768):
        X = np.full((2, Kc), 0x3F80, np.uint16)
        Y = np.full((Kc, 3), 0x3F80, np.uint16)
        C = oracle.fwd(X, Y)
        assert np.all(oracle.bf16_bits_to_f32(C) == Kc), Kc
        C32 = oracle.fwd_fp32(X, Y)
        assert np.all(C32 == Kc), Kc


def _identity_bits(n):
    I = np.zeros((n, n), np.uint16)
    I[np.arange(n), np.arange(n)] = 0x3F80
    return I


def test_identity_and_permutation_closed_forms():
    for Kc in (32, 100, 448):
        A = W.bits(W.randn_bf16((9, Kc), 1.0, 600 + Kc))
        I = _identity_bits(Kc)
        C = oracle.fwd(A, I)
        Af = oracle.bf16_bits_to_f32(A)
        assert np.array_equal(oracle.bf16_bits_to_f32(C), Af)   # -0 == +0 here
        B = W.bits(W.randn_bf16((Kc, 11), 1.0, 700 + Kc))
        C2 = oracle.fwd(I, B)
        assert np.array_equal(oracle.bf16_bits_to_f32(C2), oracle.bf16_bits_to_f32(B))
        perm = np.random.default_rng(Kc).permutation(Kc)
        P = np.zeros((Kc, Kc), np.uint16)
        P[perm, np.arange(Kc)] = 0x3F80          # (A P)[:, j] = A[:, perm[j]]
        C3 = oracle.fwd(A, P)
        assert np.array_equal(oracle.bf16_bits_to_f32(C3), Af[:, perm])
        C4 = oracle.fwd_fp32(A, P)
        assert np.array_equal(C4, Af[:, perm])


@pytest.mark.parametrize("Kc", [1, 33, 200, 256])
def test_small_integer_inputs_are_exact_for_every_entry_point(Kc):
    """Entries in {-1, 0, 1} and Kc <= 256 keep every leaf and every tree node
    an integer of magnitude <= 256, which BF16 holds exactly; so every entry
    point must equal the integer product of the operands as the page defines
    it (C = A B, dA = dC B^T, dB = A^T dC, rhs-transposed C = A W^T)."""
    M, N = 13, 10
    A = W.bits(W.randint_bf16((M, Kc), -1, 1, 800 + Kc))
    B = W.bits(W.randint_bf16((Kc, N), -1, 1, 900 + Kc))
    Wt = np.ascontiguousarray(B.T)
    dC = W.bits(W.randint_bf16((M, N), -1, 1, 1000 + Kc))
    Ai = oracle.bf16_bits_to_f32(A).astype(np.int64)
    Bi = oracle.bf16_bits_to_f32(B).astype(np.int64)
    dCi = oracle.bf16_bits_to_f32(dC).astype(np.int64)
    f = lambda h: oracle.bf16_bits_to_f32(h).astype(np.int64)
    assert np.array_equal(f(oracle.fwd(A, B)), Ai @ Bi)
    assert np.array_equal(f(oracle.fwd_rhs_transposed(A, Wt)), Ai @ Bi)
    assert np.array_equal(oracle.fwd_fp32(A, B).astype(np.int64), Ai @ Bi)
    assert np.array_equal(oracle.fwd_fp32_rhs_transposed(A, Wt).astype(np.int64), Ai @ Bi)
    # backward products: contraction over N (dA) and over M (dB)
    dCk = W.bits(W.randint_bf16((M, Kc), -1, 1, 1100 + Kc))   # dC of a [M, Kc] output
    Bk = W.bits(W.randint_bf16((N, Kc), -1, 1, 1200 + Kc))    # B [K=N, N=Kc]
    assert np.array_equal(f(oracle.da(dCk, Bk)), f(dCk) @ f(Bk).T)
    assert np.array_equal(f(oracle.db(A, np.ascontiguousarray(A))), Ai.T @ Ai)
    assert np.array_equal(f(oracle.db(dC, dC)), dCi.T @ dCi)
    assert np.array_equal(f(oracle.db_transposed(A, dC)), (Ai.T @ dCi).T)
    assert np.array_equal(f(oracle.db(A, dC)), Ai.T @ dCi)


def test_kc_zero_gives_positive_zero_and_kc_cap_is_enforced():
    X = np.zeros((3, 0), np.uint16)
    Y = np.zeros((0, 4), np.uint16)
    assert np.all(oracle.fwd(X, Y) == 0)
    assert np.all(f32_bits(oracle.fwd_fp32(X, Y)) == 0)
    Xb = np.zeros((1, 32769), np.uint16)
    Yb = np.zeros((32769, 1), np.uint16)
    with pytest.raises(ValueError):
        oracle.fwd(Xb, Yb)


def test_nan_propagates_to_its_row_only():
    A = W.bits(W.randn_bf16((4, 64), 1.0, 1300))
    B = W.bits(W.randn_bf16((64, 4), 1.0, 1301))
    A[2, 5] = 0x7FC0
    C = oracle.bf16_bits_to_f32(oracle.fwd(A, B))
    assert np.all(np.isnan(C[2])) and np.all(np.isfinite(C[[0, 1, 3]]))


def test_node_max_bounds_result_and_leaves():
    A = W.bits(W.randn_bf16((4, 300), 1.0, 1400))
    B = W.bits(W.randn_bf16((300, 6), 1.0, 1401))
    C, nm = oracle.gemm(A, B, with_node_max=True)
    Cf = oracle.bf16_bits_to_f32(C)
    assert np.all(nm >= np.abs(Cf))
    for i in range(4):
        for j in range(6):
            lv = np.abs(oracle.bf16_bits_to_f32(oracle.round_bf16(oracle.leaves_f32(A, B, i, j))))
            assert nm[i, j] >= lv.max()


def test_threads_do_not_change_bits():
    A = W.bits(W.randn_bf16((37, 500), 1.0, 1500))
    B = W.bits(W.randn_bf16((500, 9), 1.0, 1501))
    assert np.array_equal(oracle.gemm(A, B, threads=1), oracle.gemm(A, B, threads=7))


# -------------------------------------------------------------- RMSNorm --

def _ulp_bf16(v):
    v = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, (np.floor(np.log2(v)) - 7).astype(np.int64))


def test_rmsnorm_power_of_two_rows_give_the_weight_exactly():
    # x_j = +-2^k, eps = 0: every step is exact, x_j * r = +-1, so y_j = +-w_j.
    D = 96
    w = W.bits(W.randn_bf16((D,), 1.0, 31))
    for k in (-6, 0, 5):
        signs = np.where(np.arange(D) % 3 == 0, -1.0, 1.0)
        x = W.bits(torch.tensor(signs * 2.0 ** k, dtype=torch.float32).to(torch.bfloat16)).reshape(1, D)
        y = oracle.rmsnorm(x, w, 0.0)[0]
        want = np.where(signs < 0, w ^ 0x8000, w).astype(np.uint16)
        assert np.array_equal(y, want), k


def test_rmsnorm_is_invariant_to_power_of_two_scaling():
    # eps = 0: squares, sums, the mean and sqrt all scale exactly, r by 2^-k.
    x = W.randn_bf16((4, 1000), 1.0, 32)
    w = W.bits(W.randn_bf16((1000,), 1.0, 33))
    base = oracle.rmsnorm(W.bits(x), w, 0.0)
    for k in (-3, 4):
        scaled = W.bits((x.float() * 2.0 ** k).to(torch.bfloat16))
        assert np.array_equal(oracle.rmsnorm(scaled, w, 0.0), base), k


def test_rmsnorm_matches_the_exact_formula_within_one_bf16_ulp():
    x = W.randn_bf16((6, 4096), 1.0, 34)
    w = W.randn_bf16((4096,), 1.0, 35)
    eps = 1e-5
    y = oracle.bf16_bits_to_f32(oracle.rmsnorm(W.bits(x), W.bits(w), eps)).astype(np.float64)
    xd = x.double().numpy()
    wd = w.double().numpy()
    exact = xd / np.sqrt((xd * xd).mean(axis=1, keepdims=True) + eps) * wd
    # FP32 rounding before the final BF16 round is far below half a BF16 ulp
    assert np.all(np.abs(y - exact) <= _ulp_bf16(exact) * 0.5 + np.abs(exact) * 2.0 ** -20)


def test_rmsnorm_rows_are_independent_and_zero_rows_give_zero():
    x = W.bits(W.randn_bf16((5, 300), 1.0, 36))
    x[2] = 0
    w = W.bits(W.randn_bf16((300,), 1.0, 37))
    y = oracle.rmsnorm(x, w, 1e-6)
    for i in range(5):
        assert np.array_equal(oracle.rmsnorm(x[i:i + 1], w, 1e-6)[0], y[i])
    assert np.all((y[2] & 0x7FFF) == 0)          # +0 or -0 (0 * r * w keeps w's sign)


def test_rmsnorm_sum_of_squares_is_the_fp32_tree_of_the_row_with_itself():
    # With w = 1 and eps = 0, y_j = RNE_bf16(x_j * r) with r = 1 / sqrt(ss / D);
    # rebuild r from det_gemm's FP32 variant applied to the row and itself.
    D = 1000
    x = W.bits(W.randn_bf16((3, D), 1.0, 38))
    ones = W.bits(torch.ones(D, dtype=torch.bfloat16))
    y = oracle.rmsnorm(x, ones, 0.0)
    for i in range(3):
        ss = oracle.gemm(x[i:i + 1], np.ascontiguousarray(x[i:i + 1].T), out_fp32=True)[0, 0]
        m = np.float32(ss) / np.float32(D)
        r = np.float32(1.0) / np.sqrt(m, dtype=np.float32)
        want = oracle.round_bf16((oracle.bf16_bits_to_f32(x[i]) * r).astype(np.float32))
        assert np.array_equal(y[i], want), i


# -------------------------------------------------- grouped row reduction --

def test_rowdot_is_the_exact_dot_on_integer_inputs():
    # small integers: every product and partial sum is an exact FP32 integer,
    # so any order gives the exact dot product; a dropped or misplaced term,
    # a wrong row or a transposed operand does not
    C = W.bits(W.randint_bf16((7, 1000), -4, 4, 41))
    D = W.bits(W.randint_bf16((7, 1000), -4, 4, 42))
    got = oracle.rowdot(C, D)
    want = (oracle.bf16_bits_to_f32(C).astype(np.float64) * oracle.bf16_bits_to_f32(D)).sum(axis=1)
    assert np.array_equal(got.astype(np.float64), want)


def test_rowdot_order_separates_tiles_from_a_running_sum():
    # Three column tiles with dot values 1, 2^-24, 2^-24. The fixed order is
    # the mid-split tree over tiles: 1 + (2^-24 + 2^-24) = 1 + 2^-23 (exact);
    # a running sum would give (1 + 2^-24) + 2^-24 = 1 (ties to even twice).
    # The same products also fix the tile width: tiles of 256 columns give
    # slots 1 + 2^-24 = 1 and 2^-24, root 1; tiles of 64 give six slots
    # 1, 0, 2^-24, 0, 2^-24, 0 and the root (1 + (0 + 2^-24)) + (0 + (2^-24
    # + 0)) = 1.
    N = 3 * 128
    C = np.zeros((1, N), dtype=np.float32)
    D = np.zeros((1, N), dtype=np.float32)
    C[0, 0], D[0, 0] = 1.0, 1.0
    C[0, 128], D[0, 128] = 2.0 ** -12, 2.0 ** -12
    C[0, 256], D[0, 256] = 2.0 ** -12, 2.0 ** -12
    cb = W.bits(torch.from_numpy(C).to(torch.bfloat16))
    db = W.bits(torch.from_numpy(D).to(torch.bfloat16))
    assert oracle.rowdot(cb, db)[0] == np.float32(1.0 + 2.0 ** -23)


def _one_row(N, products):
    """BF16 bits of one row C and one row D whose products C[n] * D[n] are
    the given powers of two (column -> value), all other products zero."""
    C = np.zeros((1, N), dtype=np.float32)
    D = np.zeros((1, N), dtype=np.float32)
    for n, v in products.items():
        e = int(np.log2(v))
        C[0, n], D[0, n] = 2.0 ** (e // 2), 2.0 ** (e - e // 2)
    return (W.bits(torch.from_numpy(C).to(torch.bfloat16)), W.bits(torch.from_numpy(D).to(torch.bfloat16)))


def test_rowdot_sums_a_tile_in_ascending_column_order():
    """One 128-column tile holding 1 and 127 products 2^-24 (u = 2^-23).
    Ascending from column 0: each 1 + 2^-24 is a tie that stays 1, so the
    slot is 1. A descending sum gives 1 + 63.5u, a tie to the even 1 + 64u;
    32-column quarters merged in pairs give (1 + 16u) + 32u = 1 + 48u. With
    the 1 in the last column instead, ascending gives 127 x 2^-24 exactly,
    then 1 + 63.5u ties to 1 + 64u, and descending gives 1."""
    prods = {0: 1.0}
    prods.update({n: 2.0 ** -24 for n in range(1, 128)})
    c, d = _one_row(128, prods)
    assert int(f32_bits(oracle.rowdot(c, d))[0]) == 0x3F800000
    prods = {127: 1.0}
    prods.update({n: 2.0 ** -24 for n in range(0, 127)})
    c, d = _one_row(128, prods)
    assert int(f32_bits(oracle.rowdot(c, d))[0]) == 0x3F800040
