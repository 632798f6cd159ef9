"""Bit-for-bit oracle parity where the deepest pending partials are live.

The kernels keep the merge tree's pending left children ("slots") in
registers, TMEM, shared memory and, for the ones touched least often, a
per-CTA scratch in global memory. The deepest slots hold nodes of height 8
and up, so they are only used by contractions of more than 128 leaves
(Kc > 4096); a launch with few output tiles would split its contraction at
tree nodes instead (fewer leaves per work unit). Here every launch has
exactly one output tile per SM, which the library never splits, so each
CTA walks the whole contraction: 130, 448, 625 and 1024 leaves (the page's
32768 cap, RL-Kernel "Batch-Invariant Deterministic GEMM (det_gemm)",
section "Dtypes").

The inputs are integers in [-3, 3]: every FP32 leaf sum is then exact
whatever order the tensor core adds in, so the GPU must equal the oracle
bit for bit, while the leaf roundings and the tree's BF16 adds still round
(leaf sums reach 288, beyond BF16's 8 significant bits). The operands are a
gigabyte or more, so they are drawn on the device from a seeded generator
and the oracle checks sampled rows and columns: the first and last, both
sides of the first tile edge, and random ones across every tile. Every
kernel instance of the plain tiles is covered: the BF16 forward (and the
allocation-free forward), dA, dB and dB stored [N, K], both FP32-output
instances and the grouped launch."""
import numpy as np
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W
from gpu_util import check, exact_equal

pytestmark = pytest.mark.gpu

KCS = [4160, 14336, 20000, 32768]      # 130, 448 (7 -> 3 + 4 splits), 625 (odd) and 1024 leaves


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    idx = {0, n - 1, min(127, n - 1), min(128, n - 1)} | set(int(x) for x in rng.integers(0, n, k))
    return torch.tensor(sorted(idx), dtype=torch.long)


def _host_bits(t):
    return W.bits(t.contiguous().cpu())


@pytest.mark.parametrize("Kc", KCS)
def test_bf16_forward_and_the_allocation_free_forward(Kc):
    M, N = 128, 128 * _sms()                           # one 128 x 128 tile per SM
    A = W.randint_bf16_cuda((M, Kc), -3, 3, 12000 + Kc)
    B = W.randint_bf16_cuda((Kc, N), -3, 3, 12100 + Kc)
    C = dg.det_gemm_fwd(A, B)
    C2 = torch.empty_like(C)
    dg.det_gemm_fwd_noalloc(A, B, C2)
    check()
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
    r, c = _sample(M, 6, Kc), _sample(N, 60, Kc + 1)
    want = oracle.fwd(_host_bits(A[r]), _host_bits(B[:, c]))
    assert exact_equal(_host_bits(C[r][:, c]), want), Kc


@pytest.mark.parametrize("Kc", KCS)
def test_fp32_forward(Kc):
    M, N = 128, 96 * _sms()                            # one 128 x 96 FP32 tile per SM
    A = W.randint_bf16_cuda((M, Kc), -3, 3, 12200 + Kc)
    B = W.randint_bf16_cuda((Kc, N), -3, 3, 12300 + Kc)
    C = dg.det_gemm_fwd_fp32(A, B)
    check()
    r, c = _sample(M, 6, Kc), _sample(N, 60, Kc + 2)
    want = oracle.fwd_fp32(_host_bits(A[r]), _host_bits(B[:, c]))
    got = C[r][:, c].cpu().numpy()
    # exact inputs: every partial sum is an integer below 2^24, so values agree
    assert np.array_equal(got, want), Kc


@pytest.mark.parametrize("Kc", KCS)
def test_da(Kc):
    # dA[m, k] = sum_n dC[m, n] B[k, n]: the contraction is the forward N
    M, Kout = 128, 128 * _sms()
    dC = W.randint_bf16_cuda((M, Kc), -3, 3, 12400 + Kc)
    B = W.randint_bf16_cuda((Kout, Kc), -3, 3, 12500 + Kc)
    dA = dg.det_gemm_da(dC, B)
    check()
    r, c = _sample(M, 6, Kc), _sample(Kout, 60, Kc + 3)
    want = oracle.da(_host_bits(dC[r]), _host_bits(B[c]))
    assert exact_equal(_host_bits(dA[r][:, c]), want), Kc


@pytest.mark.parametrize("Kc", KCS)
def test_db_and_db_transposed(Kc):
    # dB[k, n] = sum_m A[m, k] dC[m, n]: the contraction is the forward M
    Kout, N = 128, 128 * _sms()
    A = W.randint_bf16_cuda((Kc, Kout), -3, 3, 12600 + Kc)
    dC = W.randint_bf16_cuda((Kc, N), -3, 3, 12700 + Kc)
    dB = dg.det_gemm_db(A, dC)
    check()
    r, c = _sample(Kout, 6, Kc), _sample(N, 60, Kc + 4)
    a_r, dc_c = _host_bits(A[:, r]), _host_bits(dC[:, c])
    assert exact_equal(_host_bits(dB[r][:, c]), oracle.db(a_r, dc_c)), Kc
    # dB stored [N, K]: its rows are the columns n, one 128 x 128 tile per SM
    A2 = W.randint_bf16_cuda((Kc, 128), -3, 3, 12800 + Kc)
    dC2 = W.randint_bf16_cuda((Kc, N), -3, 3, 12900 + Kc)
    dBt = dg.det_gemm_db_transposed(A2, dC2)
    check()
    want_t = oracle.db_transposed(_host_bits(A2[:, r]), _host_bits(dC2[:, c]))
    assert exact_equal(_host_bits(dBt[c][:, r]), want_t), Kc


@pytest.mark.parametrize("Kc", KCS)
def test_fp32_rhs_transposed(Kc):
    # the FP32-output instance with a K-major weight stored [N, K]
    M, N = 128, 96 * _sms()
    A = W.randint_bf16_cuda((M, Kc), -3, 3, 13000 + Kc)
    Wt = W.randint_bf16_cuda((N, Kc), -3, 3, 13100 + Kc)
    C = dg.det_gemm_fwd_fp32_rhs_transposed(A, Wt)
    check()
    r, c = _sample(M, 6, Kc), _sample(N, 60, Kc + 5)
    want = oracle.fwd_fp32_rhs_transposed(_host_bits(A[r]), _host_bits(Wt[c]))
    assert np.array_equal(C[r][:, c].cpu().numpy(), want), Kc


@pytest.mark.parametrize("Kc", [4160, 14336])
def test_grouped(Kc):
    # two groups of one row tile each, N wide enough for one tile per SM in all
    N = 64 * _sms()
    As = [W.randint_bf16_cuda((128, Kc), -3, 3, 13200 + Kc + g) for g in range(2)]
    Bs = [W.randint_bf16_cuda((Kc, N), -3, 3, 13300 + Kc + g) for g in range(2)]
    Cs = dg.det_gemm_fwd_grouped(As, Bs)
    check()
    for g in range(2):
        r, c = _sample(128, 6, Kc + g), _sample(N, 40, Kc + 6 + g)
        want = oracle.fwd(_host_bits(As[g][r]), _host_bits(Bs[g][:, c]))
        assert exact_equal(_host_bits(Cs[g][r][:, c]), want), (Kc, g)
