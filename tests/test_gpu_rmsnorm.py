"""det_rmsnorm on the GPU: bit for bit the oracle's RMSNorm (every step is a
single round-to-nearest operation in a fixed order), and a row's bits do not
depend on how many rows are normalised with it ("Comment vaincre le
non-déterminisme dans l'inférence des LLM", section "RMSNorm")."""
import numpy as np
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W
from gpu_util import check, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [8, 100, 1000, 4096, 5120, 32768])
@pytest.mark.parametrize("eps", [1e-6, 0.0])
def test_rmsnorm_matches_the_oracle_bit_for_bit(D, eps):
    M = 37 if D <= 5120 else 5
    x = W.randn_bf16((M, D), 1.0, 9100 + D)
    w = W.randn_bf16((D,), 1.0, 9200 + D)
    y = dg.det_rmsnorm(dev(x), w.cuda(), eps)
    check()
    want = oracle.rmsnorm(W.bits(x), W.bits(w), eps)
    assert np.array_equal(W.bits(y.cpu()), want)


def test_rmsnorm_rows_do_not_depend_on_the_batch_and_in_place_is_the_same():
    D = 4096
    x = W.randn_bf16((513, D), 3.0, 9301).cuda()
    w = W.randn_bf16((D,), 0.5, 9302).cuda()
    full = dg.det_rmsnorm(x, w, 1e-5)
    for M in (1, 7, 64, 129):
        assert torch.equal(dg.det_rmsnorm(x[:M], w, 1e-5).view(torch.int16), full[:M].view(torch.int16)), M
    y = x.clone()
    dg.det_rmsnorm(y, w, 1e-5, out=y)
    check()
    assert torch.equal(y.view(torch.int16), full.view(torch.int16))


def test_rmsnorm_of_zero_and_extreme_rows():
    D = 256
    x = W.randn_bf16((4, D), 1.0, 9401)
    x[0] = 0.0
    x[1] = 2.0 ** 100          # squares near the top of the FP32 range
    x[2] = 2.0 ** -60          # squares below the FP32 normal range
    w = W.randn_bf16((D,), 1.0, 9402)
    for eps in (1e-6, 0.0):
        y = dg.det_rmsnorm(x.cuda(), w.cuda(), eps)
        check()
        want = oracle.rmsnorm(W.bits(x), W.bits(w), eps)
        got = W.bits(y.cpu())
        nan_g = np.isnan(oracle.bf16_bits_to_f32(got))
        nan_w = np.isnan(oracle.bf16_bits_to_f32(want))
        assert np.array_equal(nan_g, nan_w), eps
        assert np.array_equal(got[~nan_w], want[~nan_w]), eps
