"""GPU invariance properties the page guarantees ("Guarantees": a fixed row
is bitwise identical across batch 1/N, chunked prefill on/off and padding
layouts; "Ascend NPU backend": numerics depend only on the row, never on M
or on block assignment). All comparisons are GPU against GPU, bitwise."""
import numpy as np
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import workloads as W
from gpu_util import check, dev

pytestmark = pytest.mark.gpu


def bits_equal(x, y):
    return torch.equal(x.contiguous().view(torch.int16), y.contiguous().view(torch.int16))


def test_tiny_rows_do_not_depend_on_m():
    A = dev(W.randn_bf16((64, 256), 1.0, W.seed_for(W.TINY, W.T_A)))
    B = dev(W.randn_bf16((256, 64), 1.0, W.seed_for(W.TINY, W.T_B)))
    dC = dev(W.randn_bf16((64, 64), 1.0, W.seed_for(W.TINY, W.T_DC)))
    Bt = B.t().contiguous()
    ref = dg.det_gemm_fwd(A, B)
    ref_da = dg.det_gemm_da(dC, B)
    ref_rt = dg.det_gemm_fwd_rhs_transposed(A, Bt)
    ref32 = dg.det_gemm_fwd_fp32(A, B)
    for M in (1, 7, 64):
        assert bits_equal(dg.det_gemm_fwd(A[:M], B), ref[:M]), M
        assert bits_equal(dg.det_gemm_da(dC[:M], B), ref_da[:M]), M
        assert bits_equal(dg.det_gemm_fwd_rhs_transposed(A[:M], Bt), ref_rt[:M]), M
        assert torch.equal(dg.det_gemm_fwd_fp32(A[:M], B), ref32[:M]), M
    check()


def test_a_row_gives_the_same_bits_at_every_position_of_a_tile():
    """One row copied to all 300 rows (every lane of a 128-row tile, three
    tiles): all output rows must be identical; and permuting distinct rows
    permutes the output rows."""
    K, N = 1000, 200
    x = W.randn_bf16((1, K), 1.0, 8001)
    B = dev(W.randn_bf16((K, N), 1.0, 8002))
    A = dev(x.expand(300, K).contiguous())
    C = dg.det_gemm_fwd(A, B)
    assert bits_equal(C, C[:1].expand_as(C))
    A2 = dev(W.randn_bf16((300, K), 1.0, 8003))
    perm = torch.from_numpy(np.random.default_rng(0).permutation(300)).to("cuda")
    assert bits_equal(dg.det_gemm_fwd(A2[perm], B), dg.det_gemm_fwd(A2, B)[perm])
    check()


def test_chunked_rows_and_padding_rows_do_not_change_bits():
    """Rows processed in chunks, or surrounded by zero rows or by rows of
    random 16-bit patterns (NaN and Inf included), keep their bits."""
    M, K, N = 500, 2048, 384
    A = dev(W.randn_bf16((M, K), 1.0, 8101))
    B = dev(W.randn_bf16((K, N), 0.02, 8102))
    full = dg.det_gemm_fwd(A, B)
    chunks = torch.cat([dg.det_gemm_fwd(A[i:i + 96], B) for i in range(0, M, 96)])
    assert bits_equal(chunks, full)
    pad_to = 640
    zeros = torch.zeros(pad_to - M, K, dtype=torch.bfloat16, device="cuda")
    garbage = dev(W.garbage_bf16((pad_to - M, K), 8103))
    for pad in (zeros, garbage):
        C = dg.det_gemm_fwd(torch.cat([A, pad]), B)
        assert bits_equal(C[:M], full)
        C = dg.det_gemm_fwd(torch.cat([pad, A]), B)
        assert bits_equal(C[pad_to - M:], full)
    check()


def test_output_guard_bands_stay_untouched():
    """Outputs inside a larger buffer (ldc > N, rows around it): only the
    [M, N] window is written."""
    M, N, K = 130, 72, 96
    A = dev(W.randn_bf16((M, K), 1.0, 8201))
    B = dev(W.randn_bf16((K, N), 1.0, 8202))
    big = torch.full((M + 8, N + 24), -7.0, dtype=torch.bfloat16, device="cuda")
    view = big[4:4 + M, 8:8 + N]
    dg.det_gemm_fwd(A, B, out=view)
    ref = dg.det_gemm_fwd(A, B)
    check()
    assert bits_equal(view, ref)
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[4:4 + M, 8:8 + N] = False
    assert torch.all(big[mask] == -7.0)
    big32 = torch.full((M + 8, N + 24), -7.0, dtype=torch.float32, device="cuda")
    v32 = big32[4:4 + M, 8:8 + N]
    dg.det_gemm_fwd_fp32(A, B, out=v32)
    check()
    assert torch.all(big32[mask] == -7.0)
    assert torch.equal(v32, dg.det_gemm_fwd_fp32(A, B))


def test_forced_timeout_is_reported_and_the_context_survives():
    A = dev(W.randn_bf16((256, 512), 1.0, 8301))
    B = dev(W.randn_bf16((512, 256), 1.0, 8302))
    ref = dg.det_gemm_fwd(A, B)
    assert dg.det_gemm_check() == 0
    dg.det_gemm_debug_force_timeout(True)
    try:
        dg.det_gemm_fwd(A, B)
        st = dg.det_gemm_check()
    finally:
        dg.det_gemm_debug_force_timeout(False)
    assert st == 6, dg.status_string(st)
    assert dg.det_gemm_check() == 0          # the check cleared it
    again = dg.det_gemm_fwd(A, B)
    check()
    assert bits_equal(again, ref)


def test_bad_device_arguments_raise_before_launch():
    A = dev(W.randn_bf16((64, 72), 1.0, 8401))
    B = dev(W.randn_bf16((72, 64), 1.0, 8402))
    with pytest.raises(dg.DetGemmError) as e:
        dg.det_gemm_fwd(A[:, 1:], B[1:])      # base pointer off by 2 bytes
    assert e.value.status == 3
    A2 = W.randn_bf16((64, 36), 1.0, 8403).to("cuda")   # 72-byte rows: pitch not a multiple of 16
    with pytest.raises(dg.DetGemmError) as e:
        dg.det_gemm_fwd(A2, B[:36])
    assert e.value.status == 3
    check()
