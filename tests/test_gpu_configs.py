"""The page's workloads at full size (RL-Kernel, "Batch-Invariant Deterministic
GEMM (det_gemm)", section "Why": QKV, MLP and LM-head matmuls of a 4096-hidden
transformer; "Guarantees": batch, chunked-prefill and padding invariance;
"Ascend NPU backend": the half-K TP property and the 32768 cap).

Every launch runs in the configuration the bench times. Results are checked
bitwise against the GPU itself where the page promises invariance, and
against the CPU oracle on sampled rows (and sampled columns where a full row
is too long for the oracle), within the tolerance derived in gpu_util."""
import numpy as np
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W
from gpu_util import assert_bf16_close, assert_f32_close, check, f32

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def bits_equal(x, y):
    return torch.equal(x.contiguous().view(torch.int16), y.contiguous().view(torch.int16))


def oracle_rows(X, Y, rows, out_fp32=False, cols=None):
    """Oracle on rows `rows` of X @ Y (and columns `cols` if given)."""
    Xs = np.ascontiguousarray(X[rows])
    Ys = Y if cols is None else Y[:, cols]
    return oracle.gemm(Xs, Ys, out_fp32=out_fp32, with_node_max=not out_fp32)


def check_rows(got, X, Y, rows, L, what, cols=None):
    want, nodemax = oracle_rows(X, Y, rows, cols=cols)
    g = got[rows] if cols is None else got[rows][:, cols]
    return assert_bf16_close(g, want, nodemax, L, what)


def test_qkv_rows_are_identical_for_every_batch_size():
    K, N = 4096, 12288
    A = W.randn_bf16((4096, K), W.STD_ACT, W.seed_for(W.QKV, W.T_A))
    B = W.randn_bf16((K, N), W.STD_W, W.seed_for(W.QKV, W.T_B))
    Ag, Bg = A.cuda(), B.cuda()
    full = dg.det_gemm_fwd(Ag, Bg)
    for M in (1, 3, 17, 256, 1024):
        assert bits_equal(dg.det_gemm_fwd(Ag[:M], Bg), full[:M]), M
    check()
    rows = [0, 1, 2, 16, 255, 1023, 4095]
    check_rows(W.bits(full), W.bits(A), W.bits(B), rows, K // 32, "qkv")


def test_mlp_forward_and_backward_against_oracle_rows():
    M, D, F = 8192, 4096, 14336
    x = W.randn_bf16((M, D), W.STD_ACT, W.seed_for(W.MLP, W.T_A))
    w_up = W.randn_bf16((D, F), W.STD_W, W.seed_for(W.MLP, W.T_B))
    w_down = W.randn_bf16((F, D), W.STD_W, W.seed_for(W.MLP, W.T_B) + 100)
    dy = W.randn_bf16((M, D), W.STD_DC, W.seed_for(W.MLP, W.T_DC))
    xg, wug, wdg, dyg = x.cuda(), w_up.cuda(), w_down.cuda(), dy.cuda()
    h = dg.det_gemm_fwd(xg, wug)                      # [M, F]
    y = dg.det_gemm_fwd_fp32(h, wdg)                  # [M, D]
    dh = dg.det_gemm_da(dyg, wdg)                     # [M, F] = dy w_down^T
    dwd = dg.det_gemm_db(h, dyg)                      # [F, D] = h^T dy
    dx = dg.det_gemm_da(dh, wug)                      # [M, D] = dh w_up^T
    dwu = dg.det_gemm_db(xg, dh)                      # [D, F] = x^T dh
    dwu_t = dg.det_gemm_db_transposed(xg, dh)         # [F, D]
    check()
    assert bits_equal(dwu_t, dwu.t())
    xb, wub, wdb, dyb = W.bits(x), W.bits(w_up), W.bits(w_down), W.bits(dy)
    hb, dhb = W.bits(h), W.bits(dh)
    rows = [0, 127, 128, 8191]
    check_rows(hb, xb, wub, rows, D // 32, "fwd up")
    want32 = oracle.gemm(np.ascontiguousarray(hb[rows]), wdb, out_fp32=True)
    absprod = np.abs(f32(hb[rows]).astype(np.float64)) @ np.abs(f32(wdb).astype(np.float64))
    assert_f32_close(y.cpu().numpy()[rows], want32, absprod, "fwd_fp32 down")
    check_rows(W.bits(dh), dyb, wdb.T, rows, D // 32, "da down")
    check_rows(W.bits(dx), dhb, wub.T, rows, F // 32, "da up")
    check_rows(W.bits(dwd), hb.T, dyb, [0, 5000, F - 1], M // 32, "db down")
    check_rows(W.bits(dwu), xb.T, dhb, [0, 2047, D - 1], M // 32, "db up")


def test_lm_head_bf16_and_fp32_against_oracle_samples():
    M, K, V = 2048, 4096, 151936
    A = W.randn_bf16((M, K), W.STD_ACT, W.seed_for(W.LMHEAD, W.T_A))
    Wt = W.randn_bf16((V, K), W.STD_W, W.seed_for(W.LMHEAD, W.T_B))   # weight stored [V, K]
    Ag, Wg = A.cuda(), Wt.cuda()
    C = dg.det_gemm_fwd_rhs_transposed(Ag, Wg)
    C32 = dg.det_gemm_fwd_fp32_rhs_transposed(Ag, Wg)
    part = dg.det_gemm_fwd_rhs_transposed(Ag[100:612], Wg)
    check()
    assert bits_equal(part, C[100:612])
    # decode-sized slices take the transposed tile, about eight 128-column
    # tiles per CTA
    for lo, hi in ((100, 101), (100, 112), (100, 164)):
        assert bits_equal(dg.det_gemm_fwd_rhs_transposed(Ag[lo:hi], Wg), C[lo:hi]), (lo, hi)
    check()
    rows = [0, 1000, 2047]
    cols = np.sort(np.random.default_rng(0).choice(V, 3000, replace=False))
    Ab, Wb = W.bits(A), W.bits(Wt)
    check_rows(W.bits(C), Ab, Wb.T, rows, K // 32, "lm head bf16", cols=cols)
    want32 = oracle.gemm(np.ascontiguousarray(Ab[rows]), Wb.T[:, cols], out_fp32=True)
    absprod = np.abs(f32(Ab[rows]).astype(np.float64)) @ np.abs(f32(Wb.T[:, cols]).astype(np.float64))
    assert_f32_close(C32.cpu().numpy()[rows][:, cols], want32, absprod, "lm head fp32")


def test_long_k_chunking_padding_and_half_k():
    M, K, N = 4096, 32768, 4096
    A = W.randn_bf16((M, K), 1.0, W.seed_for(W.LONGK, W.T_A))
    B = W.randn_bf16((K, N), 1.0, W.seed_for(W.LONGK, W.T_B))
    Ag, Bg = A.cuda(), B.cuda()
    full = dg.det_gemm_fwd(Ag, Bg)
    # chunked prefill: eight chunks of 512 rows
    chunks = torch.cat([dg.det_gemm_fwd(Ag[i:i + 512], Bg) for i in range(0, M, 512)])
    assert bits_equal(chunks, full)
    # ragged 500-row chunks padded to a multiple of 128 rows with zero rows
    # and, separately, with rows of random 16-bit patterns
    garbage = W.garbage_bf16((12, K), W.seed_for(W.LONGK, W.T_GARBAGE)).cuda()
    for pad in (torch.zeros(12, K, dtype=torch.bfloat16, device="cuda"), garbage):
        for i in range(0, 1500, 500):
            Cp = dg.det_gemm_fwd(torch.cat([Ag[i:i + 500], pad]), Bg)
            assert bits_equal(Cp[:500], full[i:i + 500]), i
    # tensor parallelism simulated on one GPU: two contiguous half-K GEMMs
    # are the two children of the root
    h = K // 2
    lo = W.bits(dg.det_gemm_fwd(Ag[:, :h], Bg[:h]))
    hi = W.bits(dg.det_gemm_fwd(Ag[:, h:], Bg[h:]))
    check()
    fb = W.bits(full)
    assert np.array_equal(oracle.add_bf16(lo, hi), fb)
    check_rows(fb, W.bits(A), W.bits(B), [0, 4095], K // 32, "long K")
