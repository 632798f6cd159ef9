"""det_gemm_fwd_grouped: mixture-of-experts expert GEMMs in one launch.
Each group's product is det_gemm_fwd's bit for bit (a token's result does
not depend on how many tokens its expert received), and the optional row
reduction is the oracle's fixed-order one bit for bit (Megatron Core notes,
"Kernel redesign: the grouped-GEMM epilogue": private per-tile slots and a
fixed reduction tree instead of atomics across N-tiles)."""
import numpy as np
import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W
from gpu_util import check

pytestmark = pytest.mark.gpu


def bits(t):
    return t.contiguous().view(torch.int16)


@pytest.mark.parametrize("G", [1, 3, 8, 11])
def test_grouped_products_equal_det_gemm_fwd_per_group(G):
    K, N = 1024, 768
    rng = np.random.default_rng(G)
    Ms = [int(m) for m in rng.integers(0, 700, size=G)]
    Ms[0] = max(Ms[0], 1)
    As = [W.randn_bf16((m, K), 1.0, 9500 + 10 * G + g).cuda() for g, m in enumerate(Ms)]
    Bs = [W.randn_bf16((K, N), 0.02, 9600 + 10 * G + g).cuda() for g in range(G)]
    Cs = dg.det_gemm_fwd_grouped(As, Bs)
    check()
    for g in range(G):
        assert bits(Cs[g]).shape == (Ms[g], N)
        if Ms[g]:
            assert torch.equal(bits(Cs[g]), bits(dg.det_gemm_fwd(As[g], Bs[g]))), g


def test_grouped_token_rows_do_not_depend_on_the_expert_load():
    # the same token rows routed to an expert with 5 or with 600 other tokens
    K, N = 2048, 512
    tokens = W.randn_bf16((600, K), 1.0, 9701).cuda()
    Wx = [W.randn_bf16((K, N), 0.02, 9702 + g).cuda() for g in range(3)]
    small = dg.det_gemm_fwd_grouped([tokens[:5], tokens[:1], tokens[:300]], Wx)
    big = dg.det_gemm_fwd_grouped([tokens, tokens, tokens], Wx)
    assert torch.equal(bits(small[0]), bits(big[0][:5]))
    assert torch.equal(bits(small[1]), bits(big[1][:1]))
    assert torch.equal(bits(small[2]), bits(big[2][:300]))
    check()


@pytest.mark.parametrize("N", [512, 1000])             # whole and ragged column tiles
def test_grouped_row_reduction_is_the_oracle_fixed_order(N):
    K = 512
    Ms = [300, 0, 129, 1]
    As = [W.randn_bf16((m, K), 1.0, 9800 + g).cuda() for g, m in enumerate(Ms)]
    Bs = [W.randn_bf16((K, N), 0.05, 9810 + g).cuda() for g in range(4)]
    # D with a 16-byte-aligned row pitch even when N is not a multiple of 8
    ld = (N + 7) // 8 * 8
    Ds = [torch.empty((m, ld), dtype=torch.bfloat16, device="cuda")[:, :N] for m in Ms]
    for g, d in enumerate(Ds):
        d.copy_(W.randn_bf16((Ms[g], N), 1.0, 9820 + g).cuda())
    Ds[3] = None                                          # no reduction for this group
    Cs, rd = dg.det_gemm_fwd_grouped(As, Bs, D=Ds)
    check()
    assert rd[3] is None
    for g in (0, 2):
        want = oracle.rowdot(W.bits(Cs[g].cpu()), W.bits(Ds[g].cpu()))
        assert np.array_equal(rd[g].cpu().numpy().view(np.uint32), want.view(np.uint32)), g
    assert rd[1].numel() == 0
    # and run to run
    Cs2, rd2 = dg.det_gemm_fwd_grouped(As, Bs, D=Ds)
    for g in (0, 2):
        assert torch.equal(rd[g], rd2[g])


def test_grouped_row_reduction_order_on_hand_built_rows():
    """The row reduction's order, pinned on the GPU with hand-derived bits.
    B is the identity, so C = A exactly (a one-product leaf is its own
    rounding), and D = A makes every product C*D a chosen power of two
    (u = 2^-23). Row 0: 1 then 127 products 2^-24 in one 128-column tile:
    ascending keeps 1 (each add is a tie to even). Row 1: the same with the 1
    in the tile's last column: 127 x 2^-24 = 63.5u first, then 1 + 63.5u
    ties to 1 + 64u. Row 2: products 1, 2^-24, 2^-24 at the starts of three
    tiles: the mid-split tree gives 1 + (2^-24 + 2^-24) = 1 + u, where a
    running sum would give 1."""
    N = 384
    A = torch.zeros(3, N, dtype=torch.float32)
    A[0, 0] = 1.0
    A[0, 1:128] = 2.0 ** -12
    A[1, 127] = 1.0
    A[1, 0:127] = 2.0 ** -12
    A[2, 0] = 1.0
    A[2, 128] = 2.0 ** -12
    A[2, 256] = 2.0 ** -12
    Ab = A.to(torch.bfloat16).cuda()
    eye = torch.eye(N, dtype=torch.bfloat16).cuda()
    Cs, rd = dg.det_gemm_fwd_grouped([Ab], [eye], D=[Ab])
    check()
    assert torch.equal(bits(Cs[0]), bits(Ab))
    got = rd[0].cpu().numpy().view(np.uint32)
    assert list(got) == [0x3F800000, 0x3F800040, 0x3F800001], [hex(x) for x in got]
    want = oracle.rowdot(W.bits(Ab.cpu()), W.bits(Ab.cpu()))
    assert np.array_equal(got, want.view(np.uint32))
