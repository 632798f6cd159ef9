"""det_gemm_fwd_noalloc: the forward product for callers that cannot
allocate device memory (stream capture, caller-owned memory arenas, paths
that must not synchronise the device). It must give exactly what
det_gemm_fwd gives -- the same kernel and arithmetic, with its scratch in a
fixed array of the library instead of a cudaMalloc'd buffer -- call after
call, whatever an earlier call left in that array.

The shapes make the kernel use the array: a contraction of 32768 (1024
leaves) parks the tree's highest pending partials there, and a ragged
column count sends the output of the last column tile through it.

This file is named to be collected last, so that a run stopping at its first
failure has already run every other test."""
import ctypes

import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg
import workloads as W
from gpu_util import check, dev

pytestmark = pytest.mark.gpu


def _noalloc(A, B, out):
    """Calls the C-ABI entry point directly."""
    M, K = A.shape
    N = B.shape[1]
    st = dg.lib().det_gemm_fwd_noalloc(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                                       A.stride(0), B.stride(0), out.stride(0),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0, dg.status_string(st)


@pytest.mark.parametrize("shapes", [[(200, 300, 32768), (129, 136, 5000)]])
def test_noalloc_forward_matches_det_gemm_fwd_on_two_calls_in_a_row(shapes):
    for i, (M, N, K) in enumerate(shapes):
        A = dev(W.randn_bf16((M, K), 1.0, 9100 + i))
        B = dev(W.randn_bf16((K, N), 0.02, 9200 + i))
        out = dev(torch.zeros(M, N, dtype=torch.bfloat16))
        _noalloc(A, B, out)
        ref = dg.det_gemm_fwd(A, B)
        check()
        # identical kernel and arithmetic: equal bit for bit
        assert torch.equal(out.contiguous().view(torch.int16), ref.contiguous().view(torch.int16)), (M, N, K)
