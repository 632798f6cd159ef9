"""Host-side marshalling of the Python binding, without a GPU.

The binding only turns tensors into the C-ABI's pointers, sizes and
leading dimensions. For the grouped forward it packs every per-group array
(A, B and C pointers, row counts, leading dimensions, and for the row
reduction the D pointers, their leading dimensions and the rowdot outputs)
into one host buffer and passes addresses into it. These tests replace the
library with a recorder that reads those arrays back during the call, and
the CUDA-only checks with stubs, so that the arrays the C side would see
are compared with the tensors they came from."""
import ctypes

import pytest
import torch

import invariant_deterministic_gemm_gb300 as dg


def _read(addr, n):
    return list((ctypes.c_int64 * n).from_address(addr)) if addr else None


class _Recorder:
    """Stands in for the shared library: records what det_gemm_fwd_grouped
    would read from its host arrays."""

    def __init__(self):
        self.calls = []

    def det_gemm_fwd_grouped(self, G, A, B, C, M, N, K, lda, ldb, ldc, D, ldd, rowdot, stream):
        self.calls.append(dict(G=G, A=_read(A, G), B=_read(B, G), C=_read(C, G), M=_read(M, G), N=N, K=K,
                               lda=_read(lda, G), ldb=_read(ldb, G), ldc=_read(ldc, G), D=_read(D, G),
                               ldd=_read(ldd, G), rowdot=_read(rowdot, G), stream=stream))
        return 0


@pytest.fixture
def recorder(monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(dg, "lib", lambda: rec)
    monkeypatch.setattr(dg, "_stream_handle", lambda stream: 1234)
    real_mat = dg._mat

    def mat_on_cpu(t, name, dtype=torch.bfloat16, index=-1):
        # the real checks, with only the device check lifted
        if isinstance(t, torch.Tensor) and not t.is_cuda:
            return real_mat(_AsCuda(t), name, dtype, index)
        return real_mat(t, name, dtype, index)

    monkeypatch.setattr(dg, "_mat", mat_on_cpu)
    return rec


class _AsCuda(torch.Tensor):
    """A CPU tensor that reports itself as a CUDA tensor (for _mat only)."""

    @staticmethod
    def __new__(cls, t):
        return t.as_subclass(cls)

    @property
    def is_cuda(self):
        return True


def _bf16(rows, cols):
    return torch.zeros(rows, cols, dtype=torch.bfloat16)


def test_grouped_arrays_match_the_tensors(recorder):
    N, K = 36, 24                     # 36 BF16 columns: outputs padded to a 40-element (80-byte) pitch
    Ms = [3, 0, 17]
    As = [_bf16(m, K) for m in Ms]
    Bs = [_bf16(K, N) for _ in Ms]
    Cs = dg.det_gemm_fwd_grouped(As, Bs)
    (c,) = recorder.calls
    assert c["G"] == 3 and c["N"] == N and c["K"] == K and c["stream"] == 1234
    assert c["A"] == [a.data_ptr() for a in As]
    assert c["B"] == [b.data_ptr() for b in Bs]
    assert c["C"] == [x.data_ptr() for x in Cs]
    assert c["M"] == Ms
    assert c["lda"] == [K, K, K] and c["ldb"] == [N, N, N]
    assert c["ldc"] == [40, 40, 40]
    assert [x.stride(0) for x in Cs if x.shape[0] > 1] == [40, 40]
    assert c["D"] is None and c["ldd"] is None and c["rowdot"] is None
    assert [tuple(x.shape) for x in Cs] == [(m, N) for m in Ms]


def test_grouped_row_reduction_arrays(recorder):
    N, K = 16, 32
    Ms = [5, 2]
    As = [_bf16(m, K) for m in Ms]
    Bs = [_bf16(K, N) for _ in Ms]
    outs = [_bf16(m, N) for m in Ms]
    D = [None, _bf16(2, N)]
    Cs, rowdots = dg.det_gemm_fwd_grouped(As, Bs, outs=outs, D=D)
    (c,) = recorder.calls
    assert Cs[0] is outs[0] and Cs[1] is outs[1]
    assert c["C"] == [o.data_ptr() for o in outs]
    assert c["D"] == [0, D[1].data_ptr()]
    assert c["ldd"] == [N, N]
    assert rowdots[0] is None and rowdots[1].shape == (2,) and rowdots[1].dtype == torch.float32
    assert c["rowdot"] == [0, rowdots[1].data_ptr()]


def test_grouped_argument_errors_name_the_group(recorder):
    K, N = 8, 8
    with pytest.raises(ValueError, match="group 1"):
        dg.det_gemm_fwd_grouped([_bf16(2, K), _bf16(2, K + 1)], [_bf16(K, N), _bf16(K, N)])
    with pytest.raises(TypeError, match=r"Bs\[1\] must be torch.bfloat16"):
        dg.det_gemm_fwd_grouped([_bf16(2, K), _bf16(2, K)], [_bf16(K, N), torch.zeros(K, N)])
    with pytest.raises(ValueError, match=r"D\[0\] must be \[M, N\]"):
        dg.det_gemm_fwd_grouped([_bf16(2, K)], [_bf16(K, N)], D=[_bf16(3, N)])
    with pytest.raises(ValueError, match="one entry per group"):
        dg.det_gemm_fwd_grouped([_bf16(2, K)], [_bf16(K, N), _bf16(K, N)])
    assert recorder.calls == []
    assert dg.det_gemm_fwd_grouped([], []) == []


def test_mat_reports_the_leading_dimension():
    # Real checks on CPU tensors stop at the device test, and before it at
    # the dtype test, with the element's name.
    with pytest.raises(ValueError, match=r"parts\[2\] must be a CUDA tensor"):
        dg._mat(_bf16(3, 4), "parts", torch.bfloat16, 2)
    with pytest.raises(TypeError, match="x must be torch.bfloat16"):
        dg._mat(torch.zeros(3, 4), "x")
    # With the device check lifted: the row pitch of a strided view, and a
    # one-row matrix's pitch rounded up to 16 bytes.
    big = _bf16(6, 20)
    assert dg._mat(_AsCuda(big[:, 2:9]), "v")[1] == 20
    assert dg._mat(_AsCuda(_bf16(1, 5)), "r")[1] == 8
    assert dg._mat(_AsCuda(torch.zeros(1, 5)), "r", torch.float32)[1] == 8
    with pytest.raises(ValueError, match="unit column stride"):
        dg._mat(_AsCuda(big.t()), "t")
