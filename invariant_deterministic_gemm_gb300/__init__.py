"""Python binding of the det_gemm C-ABI (libdet_gemm.so), for GB300 / sm_103a.

Argument marshalling only: every entry point takes PyTorch CUDA BF16
tensors, checks their layout, allocates the output with PyTorch when none is
given, and calls the C function of the same name on the current CUDA stream.
All arithmetic happens in the library's kernels. There is no fallback: if the
library is missing or the device is not sm_103, the call raises.

Operations (RL-Kernel, "Batch-Invariant Deterministic GEMM (det_gemm)",
sections "Guarantees", "Ascend NPU backend", "Dtypes"):
  det_gemm_fwd(A[M,K], B[K,N])                 -> C[M,N] bf16
  det_gemm_fwd_rhs_transposed(A[M,K], W[N,K])  -> C[M,N] bf16
  det_gemm_fwd_fp32(A[M,K], B[K,N])            -> C[M,N] fp32
  det_gemm_fwd_fp32_rhs_transposed(A, W[N,K])  -> C[M,N] fp32
  det_gemm_da(dC[M,N], B[K,N])                 -> dA[M,K] = dC B^T
  det_gemm_db(A[M,K], dC[M,N])                 -> dB[K,N] = A^T dC
  det_gemm_db_transposed(A[M,K], dC[M,N])      -> dB^T[N,K]
Matrices are row-major with a leading dimension (``t.stride(0)``) and unit
column stride; row-slices of bigger tensors are accepted as they are.
"""
from __future__ import annotations

import array
import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdet_gemm.so")

OK = 0
STATUS_NAMES = {
    0: "DET_GEMM_OK",
    1: "DET_GEMM_ERR_INVALID_ARG",
    2: "DET_GEMM_ERR_K_TOO_LARGE",
    3: "DET_GEMM_ERR_ALIGNMENT",
    4: "DET_GEMM_ERR_UNSUPPORTED_DEVICE",
    5: "DET_GEMM_ERR_LAUNCH",
    6: "DET_GEMM_ERR_TIMEOUT",
    7: "DET_GEMM_ERR_CUDA",
}
KC_MAX = 32768

_lib = None
_lock = threading.Lock()

_GEMM_NAMES = (
    "det_gemm_fwd", "det_gemm_fwd_rhs_transposed", "det_gemm_fwd_fp32",
    "det_gemm_fwd_fp32_rhs_transposed", "det_gemm_da", "det_gemm_db",
    "det_gemm_db_transposed", "det_gemm_fwd_noalloc",
)


class DetGemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        msg = "%s: %s" % (where, status_string(status))
        if self.status == 5:
            detail = lib().det_gemm_last_error_detail().decode()
            if detail:
                msg += " [" + detail + "]"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError("libdet_gemm.so is not built (%s); run __graft_entry__.build() "
                              "or python -m invariant_deterministic_gemm_gb300._build" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        p, i64 = ctypes.c_void_p, ctypes.c_int64
        for name in _GEMM_NAMES:
            fn = getattr(L, name)
            fn.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, p]
            fn.restype = ctypes.c_int
        for name in ("det_gemm_merge", "det_gemm_merge_fp32"):
            fn = getattr(L, name)
            fn.argtypes = [p, ctypes.c_int, p, i64, i64, i64, i64, p]
            fn.restype = ctypes.c_int
        L.det_gemm_fwd_grouped.argtypes = [ctypes.c_int, p, p, p, p, i64, i64, p, p, p, p, p, p, p]
        L.det_gemm_fwd_grouped.restype = ctypes.c_int
        L.det_rmsnorm.argtypes = [p, p, p, i64, i64, ctypes.c_float, i64, i64, p]
        L.det_rmsnorm.restype = ctypes.c_int
        L.det_gemm_check.argtypes = [p]
        L.det_gemm_check.restype = ctypes.c_int
        L.det_gemm_status_string.argtypes = [ctypes.c_int]
        L.det_gemm_status_string.restype = ctypes.c_char_p
        L.det_gemm_last_error_detail.argtypes = []
        L.det_gemm_last_error_detail.restype = ctypes.c_char_p
        L.det_gemm_abi_version.argtypes = []
        L.det_gemm_abi_version.restype = ctypes.c_int
        L.det_gemm_tree_schedule.argtypes = [i64, p]
        L.det_gemm_tree_schedule.restype = ctypes.c_int
        L.det_gemm_block_schedule.argtypes = [i64, p, p]
        L.det_gemm_block_schedule.restype = ctypes.c_int
        L.det_gemm_block_schedule8.argtypes = [i64, p, p]
        L.det_gemm_block_schedule8.restype = ctypes.c_int
        L.det_gemm_shutdown.argtypes = []
        L.det_gemm_shutdown.restype = ctypes.c_int
        L.det_gemm_debug_force_timeout.argtypes = [ctypes.c_int]
        L.det_gemm_debug_force_timeout.restype = ctypes.c_int
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().det_gemm_status_string(int(status)).decode()


# The current stream's raw handle without building a torch.cuda.Stream object
# (a measurable part of a decode-sized call); the public route otherwise.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream) -> int:
    if stream is not None:
        return int(stream.cuda_stream)
    if _raw_stream is not None:
        return int(_raw_stream(torch.cuda.current_device()))
    return int(torch.cuda.current_stream().cuda_stream)


_ELEM_SIZE = {torch.bfloat16: 2, torch.float32: 4}


def _name(name: str, index: int) -> str:
    return name if index < 0 else "%s[%d]" % (name, index)


def _mat(t: torch.Tensor, name: str, dtype=torch.bfloat16, index: int = -1):
    """(data pointer, leading dimension) of a 2-D row-major CUDA tensor
    (name, or name[index] for an element of a list, in error messages).
    Each tensor property is read once and the name is formatted only for an
    error: this marshalling is a small launch's whole host cost."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % _name(name, index))
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (_name(name, index), dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % _name(name, index))
    shape = t.shape
    if len(shape) != 2:
        raise ValueError("%s must be 2-D, got shape %s" % (_name(name, index), tuple(shape)))
    rows, cols = shape
    s0, s1 = t.stride()
    if cols > 1 and s1 != 1:
        raise ValueError("%s must be row-major with unit column stride" % _name(name, index))
    if rows > 1:
        ld = s0
    else:
        # One row: the leading dimension is never used to address anything,
        # so any value that meets the library's 16-byte pitch rule will do.
        per16 = 16 // _ELEM_SIZE[dtype]
        ld = (max(cols, s0) + per16 - 1) // per16 * per16
    return t.data_ptr(), ld


def _out(out, rows, cols, dtype, like: torch.Tensor):
    if out is None:
        # Pad the row pitch to 16 bytes (the library's rule) and hand back
        # the [rows, cols] view.
        per16 = 16 // _ELEM_SIZE[dtype]
        ld = max(per16, (cols + per16 - 1) // per16 * per16)
        if ld == cols:
            return torch.empty((rows, cols), dtype=dtype, device=like.device)
        return torch.empty((rows, ld), dtype=dtype, device=like.device)[:, :cols]
    if tuple(out.shape) != (rows, cols):
        raise ValueError("out must have shape %s, got %s" % ((rows, cols), tuple(out.shape)))
    return out


_fns = {}


def _call(name: str, x_ptr, y_ptr, out_ptr, M, N, K, ldx, ldy, ldo, stream):
    fn = _fns.get(name)
    if fn is None:
        fn = _fns[name] = getattr(lib(), name)
    st = fn(x_ptr, y_ptr, out_ptr, M, N, K, ldx, ldy, ldo, _stream_handle(stream))
    if st != OK:
        raise DetGemmError(st, name)


def det_gemm_fwd(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    """C[M,N] = A[M,K] @ B[K,N] (BF16 out)."""
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    a, lda = _mat(A, "A")
    b, ldb = _mat(B, "B")
    C = _out(out, M, N, torch.bfloat16, A)
    c, ldc = _mat(C, "out")
    _call("det_gemm_fwd", a, b, c, M, N, K, lda, ldb, ldc, stream)
    return C


def det_gemm_fwd_noalloc(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor, stream=None):
    """det_gemm_fwd without any allocation, for callers that cannot allocate
    device memory (caller-managed arenas): the output must be
    given, and the library's scratch is a fixed array in its device image
    (see det_gemm.h for its limit and for why overlapping calls race)."""
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    if out is None:
        raise ValueError("det_gemm_fwd_noalloc needs a preallocated out")
    a, lda = _mat(A, "A")
    b, ldb = _mat(B, "B")
    if tuple(out.shape) != (M, N):
        raise ValueError("out must have shape %s, got %s" % ((M, N), tuple(out.shape)))
    c, ldc = _mat(out, "out")
    _call("det_gemm_fwd_noalloc", a, b, c, M, N, K, lda, ldb, ldc, stream)
    return out


def det_gemm_fwd_rhs_transposed(A: torch.Tensor, W: torch.Tensor, out=None, stream=None):
    """C[M,N] = A[M,K] @ W[N,K]^T (BF16 out)."""
    M, K = A.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    a, lda = _mat(A, "A")
    w, ldw = _mat(W, "W")
    C = _out(out, M, N, torch.bfloat16, A)
    c, ldc = _mat(C, "out")
    _call("det_gemm_fwd_rhs_transposed", a, w, c, M, N, K, lda, ldw, ldc, stream)
    return C


def det_gemm_fwd_fp32(A: torch.Tensor, B: torch.Tensor, out=None, stream=None):
    """C[M,N] = A[M,K] @ B[K,N] with FP32 leaves, FP32 tree, FP32 out."""
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    a, lda = _mat(A, "A")
    b, ldb = _mat(B, "B")
    C = _out(out, M, N, torch.float32, A)
    c, ldc = _mat(C, "out", torch.float32)
    _call("det_gemm_fwd_fp32", a, b, c, M, N, K, lda, ldb, ldc, stream)
    return C


def det_gemm_fwd_fp32_rhs_transposed(A: torch.Tensor, W: torch.Tensor, out=None, stream=None):
    """C[M,N] = A[M,K] @ W[N,K]^T with FP32 leaves, FP32 tree, FP32 out."""
    M, K = A.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    a, lda = _mat(A, "A")
    w, ldw = _mat(W, "W")
    C = _out(out, M, N, torch.float32, A)
    c, ldc = _mat(C, "out", torch.float32)
    _call("det_gemm_fwd_fp32_rhs_transposed", a, w, c, M, N, K, lda, ldw, ldc, stream)
    return C


def det_gemm_da(dC: torch.Tensor, B: torch.Tensor, out=None, stream=None):
    """dA[M,K] = dC[M,N] @ B[K,N]^T."""
    M, N = dC.shape
    K, N2 = B.shape
    if N2 != N:
        raise ValueError("dC and B disagree on N: %d vs %d" % (N, N2))
    g, ldg = _mat(dC, "dC")
    b, ldb = _mat(B, "B")
    dA = _out(out, M, K, torch.bfloat16, dC)
    d, ldd = _mat(dA, "out")
    _call("det_gemm_da", g, b, d, M, N, K, ldg, ldb, ldd, stream)
    return dA


def det_gemm_db(A: torch.Tensor, dC: torch.Tensor, out=None, stream=None):
    """dB[K,N] = A[M,K]^T @ dC[M,N]."""
    M, K = A.shape
    M2, N = dC.shape
    if M2 != M:
        raise ValueError("A and dC disagree on M: %d vs %d" % (M, M2))
    a, lda = _mat(A, "A")
    g, ldg = _mat(dC, "dC")
    dB = _out(out, K, N, torch.bfloat16, A)
    d, ldd = _mat(dB, "out")
    _call("det_gemm_db", a, g, d, M, N, K, lda, ldg, ldd, stream)
    return dB


def det_gemm_db_transposed(A: torch.Tensor, dC: torch.Tensor, out=None, stream=None):
    """dB^T[N,K] = dC[M,N]^T @ A[M,K] (the weight gradient in [N,K] layout)."""
    M, K = A.shape
    M2, N = dC.shape
    if M2 != M:
        raise ValueError("A and dC disagree on M: %d vs %d" % (M, M2))
    a, lda = _mat(A, "A")
    g, ldg = _mat(dC, "dC")
    dBt = _out(out, N, K, torch.bfloat16, A)
    d, ldd = _mat(dBt, "out")
    _call("det_gemm_db_transposed", a, g, d, M, N, K, lda, ldg, ldd, stream)
    return dBt


def _merge(name, parts, out, dtype, stream):
    if not isinstance(parts, (list, tuple)) or len(parts) not in (2, 4, 8):
        raise ValueError("parts must be a list of 2, 4 or 8 tensors")
    mats = [_mat(t, "parts", dtype, i) for i, t in enumerate(parts)]
    shape = tuple(parts[0].shape)
    if any(tuple(t.shape) != shape for t in parts):
        raise ValueError("parts must all have the same shape")
    lds = {ld for _, ld in mats}
    if len(lds) != 1:
        raise ValueError("parts must share one row pitch")
    M, N = shape
    C = _out(out, M, N, dtype, parts[0])
    c_ptr, ldc = _mat(C, "out", dtype)
    arr = (ctypes.c_void_p * len(parts))(*[ptr for ptr, _ in mats])
    st = getattr(lib(), name)(arr, len(parts), c_ptr, M, N, lds.pop(), ldc, _stream_handle(stream))
    if st != 0:
        raise DetGemmError(st, name)
    return C


def det_gemm_merge(parts, out=None, stream=None):
    """The full-contraction det_gemm product from n = 2, 4 or 8 partial
    products over equal contiguous leaf ranges (the merge tree's top levels)."""
    return _merge("det_gemm_merge", parts, out, torch.bfloat16, stream)


def det_gemm_merge_fp32(parts, out=None, stream=None):
    """det_gemm_merge for FP32 partial products (FP32 adds)."""
    return _merge("det_gemm_merge_fp32", parts, out, torch.float32, stream)


def det_gemm_fwd_grouped(As, Bs, outs=None, D=None, stream=None):
    """C_g = A_g @ B_g for every group g (mixture-of-experts expert GEMMs):
    As[g] [M_g, K], Bs[g] [K, N] BF16. With D (a list of [M_g, N] BF16
    tensors, None entries allowed) also returns rowdot[g][i] = sum_n C_g[i, n]
    * D_g[i, n] (FP32) in a fixed order. Returns the list of C (and the list
    of rowdot tensors, None where D[g] is None, when D is given)."""
    G = len(As)
    if len(Bs) != G or (outs is not None and len(outs) != G) or (D is not None and len(D) != G):
        raise ValueError("As, Bs, outs and D must have one entry per group")
    if G == 0:
        return ([], []) if D is not None else []
    K, N = Bs[0].shape
    bf16 = torch.bfloat16
    a_ptr, a_ld, b_ptr, b_ld, c_ptr, c_ld, Ms, Cs = [], [], [], [], [], [], [], []
    for g in range(G):
        a, b = As[g], Bs[g]
        p, ld = _mat(a, "As", bf16, g)
        a_ptr.append(p)
        a_ld.append(ld)
        p, ld = _mat(b, "Bs", bf16, g)
        b_ptr.append(p)
        b_ld.append(ld)
        m, k = a.shape
        if k != K or b.shape != (K, N):
            raise ValueError("group %d: A must be [M, %d] and B [%d, %d]" % (g, K, K, N))
        c = _out(None if outs is None else outs[g], m, N, bf16, a)
        p, ld = _mat(c, "outs", bf16, g)
        c_ptr.append(p)
        c_ld.append(ld)
        Ms.append(m)
        Cs.append(c)
    rowdots = None
    vals = a_ptr + b_ptr + c_ptr + Ms + a_ld + b_ld + c_ld
    if D is not None:
        rowdots = [None if D[g] is None else torch.empty(Ms[g], dtype=torch.float32, device=As[g].device)
                   for g in range(G)]
        d_ptr, d_ld = [], []
        for g in range(G):
            d = D[g]
            if d is None:
                p, ld = 0, N
            else:
                p, ld = _mat(d, "D", bf16, g)
                if d.shape != (Ms[g], N):
                    raise ValueError("D[%d] must be [M, N]" % g)
            d_ptr.append(p)
            d_ld.append(ld)
        vals += d_ptr + d_ld + [0 if r is None else r.data_ptr() for r in rowdots]
    # All per-group arrays in one host buffer (a ctypes array per list costs
    # several times more); the call reads it before it returns.
    buf = array.array("q", vals)
    base = buf.buffer_info()[0]
    at = [base + 8 * G * i for i in range(len(vals) // G)]
    d_arr, ld_arr, rd_arr = (at[7], at[8], at[9]) if D is not None else (None, None, None)
    st = lib().det_gemm_fwd_grouped(G, at[0], at[1], at[2], at[3], N, K, at[4], at[5], at[6], d_arr, ld_arr,
                                    rd_arr, _stream_handle(stream))
    if st != 0:
        raise DetGemmError(st, "det_gemm_fwd_grouped")
    return (Cs, rowdots) if D is not None else Cs


def det_rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, out=None, stream=None):
    """Batch-invariant RMSNorm of every row of x [M, D] with weight w [D]
    (BF16 in and out). out may be x itself (in place)."""
    x_ptr, ldx = _mat(x, "x")
    if not isinstance(w, torch.Tensor) or w.dtype != torch.bfloat16 or w.dim() != 1 or w.device.type != "cuda":
        raise TypeError("w must be a 1-D bfloat16 CUDA tensor")
    if w.shape[0] != x.shape[1] or (w.numel() > 1 and w.stride(0) != 1):
        raise ValueError("w must be contiguous with x.shape[1] elements")
    M, D = x.shape
    y = _out(out, M, D, torch.bfloat16, x)
    y_ptr, ldy = _mat(y, "out")
    st = lib().det_rmsnorm(x_ptr, w.data_ptr(), y_ptr, M, D, float(eps), ldx, ldy, _stream_handle(stream))
    if st != 0:
        raise DetGemmError(st, "det_rmsnorm")
    return y


def det_gemm_check(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(lib().det_gemm_check(_stream_handle(stream)))


def det_gemm_tree_schedule(num_leaves: int) -> list[int]:
    """Host-only: the per-leaf merge schedule the kernels apply (see det_gemm.h)."""
    buf = (ctypes.c_uint16 * max(1, num_leaves))()
    st = lib().det_gemm_tree_schedule(int(num_leaves), buf)
    if st != OK:
        raise DetGemmError(st, "det_gemm_tree_schedule")
    return list(buf)[:num_leaves]


def det_gemm_block_schedule(num_leaves: int) -> list[int]:
    """Host-only: the block schedule the plain-tile kernels walk (see det_gemm.h)."""
    buf = (ctypes.c_uint16 * max(1, num_leaves))()
    nb = ctypes.c_int64(0)
    st = lib().det_gemm_block_schedule(int(num_leaves), buf, ctypes.byref(nb))
    if st != OK:
        raise DetGemmError(st, "det_gemm_block_schedule")
    return list(buf)[:nb.value]


def det_gemm_block_schedule8(num_leaves: int) -> list[int]:
    """Host-only: the eight-leaf block schedule of the transposed tile (see det_gemm.h)."""
    buf = (ctypes.c_uint16 * max(1, num_leaves))()
    nb = ctypes.c_int64(0)
    st = lib().det_gemm_block_schedule8(int(num_leaves), buf, ctypes.byref(nb))
    if st != OK:
        raise DetGemmError(st, "det_gemm_block_schedule8")
    return list(buf)[:nb.value]


def det_gemm_shutdown() -> None:
    """Free the library's cached per-stream scratch (see det_gemm.h)."""
    lib().det_gemm_shutdown()


def det_gemm_debug_force_timeout(enable: bool) -> None:
    """Test hook: make every later launch time out on purpose (see det_gemm.h)."""
    lib().det_gemm_debug_force_timeout(1 if enable else 0)


__all__ = [
    "det_gemm_fwd", "det_gemm_fwd_noalloc", "det_gemm_fwd_rhs_transposed", "det_gemm_fwd_fp32",
    "det_gemm_fwd_fp32_rhs_transposed", "det_gemm_da", "det_gemm_db",
    "det_gemm_db_transposed", "det_gemm_check", "det_gemm_tree_schedule", "det_gemm_block_schedule", "det_gemm_block_schedule8",
    "det_gemm_debug_force_timeout", "det_gemm_shutdown", "DetGemmError", "lib", "status_string",
    "det_gemm_merge",
    "det_gemm_merge_fp32",
    "det_rmsnorm",
    "det_gemm_fwd_grouped",
]
