"""CPU oracle for det_gemm -- TEST INFRASTRUCTURE ONLY.

Plain C (``det_gemm_oracle.c``) behind ctypes. Only the tests, the smoke check
and the bench's CPU-baseline leg may import this package; the GPU library and
its Python binding never do, and the two share no code.

The arithmetic follows RL-Kernel, "Batch-Invariant Deterministic GEMM
(det_gemm)", sections "Guarantees" (C = A@B, dA = dC.B^T, dB = A^T.dC; BF16 in,
FP32 accumulation, fixed K order) and "Ascend NPU backend" (32-element FP32
leaves in ascending order, each rounded once to BF16 with round-to-nearest-
even, merged by a mid-split tree of BF16 adds; backward = the forward product
on transposed operands). See the C file's header for the exact definition and
for the one reading it makes (floor split of odd ranges).

Arrays are numpy ``uint16`` holding BF16 bit patterns (row-major, any
strides) and numpy ``float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "det_gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-pthread"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, no GPU needed)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cc = os.environ.get("CC", "cc")
    subprocess.check_call([cc, *CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_det_gemm.argtypes = [p, i64, i64, p, i64, i64, i64, i64, i64,
                                        ctypes.c_int, p, i64, i64, p, ctypes.c_int]
        lib.oracle_det_gemm.restype = ctypes.c_int
        lib.oracle_leaves_f32.argtypes = [p, i64, i64, p, i64, i64, i64, i64, i64, p]
        lib.oracle_leaves_f32.restype = ctypes.c_int
        lib.oracle_tree_bf16.argtypes = [p, i64]
        lib.oracle_tree_bf16.restype = ctypes.c_uint16
        lib.oracle_tree_f32.argtypes = [p, i64]
        lib.oracle_tree_f32.restype = ctypes.c_float
        lib.oracle_round_bf16.argtypes = [p, p, i64]
        lib.oracle_round_bf16.restype = None
        lib.oracle_add_bf16.argtypes = [p, p, p, i64]
        lib.oracle_rmsnorm.argtypes = [p, i64, p, i64, i64, ctypes.c_float, p, i64]
        lib.oracle_rmsnorm.restype = ctypes.c_int
        lib.oracle_rowdot.argtypes = [p, i64, p, i64, i64, i64, p]
        lib.oracle_rowdot.restype = ctypes.c_int
        lib.oracle_add_bf16.restype = None
        _lib = lib
        return lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _strides(a: np.ndarray):
    return tuple(s // a.itemsize for s in a.strides)


def gemm(X: np.ndarray, Y: np.ndarray, out_fp32: bool = False,
         threads: int | None = None, with_node_max: bool = False):
    """det_gemm of X[M, Kc] (bf16 bits) by Y[Kc, N] (bf16 bits), any strides.

    Returns C [M, N] (uint16 bf16 bits, or float32 when ``out_fp32``), and
    when ``with_node_max`` also the [M, N] float32 array of the largest
    |node| (leaves included) seen in each element's tree.
    """
    lib = _load()
    assert X.dtype == np.uint16 and Y.dtype == np.uint16
    assert X.ndim == 2 and Y.ndim == 2 and X.shape[1] == Y.shape[0]
    M, Kc = X.shape
    N = Y.shape[1]
    xs, ys = _strides(X), _strides(Y)
    C = np.zeros((M, N), dtype=np.float32 if out_fp32 else np.uint16)
    nm = np.zeros((M, N), dtype=np.float32) if with_node_max else None
    rc = lib.oracle_det_gemm(
        X.ctypes.data, xs[0], xs[1], Y.ctypes.data, ys[0], ys[1],
        M, N, Kc, int(bool(out_fp32)), C.ctypes.data, N, 1,
        nm.ctypes.data if nm is not None else None,
        threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_det_gemm rejected its arguments")
    return (C, nm) if with_node_max else C


# The entry points of the page's surface, each as the product it defines.

def fwd(A, B, **kw):
    """C[M,N] = A[M,K] @ B[K,N]."""
    return gemm(A, B, **kw)


def fwd_rhs_transposed(A, W, **kw):
    """C[M,N] = A[M,K] @ W[N,K]^T."""
    return gemm(A, W.T, **kw)


def fwd_fp32(A, B, **kw):
    """FP32-output forward: FP32 leaves, FP32 tree."""
    return gemm(A, B, out_fp32=True, **kw)


def fwd_fp32_rhs_transposed(A, W, **kw):
    return gemm(A, W.T, out_fp32=True, **kw)


def da(dC, B, **kw):
    """dA[M,K] = dC[M,N] @ B[K,N]^T (contraction over N)."""
    return gemm(dC, B.T, **kw)


def db(A, dC, **kw):
    """dB[K,N] = A[M,K]^T @ dC[M,N] (contraction over M)."""
    return gemm(A.T, dC, **kw)


def db_transposed(A, dC, **kw):
    """dB^T[N,K] = dC[M,N]^T @ A[M,K] (contraction over M)."""
    return gemm(dC.T, A, **kw)


def leaves_f32(X, Y, i: int, j: int) -> np.ndarray:
    """The unrounded FP32 leaves of element (i, j) of X @ Y."""
    lib = _load()
    Kc = X.shape[1]
    L = (Kc + 31) // 32
    out = np.zeros(L, dtype=np.float32)
    xs, ys = _strides(X), _strides(Y)
    rc = lib.oracle_leaves_f32(X.ctypes.data, xs[0], xs[1], Y.ctypes.data, ys[0], ys[1],
                               i, j, Kc, out.ctypes.data)
    if rc != 0:
        raise ValueError("bad arguments")
    return out


def tree_bf16(leaves: np.ndarray) -> int:
    """Root of the mid-split BF16 tree over the given BF16 leaves (bits)."""
    lv = np.ascontiguousarray(leaves, dtype=np.uint16)
    return int(_load().oracle_tree_bf16(lv.ctypes.data, lv.size))


def tree_f32(leaves: np.ndarray) -> float:
    lv = np.ascontiguousarray(leaves, dtype=np.float32)
    return float(_load().oracle_tree_f32(lv.ctypes.data, lv.size))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 bits, round to nearest even."""
    xx = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(xx.shape, dtype=np.uint16)
    _load().oracle_round_bf16(xx.ctypes.data, out.ctypes.data, xx.size)
    return out


def add_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Elementwise BF16 + BF16, rounded once to BF16 (bits in, bits out)."""
    aa = np.ascontiguousarray(a, dtype=np.uint16)
    bb = np.ascontiguousarray(b, dtype=np.uint16)
    assert aa.shape == bb.shape
    out = np.empty(aa.shape, dtype=np.uint16)
    _load().oracle_add_bf16(aa.ctypes.data, bb.ctypes.data, out.ctypes.data, aa.size)
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 values (a bit shift; no rounding)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Batch-invariant RMSNorm of every row of x (BF16 bits [M, D]) with
    weight w (BF16 bits [D]): the arithmetic is spelled out in
    det_gemm_oracle.c (oracle_rmsnorm)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    M, D = x.shape
    assert w.shape == (D,)
    y = np.empty((M, D), dtype=np.uint16)
    rc = lib.oracle_rmsnorm(x.ctypes.data, D, w.ctypes.data, M, D, float(eps), y.ctypes.data, D)
    if rc != 0:
        raise ValueError("oracle_rmsnorm: bad arguments")
    return y


def rowdot(C: np.ndarray, D: np.ndarray) -> np.ndarray:
    """rowdot[i] = sum_n C[i, n] * D[i, n] (BF16 bits in, FP32 out) in the
    grouped-GEMM epilogue's fixed order: one slot per 128-column N-tile (its
    FP32 sum in ascending column order), the slots merged by the mid-split
    tree (see oracle_rowdot in det_gemm_oracle.c)."""
    lib = _load()
    C = np.ascontiguousarray(C, dtype=np.uint16)
    D = np.ascontiguousarray(D, dtype=np.uint16)
    assert C.shape == D.shape
    M, N = C.shape
    out = np.empty(M, dtype=np.float32)
    if lib.oracle_rowdot(C.ctypes.data, N, D.ctypes.data, N, M, N, out.ctypes.data) != 0:
        raise ValueError("oracle_rowdot: bad arguments")
    return out
