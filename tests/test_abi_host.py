"""Host-side checks of the C-ABI library: it loads, exports what the header
declares, rejects bad arguments before touching a GPU, and its per-leaf merge
schedule replays the mid-split tree exactly. No GPU needed."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "det_gemm.h")


@pytest.fixture(scope="module")
def dg():
    from invariant_deterministic_gemm_gb300 import _build
    _build.build()
    import invariant_deterministic_gemm_gb300 as m
    m.lib()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(det_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_page_surface():
    names = declared_functions()
    for n in ("det_gemm_fwd", "det_gemm_fwd_rhs_transposed", "det_gemm_fwd_fp32", "det_gemm_da",
              "det_gemm_db", "det_gemm_db_transposed", "det_gemm_check", "det_gemm_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(dg):
    L = dg.lib()
    for n in declared_functions():
        assert hasattr(L, n), n


def test_status_strings_and_version(dg):
    L = dg.lib()
    assert L.det_gemm_abi_version() == 1
    for code in range(8):
        s = dg.status_string(code)
        assert s.startswith(dg.STATUS_NAMES[code])
    assert "unknown" in dg.status_string(99)


P = 0x10000   # a 16-byte aligned fake device address; never dereferenced here


def call(dg, name, x, y, o, M, N, K, ldx, ldy, ldo):
    return getattr(dg.lib(), name)(x, y, o, M, N, K, ldx, ldy, ldo, None)


@pytest.mark.parametrize("name", ["det_gemm_fwd", "det_gemm_fwd_rhs_transposed", "det_gemm_fwd_fp32",
                                  "det_gemm_fwd_fp32_rhs_transposed"])
def test_forward_argument_errors_are_returned_before_any_launch(dg, name):
    ok_ld = 4096
    assert call(dg, name, P, P * 8, P * 64, 4, 8, 32769, 32776, 32776, ok_ld) == 2   # K too large
    assert call(dg, name, P, P * 8, P * 64, -1, 8, 8, 8, 8, 8) == 1                  # negative size
    assert call(dg, name, 0, P * 8, P * 64, 4, 8, 8, 8, 8, 8) == 1                   # null input
    assert call(dg, name, P, P * 8, 0, 4, 8, 8, 8, 8, 8) == 1                        # null output
    assert call(dg, name, P + 2, P * 8, P * 64, 4, 8, 8, 8, 8, 8) == 3               # misaligned base
    assert call(dg, name, P, P * 8, P * 64, 4, 8, 12, 12, 16, 16) == 3               # lda*2 not /16
    assert call(dg, name, P, P * 8, P * 64, 4, 8, 16, 8, 16, 16) == 1                # lda < K
    assert call(dg, name, P, P, P, 4, 8, 8, 8, 8, 8) == 1                            # output overlaps
    # empty outputs are fine and enqueue nothing
    assert call(dg, name, 0, 0, 0, 0, 8, 8, 8, 8, 8) == 0
    assert call(dg, name, 0, 0, 0, 4, 0, 8, 8, 8, 8) == 0


def test_backward_argument_errors(dg):
    # dA: contraction over N
    assert call(dg, "det_gemm_da", P, P * 8, P * 64, 4, 32769, 8, 32776, 32776, 8) == 2
    # dB: contraction over M
    assert call(dg, "det_gemm_db", P, P * 8, P * 64, 32769, 8, 8, 8, 8, 8) == 2
    assert call(dg, "det_gemm_db_transposed", P, P * 8, P * 64, 32769, 8, 8, 8, 8, 8) == 2
    # M = 40000 is fine for the forward (rows) but not for dB (contraction)
    assert call(dg, "det_gemm_db", P, P * 8, 0, 40000, 8, 8, 8, 8, 8) == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_valid_arguments_without_a_gpu_report_unsupported_device(dg):
    assert call(dg, "det_gemm_fwd", P, P * 8, P * 64, 4, 8, 8, 8, 8, 8) == 4


# ---------------------------------------------------------- tree schedule

def mid_split_tree(lo, hi):
    """The tree as nested tuples, written from the definition."""
    if hi - lo == 1:
        return lo
    mid = (lo + hi) // 2
    return (mid_split_tree(lo, mid), mid_split_tree(mid, hi))


def replay(sched):
    """Run the per-leaf schedule on symbolic leaves, the way the kernel does:
    merge the running value with the pending slots named in the mask (lowest
    first; the pending value is the left operand), then park it in a slot or
    emit it as the root. Checks that every slot is written before it is read
    and never overwritten while pending."""
    slots = {}
    root = None
    for leaf, e in enumerate(sched):
        mask, store = e & 0x3FF, e >> 12
        assert (e >> 10) & 3 == 0
        v = leaf
        for s in range(10):
            if mask >> s & 1:
                assert s in slots, ("read of an empty slot", leaf, s)
                v = (slots.pop(s), v)
        if store == 15:
            assert root is None
            root = v
        else:
            assert store < 10 and store not in slots, ("overwrite", leaf, store)
            assert all(store > s for s in range(10) if mask >> s & 1)
            slots[store] = v
    assert not slots, "partials left over"
    return root


def test_schedule_replays_the_mid_split_tree_for_every_leaf_count(dg):
    for L in range(1, 1025):
        sched = dg.det_gemm_tree_schedule(L)
        assert len(sched) == L
        assert replay(sched) == mid_split_tree(0, L), L


def test_schedule_slot_depth_fits_ten_slots(dg):
    for L in (512, 513, 1000, 1024):
        sched = dg.det_gemm_tree_schedule(L)
        used = set()
        for e in sched:
            m, s = e & 0x3FF, e >> 12
            used |= {b for b in range(10) if m >> b & 1}
            if s != 15:
                used.add(s)
        assert max(used) == (L - 1).bit_length() - 1


def test_schedule_rejects_bad_counts(dg):
    L = dg.lib()
    buf = (ctypes.c_uint16 * 2)()
    assert L.det_gemm_tree_schedule(0, buf) == 1
    assert L.det_gemm_tree_schedule(1025, buf) == 1
    assert L.det_gemm_tree_schedule(4, None) == 1


def block_shape(leaves):
    """The mid-split tree of a block's leaves (nested tuples)."""
    n = len(leaves)
    if n == 1:
        return leaves[0]
    mid = n // 2
    return (block_shape(leaves[:mid]), block_shape(leaves[mid:]))


def replay_blocks(blocks, L):
    """Run the block schedule on symbolic leaves the way the kernel does."""
    slots = {}
    root = None
    nxt = 0
    for e in blocks:
        n = ((e >> 10) & 3) + 1
        mask, store = e & 0x3FF, e >> 12
        v = block_shape(list(range(nxt, nxt + n)))
        nxt += n
        assert mask & 3 == 0, "blocks never merge with slots 0-1"
        for s in range(10):
            if mask >> s & 1:
                assert s in slots, ("read of an empty slot", s)
                v = (slots.pop(s), v)
        if store == 15:
            assert root is None
            root = v
        else:
            assert 2 <= store < 10 and store not in slots
            slots[store] = v
    assert nxt == L and not slots
    return root


def test_block_schedule_replays_the_mid_split_tree_for_every_leaf_count(dg):
    for L in range(1, 1025):
        blocks = dg.det_gemm_block_schedule(L)
        sizes = [((e >> 10) & 3) + 1 for e in blocks]
        if L > 4:
            assert set(sizes) <= {2, 3, 4}, L
        assert replay_blocks(blocks, L) == mid_split_tree(0, L), L
        # the BF16 kernels store the root after the walk: the last block,
        # and only it, must form the root (store value 15)
        stores = [e >> 12 for e in blocks]
        assert stores[-1] == 15 and stores.count(15) == 1, L


def four_leaf_shape(x):
    """A block half as the kernel merges it: x0, x0 + x1, x0 + (x1 + x2) or
    (x0 + x1) + (x2 + x3)."""
    if len(x) == 1:
        return x[0]
    if len(x) == 2:
        return (x[0], x[1])
    if len(x) == 3:
        return (x[0], (x[1], x[2]))
    assert len(x) == 4
    return ((x[0], x[1]), (x[2], x[3]))


def replay_blocks8(blocks, L):
    """Run the eight-leaf block schedule on symbolic leaves the way the
    transposed tile does: a block of n leaves is a left half of n // 2
    leaves and a right half of the rest."""
    slots = {}
    root = None
    nxt = 0
    for e in blocks:
        n = (e & 7) + 1
        mask, store = e & 0x3F8, e >> 12
        x = list(range(nxt, nxt + n))
        nxt += n
        nl = n // 2
        v = x[0] if n == 1 else (four_leaf_shape(x[:nl]), four_leaf_shape(x[nl:]))
        for s in range(10):
            if mask >> s & 1:
                assert s in slots, ("read of an empty slot", s)
                v = (slots.pop(s), v)
        if store == 15:
            assert root is None
            root = v
        else:
            assert 3 <= store < 10 and store not in slots
            slots[store] = v
    assert nxt == L and not slots
    return root


def test_eight_leaf_block_schedule_replays_the_mid_split_tree_for_every_leaf_count(dg):
    for L in range(1, 1025):
        blocks = dg.det_gemm_block_schedule8(L)
        sizes = [(e & 7) + 1 for e in blocks]
        if L > 8:
            assert set(sizes) <= {4, 5, 6, 7, 8}, L
        assert replay_blocks8(blocks, L) == mid_split_tree(0, L), L
        # the transposed tile stores the root after the walk too
        stores = [e >> 12 for e in blocks]
        assert stores[-1] == 15 and stores.count(15) == 1, L
        # bits 10..11 are unused in this format
        assert all(e & 0xC00 == 0 for e in blocks), L


def test_block_schedules_reject_bad_counts(dg):
    L = dg.lib()
    buf = (ctypes.c_uint16 * 2)()
    nb = ctypes.c_int64(0)
    for fn in (L.det_gemm_block_schedule, L.det_gemm_block_schedule8):
        assert fn(0, buf, ctypes.byref(nb)) == 1
        assert fn(1025, buf, ctypes.byref(nb)) == 1
        assert fn(4, None, ctypes.byref(nb)) == 1
        assert fn(4, buf, None) == 1


# ---------------------------------------------------------------- merge API

def merge_call(dg, name, parts, n, out, M, N, ldp, ldc):
    L = dg.lib()
    arr = (ctypes.c_void_p * max(1, len(parts)))(*parts) if parts else None
    return getattr(L, name)(arr, n, out, M, N, ldp, ldc, None)


@pytest.mark.parametrize("name", ["det_gemm_merge", "det_gemm_merge_fp32"])
def test_merge_argument_errors_are_returned_before_any_launch(dg, name):
    parts = [P * (i + 2) for i in range(4)]
    out = P * 64
    assert merge_call(dg, name, parts[:3], 3, out, 4, 8, 8, 8) == 1          # n must be 2, 4 or 8
    assert merge_call(dg, name, parts, 4, out, -1, 8, 8, 8) == 1             # negative size
    assert merge_call(dg, name, [], 2, out, 4, 8, 8, 8) == 1                 # no part array
    assert merge_call(dg, name, [0, parts[1]], 2, out, 4, 8, 8, 8) == 1      # null part
    assert merge_call(dg, name, parts[:2], 2, 0, 4, 8, 8, 8) == 1            # null output
    assert merge_call(dg, name, parts[:2], 2, out, 4, 8, 4, 8) == 1          # ldp < N
    assert merge_call(dg, name, [parts[0] + 4, parts[1]], 2, out, 4, 8, 8, 8) == 3   # misaligned part
    assert merge_call(dg, name, parts[:2], 2, out, 4, 8, 10, 8) == 3         # row pitch not a multiple of 16 B
    assert merge_call(dg, name, [out, parts[1]], 2, out, 4, 8, 8, 8) == 1    # output overlaps a part
    assert merge_call(dg, name, parts[:2], 2, out, 0, 8, 8, 8) == 0          # empty: nothing to do


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_merge_without_a_gpu_reports_unsupported_device(dg):
    assert merge_call(dg, "det_gemm_merge", [P * 2, P * 3], 2, P * 64, 4, 8, 8, 8) == 4


# ---------------------------------------------------------------- RMSNorm

def rms_call(dg, x, w, y, M, D, eps, ldx, ldy):
    return dg.lib().det_rmsnorm(x, w, y, M, D, eps, ldx, ldy, None)


def test_rmsnorm_argument_errors_are_returned_before_any_launch(dg):
    x, w, y = P, P * 8, P * 64
    assert rms_call(dg, x, w, y, 4, 32769, 1e-6, 32776, 32776) == 2      # D too large
    assert rms_call(dg, x, w, y, -1, 8, 1e-6, 8, 8) == 1                 # negative size
    assert rms_call(dg, x, w, y, 4, 8, -1.0, 8, 8) == 1                  # negative eps
    assert rms_call(dg, x, w, y, 4, 8, float("nan"), 8, 8) == 1          # NaN eps
    assert rms_call(dg, 0, w, y, 4, 8, 1e-6, 8, 8) == 1                  # null x
    assert rms_call(dg, x, 0, y, 4, 8, 1e-6, 8, 8) == 1                  # null w
    assert rms_call(dg, x, w + 2, y, 4, 8, 1e-6, 8, 8) == 3              # misaligned w
    assert rms_call(dg, x, w, y, 4, 12, 1e-6, 12, 12) == 3               # pitch not 16 bytes
    assert rms_call(dg, x, w, x + 16, 4, 8, 1e-6, 8, 8) == 1             # partial overlap with x
    assert rms_call(dg, x, w, w, 4, 8, 1e-6, 8, 8) == 1                  # y overlaps w
    assert rms_call(dg, x, w, y, 0, 8, 1e-6, 8, 8) == 0                  # empty


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_rmsnorm_in_place_passes_the_checks_and_needs_a_gpu(dg):
    assert rms_call(dg, P, P * 8, P, 4, 8, 1e-6, 8, 8) == 4


# ---------------------------------------------------------- grouped GEMM

def grouped_call(dg, G, A, B, C, M, N, K, lda, ldb, ldc, D=None, ldd=None, rd=None):
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs) if xs is not None else None
    i64s = lambda xs: (ctypes.c_int64 * len(xs))(*xs) if xs is not None else None
    return dg.lib().det_gemm_fwd_grouped(G, arr(A), arr(B), arr(C), i64s(M), N, K, i64s(lda), i64s(ldb),
                                         i64s(ldc), arr(D), i64s(ldd), arr(rd), None)


def test_grouped_argument_errors_are_returned_before_any_launch(dg):
    A, B, C = [P, P * 2], [P * 4, P * 8], [P * 16, P * 32]
    ok = dict(M=[4, 4], N=8, K=8, lda=[8, 8], ldb=[8, 8], ldc=[8, 8])
    assert grouped_call(dg, 0, None, None, None, None, 8, 8, None, None, None) == 0     # no groups
    assert grouped_call(dg, -1, A, B, C, ok["M"], 8, 8, ok["lda"], ok["ldb"], ok["ldc"]) == 1
    assert grouped_call(dg, 2, None, B, C, ok["M"], 8, 8, ok["lda"], ok["ldb"], ok["ldc"]) == 1
    assert grouped_call(dg, 2, A, B, C, [4, -1], 8, 8, ok["lda"], ok["ldb"], ok["ldc"]) == 1
    assert grouped_call(dg, 2, A, B, C, ok["M"], 8, 32769, [32776] * 2, [8, 8], [8, 8]) == 2
    assert grouped_call(dg, 2, [P + 2, P * 2], B, C, ok["M"], 8, 8, ok["lda"], ok["ldb"], ok["ldc"]) == 3
    assert grouped_call(dg, 2, A, B, [P * 16, P * 16], ok["M"], 8, 8, ok["lda"], ok["ldb"], ok["ldc"]) == 1
    # a row reduction without its operand
    assert grouped_call(dg, 2, A, B, C, ok["M"], 8, 8, ok["lda"], ok["ldb"], ok["ldc"],
                        D=[0, 0], ldd=[8, 8], rd=[P * 64, 0]) == 1
    assert grouped_call(dg, 2, A, B, C, ok["M"], 8, 8, ok["lda"], ok["ldb"], ok["ldc"], rd=[P * 64, 0]) == 1
