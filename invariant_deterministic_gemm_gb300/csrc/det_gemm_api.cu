// det_gemm C-ABI: argument checks, the leaf-merge schedule, TMA descriptors
// and kernel launches. The operation each entry point computes is stated in
// include/det_gemm.h (RL-Kernel, "Batch-Invariant Deterministic GEMM
// (det_gemm)", sections "Guarantees", "Ascend NPU backend" and "Dtypes").
#include "det_gemm.h"
#include "det_gemm_internal.h"

#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>

namespace detg {

// Device status word: [0] = first error code seen since the last check.
// One instance per device context; host code reaches it through
// cudaGetSymbolAddress (the host-side symbol is not a device address).
__device__ int g_status[4];

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kForcedTimeoutNs = 50ull * 1000 * 1000;

struct DeviceState {
    bool init = false;
    det_gemm_status init_status = DET_GEMM_OK;
    int sm_count = 0;
    int *status_ptr = nullptr;
    bool prepared[kVariantCount] = {};
    det_gemm_status prepare_status[kVariantCount] = {};
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Deep-slot scratch, one buffer per (device, stream) so that launches on
// different streams never share one; allocated on first use, reused by
// every later launch on that stream, freed by det_gemm_shutdown().
struct ScratchEntry {
    int device;
    cudaStream_t stream;
    void *ptr;
    size_t bytes;
};
constexpr int kMaxScratch = 64;
ScratchEntry g_scratch[kMaxScratch];
int g_scratch_count = 0;
int g_scratch_next_evict = 0;
int g_force_timeout = 0;
thread_local char g_detail[256] = "";

// Records the CUDA error behind a DET_GEMM_ERR_LAUNCH / _CUDA status.
det_gemm_status fail_cuda(det_gemm_status st, cudaError_t e, const char *where)
{
    std::snprintf(g_detail, sizeof g_detail, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
    cudaGetLastError();
    return st;
}
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

VariantOps variant_ops(Variant v)
{
    switch (v) {
    case kBf16KMN: return ops_bf16_kmn();
    case kBf16KK: return ops_bf16_kk();
    case kBf16MNMN: return ops_bf16_mnmn();
    case kF32KMN: return ops_f32_kmn();
    case kF32KK: return ops_f32_kk();
    case kBf16KMNGrouped: return ops_bf16_kmn_grouped();
    case kBf16SwapMNK: return ops_bf16_swap_mnk();
    case kBf16SwapKK: return ops_bf16_swap_kk();
    default: return VariantOps{};
    }
}

unsigned long long timeout_ns()
{
    if (g_force_timeout) return kForcedTimeoutNs;
    const char *s = std::getenv("DET_GEMM_TIMEOUT_MS");
    long long ms = s ? std::atoll(s) : 1000;
    if (ms < 1) ms = 1;
    return static_cast<unsigned long long>(ms) * 1000ull * 1000ull;
}

// smallest h with 2^h >= n, for n >= 1
int ceil_log2(int64_t n)
{
    int h = 0;
    while ((int64_t{1} << h) < n) ++h;
    return h;
}

// The per-leaf schedule of the mid-split tree (format in det_gemm.h). The
// walk descends from the root [0, L) to leaf l, splitting [lo, hi) at
// mid = (lo + hi) / 2. A node over n leaves has height ceil(log2 n); the
// left child of a node of height h waits in slot h - 1. After leaf l is
// finished the running value climbs while it is a right child, merging the
// waiting left sibling at each such node, and is parked at the first node
// where it is a left child (or is the root).
void build_schedule(int64_t L, uint16_t *out)
{
    for (int64_t l = 0; l < L; ++l) {
        int64_t lo = 0, hi = L;
        int depth = 0;
        int slot_at[32];
        bool right_at[32];
        while (hi - lo > 1) {
            const int64_t mid = (lo + hi) >> 1;
            slot_at[depth] = ceil_log2(hi - lo) - 1;
            right_at[depth] = (l >= mid);
            ++depth;
            if (l >= mid) lo = mid;
            else hi = mid;
        }
        uint32_t mask = 0;
        uint32_t store = kSlotRoot;
        for (int d = depth - 1; d >= 0; --d) {
            if (right_at[d]) {
                mask |= 1u << slot_at[d];
            } else {
                store = static_cast<uint32_t>(slot_at[d]);
                break;
            }
        }
        out[l] = static_cast<uint16_t>(mask | (store << 12));
    }
}

// The block schedule (format in det_gemm.h): the tree cut into its maximal
// subtrees of at most four leaves, in leaf order. A block's leaves are
// merged among themselves in registers; its entry says which pending
// partials to merge its value with and where to park the result, which is
// the per-leaf entry of its last leaf without the merges inside the block.
void add_blocks(const uint16_t *leaf_sched, int64_t lo, int64_t hi, int max_leaves, uint16_t *out, int64_t *nb)
{
    const int64_t n = hi - lo;
    if (n > max_leaves) {
        const int64_t mid = (lo + hi) >> 1;
        add_blocks(leaf_sched, lo, mid, max_leaves, out, nb);
        add_blocks(leaf_sched, mid, hi, max_leaves, out, nb);
        return;
    }
    const uint32_t e = leaf_sched[hi - 1];
    const int h = ceil_log2(n);                  // the block's height
    const uint32_t up = (e & 0x3FFu) & ~((1u << h) - 1u);
    if (max_leaves == 4) {
        out[(*nb)++] = static_cast<uint16_t>(up | (static_cast<uint32_t>(n - 1) << 10) | (e & 0xF000u));
    } else {
        // Blocks of up to eight leaves: a block's parent has more than eight
        // leaves (height 4 or more), so its merges and its store use slots 3
        // and up, and bits 0..2 carry the leaf count.
        out[(*nb)++] = static_cast<uint16_t>(up | static_cast<uint32_t>(n - 1) | (e & 0xF000u));
    }
}

void build_blocks(int64_t L, int max_leaves, uint16_t *out, int64_t *nb)
{
    uint16_t leaf_sched[kMaxLeaves];
    build_schedule(L, leaf_sched);
    *nb = 0;
    add_blocks(leaf_sched, 0, L, max_leaves, out, nb);
}

struct BlockSchedule {
    uint16_t *entries;
    int64_t count;
};
BlockSchedule g_block_cache[2][kMaxLeaves + 1] = {};

const BlockSchedule *blocks_for(int64_t L, int max_leaves)
{
    std::lock_guard<std::mutex> lk(g_mu);
    BlockSchedule &b = g_block_cache[max_leaves == 8][L];
    if (!b.entries) {
        uint16_t *s = static_cast<uint16_t *>(std::malloc(sizeof(uint16_t) * L));
        if (!s) return nullptr;
        int64_t nb = 0;
        build_blocks(L, max_leaves, s, &nb);
        b = BlockSchedule{s, nb};
    }
    return &b;
}

// ---------------------------------------------------------- validation

struct Mat {
    const void *ptr;
    int64_t rows, cols, ld;
    int esize;
};

det_gemm_status check_mat(const Mat &m)
{
    if (m.rows <= 0 || m.cols <= 0) return DET_GEMM_OK;   // empty: never touched
    if (m.ptr == nullptr) return DET_GEMM_ERR_INVALID_ARG;
    if (m.ld < m.cols) return DET_GEMM_ERR_INVALID_ARG;
    if (m.ld > (int64_t{1} << 36)) return DET_GEMM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(m.ptr) % 16 != 0) return DET_GEMM_ERR_ALIGNMENT;
    if ((m.ld * m.esize) % 16 != 0) return DET_GEMM_ERR_ALIGNMENT;
    return DET_GEMM_OK;
}

bool overlaps(const Mat &a, const Mat &b)
{
    if (a.rows <= 0 || a.cols <= 0 || b.rows <= 0 || b.cols <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.ptr);
    const uintptr_t a1 = a0 + static_cast<uintptr_t>(((a.rows - 1) * a.ld + a.cols) * a.esize);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b.ptr);
    const uintptr_t b1 = b0 + static_cast<uintptr_t>(((b.rows - 1) * b.ld + b.cols) * b.esize);
    return a0 < b1 && b0 < a1;
}

// ------------------------------------------------------------- devices

det_gemm_status device_state(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return DET_GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return DET_GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.init) {
        st.init = true;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            st.init_status = DET_GEMM_ERR_UNSUPPORTED_DEVICE;
        } else if (major != 10 || minor != 3) {
            st.init_status = DET_GEMM_ERR_UNSUPPORTED_DEVICE;
        } else if (cudaGetSymbolAddress(reinterpret_cast<void **>(&st.status_ptr), g_status) != cudaSuccess) {
            cudaGetLastError();
            st.init_status = DET_GEMM_ERR_LAUNCH;
        } else {
            if (!g_encode) {
                cudaDriverEntryPointQueryResult q;
                void *fn = nullptr;
                if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                                     &q) != cudaSuccess ||
                    q != cudaDriverEntryPointSuccess || fn == nullptr) {
                    cudaGetLastError();
                    st.init_status = DET_GEMM_ERR_LAUNCH;
                } else {
                    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
                }
            }
        }
    }
    if (st.init_status != DET_GEMM_OK) return st.init_status;
    *out = &st;
    return DET_GEMM_OK;
}

det_gemm_status prepare_variant(DeviceState *st, Variant v)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!st->prepared[v]) {
        st->prepared[v] = true;
        int regs = 0;
        VariantOps ops = variant_ops(v);
        cudaError_t e = ops.prepare ? ops.prepare(&regs) : cudaErrorInvalidDeviceFunction;
        if (e != cudaSuccess) {
            st->prepare_status[v] = fail_cuda(DET_GEMM_ERR_LAUNCH, e, "kernel attributes");
        } else if (ops.split_regs != 0 && regs != ops.split_regs) {
            // setmaxnreg redistributes exactly the registers the CTA is
            // launched with; any other launch allocation would make the
            // epilogue's request unsatisfiable or waste registers.
            std::snprintf(g_detail, sizeof g_detail, "kernel compiled for %d registers per thread, expected %d",
                          regs, ops.split_regs);
            st->prepare_status[v] = DET_GEMM_ERR_LAUNCH;
        }
    }
    return st->prepare_status[v];
}

// Scratch of at least `bytes` for launches on `stream` of the current device.
void *scratch_for(int device, cudaStream_t stream, size_t bytes)
{
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_scratch_count; ++i) {
        ScratchEntry &e = g_scratch[i];
        if (e.device == device && e.stream == stream) {
            if (e.bytes >= bytes) return e.ptr;
            // Grow: cudaFree waits for the device, so no launch still uses it.
            cudaFree(e.ptr);
            e.ptr = nullptr;
            if (cudaMalloc(&e.ptr, bytes) != cudaSuccess) {
                cudaGetLastError();
                e.ptr = nullptr;
                e.bytes = 0;
                return nullptr;
            }
            e.bytes = bytes;
            return e.ptr;
        }
    }
    int slot;
    if (g_scratch_count < kMaxScratch) {
        slot = g_scratch_count++;
    } else {
        slot = g_scratch_next_evict;
        g_scratch_next_evict = (g_scratch_next_evict + 1) % kMaxScratch;
        cudaFree(g_scratch[slot].ptr);   // waits for the device first
    }
    void *ptr = nullptr;
    if (cudaMalloc(&ptr, bytes) != cudaSuccess) {
        cudaGetLastError();
        g_scratch[slot] = ScratchEntry{device, stream, nullptr, 0};
        return nullptr;
    }
    g_scratch[slot] = ScratchEntry{device, stream, ptr, bytes};
    return ptr;
}

bool encode(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint64_t ld_elems,
            uint32_t box_inner, uint32_t box_outer)
{
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld_elems * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tile order (timing only; every tile is computed the same way wherever it
// falls in the walk). The smaller operand is the one kept in L2: as many of
// its 128-row (A) or BN-column (B) panels per group as fit in 32 MiB, so the
// other operand is streamed from DRAM once per group. Measured on the MLP
// dA launch (8192 x 14336 x 4096): groups of 8, 32 and 63 one-MiB A panels
// read 999, 307 and 1512 MB from DRAM; a quarter of the L2 keeps the
// resident panels from being evicted by the streamed ones and the output.
void choose_tile_order(Problem &pb, int64_t rows, int64_t cols, int64_t kc, int bn, int n_tiles)
{
    constexpr double kResidentBytes = 32.0 * 1024 * 1024;
    const double a_bytes = 2.0 * rows * kc, b_bytes = 2.0 * cols * kc;
    pb.rows_fast = a_bytes <= b_bytes ? 1 : 0;
    const double panel = 2.0 * (pb.rows_fast ? kBM : bn) * kc;
    const int tiles = pb.rows_fast ? pb.m_tiles : n_tiles;
    const int fit = panel > 0 ? static_cast<int>(kResidentBytes / panel) : tiles;
    pb.group = std::max(1, std::min(tiles, fit));
    const int slow = pb.rows_fast ? n_tiles : pb.m_tiles;
    pb.span = pb.group * slow;
    pb.div_span = make_fast_div(static_cast<unsigned>(pb.span));
    pb.div_group = make_fast_div(static_cast<unsigned>(pb.group));
    const int rem = tiles % pb.group;
    pb.div_last = make_fast_div(static_cast<unsigned>(rem == 0 ? pb.group : rem));
}

// Contraction parts per tile. A launch with few output tiles (skinny M)
// leaves SMs idle while each tile walks all its leaves; splitting every
// tile's leaves into 2, 4 or 8 equal contiguous ranges that are subtrees of
// the merge tree gives that many work units per tile, and the tree's top
// levels are applied afterwards (launch_merge_parts). The bits are the same
// for every choice. The busiest CTA walks ceil(units / SMs) * leaves-per-unit
// leaves, plus, for a split, the merge launch and the partial results'
// round trip through memory, counted as 8 leaves (fitted on GB300: it keeps
// the QKV launch at M <= 64, 96 tiles, unsplit and splits M = 256 in two,
// the faster choice for each). The fewest parts that cut that cost by a
// quarter or more are taken (each range keeps at least 8 leaves).
int choose_parts(int64_t tiles, int64_t L, int sms)
{
    auto busiest = [&](int parts) {
        return (tiles * parts + sms - 1) / sms * (L / parts) + (parts > 1 ? int64_t{8} : int64_t{0});
    };
    int best = 1;
    for (int parts = 2; parts <= 8; parts *= 2) {
        if (L % parts != 0 || L / parts < 8) break;
        if (busiest(parts) * 5 <= busiest(best) * 4) best = parts;
    }
    return best;
}

// One GEMM of a launch: out[rows, cols] = sum over kc of Aop[row, k] *
// Bop[k, col]. Aop is `a` stored either K-major ([rows, kc] row-major) or
// MN-major ([kc, rows] row-major); Bop is `b` stored K-major ([cols, kc]) or
// MN-major ([kc, cols]). d / rowdot: the optional row reduction of a grouped
// launch (rowdot[i] = sum_n out[i, n] * d[i, n], fixed order).
struct ProblemArgs {
    Mat a, b, out;
    int64_t rows;
    const void *d;
    int64_t ldd;
    float *rowdot;
};

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The launch of one or several GEMMs sharing cols and kc (a plain launch:
// g == 1; a grouped one: every group's tiles in one persistent launch).
// fixed_scratch, when given, replaces the cached per-stream scratch: the
// launch then allocates nothing at all (see det_gemm_fwd_noalloc).
det_gemm_status run_problems(Variant v, bool a_kmajor, bool b_kmajor, const ProblemArgs *pa, int g, int64_t cols,
                             int64_t kc, cudaStream_t stream, void *fixed_scratch = nullptr, size_t fixed_bytes = 0)
{
    if (g < 1 || g > kMaxProblems || cols < 0 || kc < 0) return DET_GEMM_ERR_INVALID_ARG;
    if (cols > (int64_t{1} << 31) - 256) return DET_GEMM_ERR_INVALID_ARG;
    if (kc > kKcMax) return DET_GEMM_ERR_K_TOO_LARGE;
    det_gemm_status s;
    bool any = false;
    for (int i = 0; i < g; ++i) {
        const ProblemArgs &q = pa[i];
        if (q.rows < 0 || q.rows > (int64_t{1} << 31) - 256) return DET_GEMM_ERR_INVALID_ARG;
        if (q.rows == 0 || cols == 0) continue;
        any = true;
        if ((s = check_mat(q.out)) != DET_GEMM_OK) return s;
        if (kc > 0) {
            if ((s = check_mat(q.a)) != DET_GEMM_OK) return s;
            if ((s = check_mat(q.b)) != DET_GEMM_OK) return s;
            if (overlaps(q.out, q.a) || overlaps(q.out, q.b)) return DET_GEMM_ERR_INVALID_ARG;
        }
        if (q.rowdot) {
            const Mat dm{q.d, q.rows, cols, q.ldd, 2};
            if (q.d == nullptr) return DET_GEMM_ERR_INVALID_ARG;
            if ((s = check_mat(dm)) != DET_GEMM_OK) return s;
            if (reinterpret_cast<uintptr_t>(q.rowdot) % 16 != 0) return DET_GEMM_ERR_ALIGNMENT;
            const Mat rm{q.rowdot, 1, q.rows, q.rows, 4};
            if (overlaps(rm, q.out) || overlaps(rm, dm) || overlaps(q.out, dm)) return DET_GEMM_ERR_INVALID_ARG;
        }
        for (int j = 0; j < i; ++j)
            if (pa[j].rows > 0 && overlaps(q.out, pa[j].out)) return DET_GEMM_ERR_INVALID_ARG;
    }
    if (!any) return DET_GEMM_OK;
    DeviceState *st = nullptr;
    if ((s = device_state(&st)) != DET_GEMM_OK) return s;

    if (kc == 0) {
        // Empty contraction: every element is the empty sum, +0 (and so is
        // every row reduction).
        for (int i = 0; i < g; ++i) {
            const ProblemArgs &q = pa[i];
            if (q.rows == 0 || cols == 0) continue;
            cudaError_t e = cudaMemset2DAsync(const_cast<void *>(q.out.ptr), static_cast<size_t>(q.out.ld * q.out.esize),
                                              0, static_cast<size_t>(cols * q.out.esize), static_cast<size_t>(q.rows),
                                              stream);
            if (e == cudaSuccess && q.rowdot) e = cudaMemsetAsync(q.rowdot, 0, sizeof(float) * q.rows, stream);
            if (e != cudaSuccess) return (cudaGetLastError(), DET_GEMM_ERR_LAUNCH);
        }
        return DET_GEMM_OK;
    }
    if ((s = prepare_variant(st, v)) != DET_GEMM_OK) return s;
    VariantOps ops = variant_ops(v);

    const int64_t L = (kc + kLeaf - 1) / kLeaf;
    const int64_t n_tiles = (cols + ops.bn - 1) / ops.bn;
    int64_t tiles = 0;
    for (int i = 0; i < g; ++i) tiles += (pa[i].rows + kBM - 1) / kBM * n_tiles;
    if (tiles > (int64_t{1} << 31) - 1) return DET_GEMM_ERR_INVALID_ARG;
    // Only a plain launch splits (the allocation-free path never does: the
    // partial results need memory).
    const int parts = (fixed_scratch || g > 1) ? 1 : choose_parts(tiles, L, st->sm_count);
    const int64_t Lp = L / parts;
    const BlockSchedule *blocks = nullptr;
    if (!fixed_scratch) {
        blocks = blocks_for(Lp, ops.block_leaves);
        if (!blocks) return DET_GEMM_ERR_LAUNCH;
    }

    Params p;
    std::memset(&p, 0, sizeof(p));
    uint8_t *rd_slots = nullptr;   // the row reduction's slots (scratch)
    p.num_problems = g;
    p.n_tiles = static_cast<int>(n_tiles);
    int64_t units = 0;
    size_t rd_bytes = 0;
    for (int i = 0; i < g; ++i) {
        const ProblemArgs &q = pa[i];
        Problem &pb = p.prob[i];
        pb.first_unit = static_cast<int>(units);
        pb.rows = static_cast<int>(q.rows);
        pb.m_tiles = static_cast<int>((q.rows + kBM - 1) / kBM);
        if (q.rows == 0) continue;
        units += static_cast<int64_t>(pb.m_tiles) * n_tiles * parts;
        // A K-major A operand with fewer rows than a tile is copied with a box
        // of only its rows (rounded up to 8, at least 16): on GB300 a copy
        // whose box is mostly outside the tensor, here 128 rows for fewer than
        // 16, took the QKV launch from 35 to 57 us. The tile's other rows keep
        // whatever the shared-memory slot holds; MMA row i reads only row i
        // of A, and those rows are never stored.
        const int a_box_rows =
            (a_kmajor && q.rows < kBM) ? static_cast<int>(std::max<int64_t>(16, (q.rows + 7) / 8 * 8)) : kBM;
        // The same for a K-major B operand with fewer columns than a tile
        // (the transposed tile's few output rows).
        const int b_box_rows =
            (b_kmajor && cols < ops.bn) ? static_cast<int>(std::max<int64_t>(16, (cols + 7) / 8 * 8)) : ops.bn;
        bool ok;
        if (a_kmajor) ok = encode(&pb.tmap_a, q.a.ptr, kc, q.rows, q.a.ld, 64, static_cast<uint32_t>(a_box_rows));
        else ok = encode(&pb.tmap_a, q.a.ptr, q.rows, kc, q.a.ld, 64, 64);
        if (ok) {
            if (b_kmajor) ok = encode(&pb.tmap_b, q.b.ptr, kc, cols, q.b.ld, 64, static_cast<uint32_t>(b_box_rows));
            else ok = encode(&pb.tmap_b, q.b.ptr, cols, kc, q.b.ld, 64, 64);
        }
        if (!ok) return DET_GEMM_ERR_LAUNCH;
        // An MN-major B operand is copied in boxes of 64 columns, the tile's
        // BN columns rounded up (the copy counts whole boxes).
        const int b_copy_rows = b_kmajor ? b_box_rows : (ops.bn + 63) / 64 * 64;
        pb.stage_tx = a_box_rows * kBK * 2 + b_copy_rows * kBK * 2;
        pb.out = const_cast<void *>(q.out.ptr);
        pb.ldo = q.out.ld;
        choose_tile_order(pb, q.rows, cols, kc, ops.bn, p.n_tiles);
        if (q.rowdot) rd_bytes += align256(sizeof(float) * ((cols + kRowdotTile - 1) / kRowdotTile) * q.rows);
    }
    if (units > (int64_t{1} << 31) - 1) return DET_GEMM_ERR_INVALID_ARG;
    p.units = static_cast<int>(units);
    // A split launch's part slabs: laid out like the output (out_rows x
    // part_ld each, the row pitch a multiple of 8 elements, 16 bytes). The
    // transposed tile's kernel rows are the output's columns.
    const int64_t out_rows = ops.swap ? cols : pa[0].rows;
    const int64_t out_cols = ops.swap ? pa[0].rows : cols;
    const int64_t part_ld = (out_cols + 7) / 8 * 8;
    const size_t part_bytes =
        parts > 1 ? align256(static_cast<size_t>(parts) * out_rows * part_ld * pa[0].out.esize) : 0;
    if (fixed_scratch) {
        p.scratch = fixed_scratch;
    } else {
        int dev = 0;
        cudaGetDevice(&dev);
        // The deep-slot part is sized for the largest variant and a grid of
        // one CTA per SM, so every launch on this stream can reuse it; the
        // part slabs of a split launch and the row reduction's slots follow
        // it.
        const size_t slot_bytes = static_cast<size_t>(st->sm_count) * kMaxScratchCtaBytes;
        uint8_t *base = static_cast<uint8_t *>(scratch_for(dev, stream, slot_bytes + part_bytes + rd_bytes));
        if (!base) return DET_GEMM_ERR_LAUNCH;
        p.scratch = base;
        p.part_out = parts > 1 ? base + slot_bytes : nullptr;
        rd_slots = base + slot_bytes + part_bytes;
    }
    p.parts = parts;
    p.div_parts = make_fast_div(static_cast<unsigned>(parts));
    p.div_stages = make_fast_div(static_cast<unsigned>((Lp + 1) / 2));
    p.part_ld = part_ld;
    p.part_stride = out_rows * part_ld;
    p.status = st->status_ptr;
    p.timeout_ns = timeout_ns();
    p.cols = static_cast<int>(cols);
    p.kc = static_cast<int>(kc);
    p.num_leaves = static_cast<int>(Lp);
    p.force_timeout = g_force_timeout;
    if (blocks) {
        p.num_blocks = static_cast<int>(blocks->count);
        std::memcpy(p.blocks, blocks->entries, sizeof(uint16_t) * blocks->count);
    } else {
        int64_t nb = 0;
        build_blocks(Lp, ops.block_leaves, p.blocks, &nb);
        p.num_blocks = static_cast<int>(nb);
    }

    const int grid = static_cast<int>(units < st->sm_count ? units : st->sm_count);
    if (fixed_scratch && static_cast<size_t>(grid) * static_cast<size_t>(ops.scratch_cta_bytes) > fixed_bytes) {
        std::snprintf(g_detail, sizeof g_detail,
                      "this launch needs %zu bytes of scratch (%d CTAs x %d); the fixed scratch holds %zu",
                      static_cast<size_t>(grid) * static_cast<size_t>(ops.scratch_cta_bytes), grid,
                      ops.scratch_cta_bytes, fixed_bytes);
        return DET_GEMM_ERR_INVALID_ARG;
    }
    const cudaError_t le = ops.launch(p, grid, stream);
    if (le != cudaSuccess) return fail_cuda(DET_GEMM_ERR_LAUNCH, le, "kernel launch");
    if (parts > 1) {
        const cudaError_t me = launch_merge_parts(pa[0].out.esize == 4, p.part_out, parts, static_cast<int>(out_rows),
                                                  static_cast<int>(out_cols), part_ld, p.part_stride,
                                                  const_cast<void *>(pa[0].out.ptr), pa[0].out.ld, stream);
        if (me != cudaSuccess) return fail_cuda(DET_GEMM_ERR_LAUNCH, me, "merge launch");
    }
    // Row reductions: after the product, from the stored output, all
    // groups of the launch together.
    RowdotJob jobs[kMaxProblems];
    int n_jobs = 0;
    for (int i = 0; i < g; ++i) {
        if (!pa[i].rowdot || pa[i].rows == 0) continue;
        const ProblemArgs &q = pa[i];
        jobs[n_jobs++] = RowdotJob{static_cast<const uint16_t *>(q.out.ptr), static_cast<const uint16_t *>(q.d),
                                   q.out.ld, q.ldd, static_cast<int>(q.rows), q.rowdot};
    }
    if (n_jobs > 0) {
        const cudaError_t re = launch_rowdot(jobs, n_jobs, static_cast<int>(cols), reinterpret_cast<float *>(rd_slots),
                                             stream);
        if (re != cudaSuccess) return fail_cuda(DET_GEMM_ERR_LAUNCH, re, "row reduction launch");
    }
    return DET_GEMM_OK;
}

// One plain GEMM (see run_problems).
// The argument checks of run_problems for one plain product, without a launch.
det_gemm_status validate_plain(const Mat &a, const Mat &b, const Mat &out, int64_t rows, int64_t cols, int64_t kc)
{
    if (rows < 0 || cols < 0 || kc < 0) return DET_GEMM_ERR_INVALID_ARG;
    if (cols > (int64_t{1} << 31) - 256 || rows > (int64_t{1} << 31) - 256) return DET_GEMM_ERR_INVALID_ARG;
    if (kc > kKcMax) return DET_GEMM_ERR_K_TOO_LARGE;
    if (rows == 0 || cols == 0) return DET_GEMM_OK;
    det_gemm_status s;
    if ((s = check_mat(out)) != DET_GEMM_OK) return s;
    if (kc > 0) {
        if ((s = check_mat(a)) != DET_GEMM_OK) return s;
        if ((s = check_mat(b)) != DET_GEMM_OK) return s;
        if (overlaps(out, a) || overlaps(out, b)) return DET_GEMM_ERR_INVALID_ARG;
    }
    return DET_GEMM_OK;
}

// The busiest CTA's cost, in leaves, of a launch of `tiles` tiles over L
// leaves with the contraction split that choose_parts picks (its model).
int64_t launch_cost(int64_t tiles, int64_t L, int sms)
{
    const int parts = choose_parts(tiles, L, sms);
    return (tiles * parts + sms - 1) / sms * (L / parts) + (parts > 1 ? int64_t{8} : int64_t{0});
}

// Tail split of a plain launch. When its tiles fill some rounds of one CTA
// per SM and leave only a few tiles for the last round, the output's last
// column panels run as a second launch of few tiles, which choose_parts
// then splits at tree nodes over the otherwise idle SMs: QKV at 1024 rows
// has 768 = 5 x 152 + 8 tiles of 128 leaves; 760 of them fill five rounds
// and the other 8 run as 64 units of 16 leaves. Every element keeps its
// leaves and tree (a split is tree-aligned), so the bits are those of one
// launch. Returns the first column of the tail (a multiple of the tile
// width), or 0 when one launch is as fast: the second launch and its merge
// are counted as 24 leaves, and the split must save a twentieth.
int64_t tail_split_column(Variant v, int64_t rows, int64_t cols, int64_t kc)
{
    if (v != kBf16KMN && v != kBf16KK && v != kBf16MNMN && v != kF32KMN && v != kF32KK) return 0;
    if (rows <= 0 || cols <= 0 || kc <= 0) return 0;
    DeviceState *st = nullptr;
    if (device_state(&st) != DET_GEMM_OK) return 0;
    const int sms = st->sm_count;
    const int bn = variant_ops(v).bn;
    const int64_t m_tiles = (rows + kBM - 1) / kBM, n_tiles = (cols + bn - 1) / bn;
    const int64_t L = (kc + kLeaf - 1) / kLeaf;
    const int64_t tiles = m_tiles * n_tiles;
    if (tiles <= sms) return 0;
    const int64_t whole = launch_cost(tiles, L, sms);
    int64_t best = whole, best_c = 0;
    for (int64_t c = 1; c < n_tiles && m_tiles * c <= sms; ++c) {
        const int64_t cost = launch_cost(m_tiles * (n_tiles - c), L, sms) + launch_cost(m_tiles * c, L, sms) + 24;
        if (cost < best) {
            best = cost;
            best_c = c;
        }
    }
    if (best_c == 0 || best * 20 > whole * 19) return 0;
    return (n_tiles - best_c) * bn;
}

det_gemm_status run(Variant v, Mat a, bool a_kmajor, Mat b, bool b_kmajor, Mat out, int64_t rows, int64_t cols,
                    int64_t kc, cudaStream_t stream, void *fixed_scratch = nullptr, size_t fixed_bytes = 0)
{
    if (rows < 0 || cols < 0 || kc < 0) return DET_GEMM_ERR_INVALID_ARG;
    // A BF16 launch with a K-major A and few output rows takes the
    // transposed tile: the kernel's A operand is b (its rows are the
    // output's columns), its B operand is a, and the kernel stores
    // transposed. Same leaves, same tree, same bits as the plain tile.
    if ((v == kBf16KMN || v == kBf16KK) && a_kmajor && rows >= 1 && rows <= kSwapMaxRows && cols > 0 && kc > 0) {
        const ProblemArgs sw{b, a, out, cols, nullptr, 0, nullptr};
        return run_problems(b_kmajor ? kBf16SwapKK : kBf16SwapMNK, b_kmajor, true, &sw, 1, rows, kc, stream,
                            fixed_scratch, fixed_bytes);
    }
    const ProblemArgs pa{a, b, out, rows, nullptr, 0, nullptr};
    int64_t c0 = 0;
    if (!fixed_scratch && (c0 = tail_split_column(v, rows, cols, kc)) > 0) {
        // Validate the whole product first: argument errors come back before
        // anything is enqueued, as for an unsplit launch.
        det_gemm_status s = validate_plain(a, b, out, rows, cols, kc);
        if (s != DET_GEMM_OK) return s;
        Mat b_tail = b, out_tail = out;
        const Mat b_main = b_kmajor ? Mat{b.ptr, c0, b.cols, b.ld, b.esize} : Mat{b.ptr, b.rows, c0, b.ld, b.esize};
        if (b_kmajor) {
            b_tail.ptr = static_cast<const uint8_t *>(b.ptr) + c0 * b.ld * b.esize;
            b_tail.rows = cols - c0;
        } else {
            b_tail.ptr = static_cast<const uint8_t *>(b.ptr) + c0 * b.esize;
            b_tail.cols = cols - c0;
        }
        const Mat out_main{out.ptr, out.rows, c0, out.ld, out.esize};
        out_tail.ptr = static_cast<const uint8_t *>(out.ptr) + c0 * out.esize;
        out_tail.cols = cols - c0;
        const ProblemArgs pm{a, b_main, out_main, rows, nullptr, 0, nullptr};
        if ((s = run_problems(v, a_kmajor, b_kmajor, &pm, 1, c0, kc, stream)) != DET_GEMM_OK) return s;
        const ProblemArgs pt{a, b_tail, out_tail, rows, nullptr, 0, nullptr};
        return run_problems(v, a_kmajor, b_kmajor, &pt, 1, cols - c0, kc, stream);
    }
    return run_problems(v, a_kmajor, b_kmajor, &pa, 1, cols, kc, stream, fixed_scratch, fixed_bytes);
}

Mat bf16(const void *p, int64_t r, int64_t c, int64_t ld) { return Mat{p, r, c, ld, 2}; }
Mat f32(const void *p, int64_t r, int64_t c, int64_t ld) { return Mat{p, r, c, ld, 4}; }

// det_gemm_merge / det_gemm_merge_fp32: argument checks, then the merge of
// n parts in the tree's top-level order.
det_gemm_status merge_parts(const void *const *parts, int n, void *C, int64_t M, int64_t N, int64_t ldp,
                            int64_t ldc, int esize, cudaStream_t stream)
{
    if (n != 2 && n != 4 && n != 8) return DET_GEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || parts == nullptr) return DET_GEMM_ERR_INVALID_ARG;
    if (M > (int64_t{1} << 31) - 256 || N > (int64_t{1} << 31) - 256) return DET_GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DET_GEMM_OK;
    const Mat out{C, M, N, ldc, esize};
    det_gemm_status s = check_mat(out);
    if (s != DET_GEMM_OK) return s;
    for (int i = 0; i < n; ++i) {
        const Mat part{parts[i], M, N, ldp, esize};
        if ((s = check_mat(part)) != DET_GEMM_OK) return s;
        if (overlaps(out, part)) return DET_GEMM_ERR_INVALID_ARG;
    }
    DeviceState *st = nullptr;
    if ((s = device_state(&st)) != DET_GEMM_OK) return s;
    const cudaError_t e = launch_merge_list(esize == 4, parts, n, static_cast<int>(M), static_cast<int>(N), ldp, C,
                                            ldc, stream);
    if (e != cudaSuccess) return fail_cuda(DET_GEMM_ERR_LAUNCH, e, "merge launch");
    return DET_GEMM_OK;
}

}  // namespace

det_gemm_status fwd_with_fixed_scratch(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                                       int64_t lda, int64_t ldb, int64_t ldc, cudaStream_t stream, void *scratch,
                                       size_t scratch_bytes)
{
    if (M < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    return run(kBf16KMN, bf16(A, M, K, lda), true, bf16(B, K, N, ldb), false, bf16(C, M, N, ldc), M, N, K, stream,
               scratch, scratch_bytes);
}

int fwd_with_fixed_scratch_status(const void *A, const void *B, void *C, long long M, long long N, long long K,
                                  long long lda, long long ldb, long long ldc, cudaStream_t stream, void *scratch,
                                  size_t scratch_bytes)
{
    return static_cast<int>(fwd_with_fixed_scratch(A, B, C, M, N, K, lda, ldb, ldc, stream, scratch, scratch_bytes));
}

void record_detail(const char *msg) { std::snprintf(g_detail, sizeof g_detail, "%s", msg); }

int prepare_forward_status()
{
    DeviceState *st = nullptr;
    det_gemm_status s = device_state(&st);
    if (s == DET_GEMM_OK) s = prepare_variant(st, kBf16KMN);
    if (s == DET_GEMM_OK) s = prepare_variant(st, kBf16SwapMNK);
    return static_cast<int>(s);
}

}  // namespace detg

using namespace detg;

extern "C" {

det_gemm_status det_gemm_fwd(const det_gemm_bf16 *A, const det_gemm_bf16 *B, det_gemm_bf16 *C, int64_t M,
                             int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, det_gemm_stream stream)
{
    if (M < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    return run(kBf16KMN, bf16(A, M, K, lda), true, bf16(B, K, N, ldb), false, bf16(C, M, N, ldc), M, N, K,
               reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_gemm_fwd_rhs_transposed(const det_gemm_bf16 *A, const det_gemm_bf16 *W, det_gemm_bf16 *C,
                                            int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldw,
                                            int64_t ldc, det_gemm_stream stream)
{
    if (M < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    return run(kBf16KK, bf16(A, M, K, lda), true, bf16(W, N, K, ldw), true, bf16(C, M, N, ldc), M, N, K,
               reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_gemm_fwd_fp32(const det_gemm_bf16 *A, const det_gemm_bf16 *B, float *C, int64_t M, int64_t N,
                                  int64_t K, int64_t lda, int64_t ldb, int64_t ldc, det_gemm_stream stream)
{
    if (M < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    return run(kF32KMN, bf16(A, M, K, lda), true, bf16(B, K, N, ldb), false, f32(C, M, N, ldc), M, N, K,
               reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_gemm_fwd_fp32_rhs_transposed(const det_gemm_bf16 *A, const det_gemm_bf16 *W, float *C,
                                                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldw,
                                                 int64_t ldc, det_gemm_stream stream)
{
    if (M < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    return run(kF32KK, bf16(A, M, K, lda), true, bf16(W, N, K, ldw), true, f32(C, M, N, ldc), M, N, K,
               reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_gemm_da(const det_gemm_bf16 *dC, const det_gemm_bf16 *B, det_gemm_bf16 *dA, int64_t M,
                            int64_t N, int64_t K, int64_t lddc, int64_t ldb, int64_t ldda, det_gemm_stream stream)
{
    // dA[m, k] = sum_n dC[m, n] * B[k, n]: rows M, columns K, contraction N.
    // dC is [M, N] with n contiguous (K-major); B is [K, N] with n contiguous
    // (K-major for the columns k).
    if (M < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    return run(kBf16KK, bf16(dC, M, N, lddc), true, bf16(B, K, N, ldb), true, bf16(dA, M, K, ldda), M, K, N,
               reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_gemm_db(const det_gemm_bf16 *A, const det_gemm_bf16 *dC, det_gemm_bf16 *dB, int64_t M,
                            int64_t N, int64_t K, int64_t lda, int64_t lddc, int64_t lddb, det_gemm_stream stream)
{
    // dB[k, n] = sum_m A[m, k] * dC[m, n]: rows K, columns N, contraction M.
    // A is [M, K] with k contiguous (MN-major for rows k); dC is [M, N] with n
    // contiguous (MN-major for columns n).
    if (M < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    return run(kBf16MNMN, bf16(A, M, K, lda), false, bf16(dC, M, N, lddc), false, bf16(dB, K, N, lddb), K, N, M,
               reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_gemm_db_transposed(const det_gemm_bf16 *A, const det_gemm_bf16 *dC, det_gemm_bf16 *dBt,
                                       int64_t M, int64_t N, int64_t K, int64_t lda, int64_t lddc, int64_t lddbt,
                                       det_gemm_stream stream)
{
    // dBt[n, k] = sum_m dC[m, n] * A[m, k]: rows N, columns K, contraction M.
    if (M < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    return run(kBf16MNMN, bf16(dC, M, N, lddc), false, bf16(A, M, K, lda), false, bf16(dBt, N, K, lddbt), N, K, M,
               reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_gemm_fwd_grouped(int G, const det_gemm_bf16 *const *A, const det_gemm_bf16 *const *B,
                                     det_gemm_bf16 *const *C, const int64_t *M, int64_t N, int64_t K,
                                     const int64_t *lda, const int64_t *ldb, const int64_t *ldc,
                                     const det_gemm_bf16 *const *D, const int64_t *ldd, float *const *rowdot,
                                     det_gemm_stream stream)
{
    if (G < 0 || N < 0 || K < 0) return DET_GEMM_ERR_INVALID_ARG;
    if (G == 0) return DET_GEMM_OK;
    if (!A || !B || !C || !M || !lda || !ldb || !ldc) return DET_GEMM_ERR_INVALID_ARG;
    if (rowdot && (!D || !ldd)) return DET_GEMM_ERR_INVALID_ARG;
    if (rowdot && N > int64_t{kMaxLeaves} * 128) {
        for (int i = 0; i < G; ++i)
            if (rowdot[i]) return DET_GEMM_ERR_INVALID_ARG;   // more column tiles than the tree covers
    }
    // Every argument is checked before anything is enqueued.
    for (int i = 0; i < G; ++i) {
        if (M[i] < 0) return DET_GEMM_ERR_INVALID_ARG;
        if (rowdot && rowdot[i] && (!D[i] || ldd[i] < N)) return DET_GEMM_ERR_INVALID_ARG;
    }
    for (int base = 0; base < G; base += kMaxProblems) {
        const int g = std::min(kMaxProblems, G - base);
        ProblemArgs pa[kMaxProblems];
        for (int j = 0; j < g; ++j) {
            const int i = base + j;
            const bool rd = rowdot && rowdot[i];
            pa[j] = ProblemArgs{bf16(A[i], M[i], K, lda[i]), bf16(B[i], K, N, ldb[i]), bf16(C[i], M[i], N, ldc[i]),
                                M[i], rd ? D[i] : nullptr, rd ? ldd[i] : 0, rd ? rowdot[i] : nullptr};
        }
        // One problem is a plain launch (same bits).
        const Variant v = g > 1 ? kBf16KMNGrouped : kBf16KMN;
        const det_gemm_status s = run_problems(v, true, false, pa, g, N, K, reinterpret_cast<cudaStream_t>(stream));
        if (s != DET_GEMM_OK) return s;
    }
    return DET_GEMM_OK;
}

det_gemm_status det_gemm_merge(const det_gemm_bf16 *const *parts, int n, det_gemm_bf16 *C, int64_t M, int64_t N,
                               int64_t ldp, int64_t ldc, det_gemm_stream stream)
{
    return merge_parts(reinterpret_cast<const void *const *>(parts), n, C, M, N, ldp, ldc, 2,
                       reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_gemm_merge_fp32(const float *const *parts, int n, float *C, int64_t M, int64_t N, int64_t ldp,
                                    int64_t ldc, det_gemm_stream stream)
{
    return merge_parts(reinterpret_cast<const void *const *>(parts), n, C, M, N, ldp, ldc, 4,
                       reinterpret_cast<cudaStream_t>(stream));
}

det_gemm_status det_rmsnorm(const det_gemm_bf16 *x, const det_gemm_bf16 *w, det_gemm_bf16 *y, int64_t M,
                            int64_t D, float eps, int64_t ldx, int64_t ldy, det_gemm_stream stream)
{
    if (M < 0 || D < 0 || !(eps >= 0.0f)) return DET_GEMM_ERR_INVALID_ARG;
    if (M > (int64_t{1} << 31) - 256) return DET_GEMM_ERR_INVALID_ARG;
    if (M == 0 || D == 0) return DET_GEMM_OK;
    if (D > kKcMax) return DET_GEMM_ERR_K_TOO_LARGE;
    const Mat xm = bf16(x, M, D, ldx), ym = bf16(y, M, D, ldy), wm = bf16(w, 1, D, D + (8 - D % 8) % 8);
    det_gemm_status s;
    if ((s = check_mat(xm)) != DET_GEMM_OK) return s;
    if ((s = check_mat(ym)) != DET_GEMM_OK) return s;
    if ((s = check_mat(wm)) != DET_GEMM_OK) return s;
    // In place (y == x with the same pitch) is fine: a warp reads its whole
    // row before it writes any of it. Any other overlap is not.
    const bool in_place = static_cast<const void *>(x) == static_cast<const void *>(y) && ldx == ldy;
    if ((!in_place && overlaps(xm, ym)) || overlaps(wm, ym)) return DET_GEMM_ERR_INVALID_ARG;
    DeviceState *st = nullptr;
    if ((s = device_state(&st)) != DET_GEMM_OK) return s;
    RmsParams p;
    p.x = x;
    p.w = w;
    p.y = y;
    p.ldx = ldx;
    p.ldy = ldy;
    p.rows = static_cast<int>(M);
    p.d = static_cast<int>(D);
    p.num_leaves = static_cast<int>((D + kLeaf - 1) / kLeaf);
    p.eps = eps;
    const cudaError_t e = launch_rmsnorm(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(DET_GEMM_ERR_LAUNCH, e, "rmsnorm launch");
    return DET_GEMM_OK;
}

det_gemm_status det_gemm_check(det_gemm_stream stream)
{
    DeviceState *st = nullptr;
    det_gemm_status s = device_state(&st);
    if (s != DET_GEMM_OK) return s;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return DET_GEMM_ERR_CUDA;
    }
    int code = 0;
    if (cudaMemcpyFromSymbol(&code, g_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return DET_GEMM_ERR_CUDA;
    }
    if (code != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return DET_GEMM_ERR_CUDA;
        }
    }
    return code == 0 ? DET_GEMM_OK : static_cast<det_gemm_status>(code);
}

const char *det_gemm_status_string(det_gemm_status status)
{
    switch (status) {
    case DET_GEMM_OK: return "DET_GEMM_OK";
    case DET_GEMM_ERR_INVALID_ARG: return "DET_GEMM_ERR_INVALID_ARG: null pointer, bad size or leading dimension, or overlapping output";
    case DET_GEMM_ERR_K_TOO_LARGE: return "DET_GEMM_ERR_K_TOO_LARGE: contraction length above 32768";
    case DET_GEMM_ERR_ALIGNMENT: return "DET_GEMM_ERR_ALIGNMENT: pointer not 16-byte aligned or row pitch not a multiple of 16 bytes";
    case DET_GEMM_ERR_UNSUPPORTED_DEVICE: return "DET_GEMM_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
    case DET_GEMM_ERR_LAUNCH: return "DET_GEMM_ERR_LAUNCH: kernel set-up or launch failed";
    case DET_GEMM_ERR_TIMEOUT: return "DET_GEMM_ERR_TIMEOUT: a device-side bounded wait expired";
    case DET_GEMM_ERR_CUDA: return "DET_GEMM_ERR_CUDA: CUDA runtime error on the stream";
    default: return "DET_GEMM: unknown status";
    }
}

int det_gemm_abi_version(void) { return DET_GEMM_ABI_VERSION; }

const char *det_gemm_last_error_detail(void) { return g_detail; }

det_gemm_status det_gemm_tree_schedule(int64_t num_leaves, uint16_t *out)
{
    if (out == nullptr || num_leaves < 1 || num_leaves > kMaxLeaves) return DET_GEMM_ERR_INVALID_ARG;
    build_schedule(num_leaves, out);
    return DET_GEMM_OK;
}

det_gemm_status det_gemm_block_schedule(int64_t num_leaves, uint16_t *out, int64_t *num_blocks)
{
    if (out == nullptr || num_blocks == nullptr || num_leaves < 1 || num_leaves > kMaxLeaves)
        return DET_GEMM_ERR_INVALID_ARG;
    build_blocks(num_leaves, 4, out, num_blocks);
    return DET_GEMM_OK;
}

det_gemm_status det_gemm_block_schedule8(int64_t num_leaves, uint16_t *out, int64_t *num_blocks)
{
    if (out == nullptr || num_blocks == nullptr || num_leaves < 1 || num_leaves > kMaxLeaves)
        return DET_GEMM_ERR_INVALID_ARG;
    build_blocks(num_leaves, 8, out, num_blocks);
    return DET_GEMM_OK;
}

det_gemm_status det_gemm_shutdown(void)
{
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_scratch_count; ++i) {
        if (g_scratch[i].ptr) {
            int cur = 0;
            cudaGetDevice(&cur);
            cudaSetDevice(g_scratch[i].device);
            cudaFree(g_scratch[i].ptr);
            cudaSetDevice(cur);
        }
        g_scratch[i] = ScratchEntry{0, nullptr, nullptr, 0};
    }
    g_scratch_count = 0;
    g_scratch_next_evict = 0;
    cudaGetLastError();
    return DET_GEMM_OK;
}

det_gemm_status det_gemm_debug_force_timeout(int enable)
{
    std::lock_guard<std::mutex> lk(g_mu);
    g_force_timeout = enable ? 1 : 0;
    return DET_GEMM_OK;
}

}  // extern "C"
