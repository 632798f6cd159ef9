// The last step of a split launch: the top of the merge tree.
//
// A launch with few output tiles splits the contraction of every tile into
// `parts` equal, contiguous leaf ranges, one work unit each. Each range is a
// subtree of the fixed mid-split tree (RL-Kernel, "Batch-Invariant
// Deterministic GEMM (det_gemm)", section "Ascend NPU backend": a contiguous
// half-K GEMM is one child of the tree; the same holds level by level for
// quarters and eighths when the leaf count divides evenly), so each unit
// computes exactly the subtree the unsplit kernel would. This kernel merges
// the units' roots with the tree's top levels, in the tree's order:
// ((p0 + p1) + (p2 + p3)) for four parts, each add rounded once (BF16 adds
// for the bf16 variant, FP32 adds for the fp32 one). The result is the same
// bits as the unsplit launch; only the CTA doing the work differs.
#include "det_gemm.h"
#include "det_gemm_kernel.cuh"

namespace detg {
namespace {

constexpr int kMaxParts = 8;

// The parts' base addresses, passed by value.
struct PartPtrs {
    const uint8_t *p[kMaxParts];
};

// One thread per (row, two columns) for BF16 output or (row, column) for FP32.
template <bool F32>
__global__ void merge_parts_kernel(PartPtrs parts_at, int parts, int rows, int cols, long long part_ld,
                                   uint8_t *out, long long ldo)
{
    constexpr int ES = F32 ? 4 : 2;
    const int per_row = F32 ? cols : (cols + 1) / 2;
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<long long>(rows) * per_row) return;
    const int r = static_cast<int>(idx / per_row);
    const int j = static_cast<int>(idx - static_cast<long long>(r) * per_row);
    const int col = F32 ? j : 2 * j;
    const bool pair = F32 || col + 1 < cols;
    uint32_t v[kMaxParts];
#pragma unroll
    for (int i = 0; i < kMaxParts; ++i) {
        if (i < parts) {
            const uint8_t *src = parts_at.p[i] + (r * part_ld + col) * ES;
            v[i] = pair ? *reinterpret_cast<const uint32_t *>(src) : *reinterpret_cast<const uint16_t *>(src);
        }
    }
    // balanced tree over the parts, left operand first at every node
#pragma unroll
    for (int w = 1; w < kMaxParts; w *= 2) {
#pragma unroll
        for (int i = 0; i + w < kMaxParts; i += 2 * w)
            if (i + w < parts) v[i] = merge<F32>(v[i], v[i + w]);
    }
    uint8_t *dst = out + (static_cast<long long>(r) * ldo + col) * ES;
    if (pair) *reinterpret_cast<uint32_t *>(dst) = v[0];
    else *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(v[0] & 0xFFFFu);
}

cudaError_t launch_merge(bool f32, const PartPtrs &at, int parts, int rows, int cols, long long part_ld, void *out,
                         long long ldo, cudaStream_t stream)
{
    if (parts < 2 || parts > kMaxParts || (parts & (parts - 1)) != 0) return cudaErrorInvalidValue;
    const long long per_row = f32 ? cols : (cols + 1) / 2;
    const long long n = static_cast<long long>(rows) * per_row;
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (n + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    uint8_t *dst = static_cast<uint8_t *>(out);
    if (f32)
        merge_parts_kernel<true><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(at, parts, rows, cols, part_ld,
                                                                                        dst, ldo);
    else
        merge_parts_kernel<false><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(at, parts, rows, cols,
                                                                                         part_ld, dst, ldo);
    return cudaGetLastError();
}

// Row reduction of a grouped launch (Megatron Core notes, "Kernel redesign:
// the grouped-GEMM epilogue": a private slot per N-tile, then a fixed tree,
// instead of atomic adds across N-tiles). It runs after the product, from
// the stored output: rowdot_slots_kernel forms every (row, 128-column tile)
// slot, rowdot_reduce_kernel merges each row's slots by the mid-split tree
// of FP32 adds the contraction uses, walked with its per-leaf schedule. The
// same bits every run, whichever CTA computed which tile first.
// Up to kMaxProblems row reductions (the groups of one grouped launch, all
// with the same column count) in one pair of launches; the slots of all
// groups are one array, group g's starting at slot_off[g].
struct RowdotParams {
    const uint16_t *C[kMaxProblems];
    const uint16_t *D[kMaxProblems];
    float *rowdot[kMaxProblems];
    long long ldc[kMaxProblems], ldd[kMaxProblems];
    int row_start[kMaxProblems + 1];          // prefix sums of the groups' rows
    float *slots;                             // [n_tiles][total rows]
    int groups, cols, n_tiles;
    uint16_t sched[kMaxLeaves];
};

__device__ __forceinline__ int rowdot_group(const RowdotParams &p, int r)
{
    int g = 0;
    while (g + 1 < p.groups && r >= p.row_start[g + 1]) ++g;
    return g;
}

// One slot of the row reduction per thread: slot (t, row) = the FP32 sum
// of C[i, n] * D[i, n] over the columns n of tile t in ascending order,
// from +0. A product of two BF16 values is exact in FP32, so every step is
// one rounding, as in a leaf. Rows are 16-byte aligned and tiles start on
// 256 bytes, so whole groups of eight columns are read with 16-byte loads.
__global__ void rowdot_slots_kernel(const __grid_constant__ RowdotParams p)
{
    const int total = p.row_start[p.groups];
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<long long>(total) * p.n_tiles) return;
    const int r = static_cast<int>(idx / p.n_tiles);
    const int t = static_cast<int>(idx - static_cast<long long>(r) * p.n_tiles);
    const int g = rowdot_group(p, r);
    const int i = r - p.row_start[g];
    const int c0 = kRowdotTile * t;
    const int c1 = min(c0 + kRowdotTile, p.cols);
    const uint16_t *c = p.C[g] + static_cast<long long>(i) * p.ldc[g];
    const uint16_t *d = p.D[g] + static_cast<long long>(i) * p.ldd[g];
    auto bf = [](uint32_t h) { return __uint_as_float(h << 16); };
    float s = 0.0f;
    int n = c0;
    for (; n + 8 <= c1; n += 8) {
        const uint4 x = *reinterpret_cast<const uint4 *>(c + n);
        const uint4 y = *reinterpret_cast<const uint4 *>(d + n);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
        const uint32_t ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s = __fadd_rn(s, __fmul_rn(bf(xs[k] & 0xFFFFu), bf(ys[k] & 0xFFFFu)));
            s = __fadd_rn(s, __fmul_rn(bf(xs[k] >> 16), bf(ys[k] >> 16)));
        }
    }
    for (; n < c1; ++n) s = __fadd_rn(s, __fmul_rn(bf(c[n]), bf(d[n])));
    p.slots[static_cast<long long>(t) * total + r] = s;
}

// rowdot[i]: the slots of row i merged by the mid-split tree of FP32 adds,
// walked with its per-leaf schedule (det_gemm_tree_schedule, slots for
// leaves).
__global__ void rowdot_reduce_kernel(const __grid_constant__ RowdotParams p)
{
    const int total = p.row_start[p.groups];
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= total) return;
    float slot[kMaxSlots];
    float root = 0.0f;
    for (int t = 0; t < p.n_tiles; ++t) {
        float v = p.slots[static_cast<long long>(t) * total + r];
        const uint32_t e = p.sched[t];
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s)
            if ((e >> s) & 1u) v = __fadd_rn(slot[s], v);
        const uint32_t dst = e >> 12;
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s)
            if (dst == static_cast<uint32_t>(s)) slot[s] = v;
        if (dst == kSlotRoot) root = v;
    }
    const int g = rowdot_group(p, r);
    p.rowdot[g][r - p.row_start[g]] = root;
}

}  // namespace

cudaError_t launch_merge_parts(bool f32, const void *part, int parts, int rows, int cols, long long part_ld,
                               long long part_stride, void *out, long long ldo, cudaStream_t stream)
{
    if (parts < 2 || parts > kMaxParts) return cudaErrorInvalidValue;
    PartPtrs at{};
    for (int i = 0; i < parts; ++i) at.p[i] = static_cast<const uint8_t *>(part) + i * part_stride * (f32 ? 4 : 2);
    return launch_merge(f32, at, parts, rows, cols, part_ld, out, ldo, stream);
}

cudaError_t launch_merge_list(bool f32, const void *const *parts, int n, int rows, int cols, long long ldp, void *out,
                              long long ldo, cudaStream_t stream)
{
    if (n < 2 || n > kMaxParts) return cudaErrorInvalidValue;
    PartPtrs at{};
    for (int i = 0; i < n; ++i) at.p[i] = static_cast<const uint8_t *>(parts[i]);
    return launch_merge(f32, at, n, rows, cols, ldp, out, ldo, stream);
}

cudaError_t launch_rowdot(const RowdotJob *jobs, int n, int cols, float *slots, cudaStream_t stream)
{
    if (n < 1 || n > kMaxProblems) return cudaErrorInvalidValue;
    const int n_tiles = (cols + kRowdotTile - 1) / kRowdotTile;
    if (n_tiles < 1 || n_tiles > kMaxLeaves) return cudaErrorInvalidValue;
    RowdotParams p;
    p.groups = n;
    p.cols = cols;
    p.n_tiles = n_tiles;
    p.slots = slots;
    p.row_start[0] = 0;
    for (int g = 0; g < n; ++g) {
        p.C[g] = jobs[g].C;
        p.D[g] = jobs[g].D;
        p.ldc[g] = jobs[g].ldc;
        p.ldd[g] = jobs[g].ldd;
        p.rowdot[g] = jobs[g].rowdot;
        p.row_start[g + 1] = p.row_start[g] + jobs[g].rows;
    }
    const int total = p.row_start[n];
    if (total <= 0) return cudaSuccess;
    if (det_gemm_tree_schedule(n_tiles, p.sched) != DET_GEMM_OK) return cudaErrorInvalidValue;
    const int threads = 128;
    const long long work = static_cast<long long>(total) * n_tiles;
    rowdot_slots_kernel<<<static_cast<unsigned>((work + threads - 1) / threads), threads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    rowdot_reduce_kernel<<<(total + threads - 1) / threads, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace detg
