// Internal declarations shared by the det_gemm host code and kernel
// translation units. Not part of the public C-ABI (include/det_gemm.h).
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace detg {

constexpr int kLeaf = 32;                 // contraction elements per leaf
constexpr int kKcMax = 32768;             // cap on the contraction length
constexpr int kMaxLeaves = kKcMax / kLeaf;
constexpr int kSlotRoot = 15;             // schedule "store" value for the root
constexpr int kMaxSlots = 10;             // ceil(log2(kMaxLeaves)) pending partials
constexpr int kBM = 128;                  // output rows per tile (one TMEM lane per row)
constexpr int kBK = 64;                   // contraction elements per shared-memory stage (two leaves)
constexpr int kStageWarps = 4;            // TMA copies and MMAs of the K-stages: one per SM sub-partition
constexpr int kProdRegs = 40;             // stage warpgroup after setmaxnreg

// Operand major-ness as seen by the MMA: K-major = contraction contiguous.
enum Major { kKMajor = 0, kMNMajor = 1 };

// Kernel variants: (A operand major, B operand major, output type).
enum Variant {
    kBf16KMN = 0,   // fwd: A[M,K] K-major, B[K,N] N-major
    kBf16KK,        // fwd_rhs_transposed, da: both K-major
    kBf16MNMN,      // db, db_transposed: both MN-major
    kF32KMN,        // fwd_fp32
    kF32KK,         // fwd_fp32 with a [N,K] weight
    kBf16KMNGrouped,   // fwd_grouped: several problems per launch, optional row reduction
    kBf16SwapMNK,   // fwd with at most kSwapMaxRows rows: transposed tile, A = B[K,N] (MN-major), B = A[M,K]
    kBf16SwapKK,    // fwd_rhs_transposed, da with few rows: transposed tile, both K-major
    kVariantCount
};

// Division of a non-negative int below 2^31 by a fixed divisor d >= 1 as
// one 64-bit multiply and a shift: q = (n * mul) >> shift with
// shift = 32 + ceil(log2 d) and mul = ceil(2^shift / d) (at most 2^33). The
// error term mul * d - 2^shift is below d <= 2^(shift - 32), so n * that
// error stays below 2^shift for every n < 2^32 and the floor is exact
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994). The kernels divide tile indices this way instead
// of with the runtime's integer division, a long dependent chain.
struct FastDiv {
    unsigned long long mul;
    unsigned int shift;
};

inline FastDiv make_fast_div(unsigned int d)
{
    unsigned int s = 0;
    while ((1ull << s) < d) ++s;
    FastDiv f;
    f.shift = 32 + s;
    f.mul = ((1ull << f.shift) + d - 1) / d;
    return f;
}

// Everything a launch needs; passed by value as a __grid_constant__ param.
// One GEMM of a launch. A plain launch has one; a grouped launch
// (det_gemm_fwd_grouped) has one per group, all with the same columns and
// contraction.
struct Problem {
    CUtensorMap tmap_a;           // "A operand": output rows x contraction
    CUtensorMap tmap_b;           // "B operand": contraction x output columns
    void *out;                    // row-major output, rows x cols
    long long ldo;                // output leading dimension, elements
    int rows;                     // output rows
    int m_tiles;
    int first_unit;               // index of this problem's first work unit in the launch
    int stage_tx;                 // bytes one K-stage's TMA copies bring in (A box + B box)
    int group;                    // tile order: tiles of this many row (or column) panels per group
    int rows_fast;                // 1: row tiles vary fastest (A panels stay in L2), 0: column tiles
    int span;                     // tiles per group: group x the other operand's panel count
    FastDiv div_span, div_group, div_last;   // by span, by group, by the last group's panel count
};

constexpr int kMaxProblems = 8;

struct Params {
    Problem prob[kMaxProblems];
    int num_problems;
    int units;                    // work units of the launch (all problems)
    void *scratch;                // deep-slot scratch: grid x VariantOps::scratch_cta_bytes
    int *status;                  // device status word (first int = code)
    unsigned long long timeout_ns;
    int cols, kc;
    int n_tiles;
    int num_leaves;               // leaves per work unit (the whole contraction when parts == 1)
    int parts;                    // contraction parts per tile: subtrees of the merge tree (1, 2, 4, 8)
    FastDiv div_parts, div_stages;    // by parts, by the K-stages per work unit
    void *part_out;               // parts > 1: part p of tile rows/cols goes to part_out + p * part_stride
    long long part_ld, part_stride;   // elements
    int force_timeout;
    int num_blocks;
    uint16_t blocks[kMaxLeaves];  // block schedule (see det_gemm_block_schedule)
};

struct VariantOps {
    // Sets the kernel's shared-memory attribute; reports registers per thread.
    cudaError_t (*prepare)(int *num_regs);
    cudaError_t (*launch)(const Params &p, int grid, cudaStream_t stream);
    int bn;                       // output columns per tile
    int smem_bytes;
    int scratch_cta_bytes;        // global scratch each CTA needs for its deep slots
    int split_regs;               // registers per thread the kernel must be built with (0: no register split)
    bool swap;                    // transposed tile: the kernel's rows are the output's columns
    int block_leaves;             // leaves per block of the block schedule the kernel walks (4 or 8)
};

// Output rows up to which a BF16 launch uses the transposed tile.
constexpr int kSwapMaxRows = 64;

// Merges the `parts` partial results of a split launch into the output with
// the top levels of the merge tree (parts is a power of two; part p is leaf
// range p of equal ranges, so the tree over them is the balanced one).
cudaError_t launch_merge_parts(bool f32, const void *part, int parts, int rows, int cols, long long part_ld,
                               long long part_stride, void *out, long long ldo, cudaStream_t stream);

// The same merge over n separately allocated parts (det_gemm_merge).
cudaError_t launch_merge_list(bool f32, const void *const *parts, int n, int rows, int cols, long long ldp, void *out,
                              long long ldo, cudaStream_t stream);

// Row reduction of a grouped launch: rowdot[i] = sum over n of C[i, n] *
// D[i, n] in a fixed order (one slot per 128-column tile, the FP32 sum of
// its products in ascending column order; slots merged by the mid-split
// tree), for n <= kMaxProblems groups with the same column count in one
// pair of launches. `slots` is scratch for ceil(cols / 128) floats per row
// of all groups together.
constexpr int kRowdotTile = 128;
struct RowdotJob {
    const uint16_t *C;            // [rows, cols] BF16, row pitch ldc
    const uint16_t *D;            // [rows, cols] BF16, row pitch ldd
    long long ldc, ldd;
    int rows;
    float *rowdot;                // [rows] FP32
};
cudaError_t launch_rowdot(const RowdotJob *jobs, int n, int cols, float *slots, cudaStream_t stream);

// Batch-invariant RMSNorm (det_rmsnorm): one warp per row.
struct RmsParams {
    const uint16_t *x;            // [rows, d] BF16, row pitch ldx
    const uint16_t *w;            // [d] BF16
    uint16_t *y;                  // [rows, d] BF16, row pitch ldy
    long long ldx, ldy;           // elements
    int rows, d, num_leaves;
    float eps;
};
constexpr int kRmsWarps = 8;      // rows per CTA
cudaError_t launch_rmsnorm(const RmsParams &p, cudaStream_t stream);

// Largest scratch_cta_bytes over all variants (slots 7-9 in global
// scratch: fp32 3 x 48 KiB, bf16 3 x 32 KiB).
constexpr int kMaxScratchCtaBytes = 3 * 49152;

VariantOps ops_bf16_kmn();
VariantOps ops_bf16_kk();
VariantOps ops_bf16_mnmn();
VariantOps ops_f32_kmn();
VariantOps ops_f32_kk();
VariantOps ops_bf16_kmn_grouped();
VariantOps ops_bf16_swap_mnk();
VariantOps ops_bf16_swap_kk();

// det_gemm_fwd with a caller-provided scratch buffer: nothing is allocated,
// device or host. Returns a det_gemm_status.
int fwd_with_fixed_scratch_status(const void *A, const void *B, void *C, long long M, long long N, long long K,
                                  long long lda, long long ldb, long long ldc, cudaStream_t stream, void *scratch,
                                  size_t scratch_bytes);
// Stores a message for det_gemm_last_error_detail().
void record_detail(const char *msg);
// Sets up the current device's library state and both kernels a BF16
// forward launch can take (the plain tile, and the transposed tile for at
// most kSwapMaxRows rows). Returns a det_gemm_status.
int prepare_forward_status();

}  // namespace detg
