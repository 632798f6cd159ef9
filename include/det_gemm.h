/*
 * det_gemm -- batch-invariant deterministic BF16 GEMM for GB300 (sm_103a).
 *
 * Operation (RL-Kernel, "Batch-Invariant Deterministic GEMM (det_gemm)",
 * sections "Guarantees", "Ascend NPU backend" and "Dtypes"):
 *
 *   For every output element, with contraction length Kc and pairs
 *   (x_k, y_k), the K range is cut into L = ceil(Kc / 32) leaves of 32
 *   consecutive k (the last one may be shorter). Each leaf is summed in FP32
 *   and rounded once to BF16 (round to nearest, ties to even). The L leaves
 *   are merged by a fixed mid-split binary tree of BF16 adds:
 *       T(lo, hi) = leaf[lo]                         if hi - lo == 1
 *                 = bf16(T(lo, mid) + T(mid, hi))    otherwise, mid = (lo + hi) / 2
 *   (integer division; for an odd range the left child holds the smaller
 *   half). No TF32, and no split-K that combines partial sums in a
 *   launch-dependent order (a launch with few output tiles may split its
 *   contraction, but only at nodes of this tree, which gives the same bits):
 *   the bits of an output element depend only on its own row of the left
 *   operand and its own column of the right one, never on M, on how rows are
 *   chunked or padded, or on which CTA computed it. When L is even, a contiguous half-K product is one child of the root,
 *   so bf16(first_half + second_half) equals the full product bit for bit.
 *
 *   How an output is tiled is an implementation choice that never shows in
 *   the bits: BF16 launches with at most 64 output rows (fwd,
 *   fwd_rhs_transposed, da) run a transposed tile whose MMA lanes carry the
 *   output columns, and produce the same bits as the plain tile.
 *
 *   Within a leaf the FP32 sum is formed by the tensor core; its internal
 *   summation order differs from a sequential loop, so a leaf can differ from
 *   a sequential FP32 leaf by one BF16 unit when it lies next to a rounding
 *   midpoint. The page claims batch invariance and the half-K property, not
 *   bit parity across platforms ("Ascend NPU backend", last bullet).
 *
 * Conventions for every GEMM entry point below:
 *   - All matrices are row-major with a leading dimension (ld*) counted in
 *     elements: element (r, c) of X lives at X[r * ldx + c].
 *   - Pointers are DEVICE pointers owned by the caller; the library never
 *     frees or retains them after the call returns.
 *   - M, N, K are the shapes of the forward product A[M,K] @ B[K,N] = C[M,N];
 *     the backward entry points take the same M, N, K as their forward.
 *   - The contraction length Kc (K for the forward entry points, N for dA,
 *     M for dB) must be <= DET_GEMM_KC_MAX (32768, the page's "training
 *     contract" cap on the reduction dimension).
 *   - Base pointers must be 16-byte aligned and ld * sizeof(element) must be
 *     a multiple of 16 bytes (the tensor-memory-access engine's rule).
 *   - Work is enqueued on `stream` and the call returns without waiting.
 *     Argument errors are returned synchronously before anything is
 *     enqueued. An empty output (a zero dimension) returns DET_GEMM_OK with
 *     nothing enqueued; Kc == 0 fills the output with +0.
 *   - Outputs must not overlap inputs (DET_GEMM_ERR_INVALID_ARG otherwise).
 *   - A device-side failure (a bounded wait that expired) is reported by
 *     det_gemm_check(), not by the launching call.
 *   - The library keeps one device scratch buffer per (device, stream) it has
 *     launched on: one CTA per SM x 144 KiB for the tree's most rarely
 *     touched pending partials, followed, when a launch needs them, by the
 *     part products of a launch that splits its contraction (parts x the
 *     output's size) and the grouped row reduction's per-tile slots. It is
 *     created on the first launch on that stream and reused by every later
 *     one; a launch that needs more replaces it with a larger one
 *     (cudaFree, which waits for the device, then cudaMalloc). Launches on
 *     different streams never share it. det_gemm_shutdown() releases them;
 *     det_gemm_fwd_noalloc allocates nothing.
 */
#ifndef DET_GEMM_H
#define DET_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A BF16 value as its raw 16-bit pattern. */
typedef uint16_t det_gemm_bf16;

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *det_gemm_stream;

typedef enum {
    DET_GEMM_OK = 0,
    DET_GEMM_ERR_INVALID_ARG = 1,        /* null pointer, negative size, ld too small, overlap */
    DET_GEMM_ERR_K_TOO_LARGE = 2,        /* contraction length > DET_GEMM_KC_MAX */
    DET_GEMM_ERR_ALIGNMENT = 3,          /* base not 16-byte aligned or ld*size not a multiple of 16 */
    DET_GEMM_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
    DET_GEMM_ERR_LAUNCH = 5,             /* the CUDA launch or set-up failed */
    DET_GEMM_ERR_TIMEOUT = 6,            /* a device-side bounded wait expired (det_gemm_check) */
    DET_GEMM_ERR_CUDA = 7                /* another CUDA runtime error (det_gemm_check) */
} det_gemm_status;

#define DET_GEMM_KC_MAX 32768
#define DET_GEMM_LEAF 32
#define DET_GEMM_ABI_VERSION 1

/*
 * Forward, C[M,N] = A[M,K] @ B[K,N], BF16 out.
 * ("Guarantees": forward C = A @ B; "Usage": a is [M,K], b is [K,N].)
 */
det_gemm_status det_gemm_fwd(const det_gemm_bf16 *A, const det_gemm_bf16 *B, det_gemm_bf16 *C,
                             int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldc, det_gemm_stream stream);

/*
 * Forward with the weight stored [N,K]: C[M,N] = A[M,K] @ W[N,K]^T.
 * ("Ascend NPU backend": the fwd_rhs_transposed entry point.)
 */
det_gemm_status det_gemm_fwd_rhs_transposed(const det_gemm_bf16 *A, const det_gemm_bf16 *W,
                                            det_gemm_bf16 *C, int64_t M, int64_t N, int64_t K,
                                            int64_t lda, int64_t ldw, int64_t ldc,
                                            det_gemm_stream stream);

/*
 * Forward with FP32 output, C[M,N] = A[M,K] @ B[K,N]. Same leaves and the
 * same tree, but the leaves stay FP32 and the merges are FP32 adds (round to
 * nearest even). ("Dtypes": forward_fp32 returns FP32.)
 */
det_gemm_status det_gemm_fwd_fp32(const det_gemm_bf16 *A, const det_gemm_bf16 *B, float *C,
                                  int64_t M, int64_t N, int64_t K,
                                  int64_t lda, int64_t ldb, int64_t ldc, det_gemm_stream stream);

/*
 * FP32-output forward with the weight stored [N,K]: C[M,N] = A @ W^T.
 * Not among the page's names; it is the fwd_fp32 product with the
 * fwd_rhs_transposed operand layout, for an LM head whose weight is [N,K].
 */
det_gemm_status det_gemm_fwd_fp32_rhs_transposed(const det_gemm_bf16 *A, const det_gemm_bf16 *W,
                                                 float *C, int64_t M, int64_t N, int64_t K,
                                                 int64_t lda, int64_t ldw, int64_t ldc,
                                                 det_gemm_stream stream);

/*
 * Input gradient, dA[M,K] = dC[M,N] @ B[K,N]^T (contraction over N).
 * ("Guarantees": backward dA = dC.B^T; "Ascend NPU backend": backward reuses
 * the forward product on transposed operands.)
 */
det_gemm_status det_gemm_da(const det_gemm_bf16 *dC, const det_gemm_bf16 *B, det_gemm_bf16 *dA,
                            int64_t M, int64_t N, int64_t K,
                            int64_t lddc, int64_t ldb, int64_t ldda, det_gemm_stream stream);

/*
 * Weight gradient, dB[K,N] = A[M,K]^T @ dC[M,N] (contraction over M).
 * ("Guarantees": backward dB = A^T.dC.)
 */
det_gemm_status det_gemm_db(const det_gemm_bf16 *A, const det_gemm_bf16 *dC, det_gemm_bf16 *dB,
                            int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t lddc, int64_t lddb, det_gemm_stream stream);

/*
 * Weight gradient written in the canonical weight layout [N,K]:
 * dBt[N,K] = (A^T @ dC)^T = dC[M,N]^T @ A[M,K] (contraction over M).
 * ("Ascend NPU backend": db_transposed stores the weight gradient born
 * contiguous in [N,K].) Bit for bit the transpose of det_gemm_db.
 */
det_gemm_status det_gemm_db_transposed(const det_gemm_bf16 *A, const det_gemm_bf16 *dC,
                                       det_gemm_bf16 *dBt, int64_t M, int64_t N, int64_t K,
                                       int64_t lda, int64_t lddc, int64_t lddbt,
                                       det_gemm_stream stream);

/*
 * Grouped forward product: C_g = A_g @ B_g for g < G (the expert GEMMs of a
 * mixture-of-experts layer), every group with its own rows M[g] and
 * operands, all with the same N and K. Groups are taken eight at a time,
 * each eight in one persistent launch over all their output tiles. Every
 * tile is computed end to end by one CTA with the same leaves and merge
 * tree as det_gemm_fwd, so C_g is det_gemm_fwd(A_g, B_g) bit for bit: a
 * token's result does not depend on how many tokens its expert received.
 *
 * Optional row reduction (the per-token quantity the Megatron Core notes
 * describe as accumulated atomically across N-tiles, section "Kernel
 * redesign: the grouped-GEMM epilogue"): when rowdot and rowdot[g] are not
 * NULL, rowdot[g][i] = sum over n of C_g[i, n] * D_g[i, n] in FP32, formed
 * with one private slot per 128-column N-tile and a fixed reduction order,
 * never with atomics: a tile's slot is the FP32 sum of its (exact) products
 * in ascending column order from +0, and the slots are merged by the
 * mid-split tree of FP32 adds. The reduction runs after the product, from
 * the stored C_g. Same bits every run. N must then be <= 131072 (1024
 * column tiles).
 *
 *   A[g]    device, [M[g],K] BF16, row pitch lda[g]
 *   B[g]    device, [K,N] BF16, row pitch ldb[g]
 *   C[g]    device, [M[g],N] BF16, row pitch ldc[g]
 *   D[g], ldd[g]  device, [M[g],N] BF16 (only where rowdot[g] is used)
 *   rowdot[g]     device, [M[g]] FP32, 16-byte aligned, or NULL
 * A, B, C, M, lda, ldb, ldc, D, ldd and rowdot are host arrays of G entries
 * (D, ldd and rowdot may be NULL altogether). Alignment and aliasing rules
 * are det_gemm_fwd's; the outputs of different groups must not overlap.
 * Asynchronous on `stream`. Errors as det_gemm_fwd; every group's arguments
 * are checked before the first launch of a call is enqueued only for the
 * counts and pointers above, so a later batch of eight can still fail its
 * own checks after an earlier one was enqueued.
 */
det_gemm_status det_gemm_fwd_grouped(int G, const det_gemm_bf16 *const *A, const det_gemm_bf16 *const *B,
                                     det_gemm_bf16 *const *C, const int64_t *M, int64_t N, int64_t K,
                                     const int64_t *lda, const int64_t *ldb, const int64_t *ldc,
                                     const det_gemm_bf16 *const *D, const int64_t *ldd, float *const *rowdot,
                                     det_gemm_stream stream);

/*
 * Merges partial products over contiguous contraction ranges into the full
 * product: the deterministic composition of a contraction sharded over n
 * GPUs or streams (RL-Kernel, "Batch-Invariant Deterministic GEMM
 * (det_gemm)", section "Ascend NPU backend": a contiguous half-K GEMM is one
 * child of the merge tree, so two half-K results merge to the full-K result
 * bit for bit; tensor-parallel GEMM itself is outside det_gemm, section
 * "Scope").
 *
 * parts[i] (i < n, n = 2, 4 or 8) is the det_gemm result [M,N] of the i-th
 * of n equal contiguous leaf ranges of the contraction: with L = ceil(Kc/32)
 * leaves and L divisible by n, part i covers contraction indices
 * [i*Kc/n, (i+1)*Kc/n) when Kc is a multiple of 32*n (the last part may end
 * in a partial leaf). Then every range is a subtree of the fixed mid-split
 * tree and this call applies the tree's top log2(n) levels in their order,
 * ((p0 + p1) + (p2 + p3)) for n = 4, each add rounded once to BF16 (RNE):
 * C equals the full det_gemm bit for bit. With other ranges the result is
 * still deterministic but is not that tree.
 *
 *   parts  host array of n device pointers, each [M,N] BF16, row pitch ldp
 *          elements (the same for all parts)
 *   C      device, [M,N] BF16, row pitch ldc; must not overlap any part
 * Pointers and row pitches must be 16-byte aligned. Asynchronous on
 * `stream`; nothing is allocated. Errors: DET_GEMM_ERR_INVALID_ARG (n not 2,
 * 4 or 8, null pointer, negative size, ld < N, overlap),
 * DET_GEMM_ERR_ALIGNMENT, DET_GEMM_ERR_UNSUPPORTED_DEVICE,
 * DET_GEMM_ERR_LAUNCH.
 */
det_gemm_status det_gemm_merge(const det_gemm_bf16 *const *parts, int n, det_gemm_bf16 *C, int64_t M, int64_t N,
                               int64_t ldp, int64_t ldc, det_gemm_stream stream);

/* det_gemm_merge for FP32 partial products (det_gemm_fwd_fp32 and
 * det_gemm_fwd_fp32_rhs_transposed): the same tree with FP32 adds (RNE). */
det_gemm_status det_gemm_merge_fp32(const float *const *parts, int n, float *C, int64_t M, int64_t N, int64_t ldp,
                                    int64_t ldc, det_gemm_stream stream);

/*
 * Batch-invariant RMSNorm: y[i, :] = x[i, :] / sqrt(mean_j x[i, j]^2 + eps)
 * * w, BF16 in and out ("Comment vaincre le non-déterminisme dans
 * l'inférence des LLM", section "RMSNorm": every row reduced by one core in
 * a fixed order, whatever the batch size). The pages give the strategy; the
 * arithmetic is this library's reading, each step rounded once to nearest
 * even: ss = sum of x_j^2 reduced as det_gemm's FP32 variant reduces a
 * contraction (32-element FP32 leaves, mid-split tree of FP32 adds);
 * r = 1 / sqrt(ss / D + eps) in FP32; y_j = RNE_bf16((x_j * r) * w_j).
 * A row's result therefore depends on that row, w and eps only: not on M,
 * on the other rows, or on the run.
 *
 *   x  device, [M,D] BF16, row pitch ldx elements
 *   w  device, [D] BF16
 *   y  device, [M,D] BF16, row pitch ldy; y == x with ldy == ldx (in place)
 *      is allowed, any other overlap with x or w is not
 * Pointers and row pitches must be 16-byte aligned; D <= 32768; eps >= 0.
 * Asynchronous on `stream`; nothing is allocated. Errors:
 * DET_GEMM_ERR_INVALID_ARG, DET_GEMM_ERR_K_TOO_LARGE (D > 32768),
 * DET_GEMM_ERR_ALIGNMENT, DET_GEMM_ERR_UNSUPPORTED_DEVICE,
 * DET_GEMM_ERR_LAUNCH. M == 0 or D == 0 enqueues nothing.
 */
det_gemm_status det_rmsnorm(const det_gemm_bf16 *x, const det_gemm_bf16 *w, det_gemm_bf16 *y, int64_t M,
                            int64_t D, float eps, int64_t ldx, int64_t ldy, det_gemm_stream stream);

/*
 * det_gemm_fwd for callers that cannot allocate device memory. The pages
 * describing det_gemm have no counterpart to this entry point.
 *
 * det_gemm_fwd allocates a scratch buffer with cudaMalloc on its first
 * launch on a stream. Callers that run on a memory arena they manage
 * themselves, or that must never trigger an allocation's device-wide
 * synchronisation, cannot accept that. This entry
 * point computes exactly the same product, bit for bit, with the scratch in
 * a fixed 15 MiB array compiled into the library (every GPU that loads the
 * library holds it until the process exits), and allocates nothing: no
 * cudaMalloc, no cudaFree, no host allocation.
 *
 *   - The first call on a device does all of the set-up for that device:
 *     the library's state, the attributes of both kernels a forward launch
 *     can take (the plain tile, and the transposed tile for at most 64
 *     rows), and the array's device address (cudaGetSymbolAddress). Later
 *     calls do none of it. Make that first call before any stream capture.
 *   - The array holds scratch for 160 CTAs (one per SM up to 160 SMs). A
 *     launch that would need more is rejected with DET_GEMM_ERR_INVALID_ARG
 *     before anything is enqueued (det_gemm_last_error_detail says why).
 *   - Every call shares the array and nothing in it needs to start at zero
 *     (each pending partial is written before it is read). Calls that
 *     overlap on the GPU (different streams) race on it: serialise them.
 *   - Arguments, layouts and errors are those of det_gemm_fwd.
 */
det_gemm_status det_gemm_fwd_noalloc(const det_gemm_bf16 *A, const det_gemm_bf16 *B, det_gemm_bf16 *C,
                                     int64_t M, int64_t N, int64_t K,
                                     int64_t lda, int64_t ldb, int64_t ldc, det_gemm_stream stream);

/*
 * Waits for `stream`, then reports and clears the device status word of the
 * current device: DET_GEMM_OK, DET_GEMM_ERR_TIMEOUT when a kernel gave up a
 * bounded wait since the last check, or DET_GEMM_ERR_CUDA when the stream
 * itself reports a CUDA error.
 */
det_gemm_status det_gemm_check(det_gemm_stream stream);

/* Static, human-readable name of a status code. Never NULL. */
const char *det_gemm_status_string(det_gemm_status status);

/* DET_GEMM_ABI_VERSION of the loaded library. */
int det_gemm_abi_version(void);

/*
 * The calling thread's record of the CUDA error behind its last
 * DET_GEMM_ERR_LAUNCH (name and message), or "" if none was recorded.
 * Static per-thread storage; never NULL.
 */
const char *det_gemm_last_error_detail(void);

/*
 * Host-only helper, no GPU needed: the per-leaf merge schedule the kernels
 * apply for a contraction of `num_leaves` leaves (1..1024). out[l] describes
 * what follows leaf l in an in-order walk of the mid-split tree: bits 0..9
 * are the pending-partial slots merged into the running value, lowest slot
 * first (slot s holds the left child of a node of height s + 1); bits 12..15
 * are the slot the result is parked in, or 15 when it is the root.
 * `out` is caller-owned host memory of num_leaves entries.
 * DET_GEMM_ERR_INVALID_ARG for a bad count or a NULL out.
 */
det_gemm_status det_gemm_tree_schedule(int64_t num_leaves, uint16_t *out);

/*
 * Host-only helper, no GPU needed: the block schedule the plain-tile kernels
 * walk. The tree is cut into its maximal subtrees of at most four leaves
 * (for a tree of more than four leaves these have 2, 3 or 4 leaves), in
 * leaf order;
 * out[b] describes block b: bits 10..11 hold (leaves in the block - 1);
 * bits 0..9 the pending-partial slots its value is merged with, lowest
 * first; bits 12..15 the slot its result is parked in, or 15 for the root
 * (the last block, and only it). It is the per-leaf entry of the block's last leaf (det_gemm_tree_schedule)
 * with the merges inside the block removed. `out` needs num_leaves entries;
 * *num_blocks receives the count.
 */
det_gemm_status det_gemm_block_schedule(int64_t num_leaves, uint16_t *out, int64_t *num_blocks);

/*
 * Host-only helper, no GPU needed: the block schedule of the transposed
 * tile (launches with at most 64 output rows). The tree is cut into its
 * maximal subtrees of at most eight leaves (for a tree of more than eight
 * leaves these have 4 to 8 leaves), in leaf order. Such a block's parent has
 * more than eight leaves, so its merges and its parking slot are slot 3 or
 * higher, and out[b] holds: bits 0..2 (leaves in the block - 1); bits 3..9
 * the pending-partial slots its value is merged with, lowest first; bits
 * 12..15 the slot its result is parked in, or 15 for the root (the last
 * block, and only it). The kernel evaluates a block of n leaves as a left
 * half of n/2 (rounded down) and a right half of the rest, each of one to
 * four leaves shaped as in the mid-split tree. `out` needs num_leaves
 * entries; *num_blocks receives the count. DET_GEMM_ERR_INVALID_ARG for a
 * bad count or a NULL pointer.
 */
det_gemm_status det_gemm_block_schedule8(int64_t num_leaves, uint16_t *out, int64_t *num_blocks);

/*
 * Frees the per-stream scratch buffers and forgets them; the next launch on
 * a stream allocates again. Call only when no det_gemm work is in flight
 * (it waits for the devices it frees on).
 */
det_gemm_status det_gemm_shutdown(void);

/*
 * Test hook: while `enable` is nonzero, every GEMM launch makes its MMA warp
 * wait on a barrier that nothing signals, with a short bound (about 50 ms).
 * The wait expires, the kernel abandons its work, releases its tensor
 * memory and returns, and det_gemm_check() reports DET_GEMM_ERR_TIMEOUT; the
 * CUDA context stays usable. Outputs of such launches are undefined.
 */
det_gemm_status det_gemm_debug_force_timeout(int enable);

#ifdef __cplusplus
}
#endif

#endif /* DET_GEMM_H */
