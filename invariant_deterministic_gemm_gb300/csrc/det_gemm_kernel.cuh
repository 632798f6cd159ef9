// det_gemm kernel for sm_103a: TMA -> shared memory -> tcgen05 MMA into TMEM,
// one 32-wide K leaf per accumulator, leaf rounding and the fixed mid-split
// merge tree applied by the epilogue warps.
//
// Arithmetic (RL-Kernel, "Batch-Invariant Deterministic GEMM (det_gemm)",
// sections "Guarantees" and "Ascend NPU backend"): FP32 accumulation inside
// 32-element leaves, each leaf rounded once to BF16 (RNE), leaves merged by
// BF16 adds in a fixed mid-split tree; FP32 leaves and FP32 adds for the
// fp32-output variant ("Dtypes"). Every output element is produced end to
// end by one CTA in a fixed leaf order; which CTA, and the order in which
// tiles are visited, change timing only ("Ascend NPU backend", batch-
// invariance bullet). One tile shape per variant, whatever M is: choosing a
// kernel by problem shape is what breaks batch invariance (section "Why").
//
// CTA layout (640 threads, one CTA per SM, persistent over output tiles):
//   warps 0-15 epilogue: warp w reads TMEM lanes 32*(w%4).. (rows) and the
//              column quarter w/4 of the tile; each thread owns one row and
//              BN/4 columns, and keeps the tree's pending partials for them.
//              Four epilogue warps per scheduler hide each other's waits.
//   warps 16-19 stage warps, one per scheduler: warp 16+j owns ring slot j
//              and the K-stages g = j (mod 4) of the CTA's tile sequence. It
//              copies the stage's A and B tiles in with TMA, then issues the
//              stage's MMAs; MMA issue is handed from warp to warp in stage
//              order (turn barriers). Warp 17 also allocates and frees TMEM.
//
// FP32-output tile (128 x 96): the same 640 threads and roles; each
// epilogue thread owns 32 FP32 columns (twelve epilogue warps, 512 threads).
//
// Transposed tile (launches with at most 64 output rows, BF16 out): the
// MMA's A operand is the weight, so its 128 TMEM lanes are 128 output
// columns, and its N side (64) holds the rows. 384 threads: warps 0-7
// epilogue, two per scheduler, each owning one output column per lane and
// 32 rows (a warp whose 32 rows are all past the output's only hands the
// accumulators back); warp 8 copies every stage in with TMA (and, for a
// weight stored [K, N], prefetches the weight tiles of later stages into
// L2), and warps 9-11 issue the MMAs,
// each into its own accumulator and without a turn order. The accumulators
// and all seven pending slots fit in TMEM. With at most 8 (16) output rows
// the epilogue loads, rounds and merges only the 8 (16) columns of each
// leaf that hold rows.
//
// Per tile: 64-wide K stages (two leaves) of the A and B operand tiles go
// through a ring of swizzled shared-memory slots (four; eight in the
// transposed tile). For leaf l the stage
// warp issues two K=16 MMAs into accumulator buffer l % NACC (the first one
// overwrites, so each leaf starts from zero) and commits to that buffer's
// "full" barrier. The epilogue loads the leaf, frees the buffer at once (so
// the MMAs can run NACC-1 leaves ahead), rounds it (bf16 variant) and merges
// it into its pending partials following the block schedule, and writes the
// root after the last leaf.
//
// Pending partials ("slots"): slot s holds the finished left child of a tree
// node of height s + 1, so at most ceil(log2 L) <= 10 are live. Such a node
// spans more than 2^s leaves and nodes of one height are disjoint, so slot s
// is written at most once per 2^s + 1 leaves. The epilogue evaluates the
// tree's maximal subtrees of at most four leaves ("blocks", height <= 2;
// eight leaves and height <= 3 in the transposed tile) entirely in
// registers, so only slots 2 and up ever hold a value: the next slots are
// TMEM columns past the accumulators, then shared memory, and the deepest
// (slots 7-9, touched at most once per 129 leaves) per-CTA global scratch. Global scratch is laid out chunk-major within a warp: the
// k-th 16 bytes of the 32 lanes' values are 512 contiguous bytes, so every
// vector access of a warp covers whole cache lines.
//
// Every mbarrier wait is bounded (Params::timeout_ns of %globaltimer). On
// expiry the waiter records DET_GEMM_ERR_TIMEOUT in the status word and sets
// a CTA-wide abort flag; every role then leaves its loop, outstanding TMA
// loads and MMAs are drained with bounded waits, TMEM is released and the
// CTA exits. The epilogue's per-leaf wait keeps its retry loop inside one
// inline PTX block and records a failure as data: the warp still loads and
// hands back that leaf's accumulator and finishes the tile's blocks on
// whatever the accumulators hold (the values of an aborted launch are never
// used; the accesses stay inside the CTA's TMEM, shared memory and scratch,
// and the FP32 tile's in-place root store inside the output), then leaves
// at the tile's end. Without a branch after every wait, or after every
// block, the compiler schedules one leaf's arithmetic across the next
// leaf's wait (the MLP step 627 -> 645 TFLOP/s, the FP32-output launch
// 437 -> 471).
#pragma once

#include "det_gemm_internal.h"

namespace detg {

constexpr int kStatusTimeout = 6;   // DET_GEMM_ERR_TIMEOUT
constexpr int kPrefetchRounds = 1;  // transposed tile, weight MN-major: L2 prefetch distance, in rounds of the stage ring


// ------------------------------------------------------------------ config

// SWAP: the transposed tile for launches with few output rows (at most
// BN of them). The MMA's 128 lanes then carry 128 output columns and its N
// side the rows, so the epilogue's work follows the rows that exist instead
// of a 128-row tile that is mostly padding. Every output element still comes
// out of the same leaves and the same tree: the tensor core forms the same
// products and FP32 leaf sums whichever operand is A (the bits are checked
// against the plain tile on the GPU).
template <bool F32, bool SWAP = false>
struct Cfg {
    // Epilogue warps and output columns per tile (rows when SWAP). The FP32
    // tile is 96 columns wide with three epilogue warps per scheduler, 32
    // FP32 columns each: the thread that issues an MMA of 128 rows waits
    // about as long for any N up to 256, so a wider tile does more per MMA
    // issued, and 96 columns of FP32 values and pending partials still fit
    // the registers, TMEM and shared memory. (Four warps of 24 columns ran
    // 1-3 % slower once the accumulator wait had no branch after it.)
    static constexpr int EPI_WARPS = SWAP ? 8 : (F32 ? 12 : 16);
    static constexpr int GROUPS = EPI_WARPS / 4;        // epilogue warps per TMEM lane quadrant
    static constexpr int BN = SWAP ? 64 : (F32 ? 96 : 128);
    // TMEM accumulator buffers. The BF16 tile takes three, which leaves
    // TMEM room for two pending-partial slots (with two accumulators and four
    // TMEM slots it ran 5 % slower: the MMAs then run only one leaf ahead).
    // The transposed tile takes three too, one per issuing warp.
    // The FP32 tile takes two: its 96-column slots are 48 KiB each, and with
    // three of them in TMEM a 448-leaf tree parks 12 instead of 24 values
    // per tile in shared memory and 3 instead of 7 in global memory, which
    // made that launch 4 % faster (with four accumulators it was a tenth
    // slower; with three, in the twelve-warp tile, the 448-leaf launch ran
    // 2 % faster and the 128-leaf FP32 LM head 2 % slower).
    static constexpr int NACC = 3 - (F32 ? 1 : 0);
    // Shared-memory ring depth: one slot per stage warp in the plain tiles;
    // eight in the transposed tile, whose single copy warp keeps up to 16
    // leaves of weight in flight (launches of 17 and 64 rows 2 us faster
    // than with four; one row, bound by the epilogue, unchanged).
    static constexpr int STAGES = SWAP ? 8 : kStageWarps;
    static constexpr int A_STAGE = kBM * kBK * 2;       // bytes of one A stage
    // MN-major B tiles are copied in boxes of 64 columns (one 128-byte
    // swizzle span), so a stage holds BN rounded up to 64 columns.
    static constexpr int B_COPY_COLS = (BN + 63) / 64 * 64;
    static constexpr int B_STAGE = B_COPY_COLS * kBK * 2;   // bytes of one B stage
    static constexpr int STAGE_TX = A_STAGE + B_STAGE;  // TMA bytes per stage with full boxes
    static constexpr int COLS = BN / GROUPS;            // accumulator columns per epilogue thread
    static constexpr int WORDS = F32 ? COLS : COLS / 2; // 32-bit words per value per thread (16, or 32 for fp32)
    static constexpr int TMEM_COLS = 512;
    static constexpr int TMEM_SLOT_BASE = NACC * BN;    // after the accumulators
    static constexpr int TMEM_SLOT_STRIDE = WORDS * GROUPS;   // TMEM columns of one slot
    // Leaves per block of the block schedule. The transposed tile merges up
    // to eight leaves in registers (the last leaf of a right half rounded
    // straight into its sibling), so slots 0-2 never leave its registers:
    // with half as many epilogue warps, its per-block overheads weigh more
    // (QKV at one row: 36 -> 33.4 us). The plain tiles keep blocks of four
    // leaves: eight measured 1 % slower on the large launches.
    static constexpr int BLOCK_LEAVES = SWAP ? 8 : 4;
    static constexpr int TMEM_FIRST = BLOCK_LEAVES == 8 ? 3 : 2;   // slots below never leave a block's registers
    static constexpr int TMEM_SLOTS_FIT = (TMEM_COLS - TMEM_SLOT_BASE) / TMEM_SLOT_STRIDE;
    static constexpr int TMEM_SLOTS =
        TMEM_SLOTS_FIT < kMaxSlots - TMEM_FIRST ? TMEM_SLOTS_FIT : kMaxSlots - TMEM_FIRST;
    static constexpr int SMEM_FIRST = TMEM_FIRST + TMEM_SLOTS;
    static constexpr int SMEM_SLOTS = SWAP ? 0 : (F32 ? 2 : 3);
    static constexpr int GLOBAL_FIRST = SMEM_FIRST + SMEM_SLOTS;
    static constexpr int GLOBAL_SLOTS = kMaxSlots - GLOBAL_FIRST;
    static constexpr int LINE = WORDS * 4;              // bytes of one value of one thread
    static constexpr int SLOT_BYTES = EPI_WARPS * 32 * LINE;   // one slot for the whole CTA
    static constexpr int SCRATCH_CTA_BYTES = GLOBAL_SLOTS * SLOT_BYTES;

    // Warp roles: epilogue warps first, then the stage warps.
    static constexpr int FIRST_STAGE_WARP = EPI_WARPS;
    static constexpr int TMEM_WARP = EPI_WARPS + 1;     // allocates and frees TMEM
    static constexpr int THREADS = 32 * (EPI_WARPS + kStageWarps);
    // Registers per thread at launch (the most one CTA of THREADS per SM can
    // have): the plain tile's register split redistributes exactly these,
    // kProdRegs to each stage warp and EPI_REGS to each epilogue warp; the
    // transposed tile needs no split.
    static constexpr int LAUNCH_REGS = SWAP ? 0 : (65536 / THREADS) & ~7;
    static constexpr int EPI_REGS =
        SWAP ? 0 : ((LAUNCH_REGS * THREADS - kProdRegs * 32 * kStageWarps) / (32 * EPI_WARPS)) & ~7;

    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_SLOTS = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_BAR = OFF_SLOTS + SMEM_SLOTS * SLOT_BYTES;
    // barriers: full[STAGES], empty[STAGES], acc_full[NACC], acc_empty[NACC], never,
    // drain[kStageWarps], turn[kStageWarps]
    static constexpr int NUM_BARS = 2 * STAGES + 2 * NACC + 1 + 2 * kStageWarps;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = BYTES + 1024;     // slack to align the base to 1024 B

    static_assert(SWAP ? GLOBAL_SLOTS == 0 : GLOBAL_SLOTS >= 1, "slot storage");
    static_assert(!SWAP || !F32, "the transposed tile has a BF16 output only");
    static_assert(SCRATCH_CTA_BYTES <= kMaxScratchCtaBytes, "scratch");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(A_STAGE % 1024 == 0 && B_STAGE % 1024 == 0, "swizzle atoms");
    static_assert(F32 ? WORDS == 32 : WORDS == 16, "epilogue values are 16 (BF16) or 32 (FP32) words per thread");
    static_assert(EPI_WARPS % 4 == 0, "whole TMEM lane quadrants");
};

// ----------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// mbar_arrive by the lanes for which `pred` holds, without a branch.
__device__ __forceinline__ void mbar_arrive_if(uint32_t bar, bool pred)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar),
                 "r"(static_cast<uint32_t>(pred))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a waiting thread sleeps until the
// phase completes or the hint expires instead of spinning, so it does not
// take issue slots from the warps sharing its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false when the
// CTA is aborting (another waiter gave up) or when this wait exceeds the
// launch's time bound, in which case it records the timeout and starts the
// abort. `honor_abort` = false is used by the drain waits of the teardown.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             int *status, unsigned long long timeout_ns, bool honor_abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (honor_abort && *abort_flag) return false;
        if (global_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            atomicExch(status, kStatusTimeout);
            return false;
        }
    }
}

// Wait for the phase with the given parity with no branch in the calling
// code: the test, and on failure the bounded retry loop (the same bound and
// abort protocol as wait_bounded), are one inline PTX block, so the
// compiler can schedule the caller's independent arithmetic across the
// wait. Returns 1 when the phase completed, 0 when the CTA is aborting or
// the wait timed out (which records the timeout and starts the abort).
__device__ __forceinline__ uint32_t mbar_wait_inline(uint32_t bar, uint32_t parity, uint32_t abort_flag_smem,
                                                     int *status, unsigned long long timeout_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        ".reg .u64 t0, t1;\n\t"
        ".reg .u32 ab;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "@p bra DG_WAIT_DONE;\n\t"
        "mov.u64 t0, %%globaltimer;\n"
        "DG_WAIT_LOOP:\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %6;\n\t"
        "@p bra DG_WAIT_DONE;\n\t"
        "ld.volatile.shared.u32 ab, [%3];\n\t"
        "setp.ne.u32 p, ab, 0;\n\t"
        "@p bra DG_WAIT_FAIL;\n\t"
        "mov.u64 t1, %%globaltimer;\n\t"
        "sub.u64 t1, t1, t0;\n\t"
        "setp.lt.u64 p, t1, %5;\n\t"
        "@p bra DG_WAIT_LOOP;\n\t"
        "st.volatile.shared.u32 [%3], 1;\n\t"
        "atom.exch.b32 ab, [%4], %7;\n"
        "DG_WAIT_FAIL:\n\t"
        "mov.u32 %0, 0;\n\t"
        "bra DG_WAIT_END;\n"
        "DG_WAIT_DONE:\n\t"
        "mov.u32 %0, 1;\n"
        "DG_WAIT_END:\n\t"
        "}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(abort_flag_smem), "l"(status), "l"(timeout_ns), "r"(20000u), "r"(kStatusTimeout)
        : "memory");
    return ok;
}

// The whole warp waits for the phase with the given parity. When it has
// completed already (the common case) this is one test, one vote and one
// uniform branch, with no per-lane branch; otherwise the bounded wait.
// True when every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *status,
                                          unsigned long long timeout_ns)
{
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    return __all_sync(0xFFFFFFFFu, wait_bounded(bar, parity, abort_flag, status, timeout_ns, true));
}

// One lane of the (converged) warp: the one that issues TMA copies, MMAs
// and commits while the whole warp runs the role's control flow.
__device__ __forceinline__ bool elect_one()
{
    uint32_t is_leader;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(is_leader));
    return is_leader != 0;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x,
                                            int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Prefetch of one tile of a tensor map into L2 (no shared memory, no
// completion); same coordinate rules as tma_load_2d.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void tmap_prefetch(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// UMMA shared-memory descriptor, 128-byte swizzle, sm_100 family version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;   // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;   // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: BF16 x BF16 -> FP32, M x N, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int a_major, int b_major)
{
    return (1u << 4)                                   // D format: F32
           | (1u << 7)                                 // A format: BF16
           | (1u << 10)                                // B format: BF16
           | (static_cast<uint32_t>(a_major) << 15)    // A: 0 K-major, 1 MN-major
           | (static_cast<uint32_t>(b_major) << 16)    // B: 0 K-major, 1 MN-major
           | (static_cast<uint32_t>(n >> 3) << 17)
           | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, "
        "%20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%1], {%18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33};"
        ::"r"(taddr), "r"(taddr + 16u),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

__device__ __forceinline__ void reg_fence8(uint32_t (&r)[8])
{
    asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]));
}

__device__ __forceinline__ void reg_fence4(uint32_t (&r)[4])
{
    asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Ties the registers written by tcgen05.ld to a point after tcgen05.wait::ld,
// so no use of them can be scheduled before the wait.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}

// Two FP32 values -> packed BF16 pair, each rounded to nearest even.
// The low half holds `lo` (the lower column), as memory order wants.
__device__ __forceinline__ uint32_t cvt_bf16x2(uint32_t lo, uint32_t hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    return d;
}

// One tree node: left + right, rounded once (BF16 pair, or one FP32 value).
template <bool F32>
__device__ __forceinline__ uint32_t merge(uint32_t left, uint32_t right)
{
    if constexpr (F32) {
        return __float_as_uint(__fadd_rn(__uint_as_float(left), __uint_as_float(right)));
    } else {
        uint32_t d;
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(left), "r"(right));
        return d;
    }
}

// ------------------------------------------------------------- schedule

// Tile t of the persistent walk -> (m tile, n tile). Tiles come in groups
// of `group` panels of the operand that stays in L2 (row panels of A when
// rows_fast, column panels of B otherwise) times every panel of the other
// operand; within a group the resident operand's panel varies fastest, so
// the CTAs running at the same time share the streamed operand's panel and
// each streamed panel is read from DRAM once per group. The host picks the
// order; only timing depends on it.
__device__ __forceinline__ int fdiv(int n, const FastDiv &d)
{
    return static_cast<int>((static_cast<unsigned long long>(static_cast<unsigned int>(n)) * d.mul) >> d.shift);
}

__device__ __forceinline__ void tile_coords(int t, const Problem &pb, int n_tiles, int &mt, int &nt)
{
    const int fast_tiles = pb.rows_fast ? pb.m_tiles : n_tiles;
    const int g = fdiv(t, pb.div_span);
    const int first = g * pb.group;
    const bool last = first + pb.group > fast_tiles;   // the last group may hold fewer panels
    const int gf = last ? fast_tiles - first : pb.group;
    const int r = t - g * pb.span;
    const int o = fdiv(r, last ? pb.div_last : pb.div_group);
    const int f = first + (r - o * gf);
    mt = pb.rows_fast ? f : o;
    nt = pb.rows_fast ? o : f;
}

// The problem (GEMM of a grouped launch) work unit u belongs to.
__device__ __forceinline__ int problem_of(const Params &p, int u)
{
    int pi = 0;
    while (pi + 1 < p.num_problems && u >= p.prob[pi + 1].first_unit) ++pi;
    return pi;
}

// ------------------------------------------------------------- epilogue

// Every epilogue value (a rounded leaf, a partial, the root) holds a
// thread's columns (ValW<W>): 32 columns as 16 words of BF16 pairs, or 32
// FP32 words.
template <int W>
using ValW = uint32_t[W];
using Val = ValW<16>;

// TMEM <-> registers for W (4, 8, 16 or 32) words.
template <int W>
__device__ __forceinline__ void tmem_ld_val(uint32_t taddr, ValW<W> &t)
{
    static_assert(W == 4 || W == 8 || W == 16 || W == 32, "TMEM load width");
    if constexpr (W == 4) tmem_ld4(taddr, t);
    else if constexpr (W == 8) tmem_ld8(taddr, t);
    else if constexpr (W == 16) tmem_ld16(taddr, t);
    else tmem_ld32(taddr, t);
}

template <int W>
__device__ __forceinline__ void tmem_st_val(uint32_t taddr, const ValW<W> &v)
{
    static_assert(W == 4 || W == 8 || W == 16 || W == 32, "TMEM store width");
    if constexpr (W == 4) tmem_st4(taddr, v);
    else if constexpr (W == 8) tmem_st8(taddr, v);
    else if constexpr (W == 16) tmem_st16(taddr, v);
    else tmem_st32(taddr, v);
}

template <int W>
__device__ __forceinline__ void reg_fence_val(ValW<W> &t)
{
    if constexpr (W == 4) reg_fence4(t);
    else if constexpr (W == 8) reg_fence8(t);
    else if constexpr (W == 16) reg_fence16(t);
    else reg_fence(t);
}

// What one epilogue thread needs to reach its storage.
struct EpiCtx {
    uint32_t tmem_slot;   // TMEM address of this thread's first TMEM slot
    uint32_t smem_slot;   // shared-memory address of this thread's line in the first shared slot
    uint8_t *scratch;     // this thread's first 16 bytes in the first global slot (chunk k: +512 k)
    int lane;
    int row, col;         // first output element owned by this thread
    int rows;             // rows of the output (the problem's)
    uint8_t *out;         // matrix the roots go to (the output, or this unit's part slab)
    long long ldo;        // its leading dimension, elements
};

// 16-byte chunk k of a thread's shared-memory line of CHUNKS chunks (4 or
// 8). Lines of consecutive lanes are 16*CHUNKS bytes apart; permuting the
// chunks by lane puts the eight lanes of a quarter-warp access on eight
// distinct bank groups.
template <int CHUNKS>
__device__ __forceinline__ uint32_t smem_chunk(uint32_t line, int lane, int k)
{
    static_assert(CHUNKS == 4 || CHUNKS == 8, "lines of 64 or 128 bytes");
    if constexpr (CHUNKS == 4) return line + static_cast<uint32_t>((k ^ ((lane >> 1) & 3)) * 16);
    else return line + static_cast<uint32_t>((k ^ (lane & 7)) * 16);
}

// Writes this thread's value of the root to the output, clipped to the
// matrix. A row the matrix clips goes element by element through the
// thread's part of the first global slot, which is free once the root is
// formed (every pending partial has been merged into it).
//
// Transposed tile (SWAP): the thread's TMEM lane is output column c.row and
// its 2W values are output rows c.col .. c.col+2W-1 of that column; each goes
// to out[(c.col + j) * ldo + c.row]. The 32 lanes of a warp hold 32
// consecutive columns, so every store of the warp writes 64 contiguous bytes.
template <bool F32, bool SWAP, int W = Cfg<F32, SWAP>::WORDS>
__device__ __forceinline__ void store_out(const ValW<W> &v, const Params &p, const EpiCtx &c)
{
    using C = Cfg<F32, SWAP>;
    constexpr int ES = F32 ? 4 : 2;
    if (c.row >= c.rows) return;
    if constexpr (SWAP) {
        const int nrows = p.cols - c.col;
        uint16_t *dst = reinterpret_cast<uint16_t *>(c.out) + static_cast<long long>(c.col) * c.ldo + c.row;
#pragma unroll
        for (int i = 0; i < W; ++i) {
            if (2 * i < nrows) dst[(2 * i) * c.ldo] = static_cast<uint16_t>(v[i] & 0xFFFFu);
            if (2 * i + 1 < nrows) dst[(2 * i + 1) * c.ldo] = static_cast<uint16_t>(v[i] >> 16);
        }
        return;
    }
    const int ncols = p.cols - c.col;
    if (ncols <= 0) return;
    const bool full = ncols >= C::COLS;
    uint8_t *dst = c.out + (static_cast<long long>(c.row) * c.ldo + c.col) * ES;
    uint8_t *vec = full ? dst : c.scratch;
    const int vstride = full ? 16 : 512;
#pragma unroll
    for (int k = 0; k < W / 4; ++k)
        asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(vec + vstride * k), "r"(v[4 * k]),
                     "r"(v[4 * k + 1]), "r"(v[4 * k + 2]), "r"(v[4 * k + 3])
                     : "memory");
    if (full) return;
#pragma unroll 1
    for (int j = 0; j < ncols; ++j) {
        if constexpr (F32) {
            uint32_t w;
            asm volatile("ld.global.b32 %0, [%1];" : "=r"(w) : "l"(c.scratch + (j >> 2) * 512 + 4 * (j & 3)) : "memory");
            asm volatile("st.global.b32 [%0], %1;" ::"l"(dst + 4 * j), "r"(w) : "memory");
        } else {
            uint16_t w;
            asm volatile("ld.global.u16 %0, [%1];" : "=h"(w) : "l"(c.scratch + (j >> 3) * 512 + 2 * (j & 7)) : "memory");
            asm volatile("st.global.u16 [%0], %1;" ::"l"(dst + 2 * j), "h"(w) : "memory");
        }
    }
}

// Slot s >= 2 (TMEM, shared memory or global scratch) -> t. A narrow value
// (W below the tile's words, transposed tile only) is the first W words of
// the thread's slot columns.
template <bool F32, bool SWAP, int W = Cfg<F32, SWAP>::WORDS>
__device__ __forceinline__ void load_slot(int s, ValW<W> &t, const EpiCtx &c)
{
    using C = Cfg<F32, SWAP>;
    static_assert(W == C::WORDS || C::SMEM_SLOTS + C::GLOBAL_SLOTS == 0, "narrow values live in TMEM only");
    if (C::SMEM_SLOTS + C::GLOBAL_SLOTS == 0 || s < C::SMEM_FIRST) {
        tmem_ld_val<W>(c.tmem_slot + static_cast<uint32_t>((s - C::TMEM_FIRST) * C::TMEM_SLOT_STRIDE), t);
        tmem_wait_ld();
        reg_fence_val<W>(t);
    } else if constexpr (W != C::WORDS) {
    } else if (s < C::GLOBAL_FIRST) {
        const uint32_t line = c.smem_slot + static_cast<uint32_t>((s - C::SMEM_FIRST) * C::SLOT_BYTES);
#pragma unroll
        for (int k = 0; k < W / 4; ++k)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(t[4 * k]), "=r"(t[4 * k + 1]), "=r"(t[4 * k + 2]), "=r"(t[4 * k + 3])
                         : "r"(smem_chunk<W / 4>(line, c.lane, k))
                         : "memory");
    } else {
        const uint8_t *src = c.scratch + (s - C::GLOBAL_FIRST) * C::SLOT_BYTES;
#pragma unroll
        for (int k = 0; k < W / 4; ++k)
            asm volatile("ld.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(t[4 * k]), "=r"(t[4 * k + 1]), "=r"(t[4 * k + 2]), "=r"(t[4 * k + 3])
                         : "l"(src + 512 * k)
                         : "memory");
    }
}

// v -> slot s >= 2 (TMEM, shared memory or global scratch).
template <bool F32, bool SWAP, int W = Cfg<F32, SWAP>::WORDS>
__device__ __forceinline__ void store_slot(int s, const ValW<W> &v, const EpiCtx &c)
{
    using C = Cfg<F32, SWAP>;
    static_assert(W == C::WORDS || C::SMEM_SLOTS + C::GLOBAL_SLOTS == 0, "narrow values live in TMEM only");
    if (C::SMEM_SLOTS + C::GLOBAL_SLOTS == 0 || s < C::SMEM_FIRST) {
        tmem_st_val<W>(c.tmem_slot + static_cast<uint32_t>((s - C::TMEM_FIRST) * C::TMEM_SLOT_STRIDE), v);
        tmem_wait_st();
    } else if constexpr (W != C::WORDS) {
    } else if (s < C::GLOBAL_FIRST) {
        const uint32_t line = c.smem_slot + static_cast<uint32_t>((s - C::SMEM_FIRST) * C::SLOT_BYTES);
#pragma unroll
        for (int k = 0; k < W / 4; ++k)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_chunk<W / 4>(line, c.lane, k)),
                         "r"(v[4 * k]), "r"(v[4 * k + 1]), "r"(v[4 * k + 2]), "r"(v[4 * k + 3])
                         : "memory");
    } else {
        uint8_t *dst = c.scratch + (s - C::GLOBAL_FIRST) * C::SLOT_BYTES;
#pragma unroll
        for (int k = 0; k < W / 4; ++k)
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 512 * k), "r"(v[4 * k]),
                         "r"(v[4 * k + 1]), "r"(v[4 * k + 2]), "r"(v[4 * k + 3])
                         : "memory");
    }
}

// Loads this thread's N accumulator columns (FP32) into r and waits: the
// staging registers of a BF16 leaf (32 columns), or the value itself of an
// FP32 leaf (32 columns).
template <int N>
__device__ __forceinline__ void stage_load(uint32_t acc_taddr, ValW<N> &r)
{
    tmem_ld_val<N>(acc_taddr, r);
    tmem_wait_ld();
    reg_fence_val<N>(r);
}

// A staged leaf's 2W FP32 columns -> F, rounded once to BF16 (RNE), two
// columns per word.
template <int W>
__device__ __forceinline__ void round_leaf(const uint32_t (&stg)[2 * W], ValW<W> &F)
{
#pragma unroll
    for (int i = 0; i < W; ++i) F[i] = cvt_bf16x2(stg[2 * i], stg[2 * i + 1]);
}

// ----------------------------------------------------------------- kernel

// Shared-memory and TMEM addresses of one CTA.
template <bool F32, bool SWAP>
struct Smem {
    uint32_t sA, sB, sSlots, bar0, tmem;
    volatile int *abort_flag;
    __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
    using C = Cfg<F32, SWAP>;
    __device__ uint32_t empty(int s) const { return bar0 + 8u * (C::STAGES + s); }
    __device__ uint32_t accf(int b) const { return bar0 + 8u * (2 * C::STAGES + b); }
    __device__ uint32_t acce(int b) const { return bar0 + 8u * (2 * C::STAGES + C::NACC + b); }
    __device__ uint32_t never() const { return bar0 + 8u * (2 * C::STAGES + 2 * C::NACC); }
    __device__ uint32_t drain(int j) const { return never() + 8u * (1 + j); }
    __device__ uint32_t turn(int j) const { return never() + 8u * (1 + kStageWarps + j); }
};

// Stage warps: kStageWarps warps, one per SM sub-partition. Warp j owns
// ring slot j and the K-stages g with g % kStageWarps == j: it issues the
// stage's TMA copies into its slot, waits for them, then issues the stage's
// MMAs (two K=16 MMAs per leaf into a fresh accumulator) and the commits that
// hand the accumulators to the epilogue and the slot back for the stage
// kStageWarps later. A thread that issues a tcgen05.mma waits for it to be
// taken, about 180 cycles on GB300 whatever N is (up to 256), while the
// tensor core finishes a 128 x 128 x 16 MMA in about 64. With the stages
// rotated over four warps, one warp's waits for data and accumulators
// overlap the others' issue; on GB300 this ran faster than one issuing warp,
// and faster on the large launches than issuing different leaves' MMAs
// from several warps at once (which overlaps the issue waits but slowed the
// epilogue, the tighter bound). The transposed tile, whose epilogue has half
// the work per leaf, issues that way (copy_role and issue_role below): QKV
// at 17 rows 37.5 -> 35.5 us.
//
// MMAs are still issued in leaf order: warp j issues stage g's MMAs only
// after warp j-1 has issued stage g-1's (the turn barriers). The barrier
// waits below test a phase's parity, so only one waiter may be pending per
// barrier phase pair; the turn order guarantees that for the accumulator
// barriers, and slot ownership for the ring barriers. The warp runs the loop
// and the waits; one elected lane issues copies, MMAs and commits.
template <int A_MAJOR, int B_MAJOR, bool F32, bool GROUPED, bool SWAP>
__device__ __forceinline__ void stage_role(const Params &p, const Smem<F32, SWAP> &S, int j)
{
    using C = Cfg<F32, SWAP>;
    static_assert(C::STAGES == kStageWarps, "one ring slot per stage warp");
    constexpr uint32_t IDESC = idesc_bf16(kBM, C::BN, A_MAJOR, B_MAJOR);
    // Byte offset of K step k (16 contraction elements) inside a stage:
    // K-major rows hold the stage's 64 contraction elements (128 B), so a
    // step is 32 B along the row; MN-major tiles hold one 128 B row per
    // contraction index, so a step is 16 rows = 2048 B. Descriptors address
    // in 16-byte units, so offsets are added to the start-address field.
    constexpr uint32_t A_KSTEP = ((A_MAJOR == kKMajor) ? 32u : 2048u) >> 4;
    constexpr uint32_t B_KSTEP = ((B_MAJOR == kKMajor) ? 32u : 2048u) >> 4;
    constexpr uint32_t A_LBO = (A_MAJOR == kKMajor) ? 16u : 8192u;
    constexpr uint32_t B_LBO = (B_MAJOR == kKMajor) ? 16u : 8192u;
    const bool leader = elect_one();
    const int s = j;                                  // this warp's ring slot
    const uint32_t full = S.full(s), empty = S.empty(s);
    const uint32_t my_turn = S.turn(j), next_turn = S.turn((j + 1) % kStageWarps);
    const uint32_t a_dst = S.sA + s * C::A_STAGE;
    const uint32_t b_dst = S.sB + s * C::B_STAGE;
    const uint64_t a_st = sdesc(a_dst, A_LBO, 1024u);
    const uint64_t b_st = sdesc(b_dst, B_LBO, 1024u);
    const int units = p.units;                        // work units: (problem, tile, contraction part)
    const int L = p.num_leaves;                       // leaves per unit
    const int KS = (L + 1) / 2;                       // K-stages per unit
    const int my_units = blockIdx.x < units ? (units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int total = my_units * KS;                  // K-stages of this CTA (< 2^31)
    bool tma_pending = false;     // a load into the slot may be in flight
    uint32_t tma_parity = 0;      // parity of the slot's last load
    bool mma_issued = false;
    bool ok = true;
    if (j == 0 && p.force_timeout) {
        // Test hook: a wait that nothing will end.
        ok = __all_sync(0xFFFFFFFFu, wait_bounded(S.never(), 0, S.abort_flag, p.status, p.timeout_ns, true));
    }
    // Grouped launch: the work unit's problem (a search over the problems),
    // part and tile, kept from its first stage for the rest (this warp takes
    // KS / kStageWarps stages of a unit). The plain launches recompute them
    // per stage, which measured faster for them.
    int cur_tl = -1, pi = 0, g_part = 0, g_mt = 0, g_nt = 0;
    for (int g = j; ok && g < total; g += kStageWarps) {
        const uint32_t round = static_cast<uint32_t>(g / kStageWarps) & 1u;
        const int tl = fdiv(g, p.div_stages);         // unit of this CTA
        const int ks = g - tl * KS;
        int part, mt, nt;
        if constexpr (GROUPED) {
            if (tl != cur_tl) {
                cur_tl = tl;
                const int u = blockIdx.x + tl * gridDim.x;
                pi = problem_of(p, u);
                const int ul = u - p.prob[pi].first_unit;
                const int t = fdiv(ul, p.div_parts);
                g_part = ul - t * p.parts;
                tile_coords(t, p.prob[pi], p.n_tiles, g_mt, g_nt);
            }
            part = g_part;
            mt = g_mt;
            nt = g_nt;
        } else {
            const int u = blockIdx.x + tl * gridDim.x;
            const int ul = u - p.prob[0].first_unit;
            const int t = fdiv(ul, p.div_parts);
            part = ul - t * p.parts;
            tile_coords(t, p.prob[0], p.n_tiles, mt, nt);
        }
        const Problem &pb = p.prob[pi];
        // ---- copy the stage into the slot once the MMAs of its last use are done
        if (!warp_wait(empty, round ^ 1u, S.abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
        }
        if (leader) {
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(pb.stage_tx));
            const int k0 = part * L * kLeaf + ks * kBK, m0 = mt * kBM, n0 = nt * C::BN;
            if constexpr (A_MAJOR == kKMajor) {
                tma_load_2d(a_dst, &pb.tmap_a, full, k0, m0);
            } else {
                tma_load_2d(a_dst, &pb.tmap_a, full, m0, k0);
                tma_load_2d(a_dst + 8192, &pb.tmap_a, full, m0 + 64, k0);
            }
            if constexpr (B_MAJOR == kKMajor) {
                tma_load_2d(b_dst, &pb.tmap_b, full, k0, n0);
            } else {
#pragma unroll
                for (int b = 0; b < C::B_COPY_COLS / 64; ++b)
                    tma_load_2d(b_dst + 8192 * b, &pb.tmap_b, full, n0 + 64 * b, k0);
            }
        }
        __syncwarp();
        tma_pending = true;
        tma_parity = round;
        // ---- wait for the data and for this stage's turn to issue MMAs
        bool got = warp_wait(full, round, S.abort_flag, p.status, p.timeout_ns);
        if (got && g > 0)
            got = warp_wait(my_turn, static_cast<uint32_t>((g - 1) / kStageWarps) & 1u, S.abort_flag, p.status,
                            p.timeout_ns);
        if (!got) {
            ok = false;
            break;
        }
        tma_pending = false;
        tc_fence_after();
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int leaf = 2 * ks + jj;
            if (leaf >= L) break;
            // position of the leaf in this CTA's stream -> accumulator and use
            const int G = tl * L + leaf;
            const int use = G / C::NACC;
            const int acc = G - use * C::NACC;
            if (!warp_wait(S.acce(acc), (static_cast<uint32_t>(use) & 1u) ^ 1u, S.abort_flag, p.status,
                           p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                const uint32_t d = S.tmem + static_cast<uint32_t>(acc * C::BN);
                mma_bf16(d, a_st + (2 * jj) * A_KSTEP, b_st + (2 * jj) * B_KSTEP, IDESC, 0u);   // fresh leaf
                mma_bf16(d, a_st + (2 * jj + 1) * A_KSTEP, b_st + (2 * jj + 1) * B_KSTEP, IDESC, 1u);
                mma_commit(S.accf(acc));
            }
            __syncwarp();
            mma_issued = true;
        }
        if (!ok) break;
        if (leader) {
            mma_commit(empty);
            mbar_arrive(next_turn);
        }
        __syncwarp();
    }
    if (!ok) {
        // Abandoned: let the load this warp issued land and its MMAs finish
        // before the CTA's shared memory and TMEM go away.
        if (tma_pending) wait_bounded(full, tma_parity, S.abort_flag, p.status, p.timeout_ns, false);
        if (mma_issued) {
            if (leader) mma_commit(S.drain(j));
            __syncwarp();
            wait_bounded(S.drain(j), 0, S.abort_flag, p.status, p.timeout_ns, false);
        }
    }
}

// Transposed tile: one copy warp and kSwapIssuers issuing warps. The copy
// warp fills the shared-memory ring stage by stage; issuer i issues the
// MMAs of the leaves G with G % kSwapIssuers == i into its own accumulator
// i, so the issuers' waits for MMA acceptance overlap instead of following
// a turn order. A stage's slot is released by both of its leaves' issuers
// (the empty barrier counts two commits; a stage with a single leaf commits
// twice). Only one thread waits on each accumulator-free barrier (its
// issuer) and the copy warp alone waits on the empty barriers, so no waiter
// can miss a phase.
constexpr int kSwapIssuers = 3;

// Where the K-stages of one work unit come from: its problem, the first
// contraction element of its part, and its tile's first row and column.
struct UnitAt {
    const Problem *pb;
    int k0, m0, n0;
};

template <bool F32, bool GROUPED, bool SWAP>
__device__ __forceinline__ UnitAt unit_at(const Params &p, int tl, int L)
{
    using C = Cfg<F32, SWAP>;
    const int u = blockIdx.x + tl * gridDim.x;
    const Problem &pb = p.prob[GROUPED ? problem_of(p, u) : 0];
    const int ul = u - pb.first_unit;
    const int t = fdiv(ul, p.div_parts);
    const int part = ul - t * p.parts;
    int mt, nt;
    tile_coords(t, pb, p.n_tiles, mt, nt);
    return UnitAt{&pb, part * L * kLeaf, mt * kBM, nt * C::BN};
}

// The copy warp keeps two cursors, the stage it copies and the stage it
// prefetches into L2, and finds a unit's coordinates once per unit: a
// per-stage recomputation (a chain of multiply-shift divisions) made this
// warp the launch's bottleneck, at about 850 cycles per stage.
template <int A_MAJOR, int B_MAJOR, bool F32, bool GROUPED, bool SWAP>
__device__ __forceinline__ void copy_role(const Params &p, const Smem<F32, SWAP> &S)
{
    using C = Cfg<F32, SWAP>;
    const bool leader = elect_one();
    const int units = p.units;
    const int L = p.num_leaves;
    const int KS = (L + 1) / 2;
    const int my_units = blockIdx.x < units ? (units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int total = my_units * KS;
    uint32_t loaded = 0, parity = 0;
    bool ok = true;
    if (p.force_timeout)
        ok = __all_sync(0xFFFFFFFFu, wait_bounded(S.never(), 0, S.abort_flag, p.status, p.timeout_ns, true));
    constexpr int PF = kPrefetchRounds * C::STAGES;   // prefetch distance, stages
    int tl = 0, ks = 0;                                // copy cursor: unit and K-stage
    UnitAt at{};
    if (total > 0) at = unit_at<F32, GROUPED, SWAP>(p, 0, L);
    int tlp = 0, ksp = 0;                              // prefetch cursor, PF stages ahead
    UnitAt atp{};
    if (PF < total) {
        tlp = fdiv(PF, p.div_stages);
        ksp = PF - tlp * KS;
        atp = unit_at<F32, GROUPED, SWAP>(p, tlp, L);
    }
    for (int g = 0; ok && g < total; ++g) {
        const int s = g % C::STAGES;
        const uint32_t round = static_cast<uint32_t>(g / C::STAGES) & 1u;
        if (!warp_wait(S.empty(s), round ^ 1u, S.abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
        const uint32_t full = S.full(s);
        const uint32_t a_dst = S.sA + s * C::A_STAGE;
        const uint32_t b_dst = S.sB + s * C::B_STAGE;
        if (leader) {
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(at.pb->stage_tx));
            const int k0 = at.k0 + ks * kBK;
            if constexpr (A_MAJOR == kKMajor) {
                tma_load_2d(a_dst, &at.pb->tmap_a, full, k0, at.m0);
            } else {
                tma_load_2d(a_dst, &at.pb->tmap_a, full, at.m0, k0);
                tma_load_2d(a_dst + 8192, &at.pb->tmap_a, full, at.m0 + 64, k0);
            }
            if constexpr (B_MAJOR == kKMajor) {
                tma_load_2d(b_dst, &at.pb->tmap_b, full, k0, at.n0);
            } else {
#pragma unroll
                for (int b = 0; b < C::B_COPY_COLS / 64; ++b)
                    tma_load_2d(b_dst + 8192 * b, &at.pb->tmap_b, full, at.n0 + 64 * b, k0);
            }
            // L2 prefetch of the weight PF stages ahead, for a weight stored
            // [K, N] (MN-major A) only: with the weight stored [N, K] the
            // launches ran faster without it (64 rows 35.5 -> 33.6 us), and
            // with it sixteen stages ahead slower still.
            if constexpr (SWAP && A_MAJOR != kKMajor) {
                if (g + PF < total) {
                    const int kp = atp.k0 + ksp * kBK;
                    tma_prefetch_2d(&atp.pb->tmap_a, atp.m0, kp);
                    if (atp.m0 + 64 < atp.pb->rows) tma_prefetch_2d(&atp.pb->tmap_a, atp.m0 + 64, kp);
                }
            }
        }
        __syncwarp();
        loaded |= 1u << s;
        parity = (parity & ~(1u << s)) | (round << s);
        if (++ks == KS) {
            ks = 0;
            if (++tl < my_units) at = unit_at<F32, GROUPED, SWAP>(p, tl, L);
        }
        if (++ksp == KS) {
            ksp = 0;
            if (++tlp < my_units) atp = unit_at<F32, GROUPED, SWAP>(p, tlp, L);
        }
    }
    if (!ok) {
        for (int s = 0; s < C::STAGES; ++s)
            if (loaded & (1u << s))
                wait_bounded(S.full(s), (parity >> s) & 1u, S.abort_flag, p.status, p.timeout_ns, false);
    }
}

template <int A_MAJOR, int B_MAJOR, bool F32, bool GROUPED, bool SWAP>
__device__ __forceinline__ void issue_role(const Params &p, const Smem<F32, SWAP> &S, int i)
{
    using C = Cfg<F32, SWAP>;
    static_assert(C::NACC == kSwapIssuers, "one accumulator per issuer");
    constexpr uint32_t IDESC = idesc_bf16(kBM, C::BN, A_MAJOR, B_MAJOR);
    constexpr uint32_t A_KSTEP = ((A_MAJOR == kKMajor) ? 32u : 2048u) >> 4;
    constexpr uint32_t B_KSTEP = ((B_MAJOR == kKMajor) ? 32u : 2048u) >> 4;
    constexpr uint32_t A_LBO = (A_MAJOR == kKMajor) ? 16u : 8192u;
    constexpr uint32_t B_LBO = (B_MAJOR == kKMajor) ? 16u : 8192u;
    const bool leader = elect_one();
    const uint64_t a_st0 = sdesc(S.sA, A_LBO, 1024u);
    const uint64_t b_st0 = sdesc(S.sB, B_LBO, 1024u);
    const uint32_t d = S.tmem + static_cast<uint32_t>(i * C::BN);
    const uint32_t accf = S.accf(i), acce = S.acce(i);
    const int units = p.units;
    const int L = p.num_leaves;
    const int KS = (L + 1) / 2;
    const int my_units = blockIdx.x < units ? (units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int total = my_units * L;
    uint32_t use = 0;
    bool mma_issued = false, ok = true;
    int tl = i / L, l = i - tl * L;       // position of leaf G = i; advanced by kSwapIssuers
    for (int G = i; G < total; G += kSwapIssuers, ++use) {
        const int g = tl * KS + (l >> 1);
        const int half = l & 1;
        const bool alone = (l + 1 == L) && half == 0;
        const int s = g % C::STAGES;
        if (!warp_wait(acce, (use & 1u) ^ 1u, S.abort_flag, p.status, p.timeout_ns) ||
            !warp_wait(S.full(s), static_cast<uint32_t>(g / C::STAGES) & 1u, S.abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
        }
        tc_fence_after();
        if (leader) {
            const uint64_t a = a_st0 + static_cast<uint64_t>(s * (C::A_STAGE >> 4)) + (2 * half) * A_KSTEP;
            const uint64_t b = b_st0 + static_cast<uint64_t>(s * (C::B_STAGE >> 4)) + (2 * half) * B_KSTEP;
            mma_bf16(d, a, b, IDESC, 0u);
            mma_bf16(d, a + A_KSTEP, b + B_KSTEP, IDESC, 1u);
            mma_commit(accf);
            mma_commit(S.empty(s));
            if (alone) mma_commit(S.empty(s));
        }
        __syncwarp();
        mma_issued = true;
        l += kSwapIssuers;
        while (l >= L) { l -= L; ++tl; }
    }
    if (!ok && mma_issued) {
        if (leader) mma_commit(S.drain(i));
        __syncwarp();
        wait_bounded(S.drain(i), 0, S.abort_flag, p.status, p.timeout_ns, false);
    }
}

// Epilogue warp: leaf rounding and the merge tree for one row and BN/2
// columns of every tile.
//
// The tree is walked block by block (det_gemm_block_schedule): a block's
// two to four leaves are rounded and merged in registers in straight-line
// code, then the block's value is merged with the pending partials its
// entry names and parked (one TMEM or scratch access) or written out as the
// root. The code stays small so that the loop, rare branches included,
// lives in the instruction cache.
//
// W is the number of words a thread loads, rounds, merges and stores per
// value: the tile's WORDS, or, in the transposed tile of a launch with at
// most 2W output rows, only the words that hold rows (8 or 16 columns of
// each leaf instead of 32). The slots keep their layout; a narrow value is
// the first W words of the thread's slot columns.
template <bool F32, bool GROUPED, bool SWAP, int W = Cfg<F32, SWAP>::WORDS>
__device__ __forceinline__ void epilogue_role(const Params &p, const Smem<F32, SWAP> &S, int warp, int lane)
{
    using C = Cfg<F32, SWAP>;
    static_assert(W == C::WORDS || (SWAP && (W == 4 || W == 8)), "value width");
    const int q = warp & 3;               // TMEM lane quadrant (rows 32q .. 32q+31)
    const int cq = warp >> 2;             // column group of the tile (a quarter, or a half when SWAP)
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acc0 = S.tmem + lane_bits + static_cast<uint32_t>(cq * C::COLS);
    EpiCtx c;
    c.tmem_slot = S.tmem + lane_bits + static_cast<uint32_t>(C::TMEM_SLOT_BASE + cq * C::WORDS);
    c.smem_slot = S.sSlots + static_cast<uint32_t>((warp * 32 + lane) * C::LINE);
    c.scratch = static_cast<uint8_t *>(p.scratch) + static_cast<long long>(blockIdx.x) * C::SCRATCH_CTA_BYTES +
                warp * 32 * C::LINE + lane * 16;
    c.lane = lane;
    const int units = p.units;
    const int NB = p.num_blocks;

    ValW<W> A, B, Cc;
    constexpr int SW = F32 ? W : 2 * W;   // staging registers (the FP32 tile loads its leaves into the values)
    uint32_t stg[SW];
    int acc = 0;                          // accumulator of the next leaf
    uint32_t acc_phase = 0;
    bool ok = true;
    const uint32_t abort_s = smem_u32(const_cast<int *>(S.abort_flag));
    // Waits for the next leaf's accumulator, loads it, hands it back to the
    // MMA (which may then fill it with the leaf NACC ahead) and rounds the
    // leaf into dst (an FP32 leaf is loaded into dst as is).
    auto take = [&](ValW<W> &dst) {
        ok &= mbar_wait_inline(S.accf(acc), acc_phase, abort_s, p.status, p.timeout_ns) != 0;
        tc_fence_after();
        if constexpr (F32) stage_load<W>(acc0 + static_cast<uint32_t>(acc * C::BN), dst);
        else stage_load<SW>(acc0 + static_cast<uint32_t>(acc * C::BN), stg);
        tc_fence_before();
        __syncwarp();
        mbar_arrive_if(S.acce(acc), lane == 0);
        if (++acc == C::NACC) {
            acc = 0;
            acc_phase ^= 1u;
        }
        if constexpr (!F32) round_leaf<W>(stg, dst);
    };
    // Waits for the next leaf's accumulator and hands it straight back.
    auto pass = [&]() {
        ok &= mbar_wait_inline(S.accf(acc), acc_phase, abort_s, p.status, p.timeout_ns) != 0;
        __syncwarp();
        mbar_arrive_if(S.acce(acc), lane == 0);
        if (++acc == C::NACC) {
            acc = 0;
            acc_phase ^= 1u;
        }
    };
    // The same for a BF16 leaf that is the right child of dst (eight-leaf
    // blocks): each rounded pair is added to dst as it is formed.
    auto take_into = [&](ValW<W> &dst) {
        ok &= mbar_wait_inline(S.accf(acc), acc_phase, abort_s, p.status, p.timeout_ns) != 0;
        tc_fence_after();
        stage_load<SW>(acc0 + static_cast<uint32_t>(acc * C::BN), stg);
        tc_fence_before();
        __syncwarp();
        mbar_arrive_if(S.acce(acc), lane == 0);
        if (++acc == C::NACC) {
            acc = 0;
            acc_phase ^= 1u;
        }
#pragma unroll
        for (int i = 0; i < SW / 2; ++i) dst[i] = merge<false>(dst[i], cvt_bf16x2(stg[2 * i], stg[2 * i + 1]));
    };
    auto add = [](ValW<W> &left, const ValW<W> &right) {
#pragma unroll
        for (int i = 0; i < W; ++i) left[i] = merge<F32>(left[i], right[i]);
    };

    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const Problem &pb = p.prob[GROUPED ? problem_of(p, u) : 0];
        const int ul = u - pb.first_unit;
        const int t = fdiv(ul, p.div_parts);
        const int part = ul - t * p.parts;
        int mt, nt;
        tile_coords(t, pb, p.n_tiles, mt, nt);
        c.row = mt * kBM + q * 32 + lane;
        c.col = nt * C::BN + cq * C::COLS;
        c.rows = pb.rows;
        if (p.parts > 1) {
            c.out = static_cast<uint8_t *>(p.part_out) + part * p.part_stride * (F32 ? 4 : 2);
            c.ldo = p.part_ld;
        } else {
            c.out = static_cast<uint8_t *>(pb.out);
            c.ldo = pb.ldo;
        }
        if constexpr (SWAP) {
            if (c.col >= p.cols) {
                // The warp's 32 kernel columns are all past the output's
                // rows (a launch of at most 32 rows): it has nothing to
                // round, merge or store and only hands each accumulator
                // back once the MMA has filled it.
                for (int i = 0; ok && i < p.num_leaves; ++i) pass();
                if (!ok) return;
                continue;
            }
        }
        for (int b = 0; b < NB; ++b) {
            const uint32_t e = p.blocks[b];
            if constexpr (C::BLOCK_LEAVES == 4) {
                const int n = static_cast<int>((e >> 10) & 3u) + 1;   // leaves in the block
                // n = 1: A = l0          n = 2: A = l0 + l1
                // n = 3: A = l0 + (l1 + l2)     n = 4: A = (l0 + l1) + (l2 + l3)
                take(A);
                if (n >= 2) take(B);
                if (n == 4) {
                    add(A, B);
                    take(B);
                }
                if (n >= 3) {
                    take(Cc);
                    add(B, Cc);
                }
                if (n >= 2) add(A, B);
            } else {
                // n leaves = a left half of n/2 (rounded down) and a right
                // half of the rest, each of the four-leaf shapes:
                // 1: x0   2: x0 + x1   3: x0 + (x1 + x2)   4: (x0 + x1) + (x2 + x3)
                const int n = static_cast<int>(e & 7u) + 1;
                const int nl = n >> 1, nr = n - nl;
                if (nl > 0) {                    // left half -> A
                    take(A);
                    if (nl >= 2) take(B);
                    if (nl == 4) {
                        add(A, B);
                        take(B);
                    }
                    if (nl >= 3) {
                        take(Cc);
                        add(B, Cc);
                    }
                    if (nl >= 2) add(A, B);
                }
                take(B);                         // right half -> B
                if (nr >= 2) take(Cc);
                if (nr == 4) {
                    add(B, Cc);
                    take(Cc);
                }
                if (nr >= 3) take_into(Cc);
                if (nr >= 2) add(B, Cc);
                if (nl > 0) add(A, B);
                else {
#pragma unroll
                    for (int i = 0; i < W; ++i) A[i] = B[i];
                }
            }
            // merge with the pending left siblings above the block, lowest first
#pragma unroll 1
            for (uint32_t m = (e & 0x3FFu) >> C::TMEM_FIRST; m != 0; m &= m - 1) {
                const int s = C::TMEM_FIRST + __ffs(static_cast<int>(m)) - 1;   // lowest pending slot left
                load_slot<F32, SWAP, W>(s, B, c);   // B is free once the block is merged
#pragma unroll
                for (int i = 0; i < W; ++i) A[i] = merge<F32>(B[i], A[i]);
            }
            const int st = static_cast<int>(e >> 12);
            if constexpr (F32) {
                if (st == kSlotRoot) store_out<F32, SWAP, W>(A, p, c);
                else store_slot<F32, SWAP, W>(st, A, c);
            } else {
                if (st != kSlotRoot) store_slot<F32, SWAP, W>(st, A, c);
            }
        }
        // The schedule's last block, and only it, forms the root. The BF16
        // variants store it after the walk, which keeps that once-per-tile
        // code out of the block loop (2 % faster on their launches); the
        // FP32 variant measured 6 % slower that way and stores it in place.
        if (!ok) return;   // a wait of this tile failed: the launch is aborting
        if constexpr (!F32) store_out<F32, SWAP, W>(A, p, c);
    }
}

template <int A_MAJOR, int B_MAJOR, bool F32, bool GROUPED, bool SWAP>
__global__ void __launch_bounds__(Cfg<F32, SWAP>::THREADS, 1) det_gemm_kernel(const __grid_constant__ Params p)
{
    using C = Cfg<F32, SWAP>;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms need 1024-byte aligned buffers.
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    Smem<F32, SWAP> S;
    S.sA = base + C::OFF_A;
    S.sB = base + C::OFF_B;
    S.sSlots = base + C::OFF_SLOTS;
    S.bar0 = base + C::OFF_BAR;
    uint32_t *tmem_base_smem = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    S.abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    // ---- set-up: barriers, TMEM allocation
    if (threadIdx.x == 0) {
        *S.abort_flag = 0;
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(S.full(s), 1);
            mbar_init(S.empty(s), SWAP ? 2 : 1);
        }
        for (int b = 0; b < C::NACC; ++b) {
            mbar_init(S.accf(b), 1);
            mbar_init(S.acce(b), C::EPI_WARPS);
        }
        mbar_init(S.never(), 1);
        for (int j = 0; j < kStageWarps; ++j) {
            mbar_init(S.drain(j), 1);
            mbar_init(S.turn(j), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == C::FIRST_STAGE_WARP && lane == 0) {
        for (int pi = 0; pi < (GROUPED ? p.num_problems : 1); ++pi) {
            tmap_prefetch(&p.prob[pi].tmap_a);
            tmap_prefetch(&p.prob[pi].tmap_b);
        }
    }
    if (warp == C::TMEM_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_base_smem)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    S.tmem = *tmem_base_smem;

    if constexpr (!SWAP) {
        // Register split: the stage warpgroup gives up registers and the
        // epilogue warpgroups take them (kProdRegs*128 + EPI_REGS*32*EPI_WARPS
        // fits in the LAUNCH_REGS*THREADS the CTA is launched with). Each
        // role's code sits inside its own branch so that the compiler
        // allocates it under the matching limit.
        static_assert(kProdRegs * 32 * kStageWarps + C::EPI_REGS * 32 * C::EPI_WARPS <= C::LAUNCH_REGS * C::THREADS,
                      "register split");
        if (warp < C::EPI_WARPS) {
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::EPI_REGS));
            epilogue_role<F32, GROUPED, SWAP>(p, S, warp, lane);
        } else {
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs));
            stage_role<A_MAJOR, B_MAJOR, F32, GROUPED, SWAP>(p, S, warp - C::FIRST_STAGE_WARP);
        }
    } else {
        // 384 threads: every warp has the registers it needs without a split.
        // The epilogue handles only the columns of each leaf that hold rows
        // when the launch has at most 8 or 16 of them.
        if (warp < C::EPI_WARPS) {
            if (p.cols <= 8) epilogue_role<F32, GROUPED, SWAP, 4>(p, S, warp, lane);
            else if (p.cols <= 16) epilogue_role<F32, GROUPED, SWAP, 8>(p, S, warp, lane);
            else epilogue_role<F32, GROUPED, SWAP>(p, S, warp, lane);
        } else if (warp == C::FIRST_STAGE_WARP) copy_role<A_MAJOR, B_MAJOR, F32, GROUPED, SWAP>(p, S);
        else issue_role<A_MAJOR, B_MAJOR, F32, GROUPED, SWAP>(p, S, warp - C::FIRST_STAGE_WARP - 1);
    }

    // ---- teardown
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::TMEM_WARP) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(S.tmem), "r"(C::TMEM_COLS)
                     : "memory");
    }
}

// --------------------------------------------------------- host launcher

template <int A_MAJOR, int B_MAJOR, bool F32, bool GROUPED = false, bool SWAP = false>
struct Launcher {
    using C = Cfg<F32, SWAP>;
    static cudaError_t prepare(int *num_regs)
    {
        auto fn = det_gemm_kernel<A_MAJOR, B_MAJOR, F32, GROUPED, SWAP>;
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes at;
        e = cudaFuncGetAttributes(&at, fn);
        if (e != cudaSuccess) return e;
        *num_regs = at.numRegs;
        return cudaSuccess;
    }
    static cudaError_t launch(const Params &p, int grid, cudaStream_t stream)
    {
        det_gemm_kernel<A_MAJOR, B_MAJOR, F32, GROUPED, SWAP><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
        return cudaGetLastError();
    }
    static VariantOps ops()
    {
        VariantOps o;
        o.prepare = &prepare;
        o.launch = &launch;
        o.bn = C::BN;
        o.smem_bytes = C::SMEM_BYTES;
        o.scratch_cta_bytes = C::SCRATCH_CTA_BYTES;
        o.split_regs = C::LAUNCH_REGS;
        o.swap = SWAP;
        o.block_leaves = C::BLOCK_LEAVES;
        return o;
    }
};

}  // namespace detg
