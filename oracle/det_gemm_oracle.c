/*
 * det_gemm CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the bench
 * may load this code. The GPU library never links, includes or calls it, and
 * it shares no header, table or helper with the GPU path.
 *
 * What it computes (RL-Kernel, "Batch-Invariant Deterministic GEMM (det_gemm)",
 * sections "Guarantees" and "Ascend NPU backend"):
 *
 *   For one output element with contraction pairs (x_k, y_k), k = 0 .. Kc-1:
 *     1. Leaf l covers k in [32 l, min(32 l + 32, Kc)). Its value is the FP32
 *        sum of x_k * y_k taken in ascending k, starting from +0.0f
 *        ("32-element leaves accumulate in FP32 in ascending order").
 *     2. Each leaf is rounded once to BF16, round-to-nearest-even
 *        ("round once to BF16 (round-to-nearest-even)").
 *     3. The rounded leaves over [0, L), L = ceil(Kc / 32), are merged by a
 *        fixed mid-split binary tree of BF16 adds:
 *            T(lo, hi) = leaf[lo]                                if hi - lo == 1
 *                      = bf16_add(T(lo, mid), T(mid, hi))         otherwise,
 *            mid = (lo + hi) >> 1   (left child takes floor(n/2) leaves).
 *        The page names only a "mid-split" tree; the floor split for odd
 *        ranges is this oracle's reading. It makes a contiguous half-K GEMM
 *        one child of the root whenever L is even, which the page states.
 *     4. The FP32-output variant ("forward_fp32 returns FP32", page section
 *        "Dtypes") keeps the same leaves and the same tree, but leaves are not
 *        rounded and the merges are FP32 round-to-nearest-even adds.
 *
 * Pins (tests/test_oracle_pins.py): exact rational rounding for bf16_round and
 * bf16_add; exact double sums within the sequential error bound for leaves;
 * hand-derived single-leaf sums (tests/golden/leaf_order_cases.txt) whose
 * bits differ between the ascending order and a descending or pairwise one;
 * identity / permutation / all-ones / small-integer closed forms for the
 * whole GEMM; the half-K child identity; a hand-built three-leaf example that
 * separates the floor split from the left-to-right chain and from the ceil
 * split; power-of-two trees against plain level-by-level pairwise summation.
 *
 * Build: cc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math -pthread
 * (no FMA contraction, no reassociation; a BF16 x BF16 product is exact in
 * FP32 anyway, so fused and unfused multiply-add agree).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define LEAF 32
#define KC_MAX 32768
#define L_MAX (KC_MAX / LEAF)

/* ---------------------------------------------------------------- BF16 --- */

/* BF16 bits -> FP32: a BF16 value is the top half of an FP32 word. */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * FP32 -> BF16, round to nearest, ties to even (IEEE 754 roundTiesToEven
 * applied to the 16 dropped bits). Adding 0x7FFF plus the kept LSB carries
 * into the kept half exactly when the dropped half is above one half, or is
 * exactly one half and the kept LSB is odd. Overflow carries into the
 * exponent and yields infinity, as IEEE rounding does. NaN stays NaN (quiet).
 */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        if (u & 0x007FFFFFu) return (uint16_t)((u >> 16) | 0x0040u);
        return (uint16_t)(u >> 16);
    }
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/*
 * BF16 + BF16 rounded once to BF16. The FP32 sum is correctly rounded and
 * FP32 carries 24 >= 2*8 + 2 significand bits, so rounding it again to BF16
 * equals rounding the exact sum (Figueroa 1995, double rounding for +).
 */
static uint16_t bf16_add(uint16_t a, uint16_t b)
{
    return f32_to_bf16_rne(bf16_to_f32(a) + bf16_to_f32(b));
}

/* ---------------------------------------------------------------- leaves - */

/* FP32 sum of x_k * y_k over k in [k0, k1), ascending, from +0.0f. */
static float leaf_f32(const uint16_t *x, int64_t sx, const uint16_t *y, int64_t sy,
                      int64_t k0, int64_t k1)
{
    float s = 0.0f;
    for (int64_t k = k0; k < k1; ++k) {
        float p = bf16_to_f32(x[k * sx]) * bf16_to_f32(y[k * sy]);
        s = s + p;
    }
    return s;
}

/* ---------------------------------------------------------------- trees --- */

static float fmaxabs(float m, float v)
{
    float a = fabsf(v);
    return (a > m) ? a : m;
}

/* Mid-split tree of BF16 adds over leaves[lo, hi). Tracks the largest |node|. */
static uint16_t tree_bf16(const uint16_t *leaves, int64_t lo, int64_t hi, float *maxabs)
{
    if (hi - lo == 1) {
        *maxabs = fmaxabs(*maxabs, bf16_to_f32(leaves[lo]));
        return leaves[lo];
    }
    int64_t mid = (lo + hi) >> 1;
    uint16_t left = tree_bf16(leaves, lo, mid, maxabs);
    uint16_t right = tree_bf16(leaves, mid, hi, maxabs);
    uint16_t r = bf16_add(left, right);
    *maxabs = fmaxabs(*maxabs, bf16_to_f32(r));
    return r;
}

/* Mid-split tree of FP32 adds over leaves[lo, hi). */
static float tree_f32(const float *leaves, int64_t lo, int64_t hi, float *maxabs)
{
    if (hi - lo == 1) {
        *maxabs = fmaxabs(*maxabs, leaves[lo]);
        return leaves[lo];
    }
    int64_t mid = (lo + hi) >> 1;
    float left = tree_f32(leaves, lo, mid, maxabs);
    float right = tree_f32(leaves, mid, hi, maxabs);
    float r = left + right;
    *maxabs = fmaxabs(*maxabs, r);
    return r;
}

/* ---------------------------------------------------------------- GEMM ---- */

typedef struct {
    const uint16_t *X; int64_t x_si, x_sk;   /* X[i, k] = X[i*x_si + k*x_sk] */
    const uint16_t *Y; int64_t y_sk, y_sj;   /* Y[k, j] = Y[k*y_sk + j*y_sj] */
    int64_t M, N, Kc;
    int out_fp32;
    void *C; int64_t c_si, c_sj;             /* C[i, j] = C[i*c_si + j*c_sj] */
    float *node_maxabs;                      /* optional [M, N] row-major    */
    int64_t row_begin, row_end;
} job_t;

/* One output element: leaves, then the tree. Kc >= 1. */
static void element(const job_t *jb, int64_t i, int64_t j)
{
    uint16_t leaves_bf16[L_MAX];
    float leaves_f32[L_MAX];
    const int64_t L = (jb->Kc + LEAF - 1) / LEAF;
    const uint16_t *x = jb->X + i * jb->x_si;
    const uint16_t *y = jb->Y + j * jb->y_sj;
    float maxabs = 0.0f;

    for (int64_t l = 0; l < L; ++l) {
        int64_t k0 = l * LEAF;
        int64_t k1 = (k0 + LEAF < jb->Kc) ? k0 + LEAF : jb->Kc;
        float s = leaf_f32(x, jb->x_sk, y, jb->y_sk, k0, k1);
        leaves_f32[l] = s;
        leaves_bf16[l] = f32_to_bf16_rne(s);
    }
    if (jb->out_fp32) {
        float r = tree_f32(leaves_f32, 0, L, &maxabs);
        ((float *)jb->C)[i * jb->c_si + j * jb->c_sj] = r;
    } else {
        uint16_t r = tree_bf16(leaves_bf16, 0, L, &maxabs);
        ((uint16_t *)jb->C)[i * jb->c_si + j * jb->c_sj] = r;
    }
    if (jb->node_maxabs) jb->node_maxabs[i * jb->N + j] = maxabs;
}

static void *run_rows(void *arg)
{
    const job_t *jb = (const job_t *)arg;
    for (int64_t i = jb->row_begin; i < jb->row_end; ++i)
        for (int64_t j = 0; j < jb->N; ++j)
            element(jb, i, j);
    return NULL;
}

/*
 * C[i, j] = det_gemm over k of X[i, k] * Y[k, j], for i < M, j < N.
 * Strides are in elements and may be anything (that is how the forward,
 * rhs-transposed, dA, dB and dB-transposed launches are expressed).
 * Kc == 0 writes +0. Returns 0, or -1 on bad arguments. Rows are split over
 * nthreads POSIX threads; rows are independent, so the split changes nothing.
 */
int oracle_det_gemm(const uint16_t *X, int64_t x_si, int64_t x_sk,
                    const uint16_t *Y, int64_t y_sk, int64_t y_sj,
                    int64_t M, int64_t N, int64_t Kc,
                    int out_fp32, void *C, int64_t c_si, int64_t c_sj,
                    float *node_maxabs, int nthreads)
{
    if (M < 0 || N < 0 || Kc < 0 || Kc > KC_MAX) return -1;
    if (M == 0 || N == 0) return 0;
    if (Kc == 0) {
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j) {
                if (out_fp32) ((float *)C)[i * c_si + j * c_sj] = 0.0f;
                else ((uint16_t *)C)[i * c_si + j * c_sj] = 0;
                if (node_maxabs) node_maxabs[i * N + j] = 0.0f;
            }
        return 0;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)M;
    if (nthreads > 256) nthreads = 256;

    job_t jobs[256];
    pthread_t tids[256];
    for (int t = 0; t < nthreads; ++t) {
        job_t jb = {X, x_si, x_sk, Y, y_sk, y_sj, M, N, Kc, out_fp32, C, c_si, c_sj,
                    node_maxabs, M * t / nthreads, M * (t + 1) / nthreads};
        jobs[t] = jb;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, run_rows, &jobs[t]) != 0) break;
        started = t;
    }
    run_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) run_rows(&jobs[t]); /* fallback */
    return 0;
}

/* ------------------------------------------------- pieces, for the tests -- */

/* The FP32 leaves of one element (i, j); out has ceil(Kc/32) entries. */
int oracle_leaves_f32(const uint16_t *X, int64_t x_si, int64_t x_sk,
                      const uint16_t *Y, int64_t y_sk, int64_t y_sj,
                      int64_t i, int64_t j, int64_t Kc, float *out)
{
    if (Kc < 1 || Kc > KC_MAX) return -1;
    const int64_t L = (Kc + LEAF - 1) / LEAF;
    for (int64_t l = 0; l < L; ++l) {
        int64_t k0 = l * LEAF;
        int64_t k1 = (k0 + LEAF < Kc) ? k0 + LEAF : Kc;
        out[l] = leaf_f32(X + i * x_si, x_sk, Y + j * y_sj, y_sk, k0, k1);
    }
    return 0;
}

/* The mid-split BF16 tree over n given (already rounded) leaves. */
uint16_t oracle_tree_bf16(const uint16_t *leaves, int64_t n)
{
    float m = 0.0f;
    return (n < 1) ? (uint16_t)0 : tree_bf16(leaves, 0, n, &m);
}

/* The mid-split FP32 tree over n given leaves. */
float oracle_tree_f32(const float *leaves, int64_t n)
{
    float m = 0.0f;
    return (n < 1) ? 0.0f : tree_f32(leaves, 0, n, &m);
}

void oracle_round_bf16(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t t = 0; t < n; ++t) out[t] = f32_to_bf16_rne(in[t]);
}

void oracle_add_bf16(const uint16_t *a, const uint16_t *b, uint16_t *out, int64_t n)
{
    for (int64_t t = 0; t < n; ++t) out[t] = bf16_add(a[t], b[t]);
}

/* ------------------------------------------------------------- RMSNorm ---- */

/*
 * Batch-invariant RMSNorm, one row at a time ("Comment vaincre le
 * non-déterminisme dans l'inférence des LLM", section "RMSNorm": each row is
 * handled by one core, a data-parallel strategy, so the reduction order never
 * depends on the batch). The page fixes the strategy, not the arithmetic;
 * this oracle's reading, every step rounded once to nearest even:
 *   ss  = sum of x_j * x_j over j in [0, D), reduced like det_gemm's FP32
 *         variant: FP32 leaves of 32 consecutive squares in ascending j
 *         (each square of a BF16 value is exact in FP32), merged by the
 *         mid-split tree of FP32 adds;
 *   m   = ss / D,   v = m + eps,   s = sqrt(v),   r = 1 / s   (FP32);
 *   y_j = RNE_bf16((x_j * r) * w_j)   (two FP32 products, then BF16).
 * Returns 0, or -1 on bad arguments.
 */
int oracle_rmsnorm(const uint16_t *x, int64_t ldx, const uint16_t *w, int64_t M, int64_t D, float eps,
                   uint16_t *y, int64_t ldy)
{
    if (M < 0 || D < 1 || D > KC_MAX || ldx < D || ldy < D) return -1;
    const int64_t L = (D + LEAF - 1) / LEAF;
    float *leaves = (float *)malloc(sizeof(float) * (size_t)L);
    if (!leaves) return -1;
    for (int64_t i = 0; i < M; ++i) {
        const uint16_t *xr = x + i * ldx;
        for (int64_t l = 0; l < L; ++l) {
            int64_t k0 = l * LEAF;
            int64_t k1 = (k0 + LEAF < D) ? k0 + LEAF : D;
            leaves[l] = leaf_f32(xr, 1, xr, 1, k0, k1);
        }
        float mx = 0.0f;
        const float ss = tree_f32(leaves, 0, L, &mx);
        const float m = ss / (float)D;
        const float v = m + eps;
        const float sq = sqrtf(v);
        const float r = 1.0f / sq;
        for (int64_t j = 0; j < D; ++j) {
            const float t = bf16_to_f32(xr[j]) * r;
            const float u = t * bf16_to_f32(w[j]);
            y[i * ldy + j] = f32_to_bf16_rne(u);
        }
    }
    free(leaves);
    return 0;
}

/* ----------------------------------------------------- row reduction ------ */

/*
 * rowdot[i] = sum over n of C[i, n] * D[i, n] in FP32, in the fixed order of
 * the grouped-GEMM epilogue (Megatron Core notes, "Kernel redesign: the
 * grouped-GEMM epilogue": each N-tile writes its own private slot, and the
 * slots are combined by a fixed reduction tree instead of atomic adds
 * across N-tiles). Reading: an N-tile is 128 columns (the GEMM's fixed
 * output tile width); its slot holds the FP32 sum of its products (exact:
 * BF16 x BF16) in ascending column order from +0, the same running sum a
 * leaf uses; rowdot is the mid-split tree of FP32 adds over the slots (the
 * contraction's tree, with slots for leaves).
 */
int oracle_rowdot(const uint16_t *C, int64_t ldc, const uint16_t *D, int64_t ldd, int64_t M, int64_t N,
                  float *out)
{
    if (M < 0 || N < 1 || ldc < N || ldd < N) return -1;
    const int64_t T = (N + 127) / 128;
    float *tiles = (float *)malloc(sizeof(float) * (size_t)T);
    if (!tiles) return -1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t t = 0; t < T; ++t) {
            const int64_t c0 = 128 * t;
            const int64_t c1 = (c0 + 128 < N) ? c0 + 128 : N;
            tiles[t] = leaf_f32(C + i * ldc, 1, D + i * ldd, 1, c0, c1);
        }
        float mx = 0.0f;
        out[i] = tree_f32(tiles, 0, T, &mx);
    }
    free(tiles);
    return 0;
}
