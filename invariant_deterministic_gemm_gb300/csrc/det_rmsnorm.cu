// Batch-invariant RMSNorm for sm_103a.
//
// "Comment vaincre le non-déterminisme dans l'inférence des LLM", section
// "RMSNorm": the row reduction is batch-invariant when every row is reduced
// by one core in a fixed order, whatever the number of rows. Here one warp
// owns a row and reduces it in the same order for every launch:
//   ss  = sum of x_j * x_j: 32-element FP32 leaves (the squares of BF16
//         values are exact in FP32, so the fused multiply-add the compiler
//         may form rounds exactly like add after multiply), in ascending j,
//         merged by det_gemm's mid-split tree of FP32 adds;
//   m = ss / D, v = m + eps, s = sqrt(v), r = 1 / s, each rounded once to
//   nearest even (explicit _rn intrinsics, no approximations);
//   y_j = RNE_bf16((x_j * r) * w_j).
// The tree is evaluated bottom-up by the warp's lanes, level by level; it
// is the same tree (the same nodes and operands), so the order of the adds
// within a node never changes.
// Every step is an IEEE round-to-nearest operation in a fixed order, so the
// result is a function of the row alone: identical for every batch size,
// and equal bit for bit to the CPU oracle that spells out the same steps.
#include "det_gemm_internal.h"

#include <cuda_bf16.h>

namespace detg {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_at(const uint16_t *p) { return __uint_as_float(static_cast<uint32_t>(*p) << 16); }

__device__ __forceinline__ uint16_t to_bf16(float f)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Sum of squares of x[k0, k1) in ascending order, from +0.
__device__ __forceinline__ float leaf_squares(const uint16_t *x, int k0, int k1)
{
    float s = 0.0f;
    if (k1 - k0 == kLeaf && (reinterpret_cast<uintptr_t>(x + k0) & 15u) == 0) {
        const uint4 *v = reinterpret_cast<const uint4 *>(x + k0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 c = v[q];
            const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float a = bf16_lo(words[i]), b = bf16_hi(words[i]);
                s = __fadd_rn(s, __fmul_rn(a, a));
                s = __fadd_rn(s, __fmul_rn(b, b));
            }
        }
    } else {
        for (int k = k0; k < k1; ++k) {
            const float a = bf16_at(x + k);
            s = __fadd_rn(s, __fmul_rn(a, a));
        }
    }
    return s;
}

// Node i of depth d of the mid-split tree over leaves [0, L): the path from
// the root follows the bits of i, most significant first (0 = left child).
__device__ __forceinline__ void tree_node(int L, int d, int i, int &lo, int &mid, int &hi)
{
    lo = 0;
    hi = L;
    for (int b = d - 1; b >= 0; --b) {
        const int m = (lo + hi) >> 1;
        if ((i >> b) & 1) lo = m;
        else hi = m;
    }
    mid = (lo + hi) >> 1;
}

__global__ void __launch_bounds__(32 * kRmsWarps) rmsnorm_kernel(const __grid_constant__ RmsParams p)
{
    __shared__ float leaves[kRmsWarps][kMaxLeaves];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRmsWarps + warp;
    if (row >= p.rows) return;
    const uint16_t *x = p.x + static_cast<long long>(row) * p.ldx;
    float *lv = leaves[warp];
    const int L = p.num_leaves;
    // leaves, in parallel
#pragma unroll 4
    for (int l = lane; l < L; l += 32) lv[l] = leaf_squares(x, l * kLeaf, min(l * kLeaf + kLeaf, p.d));
    __syncwarp();
    // The mid-split tree, bottom-up, in place: node (lo, hi) keeps its value
    // in lv[lo]; an internal node adds its children's values, lv[lo] (left)
    // and lv[mid] (right). Nodes of one depth cover disjoint ranges.
    int depth = 0;
    while ((1 << depth) < L) ++depth;
    for (int d = depth - 1; d >= 0; --d) {
        for (int i = lane; i < (1 << d); i += 32) {
            int lo, mid, hi;
            tree_node(L, d, i, lo, mid, hi);
            if (hi - lo >= 2) lv[lo] = __fadd_rn(lv[lo], lv[mid]);
        }
        __syncwarp();
    }
    const float m = __fdiv_rn(lv[0], static_cast<float>(p.d));
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(m, p.eps)));
    // y = RNE_bf16((x * r) * w), four 16-byte chunks per lane at a time
    uint16_t *y = p.y + static_cast<long long>(row) * p.ldy;
    const int dv = p.d / 8 * 8;
    constexpr int U = 4;
    for (int j0 = lane * 8; j0 < dv; j0 += 32 * 8 * U) {
        uint4 xv[U], wv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * 32 * 8;
            if (j < dv) {
                xv[u] = *reinterpret_cast<const uint4 *>(x + j);
                wv[u] = *reinterpret_cast<const uint4 *>(p.w + j);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * 32 * 8;
            if (j >= dv) break;
            const uint32_t xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
            const uint32_t ws[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
            uint32_t out[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float lo = __fmul_rn(__fmul_rn(bf16_lo(xs[k]), r), bf16_lo(ws[k]));
                const float hi = __fmul_rn(__fmul_rn(bf16_hi(xs[k]), r), bf16_hi(ws[k]));
                out[k] = static_cast<uint32_t>(to_bf16(lo)) | (static_cast<uint32_t>(to_bf16(hi)) << 16);
            }
            *reinterpret_cast<uint4 *>(y + j) = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
    for (int j = dv + lane; j < p.d; j += 32)
        y[j] = to_bf16(__fmul_rn(__fmul_rn(bf16_at(x + j), r), bf16_at(p.w + j)));
}

}  // namespace

cudaError_t launch_rmsnorm(const RmsParams &p, cudaStream_t stream)
{
    const long long blocks = (static_cast<long long>(p.rows) + kRmsWarps - 1) / kRmsWarps;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    rmsnorm_kernel<<<static_cast<unsigned>(blocks), 32 * kRmsWarps, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace detg
