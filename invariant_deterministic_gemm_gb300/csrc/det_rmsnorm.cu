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

__global__ void __launch_bounds__(32 * kRmsWarps) rmsnorm_kernel(const __grid_constant__ RmsParams p)
{
    __shared__ float leaves[kRmsWarps][kMaxLeaves];
    __shared__ float slots[kRmsWarps][kMaxSlots];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRmsWarps + warp;
    if (row >= p.rows) return;
    const uint16_t *x = p.x + static_cast<long long>(row) * p.ldx;
    float *lv = leaves[warp];
    // leaves, in parallel
    for (int l = lane; l < p.num_leaves; l += 32) {
        const int k0 = l * kLeaf;
        const int k1 = min(k0 + kLeaf, p.d);
        lv[l] = leaf_squares(x, k0, k1);
    }
    __syncwarp();
    // the mid-split tree, walked leaf by leaf (pending left children in slots)
    float r = 0.0f;
    if (lane == 0) {
        float* st = slots[warp];
        float root = 0.0f;
        for (int l = 0; l < p.num_leaves; ++l) {
            const uint32_t e = p.sched[l];
            float v = lv[l];
            for (uint32_t m = e & 0x3FFu, s = 0; m != 0; m >>= 1, ++s)
                if (m & 1u) v = __fadd_rn(st[s], v);
            const uint32_t dst = e >> 12;
            if (dst == kSlotRoot) root = v;
            else st[dst] = v;
        }
        const float m = __fdiv_rn(root, static_cast<float>(p.d));
        const float sq = __fsqrt_rn(__fadd_rn(m, p.eps));
        r = __fdiv_rn(1.0f, sq);
    }
    r = __shfl_sync(0xFFFFFFFFu, r, 0);
    // y = RNE_bf16((x * r) * w)
    uint16_t *y = p.y + static_cast<long long>(row) * p.ldy;
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
                       reinterpret_cast<uintptr_t>(p.w)) & 15u) == 0;
    const int dv = vec ? p.d / 8 * 8 : 0;
    for (int j = lane * 8; j < dv; j += 32 * 8) {
        const uint4 xv = *reinterpret_cast<const uint4 *>(x + j);
        const uint4 wv = *reinterpret_cast<const uint4 *>(p.w + j);
        const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, ws[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = __fmul_rn(__fmul_rn(bf16_lo(xs[i]), r), bf16_lo(ws[i]));
            const float hi = __fmul_rn(__fmul_rn(bf16_hi(xs[i]), r), bf16_hi(ws[i]));
            out[i] = static_cast<uint32_t>(to_bf16(lo)) | (static_cast<uint32_t>(to_bf16(hi)) << 16);
        }
        *reinterpret_cast<uint4 *>(y + j) = make_uint4(out[0], out[1], out[2], out[3]);
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
