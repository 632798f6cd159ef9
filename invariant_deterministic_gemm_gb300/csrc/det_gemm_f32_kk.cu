// Kernel instance: fwd_fp32 with a [N,K] weight (both K-major), FP32 out.
#include "det_gemm_kernel.cuh"

namespace detg {
VariantOps ops_f32_kk() { return Launcher<kKMajor, kKMajor, true>::ops(); }
}  // namespace detg
