// Kernel instance: fwd_fp32 (A K-major, B N-major), FP32 out.
#include "det_gemm_kernel.cuh"

namespace detg {
VariantOps ops_f32_kmn() { return Launcher<kKMajor, kMNMajor, true>::ops(); }
}  // namespace detg
