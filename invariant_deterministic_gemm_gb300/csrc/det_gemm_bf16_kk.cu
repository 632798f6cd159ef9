// Kernel instance: fwd_rhs_transposed and da (both operands K-major), BF16 out.
#include "det_gemm_kernel.cuh"

namespace detg {
VariantOps ops_bf16_kk() { return Launcher<kKMajor, kKMajor, false>::ops(); }
}  // namespace detg
