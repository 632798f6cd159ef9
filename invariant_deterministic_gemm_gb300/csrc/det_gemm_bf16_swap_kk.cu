// Kernel instance: det_gemm_fwd_rhs_transposed and det_gemm_da with few
// output rows, transposed tile: both MMA operands K-major.
#include "det_gemm_kernel.cuh"

namespace detg {
VariantOps ops_bf16_swap_kk() { return Launcher<kKMajor, kKMajor, false, false, true>::ops(); }
}  // namespace detg
