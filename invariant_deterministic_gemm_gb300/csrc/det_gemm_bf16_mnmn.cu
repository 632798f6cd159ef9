// Kernel instance: db and db_transposed (both operands MN-major), BF16 out.
#include "det_gemm_kernel.cuh"

namespace detg {
VariantOps ops_bf16_mnmn() { return Launcher<kMNMajor, kMNMajor, false>::ops(); }
}  // namespace detg
