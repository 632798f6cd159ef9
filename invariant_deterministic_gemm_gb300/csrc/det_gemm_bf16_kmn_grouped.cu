// Kernel instance: fwd_grouped (A K-major, B N-major, several problems per
// launch, optional row reduction), BF16 out.
#include "det_gemm_kernel.cuh"

namespace detg {
VariantOps ops_bf16_kmn_grouped() { return Launcher<kKMajor, kMNMajor, false, true>::ops(); }
}  // namespace detg
