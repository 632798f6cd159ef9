// Kernel instance: fwd (A K-major, B N-major), BF16 out.
#include "det_gemm_kernel.cuh"

namespace detg {
VariantOps ops_bf16_kmn() { return Launcher<kKMajor, kMNMajor, false>::ops(); }
}  // namespace detg
