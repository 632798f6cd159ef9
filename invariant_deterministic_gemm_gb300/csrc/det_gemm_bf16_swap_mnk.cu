// Kernel instance: det_gemm_fwd with few output rows, transposed tile. The
// MMA's A operand is the weight B[K,N] (N contiguous: MN-major), its B
// operand the activations A[M,K] (K-major).
#include "det_gemm_kernel.cuh"

namespace detg {
VariantOps ops_bf16_swap_mnk() { return Launcher<kMNMajor, kKMajor, false, false, true>::ops(); }
}  // namespace detg
