// det_gemm_fwd_noalloc: the forward product for callers that cannot
// allocate device memory.
//
// det_gemm_fwd keeps the tree's most rarely touched pending partials in a
// scratch buffer that it allocates with cudaMalloc the first time it runs on
// a stream. Some callers cannot let a library do that: serving and
// real-time paths that own every byte of device memory through their own
// arena and must never trigger the device-wide synchronisation an
// allocation can imply, and callers that run with the device memory they
// were given and nothing more. This entry point
// runs the same kernel with its scratch in a fixed array that is part of the
// library's device image instead.
#include "det_gemm.h"
#include "det_gemm_internal.h"

#include <mutex>

namespace {

// One CTA needs 3 x 32 KiB of scratch (its three least used pending-partial
// slots). 160 CTAs -- one per SM on a GPU of up to 160 SMs -- therefore need
// 15 MiB. Every GPU that loads this library holds this array until the
// process exits.
constexpr size_t kNoAllocScratchBytes = size_t{160} * 3 * 32768;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_done[kMaxDevices] = {};
void *g_addr[kMaxDevices] = {};
int g_setup_status[kMaxDevices] = {};

// Set-up, once per device, with that device current: the library's state
// and the kernel attributes of both kernels a forward launch can take, then
// the device address of g_noalloc_scratch (in host code the array's name is
// only a host-side handle; the address the kernel must be given is looked
// up here), so that no later call does any set-up work.
int setup(int dev, void **scratch)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_done[dev]) {
        g_done[dev] = true;
        g_setup_status[dev] = detg::prepare_forward_status();
        void *ptr = nullptr;
        if (g_setup_status[dev] == DET_GEMM_OK) {
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
                cudaGetLastError();
                detg::record_detail("cudaGetSymbolAddress failed for the no-alloc scratch array");
                g_setup_status[dev] = DET_GEMM_ERR_LAUNCH;
            } else {
                g_addr[dev] = ptr;
            }
        }
    }
    *scratch = g_addr[dev];
    return g_setup_status[dev];
}

}  // namespace

extern "C" det_gemm_status det_gemm_fwd_noalloc(const det_gemm_bf16 *A, const det_gemm_bf16 *B,
                                                det_gemm_bf16 *C, int64_t M, int64_t N, int64_t K, int64_t lda,
                                                int64_t ldb, int64_t ldc, det_gemm_stream stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return DET_GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    void *scratch = nullptr;
    const int st = setup(dev, &scratch);
    if (st != DET_GEMM_OK) return static_cast<det_gemm_status>(st);
    return static_cast<det_gemm_status>(detg::fwd_with_fixed_scratch_status(
        A, B, C, M, N, K, lda, ldb, ldc, reinterpret_cast<cudaStream_t>(stream), scratch, kNoAllocScratchBytes));
}
