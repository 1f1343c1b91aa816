// qmm_noalloc.cu -- qmm_mul_mat_id without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// expert-routed matmul: code that runs under an allocator it does not own (an
// inference engine whose memory pool is fixed up front, a plugin that may not
// call cudaMalloc, a runtime that forbids allocation between graph captures).
// This entry point gives them qmm_mul_mat_id with its scratch (status word,
// expert bounds, sorted pair list, tile list) in one file-scope device array of a
// fixed size, so the call itself allocates nothing.
//
// The array lives in every GPU that loads this library, for the life of the
// process.  Its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on that
// device; make that first call before any stream capture.  Every call on a device
// uses the same array and leaves its contents behind; the kernels rewrite every
// part they read, so no clearing is needed, but two calls whose work overlaps on
// the GPU (different streams, no ordering between them) race on the array.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "qmm.h"
#include "qmm_internal.h"
#include "qmm_moe.h"

namespace qmm {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void *g_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device (nullptr on failure).
void *scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_ptr[dev] = p;
    }
    return g_ptr[dev];
}

}  // namespace
}  // namespace qmm

using namespace qmm;

extern "C" size_t qmm_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

// The workspace variant hands Q4_K problems to the tensor-core grouped GEMM, whose
// scratch (an fp16 copy of the gathered activations) grows with the problem; this
// entry point keeps to the CUDA-core grouped GEMM, whose scratch is only the
// bucketing state, so that the fixed array stays small.
extern "C" qmm_status qmm_mul_mat_id_noalloc(const void *W_experts, qmm_type t, int64_t n_experts, int64_t n,
                                             int64_t k, const void *xq, const int32_t *ids, int64_t top_k,
                                             int64_t n_tokens, float *y, void *stream) {
    qmm_status s = moe_check_sizes(t, n_experts, n, k, top_k, n_tokens);
    if (s != QMM_OK) return s;
    const size_t need = moe_dp4a_workspace_bytes(n_tokens, n_experts, top_k);
    if (need > kNoAllocScratchBytes) return QMM_ERR_WORKSPACE;  // problem needs more than the fixed scratch
    void *ws = scratch_ptr();
    if (!ws) return QMM_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n == 0 || n_tokens == 0) return cudaMemsetAsync(ws, 0, 16, st) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
    s = moe_check_pointers(W_experts, xq, ids, y);
    if (s != QMM_OK) return s;
    return launch_mul_mat_id_dp4a(t, W_experts, n_experts, n, k, xq, ids, top_k, n_tokens, false, y, ws,
                                  kNoAllocScratchBytes, st) == cudaSuccess
               ? QMM_OK
               : QMM_ERR_CUDA;
}
