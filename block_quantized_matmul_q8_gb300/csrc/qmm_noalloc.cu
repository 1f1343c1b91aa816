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
// process.  Its device address is looked up with cudaGetSymbolAddress, with the
// device current, on the first call made in each (device, CUDA context) pair: after
// cudaDeviceReset, or from a context other than the device's primary one, the next
// call looks the address up again.  Make the first call on a device before any stream
// capture.  Every call on a device uses the same array and leaves its contents
// behind; the kernels rewrite every part they read (the bucketing kernel writes the
// counts, bounds, pair list and tile list before anything reads them), so no clearing
// is needed, but two calls whose work overlaps on the GPU (different streams, no
// ordering between them) race on the array.
#include <cuda.h>
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

// The current context, through the driver entry point the runtime exposes (no link
// against the driver library); nullptr if it cannot be had.
CUcontext current_context() {
    using Fn = CUresult (*)(CUcontext *);
    static Fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<Fn>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

constexpr int kMaxDev = 64;
std::mutex g_mu;
void *g_ptr[kMaxDev] = {};
CUcontext g_ctx[kMaxDev] = {};

// Device address of the scratch array in the current device and context (nullptr on
// failure), looked up once per (device, context).
void *scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    // cudaFree(0) makes the runtime bind the device's context, so that the driver sees
    // the context the kernels will run in
    if (cudaFree(nullptr) != cudaSuccess) return nullptr;
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ptr[dev] || ctx == nullptr || g_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_ptr[dev] = p;
        g_ctx[dev] = ctx;
    }
    return g_ptr[dev];
}

}  // namespace
}  // namespace qmm

using namespace qmm;

extern "C" size_t qmm_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

// The workspace variant hands Q4_K problems to the tensor-core grouped GEMM, whose
// scratch (an fp16 copy of the gathered activations) grows with the problem; this
// entry point keeps to the paths whose scratch is small: at decode sizes one GEMV per
// (token, slot) pair, which needs only the status word, and otherwise the CUDA-core
// grouped GEMM, whose scratch is only the bucketing state.
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
    const int64_t n_pairs = n_tokens * top_k;
    if (n_pairs <= kMoeGemvMaxPairs && gemv_id_supported(t, n, k)) {
        int32_t *status = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + kStatusOffset);
        return launch_gemv_id(t, W_experts, n_experts, n, k, xq, top_k, ids, n_pairs, y, status, st) == cudaSuccess
                   ? QMM_OK
                   : QMM_ERR_CUDA;
    }
    return launch_mul_mat_id_dp4a(t, W_experts, n_experts, n, k, xq, ids, top_k, n_tokens, false, y, ws,
                                  kNoAllocScratchBytes, st) == cudaSuccess
               ? QMM_OK
               : QMM_ERR_CUDA;
}
