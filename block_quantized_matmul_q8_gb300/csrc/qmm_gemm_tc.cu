// qmm_gemm_tc.cu -- tensor-core GEMM (placeholder until the tcgen05 kernel lands).
#include <cuda_runtime.h>

#include "qmm_internal.h"

namespace qmm {

int64_t gemm_tc_tile_m(int64_t m) { return m <= 64 ? 64 : 128; }
size_t gemm_tc_workspace_bytes(qmm_type, int64_t, int64_t, int64_t) { return 0; }
bool gemm_tc_supported(qmm_type, int64_t, int64_t, int64_t) { return false; }
cudaError_t launch_gemm_tc(qmm_type, const void *, int64_t, int64_t, const void *, int64_t, float *, void *, size_t,
                           int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace qmm
