// qmm_quantize.cu -- fp32 activations -> q8_1 blocks.
//
// One warp per 32-value block, lane i owns value i ([MMQ] section "引言": the
// activations are compressed to q8_1 on the device; the d/s pair is the one the
// dp4a fold of section "dp4a 路径的 Q4_K" consumes).  Per block:
//   amax = max |x|            (warp max, exact in any order)
//   d    = amax / 127         (IEEE fp32 division, __fdiv_rn)
//   q    = roundf(x / d)      (IEEE fp32 division, halves away from zero)
//   d_h  = fp16_rne(d),  s_h = fp16_rne(float(d_h) * sum(q))   (the product is exact)
// A block whose fp32 d is 0 is stored as all zero.  Bit-identical to the definition;
// the arithmetic is the q8_1_* helpers, which the fused GEMV staging uses as well.
#include <cuda_runtime.h>

#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_tc_ptx.cuh"

namespace qmm {

__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float *__restrict__ x, int64_t m, int64_t k,
                                                            uint8_t *__restrict__ xq) {
    // x may be written by the preceding kernel and xq read by it: wait for it first.
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nb = k / 32;
    const int64_t nblocks = m * nb;
    const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t blk = warp0; blk < nblocks; blk += nwarps) {
        const int64_t r = blk / nb, b = blk - r * nb;
        const float v = x[r * k + 32 * b + lane];
        float amax = fabsf(v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float d = q8_1_scale(amax);
        const int q = q8_1_code_fast(v, d, q8_1_recip(d));
        const int S = __reduce_add_sync(0xffffffffu, q);
        uint8_t *ob = xq + blk * kQ81Bytes;
        ob[4 + lane] = (uint8_t)(int8_t)q;
        if (lane == 0) *reinterpret_cast<uint32_t *>(ob) = q8_1_ds_word(d, S);
    }
}

cudaError_t launch_quantize_q8_1(const float *x, int64_t m, int64_t k, void *xq, cudaStream_t st) {
    const int64_t nblocks = m * (k / 32);
    if (nblocks == 0) return cudaSuccess;
    const int threads = 256;
    int64_t grid = (nblocks + 7) / 8;  // 8 warps per CTA
    const int64_t cap = int64_t(device_sm_count()) * 16;
    if (grid > cap) grid = cap;
    return launch_pdl(quantize_q8_1_kernel, dim3((unsigned)grid), dim3(threads), 0, st, x, m, k,
                      static_cast<uint8_t *>(xq));
}

}  // namespace qmm
