// qmm_quantize.cu -- fp32 activations -> q8_1 blocks.
//
// One warp per 32-value block, or (for many blocks) four lanes per block with 8 values each,
// so that a warp takes 8 consecutive blocks (1 KB of x) per step ([MMQ] section "引言": the activations are compressed to q8_1 on the device; the
// d/s pair is the one the dp4a fold of section "dp4a 路径的 Q4_K" consumes).  Per block:
//   amax = max |x|            (exact in any order)
//   d    = amax / 127         (IEEE fp32 division, __fdiv_rn)
//   q    = roundf(x / d)      (the integer of the IEEE quotient, halves away from zero)
//   d_h  = fp16_rne(d),  s_h = fp16_rne(float(d_h) * sum(q))   (the product is exact)
// A block whose fp32 d is 0 is stored as all zero.  Bit-identical to the definition; the
// arithmetic is the q8_1_* helpers (the codes through q8_1_code_rcp), which the fused GEMV
// staging uses as well.
#include <cuda_runtime.h>

#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_tc_ptx.cuh"

namespace qmm {

// One warp per block (a value per lane) while there are few blocks: the launch is then a
// single pass whose time is one lane's latency.  From kWideBlocks blocks on, 4 lanes per block
// with 8 values each: an eighth of the instructions per value (m = 512, k = 4096: 11.4 ->
// 3.8 us; m = 4 at k = 5120: 1.7 against 2.3 us the wide way).
constexpr int64_t kWideBlocks = 2048;

template <bool kWide>
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
    if constexpr (!kWide) {
        for (int64_t blk = warp0; blk < nblocks; blk += nwarps) {
            const int64_t r = blk / nb, b = blk - r * nb;
            const float v = x[r * k + 32 * b + lane];
            float amax = fabsf(v);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float d = q8_1_scale(amax);
            const int q = q8_1_code_rcp(v, d, rcp_guarded(d));
            const int S = __reduce_add_sync(0xffffffffu, q);
            uint8_t *ob = xq + blk * kQ81Bytes;
            ob[4 + lane] = (uint8_t)(int8_t)q;
            if (lane == 0) *reinterpret_cast<uint32_t *>(ob) = q8_1_ds_word(d, S);
        }
        return;
    }
    const int g = lane >> 2, l4 = lane & 3;
    for (int64_t base = 8 * warp0; base < nblocks; base += 8 * nwarps) {  // warp-uniform
        const int64_t blk = base + g;
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), b4 = a4;
        if (blk < nblocks) {
            const int64_t r = blk / nb, b = blk - r * nb;
            const float4 *src = reinterpret_cast<const float4 *>(x + r * k + 32 * b);
            a4 = src[2 * l4];
            b4 = src[2 * l4 + 1];
        }
        float amax = fmaxf(fmaxf(fmaxf(fabsf(a4.x), fabsf(a4.y)), fmaxf(fabsf(a4.z), fabsf(a4.w))),
                           fmaxf(fmaxf(fabsf(b4.x), fabsf(b4.y)), fmaxf(fabsf(b4.z), fabsf(b4.w))));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const float d = q8_1_scale(amax), rd = rcp_guarded(d);
        const float vv[8] = {a4.x, a4.y, a4.z, a4.w, b4.x, b4.y, b4.z, b4.w};
        int qq[8];
        q8_1_codes_rcp(vv, d, rd, qq);
        const int q0 = qq[0], q1 = qq[1], q2 = qq[2], q3 = qq[3], q4 = qq[4], q5 = qq[5], q6 = qq[6], q7 = qq[7];
        int S = ((q0 + q1) + (q2 + q3)) + ((q4 + q5) + (q6 + q7));
        S += __shfl_xor_sync(0xffffffffu, S, 2);
        S += __shfl_xor_sync(0xffffffffu, S, 1);
        if (blk < nblocks) {
            // the block's codes start 4 bytes in: two 4-byte stores per lane
            uint32_t *ob = reinterpret_cast<uint32_t *>(xq + blk * kQ81Bytes);
            ob[1 + 2 * l4] = (uint32_t(q0) & 0xffu) | ((uint32_t(q1) & 0xffu) << 8) | ((uint32_t(q2) & 0xffu) << 16) |
                             ((uint32_t(q3) & 0xffu) << 24);
            ob[2 + 2 * l4] = (uint32_t(q4) & 0xffu) | ((uint32_t(q5) & 0xffu) << 8) | ((uint32_t(q6) & 0xffu) << 16) |
                             ((uint32_t(q7) & 0xffu) << 24);
            if (l4 == 0) ob[0] = q8_1_ds_word(d, S);
        }
    }
}

cudaError_t launch_quantize_q8_1(const float *x, int64_t m, int64_t k, void *xq, cudaStream_t st) {
    const int64_t nblocks = m * (k / 32);
    if (nblocks == 0) return cudaSuccess;
    const int threads = 256;
    const bool wide = nblocks >= kWideBlocks;
    int64_t grid = wide ? (nblocks + 63) / 64 : (nblocks + 7) / 8;  // 8 warps per CTA, 8 or 1 blocks per warp
    const int64_t cap = int64_t(device_sm_count()) * 16;
    if (grid > cap) grid = cap;
    return wide ? launch_pdl(quantize_q8_1_kernel<true>, dim3((unsigned)grid), dim3(threads), 0, st, x, m, k,
                             static_cast<uint8_t *>(xq))
                : launch_pdl(quantize_q8_1_kernel<false>, dim3((unsigned)grid), dim3(threads), 0, st, x, m, k,
                             static_cast<uint8_t *>(xq));
}

}  // namespace qmm
