// qmm_gemv.cu -- bandwidth-bound matrix-vector path for m <= 8 columns.
//
// Every weight byte is read from HBM exactly once; each decoded weight unit is
// reused for all m columns ([P0007] section "How": the multi-column kernels unpack
// each weight once and reuse it for every column; [MMQ] table in section
// "与 MMVQ 的边界": the weight is read once and dropped, the bound is HBM).
//
// Mapping: a half-warp owns one weight row; its 16 lanes walk the row's 64-value
// units u = lane, lane+16, ... (a quarter superblock each for Q4_K/Q6_K, two blocks
// for Q8_0).  Each unit gives exact int32 dot products per 16-wide quarter (dp4a),
// combined per 32-block with the integer sub-scales and folded in fp32 with the
// block scales; the 16 partial sums are added with shuffles.
//
// The q8_1 activations are staged once per CTA in shared memory, repacked so
// that each unit's 64 int8 values start on a 16-byte boundary (80-byte stride per
// unit: 64 values + 16 bytes of padding, which keeps the 16-byte reads of the
// 8 lanes of a quarter-warp on distinct banks) and the per-block (d, s) pairs are
// fp32.  Both half-warps read the same activation addresses (broadcast).
#include <cuda_runtime.h>

#include <algorithm>

#include "qmm_common.cuh"
#include "qmm_internal.h"

namespace qmm {

constexpr int kGemvThreads = 256;
constexpr int kUnitStride = 80;  // bytes per 64-value unit in the staged activations

__host__ __device__ inline int64_t gemv_units(int64_t k) { return (k + 63) / 64; }

size_t gemv_smem_bytes(int64_t k, int ncols) {
    const int64_t U = gemv_units(k);
    return size_t(ncols) * size_t(U) * (kUnitStride + 16);
}

template <int T, int NC>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const uint8_t *__restrict__ W, int64_t n, int k,
                                                            int64_t row_bytes, const uint8_t *__restrict__ xq,
                                                            float *__restrict__ y, int64_t y_ld) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int U = (int)gemv_units(k);
    const int nb32 = k / 32;
    uint8_t *xs = smem;                                                      // [NC][U][80]
    float2 *xds = reinterpret_cast<float2 *>(smem + size_t(NC) * U * kUnitStride);  // [NC][2U]

    // ---- stage the q8_1 columns
    for (int i = threadIdx.x; i < NC * nb32; i += blockDim.x) {
        const int c = i / nb32, b = i - c * nb32;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + (size_t(c) * nb32 + b) * kQ81Bytes);
        const uint32_t dsw = src[0];
        uint32_t *dst = reinterpret_cast<uint32_t *>(xs + (size_t(c) * U + (b >> 1)) * kUnitStride + 32 * (b & 1));
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = src[1 + j];
        xds[size_t(c) * 2 * U + b] = make_float2(half_lo(dsw), half_hi(dsw));
    }
    // an odd block count leaves the second half of the last unit unset: zero it
    if (nb32 & 1) {
        for (int i = threadIdx.x; i < NC * 8; i += blockDim.x) {
            const int c = i / 8, j = i % 8;
            reinterpret_cast<uint32_t *>(xs + (size_t(c) * U + U - 1) * kUnitStride + 32)[j] = 0u;
            if (j == 0) xds[size_t(c) * 2 * U + nb32] = make_float2(0.f, 0.f);
        }
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int l16 = lane & 15;
    const int64_t npairs = (n + 1) / 2;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;

    for (int64_t pair = warp; pair < npairs; pair += nwarp) {
        const int64_t r = 2 * pair + (lane >> 4);
        const bool valid = r < n;
        const uint8_t *row = W + (valid ? r : 0) * row_bytes;
        float acc[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] = 0.f;

        for (int u = l16; u < U; u += 16) {
            Unit w;
            if (valid) {
                decode_unit<T>(row, u, nb32, w);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) w.q[i] = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) w.isc[i] = 0;
                w.fd[0] = w.fd[1] = w.fm[0] = w.fm[1] = 0.f;
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const int4 *xv = reinterpret_cast<const int4 *>(xs + (size_t(c) * U + u) * kUnitStride);
                const float4 ds = reinterpret_cast<const float4 *>(xds + size_t(c) * 2 * U)[u];
                int s[4];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int4 xw = xv[qq];
                    int a = __dp4a(w.q[4 * qq + 0], xw.x, 0);
                    a = __dp4a(w.q[4 * qq + 1], xw.y, a);
                    a = __dp4a(w.q[4 * qq + 2], xw.z, a);
                    a = __dp4a(w.q[4 * qq + 3], xw.w, a);
                    s[qq] = a;
                }
                // exact int32 per 32-block: |isc*dot16| sums stay below 2^24
                const int b0 = w.isc[0] * s[0] + w.isc[1] * s[1];
                const int b1 = w.isc[2] * s[2] + w.isc[3] * s[3];
                float a = acc[c];
                a = fmaf(w.fd[0] * ds.x, (float)b0, a);
                a = fmaf(-w.fm[0], ds.y, a);
                a = fmaf(w.fd[1] * ds.z, (float)b1, a);
                a = fmaf(-w.fm[1], ds.w, a);
                acc[c] = a;
            }
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            float a = acc[c];
            a += __shfl_xor_sync(0xffffffffu, a, 8);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            acc[c] = a;
        }
        if (valid && l16 == 0) {
#pragma unroll
            for (int c = 0; c < NC; ++c) y[c * y_ld + r] = acc[c];
        }
    }
}

template <int T, int NC>
static cudaError_t launch_gemv_nc(const void *W, int64_t n, int64_t k, const void *xq, float *y, int64_t y_ld,
                                  cudaStream_t st) {
    const size_t smem = gemv_smem_bytes(k, NC);
    auto kern = gemv_kernel<T, NC>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemvThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t npairs = (n + 1) / 2;
    const int64_t need = (npairs + kGemvThreads / 32 - 1) / (kGemvThreads / 32);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(need, int64_t(device_sm_count()) * per_sm));
    const int64_t row_bytes = int64_t(k / block_elems(T)) * block_bytes(T);
    kern<<<(unsigned)grid, kGemvThreads, smem, st>>>(static_cast<const uint8_t *>(W), n, (int)k, row_bytes,
                                                     static_cast<const uint8_t *>(xq), y, y_ld);
    return cudaGetLastError();
}

template <int T>
static cudaError_t launch_gemv_t(const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                                 cudaStream_t st) {
    const uint8_t *x = static_cast<const uint8_t *>(xq);
    const size_t xrow = size_t(k / 32) * kQ81Bytes;
    const size_t budget = size_t(device_smem_optin());
    int64_t c0 = 0;
    while (c0 < m) {
        int nc = (int)std::min<int64_t>(8, m - c0);
        while (nc > 1 && gemv_smem_bytes(k, nc) > budget) --nc;
        if (gemv_smem_bytes(k, nc) > budget) return cudaErrorInvalidValue;
        cudaError_t e;
        const void *xc = x + c0 * xrow;
        float *yc = y + c0 * n;
        switch (nc) {
        case 1: e = launch_gemv_nc<T, 1>(W, n, k, xc, yc, n, st); break;
        case 2: e = launch_gemv_nc<T, 2>(W, n, k, xc, yc, n, st); break;
        case 3: e = launch_gemv_nc<T, 3>(W, n, k, xc, yc, n, st); break;
        case 4: e = launch_gemv_nc<T, 4>(W, n, k, xc, yc, n, st); break;
        case 5: e = launch_gemv_nc<T, 5>(W, n, k, xc, yc, n, st); break;
        case 6: e = launch_gemv_nc<T, 6>(W, n, k, xc, yc, n, st); break;
        case 7: e = launch_gemv_nc<T, 7>(W, n, k, xc, yc, n, st); break;
        default: e = launch_gemv_nc<T, 8>(W, n, k, xc, yc, n, st); break;
        }
        if (e != cudaSuccess) return e;
        c0 += nc;
    }
    return cudaSuccess;
}

cudaError_t launch_gemv(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                        cudaStream_t st) {
    switch (t) {
    case QMM_Q4_K: return launch_gemv_t<QMM_Q4_K>(W, n, k, xq, m, y, st);
    case QMM_Q6_K: return launch_gemv_t<QMM_Q6_K>(W, n, k, xq, m, y, st);
    case QMM_Q8_0: return launch_gemv_t<QMM_Q8_0>(W, n, k, xq, m, y, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qmm
