// mma_sync_peak.cu -- throughput of the warp-level tensor-core MMA (mma.sync) on the
// current GPU: int8 m16n8k32 with s32 accumulation, and fp16 m16n8k16 with f32
// accumulation for comparison.  Every warp runs 8 independent accumulator chains and
// every SM holds 16 or 32 warps.  On sm_103a tcgen05 has no int8 kind, so the int8
// figure is the GPU's dense int8 tensor-core rate: the denominator that an int8 roofline
// of the quantized GEMM would use.  Not part of the library; built and run by hand:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o mma_sync_peak mma_sync_peak.cu && ./mma_sync_peak
#include <cstdio>
#include <cuda_runtime.h>
#include <stdint.h>

#define CHAINS 8

__global__ void __launch_bounds__(128) mma_s8(int iters, int32_t *out) {
    uint32_t a0 = threadIdx.x * 0x01010101u, a1 = a0 ^ 0x5a5a5a5au, a2 = a0 + 7u, a3 = a0 * 3u;
    uint32_t b0 = blockIdx.x * 0x01030507u, b1 = b0 ^ 0x3c3c3c3cu;
    int32_t c[CHAINS][4];
#pragma unroll
    for (int j = 0; j < CHAINS; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < CHAINS; ++j)
            asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                         "{%0,%1,%2,%3};"
                         : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                         : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int32_t s = 0;
#pragma unroll
    for (int j = 0; j < CHAINS; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(128) mma_f16(int iters, float *out) {
    uint32_t a0 = 0x3c003c00u, a1 = 0x3c003c00u, a2 = 0x3c003c00u, a3 = 0x3c003c00u;  // fp16 1.0 pairs
    uint32_t b0 = 0x00000000u, b1 = 0x00000000u;                                      // zeros: no growth
    float c[CHAINS][4];
#pragma unroll
    for (int j = 0; j < CHAINS; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = float(threadIdx.x);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < CHAINS; ++j)
            asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                         "{%0,%1,%2,%3};"
                         : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
                         : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < CHAINS; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

int main() {
    int dev = 0, nsm = 0;
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 128;
    void *buf = nullptr;
    for (int per_sm : {4, 8}) {
        const int blocks = nsm * per_sm;
        if (cudaMalloc(&buf, size_t(blocks) * threads * 4) != cudaSuccess) return 1;
        const int iters = 2048;
        cudaEvent_t e0, e1;
        cudaEventCreate(&e0);
        cudaEventCreate(&e1);
        for (int kind = 0; kind < 2; ++kind) {
            float best = 1e30f;
            for (int rep = 0; rep < 6; ++rep) {
                cudaEventRecord(e0);
                if (kind == 0) mma_s8<<<blocks, threads>>>(iters, (int32_t *)buf);
                else mma_f16<<<blocks, threads>>>(iters, (float *)buf);
                cudaEventRecord(e1);
                cudaEventSynchronize(e1);
                float ms = 0.f;
                cudaEventElapsedTime(&ms, e0, e1);
                if (rep > 0 && ms < best) best = ms;
            }
            cudaError_t err = cudaGetLastError();
            if (err != cudaSuccess) { printf("error %s\n", cudaGetErrorString(err)); return 1; }
            const double ops_per_mma = kind == 0 ? 2.0 * 16 * 8 * 32 : 2.0 * 16 * 8 * 16;
            const double ops = double(blocks) * (threads / 32) * iters * CHAINS * ops_per_mma;
            printf("%s mma.sync, %d CTAs/SM x 4 warps: %.3f ms, %.1f TOPS\n", kind == 0 ? "int8 m16n8k32" : "fp16 m16n8k16",
                   per_sm, best, ops / (best * 1e-3) / 1e12);
        }
        cudaFree(buf);
    }
    return 0;
}
