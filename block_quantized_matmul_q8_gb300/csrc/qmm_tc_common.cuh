// qmm_tc_common.cuh -- pieces shared by the two tensor-core kernels (the tiled GEMM and
// the skinny-activation GEMV): fp16 packing, the register split, the Q4_K nibble ->
// fp16 conversion, and the TMA descriptor encoder.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qmm {

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

template <int N> __device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N> __device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

// 8 nibbles (low or high half of bytes w0, w1) -> 8 fp16 values q*sc, exact.
// (0x6400 | q) is the fp16 value 1024 + q; fma((1024+q), sc, -1024*sc) = q*sc exactly.
__device__ __forceinline__ uint4 nibbles_to_f16(uint32_t w0, uint32_t w1, int shift, __half2 sc2, __half2 nsc2) {
    uint32_t p[4];
    const uint32_t a0 = __byte_perm(w0, 0, 0x4140), a1 = __byte_perm(w0, 0, 0x4342);
    const uint32_t b0 = __byte_perm(w1, 0, 0x4140), b1 = __byte_perm(w1, 0, 0x4342);
    p[0] = ((a0 >> shift) & 0x000F000Fu) | 0x64006400u;
    p[1] = ((a1 >> shift) & 0x000F000Fu) | 0x64006400u;
    p[2] = ((b0 >> shift) & 0x000F000Fu) | 0x64006400u;
    p[3] = ((b1 >> shift) & 0x000F000Fu) | 0x64006400u;
    uint4 r;
    r.x = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[0]), sc2, nsc2));
    r.y = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[1]), sc2, nsc2));
    r.z = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[2]), sc2, nsc2));
    r.w = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[3]), sc2, nsc2));
    return r;
}

// The same 8 values in the order 0 2 1 3 4 6 5 7 (the activation codes of the Q4_K GEMM are
// staged in that order, and an MMA's dot does not depend on the order of its k): bytes 0, 2
// of a word already sit under the two halves, bytes 1, 3 after one shift.  Low nibbles as
// (0x6400 | q) = 1024 + q with (sc, -1024 sc); high nibbles in place, (0x6400 | 16 q) =
// 1024 + 16 q, with (sc / 16, -64 sc) (both exact in fp16).  Each fma gives q sc exactly.
__device__ __forceinline__ uint4 nibbles_to_f16_0213(uint32_t w0, uint32_t w1, bool high, __half2 sc2, __half2 nsc2) {
    const uint32_t mask = high ? 0x00F000F0u : 0x000F000Fu;
    uint32_t p[4];
    p[0] = (w0 & mask) | 0x64006400u;
    p[1] = ((w0 >> 8) & mask) | 0x64006400u;
    p[2] = (w1 & mask) | 0x64006400u;
    p[3] = ((w1 >> 8) & mask) | 0x64006400u;
    uint4 r;
    r.x = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[0]), sc2, nsc2));
    r.y = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[1]), sc2, nsc2));
    r.z = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[2]), sc2, nsc2));
    r.w = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[3]), sc2, nsc2));
    return r;
}

// Q5_K: the same 8 values with their fifth bits, bit j of the 8 qh bytes that share the
// nibbles' positions (q0, q1 as w0, w1): (0x6400 | code) is the fp16 1024 + code, code <= 31.
__device__ __forceinline__ uint4 nibbles5_to_f16(uint32_t w0, uint32_t w1, uint32_t q0, uint32_t q1, int shift, int j,
                                                 __half2 sc2, __half2 nsc2) {
    const uint32_t ws[2] = {w0, w1}, qs[2] = {q0, q1};
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t a0 = __byte_perm(ws[i], 0, 0x4140), a1 = __byte_perm(ws[i], 0, 0x4342);
        const uint32_t h0 = __byte_perm(qs[i], 0, 0x4140), h1 = __byte_perm(qs[i], 0, 0x4342);
        p[2 * i] = ((a0 >> shift) & 0x000F000Fu) | (((h0 >> j) & 0x00010001u) << 4) | 0x64006400u;
        p[2 * i + 1] = ((a1 >> shift) & 0x000F000Fu) | (((h1 >> j) & 0x00010001u) << 4) | 0x64006400u;
    }
    uint4 r;
    r.x = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[0]), sc2, nsc2));
    r.y = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[1]), sc2, nsc2));
    r.z = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[2]), sc2, nsc2));
    r.w = h2bits(__hfma2(*reinterpret_cast<__half2 *>(&p[3]), sc2, nsc2));
    return r;
}

// A 2D tiled tensor map over a row-major [outer][inner] array with the given row
// stride (host; the driver's encoder is looked up once).  False on any failure.
bool tc_make_map_2d(CUtensorMap *map, CUtensorMapDataType dt, int esize, const void *base, uint64_t inner,
                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle sw);

}  // namespace qmm
