// qmm_gemv_mma.cu -- multi-column GEMV (1 <= m <= 8 activation columns) for Q4_K on the
// warp-level tensor-core MMA.
//
// The speculative-verify batch of [P0007] ("How", "Speculative decoding": 2-8 columns,
// each weight unpacked once and reused for every column) reads the weights once while
// the work per weight grows with the column count.  On CUDA cores every extra column
// costs one more set of exact dp4a dots per weight; here the columns are the N = 8 side of
// an `mma.sync m16n8k16` with fp16 operands and fp32 accumulation, so one instruction forms
// the dots of 16 weight rows with all 8 columns and the per-column cost disappears.
//
// Exactness ([MMQ] sections "dp4a 路径的 Q4_K" and "输出端: 写回与 scale 修正": exact integer
// sub-block dots, then the fp32 fold with the block scales).  The operands are integers:
//   B (activations): the q8_1 codes, |q| <= 127, exact in fp16.
//   A (weights): a nibble byte v becomes the fp16 1024 + (v & 15) for the low nibble and
//     1024 + (v & 0xf0) = 1024 + 16 q for the high one, by OR-ing the nibble bits into the
//     exponent pattern of 1024 (no conversion instructions).
//   C (accumulator input): -1024 * sum(q_x) of the 32-block, exact.
// Every product is an integer of at most 1264 * 127 and every partial sum stays below
// 4064 * 1024 + 32 * 1264 * 127 < 2^24, so the fp32 accumulator ends on exactly
// sum_i q_w,i q_x,i of a low sub-block (16 times it for a high one) in any order of
// addition.  The fold is then the method's, per 32-wide sub-block b:
//   y += d sc_b d8_b sumi_b - dmin m_b s_b,
// with the min term sum_b m_b s_b of a superblock formed by one more MMA (the 6-bit mins
// as A, the q8_1 s values as B; 8 real terms, 8 zeros).
//
// The k index inside an MMA is a free permutation as long as A and B use the same one:
// lane (g, t) supplies, for K16 step ks of a 32-byte chunk of nibbles, the 4 bytes
// 8t + 4ks .. 8t + 4ks + 3 (bytes 0, 2 at MMA positions 2t, 2t+1, bytes 1, 3 at 2t+8, 2t+9,
// which puts each nibble under its fp16 half with one shift), so a lane's weights for both
// steps are one 8-byte load per row, and its activations, staged as fp16 in the order
// 0 2 1 3 of every 4 codes, one 16-byte load.
//
// Layout.  One persistent CTA per SM owns a contiguous range of 16-row tiles.  A producer
// warp streams whole tiles (16 rows x all of k, one bulk copy per row) through a ring of
// shared-memory stages.  All 16 consumer warps work on every tile, each taking whole
// superblocks of it (superblock j of tile t goes to warp (t nsb + j) mod 16, so the warps'
// shares even out over the tiles), and writes its 16 x 8 partial results to its own slot in
// the tile's set of partial sums (set t mod (nstages + 1)).  Once all 16 have released the
// stage, the producer warp first reuses it for the next tile's copy, then sums the released
// tile's 16 slots in warp order (so the result does not depend on timing) and writes its
// outputs.  The set it reads is the one that tile t + 1 will write, whose copy the producer
// has not issued yet, so no consumer writes it meanwhile.  Every consumer warp waits for every
// tile, so a stage's earlier tile has always landed when a warp waits for its next one.
// The activations are staged once per CTA: the m columns' q8_1 codes as fp16, and per block
// d8, -1024 sum(q) and s.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_tc_ptx.cuh"

namespace qmm {
namespace {

constexpr int kMmaWarps = 16;                      // consumer warps
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;  // plus the producer warp
constexpr int kTileRows = 16;                      // MMA M: weight rows of a tile
constexpr int kCols = 8;                           // MMA N: activation columns (missing ones zero)
constexpr int kMaxStages = 8;
constexpr int kMinStages = 2;

// Shared-memory plan for a row length k: rows and activation columns padded so that their
// strides are 8 words past a multiple of 32 words (the 4 rows or columns that the 16 lanes of
// a half-warp read start on different bank groups).
struct MmaPlan {
    int nstages;
    int64_t row_stride, x_stride;
    size_t fixed, stage_bytes, smem;
};
// bytes rounded up so that bytes / 4 is `res` past a multiple of 32 (bytes a multiple of 16)
int64_t pad_to_bank(int64_t bytes, int res) {
    const int64_t w = (bytes / 4) % 32;
    return bytes + 4 * ((res - w + 32) % 32);
}
bool mma_plan(int64_t k, int m, size_t budget, MmaPlan &p) {
    if (k <= 0 || k % 256 || m < 1 || m > kCols) return false;
    if (budget <= 2048) return false;
    budget -= 1024;  // the kernel's static shared memory (barriers), rounded up
    const int64_t nb32 = k / 32, row_bytes = (k / 256) * kQ4KBytes;
    // weight rows 8 words apart in bank terms: the 4 rows a half-warp reads; fp16 activation
    // columns 16 words apart: the 2 columns a quarter-warp reads
    p.row_stride = pad_to_bank(row_bytes, 8);
    p.x_stride = pad_to_bank(2 * k, 16);
    // staged codes [m][x_stride], factors [nb32][8] float2, s [8][nb32] fp16, and the one set
    // of partial sums beyond one per stage
    p.fixed = 1024 + size_t(m) * p.x_stride + size_t(nb32) * kCols * 8 + size_t(kCols) * nb32 * 2 +
              size_t(kMmaWarps) * kTileRows * kCols * 4;
    p.stage_bytes = size_t(kTileRows) * p.row_stride;
    if (p.fixed >= budget) return false;
    // per stage: the tile's rows and each consumer warp's 16 x 8 fp32 partial sums
    const int64_t st = int64_t(budget - p.fixed) / int64_t(p.stage_bytes + kMmaWarps * kTileRows * kCols * 4);
    p.nstages = (int)std::min<int64_t>(st, kMaxStages);
    p.smem = p.fixed + size_t(p.nstages) * (p.stage_bytes + kMmaWarps * kTileRows * kCols * 4);
    return p.nstages >= kMinStages;
}

// d += A B for one m16n8k16 tile (fp16 operands, fp32 accumulator, in place).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A B + c (c0 for rows g, c1 for rows g + 8 of columns 2t, 2t+1): the first K16 step of a
// sub-block, the accumulator input read from the factor registers without copies.
__device__ __forceinline__ void mma_16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1, float c0, float c1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%10,%11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}

// (v & mask) | 0x64006400 in one logic op: the nibble bits under the fp16 pattern of 1024.
__device__ __forceinline__ uint32_t nib_f16(uint32_t v, uint32_t mask) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(0x64006400u));
    return r;
}

// Four int8 codes (one word) as two fp16 pairs in the order (0, 2), (1, 3).
__device__ __forceinline__ uint2 codes_f16_0213(uint32_t w) {
    const int q0 = (int8_t)(w & 0xffu), q1 = (int8_t)((w >> 8) & 0xffu);
    const int q2 = (int8_t)((w >> 16) & 0xffu), q3 = (int8_t)(w >> 24);
    const __half2 a = __halves2half2(__int2half_rn(q0), __int2half_rn(q2));
    const __half2 b = __halves2half2(__int2half_rn(q1), __int2half_rn(q3));
    return make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
}

// Shared-memory accesses by 32-bit shared addresses (the hot loop's address arithmetic stays
// in 32 bits and every access is a shared one).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts64(uint32_t a, float2 v) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y) : "memory");
}

// One superblock (j) of the 16-row tile: rows g and g + 8 of the lane (blk, blk8 point at the
// superblock in the two staged rows), B column g (xg: its staged fp16 codes, xv false for a
// column past m, whose codes are zero), the factor table and the s values of the column (sg).
// tot01: (row g, cols 2t, 2t+1), tot23: (row g+8, cols 2t, 2t+1).
__device__ __forceinline__ void fold_superblock(uint32_t blk, uint32_t blk8, uint32_t xg, bool xv, uint32_t fz,
                                                uint32_t sg, int j, int t, float2 &tot01, float2 &tot23) {
    const uint4 h0 = lds128(blk), h8 = lds128(blk8);
    // the 6-bit scales and mins, four per word: sub-blocks 0..3 and 4..7 (GGUF packing)
    const uint32_t sl0 = h0.y & 0x3f3f3f3fu, ml0 = h0.z & 0x3f3f3f3fu;
    const uint32_t sh0 = (h0.w & 0x0f0f0f0fu) | ((h0.y >> 2) & 0x30303030u);
    const uint32_t mh0 = ((h0.w >> 4) & 0x0f0f0f0fu) | ((h0.z >> 2) & 0x30303030u);
    const uint32_t sl8 = h8.y & 0x3f3f3f3fu, ml8 = h8.z & 0x3f3f3f3fu;
    const uint32_t sh8 = (h8.w & 0x0f0f0f0fu) | ((h8.y >> 2) & 0x30303030u);
    const uint32_t mh8 = ((h8.w >> 4) & 0x0f0f0f0fu) | ((h8.z >> 2) & 0x30303030u);
    const float d0 = half_lo(h0.x), dmin0 = half_hi(h0.x);
    const float d8r = half_lo(h8.x), dmin8 = half_hi(h8.x);
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // 32-byte chunk c of nibbles: sub-blocks 2c (low) and 2c + 1 (high)
        const uint2 w0 = lds64(blk + 16 + 32 * c + 8 * t), w8 = lds64(blk8 + 16 + 32 * c + 8 * t);
        const int blo = 8 * j + 2 * c;  // the 32-blocks of x under the two sub-blocks
        const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
        const uint4 xa = xv ? lds128(xg + 64 * blo + 16 * t) : zero4;
        const uint4 xb = xv ? lds128(xg + 64 * (blo + 1) + 16 * t) : zero4;
        // {d8, -1024 sum q} of columns 2t and 2t + 1
        const float4 fl = lds128f(fz + (blo * kCols + 2 * t) * 8);
        const float4 fh = lds128f(fz + ((blo + 1) * kCols + 2 * t) * 8);
        float clo[4], chi[4];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const uint32_t a = ks ? w0.y : w0.x, a8 = ks ? w8.y : w8.x;
            const uint32_t as = a >> 8, a8s = a8 >> 8;  // bytes 1, 3 under the halves
            const uint32_t bl0 = ks ? xa.z : xa.x, bl1 = ks ? xa.w : xa.y;
            const uint32_t bh0 = ks ? xb.z : xb.x, bh1 = ks ? xb.w : xb.y;
            const uint32_t l0 = nib_f16(a, 0x000f000fu), l1 = nib_f16(a8, 0x000f000fu);
            const uint32_t l2 = nib_f16(as, 0x000f000fu), l3 = nib_f16(a8s, 0x000f000fu);
            const uint32_t h0_ = nib_f16(a, 0x00f000f0u), h1_ = nib_f16(a8, 0x00f000f0u);
            const uint32_t h2_ = nib_f16(as, 0x00f000f0u), h3_ = nib_f16(a8s, 0x00f000f0u);
            if (ks == 0) {  // the accumulators start at -1024 sum(q) of each column's block
                mma_16816_c(clo, l0, l1, l2, l3, bl0, bl1, fl.y, fl.w);
                mma_16816_c(chi, h0_, h1_, h2_, h3_, bh0, bh1, fh.y, fh.w);
            } else {
                mma_16816(clo, l0, l1, l2, l3, bl0, bl1);
                mma_16816(chi, h0_, h1_, h2_, h3_, bh0, bh1);
            }
        }
        // d sc d8 per (row, column): the high sub-block's dot is 16 times its sumi
        const uint32_t s0w = c < 2 ? sl0 : sh0, s8w = c < 2 ? sl8 : sh8;
        const int sb0 = 8 * ((2 * c) & 3), sb1 = 8 * ((2 * c + 1) & 3);
        const float al0 = d0 * (float)((s0w >> sb0) & 0xffu), ah0 = d0 * 0.0625f * (float)((s0w >> sb1) & 0xffu);
        const float al8 = d8r * (float)((s8w >> sb0) & 0xffu), ah8 = d8r * 0.0625f * (float)((s8w >> sb1) & 0xffu);
        const float2 d8l = make_float2(fl.x, fl.z), d8h = make_float2(fh.x, fh.z);
        tot01 = __ffma2_rn(__fmul2_rn(make_float2(al0, al0), d8l), make_float2(clo[0], clo[1]), tot01);
        tot01 = __ffma2_rn(__fmul2_rn(make_float2(ah0, ah0), d8h), make_float2(chi[0], chi[1]), tot01);
        tot23 = __ffma2_rn(__fmul2_rn(make_float2(al8, al8), d8l), make_float2(clo[2], clo[3]), tot23);
        tot23 = __ffma2_rn(__fmul2_rn(make_float2(ah8, ah8), d8h), make_float2(chi[2], chi[3]), tot23);
    }
    // min term: sum_b m_b s_b by one MMA; A row g = mins of sub-blocks 2t, 2t+1 at positions
    // 2t, 2t+1 (positions 8..15 zero), B column g = the s values of the same blocks
    const uint32_t sel = (t & 1) ? 0x4342u : 0x4140u;
    uint32_t m0 = __byte_perm(t < 2 ? ml0 : mh0, 0u, sel) | 0x64006400u;
    uint32_t m8 = __byte_perm(t < 2 ? ml8 : mh8, 0u, sel) | 0x64006400u;
    const __half2 k1024 = __float2half2_rn(1024.f);
    const __half2 mf0 = __hsub2(*reinterpret_cast<__half2 *>(&m0), k1024);
    const __half2 mf8 = __hsub2(*reinterpret_cast<__half2 *>(&m8), k1024);
    const uint32_t sv = lds32(sg + 2 * (8 * j + 2 * t));
    float cm[4] = {0.f, 0.f, 0.f, 0.f};
    mma_16816(cm, *reinterpret_cast<const uint32_t *>(&mf0), *reinterpret_cast<const uint32_t *>(&mf8), 0u, 0u, sv,
              0u);
    tot01 = __ffma2_rn(make_float2(-dmin0, -dmin0), make_float2(cm[0], cm[1]), tot01);
    tot23 = __ffma2_rn(make_float2(-dmin8, -dmin8), make_float2(cm[2], cm[3]), tot23);
}

__global__ void __launch_bounds__(kMmaThreads, 1)
    gemv_q4k_mma_kernel(const uint8_t *__restrict__ W, int64_t n, int k, int m, int nstages, int64_t row_stride,
                        int64_t x_stride, const uint8_t *__restrict__ xq, float *__restrict__ y, int *status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);  // stays a shared pointer
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsb = k / 256, nb32 = k / 32;
    const int64_t row_bytes = int64_t(nsb) * kQ4KBytes;
    const size_t stage_bytes = size_t(kTileRows) * size_t(row_stride);
    uint8_t *stages = smem;                                                        // [nstages][16][row_stride]
    uint8_t *xs = stages + size_t(nstages) * stage_bytes;                          // [m][x_stride] fp16 codes
    float2 *fz = reinterpret_cast<float2 *>(xs + size_t(m) * x_stride);           // [nb32][8] {d8, -1024 sum q}
    uint16_t *sh = reinterpret_cast<uint16_t *>(fz + size_t(nb32) * kCols);        // [8][nb32] s (fp16 bits)
    float *acc = reinterpret_cast<float *>(sh + size_t(kCols) * nb32);             // [nstages + 1][16 warps][16][8]
    const int nacc = nstages + 1;
    volatile int *abortp = &abort_flag;

    // this CTA's tiles of 16 rows (the last tile of the matrix may be shorter)
    const int64_t ntile_all = (n + kTileRows - 1) / kTileRows;
    const int64_t tb = ntile_all * blockIdx.x / gridDim.x, te = ntile_all * (blockIdx.x + 1) / gridDim.x;
    const int ntiles = (int)(te - tb);

    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < nstages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty[s]), kMmaWarps);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // the weights are never written by this library's kernels: they stream before the
    // preceding kernel (the activation quantizer) has finished; x waits for it
    ptx::grid_launch_dependents();

    if (warp == kMmaWarps) {
        // ---------------- producer warp: copies in, results out
        // Tile t of the CTA goes to stage t % nstages and its partial sums to set t % nacc.
        // Once the 16 consumer warps have released a stage, the warp issues the stage's next
        // copy, then adds the released tile's slots in warp order and writes its outputs.
        auto write_tile = [&](int t) {
            const int64_t row0 = (tb + t) * kTileRows;
            const float *a = acc + size_t(t % nacc) * kMmaWarps * kTileRows * kCols;
#pragma unroll
            for (int i = 0; i < kTileRows * kCols / 32; ++i) {
                const int e = lane + 32 * i, r = e & 15, c = e >> 4;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kMmaWarps; ++w) v += a[(w * kTileRows + r) * kCols + c];
                if (c < m && row0 + r < n) y[int64_t(c) * n + row0 + r] = v;
            }
        };
        int issued = 0;
        bool ok = true;
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % nstages;
            if (t >= nstages) {
                ok = __all_sync(0xffffffffu,
                                ptx::mbar_wait_spin(ptx::smem_u32(&empty[s]), ((t / nstages) - 1) & 1, abortp));
                if (!ok) break;
            }
            const int64_t row0 = (tb + t) * kTileRows;
            const int rows = (int)min((int64_t)kTileRows, n - row0);
            const uint32_t bar = ptx::smem_u32(&full[s]);
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar, uint32_t(rows * row_bytes));
            __syncwarp();
            if (lane < rows)
                ptx::bulk_g2s(ptx::smem_u32(stages + s * stage_bytes + size_t(lane) * row_stride),
                              W + (row0 + lane) * row_bytes, uint32_t(row_bytes), bar);
            ++issued;
            if (t >= nstages) {
                write_tile(t - nstages);
                __syncwarp();
            }
        }
        // every issued copy must have landed before the CTA exits (bounded waits, independent
        // of the abort flag); then the last tiles' results
        int dummy = 0;
        for (int t = max(0, issued - nstages); t < issued; ++t)
            ptx::mbar_wait(ptx::smem_u32(&full[t % nstages]), (t / nstages) & 1, &dummy);
        for (int t = max(0, issued - nstages); ok && t < issued; ++t) {
            const int s = t % nstages;
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&empty[s]), (t / nstages) & 1, abortp));
            if (ok) write_tile(t);
        }
    } else {
        // ---------------- consumers: stage the activations, then fold the tiles
        ptx::grid_dependency_wait();
        for (int i = tid; i < kCols * nb32; i += kMmaWarps * 32) {
            const int c = i / nb32, b = i - c * nb32;
            float d8 = 0.f, z = 0.f;
            uint16_t sbits = 0;
            if (c < m) {
                const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + (size_t(c) * nb32 + b) * kQ81Bytes);
                const uint32_t dsw = src[0];
                uint32_t q[8];
                int sum = 0;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    q[jj] = src[1 + jj];
                    sum = __dp4a((int)q[jj], 0x01010101, sum);
                }
                // 32 codes as fp16, every 4 in the order 0 2 1 3: 64 bytes
                uint4 *dst = reinterpret_cast<uint4 *>(xs + size_t(c) * x_stride + size_t(b) * 64);
#pragma unroll
                for (int jj = 0; jj < 8; jj += 2) {
                    const uint2 e0 = codes_f16_0213(q[jj]), e1 = codes_f16_0213(q[jj + 1]);
                    dst[jj / 2] = make_uint4(e0.x, e0.y, e1.x, e1.y);
                }
                d8 = half_lo(dsw);
                z = -1024.f * (float)sum;
                sbits = (uint16_t)(dsw >> 16);
            }
            fz[size_t(b) * kCols + c] = make_float2(d8, z);
            sh[size_t(c) * nb32 + b] = sbits;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kMmaWarps * 32) : "memory");

        const int g = lane >> 2, t4 = lane & 3;
        const bool xv = g < m;  // columns past m: zero codes, nothing staged
        const uint32_t xg = ptx::smem_u32(xs + size_t(xv ? g : 0) * x_stride);
        const uint32_t sg = ptx::smem_u32(sh + size_t(g) * nb32);
        const uint32_t fza = ptx::smem_u32(fz);
        const uint32_t st0 = ptx::smem_u32(stages), acc0 = ptx::smem_u32(acc);
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % nstages;
            // all 16 warps wait for every tile and start on it together: probe without
            // suspending, so that no warp pays a wake-up delay per tile
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_spin(ptx::smem_u32(&full[s]), (t / nstages) & 1, abortp)))
                break;
            float2 tot01 = make_float2(0.f, 0.f), tot23 = make_float2(0.f, 0.f);
            const uint32_t rg = st0 + uint32_t(s * stage_bytes) + uint32_t(g * row_stride);
            const uint32_t rg8 = rg + uint32_t(8 * row_stride);
            int j = (int)((warp - (int64_t(t) * nsb) % kMmaWarps + kMmaWarps) % kMmaWarps);
            for (; j < nsb; j += kMmaWarps)
                fold_superblock(rg + j * kQ4KBytes, rg8 + j * kQ4KBytes, xg, xv, fza, sg, j, t4, tot01, tot23);
            // this warp's slot of the stage: rows g and g + 8, columns 2t4, 2t4 + 1
            const uint32_t a = acc0 + uint32_t((((t % nacc) * kMmaWarps + warp) * kTileRows) * kCols * 4);
            sts64(a + 4 * (g * kCols + 2 * t4), tot01);
            sts64(a + 4 * ((g + 8) * kCols + 2 * t4), tot23);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty[s]));
        }
    }
    __syncthreads();
    if (tid == 0 && abort_flag && status) atomicExch(status, (int)QMM_ERR_DEVICE);
}

}  // namespace

bool gemv_mma_supported(qmm_type t, int64_t n, int64_t k, int64_t m) {
    if (t != QMM_Q4_K || n <= 0 || m < 1 || m > 8 || k % 256 != 0) return false;
    MmaPlan p;
    return mma_plan(k, (int)m, size_t(device_smem_optin()), p);
}

cudaError_t launch_gemv_mma(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                            cudaStream_t st) {
    MmaPlan p;
    if (!gemv_mma_supported(t, n, k, m) || !mma_plan(k, (int)m, size_t(device_smem_optin()), p))
        return cudaErrorNotSupported;
    cudaError_t e = ensure_smem(gemv_q4k_mma_kernel, p.smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(device_sm_count(), (n + kTileRows - 1) / kTileRows));
    return launch_pdl(gemv_q4k_mma_kernel, dim3((unsigned)grid), dim3(kMmaThreads), p.smem, st,
                      static_cast<const uint8_t *>(W), n, (int)k, (int)m, p.nstages, p.row_stride, p.x_stride,
                      static_cast<const uint8_t *>(xq), y, static_cast<int *>(nullptr));
}

}  // namespace qmm
