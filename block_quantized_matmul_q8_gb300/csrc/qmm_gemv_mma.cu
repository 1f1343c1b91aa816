// qmm_gemv_mma.cu -- multi-column GEMV (2 <= m <= 8 activation columns) for Q4_K on the
// warp-level tensor-core MMA.
//
// The speculative-verify batch of [P0007] ("How", "Speculative decoding": 2-8 columns,
// each weight unpacked once and reused for every column) has the weight read once and
// the work per weight growing with the column count.  On CUDA cores every extra column
// costs one more set of exact dp4a dots per weight; here the columns are the N = 8 side of
// an `mma.sync m16n8k16` with fp16 operands and fp32 accumulation, so one instruction forms
// the dots of 16 weight rows with all 8 columns, and the per-column cost disappears.
//
// Exactness ([MMQ] sections "dp4a 路径的 Q4_K" and "输出端: 写回与 scale 修正": exact integer
// sub-block dots, then the fp32 fold with the block scales).  The operands are integers:
//   B (activations): the q8_1 codes, |q| <= 127, exact in fp16.
//   A (weights): a nibble byte v becomes the fp16 1024 + (v & 15) for the low nibble and
//     1024 + (v & 0xf0) = 1024 + 16 q for the high one, by OR-ing the nibble bits into the
//     exponent pattern of 1024 (two logic ops per 4 bytes, no conversion instructions).
//   C (accumulator input): -1024 * sum(q_x) of the 32-block, exact.
// Every product is an integer below 1264 * 127 and every partial sum below 2^24, so the
// fp32 accumulator ends on exactly sum_i q_w,i q_x,i of the low sub-block (16 times it for
// the high one) whatever order the tensor core adds in.  The fold is then the method's:
//   y += d sc_b d8_b sumi_b - dmin m_b s_b   per 32-wide sub-block b.
//
// Layout.  One persistent CTA per SM owns a contiguous range of rows (whole 8-row groups).
// A producer warp streams chunks of 16 rows x 4 superblocks (576 bytes of each row, one
// 2-D tensor-map box) through a ring of shared-memory stages.  Each of the 16 consumer
// warps takes one 64-value unit (two sub-blocks) of every chunk for the tile's 16 rows
// (MMA M = 16) and keeps its share of the 16 x 8 results in registers over the tile's
// chunks; at the end of a tile the 16 shares are summed through shared memory.  The
// activations are staged once per CTA as fp16 in the order of the B fragments, with the
// per-block factors d8, s and -1024 sum(q) next to them.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_tc_common.cuh"
#include "qmm_tc_ptx.cuh"

namespace qmm {
namespace {

constexpr int kMmaWarps = 16;                            // consumer warps: one unit of a chunk each
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;        // plus the producer warp
constexpr int kTileRows = 16;                            // MMA M: weight rows of a tile
constexpr int kChunkSb = 4;                              // superblocks per chunk: 16 units
constexpr int kRowChunk = kChunkSb * kQ4KBytes;          // 576 bytes of a row per chunk
constexpr int kStageBytes = kTileRows * kRowChunk;       // 9216
constexpr int kMaxStages = 16;
constexpr int kMinStages = 4;
constexpr int kFacBytes = 4 * 3 * 16;                    // per unit: 4 column pairs x 3 float4
constexpr int kRedBytes = 2 * kMmaWarps * 32 * 16;       // two buffers of 16 warps x 32 lanes x float4

__host__ __device__ inline int64_t mma_units(int64_t k) {  // units staged: whole chunks of 16
    return ((k / 256 + kChunkSb - 1) / kChunkSb) * kChunkSb * 4;
}

size_t mma_x_bytes(int64_t k, int m) { return size_t(mma_units(k)) * (size_t(m) * 128 + kFacBytes); }

int mma_stages(int64_t k, int m, size_t budget) {
    const size_t fixed = 1024 + mma_x_bytes(k, m) + kRedBytes;
    if (fixed >= budget) return 0;
    const int st = (int)std::min<size_t>(kMaxStages, (budget - fixed) / kStageBytes);
    return st >= kMinStages ? st : 0;
}

// d += A B for one m16n8k16 tile (fp16 operands, fp32 accumulator, in place).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (v & mask) | 0x64006400 in one logic op: the nibble bits under the fp16 pattern of 1024.
__device__ __forceinline__ uint32_t nib_f16(uint32_t v, uint32_t mask) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(0x64006400u));
    return r;
}

// Staged activation column c of unit u: 64 fp16 codes, 16-byte chunk j (j = 0..3 the low
// 32-block, 4..7 the high one) holding the 8 codes 8(j & 3) .. 8(j & 3) + 7 of its block in
// the order 0 2 1 3 4 6 5 7, which is the order in which the A fragments take the bytes of a
// weight word.  Odd columns swap the two halves (chunk j at j ^ 4), so that the 8 lanes of a
// quarter-warp, 2 columns x 4 chunks, read 8 different bank groups.
__device__ __forceinline__ int xh_chunk(int c, int j) { return j ^ ((c & 1) << 2); }

__global__ void __launch_bounds__(kMmaThreads, 1)
    gemv_q4k_mma_kernel(const __grid_constant__ CUtensorMap tm16, const __grid_constant__ CUtensorMap tm8,
                        int64_t n, int k, int m, int nstages, const uint8_t *__restrict__ xq, float *__restrict__ y,
                        int *status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsb = k / 256, cpt = (nsb + kChunkSb - 1) / kChunkSb;  // chunks per tile
    const int Up = (int)mma_units(k);
    uint8_t *stages = smem;
    uint8_t *xh = stages + size_t(nstages) * kStageBytes;        // [Up][m][128 B]
    uint8_t *fac = xh + size_t(Up) * m * 128;                    // [Up][4 pairs][3 float4]
    float4 *red = reinterpret_cast<float4 *>(fac + size_t(Up) * kFacBytes);  // [2][16][32]
    volatile int *abortp = &abort_flag;

    // rows of this CTA: whole groups of 8 rows; tiles of 16 rows, the last possibly 8
    const int64_t ngr = (n + 7) / 8;
    const int64_t r0 = 8 * (ngr * blockIdx.x / gridDim.x);
    const int64_t r1 = min(n, 8 * (ngr * (blockIdx.x + 1) / gridDim.x));
    const int ntiles = (int)((r1 - r0 + kTileRows - 1) / kTileRows);
    const int nchunks = ntiles * cpt;

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
        // ---------------- producer: one lane issues every chunk
        if (lane == 0) {
            ptx::prefetch_tmap(&tm16);
            ptx::prefetch_tmap(&tm8);
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % nstages;
                // all 16 consumer warps free a stage at about the same time: probe without
                // suspending, so the refill does not wait for a wake-up
                if (c >= nstages && !ptx::mbar_wait_spin(ptx::smem_u32(&empty[s]), ((c / nstages) - 1) & 1, abortp))
                    break;
                const int tile = c / cpt, kc = c - tile * cpt;
                const int64_t row0 = r0 + int64_t(tile) * kTileRows;
                const bool eight = r1 - row0 <= 8;  // the CTA's last tile holds one 8-row group
                const uint32_t bar = ptx::smem_u32(&full[s]);
                ptx::mbar_arrive_expect_tx(bar, eight ? kStageBytes / 2 : kStageBytes);
                // x: 4-byte elements; a chunk starts at superblock 4 kc, i.e. element 144 kc
                ptx::tma_load_2d(ptx::smem_u32(stages + size_t(s) * kStageBytes), eight ? &tm8 : &tm16, 144 * kc,
                                 (int)row0, bar);
                ++issued;
            }
            int dummy = 0;  // no copy may still be writing shared memory when the CTA exits
            for (int c = max(0, issued - nstages); c < issued; ++c)
                ptx::mbar_wait(ptx::smem_u32(&full[c % nstages]), (c / nstages) & 1, &dummy);
        }
    } else {
        // ---------------- consumers: stage the activations, then fold the chunks
        ptx::grid_dependency_wait();
        {
            // one thread per (unit, column, half, 8-value group): 8 codes as fp16 in fragment
            // order, and per block its d8, s and -1024 sum(q) into the factor table
            const int nb32 = k / 32;
            const int total = Up * m * 8;
            // the loads of kBatch items are issued before the first is used (one memory round
            // trip per batch, not per item)
            constexpr int kBatch = 4;
            for (int i0 = tid; i0 < total; i0 += kBatch * kMmaWarps * 32) {
              uint32_t ld[kBatch][3];
#pragma unroll
              for (int j = 0; j < kBatch; ++j) {
                const int i = i0 + j * kMmaWarps * 32;
                ld[j][0] = ld[j][1] = ld[j][2] = 0u;
                const int half = (i >> 2) & 1, uc = i >> 3, u = uc / m, c = uc - u * m;
                const int b = 2 * u + half;
                if (i < total && b < nb32) {
                    const uint8_t *blk = xq + (size_t(c) * nb32 + b) * kQ81Bytes;
                    ld[j][0] = *reinterpret_cast<const uint32_t *>(blk);
                    ld[j][1] = *reinterpret_cast<const uint32_t *>(blk + 4 + 8 * (i & 3));
                    ld[j][2] = *reinterpret_cast<const uint32_t *>(blk + 8 + 8 * (i & 3));
                }
              }
#pragma unroll
              for (int j = 0; j < kBatch; ++j) {
                const int i = i0 + j * kMmaWarps * 32;
                if (i >= total) break;  // warp-uniform: total is a multiple of 128
                const int t4 = i & 3, half = (i >> 2) & 1;
                const int uc = i >> 3, u = uc / m, c = uc - u * m;
                const uint32_t dsw = ld[j][0], lo = ld[j][1], hi = ld[j][2];
                int sum = 0;
                uint32_t h[4];
                const uint32_t wv[2] = {lo, hi};
#pragma unroll
                for (int p = 0; p < 2; ++p) {  // codes 4p .. 4p+3 of the group -> (0, 2), (1, 3)
                    const int q0 = (int8_t)(wv[p] & 0xff), q1 = (int8_t)((wv[p] >> 8) & 0xff);
                    const int q2 = (int8_t)((wv[p] >> 16) & 0xff), q3 = (int8_t)(wv[p] >> 24);
                    sum += q0 + q1 + q2 + q3;
                    h[2 * p] = h2bits(__halves2half2(__int2half_rn(q0), __int2half_rn(q2)));
                    h[2 * p + 1] = h2bits(__halves2half2(__int2half_rn(q1), __int2half_rn(q3)));
                }
                uint4 *dst = reinterpret_cast<uint4 *>(xh + (size_t(u) * m + c) * 128);
                dst[xh_chunk(c, 4 * half + t4)] = make_uint4(h[0], h[1], h[2], h[3]);
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if (t4 == 0) {
                    // pair p = c / 2: float4 0 {d8 lo c0, d8 lo c1, d8 hi c0, d8 hi c1}, 1 the same
                    // for s, 2 for -1024 sum(q)
                    float *f = reinterpret_cast<float *>(fac + size_t(u) * kFacBytes + (c >> 1) * 48);
                    const int e = 2 * half + (c & 1);
                    f[e] = half_lo(dsw);
                    f[4 + e] = half_hi(dsw);
                    f[8 + e] = -1024.0f * (float)sum;
                }
              }
            }
            // the factors of columns m..7 are never read (their B fragments are zero), except
            // in the odd pair of an odd m: clear that column
            if (m & 1) {
                for (int i = tid; i < Up * 2; i += kMmaWarps * 32) {
                    float *f = reinterpret_cast<float *>(fac + size_t(i >> 1) * kFacBytes + (m >> 1) * 48);
                    const int e = 2 * (i & 1) + 1;
                    f[e] = 0.f;
                    f[4 + e] = 0.f;
                    f[8 + e] = 0.f;
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kMmaWarps * 32) : "memory");

        const int g = lane >> 2, t = lane & 3;
        const int sbl = warp >> 2, c4 = warp & 3;  // this warp's unit: superblock sbl of the chunk, quarter c4
        const bool colv = g < m;                   // the B column this lane supplies
        float tot[4] = {0.f, 0.f, 0.f, 0.f};       // (row g, col 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % nstages;
            const int tile = c / cpt, kc = c - tile * cpt;
            const int64_t row0 = r0 + int64_t(tile) * kTileRows;
            const bool eight = r1 - row0 <= 8;
            // every consumer warp waits for every chunk, so a suspended wait's wake-up delay
            // would be paid once per chunk: probe without suspending
            if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait_spin(ptx::smem_u32(&full[s]), (c / nstages) & 1, abortp));
            const int sb = kc * kChunkSb + sbl;  // superblock within the row
            if (ok && sb < nsb) {
                // everything this warp needs from the stage, then the stage goes back
                const uint8_t *rg = stages + size_t(s) * kStageBytes + size_t(g) * kRowChunk + sbl * kQ4KBytes;
                const uint4 hd0 = *reinterpret_cast<const uint4 *>(rg);
                const uint2 wq0 = *reinterpret_cast<const uint2 *>(rg + 16 + 32 * c4 + 8 * t);
                uint4 hd1 = make_uint4(0u, 0u, 0u, 0u);
                uint2 wq1 = make_uint2(0u, 0u);
                if (!eight) {
                    const uint8_t *rg8 = rg + 8 * kRowChunk;
                    hd1 = *reinterpret_cast<const uint4 *>(rg8);
                    wq1 = *reinterpret_cast<const uint2 *>(rg8 + 16 + 32 * c4 + 8 * t);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty[s]));

                const int u = sb * 4 + c4;
                uint4 xl = make_uint4(0u, 0u, 0u, 0u), xhv = xl;
                if (colv) {
                    const uint4 *xc = reinterpret_cast<const uint4 *>(xh + (size_t(u) * m + g) * 128);
                    xl = xc[xh_chunk(g, t)];
                    xhv = xc[xh_chunk(g, 4 + t)];
                }
                const float4 *fp = reinterpret_cast<const float4 *>(fac + size_t(u) * kFacBytes + t * 48);
                const float4 f_d8 = fp[0], f_s8 = fp[1], f_z = fp[2];

                // A fragments: rows g (a0, a2) and g + 8 (a1, a3); word p of the lane's 8 bytes
                // gives K16 step p of both sub-blocks: bytes (0, 2) -> slots (2t, 2t+1), (1, 3) -> (2t+8, 2t+9)
                // the accumulators start at -1024 sum(q) of the column's 32-block
                float dlo[4] = {f_z.x, f_z.y, f_z.x, f_z.y};
                float dhi[4] = {f_z.z, f_z.w, f_z.z, f_z.w};
                {
                    const uint32_t w0[2] = {wq0.x, wq0.y}, w1[2] = {wq1.x, wq1.y};
                    const uint32_t bl[4] = {xl.x, xl.y, xl.z, xl.w}, bh[4] = {xhv.x, xhv.y, xhv.z, xhv.w};
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const uint32_t u0 = w0[p] >> 8, u1 = w1[p] >> 8;
                        mma_16816(dlo, nib_f16(w0[p], 0x000f000fu), nib_f16(w1[p], 0x000f000fu),
                                  nib_f16(u0, 0x000f000fu), nib_f16(u1, 0x000f000fu), bl[2 * p], bl[2 * p + 1]);
                        mma_16816(dhi, nib_f16(w0[p], 0x00f000f0u), nib_f16(w1[p], 0x00f000f0u),
                                  nib_f16(u0, 0x00f000f0u), nib_f16(u1, 0x00f000f0u), bh[2 * p], bh[2 * p + 1]);
                    }
                }
                // fold: y += d sc_lo d8_lo sumi_lo + d (sc_hi / 16) d8_hi (16 sumi_hi) - dmin (m_lo s_lo + m_hi s_hi)
                const uint4 hds[2] = {hd0, hd1};
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const uint4 hd = hds[rr];
                    int sc_lo, m_lo, sc_hi, m_hi;
                    q4k_scale_min(hd.y, hd.z, hd.w, 2 * c4, sc_lo, m_lo);
                    q4k_scale_min(hd.y, hd.z, hd.w, 2 * c4 + 1, sc_hi, m_hi);
                    const float d = half_lo(hd.x), dmin = half_hi(hd.x);
                    const float a_lo = d * (float)sc_lo, a_hi = d * (float)sc_hi * 0.0625f;
                    const float n_lo = -dmin * (float)m_lo, n_hi = -dmin * (float)m_hi;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int e = 2 * rr + cc;
                        const float d8l = cc ? f_d8.y : f_d8.x, d8h = cc ? f_d8.w : f_d8.z;
                        const float s8l = cc ? f_s8.y : f_s8.x, s8h = cc ? f_s8.w : f_s8.z;
                        float v = fmaf(a_lo * d8l, dlo[e], tot[e]);
                        v = fmaf(a_hi * d8h, dhi[e], v);
                        v = fmaf(n_lo, s8l, v);
                        tot[e] = fmaf(n_hi, s8h, v);
                    }
                }
            } else if (ok) {  // past the row's last superblock: nothing to fold
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty[s]));
            }
            if (kc == cpt - 1) {
                // end of a tile: the 16 warps' shares of the 16 x 8 results, summed through
                // shared memory (every consumer warp takes part, also after an abort, so the
                // named barriers always match)
                float4 *rb = red + (tile & 1) * (kMmaWarps * 32);
                rb[warp * 32 + lane] = make_float4(tot[0], tot[1], tot[2], tot[3]);
                asm volatile("bar.sync 1, %0;" ::"n"(kMmaWarps * 32) : "memory");
                if (tid < 128) {
                    const int row = tid >> 3, col = tid & 7;
                    const int hl = (row & 7) * 4 + (col >> 1), e = ((row >> 3) << 1) | (col & 1);
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < kMmaWarps; ++w) {
                        const float4 v = rb[w * 32 + hl];
                        acc += e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
                    }
                    const int64_t r = row0 + row;
                    if (ok && col < m && r < r1) y[int64_t(col) * n + r] = acc;
                }
                tot[0] = tot[1] = tot[2] = tot[3] = 0.f;
            }
        }
    }
    __syncthreads();
    if (tid == 0 && abort_flag && status) atomicExch(status, (int)QMM_ERR_DEVICE);
}

}  // namespace

bool gemv_mma_supported(qmm_type t, int64_t n, int64_t k, int64_t m) {
    if (t != QMM_Q4_K || n <= 0 || m < 2 || m > 8 || k % 256 != 0) return false;
    if (n >= (int64_t(1) << 31) || (k / 256) * int64_t(kQ4KBytes) / 4 >= (int64_t(1) << 31)) return false;
    return mma_stages(k, (int)m, size_t(device_smem_optin())) > 0;
}

cudaError_t launch_gemv_mma(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                            cudaStream_t st) {
    if (!gemv_mma_supported(t, n, k, m)) return cudaErrorNotSupported;
    const int nstages = mma_stages(k, (int)m, size_t(device_smem_optin()));
    const int64_t row_bytes = (k / 256) * kQ4KBytes;
    // the weight rows as a 2-D array of 4-byte elements; one box is 576 bytes (4
    // superblocks) of 16 or 8 rows, zero-filled past the row end and past row n
    CUtensorMap tm16, tm8;
    if (!tc_make_map_2d(&tm16, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, W, uint64_t(row_bytes / 4), uint64_t(n),
                        uint64_t(row_bytes), kRowChunk / 4, kTileRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tc_make_map_2d(&tm8, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, W, uint64_t(row_bytes / 4), uint64_t(n),
                        uint64_t(row_bytes), kRowChunk / 4, kTileRows / 2, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const size_t smem = 1024 + size_t(nstages) * kStageBytes + mma_x_bytes(k, (int)m) + kRedBytes;
    cudaError_t e = ensure_smem(gemv_q4k_mma_kernel, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(device_sm_count(), (n + 7) / 8));
    return launch_pdl(gemv_q4k_mma_kernel, dim3((unsigned)grid), dim3(kMmaThreads), smem, st, tm16, tm8, n, (int)k,
                      (int)m, nstages, static_cast<const uint8_t *>(xq), y, static_cast<int *>(nullptr));
}

}  // namespace qmm
