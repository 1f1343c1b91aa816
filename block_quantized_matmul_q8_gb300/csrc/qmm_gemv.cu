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
#include "qmm_tc_ptx.cuh"

namespace qmm {

constexpr int kGemvThreads = 256;
constexpr int kUnitStride = 80;  // bytes per 64-value unit in the staged activations

__host__ __device__ inline int64_t gemv_units(int64_t k) { return (k + 63) / 64; }

size_t gemv_smem_bytes(int64_t k, int ncols) {
    const int64_t U = gemv_units(k);
    return size_t(ncols) * size_t(U) * (kUnitStride + 16);
}

// Fold one decoded unit into the NC column accumulators.
template <int NC>
__device__ __forceinline__ void fold_unit(const Unit &w, const uint8_t *xs, const float2 *xds, int U, int u,
                                          float (&acc)[NC]) {
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

// ---- activation staging.  A launch takes its NC activation columns either as q8_1
// blocks (xq) or as fp32 values (xf, k per column), which it then quantizes itself with
// the activation quantizer's arithmetic (the q8_1_* helpers), so that the staged bytes
// are the same either way and the fp32 call needs no separate quantizer launch
// ([MMQ] section "引言": activations are compressed to q8_1 on the device).
struct XIn {
    const uint8_t *xq;
    const float *xf;  // non-null: quantize these instead of reading xq
};

template <int NC>
__device__ __forceinline__ void stage_x(const XIn &x, int k, int U, uint8_t *xs, float2 *xds, int t, int nthreads) {
    const int nb32 = k / 32;
    const int total = NC * nb32;
    if (x.xf == nullptr) {
        for (int i = t; i < total; i += nthreads) {
            const int c = i / nb32, b = i - c * nb32;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(x.xq + (size_t(c) * nb32 + b) * kQ81Bytes);
            const uint32_t dsw = src[0];
            uint32_t *dst =
                reinterpret_cast<uint32_t *>(xs + (size_t(c) * U + (b >> 1)) * kUnitStride + 32 * (b & 1));
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = src[1 + j];
            xds[size_t(c) * 2 * U + b] = make_float2(half_lo(dsw), half_hi(dsw));
        }
        return;
    }
    // 4 lanes per 32-value block, 8 values (two 16-byte loads) per lane: a warp quantizes
    // 8 blocks per pass, and the loads of kBatch passes are issued before the first is
    // used.  Max and integer sum are exact in any order, d is the quantizer's correctly
    // rounded quotient, and every code is the quantizer's integer (q8_1_code_rcp), so the
    // staged bytes are the quantizer kernel's to the bit.
    constexpr int kBatch = 2;
    const int lane = t & 31, w = t >> 5, nw = nthreads >> 5, g = lane >> 2, l4 = lane & 3;
    const int ngroups = (total + 7) / 8;
    for (int i0 = w; i0 < ngroups; i0 += nw * kBatch) {
        float4 va[kBatch], vb[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int blk = 8 * (i0 + j * nw) + g;
            va[j] = vb[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (blk < total) {
                const int c = blk / nb32, b = blk - c * nb32;
                const float4 *src = reinterpret_cast<const float4 *>(x.xf + size_t(c) * k + 32 * b);
                va[j] = src[2 * l4];
                vb[j] = src[2 * l4 + 1];
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (i0 + j * nw >= ngroups) break;  // warp-uniform
            const int blk = 8 * (i0 + j * nw) + g;
            const float4 a4 = va[j], b4 = vb[j];
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
            if (blk < total) {
                const int c = blk / nb32, b = blk - c * nb32;
                const uint32_t lo = (uint32_t(q0) & 0xffu) | ((uint32_t(q1) & 0xffu) << 8) |
                                    ((uint32_t(q2) & 0xffu) << 16) | ((uint32_t(q3) & 0xffu) << 24);
                const uint32_t hi = (uint32_t(q4) & 0xffu) | ((uint32_t(q5) & 0xffu) << 8) |
                                    ((uint32_t(q6) & 0xffu) << 16) | ((uint32_t(q7) & 0xffu) << 24);
                reinterpret_cast<uint2 *>(xs + (size_t(c) * U + (b >> 1)) * kUnitStride + 32 * (b & 1))[l4] =
                    make_uint2(lo, hi);
                if (l4 == 0) {
                    const uint32_t dsw = q8_1_ds_word(d, S);
                    xds[size_t(c) * 2 * U + b] = make_float2(half_lo(dsw), half_hi(dsw));
                }
            }
        }
    }
}

// Each lane keeps CH units' loads in flight: all loads of a chunk are issued before
// the first of them is used.  The first chunk of a warp's first row pair is issued
// before the activations are staged, so HBM traffic starts at kernel entry.
template <int T, int NC>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const uint8_t *__restrict__ W, int64_t n, int k,
                                                            int64_t row_bytes, const XIn x,
                                                            float *__restrict__ y, int64_t y_ld) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int CH = kRawChunk<T>;
    const int U = (int)gemv_units(k);
    const int nb32 = k / 32;
    uint8_t *xs = smem;                                                             // [NC][U][80]
    float2 *xds = reinterpret_cast<float2 *>(smem + size_t(NC) * U * kUnitStride);  // [NC][2U]

    const int lane = threadIdx.x & 31;
    const int l16 = lane & 15;
    const int64_t npairs = (n + 1) / 2;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;

    Raw<T> raw[CH];
    auto issue = [&](int64_t pair, int base) {
        const int64_t r = 2 * pair + (lane >> 4);
        const uint8_t *row = W + r * row_bytes;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int u = base + 16 * c;
            if (r < n && u < U) load_raw(row, u, nb32, raw[c]);
        }
    };
    if (warp < npairs) issue(warp, l16);

    // ---- stage the activation columns (the first weight loads are already in flight)
    stage_x<NC>(x, k, U, xs, xds, threadIdx.x, blockDim.x);
    // an odd block count leaves the second half of the last unit unset: zero it
    if (nb32 & 1) {
        for (int i = threadIdx.x; i < NC * 8; i += blockDim.x) {
            const int c = i / 8, j = i % 8;
            reinterpret_cast<uint32_t *>(xs + (size_t(c) * U + U - 1) * kUnitStride + 32)[j] = 0u;
            if (j == 0) xds[size_t(c) * 2 * U + nb32] = make_float2(0.f, 0.f);
        }
    }
    __syncthreads();

    bool first = true;
    for (int64_t pair = warp; pair < npairs; pair += nwarp) {
        const int64_t r = 2 * pair + (lane >> 4);
        const bool valid = r < n;
        float acc[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] = 0.f;
        for (int base = l16; base < U; base += 16 * CH) {
            if (!first) issue(pair, base);
            first = false;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int u = base + 16 * c;
                if (valid && u < U) {
                    Unit w;
                    convert_raw(raw[c], u, w);
                    fold_unit<NC>(w, xs, xds, U, u, acc);
                }
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

// ---------------------------------------------------------------------------
// Bulk-copy variant for Q4_K (rows are whole multiples of 16 bytes): one persistent
// CTA per SM owns a contiguous range of rows and streams it through a ring of
// shared-memory stages with 1D bulk copies (cp.async.bulk, completion counted on an
// mbarrier), so every byte of W moves in large contiguous transfers and up to
// nstages chunks per SM are in flight (8 chunks of 8 rows, or 6, 4 or 3 where 8 do not
// fit next to the staged activations).  A dedicated producer warp issues the copies;
// four groups of 4 consumer warps (three for rings of 6 or 3 stages) take chunks in
// turn (a half-warp per row, lane l16 takes units l16, l16+16, ...).
constexpr int kTmaMaxStages = 8;
constexpr int kTmaGroups = 4;
constexpr int kTmaGroupWarps = 4;
constexpr int kTmaConsumerWarps = kTmaGroups * kTmaGroupWarps;
constexpr int kTmaThreads = (kTmaConsumerWarps + 1) * 32;
constexpr int kTmaChunkRows = 2 * kTmaGroupWarps;  // one row per half-warp
constexpr int64_t kTwoRowMinK = 8192;              // the long-row form of the Q4_K body from here
static_assert(kTmaMaxStages == 8 && kTmaGroups == 4, "ring depths and group splits below assume 8 stages, 4 groups");

// Consumer groups that take a ring of nstages stages (0: no valid split).  Chunk c goes
// to stage c % nstages and to group c % groups, and a wait on a stage's full barrier
// names only the parity of the phase it expects.  With nstages a multiple of the group
// count, a stage is always consumed by the same group, so the stage's previous chunk is
// that group's own, already folded, and the phase waited for is the barrier's current
// one.  Otherwise a group's first chunk may sit on a stage whose earlier chunk has not
// landed: the parity of that incomplete phase reads as complete, the group reads the
// stage early and its release throws the ring's counts off (3 stages for 4 groups
// faulted on the GPU); other depths leave the same race open whenever one chunk lands
// later than the chunk issued after it.
__host__ __device__ constexpr int gemv_ring_groups(int nstages) {
    return nstages <= 0 || nstages > kTmaMaxStages ? 0 : nstages % 4 == 0 ? 4 : nstages % 3 == 0 ? 3 : 0;
}

// Stages of kTmaChunkRows rows that fit next to the staged activations: the deepest
// ring of 8, 6, 4 or 3 stages (4 consumer groups for 8 and 4, 3 for 6 and 3), or 0.
int gemv_tma_stages(int64_t row_bytes, int64_t k, int ncols, size_t budget) {
    const size_t fixed = 1024 + gemv_smem_bytes(k, ncols);
    if (fixed >= budget || row_bytes <= 0) return 0;
    const int64_t st = int64_t(budget - fixed) / (int64_t(kTmaChunkRows) * row_bytes);
    return st >= 8 ? 8 : st >= 6 ? 6 : st >= 4 ? 4 : st >= 3 ? 3 : 0;
}


// Q4_K scales and mins of sub-blocks 2c and 2c+1 (c = 0..3) from the 12 packed bytes
// q[0..11] = s0 | s1 | s2 (GGUF 6-bit rule: for j < 4, sc = q[j] & 63, m = q[j+4] & 63;
// for j >= 4, sc = (q[j+4] & 15) | (q[j-4] >> 6) << 4, m = (q[j+4] >> 4) | (q[j] >> 6) << 4).
// A lane always takes the same c, so one byte permutation per word with a per-lane
// selector gathers the bytes of both sub-blocks, and per-lane masks finish the job:
//   sc pair = (P(s0, s2) & m1) | ((P(s0, s2) >> 18) & m2)
//   m  pair = ((P(s1, s2) >> sh) & m1) | ((P(s1, s2) >> 18) & m2)
// (low byte: sub-block 2c, high byte: 2c+1).
struct Q4KPairSel {
    uint32_t sel, m1, m2, sh;
};
__device__ __forceinline__ Q4KPairSel q4k_pair_sel(int c) {
    const uint32_t b = 2u * (c & 1);
    Q4KPairSel p;
    p.sel = c < 2 ? (b | (b + 1) << 4) : ((4 + b) | (5 + b) << 4 | b << 8 | (b + 1) << 12);
    p.m1 = c < 2 ? 0x3f3fu : 0x0f0fu;
    p.m2 = c < 2 ? 0u : 0x3030u;
    p.sh = c < 2 ? 0u : 4u;
    return p;
}
__device__ __forceinline__ void q4k_pair_scales(uint32_t s0, uint32_t s1, uint32_t s2, const Q4KPairSel &p, int &sc0,
                                                int &sc1, int &m0, int &m1) {
    const uint32_t a = __byte_perm(s0, s2, p.sel), q = __byte_perm(s1, s2, p.sel);
    const uint32_t sc = (a & p.m1) | ((a >> 18) & p.m2);
    const uint32_t mn = ((q >> p.sh) & p.m1) | ((q >> 18) & p.m2);
    sc0 = sc & 0xff;
    sc1 = sc >> 8;
    m0 = mn & 0xff;
    m1 = mn >> 8;
}

// dp4a of unsigned bytes (a) with signed bytes (b).
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// One 64-value unit of two Q4_K rows against the staged activations, each unit's
// activation loads shared by both rows (the long-row form of the bulk-copy GEMV below).
// `two` false: the second row is past the end of the matrix and is not read.
template <int NC>
__device__ __forceinline__ void fold_q4k_unit2(const uint8_t *row0, const uint8_t *row1, bool two, int u, int c4,
                                               const Q4KPairSel &psel, const uint8_t *xs, const float2 *xds, int U,
                                               float (&acc0)[NC], float (&acc1)[NC]) {
    const uint8_t *b0 = row0 + (u >> 2) * kQ4KBytes;
    const uint8_t *b1 = row1 + (u >> 2) * kQ4KBytes;
    const uint4 hd0 = *reinterpret_cast<const uint4 *>(b0);
    const uint4 qa0 = *reinterpret_cast<const uint4 *>(b0 + 16 + 32 * c4);
    const uint4 qb0 = *reinterpret_cast<const uint4 *>(b0 + 32 + 32 * c4);
    uint4 hd1 = make_uint4(0u, 0u, 0u, 0u), qa1 = hd1, qb1 = hd1;
    if (two) {
        hd1 = *reinterpret_cast<const uint4 *>(b1);
        qa1 = *reinterpret_cast<const uint4 *>(b1 + 16 + 32 * c4);
        qb1 = *reinterpret_cast<const uint4 *>(b1 + 32 + 32 * c4);
    }
    const uint32_t w0[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qb0.x, qb0.y, qb0.z, qb0.w};
    const uint32_t w1[8] = {qa1.x, qa1.y, qa1.z, qa1.w, qb1.x, qb1.y, qb1.z, qb1.w};
    int sc0a, sc1a, m0a, m1a, sc0b, sc1b, m0b, m1b;
    q4k_pair_scales(hd0.y, hd0.z, hd0.w, psel, sc0a, sc1a, m0a, m1a);
    q4k_pair_scales(hd1.y, hd1.z, hd1.w, psel, sc0b, sc1b, m0b, m1b);
    const float da = half_lo(hd0.x), dmina = half_hi(hd0.x);
    const float db = half_lo(hd1.x), dminb = half_hi(hd1.x);
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) {
        const int4 *xv = reinterpret_cast<const int4 *>(xs + (size_t(cc) * U + u) * kUnitStride);
        const float4 ds = reinterpret_cast<const float4 *>(xds + size_t(cc) * 2 * U)[u];
        const int4 x0 = xv[0], x1 = xv[1], x2 = xv[2], x3 = xv[3];
        const int xl[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const int xh[8] = {x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
        int sloa = 0, shia = 0, slob = 0, shib = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            sloa = __dp4a((int)(w0[i] & 0x0f0f0f0fu), xl[i], sloa);
            slob = __dp4a((int)(w1[i] & 0x0f0f0f0fu), xl[i], slob);
            shia = dp4a_us(w0[i] & 0xf0f0f0f0u, xh[i], shia);  // high nibbles in place: 16 q
            shib = dp4a_us(w1[i] & 0xf0f0f0f0u, xh[i], shib);
        }
        shia >>= 4;
        shib >>= 4;
        float t = ds.x * (float)(sc0a * sloa);
        t = fmaf(ds.z, (float)(sc1a * shia), t);
        float mm = ds.y * (float)m0a;
        mm = fmaf(ds.w, (float)m1a, mm);
        acc0[cc] = fmaf(da, t, fmaf(-dmina, mm, acc0[cc]));
        t = ds.x * (float)(sc0b * slob);
        t = fmaf(ds.z, (float)(sc1b * shib), t);
        mm = ds.y * (float)m0b;
        mm = fmaf(ds.w, (float)m1b, mm);
        acc1[cc] = fmaf(db, t, fmaf(-dminb, mm, acc1[cc]));
    }
}

// The body of the bulk-copy GEMV for format T.  Q6_K rows (210-byte blocks) keep their
// chunks 16-byte aligned only from an even row on, so for Q6_K the CTAs' row ranges
// start on even rows (the host takes this kernel for Q6_K only when n is even or the
// rows are whole multiples of 16 bytes).
// GLU: fused gate/up with SwiGLU ([MMQ] sections "「分专家」与「整批」之间: host 侧的代价"
// and "输出端: 写回与 scale 修正": gate and up rows interleaved so that one thread holds
// both dots of an output, no stream-K).  n counts outputs; W is the gate and W2 the up
// weight, each [n] rows, or with W2 == nullptr W holds both interleaved (2n rows: gate j
// at 2j, up j at 2j+1, as qmm_repack_glu writes them).  A chunk holds 4 outputs as 8
// staged rows: the 4 gate rows and then the 4 up rows, a bulk copy each (one copy per row
// took 19.5 us for 2 x 14336 x 4096 at one column), or the interleaved pairs in one copy;
// the two half-warps of a warp fold one pair and lane 0 writes silu(gate) * up.
// kTwoRows (Q4_K, not GLU): each warp folds its two rows of a chunk together, lanes
// taking units lane + 32 j, so every unit's staged activations are read once for both
// rows; chosen by the host for long rows, where a CTA folds few chunks.
template <int T, int NC, bool GLU = false, bool kTwoRows = false, bool kRowPairs = false>
__device__ __forceinline__ void gemv_tma_body(const uint8_t *__restrict__ W, int64_t n, int k, int64_t row_bytes,
                                              int nstages, const XIn &x, float *__restrict__ y, int64_t y_ld,
                                              int *status, const uint8_t *__restrict__ W2 = nullptr) {
    constexpr int kCR = GLU ? kTmaChunkRows / 2 : kTmaChunkRows;  // outputs per chunk
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);  // stays a shared pointer
    __shared__ __align__(8) uint64_t full[kTmaMaxStages], empty[kTmaMaxStages];
    __shared__ int abort_flag;
    const int U = (int)gemv_units(k);
    const int nb32 = k / 32;
    const size_t stage_bytes = size_t(kTmaChunkRows) * size_t(row_bytes);
    uint8_t *stages = smem;
    uint8_t *xs = smem + nstages * stage_bytes;
    float2 *xds = reinterpret_cast<float2 *>(xs + size_t(NC) * U * kUnitStride);

    const int64_t ra = (T == QMM_Q6_K && (row_bytes & 15)) ? 2 : 1;  // row granularity of the split
    const int64_t nr = (n + ra - 1) / ra;
    const int64_t r0 = ra * (nr * blockIdx.x / gridDim.x);
    const int64_t r1 = min(n, ra * (nr * (blockIdx.x + 1) / gridDim.x));
    const int nchunks = (int)((r1 - r0 + kCR - 1) / kCR);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, l16 = lane & 15;
    volatile int *abortp = &abort_flag;
    // the ring protocol needs whole rounds of stages (gemv_ring_groups): any other depth
    // is refused before a copy is issued
    // kRowPairs: consumer groups of 2 warps (8 groups for a ring of 8 stages), each half-warp
    // folding two rows of a chunk with every unit's staged activations read once for both
    constexpr int kGW = kRowPairs ? 2 : kTmaGroupWarps;  // warps per consumer group
    const int ngroups = kRowPairs ? (nstages == kTmaMaxStages ? kTmaConsumerWarps / kGW : 0) : gemv_ring_groups(nstages);
    if (ngroups == 0) {
        if (tid == 0 && status) atomicExch(status, (int)QMM_ERR_DEVICE);
        return;
    }

    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < nstages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty[s]), kGW);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();

    // The weights are never written by the kernels of this library, so their copies may
    // start before the preceding kernel in the stream (typically the activation
    // quantizer) has finished; everything else waits for it.
    ptx::grid_launch_dependents();
    if (warp == kTmaConsumerWarps) {
        // ---------------- producer warp: one lane issues every copy
        if (lane == 0) {
            int issued = 0;
            const int stagger = nchunks >= 6 ? 2 : 1;  // the chunk after which the copy lane waits
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % nstages;
                if (c >= nstages && !ptx::mbar_wait(ptx::smem_u32(&empty[s]), ((c / nstages) - 1) & 1, abortp))
                    break;
                const int64_t a = r0 + int64_t(c) * kCR;
                const int64_t b = min(r1, a + kCR);
                const uint32_t bar = ptx::smem_u32(&full[s]);
                if constexpr (GLU) {
                    ptx::mbar_arrive_expect_tx(bar, uint32_t(2 * (b - a) * row_bytes));
                    if (!W2)  // interleaved gate/up rows (qmm_repack_glu): the chunk is one block
                        ptx::bulk_g2s(ptx::smem_u32(stages + s * stage_bytes), W + 2 * a * row_bytes,
                                      uint32_t(2 * (b - a) * row_bytes), bar);
                    if (W2) {  // two tensors: the chunk's gate rows, then its up rows, a copy each
                        const uint32_t dst = ptx::smem_u32(stages + s * stage_bytes);
                        ptx::bulk_g2s(dst, W + a * row_bytes, uint32_t((b - a) * row_bytes), bar);
                        ptx::bulk_g2s(dst + uint32_t(kCR * row_bytes), W2 + a * row_bytes, uint32_t((b - a) * row_bytes),
                                      bar);
                    }
                } else {
                    const uint32_t bytes = uint32_t((b - a) * row_bytes);
                    ptx::mbar_arrive_expect_tx(bar, bytes);
                    ptx::bulk_g2s(ptx::smem_u32(stages + s * stage_bytes), W + a * row_bytes, bytes, bar);
                }
                ++issued;
                // Every CTA asks for its first chunks and lets them land before asking for
                // the rest: requested all at once, the first chunks of all CTAs queue behind
                // everyone's later stages and the consumers start about 3 us late (measured:
                // one launch of the decode GEMV 12.1 -> 10.5 us).  Three first chunks where a
                // CTA has 6 or more (17408 x 5120 from q8_1 9.5 -> 9.1 us, 2-4 columns 3-5%
                // faster), two where it has fewer (4096 x 14336 and Q8_0 5120 x 5120 lose 7-8%
                // with three).
                if (c == stagger && nchunks > stagger + 1 &&
                    !ptx::mbar_wait(ptx::smem_u32(&full[stagger]), 0, abortp))
                    break;
            }
            // no copy may still be writing shared memory when the CTA exits: wait for the
            // last nstages issued chunks (each wait bounded, independent of the abort flag)
            int dummy = 0;
            for (int c = max(0, issued - nstages); c < issued; ++c)
                ptx::mbar_wait(ptx::smem_u32(&full[c % nstages]), (c / nstages) & 1, &dummy);
        }
    } else {
        // ---------------- consumers: stage the activations, then fold the chunks
        ptx::grid_dependency_wait();
        stage_x<NC>(x, k, U, xs, xds, tid, kTmaConsumerWarps * 32);
        asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumerWarps * 32) : "memory");

        const int grp = warp / kGW, gw = warp % kGW;
        // staged row of this half-warp: GLU from two tensors stages the chunk's gate rows
        // and then its up rows, so output gw's pair is rows gw and kCR + gw; interleaved
        // (and plain) chunks hold row pairs side by side
        const int rr = (GLU && W2) ? ((lane >> 4) ? kCR + gw : gw) : 2 * gw + (lane >> 4);
        const int c4 = l16 & 3;               // qs chunk of every unit this lane takes (Q4_K)
        const Q4KPairSel psel = q4k_pair_sel(c4);
        for (int c = grp; grp < ngroups && c < nchunks; c += ngroups) {
            const int s = c % nstages;
            if (!ptx::mbar_wait(ptx::smem_u32(&full[s]), (c / nstages) & 1, abortp)) break;
            const int64_t a = r0 + int64_t(c) * kCR;
            const bool valid = GLU ? a + gw < r1 : a + rr < r1;  // GLU: warp gw folds output a + gw
            float acc[NC];
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) acc[cc] = 0.f;
            if constexpr (T == QMM_Q4_K && !GLU && kRowPairs) {
                // this half-warp's rows ra, ra + 1 of the chunk, lane l16 taking units l16 + 16 j of
                // both: half the activation loads per weight row of the one-row form
                const int ra = 2 * (2 * gw + (lane >> 4));
                float acc1[NC];
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) acc1[cc] = 0.f;
                if (a + ra < r1) {
                    const uint8_t *row0 = stages + s * stage_bytes + size_t(ra) * row_bytes;
                    for (int u = l16; u < U; u += 16)
                        fold_q4k_unit2<NC>(row0, row0 + row_bytes, a + ra + 1 < r1, u, c4, psel, xs, xds, U, acc, acc1);
                }
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    float v0 = acc[cc], v1 = acc1[cc];
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) {
                        v0 += __shfl_xor_sync(0xffffffffu, v0, o);
                        v1 += __shfl_xor_sync(0xffffffffu, v1, o);
                    }
                    acc[cc] = v0;
                    acc1[cc] = v1;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty[s]));  // the stage is read: free it first
                if (l16 == 0) {
#pragma unroll
                    for (int cc = 0; cc < NC; ++cc) {
                        if (a + ra < r1) y[cc * y_ld + a + ra] = acc[cc];
                        if (a + ra + 1 < r1) y[cc * y_ld + a + ra + 1] = acc1[cc];
                    }
                }
                continue;
            }
            if constexpr (T == QMM_Q4_K && !GLU && kTwoRows) {
                const int r0w = 2 * gw;  // this warp's rows r0w, r0w + 1 of the chunk
                float acc1[NC];
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) acc1[cc] = 0.f;
                if (a + r0w < r1) {
                    const uint8_t *row0 = stages + s * stage_bytes + size_t(r0w) * row_bytes;
                    const int c4l = lane & 3;  // units lane + 32 j all take qs chunk lane % 4
                    const Q4KPairSel pl = q4k_pair_sel(c4l);
                    for (int u = lane; u < U; u += 32)
                        fold_q4k_unit2<NC>(row0, row0 + row_bytes, a + r0w + 1 < r1, u, c4l, pl, xs, xds, U, acc,
                                           acc1);
                }
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    float v0 = acc[cc], v1 = acc1[cc];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) {
                        v0 += __shfl_xor_sync(0xffffffffu, v0, o);
                        v1 += __shfl_xor_sync(0xffffffffu, v1, o);
                    }
                    acc[cc] = v0;
                    acc1[cc] = v1;
                }
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(ptx::smem_u32(&empty[s]));  // the stage is read: free it first
#pragma unroll
                    for (int cc = 0; cc < NC; ++cc) {
                        if (a + r0w < r1) y[cc * y_ld + a + r0w] = acc[cc];
                        if (a + r0w + 1 < r1) y[cc * y_ld + a + r0w + 1] = acc1[cc];
                    }
                }
                continue;
            }
            if (T == QMM_Q4_K && valid) {
                const uint8_t *row = stages + s * stage_bytes + size_t(rr) * row_bytes;
                for (int u = l16; u < U; u += 16) {
                    const uint8_t *blk = row + (u >> 2) * kQ4KBytes;
                    const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
                    const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c4);
                    const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c4);
                    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                    int sc0, sc1, m0, m1;
                    q4k_pair_scales(hd.y, hd.z, hd.w, psel, sc0, sc1, m0, m1);
                    const float d = half_lo(hd.x), dmin = half_hi(hd.x);
#pragma unroll
                    for (int cc = 0; cc < NC; ++cc) {
                        const int4 *xv = reinterpret_cast<const int4 *>(xs + (size_t(cc) * U + u) * kUnitStride);
                        const float4 ds = reinterpret_cast<const float4 *>(xds + size_t(cc) * 2 * U)[u];
                        const int4 x0 = xv[0], x1 = xv[1], x2 = xv[2], x3 = xv[3];
                        int slo = __dp4a((int)(w[0] & 0x0f0f0f0fu), x0.x, 0);
                        slo = __dp4a((int)(w[1] & 0x0f0f0f0fu), x0.y, slo);
                        slo = __dp4a((int)(w[2] & 0x0f0f0f0fu), x0.z, slo);
                        slo = __dp4a((int)(w[3] & 0x0f0f0f0fu), x0.w, slo);
                        slo = __dp4a((int)(w[4] & 0x0f0f0f0fu), x1.x, slo);
                        slo = __dp4a((int)(w[5] & 0x0f0f0f0fu), x1.y, slo);
                        slo = __dp4a((int)(w[6] & 0x0f0f0f0fu), x1.z, slo);
                        slo = __dp4a((int)(w[7] & 0x0f0f0f0fu), x1.w, slo);
                        // high nibbles in place: bytes & 0xF0 are 16 q, so the dot is 16 times
                        // the wanted one and the shift divides it exactly
                        int shi = dp4a_us(w[0] & 0xf0f0f0f0u, x2.x, 0);
                        shi = dp4a_us(w[1] & 0xf0f0f0f0u, x2.y, shi);
                        shi = dp4a_us(w[2] & 0xf0f0f0f0u, x2.z, shi);
                        shi = dp4a_us(w[3] & 0xf0f0f0f0u, x2.w, shi);
                        shi = dp4a_us(w[4] & 0xf0f0f0f0u, x3.x, shi);
                        shi = dp4a_us(w[5] & 0xf0f0f0f0u, x3.y, shi);
                        shi = dp4a_us(w[6] & 0xf0f0f0f0u, x3.z, shi);
                        shi = dp4a_us(w[7] & 0xf0f0f0f0u, x3.w, shi);
                        shi >>= 4;
                        // exact int32 sub-block dots times the 6-bit scales, folded in fp32
                        float t = ds.x * (float)(sc0 * slo);
                        t = fmaf(ds.z, (float)(sc1 * shi), t);
                        float mm = ds.y * (float)m0;
                        mm = fmaf(ds.w, (float)m1, mm);
                        acc[cc] = fmaf(d, t, fmaf(-dmin, mm, acc[cc]));
                    }
                }
            }
            if (T != QMM_Q4_K && valid) {
                // Q6_K / Q8_0: the two-phase decode of the direct kernel, reading the staged row
                const uint8_t *row = stages + s * stage_bytes + size_t(rr) * row_bytes;
                for (int u = l16; u < U; u += 16) {
                    Raw<T> raw;
                    load_raw<LdShared>(row, u, nb32, raw);
                    Unit w;
                    convert_raw(raw, u, w);
                    fold_unit<NC>(w, xs, xds, U, u, acc);
                }
            }
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                float v = acc[cc];
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                acc[cc] = v;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty[s]));  // the stage is read: free it first
            if constexpr (GLU) {
                // lane 0 holds the gate dot, lane 16 the up dot of the same output
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    const float up = __shfl_xor_sync(0xffffffffu, acc[cc], 16);
                    const float g = acc[cc];
                    if (valid && lane == 0) y[cc * y_ld + a + gw] = g / (1.0f + expf(-g)) * up;
                }
            } else if (valid && l16 == 0) {
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) y[cc * y_ld + a + rr] = acc[cc];
            }
        }
    }
    __syncthreads();
    if (tid == 0 && abort_flag && status) atomicExch(status, (int)QMM_ERR_DEVICE);
}

template <int NC>
__global__ void __launch_bounds__(kTmaThreads, 1) gemv_q4k_tma_kernel(const uint8_t *__restrict__ W, int64_t n,
                                                                      int k, int64_t row_bytes, int nstages,
                                                                      const XIn x, float *__restrict__ y,
                                                                      int64_t y_ld, int *status) {
    gemv_tma_body<QMM_Q4_K, NC>(W, n, k, row_bytes, nstages, x, y, y_ld, status);
}

// Long rows (k >= 8192) at one or two columns: the two-row fold
template <int NC>
__global__ void __launch_bounds__(kTmaThreads, 1) gemv_q4k_tma_pair_kernel(const uint8_t *__restrict__ W, int64_t n,
                                                                           int k, int64_t row_bytes, int nstages,
                                                                           const XIn x, float *__restrict__ y,
                                                                           int64_t y_ld, int *status) {
    gemv_tma_body<QMM_Q4_K, NC, false, false, true>(W, n, k, row_bytes, nstages, x, y, y_ld, status);
}
template <int NC>
__global__ void __launch_bounds__(kTmaThreads, 1) gemv_q4k_tma_long_kernel(const uint8_t *__restrict__ W, int64_t n,
                                                                           int k, int64_t row_bytes, int nstages,
                                                                           const XIn x, float *__restrict__ y,
                                                                           int64_t y_ld, int *status) {
    gemv_tma_body<QMM_Q4_K, NC, false, true>(W, n, k, row_bytes, nstages, x, y, y_ld, status);
}

template <int NC>
__global__ void __launch_bounds__(kTmaThreads, 1)
    gemv_q4k_glu_kernel(const uint8_t *__restrict__ Wg, const uint8_t *__restrict__ Wu, int64_t n, int k,
                        int64_t row_bytes, int nstages, const XIn x, float *__restrict__ y, int64_t y_ld,
                        int *status) {
    gemv_tma_body<QMM_Q4_K, NC, true>(Wg, n, k, row_bytes, nstages, x, y, y_ld, status, Wu);
}

template <int T, int NC>
__global__ void __launch_bounds__(kTmaThreads, 1) gemv_tma_kernel(const uint8_t *__restrict__ W, int64_t n, int k,
                                                                  int64_t row_bytes, int nstages, const XIn x,
                                                                  float *__restrict__ y, int64_t y_ld, int *status) {
    gemv_tma_body<T, NC>(W, n, k, row_bytes, nstages, x, y, y_ld, status);
}

// Expert-routed decode ([MMQ] section "派发路径": mul_mat_id with a handful of pairs):
// one GEMV per (token, slot) pair instead of 128-pair GEMM tiles that hold one pair
// each.  Grid (CTAs per pair, pairs); CTA (c, p) reads pair p's expert id on the device
// and streams its share of that expert's n rows with the bulk-copy body.  The ids are
// typically written by the preceding kernel (the router), so they are read after the
// grid dependency wait.  A pair whose id is outside [0, E) gets a zero output row and
// flags the call (QMM_ERR_IDS), as on the grouped paths: CTA (0, 0) scans all the ids
// and writes the call's status word, so no reset precedes the launch.  Activation row
// of pair p: xq row p / x_div (x_div = top_k: shared by a token's slots; 1: one row per
// slot).
// GLU form (Wu != nullptr): W holds the experts' gate rows and Wu their up rows, and the
// pair's row of y gets silu(gate dot) * up dot ([MMQ] section "「分专家」与「整批」之间:
// host 侧的代价": the MoE FFN's gate and up products fused, the GLU applied after the dots).
template <int T, bool GLU = false>
__global__ void __launch_bounds__(kTmaThreads, 1)
    gemv_id_kernel(const uint8_t *__restrict__ W, int n_experts, int64_t n, int k, int64_t row_bytes, int nstages,
                   const uint8_t *__restrict__ xq, int64_t x_div, const int32_t *__restrict__ ids, int n_pairs,
                   float *__restrict__ y, int *status, const uint8_t *__restrict__ Wu = nullptr) {
    const int64_t p = blockIdx.y;
    ptx::grid_dependency_wait();
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 32) {
        bool bad = false;
        for (int i = threadIdx.x; i < n_pairs; i += 32) bad |= ids[i] < 0 || ids[i] >= n_experts;
        bad = __any_sync(0xffffffffu, bad);
        if (threadIdx.x == 0) status[0] = bad ? (int)QMM_ERR_IDS : (int)QMM_OK;
    }
    const int e = ids[p];
    float *yp = y + p * n;
    if (e < 0 || e >= n_experts) {
        const int64_t r0 = n * blockIdx.x / gridDim.x, r1 = n * (blockIdx.x + 1) / gridDim.x;
        for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) yp[r] = 0.f;
        return;
    }
    XIn x;
    x.xq = xq + (p / x_div) * int64_t(k / 32) * kQ81Bytes;
    x.xf = nullptr;
    if constexpr (GLU)
        gemv_tma_body<T, 1, true>(W + int64_t(e) * n * row_bytes, n, k, row_bytes, nstages, x, yp, n, status,
                                  Wu + int64_t(e) * n * row_bytes);
    else
        gemv_tma_body<T, 1>(W + int64_t(e) * n * row_bytes, n, k, row_bytes, nstages, x, yp, n, status);
}

// Rows that a bulk-copy GEMV can stream: every chunk must start on and span whole
// 16-byte units.  Q4_K rows always are; Q8_0 rows when k/32 is a multiple of 8; Q6_K
// rows when (k/256) * 210 is, or else from an even row on when n is even.
template <int T> static int64_t gemv_tma_row_bytes(int64_t n, int64_t k) {
    const int64_t rb = (k / block_elems(T)) * block_bytes(T);
    if (rb % 16 == 0) return rb;
    if (T == QMM_Q6_K && rb % 8 == 0 && n % 2 == 0) return rb;
    return 0;
}

int gemv_ring_stages(qmm_type t, int64_t n, int64_t k, int ncols, size_t budget) {
    int64_t rb = 0;
    switch (t) {
    case QMM_Q4_K: rb = gemv_tma_row_bytes<QMM_Q4_K>(n, k); break;
    case QMM_Q6_K: rb = gemv_tma_row_bytes<QMM_Q6_K>(n, k); break;
    case QMM_Q8_0: rb = gemv_tma_row_bytes<QMM_Q8_0>(n, k); break;
    case QMM_Q4_0: rb = gemv_tma_row_bytes<QMM_Q4_0>(n, k); break;
    case QMM_Q5_K: rb = gemv_tma_row_bytes<QMM_Q5_K>(n, k); break;
    default: return 0;
    }
    return rb > 0 ? gemv_tma_stages(rb, k, ncols, budget) : 0;
}

template <int T, int NC>
static cudaError_t launch_gemv_tma_nc(const void *W, int64_t n, int64_t k, XIn x, float *y, int64_t y_ld,
                                      int nstages, cudaStream_t st, int64_t stride) {
    const int64_t row_bytes = stride > 0 ? stride : gemv_tma_row_bytes<T>(n, k);
    const size_t smem = 1024 + size_t(nstages) * kTmaChunkRows * row_bytes + gemv_smem_bytes(k, NC);
    void (*kern)(const uint8_t *, int64_t, int, int64_t, int, const XIn, float *, int64_t, int *);
    if constexpr (T == QMM_Q4_K) {
        // From k = 8192 on at 1-2 columns, each warp folds its two rows together (lanes over
        // units: 4096 x 14336 at one column 13.7 -> 12.9 us).  Below, with the full ring of 8
        // stages and q8_1 input, each half-warp folds two rows over its 16 units (17408 x 5120:
        // 10.27 -> 10.11 us at 1 column, 12.8 -> 12.5 at 2, 23.3 -> 20.2 at 5); from 6 columns
        // on the row pairs spill and the MMA GEMV takes over.  With the fp32 row quantized in
        // the prologue, the row pairs win where a CTA has at most 96 rows (14336 x 4096: 7.50 ->
        // 7.07 us, 4096 x 5120: 4.77 -> 4.53, 2048 x 4096: 3.50 -> 3.42) and the one-row form
        // where it has more (17408 x 5120, 115 rows: 9.81 against 10.00 us).  Both forms sum
        // each row in the same order, so the choice does not change y.
        const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(device_sm_count(), (n + 1) / 2));
        const bool pairs = nstages == kTmaMaxStages && NC <= 5 &&
                           (x.xf == nullptr || (NC == 1 && n <= 96 * grid));
        if constexpr (NC <= 2)
            kern = k >= kTwoRowMinK ? gemv_q4k_tma_long_kernel<NC>
                   : pairs          ? gemv_q4k_tma_pair_kernel<NC>
                                    : gemv_q4k_tma_kernel<NC>;
        else
            kern = pairs ? gemv_q4k_tma_pair_kernel<NC> : gemv_q4k_tma_kernel<NC>;
    } else {
        kern = gemv_tma_kernel<T, NC>;
    }
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(device_sm_count(), (n + 1) / 2));  // as above
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kTmaThreads), smem, st, static_cast<const uint8_t *>(W), n,
                      (int)k, row_bytes, nstages, x, y, y_ld, static_cast<int *>(nullptr));
}

template <int NC>
static cudaError_t launch_gemv_glu_nc(const void *Wg, const void *Wu, int64_t n, int64_t k, XIn x, float *y,
                                      int nstages, cudaStream_t st) {
    const int64_t row_bytes = gemv_tma_row_bytes<QMM_Q4_K>(n, k);
    const size_t smem = 1024 + size_t(nstages) * kTmaChunkRows * row_bytes + gemv_smem_bytes(k, NC);
    auto kern = gemv_q4k_glu_kernel<NC>;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(device_sm_count(), n));
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kTmaThreads), smem, st, static_cast<const uint8_t *>(Wg),
                      static_cast<const uint8_t *>(Wu), n, (int)k, row_bytes, nstages, x, y, n,
                      static_cast<int *>(nullptr));
}

template <int T>
static cudaError_t launch_gemv_id_t(const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                                    int64_t x_div, const int32_t *ids, int64_t n_pairs, float *y, int *status,
                                    cudaStream_t st) {
    const int64_t row_bytes = gemv_tma_row_bytes<T>(n, k);
    const int nstages = row_bytes > 0 ? gemv_tma_stages(row_bytes, k, 1, size_t(device_smem_optin())) : 0;
    if (nstages <= 0) return cudaErrorNotSupported;
    const size_t smem = 1024 + size_t(nstages) * kTmaChunkRows * row_bytes + gemv_smem_bytes(k, 1);
    auto kern = gemv_id_kernel<T>;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    // enough CTAs per pair to cover the SMs once, at least 2 rows each
    const int64_t per_pair = std::max<int64_t>(
        1, std::min<int64_t>((n + 1) / 2, (device_sm_count() + n_pairs - 1) / n_pairs));
    return launch_pdl(kern, dim3((unsigned)per_pair, (unsigned)n_pairs), dim3(kTmaThreads), smem, st,
                      static_cast<const uint8_t *>(W), (int)n_experts, n, (int)k, row_bytes, nstages,
                      static_cast<const uint8_t *>(xq), x_div, ids, (int)n_pairs, y, status,
                      static_cast<const uint8_t *>(nullptr));
}

template <int T, int NC>
static cudaError_t launch_gemv_nc(const void *W, int64_t n, int64_t k, XIn x, float *y, int64_t y_ld,
                                  cudaStream_t st, int64_t stride) {
    const size_t smem = gemv_smem_bytes(k, NC);
    auto kern = gemv_kernel<T, NC>;
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem(kern, smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemvThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t npairs = (n + 1) / 2;
    const int64_t need = (npairs + kGemvThreads / 32 - 1) / (kGemvThreads / 32);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(need, int64_t(device_sm_count()) * per_sm));
    const int64_t row_bytes = stride > 0 ? stride : int64_t(k / block_elems(T)) * block_bytes(T);
    kern<<<(unsigned)grid, kGemvThreads, smem, st>>>(static_cast<const uint8_t *>(W), n, (int)k, row_bytes, x, y,
                                                     y_ld);
    return cudaGetLastError();
}

template <int T>
static cudaError_t launch_gemv_t(const void *W, int64_t n, int64_t k, const void *xq, const float *xf, int64_t m,
                                 float *y, cudaStream_t st, int64_t stride) {
    const size_t xrow = size_t(k / 32) * kQ81Bytes;
    const size_t budget = size_t(device_smem_optin());
    int64_t c0 = 0;
    while (c0 < m) {
        int nc = (int)std::min<int64_t>(8, m - c0);
        while (nc > 1 && gemv_smem_bytes(k, nc) > budget) --nc;
        if (gemv_smem_bytes(k, nc) > budget) return cudaErrorInvalidValue;
        cudaError_t e;
        XIn xc;
        xc.xq = xf ? nullptr : static_cast<const uint8_t *>(xq) + c0 * xrow;
        xc.xf = xf ? xf + c0 * k : nullptr;
        float *yc = y + c0 * n;
        // rows padded to a 16-byte multiple (stride > 0) always stream in whole units
        const int64_t trb = stride > 0 ? stride : gemv_tma_row_bytes<T>(n, k);
        const int nst = trb > 0 ? gemv_tma_stages(trb, k, nc, budget) : 0;
        if (nst > 0 && gemv_tma_enabled()) {
            switch (nc) {
            case 1: e = launch_gemv_tma_nc<T, 1>(W, n, k, xc, yc, n, nst, st, stride); break;
            case 2: e = launch_gemv_tma_nc<T, 2>(W, n, k, xc, yc, n, nst, st, stride); break;
            case 3: e = launch_gemv_tma_nc<T, 3>(W, n, k, xc, yc, n, nst, st, stride); break;
            case 4: e = launch_gemv_tma_nc<T, 4>(W, n, k, xc, yc, n, nst, st, stride); break;
            case 5: e = launch_gemv_tma_nc<T, 5>(W, n, k, xc, yc, n, nst, st, stride); break;
            case 6: e = launch_gemv_tma_nc<T, 6>(W, n, k, xc, yc, n, nst, st, stride); break;
            case 7: e = launch_gemv_tma_nc<T, 7>(W, n, k, xc, yc, n, nst, st, stride); break;
            default: e = launch_gemv_tma_nc<T, 8>(W, n, k, xc, yc, n, nst, st, stride); break;
            }
            if (e != cudaSuccess) return e;
            c0 += nc;
            continue;
        }
        switch (nc) {
        case 1: e = launch_gemv_nc<T, 1>(W, n, k, xc, yc, n, st, stride); break;
        case 2: e = launch_gemv_nc<T, 2>(W, n, k, xc, yc, n, st, stride); break;
        case 3: e = launch_gemv_nc<T, 3>(W, n, k, xc, yc, n, st, stride); break;
        case 4: e = launch_gemv_nc<T, 4>(W, n, k, xc, yc, n, st, stride); break;
        case 5: e = launch_gemv_nc<T, 5>(W, n, k, xc, yc, n, st, stride); break;
        case 6: e = launch_gemv_nc<T, 6>(W, n, k, xc, yc, n, st, stride); break;
        case 7: e = launch_gemv_nc<T, 7>(W, n, k, xc, yc, n, st, stride); break;
        default: e = launch_gemv_nc<T, 8>(W, n, k, xc, yc, n, st, stride); break;
        }
        if (e != cudaSuccess) return e;
        c0 += nc;
    }
    return cudaSuccess;
}

cudaError_t launch_gemv(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, const float *xf, int64_t m,
                        float *y, cudaStream_t st, int64_t stride) {
    switch (t) {
    case QMM_Q4_K: return launch_gemv_t<QMM_Q4_K>(W, n, k, xq, xf, m, y, st, stride);
    case QMM_Q6_K: return launch_gemv_t<QMM_Q6_K>(W, n, k, xq, xf, m, y, st, stride);
    case QMM_Q8_0: return launch_gemv_t<QMM_Q8_0>(W, n, k, xq, xf, m, y, st, stride);
    case QMM_Q4_0: return launch_gemv_t<QMM_Q4_0>(W, n, k, xq, xf, m, y, st, stride);
    case QMM_Q5_K: return launch_gemv_t<QMM_Q5_K>(W, n, k, xq, xf, m, y, st, stride);
    }
    return cudaErrorInvalidValue;
}

bool gemv_glu_supported(qmm_type t, int64_t n, int64_t k, int64_t m) {
    if (t != QMM_Q4_K || n <= 0 || m <= 0 || m > 8 || k % 256 != 0) return false;
    const int64_t rb = gemv_tma_row_bytes<QMM_Q4_K>(n, k);
    const size_t budget = size_t(device_smem_optin());
    return gemv_tma_stages(rb, k, (int)std::min<int64_t>(m, 8), budget) > 0;
}

cudaError_t launch_gemv_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n, int64_t k, const void *xq,
                            int64_t m, float *y, cudaStream_t st) {
    if (!gemv_glu_supported(t, n, k, m)) return cudaErrorNotSupported;
    const int64_t rb = gemv_tma_row_bytes<QMM_Q4_K>(n, k);
    const int nst = gemv_tma_stages(rb, k, (int)m, size_t(device_smem_optin()));
    XIn x;
    x.xq = static_cast<const uint8_t *>(xq);
    x.xf = nullptr;
    switch (m) {
    case 1: return launch_gemv_glu_nc<1>(Wg, Wu, n, k, x, y, nst, st);
    case 2: return launch_gemv_glu_nc<2>(Wg, Wu, n, k, x, y, nst, st);
    case 3: return launch_gemv_glu_nc<3>(Wg, Wu, n, k, x, y, nst, st);
    case 4: return launch_gemv_glu_nc<4>(Wg, Wu, n, k, x, y, nst, st);
    case 5: return launch_gemv_glu_nc<5>(Wg, Wu, n, k, x, y, nst, st);
    case 6: return launch_gemv_glu_nc<6>(Wg, Wu, n, k, x, y, nst, st);
    case 7: return launch_gemv_glu_nc<7>(Wg, Wu, n, k, x, y, nst, st);
    default: return launch_gemv_glu_nc<8>(Wg, Wu, n, k, x, y, nst, st);
    }
}

bool gemv_id_supported(qmm_type t, int64_t n, int64_t k) {
    int64_t rb = 0;
    switch (t) {
    case QMM_Q4_K: rb = gemv_tma_row_bytes<QMM_Q4_K>(n, k); break;
    case QMM_Q6_K: rb = gemv_tma_row_bytes<QMM_Q6_K>(n, k); break;
    case QMM_Q8_0: rb = gemv_tma_row_bytes<QMM_Q8_0>(n, k); break;
    case QMM_Q4_0: rb = gemv_tma_row_bytes<QMM_Q4_0>(n, k); break;
    case QMM_Q5_K: rb = gemv_tma_row_bytes<QMM_Q5_K>(n, k); break;
    }
    return n > 0 && rb > 0 && gemv_tma_stages(rb, k, 1, size_t(device_smem_optin())) > 0;
}

cudaError_t launch_gemv_id(qmm_type t, const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                           int64_t x_div, const int32_t *ids, int64_t n_pairs, float *y, int *status,
                           cudaStream_t st) {
    switch (t) {
    case QMM_Q4_K: return launch_gemv_id_t<QMM_Q4_K>(W, n_experts, n, k, xq, x_div, ids, n_pairs, y, status, st);
    case QMM_Q6_K: return launch_gemv_id_t<QMM_Q6_K>(W, n_experts, n, k, xq, x_div, ids, n_pairs, y, status, st);
    case QMM_Q8_0: return launch_gemv_id_t<QMM_Q8_0>(W, n_experts, n, k, xq, x_div, ids, n_pairs, y, status, st);
    case QMM_Q4_0: return launch_gemv_id_t<QMM_Q4_0>(W, n_experts, n, k, xq, x_div, ids, n_pairs, y, status, st);
    case QMM_Q5_K: return launch_gemv_id_t<QMM_Q5_K>(W, n_experts, n, k, xq, x_div, ids, n_pairs, y, status, st);
    }
    return cudaErrorInvalidValue;
}

// The fused gate/up form of the decode MoE GEMV (Q4_K; both tensors [E][n] rows).
bool gemv_id_glu_supported(qmm_type t, int64_t n, int64_t k) { return gemv_glu_supported(t, n, k, 1); }

cudaError_t launch_gemv_id_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n_experts, int64_t n, int64_t k,
                               const void *xq, int64_t x_div, const int32_t *ids, int64_t n_pairs, float *y,
                               int *status, cudaStream_t st) {
    if (!gemv_id_glu_supported(t, n, k)) return cudaErrorNotSupported;
    const int64_t row_bytes = gemv_tma_row_bytes<QMM_Q4_K>(n, k);
    const int nstages = gemv_tma_stages(row_bytes, k, 1, size_t(device_smem_optin()));
    const size_t smem = 1024 + size_t(nstages) * kTmaChunkRows * row_bytes + gemv_smem_bytes(k, 1);
    auto kern = gemv_id_kernel<QMM_Q4_K, true>;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    // enough CTAs per pair to cover the SMs once, at least one output each
    const int64_t per_pair =
        std::max<int64_t>(1, std::min<int64_t>(n, (device_sm_count() + n_pairs - 1) / n_pairs));
    return launch_pdl(kern, dim3((unsigned)per_pair, (unsigned)n_pairs), dim3(kTmaThreads), smem, st,
                      static_cast<const uint8_t *>(Wg), (int)n_experts, n, (int)k, row_bytes, nstages,
                      static_cast<const uint8_t *>(xq), x_div, ids, (int)n_pairs, y, status,
                      static_cast<const uint8_t *>(Wu));
}

}  // namespace qmm
