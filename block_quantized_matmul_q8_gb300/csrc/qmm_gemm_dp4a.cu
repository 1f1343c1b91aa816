// qmm_gemm_dp4a.cu -- CUDA-core tiled GEMM on exact dp4a integer dots.
//
// Tile = 64 weight rows x 64 activation rows; K advances 256 values per stage
// ([MMQ] section "分块的骨架: I、J 与 K 三根轴": a block owns an I x J output tile
// and loads the weight tile once per K slab; section "加载端": the weight tile is
// unpacked to 8-bit codes plus per-sub-block scales at load time).  Each thread
// owns 4 x 4 outputs (rows tr+16i, activation rows tc+16j).  Per 32-block the
// thread forms exact int32 dots (two 16-wide quarters combined with the integer
// sub-scales) and folds them in fp32 with the block scales.
//
// The same kernel serves the expert-grouped path: a work item then names an
// expert and a run of up to 64 (token, slot) pairs of that expert in the sorted
// order; activation rows are gathered through the pair list and outputs scattered
// back to y[pair][:] ([MMQ] section "专家边界": expert_bounds, ids_dst and the
// scattered write-back).  CTAs are persistent and walk the work items in order.
#include <cuda_runtime.h>

#include <algorithm>

#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_moe.h"

namespace qmm {

constexpr int kTN = 64;       // weight rows per tile
constexpr int kTM = 64;       // activation rows per tile
constexpr int kStride = 68;   // words per smem row (64 + 4 pad)
constexpr int kThreads = 256;

struct DP4AGemmArgs {
    const uint8_t *W;
    int64_t n;
    int k;
    int64_t row_bytes;
    const uint8_t *xq;
    float *y;
    int64_t m;            // dense: activation rows
    // grouped (MoE) mode when tiles != nullptr
    const MoETile *tiles;
    const int32_t *ntiles;
    const int32_t *bounds;
    const int32_t *perm;
    int top_k;
    int64_t expert_stride;  // bytes between experts' weight matrices
};

struct DP4ASmem {
    int wq[kTN][kStride];
    int wisc[kTN][16];
    float wfd[kTN][8];
    float wfm[kTN][8];
    int xqs[kTM][kStride];
    float xd[kTM][8];
    float xs[kTM][8];
    int tok_x[kTM];
    int64_t tok_y[kTM];
};

template <int T>
__global__ void __launch_bounds__(kThreads, 2) gemm_dp4a_kernel(DP4AGemmArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    DP4ASmem &S = *reinterpret_cast<DP4ASmem *>(smem_raw);
    const int tid = threadIdx.x;
    const int tr = tid >> 4, tc = tid & 15;
    const int U = (a.k + 63) / 64;
    const int nb32 = a.k / 32;
    const int nstage = (a.k + 255) / 256;
    const int64_t row_tiles = (a.n + kTN - 1) / kTN;
    const bool grouped = a.tiles != nullptr;
    const int64_t col_items = grouped ? int64_t(*a.ntiles) : (a.m + kTM - 1) / kTM;
    const int64_t total = row_tiles * col_items;

    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int64_t ci = w / row_tiles;
        const int64_t rt = w - ci * row_tiles;
        const int64_t row0 = rt * kTN;
        const uint8_t *Wb = a.W;
        __syncthreads();  // previous item's smem reads are done
        if (tid < kTM) {
            int xr = -1;
            int64_t yr = -1;
            if (grouped) {
                const MoETile t = a.tiles[ci];
                const int idx = a.bounds[t.expert] + t.first + tid;
                if (t.first + tid < t.count) {
                    const int p = a.perm[idx];
                    xr = p / a.top_k;
                    yr = p;
                }
            } else {
                const int64_t tok = ci * kTM + tid;
                if (tok < a.m) {
                    xr = (int)tok;
                    yr = tok;
                }
            }
            S.tok_x[tid] = xr;
            S.tok_y[tid] = yr;
        }
        if (grouped) Wb += int64_t(a.tiles[ci].expert) * a.expert_stride;

        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

        for (int st = 0; st < nstage; ++st) {
            __syncthreads();  // tok_* visible; previous stage consumed
            {   // weight tile: thread -> (row, unit within the stage)
                const int r = tid >> 2, uu = tid & 3;
                const int u = 4 * st + uu;
                const int64_t row = row0 + r;
                Unit o;
                if (row < a.n && u < U) {
                    decode_unit<T>(Wb + row * a.row_bytes, u, nb32, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) o.q[i] = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) o.isc[i] = 0;
                    o.fd[0] = o.fd[1] = o.fm[0] = o.fm[1] = 0.f;
                }
                int4 *dst = reinterpret_cast<int4 *>(&S.wq[r][16 * uu]);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_int4(o.q[4 * i], o.q[4 * i + 1], o.q[4 * i + 2], o.q[4 * i + 3]);
                *reinterpret_cast<int4 *>(&S.wisc[r][4 * uu]) = make_int4(o.isc[0], o.isc[1], o.isc[2], o.isc[3]);
                S.wfd[r][2 * uu] = o.fd[0];
                S.wfd[r][2 * uu + 1] = o.fd[1];
                S.wfm[r][2 * uu] = o.fm[0];
                S.wfm[r][2 * uu + 1] = o.fm[1];
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // activation tile: 64 rows x 8 q8_1 blocks
                const int idx = tid + h * kThreads;
                const int j = idx >> 3, b = idx & 7;
                const int gb = 8 * st + b;
                const int xr = S.tok_x[j];
                int4 q0 = make_int4(0, 0, 0, 0), q1 = q0;
                float d = 0.f, s = 0.f;
                if (xr >= 0 && gb < nb32) {
                    const uint32_t *src = reinterpret_cast<const uint32_t *>(a.xq + (int64_t(xr) * nb32 + gb) * kQ81Bytes);
                    const uint32_t dsw = ldg4(src);
                    q0 = make_int4(ldg4(src + 1), ldg4(src + 2), ldg4(src + 3), ldg4(src + 4));
                    q1 = make_int4(ldg4(src + 5), ldg4(src + 6), ldg4(src + 7), ldg4(src + 8));
                    d = half_lo(dsw);
                    s = half_hi(dsw);
                }
                *reinterpret_cast<int4 *>(&S.xqs[j][8 * b]) = q0;
                *reinterpret_cast<int4 *>(&S.xqs[j][8 * b + 4]) = q1;
                S.xd[j][b] = d;
                S.xs[j][b] = s;
            }
            __syncthreads();
#pragma unroll 2
            for (int b = 0; b < 8; ++b) {
                int wv[4][8], xv[4][8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int4 p0 = *reinterpret_cast<const int4 *>(&S.wq[tr + 16 * i][8 * b]);
                    const int4 p1 = *reinterpret_cast<const int4 *>(&S.wq[tr + 16 * i][8 * b + 4]);
                    wv[i][0] = p0.x; wv[i][1] = p0.y; wv[i][2] = p0.z; wv[i][3] = p0.w;
                    wv[i][4] = p1.x; wv[i][5] = p1.y; wv[i][6] = p1.z; wv[i][7] = p1.w;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int4 p0 = *reinterpret_cast<const int4 *>(&S.xqs[tc + 16 * j][8 * b]);
                    const int4 p1 = *reinterpret_cast<const int4 *>(&S.xqs[tc + 16 * j][8 * b + 4]);
                    xv[j][0] = p0.x; xv[j][1] = p0.y; xv[j][2] = p0.z; xv[j][3] = p0.w;
                    xv[j][4] = p1.x; xv[j][5] = p1.y; xv[j][6] = p1.z; xv[j][7] = p1.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = tr + 16 * i;
                    const int isc0 = S.wisc[r][2 * b], isc1 = S.wisc[r][2 * b + 1];
                    const float fd = S.wfd[r][b], fm = S.wfm[r][b];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int t = tc + 16 * j;
                        int s0 = __dp4a(wv[i][0], xv[j][0], 0);
                        s0 = __dp4a(wv[i][1], xv[j][1], s0);
                        s0 = __dp4a(wv[i][2], xv[j][2], s0);
                        s0 = __dp4a(wv[i][3], xv[j][3], s0);
                        int s1 = __dp4a(wv[i][4], xv[j][4], 0);
                        s1 = __dp4a(wv[i][5], xv[j][5], s1);
                        s1 = __dp4a(wv[i][6], xv[j][6], s1);
                        s1 = __dp4a(wv[i][7], xv[j][7], s1);
                        const int blk = isc0 * s0 + isc1 * s1;
                        float v = acc[i][j];
                        v = fmaf(fd * S.xd[t][b], (float)blk, v);
                        v = fmaf(-fm, S.xs[t][b], v);
                        acc[i][j] = v;
                    }
                }
            }
        }
        // write-back (scattered through the pair list in grouped mode)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t yr = S.tok_y[tc + 16 * j];
            if (yr < 0) continue;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t row = row0 + tr + 16 * i;
                if (row < a.n) a.y[yr * a.n + row] = acc[i][j];
            }
        }
    }
}

template <int T>
static cudaError_t launch_dp4a_t(const DP4AGemmArgs &args, int64_t total_hint, cudaStream_t st) {
    const size_t smem = sizeof(DP4ASmem);
    auto kern = gemm_dp4a_kernel<T>;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm = std::max(per_sm, 1);
    int64_t grid = int64_t(device_sm_count()) * per_sm;
    if (total_hint > 0) grid = std::min(grid, total_hint);
    kern<<<(unsigned)std::max<int64_t>(grid, 1), kThreads, smem, st>>>(args);
    return cudaGetLastError();
}

static cudaError_t launch_dp4a(qmm_type t, const DP4AGemmArgs &args, int64_t total_hint, cudaStream_t st) {
    switch (t) {
    case QMM_Q4_K: return launch_dp4a_t<QMM_Q4_K>(args, total_hint, st);
    case QMM_Q6_K: return launch_dp4a_t<QMM_Q6_K>(args, total_hint, st);
    case QMM_Q8_0: return launch_dp4a_t<QMM_Q8_0>(args, total_hint, st);
    case QMM_Q4_0: return launch_dp4a_t<QMM_Q4_0>(args, total_hint, st);
    case QMM_Q5_K: return launch_dp4a_t<QMM_Q5_K>(args, total_hint, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_dp4a(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                             cudaStream_t st, int64_t stride) {
    DP4AGemmArgs a{};
    a.W = static_cast<const uint8_t *>(W);
    a.n = n;
    a.k = (int)k;
    a.row_bytes = stride > 0 ? stride : (k / block_elems(t)) * block_bytes(t);
    a.xq = static_cast<const uint8_t *>(xq);
    a.y = y;
    a.m = m;
    const int64_t total = ((n + kTN - 1) / kTN) * ((m + kTM - 1) / kTM);
    return launch_dp4a(t, a, total, st);
}

cudaError_t launch_gemm_dp4a_grouped(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, float *y,
                                     const MoETile *tiles, const int32_t *ntiles, const int32_t *bounds,
                                     const int32_t *perm, int top_k, cudaStream_t st) {
    DP4AGemmArgs a{};
    a.W = static_cast<const uint8_t *>(W);
    a.n = n;
    a.k = (int)k;
    a.row_bytes = (k / block_elems(t)) * block_bytes(t);
    a.xq = static_cast<const uint8_t *>(xq);
    a.y = y;
    a.m = 0;
    a.tiles = tiles;
    a.ntiles = ntiles;
    a.bounds = bounds;
    a.perm = perm;
    a.top_k = top_k;
    a.expert_stride = n * a.row_bytes;
    return launch_dp4a(t, a, 0, st);
}

}  // namespace qmm
