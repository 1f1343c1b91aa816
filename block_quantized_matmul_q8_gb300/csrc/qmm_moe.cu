// qmm_moe.cu -- expert-routed matmul: device bucketing and the grouped launch.
//
// [MMQ] sections "专家边界: 在 GPU 上做分段, 而不是在 host 上" and "MoE 的二次账":
// the (token, slot) pairs are sorted by expert on the device into expert_bounds and
// a pair list, so the host never reads the routing ids and the call stays
// asynchronous; each expert's pairs are cut into tiles of up to `tile_tokens`
// columns and every tile of every expert goes into one work list, which one
// persistent launch walks ([MMQ] section "局限与工程含义": merging the experts'
// small GEMMs into one schedule).
//
// Bucketing is a stable counting sort done by one CTA:
//   pass 1  counts per expert (shared-memory atomics) and invalid ids;
//   scan    bounds[e] (exclusive prefix), each expert's tile offset and the cold list,
//           one warp-wide scan over runs of consecutive experts;
//   pass 2  rounds of 1024 pairs; within a warp, lanes with the same expert find
//           each other with __match_any_sync, a per-(warp, expert) count table is
//           scanned over warps (one shuffle scan per expert), and each pair lands at
//           bounds[e] + (earlier rounds) + (earlier warps) + (earlier lanes).
//   Invalid pairs are appended after the valid ones; their output rows are zeroed.
#include <cuda_runtime.h>

#include <algorithm>

#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_moe.h"

namespace qmm {

constexpr int kBucketThreads = 1024;
constexpr int kBucketWarps = kBucketThreads / 32;

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

MoELayout moe_layout(int64_t n_pairs, int64_t n_experts, int tile_tokens, size_t gemm_bytes, size_t cold_bytes) {
    MoELayout L{};
    size_t off = 0;
    L.status = off;
    off += 256;
    L.bounds = off;
    off = align256(off + sizeof(int32_t) * size_t(n_experts + 1));
    L.perm = off;
    off = align256(off + sizeof(int32_t) * size_t(n_pairs));
    L.tiles = off;
    const int64_t max_tiles = n_pairs / tile_tokens + n_experts + 1;
    off = align256(off + sizeof(MoETile) * size_t(max_tiles));
    L.cold = off;
    off = align256(off + sizeof(int32_t) * size_t(n_experts));
    L.gemm = off;
    off = align256(off + gemm_bytes);
    L.cold_gemm = off;
    off = align256(off + cold_bytes);
    L.total = off;
    return L;
}

// Exclusive prefix sum over a warp of one int per lane; returns this lane's prefix and
// sets total to the sum of all lanes.
__device__ __forceinline__ int warp_exclusive_scan(int v, int lane, int &total) {
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - v;
}

__global__ void __launch_bounds__(kBucketThreads) moe_bucket_kernel(const int32_t *__restrict__ ids, int64_t n_pairs,
                                                                    int E, int tile_tokens, int cold_max,
                                                                    int32_t *status, int32_t *bounds, int32_t *perm,
                                                                    MoETile *tiles, int32_t *cold) {
    extern __shared__ __align__(16) int32_t sm[];
    const int Ep = (E & ~1) + 1;               // odd row stride of the per-warp tables: no bank conflicts
    int32_t *cnt = sm;                          // [E]   counts, then running bases
    int32_t *toff = cnt + E;                    // [E]   tile offsets
    int32_t *wcnt = toff + E;                   // [32][Ep] per-warp counts of a round
    int32_t *wofs = wcnt + kBucketWarps * Ep;   // [32][Ep] per-warp offsets of a round
    __shared__ int32_t s_bad, s_bad_pos;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int i = tid; i < E; i += kBucketThreads) cnt[i] = 0;
    for (int i = tid; i < kBucketWarps * Ep; i += kBucketThreads) wcnt[i] = 0;
    if (tid == 0) {
        s_bad = 0;
        s_bad_pos = 0;
    }
    __syncthreads();

    // pass 1: counts
    for (int64_t i = tid; i < n_pairs; i += kBucketThreads) {
        const int e = ids[i];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else atomicAdd(&s_bad, 1);
    }
    __syncthreads();

    // scan (warp 0, E <= kMaxExperts): lane l takes the experts [l * per, (l + 1) * per)
    // in order, so bounds, tile offsets and the cold list (experts with 1..cold_max
    // pairs, which get no tiles) all come out in expert order.
    if (warp == 0) {
        const int per = (E + 31) / 32, e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int pairs = 0, ntile = 0, ncold = 0;
        for (int e = e0; e < e1; ++e) {
            const int c = cnt[e];
            pairs += c;
            if (c > 0 && c <= cold_max) ++ncold;
            else ntile += (c + tile_tokens - 1) / tile_tokens;
        }
        int tot_pairs, tot_tiles, tot_cold;
        int run = warp_exclusive_scan(pairs, lane, tot_pairs);
        int trun = warp_exclusive_scan(ntile, lane, tot_tiles);
        int crun = warp_exclusive_scan(ncold, lane, tot_cold);
        for (int e = e0; e < e1; ++e) {
            const int c = cnt[e];
            bounds[e] = run;
            cnt[e] = run;  // running base for pass 2
            toff[e] = trun;
            run += c;
            if (c > 0 && c <= cold_max) cold[crun++] = e;
            else trun += (c + tile_tokens - 1) / tile_tokens;
        }
        if (lane == 0) {
            bounds[E] = tot_pairs;
            status[0] = s_bad ? (int32_t)QMM_ERR_IDS : (int32_t)QMM_OK;
            status[1] = tot_tiles;
            status[2] = s_bad;
            status[3] = tot_cold;
        }
    }
    __syncthreads();

    // tile list
    for (int e = warp; e < E; e += kBucketWarps) {
        const int b0 = bounds[e], c = bounds[e + 1] - b0;
        const int nt = c <= cold_max ? 0 : (c + tile_tokens - 1) / tile_tokens;
        for (int t = lane; t < nt; t += 32) {
            MoETile mt;
            mt.expert = e;
            mt.first = t * tile_tokens;
            mt.count = c;
            mt.pad = 0;
            tiles[toff[e] + t] = mt;
        }
    }

    // pass 2: stable scatter, rounds of kBucketThreads pairs
    const int nvalid = bounds[E];
    for (int64_t base = 0; base < n_pairs; base += kBucketThreads) {
        const int64_t i = base + tid;
        const int e = i < n_pairs ? ids[i] : -1;
        const bool valid = e >= 0 && e < E;
        const unsigned key = valid ? (unsigned)e : (unsigned)(E + lane);  // invalid lanes stay alone
        const unsigned grp = __match_any_sync(0xffffffffu, key);
        const unsigned lt = grp & ((1u << lane) - 1u);
        const int rank = __popc(lt);
        if (valid && lt == 0) wcnt[warp * Ep + e] = __popc(grp);
        __syncthreads();
        // per expert, the warps' counts of this round scanned in warp order: warp w takes
        // experts w, w + 32, ..., lane l the count of warp l
        for (int x = warp; x < E; x += kBucketWarps) {
            const int c = wcnt[lane * Ep + x];
            int total;
            const int ex = warp_exclusive_scan(c, lane, total);
            wofs[lane * Ep + x] = cnt[x] + ex;
            wcnt[lane * Ep + x] = 0;
            __syncwarp();
            if (lane == 0) cnt[x] += total;
        }
        __syncthreads();
        if (valid) perm[wofs[warp * Ep + e] + rank] = (int32_t)i;
        // invalid pairs go after the valid ones, in index order
        const unsigned bad = __ballot_sync(0xffffffffu, i < n_pairs && !valid);
        if (bad) {
            int wbase = 0;
            if (lane == 0) wbase = atomicAdd(&s_bad_pos, __popc(bad));  // warps may interleave; order within a warp kept
            wbase = __shfl_sync(0xffffffffu, wbase, 0);
            if (i < n_pairs && !valid) perm[nvalid + wbase + __popc(bad & ((1u << lane) - 1u))] = (int32_t)i;
        }
        __syncthreads();
    }
}

__global__ void moe_zero_invalid_kernel(const int32_t *status, const int32_t *perm, const int32_t *bounds, int E,
                                        float *y, int64_t n) {
    const int nbad = status[2];
    const int nvalid = bounds[E];
    for (int b = blockIdx.x; b < nbad; b += gridDim.x) {
        float *row = y + int64_t(perm[nvalid + b]) * n;
        for (int64_t j = threadIdx.x; j < n; j += blockDim.x) row[j] = 0.f;
    }
}

cudaError_t launch_moe_bucket(const int32_t *ids, int64_t n_pairs, int n_experts, int tile_tokens, int cold_max,
                              void *ws, const MoELayout &L, cudaStream_t st) {
    uint8_t *base = static_cast<uint8_t *>(ws);
    const size_t smem = sizeof(int32_t) * (size_t(n_experts) * 2 + size_t(2 * kBucketWarps) * ((n_experts & ~1) + 1));
    cudaError_t e = ensure_smem(moe_bucket_kernel, smem);
    if (e != cudaSuccess) return e;
    moe_bucket_kernel<<<1, kBucketThreads, smem, st>>>(
        ids, n_pairs, n_experts, tile_tokens, cold_max, reinterpret_cast<int32_t *>(base + L.status),
        reinterpret_cast<int32_t *>(base + L.bounds), reinterpret_cast<int32_t *>(base + L.perm),
        reinterpret_cast<MoETile *>(base + L.tiles), reinterpret_cast<int32_t *>(base + L.cold));
    return cudaGetLastError();
}

constexpr int kDp4aTileTokens = 64;   // pairs per token tile of the CUDA-core grouped GEMM
constexpr int kTcTileTokens = 128;    // pairs per token tile of the tensor-core grouped GEMM
// Experts with at most this many pairs skip the 128-pair tiles of the tensor-core grouped
// GEMM (which would hold them in 128 rows) and run on the skinny tensor-core kernel,
// their pairs as its N = 16 columns.
constexpr int kColdMaxPairs = 16;

static size_t cold_bytes(qmm_type t, int64_t n_experts, int64_t n, int64_t k) {
    return gemv_tc_grouped_supported(t, n_experts, n, k) ? gemv_tc_grouped_bytes(n_experts, k) : 0;
}

size_t moe_dp4a_workspace_bytes(int64_t n_tokens, int64_t n_experts, int64_t top_k) {
    return moe_layout(n_tokens * top_k, n_experts, kDp4aTileTokens, 0, 0).total;
}

size_t moe_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t n_tokens, int64_t n_experts, int64_t top_k) {
    const int64_t n_pairs = n_tokens * top_k;
    if (gemm_tc_grouped_supported(t, n_experts, n, k))
        return moe_layout(n_pairs, n_experts, kTcTileTokens, gemm_tc_grouped_bytes(n_pairs, k),
                          cold_bytes(t, n_experts, n, k))
            .total;
    return moe_dp4a_workspace_bytes(n_tokens, n_experts, top_k);
}

cudaError_t launch_mul_mat_id_dp4a(qmm_type t, const void *W, int64_t n_experts, int64_t n, int64_t k,
                                   const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens,
                                   bool x_per_slot, float *y, void *ws, size_t ws_bytes, cudaStream_t st) {
    const int64_t n_pairs = n_tokens * top_k;
    const MoELayout L = moe_layout(n_pairs, n_experts, kDp4aTileTokens, 0, 0);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    cudaError_t e = launch_moe_bucket(ids, n_pairs, (int)n_experts, kDp4aTileTokens, 0, ws, L, st);
    if (e != cudaSuccess) return e;
    uint8_t *base = static_cast<uint8_t *>(ws);
    const int32_t *status = reinterpret_cast<const int32_t *>(base + L.status);
    const int32_t *bounds = reinterpret_cast<const int32_t *>(base + L.bounds);
    const int32_t *perm = reinterpret_cast<const int32_t *>(base + L.perm);
    const MoETile *tiles = reinterpret_cast<const MoETile *>(base + L.tiles);
    moe_zero_invalid_kernel<<<64, 256, 0, st>>>(status, perm, bounds, (int)n_experts, y, n);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_gemm_dp4a_grouped(t, W, n, k, xq, y, tiles, status + 1, bounds, perm, x_per_slot ? 1 : (int)top_k,
                                    st);
}


cudaError_t launch_mul_mat_id(qmm_type t, const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                              const int32_t *ids, int64_t top_k, int64_t n_tokens, bool x_per_slot, float *y,
                              void *ws, size_t ws_bytes, cudaStream_t st) {
    const int64_t n_pairs = n_tokens * top_k;
    if (n_pairs <= kMoeGemvMaxPairs && gemv_id_supported(t, n, k)) {
        int32_t *status = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + kStatusOffset);
        return launch_gemv_id(t, W, n_experts, n, k, xq, x_per_slot ? 1 : top_k, ids, n_pairs, y, status, st);
    }
    if (!gemm_tc_grouped_supported(t, n_experts, n, k))
        return launch_mul_mat_id_dp4a(t, W, n_experts, n, k, xq, ids, top_k, n_tokens, x_per_slot, y, ws, ws_bytes,
                                      st);
    const bool split = gemv_tc_grouped_supported(t, n_experts, n, k);
    const MoELayout L = moe_layout(n_pairs, n_experts, kTcTileTokens, gemm_tc_grouped_bytes(n_pairs, k),
                                   cold_bytes(t, n_experts, n, k));
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    cudaError_t e =
        launch_moe_bucket(ids, n_pairs, (int)n_experts, kTcTileTokens, split ? kColdMaxPairs : 0, ws, L, st);
    if (e != cudaSuccess) return e;
    uint8_t *base = static_cast<uint8_t *>(ws);
    int32_t *status = reinterpret_cast<int32_t *>(base + L.status);
    const int32_t *bounds = reinterpret_cast<const int32_t *>(base + L.bounds);
    const int32_t *perm = reinterpret_cast<const int32_t *>(base + L.perm);
    const MoETile *tiles = reinterpret_cast<const MoETile *>(base + L.tiles);
    moe_zero_invalid_kernel<<<64, 256, 0, st>>>(status, perm, bounds, (int)n_experts, y, n);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t x_div = x_per_slot ? 1 : top_k;
    const int64_t max_token_tiles = n_pairs / kTcTileTokens + n_experts + 1;
    e = launch_gemm_tc_grouped(t, W, n_experts, n, k, xq, x_div, n_pairs, y, tiles, status + 1, max_token_tiles, bounds,
                               perm, status, base + L.gemm, L.cold_gemm - L.gemm, st);
    if (e != cudaSuccess || !split) return e;
    // the cold experts: 16-column slabs on the skinny tensor-core kernel
    return launch_gemv_tc_grouped(W, n_experts, n, k, xq, x_div, reinterpret_cast<const int32_t *>(base + L.cold),
                                  status + 3, bounds, perm, y, status, base + L.cold_gemm, L.total - L.cold_gemm, st);
}

// ---------------------------------------------------------------- fused gate/up (SwiGLU)

// Unfused SwiGLU of two products in the workspace: y = silu(g) * u.
__global__ void moe_glu_combine_kernel(const float *__restrict__ g, const float *__restrict__ u, int64_t total,
                                       float *__restrict__ y) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x)
        y[i] = g[i] / (1.0f + expf(-g[i])) * u[i];
}

// The cold experts' SwiGLU: rows of their pairs from the gate and up products.  Block (p, c)
// takes pair p of cold expert c (a cold expert has at most kColdMaxPairs pairs), so every row
// has its own block (one block per expert walking its rows one after another took ~95 us).
__global__ void moe_glu_cold_combine_kernel(const int32_t *__restrict__ cold, const int32_t *__restrict__ ncold,
                                            const int32_t *__restrict__ bounds, const int32_t *__restrict__ perm,
                                            const float *__restrict__ g, const float *__restrict__ u,
                                            float *__restrict__ y, int64_t n) {
    const int nc = *ncold;
    for (int c = blockIdx.y; c < nc; c += gridDim.y) {
        const int e = cold[c];
        const int j = bounds[e] + (int)blockIdx.x;
        if (j >= bounds[e + 1]) continue;
        const int64_t off = int64_t(perm[j]) * n;
        for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
            const float gv = g[off + i];
            y[off + i] = gv / (1.0f + expf(-gv)) * u[off + i];
        }
    }
}

enum MoeGluPath { kMoeGluGemv = 1, kMoeGluTc = 2, kMoeGluUnfused = 3 };
static int moe_glu_path(qmm_type t, int64_t n_experts, int64_t n, int64_t k, int64_t n_pairs) {
    if (n_pairs <= kMoeGemvMaxPairs && gemv_id_glu_supported(t, n, k)) return kMoeGluGemv;
    if (gemm_tc_grouped_glu_supported(t, n_experts, n, k)) return kMoeGluTc;
    return kMoeGluUnfused;
}

// Unfused layout: the mul_mat_id workspace first (its status word stays at offset 0),
// then the gate and up products [pairs][n].
size_t moe_glu_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t n_tokens, int64_t n_experts, int64_t top_k) {
    const int64_t n_pairs = n_tokens * top_k;
    switch (moe_glu_path(t, n_experts, n, k, n_pairs)) {
    case kMoeGluGemv: return 256;  // the status word
    case kMoeGluTc: {
        // the cold experts' gate and up products after the layout, when they take the skinny kernel
        const bool split = gemv_tc_grouped_supported(t, n_experts, n, k);
        return moe_layout(n_pairs, n_experts, kTcTileTokens, gemm_tc_grouped_bytes(n_pairs, k),
                          cold_bytes(t, n_experts, n, k))
                   .total +
               (split ? 2 * align256(size_t(n_pairs) * size_t(n) * 4) : 0);
    }
    default:
        return align256(moe_workspace_bytes(t, n, k, n_tokens, n_experts, top_k)) +
               2 * align256(size_t(n_pairs) * size_t(n) * 4);
    }
}

cudaError_t launch_mul_mat_id_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n_experts, int64_t n, int64_t k,
                                  const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens, bool x_per_slot,
                                  float *y, void *ws, size_t ws_bytes, cudaStream_t st) {
    const int64_t n_pairs = n_tokens * top_k;
    const int64_t x_div = x_per_slot ? 1 : top_k;
    const int path = moe_glu_path(t, n_experts, n, k, n_pairs);
    if (ws_bytes < moe_glu_workspace_bytes(t, n, k, n_tokens, n_experts, top_k)) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    if (path == kMoeGluGemv)
        return launch_gemv_id_glu(t, Wg, Wu, n_experts, n, k, xq, x_div, ids, n_pairs, y,
                                  reinterpret_cast<int32_t *>(base + kStatusOffset), st);
    if (path == kMoeGluTc) {
        // experts with more than 16 pairs on the fused grouped GEMM; the others (cold) on the
        // skinny kernel, once for the gate and once for the up weights, then the combine
        const bool split = gemv_tc_grouped_supported(t, n_experts, n, k);
        const MoELayout L = moe_layout(n_pairs, n_experts, kTcTileTokens, gemm_tc_grouped_bytes(n_pairs, k),
                                       cold_bytes(t, n_experts, n, k));
        cudaError_t e =
            launch_moe_bucket(ids, n_pairs, (int)n_experts, kTcTileTokens, split ? kColdMaxPairs : 0, ws, L, st);
        if (e != cudaSuccess) return e;
        int32_t *status = reinterpret_cast<int32_t *>(base + L.status);
        const int32_t *bounds = reinterpret_cast<const int32_t *>(base + L.bounds);
        const int32_t *perm = reinterpret_cast<const int32_t *>(base + L.perm);
        const MoETile *tiles = reinterpret_cast<const MoETile *>(base + L.tiles);
        moe_zero_invalid_kernel<<<64, 256, 0, st>>>(status, perm, bounds, (int)n_experts, y, n);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = launch_gemm_tc_grouped_glu(t, Wg, Wu, n_experts, n, k, xq, x_div, n_pairs, y, tiles, status + 1, bounds,
                                       perm, status, base + L.gemm, L.cold_gemm - L.gemm, st);
        if (e != cudaSuccess || !split) return e;
        const int32_t *cold = reinterpret_cast<const int32_t *>(base + L.cold);
        float *g = reinterpret_cast<float *>(base + L.total);
        float *u = reinterpret_cast<float *>(base + L.total + align256(size_t(n_pairs) * size_t(n) * 4));
        for (int h = 0; h < 2; ++h) {
            e = launch_gemv_tc_grouped(h ? Wu : Wg, n_experts, n, k, xq, x_div, cold, status + 3, bounds, perm,
                                       h ? u : g, status, base + L.cold_gemm, L.total - L.cold_gemm, st);
            if (e != cudaSuccess) return e;
        }
        const dim3 grid(kColdMaxPairs, (unsigned)std::min<int64_t>(std::max<int64_t>(n_experts, 1), 65535));
        moe_glu_cold_combine_kernel<<<grid, 256, 0, st>>>(cold, status + 3, bounds, perm, g, u, y, n);
        return cudaGetLastError();
    }
    // unfused: both products through mul_mat_id, then y = silu(g) * u (invalid pairs: 0 * 0)
    const size_t inner = align256(moe_workspace_bytes(t, n, k, n_tokens, n_experts, top_k));
    float *g = reinterpret_cast<float *>(base + inner);
    float *u = reinterpret_cast<float *>(base + inner + align256(size_t(n_pairs) * size_t(n) * 4));
    cudaError_t e = launch_mul_mat_id(t, Wg, n_experts, n, k, xq, ids, top_k, n_tokens, x_per_slot, g, ws, inner, st);
    if (e != cudaSuccess) return e;
    e = launch_mul_mat_id(t, Wu, n_experts, n, k, xq, ids, top_k, n_tokens, x_per_slot, u, ws, inner, st);
    if (e != cudaSuccess) return e;
    const int64_t total = n_pairs * n;
    const int grid = (int)std::min<int64_t>((total + 255) / 256, int64_t(device_sm_count()) * 8);
    moe_glu_combine_kernel<<<std::max(grid, 1), 256, 0, st>>>(g, u, total, y);
    return cudaGetLastError();
}

}  // namespace qmm
