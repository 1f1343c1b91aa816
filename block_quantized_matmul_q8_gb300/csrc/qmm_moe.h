// qmm_moe.h -- device-side expert bucketing shared by the MoE kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm.h"

namespace qmm {

// One work item of the expert-grouped GEMM: pairs [first, min(first + tile, count))
// of expert `expert` in the sorted order (count = that expert's pair count).
struct MoETile {
    int32_t expert;
    int32_t first;
    int32_t count;
    int32_t pad;
};

// Largest expert count the single-CTA bucketing kernel supports.
constexpr int kMaxExperts = 512;

// Up to this many (token, slot) pairs, one GEMV per pair beats the grouped GEMM, whose
// 128-pair tiles would each hold one or two pairs.
constexpr int64_t kMoeGemvMaxPairs = 32;

// Workspace layout of qmm_mul_mat_id (offsets in bytes, 256-byte aligned pieces).
struct MoELayout {
    size_t status;   // int32 status word, tile count, invalid-pair count, cold-expert count
    size_t bounds;   // int32 [E + 1]
    size_t perm;     // int32 [pairs]: valid pairs sorted by expert, then invalid pairs
    size_t tiles;    // MoETile [max tiles]
    size_t cold;     // int32 [E]: the cold experts (1..cold_max pairs, no tiles), count in status[3]
    size_t gemm;       // scratch of the grouped GEMM
    size_t cold_gemm;  // scratch of the cold experts' skinny kernel
    size_t total;
};
MoELayout moe_layout(int64_t n_pairs, int64_t n_experts, int tile_tokens, size_t gemm_bytes, size_t cold_bytes);

// cold_max > 0: experts with 1..cold_max pairs are left out of the tile list and listed
// in L.cold instead (their count in status[3]); 0: every expert with pairs gets tiles.
cudaError_t launch_moe_bucket(const int32_t *ids, int64_t n_pairs, int n_experts, int tile_tokens, int cold_max,
                              void *ws, const MoELayout &L, cudaStream_t st);

cudaError_t launch_gemm_dp4a_grouped(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, float *y,
                                     const MoETile *tiles, const int32_t *ntiles, const int32_t *bounds,
                                     const int32_t *perm, int top_k, cudaStream_t st);

}  // namespace qmm
