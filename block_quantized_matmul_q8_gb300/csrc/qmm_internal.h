// qmm_internal.h -- host-side declarations shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "qmm.h"

namespace qmm {

// SM count of the current device (cached per device).
int device_sm_count();
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for kern on the current device, skipped
// when an equal or larger size was already granted
cudaError_t ensure_max_dynamic_smem(const void *kern, size_t bytes);
template <class K> inline cudaError_t ensure_smem(K *kern, size_t bytes) {
    return ensure_max_dynamic_smem(reinterpret_cast<const void *>(kern), bytes);
}

// Launch kern<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization, so that it may start while the previous kernel in the stream is
// still running; the kernel itself waits (griddepcontrol.wait) before it touches
// anything that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
// Opt-in shared memory per block of the current device (cached per device).
int device_smem_optin();

// ---------------------------------------------------------------- launchers
cudaError_t launch_quantize_q8_1(const float *x, int64_t m, int64_t k, void *xq, cudaStream_t st);

// False when the test switch asks for the direct-load GEMV only.
bool gemv_tma_enabled();

// GEMV, m <= 8: y[m][n] from W rows and the activations, given either as q8_1 blocks
// (xq) or as fp32 values (xf != nullptr), which each CTA then quantizes itself to the
// same bytes as launch_quantize_q8_1.  Columns are taken in groups of up to 8 per launch.
size_t gemv_smem_bytes(int64_t k, int ncols);
// ring depth of the bulk-copy GEMV for ncols columns in budget bytes (0: direct kernel)
int gemv_ring_stages(qmm_type t, int64_t n, int64_t k, int ncols, size_t budget);
// stride: bytes from one weight row to the next (0: the natural k/QK blocks; > 0: rows
// padded to a multiple of 16 bytes by qmm_repack_aligned).
cudaError_t launch_gemv(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, const float *xf, int64_t m,
                        float *y, cudaStream_t st, int64_t stride = 0);
// Fused gate/up + SwiGLU GEMV (Q4_K, m <= 8): y[m][n] = silu(x Wg^T) * (x Wu^T) from
// q8_1 activations, both weights read once.
// Fused gate/up launches take Wu == nullptr for one interleaved tensor (gate row j at
// 2j, up row j at 2j+1, as qmm_repack_glu writes it) in Wg.
bool gemv_glu_supported(qmm_type t, int64_t n, int64_t k, int64_t m);
cudaError_t launch_gemv_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n, int64_t k, const void *xq,
                            int64_t m, float *y, cudaStream_t st);
// Expert-routed decode: one bulk-copy GEMV per (token, slot) pair, expert ids read on the
// device; pair p's activation row is xq row p / x_div.  Invalid ids give zero rows; the
// kernel writes *status (QMM_OK, or QMM_ERR_IDS if any id is invalid).
bool gemv_id_supported(qmm_type t, int64_t n, int64_t k);
cudaError_t launch_gemv_id(qmm_type t, const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                           int64_t x_div, const int32_t *ids, int64_t n_pairs, float *y, int *status,
                           cudaStream_t st);
// Its fused gate/up form (Q4_K): pair p's row of y is silu(gate dot) * up dot, with the
// experts' gate rows in Wg and their up rows in Wu (both [E][n] rows).
bool gemv_id_glu_supported(qmm_type t, int64_t n, int64_t k);
cudaError_t launch_gemv_id_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n_experts, int64_t n, int64_t k,
                               const void *xq, int64_t x_div, const int32_t *ids, int64_t n_pairs, float *y,
                               int *status, cudaStream_t st);

// Multi-column GEMV on the warp-level MMA (Q4_K, 2 <= m <= 8, q8_1 activations): 16 weight
// rows x 8 columns per mma.sync m16n8k16 on exact integer operands, then the fp32 fold.
bool gemv_mma_supported(qmm_type t, int64_t n, int64_t k, int64_t m);
cudaError_t launch_gemv_mma(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                            cudaStream_t st);

// Tensor-core path for skinny activations (Q4_K, 1 <= m <= 16): weights as the MMA's
// 128-row M side, activations as N = 16; stream-K over (row tile, superblock) units.
bool gemv_tc_supported(qmm_type t, int64_t n, int64_t k, int64_t m);
// Expert-grouped skinny path for the cold experts of mul_mat_id (1..16 pairs each): the
// cold list and its count (on the device) come from the bucketing kernel; x_div as in
// gemv_id.  y rows are pairs; status receives QMM_ERR_DEVICE if a wait gives up.
bool gemv_tc_grouped_supported(qmm_type t, int64_t n_experts, int64_t n, int64_t k);
size_t gemv_tc_grouped_bytes(int64_t n_experts, int64_t k);
cudaError_t launch_gemv_tc_grouped(const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                                   int64_t x_div, const int32_t *cold, const int32_t *ncold, const int32_t *bounds,
                                   const int32_t *perm, float *y, int *status, void *ws, size_t ws_bytes,
                                   cudaStream_t st);
size_t gemv_tc_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t m);
cudaError_t launch_gemv_tc(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                           void *ws, size_t ws_bytes, cudaStream_t st);

// CUDA-core tiled GEMM (dp4a), any m.
cudaError_t launch_gemm_dp4a(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                             cudaStream_t st, int64_t stride = 0);

// Tensor-core GEMM (tcgen05, kind::f16 on integer-valued operands).
int64_t gemm_tc_tile_m(int64_t m);
size_t gemm_tc_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t m, int64_t stride = 0);
bool gemm_tc_supported(qmm_type t, int64_t n, int64_t k, int64_t m, int64_t stride = 0);
cudaError_t launch_gemm_tc(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                           void *ws, size_t ws_bytes, int stream_k_mode, cudaStream_t st, int64_t stride = 0);
// Row stride of the padded layout of qmm_repack_aligned (0 for bad arguments).
int64_t aligned_row_bytes(qmm_type t, int64_t k);

// Fused gate/up + SwiGLU on the tensor-core GEMM (Q4_K): y[m][n_out] = silu(x Wg^T) * (x Wu^T),
// one whole 128-column tile (64 outputs) per CTA.
bool gemm_tc_glu_supported(qmm_type t, int64_t n_out, int64_t k, int64_t m);
size_t gemm_tc_glu_workspace_bytes(qmm_type t, int64_t n_out, int64_t k, int64_t m);
cudaError_t launch_gemm_tc_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n_out, int64_t k, const void *xq,
                               int64_t m, float *y, void *ws, size_t ws_bytes, cudaStream_t st);

// Expert-grouped tensor-core GEMM over a device-built tile list (see qmm_moe.h); sorted
// pair row j takes xq row perm[j] / x_div.
struct MoETile;
bool gemm_tc_grouped_supported(qmm_type t, int64_t n_experts, int64_t n, int64_t k);
size_t gemm_tc_grouped_bytes(int64_t n_pairs, int64_t k);
cudaError_t launch_gemm_tc_grouped(qmm_type t, const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                                   int64_t x_div, int64_t n_pairs, float *y, const MoETile *tiles,
                                   const int32_t *ntiles, int64_t max_token_tiles, const int32_t *bounds,
                                   const int32_t *perm, int *status, void *ws, size_t ws_bytes, cudaStream_t st);
// Its fused gate/up form (Q4_K): y[pair][n] = silu(gate dot) * up dot, whole tiles only.
bool gemm_tc_grouped_glu_supported(qmm_type t, int64_t n_experts, int64_t n, int64_t k);
cudaError_t launch_gemm_tc_grouped_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n_experts, int64_t n,
                                       int64_t k, const void *xq, int64_t x_div, int64_t n_pairs, float *y,
                                       const MoETile *tiles, const int32_t *ntiles, const int32_t *bounds,
                                       const int32_t *perm, int *status, void *ws, size_t ws_bytes, cudaStream_t st);

// MoE: device bucketing + grouped GEMM, or one GEMV per pair for a handful of pairs.
// x_per_slot: xq holds one activation row per (token, slot) pair instead of one per token.
size_t moe_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t n_tokens, int64_t n_experts, int64_t top_k);
cudaError_t launch_mul_mat_id(qmm_type t, const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                              const int32_t *ids, int64_t top_k, int64_t n_tokens, bool x_per_slot, float *y,
                              void *ws, size_t ws_bytes, cudaStream_t st);
// Fused gate/up + SwiGLU of mul_mat_id: y[t][s][n] = silu(x Wg[e]^T) * (x Wu[e]^T) with
// e = ids[t][s]: one fused GEMV per pair for a handful of pairs, the fused grouped
// tensor-core GEMM (Q4_K), else both products into the workspace and a combine pass.
size_t moe_glu_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t n_tokens, int64_t n_experts, int64_t top_k);
cudaError_t launch_mul_mat_id_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n_experts, int64_t n, int64_t k,
                                  const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens, bool x_per_slot,
                                  float *y, void *ws, size_t ws_bytes, cudaStream_t st);
// Argument checks of qmm_mul_mat_id shared by its entry points.
qmm_status moe_check_sizes(qmm_type t, int64_t n_experts, int64_t n, int64_t k, int64_t top_k, int64_t n_tokens);
qmm_status moe_check_pointers(const void *W_experts, const void *xq, const int32_t *ids, const float *y);
// The same computation on CUDA-core tiles only; its scratch is small (bucketing only).
size_t moe_dp4a_workspace_bytes(int64_t n_tokens, int64_t n_experts, int64_t top_k);
cudaError_t launch_mul_mat_id_dp4a(qmm_type t, const void *W, int64_t n_experts, int64_t n, int64_t k,
                                   const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens,
                                   bool x_per_slot, float *y, void *ws, size_t ws_bytes, cudaStream_t st);

// Test switch of qmm_set_test_fault (0: off).
int test_fault_mode();

// Offset of the device status word inside a mul_mat_id workspace.
constexpr size_t kStatusOffset = 0;

}  // namespace qmm
