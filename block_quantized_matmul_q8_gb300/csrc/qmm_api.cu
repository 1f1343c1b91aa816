// qmm_api.cu -- the C ABI (include/qmm.h): argument checks, path choice, planning.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <map>
#include <mutex>
#include <utility>

#include "qmm.h"
#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_moe.h"

namespace qmm {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_optin[kMaxDevices];
std::atomic<int> g_force_path{0};
std::atomic<int> g_stream_k_mode{0};
std::atomic<int> g_test_fault{0};

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return dev;
}
}  // namespace

// The largest dynamic shared-memory size already granted to each kernel on each device:
// the attribute is set once per (kernel, device, larger size), not on every call.
cudaError_t ensure_max_dynamic_smem(const void *kern, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, size_t> granted;
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = granted.find({kern, dev});
        if (it != granted.end() && it->second >= bytes) return cudaSuccess;
    }
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lock(mu);
        size_t &g = granted[{kern, dev}];
        g = std::max(g, bytes);
    }
    return e;
}

int device_sm_count() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 1;
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
        g_sm_count[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

int device_smem_optin() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 48 * 1024;
    int v = g_smem_optin[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || v <= 0)
            v = 48 * 1024;
        g_smem_optin[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

static bool type_ok(qmm_type t) {
    return t == QMM_Q4_K || t == QMM_Q5_K || t == QMM_Q6_K || t == QMM_Q8_0 || t == QMM_Q4_0;
}
static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
static bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

constexpr int64_t kMaxK = int64_t(1) << 20;
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;

static qmm_status check_k(qmm_type t, int64_t k) {
    if (!type_ok(t)) return QMM_ERR_TYPE;
    if (k <= 0) return QMM_ERR_ARG;
    if (k % block_elems(t) != 0 || k % 32 != 0 || k > kMaxK) return QMM_ERR_SHAPE;
    return QMM_OK;
}

static qmm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA; }

// Which kernel family qmm_mul_mat uses for these sizes.
enum Path { kGemv = 1, kGemmDp4a = 2, kGemmTc = 3, kGemvDirect = 4, kGemvTc = 5, kGemvMma = 6 };

int test_fault_mode() { return g_test_fault.load(std::memory_order_relaxed); }

bool gemv_tma_enabled() { return g_force_path.load(std::memory_order_relaxed) != kGemvDirect; }

// stride: the row stride of padded rows (qmm_repack_aligned), 0 for natural rows.
static int choose_path(qmm_type t, int64_t n, int64_t k, int64_t m, int64_t stride = 0) {
    const int force = g_force_path.load(std::memory_order_relaxed);
    const bool gemv_fits = gemv_smem_bytes(k, 1) <= size_t(device_smem_optin());
    if ((force == kGemv || force == kGemvDirect) && gemv_fits && m <= 64) return kGemv;
    if (force == kGemmDp4a) return kGemmDp4a;
    if (force == kGemmTc && gemm_tc_supported(t, n, k, m, stride)) return kGemmTc;
    if (force == kGemvTc && gemv_tc_supported(t, n, k, m)) return kGemvTc;
    if (force == kGemvMma && gemv_mma_supported(t, n, k, m)) return kGemvMma;
    // Q4_K from 6 columns on (natural rows): the MMA GEMV's cost hardly grows with the
    // columns, the dp4a GEMV's does (17408 x 5120: 21.9 against 22.5 us at 6 columns, 22.6
    // against 32.3 at 8; at 5 columns the row-pair dp4a GEMV is faster, 20.2 against 21.8)
    if (m >= 6 && m <= 8 && stride == 0 && gemv_mma_supported(t, n, k, m)) return kGemvMma;
    if (m <= 8 && gemv_fits) return kGemv;
    // skinny activations on the tensor cores (weights as the MMA's M side; Q4_K, whose rows
    // are whole 16-byte units and so never padded)
    if (gemv_tc_supported(t, n, k, m)) return kGemvTc;
    if (gemm_tc_supported(t, n, k, m, stride)) return kGemmTc;
    return kGemmDp4a;
}

// Bytes at the head of the qmm_mul_mat_f32 workspace that hold the q8_1 activations.
size_t q8_region_bytes(int64_t m, int64_t k) { return ((size_t(m) * size_t(k / 32) * kQ81Bytes) + 255) & ~size_t(255); }

qmm_status mul_mat_q8(const void *W, qmm_type t, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                      void *workspace, size_t ws_bytes, cudaStream_t st, int64_t stride = 0);

qmm_status moe_check_sizes(qmm_type t, int64_t n_experts, int64_t n, int64_t k, int64_t top_k, int64_t n_tokens) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n_experts <= 0 || top_k <= 0 || n < 0 || n_tokens < 0) return QMM_ERR_ARG;
    // the pair count n_tokens * top_k, compared without forming a product that could overflow
    if (n_experts > kMaxExperts || n > kMaxRows || top_k > kMaxRows || n_tokens > kMaxRows / top_k)
        return QMM_ERR_SHAPE;
    return QMM_OK;
}

qmm_status moe_check_pointers(const void *W_experts, const void *xq, const int32_t *ids, const float *y) {
    if (!W_experts || !xq || !ids || !y) return QMM_ERR_ARG;
    if (!aligned16(W_experts) || !aligned16(xq) || !aligned16(y) || (reinterpret_cast<uintptr_t>(ids) & 3u))
        return QMM_ERR_ALIGN;
    return QMM_OK;
}

}  // namespace qmm

using namespace qmm;

// Unfused SwiGLU for the shapes the fused kernels do not take: y = silu(g) * u.
__global__ void glu_combine_kernel(const float *__restrict__ g, const float *__restrict__ u, int64_t total,
                                   float *__restrict__ y) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x)
        y[i] = g[i] / (1.0f + expf(-g[i])) * u[i];
}

// The same from one product of an interleaved gate/up tensor: z is [m][2n] with the gate
// dot of output j in column 2j and the up dot in column 2j+1.
__global__ void glu_combine_pairs_kernel(const float2 *__restrict__ z, int64_t total, float *__restrict__ y) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const float2 gu = z[i];
        y[i] = gu.x / (1.0f + expf(-gu.x)) * gu.y;
    }
}

// Interleave a gate/up pair row by row: dst row 2j = gate row j, 2j+1 = up row j.  rows
// of rb bytes; copied in 16-byte units when rb allows (all pointers are 16-byte aligned),
// else in 2-byte units (every block size is even).
__global__ void repack_glu_kernel(const uint8_t *__restrict__ wg, const uint8_t *__restrict__ wu, int64_t n,
                                  int64_t rb, uint8_t *__restrict__ dst) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    if (rb % 16 == 0) {
        const int64_t per_row = rb / 16, total = 2 * n * per_row;
        for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
            const int64_t row = i / per_row, c = i - row * per_row;
            const uint8_t *src = ((row & 1) ? wu : wg) + (row >> 1) * rb;
            reinterpret_cast<uint4 *>(dst + row * rb)[c] = reinterpret_cast<const uint4 *>(src)[c];
        }
    } else {
        const int64_t per_row = rb / 2, total = 2 * n * per_row;
        for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
            const int64_t row = i / per_row, c = i - row * per_row;
            const uint8_t *src = ((row & 1) ? wu : wg) + (row >> 1) * rb;
            reinterpret_cast<uint16_t *>(dst + row * rb)[c] = reinterpret_cast<const uint16_t *>(src)[c];
        }
    }
}

// Rows of rb bytes copied to rows of `stride` bytes (a multiple of 16), the tail of each
// row zero; in units of U bytes, U dividing rb (every block size is even).
template <int U>
__global__ void repack_aligned_kernel(const uint8_t *__restrict__ src, int64_t n, int64_t rb, int64_t stride,
                                      uint8_t *__restrict__ dst) {
    using V = typename std::conditional<U == 8, uint2, typename std::conditional<U == 4, uint32_t, uint16_t>::type>::type;
    const int64_t per_row = stride / U, total = n * per_row;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = i / per_row, c = i - row * per_row;
        V v{};
        if (c * U < rb) v = reinterpret_cast<const V *>(src + row * rb)[c];
        reinterpret_cast<V *>(dst + row * stride)[c] = v;
    }
}

enum GluPath { kGluGemv = 1, kGluTc = 2, kGluUnfused = 3 };
static int choose_glu_path(qmm_type t, int64_t n, int64_t k, int64_t m) {
    const int force = g_force_path.load(std::memory_order_relaxed);
    if (force == kGemmDp4a) return kGluUnfused;
    if (force == kGemmTc && gemm_tc_glu_supported(t, n, k, m)) return kGluTc;
    if (force == kGemv && gemv_glu_supported(t, n, k, m)) return kGluGemv;
    if (m <= 8 && gemv_glu_supported(t, n, k, m)) return kGluGemv;
    if (gemm_tc_glu_supported(t, n, k, m)) return kGluTc;
    return kGluUnfused;
}

static qmm_status mul_mat_id_common(const void *W_experts, qmm_type t, int64_t n_experts, int64_t n, int64_t k,
                                    const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens,
                                    bool x_per_slot, float *y, void *workspace, size_t ws_bytes, void *stream) {
    qmm_status s = moe_check_sizes(t, n_experts, n, k, top_k, n_tokens);
    if (s != QMM_OK) return s;
    if (!workspace) return QMM_ERR_WORKSPACE;
    if (!aligned256(workspace)) return QMM_ERR_ALIGN;
    const size_t need = moe_workspace_bytes(t, n, k, n_tokens, n_experts, top_k);
    if (ws_bytes < need) return QMM_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n == 0 || n_tokens == 0) {
        // empty problem: only reset the status word
        return cuda_status(cudaMemsetAsync(workspace, 0, 16, st));
    }
    s = moe_check_pointers(W_experts, xq, ids, y);
    if (s != QMM_OK) return s;
    return cuda_status(launch_mul_mat_id(t, W_experts, n_experts, n, k, xq, ids, top_k, n_tokens, x_per_slot, y,
                                         workspace, ws_bytes, st));
}

extern "C" {

const char *qmm_status_string(qmm_status s) {
    switch (s) {
    case QMM_OK: return "QMM_OK";
    case QMM_ERR_ARG: return "QMM_ERR_ARG";
    case QMM_ERR_SHAPE: return "QMM_ERR_SHAPE";
    case QMM_ERR_TYPE: return "QMM_ERR_TYPE";
    case QMM_ERR_ALIGN: return "QMM_ERR_ALIGN";
    case QMM_ERR_WORKSPACE: return "QMM_ERR_WORKSPACE";
    case QMM_ERR_CUDA: return "QMM_ERR_CUDA";
    case QMM_ERR_IDS: return "QMM_ERR_IDS";
    case QMM_ERR_DEVICE: return "QMM_ERR_DEVICE";
    }
    return "QMM_ERR_UNKNOWN";
}

size_t qmm_q8_1_bytes(int64_t m, int64_t k) {
    if (m < 0 || k < 0) return 0;
    return size_t(m) * size_t(k / 32) * kQ81Bytes;
}

size_t qmm_row_bytes(qmm_type t, int64_t k) {
    if (!type_ok(t) || k < 0 || k % block_elems(t)) return 0;
    return size_t(k / block_elems(t)) * size_t(block_bytes(t));
}

size_t qmm_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t m, int64_t n_experts, int64_t top_k) {
    if (!type_ok(t) || n < 0 || k <= 0 || m < 0) return 0;
    if (n_experts > 0)
        return moe_check_sizes(t, n_experts, n, k, top_k, m) == QMM_OK ? moe_workspace_bytes(t, n, k, m, n_experts, top_k)
                                                                        : 0;
    if (n > kMaxRows || m > kMaxRows || check_k(t, k) != QMM_OK) return 0;
    // enough for every path the call may take (the forced ones included)
    const size_t gemm = gemm_tc_supported(t, n, k, m) ? gemm_tc_workspace_bytes(t, n, k, m) : 0;
    return std::max(gemm, gemv_tc_workspace_bytes(t, n, k, m));
}

qmm_status qmm_quantize_q8_1(const float *x, int64_t m, int64_t k, void *xq, void *stream) {
    if (m < 0 || k <= 0) return QMM_ERR_ARG;
    if (k % 32 || k > kMaxK || m > kMaxRows) return QMM_ERR_SHAPE;
    if (m == 0) return QMM_OK;
    if (!x || !xq) return QMM_ERR_ARG;
    if (!aligned16(x) || !aligned16(xq)) return QMM_ERR_ALIGN;
    return cuda_status(launch_quantize_q8_1(x, m, k, xq, static_cast<cudaStream_t>(stream)));
}

qmm_status qmm_mul_mat(const void *W, qmm_type t, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                       void *workspace, size_t ws_bytes, void *stream) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n < 0 || m < 0) return QMM_ERR_ARG;
    if (n > kMaxRows || m > kMaxRows) return QMM_ERR_SHAPE;
    if (n == 0 || m == 0) return QMM_OK;
    if (!W || !xq || !y) return QMM_ERR_ARG;
    if (!aligned16(W) || !aligned16(xq) || !aligned16(y)) return QMM_ERR_ALIGN;
    return mul_mat_q8(W, t, n, k, xq, m, y, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

size_t qmm_workspace_bytes_glu(qmm_type t, int64_t n, int64_t k, int64_t m) {
    if (!type_ok(t) || n <= 0 || k <= 0 || m <= 0 || check_k(t, k) != QMM_OK) return 0;
    switch (choose_glu_path(t, n, k, m)) {
    case kGluGemv: return 0;
    case kGluTc: return gemm_tc_glu_workspace_bytes(t, n, k, m);
    // unfused: two products of n rows, or one of 2n rows for the interleaved tensor
    default: return align256(size_t(2) * m * n * 4) + qmm_workspace_bytes(t, 2 * n, k, m, 0, 0);
    }
}

static qmm_status mul_mat_glu_common(const void *W_gate, const void *W_up, bool packed, qmm_type t, int64_t n,
                                     int64_t k, const void *xq, int64_t m, float *y, void *workspace, size_t ws_bytes,
                                     void *stream) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n < 0 || m < 0) return QMM_ERR_ARG;
    if (n > kMaxRows / 2 || m > kMaxRows) return QMM_ERR_SHAPE;
    if (n == 0 || m == 0) return QMM_OK;
    if (!W_gate || (!packed && !W_up) || !xq || !y) return QMM_ERR_ARG;
    if (!aligned16(W_gate) || (!packed && !aligned16(W_up)) || !aligned16(xq) || !aligned16(y)) return QMM_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const void *wu = packed ? nullptr : W_up;
    const int path = choose_glu_path(t, n, k, m);
    if (path == kGluGemv) return cuda_status(launch_gemv_glu(t, W_gate, wu, n, k, xq, m, y, st));
    const size_t need = qmm_workspace_bytes_glu(t, n, k, m);
    if (!workspace || ws_bytes < need) return QMM_ERR_WORKSPACE;
    if (!aligned256(workspace)) return QMM_ERR_ALIGN;
    if (path == kGluTc) return cuda_status(launch_gemm_tc_glu(t, W_gate, wu, n, k, xq, m, y, workspace, ws_bytes, st));
    // unfused: the dots into the workspace, then the combine pass
    float *g = static_cast<float *>(workspace), *u = g + m * n;
    uint8_t *rest = static_cast<uint8_t *>(workspace) + align256(size_t(2) * m * n * 4);
    const size_t rest_bytes = ws_bytes - align256(size_t(2) * m * n * 4);
    const int64_t total = m * n;
    const int grid = (int)std::min<int64_t>((total + 255) / 256, int64_t(device_sm_count()) * 8);
    if (packed) {  // one product of the 2n interleaved rows: [m][2n], gate and up side by side
        s = mul_mat_q8(W_gate, t, 2 * n, k, xq, m, g, rest, rest_bytes, st);
        if (s != QMM_OK) return s;
        glu_combine_pairs_kernel<<<std::max(grid, 1), 256, 0, st>>>(reinterpret_cast<const float2 *>(g), total, y);
        return cuda_status(cudaGetLastError());
    }
    s = mul_mat_q8(W_gate, t, n, k, xq, m, g, rest, rest_bytes, st);
    if (s != QMM_OK) return s;
    s = mul_mat_q8(W_up, t, n, k, xq, m, u, rest, rest_bytes, st);
    if (s != QMM_OK) return s;
    glu_combine_kernel<<<std::max(grid, 1), 256, 0, st>>>(g, u, total, y);
    return cuda_status(cudaGetLastError());
}

qmm_status qmm_mul_mat_glu(const void *W_gate, const void *W_up, qmm_type t, int64_t n, int64_t k, const void *xq,
                           int64_t m, float *y, void *workspace, size_t ws_bytes, void *stream) {
    return mul_mat_glu_common(W_gate, W_up, false, t, n, k, xq, m, y, workspace, ws_bytes, stream);
}

qmm_status qmm_mul_mat_glu_packed(const void *W_gu, qmm_type t, int64_t n, int64_t k, const void *xq, int64_t m,
                                  float *y, void *workspace, size_t ws_bytes, void *stream) {
    return mul_mat_glu_common(W_gu, nullptr, true, t, n, k, xq, m, y, workspace, ws_bytes, stream);
}

qmm_status qmm_repack_glu(const void *W_gate, const void *W_up, qmm_type t, int64_t n, int64_t k, void *W_gu,
                          void *stream) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n < 0) return QMM_ERR_ARG;
    if (n > kMaxRows / 2) return QMM_ERR_SHAPE;
    if (n == 0) return QMM_OK;
    if (!W_gate || !W_up || !W_gu) return QMM_ERR_ARG;
    if (!aligned16(W_gate) || !aligned16(W_up) || !aligned16(W_gu)) return QMM_ERR_ALIGN;
    const int64_t rb = int64_t(qmm_row_bytes(t, k));
    const int64_t units = 2 * n * (rb % 16 == 0 ? rb / 16 : rb / 2);
    const int grid = (int)std::min<int64_t>((units + 255) / 256, int64_t(device_sm_count()) * 8);
    repack_glu_kernel<<<std::max(grid, 1), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(W_gate), static_cast<const uint8_t *>(W_up), n, rb, static_cast<uint8_t *>(W_gu));
    return cuda_status(cudaGetLastError());
}

size_t qmm_workspace_bytes_f32(qmm_type t, int64_t n, int64_t k, int64_t m) {
    if (!type_ok(t) || n < 0 || k <= 0 || m < 0 || k % 32) return 0;
    return q8_region_bytes(m, k) + qmm_workspace_bytes(t, n, k, m, 0, 0);
}

qmm_status qmm_mul_mat_f32(const void *W, qmm_type t, int64_t n, int64_t k, const float *x, int64_t m, float *y,
                           void *workspace, size_t ws_bytes, void *stream) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n < 0 || m < 0) return QMM_ERR_ARG;
    if (n > kMaxRows || m > kMaxRows) return QMM_ERR_SHAPE;
    if (n == 0 || m == 0) return QMM_OK;
    if (!W || !x || !y) return QMM_ERR_ARG;
    if (!aligned16(W) || !aligned16(x) || !aligned16(y)) return QMM_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // m == 1: one launch; every CTA quantizes the activation row into its shared memory
    // while its first weight copies are in flight.  For m > 1 the redundant per-CTA
    // quantization (m*k values on every CTA, its loads exposed before the first fold)
    // costs more than the separate quantizer launch, so the q8_1 route below is taken.
    const int path = choose_path(t, n, k, m);
    if (path == kGemv && m == 1) return cuda_status(launch_gemv(t, W, n, k, nullptr, x, m, y, st));
    // otherwise: the quantizer writes q8_1 into the head of the workspace, then the product
    if (!workspace || ws_bytes < qmm_workspace_bytes_f32(t, n, k, m)) return QMM_ERR_WORKSPACE;
    if (!aligned256(workspace)) return QMM_ERR_ALIGN;
    const size_t off = q8_region_bytes(m, k);
    uint8_t *xq = static_cast<uint8_t *>(workspace);
    cudaError_t e = launch_quantize_q8_1(x, m, k, xq, st);
    if (e != cudaSuccess) return QMM_ERR_CUDA;
    return mul_mat_q8(W, t, n, k, xq, m, y, xq + off, ws_bytes - off, st);
}

// Host-buffer form: x_dev [m][k] and y_dev [m][n] at the head of the workspace, each
// 256-byte aligned, then the qmm_mul_mat_f32 workspace.
constexpr size_t kMappedOutMax = size_t(1) << 20;  // y written in place up to 1 MB

// The device address of a page-locked (registered or cudaHostAlloc'd) host buffer, if it
// has one and it is `align`-byte aligned; nullptr otherwise (pageable memory, device
// memory, or a query error, which is cleared).
static const void *mapped_host(const void *p, size_t align) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
    if (reinterpret_cast<uintptr_t>(a.devicePointer) % align) return nullptr;
    return a.devicePointer;
}
static size_t host_io_bytes(int64_t n, int64_t k, int64_t m) {
    return align256(size_t(m) * size_t(k) * 4) + align256(size_t(m) * size_t(n) * 4);
}

size_t qmm_workspace_bytes_f32_host(qmm_type t, int64_t n, int64_t k, int64_t m) {
    if (!type_ok(t) || n < 0 || k <= 0 || m < 0 || k % 32) return 0;
    return host_io_bytes(n, k, m) + qmm_workspace_bytes_f32(t, n, k, m);
}

qmm_status qmm_mul_mat_f32_host(const void *W, qmm_type t, int64_t n, int64_t k, const float *x_host, int64_t m,
                                float *y_host, void *workspace, size_t ws_bytes, void *stream) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n < 0 || m < 0) return QMM_ERR_ARG;
    if (n > kMaxRows || m > kMaxRows) return QMM_ERR_SHAPE;
    if (n == 0 || m == 0) return QMM_OK;
    if (!W || !x_host || !y_host) return QMM_ERR_ARG;
    if (!aligned16(W)) return QMM_ERR_ALIGN;
    if (!workspace || ws_bytes < qmm_workspace_bytes_f32_host(t, n, k, m)) return QMM_ERR_WORKSPACE;
    if (!aligned256(workspace)) return QMM_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(workspace);
    const size_t io = host_io_bytes(n, k, m);
    // Page-locked host buffers are mapped into the device's address space: the kernels read
    // x and write y there in place, over the CPU-GPU link, instead of a copy engine moving
    // them before and after (a copy is a separate operation on the stream, with its own
    // start-up, between which the kernel cannot begin).  y goes through a device copy when
    // it is large.  Pageable buffers always take the copies.
    const float *x_in = static_cast<const float *>(mapped_host(x_host, 16));
    float *y_out = size_t(m) * size_t(n) * 4 <= kMappedOutMax ? static_cast<float *>(const_cast<void *>(mapped_host(y_host, 16))) : nullptr;
    if (!x_in) {
        float *x_dev = reinterpret_cast<float *>(base);
        if (cudaMemcpyAsync(x_dev, x_host, size_t(m) * size_t(k) * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return QMM_ERR_CUDA;
        x_in = x_dev;
    }
    float *y_dev = y_out ? y_out : reinterpret_cast<float *>(base + align256(size_t(m) * size_t(k) * 4));
    s = qmm_mul_mat_f32(W, t, n, k, x_in, m, y_dev, base + io, ws_bytes - io, stream);
    if (s != QMM_OK) return s;
    if (!y_out &&
        cudaMemcpyAsync(y_host, y_dev, size_t(m) * size_t(n) * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return QMM_ERR_CUDA;
    return QMM_OK;
}

}  // extern "C"

namespace qmm {
qmm_status mul_mat_q8(const void *W, qmm_type t, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                      void *workspace, size_t ws_bytes, cudaStream_t st, int64_t stride) {
    switch (choose_path(t, n, k, m, stride)) {
    case kGemv: return cuda_status(launch_gemv(t, W, n, k, xq, nullptr, m, y, st, stride));
    case kGemvMma: return cuda_status(launch_gemv_mma(t, W, n, k, xq, m, y, st));
    case kGemvTc: {
        const size_t need = gemv_tc_workspace_bytes(t, n, k, m);
        if (!workspace || ws_bytes < need) return QMM_ERR_WORKSPACE;
        if (!aligned256(workspace)) return QMM_ERR_ALIGN;
        return cuda_status(launch_gemv_tc(t, W, n, k, xq, m, y, workspace, ws_bytes, st));
    }
    case kGemmTc: {
        const size_t need = gemm_tc_workspace_bytes(t, n, k, m, stride);
        if (need > 0) {
            if (!workspace || ws_bytes < need) return QMM_ERR_WORKSPACE;
            if (!aligned256(workspace)) return QMM_ERR_ALIGN;
        }
        return cuda_status(launch_gemm_tc(t, W, n, k, xq, m, y, workspace, ws_bytes,
                                          g_stream_k_mode.load(std::memory_order_relaxed), st, stride));
    }
    default: return cuda_status(launch_gemm_dp4a(t, W, n, k, xq, m, y, st, stride));
    }
}
}  // namespace qmm

extern "C" {

qmm_status qmm_mul_mat_id(const void *W_experts, qmm_type t, int64_t n_experts, int64_t n, int64_t k,
                          const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens, float *y,
                          void *workspace, size_t ws_bytes, void *stream) {
    return mul_mat_id_common(W_experts, t, n_experts, n, k, xq, ids, top_k, n_tokens, false, y, workspace, ws_bytes,
                             stream);
}

qmm_status qmm_mul_mat_id_slot(const void *W_experts, qmm_type t, int64_t n_experts, int64_t n, int64_t k,
                               const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens, float *y,
                               void *workspace, size_t ws_bytes, void *stream) {
    return mul_mat_id_common(W_experts, t, n_experts, n, k, xq, ids, top_k, n_tokens, true, y, workspace, ws_bytes,
                             stream);
}

size_t qmm_workspace_bytes_id_glu(qmm_type t, int64_t n, int64_t k, int64_t n_tokens, int64_t n_experts,
                                  int64_t top_k) {
    if (moe_check_sizes(t, n_experts, n, k, top_k, n_tokens) != QMM_OK) return 0;
    return moe_glu_workspace_bytes(t, n, k, n_tokens, n_experts, top_k);
}

qmm_status qmm_mul_mat_id_glu(const void *W_gate, const void *W_up, qmm_type t, int64_t n_experts, int64_t n, int64_t k,
                              const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens, float *y,
                              void *workspace, size_t ws_bytes, void *stream) {
    qmm_status s = moe_check_sizes(t, n_experts, n, k, top_k, n_tokens);
    if (s != QMM_OK) return s;
    if (!workspace) return QMM_ERR_WORKSPACE;
    if (!aligned256(workspace)) return QMM_ERR_ALIGN;
    if (ws_bytes < moe_glu_workspace_bytes(t, n, k, n_tokens, n_experts, top_k)) return QMM_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n == 0 || n_tokens == 0) return cuda_status(cudaMemsetAsync(workspace, 0, 16, st));
    s = moe_check_pointers(W_gate, xq, ids, y);
    if (s != QMM_OK) return s;
    if (!W_up) return QMM_ERR_ARG;
    if (!aligned16(W_up)) return QMM_ERR_ALIGN;
    return cuda_status(launch_mul_mat_id_glu(t, W_gate, W_up, n_experts, n, k, xq, ids, top_k, n_tokens, false, y,
                                             workspace, ws_bytes, st));
}

qmm_status qmm_read_device_status(const void *workspace, int32_t *status, void *stream) {
    if (!workspace || !status) return QMM_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, static_cast<const uint8_t *>(workspace) + kStatusOffset, sizeof(v),
                        cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return QMM_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return QMM_ERR_CUDA;
    *status = v;
    return QMM_OK;
}

size_t qmm_aligned_row_bytes(qmm_type t, int64_t k) { return type_ok(t) ? size_t(aligned_row_bytes(t, k)) : 0; }

size_t qmm_workspace_bytes_aligned(qmm_type t, int64_t n, int64_t k, int64_t m) {
    if (!type_ok(t) || n < 0 || k <= 0 || m < 0 || check_k(t, k) != QMM_OK) return 0;
    const int64_t stride = aligned_row_bytes(t, k);
    const size_t gemm = gemm_tc_supported(t, n, k, m, stride) ? gemm_tc_workspace_bytes(t, n, k, m, stride) : 0;
    return std::max(gemm, gemv_tc_workspace_bytes(t, n, k, m));
}

qmm_status qmm_repack_aligned(const void *W, qmm_type t, int64_t n, int64_t k, void *W_aligned, void *stream) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n < 0) return QMM_ERR_ARG;
    if (n > kMaxRows) return QMM_ERR_SHAPE;
    if (n == 0) return QMM_OK;
    if (!W || !W_aligned) return QMM_ERR_ARG;
    if (!aligned16(W) || !aligned16(W_aligned)) return QMM_ERR_ALIGN;
    const int64_t rb = int64_t(qmm_row_bytes(t, k)), stride = aligned_row_bytes(t, k);
    const int unit = rb % 8 == 0 ? 8 : rb % 4 == 0 ? 4 : 2;
    const int64_t total = n * (stride / unit);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, int64_t(device_sm_count()) * 8));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t *src = static_cast<const uint8_t *>(W);
    uint8_t *dst = static_cast<uint8_t *>(W_aligned);
    if (unit == 8) repack_aligned_kernel<8><<<grid, 256, 0, st>>>(src, n, rb, stride, dst);
    else if (unit == 4) repack_aligned_kernel<4><<<grid, 256, 0, st>>>(src, n, rb, stride, dst);
    else repack_aligned_kernel<2><<<grid, 256, 0, st>>>(src, n, rb, stride, dst);
    return cuda_status(cudaGetLastError());
}

qmm_status qmm_mul_mat_aligned(const void *W_aligned, qmm_type t, int64_t n, int64_t k, const void *xq, int64_t m,
                               float *y, void *workspace, size_t ws_bytes, void *stream) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n < 0 || m < 0) return QMM_ERR_ARG;
    if (n > kMaxRows || m > kMaxRows) return QMM_ERR_SHAPE;
    if (n == 0 || m == 0) return QMM_OK;
    if (!W_aligned || !xq || !y) return QMM_ERR_ARG;
    if (!aligned16(W_aligned) || !aligned16(xq) || !aligned16(y)) return QMM_ERR_ALIGN;
    return mul_mat_q8(W_aligned, t, n, k, xq, m, y, workspace, ws_bytes, static_cast<cudaStream_t>(stream),
                      aligned_row_bytes(t, k));
}

qmm_status qmm_get_device_status(const void *workspace, void *stream) {
    int32_t v = 0;
    const qmm_status s = qmm_read_device_status(workspace, &v, stream);
    return s != QMM_OK ? s : static_cast<qmm_status>(v);
}

int qmm_tile_efficiency_percent(int64_t ntiles, int64_t nsm) {
    if (ntiles <= 0 || nsm <= 0) return 0;
    const int64_t nwaves = (ntiles + nsm - 1) / nsm;
    return (int)(100 * ntiles / (nsm * nwaves));
}

int qmm_gemv_ring_stages(qmm_type t, int64_t n, int64_t k, int32_t ncols, int64_t smem_bytes) {
    if (n <= 0 || ncols < 1 || ncols > 8 || smem_bytes <= 0 || check_k(t, k) != QMM_OK) return 0;
    return gemv_ring_stages(t, n, k, ncols, size_t(smem_bytes));
}

qmm_status qmm_plan_gemm(qmm_type t, int64_t n, int64_t k, int64_t m, int32_t nsm, int32_t stream_k_mode,
                         qmm_gemm_plan *plan) {
    qmm_status s = check_k(t, k);
    if (s != QMM_OK) return s;
    if (n <= 0 || m <= 0 || nsm <= 0 || !plan) return QMM_ERR_ARG;
    qmm_gemm_plan p{};
    p.tile_n = 128;
    p.tile_m = (int32_t)gemm_tc_tile_m(m);
    p.iter_k = 256;
    p.tiles_n = (n + p.tile_n - 1) / p.tile_n;
    p.tiles_m = (m + p.tile_m - 1) / p.tile_m;
    p.ntiles = p.tiles_n * p.tiles_m;
    p.iters_per_tile = (k + p.iter_k - 1) / p.iter_k;
    p.nwork = p.ntiles * p.iters_per_tile;
    p.efficiency_percent = qmm_tile_efficiency_percent(p.ntiles, nsm);
    const bool sk = stream_k_mode == 2 || (stream_k_mode == 0 && p.efficiency_percent < 90);
    if (!sk) {
        p.stream_k = 0;
        p.ctas = (int32_t)std::min<int64_t>(p.ntiles, kMaxRows);
        p.fixup = 0;
    } else {
        p.stream_k = 1;
        p.ctas = (int32_t)std::min<int64_t>(nsm, p.nwork);
        p.fixup = 0;
        for (int32_t c = 1; c < p.ctas; ++c) {
            const int64_t b = (int64_t)c * p.nwork / p.ctas;
            if (b % p.iters_per_tile) {
                p.fixup = 1;
                break;
            }
        }
    }
    *plan = p;
    return QMM_OK;
}

void qmm_plan_cta_range(const qmm_gemm_plan *plan, int32_t cta, int64_t *begin, int64_t *end) {
    if (!plan || !begin || !end || cta < 0 || cta >= plan->ctas) {
        if (begin) *begin = 0;
        if (end) *end = 0;
        return;
    }
    if (!plan->stream_k) {
        *begin = (int64_t)cta * plan->iters_per_tile;
        *end = *begin + plan->iters_per_tile;
        return;
    }
    *begin = (int64_t)cta * plan->nwork / plan->ctas;
    *end = (int64_t)(cta + 1) * plan->nwork / plan->ctas;
}

void qmm_set_force_path(int path) { g_force_path.store(path, std::memory_order_relaxed); }
void qmm_set_stream_k_mode(int mode) { g_stream_k_mode.store(mode, std::memory_order_relaxed); }
void qmm_set_test_fault(int mode) { g_test_fault.store(mode, std::memory_order_relaxed); }

}  // extern "C"
