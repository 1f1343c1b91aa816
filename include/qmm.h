/*
 * qmm.h -- C ABI of the block-quantized matmul library for GB300 (sm_103a).
 *
 * The library computes y[m][n] = sum_k x[m][k] * dequant(W)[n][k] with W kept in
 * its block-quantized form (Q4_K, Q5_K, Q6_K, Q8_0 or Q4_0) and x quantized to q8_1 first.
 * Every product is formed from exact integer sub-block dot products that are
 * then folded with the block scales in fp32.
 *
 * Sources (web pages on block-quantized matmul), cited by title and section:
 *   [MMQ]   "llama.cpp 源码完全拆解(十五): 量化 GEMM 的矩阵编队 -- MMQ 如何把 MoE 与预填充塞满 GPU"
 *   [P0007] "Patch 0007: an fp16 matrix-vector path for GP100"
 *   [QMM]   "QTensor 与 QMatMul" (candle 0.11.0 notes)
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller, except the host
 *     buffers of qmm_mul_mat_f32_host.  The library keeps no reference to them after
 *     a call returns and allocates no device memory per call: scratch lives in the
 *     caller's workspace.
 *   - Every call enqueues its work on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns without synchronising the host, except the two
 *     status reads and qmm_mul_mat_f32_host with a pageable y_host.
 *   - Row-major layouts.  W is [n] rows of k/QK blocks, one row per output
 *     feature, as PyTorch Linear stores weights ([QMM] section "QMatMul:
 *     三种形态": weights are stored [n, k]).  x is [m][k] fp32, y is [m][n] fp32.
 *   - Argument errors are returned synchronously and nothing is enqueued.
 *     QMM_ERR_CUDA reports a failed launch (cudaGetLastError after the launch).
 *   - The library works on the CUDA device that is current when a call is made.
 *
 * Block formats (bytes, little-endian fp16 fields):
 *   q8_1 (36 B / 32 values): fp16 d, fp16 s, int8 q[32]; s = d * sum(q)
 *        ([MMQ] section "dp4a 路径的 Q4_K": the activation block carries d and s).
 *   Q4_K (144 B / 256):      fp16 d, fp16 dmin, 12 B of 6-bit sub-block scales
 *        and mins, 128 B of nibbles; w = d*sc*q - dmin*m
 *        ([MMQ] section "Q4_K: 在加载期就把两层 scale 合并成 half2").
 *   Q5_K (176 B / 256):      fp16 d, fp16 dmin, 12 B of scales/mins (Q4_K's rule), qh[32],
 *        128 B of nibbles in Q4_K's order; the fifth bit of weight 32j + l is bit j of
 *        qh[l]; w = d*sc*q - dmin*m with q in 0..31 ([MMQ] section "Q4_K: 在加载期就把两层
 *        scale 合并成 half2": Q4_K and Q5_K share the scale unpack; the bit plane's layout
 *        is this library's reading).
 *   Q6_K (210 B / 256):      ql[128], qh[64], int8 scales[16], fp16 d;
 *        w = d*sc*(code-32) ([MMQ] section "Q6_K: 6 位数据要多占一半的共享内存").
 *   Q8_0 (34 B / 32):        fp16 d, int8 q[32]; w = d*q.
 *   Q4_0 (18 B / 32):        fp16 d, 16 B of nibbles, byte i holding weight i in its
 *        low nibble and weight 16+i in its high nibble; w = d*(q-8), and the integer
 *        dot runs on the offset codes q-8 ([MMQ] sections "tile_x_sizes" and
 *        "Q4_0: 一个 get_int_b2 搬进 8 个 4-bit").
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { QMM_Q4_0 = 2, QMM_Q8_0 = 8, QMM_Q4_K = 12, QMM_Q5_K = 13, QMM_Q6_K = 14 } qmm_type;

typedef enum {
    QMM_OK = 0,
    QMM_ERR_ARG = 1,       /* null pointer, m/n/k/top_k/n_experts <= 0 where not allowed */
    QMM_ERR_SHAPE = 2,     /* k not a multiple of the block size, or a size above the library limits */
    QMM_ERR_TYPE = 3,      /* unknown qmm_type */
    QMM_ERR_ALIGN = 4,     /* a pointer not 16-byte aligned */
    QMM_ERR_WORKSPACE = 5, /* workspace smaller than qmm_workspace_bytes() */
    QMM_ERR_CUDA = 6,      /* a CUDA runtime call or kernel launch failed */
    QMM_ERR_IDS = 7,       /* device status only: a routing id was outside [0, n_experts) */
    QMM_ERR_DEVICE = 8     /* device status only: a kernel gave up on a bounded wait */
} qmm_status;

/* Human-readable name of a status code (static string). */
QMM_API const char *qmm_status_string(qmm_status s);

/* Bytes of the q8_1 blocks for an [m][k] activation: m * (k/32) * 36. */
QMM_API size_t qmm_q8_1_bytes(int64_t m, int64_t k);

/* Bytes of one weight row of k values in format t (k/QK blocks), 0 if k is not a
 * multiple of the block size or t is unknown. */
QMM_API size_t qmm_row_bytes(qmm_type t, int64_t k);

/* Workspace bytes that qmm_mul_mat (n_experts == 0) or qmm_mul_mat_id
 * (n_experts > 0) needs for these sizes on the CURRENT device (the tensor-core
 * paths keep one partial-sum slot per SM, so the figure depends on the SM count:
 * size the workspace with the device current on which the call will run).  The
 * workspace must be 256-byte aligned device memory; its contents need no
 * initialisation.  0 for a type or sizes that the call rejects. */
QMM_API size_t qmm_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t m, int64_t n_experts, int64_t top_k);

/*
 * Quantize fp32 activations to q8_1 ([MMQ] sections "引言" and
 * "mul_mat_id 的第三条路": activations stay fp32 and are compressed to q8_1 on
 * the device; [QMM] section "CPU: 先量化激活, 再逐行点积").
 *   x   : fp32 [m][k], 16-byte aligned, k % 32 == 0.
 *   xq  : output, qmm_q8_1_bytes(m, k) bytes, 16-byte aligned; block (r, b)
 *         at byte (r*(k/32) + b)*36.
 * Per 32-block: d = amax/127 (fp32), q = round-half-away(x/d) (IEEE fp32 division),
 * stored fp16 d and s = fp16(d_stored * sum(q)); a block whose fp32 d is 0 is all
 * zero.  The result is bit-identical on every run.  Non-finite x is outside the
 * contract (the q values of such a block are unspecified).
 */
QMM_API qmm_status qmm_quantize_q8_1(const float *x, int64_t m, int64_t k, void *xq, void *stream);

/*
 * y = x * dequant(W)^T with x given as q8_1 blocks ([MMQ] sections "形状判据",
 * "dp4a 路径的 Q4_K", "Q6_K: 子块尺度与 q8_1 块长错位"; [QMM] section "QMatMul").
 *   W      : [n][k/QK] blocks of type t, contiguous rows, 16-byte aligned.
 *   xq     : q8_1 blocks of x [m][k] as written by qmm_quantize_q8_1.
 *   y      : fp32 [m][n] output, 16-byte aligned; every element is written.
 *   workspace, ws_bytes: at least qmm_workspace_bytes(t, n, k, m, 0, 0) bytes.
 * k % 256 == 0 for Q4_K/Q5_K/Q6_K, k % 32 == 0 for Q8_0/Q4_0.  Paths (each weight byte is
 * read once, every column reusing the decoded weight):
 *   Q4_K, m <= 5:       the bulk-copy GEMV (dp4a);
 *   Q4_K, 6 <= m <= 8:  the multi-column GEMV on the warp-level MMA (the columns as its N
 *                       side) where its two tile stages fit shared memory, else the above;
 *   Q4_K, 9 <= m <= 16: the skinny tensor-core path (weight rows as the MMA's M side);
 *   Q4_K, m > 16:       the tiled tensor-core GEMM;
 *   Q5_K, m <= 8:       the bulk-copy GEMV; m > 8: the tiled tensor-core GEMM;
 *   Q6_K/Q8_0, m <= 8:  the bulk-copy GEMV;
 *   Q6_K/Q8_0, m > 8:   the tiled tensor-core GEMM (Q8_0: k % 256 == 0; Q6_K: n % 8
 *                       == 0), otherwise the CUDA-core tiled GEMM;
 *   Q4_0, m <= 8:       the bulk-copy GEMV (k % 256 == 0, else the direct-load GEMV);
 *   Q4_0, m > 8:        the tiled tensor-core GEMM when k % 256 == 0, otherwise the
 *                       CUDA-core tiled GEMM;
 * the tensor-core paths split their work with a stream-K schedule.
 * Accuracy: |y - y_exact| <= 1e-5 * sum over blocks of |block term| per element.
 */
QMM_API qmm_status qmm_mul_mat(const void *W, qmm_type t, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                       void *workspace, size_t ws_bytes, void *stream);

/*
 * The same product from fp32 activations: the call quantizes x to q8_1 itself
 * (qmm_quantize_q8_1's arithmetic, to the bit) and then multiplies, so that
 *   qmm_mul_mat_f32(W, t, n, k, x, m, y, ...)
 * gives exactly the y of qmm_quantize_q8_1(x) followed by qmm_mul_mat ([MMQ]
 * section "引言": the activations stay fp32 and are quantized on the device).
 *   x  : fp32 [m][k], 16-byte aligned, k % 32 == 0 (and the format's block size).
 *   W, y, stream: as qmm_mul_mat.
 *   workspace: at least qmm_workspace_bytes_f32(t, n, k, m) bytes, 256-byte aligned.
 *              When m == 1 and the GEMV runs, the workspace is not used (may be NULL):
 *              that case is ONE launch in which every CTA quantizes x into its shared
 *              memory while its first weight copies are in flight.  Otherwise the
 *              q8_1 blocks go to the head of the workspace (the quantizer kernel writes
 *              them) and the rest is the qmm_mul_mat workspace.
 * Errors as qmm_mul_mat (QMM_ERR_WORKSPACE when the workspace is needed and short).
 */
QMM_API size_t qmm_workspace_bytes_f32(qmm_type t, int64_t n, int64_t k, int64_t m);
QMM_API qmm_status qmm_mul_mat_f32(const void *W, qmm_type t, int64_t n, int64_t k, const float *x, int64_t m,
                                   float *y, void *workspace, size_t ws_bytes, void *stream);

/*
 * qmm_mul_mat_f32 with x and y in HOST memory, all on `stream` (an interface of this
 * library; the pages have no counterpart).  The same y as qmm_mul_mat_f32 to the bit.
 *   x_host : fp32 [m][k]; y_host : fp32 [m][n].  A page-locked buffer (16-byte aligned;
 *            y up to 1 MB) is read or written by the kernels in place through its mapped
 *            device address; any other buffer goes through a copy into or out of the
 *            workspace.  The host buffers must stay valid, and y_host unread, until the
 *            stream has passed the call.  With pageable y_host the runtime makes the copy
 *            back synchronous, so the call returns with y in y_host.
 *   workspace : at least qmm_workspace_bytes_f32_host(t, n, k, m) bytes, 256-byte
 *            aligned: room for device copies of x and y at its head (used by the
 *            buffers that are copied), then the qmm_mul_mat_f32
 *            workspace.
 * Errors as qmm_mul_mat_f32; QMM_ERR_CUDA if a copy cannot be enqueued.
 */
QMM_API size_t qmm_workspace_bytes_f32_host(qmm_type t, int64_t n, int64_t k, int64_t m);
QMM_API qmm_status qmm_mul_mat_f32_host(const void *W, qmm_type t, int64_t n, int64_t k, const float *x_host,
                                        int64_t m, float *y_host, void *workspace, size_t ws_bytes, void *stream);

/*
 * Fused gate/up matmul with SwiGLU ([MMQ] sections "「分专家」与「整批」之间: host 侧的
 * 代价" and "输出端: 写回与 scale 修正": the gate and up weights are loaded and dotted
 * together and the GLU is applied right after the dots; [P0007]: fused ffn
 * gate/up/SWIGLU):
 *   y[m][n] = silu(x * dequant(W_gate)^T) * (x * dequant(W_up)^T),  silu(g) = g / (1 + e^-g)
 *   W_gate, W_up : [n][k/QK] blocks of type t each, 16-byte aligned.
 *   xq, m, y, stream : as qmm_mul_mat (y is [m][n]).
 *   workspace : at least qmm_workspace_bytes_glu(t, n, k, m) bytes, 256-byte aligned
 *               (may be NULL when that is 0).
 * Paths: Q4_K, m <= 8: one bulk-copy GEMV reading both weights once (each output's
 * gate and up rows are folded by the two halves of one warp); Q4_K, m > 8: the
 * tensor-core GEMM with gate and up rows interleaved in its tile (one thread holds both
 * dots of an output), whole tiles only, no stream-K; other types and shapes: the two
 * products into the workspace, then a combine pass.  Accuracy: each dot within 1e-5
 * of its sum of |block terms|, carried through silu(g) * u to first order, plus
 * 2^-20 |y| for evaluating silu and the product in fp32, plus 2^-120 |u| where silu
 * underflows fp32 (gate dots below -88.7 give 0).
 */
QMM_API size_t qmm_workspace_bytes_glu(qmm_type t, int64_t n, int64_t k, int64_t m);
QMM_API qmm_status qmm_mul_mat_glu(const void *W_gate, const void *W_up, qmm_type t, int64_t n, int64_t k,
                                   const void *xq, int64_t m, float *y, void *workspace, size_t ws_bytes,
                                   void *stream);

/*
 * One-time repack of a gate/up pair into one interleaved tensor (the optional weight
 * repack; llama.cpp interleaves up and gate rows when it loads its fused tile, [MMQ]
 * section "输出端: 写回与 scale 修正"; [QMM] section "Q4K 的 8 列重排": a repack keeps a
 * second copy of the weights, so the caller owns both and may free the pair after):
 *   W_gu row 2j = W_gate row j, row 2j+1 = W_up row j, bytes copied unchanged.
 *   W_gate, W_up : [n][k/QK] blocks of type t; W_gu : [2n][k/QK], all 16-byte aligned.
 * Enqueued on stream like every call; W_gu is ready when the stream reaches it.
 */
QMM_API qmm_status qmm_repack_glu(const void *W_gate, const void *W_up, qmm_type t, int64_t n, int64_t k, void *W_gu,
                                  void *stream);

/*
 * qmm_mul_mat_glu on the interleaved tensor of qmm_repack_glu: the same y, and to the
 * bit on the fused paths (Q4_K), which fold the same rows in the same order: the GEMV
 * then streams each chunk of 4 outputs (gate and up rows) with one copy instead of two,
 * and the tensor-core GEMM loads a tile's gate and up rows as one box.  Other types
 * and shapes: one product of the 2n rows into the workspace and a combine pass, within
 * the bound of qmm_mul_mat_glu.  workspace: qmm_workspace_bytes_glu(t, n, k, m).
 */
QMM_API qmm_status qmm_mul_mat_glu_packed(const void *W_gu, qmm_type t, int64_t n, int64_t k, const void *xq,
                                          int64_t m, float *y, void *workspace, size_t ws_bytes, void *stream);

/*
 * One-time repack of W into rows padded to whole 16-byte units (the optional weight
 * repack; [QMM] section "Q4K 的 8 列重排": a one-time repack done when the weights are
 * loaded, kept as a second copy, so the caller owns both and may free the original).
 * Blocks are copied unchanged; row r of W_aligned starts at r * qmm_aligned_row_bytes(t, k)
 * and the bytes after its k/QK blocks are zero.  Q6_K rows (210-byte blocks) and Q8_0/Q4_0
 * rows (34/18-byte blocks) are generally not whole 16-byte units: padded, every row can
 * be streamed by 16-byte bulk copies.  Q6_K rows get room for the 14 bytes by which the
 * tensor-core GEMM's 16-byte-aligned copy window of a superblock can run past its row,
 * which lifts that path's n % 8 == 0 condition.  Q4_K rows are whole units already, and
 * padded rows equal W.
 *   W : [n][k/QK] blocks, 16-byte aligned; W_aligned : n * qmm_aligned_row_bytes(t, k)
 *       bytes, 16-byte aligned.  Enqueued on stream.
 */
QMM_API size_t qmm_aligned_row_bytes(qmm_type t, int64_t k);
QMM_API qmm_status qmm_repack_aligned(const void *W, qmm_type t, int64_t n, int64_t k, void *W_aligned,
                                      void *stream);

/*
 * qmm_mul_mat on the padded rows of qmm_repack_aligned: the same product within the same
 * bound (the kernels decode the same blocks; only where each row starts differs), with the
 * bulk-copy GEMV for every Q6_K/Q8_0/Q4_0 shape and the tensor-core GEMM for Q6_K at any n.
 *   workspace : at least qmm_workspace_bytes_aligned(t, n, k, m) bytes, 256-byte aligned.
 * Other arguments and errors as qmm_mul_mat.
 */
QMM_API size_t qmm_workspace_bytes_aligned(qmm_type t, int64_t n, int64_t k, int64_t m);
QMM_API qmm_status qmm_mul_mat_aligned(const void *W_aligned, qmm_type t, int64_t n, int64_t k, const void *xq,
                                       int64_t m, float *y, void *workspace, size_t ws_bytes, void *stream);

/*
 * Expert-routed matmul ([MMQ] sections "派发路径", "专家边界: 在 GPU 上做分段,
 * 而不是在 host 上", "MoE 的二次账"):
 *   y[t][s][:] = x[t] * dequant(W_experts[ids[t][s]])^T
 *   W_experts : [n_experts][n][k/QK] blocks of type t, 16-byte aligned.
 *   xq        : q8_1 blocks of x [n_tokens][k]; a token's row is shared by all
 *               of its top_k slots.
 *   ids       : int32 [n_tokens][top_k] expert ids (device memory).
 *   y         : fp32 [n_tokens][top_k][n]; every element is written.
 *   workspace : at least qmm_workspace_bytes(t, n, k, n_tokens, n_experts, top_k)
 *               bytes; it also holds the device status word read by
 *               qmm_read_device_status.
 * The host never reads ids, so the call does not synchronise.  A pair whose id is
 * outside [0, n_experts) gets a zero output row and sets QMM_ERR_IDS in the status
 * word.  Paths:
 *   n_tokens * top_k <= 32 (decode): one bulk-copy GEMV per (token, slot) pair, the
 *     pair's expert id read on the device (for the shapes the GEMV streams: Q4_K
 *     always, Q8_0 and Q4_0 with k/32 % 8 == 0, Q6_K with 16-byte rows or even n);
 *   otherwise the pairs are bucketed by expert on the device (a stable counting sort)
 *     and the per-expert tiles are walked by one persistent launch: with k % 256 == 0
 *     (and for Q6_K n % 8 == 0) on the tensor cores (128-pair tiles from a device-built
 *     list, whole tiles per CTA when they fill 90% of the CTAs' rounds, else stream-K;
 *     the workspace then also holds an fp16 copy of the gathered activations), other
 *     shapes on the CUDA-core grouped GEMM.  For Q4_K the
 *     experts with 1..16 pairs ([MMQ] section "MoE 的二次账": experts whose few columns
 *     leave the tiles mostly empty) skip the 128-pair tiles: a second launch runs them
 *     as 16-column slabs on the skinny tensor-core kernel, the expert list and its
 *     length read on the device.
 */
QMM_API qmm_status qmm_mul_mat_id(const void *W_experts, qmm_type t, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                          const int32_t *ids, int64_t top_k, int64_t n_tokens, float *y, void *workspace,
                          size_t ws_bytes, void *stream);

/*
 * qmm_mul_mat_id with one activation row per (token, slot) pair, as in a MoE down
 * projection, where each slot's input is that expert's own up/gate output:
 *   y[t][s][:] = x[t][s] * dequant(W_experts[ids[t][s]])^T
 *   xq : q8_1 blocks of x [n_tokens][top_k][k] (pair (t, s) at row t*top_k + s).
 * Everything else (arguments, workspace size, status word, paths) is as for
 * qmm_mul_mat_id.
 */
QMM_API qmm_status qmm_mul_mat_id_slot(const void *W_experts, qmm_type t, int64_t n_experts, int64_t n, int64_t k,
                                       const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens, float *y,
                                       void *workspace, size_t ws_bytes, void *stream);

/*
 * Expert-routed fused gate/up with SwiGLU ([MMQ] section "「分专家」与「整批」之间: host
 * 侧的代价": in the MoE FFN the gate and up products of a tile are formed together and
 * the GLU applied right after the dots; [P0007] Coverage: fused ffn gate/up/SWIGLU):
 *   y[t][s][j] = silu(g) * u,  g = x[t] . dequant(W_gate[e])[j],  u = x[t] . dequant(W_up[e])[j],
 *   e = ids[t][s], silu(g) = g / (1 + exp(-g)).
 *   W_gate, W_up : device, each [n_experts][n][k/QK] blocks of type t (the experts' gate
 *                  and up weights, one tensor each), 16-byte aligned
 *   xq, ids, top_k, n_tokens, y : as qmm_mul_mat_id (x shared by a token's slots)
 *   workspace    : device, 256-byte aligned, at least qmm_workspace_bytes_id_glu(...)
 *                  bytes; its status word reads as for qmm_mul_mat_id
 * Paths: one fused GEMV per (token, slot) pair for n_tokens * top_k <= 32 (Q4_K); the
 * fused expert-grouped tensor-core GEMM (Q4_K; every expert on 128-pair tiles, each tile
 * computed whole); otherwise both products into the workspace and a combine pass.  An id
 * outside [0, n_experts) gives a zero row and QMM_ERR_IDS in the status word.  Errors as
 * qmm_mul_mat_id; W_up must be given.
 */
QMM_API size_t qmm_workspace_bytes_id_glu(qmm_type t, int64_t n, int64_t k, int64_t n_tokens, int64_t n_experts,
                                          int64_t top_k);
QMM_API qmm_status qmm_mul_mat_id_glu(const void *W_gate, const void *W_up, qmm_type t, int64_t n_experts, int64_t n,
                                      int64_t k, const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens,
                                      float *y, void *workspace, size_t ws_bytes, void *stream);

/*
 * qmm_mul_mat_id without a workspace argument, for callers that cannot allocate
 * device memory where they make this call (a fixed memory pool owned by someone
 * else, a plugin that may not call cudaMalloc, code that runs between graph
 * captures).  The pages have no counterpart of this call.
 *   Arguments, layouts and results are those of qmm_mul_mat_id.
 *   Scratch: one file-scope device array of qmm_noalloc_scratch_bytes() (1 MiB),
 *   present in every GPU that loads the library until the process exits.  Up to 32
 *   (token, slot) pairs this call runs one GEMV per pair (as qmm_mul_mat_id does),
 *   which needs only the status word; beyond that it runs the CUDA-core grouped
 *   GEMM, whose scratch is the bucketing state alone: 256 B of status,
 *   4*(n_experts+1) B of bounds, 4 B per (token, slot) pair, 16 B per tile
 *   (pairs/64 + n_experts + 1 tiles) and 4*n_experts B of cold-expert list, each
 *   piece rounded up to 256 B, so up to about 240K pairs fit (fewer with many
 *   experts).  A larger problem is rejected with QMM_ERR_WORKSPACE and nothing is
 *   enqueued.  The call allocates nothing and frees nothing.
 *   The first call in a device and CUDA context looks up the array's device
 *   address (with that device current); make that first call before any stream
 *   capture.  Every call on a device shares the array: calls whose work can
 *   overlap on the GPU (different streams without ordering) race on it.
 *   The device status word is kept in the array and is not reported.
 */
QMM_API qmm_status qmm_mul_mat_id_noalloc(const void *W_experts, qmm_type t, int64_t n_experts, int64_t n, int64_t k,
                                          const void *xq, const int32_t *ids, int64_t top_k, int64_t n_tokens,
                                          float *y, void *stream);

/* Size in bytes of the fixed scratch array used by qmm_mul_mat_id_noalloc. */
QMM_API size_t qmm_noalloc_scratch_bytes(void);

/* Copy the device status word of the last qmm_mul_mat_id on this workspace to
 * *status (QMM_OK, QMM_ERR_IDS or QMM_ERR_DEVICE).  This call synchronises
 * `stream`.  Returns QMM_ERR_CUDA if the copy fails. */
QMM_API qmm_status qmm_read_device_status(const void *workspace, int32_t *status, void *stream);

/* The same status word as the return value: QMM_OK, QMM_ERR_IDS (a routing id was
 * outside [0, n_experts)) or QMM_ERR_DEVICE (a kernel gave up on a bounded wait), as
 * written by the last qmm_mul_mat_id / qmm_mul_mat_id_slot / qmm_mul_mat_id_glu enqueued on this workspace
 * and `stream`.  Synchronises `stream` (a host read of a device flag has to wait for
 * the writer).  QMM_ERR_ARG for a NULL workspace, QMM_ERR_CUDA if the read fails, so a
 * caller that must tell a failed read from a device error uses qmm_read_device_status. */
QMM_API qmm_status qmm_get_device_status(const void *workspace, void *stream);

/* ------------------------------------------------------------------ host-side planning
 * These functions run on the host only and never touch a GPU. */

/* Tile efficiency of one-tile-per-CTA scheduling ([MMQ] section
 * "朴素切法的负载缺口"): nwaves = ceil(ntiles/nsm), percent = 100*ntiles/(nsm*nwaves). */
QMM_API int qmm_tile_efficiency_percent(int64_t ntiles, int64_t nsm);

/* Schedule of one GEMM launch ([MMQ] sections "stream-K 的切法",
 * "fixup: 部分和的归约", "什么时候不用 stream-K"). */
typedef struct {
    int64_t tiles_n;      /* tiles along the W rows (n) */
    int64_t tiles_m;      /* tiles along the activation rows (m) */
    int64_t ntiles;       /* tiles_n * tiles_m */
    int64_t iters_per_tile; /* K iterations per tile */
    int64_t nwork;        /* ntiles * iters_per_tile */
    int32_t ctas;         /* CTAs launched */
    int32_t stream_k;     /* 1: the flattened (tile, k-iteration) stream is split evenly over ctas */
    int32_t fixup;        /* 1: some tile is shared by two or more CTAs and needs the fixup pass */
    int32_t efficiency_percent; /* qmm_tile_efficiency_percent(ntiles, nsm) */
    int32_t tile_n;       /* W rows per tile */
    int32_t tile_m;       /* activation rows per tile */
    int32_t iter_k;       /* K values per iteration */
} qmm_gemm_plan;

/* Fill *plan for a dense GEMM of these sizes on a GPU with nsm SMs.
 * stream_k_mode: 0 = automatic (stream-K only when the tile efficiency is below 90%),
 * 1 = never, 2 = always.  Returns QMM_ERR_ARG/SHAPE/TYPE on bad sizes. */
QMM_API qmm_status qmm_plan_gemm(qmm_type t, int64_t n, int64_t k, int64_t m, int32_t nsm, int32_t stream_k_mode,
                         qmm_gemm_plan *plan);

/* The half-open range [*begin, *end) of flattened work units (tile * iters_per_tile
 * + k-iteration) that CTA `cta` of the plan processes. */
QMM_API void qmm_plan_cta_range(const qmm_gemm_plan *plan, int32_t cta, int64_t *begin, int64_t *end);

/* Ring depth of the bulk-copy GEMV, which streams the weight rows once through
 * shared-memory stages ([MMQ] section "与 MMVQ 的边界": the m <= 8 path is bound by
 * reading W), for one launch of ncols (1..8) activation columns,
 * given smem_bytes of shared memory per block: the deepest of 8, 6, 4 or 3 stages of 8
 * weight rows that fits.  The consumer groups take the stages in turn, 4 groups for 8
 * and 4 stages (8 groups of 2 warps in the Q4_K row-pair form), 3 for 6 and 3, so that
 * each stage always goes to the same group.  0
 * when the rows cannot be streamed in whole 16-byte units (Q8_0 and Q4_0 unless k/32
 * is a multiple of 8; Q6_K unless k/256 is a multiple of 8, or of 4 with n even) or
 * when not even 3 stages fit next to the staged activations (Q4_K at one column from
 * k = 15616 on, with 227 KB): the call then runs on the direct-load GEMV kernel.  Bad
 * arguments give 0. */
QMM_API int qmm_gemv_ring_stages(qmm_type t, int64_t n, int64_t k, int32_t ncols, int64_t smem_bytes);

/* ------------------------------------------------------------------ test controls
 * Process-wide switches for tests and benchmarks; read at every call. */

/* Path override for qmm_mul_mat: 0 = automatic, 1 = GEMV for any m <= 64,
 * 2 = the CUDA-core (dp4a) tiled GEMM, 3 = the tensor-core GEMM for any m,
 * 4 = GEMV for any m <= 64 with direct global loads only (no bulk copies),
 * 5 = the skinny tensor-core path (Q4_K, m <= 16), 6 = the multi-column mma.sync GEMV
 * (Q4_K, 1 <= m <= 8).  A forced path that does not
 * support the call's type or sizes falls back to the automatic choice. */
QMM_API void qmm_set_force_path(int path);

/* Stream-K mode for the tensor-core GEMM: 0 = automatic, 1 = never, 2 = always. */
QMM_API void qmm_set_stream_k_mode(int mode);

/* Failure-detection test switch (an interface of this library; the pages have no
 * counterpart).  0 = off.  1 = every tensor-core GEMM launch made while it is set
 * (qmm_mul_mat and the grouped mul_mat_id paths with m > 16) withholds its
 * activation copies, so that the MMA issuer's bounded wait for the first stage runs
 * out (after about 10^5 cycles instead of about a second): the kernel stops, frees
 * its tensor memory and sets QMM_ERR_DEVICE in the workspace's status word, which
 * qmm_read_device_status / qmm_get_device_status return.  No copy is in flight when
 * the kernel leaves and the context stays usable; y is unspecified for that call. */
QMM_API void qmm_set_test_fault(int mode);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
