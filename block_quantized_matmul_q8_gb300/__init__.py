"""Python binding of libqmm (the C ABI in include/qmm.h).

Argument marshalling only: every step of the matmul runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  The functions keep the C
names; tensors are passed as device pointers of contiguous CUDA tensors and the
current torch stream is used unless one is given.

If libqmm.so is missing or cannot be loaded, every call raises QMMError; there is
no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmm.so")

TYPES = {"q4_0": 2, "q8_0": 8, "q4_K": 12, "q5_K": 13, "q6_K": 14}
BLOCK = {"q4_0": (32, 18), "q8_0": (32, 34), "q4_K": (256, 144), "q5_K": (256, 176), "q6_K": (256, 210)}
STATUS = {0: "QMM_OK", 1: "QMM_ERR_ARG", 2: "QMM_ERR_SHAPE", 3: "QMM_ERR_TYPE", 4: "QMM_ERR_ALIGN",
          5: "QMM_ERR_WORKSPACE", 6: "QMM_ERR_CUDA", 7: "QMM_ERR_IDS", 8: "QMM_ERR_DEVICE"}
PATH_AUTO, PATH_GEMV, PATH_GEMM_DP4A, PATH_GEMM_TC, PATH_GEMV_DIRECT, PATH_GEMV_TC, PATH_GEMV_MMA = 0, 1, 2, 3, 4, 5, 6

# Every function that include/qmm.h declares.
EXPORTS = ("qmm_status_string", "qmm_q8_1_bytes", "qmm_row_bytes", "qmm_workspace_bytes", "qmm_quantize_q8_1",
           "qmm_mul_mat", "qmm_mul_mat_id", "qmm_read_device_status", "qmm_tile_efficiency_percent",
           "qmm_plan_gemm", "qmm_plan_cta_range", "qmm_set_force_path", "qmm_set_stream_k_mode",
           "qmm_mul_mat_id_noalloc", "qmm_noalloc_scratch_bytes", "qmm_workspace_bytes_f32", "qmm_mul_mat_f32",
           "qmm_mul_mat_id_slot", "qmm_workspace_bytes_glu", "qmm_mul_mat_glu", "qmm_gemv_ring_stages",
           "qmm_repack_glu", "qmm_mul_mat_glu_packed", "qmm_workspace_bytes_f32_host", "qmm_mul_mat_f32_host",
           "qmm_get_device_status", "qmm_set_test_fault", "qmm_aligned_row_bytes", "qmm_repack_aligned",
           "qmm_workspace_bytes_aligned", "qmm_mul_mat_aligned", "qmm_workspace_bytes_id_glu", "qmm_mul_mat_id_glu")


class QMMError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = int(code)
        super().__init__(f"{what}: {STATUS.get(self.code, self.code)}" if what else STATUS.get(self.code, str(code)))


class GemmPlan(ctypes.Structure):
    _fields_ = [("tiles_n", ctypes.c_int64), ("tiles_m", ctypes.c_int64), ("ntiles", ctypes.c_int64),
                ("iters_per_tile", ctypes.c_int64), ("nwork", ctypes.c_int64), ("ctas", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("fixup", ctypes.c_int32), ("efficiency_percent", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("iter_k", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_lib = None


def lib():
    """The loaded libqmm (ctypes.CDLL).  Raises QMMError if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise QMMError(6, f"libqmm.so not found at {LIB_PATH}; run block_quantized_matmul_q8_gb300._build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    L.qmm_status_string.restype = ctypes.c_char_p
    L.qmm_status_string.argtypes = [ctypes.c_int]
    L.qmm_q8_1_bytes.restype = SZ
    L.qmm_q8_1_bytes.argtypes = [I64, I64]
    L.qmm_row_bytes.restype = SZ
    L.qmm_row_bytes.argtypes = [ctypes.c_int, I64]
    L.qmm_workspace_bytes.restype = SZ
    L.qmm_workspace_bytes.argtypes = [ctypes.c_int, I64, I64, I64, I64, I64]
    L.qmm_quantize_q8_1.restype = ctypes.c_int
    L.qmm_quantize_q8_1.argtypes = [P, I64, I64, P, P]
    L.qmm_mul_mat.restype = ctypes.c_int
    L.qmm_mul_mat.argtypes = [P, ctypes.c_int, I64, I64, P, I64, P, P, SZ, P]
    L.qmm_mul_mat_id.restype = ctypes.c_int
    L.qmm_mul_mat_id.argtypes = [P, ctypes.c_int, I64, I64, I64, P, P, I64, I64, P, P, SZ, P]
    L.qmm_read_device_status.restype = ctypes.c_int
    L.qmm_read_device_status.argtypes = [P, ctypes.POINTER(I32), P]
    L.qmm_get_device_status.restype = ctypes.c_int
    L.qmm_get_device_status.argtypes = [P, P]
    L.qmm_tile_efficiency_percent.restype = ctypes.c_int
    L.qmm_tile_efficiency_percent.argtypes = [I64, I64]
    L.qmm_gemv_ring_stages.restype = ctypes.c_int
    L.qmm_gemv_ring_stages.argtypes = [ctypes.c_int, I64, I64, I32, I64]
    L.qmm_plan_gemm.restype = ctypes.c_int
    L.qmm_plan_gemm.argtypes = [ctypes.c_int, I64, I64, I64, I32, I32, ctypes.POINTER(GemmPlan)]
    L.qmm_plan_cta_range.restype = None
    L.qmm_plan_cta_range.argtypes = [ctypes.POINTER(GemmPlan), I32, ctypes.POINTER(I64), ctypes.POINTER(I64)]
    L.qmm_set_force_path.restype = None
    L.qmm_set_force_path.argtypes = [ctypes.c_int]
    L.qmm_aligned_row_bytes.restype = SZ
    L.qmm_aligned_row_bytes.argtypes = [ctypes.c_int, I64]
    L.qmm_repack_aligned.restype = ctypes.c_int
    L.qmm_repack_aligned.argtypes = [P, ctypes.c_int, I64, I64, P, P]
    L.qmm_workspace_bytes_aligned.restype = SZ
    L.qmm_workspace_bytes_aligned.argtypes = [ctypes.c_int, I64, I64, I64]
    L.qmm_mul_mat_aligned.restype = ctypes.c_int
    L.qmm_mul_mat_aligned.argtypes = [P, ctypes.c_int, I64, I64, P, I64, P, P, SZ, P]
    L.qmm_set_test_fault.restype = None
    L.qmm_set_test_fault.argtypes = [ctypes.c_int]
    L.qmm_set_stream_k_mode.restype = None
    L.qmm_set_stream_k_mode.argtypes = [ctypes.c_int]
    L.qmm_mul_mat_id_noalloc.restype = ctypes.c_int
    L.qmm_mul_mat_id_noalloc.argtypes = [P, ctypes.c_int, I64, I64, I64, P, P, I64, I64, P, P]
    L.qmm_workspace_bytes_glu.restype = ctypes.c_size_t
    L.qmm_workspace_bytes_glu.argtypes = [ctypes.c_int, I64, I64, I64]
    L.qmm_mul_mat_glu.restype = ctypes.c_int
    L.qmm_mul_mat_glu.argtypes = [P, P, ctypes.c_int, I64, I64, P, I64, P, P, ctypes.c_size_t, P]
    L.qmm_mul_mat_glu_packed.restype = ctypes.c_int
    L.qmm_mul_mat_glu_packed.argtypes = [P, ctypes.c_int, I64, I64, P, I64, P, P, ctypes.c_size_t, P]
    L.qmm_repack_glu.restype = ctypes.c_int
    L.qmm_repack_glu.argtypes = [P, P, ctypes.c_int, I64, I64, P, P]
    L.qmm_mul_mat_id_slot.restype = ctypes.c_int
    L.qmm_mul_mat_id_slot.argtypes = [P, ctypes.c_int, I64, I64, I64, P, P, I64, I64, P, P, ctypes.c_size_t, P]
    L.qmm_workspace_bytes_id_glu.restype = SZ
    L.qmm_workspace_bytes_id_glu.argtypes = [ctypes.c_int, I64, I64, I64, I64, I64]
    L.qmm_mul_mat_id_glu.restype = ctypes.c_int
    L.qmm_mul_mat_id_glu.argtypes = [P, P, ctypes.c_int, I64, I64, I64, P, P, I64, I64, P, P, ctypes.c_size_t, P]
    L.qmm_noalloc_scratch_bytes.restype = SZ
    L.qmm_noalloc_scratch_bytes.argtypes = []
    L.qmm_workspace_bytes_f32.restype = SZ
    L.qmm_workspace_bytes_f32_host.restype = SZ
    L.qmm_workspace_bytes_f32_host.argtypes = [ctypes.c_int, I64, I64, I64]
    L.qmm_mul_mat_f32_host.restype = ctypes.c_int
    L.qmm_mul_mat_f32_host.argtypes = [P, ctypes.c_int, I64, I64, P, I64, P, P, SZ, P]
    L.qmm_workspace_bytes_f32.argtypes = [ctypes.c_int, I64, I64, I64]
    L.qmm_mul_mat_f32.restype = ctypes.c_int
    L.qmm_mul_mat_f32.argtypes = [P, ctypes.c_int, I64, I64, P, I64, P, P, SZ, P]
    _lib = L
    return L


def _check(rc, what):
    if rc != 0:
        raise QMMError(rc, what)


def _qtype(t) -> int:
    return TYPES[t] if isinstance(t, str) else int(t)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise QMMError(1, f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise QMMError(3, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise QMMError(1, f"{name} must be contiguous")
    return t


def qmm_status_string(code: int) -> str:
    return lib().qmm_status_string(int(code)).decode()


def qmm_q8_1_bytes(m: int, k: int) -> int:
    return lib().qmm_q8_1_bytes(m, k)


def qmm_row_bytes(qtype, k: int) -> int:
    return lib().qmm_row_bytes(_qtype(qtype), k)


def qmm_workspace_bytes(qtype, n: int, k: int, m: int, n_experts: int = 0, top_k: int = 0) -> int:
    return lib().qmm_workspace_bytes(_qtype(qtype), n, k, m, n_experts, top_k)


def qmm_quantize_q8_1(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 [m, k] CUDA tensor -> uint8 [m, k/32*36] q8_1 blocks."""
    _dev(x, "x", torch.float32)
    m, k = x.shape
    if out is None:
        out = torch.empty((m, (k // 32) * 36), dtype=torch.uint8, device=x.device)
    _dev(out, "out", torch.uint8)
    if out.numel() < qmm_q8_1_bytes(m, k):
        raise QMMError(1, "out too small")
    _check(lib().qmm_quantize_q8_1(_ptr(x), m, k, _ptr(out), _stream(stream)), "qmm_quantize_q8_1")
    return out


def qmm_mul_mat(W: torch.Tensor, qtype, n: int, k: int, xq: torch.Tensor, m: int, y: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[m, n] fp32 = x * dequant(W)^T from q8_1 activations xq."""
    _dev(W, "W")
    _dev(xq, "xq")
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=W.device)
    _dev(y, "y", torch.float32)
    need = qmm_workspace_bytes(qtype, n, k, m)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=W.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().qmm_mul_mat(_ptr(W), _qtype(qtype), n, k, _ptr(xq), m, _ptr(y), _ptr(workspace), ws_bytes,
                             _stream(stream)), "qmm_mul_mat")
    return y


def qmm_aligned_row_bytes(qtype, k: int) -> int:
    return int(lib().qmm_aligned_row_bytes(_qtype(qtype), k))


def qmm_repack_aligned(W: torch.Tensor, qtype, n: int, k: int, W_aligned: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """W with its rows padded to whole 16-byte units: uint8 [n, qmm_aligned_row_bytes]."""
    _dev(W, "W")
    if W_aligned is None:
        W_aligned = torch.empty((n, qmm_aligned_row_bytes(qtype, k)), dtype=torch.uint8, device=W.device)
    _dev(W_aligned, "W_aligned")
    _check(lib().qmm_repack_aligned(_ptr(W), _qtype(qtype), n, k, _ptr(W_aligned), _stream(stream)),
           "qmm_repack_aligned")
    return W_aligned


def qmm_workspace_bytes_aligned(qtype, n: int, k: int, m: int) -> int:
    return int(lib().qmm_workspace_bytes_aligned(_qtype(qtype), n, k, m))


def qmm_mul_mat_aligned(W_aligned: torch.Tensor, qtype, n: int, k: int, xq: torch.Tensor, m: int,
                        y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """qmm_mul_mat on the padded rows of qmm_repack_aligned."""
    _dev(W_aligned, "W_aligned")
    _dev(xq, "xq")
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=W_aligned.device)
    _dev(y, "y", torch.float32)
    need = qmm_workspace_bytes_aligned(qtype, n, k, m)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=W_aligned.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().qmm_mul_mat_aligned(_ptr(W_aligned), _qtype(qtype), n, k, _ptr(xq), m, _ptr(y), _ptr(workspace),
                                     ws_bytes, _stream(stream)), "qmm_mul_mat_aligned")
    return y


def qmm_workspace_bytes_glu(qtype, n: int, k: int, m: int) -> int:
    return lib().qmm_workspace_bytes_glu(_qtype(qtype), n, k, m)


def qmm_mul_mat_glu(W_gate: torch.Tensor, W_up: torch.Tensor, qtype, n: int, k: int, xq: torch.Tensor, m: int,
                    y: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[m, n] fp32 = silu(x * dequant(W_gate)^T) * (x * dequant(W_up)^T) from q8_1 activations."""
    _dev(W_gate, "W_gate")
    _dev(W_up, "W_up")
    _dev(xq, "xq")
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=W_gate.device)
    _dev(y, "y", torch.float32)
    need = qmm_workspace_bytes_glu(qtype, n, k, m)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=W_gate.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().qmm_mul_mat_glu(_ptr(W_gate), _ptr(W_up), _qtype(qtype), n, k, _ptr(xq), m, _ptr(y),
                                 _ptr(workspace) if workspace is not None else None, ws_bytes, _stream(stream)),
           "qmm_mul_mat_glu")
    return y


def qmm_repack_glu(W_gate: torch.Tensor, W_up: torch.Tensor, qtype, n: int, k: int,
                   W_gu: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Interleaved copy of a gate/up pair: row 2j = gate row j, row 2j+1 = up row j."""
    _dev(W_gate, "W_gate")
    _dev(W_up, "W_up")
    if W_gu is None:
        W_gu = torch.empty(2 * W_gate.numel(), dtype=torch.uint8, device=W_gate.device)
    _dev(W_gu, "W_gu")
    _check(lib().qmm_repack_glu(_ptr(W_gate), _ptr(W_up), _qtype(qtype), n, k, _ptr(W_gu), _stream(stream)),
           "qmm_repack_glu")
    return W_gu


def qmm_mul_mat_glu_packed(W_gu: torch.Tensor, qtype, n: int, k: int, xq: torch.Tensor, m: int,
                           y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """qmm_mul_mat_glu on the interleaved tensor of qmm_repack_glu."""
    _dev(W_gu, "W_gu")
    _dev(xq, "xq")
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=W_gu.device)
    _dev(y, "y", torch.float32)
    need = qmm_workspace_bytes_glu(qtype, n, k, m)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=W_gu.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().qmm_mul_mat_glu_packed(_ptr(W_gu), _qtype(qtype), n, k, _ptr(xq), m, _ptr(y),
                                        _ptr(workspace) if workspace is not None else None, ws_bytes,
                                        _stream(stream)), "qmm_mul_mat_glu_packed")
    return y


def qmm_workspace_bytes_f32_host(qtype, n: int, k: int, m: int) -> int:
    return int(lib().qmm_workspace_bytes_f32_host(_qtype(qtype), n, k, m))


def qmm_mul_mat_f32_host(W: torch.Tensor, qtype, n: int, k: int, x_host: torch.Tensor, m: int, y_host: torch.Tensor,
                         workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """qmm_mul_mat_f32 with x and y in host memory (pinned for asynchronous copies):
    the copies and the product are enqueued on the stream by one C call."""
    _dev(W, "W")
    _dev(workspace, "workspace", torch.uint8)
    for t_, name in ((x_host, "x_host"), (y_host, "y_host")):
        if t_.is_cuda or t_.dtype != torch.float32 or not t_.is_contiguous():
            raise QMMError(1, f"{name} must be a contiguous fp32 host tensor")
    _check(lib().qmm_mul_mat_f32_host(_ptr(W), _qtype(qtype), n, k, _ptr(x_host), m, _ptr(y_host), _ptr(workspace),
                                      workspace.numel(), _stream(stream)), "qmm_mul_mat_f32_host")
    return y_host


def qmm_workspace_bytes_f32(qtype, n: int, k: int, m: int) -> int:
    return int(lib().qmm_workspace_bytes_f32(_qtype(qtype), n, k, m))


def qmm_mul_mat_f32(W: torch.Tensor, qtype, n: int, k: int, x: torch.Tensor, m: int, y: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[m, n] fp32 = x * dequant(W)^T from fp32 activations x, quantized to q8_1 inside
    the call (one launch for m == 1, which needs no workspace; a workspace is made here
    for m > 1 when none is given)."""
    _dev(W, "W")
    _dev(x, "x", torch.float32)
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=W.device)
    _dev(y, "y", torch.float32)
    if workspace is None and m > 1:
        workspace = torch.empty(qmm_workspace_bytes_f32(qtype, n, k, m), dtype=torch.uint8, device=W.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().qmm_mul_mat_f32(_ptr(W), _qtype(qtype), n, k, _ptr(x), m, _ptr(y), _ptr(workspace), ws_bytes,
                                 _stream(stream)), "qmm_mul_mat_f32")
    return y


def _mul_mat_id(fn, name, W, qtype, n_experts, n, k, xq, ids, top_k, n_tokens, y, workspace, stream):
    _dev(W, "W")
    _dev(xq, "xq")
    _dev(ids, "ids", torch.int32)
    if y is None:
        y = torch.empty((n_tokens, top_k, n), dtype=torch.float32, device=W.device)
    _dev(y, "y", torch.float32)
    if workspace is None:
        workspace = torch.empty(qmm_workspace_bytes(qtype, n, k, n_tokens, n_experts, top_k), dtype=torch.uint8,
                                device=W.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(fn(_ptr(W), _qtype(qtype), n_experts, n, k, _ptr(xq), _ptr(ids), top_k, n_tokens, _ptr(y),
              _ptr(workspace), ws_bytes, _stream(stream)), name)
    return y


def qmm_mul_mat_id(W: torch.Tensor, qtype, n_experts: int, n: int, k: int, xq: torch.Tensor, ids: torch.Tensor,
                   top_k: int, n_tokens: int, y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """y[n_tokens, top_k, n] fp32 with y[t, s] = x[t] * dequant(W[ids[t, s]])^T."""
    return _mul_mat_id(lib().qmm_mul_mat_id, "qmm_mul_mat_id", W, qtype, n_experts, n, k, xq, ids, top_k, n_tokens,
                       y, workspace, stream)


def qmm_mul_mat_id_slot(W: torch.Tensor, qtype, n_experts: int, n: int, k: int, xq: torch.Tensor, ids: torch.Tensor,
                        top_k: int, n_tokens: int, y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """y[n_tokens, top_k, n] fp32 with y[t, s] = x[t, s] * dequant(W[ids[t, s]])^T: xq holds
    one q8_1 row per (token, slot) pair, row t*top_k + s."""
    return _mul_mat_id(lib().qmm_mul_mat_id_slot, "qmm_mul_mat_id_slot", W, qtype, n_experts, n, k, xq, ids, top_k,
                       n_tokens, y, workspace, stream)


def qmm_workspace_bytes_id_glu(qtype, n: int, k: int, n_tokens: int, n_experts: int, top_k: int) -> int:
    return lib().qmm_workspace_bytes_id_glu(_qtype(qtype), n, k, n_tokens, n_experts, top_k)


def qmm_mul_mat_id_glu(W_gate: torch.Tensor, W_up: torch.Tensor, qtype, n_experts: int, n: int, k: int,
                       xq: torch.Tensor, ids: torch.Tensor, top_k: int, n_tokens: int, y: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[n_tokens, top_k, n] fp32 with y[t, s] = silu(x[t] Wg[e]^T) * (x[t] Wu[e]^T), e = ids[t, s]."""
    _dev(W_gate, "W_gate")
    _dev(W_up, "W_up")
    _dev(xq, "xq")
    _dev(ids, "ids", torch.int32)
    if y is None:
        y = torch.empty((n_tokens, top_k, n), dtype=torch.float32, device=W_gate.device)
    _dev(y, "y", torch.float32)
    if workspace is None:
        workspace = torch.empty(max(qmm_workspace_bytes_id_glu(qtype, n, k, n_tokens, n_experts, top_k), 256),
                                dtype=torch.uint8, device=W_gate.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().qmm_mul_mat_id_glu(_ptr(W_gate), _ptr(W_up), _qtype(qtype), n_experts, n, k, _ptr(xq), _ptr(ids),
                                    top_k, n_tokens, _ptr(y), _ptr(workspace), ws_bytes, _stream(stream)),
           "qmm_mul_mat_id_glu")
    return y


def qmm_mul_mat_id_noalloc(W: torch.Tensor, qtype, n_experts: int, n: int, k: int, xq: torch.Tensor,
                           ids: torch.Tensor, top_k: int, n_tokens: int, y: torch.Tensor, stream=None) -> torch.Tensor:
    """qmm_mul_mat_id with the library's fixed device scratch instead of a workspace;
    y must be given (the call allocates nothing)."""
    _dev(W, "W")
    _dev(xq, "xq")
    _dev(ids, "ids", torch.int32)
    _dev(y, "y", torch.float32)
    _check(lib().qmm_mul_mat_id_noalloc(_ptr(W), _qtype(qtype), n_experts, n, k, _ptr(xq), _ptr(ids), top_k,
                                        n_tokens, _ptr(y), _stream(stream)), "qmm_mul_mat_id_noalloc")
    return y


def qmm_noalloc_scratch_bytes() -> int:
    return lib().qmm_noalloc_scratch_bytes()


def qmm_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(-1)
    _check(lib().qmm_read_device_status(_ptr(workspace), ctypes.byref(v), _stream(stream)), "qmm_read_device_status")
    return v.value


def qmm_get_device_status(workspace: torch.Tensor, stream=None) -> int:
    """The status word of the last mul_mat_id on this workspace (synchronises the stream)."""
    return int(lib().qmm_get_device_status(_ptr(workspace), _stream(stream)))


def qmm_tile_efficiency_percent(ntiles: int, nsm: int) -> int:
    return lib().qmm_tile_efficiency_percent(ntiles, nsm)


def qmm_gemv_ring_stages(t, n: int, k: int, ncols: int, smem_bytes: int) -> int:
    return lib().qmm_gemv_ring_stages(_qtype(t), n, k, ncols, smem_bytes)


def qmm_plan_gemm(qtype, n: int, k: int, m: int, nsm: int, stream_k_mode: int = 0) -> GemmPlan:
    p = GemmPlan()
    _check(lib().qmm_plan_gemm(_qtype(qtype), n, k, m, nsm, stream_k_mode, ctypes.byref(p)), "qmm_plan_gemm")
    return p


def qmm_plan_cta_range(plan: GemmPlan, cta: int):
    b, e = ctypes.c_int64(), ctypes.c_int64()
    lib().qmm_plan_cta_range(ctypes.byref(plan), cta, ctypes.byref(b), ctypes.byref(e))
    return b.value, e.value


def qmm_set_force_path(path: int) -> None:
    lib().qmm_set_force_path(int(path))


def qmm_set_stream_k_mode(mode: int) -> None:
    lib().qmm_set_stream_k_mode(int(mode))


def qmm_set_test_fault(mode: int) -> None:
    lib().qmm_set_test_fault(int(mode))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libqmm.so in-tree (nvcc, sm_103a)."""
    from ._build import build as _b
    global _lib
    path = _b(force=force, verbose=verbose)
    _lib = None
    return path
