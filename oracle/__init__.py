"""CPU oracle for the block-quantized matmul (ctypes wrapper over qmm_oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, the smoke check in __graft_entry__.py and the
CPU-baseline leg of bench.py use it; the product package never imports it and
shares no code with it.

Every function returns fp64 results of the plain definitions (see the C file's
header for the readings of the pages that it takes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_qmm.so")

TYPES = {"q4_0": 2, "q8_0": 8, "q4_K": 12, "q5_K": 13, "q6_K": 14}
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no fast-math, no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load(_LIB_PATH)
    return _lib


def load(path: str):
    """A ctypes handle on an oracle library at `path` with every signature declared
    (lib() uses it for the in-tree build; the mutation tests load planted copies)."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    L.oracle_half_to_double.restype = ctypes.c_double
    L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_float_to_half.restype = ctypes.c_uint16
    L.oracle_float_to_half.argtypes = [ctypes.c_float]
    L.oracle_quantize_q8_1.argtypes = [P, I64, I64, P]
    L.oracle_dequant_q8_1.argtypes = [P, I64, I64, P]
    L.oracle_block_bytes.argtypes = [ctypes.c_int]
    L.oracle_block_elems.argtypes = [ctypes.c_int]
    L.oracle_q4_K_fields.argtypes = [P, P, P, P, P, P]
    L.oracle_q5_K_fields.argtypes = [P, P, P, P, P, P]
    L.oracle_q6_K_fields.argtypes = [P, P, P, P]
    L.oracle_dequant.argtypes = [ctypes.c_int, P, I64, I64, P]
    L.oracle_mul_mat.argtypes = [ctypes.c_int, P, I64, I64, P, I64, P, P]
    L.oracle_mul_mat_at.argtypes = [ctypes.c_int, P, I64, I64, P, I64, P, P, I64, P, P]
    L.oracle_brute.argtypes = [ctypes.c_int, P, I64, I64, P, I64, P]
    L.oracle_bucket.restype = I64
    L.oracle_bucket.argtypes = [P, I64, I64, I64, P, P]
    L.oracle_mul_mat_id.restype = I64
    L.oracle_mul_mat_id.argtypes = [ctypes.c_int, P, I64, I64, I64, P, P, I64, I64, P, P]
    L.oracle_mul_mat_id_slot.restype = I64
    L.oracle_mul_mat_id_slot.argtypes = [ctypes.c_int, P, I64, I64, I64, P, P, I64, I64, P, P]
    L.oracle_set_threads.argtypes = [ctypes.c_int]
    return L


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view(np.uint8) if a.dtype != np.uint8 else a


def _check(rc):
    if rc < 0:
        raise ValueError(f"oracle call failed with code {rc}")
    return rc


def set_threads(n: int) -> int:
    return lib().oracle_set_threads(int(n))


def half_to_double(h: int) -> float:
    return lib().oracle_half_to_double(int(h))


def float_to_half(x: float) -> int:
    return lib().oracle_float_to_half(float(np.float32(x)))


def block_bytes(fmt: str) -> int:
    return lib().oracle_block_bytes(TYPES[fmt])


def block_elems(fmt: str) -> int:
    return lib().oracle_block_elems(TYPES[fmt])


def quantize_q8_1(x: np.ndarray) -> np.ndarray:
    """fp32 [m][k] -> q8_1 bytes uint8 [m][k/32*36]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    m, k = x.shape
    out = np.empty((m, (k // 32) * 36), dtype=np.uint8)
    _check(lib().oracle_quantize_q8_1(_p(x), m, k, _p(out)))
    return out


def dequant_q8_1(xq: np.ndarray, m: int, k: int) -> np.ndarray:
    xq = _u8(xq)
    out = np.empty((m, k), dtype=np.float64)
    _check(lib().oracle_dequant_q8_1(_p(xq), m, k, _p(out)))
    return out


def dequant(W: np.ndarray, fmt: str, n: int, k: int) -> np.ndarray:
    W = _u8(W)
    out = np.empty((n, k), dtype=np.float64)
    _check(lib().oracle_dequant(TYPES[fmt], _p(W), n, k, _p(out)))
    return out


def q4_K_fields(blk: np.ndarray):
    blk = _u8(blk)
    d = ctypes.c_double()
    dmin = ctypes.c_double()
    sc = np.empty(8, np.int32)
    mn = np.empty(8, np.int32)
    q = np.empty(256, np.int32)
    lib().oracle_q4_K_fields(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(mn), _p(q))
    return d.value, dmin.value, sc, mn, q


def q5_K_fields(blk: np.ndarray):
    blk = _u8(blk)
    d = ctypes.c_double()
    dmin = ctypes.c_double()
    sc = np.empty(8, np.int32)
    mn = np.empty(8, np.int32)
    q = np.empty(256, np.int32)
    lib().oracle_q5_K_fields(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(mn), _p(q))
    return d.value, dmin.value, sc, mn, q


def q6_K_fields(blk: np.ndarray):
    blk = _u8(blk)
    d = ctypes.c_double()
    sc = np.empty(16, np.int32)
    q = np.empty(256, np.int32)
    lib().oracle_q6_K_fields(_p(blk), ctypes.byref(d), _p(sc), _p(q))
    return d.value, sc, q


def mul_mat(W: np.ndarray, fmt: str, n: int, k: int, xq: np.ndarray, m: int):
    """(y, T), both fp64 [m][n]: the fold and the sum of |block terms|."""
    W = _u8(W)
    xq = _u8(xq)
    y = np.empty((m, n), dtype=np.float64)
    T = np.empty((m, n), dtype=np.float64)
    _check(lib().oracle_mul_mat(TYPES[fmt], _p(W), n, k, _p(xq), m, _p(y), _p(T)))
    return y, T


def silu(v):
    """v * sigmoid(v) in fp64: the SwiGLU gate ([MMQ] section "「分专家」与「整批」之间: host
    侧的代价": the fused gate/up kernel applies the GLU right after the dots; [P0007]'s
    coverage list: fused ffn gate/up/SWIGLU)."""
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def mul_mat_glu(W_gate, W_up, fmt, n, k, xq, m):
    """(y, tol), both fp64 [m][n]: y = silu(g) * u with g, u the folds of the gate and up
    rows (each W [n][k]).  tol is the per-element bound that the GPU result must meet:
    the fold bound of each dot (1e-5 of its sum of |block terms|) carried through the
    product to first order, plus 2^-20 of |y| for evaluating silu and the product in fp32,
    plus 2^-120 |u| for the fp32 range: e^-g overflows fp32 for g < -88.7, where the true
    silu(g) is below 88.7 e^-88.7 < 3e-37 in magnitude and fp32 gives 0:
        tol = 1e-5 * (|silu'(g)| T_g |u| + |silu(g)| T_u) + 2^-20 |y| + 2^-120 |u|."""
    g, Tg = mul_mat(W_gate, fmt, n, k, xq, m)
    u, Tu = mul_mat(W_up, fmt, n, k, xq, m)
    return _glu(g, Tg, u, Tu)


def _glu(g, Tg, u, Tu):
    sg = 1.0 / (1.0 + np.exp(-g))
    a = g * sg
    da = sg * (1.0 + g * (1.0 - sg))
    y = a * u
    tol = 1e-5 * (np.abs(da) * Tg * np.abs(u) + np.abs(a) * Tu) + 2.0 ** -20 * np.abs(y) + 2.0 ** -120 * np.abs(u)
    return y, tol


def mul_mat_glu_at(W_gate, W_up, fmt, n, k, xq, m, rows, cols):
    """mul_mat_glu at selected output positions (rows = output features, cols =
    activation rows): (y, tol) of length len(rows)."""
    g, Tg = mul_mat_at(W_gate, fmt, n, k, xq, m, rows, cols)
    u, Tu = mul_mat_at(W_up, fmt, n, k, xq, m, rows, cols)
    return _glu(g, Tg, u, Tu)


def repack_glu(W_gate, W_up) -> np.ndarray:
    """The interleaved gate/up tensor, bytes unchanged: row 2j is gate row j and row 2j+1
    up row j (the row order of the fused tile in [MMQ] section "输出端: 写回与 scale 修正",
    there in groups of 8 rows, here single rows)."""
    g = _u8(W_gate)
    u = _u8(W_up)
    if g.shape != u.shape or g.ndim != 2:
        raise ValueError("gate and up must be [n][row bytes] of the same shape")
    out = np.empty((2 * g.shape[0], g.shape[1]), dtype=np.uint8)
    out[0::2] = g
    out[1::2] = u
    return out


def aligned_row_bytes(fmt: str, k: int) -> int:
    """Row stride of the padded layout: the row's k/QK blocks rounded up to whole 16-byte
    units, for Q6_K after 14 more bytes (a superblock's 16-byte-aligned 224-byte copy window
    can reach 14 bytes past the row's last block)."""
    rb = (k // block_elems(fmt)) * block_bytes(fmt)
    return -(-(rb + (14 if fmt == "q6_K" else 0)) // 16) * 16


def repack_aligned(W, fmt, n, k) -> np.ndarray:
    """W [n][k/QK blocks] as rows of aligned_row_bytes bytes: the blocks unchanged, the
    rest of each row zero (the one-time repack of [QMM] section "Q4K 的 8 列重排", here
    only a change of row stride)."""
    W = _u8(W).reshape(n, -1)
    rb = (k // block_elems(fmt)) * block_bytes(fmt)
    if W.shape[1] != rb:
        raise ValueError("W must be [n][row bytes]")
    out = np.zeros((n, aligned_row_bytes(fmt, k)), dtype=np.uint8)
    out[:, :rb] = W
    return out


def mul_mat_at(W, fmt, n, k, xq, m, rows, cols):
    """Fold at selected output positions (rows = W rows, cols = activation rows)."""
    W = _u8(W)
    xq = _u8(xq)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    y = np.empty(len(rows), dtype=np.float64)
    T = np.empty(len(rows), dtype=np.float64)
    _check(lib().oracle_mul_mat_at(TYPES[fmt], _p(W), n, k, _p(xq), m, _p(rows), _p(cols), len(rows), _p(y), _p(T)))
    return y, T


def brute(W, fmt, n, k, xq, m) -> np.ndarray:
    W = _u8(W)
    xq = _u8(xq)
    y = np.empty((m, n), dtype=np.float64)
    _check(lib().oracle_brute(TYPES[fmt], _p(W), n, k, _p(xq), m, _p(y)))
    return y


def bucket(ids: np.ndarray, n_experts: int):
    """(bounds int32 [E+1], perm int32 [valid pairs], n_invalid)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    t, kk = ids.shape
    bounds = np.empty(n_experts + 1, np.int32)
    perm = np.empty(t * kk, np.int32)
    bad = lib().oracle_bucket(_p(ids), t, kk, n_experts, _p(bounds), _p(perm))
    return bounds, perm[: bounds[-1]], int(bad)


def mul_mat_id(W, fmt, n_experts, n, k, xq, ids, per_slot=False):
    """(y, T, n_invalid) with y, T fp64 [n_tokens][top_k][n].  xq holds one q8_1 row
    per token, or with per_slot one row per (token, slot) pair (row t*top_k + s)."""
    W = _u8(W)
    xq = _u8(xq)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    t, kk = ids.shape
    y = np.empty((t, kk, n), np.float64)
    T = np.empty((t, kk, n), np.float64)
    fn = lib().oracle_mul_mat_id_slot if per_slot else lib().oracle_mul_mat_id
    bad = fn(TYPES[fmt], _p(W), n_experts, n, k, _p(xq), _p(ids), kk, t, _p(y), _p(T))
    _check(bad)
    return y, T, int(bad)


def mul_mat_id_glu(W_gate, W_up, fmt, n_experts, n, k, xq, ids):
    """(y, tol, n_invalid), y and tol fp64 [n_tokens][top_k][n]: the expert-routed SwiGLU
    y[t][s] = silu(g) * u with g, u the folds of expert ids[t][s]'s gate and up rows
    against token t's row of xq, and tol the bound of mul_mat_glu per element.  Pairs with
    an invalid id have g = u = 0, hence y = 0 and tol = 0."""
    g, Tg, bad = mul_mat_id(W_gate, fmt, n_experts, n, k, xq, ids)
    u, Tu, _ = mul_mat_id(W_up, fmt, n_experts, n, k, xq, ids)
    y, tol = _glu(g, Tg, u, Tu)
    return y, tol, bad


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
