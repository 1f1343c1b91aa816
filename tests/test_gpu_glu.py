"""Fused gate/up + SwiGLU (qmm_mul_mat_glu) against the oracle's silu(g) * u and its
propagated bound: the bulk-copy GEMV (Q4_K, m <= 8), the tensor-core GEMM with gate and
up rows interleaved in the tile (Q4_K, m > 8, whole tiles, ragged n), and the unfused
fallback (the other formats, or forced)."""
import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qmm.build()
    yield
    qmm.qmm_set_force_path(0)


def run_glu(oracle_mod, fmt, n, k, m, path=0, seed=0, x_scale=1.0):
    W, x = qmm_synth.make_dense(fmt, 2 * n, k, m, seed=seed)
    row = W.shape[1]
    Wg, Wu = W[:n].copy(), W[n:].copy()
    xq = oracle_mod.quantize_q8_1((x * np.float32(x_scale)).astype(np.float32))
    qmm.qmm_set_force_path(path)
    try:
        y = torch.full((m, n), float("nan"), device=DEV)
        qmm.qmm_mul_mat_glu(torch.from_numpy(Wg).to(DEV), torch.from_numpy(Wu).to(DEV), fmt, n, k,
                            torch.from_numpy(xq).to(DEV), m, y=y)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    y_ref, tol = oracle_mod.mul_mat_glu(Wg, Wu, fmt, n, k, xq, m)
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - y_ref)
    bad = err > tol
    assert not bad.any(), (f"glu {fmt} n={n} k={k} m={m} path={path}: {int(bad.sum())} outside the bound; "
                           f"worst {np.unravel_index(np.argmax(err - tol), err.shape)}")
    assert row == W.shape[1]


@pytest.mark.parametrize("n,k,m", [(1000, 2048, 1), (1001, 512, 2), (64, 256, 3), (777, 1024, 5), (2048, 5120, 8)])
def test_glu_gemv(oracle_mod, n, k, m):
    run_glu(oracle_mod, "q4_K", n, k, m, seed=n + m)


@pytest.mark.parametrize("n,k,m", [(64, 256, 9), (130, 512, 64), (300, 1024, 129), (1000, 2048, 200),
                                   (65, 256, 513), (1000, 256, 1290)])
def test_glu_tensor_core(oracle_mod, n, k, m):
    run_glu(oracle_mod, "q4_K", n, k, m, seed=2 * n + m)


def test_glu_tensor_core_forced_small_m(oracle_mod):
    run_glu(oracle_mod, "q4_K", 200, 512, 4, path=qmm.PATH_GEMM_TC, seed=3)


def test_glu_saturated_gate(oracle_mod):
    """Activations scaled so that the gate dots reach large magnitudes: silu saturates to
    g for g >> 0 and to -0 for g << 0, on both fused paths."""
    run_glu(oracle_mod, "q4_K", 130, 512, 3, seed=5, x_scale=40.0)
    run_glu(oracle_mod, "q4_K", 130, 512, 40, seed=6, x_scale=40.0)


@pytest.mark.parametrize("fmt,n,k,m", [("q6_K", 130, 512, 3), ("q6_K", 96, 1024, 40), ("q8_0", 200, 256, 1),
                                       ("q8_0", 136, 512, 100), ("q4_K", 300, 512, 20)])
def test_glu_unfused(oracle_mod, fmt, n, k, m):
    path = qmm.PATH_GEMM_DP4A if fmt == "q4_K" else 0
    run_glu(oracle_mod, fmt, n, k, m, path=path, seed=n + k)



# ---------------------------------------------------------------- interleaved gate/up

@pytest.mark.parametrize("fmt,n,k", [("q4_K", 130, 512), ("q6_K", 33, 256), ("q6_K", 8, 2048), ("q8_0", 17, 96),
                                     ("q8_0", 40, 256), ("q4_0", 9, 1056)])
def test_repack_glu_bytes(oracle_mod, fmt, n, k):
    """The repack is byte work: bit-exact against the oracle's interleave (16-byte and
    2-byte copy units)."""
    W, _ = qmm_synth.make_dense(fmt, 2 * n, k, 1, seed=n)
    Wg, Wu = W[:n].copy(), W[n:].copy()
    got = qmm.qmm_repack_glu(torch.from_numpy(Wg).to(DEV), torch.from_numpy(Wu).to(DEV), fmt, n, k)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().reshape(2 * n, -1), oracle_mod.repack_glu(Wg, Wu))


def run_packed(oracle_mod, fmt, n, k, m, path=0, seed=0):
    W, x = qmm_synth.make_dense(fmt, 2 * n, k, m, seed=seed)
    Wg, Wu = W[:n].copy(), W[n:].copy()
    xq = oracle_mod.quantize_q8_1(x)
    Wg_d, Wu_d, xq_d = (torch.from_numpy(a).to(DEV) for a in (Wg, Wu, xq))
    W_gu = qmm.qmm_repack_glu(Wg_d, Wu_d, fmt, n, k)
    qmm.qmm_set_force_path(path)
    try:
        y_packed = qmm.qmm_mul_mat_glu_packed(W_gu, fmt, n, k, xq_d, m)
        y_pair = qmm.qmm_mul_mat_glu(Wg_d, Wu_d, fmt, n, k, xq_d, m)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    a, b = y_packed.cpu().numpy(), y_pair.cpu().numpy()
    y_ref, tol = oracle_mod.mul_mat_glu(Wg, Wu, fmt, n, k, xq, m)
    err = np.abs(a.astype(np.float64) - y_ref)
    assert np.all(np.isfinite(a)) and not (err > tol).any(), f"packed glu {fmt} n={n} k={k} m={m} path={path}"
    return a, b


# The fused paths fold the same rows in the same order from either layout: equal to the bit
@pytest.mark.parametrize("n,k,m,path", [(1000, 2048, 1, 0), (1001, 512, 3, 0), (777, 1024, 8, 0),
                                        (64, 256, 9, 0), (300, 1024, 129, 0), (65, 256, 513, 0),
                                        (200, 512, 4, 3), (1000, 256, 1290, 0)])
def test_glu_packed_fused_bitexact(oracle_mod, n, k, m, path):
    a, b = run_packed(oracle_mod, "q4_K", n, k, m, path=path, seed=n + m)
    assert np.array_equal(a, b)


# Elsewhere one product of the 2n interleaved rows and a combine pass: within the bound
@pytest.mark.parametrize("fmt,n,k,m,path", [("q6_K", 130, 512, 3, 0), ("q8_0", 100, 256, 20, 0),
                                            ("q4_0", 70, 1056, 2, 0), ("q4_K", 300, 1024, 40, 2)])
def test_glu_packed_unfused(oracle_mod, fmt, n, k, m, path):
    run_packed(oracle_mod, fmt, n, k, m, path=path, seed=3 * n + m)
