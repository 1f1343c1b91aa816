"""GPU parity of the expert-routed fused gate/up with SwiGLU (qmm_mul_mat_id_glu) against
the oracle's bound per element (the dense SwiGLU bound of each pair, itself pinned), on
each of its paths: one fused GEMV per pair (a handful of pairs, Q4_K), the fused grouped
tensor-core GEMM (Q4_K: ragged expert sizes, tiles of one pair, experts with several
128-pair tiles, n not a multiple of the 64 outputs of a tile), and the unfused form (other
formats: both products, then the combine).  Invalid ids give zero rows and QMM_ERR_IDS."""
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
    qmm.lib()


def _problem(fmt, E, n, k, T_, K, seed, invalid=0):
    rng = np.random.default_rng(seed)
    rw, rx, ri = qmm_synth.streams(seed)
    Wg = qmm_synth.gen_weights(fmt, rw, E * n, k).reshape(E, n, -1)
    Wu = qmm_synth.gen_weights(fmt, rw, E * n, k).reshape(E, n, -1)
    x = qmm_synth.gen_x(rx, T_, k)
    ids = qmm_synth.gen_moe_ids(ri, T_, K, E, 1.1)
    for i in range(invalid):
        ids[rng.integers(T_), rng.integers(K)] = -1 if i % 2 else E
    return Wg, Wu, x, ids


@pytest.mark.parametrize("fmt,E,n,k,T_,K,invalid", [
    ("q4_K", 8, 256, 1024, 2, 4, 0),     # 8 pairs: one fused GEMV per pair
    ("q4_K", 16, 130, 512, 3, 8, 2),     # 24 pairs, ragged n, invalid ids
    ("q4_K", 8, 256, 1024, 40, 4, 0),    # 160 pairs: grouped tensor-core GLU
    ("q4_K", 5, 200, 1024, 333, 3, 3),   # experts with several 128-pair tiles, n % 64 != 0
    ("q4_K", 64, 96, 256, 70, 4, 0),     # many experts with a pair or two
    ("q8_0", 6, 128, 512, 20, 4, 1),     # unfused
    ("q6_K", 4, 64, 512, 3, 2, 0),       # unfused, decode size
])
def test_mul_mat_id_glu_matches_oracle(oracle_mod, fmt, E, n, k, T_, K, invalid):
    Wg, Wu, x, ids = _problem(fmt, E, n, k, T_, K, seed=E + n + T_, invalid=invalid)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, tol, bad = oracle_mod.mul_mat_id_glu(Wg, Wu, fmt, E, n, k, xq, ids)
    ws = torch.empty(max(qmm.qmm_workspace_bytes_id_glu(fmt, n, k, T_, E, K), 256), dtype=torch.uint8, device=DEV)
    y = torch.full((T_, K, n), float("nan"), device=DEV)
    qmm.qmm_mul_mat_id_glu(torch.from_numpy(Wg).to(DEV), torch.from_numpy(Wu).to(DEV), fmt, E, n, k,
                           torch.from_numpy(xq).to(DEV), torch.from_numpy(ids).to(DEV), K, T_, y=y, workspace=ws)
    assert qmm.qmm_read_device_status(ws) == (7 if bad else 0)
    yg = y.cpu().numpy().astype(np.float64)
    assert np.isfinite(yg).all()
    err = np.abs(yg - y_ref)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert (err <= tol).all(), f"{fmt} E={E} n={n} k={k} T={T_} K={K}: worst {worst} err {err[worst]:.3e} tol {tol[worst]:.3e}"
    if invalid:
        rows = (ids < 0) | (ids >= E)
        assert not yg[rows].any()


def test_mul_mat_id_glu_equals_its_parts(oracle_mod):
    """The fused grouped GEMM against silu(g) * u of the plain mul_mat_id products of the
    gate and up experts: both meet the oracle's bound, so they agree within twice it (the
    fused tiles may add in another order, so bit equality is not required)."""
    fmt, E, n, k, T_, K = "q4_K", 8, 192, 1024, 64, 4
    Wg, Wu, x, ids = _problem(fmt, E, n, k, T_, K, seed=11)
    xq = oracle_mod.quantize_q8_1(x)
    _, tol, _ = oracle_mod.mul_mat_id_glu(Wg, Wu, fmt, E, n, k, xq, ids)
    d = lambda a: torch.from_numpy(a).to(DEV)
    y = qmm.qmm_mul_mat_id_glu(d(Wg), d(Wu), fmt, E, n, k, d(xq), d(ids), K, T_).cpu().numpy().astype(np.float64)
    g = qmm.qmm_mul_mat_id(d(Wg), fmt, E, n, k, d(xq), d(ids), K, T_).cpu().numpy().astype(np.float64)
    u = qmm.qmm_mul_mat_id(d(Wu), fmt, E, n, k, d(xq), d(ids), K, T_).cpu().numpy().astype(np.float64)
    assert (np.abs(y - g / (1.0 + np.exp(-g)) * u) <= 2 * tol).all()


def test_mul_mat_id_glu_rejects_bad_arguments():
    d = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    ids = torch.zeros((1, 1), dtype=torch.int32, device=DEV)
    y = torch.zeros((1, 1, 256), device=DEV)
    ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
    with pytest.raises(qmm.QMMError):  # no up tensor
        qmm.lib()
        code = qmm.lib().qmm_mul_mat_id_glu(qmm._ptr(d), None, 12, 1, 256, 256, qmm._ptr(d), qmm._ptr(ids), 1, 1,
                                            qmm._ptr(y), qmm._ptr(ws), 4096, None)
        qmm._check(code, "qmm_mul_mat_id_glu")
