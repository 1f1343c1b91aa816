"""Parity of the skinny tensor-core path (Q4_K, 1 <= m <= 16: weight rows as the MMA's
128-row M side, activation rows as N = 16) against the oracle.  Shapes cover ragged
row tiles, one to many superblocks, every m from 1 to 16 and stream-K splits of a tile
between CTAs (few units per CTA, and tiles fewer than CTAs)."""
import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth
from parity import adversarial_x_rows, assert_within

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qmm.build()
    yield
    qmm.qmm_set_force_path(0)


def run_skinny(oracle_mod, n, k, m, seed=0, x=None, path=qmm.PATH_GEMV_TC):
    W, xr = qmm_synth.make_dense("q4_K", n, k, m, seed=seed)
    if x is not None:
        xr = x
    xq = oracle_mod.quantize_q8_1(xr)
    qmm.qmm_set_force_path(path)
    try:
        ws = torch.empty(max(256, qmm.qmm_workspace_bytes("q4_K", n, k, m)), dtype=torch.uint8, device=DEV)
        y = torch.full((m, n), float("nan"), device=DEV)
        qmm.qmm_mul_mat(torch.from_numpy(W).to(DEV), "q4_K", n, k, torch.from_numpy(xq).to(DEV), m, y=y,
                        workspace=ws)
        torch.cuda.synchronize()
        status = qmm.qmm_read_device_status(ws)
    finally:
        qmm.qmm_set_force_path(0)
    assert status == 0, f"device status {status}"
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    assert_within(y.cpu().numpy(), y_ref, T, f"skinny n={n} k={k} m={m}")
    return y.cpu().numpy()


@pytest.mark.parametrize("m", list(range(1, 17)))
def test_skinny_every_m(oracle_mod, m):
    run_skinny(oracle_mod, 300, 1024, m, seed=m)


@pytest.mark.parametrize("n,k,m", [(1, 256, 3), (128, 256, 16), (129, 512, 2), (1000, 2304, 8), (4100, 512, 5),
                                   (2000, 4096, 11), (64, 5120, 4)])
def test_skinny_shapes(oracle_mod, n, k, m):
    """(1, 256): a single weight row; (64, 5120): one tile split over 20 CTAs;
    (4100, 512): a ragged last tile among many."""
    run_skinny(oracle_mod, n, k, m, seed=n + k + m)


def test_skinny_adversarial_activations(oracle_mod):
    k = 512
    xa = np.resize(adversarial_x_rows().reshape(-1), k)
    x = (np.stack([xa, -xa, 1e-3 * xa]) * np.float32(1)).astype(np.float32)
    run_skinny(oracle_mod, 333, k, 3, seed=1, x=x)


def test_skinny_zero_activations_give_zero():
    n, k, m = 200, 512, 4
    W, _ = qmm_synth.make_dense("q4_K", n, k, m)
    xq = torch.zeros((m, k // 32 * 36), dtype=torch.uint8, device=DEV)
    qmm.qmm_set_force_path(qmm.PATH_GEMV_TC)
    try:
        y = qmm.qmm_mul_mat(torch.from_numpy(W).to(DEV), "q4_K", n, k, xq, m)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    assert torch.all(y == 0)


@pytest.mark.parametrize("m", [2, 8])
def test_skinny_agrees_with_dp4a_gemv(oracle_mod, m):
    """The same problem through the skinny path and the dp4a GEMV: both within the
    bound, and within 2x the bound of each other."""
    n, k = 777, 2048
    W, x = qmm_synth.make_dense("q4_K", n, k, m, seed=9 + m)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    a = run_skinny(oracle_mod, n, k, m, seed=9 + m)
    b = run_skinny(oracle_mod, n, k, m, seed=9 + m, path=qmm.PATH_GEMV)
    assert np.all(np.abs(a.astype(np.float64) - b) <= 2e-5 * T)
