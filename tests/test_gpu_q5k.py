"""GPU parity of Q5_K (the 5-bit k-quant: Q4_K's scales and nibbles plus a plane of fifth
bits) against the oracle, |y - y_oracle| <= 1e-5 T per element, on every path that takes
the format: the bulk-copy and direct GEMVs (m <= 8), the dp4a GEMM and the tensor-core
GEMM (m > 8), the grouped MoE GEMM and the MoE decode GEMV.  The extreme-code case sets
every fifth bit (codes 16..31, the largest operand values) with scales and mins 63, and
the plane-only case isolates the fifth bits (low nibbles 0) so that a fifth bit read from
the wrong byte or bit of the plane changes the result."""
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
    qmm.lib()
    yield
    qmm.qmm_set_force_path(0)


def _run(W, n, k, xq, m, path):
    qmm.qmm_set_force_path(path)
    try:
        y = qmm.qmm_mul_mat(torch.from_numpy(W).to(DEV), "q5_K", n, k, torch.from_numpy(xq).to(DEV), m)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    return y.cpu().numpy()


@pytest.mark.parametrize("n,k,m,path", [
    (300, 1024, 1, qmm.PATH_AUTO), (300, 1024, 1, qmm.PATH_GEMV_DIRECT), (77, 2560, 5, qmm.PATH_GEMV),
    (300, 1024, 8, qmm.PATH_AUTO),
    (300, 1024, 40, qmm.PATH_GEMM_DP4A), (300, 1024, 40, qmm.PATH_GEMM_TC),
    (1000, 1280, 200, qmm.PATH_GEMM_TC),   # several 128-row tiles each way, ragged in n and m
    (130, 256, 129, qmm.PATH_AUTO),        # one superblock per row
])
def test_q5_K_matches_oracle(oracle_mod, n, k, m, path):
    W, x = qmm_synth.make_dense("q5_K", n, k, m, seed=n + 3 * k + m)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q5_K", n, k, xq, m)
    assert_within(_run(W, n, k, xq, m, path), y_ref, T, f"q5_K n={n} k={k} m={m} path={path}")


def _extreme_weights(n, k, seed):
    W = qmm_synth.gen_q5_K(np.random.default_rng(seed), n, k)
    blk = W.reshape(n, k // 256, 176)
    blk[:8, :, 4:16] = 0xFF   # every 6-bit scale and min 63
    blk[:8, :, 16:48] = 0xFF  # every fifth bit set
    blk[:8, :, 48:] = 0xFF    # every nibble 15: code 31
    blk[8:16, :, 48:] = 0x00  # nibbles 0: the codes are the fifth bits alone (0 or 16)
    return W


@pytest.mark.parametrize("m,path", [(1, qmm.PATH_AUTO), (4, qmm.PATH_GEMV), (40, qmm.PATH_GEMM_DP4A),
                                    (40, qmm.PATH_GEMM_TC)])
def test_q5_K_extreme_codes(oracle_mod, m, path):
    n, k = 64, 2048
    W = _extreme_weights(n, k, seed=9)
    x = qmm_synth.gen_x(np.random.default_rng(10), m, k)
    x[0, :] = 127.0
    if m > 1:
        x[1, :] = -1.0
    if m > 3:
        adv = adversarial_x_rows().reshape(-1)
        x[3, :min(adv.size, k)] = adv[:k]
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q5_K", n, k, xq, m)
    assert_within(_run(W, n, k, xq, m, path), y_ref, T, f"q5_K extreme m={m} path={path}")


@pytest.mark.parametrize("E,n,k,T_,K", [(4, 64, 256, 9, 2), (8, 200, 1024, 300, 2), (16, 130, 512, 3, 4)])
def test_q5_K_moe(oracle_mod, E, n, k, T_, K):
    W, x, ids = qmm_synth.make_moe(E, n, k, T_, K, seed=E + n + T_, fmt="q5_K")
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, Tr, bad = oracle_mod.mul_mat_id(W, "q5_K", E, n, k, xq, ids)
    ws = torch.empty(qmm.qmm_workspace_bytes("q5_K", n, k, T_, E, K), dtype=torch.uint8, device=DEV)
    y = torch.full((T_, K, n), float("nan"), device=DEV)
    qmm.qmm_mul_mat_id(torch.from_numpy(W).to(DEV), "q5_K", E, n, k, torch.from_numpy(xq).to(DEV),
                       torch.from_numpy(ids).to(DEV), K, T_, y=y, workspace=ws)
    assert qmm.qmm_read_device_status(ws) == (7 if bad else 0)
    assert_within(y.cpu().numpy(), y_ref, Tr, f"q5_K moe E={E} n={n} k={k} T={T_} K={K}")
