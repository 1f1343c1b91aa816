"""GPU parity of the multi-column GEMV on mma.sync (Q4_K, 1 <= m <= 8) against the
oracle, |y - y_oracle| <= 1e-5 T per element, and the dp4a GEMV on the same inputs.
Shapes cover ragged row counts (tiles of fewer than 16 rows at the end of the matrix and
of a CTA), one superblock per row (most warps without work in a tile), superblock counts
below, at and above the 16 consumer warps, every column count, and activation blocks that
stress the exact-integer operands (all-zero blocks, |q| = 127 everywhere)."""
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
        y = qmm.qmm_mul_mat(torch.from_numpy(W).to(DEV), "q4_K", n, k, torch.from_numpy(xq).to(DEV), m)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    return y.cpu().numpy()


@pytest.mark.parametrize("n,k,m", [
    (300, 1024, 1), (300, 1024, 2), (300, 1024, 3), (300, 1024, 4), (300, 1024, 5), (300, 1024, 6),
    (300, 1024, 7), (300, 1024, 8),
    (17408 // 8, 5120, 8),  # 20 superblocks: more than the 16 consumer warps
    (1000, 4096, 4),       # 16 superblocks: one per warp
    (4111, 2048, 1),
    (1000, 1280, 3),   # 5 superblocks per row
    (17, 256, 5),      # one superblock, 17 rows: a tile of 16 and a tile of 1
    (4104, 5120, 8),   # several 16-row tiles per CTA, the last tile 8 rows
    (2440, 2048, 2),   # 152.5 tiles: CTAs with 1 or 2 tiles, the last one 8 rows
    (8, 768, 7),       # a single tile of 8 rows
])
def test_gemv_mma_matches_oracle(oracle_mod, n, k, m):
    W, x = qmm_synth.make_dense("q4_K", n, k, m, seed=n + k + m)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    y = _run(W, n, k, xq, m, qmm.PATH_GEMV_MMA)
    assert_within(y, y_ref, T, f"mma gemv n={n} k={k} m={m}")
    y_dp4a = _run(W, n, k, xq, m, qmm.PATH_GEMV)
    assert_within(y_dp4a, y_ref, T, "dp4a gemv")


def test_gemv_mma_extreme_codes(oracle_mod):
    """Weight codes 15 with scales 63 and activation codes +-127 (the largest integer
    sums the operands can form), all-zero activation blocks, and adversarial blocks."""
    n, k, m = 64, 2048, 8
    rng = np.random.default_rng(5)
    W = qmm_synth.gen_q4_K(rng, n, k)
    blk = W.reshape(n, k // 256, 144)
    blk[:8, :, 4:16] = 0xFF  # every 6-bit scale and min 63
    blk[:8, :, 16:] = 0xFF   # every nibble 15
    x = qmm_synth.gen_x(rng, m, k)
    x[0, :] = 127.0           # amax 127: q = 127 everywhere
    x[1, :] = -1.0            # q = -127 everywhere
    x[2, :64] = 0.0           # two zero blocks
    adv = adversarial_x_rows().reshape(-1)
    x[3, :adv.size] = adv[:k]
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    assert_within(_run(W, n, k, xq, m, qmm.PATH_GEMV_MMA), y_ref, T, "extreme codes")


@pytest.mark.slow
@pytest.mark.parametrize("m", [2, 8])
def test_gemv_mma_long_rows(oracle_mod, m):
    """k = 14336 (a down projection): the staged activations of 2 columns still fit, of 8
    they do not, and the call falls back to the dp4a GEMV; either way within the bound."""
    n, k = 512, 14336
    W, x = qmm_synth.make_dense("q4_K", n, k, m, seed=77)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    assert_within(_run(W, n, k, xq, m, qmm.PATH_AUTO), y_ref, T, f"long rows m={m}")


@pytest.mark.parametrize("m", [6, 8])
def test_gemv_mma_repeats_bit_exact(oracle_mod, m):
    """The automatic path at 6..8 columns is the MMA GEMV; its partial sums of a tile are
    added in a fixed warp order, so two calls give the same bits."""
    n, k = 3000, 5120
    W, x = qmm_synth.make_dense("q4_K", n, k, m, seed=3 + m)
    xq = oracle_mod.quantize_q8_1(x)
    a = _run(W, n, k, xq, m, qmm.PATH_AUTO)
    b = _run(W, n, k, xq, m, qmm.PATH_AUTO)
    assert np.array_equal(a, b)
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    assert_within(a, y_ref, T, f"auto m={m}")
