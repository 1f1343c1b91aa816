"""GPU parity of the padded-row layout: qmm_repack_aligned must write the oracle's padded
rows byte for byte, and qmm_mul_mat_aligned must meet the oracle's bound (1e-5 T per
element, the oracle multiplying the original rows) on every path the layout opens:
the bulk-copy GEMV for any Q6_K/Q8_0/Q4_0 row length and the tensor-core GEMM for Q6_K at
any n."""
import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth
from parity import assert_within

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _reset():
    yield
    qmm.qmm_set_force_path(0)


# Q6_K with n % 8 == 0 takes the row-group boxes on the padded stride as well
@pytest.mark.parametrize("fmt,n,k", [("q6_K", 300, 1280), ("q6_K", 17, 5120), ("q6_K", 136, 1280), ("q8_0", 300, 96),
                                     ("q8_0", 257, 2080), ("q4_0", 130, 224), ("q4_K", 40, 512)])
@pytest.mark.parametrize("m,path", [(1, 0), (5, 1), (40, 0), (40, 2), (40, 3)])
def test_aligned_matches_oracle(oracle_mod, fmt, n, k, m, path):
    W, x = qmm_synth.make_dense(fmt, n, k, m, seed=n * 7 + k + m)
    xq = oracle_mod.quantize_q8_1(x)
    Wa = qmm.qmm_repack_aligned(torch.from_numpy(W).to(DEV), fmt, n, k)
    torch.cuda.synchronize()
    assert np.array_equal(Wa.cpu().numpy(), oracle_mod.repack_aligned(W, fmt, n, k))
    qmm.qmm_set_force_path(path)
    y = qmm.qmm_mul_mat_aligned(Wa, fmt, n, k, torch.from_numpy(xq).to(DEV), m)
    torch.cuda.synchronize()
    y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
    assert_within(y.cpu().numpy(), y_ref, T, f"aligned {fmt} n={n} k={k} m={m} path={path}")
