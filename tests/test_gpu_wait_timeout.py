"""Failure detection on the GPU without a fault: a bounded device wait is made to run
out, the kernel must report QMM_ERR_DEVICE through the workspace's status word, and the
next normal call on the same stream and workspace must be correct.

The test switch qmm_set_test_fault(1) makes the tensor-core GEMM's activation producer
issue no copy at all, so the MMA issuer's wait for the first stage (shortened to about
10^5 cycles under the switch) gives up.  Nothing is in flight when the kernel leaves."""
import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth
from parity import assert_within

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
QMM_ERR_DEVICE = 8


@pytest.fixture(autouse=True)
def _switches_off():
    yield
    qmm.qmm_set_test_fault(0)
    qmm.qmm_set_force_path(qmm.PATH_AUTO)


@pytest.mark.parametrize("fmt", ["q4_K", "q6_K"])
def test_bounded_wait_runs_out_then_recovers(oracle_mod, fmt):
    n, k, m = 256, 1024, 96
    W, x = qmm_synth.make_dense(fmt, n, k, m, seed=11)
    Wd = torch.from_numpy(W).to(DEV)
    xq = qmm.qmm_quantize_q8_1(torch.from_numpy(x).to(DEV))
    ws = torch.empty(qmm.qmm_workspace_bytes(fmt, n, k, m), dtype=torch.uint8, device=DEV)
    qmm.qmm_set_force_path(qmm.PATH_GEMM_TC)
    qmm.qmm_set_test_fault(1)
    qmm.qmm_mul_mat(Wd, fmt, n, k, xq, m, workspace=ws)
    assert qmm.qmm_read_device_status(ws) == QMM_ERR_DEVICE
    assert qmm.qmm_get_device_status(ws) == QMM_ERR_DEVICE
    qmm.qmm_set_test_fault(0)
    # the context is usable and the same stream and workspace give the right answer
    y = qmm.qmm_mul_mat(Wd, fmt, n, k, xq, m, workspace=ws)
    assert qmm.qmm_get_device_status(ws) == 0
    torch.cuda.synchronize()
    y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, xq.cpu().numpy(), m)
    assert_within(y.cpu().numpy(), y_ref, T, f"{fmt} after a wait ran out")


def test_bounded_wait_in_grouped_moe(oracle_mod):
    """The same through mul_mat_id: the hot experts' tiles run on the tensor-core GEMM."""
    E, n, k, T_, K = 8, 128, 512, 96, 4
    W, x, ids = qmm_synth.make_moe(E, n, k, T_, K, seed=12)
    Wd = torch.from_numpy(W).to(DEV)
    idd = torch.from_numpy(ids).to(DEV)
    xq = qmm.qmm_quantize_q8_1(torch.from_numpy(x).to(DEV))
    ws = torch.empty(qmm.qmm_workspace_bytes("q4_K", n, k, T_, E, K), dtype=torch.uint8, device=DEV)
    assert np.bincount(ids.ravel(), minlength=E).max() > 16  # some expert takes the tensor-core tiles
    qmm.qmm_set_test_fault(1)
    qmm.qmm_mul_mat_id(Wd, "q4_K", E, n, k, xq, idd, K, T_, workspace=ws)
    assert qmm.qmm_get_device_status(ws) == QMM_ERR_DEVICE
    qmm.qmm_set_test_fault(0)
    y = qmm.qmm_mul_mat_id(Wd, "q4_K", E, n, k, xq, idd, K, T_, workspace=ws)
    assert qmm.qmm_get_device_status(ws) == 0
    y_ref, Tr, _ = oracle_mod.mul_mat_id(W, "q4_K", E, n, k, xq.cpu().numpy(), ids)
    assert_within(y.cpu().numpy(), y_ref, Tr, "mul_mat_id after a wait ran out")
