"""The workspace-free expert-routed matmul (qmm_mul_mat_id_noalloc), called through
the C ABI, must give the same output as qmm_mul_mat_id with a workspace, on two
calls in a row (the second call finds the first call's contents in the shared
scratch array).  This file is collected last so that a failure here comes after
every other test has run."""
import ctypes

import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth
from parity import TOL

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_call_twice():
    qmm.build()
    L = qmm.lib()
    cases = [(16, 96, 512, 40, 4, 1), (128, 64, 256, 512, 8, 2)]
    for (E, n, k, T_, K, seed) in cases:
        W, x, ids = qmm_synth.make_moe(E, n, k, T_, K, seed=seed)
        Wd = torch.from_numpy(W).to(DEV)
        idd = torch.from_numpy(ids).to(DEV)
        xq = qmm.qmm_quantize_q8_1(torch.from_numpy(x).to(DEV))
        ws = torch.empty(qmm.qmm_workspace_bytes("q4_K", n, k, T_, E, K), dtype=torch.uint8, device=DEV)
        y_ref = qmm.qmm_mul_mat_id(Wd, "q4_K", E, n, k, xq, idd, K, T_, workspace=ws)
        torch.cuda.synchronize()
        ref = y_ref.cpu().numpy().astype(np.float64)
        scale = np.abs(ref).max() + 1e-30
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for call in range(2):
            y = torch.full((T_, K, n), float("nan"), device=DEV)
            rc = L.qmm_mul_mat_id_noalloc(_p(Wd), 12, E, n, k, _p(xq), _p(idd), K, T_, _p(y), stream)
            assert rc == 0, qmm.qmm_status_string(rc)
            torch.cuda.synchronize()
            got = y.cpu().numpy().astype(np.float64)
            assert np.all(np.isfinite(got)), f"call {call}: unwritten outputs"
            # the workspace call may take the tensor-core grouped GEMM and this one the
            # CUDA-core one: both sum the same exact integer dots and differ only in the
            # fp32 order of the fold, far inside the parity tolerance
            assert np.all(np.abs(got - ref) <= TOL * scale), f"call {call}: differs from the workspace call"


def test_noalloc_rejects_problems_beyond_the_scratch():
    L = qmm.lib()
    n_tokens, top_k = 1 << 20, 8  # 8M pairs: far more than 1 MiB of scratch holds
    rc = L.qmm_mul_mat_id_noalloc(ctypes.c_void_p(256), 12, 128, 64, 256, ctypes.c_void_p(256),
                                  ctypes.c_void_p(256), top_k, n_tokens, ctypes.c_void_p(256), None)
    assert rc == 5  # QMM_ERR_WORKSPACE, nothing enqueued
