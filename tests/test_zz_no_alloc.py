"""The workspace-free expert-routed matmul (qmm_mul_mat_id_noalloc), called through
the C ABI, against the oracle with the per-element bound |y - y_oracle| <= 1e-5 T, on
two calls in a row (the second call finds the first call's contents in the shared
scratch array), and against the workspace call qmm_mul_mat_id on the same inputs.
Cases: the grouped path with a few routing ids outside [0, E) (their rows must be
zero on both calls), the per-pair GEMV of decode sizes, and the empty problem.  This
file is collected last so that a failure here comes after every other test has run."""
import ctypes

import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import oracle
import qmm_synth
from parity import assert_within

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("E,n,k,T_,K,seed,bad", [
    (16, 96, 512, 40, 4, 1, 3),     # grouped CUDA-core GEMM, three invalid ids
    (128, 64, 256, 512, 8, 2, 0),   # grouped, many experts
    (16, 80, 512, 3, 4, 3, 1),      # 12 pairs: one GEMV per pair, one invalid id
])
def test_noalloc_matches_oracle_twice(oracle_mod, E, n, k, T_, K, seed, bad):
    qmm.build()
    L = qmm.lib()
    W, x, ids = qmm_synth.make_moe(E, n, k, T_, K, seed=seed)
    rng = np.random.default_rng(seed)
    for i in range(bad):  # ids outside [0, E): -1 and E + something
        ids[rng.integers(0, T_), rng.integers(0, K)] = -1 if i % 2 == 0 else E + i
    Wd = torch.from_numpy(W).to(DEV)
    idd = torch.from_numpy(ids).to(DEV)
    xq = qmm.qmm_quantize_q8_1(torch.from_numpy(x).to(DEV))
    torch.cuda.synchronize()
    y_ref, T, n_bad = oracle_mod.mul_mat_id(W, "q4_K", E, n, k, xq.cpu().numpy(), ids)
    assert n_bad == int(((ids < 0) | (ids >= E)).sum())
    ws = torch.empty(qmm.qmm_workspace_bytes("q4_K", n, k, T_, E, K), dtype=torch.uint8, device=DEV)
    y_ws = qmm.qmm_mul_mat_id(Wd, "q4_K", E, n, k, xq, idd, K, T_, workspace=ws)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    invalid = (ids < 0) | (ids >= E)
    for call in range(2):
        y = torch.full((T_, K, n), float("nan"), device=DEV)
        rc = L.qmm_mul_mat_id_noalloc(_p(Wd), 12, E, n, k, _p(xq), _p(idd), K, T_, _p(y), stream)
        assert rc == 0, qmm.qmm_status_string(rc)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert_within(got, y_ref, T, f"noalloc call {call}")
        assert np.all(got[invalid] == 0), f"call {call}: rows of invalid ids are not zero"
        # the workspace call meets the same bound on the same inputs
        assert_within(y_ws.cpu().numpy(), y_ref, T, "workspace call")


def test_noalloc_empty_problem():
    L = qmm.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y = torch.empty(0, device=DEV)
    rc = L.qmm_mul_mat_id_noalloc(ctypes.c_void_p(256), 12, 8, 64, 256, ctypes.c_void_p(256),
                                  ctypes.c_void_p(256), 4, 0, _p(y), stream)
    assert rc == 0
    torch.cuda.synchronize()


def test_noalloc_rejects_problems_beyond_the_scratch():
    L = qmm.lib()
    n_tokens, top_k = 1 << 20, 8  # 8M pairs: far more than 1 MiB of scratch holds
    rc = L.qmm_mul_mat_id_noalloc(ctypes.c_void_p(256), 12, 128, 64, 256, ctypes.c_void_p(256),
                                  ctypes.c_void_p(256), top_k, n_tokens, ctypes.c_void_p(256), None)
    assert rc == 5  # QMM_ERR_WORKSPACE, nothing enqueued
