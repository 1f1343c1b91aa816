"""GPU parity at the full sizes of the pages' workloads, through the same calls the
benchmark times.  Whole outputs are compared where the oracle finishes in seconds
(m = 1..8 and the small PR1 case); larger products are compared on sampled
outputs, always including the edge rows and columns of the last tiles."""
import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth
from parity import assert_within

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib(oracle_mod):
    qmm.build()
    oracle_mod.set_threads(0)
    yield
    qmm.qmm_set_force_path(0)


def sample_positions(rng, n, m, count):
    rows = np.concatenate([rng.integers(0, n, count), [0, n - 1, n - 2, max(0, n - 129)]])
    cols = np.concatenate([rng.integers(0, m, count), [m - 1, 0, m - 1, m // 2]])
    return rows.astype(np.int64), cols.astype(np.int64)


def dense_case(oracle_mod, fmt, n, k, ms, full_upto=8, samples=3000, seed=0):
    W, x = qmm_synth.make_dense(fmt, n, k, max(ms), seed=seed)
    Wd = torch.from_numpy(W).to(DEV)
    xd = torch.from_numpy(x).to(DEV)
    xq_gpu = qmm.qmm_quantize_q8_1(xd)
    xq = oracle_mod.quantize_q8_1(x)
    assert np.array_equal(xq_gpu.cpu().numpy(), xq), "q8_1 not bit-exact"
    for m in ms:
        y = qmm.qmm_mul_mat(Wd, fmt, n, k, xq_gpu[:m].contiguous(), m)
        torch.cuda.synchronize()
        y = y.cpu().numpy()
        if m <= full_upto:
            y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, xq[:m], m)
            assert_within(y, y_ref, T, f"{fmt} n={n} k={k} m={m}")
        else:
            rng = np.random.default_rng(m)
            rows, cols = sample_positions(rng, n, m, samples)
            y_ref, T = oracle_mod.mul_mat_at(W, fmt, n, k, xq[:m], m, rows, cols)
            assert_within(y[cols, rows], y_ref, T, f"{fmt} n={n} k={k} m={m} (sampled)")


def test_pr1_q4K_n1024_k2048_m16(oracle_mod):
    dense_case(oracle_mod, "q4_K", 1024, 2048, [16], full_upto=16)


def test_decode_q4K_n17408_k5120(oracle_mod):
    dense_case(oracle_mod, "q4_K", 17408, 5120, [1, 2, 4, 5, 8])


def test_decode_q4K_direct_loads(oracle_mod):
    qmm.qmm_set_force_path(qmm.PATH_GEMV_DIRECT)
    try:
        dense_case(oracle_mod, "q4_K", 17408, 5120, [1, 8])
    finally:
        qmm.qmm_set_force_path(0)


def test_prefill_q4K_n14336_k4096(oracle_mod):
    dense_case(oracle_mod, "q4_K", 14336, 4096, [512, 2048])


def test_prefill_q4K_n4100_edge_tiles(oracle_mod):
    dense_case(oracle_mod, "q4_K", 4100, 4096, [512], samples=2000)


def test_mixed_q6K_n151936_k5120(oracle_mod):
    dense_case(oracle_mod, "q6_K", 151936, 5120, [1, 512], full_upto=1, samples=2000)


def test_mixed_q80_n5120_k5120(oracle_mod):
    dense_case(oracle_mod, "q8_0", 5120, 5120, [1, 512], full_upto=1)


def test_moe_e128_n1536_k4096_t512_top8(oracle_mod):
    E, n, k, T_, K = 128, 1536, 4096, 512, 8
    W, x, ids = qmm_synth.make_moe(E, n, k, T_, K, seed=0)
    xq = oracle_mod.quantize_q8_1(x)
    ws = torch.empty(qmm.qmm_workspace_bytes("q4_K", n, k, T_, E, K), dtype=torch.uint8, device=DEV)
    y = qmm.qmm_mul_mat_id(torch.from_numpy(W).to(DEV), "q4_K", E, n, k, torch.from_numpy(xq).to(DEV),
                           torch.from_numpy(ids).to(DEV), K, T_, workspace=ws)
    assert qmm.qmm_read_device_status(ws) == 0
    y = y.cpu().numpy()
    rng = np.random.default_rng(1)
    t = rng.integers(0, T_, 3000)
    s = rng.integers(0, K, 3000)
    r = rng.integers(0, n, 3000)
    r[:4] = [0, n - 1, 0, n - 1]
    # include the hottest and the coldest experts
    counts = np.bincount(ids.ravel(), minlength=E)
    for e in (int(np.argmax(counts)), int(np.argmin(counts))):
        tt, ss = np.argwhere(ids == e)[0]
        t[4 + e % 4], s[4 + e % 4] = tt, ss
    y_ref = np.empty(len(t))
    T = np.empty(len(t))
    for e in np.unique(ids[t, s]):
        sel = np.nonzero(ids[t, s] == e)[0]
        yy, TT = oracle_mod.mul_mat_at(W[e], "q4_K", n, k, xq, T_, r[sel], t[sel])
        y_ref[sel] = yy
        T[sel] = TT
    assert_within(y[t, s, r], y_ref, T, "moe full size (sampled)")


def test_q40_n8192_k4096(oracle_mod):
    dense_case(oracle_mod, "q4_0", 8192, 4096, [1, 512], full_upto=1)


def test_moe_decode_e128_n1536_k4096_t1_top8(oracle_mod):
    """The decode form of the MoE workload (one token, top-8: one GEMV per pair), whole output."""
    E, n, k, T_, K = 128, 1536, 4096, 1, 8
    W, x, ids = qmm_synth.make_moe(E, n, k, T_, K, seed=2)
    xq = oracle_mod.quantize_q8_1(x)
    ws = torch.empty(max(256, qmm.qmm_workspace_bytes("q4_K", n, k, T_, E, K)), dtype=torch.uint8, device=DEV)
    y = qmm.qmm_mul_mat_id(torch.from_numpy(W).to(DEV), "q4_K", E, n, k, torch.from_numpy(xq).to(DEV),
                           torch.from_numpy(ids).to(DEV), K, T_, workspace=ws)
    assert qmm.qmm_read_device_status(ws) == 0
    y_ref, T, bad = oracle_mod.mul_mat_id(W, "q4_K", E, n, k, xq, ids)
    assert bad == 0
    assert_within(y.cpu().numpy(), y_ref, T, "moe decode full size")


@pytest.mark.parametrize("m", [1, 512])
def test_glu_packed_n14336_k4096(oracle_mod, m):
    """The fused gate/up rows of the bench on the interleaved tensor: m = 1 whole, m = 512
    sampled; the same bits as the two-tensor call."""
    n, k = 14336, 4096
    W, x = qmm_synth.make_dense("q4_K", 2 * n, k, m, seed=0)
    Wg, Wu = W[:n].copy(), W[n:].copy()
    xq = oracle_mod.quantize_q8_1(x)
    Wg_d, Wu_d, xq_d = (torch.from_numpy(a).to(DEV) for a in (Wg, Wu, xq))
    y_p = qmm.qmm_mul_mat_glu_packed(qmm.qmm_repack_glu(Wg_d, Wu_d, "q4_K", n, k), "q4_K", n, k, xq_d, m)
    y_2 = qmm.qmm_mul_mat_glu(Wg_d, Wu_d, "q4_K", n, k, xq_d, m)
    torch.cuda.synchronize()
    a = y_p.cpu().numpy()
    assert np.array_equal(a, y_2.cpu().numpy())
    if m == 1:
        y_ref, tol = oracle_mod.mul_mat_glu(Wg, Wu, "q4_K", n, k, xq, m)
        assert not (np.abs(a - y_ref) > tol).any()
    else:
        rng = np.random.default_rng(5)
        rows, cols = sample_positions(rng, n, m, 1500)
        ref, tol = oracle_mod.mul_mat_glu_at(Wg, Wu, "q4_K", n, k, xq, m, rows, cols)
        assert not (np.abs(a[cols, rows] - ref) > tol).any()
