"""Parity of the tensor-core GEMM (tcgen05, kind::f16 on integer-valued operands)
against the oracle: ragged tile edges in both dimensions, one to many superblocks,
with and without the stream-K split and its fixup pass."""
import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth
from parity import assert_within

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qmm.build()
    yield
    qmm.qmm_set_force_path(0)
    qmm.qmm_set_stream_k_mode(0)


def run_tc(oracle_mod, n, k, m, sk_mode, seed=0, x=None, fmt="q4_K", W=None):
    Wr, xr = qmm_synth.make_dense(fmt, n, k, m, seed=seed)
    W = Wr if W is None else W
    if x is not None:
        xr = x
    xq = oracle_mod.quantize_q8_1(xr)
    qmm.qmm_set_force_path(qmm.PATH_GEMM_TC)
    qmm.qmm_set_stream_k_mode(sk_mode)
    try:
        ws = torch.empty(max(256, qmm.qmm_workspace_bytes(fmt, n, k, m)), dtype=torch.uint8, device=DEV)
        y = torch.full((m, n), float("nan"), device=DEV)
        qmm.qmm_mul_mat(torch.from_numpy(W).to(DEV), fmt, n, k, torch.from_numpy(xq).to(DEV), m, y=y,
                        workspace=ws)
        torch.cuda.synchronize()
        status = qmm.qmm_read_device_status(ws)
    finally:
        qmm.qmm_set_force_path(0)
        qmm.qmm_set_stream_k_mode(0)
    assert status == 0, f"device status {status}"
    y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
    assert_within(y.cpu().numpy(), y_ref, T, f"tc {fmt} n={n} k={k} m={m} sk={sk_mode}")


def test_tc_single_tile_smallest(oracle_mod):
    run_tc(oracle_mod, 128, 256, 128, 1)


@pytest.mark.parametrize("n,k,m", [(128, 512, 128), (129, 256, 9), (1, 256, 17), (300, 1024, 130), (256, 768, 256),
                                   (77, 2048, 200)])
@pytest.mark.parametrize("sk", [1, 2])
def test_tc_parity(oracle_mod, n, k, m, sk):
    run_tc(oracle_mod, n, k, m, sk, seed=n + k + m)


def test_tc_auto_schedule(oracle_mod):
    run_tc(oracle_mod, 1000, 1024, 300, 0, seed=3)


@pytest.mark.parametrize("fmt", ["q4_K", "q6_K", "q8_0", "q4_0", "q5_K"])
def test_tc_persistent_whole_tiles(oracle_mod, fmt):
    """More whole tiles than SMs (16 x 11 = 176, ragged in both dimensions): persistent CTAs
    that each take a contiguous run of tiles (Q5_K keeps one CTA per tile)."""
    run_tc(oracle_mod, 2000, 256, 1290, 1, seed=17, fmt=fmt)


def test_tc_integer_exactness(oracle_mod):
    """Activations whose q8_1 codes hit +-127 everywhere: the largest integer dots
    (32 * 945 * 127 per sub-block) must still be exact in the fp32 accumulators."""
    n, k, m = 130, 512, 20
    x = np.where(np.random.default_rng(5).random((m, k)) < 0.5, -1.0, 1.0).astype(np.float32)
    run_tc(oracle_mod, n, k, m, 1, seed=9, x=x)


# Q8_0 on the tensor cores: int8 codes as exact fp16, a d per 32-block folded with d8
@pytest.mark.parametrize("n,k,m", [(128, 256, 128), (129, 512, 9), (300, 1024, 130), (77, 2048, 200),
                                   (1000, 1024, 300)])
@pytest.mark.parametrize("sk", [1, 2])
def test_tc_q8_0_parity(oracle_mod, n, k, m, sk):
    run_tc(oracle_mod, n, k, m, sk, seed=n + k + m, fmt="q8_0")


def test_tc_q8_0_extreme_codes(oracle_mod):
    """Codes -128 and 127 everywhere: the fp16 conversion must keep both ends exact."""
    n, k, m = 130, 512, 20
    W, x = qmm_synth.make_dense("q8_0", n, k, m, seed=4)
    blk = W.reshape(n, k // 32, 34)
    blk[:, ::2, 2:] = np.uint8(0x80)   # -128
    blk[:, 1::2, 2:] = np.uint8(0x7f)  # 127
    xq = oracle_mod.quantize_q8_1(x)
    qmm.qmm_set_force_path(qmm.PATH_GEMM_TC)
    try:
        y = qmm.qmm_mul_mat(torch.from_numpy(W).to(DEV), "q8_0", n, k, torch.from_numpy(xq).to(DEV), m)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    y_ref, T = oracle_mod.mul_mat(W, "q8_0", n, k, xq, m)
    assert_within(y.cpu().numpy(), y_ref, T, "tc q8_0 extreme codes")


# Q6_K on the tensor cores: 6-bit codes q - 32 in two exact fp16 planes per 32-block slot,
# d folded with d8.  n a multiple of 8: the raw superblocks arrive as boxes of row groups
# (one map row per 8 weight rows) and the tile columns are permuted to match, through
# whole tiles and stream-K partial slots alike.
@pytest.mark.parametrize("n,k,m", [(128, 256, 128), (136, 512, 9), (8, 256, 17), (1000, 1024, 300),
                                   (2048, 768, 200)])
@pytest.mark.parametrize("sk", [1, 2])
def test_tc_q6_k_parity(oracle_mod, n, k, m, sk):
    run_tc(oracle_mod, n, k, m, sk, seed=3 * n + k + m, fmt="q6_K")


def test_tc_q6_k_extreme_scales_and_codes(oracle_mod):
    """int8 sub-scales -128 and 127, codes 63 and 15 (q - 32 = 31 and -17): the largest
    per-16 dots and the fold with d * sc must stay within the bound."""
    n, k, m = 136, 512, 20
    W, x = qmm_synth.make_dense("q6_K", n, k, m, seed=8)
    blk = W.reshape(n, k // 256, 210)
    blk[:, :, 0:128] = np.uint8(0xFF)                      # low nibbles 15
    blk[:, 0::2, 128:192] = np.uint8(0xFF)                 # high bits 3 -> code 63
    blk[:, 1::2, 128:192] = np.uint8(0x00)                 # code 15
    blk[:, :, 192:200] = np.uint8(0x80)                    # sc = -128
    blk[:, :, 200:208] = np.uint8(0x7F)                    # sc = 127
    xq = oracle_mod.quantize_q8_1(x)
    qmm.qmm_set_force_path(qmm.PATH_GEMM_TC)
    try:
        y = qmm.qmm_mul_mat(torch.from_numpy(W).to(DEV), "q6_K", n, k, torch.from_numpy(xq).to(DEV), m)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    y_ref, T = oracle_mod.mul_mat(W, "q6_K", n, k, xq, m)
    assert_within(y.cpu().numpy(), y_ref, T, "tc q6_K extreme scales")


def test_tc_q6_k_odd_n_falls_back(oracle_mod):
    """n not a multiple of 8: the forced tensor-core path is not available for Q6_K and
    the call still returns the right product (CUDA-core GEMM)."""
    n, k, m = 130, 512, 40
    W, x = qmm_synth.make_dense("q6_K", n, k, m, seed=11)
    xq = oracle_mod.quantize_q8_1(x)
    qmm.qmm_set_force_path(qmm.PATH_GEMM_TC)
    try:
        y = qmm.qmm_mul_mat(torch.from_numpy(W).to(DEV), "q6_K", n, k, torch.from_numpy(xq).to(DEV), m)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    y_ref, T = oracle_mod.mul_mat(W, "q6_K", n, k, xq, m)
    assert_within(y.cpu().numpy(), y_ref, T, "q6_K odd n")


# Q4_0 on the tensor cores: offset codes q - 8 as exact fp16, a d per 32-block folded
# with d8 (k % 256 == 0: a row's 256 values are 144 bytes, one box of the raw map)
@pytest.mark.parametrize("n,k,m", [(128, 256, 128), (129, 512, 9), (1, 256, 17), (300, 1024, 130), (77, 2048, 200),
                                   (1000, 4096, 300)])
@pytest.mark.parametrize("sk", [1, 2])
def test_tc_q4_0_parity(oracle_mod, n, k, m, sk):
    run_tc(oracle_mod, n, k, m, sk, seed=5 * n + k + m, fmt="q4_0")


def test_tc_q4_0_extreme_codes(oracle_mod):
    """Codes 0 and 15 (values -8 and 7) against activations at +-127."""
    n, k, m = 130, 512, 20
    W, _ = qmm_synth.make_dense("q4_0", n, k, m, seed=4)
    blk = W.reshape(n, k // 32, 18)
    blk[:, ::2, 2:] = np.uint8(0x00)
    blk[:, 1::2, 2:] = np.uint8(0xFF)
    x = np.where(np.random.default_rng(8).random((m, k)) < 0.5, -1.0, 1.0).astype(np.float32)
    run_tc(oracle_mod, n, k, m, 1, x=x, W=W, fmt="q4_0")
