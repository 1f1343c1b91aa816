"""GPU parity: every path of the CUDA library against the CPU oracle on the same
seeded inputs.  q8_1 must be bit-exact; y must satisfy |y - y_oracle| <= 1e-5 * T
with T the per-element sum of |block terms|."""
import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth
from parity import TOL, adversarial_x_rows, assert_within, near_tie_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qmm.build()
    qmm.lib()
    yield
    qmm.qmm_set_force_path(0)
    qmm.qmm_set_stream_k_mode(0)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_mul_mat(W, fmt, n, k, xq, m, path=0):
    qmm.qmm_set_force_path(path)
    try:
        y = qmm.qmm_mul_mat(to_dev(W), fmt, n, k, to_dev(xq), m)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_force_path(0)
    return y.cpu().numpy()


# ---------------------------------------------------------------- quantizer

@pytest.mark.parametrize("m,k", [(1, 32), (3, 5120), (16, 2048), (2048, 4096), (7, 96)])
def test_quantize_bitexact_random(oracle_mod, m, k):
    x = qmm_synth.gen_x(np.random.default_rng(m * 1000 + k), m, k)
    x[0, :32] *= 1000.0
    got = qmm.qmm_quantize_q8_1(to_dev(x)).cpu().numpy()
    assert np.array_equal(got, oracle_mod.quantize_q8_1(x))


def test_quantize_bitexact_adversarial(oracle_mod):
    x = adversarial_x_rows().reshape(1, -1)
    got = qmm.qmm_quantize_q8_1(to_dev(x)).cpu().numpy()
    assert np.array_equal(got, oracle_mod.quantize_q8_1(x))


def test_quantize_tie_and_scale_edges(oracle_mod):
    """Values that land exactly on .5 after the fp32 division, for many scales."""
    rng = np.random.default_rng(9)
    rows = []
    for _ in range(64):
        amax = np.float32(rng.uniform(0.01, 100))
        d = amax / np.float32(127)
        q = rng.integers(-126, 127, 32).astype(np.float32)
        x = ((q + np.float32(0.5)) * d).astype(np.float32)
        x[rng.integers(0, 32)] = amax
        rows.append(x)
    x = np.stack(rows).reshape(2, -1)
    got = qmm.qmm_quantize_q8_1(to_dev(x)).cpu().numpy()
    assert np.array_equal(got, oracle_mod.quantize_q8_1(x))


@pytest.mark.parametrize("nrows,shape", [(4096, (8, -1)), (512, (1, -1))])
def test_quantize_near_ties_bitexact(oracle_mod, nrows, shape):
    """Quotients within a few ulps of the rounding ties, over scales from 2^-20 to 2^20: 4096
    blocks (4 lanes per block) and 512 (a warp per block)."""
    x = near_tie_rows(21, nrows).reshape(*shape)
    got = qmm.qmm_quantize_q8_1(to_dev(x)).cpu().numpy()
    assert np.array_equal(got, oracle_mod.quantize_q8_1(x))


def test_quantize_adversarial_many_blocks(oracle_mod):
    """The adversarial rows repeated past 2048 blocks, so the 4-lanes-per-block form runs."""
    row = adversarial_x_rows().reshape(1, -1)
    x = np.tile(row, (max(1, -(-2048 * 32 // row.size)), 1))
    got = qmm.qmm_quantize_q8_1(to_dev(x)).cpu().numpy()
    assert np.array_equal(got, oracle_mod.quantize_q8_1(x))


# ---------------------------------------------------------------- GEMV (m <= 8)

# Q6_K with an even n and Q8_0 with k/32 a multiple of 8 stream their rows with bulk
# copies; the other shapes take the direct-load kernel.
# Long rows get shallower rings: at one column Q4_K k = 11776 takes 4 stages, k = 14336
# and Q8_0 k = 8192 take 3 (three consumer groups), Q4_K k = 16384 none (the direct
# kernel); Q6_K k = 5120 takes 6 stages (three groups).  Q4_K rows from k = 8192 on at
# one or two columns take the two-row fold (a warp's two rows share each unit's x loads).
GEMV_SHAPES = {"q4_K": [(1, 256), (7, 512), (129, 2304), (45, 8192), (64, 11776), (33, 14336), (20, 16384)],
               "q6_K": [(1, 256), (7, 512), (129, 2304), (130, 2304), (64, 512), (2, 5120)],
               "q8_0": [(1, 32), (7, 96), (129, 1056), (33, 2048), (130, 256), (64, 5120), (40, 8192)],
               # odd block counts (k = 96, 1056: rows only 2-byte aligned, a last unit of one
               # block) take the direct-load kernel; k % 256 == 0 the bulk copies
               "q4_0": [(1, 32), (7, 96), (129, 1056), (33, 2048), (130, 256), (64, 4096), (40, 8192)]}


@pytest.mark.parametrize("fmt", ["q4_K", "q6_K", "q8_0", "q4_0"])
@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 6, 7, 8])
def test_gemv_parity(oracle_mod, fmt, m):
    for (n, k) in GEMV_SHAPES[fmt]:
        W, x = qmm_synth.make_dense(fmt, n, k, m, seed=n + k + m)
        xq = oracle_mod.quantize_q8_1(x)
        y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
        assert_within(run_mul_mat(W, fmt, n, k, xq, m, path=1), y_ref, T, f"gemv {fmt} n={n} k={k} m={m}")


# ---------------------------------------------------------------- tiled GEMM paths

GEMM_CASES = [("q4_K", 129, 512, 9), ("q4_K", 300, 1024, 65), ("q4_K", 64, 256, 130), ("q4_K", 1, 256, 17),
              ("q6_K", 129, 512, 17), ("q6_K", 200, 768, 64), ("q8_0", 129, 1056, 33), ("q8_0", 70, 96, 127),
              ("q4_0", 129, 512, 9), ("q4_0", 300, 1056, 65), ("q4_0", 64, 96, 130), ("q4_0", 1000, 4096, 300)]


@pytest.mark.parametrize("fmt,n,k,m", GEMM_CASES)
@pytest.mark.parametrize("path", [2, 0])
def test_gemm_parity(oracle_mod, fmt, n, k, m, path):
    W, x = qmm_synth.make_dense(fmt, n, k, m, seed=3 * n + k + m)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
    assert_within(run_mul_mat(W, fmt, n, k, xq, m, path=path), y_ref, T, f"gemm path={path} {fmt} n={n} k={k} m={m}")


@pytest.mark.parametrize("m", [1, 4, 8, 9, 16])
def test_gemv_and_gemm_agree(oracle_mod, m):
    """The same m through the GEMV and the tiled GEMM: both within the bound, and
    within 2x the bound of each other."""
    n, k = 257, 1024
    W, x = qmm_synth.make_dense("q4_K", n, k, m, seed=77 + m)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    a = run_mul_mat(W, "q4_K", n, k, xq, m, path=1)
    b = run_mul_mat(W, "q4_K", n, k, xq, m, path=2)
    assert_within(a, y_ref, T, "gemv")
    assert_within(b, y_ref, T, "gemm")
    assert np.all(np.abs(a.astype(np.float64) - b) <= 2 * TOL * T)


def test_zero_activation_gives_exact_zero(oracle_mod):
    n, k, m = 65, 512, 12
    W, _ = qmm_synth.make_dense("q4_K", n, k, m)
    xq = oracle_mod.quantize_q8_1(np.zeros((m, k), np.float32))
    for path in (1, 2, 0):
        if path == 1 and m > 8:
            continue
        y = run_mul_mat(W, "q4_K", n, k, xq, m, path=path)
        assert np.all(y == 0)


# ---------------------------------------------------------------- MoE

def moe_check(oracle_mod, E, n, k, T_, K, seed, corrupt=0, fmt="q4_K", per_slot=False):
    W, x, ids = qmm_synth.make_moe(E, n, k, T_, K, seed=seed, fmt=fmt)
    if corrupt:
        rng = np.random.default_rng(seed)
        for _ in range(corrupt):
            ids[rng.integers(0, T_), rng.integers(0, K)] = rng.choice([-1, E, E + 5])
    if per_slot:  # one activation row per (token, slot): fresh rows, seeded
        x = qmm_synth.gen_x(np.random.default_rng(seed + 1), T_ * K, k)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, Tr, bad = oracle_mod.mul_mat_id(W, fmt, E, n, k, xq, ids, per_slot=per_slot)
    ws = torch.empty(qmm.qmm_workspace_bytes(fmt, n, k, T_, E, K), dtype=torch.uint8, device=DEV)
    y = torch.full((T_, K, n), float("nan"), device=DEV)
    call = qmm.qmm_mul_mat_id_slot if per_slot else qmm.qmm_mul_mat_id
    call(to_dev(W), fmt, E, n, k, to_dev(xq), to_dev(ids), K, T_, y=y, workspace=ws)
    status = qmm.qmm_read_device_status(ws)
    assert status == (7 if bad else 0)
    assert_within(y.cpu().numpy(), y_ref, Tr, f"moe {fmt} E={E} n={n} k={k} T={T_} K={K} per_slot={per_slot}")


# The last two put several 128-pair tiles on each expert and split tiles between
# CTAs of the stream-K schedule of the tensor-core grouped GEMM (partials + fixup).
@pytest.mark.parametrize("E,n,k,T_,K", [(4, 64, 256, 9, 2), (16, 130, 512, 70, 4), (128, 96, 256, 512, 8),
                                        (3, 33, 512, 200, 3), (8, 384, 2048, 600, 2), (5, 200, 1024, 333, 3)])
def test_moe_parity(oracle_mod, E, n, k, T_, K):
    moe_check(oracle_mod, E, n, k, T_, K, seed=E + n + T_)


def test_moe_invalid_ids_flagged_and_zeroed(oracle_mod):
    moe_check(oracle_mod, 8, 64, 256, 40, 4, seed=5, corrupt=6)


@pytest.mark.parametrize("fmt,n,k", [("q6_K", 130, 2304), ("q6_K", 1000, 5120), ("q8_0", 130, 256),
                                     ("q8_0", 512, 5120), ("q4_0", 130, 2048), ("q4_0", 512, 4096)])
@pytest.mark.parametrize("m", [1, 3, 8])
def test_gemv_bulk_and_direct_agree(oracle_mod, fmt, n, k, m):
    """The bulk-copy GEMV (path 1) and the direct-load GEMV (path 4) fold the same
    decoded units in the same order: their outputs agree to the bit."""
    W, x = qmm_synth.make_dense(fmt, n, k, m, seed=n + m)
    xq = oracle_mod.quantize_q8_1(x)
    a = run_mul_mat(W, fmt, n, k, xq, m, path=1)
    b = run_mul_mat(W, fmt, n, k, xq, m, path=4)
    assert np.array_equal(a, b)
    y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
    assert_within(a, y_ref, T, f"bulk gemv {fmt} n={n} k={k} m={m}")


# Decode-size routing (tokens x top_k <= 32 pairs): one GEMV per pair, expert ids read on
# the device.  32 pairs is the largest such call, 33 goes back to the grouped GEMM; Q6_K
# rows of 9 superblocks (k = 2304) are not bulk-copy aligned and take the grouped GEMM too.
@pytest.mark.parametrize("fmt,E,n,k,T_,K", [("q4_K", 32, 384, 2048, 1, 8), ("q4_K", 16, 1000, 512, 3, 8),
                                            ("q4_K", 8, 256, 256, 4, 8), ("q4_K", 8, 256, 256, 11, 3),
                                            ("q6_K", 16, 130, 1024, 2, 4), ("q6_K", 8, 96, 2048, 1, 8),
                                            ("q6_K", 8, 96, 2304, 1, 8),
                                            ("q8_0", 16, 136, 256, 2, 8), ("q8_0", 8, 100, 512, 1, 2),
                                            ("q4_0", 16, 136, 256, 2, 8), ("q4_0", 8, 100, 96, 1, 8)])
def test_moe_decode_gemv_parity(oracle_mod, fmt, E, n, k, T_, K):
    moe_check(oracle_mod, E, n, k, T_, K, seed=E + n + T_ + K, fmt=fmt)


def test_moe_decode_gemv_invalid_ids_flagged_and_zeroed(oracle_mod):
    moe_check(oracle_mod, 16, 200, 512, 2, 8, seed=17, corrupt=3)


# One activation row per (token, slot) pair (a down projection): the decode GEMV, the
# tensor-core grouped GEMM and the CUDA-core grouped GEMM
@pytest.mark.parametrize("fmt,E,n,k,T_,K", [("q4_K", 16, 256, 512, 2, 4), ("q4_K", 16, 130, 512, 64, 4),
                                            ("q4_K", 8, 384, 1024, 300, 2), ("q6_K", 8, 130, 512, 40, 2),
                                            ("q8_0", 8, 64, 256, 50, 3), ("q4_0", 8, 64, 256, 50, 3),
                                            ("q4_0", 16, 100, 512, 2, 4)])
def test_moe_per_slot_parity(oracle_mod, fmt, E, n, k, T_, K):
    moe_check(oracle_mod, E, n, k, T_, K, seed=2 * E + n + T_, fmt=fmt, per_slot=True)


# Q4_0 through the grouped CUDA-core MoE GEMM (more than 32 pairs), with skewed routing
@pytest.mark.parametrize("E,n,k,T_,K", [(8, 130, 512, 70, 4), (16, 64, 1056, 100, 2)])
def test_moe_q4_0_grouped_parity(oracle_mod, E, n, k, T_, K):
    moe_check(oracle_mod, E, n, k, T_, K, seed=3 * E + n, fmt="q4_0")


@pytest.mark.parametrize("path", [1, 2, 4])
def test_q4_0_extreme_codes(oracle_mod, path):
    """Codes 0 and 15 (values -8 and 7) against activations at +-127: the largest
    integer dots of the format must stay exact on every path."""
    n, k, m = 130, 512, 9 if path == 2 else 4
    W, _ = qmm_synth.make_dense("q4_0", n, k, m, seed=6)
    blk = W.reshape(n, k // 32, 18)
    blk[0::2, :, 2:] = np.uint8(0x00)
    blk[1::2, :, 2:] = np.uint8(0xFF)
    x = np.where(np.random.default_rng(7).random((m, k)) < 0.5, -1.0, 1.0).astype(np.float32)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q4_0", n, k, xq, m)
    assert_within(run_mul_mat(W, "q4_0", n, k, xq, m, path=path), y_ref, T, f"q4_0 extreme path={path}")


# Cold experts (1..16 pairs) run as 16-column slabs on the skinny tensor-core kernel, the
# others on 128-pair tiles of the grouped GEMM; hand-built routings pin the boundary.
def moe_check_ids(oracle_mod, E, n, k, ids, seed, per_slot=False):
    T_, K = ids.shape
    W = qmm_synth.gen_weights("q4_K", np.random.default_rng(seed), E * n, k).reshape(E, n, -1)
    x = qmm_synth.gen_x(np.random.default_rng(seed + 1), T_ * K if per_slot else T_, k)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, Tr, bad = oracle_mod.mul_mat_id(W, "q4_K", E, n, k, xq, ids, per_slot=per_slot)
    ws = torch.empty(qmm.qmm_workspace_bytes("q4_K", n, k, T_, E, K), dtype=torch.uint8, device=DEV)
    y = torch.full((T_, K, n), float("nan"), device=DEV)
    call = qmm.qmm_mul_mat_id_slot if per_slot else qmm.qmm_mul_mat_id
    call(to_dev(W), "q4_K", E, n, k, to_dev(xq), to_dev(ids), K, T_, y=y, workspace=ws)
    assert qmm.qmm_read_device_status(ws) == (7 if bad else 0)
    assert_within(y.cpu().numpy(), y_ref, Tr, f"moe ids E={E} n={n} k={k} T={T_} K={K} per_slot={per_slot}")


def routing(counts, K, seed, extra_invalid=0):
    """ids [T][K] giving expert e exactly counts[e] pairs (shuffled), invalid ids appended."""
    flat = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)] +
                          [np.full(extra_invalid, -1, np.int32)])
    pad = (-len(flat)) % K
    flat = np.concatenate([flat, np.full(pad, len(counts), np.int32)])  # id E: invalid
    np.random.default_rng(seed).shuffle(flat)
    return flat.reshape(-1, K)


@pytest.mark.parametrize("per_slot", [False, True])
def test_moe_cold_hot_boundary(oracle_mod, per_slot):
    counts = [16, 17, 1, 0, 15, 2, 130, 16, 3, 40]
    moe_check_ids(oracle_mod, len(counts), 130, 512, routing(counts, 4, seed=3), seed=4, per_slot=per_slot)


def test_moe_all_cold(oracle_mod):
    counts = [1 + (e * 7) % 16 for e in range(40)]
    moe_check_ids(oracle_mod, 40, 256, 768, routing(counts, 8, seed=5), seed=6)


def test_moe_cold_with_invalid_ids(oracle_mod):
    counts = [5, 0, 12, 16, 3, 200]
    moe_check_ids(oracle_mod, 6, 96, 1024, routing(counts, 2, seed=7, extra_invalid=9), seed=8)


@pytest.mark.parametrize("E,n,k,T_,K", [(64, 256, 512, 40, 8), (32, 130, 768, 20, 4), (128, 1536, 256, 64, 8)])
def test_moe_mostly_cold_parity(oracle_mod, E, n, k, T_, K):
    moe_check(oracle_mod, E, n, k, T_, K, seed=E + T_)


# Long rows: the GEMV stages x in shared memory ((k/64) * 96 bytes per column), so from
# k = 155136 on a single column no longer fits and m <= 8 goes to the GEMM paths; the
# largest k the ABI accepts is 2^20.
@pytest.mark.parametrize("fmt,n,k,m", [("q4_K", 40, 154880, 1), ("q4_K", 40, 155136, 1), ("q4_K", 9, 1 << 20, 1),
                                       ("q4_K", 9, 1 << 20, 3), ("q8_0", 17, 155136, 2), ("q6_K", 16, 1 << 19, 1),
                                       ("q4_0", 24, 1 << 20, 2)])
def test_long_rows_up_to_the_k_limit(oracle_mod, fmt, n, k, m):
    W, x = qmm_synth.make_dense(fmt, n, k, m, seed=k % 1000 + m)
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
    assert_within(run_mul_mat(W, fmt, n, k, xq, m), y_ref, T, f"long rows {fmt} n={n} k={k} m={m}")


def test_k_above_the_limit_is_refused():
    W = torch.zeros(16 * ((1 << 20) + 256) // 256 * 144, dtype=torch.uint8, device=DEV)
    xq = torch.zeros(((1 << 20) + 256) // 32 * 36, dtype=torch.uint8, device=DEV)
    with pytest.raises(qmm.QMMError) as e:
        qmm.qmm_mul_mat(W, "q4_K", 16, (1 << 20) + 256, xq, 1)
    assert e.value.code == 2


# The grouped tensor-core GEMM for every format it supports (Q6_K: n % 8 == 0), with
# stream-K splitting tiles over CTAs; Q6_K with n % 8 != 0 stays on the CUDA-core path.
@pytest.mark.parametrize("fmt,E,n,k,T_,K", [("q8_0", 16, 200, 768, 300, 4), ("q8_0", 8, 64, 256, 50, 3),
                                            ("q4_0", 12, 130, 1024, 400, 3), ("q6_K", 8, 136, 512, 60, 4),
                                            ("q6_K", 16, 256, 1024, 300, 2), ("q6_K", 8, 130, 512, 60, 4)])
def test_moe_grouped_tc_other_formats(oracle_mod, fmt, E, n, k, T_, K):
    moe_check(oracle_mod, E, n, k, T_, K, seed=E + n + k + T_, fmt=fmt)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0", "q6_K"])
def test_moe_grouped_tc_other_formats_per_slot(oracle_mod, fmt):
    moe_check(oracle_mod, 8, 136, 512, 90, 3, seed=11, fmt=fmt, per_slot=True)
