"""Pins for the oracle's fold: special cases that reduce to an integer matmul,
brute force against the dequantized fp64 matmul, the min term's sign and
indexing, MoE reduction to the dense routine, and bucketing against a stable
sort."""
import numpy as np
import pytest

import qmm_synth
from blockpack import pack_q4_0, pack_q4_K, pack_q5_K, pack_q6_K, pack_q8_0, pack_q8_1


def _q8_1_rows(q: np.ndarray, d: np.ndarray, s: np.ndarray) -> np.ndarray:
    """q8_1 bytes from int8 q [m][k] and per-block fp16 d, s [m][k/32]."""
    m, k = q.shape
    out = np.zeros((m, k // 32, 36), np.uint8)
    for r in range(m):
        for b in range(k // 32):
            out[r, b] = pack_q8_1(d[r, b], s[r, b], q[r, 32 * b:32 * b + 32])
    return out.reshape(m, -1)


def test_q4_K_integer_matmul_special_case(oracle_mod):
    """d = 1, dmin = 0, all sub-block scales 1 and q8_1 d = 1: the fold is the
    plain integer matmul of the nibble codes with the int8 activations."""
    rng = np.random.default_rng(21)
    n, k, m = 5, 512, 3
    Qw = rng.integers(0, 16, (n, k))
    rows = []
    for r in range(n):
        rows.append(np.concatenate([pack_q4_K(1.0, 0.0, np.ones(8, int), rng.integers(0, 64, 8), Qw[r, 256 * s:256 * s + 256])
                                    for s in range(k // 256)]))
    W = np.stack(rows)
    Qx = rng.integers(-127, 128, (m, k))
    xq = _q8_1_rows(Qx, np.ones((m, k // 32)), rng.uniform(-3, 3, (m, k // 32)))
    y, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    assert np.array_equal(y, (Qx @ Qw.T).astype(np.float64))


def test_q4_K_min_term_special_case(oracle_mod):
    """All scales 0, d = 0, dmin = 1: y[c][r] = -sum_b m[r,b] * s[c,b]."""
    rng = np.random.default_rng(22)
    n, k, m = 4, 768, 3
    M = rng.integers(0, 64, (n, k // 32))
    rows = []
    for r in range(n):
        rows.append(np.concatenate([pack_q4_K(0.0, 1.0, np.zeros(8, int), M[r, 8 * s:8 * s + 8], rng.integers(0, 16, 256))
                                    for s in range(k // 256)]))
    W = np.stack(rows)
    S = rng.uniform(-4, 4, (m, k // 32)).astype(np.float16).astype(np.float64)
    xq = _q8_1_rows(rng.integers(-127, 128, (m, k)), rng.uniform(0, 1, (m, k // 32)), S)
    y, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    assert np.allclose(y, -(S @ M.T), rtol=1e-15, atol=0)
    assert np.allclose(T, np.abs(S) @ M.T, rtol=1e-15, atol=0)


def test_q6_K_integer_matmul_special_case(oracle_mod):
    """d = 1, q8_1 d = 1: the fold is sum_j sc_j * (int dot of sub-block j)."""
    rng = np.random.default_rng(23)
    n, k, m = 4, 512, 3
    V = rng.integers(-32, 32, (n, k))
    SC = rng.integers(-128, 128, (n, k // 16))
    W = np.stack([np.concatenate([pack_q6_K(1.0, SC[r, 16 * s:16 * s + 16], V[r, 256 * s:256 * s + 256])
                                  for s in range(k // 256)]) for r in range(n)])
    Qx = rng.integers(-127, 128, (m, k))
    xq = _q8_1_rows(Qx, np.ones((m, k // 32)), np.zeros((m, k // 32)))
    y, _ = oracle_mod.mul_mat(W, "q6_K", n, k, xq, m)
    assert np.array_equal(y, (Qx @ (V * np.repeat(SC, 16, axis=1)).T).astype(np.float64))


def test_q8_0_integer_matmul_special_case(oracle_mod):
    rng = np.random.default_rng(24)
    n, k, m = 6, 320, 4
    Qw = rng.integers(-128, 128, (n, k))
    W = np.stack([np.concatenate([pack_q8_0(1.0, Qw[r, 32 * b:32 * b + 32]) for b in range(k // 32)]) for r in range(n)])
    Qx = rng.integers(-127, 128, (m, k))
    xq = _q8_1_rows(Qx, np.ones((m, k // 32)), np.zeros((m, k // 32)))
    y, _ = oracle_mod.mul_mat(W, "q8_0", n, k, xq, m)
    assert np.array_equal(y, (Qx @ Qw.T).astype(np.float64))


def test_q4_0_integer_matmul_special_case(oracle_mod):
    """d = 1 and q8_1 d = 1: the fold is the integer matmul of the offset codes q - 8
    with the int8 activations (the q8_1 s plays no part)."""
    rng = np.random.default_rng(25)
    n, k, m = 5, 384, 3
    Qw = rng.integers(0, 16, (n, k))
    W = np.stack([np.concatenate([pack_q4_0(1.0, Qw[r, 32 * b:32 * b + 32]) for b in range(k // 32)]) for r in range(n)])
    Qx = rng.integers(-127, 128, (m, k))
    xq = _q8_1_rows(Qx, np.ones((m, k // 32)), rng.uniform(-3, 3, (m, k // 32)))
    y, T = oracle_mod.mul_mat(W, "q4_0", n, k, xq, m)
    assert np.array_equal(y, (Qx @ (Qw - 8).T).astype(np.float64))
    # T: per 32-block |d_w d8 sumi|
    blk = np.abs(np.einsum("mbi,nbi->mnb", Qx.reshape(m, -1, 32), (Qw - 8).reshape(n, -1, 32)))
    assert np.array_equal(T, blk.sum(axis=2).astype(np.float64))


# ---------------------------------------------------------------- the tolerance sum T
# T is the sum of |block term| over an output's blocks, the scale of the parity bound
# 1e-5 * T.  With power-of-two d, dmin and d8, int codes and fp16 s, every term is exact
# in fp64, so T has a closed form in the integer fields: numpy's einsum of the codes
# gives the per-sub-block dots, and the sums may differ from the oracle's only by the
# order of fp64 additions.


def _pow2(rng, lo, hi, shape):
    return 2.0 ** rng.integers(lo, hi, shape)


def test_q4_K_tolerance_sum_closed_form(oracle_mod):
    """Q4_K: T = sum_b |d sc_b d8_b sumi_b| + |dmin m_b s_b|, the scale and min terms of
    each 32-wide sub-block counted separately, with non-unit d, dmin, d8 and s."""
    rng = np.random.default_rng(27)
    n, k, m = 4, 512, 3
    nsb = k // 256
    D, DM = _pow2(rng, -6, 1, (n, nsb)), _pow2(rng, -6, 1, (n, nsb))
    SC, MN = rng.integers(0, 64, (n, k // 32)), rng.integers(0, 64, (n, k // 32))
    Qw = rng.integers(0, 16, (n, k))
    W = np.stack([np.concatenate([pack_q4_K(D[r, s], DM[r, s], SC[r, 8 * s:8 * s + 8], MN[r, 8 * s:8 * s + 8],
                                            Qw[r, 256 * s:256 * s + 256]) for s in range(nsb)]) for r in range(n)])
    Qx = rng.integers(-127, 128, (m, k))
    D8 = _pow2(rng, -8, -1, (m, k // 32))
    S8 = rng.uniform(-4, 4, (m, k // 32)).astype(np.float16).astype(np.float64)
    xq = _q8_1_rows(Qx, D8, S8)
    y, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    sumi = np.einsum("mbi,nbi->mnb", Qx.reshape(m, -1, 32), Qw.reshape(n, -1, 32))
    t1 = np.repeat(D, 8, axis=1)[None] * SC[None] * D8[:, None, :] * sumi
    t2 = np.repeat(DM, 8, axis=1)[None] * MN[None] * S8[:, None, :]
    np.testing.assert_allclose(T, (np.abs(t1) + np.abs(t2)).sum(axis=2), rtol=1e-15, atol=0)
    assert np.all(np.abs(y - (t1 - t2).sum(axis=2)) <= 1e-14 * T)


def test_q6_K_tolerance_sum_closed_form(oracle_mod):
    """Q6_K: T = sum_j |d sc_j d8_(j/2) sumi_j| over 16-wide sub-blocks j, the q8_1 d
    of the 32-block that holds sub-block j."""
    rng = np.random.default_rng(28)
    n, k, m = 4, 512, 3
    nsb = k // 256
    D = _pow2(rng, -6, 1, (n, nsb))
    SC = rng.integers(-128, 128, (n, k // 16))
    V = rng.integers(-32, 32, (n, k))
    W = np.stack([np.concatenate([pack_q6_K(D[r, s], SC[r, 16 * s:16 * s + 16], V[r, 256 * s:256 * s + 256])
                                  for s in range(nsb)]) for r in range(n)])
    Qx = rng.integers(-127, 128, (m, k))
    D8 = _pow2(rng, -8, -1, (m, k // 32))
    xq = _q8_1_rows(Qx, D8, rng.uniform(-3, 3, (m, k // 32)))
    y, T = oracle_mod.mul_mat(W, "q6_K", n, k, xq, m)
    sumi = np.einsum("mji,nji->mnj", Qx.reshape(m, -1, 16), V.reshape(n, -1, 16))
    t = np.repeat(D, 16, axis=1)[None] * SC[None] * np.repeat(D8, 2, axis=1)[:, None, :] * sumi
    np.testing.assert_allclose(T, np.abs(t).sum(axis=2), rtol=1e-15, atol=0)
    assert np.all(np.abs(y - t.sum(axis=2)) <= 1e-14 * T)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_32_block_tolerance_sum_closed_form(oracle_mod, fmt):
    """Q8_0 and Q4_0: T = sum_b |d_b d8_b sumi_b| over 32-blocks, with non-unit d and d8
    (Q4_0's integers are the offset codes q - 8)."""
    rng = np.random.default_rng(29)
    n, k, m = 5, 320, 3
    D = _pow2(rng, -6, 1, (n, k // 32))
    if fmt == "q8_0":
        Qw = rng.integers(-128, 128, (n, k))
        V = Qw
        W = np.stack([np.concatenate([pack_q8_0(D[r, b], Qw[r, 32 * b:32 * b + 32]) for b in range(k // 32)])
                      for r in range(n)])
    else:
        Qw = rng.integers(0, 16, (n, k))
        V = Qw - 8
        W = np.stack([np.concatenate([pack_q4_0(D[r, b], Qw[r, 32 * b:32 * b + 32]) for b in range(k // 32)])
                      for r in range(n)])
    Qx = rng.integers(-127, 128, (m, k))
    D8 = _pow2(rng, -8, -1, (m, k // 32))
    xq = _q8_1_rows(Qx, D8, rng.uniform(-3, 3, (m, k // 32)))
    y, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
    sumi = np.einsum("mbi,nbi->mnb", Qx.reshape(m, -1, 32), V.reshape(n, -1, 32))
    t = D[None] * D8[:, None, :] * sumi
    np.testing.assert_allclose(T, np.abs(t).sum(axis=2), rtol=1e-15, atol=0)
    assert np.all(np.abs(y - t.sum(axis=2)) <= 1e-14 * T)


def test_q5_K_integer_matmul_special_case(oracle_mod):
    """d = 1, dmin = 0, all sub-block scales 1 and q8_1 d = 1: the fold is the integer
    matmul of the 5-bit codes with the int8 activations."""
    rng = np.random.default_rng(26)
    n, k, m = 5, 512, 3
    Qw = rng.integers(0, 32, (n, k))
    W = np.stack([np.concatenate([pack_q5_K(1.0, 0.0, np.ones(8, int), rng.integers(0, 64, 8),
                                            Qw[r, 256 * s:256 * s + 256]) for s in range(k // 256)]) for r in range(n)])
    Qx = rng.integers(-127, 128, (m, k))
    xq = _q8_1_rows(Qx, np.ones((m, k // 32)), rng.uniform(-3, 3, (m, k // 32)))
    y, T = oracle_mod.mul_mat(W, "q5_K", n, k, xq, m)
    assert np.array_equal(y, (Qx @ Qw.T).astype(np.float64))


def test_q5_K_tolerance_sum_and_min_term(oracle_mod):
    """Q5_K with non-unit power-of-two d, dmin, d8 and fp16 s: y and T in closed form,
    T = sum_b |d sc_b d8_b sumi_b| + |dmin m_b s_b|."""
    rng = np.random.default_rng(29)
    n, k, m = 4, 512, 3
    nsb = k // 256
    D, DM = _pow2(rng, -6, 1, (n, nsb)), _pow2(rng, -6, 1, (n, nsb))
    SC, MN = rng.integers(0, 64, (n, k // 32)), rng.integers(0, 64, (n, k // 32))
    Qw = rng.integers(0, 32, (n, k))
    W = np.stack([np.concatenate([pack_q5_K(D[r, s], DM[r, s], SC[r, 8 * s:8 * s + 8], MN[r, 8 * s:8 * s + 8],
                                            Qw[r, 256 * s:256 * s + 256]) for s in range(nsb)]) for r in range(n)])
    Qx = rng.integers(-127, 128, (m, k))
    D8 = _pow2(rng, -8, -1, (m, k // 32))
    S8 = rng.uniform(-4, 4, (m, k // 32)).astype(np.float16).astype(np.float64)
    xq = _q8_1_rows(Qx, D8, S8)
    y, T = oracle_mod.mul_mat(W, "q5_K", n, k, xq, m)
    sumi = np.einsum("mbi,nbi->mnb", Qx.reshape(m, -1, 32), Qw.reshape(n, -1, 32))
    t1 = np.repeat(D, 8, axis=1)[None] * SC[None] * D8[:, None, :] * sumi
    t2 = np.repeat(DM, 8, axis=1)[None] * MN[None] * S8[:, None, :]
    np.testing.assert_allclose(T, (np.abs(t1) + np.abs(t2)).sum(axis=2), rtol=1e-15, atol=0)
    assert np.all(np.abs(y - (t1 - t2).sum(axis=2)) <= 1e-14 * T)


@pytest.mark.parametrize("fmt", ["q6_K", "q8_0", "q4_0"])
def test_brute_force_agrees(oracle_mod, fmt):
    """Without a min term the fold equals the fp64 matmul of dequantized W and
    dequantized q8_1 x up to fp64 rounding; and the brute force itself equals
    numpy's matmul of the two dequantized matrices."""
    rng = np.random.default_rng(31)
    n, k, m = 9, 512, 5
    W = qmm_synth.gen_weights(fmt, rng, n, k)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, m, k))
    yA, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
    yB = oracle_mod.brute(W, fmt, n, k, xq, m)
    assert np.all(np.abs(yA - yB) <= 1e-12 * T)
    ref = oracle_mod.dequant_q8_1(xq, m, k) @ oracle_mod.dequant(W, fmt, n, k).T
    assert np.allclose(yB, ref, rtol=0, atol=1e-12 * np.abs(T).max())


def test_brute_force_agrees_q4_K_exact_s(oracle_mod):
    """Q4_K: when s = d*sum(q) is exact in fp16 the fold equals the brute force
    to fp64 rounding (power-of-two d and small sums make d*sum(q) exact)."""
    rng = np.random.default_rng(32)
    n, k, m = 7, 512, 4
    W = qmm_synth.gen_q4_K(rng, n, k)
    Qx = rng.integers(-60, 61, (m, k))
    d = 2.0 ** rng.integers(-8, -2, (m, k // 32))
    S = Qx.reshape(m, k // 32, 32).sum(axis=2)
    xq = _q8_1_rows(Qx, d, d * S)
    yA, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    yB = oracle_mod.brute(W, "q4_K", n, k, xq, m)
    assert np.all(np.abs(yA - yB) <= 1e-12 * T)


@pytest.mark.parametrize("fmt", ["q4_K", "q5_K"])
def test_brute_force_q4_K_s_rounding_bound(oracle_mod, fmt):
    """Q4_K and Q5_K with quantized activations: the fold uses the stored fp16 s, the brute
    force d*sum(q); they differ by at most the fp16 rounding of s in the min terms."""
    rng = np.random.default_rng(33)
    n, k, m = 8, 1024, 3
    W = qmm_synth.gen_weights(fmt, rng, n, k)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, m, k))
    yA, T = oracle_mod.mul_mat(W, fmt, n, k, xq, m)
    yB = oracle_mod.brute(W, fmt, n, k, xq, m)
    assert np.all(np.abs(yA - yB) <= 2.0 ** -10 * T)


def test_activation_quantization_error_reported(oracle_mod, capsys):
    """Reported, not a pass criterion: relative RMS of the q8_1 path against the
    fp64 product of dequantized W with the raw fp32 activations."""
    rng = np.random.default_rng(34)
    res = {}
    for fmt in ("q4_K", "q6_K", "q8_0"):
        n, k, m = 64, 2048, 4
        W = qmm_synth.gen_weights(fmt, rng, n, k)
        x = qmm_synth.gen_x(rng, m, k)
        yA, _ = oracle_mod.mul_mat(W, fmt, n, k, oracle_mod.quantize_q8_1(x), m)
        yR = x.astype(np.float64) @ oracle_mod.dequant(W, fmt, n, k).T
        res[fmt] = float(np.sqrt(np.mean((yA - yR) ** 2) / np.mean(yR ** 2)))
    print("activation-quantization rel RMS:", res)
    assert all(v < 0.05 for v in res.values())


def test_mul_mat_at_matches_full(oracle_mod):
    rng = np.random.default_rng(41)
    n, k, m = 33, 512, 3
    W = qmm_synth.gen_q4_K(rng, n, k)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, m, k))
    y, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    rows = rng.integers(0, n, 50)
    cols = rng.integers(0, m, 50)
    y2, T2 = oracle_mod.mul_mat_at(W, "q4_K", n, k, xq, m, rows, cols)
    assert np.array_equal(y2, y[cols, rows]) and np.array_equal(T2, T[cols, rows])


def test_bucket_is_stable_sort(oracle_mod):
    rng = np.random.default_rng(51)
    ids = qmm_synth.gen_moe_ids(rng, 200, 8, 32)
    ids[3, 2] = -1
    ids[7, 0] = 32
    bounds, perm, bad = oracle_mod.bucket(ids, 32)
    assert bad == 2
    flat = ids.ravel()
    valid = np.nonzero((flat >= 0) & (flat < 32))[0]
    order = valid[np.argsort(flat[valid], kind="stable")]
    assert np.array_equal(perm, order)
    assert np.array_equal(np.diff(bounds), np.bincount(flat[valid], minlength=32))


def test_mul_mat_id_reduces_to_dense(oracle_mod):
    rng = np.random.default_rng(52)
    E, n, k, T_, K = 6, 16, 512, 5, 3
    W = qmm_synth.gen_q4_K(rng, E * n, k).reshape(E, n, -1)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, T_, k))
    ids = qmm_synth.gen_moe_ids(rng, T_, K, E)
    ids[1, 1] = 99
    y, T, bad = oracle_mod.mul_mat_id(W, "q4_K", E, n, k, xq, ids)
    assert bad == 1
    for t in range(T_):
        for s in range(K):
            e = ids[t, s]
            if e >= E:
                assert np.all(y[t, s] == 0) and np.all(T[t, s] == 0)
                continue
            yd, Td = oracle_mod.mul_mat(W[e], "q4_K", n, k, xq[t:t + 1], 1)
            assert np.array_equal(y[t, s], yd[0]) and np.array_equal(T[t, s], Td[0])


def test_synthetic_moe_histogram_is_skewed():
    """The MoE workload recipe (seed 0) is as skewed as intended: one hot expert,
    many cold ones, every expert used."""
    _, _, ids = qmm_synth.make_moe(128, 8, 256, 512, 8)
    c = np.bincount(ids.ravel(), minlength=128)
    assert c.sum() == 4096 and c.max() > 300 and np.median(c) < 32 and c.min() >= 1
    assert all(len(set(r)) == 8 for r in ids)


def test_mul_mat_id_per_slot_reduces_to_dense(oracle_mod):
    """One activation row per (token, slot): each output row is the dense routine on that
    pair's own row and expert; with every slot's row equal to its token's row it is the
    shared-row call, to the bit."""
    rng = np.random.default_rng(53)
    E, n, k, T_, K = 5, 24, 512, 4, 3
    W = qmm_synth.gen_q4_K(rng, E * n, k).reshape(E, n, -1)
    xs = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, T_ * K, k))
    ids = qmm_synth.gen_moe_ids(rng, T_, K, E)
    ids[2, 0] = -1
    y, T, bad = oracle_mod.mul_mat_id(W, "q4_K", E, n, k, xs, ids, per_slot=True)
    assert bad == 1
    for t in range(T_):
        for s in range(K):
            e = ids[t, s]
            if e < 0:
                assert np.all(y[t, s] == 0) and np.all(T[t, s] == 0)
                continue
            yd, Td = oracle_mod.mul_mat(W[e], "q4_K", n, k, xs[t * K + s:t * K + s + 1], 1)
            assert np.array_equal(y[t, s], yd[0]) and np.array_equal(T[t, s], Td[0])
    xt = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, T_, k))
    rep = np.repeat(xt, K, axis=0)
    y1, T1, _ = oracle_mod.mul_mat_id(W, "q4_K", E, n, k, rep, ids, per_slot=True)
    y2, T2, _ = oracle_mod.mul_mat_id(W, "q4_K", E, n, k, xt, ids)
    assert np.array_equal(y1, y2) and np.array_equal(T1, T2)


def test_silu_closed_forms(oracle_mod):
    """silu(0) = 0, silu(v) - silu(-v) = v, silu(1) = 1 / (1 + 1/e), and silu(v) -> v for
    large v, -> 0 for very negative v."""
    v = np.linspace(-30, 30, 121)
    s = oracle_mod.silu(v)
    assert oracle_mod.silu(0.0) == 0.0
    np.testing.assert_allclose(s - oracle_mod.silu(-v), v, rtol=0, atol=1e-12)
    assert abs(oracle_mod.silu(1.0) - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15
    assert abs(oracle_mod.silu(40.0) - 40.0) < 1e-12 and abs(oracle_mod.silu(-40.0)) < 1e-15


def test_mul_mat_glu_pins(oracle_mod):
    """The GLU oracle against a hand-built case: gate rows equal to the up rows give
    silu(u) * u; a zero gate row gives exactly 0; the bound is non-negative and shrinks
    to the fp32 term when the gate's dots carry no error bound."""
    rng = np.random.default_rng(61)
    n, k, m = 6, 512, 3
    Wu = qmm_synth.gen_q4_K(rng, n, k)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, m, k))
    u, _ = oracle_mod.mul_mat(Wu, "q4_K", n, k, xq, m)
    y, tol = oracle_mod.mul_mat_glu(Wu, Wu, "q4_K", n, k, xq, m)
    np.testing.assert_allclose(y, u * u / (1.0 + np.exp(-u)), rtol=1e-14, atol=0)
    assert np.all(tol >= 0)
    Wg = Wu.copy()
    Wg.reshape(n, k // 256, 144)[2, :, :4] = 0  # row 2: d = dmin = 0, every term 0
    y2, tol2 = oracle_mod.mul_mat_glu(Wg, Wu, "q4_K", n, k, xq, m)
    assert np.all(y2[:, 2] == 0) and np.all(tol2[:, 2] >= 0)


def test_repack_glu_row_order(oracle_mod):
    """Row 2j of the interleaved tensor is gate row j and row 2j+1 up row j, bytes
    unchanged; its even and odd rows multiply exactly as the gate and up tensors."""
    g = np.arange(3 * 4, dtype=np.uint8).reshape(3, 4)
    u = (100 + np.arange(3 * 4)).astype(np.uint8).reshape(3, 4)
    p = oracle_mod.repack_glu(g, u)
    assert p.tolist() == [g[0].tolist(), u[0].tolist(), g[1].tolist(), u[1].tolist(), g[2].tolist(), u[2].tolist()]
    rng = np.random.default_rng(41)
    n, k, m = 5, 512, 2
    Wg = qmm_synth.gen_weights("q4_K", rng, n, k)
    Wu = qmm_synth.gen_weights("q4_K", rng, n, k)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, m, k))
    y2, _ = oracle_mod.mul_mat(oracle_mod.repack_glu(Wg, Wu), "q4_K", 2 * n, k, xq, m)
    assert np.array_equal(y2[:, 0::2], oracle_mod.mul_mat(Wg, "q4_K", n, k, xq, m)[0])
    assert np.array_equal(y2[:, 1::2], oracle_mod.mul_mat(Wu, "q4_K", n, k, xq, m)[0])


def test_mul_mat_glu_at_matches_full(oracle_mod):
    rng = np.random.default_rng(43)
    n, k, m = 7, 512, 3
    Wg = qmm_synth.gen_weights("q4_K", rng, n, k)
    Wu = qmm_synth.gen_weights("q4_K", rng, n, k)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, m, k))
    y, tol = oracle_mod.mul_mat_glu(Wg, Wu, "q4_K", n, k, xq, m)
    rows = np.array([0, 6, 3, 5])
    cols = np.array([2, 0, 1, 2])
    ya, ta = oracle_mod.mul_mat_glu_at(Wg, Wu, "q4_K", n, k, xq, m, rows, cols)
    assert np.array_equal(ya, y[cols, rows]) and np.array_equal(ta, tol[cols, rows])


@pytest.mark.parametrize("fmt", ["q4_K", "q8_0"])
def test_mul_mat_id_glu_is_the_dense_glu_per_pair(oracle_mod, fmt):
    """The expert-routed SwiGLU is the (pinned) dense SwiGLU of each pair's expert and
    token: y[t][s] and its bound equal mul_mat_glu on W_gate[e], W_up[e] and x[t]; a pair
    with an invalid id has y = 0 and bound 0."""
    E, n, k, T_, K = 5, 9, 512, 4, 3
    rng = np.random.default_rng(47)
    Wg = qmm_synth.gen_weights(fmt, rng, E * n, k).reshape(E, n, -1)
    Wu = qmm_synth.gen_weights(fmt, rng, E * n, k).reshape(E, n, -1)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, T_, k))
    ids = rng.integers(0, E, size=(T_, K)).astype(np.int32)
    ids[1, 2] = E  # invalid
    y, tol, bad = oracle_mod.mul_mat_id_glu(Wg, Wu, fmt, E, n, k, xq, ids)
    assert bad == 1
    rb = xq.reshape(T_, -1)
    for t in range(T_):
        for s_ in range(K):
            e = ids[t, s_]
            if e >= E:
                assert not y[t, s_].any() and not tol[t, s_].any()
                continue
            yd, td = oracle_mod.mul_mat_glu(Wg[e], Wu[e], fmt, n, k, rb[t:t + 1], 1)
            assert np.array_equal(y[t, s_], yd[0]) and np.array_equal(tol[t, s_], td[0])


def test_mul_mat_glu_gate_and_up_roles(oracle_mod):
    """Gate rows equal to the up rows with d and dmin doubled (exact in fp16) make every
    gate dot exactly twice the up dot, so y = silu(2u) * u: a reference that swapped the
    two roles (silu(u) * 2u) or ignored the up dot (silu(2u) * 2u) fails; an all-zero up
    row gives exactly 0 whatever the gate."""
    rng = np.random.default_rng(62)
    n, k, m = 5, 512, 3
    Wu = qmm_synth.gen_q4_K(rng, n, k)
    blk = Wu.reshape(n, k // 256, 144)
    blk[:, :, 0:4] = np.minimum(blk[:, :, 0:4], 0x20)  # keep d, dmin small: doubling stays exact
    Wg = Wu.copy()
    hv = Wg.reshape(n, k // 256, 144)[:, :, 0:4].copy().view(np.float16)
    Wg.reshape(n, k // 256, 144)[:, :, 0:4] = (hv * np.float16(2)).view(np.uint8)
    xq = oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, m, k))
    u, _ = oracle_mod.mul_mat(Wu, "q4_K", n, k, xq, m)
    g, _ = oracle_mod.mul_mat(Wg, "q4_K", n, k, xq, m)
    np.testing.assert_allclose(g, 2 * u, rtol=1e-15, atol=0)
    y, _ = oracle_mod.mul_mat_glu(Wg, Wu, "q4_K", n, k, xq, m)
    np.testing.assert_allclose(y, 2 * u / (1.0 + np.exp(-2 * u)) * u, rtol=1e-14, atol=0)
    Wz = Wu.copy()
    Wz.reshape(n, k // 256, 144)[3, :, 0:4] = 0  # up row 3: d = dmin = 0
    y3, _ = oracle_mod.mul_mat_glu(Wg, Wz, "q4_K", n, k, xq, m)
    assert np.all(y3[:, 3] == 0)


def test_mul_mat_glu_tolerance_closed_forms(oracle_mod):
    """The SwiGLU bound at gate dots where fp64 gives silu and its slope exactly.  Q8_0
    rows with d = 1 and q8_1 d = 1 make every dot an integer (numpy's int matmul), and:
      - row 0 holds a gate dot of exactly 0 from two blocks that cancel (T_g > 0):
        silu(0) = 0 and silu'(0) = 1/2, so y = 0 and tol = 1e-5 T_g |u| / 2 + 2^-120 |u|;
      - row 1 a gate dot of 40 or more, where e^-g < 2^-57 leaves the fp64 sigmoid at
        exactly 1: silu(g) = g and silu'(g) = 1, so y = g u and
        tol = 1e-5 (T_g |u| + g T_u) + 2^-20 |g u| + 2^-120 |u|;
      - row 2 a gate dot of -746 or less, where e^-g overflows and the sigmoid is exactly
        0: y = 0 and tol = 2^-120 |u|."""
    rng = np.random.default_rng(63)
    n, k, m = 3, 64, 2
    Qx = rng.integers(-127, 128, (m, 32))
    Qx[:, 0] = 127                       # no all-zero row
    Qx = np.concatenate([Qx, Qx], axis=1)  # blocks 0 and 1 of x are equal
    a = rng.integers(-128, 128, 32)
    sx = np.sign(Qx[0, :32])
    Qg = np.stack([np.concatenate([a, -a]),
                   np.concatenate([sx * 100, sx * 100]),
                   np.concatenate([-sx * 127, -sx * 127])])
    Qu = rng.integers(-128, 128, (n, k))

    def rows(Q):
        return np.stack([np.concatenate([pack_q8_0(1.0, Q[r, 32 * b:32 * b + 32]) for b in range(k // 32)])
                         for r in range(n)])
    xq = _q8_1_rows(Qx, np.ones((m, 2)), np.zeros((m, 2)))
    with np.errstate(over="ignore"):
        y, tol = oracle_mod.mul_mat_glu(rows(Qg), rows(Qu), "q8_0", n, k, xq, m)
    g = (Qx @ Qg.T).astype(np.float64)
    u = (Qx @ Qu.T).astype(np.float64)
    Tg = np.abs(np.einsum("mbi,nbi->mnb", Qx.reshape(m, 2, 32), Qg.reshape(n, 2, 32))).sum(axis=2)
    Tu = np.abs(np.einsum("mbi,nbi->mnb", Qx.reshape(m, 2, 32), Qu.reshape(n, 2, 32))).sum(axis=2)
    assert np.all(g[:, 0] == 0) and np.all(Tg[:, 0] > 0)
    assert g[0, 1] >= 40 and g[0, 2] <= -746
    eps = 2.0 ** -120
    # row 0: silu(0) = 0, slope 1/2
    assert np.all(y[:, 0] == 0)
    np.testing.assert_allclose(tol[:, 0], 1e-5 * Tg[:, 0] * np.abs(u[:, 0]) / 2 + eps * np.abs(u[:, 0]), rtol=1e-14)
    # row 1 (x row 0, whose signs built it): silu(g) = g, slope 1
    assert y[0, 1] == g[0, 1] * u[0, 1]
    np.testing.assert_allclose(tol[0, 1], 1e-5 * (Tg[0, 1] * abs(u[0, 1]) + g[0, 1] * Tu[0, 1])
                               + 2.0 ** -20 * abs(g[0, 1] * u[0, 1]) + eps * abs(u[0, 1]), rtol=1e-14)
    # row 2: the sigmoid is 0
    assert y[0, 2] == 0
    np.testing.assert_allclose(tol[0, 2], eps * abs(u[0, 2]), rtol=1e-14)
