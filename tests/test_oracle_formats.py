"""Pins for the oracle's formats: byte sizes the pages print, fp16 conversion
against numpy, the q8_1 quantizer's invariants, and hand-built blocks with
closed-form decodes."""
import json
import os

import numpy as np
import pytest

import qmm_synth
from blockpack import pack_q4_0, pack_q4_K, pack_q5_K, pack_q6_K, pack_q8_0, pack_q8_1, unpack_q8_1

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- sizes

def test_block_sizes_match_pages(oracle_mod):
    g = golden("page_facts.json")
    assert oracle_mod.block_bytes("q4_K") == g["q4_K_bytes_per_256"]["value"]
    assert oracle_mod.block_elems("q4_K") * 2 == g["q4_K_bytes_per_256"]["fp16_bytes_per_256"]
    assert 8 * oracle_mod.block_bytes("q4_K") == g["q4_K_x8_bytes"]["value"]
    mb = g["matrix_8192x4096_MB"]
    n, k = 8192, 4096
    q80 = n * (k // oracle_mod.block_elems("q8_0")) * oracle_mod.block_bytes("q8_0")
    assert round(q80 / 1e6, 1) == mb["q8_0"]
    assert round(n * k * 4 / 1e6) == mb["f32"] and round(n * k * 2 / 1e6) == mb["f16"]
    # q8_1: 128 values = 32 ints of int8 + 4 ints of (d, s) -> 36 bytes per 32 values.
    t = g["q8_1_ints_per_128_values"]
    assert (t["qs_ints"] + t["scale_ints"]) * 4 // 4 == t["value"]
    x = np.zeros((1, 128), np.float32)
    assert oracle_mod.quantize_q8_1(x).nbytes == t["value"] * 4
    # Q6_K: 128 B ql + 64 B qh + 16 B scales + 2 B d (by construction of the reading).
    assert oracle_mod.block_bytes("q6_K") == 210
    q40 = n * (k // oracle_mod.block_elems("q4_0")) * oracle_mod.block_bytes("q4_0")
    assert round(q40 / 1e6, 1) == mb["q4_0"]
    assert oracle_mod.block_elems("q4_0") == 32
    for fmt in ("q4_K", "q5_K", "q6_K", "q8_0", "q4_0"):
        assert qmm_synth.BLOCK_BYTES[fmt] == oracle_mod.block_bytes(fmt)
    # Q5_K: Q4_K's 144 bytes plus a 32-byte plane of fifth bits (one per weight)
    assert oracle_mod.block_bytes("q5_K") == oracle_mod.block_bytes("q4_K") + 256 // 8


# ---------------------------------------------------------------- fp16

def test_half_decode_all_patterns(oracle_mod):
    pats = np.arange(65536, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(p)) for p in pats])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_float_to_half_matches_numpy_rne(oracle_mod):
    rng = np.random.default_rng(1)
    vals = [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, 2.0 ** -24, 2.0 ** -25,
            2.0 ** -25 * 1.0000001, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -11), 1e-8, 6.1e-5]
    # exact midpoints between consecutive fp16 values (ties -> even), normal and subnormal
    h = np.arange(0, 0x7bff, 37, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    vals += list(((lo + hi) / 2).astype(np.float32))
    vals += list(rng.standard_normal(2000).astype(np.float32) * 10.0 ** rng.integers(-9, 5, 2000))
    vals = np.array(vals, dtype=np.float32)
    with np.errstate(over="ignore"):  # 65520 and above round to infinity, as intended
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref), np.nonzero(got != ref)


# ---------------------------------------------------------------- q8_1 quantizer

def _adversarial_rows():
    """Blocks of 32 that stress the quantizer: zeros, signed zeros, ties, extremes."""
    rows = []
    z = np.zeros(32, np.float32)
    rows.append(z.copy())
    nz = z.copy(); nz[:] = -0.0; rows.append(nz)
    one = z.copy(); one[7] = 3.5; rows.append(one)
    neg = z.copy(); neg[31] = -2.0; neg[0] = 1.0; rows.append(neg)
    # x/d lands exactly on .5: amax=127 -> d=1, x = k + 0.5
    tie = np.arange(32, dtype=np.float32) - 15.5; tie[0] = 127.0; rows.append(tie)
    tie2 = -tie; rows.append(tie2)
    big = np.linspace(-60000, 60000, 32).astype(np.float32); rows.append(big)
    tiny = (np.arange(32, dtype=np.float32) - 16) * np.float32(1e-40); rows.append(tiny)  # denormals
    tiny2 = np.full(32, np.float32(1.4e-45)); tiny2[3] = -np.float32(2.8e-45); rows.append(tiny2)
    same = np.full(32, np.float32(0.3)); rows.append(same)
    for pos in (0, 13, 31):
        r = np.random.default_rng(pos).standard_normal(32).astype(np.float32)
        r[pos] = 9.0
        rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("kind", ["normal", "adversarial"])
def test_q8_1_invariants(oracle_mod, kind):
    if kind == "normal":
        x = np.random.default_rng(3).standard_normal((7, 32 * 40)).astype(np.float32)
    else:
        x = _adversarial_rows()
    m, k = x.shape
    xq = oracle_mod.quantize_q8_1(x)
    d, s, q = unpack_q8_1(xq, m, k)
    q = q.astype(np.int64)
    xb = x.reshape(m, k // 32, 32).astype(np.float64)
    qb = q.reshape(m, k // 32, 32)
    amax = np.abs(xb).max(axis=2)
    S = qb.sum(axis=2)
    # |q| <= 127; some |q| == 127 whenever the fp32 scale amax/127 is not zero
    # (a block of a few minimum denormals has amax > 0 but amax/127 == 0 in fp32;
    # such a block is stored as all zero)
    assert np.abs(qb).max() <= 127
    nzb = (amax.astype(np.float32) / np.float32(127.0)) > 0
    assert np.all(np.abs(qb).max(axis=2)[nzb] == 127)
    assert np.all(qb[~nzb] == 0) and np.all(d[~nzb] == 0) and np.all(s[~nzb] == 0)
    # stored d is amax/127 to within fp16 rounding (half an fp16 ulp, plus the fp32 step)
    dd = amax / 127.0
    rel = np.abs(d.astype(np.float64) - dd) / np.where(dd > 0, dd, 1)
    normal = dd >= 2.0 ** -14
    assert np.all(rel[normal] <= 2.0 ** -11 + 2.0 ** -23)
    # s = d * sum(q) from the stored fields, rounded once to fp16 (the page's invariant)
    exact = d.astype(np.float64) * S
    assert np.all(np.abs(s.astype(np.float64) - exact) <= np.abs(exact) * 2.0 ** -11 + 2.0 ** -25)
    # q is the integer nearest to x/d (using the fp32 d the block was quantized with),
    # with halves rounded away from zero.
    d32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d32[..., None] > 0, xb / d32[..., None], 0.0)
    err = np.abs(r - qb)
    assert np.all(err <= 0.5 + 1e-6 * np.maximum(1, np.abs(r)))
    ties = np.abs(np.abs(r - np.trunc(r)) - 0.5) < 1e-9
    if ties.any():
        assert np.all(np.abs(qb[ties]) == np.ceil(np.abs(r[ties])))


def test_q8_1_fp32_division_path(oracle_mod):
    """The quantizer follows the fp32 definition bit for bit: fp32 amax/127,
    fp32 x/d, round half away from zero (checked with numpy's IEEE fp32 ops)."""
    x = np.concatenate([np.random.default_rng(5).standard_normal((5, 256)).astype(np.float32),
                        np.random.default_rng(6).uniform(-3, 3, (3, 256)).astype(np.float32)])
    m, k = x.shape
    d, s, q = unpack_q8_1(oracle_mod.quantize_q8_1(x), m, k)
    xb = x.reshape(m, k // 32, 32)
    d32 = np.abs(xb).max(axis=2) / np.float32(127.0)
    v = (xb / d32[..., None]).astype(np.float64)
    qq = (np.sign(v) * np.floor(np.abs(v) + 0.5)).astype(np.int64)
    assert np.array_equal(qq.reshape(m, k), q.astype(np.int64))
    assert np.array_equal(d32.astype(np.float16).astype(np.float32), d)


# ---------------------------------------------------------------- weight decode

def test_q4_K_scale_packing_roundtrip(oracle_mod):
    rng = np.random.default_rng(11)
    cases = [np.zeros(8, int), np.full(8, 63), np.arange(8) * 9]
    cases += [rng.integers(0, 64, 8) for _ in range(50)]
    for sc in cases:
        mn = rng.integers(0, 64, 8)
        q = rng.integers(0, 16, 256)
        blk = pack_q4_K(0.5, 0.25, sc, mn, q)
        d, dmin, sc2, mn2, q2 = oracle_mod.q4_K_fields(blk)
        assert d == 0.5 and dmin == 0.25
        assert np.array_equal(sc2, sc) and np.array_equal(mn2, mn) and np.array_equal(q2, q)


@pytest.mark.parametrize("j", range(8))
def test_q4_K_single_subblock_closed_form(oracle_mod, j):
    """Only sub-block j has a scale (and a min): every other decoded weight is 0,
    and sub-block j decodes to d*sc*q - dmin*m."""
    sc = np.zeros(8, int); sc[j] = 37
    mn = np.zeros(8, int); mn[j] = 5
    q = (np.arange(256) * 7 + 3) % 16
    blk = pack_q4_K(0.125, 0.5, sc, mn, q)
    w = oracle_mod.dequant(blk, "q4_K", 1, 256)[0]
    expect = np.zeros(256)
    expect[32 * j:32 * j + 32] = 0.125 * 37 * q[32 * j:32 * j + 32] - 0.5 * 5
    assert np.array_equal(w, expect)


def test_q4_K_nibble_positions(oracle_mod):
    """Raw bytes, no packer: qs byte 32c+l low nibble is weight 64c+l, high nibble 64c+32+l."""
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([1.0], np.float16).view(np.uint8)
    blk[4:8] = 1                       # sc[0..3] = 1, mins 0
    blk[12:16] = 1                     # low nibble of bytes 8..11 -> sc[4..7] = 1
    c, l = 2, 9
    blk[16 + 32 * c + l] = 0xA3        # low nibble 3, high nibble 10
    w = oracle_mod.dequant(blk, "q4_K", 1, 256)[0]
    nz = np.nonzero(w)[0]
    assert list(nz) == [64 * c + l, 64 * c + 32 + l]
    assert w[64 * c + l] == 3 and w[64 * c + 32 + l] == 10


def test_q6_K_fields_roundtrip(oracle_mod):
    rng = np.random.default_rng(12)
    for _ in range(20):
        v = rng.integers(-32, 32, 256)
        sc = rng.integers(-128, 128, 16)
        blk = pack_q6_K(0.25, sc, v)
        d, sc2, v2 = oracle_mod.q6_K_fields(blk)
        assert d == 0.25 and np.array_equal(sc2, sc) and np.array_equal(v2, v)
        w = oracle_mod.dequant(blk, "q6_K", 1, 256)[0]
        assert np.array_equal(w, 0.25 * np.repeat(sc, 16) * v)


def test_q6_K_raw_bit_positions(oracle_mod):
    """Raw bytes, no packer: weight 128h+32t+l takes ql[64h+32(t&1)+l] nibble t>>1 and qh[32h+l] bits 2t..2t+1."""
    for (h, t, l) in [(0, 0, 0), (0, 3, 31), (1, 1, 5), (1, 2, 17)]:
        blk = np.zeros(210, np.uint8)
        blk[0:128] = 0x00
        blk[128:192] = 0xAA             # every 2-bit field = 2 -> codes 32 -> value 0 everywhere
        blk[192:208] = 1
        blk[208:210] = np.array([1.0], np.float16).view(np.uint8)
        i = 128 * h + 32 * t + l
        blk[64 * h + 32 * (t & 1) + l] |= 0x5 << (4 * (t >> 1))   # low bits 5 -> code 37 -> value 5
        w = oracle_mod.dequant(blk, "q6_K", 1, 256)[0]
        assert list(np.nonzero(w)[0]) == [i] and w[i] == 5


def test_q8_0_decode(oracle_mod):
    q = np.arange(-16, 16)
    w = oracle_mod.dequant(pack_q8_0(0.5, q), "q8_0", 1, 32)[0]
    assert np.array_equal(w, 0.5 * q)


def test_q4_0_nibble_positions_and_offset(oracle_mod):
    """Byte i's low nibble is weight i and its high nibble weight 16 + i; the value is
    d * (code - 8), so code 8 everywhere decodes to exact zeros."""
    w = oracle_mod.dequant(pack_q4_0(0.25, np.full(32, 8)), "q4_0", 1, 32)[0]
    assert np.array_equal(w, np.zeros(32))
    for i in range(32):
        q = np.full(32, 8)
        q[i] = 15
        w = oracle_mod.dequant(pack_q4_0(0.25, q), "q4_0", 1, 32)[0]
        assert list(np.nonzero(w)[0]) == [i] and w[i] == 0.25 * 7
    # raw bytes: byte 3 = 0x1f puts code 15 at weight 3 and code 1 at weight 19
    blk = pack_q4_0(1.0, np.full(32, 8))
    blk[2 + 3] = 0x1F
    w = oracle_mod.dequant(blk, "q4_0", 1, 32)[0]
    assert w[3] == 7 and w[19] == -7 and np.count_nonzero(w) == 2


def test_q4_0_decode_all_codes(oracle_mod):
    q = np.concatenate([np.arange(16), np.arange(15, -1, -1)])
    w = oracle_mod.dequant(pack_q4_0(-0.5, q), "q4_0", 1, 32)[0]
    assert np.array_equal(w, -0.5 * (q - 8))


# ---------------------------------------------------------------- padded rows

@pytest.mark.parametrize("fmt,k", [("q6_K", 5120), ("q6_K", 1280), ("q8_0", 5120), ("q8_0", 96), ("q4_0", 224),
                                   ("q4_K", 4096)])
def test_repack_aligned_round_trip(oracle_mod, fmt, k):
    """The padded rows hold the original blocks byte for byte, then zeros; the stride is a
    whole number of 16-byte units, and for Q6_K every superblock's 224-byte copy window
    (from the 16-byte boundary at or below the superblock) ends inside its own row."""
    rng = np.random.default_rng(k)
    n = 7
    W = qmm_synth.gen_weights(fmt, rng, n, k)
    rb = (k // oracle_mod.block_elems(fmt)) * oracle_mod.block_bytes(fmt)
    stride = oracle_mod.aligned_row_bytes(fmt, k)
    A = oracle_mod.repack_aligned(W, fmt, n, k)
    assert A.shape == (n, stride) and stride % 16 == 0 and rb <= stride < rb + 16 + (14 if fmt == "q6_K" else 0)
    assert np.array_equal(A[:, :rb], W.reshape(n, rb)) and not A[:, rb:].any()
    if fmt == "q6_K":
        for sb in range(k // 256):
            assert (210 * sb) // 16 * 16 + 224 <= stride
    yA, TA = oracle_mod.mul_mat(A[:, :rb].copy(), fmt, n, k, oracle_mod.quantize_q8_1(qmm_synth.gen_x(rng, 2, k)), 2)
    assert np.all(np.isfinite(yA))


# ---------------------------------------------------------------- Q5_K

def test_q5_K_raw_bit_positions(oracle_mod):
    """Raw bytes, no packer: with every scale 1 and d = 1, qs byte 32c + l gives weights
    64c + l (low nibble) and 64c + 32 + l (high nibble), and bit j of qh[l] adds 16 to
    weight 32j + l and to no other."""
    blk = np.zeros(176, np.uint8)
    blk[0:2] = np.array([1.0], np.float16).view(np.uint8)
    blk[4:8] = 1                       # sc[0..3] = 1, mins 0
    blk[12:16] = 1                     # sc[4..7] = 1
    c, l = 1, 5
    blk[48 + 32 * c + l] = 0x72        # low nibble 2, high nibble 7
    j, l2 = 6, 20
    blk[16 + l2] = 1 << j              # fifth bit of weight 32j + l2
    w = oracle_mod.dequant(blk, "q5_K", 1, 256)[0]
    nz = sorted(np.nonzero(w)[0])
    assert nz == sorted([64 * c + l, 64 * c + 32 + l, 32 * j + l2])
    assert w[64 * c + l] == 2 and w[64 * c + 32 + l] == 7 and w[32 * j + l2] == 16


def test_q5_K_fields_roundtrip(oracle_mod):
    rng = np.random.default_rng(15)
    for _ in range(20):
        q = rng.integers(0, 32, 256)
        sc, mn = rng.integers(0, 64, 8), rng.integers(0, 64, 8)
        blk = pack_q5_K(0.5, 0.25, sc, mn, q)
        d, dmin, sc2, mn2, q2 = oracle_mod.q5_K_fields(blk)
        assert (d, dmin) == (0.5, 0.25) and np.array_equal(sc2, sc) and np.array_equal(mn2, mn)
        assert np.array_equal(q2, q)
        w = oracle_mod.dequant(blk, "q5_K", 1, 256)[0]
        assert np.array_equal(w, 0.5 * np.repeat(sc, 32) * q - 0.25 * np.repeat(mn, 32))
