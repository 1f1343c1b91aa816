"""Hand-built blocks for tests: pack integer fields into the block byte layouts.

These packers are the tests' own statement of each layout (the same readings the
oracle and the kernels take), used to build inputs whose results have closed
forms.  They hold no matmul arithmetic.

* Q4_K: {fp16 d, fp16 dmin, 12 B scales/mins, 128 B nibbles}.  Sub-blocks 0..3
  keep their 6-bit scale in the low 6 bits of bytes 0..3 and their 6-bit min in
  the low 6 bits of bytes 4..7.  Sub-blocks 4..7 keep the low 4 bits of the scale
  in the low nibble of bytes 8..11, the low 4 bits of the min in the high nibble
  of bytes 8..11, and the top 2 bits of scale / min in the top 2 bits of bytes
  0..3 / 4..7.  Nibbles: weight 64c + l is the low nibble of qs byte 32c + l and
  weight 64c + 32 + l its high nibble (c = 0..3, l = 0..31).
* Q5_K: {fp16 d, fp16 dmin, 12 B scales/mins, qh[32], qs[128]}: Q4_K's scale rule and
  nibble order for the low 4 bits; the fifth bit of weight 32j + l is bit j of qh[l].
* Q6_K: {ql[128], qh[64], int8 sc[16], fp16 d}.  Weight 128h + 32t + l (h = 0..1,
  t = 0..3, l = 0..31) takes its low 4 bits from ql[64h + 32(t&1) + l] (low nibble
  for t < 2, high nibble for t >= 2) and its high 2 bits from bits 2t..2t+1 of
  qh[32h + l]; the stored code is value + 32.
* Q8_0: {fp16 d, int8 q[32]}.   q8_1: {fp16 d, fp16 s, int8 q[32]}.
* Q4_0: {fp16 d, 16 B nibbles}: weight i (i < 16) is the low nibble of byte i and
  weight 16 + i its high nibble; the stored code is value + 8.
"""
from __future__ import annotations

import numpy as np


def f16_bytes(v) -> np.ndarray:
    return np.array([v], dtype=np.float16).view(np.uint8)


def pack_q4_K(d: float, dmin: float, sc: np.ndarray, mn: np.ndarray, q: np.ndarray) -> np.ndarray:
    sc = np.asarray(sc, dtype=np.int64)
    mn = np.asarray(mn, dtype=np.int64)
    q = np.asarray(q, dtype=np.int64)
    assert sc.shape == (8,) and mn.shape == (8,) and q.shape == (256,)
    assert sc.min() >= 0 and sc.max() < 64 and mn.min() >= 0 and mn.max() < 64
    assert q.min() >= 0 and q.max() < 16
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = f16_bytes(d)
    b[2:4] = f16_bytes(dmin)
    s = np.zeros(12, dtype=np.int64)
    for j in range(4):
        s[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = mn[j] | ((mn[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    b[4:16] = s.astype(np.uint8)
    qs = np.zeros(128, dtype=np.int64)
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    b[16:] = qs.astype(np.uint8)
    return b


def pack_q5_K(d: float, dmin: float, sc: np.ndarray, mn: np.ndarray, q: np.ndarray) -> np.ndarray:
    """q: 256 codes in 0..31.  Q4_K's layout for the low 4 bits (and the scales), with the
    fifth bit of weight 32j + l in bit j of qh[l]: {d, dmin, 12 B scales, qh[32], qs[128]}."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() < 32
    b4 = pack_q4_K(d, dmin, sc, mn, q & 15)
    qh = np.zeros(32, dtype=np.int64)
    for i in range(256):
        qh[i % 32] |= (q[i] >> 4) << (i // 32)
    b = np.zeros(176, dtype=np.uint8)
    b[0:16] = b4[0:16]
    b[16:48] = qh.astype(np.uint8)
    b[48:] = b4[16:]
    return b


def pack_q6_K(d: float, sc: np.ndarray, v: np.ndarray) -> np.ndarray:
    """v: 256 values in -32..31; sc: 16 int8 scales."""
    sc = np.asarray(sc, dtype=np.int64)
    code = np.asarray(v, dtype=np.int64) + 32
    assert code.min() >= 0 and code.max() < 64 and sc.shape == (16,)
    ql = np.zeros(128, dtype=np.int64)
    qh = np.zeros(64, dtype=np.int64)
    for h in range(2):
        for t in range(4):
            for l in range(32):
                c = code[128 * h + 32 * t + l]
                ql[64 * h + 32 * (t & 1) + l] |= (c & 15) << (4 * (t >> 1))
                qh[32 * h + l] |= (c >> 4) << (2 * t)
    b = np.zeros(210, dtype=np.uint8)
    b[0:128] = ql.astype(np.uint8)
    b[128:192] = qh.astype(np.uint8)
    b[192:208] = sc.astype(np.int8).view(np.uint8)
    b[208:210] = f16_bytes(d)
    return b


def pack_q8_0(d: float, q: np.ndarray) -> np.ndarray:
    b = np.zeros(34, dtype=np.uint8)
    b[0:2] = f16_bytes(d)
    b[2:] = np.asarray(q, dtype=np.int8).view(np.uint8)
    return b


def pack_q4_0(d: float, q: np.ndarray) -> np.ndarray:
    """q: 32 codes in 0..15 (value + 8)."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,) and q.min() >= 0 and q.max() < 16
    b = np.zeros(18, dtype=np.uint8)
    b[0:2] = f16_bytes(d)
    b[2:] = (q[:16] | (q[16:] << 4)).astype(np.uint8)
    return b


def pack_q8_1(d: float, s: float, q: np.ndarray) -> np.ndarray:
    b = np.zeros(36, dtype=np.uint8)
    b[0:2] = f16_bytes(d)
    b[2:4] = f16_bytes(s)
    b[4:] = np.asarray(q, dtype=np.int8).view(np.uint8)
    return b


def unpack_q8_1(xq: np.ndarray, m: int, k: int):
    """(d fp32 [m][k/32], s fp32 [m][k/32], q int8 [m][k]) read from q8_1 bytes."""
    b = np.ascontiguousarray(xq).reshape(m, k // 32, 36)
    d = b[:, :, 0:2].copy().view(np.float16).reshape(m, k // 32).astype(np.float32)
    s = b[:, :, 2:4].copy().view(np.float16).reshape(m, k // 32).astype(np.float32)
    q = b[:, :, 4:].copy().view(np.int8).reshape(m, k)
    return d, s, q
