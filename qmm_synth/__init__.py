"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle runs.

This module holds none of the method's arithmetic: it draws random bytes and
random block fields and lays them out at the byte offsets of each block format,
so that the CUDA path and the CPU oracle consume identical bytes.

Block byte layouts (what each generator fills):

* Q4_K, 144 bytes per 256 weights: fp16 ``d`` at 0, fp16 ``dmin`` at 2, 12 bytes
  of packed 6-bit sub-block scales/mins at 4, 128 bytes of nibbles at 16.
  Any 12-byte pattern is a valid packing of sixteen 6-bit fields and any byte is
  two nibbles, so uniform random bytes give scales/mins uniform on 0..63 and
  nibbles uniform on 0..15 without any packing code here.
* Q6_K, 210 bytes per 256 weights: ``ql[128]`` at 0, ``qh[64]`` at 128, sixteen
  int8 sub-block scales at 192, fp16 ``d`` at 208.  Uniform ql/qh bytes give
  uniform 6-bit codes.
* Q8_0, 34 bytes per 32 weights: fp16 ``d`` at 0, 32 int8 at 2.
* Q4_0, 18 bytes per 32 weights: fp16 ``d`` at 0, 16 bytes of nibbles at 2.  Uniform
  bytes give nibble codes uniform on 0..15.

Workload shapes and value ranges follow the pages' workloads: Q4_K with
d, dmin uniform on [1e-4, 1e-3]; Q6_K with int8 sub-scales uniform on -64..63 and
d uniform on [1e-5, 1e-4]; Q8_0 with int8 uniform and d uniform on [1e-3, 1e-2];
Q4_0 (the pages time it at 8192 x 4096 without giving a value distribution) with
nibbles uniform and d uniform on [1e-3, 1e-2];
activations N(0, 1) in fp32; MoE routing top-8 of 128 experts drawn without
replacement with Zipf(1.1) weights.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
QK8_0 = 32
QK8_1 = 32
BLOCK_BYTES = {"q4_K": 144, "q5_K": 176, "q6_K": 210, "q8_0": 34, "q4_0": 18}
BLOCK_ELEMS = {"q4_K": QK_K, "q5_K": QK_K, "q6_K": QK_K, "q8_0": QK8_0, "q4_0": QK8_0}
Q8_1_BLOCK_BYTES = 36


def streams(seed: int = 0, n: int = 3):
    """Independent child generators (W, x, ids, ...) from one seed."""
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def row_bytes(fmt: str, k: int) -> int:
    qk = BLOCK_ELEMS[fmt]
    if k % qk:
        raise ValueError(f"k={k} is not a multiple of the {fmt} block size {qk}")
    return (k // qk) * BLOCK_BYTES[fmt]


def _fp16_uniform(rng, size, lo, hi):
    return rng.uniform(lo, hi, size=size).astype(np.float32).astype(np.float16)


def gen_q4_K(rng, n: int, k: int, d_range=(1e-4, 1e-3), dmin_range=(1e-4, 1e-3)) -> np.ndarray:
    """Random Q4_K matrix [n][k/256 blocks] as uint8 of shape (n, k/256*144)."""
    nb = k // QK_K
    if k % QK_K:
        raise ValueError("k must be a multiple of 256 for Q4_K")
    blk = np.empty((n, nb, 144), dtype=np.uint8)
    blk[:, :, 4:] = rng.integers(0, 256, size=(n, nb, 140), dtype=np.uint8)
    blk[:, :, 0:2] = _fp16_uniform(rng, (n, nb), *d_range).view(np.uint8).reshape(n, nb, 2)
    blk[:, :, 2:4] = _fp16_uniform(rng, (n, nb), *dmin_range).view(np.uint8).reshape(n, nb, 2)
    return blk.reshape(n, nb * 144)


def gen_q5_K(rng, n: int, k: int, d_range=(1e-4, 1e-3), dmin_range=(1e-4, 1e-3)) -> np.ndarray:
    """Random Q5_K matrix as uint8 of shape (n, k/256*176): the Q4_K recipe (d, dmin fp16
    uniform, every 12-byte scale pattern, uniform nibbles) with a uniform fifth-bit plane."""
    nb = k // QK_K
    if k % QK_K:
        raise ValueError("k must be a multiple of 256 for Q5_K")
    blk = np.empty((n, nb, 176), dtype=np.uint8)
    blk[:, :, 4:] = rng.integers(0, 256, size=(n, nb, 172), dtype=np.uint8)
    blk[:, :, 0:2] = _fp16_uniform(rng, (n, nb), *d_range).view(np.uint8).reshape(n, nb, 2)
    blk[:, :, 2:4] = _fp16_uniform(rng, (n, nb), *dmin_range).view(np.uint8).reshape(n, nb, 2)
    return blk.reshape(n, nb * 176)


def gen_q6_K(rng, n: int, k: int, d_range=(1e-5, 1e-4), sc_range=(-64, 63)) -> np.ndarray:
    """Random Q6_K matrix as uint8 of shape (n, k/256*210)."""
    nb = k // QK_K
    if k % QK_K:
        raise ValueError("k must be a multiple of 256 for Q6_K")
    blk = np.empty((n, nb, 210), dtype=np.uint8)
    blk[:, :, 0:192] = rng.integers(0, 256, size=(n, nb, 192), dtype=np.uint8)
    blk[:, :, 192:208] = rng.integers(sc_range[0], sc_range[1] + 1, size=(n, nb, 16)).astype(np.int8).view(np.uint8)
    blk[:, :, 208:210] = _fp16_uniform(rng, (n, nb), *d_range).view(np.uint8).reshape(n, nb, 2)
    return blk.reshape(n, nb * 210)


def gen_q8_0(rng, n: int, k: int, d_range=(1e-3, 1e-2)) -> np.ndarray:
    """Random Q8_0 matrix as uint8 of shape (n, k/32*34); int8 values uniform on -128..127."""
    nb = k // QK8_0
    if k % QK8_0:
        raise ValueError("k must be a multiple of 32 for Q8_0")
    blk = np.empty((n, nb, 34), dtype=np.uint8)
    blk[:, :, 2:] = rng.integers(0, 256, size=(n, nb, 32), dtype=np.uint8)
    blk[:, :, 0:2] = _fp16_uniform(rng, (n, nb), *d_range).view(np.uint8).reshape(n, nb, 2)
    return blk.reshape(n, nb * 34)


def gen_q4_0(rng, n: int, k: int, d_range=(1e-3, 1e-2)) -> np.ndarray:
    """Random Q4_0 matrix as uint8 of shape (n, k/32*18); nibble codes uniform on 0..15."""
    nb = k // QK8_0
    if k % QK8_0:
        raise ValueError("k must be a multiple of 32 for Q4_0")
    blk = np.empty((n, nb, 18), dtype=np.uint8)
    blk[:, :, 2:] = rng.integers(0, 256, size=(n, nb, 16), dtype=np.uint8)
    blk[:, :, 0:2] = _fp16_uniform(rng, (n, nb), *d_range).view(np.uint8).reshape(n, nb, 2)
    return blk.reshape(n, nb * 18)


GEN = {"q4_K": gen_q4_K, "q5_K": gen_q5_K, "q6_K": gen_q6_K, "q8_0": gen_q8_0, "q4_0": gen_q4_0}


def gen_weights(fmt: str, rng, n: int, k: int) -> np.ndarray:
    return GEN[fmt](rng, n, k)


def gen_x(rng, m: int, k: int) -> np.ndarray:
    """Activations, fp32 N(0, 1), shape (m, k)."""
    return rng.standard_normal(size=(m, k), dtype=np.float32)


def zipf_weights(n_experts: int, s: float = 1.1) -> np.ndarray:
    r = np.arange(1, n_experts + 1, dtype=np.float64)
    w = r ** (-s)
    return w / w.sum()


def gen_moe_ids(rng, n_tokens: int, top_k: int, n_experts: int, s: float = 1.1) -> np.ndarray:
    """Routing ids int32 [n_tokens][top_k]: top_k distinct experts per token,
    drawn without replacement with probability proportional to rank^-s
    (expert id = rank - 1), via the Gumbel-top-k construction."""
    if top_k > n_experts:
        raise ValueError("top_k > n_experts")
    logw = np.log(zipf_weights(n_experts, s))
    g = rng.gumbel(size=(n_tokens, n_experts))
    keys = logw[None, :] + g
    ids = np.argsort(-keys, axis=1, kind="stable")[:, :top_k]
    return ids.astype(np.int32)


# Named workloads (shapes of the pages' workloads; seed 0 unless stated).
WORKLOADS = {
    "pr1_q4K_n1024_k2048_m16": dict(fmt="q4_K", n=1024, k=2048, m=16),
    "decode_q4K_n17408_k5120": dict(fmt="q4_K", n=17408, k=5120, m=(1, 2, 4, 5, 8)),
    "prefill_q4K_n14336_k4096": dict(fmt="q4_K", n=14336, k=4096, m=(512, 2048)),
    "prefill_q4K_n4100_k4096": dict(fmt="q4_K", n=4100, k=4096, m=(512,)),
    "mixed_q6K_n151936_k5120": dict(fmt="q6_K", n=151936, k=5120, m=(1, 512)),
    "mixed_q80_n5120_k5120": dict(fmt="q8_0", n=5120, k=5120, m=(1, 512)),
    "q40_n8192_k4096": dict(fmt="q4_0", n=8192, k=4096, m=(1, 512)),
    "moe_q4K_e128_n1536_k4096_t512_top8": dict(fmt="q4_K", n=1536, k=4096, n_experts=128, n_tokens=512, top_k=8),
}


def make_dense(fmt: str, n: int, k: int, m: int, seed: int = 0):
    """(W bytes, x fp32) for one dense problem."""
    rw, rx, _ = streams(seed)
    return gen_weights(fmt, rw, n, k), gen_x(rx, m, k)


def make_moe(n_experts: int, n: int, k: int, n_tokens: int, top_k: int, seed: int = 0, fmt: str = "q4_K", s: float = 1.1):
    """(W bytes [E][n][row], x fp32 [T][k], ids int32 [T][top_k]) for one MoE problem."""
    rw, rx, ri = streams(seed)
    W = gen_weights(fmt, rw, n_experts * n, k).reshape(n_experts, n, -1)
    x = gen_x(rx, n_tokens, k)
    ids = gen_moe_ids(ri, n_tokens, top_k, n_experts, s)
    return W, x, ids
