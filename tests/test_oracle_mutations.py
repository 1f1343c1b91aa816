"""Planted mistakes: each plausible slip in the oracle's arithmetic, made in a temporary
copy of its C source (on the CPU, never on the product path), must make at least one of
the oracle's pins fail.  This is what makes the pins evidence: a pin set that a dropped
term, a wrong sign, a wrong index or a swapped operand slips through would not be."""
import ctypes
import os
import subprocess

import numpy as np

import pytest

import oracle
import test_oracle_formats as F
import test_oracle_matmul as M

SRC = os.path.join(os.path.dirname(oracle.__file__), "qmm_oracle.c")

# (name, original text, planted text, pins that must catch it)
MUTATIONS = [
    ("Q4_0 nibble halves swapped",
     "return (i < 16 ? (qs[i] & 0x0f) : (qs[i - 16] >> 4)) - 8;",
     "return (i < 16 ? (qs[i] >> 4) : (qs[i - 16] & 0x0f)) - 8;",
     [F.test_q4_0_nibble_positions_and_offset, F.test_q4_0_decode_all_codes]),
    ("Q4_0 offset dropped",
     "return (i < 16 ? (qs[i] & 0x0f) : (qs[i - 16] >> 4)) - 8;",
     "return (i < 16 ? (qs[i] & 0x0f) : (qs[i - 16] >> 4));",
     [F.test_q4_0_nibble_positions_and_offset, M.test_q4_0_integer_matmul_special_case]),
    ("Q4_K min term added instead of subtracted",
     "acc += t1 - t2;", "acc += t1 + t2;",
     [M.test_q4_K_min_term_special_case]),
    ("Q4_K scale of sub-blocks 0-3 read from the min bytes",
     "*sc = s12[j] & 63;", "*sc = s12[j + 4] & 63;",
     [F.test_q4_K_scale_packing_roundtrip, M.test_q4_K_integer_matmul_special_case]),
    ("Q6_K high-bit pair taken from the wrong shift",
     "int high = (qh[32 * h + l] >> (2 * t)) & 3;", "int high = (qh[32 * h + l] >> t) & 3;",
     [F.test_q6_K_fields_roundtrip, F.test_q6_K_raw_bit_positions, M.test_q6_K_integer_matmul_special_case]),
    ("Q8_0 weights read as unsigned",
     "sumi += (int64_t)(int8_t)blk[2 + i] * (int8_t)xb[4 + i];",
     "sumi += (int64_t)blk[2 + i] * (int8_t)xb[4 + i];",
     [M.test_q8_0_integer_matmul_special_case]),
    ("Q4_K low and high nibbles swapped",
     "return t < 32 ? (qs[32 * c + t] & 0x0f) : (qs[32 * c + t - 32] >> 4);",
     "return t < 32 ? (qs[32 * c + t] >> 4) : (qs[32 * c + t - 32] & 0x0f);",
     [F.test_q4_K_nibble_positions, M.test_q4_K_integer_matmul_special_case]),
    ("MoE bucketing not stable (pairs of an expert in reverse order)",
     "            if (ids[i] == e) perm[pos++] = (int32_t)i;",
     "            if (ids[n_tokens * top_k - 1 - i] == e) perm[pos++] = (int32_t)(n_tokens * top_k - 1 - i);",
     [M.test_bucket_is_stable_sort]),
    ("mul_mat_id per-slot x read from the token's row",
     "int64_t xrow = x_per_slot ? i : i / top_k;",
     "int64_t xrow = i / top_k;",
     [M.test_mul_mat_id_per_slot_reduces_to_dense]),
    ("Q4_K d and dmin swapped in the fold",
     "\n            double d = h2d(blk), dmin = h2d(blk + 2);",
     "\n            double dmin = h2d(blk), d = h2d(blk + 2);",
     [M.test_q4_K_integer_matmul_special_case, M.test_q4_K_min_term_special_case]),
    ("Q6_K sub-scale of the 32-block instead of the 16-block",
     "double t = d * (int8_t)blk[192 + j] * d8 * (double)sumi;",
     "double t = d * (int8_t)blk[192 + j / 2] * d8 * (double)sumi;",
     [M.test_q6_K_integer_matmul_special_case]),
    ("mul_mat_id shared x read from the wrong row",
     "int64_t xrow = x_per_slot ? i : i / top_k;",
     "int64_t xrow = x_per_slot ? i : i % top_k;",
     [M.test_mul_mat_id_reduces_to_dense]),
    ("q8_1 s from the fp32 d instead of the stored fp16 d",
     "uint16_t sh = oracle_float_to_half(dhf * (float)S);",
     "uint16_t sh = oracle_float_to_half(d * (float)S);",
     [lambda o: F.test_q8_1_invariants(o, "normal"), lambda o: F.test_q8_1_invariants(o, "adversarial")]),
    ("Q5_K fifth bit taken from bit l % 8 of qh[i / 8] instead of bit i / 32 of qh[i % 32]",
     "int high = (qh[i % 32] >> (i / 32)) & 1;", "int high = (qh[i / 8] >> (i % 8)) & 1;",
     [F.test_q5_K_raw_bit_positions, F.test_q5_K_fields_roundtrip, M.test_q5_K_integer_matmul_special_case]),
    ("Q5_K fifth bit worth 32 instead of 16",
     "return low | (high << 4);", "return low | (high << 5);",
     [F.test_q5_K_raw_bit_positions, M.test_q5_K_integer_matmul_special_case]),
    ("Q5_K codes read at Q4_K's nibble offset (the qh plane ignored)",
     "const uint8_t *qh = blk + 16, *qs = blk + 48;", "const uint8_t *qh = blk + 16, *qs = blk + 16;",
     [F.test_q5_K_raw_bit_positions, M.test_q5_K_integer_matmul_special_case]),
    # the tolerance sum T, which scales every parity bound: a slip that inflates it would
    # loosen every GPU comparison without failing any of them
    ("T taken as |y| instead of the sum of |block terms|",
     "if (T) *T = tabs;", "if (T) *T = fabs(acc);",
     [M.test_q4_K_tolerance_sum_closed_form, M.test_q6_K_tolerance_sum_closed_form,
      lambda o: M.test_32_block_tolerance_sum_closed_form(o, "q8_0")]),
    ("Q4_K T from the net sub-block term |t1 - t2|",
     "tabs += fabs(t1) + fabs(t2);", "tabs += fabs(t1 - t2);",
     [M.test_q4_K_tolerance_sum_closed_form, M.test_q4_K_min_term_special_case]),
    ("Q4_K T without the scale term",
     "tabs += fabs(t1) + fabs(t2);", "tabs += fabs(t2);",
     [M.test_q4_K_tolerance_sum_closed_form, M.test_q4_K_min_term_special_case]),
    ("Q4_K T as |sum| per superblock",
     ("double d = h2d(blk), dmin = h2d(blk + 2);\n            for (int b = 0; b < 8; ++b) {",
      "                tabs += fabs(t1) + fabs(t2);\n            }\n"),
     ("double d = h2d(blk), dmin = h2d(blk + 2), sb = 0.0;\n            for (int b = 0; b < 8; ++b) {",
      "                sb += t1 - t2;\n            }\n            tabs += fabs(sb);\n"),
     [M.test_q4_K_tolerance_sum_closed_form, M.test_q4_K_min_term_special_case]),
    ("Q6_K T without the q8_1 d",
     "                acc += t;\n                tabs += fabs(t);",
     "                acc += t;\n                tabs += fabs(d * (int8_t)blk[192 + j] * (double)sumi);",
     [M.test_q6_K_tolerance_sum_closed_form]),
    ("Q8_0 T from |q_w| |q_x| instead of |sumi|",
     "            for (int i = 0; i < 32; ++i) sumi += (int64_t)(int8_t)blk[2 + i] * (int8_t)xb[4 + i];\n"
     "            double t = h2d(blk) * h2d(xb) * (double)sumi;\n"
     "            acc += t;\n"
     "            tabs += fabs(t);",
     "            int64_t sabs = 0;\n"
     "            for (int i = 0; i < 32; ++i) sumi += (int64_t)(int8_t)blk[2 + i] * (int8_t)xb[4 + i];\n"
     "            for (int i = 0; i < 32; ++i) sabs += llabs((int64_t)(int8_t)blk[2 + i] * (int8_t)xb[4 + i]);\n"
     "            double t = h2d(blk) * h2d(xb) * (double)sumi;\n"
     "            acc += t;\n"
     "            tabs += fabs(h2d(blk) * h2d(xb)) * (double)sabs;",
     [lambda o: M.test_32_block_tolerance_sum_closed_form(o, "q8_0")]),
]


def _catches(pin, mod):
    try:
        pin(mod)
    except AssertionError:
        return True
    return False


@pytest.mark.parametrize("name,orig,planted,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, oracle_mod, name, orig, planted, pins):
    src = open(SRC).read()
    # a mistake is one replacement, or a tuple of them made together
    origs, planteds = (orig, planted) if isinstance(orig, tuple) else ((orig,), (planted,))
    for o, p in zip(origs, planteds):
        assert src.count(o) == 1, f"the line to plant in is gone: {o}"
        src = src.replace(o, p)
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", "-std=c11",
                    "-o", str(so), str(mutant_c), "-lm"], check=True)
    real = oracle.lib()
    # every pin passes on the real oracle ...
    for pin in pins:
        pin(oracle)
    # ... and at least one fails on the planted copy
    oracle._lib = oracle.load(str(so))
    try:
        caught = [_catches(pin, oracle) for pin in pins]
    finally:
        oracle._lib = real
    assert any(caught), f"no pin catches: {name}"


# The SwiGLU reference is numpy code: its planted mistakes replace a function of the
# oracle module for the duration of the check.
def _glu_mutant(combine):
    real = oracle._glu

    def glu(g, Tg, u, Tu):
        _, tol = real(g, Tg, u, Tu)
        return combine(g, u), tol
    return glu


def _silu(v):
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


_real_glu = oracle._glu


def _glu_tol_mutant(bound):
    """The real SwiGLU value with a planted mistake in its bound."""
    def glu(g, Tg, u, Tu):
        y, tol = _real_glu(g, Tg, u, Tu)
        return y, bound(g, Tg, u, Tu, tol)
    return glu


PY_MUTATIONS = [
    ("silu with the sigmoid's sign flipped", "silu",
     lambda v: np.asarray(v, dtype=np.float64) / (1.0 + np.exp(np.asarray(v, dtype=np.float64))),
     [M.test_silu_closed_forms]),
    ("SwiGLU ignoring the up dot", "_glu", _glu_mutant(lambda g, u: _silu(g) * g),
     [M.test_mul_mat_glu_pins, M.test_mul_mat_glu_gate_and_up_roles]),
    ("SwiGLU with gate and up swapped", "_glu", _glu_mutant(lambda g, u: _silu(u) * g),
     [M.test_mul_mat_glu_pins, M.test_mul_mat_glu_gate_and_up_roles]),
    ("SwiGLU without the silu", "_glu", _glu_mutant(lambda g, u: g * u),
     [M.test_mul_mat_glu_pins, M.test_mul_mat_glu_gate_and_up_roles]),
    ("SwiGLU bound 100 times too wide", "_glu", _glu_tol_mutant(lambda g, Tg, u, Tu, tol: 100 * tol),
     [M.test_mul_mat_glu_tolerance_closed_forms]),
    ("SwiGLU bound without the slope of silu", "_glu",
     _glu_tol_mutant(lambda g, Tg, u, Tu, tol: 1e-5 * (np.abs(_silu(g)) * Tg * np.abs(u) + np.abs(_silu(g)) * Tu)
                     + 2.0 ** -20 * np.abs(_silu(g) * u) + 2.0 ** -120 * np.abs(u)),
     [M.test_mul_mat_glu_tolerance_closed_forms]),
    ("SwiGLU bound without the fp32 evaluation term", "_glu",
     _glu_tol_mutant(lambda g, Tg, u, Tu, tol: tol - 2.0 ** -20 * np.abs(_silu(g) * u)),
     [M.test_mul_mat_glu_tolerance_closed_forms]),
    ("SwiGLU bound with gate and up bounds swapped", "_glu",
     _glu_tol_mutant(lambda g, Tg, u, Tu, tol: _real_glu(g, Tu, u, Tg)[1]),
     [M.test_mul_mat_glu_tolerance_closed_forms]),
]


@pytest.mark.parametrize("name,attr,mutant,pins", PY_MUTATIONS, ids=[m[0] for m in PY_MUTATIONS])
def test_planted_python_mistake_is_caught(oracle_mod, name, attr, mutant, pins):
    for pin in pins:
        pin(oracle)
    real = getattr(oracle, attr)
    setattr(oracle, attr, mutant)
    try:
        caught = [_catches(pin, oracle) for pin in pins]
    finally:
        setattr(oracle, attr, real)
    assert any(caught), f"no pin catches: {name}"
