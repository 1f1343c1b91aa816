"""qmm_mul_mat_f32 (fp32 activations, quantized inside the call) against the oracle
and against qmm_quantize_q8_1 followed by qmm_mul_mat.  For m == 1 the GEMV kernels
quantize the activations in their own prologue; the staged q8_1 bytes must be those of
the quantizer kernel, so y must equal the two-call result to the bit."""
import numpy as np
import pytest
import torch

import block_quantized_matmul_q8_gb300 as qmm
import qmm_synth
from parity import adversarial_x_rows, assert_within, near_tie_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qmm.build()
    qmm.lib()
    yield
    qmm.qmm_set_force_path(0)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def two_calls(Wd, fmt, n, k, xd, m):
    xq = qmm.qmm_quantize_q8_1(xd)
    return qmm.qmm_mul_mat(Wd, fmt, n, k, xq, m)


# (n, k): several 8-row chunks with a ragged tail; k=160 has an odd block count
SHAPES = {"q4_K": [(129, 2304), (1000, 512)], "q6_K": [(129, 2304), (37, 256)],
          "q8_0": [(129, 1056), (33, 160)], "q4_0": [(129, 2048), (33, 160)]}


@pytest.mark.parametrize("fmt", ["q4_K", "q6_K", "q8_0", "q4_0"])
@pytest.mark.parametrize("m", [1, 2, 3, 5, 8, 9, 20])
@pytest.mark.parametrize("path", [0, 4])
def test_f32_equals_two_calls_and_oracle(oracle_mod, fmt, m, path):
    for (n, k) in SHAPES[fmt]:
        W, x = qmm_synth.make_dense(fmt, n, k, m, seed=n + m)
        if m >= 2:
            x[1, :] = 0.0                                   # an all-zero column
        x[0, :32] *= 50.0                                  # a large scale (d*sum q stays in fp16 range)
        Wd, xd = to_dev(W), to_dev(x)
        qmm.qmm_set_force_path(path)
        try:
            y1 = qmm.qmm_mul_mat_f32(Wd, fmt, n, k, xd, m)
            y2 = two_calls(Wd, fmt, n, k, xd, m)
            torch.cuda.synchronize()
        finally:
            qmm.qmm_set_force_path(0)
        a, b = y1.cpu().numpy(), y2.cpu().numpy()
        assert np.array_equal(a, b), f"{fmt} n={n} k={k} m={m} path={path}: differs from quantize + mul_mat"
        y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, oracle_mod.quantize_q8_1(x), m)
        assert_within(a, y_ref, T, f"f32 {fmt} n={n} k={k} m={m}")


def test_f32_adversarial_activations(oracle_mod):
    """Ties after the division, denormal blocks, single spikes: the in-kernel quantizer
    must take every integer decision the oracle takes."""
    k = 512
    xa = np.resize(adversarial_x_rows().reshape(-1), k)   # every adversarial block, then repeats
    x = (np.stack([xa] * 3) * np.float32([[1], [-1], [1e-3]])).astype(np.float32)
    n = 77
    W, _ = qmm_synth.make_dense("q4_K", n, k, 3, seed=3)
    y = qmm.qmm_mul_mat_f32(to_dev(W), "q4_K", n, k, to_dev(x), 3).cpu().numpy()
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, oracle_mod.quantize_q8_1(x), 3)
    assert_within(y, y_ref, T, "f32 adversarial")


def test_f32_workspace_errors():
    n, k, m = 256, 512, 20
    W, x = qmm_synth.make_dense("q4_K", n, k, m, seed=1)
    Wd, xd = to_dev(W), to_dev(x)
    need = qmm.qmm_workspace_bytes_f32("q4_K", n, k, m)
    assert need >= qmm.qmm_q8_1_bytes(m, k) + qmm.qmm_workspace_bytes("q4_K", n, k, m)
    short = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(qmm.QMMError) as e:
        qmm.qmm_mul_mat_f32(Wd, "q4_K", n, k, xd, m, workspace=short)
    assert e.value.code == 5
    # m == 1 runs the one-launch GEMV and needs no workspace
    y = qmm.qmm_mul_mat_f32(Wd, "q4_K", n, k, xd[:1].contiguous(), 1)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("m", [1, 4, 8])
def test_f32_near_ties_equal_two_calls(oracle_mod, m):
    """Activations whose quotients sit on or next to the rounding ties: the in-kernel
    quantizer must pick the integers the quantizer kernel and the oracle pick."""
    k, n = 2048, 200
    x = near_tie_rows(100 + m, m * k // 32, exp_range=(-12, 1)).reshape(m, k)  # s = d * sum q stays finite
    W, _ = qmm_synth.make_dense("q4_K", n, k, m, seed=m)
    Wd, xd = to_dev(W), to_dev(x)
    y1 = qmm.qmm_mul_mat_f32(Wd, "q4_K", n, k, xd, m)
    y2 = two_calls(Wd, "q4_K", n, k, xd, m)
    torch.cuda.synchronize()
    assert np.array_equal(y1.cpu().numpy(), y2.cpu().numpy())
    xq = oracle_mod.quantize_q8_1(x)
    y_ref, T = oracle_mod.mul_mat(W, "q4_K", n, k, xq, m)
    assert_within(y1.cpu().numpy(), y_ref, T, "f32 near ties")


@pytest.mark.parametrize("fmt,n,k,m", [("q4_K", 1000, 512, 1), ("q4_K", 129, 2304, 5), ("q8_0", 33, 160, 20),
                                       ("q4_0", 129, 2048, 1), ("q4_K", 14336, 256, 20)])
@pytest.mark.parametrize("pinned", ["both", "x", "none"])
def test_f32_host_buffers(oracle_mod, fmt, n, k, m, pinned):
    """The host-buffer call gives the bits of the device call, from pinned or pageable host
    memory: page-locked buffers are read and written in place (y only up to 1 MB; the
    14336-column case takes the copy back), pageable ones through copies."""
    W, x = qmm_synth.make_dense(fmt, n, k, m, seed=n + 3 * m)
    Wd = to_dev(W)
    x_h = torch.from_numpy(x)
    y_h = torch.full((m, n), float("nan"))
    if pinned in ("both", "x"):
        x_h = x_h.pin_memory()
    if pinned == "both":
        y_h = y_h.pin_memory()
    ws = torch.empty(max(256, qmm.qmm_workspace_bytes_f32_host(fmt, n, k, m)), dtype=torch.uint8, device=DEV)
    qmm.qmm_mul_mat_f32_host(Wd, fmt, n, k, x_h, m, y_h, ws)
    y_d = qmm.qmm_mul_mat_f32(Wd, fmt, n, k, to_dev(x), m)
    torch.cuda.synchronize()
    assert np.array_equal(y_h.numpy(), y_d.cpu().numpy())
    y_ref, T = oracle_mod.mul_mat(W, fmt, n, k, oracle_mod.quantize_q8_1(x), m)
    assert_within(y_h.numpy(), y_ref, T, f"f32 host {fmt} n={n} k={k} m={m}")


def test_f32_host_workspace_errors():
    n, k, m = 64, 256, 2
    W, x = qmm_synth.make_dense("q4_K", n, k, m, seed=1)
    Wd = to_dev(W)
    need = qmm.qmm_workspace_bytes_f32_host("q4_K", n, k, m)
    assert need >= 256 * 2
    short = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(qmm.QMMError) as e:
        qmm.qmm_mul_mat_f32_host(Wd, "q4_K", n, k, torch.from_numpy(x), m, torch.empty((m, n)), short)
    assert e.value.code == 5
