"""Shared helpers for the GPU parity tests (inputs from qmm_synth, expected values from the oracle)."""
from __future__ import annotations

import numpy as np

# |y_gpu - y_oracle| <= TOL * (sum over blocks of |block term|), per element.
TOL = 1e-5


def assert_within(y_gpu, y_ref, T, what=""):
    y = np.asarray(y_gpu, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    bad = err > TOL * T
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.unravel_index(np.argmax(err / np.maximum(T, 1e-300)), y.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{y.size} outside {TOL}*T; first {idx.tolist()}; "
                             f"worst {worst}: gpu={y[worst]!r} ref={y_ref[worst]!r} T={T[worst]!r}")
    return float((err / np.where(T > 0, T, 1)).max()) if y.size else 0.0


def adversarial_x_rows():
    """32-value blocks that stress the quantizer: zeros, signed zeros, exact ties,
    extremes near the fp16 range, denormals, constant blocks, amax at several places."""
    rows = []
    z = np.zeros(32, np.float32)
    rows.append(z.copy())
    nz = z.copy(); nz[:] = -0.0; rows.append(nz)
    one = z.copy(); one[7] = 3.5; rows.append(one)
    neg = z.copy(); neg[31] = -2.0; neg[0] = 1.0; rows.append(neg)
    tie = np.arange(32, dtype=np.float32) - 15.5; tie[0] = 127.0; rows.append(tie)
    rows.append(-tie)
    rows.append(np.linspace(-60000, 60000, 32).astype(np.float32))
    rows.append((np.arange(32, dtype=np.float32) - 16) * np.float32(1e-40))
    t2 = np.full(32, np.float32(1.4e-45)); t2[3] = -np.float32(2.8e-45); rows.append(t2)
    rows.append(np.full(32, np.float32(0.3)))
    for pos in (0, 13, 31):
        r = np.random.default_rng(pos).standard_normal(32).astype(np.float32)
        r[pos] = 9.0
        rows.append(r)
    return np.stack(rows)


def near_tie_rows(seed, nblocks, exp_range=(-20, 20)):
    """Blocks whose values sit within a few ulps of (q + 1/2) * d, d = amax/127 in fp32:
    the quotients x/d land on or next to the rounding ties, where a quantizer that does
    not divide exactly in IEEE fp32 would pick another integer.  amax is uniform in
    [1e-3, 1e3] times 2^e, e drawn from exp_range."""
    rng = np.random.default_rng(seed)
    out = np.empty((nblocks, 32), np.float32)
    for b in range(nblocks):
        amax = np.float32(rng.uniform(1e-3, 1e3)) * np.float32(2.0) ** int(rng.integers(*exp_range))
        d = np.float32(amax / np.float32(127))
        q = rng.integers(-127, 127, 32).astype(np.float32)
        v = ((q + np.float32(0.5)) * d).astype(np.float32)
        steps = rng.integers(-6, 7, 32)
        for i in range(32):
            s = int(steps[i])
            while s > 0:
                v[i] = np.nextafter(v[i], np.float32(np.inf)); s -= 1
            while s < 0:
                v[i] = np.nextafter(v[i], np.float32(-np.inf)); s += 1
        v = np.clip(v, -amax, amax)
        v[rng.integers(0, 32)] = amax if rng.random() < 0.5 else -amax
        out[b] = v
    return out
