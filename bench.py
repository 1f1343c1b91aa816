#!/usr/bin/env python3
"""Benchmark of the block-quantized matmul on GB300.

One step = one pass of the hot path over one batch of synthetic input:
q8_1 quantization of x followed by y = x * dequant(W)^T.

Headline workload (the pages' decode GEMV shape): Q4_K W n=17408 x k=5120, m=1
fp32 activation row.  The metric is HBM GB/s of algorithmic bytes; the roofline
object reports the GEMV kernel against the measured HBM copy bandwidth.  The
"secondary" object reports the prefill GEMM (m=512) and the MoE mul_mat_id in
TOPS (2*m*n*k integer multiply-adds), and every other workload shape of the pages is
timed the same way.

Timing: the K timed steps (and, separately, the W warm-up steps) are captured once
into a CUDA graph and replayed, so the device-side numbers carry no Python launch
overhead; CUDA events on the launching stream bracket exactly the K steps, with a
barrier and a device synchronise on both sides, max over ranks.  The roofline
kernel time comes from a second graph holding K back-to-back launches of the GEMV
alone.  The end-to-end number is measured without graphs, through the Python API a
user calls, with the host-to-device copy of x and the device-to-host copy of y
inside the timed region.  L2 is defeated by rotating among weight copies whose
total size exceeds 3x the 129 MB L2.

--impl reference times the CPU oracle (test infrastructure, plain fp64 C) on the
host cores, on a bounded sample of the same workload, and prints the same JSON line
with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import qmm_synth  # noqa: E402

METRIC = "Q4_K matmul HBM GB/s at m=1 and int8 TOPS at m=512/MoE, % of GB300 roofline"
UNIT = "GB/s"
N, K, M = 17408, 5120, 1
WORKLOAD = "decode GEMV Q4_K n=17408 k=5120 m=1 (fp32 x in, quantized in the GEMV prologue, y out: one launch)"
L2_BYTES = 129 * 1024 * 1024


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings over all ranks (identity with one rank)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate_rate(world, bytes_per_step, ms_per_step):
    """Whole-job throughput in GB/s: every rank processes bytes_per_step per step;
    the job's step time is the slowest rank's."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def step_bytes(n, k, m, row_bytes):
    """Algorithmic bytes of one step (fp32 x in, quantized on chip, y out): W once, x
    read, y written.  At m <= 8 the step is one launch, so these are also the bytes of
    that launch."""
    return n * row_bytes + m * k * 4 + m * n * 4


def gemv_q8_bytes(n, k, m, row_bytes):
    """Algorithmic bytes of one GEMV launch from q8_1 activations: W once, q8_1 read, y written."""
    return n * row_bytes + m * (k // 32) * 36 + m * n * 4


def int8_tensor_peak():
    """The GPU's dense int8 tensor-core rate in TOPS: on sm_103a tcgen05 has no int8 kind,
    so it is the mma.sync s8 rate, measured once by a stand-alone probe and recorded in
    profiles/mma_sync_peak.json (None when the record is missing)."""
    p = os.path.join(ROOT, "profiles", "mma_sync_peak.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        return json.load(f).get("int8_mma_sync_tops")


def tensor_fracs(tops):
    """A GEMM row's fractions of the int8 tensor-core rate and of the measured bf16
    (tcgen05) rate; the path runs kind::f16 MMAs, the bf16 figure is its own dtype's."""
    out = {}
    i8 = int8_tensor_peak()
    if i8:
        out["int8_tc_frac"] = tops / i8
    out["fp16_tc_frac"] = tops / measured_peaks()[1]
    return out


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# the sources each profiled kernel is built from (its own file and the headers it includes)
_HEADERS = ["qmm_common.cuh", "qmm_tc_ptx.cuh", "qmm_internal.h", "qmm_moe.h", "../../include/qmm.h"]
KERNEL_SOURCES = {"gemv_q4k_tma_kernel<1>": ["qmm_gemv.cu"] + _HEADERS,
                  "gemm_tc_q4k_kernel": ["qmm_gemm_tc.cu"] + _HEADERS}


def kernel_source_sha(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_matmul_q8_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(os.path.basename(name).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from a committed ncu summary, if taken on the kernel's
    current sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_sha") != kernel_source_sha(kernel):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
        if not self.path or not os.path.exists(self.path):
            return out
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if sm:
            loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
            out = {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                   "samples": len(sm)}
        return out


def oracle_baseline(W, x, n, k, m, row_bytes, budget_s=12.0):
    """The CPU oracle (as it stands) on the host cores: quantize + fold over whole rows,
    repeated over row slices until about budget_s seconds of work; returns GB/s of
    the same algorithmic bytes."""
    import oracle
    threads = oracle.set_threads(os.cpu_count() or 1)
    rows_per = max(1, n // 8)
    done_rows, t0, reps = 0, time.perf_counter(), 0
    while True:
        r0 = (reps * rows_per) % n
        r1 = min(n, r0 + rows_per)
        xq = oracle.quantize_q8_1(x)
        oracle.mul_mat(W[r0:r1], "q4_K", r1 - r0, k, xq, m)
        done_rows += r1 - r0
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    bytes_done = done_rows * row_bytes + reps * (m * k * 4 + 2 * m * (k // 32) * 36) + done_rows * m * 4
    return {"value": bytes_done / el / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done_rows} weight rows of the n={n} k={k} m={m} Q4_K problem in {reps} slices "
                      f"(quantize + fp64 fold), {el:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    row_bytes = (K // 256) * 144
    W, x = qmm_synth.make_dense("q4_K", N, K, M, seed=0)
    import oracle
    oracle.build()
    steps = []
    for i in range(args.warmup + args.steps):
        r = oracle_baseline(W, x, N, K, M, row_bytes, budget_s=max(2.0, 20.0 / max(1, args.steps + args.warmup)))
        if i >= args.warmup:
            steps.append(r)
    val = statistics.median(s["value"] for s in steps)
    # time one whole step of the workload would take at the measured rate
    ms_step = step_bytes(N, K, M, row_bytes) / (val * 1e9) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n": N, "k": K, "m": M, "format": "Q4_K", "seed": 0,
                       "sample": "each step times bounded slices of the workload on the host cores"},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": steps[0]["cores"], "kind": "oracle",
                             "sample": steps[0]["sample"]},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_region(torch, fn, steps, warmup, stream, barrier):
    """Eager timing: W warm-up steps, then exactly K steps between two events."""
    for i in range(warmup):
        fn(i)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        fn(warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1)


def capture(torch, fn, first, count):
    """A CUDA graph holding steps first .. first+count-1 of fn."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(first, first + count):
            fn(i)
    return g


HOLD_CYCLES = 200_000  # ~0.1 ms of device time at 2 GHz


def time_graphs(torch, fn, steps, warmup, barrier):
    """Graph timing: eager warm-up, a graph of the W warm-up steps replayed, then a
    graph of exactly K steps replayed once between two events.  A short device-side
    hold is queued in front of the first event, so that the GPU is still busy while the
    host submits the graph: the events then time the K steps on the device, not the
    host's graph-submission latency."""
    for i in range(2):
        fn(i)
    torch.cuda.synchronize()
    gw = capture(torch, fn, 0, warmup)
    gt = capture(torch, fn, warmup, steps)
    gw.replay()
    barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(HOLD_CYCLES)
    e0.record(stream)
    gt.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1)


def secondary(torch, qmm, dev, stream, steps, hbm_peak, only=""):
    """Every other workload of the pages, device-timed by graph replay: GEMV rows in
    GB/s (and fraction of the HBM peak), GEMM and MoE rows in TOPS (2*m*n*k).  `only`
    keeps the rows whose name contains it."""
    out = {}

    def dense(fmt, n, k, ms, q8_input=False):
        ms = [m for m in ms if only in f"{fmt}_n{n}_k{k}_m{m}" + ("_q8_1_input" if q8_input else "")]
        if not ms:
            return {}
        """Whole path from fp32 x (qmm_mul_mat_f32); q8_input times qmm_mul_mat on
        pre-quantized activations instead."""
        rows = {}
        W, x = qmm_synth.make_dense(fmt, n, k, max(ms), seed=0)
        copies = max(1, int(3 * L2_BYTES // W.nbytes) + 1)
        Wd = [torch.from_numpy(W).to(dev) for _ in range(copies)]
        x_all = torch.from_numpy(x).to(dev)
        xq_all = qmm.qmm_quantize_q8_1(x_all)
        for m in ms:
            xm = x_all[:m].contiguous()
            xq = xq_all[:m].contiguous()
            y = torch.empty((m, n), device=dev)
            if q8_input:
                ws = torch.empty(max(1, qmm.qmm_workspace_bytes(fmt, n, k, m)), dtype=torch.uint8, device=dev)
                fn = lambda i: qmm.qmm_mul_mat(Wd[i % copies], fmt, n, k, xq, m, y=y, workspace=ws)
                xb = m * (k // 32) * 36
            else:
                ws = torch.empty(max(1, qmm.qmm_workspace_bytes_f32(fmt, n, k, m)), dtype=torch.uint8, device=dev)
                fn = lambda i: qmm.qmm_mul_mat_f32(Wd[i % copies], fmt, n, k, xm, m, y=y, workspace=ws)
                xb = m * k * 4
            ms_call = time_graphs(torch, fn, steps, 3, lambda: None) / steps
            key = f"{fmt}_n{n}_k{k}_m{m}" + ("_q8_1_input" if q8_input else "")
            if m <= 8:
                b = W.nbytes + xb + m * n * 4
                rows[key] = {"GB/s": b / (ms_call * 1e-3) / 1e9, "hbm_frac": b / (ms_call * 1e-3) / 1e9 / hbm_peak,
                             "ms": ms_call}
            else:
                rows[key] = {"tops": 2 * m * n * k / (ms_call * 1e-3) / 1e12, "ms": ms_call}
                rows[key].update(tensor_fracs(rows[key]["tops"]))
            rows[key]["l2"] = f"{copies} weight copies ({copies * W.nbytes / 1e6:.0f} MB)"
        del Wd
        return rows

    def glu(n, k, ms, packed=False):
        """Fused gate/up + SwiGLU from q8_1 input: both weights (n rows each) in GB/s at
        m <= 8, TOPS over both products (2 * m * 2n * k) above.  packed: the interleaved
        tensor of qmm_repack_glu (the repack itself is outside the timed region)."""
        name = "glu_packed" if packed else "glu"
        ms = [m for m in ms if only in f"{name}_q4_K_n{n}_k{k}_m{m}"]
        if not ms:
            return {}
        rows = {}
        W, x = qmm_synth.make_dense("q4_K", 2 * n, k, max(ms), seed=0)
        copies = max(1, int(3 * L2_BYTES // W.nbytes) + 1)
        Wg = [torch.from_numpy(W[:n].copy()).to(dev) for _ in range(copies)]
        Wu = [torch.from_numpy(W[n:].copy()).to(dev) for _ in range(copies)]
        if packed:
            Wg = [qmm.qmm_repack_glu(g, u, "q4_K", n, k) for g, u in zip(Wg, Wu)]
            Wu = None
        xq_all = qmm.qmm_quantize_q8_1(torch.from_numpy(x).to(dev))
        for m in ms:
            xq = xq_all[:m].contiguous()
            y = torch.empty((m, n), device=dev)
            need = qmm.qmm_workspace_bytes_glu("q4_K", n, k, m)
            ws = torch.empty(max(1, need), dtype=torch.uint8, device=dev)
            if packed:
                fn = lambda i: qmm.qmm_mul_mat_glu_packed(Wg[i % copies], "q4_K", n, k, xq, m, y=y, workspace=ws)
            else:
                fn = lambda i: qmm.qmm_mul_mat_glu(Wg[i % copies], Wu[i % copies], "q4_K", n, k, xq, m, y=y,
                                                   workspace=ws)
            ms_call = time_graphs(torch, fn, steps, 3, lambda: None) / steps
            key = f"{name}_q4_K_n{n}_k{k}_m{m}"
            if m <= 8:
                b = W.nbytes + m * (k // 32) * 36 + m * n * 4
                rows[key] = {"GB/s": b / (ms_call * 1e-3) / 1e9, "hbm_frac": b / (ms_call * 1e-3) / 1e9 / hbm_peak,
                             "ms": ms_call}
            else:
                rows[key] = {"tops": 2 * m * 2 * n * k / (ms_call * 1e-3) / 1e12, "ms": ms_call}
                rows[key].update(tensor_fracs(rows[key]["tops"]))
            rows[key]["l2"] = f"{copies} copies of both weights ({copies * W.nbytes / 1e6:.0f} MB)"
        del Wg, Wu
        return rows

    out.update(dense("q4_K", 17408, 5120, [1], q8_input=True))
    out.update(dense("q4_K", 17408, 5120, [2, 4, 5, 8]))
    out.update(dense("q4_K", 1024, 2048, [16]))
    out.update(dense("q4_K", 17408, 5120, [16]))
    out.update(dense("q4_K", 4096, 14336, [1]))  # the prefill shape's down projection: long rows
    out.update(dense("q4_K", 14336, 4096, [512, 2048]))
    out.update(dense("q4_K", 4100, 4096, [512]))
    out.update(dense("q6_K", 151936, 5120, [1, 512]))
    out.update(dense("q8_0", 5120, 5120, [1, 512]))
    out.update(dense("q4_0", 8192, 4096, [1, 512]))
    out.update(glu(14336, 4096, [1, 512]))
    out.update(glu(14336, 4096, [1, 512], packed=True))
    # MoE: 128 experts x Q4_K n=1536 k=4096, 512 tokens top-8 Zipf(1.1); and its decode
    # form, one token top-8, whose calls route to disjoint sets of 8 experts in turn (16
    # calls cover all 128 experts, 453 MB, so no call finds its experts in L2)
    key_p, key_d = "moe_q4K_e128_n1536_k4096_t512_top8", "moe_decode_q4K_e128_n1536_k4096_t1_top8"
    key_g, key_gd = "moe_glu_q4K_e128_n1536_k4096_t512_top8", "moe_glu_decode_q4K_e128_n1536_k4096_t1_top8"
    if not any(only in key for key in (key_p, key_d, key_g, key_gd)):
        return out
    E, n, k, T_, Kt = 128, 1536, 4096, 512, 8
    W, x, ids = qmm_synth.make_moe(E, n, k, T_, Kt, seed=0)
    Wd = torch.from_numpy(W).to(dev)
    if only in key_p:
        xq = qmm.qmm_quantize_q8_1(torch.from_numpy(x).to(dev))
        idd = torch.from_numpy(ids).to(dev)
        y = torch.empty((T_, Kt, n), device=dev)
        ws = torch.empty(qmm.qmm_workspace_bytes("q4_K", n, k, T_, E, Kt), dtype=torch.uint8, device=dev)
        fn = lambda i: qmm.qmm_mul_mat_id(Wd, "q4_K", E, n, k, xq, idd, Kt, T_, y=y, workspace=ws)
        ms = time_graphs(torch, fn, steps, 3, lambda: None) / steps
        out[key_p] = {"tops": 2 * T_ * Kt * n * k / (ms * 1e-3) / 1e12, "ms": ms, "l2": "weights 453 MB > 3x L2"}
        out[key_p].update(tensor_fracs(out[key_p]["tops"]))
    if only in key_d:
        order = np.random.default_rng(7).permutation(E).astype(np.int32)
        ids_d = [torch.from_numpy(order[8 * j:8 * j + 8].reshape(1, Kt).copy()).to(dev) for j in range(E // Kt)]
        xq1 = qmm.qmm_quantize_q8_1(torch.from_numpy(x[:1]).to(dev))
        y1 = torch.empty((1, Kt, n), device=dev)
        ws1 = torch.empty(qmm.qmm_workspace_bytes("q4_K", n, k, 1, E, Kt), dtype=torch.uint8, device=dev)
        fn = lambda i: qmm.qmm_mul_mat_id(Wd, "q4_K", E, n, k, xq1, ids_d[i % len(ids_d)], Kt, 1, y=y1, workspace=ws1)
        ms = time_graphs(torch, fn, steps, 3, lambda: None) / steps
        b = Kt * n * (k // 256) * 144 + (k // 32) * 36 + Kt * n * 4
        out[key_d] = {"GB/s": b / (ms * 1e-3) / 1e9, "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_peak, "ms": ms,
                      "l2": "16 routings cycle through the 128 experts (453 MB)"}
    if only in key_g or only in key_gd:
        # the fused gate/up + SwiGLU of the same MoE FFN: a second expert tensor as the up weights
        Wu = torch.from_numpy(qmm_synth.gen_weights("q4_K", np.random.default_rng(5), E * n, k)).to(dev)
    if only in key_g:
        xq = qmm.qmm_quantize_q8_1(torch.from_numpy(x).to(dev))
        idd = torch.from_numpy(ids).to(dev)
        y = torch.empty((T_, Kt, n), device=dev)
        ws = torch.empty(qmm.qmm_workspace_bytes_id_glu("q4_K", n, k, T_, E, Kt), dtype=torch.uint8, device=dev)
        fn = lambda i: qmm.qmm_mul_mat_id_glu(Wd, Wu, "q4_K", E, n, k, xq, idd, Kt, T_, y=y, workspace=ws)
        ms = time_graphs(torch, fn, steps, 3, lambda: None) / steps
        out[key_g] = {"tops": 2 * 2 * T_ * Kt * n * k / (ms * 1e-3) / 1e12, "ms": ms,
                      "l2": "gate and up weights 906 MB > 3x L2"}
        out[key_g].update(tensor_fracs(out[key_g]["tops"]))
    if only in key_gd:
        order = np.random.default_rng(7).permutation(E).astype(np.int32)
        ids_d = [torch.from_numpy(order[8 * j:8 * j + 8].reshape(1, Kt).copy()).to(dev) for j in range(E // Kt)]
        xq1 = qmm.qmm_quantize_q8_1(torch.from_numpy(x[:1]).to(dev))
        y1 = torch.empty((1, Kt, n), device=dev)
        ws1 = torch.empty(max(qmm.qmm_workspace_bytes_id_glu("q4_K", n, k, 1, E, Kt), 256), dtype=torch.uint8,
                          device=dev)
        fn = lambda i: qmm.qmm_mul_mat_id_glu(Wd, Wu, "q4_K", E, n, k, xq1, ids_d[i % len(ids_d)], Kt, 1, y=y1,
                                              workspace=ws1)
        ms = time_graphs(torch, fn, steps, 3, lambda: None) / steps
        b = 2 * Kt * n * (k // 256) * 144 + (k // 32) * 36 + Kt * n * 4
        out[key_gd] = {"GB/s": b / (ms * 1e-3) / 1e9, "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_peak, "ms": ms,
                       "l2": "16 routings cycle through the 128 experts (906 MB of gate and up weights)"}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="qmm", choices=["qmm", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--rows", default="", help="only the secondary rows whose name contains this text")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        args.warmup = 3

    import torch
    import torch.distributed as dist

    import block_quantized_matmul_q8_gb300 as qmm

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qmm.build()

    def barrier():
        if world > 1:
            dist.barrier()

    row_bytes = qmm.qmm_row_bytes("q4_K", K)
    W, x = qmm_synth.make_dense("q4_K", N, K, M, seed=0)
    copies = max(2, int(3 * L2_BYTES // W.nbytes) + 1)
    Wd = [torch.from_numpy(W).to(dev) for _ in range(copies)]
    x_h = torch.from_numpy(x).pin_memory()
    x_d = x_h.to(dev)
    y = torch.empty((M, N), device=dev)
    y_h = torch.empty((M, N), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()

    # --- device-resident steps (graph-replayed): one call from fp32 x, which at m = 1 is
    # one launch of the GEMV that quantizes x in its prologue
    def step(i):
        qmm.qmm_mul_mat_f32(Wd[i % copies], "q4_K", N, K, x_d, M, y=y)

    with ClockSampler(local) as clk:
        ms_total = time_graphs(torch, step, args.steps, args.warmup, barrier)
    clocks = clk.summary()

    # --- end to end through the C ABI's host-buffer call: each step one qmm_mul_mat_f32_host
    # call that enqueues the copy of the pinned host x, the product and the copy of y back
    ws_host = torch.empty(max(256, qmm.qmm_workspace_bytes_f32_host("q4_K", N, K, M)), dtype=torch.uint8, device=dev)

    def step_e2e(i):
        qmm.qmm_mul_mat_f32_host(Wd[i % copies], "q4_K", N, K, x_h, M, y_h, ws_host, stream=stream)

    ms_e2e = time_region(torch, step_e2e, args.steps, args.warmup, stream, barrier)

    ms_total, ms_e2e = max_over_ranks([ms_total, ms_e2e], device=dev)
    ms_step = ms_total / args.steps
    sb = step_bytes(N, K, M, row_bytes)
    value = aggregate_rate(world, sb, ms_step)
    e2e_value = aggregate_rate(world, sb, ms_e2e / args.steps)
    hbm_peak, tf_peak, peak_src = measured_peaks()
    # the step is one launch of the GEMV kernel: its duration is the step's
    gemv_ms = ms_step
    kb = sb
    achieved = kb / (gemv_ms * 1e-3) / 1e9
    traffic = recorded_traffic("gemv_q4k_tma_kernel<1>")

    sec = None
    if rank == 0 and not args.no_secondary:
        sec = secondary(torch, qmm, dev, stream, steps=10, hbm_peak=measured_peaks()[0], only=args.rows)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(W, x, N, K, M, row_bytes)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8 dot (exact int32) + fp32 fold", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n": N, "k": K, "m": M, "format": "Q4_K", "seed": 0,
                       "timing": "CUDA graph replay of exactly K steps between events (device-side hold "
                                 "queued before the first event hides the host's graph submission)",
                       "l2": f"rotating {copies} weight copies ({copies * W.nbytes / 1e6:.0f} MB > 3x L2)",
                       "replicas": world},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic, "kernel": "gemv_q4k_tma_kernel<1>",
                         "peak_source": f"{peak_src} HBM copy bandwidth", "kernel_ms": gemv_ms,
                         "kernel_timing": "graph of K back-to-back steps (one GEMV launch each) between events",
                         "algorithmic_bytes": kb},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": M * K * 4,
                    "d2h_bytes_per_step": M * N * 4, "ms_per_step": ms_e2e / args.steps,
                    "how": "one qmm_mul_mat_f32_host call per step (eager, no graph) on page-locked host x and y: the GEMV reads x and writes y in host memory in place (the bytes cross the CPU-GPU link inside the timed region)"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "secondary": sec,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
