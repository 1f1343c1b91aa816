"""Host-side checks of the C ABI: the library loads, exports every declared symbol,
rejects bad arguments before touching a GPU, and plans schedules as the pages'
worked examples say.  No kernel runs here."""
import ctypes
import json
import os
import re

import pytest

import block_quantized_matmul_q8_gb300 as qmm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    qmm.build()
    return qmm.lib()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "qmm.h")).read()
    return sorted(set(re.findall(r"QMM_API\s+[\w\s\*]*?\b(qmm_\w+)\s*\(", txt)))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 13
    assert sorted(qmm.EXPORTS) == names
    for name in names:
        assert hasattr(L, name), name


def test_status_strings(L):
    for code, name in qmm.STATUS.items():
        assert qmm.qmm_status_string(code) == name


def test_sizes():
    assert qmm.qmm_q8_1_bytes(3, 256) == 3 * 8 * 36
    assert qmm.qmm_row_bytes("q4_K", 5120) == 20 * 144
    assert qmm.qmm_row_bytes("q6_K", 5120) == 20 * 210
    assert qmm.qmm_row_bytes("q8_0", 96) == 3 * 34
    assert qmm.qmm_row_bytes("q4_0", 96) == 3 * 18
    assert qmm.qmm_row_bytes("q4_0", 100) == 0
    assert qmm.qmm_row_bytes("q4_K", 100) == 0
    assert qmm.qmm_row_bytes(99, 256) == 0


def test_workspace_bytes_zero_for_rejected_sizes(L):
    # the sizes the calls reject get 0, not a figure computed from them
    assert L.qmm_workspace_bytes(99, 8, 256, 4, 0, 0) == 0            # unknown type
    assert L.qmm_workspace_bytes(12, 8, 100, 4, 0, 0) == 0            # k not whole superblocks
    assert L.qmm_workspace_bytes(12, 8, 1 << 21, 4, 0, 0) == 0        # k above the limit
    assert L.qmm_workspace_bytes(12, 1 << 31, 256, 4, 0, 0) == 0      # n above 2^31 - 1
    assert L.qmm_workspace_bytes(12, 8, 256, 1 << 31, 0, 0) == 0      # m above 2^31 - 1
    assert L.qmm_workspace_bytes(12, 8, 256, 1 << 62, 4, 4) == 0      # pairs past 2^31 - 1, product overflows
    assert L.qmm_workspace_bytes(12, 8, 256, 3, 100000, 2) == 0       # too many experts
    assert L.qmm_workspace_bytes(12, 8, 256, 3, 4, 2) > 0
    assert L.qmm_workspace_bytes_id_glu(12, 8, 256, 1 << 62, 4, 4) == 0


def _mm(L, W=1024, t=12, n=8, k=256, xq=2048, m=4, y=4096, ws=None, wsb=0):
    P = ctypes.c_void_p
    return L.qmm_mul_mat(P(W), t, n, k, P(xq), m, P(y), P(ws) if ws else None, wsb, None)


def test_argument_errors_need_no_gpu(L):
    assert _mm(L, t=99) == 3                      # unknown type
    assert _mm(L, k=100) == 2                     # not a multiple of 256
    assert _mm(L, t=8, k=48) == 2                 # Q8_0 needs k % 32
    assert _mm(L, k=0) == 1
    assert _mm(L, n=-1) == 1
    assert _mm(L, W=0) == 1                       # null pointer
    assert _mm(L, W=1032) == 4                    # misaligned
    assert _mm(L, y=4100) == 4
    assert _mm(L, n=0) == 0 and _mm(L, m=0) == 0  # empty problems are no-ops
    P = ctypes.c_void_p
    assert L.qmm_quantize_q8_1(P(1024), 2, 48, P(2048), None) == 2
    assert L.qmm_quantize_q8_1(P(1024), 0, 64, P(2048), None) == 0
    assert L.qmm_quantize_q8_1(P(1028), 2, 64, P(2048), None) == 4
    # mul_mat_id: workspace and expert checks
    args = [P(1024), 12, 4, 8, 256, P(2048), P(4096), 2, 3, P(8192)]
    assert L.qmm_mul_mat_id(*args, None, 0, None) == 5
    ws_need = L.qmm_workspace_bytes(12, 8, 256, 3, 4, 2)
    assert ws_need > 0
    assert L.qmm_mul_mat_id(*args, P(1 << 20), ws_need - 1, None) == 5
    assert L.qmm_mul_mat_id(*args, P((1 << 20) + 16), ws_need, None) == 4
    bad_e = [P(1024), 12, 0, 8, 256, P(2048), P(4096), 2, 3, P(8192)]
    assert L.qmm_mul_mat_id(*bad_e, P(1 << 20), ws_need, None) == 1
    many = [P(1024), 12, 100000, 8, 256, P(2048), P(4096), 2, 3, P(8192)]
    assert L.qmm_mul_mat_id(*many, P(1 << 20), 1 << 40, None) == 2
    # pair counts past 2^31 - 1, including ones whose product overflows int64
    for T_, K in ((1 << 31, 1), (1 << 30, 2), (1 << 62, 4), (3, 1 << 62), (1 << 40, 1 << 40)):
        huge = [P(1024), 12, 4, 8, 256, P(2048), P(4096), K, T_, P(8192)]
        assert L.qmm_mul_mat_id(*huge, P(1 << 20), 1 << 40, None) == 2, (T_, K)


def test_f32_call_argument_errors_need_no_gpu(L):
    P = ctypes.c_void_p

    def mm(W=1024, t=12, n=8, k=256, x=2048, m=4, y=4096, ws=None, wsb=0):
        return L.qmm_mul_mat_f32(P(W), t, n, k, P(x), m, P(y), P(ws) if ws else None, wsb, None)

    assert mm(t=99) == 3
    assert mm(k=100) == 2
    assert mm(t=8, k=48) == 2
    assert mm(x=0) == 1
    assert mm(x=2052) == 4                        # fp32 activations need 16-byte alignment
    assert mm(n=0) == 0 and mm(m=0) == 0
    # m > 8 needs the workspace (q8_1 head + GEMM scratch)
    need = L.qmm_workspace_bytes_f32(12, 8, 256, 20)
    assert need == ((20 * 8 * 36 + 255) // 256) * 256 + L.qmm_workspace_bytes(12, 8, 256, 20, 0, 0)
    assert mm(m=20) == 5
    assert mm(m=20, ws=1 << 20, wsb=need - 1) == 5
    assert mm(m=20, ws=(1 << 20) + 16, wsb=need) == 4
    assert L.qmm_workspace_bytes_f32(12, 8, 100, 20) == 0


def test_tile_efficiency_matches_page_examples():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "schedule_examples.json")))
    for c in g["tile_efficiency"]["cases"]:
        assert qmm.qmm_tile_efficiency_percent(c["ntiles"], c["nsm"]) == c["percent"]


def test_plan_tile_counts_match_prefill_example():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "schedule_examples.json")))["prefill_8k_gate_up"]
    p = qmm.qmm_plan_gemm("q4_K", g["n_rows"], 4096, g["ncols"], 108)
    assert p.tile_n == g["I"] == 128
    assert p.tiles_n == g["row_tiles"]
    assert p.tiles_n * ((g["ncols"] + g["J"] - 1) // g["J"]) == g["tiles"]
    assert p.ntiles == p.tiles_n * p.tiles_m


@pytest.mark.parametrize("n,k,m,nsm,mode", [(14336, 4096, 512, 152, 0), (4100, 4096, 512, 152, 0),
                                            (1024, 2048, 16, 152, 0), (1024, 2048, 16, 152, 2),
                                            (151936, 5120, 512, 152, 0), (1536, 4096, 700, 13, 2),
                                            (5120, 5120, 512, 152, 1)])
def test_plan_partitions_all_work_exactly_once(n, k, m, nsm, mode):
    p = qmm.qmm_plan_gemm("q4_K", n, k, m, nsm, mode)
    eff = qmm.qmm_tile_efficiency_percent(p.ntiles, nsm)
    assert p.efficiency_percent == eff
    assert p.stream_k == (mode == 2 or (mode == 0 and eff < 90))
    covered = 0
    prev_end = 0
    split_tiles = set()
    for c in range(p.ctas):
        b, e = qmm.qmm_plan_cta_range(p, c)
        assert b == prev_end and e >= b
        if b % p.iters_per_tile:
            split_tiles.add(b // p.iters_per_tile)
        prev_end = e
        covered += e - b
    assert covered == p.nwork and prev_end == p.nwork
    assert p.fixup == (len(split_tiles) > 0)
    if p.stream_k:
        assert p.ctas == min(nsm, p.nwork)
        sizes = [qmm.qmm_plan_cta_range(p, c)[1] - qmm.qmm_plan_cta_range(p, c)[0] for c in range(p.ctas)]
        assert max(sizes) - min(sizes) <= 1


# Ring depth of the bulk-copy GEMV: stages of 8 weight rows next to the staged
# activations (ncols units of 64 values, 96 bytes each, plus 1 KB of alignment slack),
# at most 8, and only depths that 4 or 3 consumer groups split into whole stages each.
ROW = {"q4_K": lambda k: k // 256 * 144, "q6_K": lambda k: k // 256 * 210, "q8_0": lambda k: k // 32 * 34,
       "q4_0": lambda k: k // 32 * 18}


def expected_depth(fmt, n, k, ncols, budget):
    rb = ROW[fmt](k)
    if rb % 16 and not (fmt == "q6_K" and rb % 8 == 0 and n % 2 == 0):
        return 0
    fixed = 1024 + ncols * ((k + 63) // 64) * 96
    if fixed >= budget:
        return 0
    st = (budget - fixed) // (8 * rb)
    return max([d for d in (8, 6, 4, 3) if d <= st], default=0)


def test_gemv_ring_depth_whole_rounds(L):
    budget = 227 * 1024
    seen = set()
    for fmt, ks in (("q4_K", range(256, 40000, 256)), ("q6_K", range(256, 30000, 256)),
                    ("q8_0", range(32, 20000, 32)), ("q4_0", range(32, 30000, 32))):
        for k in ks:
            for ncols in (1, 2, 5, 8):
                for n in (4096, 4097):
                    d = qmm.qmm_gemv_ring_stages(fmt, n, k, ncols, budget)
                    assert d in (0, 3, 4, 6, 8), (fmt, n, k, ncols, d)
                    assert d == expected_depth(fmt, n, k, ncols, budget), (fmt, n, k, ncols, d)
                    seen.add(d)
    assert seen == {0, 3, 4, 6, 8}
    # shapes where 3, 5, 6 or 7 stages fit
    assert qmm.qmm_gemv_ring_stages("q4_K", 4096, 14336, 1, budget) == 3
    assert qmm.qmm_gemv_ring_stages("q8_0", 5120, 8192, 1, budget) == 3
    assert qmm.qmm_gemv_ring_stages("q8_0", 5120, 5120, 1, budget) == 4
    assert qmm.qmm_gemv_ring_stages("q6_K", 151936, 5120, 1, budget) == 6
    assert qmm.qmm_gemv_ring_stages("q4_K", 4096, 15616, 1, budget) == 0
    assert qmm.qmm_gemv_ring_stages("q4_K", 17408, 5120, 1, budget) == 8
    # bad arguments
    assert qmm.qmm_gemv_ring_stages("q4_K", 0, 5120, 1, budget) == 0
    assert qmm.qmm_gemv_ring_stages("q4_K", 16, 5000, 1, budget) == 0
    assert qmm.qmm_gemv_ring_stages("q4_K", 16, 5120, 9, budget) == 0


def test_newer_calls_argument_errors_need_no_gpu(L):
    """The fused gate/up calls, the repack, the host-buffer call and the per-slot MoE call
    refuse bad arguments before anything is enqueued."""
    P = ctypes.c_void_p
    # qmm_mul_mat_glu(W_gate, W_up, t, n, k, xq, m, y, ws, ws_bytes, stream)
    glu = lambda Wg=1024, Wu=2048, t=12, n=8, k=256, xq=4096, m=4, y=8192: L.qmm_mul_mat_glu(
        P(Wg), P(Wu), t, n, k, P(xq), m, P(y), None, 0, None)
    assert glu(t=99) == 3 and glu(k=100) == 2 and glu(k=0) == 1 and glu(n=-1) == 1
    assert glu(Wu=0) == 1 and glu(xq=0) == 1 and glu(Wg=1030) == 4 and glu(y=8196) == 4
    assert glu(n=0) == 0 and glu(m=0) == 0
    packed = lambda W=1024, t=12, n=8, k=256, xq=4096, m=4, y=8192: L.qmm_mul_mat_glu_packed(
        P(W), t, n, k, P(xq), m, P(y), None, 0, None)
    assert packed(t=99) == 3 and packed(k=100) == 2 and packed(W=0) == 1 and packed(W=1032) == 4
    assert packed(n=0) == 0 and packed(m=0) == 0
    # qmm_repack_glu(W_gate, W_up, t, n, k, W_gu, stream)
    rp = lambda Wg=1024, Wu=2048, t=12, n=8, k=256, out=4096: L.qmm_repack_glu(P(Wg), P(Wu), t, n, k, P(out), None)
    assert rp(t=99) == 3 and rp(t=2, k=48) == 2 and rp(out=0) == 1 and rp(Wu=2056) == 4 and rp(n=0) == 0
    # qmm_mul_mat_f32_host(W, t, n, k, x_host, m, y_host, ws, ws_bytes, stream)
    host = lambda W=1024, t=12, n=8, k=256, x=4096, m=2, y=8192, ws=None, wsb=0: L.qmm_mul_mat_f32_host(
        P(W), t, n, k, P(x), m, P(y), P(ws) if ws else None, wsb, None)
    assert host(t=99) == 3 and host(k=100) == 2 and host(x=0) == 1 and host(y=0) == 1
    assert host(W=1028) == 4 and host(n=0) == 0 and host(m=0) == 0
    need = L.qmm_workspace_bytes_f32_host(12, 8, 256, 2)
    assert need >= 2 * 256 and host(ws=1 << 20, wsb=need - 1) == 5 and host(ws=(1 << 20) + 16, wsb=need) == 4
    # qmm_mul_mat_id_slot: the same checks as qmm_mul_mat_id
    args = [P(1024), 12, 4, 8, 256, P(2048), P(4096), 2, 3, P(8192)]
    assert L.qmm_mul_mat_id_slot(*args, None, 0, None) == 5
    bad_t = [P(1024), 99, 4, 8, 256, P(2048), P(4096), 2, 3, P(8192)]
    assert L.qmm_mul_mat_id_slot(*bad_t, None, 0, None) == 3


def test_q4_0_sizes_and_shapes(L):
    assert qmm.qmm_row_bytes("q4_0", 4096) == 128 * 18
    assert qmm.qmm_q8_1_bytes(3, 4096) == 3 * 128 * 36
    P = ctypes.c_void_p
    # k must be a multiple of the 32-value block
    assert L.qmm_mul_mat(P(1024), 2, 8, 48, P(2048), 4, P(4096), None, 0, None) == 2


def test_aligned_row_bytes_matches_oracle(oracle_mod):
    for fmt, k in [("q6_K", 5120), ("q6_K", 256), ("q8_0", 5120), ("q8_0", 96), ("q4_0", 224), ("q4_K", 4096)]:
        assert qmm.qmm_aligned_row_bytes(fmt, k) == oracle_mod.aligned_row_bytes(fmt, k)
    assert qmm.qmm_aligned_row_bytes("q6_K", 100) == 0  # not a whole number of blocks
