// qmm_gemv_tc.cu -- tensor-core path for skinny activations (1 <= m <= 16), Q4_K.
//
// What it computes is the tiled GEMM's exact-integer fold ([MMQ] sections "dp4a 路径的
// Q4_K" and "输出端"): per 32-wide sub-block an exact integer dot (kind::f16 MMA on
// integer-valued fp16 operands, exact in the fp32 accumulator), folded in fp32 with d8,
// then d * acc - dmin * sum_b m_b s_b per superblock.
//
// The roles of the operands are swapped against the tiled GEMM: the 128 weight rows of
// a tile are the MMA's M side (TMEM lanes) and the m <= 16 activation rows its N side
// (16 TMEM columns per accumulator), so the per-element fold is 16 columns wide instead
// of 128 and the cost per weight byte is the nibble unpack, not the epilogue
// ([P0007] section "How": for 2..8 columns the weights are decoded once and reused
// for every column; [MMQ] "与 MMVQ 的边界": the weight is read once, the bound is HBM).
//
// Work is the flattened stream of (128-row tile, superblock) units split evenly over one
// CTA per SM ([MMQ] section "stream-K 的切法"); tiles shared by CTAs are summed by a fixup
// kernel in CTA order.  The same kernel serves the cold experts of an expert-routed
// matmul ([MMQ] section "MoE 的二次账": experts with a few pairs leave wide tiles mostly
// empty): a tile is then (cold expert, 128 weight rows of it), its 16 columns that
// expert's pairs, gathered into a 16-row slab, and its outputs go to the pairs' rows;
// the list of cold experts and its length are read on the device.  16 warps:
//   warp 0      TMA: fp16 activation slabs (128-byte swizzle, 8 half-superblocks in
//               flight, since they come from L2 and every superblock needs new ones), the
//               s tile of the min term, and d8 per superblock (transposed:
//               [sub-block][token]).
//   warp 1      TMEM allocation; one lane issues the MMAs: per superblock 8 sub-blocks
//               of two K=16 MMAs each (A, the weights, read from TMEM; B, the
//               activations, from shared memory) into 8 accumulator slots, plus one K=16
//               MMA for sum_b min * s; slots form a ring of 2 superblocks.
//   warp 2      TMA: raw Q4_K superblocks of the tile's 128 rows, an 8-deep ring (the HBM
//               stream).
//   warps 4-11  unpack, two groups of 4 warps: group h converts half h of every
//               superblock, one weight row per thread, and stores it with tcgen05.st into
//               that row's TMEM lane (the MMA's A operand: fp16 pairs along the columns),
//               so the unpacked weights never pass through shared memory; group 1 also
//               writes the fp16 mins (shared memory), group 0 (d, -dmin) for the epilogue.
//               A group hands a half to the MMA only once that half's activation slabs
//               have landed too, so the MMA thread observes one barrier per half (each
//               completion it waits for idles the tensor pipe for a few hundred cycles).
//   warps 12-15 epilogue: one weight row per thread, 16 activation columns, the running
//               sums in registers.
// Every wait is bounded (qmm_tc_ptx.cuh); a wait that gives up raises the CTA's abort
// flag, the roles leave their loops, copies in flight are drained and TMEM is freed.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_tc_common.cuh"
#include "qmm_tc_ptx.cuh"

namespace qmm {

namespace {

constexpr int kRows = 128;        // weight rows per tile: MMA M, TMEM lanes
constexpr int kNT = 16;           // activation rows per tile: MMA N, TMEM columns per slot
constexpr int kMaxM = kNT;
constexpr int kRawStages = 8;
constexpr int kXStages = 8;       // activation half-superblocks in flight (they come from L2)
constexpr int kSdRing = 4;        // superblocks of d8 / (d, -dmin) in flight
constexpr int kSbRing = 2;        // superblocks of accumulator slots in TMEM
constexpr int kSlotsPerSb = 9;    // 8 sub-blocks + the min term
constexpr int kThreads = 512;
constexpr int kUnpackWarp0 = 4;
constexpr int kEpiWarp0 = 12;
constexpr int kEpiWarps = 4;
constexpr int kMaxPartialCtas = 256;
// TMEM columns: a ring of kABufs half-superblocks of unpacked weights (the MMA's A
// operand, 64 columns of fp16 pairs each), then the accumulator slots
constexpr uint32_t kAColsHalf = 64;
constexpr int kABufs = 3;
constexpr uint32_t kSlotCol0 = kABufs * kAColsHalf;
static_assert(kSlotCol0 + kSbRing * kSlotsPerSb * kNT <= 512, "accumulator ring exceeds TMEM");

// dynamic shared memory map (offsets from a 1024-aligned base)
constexpr uint32_t kXSlab = kNT * 128;                        // 16 rows x 64 fp16
constexpr uint32_t kOffX = 0;                                 // [kXStages][2 slabs]
constexpr uint32_t kOffWmin = kOffX + kXStages * 2 * kXSlab;  // [2][128][32 B], by superblock parity
constexpr uint32_t kOffXmin = kOffWmin + 2 * kRows * 32;      // [kSdRing][16][32 B]
constexpr uint32_t kOffDX = kOffXmin + kSdRing * kNT * 32;    // [kSdRing][8][16] fp32
constexpr uint32_t kDXBytes = 8 * kNT * 4;
constexpr uint32_t kOffDD = kOffDX + kSdRing * kDXBytes;      // [kSdRing][d[128], -dmin[128]] fp32
constexpr uint32_t kDDBytes = 2 * kRows * 4;
constexpr uint32_t kRawBytes = kRows * kQ4KBytes;
constexpr uint32_t kOffRaw = (kOffDD + kSdRing * kDDBytes + 1023) & ~1023u;
constexpr uint32_t kSmemBytes = kOffRaw + kRawStages * kRawBytes;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 227 * 1024, "shared memory map exceeds the per-CTA limit");

struct SkArgs {
    int64_t n;      // weight rows (grouped: per expert)
    int m;          // activation rows (1..16)
    int64_t nsb;    // superblocks per row
    int64_t ntiles; // 128-row tiles (grouped: per expert)
    int64_t nwork;  // ntiles * nsb (grouped: set in the kernel from *ncold)
    int ctas;
    float *y;       // [m][n] (grouped: [pairs][n])
    float *partial; // [ctas][2][128][16]
    int *status;
    // Expert-grouped mode (cold != nullptr, MoE experts with 1..16 pairs): tile c * ntiles
    // + t is the 128-row tile t of expert cold[c]; its activations are the 16-row slab c
    // of the gathered buffers, its output column j < count the pair perm[bounds[e] + j].
    const int32_t *cold;
    const int32_t *ncold;
    const int32_t *bounds;
    const int32_t *perm;
};

// What a tile addresses: the first W row (in the map over all experts' rows), the first
// row of its activation slab and of its d8 rows, and the output columns it holds.
struct SkTile {
    int64_t wrow0, xrow0, dxrow0;
    int64_t row0;   // first weight row within its expert (the output feature)
    int cols;       // valid activation columns
    int32_t pair0;  // grouped: offset of the expert's pairs in perm
};
// the y row of activation column j of a tile: j itself, or its pair
__device__ __forceinline__ int64_t sk_out_row(const SkArgs &a, const SkTile &tt, int j) {
    return a.cold ? int64_t(a.perm[tt.pair0 + j]) : int64_t(j);
}
__device__ __forceinline__ SkTile sk_tile(const SkArgs &a, int64_t tile) {
    SkTile r;
    if (!a.cold) {
        r.wrow0 = r.row0 = tile * kRows;
        r.xrow0 = r.dxrow0 = 0;
        r.cols = a.m;
        r.pair0 = 0;
        return r;
    }
    const int64_t c = tile / a.ntiles, t = tile - c * a.ntiles;
    const int e = a.cold[c];
    r.row0 = t * kRows;
    r.wrow0 = int64_t(e) * a.n + r.row0;
    r.xrow0 = c * kNT;
    r.dxrow0 = c * (a.nsb * 8);
    r.pair0 = a.bounds[e];
    r.cols = a.bounds[e + 1] - r.pair0;
    return r;
}

struct Barriers {
    uint64_t x_full[kXStages], x_empty[kXStages], w_full[kABufs], w_empty[kABufs];
    uint64_t raw_full[kRawStages], raw_empty[kRawStages];
    uint64_t sd_full[kSdRing], sd_empty[kSdRing];
    uint64_t acc_full[kSbRing], acc_empty[kSbRing];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void cta_range(const SkArgs &a, int cta, int64_t &b, int64_t &e) {
    b = a.nwork * cta / a.ctas;
    e = a.nwork * (cta + 1) / a.ctas;
}

// the segments of a CTA's unit range: (tile, s0, s1), superblocks s0 <= s < s1
struct Seg {
    int64_t tile, s0, s1;
};
__device__ __forceinline__ bool next_seg(const SkArgs &a, int64_t &u, int64_t end, Seg &sg) {
    if (u >= end) return false;
    sg.tile = u / a.nsb;
    sg.s0 = u - sg.tile * a.nsb;
    sg.s1 = min(a.nsb, sg.s0 + (end - u));
    u += sg.s1 - sg.s0;
    return true;
}

__device__ __forceinline__ uint32_t slot_col(uint32_t sbs, int G) { return kSlotCol0 + (sbs * kSlotsPerSb + G) * kNT; }

__global__ void __launch_bounds__(kThreads, 1)
    gemv_tc_q4k_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xmin,
                       const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_w,
                       const SkArgs a_in) {
    SkArgs a = a_in;
    if (a.cold) {
        // the cold list and the gathered activations come from the preceding kernels
        ptx::grid_dependency_wait();
        a.nwork = int64_t(*a.ncold) * a.ntiles * a.nsb;
    }
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ Barriers B;
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);  // stays a shared pointer
    const uint32_t sbase = ptx::smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abortp = &B.abort;

    if (tid == 0) {
        B.abort = 0;
        for (int s = 0; s < kABufs; ++s) {
            ptx::mbar_init(ptx::smem_u32(&B.w_full[s]), kRows);
            ptx::mbar_init(ptx::smem_u32(&B.w_empty[s]), 1);
        }
        for (int s = 0; s < kXStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&B.x_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&B.x_empty[s]), 1);
        }
        for (int s = 0; s < kSdRing; ++s) {
            ptx::mbar_init(ptx::smem_u32(&B.sd_full[s]), 1 + kRows);
            ptx::mbar_init(ptx::smem_u32(&B.sd_empty[s]), kEpiWarps);
        }
        for (int s = 0; s < kRawStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&B.raw_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&B.raw_empty[s]), 2 * kRows);
        }
        for (int s = 0; s < kSbRing; ++s) {
            ptx::mbar_init(ptx::smem_u32(&B.acc_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&B.acc_empty[s]), kEpiWarps);
        }
        ptx::mbar_init(ptx::smem_u32(&B.done), 1);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&B.tmem_base), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = B.tmem_base;

    int64_t ubeg, uend;
    cta_range(a, blockIdx.x, ubeg, uend);

    if (warp == 0) {
        // ------------------------------------------------------------ activation TMA
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_x);
            ptx::prefetch_tmap(&tm_xmin);
            ptx::prefetch_tmap(&tm_dx);
            // the activations were written by the preceding kernel (the prep pass)
            ptx::grid_dependency_wait();
            int64_t u = ubeg;
            Seg sg;
            uint32_t sbc = 0;
            bool ok = true;
            while (ok && next_seg(a, u, uend, sg)) {
                const SkTile tt = sk_tile(a, sg.tile);
                for (int64_t sb = sg.s0; ok && sb < sg.s1; ++sb, ++sbc) {
                    const uint32_t sdi = sbc % kSdRing, ph = (sbc / kSdRing) & 1;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.sd_empty[sdi]), ph ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sdbar = ptx::smem_u32(&B.sd_full[sdi]);
                    ptx::mbar_arrive_expect_tx(sdbar, kDXBytes);
                    ptx::tma_load_2d(sbase + kOffDX + sdi * kDXBytes, &tm_dx, 0, (int)(tt.dxrow0 + 8 * sb), sdbar);
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t xi = (2 * sbc + h) % kXStages, xph = ((2 * sbc + h) / kXStages) & 1;
                        if (!ptx::mbar_wait(ptx::smem_u32(&B.x_empty[xi]), xph ^ 1, abortp)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bar = ptx::smem_u32(&B.x_full[xi]);
                        ptx::mbar_arrive_expect_tx(bar, 2 * kXSlab + (h ? kNT * 32u : 0u));
                        const int kx = (int)(256 * sb + 128 * h);
                        const int xr = (int)tt.xrow0;
                        ptx::tma_load_2d(sbase + kOffX + xi * 2 * kXSlab, &tm_x, kx, xr, bar);
                        ptx::tma_load_2d(sbase + kOffX + xi * 2 * kXSlab + kXSlab, &tm_x, kx + 64, xr, bar);
                        if (h) ptx::tma_load_2d(sbase + kOffXmin + sdi * (kNT * 32), &tm_xmin, (int)(16 * sb), xr, bar);
                    }
                }
            }
            // drain: every armed copy must have landed before the CTA may exit
            int dummy = 0;
            const uint32_t nx = 2 * sbc;
            for (uint32_t i = (nx > kXStages ? nx - kXStages : 0); i < nx; ++i)
                ptx::mbar_wait(ptx::smem_u32(&B.x_full[i % kXStages]), (i / kXStages) & 1, &dummy);
            for (uint32_t i = (sbc > kSdRing ? sbc - kSdRing : 0); i < sbc; ++i)
                ptx::mbar_wait(ptx::smem_u32(&B.sd_full[i % kSdRing]), (i / kSdRing) & 1, &dummy);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_f16_f32(kRows, kNT);
            int64_t u = ubeg;
            Seg sg;
            uint32_t sbc = 0;
            bool ok = true;
            while (ok && next_seg(a, u, uend, sg)) {
                for (int64_t sb = sg.s0; ok && sb < sg.s1; ++sb, ++sbc) {
                    const uint32_t sbs = sbc % kSbRing, aph = (sbc / kSbRing) & 1;
                    if (!ptx::mbar_wait_spin(ptx::smem_u32(&B.acc_empty[sbs]), aph ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    for (int h = 0; ok && h < 2; ++h) {
                        const uint32_t xi = (2 * sbc + h) % kXStages;
                        const uint32_t ai = (2 * sbc + h) % kABufs, aph2 = ((2 * sbc + h) / kABufs) & 1;
                        // w_full covers the activation half too: its unpack group waited for it
                        if (!ptx::mbar_wait_spin(ptx::smem_u32(&B.w_full[ai]), aph2, abortp)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        // descriptors of the two activation slabs, built once; a K16 step of 32
                        // bytes inside the 128-byte swizzled row adds 2 to the start-address field
                        const uint64_t xd0 = ptx::smem_desc(sbase + kOffX + xi * 2 * kXSlab, 1024, 2);
                        const uint64_t xd1 = ptx::smem_desc(sbase + kOffX + xi * 2 * kXSlab + kXSlab, 1024, 2);
                        const uint32_t dcol = tmem + slot_col(sbs, 4 * h), acol = tmem + ai * kAColsHalf;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {  // sub-block 4h + q: K = 128h + 32q ..
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                const uint32_t kstep = (q & 1) * 2 + t;  // K16 step in the 128-byte row
                                ptx::mma_f16_tmem_a(dcol + kNT * q, acol + 16 * q + 8 * t,
                                                    ((q >> 1) ? xd1 : xd0) + 2 * kstep, idesc, t);
                            }
                        }
                        if (h == 1)
                            ptx::mma_f16(tmem + slot_col(sbs, 8),
                                         ptx::smem_desc(sbase + kOffWmin + (sbc & 1) * (kRows * 32), 256, 6),
                                         ptx::smem_desc(sbase + kOffXmin + (sbc % kSdRing) * (kNT * 32), 256, 6),
                                         idesc, 0);
                        ptx::mma_commit(ptx::smem_u32(&B.x_empty[xi]));
                        ptx::mma_commit(ptx::smem_u32(&B.w_empty[ai]));
                    }
                    if (ok) ptx::mma_commit(ptx::smem_u32(&B.acc_full[sbs]));
                }
            }
            // every MMA must be complete before TMEM is freed
            ptx::mma_commit(ptx::smem_u32(&B.done));
            int dummy = 0;
            ptx::mbar_wait(ptx::smem_u32(&B.done), 0, &dummy);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ raw weight TMA
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_w);
            int64_t u = ubeg;
            Seg sg;
            uint32_t r_it = 0;
            bool ok = true;
            while (ok && next_seg(a, u, uend, sg)) {
                const int n0 = (int)sk_tile(a, sg.tile).wrow0;
                for (int64_t sb = sg.s0; sb < sg.s1; ++sb, ++r_it) {
                    const uint32_t ri = r_it % kRawStages, ph = (r_it / kRawStages) & 1;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.raw_empty[ri]), ph ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    const uint32_t rbar = ptx::smem_u32(&B.raw_full[ri]);
                    ptx::mbar_arrive_expect_tx(rbar, kRawBytes);
                    ptx::tma_load_2d(sbase + kOffRaw + ri * kRawBytes, &tm_w, (int)(sb * kQ4KBytes), n0, rbar);
                }
            }
            int dummy = 0;
            for (uint32_t i = (r_it > kRawStages ? r_it - kRawStages : 0); i < r_it; ++i)
                ptx::mbar_wait(ptx::smem_u32(&B.raw_full[i % kRawStages]), (i / kRawStages) & 1, &dummy);
        }
    } else if (warp == 3) {
        // no role
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------ weight unpack
        const int h = (warp - kUnpackWarp0) >> 2;            // half of every superblock
        const int r = tid - 32 * kUnpackWarp0 - kRows * h;   // weight row within the tile
        int64_t u = ubeg;
        Seg sg;
        uint32_t sbc = 0;
        bool ok = true;
        while (ok && next_seg(a, u, uend, sg)) {
            for (int64_t sb = sg.s0; ok && sb < sg.s1; ++sb, ++sbc) {
                const uint32_t ri = sbc % kRawStages;
                if (!ptx::mbar_wait(ptx::smem_u32(&B.raw_full[ri]), (sbc / kRawStages) & 1, abortp)) {
                    ok = false;
                    break;
                }
                const uint8_t *blk = smem + kOffRaw + ri * kRawBytes + r * kQ4KBytes;
                const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
                if (h == 0) {  // (d, -dmin) for the epilogue
                    const uint32_t sdi = sbc % kSdRing;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.sd_empty[sdi]), ((sbc / kSdRing) & 1) ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    float *dd = reinterpret_cast<float *>(smem + kOffDD + sdi * kDDBytes);
                    dd[r] = half_lo(hd.x);
                    dd[kRows + r] = -half_hi(hd.x);
                    ptx::mbar_arrive(ptx::smem_u32(&B.sd_full[sdi]));
                }
                const uint32_t ai = (2 * sbc + h) % kABufs;
                if (!ptx::mbar_wait(ptx::smem_u32(&B.w_empty[ai]), (((2 * sbc + h) / kABufs) & 1) ^ 1, abortp)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();  // after the MMAs that read the previous contents
                // this thread's row is TMEM lane r: the warp's lane quarter is r / 32 = warp % 4
                const uint32_t arow = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + ai * kAColsHalf;
#pragma unroll
                for (int j2 = 0; j2 < 2; ++j2) {  // qs chunk c = 2h + j2: sub-blocks 2c (low), 2c+1 (high)
                    const int c = 2 * h + j2;
                    const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
                    const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
                    int sc_lo, m_lo, sc_hi, m_hi;
                    q4k_scale_min(hd.y, hd.z, hd.w, 2 * c, sc_lo, m_lo);
                    q4k_scale_min(hd.y, hd.z, hd.w, 2 * c + 1, sc_hi, m_hi);
                    const __half2 s_lo = __float2half2_rn((float)sc_lo), ns_lo = __float2half2_rn(-1024.f * sc_lo);
                    const __half2 s_hi = __float2half2_rn((float)sc_hi), ns_hi = __float2half2_rn(-1024.f * sc_hi);
                    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                    uint32_t lo[16], hi[16];  // 32 fp16 values each, two per column
#pragma unroll
                    for (int cq = 0; cq < 4; ++cq) {
                        const uint4 l4 = nibbles_to_f16(w[2 * cq], w[2 * cq + 1], 0, s_lo, ns_lo);
                        const uint4 h4 = nibbles_to_f16(w[2 * cq], w[2 * cq + 1], 4, s_hi, ns_hi);
                        lo[4 * cq] = l4.x; lo[4 * cq + 1] = l4.y; lo[4 * cq + 2] = l4.z; lo[4 * cq + 3] = l4.w;
                        hi[4 * cq] = h4.x; hi[4 * cq + 1] = h4.y; hi[4 * cq + 2] = h4.z; hi[4 * cq + 3] = h4.w;
                    }
                    ptx::tmem_st_32x32b_x16(arow + 32 * j2, lo);
                    ptx::tmem_st_32x32b_x16(arow + 32 * j2 + 16, hi);
                }
                if (h == 1) {  // mins of the 8 sub-blocks as fp16, then 8 zeros (32-byte swizzle)
                    uint32_t mm[4];
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2) {
                        int s0_, m0_, s1_, m1_;
                        q4k_scale_min(hd.y, hd.z, hd.w, 2 * i2, s0_, m0_);
                        q4k_scale_min(hd.y, hd.z, hd.w, 2 * i2 + 1, s1_, m1_);
                        mm[i2] = h2bits(__floats2half2_rn((float)m0_, (float)m1_));
                    }
                    // by superblock parity: this group may write superblock s+1's mins while
                    // the MMA of superblock s is still to read its own (the A ring lets it
                    // run one half ahead); the buffer of s-1 is free, since the use of the
                    // A buffer waited for the MMAs of (s, half 0), issued after (s-1, half 1)
                    uint8_t *mdst = smem + kOffWmin + (sbc & 1) * (kRows * 32) + r * 32;
                    const int sw = (r >> 2) & 1;
                    *reinterpret_cast<uint4 *>(mdst + ((0 ^ sw) << 4)) = make_uint4(mm[0], mm[1], mm[2], mm[3]);
                    *reinterpret_cast<uint4 *>(mdst + ((1 ^ sw) << 4)) = make_uint4(0, 0, 0, 0);
                }
                ptx::tmem_st_wait();
                ptx::fence_proxy_async_smem();  // the mins are read by the MMA (async proxy)
                ptx::tc_fence_before();
                // The MMA thread waits only on w_full, so the group first waits for this half's
                // activation slabs (and, for half 1, the s tile): group h alone waits on the
                // x barriers of the halves 2s + h, since the x ring is 8 deep.
                {
                    const uint32_t xi = (2 * sbc + h) % kXStages, xph = ((2 * sbc + h) / kXStages) & 1;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.x_full[xi]), xph, abortp)) {
                        ok = false;
                        break;
                    }
                }
                ptx::mbar_arrive(ptx::smem_u32(&B.w_full[ai]));
                ptx::mbar_arrive(ptx::smem_u32(&B.raw_empty[ri]));
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // warp w reads TMEM lanes 32*(w%4).. : one weight row per thread, 16 columns.
        const int qd = warp & 3;
        const int tl = 32 * qd + lane;  // weight row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        int64_t u = ubeg;
        Seg sg;
        uint32_t sbc = 0;
        int seg_i = 0;
        bool ok = true;
        while (ok && next_seg(a, u, uend, sg)) {
            float2 tot[kNT / 2];
#pragma unroll
            for (int i = 0; i < kNT / 2; ++i) tot[i] = make_float2(0.f, 0.f);
            for (int64_t sb = sg.s0; ok && sb < sg.s1; ++sb, ++sbc) {
                const uint32_t sdi = sbc % kSdRing, sbs = sbc % kSbRing;
                if (!ptx::mbar_wait(ptx::smem_u32(&B.sd_full[sdi]), (sbc / kSdRing) & 1, abortp) ||
                    !ptx::mbar_wait(ptx::smem_u32(&B.acc_full[sbs]), (sbc / kSbRing) & 1, abortp)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const float4 *dx = reinterpret_cast<const float4 *>(smem + kOffDX + sdi * kDXBytes);
                const float *dd = reinterpret_cast<const float *>(smem + kOffDD + sdi * kDDBytes);
                const float d = dd[tl], nd = dd[kRows + tl];
                float2 acc[kNT / 2];
#pragma unroll
                for (int i = 0; i < kNT / 2; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
                for (int G = 0; G < 8; ++G) {
                    float v[16];
                    ptx::tmem_ld_32x32b_x16(lane_base + slot_col(sbs, G), v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i4 = 0; i4 < kNT / 4; ++i4) {  // d8 of sub-block G, columns 4 i4 .. 4 i4 + 3
                        const float4 s4 = dx[G * (kNT / 4) + i4];
                        acc[2 * i4] = __ffma2_rn(make_float2(s4.x, s4.y), make_float2(v[4 * i4], v[4 * i4 + 1]),
                                                 acc[2 * i4]);
                        acc[2 * i4 + 1] = __ffma2_rn(make_float2(s4.z, s4.w),
                                                     make_float2(v[4 * i4 + 2], v[4 * i4 + 3]), acc[2 * i4 + 1]);
                    }
                }
                float vm[16];
                ptx::tmem_ld_32x32b_x16(lane_base + slot_col(sbs, 8), vm);
                ptx::tmem_ld_wait();
                // tot += d * acc - dmin * sum_b m_b s_b
#pragma unroll
                for (int i = 0; i < kNT / 2; ++i)
                    tot[i] = __ffma2_rn(make_float2(nd, nd), make_float2(vm[2 * i], vm[2 * i + 1]),
                                        __ffma2_rn(make_float2(d, d), acc[i], tot[i]));
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(ptx::smem_u32(&B.acc_empty[sbs]));
                    ptx::mbar_arrive(ptx::smem_u32(&B.sd_empty[sdi]));
                }
            }
            if (!ok) break;
            // the segment's result: whole tile -> y, part of a tile -> this CTA's partial slot
            const bool full = sg.s0 == 0 && sg.s1 == a.nsb;
            if (full) {
                const SkTile tt = sk_tile(a, sg.tile);
                const int64_t row = tt.row0 + tl;
                if (row < a.n) {
#pragma unroll
                    for (int i = 0; i < kNT / 2; ++i) {
                        if (2 * i < tt.cols) a.y[sk_out_row(a, tt, 2 * i) * a.n + row] = tot[i].x;
                        if (2 * i + 1 < tt.cols) a.y[sk_out_row(a, tt, 2 * i + 1) * a.n + row] = tot[i].y;
                    }
                }
            } else {
                const int slotidx = seg_i == 0 ? 0 : 1;
                float4 *dst = reinterpret_cast<float4 *>(
                    a.partial + ((int64_t(blockIdx.x) * 2 + slotidx) * kRows + tl) * kNT);
#pragma unroll
                for (int i4 = 0; i4 < kNT / 4; ++i4)
                    dst[i4] = make_float4(tot[2 * i4].x, tot[2 * i4].y, tot[2 * i4 + 1].x, tot[2 * i4 + 1].y);
            }
            ++seg_i;
        }
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, 512);
    if (tid == 0 && B.abort && a.status) atomicExch(a.status, (int)QMM_ERR_DEVICE);
}

// q8_1 blocks -> fp16 activation codes [m][k], fp16 s tile [m][k/256][16] (8 values
// then 8 zeros), and d8 transposed and padded to 16 columns, [k/32][16] (zeros for the
// rows m..15).
__global__ void gemv_tc_prep_kernel(const uint8_t *__restrict__ xq, int m, int k, __half *__restrict__ xh,
                                    __half *__restrict__ smin, float *__restrict__ dxt, int *status) {
    // xq may have been written by the preceding kernel (the quantizer)
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    const int nb32 = k / 32;
    const int64_t total = int64_t(kNT) * nb32;
    if (blockIdx.x == 0 && threadIdx.x == 0 && status) *status = (int)QMM_OK;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int b = (int)(i / kNT), r = (int)(i - int64_t(b) * kNT);
        if (r >= m) {
            dxt[i] = 0.f;
            continue;
        }
        const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + (int64_t(r) * nb32 + b) * kQ81Bytes);
        const uint32_t dsw = ldg4(src);
        uint4 *dst = reinterpret_cast<uint4 *>(xh + int64_t(r) * k + 32 * b);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t w0 = ldg4(src + 1 + 2 * j), w1 = ldg4(src + 2 + 2 * j);
            const int8_t *c0 = reinterpret_cast<const int8_t *>(&w0);
            const int8_t *c1 = reinterpret_cast<const int8_t *>(&w1);
            uint4 o;
            o.x = h2bits(__halves2half2(__int2half_rn(c0[0]), __int2half_rn(c0[1])));
            o.y = h2bits(__halves2half2(__int2half_rn(c0[2]), __int2half_rn(c0[3])));
            o.z = h2bits(__halves2half2(__int2half_rn(c1[0]), __int2half_rn(c1[1])));
            o.w = h2bits(__halves2half2(__int2half_rn(c1[2]), __int2half_rn(c1[3])));
            dst[j] = o;
        }
        dxt[i] = half_lo(dsw);
        __half *sp = smin + (int64_t(r) * (nb32 / 8) + b / 8) * 16;
        sp[b % 8] = __ushort_as_half((unsigned short)(dsw >> 16));
        sp[8 + b % 8] = __ushort_as_half(0);
    }
}

// The same for the cold experts of an expert-grouped call: slab c (rows 16c .. 16c+15 of
// xh and smin, d8 rows c*k/32 .. of dxt) holds the activation rows of expert cold[c]'s
// pairs in their sorted order, zeros past its pair count.  Activation row of pair p:
// xq row p / x_div.
__global__ void gemv_tc_prep_grouped_kernel(const uint8_t *__restrict__ xq, int64_t x_div, int k,
                                            const int32_t *__restrict__ cold, const int32_t *__restrict__ ncold,
                                            const int32_t *__restrict__ bounds, const int32_t *__restrict__ perm,
                                            __half *__restrict__ xh, __half *__restrict__ smin,
                                            float *__restrict__ dxt) {
    // the pair lists come from the bucketing kernel before this one
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    const int nb32 = k / 32;
    const int64_t per_slot = int64_t(kNT) * nb32;
    const int64_t total = int64_t(*ncold) * per_slot;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t c = i / per_slot, rem = i - c * per_slot;
        const int b = (int)(rem / kNT), r = (int)(rem - int64_t(b) * kNT);
        const int e = cold[c];
        const int cnt = bounds[e + 1] - bounds[e];
        const int64_t xr = c * kNT + r;  // row of the gathered buffers
        uint4 *dst = reinterpret_cast<uint4 *>(xh + xr * k + 32 * b);
        __half *sp = smin + (xr * (nb32 / 8) + b / 8) * 16;
        if (r >= cnt) {
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(0u, 0u, 0u, 0u);
            dxt[i] = 0.f;
            sp[b % 8] = __ushort_as_half(0);
            sp[8 + b % 8] = __ushort_as_half(0);
            continue;
        }
        const int64_t row = int64_t(perm[bounds[e] + r]) / x_div;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + (row * nb32 + b) * kQ81Bytes);
        const uint32_t dsw = ldg4(src);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t w0 = ldg4(src + 1 + 2 * j), w1 = ldg4(src + 2 + 2 * j);
            const int8_t *c0 = reinterpret_cast<const int8_t *>(&w0);
            const int8_t *c1 = reinterpret_cast<const int8_t *>(&w1);
            uint4 o;
            o.x = h2bits(__halves2half2(__int2half_rn(c0[0]), __int2half_rn(c0[1])));
            o.y = h2bits(__halves2half2(__int2half_rn(c0[2]), __int2half_rn(c0[3])));
            o.z = h2bits(__halves2half2(__int2half_rn(c1[0]), __int2half_rn(c1[1])));
            o.w = h2bits(__halves2half2(__int2half_rn(c1[2]), __int2half_rn(c1[3])));
            dst[j] = o;
        }
        dxt[i] = half_lo(dsw);
        sp[b % 8] = __ushort_as_half((unsigned short)(dsw >> 16));
        sp[8 + b % 8] = __ushort_as_half(0);
    }
}

// stream-K fixup: every tile that several CTAs share is summed in CTA order; one thread
// per weight row, 16 columns.
__global__ void __launch_bounds__(kRows) gemv_tc_fixup_kernel(const SkArgs a_in) {
    SkArgs a = a_in;
    int64_t ntiles = gridDim.x;  // dense: one block per tile
    if (a.cold) {                // grouped: the cold experts' tiles, counted on the device
        ntiles = int64_t(*a.ncold) * a.ntiles;
        a.nwork = ntiles * a.nsb;
    }
    auto owner = [&](int64_t uu) {
        int64_t c = uu * a.ctas / a.nwork;
        while (c + 1 < a.ctas && a.nwork * (c + 1) / a.ctas <= uu) ++c;
        while (c > 0 && a.nwork * c / a.ctas > uu) --c;
        return c;
    };
    const int tl = threadIdx.x;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t u0 = t * a.nsb, u1 = u0 + a.nsb - 1;
        const int64_t c0 = owner(u0), c1 = owner(u1);
        if (c0 == c1) continue;  // the tile was written whole by one CTA
        float s[kNT];
#pragma unroll
        for (int i = 0; i < kNT; ++i) s[i] = 0.f;
        for (int64_t c = c0; c <= c1; ++c) {
            const int64_t cb = a.nwork * c / a.ctas;
            if (a.nwork * (c + 1) / a.ctas == cb) continue;  // c owns no units
            const int slotidx = (cb / a.nsb == t) ? 0 : 1;   // tile t is this CTA's first segment?
            const float4 *p = reinterpret_cast<const float4 *>(a.partial + ((c * 2 + slotidx) * kRows + tl) * kNT);
#pragma unroll
            for (int i4 = 0; i4 < kNT / 4; ++i4) {
                const float4 v = p[i4];
                s[4 * i4] += v.x;
                s[4 * i4 + 1] += v.y;
                s[4 * i4 + 2] += v.z;
                s[4 * i4 + 3] += v.w;
            }
        }
        const SkTile tt = sk_tile(a, t);
        const int64_t row = tt.row0 + tl;
        if (row >= a.n) continue;
#pragma unroll
        for (int i = 0; i < kNT; ++i)
            if (i < tt.cols) a.y[sk_out_row(a, tt, i) * a.n + row] = s[i];
    }
}

struct SkLayout {
    size_t status, xh, smin, dxt, partial, total;
};
SkLayout sk_layout(int64_t m, int64_t k, int64_t ctas) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    SkLayout L{};
    size_t off = 256;
    L.status = 0;
    L.xh = off;
    off = al(off + size_t(m) * k * 2);
    L.smin = off;
    off = al(off + size_t(m) * (k / 256) * 32);
    L.dxt = off;
    off = al(off + size_t(k / 32) * kNT * 4);
    L.partial = off;
    off = al(off + size_t(ctas) * 2 * kRows * kNT * 4);
    L.total = off;
    return L;
}

int sk_ctas(int64_t n, int64_t k) {
    const int64_t nwork = ((n + kRows - 1) / kRows) * (k / 256);
    return (int)std::min<int64_t>(std::min<int64_t>(device_sm_count(), kMaxPartialCtas), nwork);
}

}  // namespace

bool gemv_tc_grouped_supported(qmm_type t, int64_t n_experts, int64_t n, int64_t k) {
    // TMA coordinates are 32-bit: the map over all experts' rows and the gathered slabs
    return t == QMM_Q4_K && k % 256 == 0 && n > 0 && n_experts > 0 && n_experts * n < (int64_t(1) << 31) &&
           n_experts * kNT * (k / 32) < (int64_t(1) << 31);
}

namespace {
struct SkGroupedLayout {
    size_t xh, smin, dxt, partial, total;
};
SkGroupedLayout sk_grouped_layout(int64_t n_experts, int64_t k) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    SkGroupedLayout L{};
    size_t off = 0;
    L.xh = off;
    off = al(off + size_t(n_experts) * kNT * k * 2);
    L.smin = off;
    off = al(off + size_t(n_experts) * kNT * (k / 256) * 32);
    L.dxt = off;
    off = al(off + size_t(n_experts) * (k / 32) * kNT * 4);
    L.partial = off;
    off = al(off + size_t(kMaxPartialCtas) * 2 * kRows * kNT * 4);
    L.total = off;
    return L;
}
}  // namespace

size_t gemv_tc_grouped_bytes(int64_t n_experts, int64_t k) { return sk_grouped_layout(n_experts, k).total; }

cudaError_t launch_gemv_tc_grouped(const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                                   int64_t x_div, const int32_t *cold, const int32_t *ncold, const int32_t *bounds,
                                   const int32_t *perm, float *y, int *status, void *ws, size_t ws_bytes,
                                   cudaStream_t st) {
    if (!gemv_tc_grouped_supported(QMM_Q4_K, n_experts, n, k)) return cudaErrorNotSupported;
    const SkGroupedLayout L = sk_grouped_layout(n_experts, k);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    __half *xh = reinterpret_cast<__half *>(base + L.xh);
    __half *smin = reinterpret_cast<__half *>(base + L.smin);
    float *dxt = reinterpret_cast<float *>(base + L.dxt);
    const int64_t nprep = n_experts * kNT * (k / 32);
    const int pgrid = (int)std::min<int64_t>((nprep + 255) / 256, int64_t(device_sm_count()) * 4);
    cudaError_t e = launch_pdl(gemv_tc_prep_grouped_kernel, dim3(std::max(pgrid, 1)), dim3(256), 0, st,
                               static_cast<const uint8_t *>(xq), x_div, (int)k, cold, ncold, bounds, perm, xh, smin,
                               dxt);
    if (e != cudaSuccess) return e;

    CUtensorMap tm_x, tm_xmin, tm_dx, tm_w;
    const uint64_t row_bytes = uint64_t(k / 256) * kQ4KBytes;
    const int64_t xrows = n_experts * kNT;
    if (!tc_make_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xh, k, xrows, uint64_t(k) * 2, 64, kNT,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tc_make_map_2d(&tm_xmin, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, smin, (k / 256) * 16, xrows,
                        uint64_t(k / 256) * 32, 16, kNT, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !tc_make_map_2d(&tm_dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dxt, kNT, n_experts * (k / 32), kNT * 4, kNT, 8,
                        CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tc_make_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, row_bytes, n_experts * n, row_bytes, kQ4KBytes,
                        kRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    SkArgs a{};
    a.n = n;
    a.m = kNT;
    a.nsb = k / 256;
    a.ntiles = (n + kRows - 1) / kRows;
    a.nwork = 0;  // set on the device from *ncold
    a.ctas = std::min(device_sm_count(), kMaxPartialCtas);
    a.y = y;
    a.partial = reinterpret_cast<float *>(base + L.partial);
    a.status = status;
    a.cold = cold;
    a.ncold = ncold;
    a.bounds = bounds;
    a.perm = perm;

    e = ensure_smem(gemv_tc_q4k_kernel, kSmemAlloc);
    if (e != cudaSuccess) return e;
    e = launch_pdl(gemv_tc_q4k_kernel, dim3(a.ctas), dim3(kThreads), kSmemAlloc, st, tm_x, tm_xmin, tm_dx, tm_w, a);
    if (e != cudaSuccess) return e;
    // at most every expert's tiles are cold: a bounded grid strides over those that are
    const int64_t fx = std::min<int64_t>(n_experts * a.ntiles, int64_t(device_sm_count()) * 4);
    gemv_tc_fixup_kernel<<<(unsigned)fx, kRows, 0, st>>>(a);
    return cudaGetLastError();
}

bool gemv_tc_supported(qmm_type t, int64_t n, int64_t k, int64_t m) {
    return t == QMM_Q4_K && k % 256 == 0 && n > 0 && m >= 1 && m <= kMaxM;
}

size_t gemv_tc_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t m) {
    if (!gemv_tc_supported(t, n, k, m)) return 0;
    return sk_layout(m, k, sk_ctas(n, k)).total;
}

cudaError_t launch_gemv_tc(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                           void *ws, size_t ws_bytes, cudaStream_t st) {
    if (!gemv_tc_supported(t, n, k, m)) return cudaErrorNotSupported;
    const int ctas = sk_ctas(n, k);
    const SkLayout L = sk_layout(m, k, ctas);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    int *status = reinterpret_cast<int *>(base + L.status);
    __half *xh = reinterpret_cast<__half *>(base + L.xh);
    __half *smin = reinterpret_cast<__half *>(base + L.smin);
    float *dxt = reinterpret_cast<float *>(base + L.dxt);

    const int64_t nprep = int64_t(kNT) * (k / 32);
    const int pgrid = (int)std::min<int64_t>((nprep + 255) / 256, int64_t(device_sm_count()) * 4);
    cudaError_t e = launch_pdl(gemv_tc_prep_kernel, dim3(std::max(pgrid, 1)), dim3(256), 0, st,
                               static_cast<const uint8_t *>(xq), (int)m, (int)k, xh, smin, dxt, status);
    if (e != cudaSuccess) return e;

    CUtensorMap tm_x, tm_xmin, tm_dx, tm_w;
    const uint64_t row_bytes = uint64_t(k / 256) * kQ4KBytes;
    if (!tc_make_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xh, k, m, uint64_t(k) * 2, 64, kNT,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tc_make_map_2d(&tm_xmin, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, smin, (k / 256) * 16, m, uint64_t(k / 256) * 32,
                        16, kNT, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !tc_make_map_2d(&tm_dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dxt, kNT, k / 32, kNT * 4, kNT, 8,
                        CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tc_make_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, row_bytes, n, row_bytes, kQ4KBytes, kRows,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    SkArgs a{};
    a.n = n;
    a.m = (int)m;
    a.nsb = k / 256;
    a.ntiles = (n + kRows - 1) / kRows;
    a.nwork = a.ntiles * a.nsb;
    a.ctas = ctas;
    a.y = y;
    a.partial = reinterpret_cast<float *>(base + L.partial);
    a.status = status;

    e = ensure_smem(gemv_tc_q4k_kernel, kSmemAlloc);
    if (e != cudaSuccess) return e;
    e = launch_pdl(gemv_tc_q4k_kernel, dim3(ctas), dim3(kThreads), kSmemAlloc, st, tm_x, tm_xmin, tm_dx, tm_w, a);
    if (e != cudaSuccess) return e;
    gemv_tc_fixup_kernel<<<(unsigned)a.ntiles, kRows, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qmm
