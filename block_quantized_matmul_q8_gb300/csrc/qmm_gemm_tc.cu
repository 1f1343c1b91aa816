// qmm_gemm_tc.cu -- tensor-core GEMM for m > 8 (tcgen05, TMEM accumulators, TMA).
//
// What it computes is the exact-integer fold of [MMQ] sections "dp4a 路径的 Q4_K"
// and "输出端": per 32-wide sub-block an exact integer dot, folded in fp32 with the
// activation scale d8 and the weight scales d*sc, minus dmin*m*s.
//
// How, on sm_103a (where tcgen05 has no int8 kind): the integer dots run as
// kind::f16 MMAs on integer-valued fp16 operands with fp32 accumulators.  Every
// operand value is an exact fp16 integer (activation codes |q| <= 127, weight codes
// times the 6-bit sub-block scale <= 15*63 = 945) and every partial sum of one
// 32-wide sub-block is an integer below 32*945*127 < 2^24, so the fp32 accumulator
// holds the exact int32 dot whatever order the tensor core adds in.
//
// Tile: 128 activation rows (MMA M, TMEM lanes) x 128 weight rows (MMA N, TMEM
// columns); K advances by half a superblock (128 values) per pipeline stage.
// Each 32-wide sub-block accumulates into its own TMEM slot of 128 columns.  The
// four slots are handed between the MMA issuer and the epilogue in pairs (one commit,
// one wait and one release per two sub-blocks, double-buffered): on this part every
// barrier completion that the lone MMA thread has to observe costs a few hundred
// cycles during which the tensor pipe idles, so the kernel is built to need as few
// of them as possible (one per stage, one per pair of sub-blocks).
// 24 warps, registers split with setmaxnreg (32 / 64 / 96 per thread):
//   warp 0      TMA: fp16 activation slabs (128-byte swizzle), per superblock the
//               fp32 d8 tile and, for Q4_K, the fp16 s tile of the min term.
//   warp 1      TMEM allocation; one lane issues the MMAs.
//   warp 2      TMA: the raw superblocks of the tile's 128 weight rows.
//   warps 4-7   unpack: one weight row each, from the raw bytes in shared memory;
//               weight codes -> fp16 written straight into the 128-byte-swizzled
//               K-major layout the MMA reads, the 6-bit mins as fp16 for the min-term
//               MMA, and the per-row fp32 factors of the epilogue (Q4_K: d and -dmin;
//               Q8_0: d per block).
//   warps 8-23  epilogue: one activation row (TMEM lane) and 32 weight columns per
//               thread; Q4_K: per sub-block acc += d8 * slot, per superblock
//               total += d * acc - dmin * minslot, where one more K=16 MMA (a group of
//               its own) forms minslot = sum_b s[m,b] * m[n,b] (8 real terms, 8 zeros);
//               Q8_0: total += d8 d * slot.  The total stays in registers for the
//               whole segment.
// Work is a flattened stream of (tile, superblock) units split over the CTAs
// ([MMQ] section "stream-K 的切法"); a tile shared by several CTAs is summed by a
// separate fixup kernel in CTA order ([MMQ] section "fixup: 部分和的归约"), so no
// CTA ever waits on another.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "qmm_common.cuh"
#include "qmm_internal.h"
#include "qmm_moe.h"
#include "qmm_tc_common.cuh"
#include "qmm_tc_ptx.cuh"

namespace qmm {

namespace {

constexpr int kTM = 128;  // activation rows per tile
constexpr int kTN = 128;  // weight rows per tile
constexpr int kMaxStages = 3;  // deepest activation/weight stage ring of any format
constexpr int kSlots = 4;          // accumulator slots of 128 TMEM columns: all of TMEM
constexpr int kPair = 2;           // slots handed over per barrier round trip
constexpr int kThreads = 768;      // 24 warps = 6 warpgroups
constexpr int kUnpackWarp0 = 4;
constexpr int kEpiWarp0 = 8;
constexpr int kEpiWarps = 16;
// Registers per thread after the split.  The block is launched with 80 registers per
// thread (65536 / 768 rounded down to a multiple of 8), so the split may hand out at
// most 768 x 80 registers; setmaxnreg.inc would otherwise wait forever.
constexpr int kLaunchRegs = 80;
constexpr int kRegsProducer = 32, kRegsUnpack = 64, kRegsEpilogue = 96;
static_assert(128 * kRegsProducer + 128 * kRegsUnpack + 32 * kEpiWarps * kRegsEpilogue <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kMaxPartialCtas = 256;

// Per-format constants.  Q4_K: 144-byte superblocks and a min-term MMA per superblock.
// Q8_0: the 256 k values of a step are eight 34-byte blocks, a d per 32-block and row.
// kUses counts the sub-block slots of one superblock (whole pairs), kDDBytes the
// per-row factors the unpack hands to the epilogue, raw_x the raw tensor map's x
// coordinate of superblock sb (in its elements).
template <int T> struct TcFmt;
// Stage geometry (all formats but Q6_K): 2 stages of half a superblock, each 2 activation
// slabs of 64 k values and 2 weight slabs; kScaleD: the weight row's d multiplies the
// superblock's sum of d8 * slot once, instead of a factor per slot.
struct TcStages2 {
    static constexpr int kStages = 2, kStagesPerSb = 2, kXSlabs = 2, kPlanes = 1;
};
template <> struct TcFmt<QMM_Q4_K> : TcStages2 {
    static constexpr uint32_t kRawRow = kQ4KBytes;  // raw bytes of one weight row per 256 k
    static constexpr uint32_t kRawBuf = 128 * kRawRow;  // one raw buffer: the tile's 128 rows
    static constexpr bool kMin = true, kScaleD = true;
    static constexpr int kUses = 8;
    static constexpr int kSub = 32;  // k values per slot
    static constexpr uint32_t kDDBytes = 2 * 128 * 2;  // fp16 d[128], -dmin[128]
    static __device__ __forceinline__ int raw_x(int64_t sb) { return (int)(sb * kQ4KBytes); }
};
// Q5_K: Q4_K's superblock with a 32-byte plane of fifth bits (176 bytes, a whole number
// of 16-byte units, one tensor-map box per superblock); the operand code * sc stays exact
// in fp16 (31 * 63 = 1953 < 2048).
template <> struct TcFmt<QMM_Q5_K> : TcStages2 {
    static constexpr uint32_t kRawRow = kQ5KBytes;
    static constexpr uint32_t kRawBuf = 128 * kRawRow;
    static constexpr bool kMin = true, kScaleD = true;
    static constexpr int kUses = 8;
    static constexpr int kSub = 32;
    static constexpr uint32_t kDDBytes = 2 * 128 * 2;  // fp16 d[128], -dmin[128]
    static __device__ __forceinline__ int raw_x(int64_t sb) { return (int)(sb * kQ5KBytes); }
};
template <> struct TcFmt<QMM_Q8_0> : TcStages2 {
    static constexpr uint32_t kRawRow = 8 * kQ80Bytes;  // 272
    static constexpr uint32_t kRawBuf = 128 * kRawRow;
    static constexpr bool kMin = false, kScaleD = false;
    static constexpr int kUses = 8;
    static constexpr int kSub = 32;
    static constexpr uint32_t kDDBytes = 8 * 128 * 2;  // fp16 d[8 blocks][128 rows]
    static __device__ __forceinline__ int raw_x(int64_t sb) { return (int)(sb * 136); }
};
// Q4_0: the 256 k values of a step are eight 18-byte blocks (144 bytes, as a Q4_K
// superblock), a d per 32-block and row; the codes q - 8 are exact fp16 integers.
template <> struct TcFmt<QMM_Q4_0> : TcStages2 {
    static constexpr uint32_t kRawRow = 8 * kQ40Bytes;  // 144
    static constexpr uint32_t kRawBuf = 128 * kRawRow;
    static constexpr bool kMin = false, kScaleD = false;
    static constexpr int kUses = 8;
    static constexpr int kSub = 32;
    static constexpr uint32_t kDDBytes = 8 * 128 * 2;  // fp16 d[8 blocks][128 rows]
    static __device__ __forceinline__ int raw_x(int64_t sb) { return (int)(sb * 144); }
};
// Q6_K: a row is 210 bytes per superblock, so neither a row (210 * k/256 bytes) nor a
// superblock is a whole number of 16-byte units and the rows cannot be the rows of a 2-D
// tensor map; 8 rows always are.  With n a multiple of 8 the map's row is a group of 8 weight
// rows and the raw warp loads 8 boxes per superblock (TcArgs::q6_groups); otherwise it issues
// one 224-byte bulk copy per row.  Either way a row's data is the window starting at the
// 16-byte boundary at or below its superblock (offset <= 14 inside it, the bytes after it
// belong to the next row), and windows sit 240 bytes apart in shared memory.
// The int8 sub-scale of every 16 values goes into the operands: with sc = 16 a + b
// (a = sc >> 4 in -8..7, b = sc & 15), the weight code q (-32..31) becomes two exact fp16
// planes, 16 q a and q b, and the MMA runs over the same activations once per plane into
// the same accumulator, which then holds sum sc q x of a whole 32-block (each element adds
// 0, 16 q a, q b or q sc, all at most 128 |q| in magnitude, so every partial sum stays
// below 32 * 127 * 32 * 128 < 2^24 and is exact in any order).  One slot per 32-block, as
// for Q4_K, and only d is left for the fold: twice the MMAs, half the slots and a quarter
// of the fold work of one slot per 16-wide sub-block.  Stages are a quarter superblock
// (one activation slab, two weight planes), three deep.
template <> struct TcFmt<QMM_Q6_K> {
    static constexpr int kStages = 3, kStagesPerSb = 4, kXSlabs = 1, kPlanes = 2;
    static constexpr uint32_t kRawRow = 240;    // shared-memory stride of the row windows
    static constexpr uint32_t kCopyBytes = 224;  // window bytes per row
    static constexpr uint32_t kRawBuf = 128 * kRawRow;
    static constexpr bool kMin = false, kScaleD = true;
    static constexpr int kUses = 8;
    static constexpr int kSub = 32;
    static constexpr uint32_t kDDBytes = 128 * 2;  // fp16 d[128 rows]
    // byte offset of superblock sb of weight row `row` from the start of W
    static __device__ __forceinline__ int64_t pos(int64_t row, int64_t sb, int64_t row_bytes) {
        return row * row_bytes + sb * kQ6KBytes;
    }
};

// Q6_K row groups: one box of 16 rows x 240 bytes per row residue mod 8
constexpr uint32_t kQ6GroupBox = 16 * TcFmt<QMM_Q6_K>::kRawRow;
static_assert(8 * kQ6GroupBox == TcFmt<QMM_Q6_K>::kRawBuf && kQ6GroupBox % 128 == 0, "Q6_K group boxes");

// dynamic shared memory map (offsets from a 1024-aligned base)
constexpr uint32_t kSlabBytes = 128 * 128;  // 128 rows x 64 fp16
template <int T> struct TcMap {
    using F = TcFmt<T>;
    static_assert(F::kUses % (2 * kPair) == 0, "a superblock must start on the first pair of the ring");
    static_assert(F::kRawBuf % 16 == 0, "raw buffers must keep TMA destinations 16-byte aligned");
    static_assert(F::kStages <= kMaxStages && (F::kUses / kPair) % F::kStagesPerSb == 0, "stage geometry");
    static constexpr uint32_t kXStage = F::kXSlabs * kSlabBytes;      // activation slabs of a stage
    static constexpr uint32_t kWStage = F::kPlanes * kXStage;         // weight slabs of a stage (all planes)
    static constexpr uint32_t kOffX = 0;                                  // [stage][kXSlabs slabs]
    static constexpr uint32_t kOffW = kOffX + F::kStages * kXStage;       // [stage][plane][kXSlabs slabs]
    static constexpr uint32_t kMinBytes = F::kMin ? F::kStages * 4096 : 0;
    static constexpr uint32_t kOffXmin = kOffW + F::kStages * kWStage;    // [stage][128][32 B]
    static constexpr uint32_t kOffWmin = kOffXmin + kMinBytes;              // [stage][128][32 B]
    static constexpr uint32_t kOffDX = kOffWmin + kMinBytes;                // [2][128][8] fp32 d8
    static constexpr uint32_t kOffDD = kOffDX + 2 * 4096;                   // [2][kDDBytes]
    static constexpr uint32_t kRawBytes = F::kRawBuf;                    // raw weights of 128 rows
    static constexpr uint32_t kOffRaw = (kOffDD + 2 * F::kDDBytes + 1023) & ~1023u;
    static constexpr uint32_t kSmemAlloc = kOffRaw + 2 * kRawBytes + 1024;
    static_assert(kSmemAlloc <= 227 * 1024, "shared memory map exceeds the per-CTA limit");
};

struct TcArgs {
    const uint8_t *W;
    int64_t n;
    int64_t m;
    int k;
    int64_t row_bytes;
    float *y;
    float *partial;
    int *status;
    int64_t tiles_n;
    int64_t nsb;
    int64_t nwork;
    int ctas;
    // 0: one tile per CTA; 1: stream-K; 2 (expert-grouped): whole tiles when the tile
    // count read on the device fills the CTAs' waves to at least 90%, else stream-K;
    // 3 (expert-grouped): whole tiles always (the fused gate/up needs both dots whole)
    int stream_k;
    // expert-grouped mode (tiles != nullptr): the activation arrays hold the (token,
    // slot) pairs in expert-sorted order, W is [E][n] rows, y is [pairs][n]
    const MoETile *tiles;
    const int32_t *ntiles;  // device: number of token tiles in `tiles`
    const int32_t *bounds;
    const int32_t *perm;
    // fused gate/up + SwiGLU (n_out > 0, Q4_K): the tile space has n = 2 n_out columns,
    // column 2j the gate row j (tm_w) and 2j+1 the up row j (tm_w2); y is [m][n_out].
    // glu_packed: the rows are stored interleaved (qmm_repack_glu), so column c is row c
    // of tm_w and the tile loads as in the plain GEMM
    int64_t n_out;
    int glu_packed;
    // test switch (qmm_set_test_fault): the activation producer issues nothing, and the
    // MMA issuer's wait for the first stage gives up after mma_wait_cycles, so the
    // kernel reports QMM_ERR_DEVICE with no copy in flight
    int withhold_x;
    long long mma_wait_cycles;
    // Q6_K with its rows in whole groups of 8 (tm_w maps each group as one row of 8 row
    // lengths): the raw superblock of a tile's 128 rows comes as 8 boxes, one per row
    // residue mod 8, instead of 128 bulk copies
    int q6_groups;
};

// Where tile t lives: m0 = first activation row (sorted row in grouped mode), rows =
// valid activation rows, n0w = first row in the weight tensor map, col0 = first output
// column.
struct TileInfo {
    int m0, rows, n0w;
    int64_t col0;
};
__device__ __forceinline__ TileInfo resolve_tile(const TcArgs &a, int64_t t) {
    TileInfo ti;
    const int64_t tn = t % a.tiles_n;
    ti.col0 = tn * kTN;
    if (a.tiles) {
        const MoETile mt = a.tiles[t / a.tiles_n];
        ti.m0 = a.bounds[mt.expert] + mt.first;
        ti.rows = min(kTM, mt.count - mt.first);
        ti.n0w = (int)(int64_t(mt.expert) * a.n + ti.col0);
    } else {
        ti.m0 = (int)((t / a.tiles_n) * kTM);
        ti.rows = a.m - ti.m0 < kTM ? (int)(a.m - ti.m0) : kTM;
        ti.n0w = (int)ti.col0;
    }
    return ti;
}

// Stage barriers: st_full completes when the activation slabs have landed (TMA
// transaction bytes) and all 128 unpack threads have written the weight slabs;
// st_empty when the MMAs reading the stage are done (TMA producer and unpack both wait
// on it).  sd_full / sd_empty guard the per-superblock scale tiles the same way.
struct Barriers {
    uint64_t st_full[kMaxStages], st_empty[kMaxStages];
    uint64_t acc_full[kSlots / kPair], acc_empty[kSlots / kPair];
    uint64_t sd_full[2], sd_empty[2];
    uint64_t raw_full[2], raw_empty[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

// Mode 2: whole tiles are worth it when the last wave is nearly full, i.e. when the tiles
// fill at least 90% of ceil(tiles / ctas) rounds of the CTAs; the fixup kernel takes the
// same decision from the same numbers.
__device__ __forceinline__ bool whole_tiles(const TcArgs &a) {
    if (a.stream_k == 3) return true;
    if (a.stream_k != 2) return false;
    const int64_t t = a.nwork / a.nsb, rounds = (t + a.ctas - 1) / a.ctas;
    return 10 * t >= 9 * rounds * a.ctas;
}

__device__ __forceinline__ void cta_range(const TcArgs &a, int cta, int64_t &b, int64_t &e) {
    if (whole_tiles(a)) {  // a contiguous run of whole tiles: nothing left for the fixup
        const int64_t t = a.nwork / a.nsb;
        b = (t * cta / a.ctas) * a.nsb;
        e = (t * (cta + 1) / a.ctas) * a.nsb;
    } else if (a.stream_k) {
        b = a.nwork * cta / a.ctas;
        e = a.nwork * (cta + 1) / a.ctas;
    } else {
        b = int64_t(cta) * a.nsb;
        e = b + a.nsb;
    }
}

// the segments of a CTA's unit range: (tile, s0, s1) with s in [s0, s1) superblocks
struct Seg {
    int64_t tile, s0, s1;
};
__device__ __forceinline__ bool next_seg(const TcArgs &a, int64_t &u, int64_t end, Seg &sg) {
    if (u >= end) return false;
    sg.tile = u / a.nsb;
    sg.s0 = u - sg.tile * a.nsb;
    sg.s1 = min(a.nsb, sg.s0 + (end - u));
    u += sg.s1 - sg.s0;
    return true;
}

// Q6_K by row groups (TcArgs::q6_groups): tile column c holds weight row q6_perm(c), so that
// the 8 unpack threads of a quarter warp, which take 8 consecutive columns, read 8 different
// rows of one row-group box (distinct banks) while writing their own columns as before.
__device__ __forceinline__ int q6_perm(int c) { return 64 * (c >> 6) + 8 * (c & 7) + ((c >> 3) & 7); }

// One epilogue thread's 32 results of a segment: a whole tile goes to y, part of a
// tile to this CTA's partial slot (0 for its first segment, 1 for its last).  With row
// groups (rowgrp) column 32 cq + 8 jj + j is weight row 64 (cq / 2) + 4 (cq % 2) + 8 j + jj:
// four consecutive rows for each j; partial slots are kept in weight-row order.
__device__ __forceinline__ void store_segment(const TcArgs &a, const Seg &sg, int seg_i, int tl, int cq,
                                              const float2 (&tot)[16], bool rowgrp) {
    const TileInfo ti = resolve_tile(a, sg.tile);
    const int64_t col0 = ti.col0 + 32 * cq;
    auto val = [&](int i) { return (i & 1) ? tot[i >> 1].y : tot[i >> 1].x; };
    const int gbase = 64 * (cq >> 1) + 4 * (cq & 1);  // rowgrp: first weight row of the thread's groups
    if (a.n_out) {  // GLU (whole tiles only): columns 2i, 2i+1 are the gate and up dots of output col0/2 + i
        if (tl >= ti.rows) return;
        const int64_t yrow = a.tiles ? int64_t(a.perm[ti.m0 + tl]) : int64_t(ti.m0 + tl);
        float *dst = a.y + yrow * a.n_out + col0 / 2;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (col0 / 2 + i < a.n_out) dst[i] = tot[i].x / (1.0f + expf(-tot[i].x)) * tot[i].y;
        return;
    }
    if (sg.s0 == 0 && sg.s1 == a.nsb) {
        if (tl >= ti.rows) return;
        const int64_t yrow = a.tiles ? int64_t(a.perm[ti.m0 + tl]) : int64_t(ti.m0 + tl);
        if (rowgrp) {
            float *dst = a.y + yrow * a.n + ti.col0 + gbase;
            if ((a.n % 4 == 0) && (ti.col0 + 128 <= a.n)) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4 *>(dst + 8 * j) = make_float4(val(j), val(8 + j), val(16 + j), val(24 + j));
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (ti.col0 + gbase + 8 * j + jj < a.n) dst[8 * j + jj] = val(8 * jj + j);
            }
            return;
        }
        float *dst = a.y + yrow * a.n + col0;
        if ((a.n % 4 == 0) && (col0 + 32 <= a.n)) {
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4)
                reinterpret_cast<float4 *>(dst)[i4] =
                    make_float4(tot[2 * i4].x, tot[2 * i4].y, tot[2 * i4 + 1].x, tot[2 * i4 + 1].y);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (col0 + 2 * i < a.n) dst[2 * i] = tot[i].x;
                if (col0 + 2 * i + 1 < a.n) dst[2 * i + 1] = tot[i].y;
            }
        }
    } else {
        const int slotidx = seg_i == 0 ? 0 : 1;
        float *prow = a.partial + ((int64_t(blockIdx.x) * 2 + slotidx) * kTM + tl) * kTN;
        if (rowgrp) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4 *>(prow + gbase + 8 * j) = make_float4(val(j), val(8 + j), val(16 + j), val(24 + j));
            return;
        }
        float4 *dst = reinterpret_cast<float4 *>(prow + 32 * cq);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4)
            dst[i4] = make_float4(tot[2 * i4].x, tot[2 * i4].y, tot[2 * i4 + 1].x, tot[2 * i4 + 1].y);
    }
}

template <int T>
__device__ __forceinline__ void gemm_tc_body(const CUtensorMap &tm_x, const CUtensorMap &tm_xmin,
                                             const CUtensorMap &tm_dx, const CUtensorMap &tm_w,
                                             const CUtensorMap &tm_w2, TcArgs a) {
    using F = TcFmt<T>;
    using Mp = TcMap<T>;
    constexpr uint32_t kOffX = Mp::kOffX, kOffW = Mp::kOffW, kOffXmin = Mp::kOffXmin, kOffWmin = Mp::kOffWmin;
    constexpr uint32_t kOffDX = Mp::kOffDX, kOffDD = Mp::kOffDD, kOffRaw = Mp::kOffRaw, kRawBytes = Mp::kRawBytes;
    constexpr int kGroups = F::kUses / kPair;  // slot pairs per superblock (the min group comes on top)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ Barriers B;
    // 1024-byte aligned, derived from the shared array by an offset so that the compiler keeps
    // every access through it a shared-memory one (a round trip through an integer turned them
    // into generic loads and stores)
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abortp = &B.abort;

    if (tid == 0) {
        B.abort = 0;
        for (int s = 0; s < F::kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&B.st_full[s]), 1 + 128);
            ptx::mbar_init(ptx::smem_u32(&B.st_empty[s]), 1);
        }
        for (int s = 0; s < kSlots / kPair; ++s) {
            ptx::mbar_init(ptx::smem_u32(&B.acc_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&B.acc_empty[s]), kEpiWarps);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(ptx::smem_u32(&B.raw_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&B.raw_empty[s]), 128);
            ptx::mbar_init(ptx::smem_u32(&B.sd_full[s]), 1 + 128);
            ptx::mbar_init(ptx::smem_u32(&B.sd_empty[s]), kEpiWarps);
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

    if (a.tiles) a.nwork = int64_t(*a.ntiles) * a.tiles_n * a.nsb;
    int64_t ubeg, uend;
    cta_range(a, blockIdx.x, ubeg, uend);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        regs_dec<kRegsProducer>();
        if (lane == 0 && !a.withhold_x) {
            ptx::prefetch_tmap(&tm_x);
            if (F::kMin) ptx::prefetch_tmap(&tm_xmin);
            ptx::prefetch_tmap(&tm_dx);
            int64_t u = ubeg;
            Seg sg;
            uint32_t x_it = 0, sd_it = 0;
            bool ok = true;
            while (ok && next_seg(a, u, uend, sg)) {
                const int m0 = resolve_tile(a, sg.tile).m0;
                for (int64_t sb = sg.s0; ok && sb < sg.s1; ++sb) {
                    const uint32_t sdi = sd_it & 1;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.sd_empty[sdi]), ((sd_it >> 1) & 1) ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sdbar = ptx::smem_u32(&B.sd_full[sdi]);
                    ptx::mbar_arrive_expect_tx(sdbar, 4096);
                    ptx::tma_load_2d(sbase + kOffDX + sdi * 4096, &tm_dx, (int)(8 * sb), m0, sdbar);
                    ++sd_it;
                    for (int h = 0; h < F::kStagesPerSb; ++h) {
                        const uint32_t st = x_it % F::kStages;
                        if (!ptx::mbar_wait(ptx::smem_u32(&B.st_empty[st]), ((x_it / F::kStages) & 1) ^ 1, abortp)) {
                            ok = false;
                            break;
                        }
                        const bool last = h == F::kStagesPerSb - 1;
                        const uint32_t bar = ptx::smem_u32(&B.st_full[st]);
                        ptx::mbar_arrive_expect_tx(bar, Mp::kXStage + ((F::kMin && last) ? 4096u : 0u));
                        const int kx = (int)(256 * sb + 64 * F::kXSlabs * h);
#pragma unroll
                        for (int i = 0; i < F::kXSlabs; ++i)
                            ptx::tma_load_2d(sbase + kOffX + st * Mp::kXStage + i * kSlabBytes, &tm_x, kx + 64 * i, m0, bar);
                        if (F::kMin && last)
                            ptx::tma_load_2d(sbase + kOffXmin + st * 4096, &tm_xmin, (int)(16 * sb), m0, bar);
                        ++x_it;
                    }
                }
            }
            // drain: every armed copy must have landed before the CTA may exit
            int dummy = 0;
            for (uint32_t i = (x_it > F::kStages ? x_it - F::kStages : 0); i < x_it; ++i)
                ptx::mbar_wait(ptx::smem_u32(&B.st_full[i % F::kStages]), (i / F::kStages) & 1, &dummy);
            for (uint32_t i = (sd_it > 2 ? sd_it - 2 : 0); i < sd_it; ++i)
                ptx::mbar_wait(ptx::smem_u32(&B.sd_full[i & 1]), (i >> 1) & 1, &dummy);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Per stage: one wait for the stage, then per pair of slots one wait for the
        // pair's release, the MMAs of both sub-blocks and one commit; for Q4_K the min
        // MMA follows the last pair as a group of its own.
        regs_dec<kRegsProducer>();
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_f16_f32(kTM, kTN);
            int64_t u = ubeg;
            Seg sg;
            uint32_t x_it = 0, gq = 0;
            bool ok = true;
            while (ok && next_seg(a, u, uend, sg)) {
                for (int64_t sb = sg.s0; ok && sb < sg.s1; ++sb) {
                    for (int h = 0; ok && h < F::kStagesPerSb; ++h) {
                        const uint32_t st = x_it % F::kStages, par = (x_it / F::kStages) & 1;
                        if (!ptx::mbar_wait_spin(ptx::smem_u32(&B.st_full[st]), par, abortp, a.mma_wait_cycles)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t xa = sbase + kOffX + st * Mp::kXStage;
                        const uint32_t wa = sbase + kOffW + st * Mp::kWStage;
                        for (int q = 0; q < kGroups / F::kStagesPerSb; ++q) {  // the pairs of this stage
                            const uint32_t e = gq & 1;
                            if (!ptx::mbar_wait_spin(ptx::smem_u32(&B.acc_empty[e]), ((gq >> 1) & 1) ^ 1, abortp)) {
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
#pragma unroll
                            for (int b2 = 0; b2 < kPair; ++b2) {
                                const uint32_t d = tmem + (kPair * e + b2) * kTN;
#pragma unroll
                                for (int t = 0; t < F::kSub / 16; ++t) {  // K16 steps per slot
                                    const int step = (q * kPair + b2) * (F::kSub / 16) + t;  // slab step/4, 32 bytes each
                                    const uint32_t off = (step >> 2) * kSlabBytes + (step & 3) * 32;
#pragma unroll
                                    for (int pl = 0; pl < F::kPlanes; ++pl)  // Q6_K: both weight planes, same activations
                                        ptx::mma_f16(d, ptx::smem_desc(xa + off, 1024, 2),
                                                     ptx::smem_desc(wa + pl * Mp::kXStage + off, 1024, 2), idesc,
                                                     (t | pl) != 0);
                                }
                            }
                            ptx::mma_commit(ptx::smem_u32(&B.acc_full[e]));
                            ++gq;
                        }
                        if (F::kMin && ok && h == F::kStagesPerSb - 1) {  // the min term: a group of one slot
                            const uint32_t e = gq & 1;
                            if (!ptx::mbar_wait_spin(ptx::smem_u32(&B.acc_empty[e]), ((gq >> 1) & 1) ^ 1, abortp)) {
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
                            ptx::mma_f16(tmem + kPair * e * kTN, ptx::smem_desc(sbase + kOffXmin + st * 4096, 256, 6),
                                         ptx::smem_desc(sbase + kOffWmin + st * 4096, 256, 6), idesc, 0);
                            ptx::mma_commit(ptx::smem_u32(&B.acc_full[e]));
                            ++gq;
                        }
                        ptx::mma_commit(ptx::smem_u32(&B.st_empty[st]));
                        ++x_it;
                    }
                }
            }
            // every MMA must be complete before TMEM is freed
            ptx::mma_commit(ptx::smem_u32(&B.done));
            int dummy = 0;
            ptx::mbar_wait(ptx::smem_u32(&B.done), 0, &dummy);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ raw weight TMA
        // The raw superblock of the tile's 128 weight rows, one per superblock, into a
        // 2-deep ring; independent of the activation stream so neither waits on the other.
        // Q4_K / Q8_0: one tensor-map box (lane 0); Q6_K: 8 row-group boxes (lane 0), or
        // one bulk copy per valid row spread over the 32 lanes.
        regs_dec<kRegsProducer>();
        if (T == QMM_Q6_K || lane == 0) {
            if (T != QMM_Q6_K || a.q6_groups) ptx::prefetch_tmap(&tm_w);
            if (a.n_out && !a.glu_packed) ptx::prefetch_tmap(&tm_w2);
            int64_t u = ubeg;
            Seg sg;
            uint32_t r_it = 0;
            bool ok = true;
            while (ok && next_seg(a, u, uend, sg)) {
                const int n0 = resolve_tile(a, sg.tile).n0w;
                for (int64_t sb = sg.s0; sb < sg.s1; ++sb) {
                    const uint32_t ri = r_it & 1;
                    const bool got = ptx::mbar_wait(ptx::smem_u32(&B.raw_empty[ri]), ((r_it >> 1) & 1) ^ 1, abortp);
                    // Q6_K: all 32 lanes take part, so they must agree before the warp barrier
                    if (!(T == QMM_Q6_K ? __all_sync(0xffffffffu, got) != 0 : got)) {
                        ok = false;
                        break;
                    }
                    const uint32_t rbar = ptx::smem_u32(&B.raw_full[ri]);
                    if constexpr (T == QMM_Q6_K) {
                      if (a.q6_groups) {
                        // box res: rows n0 + res, n0 + res + 8, ... (16 of them, 240 bytes each
                        // from the 16-byte boundary at or below the superblock), where rows
                        // past the matrix read as zeros.  One copy per 128 rows instead of
                        // 128 (151936 x 5120 at m = 512: the per-row copies cost about 24%).
                        if (lane == 0) {
                            ptx::mbar_arrive_expect_tx(rbar, kRawBytes);
#pragma unroll 1
                            for (int res = 0; res < 8; ++res)
                                ptx::tma_load_2d(sbase + kOffRaw + ri * kRawBytes + res * kQ6GroupBox, &tm_w,
                                                 (int)(((int64_t)res * a.row_bytes + sb * kQ6KBytes) & ~int64_t(15)),
                                                 n0 / 8, rbar);
                        }
                        __syncwarp();
                      } else {
                        // rows of W in this tile: its columns within the expert's (or the matrix's) n
                        const int64_t cols = a.n - resolve_tile(a, sg.tile).col0;
                        const int64_t nval = cols < 128 ? cols : 128;
                        if (lane == 0) ptx::mbar_arrive_expect_tx(rbar, (uint32_t)nval * F::kCopyBytes);
                        __syncwarp();
#pragma unroll 1
                        for (int r = lane; r < nval; r += 32) {
                            const int64_t p = F::pos(n0 + r, sb, a.row_bytes);
                            ptx::bulk_g2s(sbase + kOffRaw + ri * kRawBytes + r * F::kRawRow, a.W + (p & ~int64_t(15)),
                                          F::kCopyBytes, rbar);
                        }
                      }
                    } else if (a.n_out && !a.glu_packed) {  // GLU: 64 gate rows, then the 64 up rows of the same outputs
                        ptx::mbar_arrive_expect_tx(rbar, kRawBytes);
                        ptx::tma_load_2d(sbase + kOffRaw + ri * kRawBytes, &tm_w, F::raw_x(sb), n0 / 2, rbar);
                        ptx::tma_load_2d(sbase + kOffRaw + ri * kRawBytes + 64 * F::kRawRow, &tm_w2, F::raw_x(sb),
                                         n0 / 2, rbar);
                    } else {
                        ptx::mbar_arrive_expect_tx(rbar, kRawBytes);
                        ptx::tma_load_2d(sbase + kOffRaw + ri * kRawBytes, &tm_w, F::raw_x(sb), n0, rbar);
                    }
                    ++r_it;
                }
            }
            int dummy = 0;
            for (uint32_t i = (r_it > 2 ? r_it - 2 : 0); i < r_it; ++i)
                ptx::mbar_wait(ptx::smem_u32(&B.raw_full[i & 1]), (i >> 1) & 1, &dummy);
        }
    } else if (warp < kUnpackWarp0) {
        regs_dec<kRegsProducer>();  // warp 3: no role, gives its registers away
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------ weight unpack
        // One weight row per thread, reading the raw superblock that the TMA warp put in
        // shared memory (rows 144 bytes apart: 8 consecutive rows hit distinct banks); with
        // Q6_K row groups the thread of tile column r takes weight row q6_perm(r).
        regs_dec<kRegsUnpack>();
        const int r = tid - 32 * kUnpackWarp0;  // tile column (weight row within the tile)
        int64_t u = ubeg;
        Seg sg;
        uint32_t w_it = 0, sb_it = 0;
        bool ok = true;
        while (ok && next_seg(a, u, uend, sg)) {
            // this thread's row of W: tile column r, or with Q6_K row groups weight row q6_perm(r)
            const int wr = (T == QMM_Q6_K && a.q6_groups) ? q6_perm(r) : r;
            const int64_t n0w = resolve_tile(a, sg.tile).n0w + wr;
            (void)n0w;
            for (int64_t sb = sg.s0; ok && sb < sg.s1; ++sb) {
                const uint32_t ri = sb_it & 1;
                if (!ptx::mbar_wait(ptx::smem_u32(&B.raw_full[ri]), (sb_it >> 1) & 1, abortp) ||
                    !ptx::mbar_wait(ptx::smem_u32(&B.sd_empty[ri]), ((sb_it >> 1) & 1) ^ 1, abortp)) {
                    ok = false;
                    break;
                }
                // GLU from two tensors: tile column r is gate row r/2 (r even) or up row r/2 (r odd)
                const int rsrc = a.n_out && !a.glu_packed ? (r & 1) * 64 + (r >> 1) : r;
                const uint8_t *blk = smem + kOffRaw + ri * kRawBytes + rsrc * F::kRawRow;
                if constexpr (T == QMM_Q6_K) {
                    if (a.q6_groups)  // weight row wr: box wr % 8, its row wr / 8
                        blk = smem + kOffRaw + ri * kRawBytes + (wr & 7) * kQ6GroupBox + (wr >> 3) * F::kRawRow;
                    blk += (int)(F::pos(n0w, sb, a.row_bytes) & 15);  // the superblock's offset inside its window
                }
                float *dd = reinterpret_cast<float *>(smem + kOffDD + ri * F::kDDBytes);
                if constexpr (T == QMM_Q4_K || T == QMM_Q5_K) {
                // Q5_K: the nibbles start 32 bytes later, after the plane of fifth bits
                constexpr int kQs = T == QMM_Q4_K ? 16 : 48;
                const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
                // (d, -dmin) for the epilogue as fp16: d of the 128 rows, then -dmin
                reinterpret_cast<uint16_t *>(dd)[r] = (uint16_t)(hd.x & 0xffffu);
                reinterpret_cast<uint16_t *>(dd)[128 + r] = (uint16_t)((hd.x >> 16) ^ 0x8000u);
                ptx::mbar_arrive(ptx::smem_u32(&B.sd_full[ri]));
                for (int h = 0; h < 2; ++h) {
                    const uint32_t st = w_it % F::kStages;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.st_empty[st]), ((w_it / F::kStages) & 1) ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    uint8_t *wst = smem + kOffW + st * Mp::kWStage;
#pragma unroll
                    for (int j2 = 0; j2 < 2; ++j2) {  // slab j2 <-> qs chunk c = 2h + j2
                        const int c = 2 * h + j2;
                        const uint4 qa = *reinterpret_cast<const uint4 *>(blk + kQs + 32 * c);
                        const uint4 qb = *reinterpret_cast<const uint4 *>(blk + kQs + 16 + 32 * c);
                        int sc_lo, m_lo, sc_hi, m_hi;
                        q4k_scale_min(hd.y, hd.z, hd.w, 2 * c, sc_lo, m_lo);
                        q4k_scale_min(hd.y, hd.z, hd.w, 2 * c + 1, sc_hi, m_hi);
                        const __half2 s_lo = __float2half2_rn((float)sc_lo), ns_lo = __float2half2_rn(-1024.f * sc_lo);
                        // Q4_K takes the high nibbles in place (16 q): scale sc / 16, offset -64 sc
                        const __half2 s_hi = __float2half2_rn(T == QMM_Q4_K ? 0.0625f * sc_hi : (float)sc_hi);
                        const __half2 ns_hi = __float2half2_rn(T == QMM_Q4_K ? -64.f * sc_hi : -1024.f * sc_hi);
                        const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                        uint8_t *rowdst = wst + j2 * kSlabBytes + r * 128;
                        if constexpr (T == QMM_Q4_K) {
#pragma unroll
                            for (int cq = 0; cq < 4; ++cq) {  // codes in the order 0 2 1 3 of every 4
                                const uint4 lo = nibbles_to_f16_0213(w[2 * cq], w[2 * cq + 1], false, s_lo, ns_lo);
                                const uint4 hi = nibbles_to_f16_0213(w[2 * cq], w[2 * cq + 1], true, s_hi, ns_hi);
                                *reinterpret_cast<uint4 *>(rowdst + ((cq ^ (r & 7)) << 4)) = lo;
                                *reinterpret_cast<uint4 *>(rowdst + (((cq + 4) ^ (r & 7)) << 4)) = hi;
                            }
                        } else {  // the fifth bits of the same 32 positions: bits 2c and 2c+1 of qh
                            const uint4 ha = *reinterpret_cast<const uint4 *>(blk + 16);
                            const uint4 hb = *reinterpret_cast<const uint4 *>(blk + 32);
                            const uint32_t q[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
#pragma unroll
                            for (int cq = 0; cq < 4; ++cq) {
                                const uint4 lo = nibbles5_to_f16(w[2 * cq], w[2 * cq + 1], q[2 * cq], q[2 * cq + 1], 0,
                                                                 2 * c, s_lo, ns_lo);
                                const uint4 hi = nibbles5_to_f16(w[2 * cq], w[2 * cq + 1], q[2 * cq], q[2 * cq + 1], 4,
                                                                 2 * c + 1, s_hi, ns_hi);
                                *reinterpret_cast<uint4 *>(rowdst + ((cq ^ (r & 7)) << 4)) = lo;
                                *reinterpret_cast<uint4 *>(rowdst + (((cq + 4) ^ (r & 7)) << 4)) = hi;
                            }
                        }
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
                        uint8_t *mdst = smem + kOffWmin + st * 4096 + r * 32;
                        const int sw = (r >> 2) & 1;
                        *reinterpret_cast<uint4 *>(mdst + ((0 ^ sw) << 4)) = make_uint4(mm[0], mm[1], mm[2], mm[3]);
                        *reinterpret_cast<uint4 *>(mdst + ((1 ^ sw) << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(ptx::smem_u32(&B.st_full[st]));
                    ++w_it;
                }
                } else if constexpr (T == QMM_Q6_K) {
                // Q6_K: d for the epilogue (the superblock starts 0 or 2 bytes past a word
                // boundary: its words are read from the boundary below and shifted), then per
                // quarter superblock the 64-value unit as two planes of exact fp16 integers,
                // 16 q (sc >> 4) and q (sc & 15), with q the code - 32 and sc the int8 scale of
                // its 16 values (sc = 16 (sc >> 4) + (sc & 15)).
                {
                    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(blk) & 2u);
                    const uint32_t dw = LdShared::u32(blk + 208 - mis);
                    reinterpret_cast<uint16_t *>(dd)[r] = (uint16_t)(mis ? (dw >> 16) : (dw & 0xffffu));
                }
                ptx::mbar_arrive(ptx::smem_u32(&B.sd_full[ri]));
                const __half2 bias = __float2half2_rn(-1152.f);
                for (int h = 0; h < F::kStagesPerSb; ++h) {  // unit h (64 k values) is stage h of the superblock
                    const uint32_t st = w_it % F::kStages;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.st_empty[st]), ((w_it / F::kStages) & 1) ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    uint8_t *wst = smem + kOffW + st * Mp::kWStage;
                    // Unit h covers k = 64h .. 64h+63: half hh = h >> 1 of the superblock,
                    // quarters t = 2 (h & 1) and 2 (h & 1) + 1; weight 128 hh + 32 t + l takes the
                    // nibble t >> 1 of ql[64 hh + 32 (t & 1) + l] and bits 2t, 2t+1 of qh[32 hh + l].
                    // The 32 qh bytes stay in registers for the unit, the ql bytes are read 32 at
                    // a time (one quarter t).
                    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(blk) & 2u), fsh2 = 8u * mis;
                    const uint8_t *blk4 = blk - mis;
                    auto wd = [&](int off) {  // the 32-bit word at byte off of the superblock
                        return __funnelshift_r(LdShared::u32(blk4 + off), LdShared::u32(blk4 + off + 4), fsh2);
                    };
                    // Eight consecutive words of the superblock from byte X (a multiple of 16):
                    // three aligned 16-byte loads of the window (rows 240 bytes apart, so the 8
                    // lanes of a quarter warp hit distinct banks), rotated by the superblock's
                    // word offset in the window and shifted by its odd half-word.
                    const uint32_t o = (uint32_t)(reinterpret_cast<uintptr_t>(blk) & 15u);
                    const uint8_t *win = blk - o;
                    const bool rot1 = (o & 4u) != 0, rot2 = (o & 8u) != 0;
                    const uint32_t fsh = 8u * (o & 3u);
                    auto span8 = [&](int X, uint32_t(&out)[8]) {
                        uint32_t v[12];
#pragma unroll
                        for (int c = 0; c < 3; ++c) {
                            const uint4 t4 = *reinterpret_cast<const uint4 *>(win + X + 16 * c);
                            v[4 * c] = t4.x;
                            v[4 * c + 1] = t4.y;
                            v[4 * c + 2] = t4.z;
                            v[4 * c + 3] = t4.w;
                        }
#pragma unroll
                        for (int i = 0; i < 11; ++i) v[i] = rot1 ? v[i + 1] : v[i];
#pragma unroll
                        for (int i = 0; i < 9; ++i) v[i] = rot2 ? v[i + 2] : v[i];
#pragma unroll
                        for (int j = 0; j < 8; ++j) out[j] = __funnelshift_r(v[j], v[j + 1], fsh);
                    };
                    const uint32_t scw = wd(192 + 4 * h);  // the 4 int8 scales of the unit's 16-value sub-blocks
                    __half2 ha[4], hb[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int sc = (int)(int8_t)((scw >> (8 * j)) & 0xffu);
                        ha[j] = __float2half2_rn((float)(16 * (sc >> 4)));
                        hb[j] = __float2half2_rn((float)(sc & 15));
                    }
                    const int hh = h >> 1;
                    uint8_t *rowa = wst + r * 128, *rowb = wst + kSlabBytes + r * 128;
                    uint32_t QH[8];
                    span8(128 + 32 * hh, QH);  // qh[32 hh + l], l = 0..31
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t QL[8];
                    span8(64 * hh + 32 * c2, QL);  // ql[64 hh + 32 c2 + l]
#pragma unroll
                    for (int cq4 = 0; cq4 < 4; ++cq4) {  // 16-byte chunk cq: codes 8cq .. 8cq+7, sub-block cq / 2
                        const int cq = 4 * c2 + cq4;
                        const int tt = 2 * (h & 1) + c2;
                        uint32_t code[2];
#pragma unroll
                        for (int e2 = 0; e2 < 2; ++e2) {
                            const uint32_t ql = QL[2 * cq4 + e2];
                            const uint32_t qh = QH[2 * cq4 + e2];
                            const uint32_t lo = (ql >> (4 * (tt >> 1))) & 0x0f0f0f0fu;
                            const uint32_t hi2 = ((qh >> (2 * tt)) & 0x03030303u) << 4;
                            code[e2] = __vsub4(lo | hi2, 0x20202020u);  // q - 32 as signed bytes
                        }
                        uint32_t pa[4], pb[4];
#pragma unroll
                        for (int e2 = 0; e2 < 2; ++e2) {
                            const uint32_t uu = code[e2] ^ 0x80808080u;
                            uint32_t lo = __byte_perm(uu, 0x64646464u, 0x4140);
                            uint32_t hi = __byte_perm(uu, 0x64646464u, 0x4342);
                            const __half2 ql = __hadd2(*reinterpret_cast<__half2 *>(&lo), bias);
                            const __half2 qh = __hadd2(*reinterpret_cast<__half2 *>(&hi), bias);
                            pa[2 * e2] = h2bits(__hmul2(ql, ha[cq >> 1]));
                            pa[2 * e2 + 1] = h2bits(__hmul2(qh, ha[cq >> 1]));
                            pb[2 * e2] = h2bits(__hmul2(ql, hb[cq >> 1]));
                            pb[2 * e2 + 1] = h2bits(__hmul2(qh, hb[cq >> 1]));
                        }
                        const int sw = (cq ^ (r & 7)) << 4;
                        *reinterpret_cast<uint4 *>(rowa + sw) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
                        *reinterpret_cast<uint4 *>(rowb + sw) = make_uint4(pb[0], pb[1], pb[2], pb[3]);
                    }
                    }
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(ptx::smem_u32(&B.st_full[st]));
                    ++w_it;
                }
                } else if constexpr (T == QMM_Q4_0) {
                // Q4_0: the row's 256 k values are 8 blocks of {fp16 d, 16 nibble bytes}, block
                // b at byte 18b; byte i of a block holds its weight i (low nibble) and 16 + i
                // (high).  The d of every block goes to the epilogue; a nibble v becomes the
                // fp16 1024 + v (v | 0x6400), and adding -1032 leaves the exact code v - 8.
#pragma unroll
                for (int b = 0; b < 8; ++b)
                    reinterpret_cast<__half *>(dd)[b * 128 + r] = *reinterpret_cast<const __half *>(blk + 18 * b);
                ptx::mbar_arrive(ptx::smem_u32(&B.sd_full[ri]));
                const __half2 bias = __float2half2_rn(-1032.f);
                for (int h = 0; h < 2; ++h) {
                    const uint32_t st = w_it % F::kStages;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.st_empty[st]), ((w_it / F::kStages) & 1) ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    // blocks 4h .. 4h+3: 72 bytes from byte 72h (rows are 144 bytes apart, so the
                    // range is 8-byte aligned); block b2's nibbles start at byte 18 b2 + 2 of it,
                    // on a word boundary for odd b2 and 2 bytes past one for even b2
                    uint32_t w[18];
                    const uint2 *src = reinterpret_cast<const uint2 *>(blk + 72 * h);
#pragma unroll
                    for (int i2 = 0; i2 < 9; ++i2) {
                        const uint2 t2 = src[i2];
                        w[2 * i2] = t2.x;
                        w[2 * i2 + 1] = t2.y;
                    }
                    uint8_t *wst = smem + kOffW + st * Mp::kWStage;
#pragma unroll
                    for (int b2 = 0; b2 < 4; ++b2) {
                        const int o = (b2 >> 1) * 9;
                        uint32_t q[4];
#pragma unroll
                        for (int i2 = 0; i2 < 4; ++i2)
                            q[i2] = (b2 & 1) ? w[o + 5 + i2] : __funnelshift_r(w[o + i2], w[o + i2 + 1], 16);
                        uint8_t *rowdst = wst + (b2 >> 1) * kSlabBytes + r * 128;
#pragma unroll
                        for (int cq = 0; cq < 4; ++cq) {  // 16-byte chunk cq: weights 8cq .. 8cq+7
                            uint32_t pr[4];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const uint32_t src4 = q[2 * (cq & 1) + e2];
                                const uint32_t nib = (cq < 2 ? src4 : src4 >> 4) & 0x0f0f0f0fu;
                                uint32_t lo = __byte_perm(nib, 0x64646464u, 0x4140);
                                uint32_t hi = __byte_perm(nib, 0x64646464u, 0x4342);
                                lo = h2bits(__hadd2(*reinterpret_cast<__half2 *>(&lo), bias));
                                hi = h2bits(__hadd2(*reinterpret_cast<__half2 *>(&hi), bias));
                                pr[2 * e2] = lo;
                                pr[2 * e2 + 1] = hi;
                            }
                            const int chunk = (b2 & 1) * 4 + cq;  // 16-byte chunk of the 128-byte row
                            *reinterpret_cast<uint4 *>(rowdst + ((chunk ^ (r & 7)) << 4)) =
                                make_uint4(pr[0], pr[1], pr[2], pr[3]);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(ptx::smem_u32(&B.st_full[st]));
                    ++w_it;
                }
                } else {
                // Q8_0: the row's 256 k values are 8 blocks of {fp16 d, int8 q[32]}, block b at
                // byte 34b.  The d of every block goes to the epilogue; the codes become
                // exact fp16 integers: (q ^ 0x80) | 0x6400 is the fp16 1024 + q + 128.
#pragma unroll
                for (int b = 0; b < 8; ++b)
                    reinterpret_cast<__half *>(dd)[b * 128 + r] = *reinterpret_cast<const __half *>(blk + 34 * b);
                ptx::mbar_arrive(ptx::smem_u32(&B.sd_full[ri]));
                const __half2 bias = __float2half2_rn(-1152.f);
                for (int h = 0; h < 2; ++h) {
                    const uint32_t st = w_it % F::kStages;
                    if (!ptx::mbar_wait(ptx::smem_u32(&B.st_empty[st]), ((w_it / F::kStages) & 1) ^ 1, abortp)) {
                        ok = false;
                        break;
                    }
                    // blocks 4h .. 4h+3: 136 bytes from byte 136h (rows are 272 = 16*17 bytes apart,
                    // so the range is 8-byte aligned); block b2 starts at byte 34 b2 of it
                    uint32_t w[34];
                    const uint2 *src = reinterpret_cast<const uint2 *>(blk + 136 * h);
#pragma unroll
                    for (int i2 = 0; i2 < 17; ++i2) {
                        const uint2 t2 = src[i2];
                        w[2 * i2] = t2.x;
                        w[2 * i2 + 1] = t2.y;
                    }
                    uint8_t *wst = smem + kOffW + st * Mp::kWStage;
#pragma unroll
                    for (int b2 = 0; b2 < 4; ++b2) {
                        const int o = (b2 >> 1) * 17;
                        uint32_t q[8];
#pragma unroll
                        for (int i2 = 0; i2 < 8; ++i2)  // codes at byte 34 b2 + 2: word-aligned for odd b2
                            q[i2] = (b2 & 1) ? w[o + 9 + i2] : __funnelshift_r(w[o + i2], w[o + i2 + 1], 16);
                        uint8_t *rowdst = wst + (b2 >> 1) * kSlabBytes + r * 128;
#pragma unroll
                        for (int cq = 0; cq < 4; ++cq) {
                            uint32_t pr[4];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const uint32_t uu = q[2 * cq + e2] ^ 0x80808080u;
                                uint32_t lo = __byte_perm(uu, 0x64646464u, 0x4140);
                                uint32_t hi = __byte_perm(uu, 0x64646464u, 0x4342);
                                lo = h2bits(__hadd2(*reinterpret_cast<__half2 *>(&lo), bias));
                                hi = h2bits(__hadd2(*reinterpret_cast<__half2 *>(&hi), bias));
                                pr[2 * e2] = lo;
                                pr[2 * e2 + 1] = hi;
                            }
                            const int chunk = (b2 & 1) * 4 + cq;  // 16-byte chunk of the 128-byte row
                            *reinterpret_cast<uint4 *>(rowdst + ((chunk ^ (r & 7)) << 4)) =
                                make_uint4(pr[0], pr[1], pr[2], pr[3]);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(ptx::smem_u32(&B.st_full[st]));
                    ++w_it;
                }
                }
                ptx::mbar_arrive(ptx::smem_u32(&B.raw_empty[ri]));
                ++sb_it;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // 16 warps: warp w reads TMEM lanes 32*(w%4).. (one activation row per thread)
        // and one quarter of the 128 columns (32 weight rows).  Slots arrive in pairs;
        // both are read (16 columns at a time) and the pair is handed back before the
        // next pair is awaited.  The waits suspend: 16 warps probing the barrier take issue
        // slots from the unpack warps (Q6_K at 151936 x 5120, m = 512: 3.45 -> 3.29 ms;
        // the other formats unchanged).  The segment's total stays in registers.
        regs_inc<kRegsEpilogue>();
        const int ew = warp - kEpiWarp0;  // 0..15
        const int cq = ew >> 2;           // column quarter: columns 32cq .. 32cq+31
        const int qd = warp & 3;          // TMEM lane quarter this warp may access
        const int tl = 32 * qd + lane;    // activation row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        int64_t u = ubeg;
        Seg sg;
        uint32_t ge = 0, sd_it = 0;
        int seg_i = 0;
        bool ok = true;
        while (ok && next_seg(a, u, uend, sg)) {
            float2 tot[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) tot[i] = make_float2(0.f, 0.f);
            for (int64_t sb = sg.s0; ok && sb < sg.s1; ++sb) {
                const uint32_t sdi = sd_it & 1;
                if (!ptx::mbar_wait(ptx::smem_u32(&B.sd_full[sdi]), (sd_it >> 1) & 1, abortp)) {
                    ok = false;
                    break;
                }
                // the row's 8 d8 values as two 16-byte chunks; the tile comes with the 32-byte
                // swizzle (chunk c of row tl at chunk c ^ (tl >> 2 & 1)), so the 8 lanes of a
                // quarter warp read 8 different bank groups
                const uint8_t *dxrow = smem + kOffDX + sdi * 4096 + tl * 32;
                const int dxsw = (tl >> 2) & 1;
                auto dxv = [&](int c) { return *reinterpret_cast<const float4 *>(dxrow + ((c ^ dxsw) << 4)); };
                const float *dd = reinterpret_cast<const float *>(smem + kOffDD + sdi * F::kDDBytes);
                if constexpr (F::kScaleD) {
                    float2 acc[16];  // columns 2i, 2i+1 of this thread's 32
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < kGroups; ++j) {
                        const uint32_t e = ge & 1;
                        if (!ptx::mbar_wait(ptx::smem_u32(&B.acc_full[e]), (ge >> 1) & 1, abortp)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const float4 d4 = dxv(j >> 1);
                        const float d8a = (j & 1) ? d4.z : d4.x, d8b = (j & 1) ? d4.w : d4.y;
#pragma unroll
                        for (int b2 = 0; b2 < kPair; ++b2) {
                            const float2 dg = b2 ? make_float2(d8b, d8b) : make_float2(d8a, d8a);
#pragma unroll
                            for (int hv = 0; hv < 2; ++hv) {
                                float v[16];
                                ptx::tmem_ld_32x32b_x16(lane_base + (kPair * e + b2) * kTN + 32 * cq + 16 * hv, v);
                                ptx::tmem_ld_wait();
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    acc[8 * hv + i] = __ffma2_rn(dg, make_float2(v[2 * i], v[2 * i + 1]), acc[8 * hv + i]);
                            }
                        }
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&B.acc_empty[e]));
                        ++ge;
                    }
                    if (!ok) break;
                    if constexpr (F::kMin) {
                        // the superblock's fold: total += d * acc + (-dmin) * minslot, with d
                        // and -dmin the fp16 factors of this thread's 32 weight rows.  d * acc
                        // is added before the min slot is awaited, and each factor comes as
                        // four 16-byte loads issued together (loaded one column group at a
                        // time after the wait, they held each superblock up by ~1K cycles).
                        const uint4 *dh = reinterpret_cast<const uint4 *>(dd) + 4 * cq;
                        const uint4 *mh = reinterpret_cast<const uint4 *>(dd) + 16 + 4 * cq;
                        uint4 hq[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) hq[i] = dh[i];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const __half2 *h = reinterpret_cast<const __half2 *>(&hq[i]);
#pragma unroll
                            for (int p = 0; p < 4; ++p)
                                tot[4 * i + p] = __ffma2_rn(__half22float2(h[p]), acc[4 * i + p], tot[4 * i + p]);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) hq[i] = mh[i];
                        const uint32_t e = ge & 1;
                        if (!ptx::mbar_wait(ptx::smem_u32(&B.acc_full[e]), (ge >> 1) & 1, abortp)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        float vm[32];
                        ptx::tmem_ld_32x32b_x32(lane_base + kPair * e * kTN + 32 * cq, vm);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const __half2 *h = reinterpret_cast<const __half2 *>(&hq[i]);
#pragma unroll
                            for (int p = 0; p < 4; ++p)
                                tot[4 * i + p] = __ffma2_rn(__half22float2(h[p]),
                                                            make_float2(vm[8 * i + 2 * p], vm[8 * i + 2 * p + 1]),
                                                            tot[4 * i + p]);
                        }
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&B.acc_empty[e]));
                        ++ge;
                    } else {
                        // Q6_K: total += d * acc, d the fp16 factor of each weight row (column)
                        const uint4 *dh = reinterpret_cast<const uint4 *>(dd) + 4 * cq;
                        uint4 hq[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) hq[i] = dh[i];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const __half2 *h = reinterpret_cast<const __half2 *>(&hq[i]);
#pragma unroll
                            for (int p = 0; p < 4; ++p)
                                tot[4 * i + p] = __ffma2_rn(__half22float2(h[p]), acc[4 * i + p], tot[4 * i + p]);
                        }
                    }
                } else {
                    // Q8_0 / Q4_0: total += (d8 * w) * slot with w the block's d of the slot's
                    // row, two columns per packed op
#pragma unroll
                    for (int j = 0; j < kGroups; ++j) {
                        const uint32_t e = ge & 1;
                        if (!ptx::mbar_wait(ptx::smem_u32(&B.acc_full[e]), (ge >> 1) & 1, abortp)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
#pragma unroll
                        for (int b2 = 0; b2 < kPair; ++b2) {
                            const int G = kPair * j + b2;
                            const int g32 = G * F::kSub / 32;  // the sub-block's 32-block: its d8
                            const float4 d4 = dxv(g32 >> 2);
                            const float dgs = (g32 & 3) == 0 ? d4.x : (g32 & 3) == 1 ? d4.y : (g32 & 3) == 2 ? d4.z : d4.w;
                            const float2 d8 = make_float2(dgs, dgs);
                            // the block's fp16 d of this thread's 32 weight rows, loaded together
                            const uint4 *dwg = reinterpret_cast<const uint4 *>(dd) + G * 16 + 4 * cq;
                            uint4 hq[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) hq[i] = dwg[i];
#pragma unroll
                            for (int hv = 0; hv < 2; ++hv) {
                                float v[16];
                                ptx::tmem_ld_32x32b_x16(lane_base + (kPair * e + b2) * kTN + 32 * cq + 16 * hv, v);
                                ptx::tmem_ld_wait();
#pragma unroll
                                for (int i = 0; i < 2; ++i) {
                                    const __half2 *h = reinterpret_cast<const __half2 *>(&hq[2 * hv + i]);
#pragma unroll
                                    for (int p = 0; p < 4; ++p) {
                                        const float2 sc = __fmul2_rn(d8, __half22float2(h[p]));
                                        tot[8 * hv + 4 * i + p] = __ffma2_rn(
                                            sc, make_float2(v[8 * i + 2 * p], v[8 * i + 2 * p + 1]), tot[8 * hv + 4 * i + p]);
                                    }
                                }
                            }
                        }
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&B.acc_empty[e]));
                        ++ge;
                    }
                    if (!ok) break;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&B.sd_empty[sdi]));
                ++sd_it;
            }
            if (!ok) break;
            store_segment(a, sg, seg_i, tl, cq, tot, T == QMM_Q6_K && a.q6_groups);
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

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_q4k_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xmin,
                       const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_w2, TcArgs a) {
    gemm_tc_body<QMM_Q4_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w2, a);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_q5k_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xmin,
                       const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_w2, TcArgs a) {
    gemm_tc_body<QMM_Q5_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w2, a);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_q80_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xmin,
                       const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_w2, TcArgs a) {
    gemm_tc_body<QMM_Q8_0>(tm_x, tm_xmin, tm_dx, tm_w, tm_w2, a);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_q40_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xmin,
                       const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_w2, TcArgs a) {
    gemm_tc_body<QMM_Q4_0>(tm_x, tm_xmin, tm_dx, tm_w, tm_w2, a);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_q6k_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xmin,
                       const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_w2, TcArgs a) {
    gemm_tc_body<QMM_Q6_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w2, a);
}

// Four int8 codes (one word) as two fp16 pairs: (0, 1), (2, 3), or with perm4 (0, 2), (1, 3).
__device__ __forceinline__ uint2 codes4_f16(uint32_t w, int perm4) {
    const int8_t *c = reinterpret_cast<const int8_t *>(&w);
    const int i1 = perm4 ? 2 : 1, i2 = perm4 ? 1 : 2;
    return make_uint2(h2bits(__halves2half2(__int2half_rn(c[0]), __int2half_rn(c[i1]))),
                      h2bits(__halves2half2(__int2half_rn(c[i2]), __int2half_rn(c[3]))));
}

// q8_1 blocks -> fp16 activation codes [m][k], fp32 d8 [m][k/32], fp16 s tile
// [m][k/256][16] (8 values then 8 zeros) for the tensor-core GEMM.  perm4: every 4 codes in
// the order 0 2 1 3 (the order of the Q4_K unpack; a slot's dot is the same in any order).
__global__ void tc_prep_kernel(const uint8_t *__restrict__ xq, int64_t m, int k, __half *__restrict__ xh,
                               float *__restrict__ dx, __half *__restrict__ smin, int *status, int perm4) {
    const int nb32 = k / 32;
    const int64_t total = m * nb32;
    if (blockIdx.x == 0 && threadIdx.x == 0 && status) *status = (int)QMM_OK;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = i / nb32;
        const int b = (int)(i - r * nb32);
        const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + i * kQ81Bytes);
        const uint32_t dsw = ldg4(src);
        uint4 *dst = reinterpret_cast<uint4 *>(xh + r * k + 32 * b);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint2 a = codes4_f16(ldg4(src + 1 + 2 * j), perm4), b = codes4_f16(ldg4(src + 2 + 2 * j), perm4);
            dst[j] = make_uint4(a.x, a.y, b.x, b.y);
        }
        dx[i] = half_lo(dsw);
        __half *sp = smin + (r * (nb32 / 8) + b / 8) * 16;
        sp[b % 8] = __ushort_as_half((unsigned short)(dsw >> 16));
        sp[8 + b % 8] = __ushort_as_half(0);
    }
}

// Expert-grouped variant of tc_prep_kernel: sorted row j holds activation row
// perm[j] / x_div of xq (x_div = top_k: the pair's token; 1: one row per pair).
// Rows of invalid pairs are left as they are:
// the GEMM computes them but never stores them.
__global__ void tc_prep_gather_kernel(const uint8_t *__restrict__ xq, int k, const int32_t *__restrict__ perm,
                                      const int32_t *__restrict__ bounds, int E, int x_div, int64_t n_pairs,
                                      __half *__restrict__ xh, float *__restrict__ dx, __half *__restrict__ smin,
                                      int perm4) {
    const int nb32 = k / 32;
    const int64_t nvalid = bounds[E];
    const int64_t total = n_pairs * nb32;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t j = i / nb32;
        if (j >= nvalid) continue;
        const int b = (int)(i - j * nb32);
        const int64_t tok = perm[j] / x_div;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + (tok * nb32 + b) * kQ81Bytes);
        const uint32_t dsw = ldg4(src);
        uint4 *dst = reinterpret_cast<uint4 *>(xh + j * k + 32 * b);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint2 a = codes4_f16(ldg4(src + 1 + 2 * q), perm4), b = codes4_f16(ldg4(src + 2 + 2 * q), perm4);
            dst[q] = make_uint4(a.x, a.y, b.x, b.y);
        }
        dx[i] = half_lo(dsw);
        __half *sp = smin + (j * (nb32 / 8) + b / 8) * 16;
        sp[b % 8] = __ushort_as_half((unsigned short)(dsw >> 16));
        sp[8 + b % 8] = __ushort_as_half(0);
    }
}

// stream-K fixup: every tile that several CTAs share is summed in CTA order.
// Grid (tiles, 16): CTA (t, part) owns 8 activation rows of tile t, one float4 of
// 4 weight columns per thread.
constexpr int kFixupParts = 16;
__global__ void __launch_bounds__(256) tc_fixup_kernel(TcArgs a) {
    int64_t ntiles = int64_t(gridDim.x);  // dense: one block column per tile
    if (a.tiles) {  // grouped: the tile count is on the device; the grid strides over it
        ntiles = int64_t(*a.ntiles) * a.tiles_n;
        a.nwork = ntiles * a.nsb;
        if (whole_tiles(a)) return;  // every tile was written whole
    }
    auto owner = [&](int64_t uu) {
        int64_t c = uu * a.ctas / a.nwork;
        while (c + 1 < a.ctas && a.nwork * (c + 1) / a.ctas <= uu) ++c;
        while (c > 0 && a.nwork * c / a.ctas > uu) --c;
        return c;
    };
    const int tl = blockIdx.y * (kTM / kFixupParts) + (threadIdx.x >> 5);  // 8 rows per CTA
    const int cl = 4 * (threadIdx.x & 31);                                 // 4 columns per thread
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t u0 = t * a.nsb, u1 = u0 + a.nsb - 1;
        const int64_t c0 = owner(u0), c1 = owner(u1);
        if (c0 == c1) continue;  // the tile was written whole by one CTA
        const TileInfo ti = resolve_tile(a, t);
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t c = c0; c <= c1; ++c) {
            const int64_t cb = a.nwork * c / a.ctas;
            if (a.nwork * (c + 1) / a.ctas == cb) continue;  // fewer units than CTAs: c owns nothing
            const int slotidx = (cb / a.nsb == t) ? 0 : 1;  // tile t is this CTA's first segment?
            const float4 p = *reinterpret_cast<const float4 *>(a.partial + ((c * 2 + slotidx) * kTM + tl) * kTN + cl);
            s.x += p.x;
            s.y += p.y;
            s.z += p.z;
            s.w += p.w;
        }
        const int64_t col = ti.col0 + cl;
        if (tl >= ti.rows) continue;
        const int64_t yrow = a.tiles ? int64_t(a.perm[ti.m0 + tl]) : int64_t(ti.m0 + tl);
        float *dst = a.y + yrow * a.n + col;
        const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (col + j < a.n) dst[j] = sv[j];
    }
}

// ---------------------------------------------------------------- host side

bool make_map_2d(CUtensorMap *map, CUtensorMapDataType dt, int esize, const void *base, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    return tc_make_map_2d(map, dt, esize, base, inner, outer, inner * esize, box_inner, box_outer, sw);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The test switch of qmm_set_test_fault, copied into a launch's arguments.
void tc_test_fault(TcArgs &a) {
    a.withhold_x = test_fault_mode() == 1 ? 1 : 0;
    a.mma_wait_cycles = a.withhold_x ? 100000LL : ptx::kWaitCycles;
}

struct TcLayout {
    size_t status, xh, dx, smin, partial, total;
};
TcLayout tc_layout(int64_t m, int64_t k, int64_t partial_ctas) {
    TcLayout L{};
    size_t off = 256;
    L.status = 0;
    L.xh = off;
    off = align256(off + size_t(m) * k * 2);
    L.dx = off;
    off = align256(off + size_t(m) * (k / 32) * 4);
    L.smin = off;
    off = align256(off + size_t(m) * (k / 256) * 32);
    L.partial = off;
    off = align256(off + size_t(partial_ctas) * 2 * kTM * kTN * 4);
    L.total = off;
    return L;
}

}  // namespace

// Bytes of one weight row, and the raw map of `rows` weight rows: one box is the 256 k
// values of 128 rows (Q8_0 read as uint16, so that a step's 272 bytes are a box of 136).
// Q6_K has no map: its raw warp bulk-copies from W, which must start on a 16-byte boundary.
// The Q4_K unpack writes every 4 weights in the order 0 2 1 3; its activations are staged so.
int tc_perm4(qmm_type t) { return t == QMM_Q4_K ? 1 : 0; }

int64_t tc_row_bytes(qmm_type t, int64_t k) { return (k / 256) * block_bytes(t) * (256 / block_elems(t)); }

// Q6_K raw superblocks by row-group boxes (TcArgs::q6_groups): rows in whole groups of 8
// whose 8 row lengths make a multiple of 16 bytes
bool q6_row_groups(qmm_type t, int64_t rows, int64_t row_bytes) {
    return t == QMM_Q6_K && rows % 8 == 0 && (8 * row_bytes) % 16 == 0;
}

bool tc_weight_map(qmm_type t, const void *W, int64_t rows, int64_t k, CUtensorMap *tm_w, int64_t stride = 0) {
    const int64_t row_bytes = stride > 0 ? stride : tc_row_bytes(t, k);
    if (t == QMM_Q8_0)
        return make_map_2d(tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, W, row_bytes / 2, rows, TcFmt<QMM_Q8_0>::kRawRow / 2,
                           kTN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (t == QMM_Q6_K) {
        // rows in whole groups of 8: each group is one row of the map (8 row lengths, a
        // multiple of 16 bytes), read as 240-byte boxes of 16 groups; otherwise the kernel
        // copies each row's window itself
        memset(tm_w, 0, sizeof(*tm_w));
        if ((reinterpret_cast<uintptr_t>(W) & 15u) != 0) return false;
        if (!q6_row_groups(t, rows, row_bytes)) return true;
        return make_map_2d(tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, uint64_t(8 * row_bytes), uint64_t(rows / 8),
                           TcFmt<QMM_Q6_K>::kRawRow, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    // Q4_K, Q5_K and Q4_0: a box of one superblock's raw bytes (144, 176, 144) per row
    return make_map_2d(tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, row_bytes, rows, (uint32_t)tc_row_bytes(t, 256), kTN,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
}

int64_t gemm_tc_tile_m(int64_t) { return kTM; }

bool gemm_tc_supported(qmm_type t, int64_t n, int64_t k, int64_t m, int64_t stride) {
    if (!(k % 256 == 0 && n > 0 && m > 0 && m <= (int64_t(1) << 30))) return false;
    if (t == QMM_Q4_K || t == QMM_Q5_K || t == QMM_Q8_0 || t == QMM_Q4_0) return true;
    // Q6_K's raw windows reach up to 14 bytes past a row's last block: with natural rows the
    // last row's window must end at the end of W, which n % 8 == 0 gives; rows padded by
    // qmm_repack_aligned keep every window inside its own row
    return t == QMM_Q6_K && (n % 8 == 0 || (stride > 0 && stride >= aligned_row_bytes(t, k)));
}

int64_t aligned_row_bytes(qmm_type t, int64_t k) {
    if (block_bytes(t) <= 0 || k <= 0 || k % block_elems(t)) return 0;
    const int64_t rb = (k / block_elems(t)) * block_bytes(t);
    // Q6_K: room for the 14 bytes that a superblock's 16-byte-aligned copy window can overrun
    return ((rb + (t == QMM_Q6_K ? 14 : 0) + 15) / 16) * 16;
}

size_t gemm_tc_workspace_bytes(qmm_type t, int64_t n, int64_t k, int64_t m, int64_t stride) {
    if (!gemm_tc_supported(t, n, k, m, stride)) return 0;
    const int64_t nwork = ((n + kTN - 1) / kTN) * ((m + kTM - 1) / kTM) * (k / 256);
    return tc_layout(m, k, std::min<int64_t>(kMaxPartialCtas, nwork)).total;
}

namespace {

// Launch the GEMM kernel of format T (and the fixup pass when asked) once the maps are built.
template <int T>
cudaError_t run_tc(const CUtensorMap &tm_x, const CUtensorMap &tm_xmin, const CUtensorMap &tm_dx,
                   const CUtensorMap &tm_w, const CUtensorMap &tm_w2, const TcArgs &args, int ctas, int64_t fixup_tiles,
                   cudaStream_t st) {
    auto kern = T == QMM_Q4_K   ? gemm_tc_q4k_kernel
                : T == QMM_Q5_K ? gemm_tc_q5k_kernel
                : T == QMM_Q6_K ? gemm_tc_q6k_kernel
                : T == QMM_Q4_0 ? gemm_tc_q40_kernel
                                : gemm_tc_q80_kernel;
    constexpr uint32_t smem = TcMap<T>::kSmemAlloc;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    // The setmaxnreg split hands out exactly kThreads x kLaunchRegs registers; a build that
    // launches with fewer registers per thread would leave setmaxnreg.inc waiting forever.
    static int launch_regs = -1;
    if (launch_regs < 0) {
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return cudaErrorInvalidValue;
        launch_regs = fa.numRegs;
    }
    if (launch_regs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    kern<<<ctas, kThreads, smem, st>>>(tm_x, tm_xmin, tm_dx, tm_w, tm_w2, args);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (fixup_tiles > 0) {
        // dense: one block column per tile; grouped (the count known on the device only, up
        // to fixup_tiles): a bounded grid that strides over the tiles
        const int64_t gx = args.tiles ? std::min<int64_t>(fixup_tiles, int64_t(device_sm_count()) * 2) : fixup_tiles;
        tc_fixup_kernel<<<dim3((unsigned)gx, kFixupParts), 256, 0, st>>>(args);
        e = cudaGetLastError();
    }
    return e;
}

bool make_act_maps(CUtensorMap &tm_x, CUtensorMap &tm_xmin, CUtensorMap &tm_dx, const __half *xh, const float *dx,
                   const __half *smin, int64_t rows, int64_t k) {
    return make_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xh, k, rows, 64, kTM, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map_2d(&tm_xmin, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, smin, (k / 256) * 16, rows, 16, kTM,
                       CU_TENSOR_MAP_SWIZZLE_32B) &&
           make_map_2d(&tm_dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dx, k / 32, rows, 8, kTM, CU_TENSOR_MAP_SWIZZLE_32B);
}

}  // namespace

// More whole tiles than SMs: one persistent CTA per SM takes a contiguous run of them
// (mode 3), so each SM's pipeline runs on from one tile into the next instead of being
// refilled by a new CTA (Q4_K 14336 x 4096 at m = 512: 146 -> 141 us, m = 2048: 572 ->
// 544 us; Q6_K 151936 x 5120: 3.30 -> 3.07 ms; Q4_0: 184 -> 179 us).  Q5_K stays on one CTA
// per tile, which balances better across SMs for its longer unpack (187 against 198 us).
static int persistent_whole_tiles(qmm_type t, const qmm_gemm_plan &p, int nsm, TcArgs &args) {
    if (p.stream_k || p.ntiles <= nsm || t == QMM_Q5_K) return p.ctas;
    args.stream_k = 3;
    args.ctas = nsm;
    return nsm;
}

cudaError_t launch_gemm_tc(qmm_type t, const void *W, int64_t n, int64_t k, const void *xq, int64_t m, float *y,
                           void *ws, size_t ws_bytes, int stream_k_mode, cudaStream_t st, int64_t stride) {
    if (!gemm_tc_supported(t, n, k, m, stride)) return cudaErrorNotSupported;
    qmm_gemm_plan p{};
    const int nsm = std::min(device_sm_count(), kMaxPartialCtas);
    if (qmm_plan_gemm(t, n, k, m, nsm, stream_k_mode, &p) != QMM_OK) return cudaErrorInvalidValue;
    const TcLayout L = tc_layout(m, k, std::min<int64_t>(kMaxPartialCtas, p.nwork));
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    int *status = reinterpret_cast<int *>(base + L.status);
    __half *xh = reinterpret_cast<__half *>(base + L.xh);
    float *dx = reinterpret_cast<float *>(base + L.dx);
    __half *smin = reinterpret_cast<__half *>(base + L.smin);

    const int64_t nblk = m * (k / 32);
    const int pgrid = (int)std::min<int64_t>((nblk + 255) / 256, int64_t(device_sm_count()) * 8);
    tc_prep_kernel<<<std::max(pgrid, 1), 256, 0, st>>>(static_cast<const uint8_t *>(xq), m, (int)k, xh, dx, smin,
                                                      status, tc_perm4(t));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap tm_x, tm_xmin, tm_dx, tm_w;
    const int64_t row_bytes = stride > 0 ? stride : tc_row_bytes(t, k);
    if (!make_act_maps(tm_x, tm_xmin, tm_dx, xh, dx, smin, m, k) || !tc_weight_map(t, W, n, k, &tm_w, stride))
        return cudaErrorInvalidValue;

    TcArgs args{};
    tc_test_fault(args);
    args.q6_groups = q6_row_groups(t, n, row_bytes) ? 1 : 0;
    args.W = static_cast<const uint8_t *>(W);
    args.n = n;
    args.m = m;
    args.k = (int)k;
    args.row_bytes = row_bytes;
    args.y = y;
    args.partial = reinterpret_cast<float *>(base + L.partial);
    args.status = status;
    args.tiles_n = p.tiles_n;
    args.nsb = p.iters_per_tile;
    args.nwork = p.nwork;
    args.ctas = p.ctas;
    args.stream_k = p.stream_k;
    const int ctas = persistent_whole_tiles(t, p, nsm, args);
    const int64_t fixup_tiles = (p.stream_k && p.fixup) ? p.ntiles : 0;
    if (t == QMM_Q8_0) return run_tc<QMM_Q8_0>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup_tiles, st);
    if (t == QMM_Q4_0) return run_tc<QMM_Q4_0>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup_tiles, st);
    if (t == QMM_Q5_K) return run_tc<QMM_Q5_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup_tiles, st);
    if (t == QMM_Q6_K) return run_tc<QMM_Q6_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup_tiles, st);
    return run_tc<QMM_Q4_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup_tiles, st);
}

// ---------------------------------------------------------------- fused gate/up + SwiGLU

bool gemm_tc_glu_supported(qmm_type t, int64_t n_out, int64_t k, int64_t m) {
    return t == QMM_Q4_K && n_out > 0 && gemm_tc_supported(t, 2 * n_out, k, m);
}

size_t gemm_tc_glu_workspace_bytes(qmm_type t, int64_t n_out, int64_t k, int64_t m) {
    return gemm_tc_glu_supported(t, n_out, k, m) ? tc_layout(m, k, 0).total : 0;
}

// Whole tiles only (the GLU needs both complete dots in one thread, [MMQ] section
// "「分专家」与「整批」之间: host 侧的代价"): one tile per CTA, or runs of whole tiles on
// persistent CTAs when there are more tiles than SMs.
cudaError_t launch_gemm_tc_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n_out, int64_t k, const void *xq,
                               int64_t m, float *y, void *ws, size_t ws_bytes, cudaStream_t st) {
    // Wu == nullptr: Wg holds the gate and up rows interleaved (2 n_out rows)
    const bool packed = Wu == nullptr;
    if (!gemm_tc_glu_supported(t, n_out, k, m)) return cudaErrorNotSupported;
    qmm_gemm_plan p{};
    const int nsm = std::min(device_sm_count(), kMaxPartialCtas);
    if (qmm_plan_gemm(t, 2 * n_out, k, m, nsm, 1, &p) != QMM_OK || p.stream_k) return cudaErrorInvalidValue;
    const TcLayout L = tc_layout(m, k, 0);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    int *status = reinterpret_cast<int *>(base + L.status);
    __half *xh = reinterpret_cast<__half *>(base + L.xh);
    float *dx = reinterpret_cast<float *>(base + L.dx);
    __half *smin = reinterpret_cast<__half *>(base + L.smin);
    const int64_t nblk = m * (k / 32);
    const int pgrid = (int)std::min<int64_t>((nblk + 255) / 256, int64_t(device_sm_count()) * 8);
    tc_prep_kernel<<<std::max(pgrid, 1), 256, 0, st>>>(static_cast<const uint8_t *>(xq), m, (int)k, xh, dx, smin,
                                                      status, 1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t row_bytes = (k / 256) * kQ4KBytes;
    CUtensorMap tm_x, tm_xmin, tm_dx, tm_w, tm_w2;
    if (!make_act_maps(tm_x, tm_xmin, tm_dx, xh, dx, smin, m, k)) return cudaErrorInvalidValue;
    if (packed) {
        if (!make_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wg, row_bytes, 2 * n_out, kQ4KBytes, kTN,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        tm_w2 = tm_w;
    } else if (!make_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wg, row_bytes, n_out, kQ4KBytes, kTN / 2,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
               !make_map_2d(&tm_w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wu, row_bytes, n_out, kQ4KBytes, kTN / 2,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TcArgs args{};
    tc_test_fault(args);
    args.W = static_cast<const uint8_t *>(Wg);
    args.n = 2 * n_out;
    args.m = m;
    args.k = (int)k;
    args.row_bytes = row_bytes;
    args.y = y;
    args.partial = nullptr;
    args.status = status;
    args.tiles_n = p.tiles_n;
    args.nsb = p.iters_per_tile;
    args.nwork = p.nwork;
    args.ctas = p.ctas;
    args.stream_k = 0;
    args.n_out = n_out;
    args.glu_packed = packed ? 1 : 0;
    const int ctas = persistent_whole_tiles(t, p, nsm, args);
    return run_tc<QMM_Q4_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w2, args, ctas, 0, st);
}

// ---------------------------------------------------------------- expert-grouped mode

bool gemm_tc_grouped_supported(qmm_type t, int64_t n_experts, int64_t n, int64_t k) {
    // the experts' rows are one W of n_experts * n rows, so the dense conditions apply per
    // expert (Q6_K: n % 8 == 0 keeps every expert's rows, and the end of W, on 16 bytes)
    return n_experts > 0 && n_experts * n < (int64_t(1) << 31) && gemm_tc_supported(t, n, k, 1);
}

size_t gemm_tc_grouped_bytes(int64_t n_pairs, int64_t k) {
    return tc_layout(n_pairs, k, device_sm_count() < kMaxPartialCtas ? device_sm_count() : kMaxPartialCtas).total;
}

cudaError_t launch_gemm_tc_grouped(qmm_type t, const void *W, int64_t n_experts, int64_t n, int64_t k, const void *xq,
                                   int64_t x_div, int64_t n_pairs, float *y, const MoETile *tiles,
                                   const int32_t *ntiles, int64_t max_token_tiles, const int32_t *bounds,
                                   const int32_t *perm, int *status, void *ws, size_t ws_bytes, cudaStream_t st) {
    const int ctas = std::min(device_sm_count(), kMaxPartialCtas);
    const TcLayout L = tc_layout(n_pairs, k, ctas);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    __half *xh = reinterpret_cast<__half *>(base + L.xh);
    float *dx = reinterpret_cast<float *>(base + L.dx);
    __half *smin = reinterpret_cast<__half *>(base + L.smin);

    const int64_t nblk = n_pairs * (k / 32);
    const int pgrid = (int)std::min<int64_t>((nblk + 255) / 256, int64_t(device_sm_count()) * 8);
    tc_prep_gather_kernel<<<std::max(pgrid, 1), 256, 0, st>>>(static_cast<const uint8_t *>(xq), (int)k, perm, bounds,
                                                             (int)n_experts, (int)x_div, n_pairs, xh, dx, smin,
                                                             tc_perm4(t));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap tm_x, tm_xmin, tm_dx, tm_w;
    if (!gemm_tc_grouped_supported(t, n_experts, n, k) || !make_act_maps(tm_x, tm_xmin, tm_dx, xh, dx, smin, n_pairs, k) ||
        !tc_weight_map(t, W, n_experts * n, k, &tm_w))
        return cudaErrorInvalidValue;

    TcArgs args{};
    tc_test_fault(args);
    args.W = static_cast<const uint8_t *>(W);
    args.n = n;
    args.m = n_pairs;
    args.k = (int)k;
    args.row_bytes = tc_row_bytes(t, k);
    args.q6_groups = q6_row_groups(t, n_experts * n, args.row_bytes) ? 1 : 0;
    args.y = y;
    args.partial = reinterpret_cast<float *>(base + L.partial);
    args.status = status;
    args.tiles_n = (n + kTN - 1) / kTN;
    args.nsb = k / 256;
    args.nwork = 0;  // read from the device tile count by the kernels
    args.ctas = ctas;
    args.stream_k = 2;
    args.tiles = tiles;
    args.ntiles = ntiles;
    args.bounds = bounds;
    args.perm = perm;
    const int64_t fixup = max_token_tiles * args.tiles_n;
    switch (t) {
    case QMM_Q8_0: return run_tc<QMM_Q8_0>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup, st);
    case QMM_Q4_0: return run_tc<QMM_Q4_0>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup, st);
    case QMM_Q5_K: return run_tc<QMM_Q5_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup, st);
    case QMM_Q6_K: return run_tc<QMM_Q6_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup, st);
    default: return run_tc<QMM_Q4_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w, args, ctas, fixup, st);
    }
}

// The fused gate/up form of the grouped GEMM (Q4_K): the tile space of an expert has 2 n
// columns, column 2j its gate row j (tm_w over the experts' E n gate rows) and 2j + 1 its
// up row j (tm_w2); a tile's raw rows are 64 gate rows and the 64 up rows of the same
// outputs, and every tile is computed whole by one CTA (the GLU needs both dots).
bool gemm_tc_grouped_glu_supported(qmm_type t, int64_t n_experts, int64_t n, int64_t k) {
    return t == QMM_Q4_K && n_experts > 0 && n_experts * n < (int64_t(1) << 30) && k % 256 == 0 && n > 0;
}

cudaError_t launch_gemm_tc_grouped_glu(qmm_type t, const void *Wg, const void *Wu, int64_t n_experts, int64_t n,
                                       int64_t k, const void *xq, int64_t x_div, int64_t n_pairs, float *y,
                                       const MoETile *tiles, const int32_t *ntiles, const int32_t *bounds,
                                       const int32_t *perm, int *status, void *ws, size_t ws_bytes, cudaStream_t st) {
    if (!gemm_tc_grouped_glu_supported(t, n_experts, n, k)) return cudaErrorNotSupported;
    const int ctas = std::min(device_sm_count(), kMaxPartialCtas);
    const TcLayout L = tc_layout(n_pairs, k, 0);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    __half *xh = reinterpret_cast<__half *>(base + L.xh);
    float *dx = reinterpret_cast<float *>(base + L.dx);
    __half *smin = reinterpret_cast<__half *>(base + L.smin);
    const int64_t nblk = n_pairs * (k / 32);
    const int pgrid = (int)std::min<int64_t>((nblk + 255) / 256, int64_t(device_sm_count()) * 8);
    tc_prep_gather_kernel<<<std::max(pgrid, 1), 256, 0, st>>>(static_cast<const uint8_t *>(xq), (int)k, perm, bounds,
                                                             (int)n_experts, (int)x_div, n_pairs, xh, dx, smin,
                                                             1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t row_bytes = (k / 256) * kQ4KBytes;
    CUtensorMap tm_x, tm_xmin, tm_dx, tm_w, tm_w2;
    if (!make_act_maps(tm_x, tm_xmin, tm_dx, xh, dx, smin, n_pairs, k) ||
        !make_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wg, row_bytes, n_experts * n, kQ4KBytes, kTN / 2,
                     CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map_2d(&tm_w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wu, row_bytes, n_experts * n, kQ4KBytes, kTN / 2,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TcArgs args{};
    tc_test_fault(args);
    args.W = static_cast<const uint8_t *>(Wg);
    args.n = 2 * n;  // tile space: gate and up columns of every output
    args.m = n_pairs;
    args.k = (int)k;
    args.row_bytes = row_bytes;
    args.y = y;
    args.partial = nullptr;
    args.status = status;
    args.tiles_n = (2 * n + kTN - 1) / kTN;
    args.nsb = k / 256;
    args.nwork = 0;  // read from the device tile count by the kernels
    args.ctas = ctas;
    args.stream_k = 3;
    args.tiles = tiles;
    args.ntiles = ntiles;
    args.bounds = bounds;
    args.perm = perm;
    args.n_out = n;
    args.glu_packed = 0;
    return run_tc<QMM_Q4_K>(tm_x, tm_xmin, tm_dx, tm_w, tm_w2, args, ctas, 0, st);
}

// ---------------------------------------------------------------- shared with the skinny path

bool tc_make_map_2d(CUtensorMap *map, CUtensorMapDataType dt, int esize, const void *base, uint64_t inner,
                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle sw) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn) return false;
    (void)esize;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qmm
