// qmm_common.cuh -- block formats and shared device helpers of the CUDA path.
//
// Block layouts (see include/qmm.h):
//   q8_1 36 B: fp16 d | fp16 s | int8 q[32]
//   Q4_K 144 B: fp16 d | fp16 dmin | 12 B packed 6-bit scales/mins | 128 B nibbles
//   Q5_K 176 B: fp16 d | fp16 dmin | 12 B scales/mins | qh[32] | 128 B nibbles (the fifth
//               bit of weight 32j + l is bit j of qh[l])
//   Q6_K 210 B: ql[128] | qh[64] | int8 sc[16] | fp16 d
//   Q8_0 34 B: fp16 d | int8 q[32]
//   Q4_0 18 B: fp16 d | 16 B nibbles (byte i: weight i low, weight 16+i high; d*(q-8))
//
// Work is cut into "units" of 64 consecutive k values of one weight row: a quarter
// superblock for Q4_K / Q6_K, two blocks for Q8_0 and Q4_0.  A unit always lines up with two
// q8_1 activation blocks (2u, 2u+1), so one decode routine serves the GEMV and the
// CUDA-core GEMM.  A decoded unit holds
//   q[16]   : 64 signed 8-bit weight codes, 4 per word, in k order
//   isc[4]  : integer scale of each 16-wide quarter (Q4_K: the 6-bit sub-block scale,
//             twice per 32-block; Q6_K: the int8 sub-scale; Q8_0, Q4_0: 1)
//   fd[2]   : fp32 factor of each 32-block's integer dot (Q4_K/Q6_K: d, Q8_0/Q4_0: d of
//             the block)
//   fm[2]   : fp32 factor of each 32-block's min term (Q4_K: dmin*m, otherwise 0)
// so that one 32-block's term is  fd * d8 * (isc0*dot16_0 + isc1*dot16_1) - fm * s8
// ([MMQ] sections "dp4a 路径的 Q4_K" and "Q6_K: 子块尺度与 q8_1 块长错位").
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "qmm.h"

namespace qmm {

constexpr int kQ4KBytes = 144;
constexpr int kQ5KBytes = 176;
constexpr int kQ6KBytes = 210;
constexpr int kQ80Bytes = 34;
constexpr int kQ40Bytes = 18;
constexpr int kQ81Bytes = 36;

struct Unit {
    int q[16];
    int isc[4];
    float fd[2];
    float fm[2];
};

__host__ __device__ constexpr int block_bytes(int t) {
    return t == QMM_Q4_K ? kQ4KBytes
           : t == QMM_Q5_K ? kQ5KBytes
           : t == QMM_Q6_K ? kQ6KBytes
           : t == QMM_Q8_0 ? kQ80Bytes
           : t == QMM_Q4_0 ? kQ40Bytes
                           : 0;
}
__host__ __device__ constexpr int block_elems(int t) { return t == QMM_Q8_0 || t == QMM_Q4_0 ? 32 : 256; }

__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

__device__ __forceinline__ uint4 ldg16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
// ---- q8_1 arithmetic, shared by every kernel that quantizes activations so that all
// of them give the same bytes ([MMQ] section "引言"; [QMM] section "CPU: 先量化激活,
// 再逐行点积"): d = amax/127 and q = round-half-away(v/d), both IEEE fp32 divisions;
// stored d_h = fp16(d), s_h = fp16(float(d_h) * sum q); a block with d == 0 is all zero.
__device__ __forceinline__ float q8_1_scale(float amax) { return __fdiv_rn(amax, 127.0f); }
__device__ __forceinline__ int q8_1_code(float v, float d) { return d != 0.0f ? (int)roundf(__fdiv_rn(v, d)) : 0; }
// The code without a division wherever that cannot change the integer: rd is 1/d within
// 2^-22 (rcp.approx: at most 1 ulp), or 0 where d is outside [2^-100, 2^125) and the quotient
// must be taken (1/d would be subnormal or huge there, and NaN and infinities fail the test).
__device__ __forceinline__ float rcp_guarded(float d) {
    if (!(d >= 0x1p-100f && d < 0x1p+125f)) return 0.0f;
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}
// The q8_1 code of v (the integer of q8_1_code) from that reciprocal.  With |v| <= 127.00001 d,
// t = v rd is within 128 (2^-22 + 2^-24) < 2^-14 of v/d and the IEEE quotient within 2^-17
// of it, so both round to the same integer unless |t| lies within 2^-11 of a half-integer;
// there, or when rd == 0, the quotient is computed.
__device__ __forceinline__ int q8_1_code_rcp(float v, float d, float rd) {
    if (rd == 0.0f) return q8_1_code(v, d);
    const float t = v * rd;
    const float a = fabsf(t);
    if (fabsf((a - truncf(a)) - 0.5f) < 0x1p-11f) return q8_1_code(v, d);
    return (int)rintf(t);
}

// The codes of N values of one block (a lane's share of it), as q8_1_code_rcp gives them
// but with one test per share: r = rint(v rd) is the code unless some product lies within
// 2^-11 of a half-integer (|t - r| > 1/2 - 2^-11) or rd == 0, and then every code of the
// share is taken from the quotient.
template <int N>
__device__ __forceinline__ void q8_1_codes_rcp(const float (&v)[N], float d, float rd, int (&q)[N]) {
    float far = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float t = v[i] * rd;
        const float r = rintf(t);
        far = fmaxf(far, fabsf(t - r));
        q[i] = (int)r;
    }
    if (rd == 0.0f || far > 0.5f - 0x1p-11f) {
#pragma unroll
        for (int i = 0; i < N; ++i) q[i] = q8_1_code(v[i], d);
    }
}

// The (d_h, s_h) word of a block: d_h in the low half, s_h in the high half.
__device__ __forceinline__ uint32_t q8_1_ds_word(float d, int sum_q) {
    if (d == 0.0f) return 0u;
    const __half dh = __float2half_rn(d);
    const __half sh = __float2half_rn(__half2float(dh) * (float)sum_q);
    return uint32_t(__half_as_ushort(dh)) | (uint32_t(__half_as_ushort(sh)) << 16);
}

__device__ __forceinline__ uint32_t ldg4(const void *p) {
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ldg2(const void *p) {
    unsigned short r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// Load policies of the two-phase decode below: rows read from global memory (read-only
// path) or rows staged in shared memory by a bulk copy.
struct LdGlobal {
    static __device__ __forceinline__ uint32_t u32(const void *p) { return ldg4(p); }
    static __device__ __forceinline__ uint32_t u16(const void *p) { return ldg2(p); }
    static __device__ __forceinline__ uint4 u128(const void *p) { return ldg16(p); }
};
struct LdShared {
    static __device__ __forceinline__ uint32_t saddr(const void *p) {
        return static_cast<uint32_t>(__cvta_generic_to_shared(p));
    }
    static __device__ __forceinline__ uint32_t u32(const void *p) {
        uint32_t r;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(saddr(p)));
        return r;
    }
    static __device__ __forceinline__ uint32_t u16(const void *p) {
        unsigned short r;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(saddr(p)));
        return r;
    }
    static __device__ __forceinline__ uint4 u128(const void *p) {
        uint4 r;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                     : "r"(saddr(p)));
        return r;
    }
};

// Q4_K: 6-bit scale and min of sub-block j from the 12 packed bytes held in three
// little-endian words s0 (bytes 0..3), s1 (4..7), s2 (8..11).
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j, int &sc, int &mn) {
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63;
        mn = (s1 >> (8 * j)) & 63;
    } else {
        const int jj = 8 * (j - 4);
        sc = ((s2 >> jj) & 15) | (((s0 >> (jj + 6)) & 3) << 4);
        mn = ((s2 >> (jj + 4)) & 15) | (((s1 >> (jj + 6)) & 3) << 4);
    }
}

// Q4_K unit u (chunk c = u % 4 of superblock u / 4): qs bytes 32c..32c+31 hold
// weights 64c+l (low nibble, sub-block 2c) and 64c+32+l (high nibble, sub-block 2c+1).
__device__ __forceinline__ void decode_q4_K(const uint8_t *row, int u, Unit &o) {
    const uint8_t *blk = row + (u >> 2) * kQ4KBytes;
    const int c = u & 3;
    const uint4 h = ldg16(blk);
    const uint4 a = ldg16(blk + 16 + 32 * c);
    const uint4 b = ldg16(blk + 32 + 32 * c);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        o.q[i] = (int)(w[i] & 0x0f0f0f0fu);
        o.q[8 + i] = (int)((w[i] >> 4) & 0x0f0f0f0fu);
    }
    const float d = half_lo(h.x), dmin = half_hi(h.x);
    int sc0, m0, sc1, m1;
    q4k_scale_min(h.y, h.z, h.w, 2 * c, sc0, m0);
    q4k_scale_min(h.y, h.z, h.w, 2 * c + 1, sc1, m1);
    o.isc[0] = o.isc[1] = sc0;
    o.isc[2] = o.isc[3] = sc1;
    o.fd[0] = o.fd[1] = d;
    o.fm[0] = dmin * (float)m0;
    o.fm[1] = dmin * (float)m1;
}

// Load n 4-byte words starting at a 2-byte aligned address p into w[0..n-1]
// (byte i of the stream = byte p[i]).  Reads whole aligned words only: when p is
// not 4-byte aligned it also touches the 2 bytes before p and the 2 bytes after
// p + 4n, so callers keep [p-2, p+4n+2) inside the buffer.
template <int N>
__device__ __forceinline__ void ldg_words_a2(const uint8_t *p, uint32_t (&w)[N]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *base = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
    if ((a & 3) == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = ldg4(base + i);
    } else {
        uint32_t prev = ldg4(base);
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const uint32_t next = ldg4(base + i + 1);
            w[i] = __funnelshift_r(prev, next, 16);
            prev = next;
        }
    }
}

// Q6_K unit u (v = u % 4 of superblock u / 4) covers weights 64v..64v+63 of the
// superblock: half h = v/2, groups t = 2(v%2) and 2(v%2)+1.  Weight 128h+32t+l takes
// its low 4 bits from ql[64h + 32(t&1) + l] (nibble t>>1) and its top 2 bits from
// bits 2t..2t+1 of qh[32h + l] ([MMQ] section "Q6_K: 6 位数据要多占一半的共享内存").
__device__ __forceinline__ void decode_q6_K(const uint8_t *row, int u, Unit &o) {
    const uint8_t *blk = row + (u >> 2) * kQ6KBytes;
    const int v = u & 3, h = v >> 1, p = v & 1;
    // A block that is not 4-byte aligned starts 2 bytes past a word boundary, so the
    // 2 bytes before it belong to the previous block of the same buffer; every word
    // read below ends at or before byte 210 of this block.
    uint32_t ql[16], qh[8], tail[4];
    ldg_words_a2<16>(blk + 64 * h, ql);        // ql[64h .. 64h+64)
    ldg_words_a2<8>(blk + 128 + 32 * h, qh);   // qh[32h .. 32h+32)
    ldg_words_a2<4>(blk + 192, tail);          // 16 int8 sub-scales
    const int shift_l = 4 * p;
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
        const int t = 2 * p + tt;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = (ql[8 * tt + i] >> shift_l) & 0x0f0f0f0fu;
            const uint32_t hi = ((qh[i] >> (2 * t)) & 0x03030303u) << 4;
            o.q[8 * tt + i] = (int)__vsub4(lo | hi, 0x20202020u);
        }
    }
    const int j0 = 4 * v;  // first 16-wide sub-block of this unit
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = j0 + i;
        o.isc[i] = (int)(int8_t)((tail[j >> 2] >> (8 * (j & 3))) & 0xff);
    }
    const float d = half_lo(ldg2(blk + 208));
    o.fd[0] = o.fd[1] = d;
    o.fm[0] = o.fm[1] = 0.f;
}

// Q8_0 unit u: blocks 2u and 2u+1 (68 bytes at offset 68u of the row).  Rows with an
// odd number of blocks are only 2-byte aligned, so the words come through
// ldg_words_a2: a two-block unit is never the last unit of its row, so the 2 bytes
// after it exist; a single-block unit (odd block count, last unit of the row) reads
// its 34 bytes as 8 words plus one 2-byte load.
__device__ __forceinline__ void decode_q8_0(const uint8_t *row, int u, bool two, Unit &o) {
    const uint8_t *p = row + 68 * u;
    uint32_t w[17];
    if (two) {
        ldg_words_a2<17>(p, w);
    } else {
        uint32_t a[8];
        ldg_words_a2<8>(p, a);
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = a[i];
        w[8] = ldg2(p + 32);
#pragma unroll
        for (int i = 9; i < 17; ++i) w[i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) o.q[i] = (int)__funnelshift_r(w[i], w[i + 1], 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) o.q[8 + i] = (int)w[9 + i];
    o.isc[0] = o.isc[1] = o.isc[2] = o.isc[3] = 1;
    o.fd[0] = half_lo(w[0]);
    o.fd[1] = two ? half_hi(w[8]) : 0.f;
    o.fm[0] = o.fm[1] = 0.f;
}

// Q4_0 codes of one block from its 16 nibble bytes held in 4 words: the low nibbles
// are weights 0..15, the high nibbles weights 16..31 ([MMQ] section "Q4_0: 一个
// get_int_b2 搬进 8 个 4-bit": the two nibble halves of a word go to the front and back
// halves of the block); q - 8 per byte with one __vsub4, as the load side there does.
__device__ __forceinline__ void q4_0_codes(const uint32_t (&qs)[4], int *q8) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        q8[i] = (int)__vsub4(qs[i] & 0x0f0f0f0fu, 0x08080808u);
        q8[4 + i] = (int)__vsub4((qs[i] >> 4) & 0x0f0f0f0fu, 0x08080808u);
    }
}

// Q4_0 unit u: blocks 2u and 2u+1 (36 bytes at offset 36u of the row).  Words w[0..8]
// of a two-block unit: w[0] = d0 | qs0[0..1], w[1..3] = qs0[2..13], w[4] = qs0[14..15] |
// d1, w[5..8] = qs1.  Rows with an odd block count are only 2-byte aligned; as for
// Q8_0, a two-block unit is then never the last of its row, and a single-block unit
// reads its 18 bytes as 4 words plus one 2-byte load.
__device__ __forceinline__ void q4_0_unit_from_words(const uint32_t (&w)[9], bool two, Unit &o) {
    uint32_t qa[4], qb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) qa[i] = __funnelshift_r(w[i], w[i + 1], 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) qb[i] = w[5 + i];
    q4_0_codes(qa, o.q);
    q4_0_codes(qb, o.q + 8);
    o.isc[0] = o.isc[1] = o.isc[2] = o.isc[3] = 1;
    o.fd[0] = half_lo(w[0]);
    o.fd[1] = two ? half_hi(w[4]) : 0.f;
    o.fm[0] = o.fm[1] = 0.f;
}

__device__ __forceinline__ void decode_q4_0(const uint8_t *row, int u, bool two, Unit &o) {
    const uint8_t *p = row + 36 * u;
    uint32_t w[9];
    if (two) {
        ldg_words_a2<9>(p, w);
    } else {
        uint32_t a[4];
        ldg_words_a2<4>(p, a);
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = a[i];
        w[4] = ldg2(p + 16);
#pragma unroll
        for (int i = 5; i < 9; ++i) w[i] = 0u;
    }
    q4_0_unit_from_words(w, two, o);
}

// ---------------------------------------------------------------------------
// Two-phase decode for latency hiding: load_raw<T> issues only the loads of one unit
// (no arithmetic on loaded data, so a caller can put many units' loads in flight
// before the first one is used), convert_raw<T> turns the words into a Unit.
// The loads stay inside the same byte ranges as the one-phase decoders above.

template <int T> struct Raw;
template <> struct Raw<QMM_Q4_K> { uint4 h, a, b; };
template <> struct Raw<QMM_Q5_K> { uint4 h, qh0, qh1, a, b; };
template <> struct Raw<QMM_Q6_K> { uint32_t ql[17], qh[9], sc[5]; uint32_t shift; };
template <> struct Raw<QMM_Q8_0> { uint32_t w[18]; uint32_t shift; bool two; };
template <> struct Raw<QMM_Q4_0> { uint32_t w[10]; uint32_t shift; bool two; };

// units per lane kept in flight by the GEMV
template <int T> constexpr int kRawChunk = T == QMM_Q4_K ? 5 : T == QMM_Q6_K ? 2 : T == QMM_Q4_0 ? 5 : 3;

// Q5_K unit u (chunk c = u % 4 of superblock u / 4): the codes of Q4_K's nibbles, each with
// its fifth bit from the qh plane: weights 64c + l (sub-block 2c) take bit 2c of qh[l],
// weights 64c + 32 + l (sub-block 2c + 1) bit 2c + 1.  a, b: qs bytes 32c..32c+31; q0, q1:
// qh bytes 0..31.
__device__ __forceinline__ void q5k_unit(const uint4 &h, const uint4 &q0, const uint4 &q1, const uint4 &a,
                                         const uint4 &b, int c, Unit &o) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const uint32_t qh[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        o.q[i] = (int)((w[i] & 0x0f0f0f0fu) | (((qh[i] >> (2 * c)) & 0x01010101u) << 4));
        o.q[8 + i] = (int)(((w[i] >> 4) & 0x0f0f0f0fu) | (((qh[i] >> (2 * c + 1)) & 0x01010101u) << 4));
    }
    const float d = half_lo(h.x), dmin = half_hi(h.x);
    int sc0, m0, sc1, m1;
    q4k_scale_min(h.y, h.z, h.w, 2 * c, sc0, m0);
    q4k_scale_min(h.y, h.z, h.w, 2 * c + 1, sc1, m1);
    o.isc[0] = o.isc[1] = sc0;
    o.isc[2] = o.isc[3] = sc1;
    o.fd[0] = o.fd[1] = d;
    o.fm[0] = dmin * (float)m0;
    o.fm[1] = dmin * (float)m1;
}

// Q5_K rows are whole 16-byte units (176-byte blocks): every load is 16 bytes, aligned.
__device__ __forceinline__ void decode_q5_K(const uint8_t *row, int u, Unit &o) {
    const uint8_t *blk = row + (u >> 2) * kQ5KBytes;
    const int c = u & 3;
    q5k_unit(ldg16(blk), ldg16(blk + 16), ldg16(blk + 32), ldg16(blk + 48 + 32 * c), ldg16(blk + 64 + 32 * c), c, o);
}

template <class Ld = LdGlobal>
__device__ __forceinline__ void load_raw(const uint8_t *row, int u, int, Raw<QMM_Q5_K> &r) {
    const uint8_t *blk = row + (u >> 2) * kQ5KBytes;
    const int c = u & 3;
    r.h = Ld::u128(blk);
    r.qh0 = Ld::u128(blk + 16);
    r.qh1 = Ld::u128(blk + 32);
    r.a = Ld::u128(blk + 48 + 32 * c);
    r.b = Ld::u128(blk + 64 + 32 * c);
}

__device__ __forceinline__ void convert_raw(const Raw<QMM_Q5_K> &r, int u, Unit &o) {
    q5k_unit(r.h, r.qh0, r.qh1, r.a, r.b, u & 3, o);
}

template <class Ld = LdGlobal>
__device__ __forceinline__ void load_raw(const uint8_t *row, int u, int, Raw<QMM_Q4_K> &r) {
    const uint8_t *blk = row + (u >> 2) * kQ4KBytes;
    const int c = u & 3;
    r.h = Ld::u128(blk);
    r.a = Ld::u128(blk + 16 + 32 * c);
    r.b = Ld::u128(blk + 32 + 32 * c);
}

__device__ __forceinline__ void convert_raw(const Raw<QMM_Q4_K> &r, int u, Unit &o) {
    const int c = u & 3;
    const uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        o.q[i] = (int)(w[i] & 0x0f0f0f0fu);
        o.q[8 + i] = (int)((w[i] >> 4) & 0x0f0f0f0fu);
    }
    const float d = half_lo(r.h.x), dmin = half_hi(r.h.x);
    int sc0, m0, sc1, m1;
    q4k_scale_min(r.h.y, r.h.z, r.h.w, 2 * c, sc0, m0);
    q4k_scale_min(r.h.y, r.h.z, r.h.w, 2 * c + 1, sc1, m1);
    o.isc[0] = o.isc[1] = sc0;
    o.isc[2] = o.isc[3] = sc1;
    o.fd[0] = o.fd[1] = d;
    o.fm[0] = dmin * (float)m0;
    o.fm[1] = dmin * (float)m1;
}

// Q6_K: a block is either 4-byte aligned or 2 bytes past a word boundary (then the
// 2 bytes before it belong to the previous block).  Aligned: ql/qh load one word past
// their range (still inside the block), the scales load 4 words + the fp16 d as a
// 2-byte load.  Misaligned: every part starts one halfword early; the scale words
// [190, 210) end exactly at the block end.
template <class Ld = LdGlobal>
__device__ __forceinline__ void load_raw(const uint8_t *row, int u, int, Raw<QMM_Q6_K> &r) {
    const uint8_t *blk = row + (u >> 2) * kQ6KBytes;
    const int v = u & 3, h = v >> 1;
    const uintptr_t a = reinterpret_cast<uintptr_t>(blk);
    const uint32_t mis = (uint32_t)(a & 2u);  // 0 or 2
    r.shift = mis * 8u;                       // 0 or 16 bits
    const uint32_t *ql = reinterpret_cast<const uint32_t *>((a + 64 * h) - mis);
    const uint32_t *qh = reinterpret_cast<const uint32_t *>((a + 128 + 32 * h) - mis);
    const uint32_t *sc = reinterpret_cast<const uint32_t *>((a + 192) - mis);
#pragma unroll
    for (int i = 0; i < 17; ++i) r.ql[i] = Ld::u32(ql + i);
#pragma unroll
    for (int i = 0; i < 9; ++i) r.qh[i] = Ld::u32(qh + i);
#pragma unroll
    for (int i = 0; i < 4; ++i) r.sc[i] = Ld::u32(sc + i);
    r.sc[4] = mis ? Ld::u32(sc + 4) : Ld::u16(sc + 4);
}

__device__ __forceinline__ void convert_raw(const Raw<QMM_Q6_K> &r, int u, Unit &o) {
    const int v = u & 3, p = v & 1;
    uint32_t ql[16], qh[8], sc[5];
#pragma unroll
    for (int i = 0; i < 16; ++i) ql[i] = __funnelshift_r(r.ql[i], r.ql[i + 1], r.shift);
#pragma unroll
    for (int i = 0; i < 8; ++i) qh[i] = __funnelshift_r(r.qh[i], r.qh[i + 1], r.shift);
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] = __funnelshift_r(r.sc[i], r.sc[i + 1], r.shift);
    sc[4] = r.shift ? (r.sc[4] >> 16) : r.sc[4];  // the fp16 d
    const int shift_l = 4 * p;
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
        const int t = 2 * p + tt;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = (ql[8 * tt + i] >> shift_l) & 0x0f0f0f0fu;
            const uint32_t hi = ((qh[i] >> (2 * t)) & 0x03030303u) << 4;
            o.q[8 * tt + i] = (int)__vsub4(lo | hi, 0x20202020u);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = 4 * v + i;
        o.isc[i] = (int)(int8_t)((sc[j >> 2] >> (8 * (j & 3))) & 0xff);
    }
    o.fd[0] = o.fd[1] = half_lo(sc[4]);
    o.fm[0] = o.fm[1] = 0.f;
}

// Q8_0: a unit of two blocks is 68 bytes at 68u; rows with an odd block count are
// only 2-byte aligned.  Two-block units are never the last unit of their row, so a
// misaligned load of 18 words [68u-2, 68u+70) stays inside the row's bytes plus the
// next unit's; a single-block unit reads exactly [68u, 68u+34) (or from 68u-2).
template <class Ld = LdGlobal>
__device__ __forceinline__ void load_raw(const uint8_t *row, int u, int nblk32, Raw<QMM_Q8_0> &r) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(row + 68 * u);
    const uint32_t mis = (uint32_t)(a & 2u);
    r.shift = mis * 8u;
    r.two = 2 * u + 1 < nblk32;
    const uint32_t *p = reinterpret_cast<const uint32_t *>(a - mis);
    if (r.two) {
#pragma unroll
        for (int i = 0; i < 17; ++i) r.w[i] = Ld::u32(p + i);
        r.w[17] = mis ? Ld::u32(p + 17) : 0u;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) r.w[i] = Ld::u32(p + i);
        r.w[8] = mis ? Ld::u32(p + 8) : Ld::u16(p + 8);
#pragma unroll
        for (int i = 9; i < 18; ++i) r.w[i] = 0u;
    }
}

__device__ __forceinline__ void convert_raw(const Raw<QMM_Q8_0> &r, int, Unit &o) {
    uint32_t w[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) w[i] = __funnelshift_r(r.w[i], r.w[i + 1], r.shift);
    if (!r.two) {
        w[8] &= 0xffffu;
#pragma unroll
        for (int i = 9; i < 17; ++i) w[i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) o.q[i] = (int)__funnelshift_r(w[i], w[i + 1], 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) o.q[8 + i] = (int)w[9 + i];
    o.isc[0] = o.isc[1] = o.isc[2] = o.isc[3] = 1;
    o.fd[0] = half_lo(w[0]);
    o.fd[1] = r.two ? half_hi(w[8]) : 0.f;
    o.fm[0] = o.fm[1] = 0.f;
}

// Q4_0: a unit of two blocks is 36 bytes at 36u, 2-byte aligned when the row's block
// count is odd (then only single-block units end a row).  Misaligned, the 10 words
// [36u-2, 36u+38) stay inside the row's bytes plus the next unit's; a single-block unit
// reads exactly [36u, 36u+18) (or from 36u-2).
template <class Ld = LdGlobal>
__device__ __forceinline__ void load_raw(const uint8_t *row, int u, int nblk32, Raw<QMM_Q4_0> &r) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(row + 36 * u);
    const uint32_t mis = (uint32_t)(a & 2u);
    r.shift = mis * 8u;
    r.two = 2 * u + 1 < nblk32;
    const uint32_t *p = reinterpret_cast<const uint32_t *>(a - mis);
    if (r.two) {
#pragma unroll
        for (int i = 0; i < 9; ++i) r.w[i] = Ld::u32(p + i);
        r.w[9] = mis ? Ld::u32(p + 9) : 0u;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) r.w[i] = Ld::u32(p + i);
        r.w[4] = mis ? Ld::u32(p + 4) : Ld::u16(p + 4);
#pragma unroll
        for (int i = 5; i < 10; ++i) r.w[i] = 0u;
    }
}

__device__ __forceinline__ void convert_raw(const Raw<QMM_Q4_0> &r, int, Unit &o) {
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = __funnelshift_r(r.w[i], r.w[i + 1], r.shift);
    if (!r.two) {
        w[4] &= 0xffffu;
#pragma unroll
        for (int i = 5; i < 9; ++i) w[i] = 0u;
    }
    q4_0_unit_from_words(w, r.two, o);
}

template <int T>
__device__ __forceinline__ void decode_unit(const uint8_t *row, int u, int nblk32, Unit &o) {
    if constexpr (T == QMM_Q4_K) decode_q4_K(row, u, o);
    else if constexpr (T == QMM_Q5_K) decode_q5_K(row, u, o);
    else if constexpr (T == QMM_Q6_K) decode_q6_K(row, u, o);
    else if constexpr (T == QMM_Q4_0) decode_q4_0(row, u, 2 * u + 1 < nblk32, o);
    else decode_q8_0(row, u, 2 * u + 1 < nblk32, o);
}

}  // namespace qmm
