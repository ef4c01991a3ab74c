// qdot_k56.cuh -- Q5_K, Q6_K and Q3_K rows against integer activation planes (the GEMV kernels).
//
// These are the next card-expert types the pages list after Q4_K ("bloomery README 0.3.1",
// Status table, "Quant types" row: card experts in Q4_K-Q6_K; "bloomery README 0.3.11", limits
// list: the large model's routed experts as Q3_K gate and up with a Q4_K down).  The activations are
// the staged vectors of qdot.cuh (per 32-value sub-block: NPL byte planes, an fp32 step and the
// sub-block sum; group g = values 64g .. 64g + 63 = sub-blocks 2c, 2c + 1 of super-block g/4,
// c = g % 4).  A lane takes one (row, group) item, builds the weights' integer codes as bytes
// and multiplies them with dp4a, as the Q4_K walk does.
//
// Q5_K (176 bytes per 256 weights): the Q4_K header (fp16 d, fp16 dmin, 12 bytes of 6-bit
// scales and mins), then 32 bytes qh whose byte i holds in bit j the 16s digit of element i of
// sub-block j, then Q4_K's 128 nibble bytes.  q = nibble + 16 * bit in [0, 31];
// w = d*sc_j*q - dmin*m_j.  Blocks are 11 x 16 bytes: every load is 16-byte aligned.
//
// Q6_K (210 bytes per 256 weights): 128 bytes of low nibbles, 64 bytes of 2-bit high parts,
// 16 int8 scales (one per 16 weights), fp16 d.  Element 128h + 32r + l (r < 4, l < 32) takes
// the low nibble (r < 2) or high nibble (r >= 2) of byte 64h + 32(r % 2) + l and bits 2r, 2r+1
// of byte 128 + 32h + l; w = d * sc[n / 16] * (u - 32), u = nibble + 16 * high bits.  In group
// c, sub-block 2c is r = 2(c % 2) of half h = c / 2 and sub-block 2c + 1 is r + 1.  A block
// starts on a 2-byte boundary only, so its fields are read as aligned 4-byte words from at
// most 2 bytes before a field and funnel-shifted into place; no read leaves the block's row
// past its end.  The codes u - 32 enter dp4a as signed bytes; the two 16-weight halves of a
// sub-block have their own scales, so their integer sums are kept apart.
//
// Q3_K (110 bytes per 256 weights): 32 bytes hmask, 64 bytes of 2-bit low parts, 12 bytes of
// sixteen 6-bit scales stored + 32, fp16 d.  Element 128h + 32r + l takes bits 2r, 2r + 1 of
// byte 32 + 32h + l and bit 4h + r of byte l; v = low + 4 * bit, q = v - 4 in [-4, 3]; scale j
// has its low nibble in byte 96 + j (j < 8, low) or 96 + j - 8 (high nibble) and bits 4-5 in bits
// 2(j / 4), 2(j / 4) + 1 of byte 104 + j % 4; w = d * (s_j - 32) * q.  Read and multiplied as
// Q6_K (2-byte aligned blocks, signed codes, one scale per 16 weights).
//
// MXFP4 (17 bytes per 32 weights, OCP Microscaling): an E8M0 scale byte e, then 16 bytes whose
// byte j holds E2M1 element j (low nibble) and j + 16 (high nibble); w = 2^(e - 127) * value.
// The codes enter dp4a as signed bytes of twice their value (exact integers), one scale per
// block, i.e. per staged sub-block of x.  Rows must be a multiple of 4 bytes (K % 128 == 0), so
// that the aligned word loads of the byte-aligned blocks stay inside the row.
#pragma once

#include <type_traits>

#include "qdot.cuh"

namespace moe {

constexpr int kQ5KBytes = 176;
constexpr int kQ6KBytes = 210;
constexpr int kQ3KBytes = 110;
constexpr int kMxfp4Bytes = 17;

template <>
struct Walk<MOE_Q5_K> {
    static constexpr int kBlockWeights = 256;
    static constexpr int kBlockBytes = kQ5KBytes;
};
template <>
struct Walk<MOE_Q6_K> {
    static constexpr int kBlockWeights = 256;
    static constexpr int kBlockBytes = kQ6KBytes;
};
template <>
struct Walk<MOE_Q3_K> {
    static constexpr int kBlockWeights = 256;
    static constexpr int kBlockBytes = kQ3KBytes;
};
template <>
struct Walk<MOE_MXFP4> {
    static constexpr int kBlockWeights = 32;
    static constexpr int kBlockBytes = kMxfp4Bytes;
};

__device__ __forceinline__ int qd_dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int qd_dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------------------- Q5_K

// acc[r0 + i][t] += row i . vector vidx[t] over group g (RPL rows of rowp from r0; NULL rows
// skipped).  The same walk as qd4_group with the fifth bit of every code.
template <int NT, int RPL, int NPL>
__device__ __forceinline__ void qd5_group(const uint8_t* const (&rowp)[4], int r0, int g, int G, const uint4* X,
                                          const float4* XS, int nt, float (&acc)[4][NT], const int* vidx) {
    const int b = g >> 2, c = g & 3;
    uint32_t lo[RPL][8], hi[RPL][8];                 // code bytes of sub-blocks 2c and 2c + 1
    float fs[RPL][2], fm[RPL][2];
    bool live[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        const uint8_t* rp = rowp[r0 + i];
        live[i] = rp != nullptr;
        uint4 hd = make_uint4(0u, 0u, 0u, 0u), h0 = hd, h1 = hd, q0 = hd, q1 = hd;
        if (live[i]) {
            const uint8_t* blk = rp + (int64_t)b * kQ5KBytes;
            hd = __ldg(reinterpret_cast<const uint4*>(blk));
            h0 = __ldg(reinterpret_cast<const uint4*>(blk + 16));
            h1 = __ldg(reinterpret_cast<const uint4*>(blk + 32));
            q0 = __ldg(reinterpret_cast<const uint4*>(blk + 48 + 32 * c));
            q1 = __ldg(reinterpret_cast<const uint4*>(blk + 64 + 32 * c));
        }
        qd4_scales(hd, c, fs[i], fm[i]);
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int qd = 0; qd < 8; ++qd) {
            lo[i][qd] = (qw[qd] & 0x0F0F0F0Fu) | (((hw[qd] >> (2 * c)) & 0x01010101u) << 4);
            hi[i][qd] = ((qw[qd] >> 4) & 0x0F0F0F0Fu) | (((hw[qd] >> (2 * c + 1)) & 0x01010101u) << 4);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t < nt) {
            const int v = vidx ? vidx[t] : t;
            const uint4* Xv = X + (size_t)v * 16 * G + g;
            int ah[RPL][2], am[RPL][2], al[RPL][2];
#pragma unroll
            for (int i = 0; i < RPL; ++i) ah[i][0] = ah[i][1] = am[i][0] = am[i][1] = al[i][0] = al[i][1] = 0;
#pragma unroll
            for (int qd = 0; qd < 8; ++qd) {
                const uint4 xl = Xv[qd * G], xh = Xv[(8 + qd) * G];
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    ah[i][0] = qd_dp4a_us(lo[i][qd], xl.x, ah[i][0]);
                    ah[i][1] = qd_dp4a_us(hi[i][qd], xh.x, ah[i][1]);
                    if constexpr (NPL == 3) {
                        am[i][0] = qd_dp4a_uu(lo[i][qd], xl.y, am[i][0]);
                        am[i][1] = qd_dp4a_uu(hi[i][qd], xh.y, am[i][1]);
                        al[i][0] = qd_dp4a_uu(lo[i][qd], xl.z, al[i][0]);
                        al[i][1] = qd_dp4a_uu(hi[i][qd], xh.z, al[i][1]);
                    } else {
                        al[i][0] = qd_dp4a_uu(lo[i][qd], xl.y, al[i][0]);
                        al[i][1] = qd_dp4a_uu(hi[i][qd], xh.y, al[i][1]);
                    }
                }
            }
            const float4 xs = XS[(size_t)v * G + g];
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
                if (live[i]) {
                    float d0, d1;
                    if constexpr (NPL == 3) {
                        d0 = fmaf((float)(ah[i][0] * 256 + am[i][0]), 256.0f, (float)al[i][0]) * xs.x;
                        d1 = fmaf((float)(ah[i][1] * 256 + am[i][1]), 256.0f, (float)al[i][1]) * xs.y;
                    } else {
                        d0 = (float)(ah[i][0] * 256 + al[i][0]) * xs.x;
                        d1 = (float)(ah[i][1] * 256 + al[i][1]) * xs.y;
                    }
                    float part = fs[i][0] * d0;
                    part = fmaf(fs[i][1], d1, part);
                    part = fmaf(-fm[i][0], xs.z, part);
                    part = fmaf(-fm[i][1], xs.w, part);
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
                        if (rr == r0 + i) acc[rr][t] += part;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------- Q6_K

// n (<= 8) consecutive 4-byte words of a field starting at byte p (2-byte aligned): aligned
// word loads from p rounded down to 4 bytes, shifted into place.  Reads stay inside
// [p - 2, p + 4n + 2) and, for a 4-byte aligned p, inside [p, p + 4n).
template <int N>
__device__ __forceinline__ void q6_words(const uint8_t* p, uint32_t (&out)[N]) {
    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 3u);        // 0 or 2
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p - mis);
    uint32_t a[N + 1];
#pragma unroll
    for (int j = 0; j < N; ++j) a[j] = __ldg(w + j);
    a[N] = mis ? __ldg(w + N) : 0u;
#pragma unroll
    for (int j = 0; j < N; ++j) out[j] = __funnelshift_r(a[j], a[j + 1], 8u * mis);
}

// Signed codes (as bytes) of sub-blocks 2c and 2c + 1 of group g of one row, and d * scale of the
// group's four 16-weight quarters.  Q6_K: u - 32 from a nibble and two high bits; Q3_K: v - 4
// from two low bits and a high bit, with 6-bit scales stored + 32.
// n consecutive 4-byte words from byte p at any alignment (aligned loads, funnel-shifted).
// Reads stay inside [p & ~3, p + 4n) and, when p is not 4-byte aligned, up to the next
// 4-byte boundary after p + 4n - 1.
template <int N>
__device__ __forceinline__ void q_words_any(const uint8_t* p, uint32_t (&out)[N]) {
    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 3u);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p - mis);
    uint32_t a[N + 1];
#pragma unroll
    for (int j = 0; j < N; ++j) a[j] = __ldg(w + j);
    a[N] = mis ? __ldg(w + N) : 0u;
#pragma unroll
    for (int j = 0; j < N; ++j) out[j] = __funnelshift_r(a[j], a[j + 1], 8u * mis);
}

// Four E2M1 codes (one per byte, low nibble) as signed bytes of twice their value: magnitudes
// 0, 0.5, 1, 1.5, 2, 3, 4, 6 become 0, 1, 2, 3, 4, 6, 8, 12 (byte permutes from two 8-byte
// tables, the negative table chosen by the sign bit).
__device__ __forceinline__ uint32_t e2m1x2_bytes(uint32_t nib) {
    const uint32_t mag = nib & 0x07070707u;
    const uint32_t sel = (mag & 0x7u) | ((mag >> 4) & 0x70u) | ((mag >> 8) & 0x700u) | ((mag >> 12) & 0x7000u);
    const uint32_t pos = __byte_perm(0x03020100u, 0x0C080604u, sel);
    const uint32_t neg = __byte_perm(0xFDFEFF00u, 0xF4F8FAFCu, sel);
    const uint32_t sgn = ((nib >> 3) & 0x01010101u) * 0xFFu;
    return (pos & ~sgn) | (neg & sgn);
}

template <int QT>
__device__ __forceinline__ void q_signed_codes(const uint8_t* rp, int g, uint32_t (&cw)[2][8], float (&sd)[4]) {
    if constexpr (QT == MOE_MXFP4) {
        // group g = blocks 2g (sub-block 0) and 2g + 1: an E8M0 scale byte, then byte j holds
        // element j (low nibble) and element j + 16 (high nibble); codes are twice the value, so
        // the scale is 2^(e - 128) (e = 255: NaN)
#pragma unroll
        for (int sb = 0; sb < 2; ++sb) {
            const uint8_t* blk = rp + (int64_t)(2 * g + sb) * kMxfp4Bytes;
            const uint32_t e = __ldg(blk);
            const float s = e == 255u ? __int_as_float(0x7FC00000) : ldexpf(0.5f, (int)e - 127);
            sd[2 * sb] = sd[2 * sb + 1] = s;
            uint32_t q[4];
            q_words_any<4>(blk + 1, q);
#pragma unroll
            for (int qd = 0; qd < 8; ++qd)
                cw[sb][qd] = e2m1x2_bytes(qd < 4 ? (q[qd] & 0x0F0F0F0Fu) : ((q[qd - 4] >> 4) & 0x0F0F0F0Fu));
        }
    } else {
    const int b = g >> 2, c = g & 3, h = c >> 1, rlo = 2 * (c & 1);   // sub-block 2c: r = rlo; 2c+1: rlo+1
    if constexpr (QT == MOE_Q6_K) {
        const uint8_t* blk = rp + (int64_t)b * kQ6KBytes;
        uint32_t l0[8], l1[8], hb[8], sw[1];
        q6_words<8>(blk + 64 * h, l0);
        q6_words<8>(blk + 64 * h + 32, l1);
        q6_words<8>(blk + 128 + 32 * h, hb);
        q6_words<1>(blk + 192 + 4 * c, sw);
        const float d = __half2float(__ushort_as_half((unsigned short)qd_ldg_u16(blk + 208)));
#pragma unroll
        for (int j = 0; j < 4; ++j) sd[j] = d * (float)(int8_t)((sw[0] >> (8 * j)) & 0xFFu);
        const int ns = 4 * (c & 1);                  // nibble: low for r < 2, high for r >= 2
#pragma unroll
        for (int qd = 0; qd < 8; ++qd) {
            const uint32_t u0 = ((l0[qd] >> ns) & 0x0F0F0F0Fu) | (((hb[qd] >> (2 * rlo)) & 0x03030303u) << 4);
            const uint32_t u1 = ((l1[qd] >> ns) & 0x0F0F0F0Fu) | (((hb[qd] >> (2 * rlo + 2)) & 0x03030303u) << 4);
            cw[0][qd] = __vsub4(u0, 0x20202020u);
            cw[1][qd] = __vsub4(u1, 0x20202020u);
        }
    } else {                                         // MOE_Q3_K, 110 bytes
        const uint8_t* blk = rp + (int64_t)b * kQ3KBytes;
        uint32_t hm[8], qs[8], sw[3];
        q6_words<8>(blk, hm);                        // bit 4h + r of byte l: the high bit of element 128h + 32r + l
        q6_words<8>(blk + 32 + 32 * h, qs);          // bits 2r, 2r + 1 of byte 32h + l: its low bits
        q6_words<3>(blk + 96, sw);
        const float d = __half2float(__ushort_as_half((unsigned short)qd_ldg_u16(blk + 108)));
        auto S = [&](int i) -> int {                  // scale byte i (registers, no indexed array)
            const uint32_t w = i < 4 ? sw[0] : i < 8 ? sw[1] : sw[2];
            return (int)((w >> (8 * (i & 3))) & 0xFFu);
        };
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * c + jj;
            const int lo4 = j < 8 ? (S(j) & 15) : (S(j - 8) >> 4);
            const int hi2 = (S(8 + (j & 3)) >> (2 * (j >> 2))) & 3;
            sd[jj] = d * (float)((lo4 | (hi2 << 4)) - 32);
        }
#pragma unroll
        for (int qd = 0; qd < 8; ++qd) {
            const uint32_t v0 = ((qs[qd] >> (2 * rlo)) & 0x03030303u) | (((hm[qd] >> (4 * h + rlo)) & 0x01010101u) << 2);
            const uint32_t v1 =
                ((qs[qd] >> (2 * rlo + 2)) & 0x03030303u) | (((hm[qd] >> (4 * h + rlo + 1)) & 0x01010101u) << 2);
            cw[0][qd] = __vsub4(v0, 0x04040404u);
            cw[1][qd] = __vsub4(v1, 0x04040404u);
        }
    }
    }
}

// Rows of signed codes with one scale per 16 weights (Q6_K, Q3_K) over group g.
template <int QT, int NT, int RPL, int NPL>
__device__ __forceinline__ void qd_signed_group(const uint8_t* const (&rowp)[4], int r0, int g, int G, const uint4* X,
                                                const float4* XS, int nt, float (&acc)[4][NT], const int* vidx) {
    uint32_t cw[RPL][2][8];                          // signed code bytes, sub-blocks 2c, 2c + 1
    float sd[RPL][4];                                // d * scale of the group's four 16-weight quarters
    bool live[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        const uint8_t* rp = rowp[r0 + i];
        live[i] = rp != nullptr;
        if (live[i]) {
            q_signed_codes<QT>(rp, g, cw[i], sd[i]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) cw[i][0][j] = cw[i][1][j] = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) sd[i][j] = 0.f;
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t < nt) {
            const int v = vidx ? vidx[t] : t;
            const uint4* Xv = X + (size_t)v * 16 * G + g;
            const float4 xs = XS[(size_t)v * G + g];
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
                float part = 0.f;
#pragma unroll
                for (int sb = 0; sb < 2; ++sb) {                 // sub-block 2c + sb
#pragma unroll
                    for (int hq = 0; hq < 2; ++hq) {             // its 16-weight halves
                        int ah = 0, am = 0, al = 0;
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            const int qd = 4 * hq + qq;
                            const uint4 xv = Xv[(8 * sb + qd) * G];
                            ah = qd_dp4a_ss(cw[i][sb][qd], xv.x, ah);
                            if constexpr (NPL == 3) {
                                am = qd_dp4a_su(cw[i][sb][qd], xv.y, am);
                                al = qd_dp4a_su(cw[i][sb][qd], xv.z, al);
                            } else {
                                al = qd_dp4a_su(cw[i][sb][qd], xv.y, al);
                            }
                        }
                        float dot;
                        if constexpr (NPL == 3) {
                            dot = fmaf((float)(ah * 256 + am), 256.0f, (float)al);
                        } else {
                            dot = (float)(ah * 256 + al);
                        }
                        part = fmaf(sd[i][2 * sb + hq] * (sb ? xs.y : xs.x), dot, part);
                    }
                }
                if (live[i]) {
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
                        if (rr == r0 + i) acc[rr][t] += part;
                }
            }
        }
    }
}

// acc[r][t] += row r . vector vidx[t] (t < nt) for 4 rows of nblk blocks of type QT
// (MOE_Q5_K, MOE_Q6_K, MOE_Q3_K or MOE_MXFP4), lanes split into row subsets as in qd4_rows4.
template <int QT, int NT, int NPL>
__device__ __forceinline__ void qd56_rows4(const uint8_t* const (&rowp)[4], int nblk, const uint4* X,
                                           const float4* XS, int nt, int lane, float (&acc)[4][NT]) {
    const int G = QT == MOE_MXFP4 ? nblk / 2 : nblk * 4;        // groups of 64 weights
    auto grp = [&](auto rpl, int r0, int g) {
        constexpr int RPL = decltype(rpl)::value;
        if constexpr (QT == MOE_Q5_K) qd5_group<NT, RPL, NPL>(rowp, r0, g, G, X, XS, nt, acc, nullptr);
        else qd_signed_group<QT, NT, RPL, NPL>(rowp, r0, g, G, X, XS, nt, acc, nullptr);
    };
    if (G >= 24) {
        for (int g = lane; g < G; g += 32) grp(std::integral_constant<int, 4>{}, 0, g);
    } else if (G >= 12) {
        const int rs = lane >> 4;
        for (int g = lane & 15; g < G; g += 16) grp(std::integral_constant<int, 2>{}, 2 * rs, g);
    } else {
        const int rs = lane >> 3;
        for (int g = lane & 7; g < G; g += 8) grp(std::integral_constant<int, 1>{}, rs, g);
    }
}

}  // namespace moe
