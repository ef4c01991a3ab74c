// qdot.cuh -- per-lane dequant-dot of quantized rows against staged fp32 vectors.
//
// One warp reads 4 weight rows at a time; per warp iteration every lane covers
// 32 weights of each row: Q4_K one 16-byte quant chunk (8 lanes per 256-weight
// super-block: w = d*sc_j*q - dmin*m_j), Q8_0 one 34-byte block (w = d*q).
// The vectors are staged in shared memory in exactly the order of that walk
// (float4 slot (it*8 + i4)*32 + lane), so every lane reads 16 bytes at a time
// without bank conflicts, and for Q4_K each lane also finds the sums of its two
// 16-element halves (the min term).  Used by the decode GEMV kernels and the
// fused decode-layer kernel.
#pragma once

#include "internal.cuh"

namespace moe {

__device__ __forceinline__ float qd_byte_to_float(uint32_t word, int b) {
    // 0x4B0000bb is 2^23 + bb as an fp32; subtracting 2^23 leaves bb exactly.
    return __int_as_float(__byte_perm(word, 0x4B00u, 0x5440u | (uint32_t)b)) - 8388608.0f;
}
// Same for a byte that holds int8 + 128: leaves the signed value exactly.
__device__ __forceinline__ float qd_sbyte_to_float(uint32_t word, int b) {
    return __int_as_float(__byte_perm(word, 0x4B00u, 0x5440u | (uint32_t)b)) - 8388736.0f;
}
__device__ __forceinline__ uint32_t qd_ldg_u16(const uint8_t* p) {
    return __ldg(reinterpret_cast<const unsigned short*>(p));
}

template <int QT>
struct Walk;

// Q4_K: lane l of iteration it covers super-block it*4 + l/8, quant chunk l%8.
template <>
struct Walk<MOE_Q4_K> {
    static constexpr int kBlockWeights = kQ4KWeights;
    static constexpr int kBlockBytes = kQ4KBytes;
    static constexpr int kBlocksPerIter = 4;
    __device__ static int blk(int it, int lane) { return it * 4 + (lane >> 3); }
    // element offset inside the row of the first of the 4 values of slot i4
    __device__ static int pos(int it, int lane, int i4) {
        const int ch = lane & 7, c = ch >> 1, half = ch & 1, hi = i4 >> 2;
        return blk(it, lane) * 256 + 64 * c + 32 * hi + 16 * half + 4 * (i4 & 3);
    }
};

// Q8_0: lane l of iteration it covers block it*32 + l.
template <>
struct Walk<MOE_Q8_0> {
    static constexpr int kBlockWeights = kQ80Weights;
    static constexpr int kBlockBytes = kQ80Bytes;
    static constexpr int kBlocksPerIter = 32;
    __device__ static int blk(int it, int lane) { return it * 32 + lane; }
    __device__ static int pos(int it, int lane, int i4) { return blk(it, lane) * 32 + 4 * i4; }
};

template <int QT>
__host__ __device__ inline int walk_iters(int K) {
    const int nblk = K / (QT == MOE_Q4_K ? kQ4KWeights : kQ80Weights);
    const int bpi = QT == MOE_Q4_K ? 4 : 32;
    return (nblk + bpi - 1) / bpi;
}

__device__ __forceinline__ float4 qd_load_vec4(const void* v, bool bf16, int64_t idx) {
    float4 out;
    if (bf16) {
        const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(v) + idx);
        out.x = __uint_as_float(raw.x << 16);
        out.y = __uint_as_float(raw.x & 0xFFFF0000u);
        out.z = __uint_as_float(raw.y << 16);
        out.w = __uint_as_float(raw.y & 0xFFFF0000u);
    } else {
        out = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(v) + idx);
    }
    return out;
}

// Stage one length-K vector (src: bf16 or fp32, global) into xs (iters*256 float4
// slots, walk order) with threads [tid0, tid0+nthr).  Call qd_stage_sums after a
// barrier for Q4_K.  `coherent` reads through L2 (data written by other CTAs).
template <int QT>
__device__ __forceinline__ void qd_stage(const void* src, bool bf16, bool coherent, int K, int iters, float4* xs,
                                         int tid, int nthr) {
    const int nblk = K / Walk<QT>::kBlockWeights;
    constexpr int kB = 8;                             // loads in flight per thread before any store
    for (int s0 = tid; s0 < iters * 256; s0 += kB * nthr) {
        float4 v[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int s = s0 + b * nthr;
            v[b] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s < iters * 256) {
                const int it = s >> 8, i4 = (s >> 5) & 7, ln = s & 31;
                if (Walk<QT>::blk(it, ln) < nblk) {
                    const int p = Walk<QT>::pos(it, ln, i4);
                    if (coherent && !bf16)
                        v[b] = __ldcg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + p));
                    else
                        v[b] = qd_load_vec4(src, bf16, p);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int s = s0 + b * nthr;
            if (s < iters * 256) xs[s] = v[b];
        }
    }
}

// Stage n vectors at once (vector i from base + i*row_elems, fp32, written by other
// CTAs: read through L2) into xs + i*iters*256: every load is issued before any store.
template <int QT>
__device__ __forceinline__ void qd_stage_many_f32(const float* base, int64_t row_elems, int n, int K, int iters,
                                                  float4* xs, int tid, int nthr) {
    const int nblk = K / Walk<QT>::kBlockWeights;
    const int per = iters * 256;
    const int total = n * per;
    constexpr int kB = 8;                             // loads in flight per thread
    for (int s0 = tid; s0 < total; s0 += kB * nthr) {
        float4 v[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int s = s0 + b * nthr;
            v[b] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s < total) {
                const int i = s / per, r = s - i * per;
                const int it = r >> 8, i4 = (r >> 5) & 7, ln = r & 31;
                if (Walk<QT>::blk(it, ln) < nblk)
                    v[b] = __ldcg(reinterpret_cast<const float4*>(base + (int64_t)i * row_elems + Walk<QT>::pos(it, ln, i4)));
            }
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int s = s0 + b * nthr;
            if (s < total) xs[s] = v[b];
        }
    }
}

// Half sums of n consecutive staged vectors at once (vector i at xs + i*iters*256,
// sums at xsum + i*iters*32).
__device__ __forceinline__ void qd_stage_sums_many(const float4* xs, float2* xsum, int n, int iters, int tid,
                                                   int nthr) {
    for (int r = tid; r < n * iters * 32; r += nthr) {
        const int i = r / (iters * 32), rr = r - i * iters * 32;
        const int it = rr >> 5, ln = rr & 31;
        const float4* base = xs + (size_t)i * iters * 256 + it * 256 + ln;
        float lo = 0.f, hi = 0.f;
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
            const float4 v = base[i4 * 32];
            lo += (v.x + v.y) + (v.z + v.w);
            const float4 u = base[(i4 + 4) * 32];
            hi += (u.x + u.y) + (u.z + u.w);
        }
        xsum[r] = make_float2(lo, hi);
    }
}

// 16-element half sums of each lane's slice (Q4_K min term): xsum[it*32 + lane].
__device__ __forceinline__ void qd_stage_sums(const float4* xs, float2* xsum, int iters, int tid, int nthr) {
    for (int r = tid; r < iters * 32; r += nthr) {
        const int it = r >> 5, ln = r & 31;
        const float4* base = xs + it * 256 + ln;
        float lo = 0.f, hi = 0.f;
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
            const float4 v = base[i4 * 32];
            lo += (v.x + v.y) + (v.z + v.w);
            const float4 u = base[(i4 + 4) * 32];
            hi += (u.x + u.y) + (u.z + u.w);
        }
        xsum[r] = make_float2(lo, hi);
    }
}

// acc[r][t] += lane's part of row r . vector t, for 4 rows and nt <= NT staged vectors.
// Vector t lives at xs + t*vstride (float4 slots) and xsum + t*sstride.  Rows may be
// NULL (skipped, accumulators untouched).
template <bool kSmemRows>
__device__ __forceinline__ uint4 qd_ld16(const uint8_t* p) {
    if (kSmemRows) return *reinterpret_cast<const uint4*>(p);
    return __ldg(reinterpret_cast<const uint4*>(p));
}
template <bool kSmemRows>
__device__ __forceinline__ uint32_t qd_ld2(const uint8_t* p) {
    if (kSmemRows) return *reinterpret_cast<const unsigned short*>(p);
    return qd_ldg_u16(p);
}

// Q8_0 rows are GGUF blocks (34 bytes, read as halfwords), or with q80r the repacked row
// layout (the block's 32 quants at 32*b, 16-byte aligned; its scale at 32*nblk + 2*b).
template <int QT, int NT, bool kSmemRows = false>
__device__ __forceinline__ void qd_rows4(const uint8_t* const (&rowp)[4], int nblk, int iters, const float4* xs,
                                         int vstride, const float2* xsum, int sstride, int nt, int lane,
                                         float (&acc)[4][NT], const int* vidx = nullptr, bool q80r = false) {
    for (int it = 0; it < iters; ++it) {
        const int b = Walk<QT>::blk(it, lane);
        if (b >= nblk) continue;
        if (QT == MOE_Q4_K) {
            const int ch = lane & 7, jj = (ch >> 1) & 1, upper = ch >> 2;
            uint4 q[4], hd[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (rowp[r]) {
                    const uint8_t* bp = rowp[r] + (int64_t)b * kQ4KBytes;
                    hd[r] = qd_ld16<kSmemRows>(bp);
                    q[r] = qd_ld16<kSmemRows>(bp + 16 + 16 * ch);
                } else {
                    hd[r] = make_uint4(0, 0, 0, 0);
                    q[r] = make_uint4(0, 0, 0, 0);
                }
            }
            float fsc[4][2], fm[4][2];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float d = __half2float(__ushort_as_half((unsigned short)(hd[r].x & 0xFFFFu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hd[r].x >> 16)));
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const int j = 2 * jj + s;
                    const uint32_t by = (hd[r].y >> (8 * j)) & 0xFFu;
                    const uint32_t bz = (hd[r].z >> (8 * j)) & 0xFFu;
                    const uint32_t bw = (hd[r].w >> (8 * j)) & 0xFFu;
                    uint32_t sc, m;
                    if (!upper) { sc = by & 63u; m = bz & 63u; }
                    else { sc = (bw & 15u) | ((by >> 6) << 4); m = (bw >> 4) | ((bz >> 6) << 4); }
                    fsc[r][s] = d * (float)sc;
                    fm[r][s] = dmin * (float)m;
                }
            }
            const float4* xb = xs + it * 256 + lane;
            const float2* xsb = xsum + it * 32 + lane;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (t < nt) {
                    float dl[4], dh[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) { dl[r] = 0.f; dh[r] = 0.f; }
                    const size_t vt = (size_t)(vidx ? vidx[t] : t);
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) {
                        const float4 xl = xb[vt * vstride + w4 * 32];
                        const float4 xh = xb[vt * vstride + (w4 + 4) * 32];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t word = w4 == 0 ? q[r].x : w4 == 1 ? q[r].y : w4 == 2 ? q[r].z : q[r].w;
                            const uint32_t lo = word & 0x0F0F0F0Fu, hi = (word >> 4) & 0x0F0F0F0Fu;
                            dl[r] = fmaf(qd_byte_to_float(lo, 0), xl.x, dl[r]);
                            dl[r] = fmaf(qd_byte_to_float(lo, 1), xl.y, dl[r]);
                            dl[r] = fmaf(qd_byte_to_float(lo, 2), xl.z, dl[r]);
                            dl[r] = fmaf(qd_byte_to_float(lo, 3), xl.w, dl[r]);
                            dh[r] = fmaf(qd_byte_to_float(hi, 0), xh.x, dh[r]);
                            dh[r] = fmaf(qd_byte_to_float(hi, 1), xh.y, dh[r]);
                            dh[r] = fmaf(qd_byte_to_float(hi, 2), xh.z, dh[r]);
                            dh[r] = fmaf(qd_byte_to_float(hi, 3), xh.w, dh[r]);
                        }
                    }
                    const float2 sx = xsb[vt * sstride];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        float v = fsc[r][0] * dl[r];
                        v = fmaf(fsc[r][1], dh[r], v);
                        v = fmaf(-fm[r][0], sx.x, v);
                        v = fmaf(-fm[r][1], sx.y, v);
                        acc[r][t] += v;
                    }
                }
            }
        } else {
            uint32_t qw[4][8];
            float dd[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (rowp[r] && q80r) {
                    const uint8_t* qp = rowp[r] + (int64_t)b * 32;
                    dd[r] = __half2float(__ushort_as_half((unsigned short)qd_ld2<kSmemRows>(rowp[r] + (int64_t)nblk * 32 + 2 * b)));
                    const uint4 a0 = qd_ld16<kSmemRows>(qp), a1 = qd_ld16<kSmemRows>(qp + 16);
                    qw[r][0] = a0.x ^ 0x80808080u; qw[r][1] = a0.y ^ 0x80808080u;   // int8 + 128 as bytes
                    qw[r][2] = a0.z ^ 0x80808080u; qw[r][3] = a0.w ^ 0x80808080u;
                    qw[r][4] = a1.x ^ 0x80808080u; qw[r][5] = a1.y ^ 0x80808080u;
                    qw[r][6] = a1.z ^ 0x80808080u; qw[r][7] = a1.w ^ 0x80808080u;
                } else if (rowp[r]) {
                    const uint8_t* bp = rowp[r] + (int64_t)b * kQ80Bytes;
                    dd[r] = __half2float(__ushort_as_half((unsigned short)qd_ld2<kSmemRows>(bp)));
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const uint32_t lo16 = qd_ld2<kSmemRows>(bp + 2 + 4 * w);
                        const uint32_t hi16 = qd_ld2<kSmemRows>(bp + 4 + 4 * w);
                        qw[r][w] = (lo16 | (hi16 << 16)) ^ 0x80808080u;   // int8 + 128 as bytes
                    }
                } else {
                    dd[r] = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w) qw[r][w] = 0x80808080u;
                }
            }
            const float4* xb = xs + it * 256 + lane;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (t < nt) {
                    float dt[4] = {0.f, 0.f, 0.f, 0.f};
                    const size_t vt = (size_t)(vidx ? vidx[t] : t);
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const float4 xv = xb[vt * vstride + w * 32];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            dt[r] = fmaf(qd_sbyte_to_float(qw[r][w], 0), xv.x, dt[r]);
                            dt[r] = fmaf(qd_sbyte_to_float(qw[r][w], 1), xv.y, dt[r]);
                            dt[r] = fmaf(qd_sbyte_to_float(qw[r][w], 2), xv.z, dt[r]);
                            dt[r] = fmaf(qd_sbyte_to_float(qw[r][w], 3), xv.w, dt[r]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[r][t] = fmaf(dd[r], dt[r], acc[r][t]);
                }
            }
        }
    }
}

// Transposed warp sum of acc[4][NT] (NT = 1, 2, 4 or 8).  Each halving step sends one half
// of the lane's entries to the partner lane and keeps the other, so the 4*NT sums cost
// 4*NT - 1 shuffles plus the butterfly steps left over, not 4*NT*5.  Afterwards lane L
// holds the warp total of entry i = L >> qd_red_shift<NT>() of acc, i = r * NT + t, and
// the 2^shift lanes sharing i hold the same value.
template <int NT>
__host__ __device__ constexpr int qd_red_shift() { return NT >= 8 ? 0 : NT == 4 ? 1 : NT == 2 ? 2 : 3; }

template <int NT>
__device__ __forceinline__ float qd_warp_reduce_t(const float (&acc)[4][NT]) {
    constexpr int V = 4 * NT;
    float v[V];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) v[r * NT + t] = acc[r][t];
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int n = V, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = up ? v[i + n / 2] : v[i];
            const float send = up ? v[i] : v[i + n / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float s = v[0];
#pragma unroll
    for (int o = (1 << qd_red_shift<NT>()) >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}



// ============================================================================
// Q4_K against integer activations (the path both GEMV kernels use).
//
// A row is walked in groups of 64 weights: group g = (super-block b, quant group
// c), i.e. 32 quant bytes holding sub-blocks 2c (low nibbles) and 2c+1 (high
// nibbles).  One lane takes one (row, group) item, so it decodes its two
// sub-block scales once per 64 weights.  Each activation sub-block of 32 values
// (largest magnitude m) is scaled to integers and stored as NPL byte planes (the
// signed high byte first, then unsigned bytes):
//   NPL = 3, any input: x24 = round(x * (2^23-1) / m), planes {hi, mid, lo};
//   NPL = 2, bf16 input: x16 = round(x * 2^(15-e)) with 2^(e-1) <= m < 2^e, planes
//     {hi, lo}.  The step is a power of two, so a bf16 value (8 significant bits)
//     within 7 binades of m is held exactly; only smaller ones round, by at most
//     2^-16 of 2^e.
// The lane multiplies its 4-bit codes with dp4a (exact integer sums), recombines
// the planes and applies the scales in fp32:
//   dot_j = (65536*sum(q*hi) + 256*sum(q*mid) + sum(q*lo)) * sx_j      (NPL = 3)
//   dot_j = (256*sum(q*hi) + sum(q*lo)) * sx_j                         (NPL = 2)
//   row . x += d*sc_j*dot_j - dmin*m_j*sum(x over sub-block j)
// The high nibbles enter dp4a unshifted (byte = 16 q), so their sums are 16x the
// codes' sums and the factor 1/16 joins the sub-block scale (exact).  Plane sums
// are joined in integers (|256*hi + next| < 2^31) before the conversion to fp32.
// The sums over sub-block j carry the unrounded values, so the min term is exact;
// the rounding of x is at most 2^-24 (NPL = 3) or 2^-16 (NPL = 2, bf16 values
// more than 7 binades below m only) of the sub-block's range.
// Staged vector layout (G = K/64 groups): X[q*G + g] (q = 0..15) holds the
// planes {hi, mid, lo, 0} or {hi, lo, 0, 0} of 4 values: q < 8 values 4q.. of
// sub-block 2c, q >= 8 values 4(q-8).. of sub-block 2c+1;
// XS[g] = {sx_lo, sx_hi, sum_lo, sum_hi}.
// ============================================================================

__host__ __device__ inline int qd4_groups(int K) { return K / 64; }
// Staging of one sub-block with largest magnitude m (NPL planes, see above): the
// factor inv that maps a value to its integer and the step sx that maps it back.
template <int NPL>
__device__ __forceinline__ float2 qx_scale(float m) {
    if (!(m > 0.f)) return make_float2(0.f, 0.f);
    if constexpr (NPL == 3) {
        return make_float2(8388607.0f / m, m / 8388607.0f);
    } else {
        int e;
        (void)frexpf(m, &e);                         // m = f * 2^e, 1/2 <= f < 1
        return make_float2(ldexpf(1.0f, 15 - e), ldexpf(1.0f, e - 15));
    }
}
template <int NPL>
__device__ __forceinline__ int qx_int(float v, float inv) {
    constexpr int kLim = NPL == 3 ? 8388607 : 32767;
    return max(-kLim, min(kLim, __float2int_rn(v * inv)));
}
// byte plane p (0 = the signed high byte) of a staged integer
template <int NPL>
__device__ __forceinline__ uint32_t qx_plane(int x, int p) {
    return ((uint32_t)x >> (8 * (NPL - 1 - p))) & 0xFFu;
}
// the staged uint4 of 4 values (planes in .x, .y[, .z])
template <int NPL>
__device__ __forceinline__ uint4 qx_pack4(const float (&v)[4], float inv) {
    uint32_t w[3] = {0u, 0u, 0u};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int x = qx_int<NPL>(v[b], inv);
#pragma unroll
        for (int pl = 0; pl < NPL; ++pl) w[pl] |= qx_plane<NPL>(x, pl) << (8 * b);
    }
    return make_uint4(w[0], w[1], NPL == 3 ? w[2] : 0u, 0u);
}
// bytes of one staged vector
__host__ __device__ inline size_t qd4_vec_bytes(int K) { return (size_t)qd4_groups(K) * 17 * 16; }

__device__ __forceinline__ int qd_dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int qd_dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// RMSNorm of one fp32 row, r = 1 / sqrt(mean(x^2) + eps), in the summation order of
// moe_rmsnorm_bf16's kernel: its thread i (of 256) accumulates x[4i + 1024 j .. + 3] with fmaf,
// each of its 8 warps reduces its 32 partial sums by a xor butterfly, and the 8 warp sums are
// added in order.  rms_vwarp_sum is that kernel's warp vw (lanes playing threads 32 vw ..
// 32 vw + 31; every lane gets the sum); rms_scale adds the 8 sums in order.  H <= 2048, so a
// lane's two loads are issued before any arithmetic.  A layer that normalizes its own input
// thus gives the bits of the separate kernel.
__device__ __forceinline__ float rms_vwarp_sum(const float* row, int H, int vw) {
    const int lane = threadIdx.x & 31;
    const int h0 = (vw * 32 + lane) * 4;
    const float4 a = h0 < H ? __ldcg(reinterpret_cast<const float4*>(row + h0)) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 b = h0 + 1024 < H ? __ldcg(reinterpret_cast<const float4*>(row + h0 + 1024))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    float ss = 0.f;
    if (h0 < H) {
        ss = fmaf(a.x, a.x, ss);
        ss = fmaf(a.y, a.y, ss);
        ss = fmaf(a.z, a.z, ss);
        ss = fmaf(a.w, a.w, ss);
    }
    if (h0 + 1024 < H) {
        ss = fmaf(b.x, b.x, ss);
        ss = fmaf(b.y, b.y, ss);
        ss = fmaf(b.z, b.z, ss);
        ss = fmaf(b.w, b.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    return ss;
}
__device__ __forceinline__ float rms_scale(const float* part8, int H, float eps) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part8[w];
    return 1.0f / sqrtf(s / (float)H + eps);
}
// The scales of T rows of x (stride H) into s_r[t], by all warps of the CTA (part: [T][8]
// shared scratch).  Every thread of the CTA must call it.
__device__ __forceinline__ void rms_scales_cta(const float* x, int T, int H, float eps, float (*part)[8],
                                               float* s_r) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int it = warp; it < T * 8; it += nw) {
        const float v = rms_vwarp_sum(x + (int64_t)(it >> 3) * H, H, it & 7);
        if (lane == 0) part[it >> 3][it & 7] = v;
    }
    __syncthreads();
    if ((int)threadIdx.x < T) s_r[threadIdx.x] = rms_scale(part[threadIdx.x], H, eps);
    __syncthreads();
}
// u = bf16(x * r * gamma) per component, as a float (the normalized layer input).
__device__ __forceinline__ float4 rms_apply4(float4 x, float r, float4 g) {
    return make_float4(__bfloat162float(__float2bfloat16_rn(x.x * r * g.x)),
                       __bfloat162float(__float2bfloat16_rn(x.y * r * g.y)),
                       __bfloat162float(__float2bfloat16_rn(x.z * r * g.z)),
                       __bfloat162float(__float2bfloat16_rn(x.w * r * g.w)));
}

// Stage n vectors (vector i at src + row*row_elems, bf16 or fp32; `coherent` reads fp32
// through L2; rows (nullable): vector i is source row rows[i]) into X + i*16*G, XS + i*G
// as NPL planes (NPL = 2 only for bf16 values: bf16 src, or the normalized input below).
// Work is split in chunks of 32 values (4 sub-blocks of 8 threads, 4 values per thread,
// max and sum by butterfly within the 8); warp w of nw takes chunks w, w + nw, ... with
// four chunks' loads in flight.  Every lane of every warp in [0, nw) must call it.  With
// ngamma, src is fp32 and vector i is staged as its RMSNorm output bf16(x * nscale[i] *
// gamma) (nscale: the vectors' scales, shared memory).
template <int NPL>
__device__ __forceinline__ void qd4_stage_par(const void* src, bool bf16, bool coherent, int64_t row_elems, int n,
                                              const int* rows, int K, uint4* X, float4* XS, int tid, int nthr,
                                              const float* ngamma = nullptr, const float* nscale = nullptr) {
    const int G = qd4_groups(K);
    const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    const int cpv = G / 2;                            // chunks per vector (G = K/64 is a multiple of 4)
    const int total = n * cpv;
    constexpr int kU = 4;
    const int sbl = lane >> 3, q8 = lane & 7;         // sub-block within the chunk, quad within it
    for (int c0 = warp; c0 < total; c0 += kU * nw) {
        float4 v[kU];
        int iv[kU], sbv[kU];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            const int c = c0 + j * nw;
            v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            iv[j] = -1;
            sbv[j] = 0;
            if (c < total) {
                const int i = c / cpv;
                const int sb = (c - i * cpv) * 4 + sbl;   // sub-block index 0..2G-1 in the vector
                iv[j] = i;
                sbv[j] = sb;
                const int g = sb >> 1, hh = sb & 1;
                const int64_t row = rows ? rows[i] : i;
                const int64_t e = row * row_elems + (g >> 2) * 256 + (2 * (g & 3) + hh) * 32 + 4 * q8;
                if (bf16) {
                    const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(src) + e);
                    v[j] = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                                       __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
                } else {
                    const float4* p4 = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + e);
                    v[j] = coherent ? __ldcg(p4) : *p4;
                    if (ngamma)
                        v[j] = rms_apply4(v[j], nscale[i],
                                          *reinterpret_cast<const float4*>(ngamma + (e - row * row_elems)));
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            if (c0 + j * nw >= total) break;              // warp-uniform
            float m = fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w)));
            float sum = (v[j].x + v[j].y) + (v[j].z + v[j].w);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                sum += __shfl_xor_sync(0xffffffffu, sum, o);
            }
            const int i = iv[j], sb = sbv[j], g = sb >> 1, hh = sb & 1;
            const float2 sc = qx_scale<NPL>(m);
            const float vv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            X[(size_t)i * 16 * G + (hh * 8 + q8) * G + g] = qx_pack4<NPL>(vv, sc.x);
            if (q8 == 0) {
                float* xsf = reinterpret_cast<float*>(XS + (size_t)i * G + g);
                xsf[hh] = sc.y;
                xsf[2 + hh] = sum;
            }
        }
    }
}

// Exact float of an integer 0 <= v < 2^23 (2^23 + v as fp32 bit pattern, minus 2^23).
__device__ __forceinline__ float qd_small_u2f(uint32_t v) { return __uint_as_float(0x4B000000u | v) - 8388608.0f; }

// Scales of sub-blocks 2c and 2c+1 of a Q4_K block header: fs = d*sc_j, fm = dmin*m_j.
// Sub-blocks 0..3 keep sc and m in the low 6 bits of bytes 0..3 / 4..7 of the 12 scale
// bytes; sub-blocks 4..7 take their low 4 bits from the nibbles of bytes 8..11 and the
// top 2 bits from bits 6..7 of bytes 0..3 / 4..7.  Both sub-blocks of the pair come out
// of one 16-bit window of each scale word.
__device__ __forceinline__ void qd4_scales(const uint4& hd, int c, float (&fs)[2], float (&fm)[2]) {
    const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
    const int sh = (c & 1) * 16;
    const uint32_t y = hd.y >> sh, z = hd.z >> sh, w = hd.w >> sh;
    const uint32_t sc_lo = y & 0x3F3Fu, m_lo = z & 0x3F3Fu;
    const uint32_t sc_hi = (w & 0x0F0Fu) | ((y >> 2) & 0x3030u);
    const uint32_t m_hi = ((w >> 4) & 0x0F0Fu) | ((z >> 2) & 0x3030u);
    const bool upper = c >= 2;
    const uint32_t sc = upper ? sc_hi : sc_lo, m = upper ? m_hi : m_lo;
    fs[0] = d * qd_small_u2f(sc & 0xFFu);
    fs[1] = d * qd_small_u2f(sc >> 8);
    fm[0] = dmin * qd_small_u2f(m & 0xFFu);
    fm[1] = dmin * qd_small_u2f(m >> 8);
}

// One lane, one group g (64 weights: sub-blocks 2c, 2c+1 of super-block g/4, c = g%4),
// RPL rows whose bytes are already loaded: hd = the 16-byte block header, q0/q1 = the
// 32 quant bytes of the group.  acc[r0 + i][t] += row i . vector vidx[t] (t < nt); the
// activation planes of the group are read once and serve every row.
template <int NT, int RPL, int NPL>
__device__ __forceinline__ void qd4_group_math(const uint4 (&hd)[RPL], const uint4 (&q0)[RPL], const uint4 (&q1)[RPL],
                                               const bool (&live)[RPL], int r0, int g, int G, const uint4* X,
                                               const float4* XS, int nt, float (&acc)[4][NT], const int* vidx) {
    const int c = g & 3;
    uint32_t qw[RPL][8];
    float fs[RPL][2], fm[RPL][2];
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        qw[i][0] = q0[i].x; qw[i][1] = q0[i].y; qw[i][2] = q0[i].z; qw[i][3] = q0[i].w;
        qw[i][4] = q1[i].x; qw[i][5] = q1[i].y; qw[i][6] = q1[i].z; qw[i][7] = q1[i].w;
        qd4_scales(hd[i], c, fs[i], fm[i]);
        fs[i][1] *= 0.0625f;                       // the high nibbles' sums carry a factor 16
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t < nt) {
            const int v = vidx ? vidx[t] : t;
            const uint4* Xv = X + (size_t)v * 16 * G + g;
            int ah[RPL][2], am[RPL][2], al[RPL][2];       // am: the middle plane (NPL = 3)
#pragma unroll
            for (int i = 0; i < RPL; ++i) ah[i][0] = ah[i][1] = am[i][0] = am[i][1] = al[i][0] = al[i][1] = 0;
#pragma unroll
            for (int qd = 0; qd < 8; ++qd) {
                const uint4 xl = Xv[qd * G], xh = Xv[(8 + qd) * G];
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    const uint32_t ql = qw[i][qd] & 0x0F0F0F0Fu, qh = qw[i][qd] & 0xF0F0F0F0u;
                    ah[i][0] = qd_dp4a_us(ql, xl.x, ah[i][0]);
                    ah[i][1] = qd_dp4a_us(qh, xh.x, ah[i][1]);
                    if constexpr (NPL == 3) {
                        am[i][0] = qd_dp4a_uu(ql, xl.y, am[i][0]);
                        am[i][1] = qd_dp4a_uu(qh, xh.y, am[i][1]);
                        al[i][0] = qd_dp4a_uu(ql, xl.z, al[i][0]);
                        al[i][1] = qd_dp4a_uu(qh, xh.z, al[i][1]);
                    } else {
                        al[i][0] = qd_dp4a_uu(ql, xl.y, al[i][0]);
                        al[i][1] = qd_dp4a_uu(qh, xh.y, al[i][1]);
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

// qd4_group_math with the rows' bytes read here (rows r0..r0+RPL-1 of rowp; NULL rows skipped).
template <int NT, int RPL, bool kSmemRows, int NPL>
__device__ __forceinline__ void qd4_group(const uint8_t* const (&rowp)[4], int r0, int g, int G, const uint4* X,
                                          const float4* XS, int nt, float (&acc)[4][NT], const int* vidx) {
    const int b = g >> 2, c = g & 3;
    uint4 hd[RPL], q0[RPL], q1[RPL];
    bool live[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        const uint8_t* rp = rowp[r0 + i];
        live[i] = rp != nullptr;
        if (live[i]) {
            const uint8_t* blk = rp + (int64_t)b * kQ4KBytes;
            hd[i] = qd_ld16<kSmemRows>(blk);
            q0[i] = qd_ld16<kSmemRows>(blk + 16 + 32 * c);
            q1[i] = qd_ld16<kSmemRows>(blk + 32 + 32 * c);
        } else {
            hd[i] = q0[i] = q1[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    qd4_group_math<NT, RPL, NPL>(hd, q0, q1, live, r0, g, G, X, XS, nt, acc, vidx);
}

// acc[r][t] += row r . vector vidx[t] (t < nt) for 4 Q4_K rows of nblk super-blocks.
// Rows may be NULL (skipped).  Vector v lives at X + v*16*G, XS + v*G.  Lanes split
// into row subsets so that every lane reuses one group's activations over 4, 2 or 1
// rows (long rows: 4; 12-23 groups: 2; shorter: 1).
template <int NT, bool kSmemRows, int NPL>
__device__ __forceinline__ void qd4_rows4(const uint8_t* const (&rowp)[4], int nblk, const uint4* X,
                                          const float4* XS, int nt, int lane, float (&acc)[4][NT],
                                          const int* vidx = nullptr) {
    const int G = nblk * 4;
    if (G >= 24) {
        for (int g = lane; g < G; g += 32) qd4_group<NT, 4, kSmemRows, NPL>(rowp, 0, g, G, X, XS, nt, acc, vidx);
    } else if (G >= 12) {
        const int rs = lane >> 4;
        for (int g = lane & 15; g < G; g += 16) qd4_group<NT, 2, kSmemRows, NPL>(rowp, 2 * rs, g, G, X, XS, nt, acc, vidx);
    } else {
        const int rs = lane >> 3;
        for (int g = lane & 7; g < G; g += 8) qd4_group<NT, 1, kSmemRows, NPL>(rowp, rs, g, G, X, XS, nt, acc, vidx);
    }
}

}  // namespace moe
