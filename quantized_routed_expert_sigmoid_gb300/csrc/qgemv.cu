// qgemv.cu -- fused dequant-GEMV for the experts at decode sizes.
//
// The pages run the card experts on the stored GGUF quantization ("bloomery
// README 0.3.1", Status table, "Quant types" row; "Why it is fast": kernels
// "on the stored quantization").  At a few tokens per expert the expert FFN
// is a matrix-vector product bound by HBM bandwidth: every weight byte of the
// chosen experts is read once, dequantized in registers and multiplied in
// fp32.  One launch covers all active experts:
//   GATEUP : h[i, r] = silu(Wg[e][r] . v_i) * (Wu[e][r] . v_i)   (r < I)
//   DOWN   : y[i, n] = Wd[e][n] . v_i                            (n < H)
// Block formats (public GGUF layout):
//   Q4_K  w = d*sc_j*q - dmin*m_j  per 256-weight super-block of 144 bytes,
//   Q8_0  w = d*q                  per 32-weight block of 34 bytes.
// Work split: grid.y = active-expert slot, grid.x = tiles of rows.  Each warp
// takes 4 weight rows at a time (gate/up: 2 rows of each matrix) so that one
// read of the staged activation feeds four rows.  Per warp iteration every
// lane covers 32 weights: Q4_K one 16-byte quant chunk (8 lanes per
// super-block), Q8_0 one whole block.  The activations of up to NT pairs are
// staged in shared memory in exactly the per-lane order of that walk
// (conflict-free 16-byte reads), with their 16-element sums for the Q4_K min
// term.  Reductions run in a fixed order: the same bits on every run.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerUnit = 4;  // weight rows a warp holds at once

__device__ __forceinline__ float byte_to_float(uint32_t word, int b) {
    // 0x4B0000bb is 2^23 + bb as an fp32; subtracting 2^23 leaves bb exactly.
    return __int_as_float(__byte_perm(word, 0x4B00u, 0x5440u | (uint32_t)b)) - 8388608.0f;
}

// Same for a byte that holds int8 + 128: leaves the signed value exactly.
__device__ __forceinline__ float sbyte_to_float(uint32_t word, int b) {
    return __int_as_float(__byte_perm(word, 0x4B00u, 0x5440u | (uint32_t)b)) - 8388736.0f;
}

__device__ __forceinline__ uint16_t ldg_u16(const uint8_t* p) {
    return __ldg(reinterpret_cast<const unsigned short*>(p));
}

template <int QT>
struct Walk;

// Q4_K: lane l of iteration it covers super-block it*4 + l/8, quant chunk l%8.
template <>
struct Walk<MOE_Q4_K> {
    static constexpr int kBlocksPerIter = 4;
    static constexpr int kBlockWeights = kQ4KWeights;
    __device__ static int blk(int it, int lane) { return it * 4 + (lane >> 3); }
    // element offset inside the row of the first of 4 values of slot i4
    __device__ static int pos(int it, int lane, int i4) {
        const int ch = lane & 7, c = ch >> 1, half = ch & 1, hi = i4 >> 2;
        return blk(it, lane) * 256 + 64 * c + 32 * hi + 16 * half + 4 * (i4 & 3);
    }
};

// Q8_0: lane l of iteration it covers block it*32 + l.
template <>
struct Walk<MOE_Q8_0> {
    static constexpr int kBlocksPerIter = 32;
    static constexpr int kBlockWeights = kQ80Weights;
    __device__ static int blk(int it, int lane) { return it * 32 + lane; }
    __device__ static int pos(int it, int lane, int i4) { return blk(it, lane) * 32 + 4 * i4; }
};

__device__ __forceinline__ void load_vec4(const void* v, bool bf16, int64_t idx, float4& out) {
    if (bf16) {
        const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(v) + idx);
        out.x = __uint_as_float(raw.x << 16);
        out.y = __uint_as_float(raw.x & 0xFFFF0000u);
        out.z = __uint_as_float(raw.y << 16);
        out.w = __uint_as_float(raw.y & 0xFFFF0000u);
    } else {
        out = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(v) + idx);
    }
}

template <int QT, bool GATEUP, int NT>
__global__ void __launch_bounds__(kThreads) qgemv_kernel(GemvArgs a, int iters, int units_per_warp) {
    using W = Walk<QT>;
    extern __shared__ float4 xs[];                    // [NT][iters*256] float4
    float2* xsum = reinterpret_cast<float2*>(xs + (size_t)NT * iters * 256);  // [NT][iters*32]
    __shared__ int s_e, s_start, s_n;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // ---- which expert this CTA serves: the blockIdx.y-th expert with pairs
    if (warp == 0) {
        if (a.offsets == nullptr) {
            if (lane == 0) { s_e = blockIdx.y == 0 ? 0 : -1; s_start = 0; s_n = a.n_pairs; }
        } else {
            const int want = blockIdx.y;
            int seen = 0, found = -1, fstart = 0, fn = 0;
            for (int base = 0; base < a.E && found < 0; base += 32) {
                const int e = base + lane;
                int o0 = 0, cnt = 0;
                if (e < a.E) { o0 = a.offsets[e]; cnt = a.offsets[e + 1] - o0; }
                const unsigned nz = __ballot_sync(0xffffffffu, cnt > 0);
                const int here = __popc(nz);
                if (seen + here > want) {
                    const int idx = want - seen;
                    const bool me = cnt > 0 && __popc(nz & ((1u << lane) - 1u)) == idx;
                    const unsigned who = __ballot_sync(0xffffffffu, me);
                    const int src = __ffs(who) - 1;
                    found = __shfl_sync(0xffffffffu, e, src);
                    fstart = __shfl_sync(0xffffffffu, o0, src);
                    fn = __shfl_sync(0xffffffffu, cnt, src);
                }
                seen += here;
            }
            if (lane == 0) { s_e = found; s_start = fstart; s_n = fn; }
        }
    }
    __syncthreads();
    const int e = s_e;
    if (e < 0) return;
    const int start = s_start, n_tot = s_n;

    const int nblk = a.K / W::kBlockWeights;
    const int64_t rb = (int64_t)nblk * (QT == MOE_Q4_K ? kQ4KBytes : kQ80Bytes);
    const uint8_t* w0 = a.w0 + (int64_t)e * a.expert_stride;
    const uint8_t* w1 = GATEUP ? a.w1 + (int64_t)e * a.expert_stride : nullptr;
    const int row_step = GATEUP ? 2 : 4;              // output rows per unit
    const int n_units = a.rows / row_step;
    const int slots = iters * 256;                    // float4 slots per staged vector

    for (int pb = 0; pb < n_tot; pb += NT) {
        const int nt = min(NT, n_tot - pb);
        // ---- stage the activation vectors of pairs start+pb .. +nt in walk order
        for (int idx = threadIdx.x; idx < nt * slots; idx += kThreads) {
            const int t = idx / slots, s = idx - t * slots;
            const int it = s >> 8, i4 = (s >> 5) & 7, ln = s & 31;
            const int p = W::pos(it, ln, i4);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (W::blk(it, ln) < nblk) {
                const int i = start + pb + t;
                int64_t row;
                if (GATEUP) row = a.sorted_pairs ? (int64_t)(a.sorted_pairs[i] / a.k) : (int64_t)i;
                else row = i;
                load_vec4(a.vin, a.vin_bf16, row * a.K + p, v);
            }
            xs[(size_t)t * slots + s] = v;
        }
        __syncthreads();
        if (QT == MOE_Q4_K) {
            for (int idx = threadIdx.x; idx < nt * iters * 32; idx += kThreads) {
                const int t = idx / (iters * 32), r = idx - t * iters * 32;
                const int it = r >> 5, ln = r & 31;
                const float4* base = xs + (size_t)t * slots + it * 256 + ln;
                float lo = 0.f, hi = 0.f;
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    const float4 v = base[i4 * 32];
                    lo += (v.x + v.y) + (v.z + v.w);
                    const float4 u = base[(i4 + 4) * 32];
                    hi += (u.x + u.y) + (u.z + u.w);
                }
                xsum[(size_t)t * iters * 32 + r] = make_float2(lo, hi);
            }
            __syncthreads();
        }

        // ---- each warp: units of 4 weight rows
        for (int ui = 0; ui < units_per_warp; ++ui) {
            const int unit = (blockIdx.x * kWarps + warp) * units_per_warp + ui;
            if (unit >= n_units) break;
            const uint8_t* rowp[kRowsPerUnit];
            if (GATEUP) {
                const int r0 = unit * 2;
                rowp[0] = w0 + (int64_t)r0 * rb;
                rowp[1] = w0 + (int64_t)(r0 + 1) * rb;
                rowp[2] = w1 + (int64_t)r0 * rb;
                rowp[3] = w1 + (int64_t)(r0 + 1) * rb;
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) rowp[r] = w0 + (int64_t)(unit * 4 + r) * rb;
            }
            float acc[kRowsPerUnit][NT];
#pragma unroll
            for (int r = 0; r < kRowsPerUnit; ++r)
#pragma unroll
                for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;

            for (int it = 0; it < iters; ++it) {
                const int b = W::blk(it, lane);
                if (b >= nblk) continue;
                if (QT == MOE_Q4_K) {
                    const int ch = lane & 7, jj = (ch >> 1) & 1, upper = ch >> 2;  // c = ch>>1: j0 = 2c
                    uint4 q[kRowsPerUnit], hd[kRowsPerUnit];
#pragma unroll
                    for (int r = 0; r < kRowsPerUnit; ++r) {
                        const uint8_t* bp = rowp[r] + (int64_t)b * kQ4KBytes;
                        hd[r] = __ldg(reinterpret_cast<const uint4*>(bp));
                        q[r] = __ldg(reinterpret_cast<const uint4*>(bp + 16 + 16 * ch));
                    }
                    // per row: d*sc and dmin*m for sub-blocks j0 = 2c (low nibbles), j1 = 2c+1 (high)
                    float fsc[kRowsPerUnit][2], fm[kRowsPerUnit][2];
#pragma unroll
                    for (int r = 0; r < kRowsPerUnit; ++r) {
                        const float d = __half2float(__ushort_as_half((unsigned short)(hd[r].x & 0xFFFFu)));
                        const float dmin = __half2float(__ushort_as_half((unsigned short)(hd[r].x >> 16)));
#pragma unroll
                        for (int s = 0; s < 2; ++s) {
                            const int j = 2 * jj + s;              // j & 3 for sub-block 2c+s
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
                            float dl[kRowsPerUnit], dh[kRowsPerUnit];
#pragma unroll
                            for (int r = 0; r < kRowsPerUnit; ++r) { dl[r] = 0.f; dh[r] = 0.f; }
#pragma unroll
                            for (int w4 = 0; w4 < 4; ++w4) {
                                const float4 xl = xb[(size_t)t * slots + w4 * 32];
                                const float4 xh = xb[(size_t)t * slots + (w4 + 4) * 32];
#pragma unroll
                                for (int r = 0; r < kRowsPerUnit; ++r) {
                                    const uint32_t word = w4 == 0 ? q[r].x : w4 == 1 ? q[r].y : w4 == 2 ? q[r].z : q[r].w;
                                    const uint32_t lo = word & 0x0F0F0F0Fu, hi = (word >> 4) & 0x0F0F0F0Fu;
                                    dl[r] = fmaf(byte_to_float(lo, 0), xl.x, dl[r]);
                                    dl[r] = fmaf(byte_to_float(lo, 1), xl.y, dl[r]);
                                    dl[r] = fmaf(byte_to_float(lo, 2), xl.z, dl[r]);
                                    dl[r] = fmaf(byte_to_float(lo, 3), xl.w, dl[r]);
                                    dh[r] = fmaf(byte_to_float(hi, 0), xh.x, dh[r]);
                                    dh[r] = fmaf(byte_to_float(hi, 1), xh.y, dh[r]);
                                    dh[r] = fmaf(byte_to_float(hi, 2), xh.z, dh[r]);
                                    dh[r] = fmaf(byte_to_float(hi, 3), xh.w, dh[r]);
                                }
                            }
                            const float2 sx = xsb[(size_t)t * iters * 32];
#pragma unroll
                            for (int r = 0; r < kRowsPerUnit; ++r) {
                                float v = fsc[r][0] * dl[r];
                                v = fmaf(fsc[r][1], dh[r], v);
                                v = fmaf(-fm[r][0], sx.x, v);
                                v = fmaf(-fm[r][1], sx.y, v);
                                acc[r][t] += v;
                            }
                        }
                    }
                } else {
                    // Q8_0: one 34-byte block per lane (2-byte aligned): fp16 d + 32 int8.
                    uint32_t qw[kRowsPerUnit][8];
                    float dd[kRowsPerUnit];
#pragma unroll
                    for (int r = 0; r < kRowsPerUnit; ++r) {
                        const uint8_t* bp = rowp[r] + (int64_t)b * kQ80Bytes;
                        dd[r] = __half2float(__ushort_as_half(ldg_u16(bp)));
#pragma unroll
                        for (int w = 0; w < 8; ++w) {
                            const uint32_t lo16 = ldg_u16(bp + 2 + 4 * w);
                            const uint32_t hi16 = ldg_u16(bp + 4 + 4 * w);
                            qw[r][w] = (lo16 | (hi16 << 16)) ^ 0x80808080u;  // int8 + 128 as bytes
                        }
                    }
                    const float4* xb = xs + it * 256 + lane;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (t < nt) {
                            float dt[kRowsPerUnit];
#pragma unroll
                            for (int r = 0; r < kRowsPerUnit; ++r) dt[r] = 0.f;
#pragma unroll
                            for (int w = 0; w < 8; ++w) {
                                const float4 xv = xb[(size_t)t * slots + w * 32];
#pragma unroll
                                for (int r = 0; r < kRowsPerUnit; ++r) {
                                    dt[r] = fmaf(sbyte_to_float(qw[r][w], 0), xv.x, dt[r]);
                                    dt[r] = fmaf(sbyte_to_float(qw[r][w], 1), xv.y, dt[r]);
                                    dt[r] = fmaf(sbyte_to_float(qw[r][w], 2), xv.z, dt[r]);
                                    dt[r] = fmaf(sbyte_to_float(qw[r][w], 3), xv.w, dt[r]);
                                }
                            }
#pragma unroll
                            for (int r = 0; r < kRowsPerUnit; ++r) acc[r][t] = fmaf(dd[r], dt[r], acc[r][t]);
                        }
                    }
                }
            }
            // ---- reduce across the warp (fixed butterfly) and write
#pragma unroll
            for (int r = 0; r < kRowsPerUnit; ++r)
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    float v = acc[r][t];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    acc[r][t] = v;
                }
            if (GATEUP) {
                if (lane < 2 * NT) {
                    const int t = lane >> 1, ri = lane & 1;
                    if (t < nt) {
                        float g = 0.f, u = 0.f;
#pragma unroll
                        for (int tt = 0; tt < NT; ++tt)
                            if (tt == t) { g = ri ? acc[1][tt] : acc[0][tt]; u = ri ? acc[3][tt] : acc[2][tt]; }
                        const float hval = g / (1.0f + expf(-g)) * u;
                        a.out[(int64_t)(start + pb + t) * a.rows + unit * 2 + ri] = hval;
                    }
                }
            } else {
                if (lane < 4 * NT) {
                    const int t = lane >> 2, ri = lane & 3;
                    if (t < nt) {
                        float v = 0.f;
#pragma unroll
                        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                            for (int r = 0; r < 4; ++r)
                                if (tt == t && r == ri) v = acc[r][tt];
                        a.out[(int64_t)(start + pb + t) * a.rows + unit * 4 + ri] = v;
                    }
                }
            }
        }
        __syncthreads();
    }
}

template <int QT, bool GU, int NT>
cudaError_t launch_one(const GemvArgs& a, int iters, int grid_y, cudaStream_t s) {
    const size_t smem = (size_t)NT * iters * 256 * sizeof(float4) + (size_t)NT * iters * 32 * sizeof(float2);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(qgemv_kernel<QT, GU, NT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    const int row_step = GU ? 2 : 4;
    const int n_units = a.rows / row_step;
    const int upw = 1;
    const int grid_x = (n_units + kWarps * upw - 1) / (kWarps * upw);
    qgemv_kernel<QT, GU, NT><<<dim3(grid_x, grid_y), kThreads, smem, s>>>(a, iters, upw);
    return cudaGetLastError();
}

template <int QT, bool GU>
cudaError_t launch_nt(const GemvArgs& a, int nt, int iters, int grid_y, cudaStream_t s) {
    switch (nt) {
        case 1: return launch_one<QT, GU, 1>(a, iters, grid_y, s);
        case 2: return launch_one<QT, GU, 2>(a, iters, grid_y, s);
        case 4: return launch_one<QT, GU, 4>(a, iters, grid_y, s);
        default: return launch_one<QT, GU, 8>(a, iters, grid_y, s);
    }
}

}  // namespace

cudaError_t launch_qgemv(const GemvArgs& a, cudaStream_t s) {
    if (a.n_pairs <= 0) return cudaSuccess;
    const int bw = a.qtype == MOE_Q4_K ? kQ4KWeights : kQ80Weights;
    const int bpi = a.qtype == MOE_Q4_K ? 4 : 32;
    const int nblk = a.K / bw;
    const int iters = (nblk + bpi - 1) / bpi;
    // Tokens per pass: at most the pairs one expert can hold (distinct ids per
    // token: <= tokens), at most 8, and a staged tile of at most ~64 KB.
    const int per_expert_max = a.sorted_pairs ? (a.n_pairs / a.k) : a.n_pairs;
    int nt = 8;
    while (nt > 1 && ((size_t)nt * iters * 4096 > 64 * 1024 || nt / 2 >= per_expert_max)) nt /= 2;
    const int grid_y = a.offsets ? (a.n_pairs < a.E ? a.n_pairs : a.E) : 1;
    if (a.qtype == MOE_Q4_K)
        return a.gateup ? launch_nt<MOE_Q4_K, true>(a, nt, iters, grid_y, s)
                        : launch_nt<MOE_Q4_K, false>(a, nt, iters, grid_y, s);
    return a.gateup ? launch_nt<MOE_Q8_0, true>(a, nt, iters, grid_y, s)
                    : launch_nt<MOE_Q8_0, false>(a, nt, iters, grid_y, s);
}

}  // namespace moe
