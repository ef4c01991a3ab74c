// qgemv.cu -- fused dequant-GEMV for the experts at decode sizes where the segmented
// kernels of gemv_seg.cu do not apply (Q8_0 weights, such as a Q8_0 shared expert, in the
// stored GGUF blocks or repacked by moe_weights_prepare, or more than 256 experts).
//
// The pages run the card experts on the stored GGUF quantization ("bloomery
// README 0.3.1", Status table, "Quant types" row; "Why it is fast": kernels
// on the stored quantization).  At a few tokens per expert the expert FFN is a
// matrix-vector product bound by HBM bandwidth: every weight byte of the
// chosen experts is read once, dequantized in registers and multiplied in
// fp32.  One launch covers all active experts:
//   GATEUP : h[i, r] = silu(Wg[e][r] . v_i) * (Wu[e][r] . v_i)   (r < I)
//   DOWN   : y[i, n] = Wd[e][n] . v_i                            (n < H)
// Work split: grid.y = active-expert slot, grid.x = tiles of rows; each warp
// takes 4 weight rows at a time (gate/up: 2 rows of each matrix) so one read
// of the staged activations feeds four rows (see qdot.cuh for the walk).
// Reductions run in a fixed order: the same bits on every run.
#include <algorithm>

#include "internal.cuh"
#include "qdot.cuh"
#include "qdot_k56.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// Requests [src, src + bytes) into L2 (a hint; 16-byte multiples, pieces of at most 64 KB).
__device__ __forceinline__ void prefetch_rows_l2(const uint8_t* src, int64_t bytes) {
    for (int64_t o = 0; o < bytes; o += 65536) {
        const uint32_t n = (uint32_t)(bytes - o < 65536 ? bytes - o : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + o), "r"(n) : "memory");
    }
}

// Sum a unit's acc over the warp and store it.  Gate/up: rows 0, 1 = gate of the unit's
// rows 2 unit, 2 unit + 1, rows 2, 3 = up of the same rows -> h[t][row] = SiLU(gate) * up;
// down: rows 0..3 -> y[t][4 unit + r].
template <int NT, bool GATEUP>
__device__ __forceinline__ void qd_store_units(const float (&acc)[4][NT], int lane, int nt, float* out, int rows,
                                               int unit) {
    constexpr int sh = qd_red_shift<NT>();
    const float v = qd_warp_reduce_t<NT>(acc);
    const int i = lane >> sh, r = i / NT, t = i - r * NT;
    const bool lead = (lane & ((1 << sh) - 1)) == 0 && t < nt;
    if (GATEUP) {
        const float u = __shfl_xor_sync(0xffffffffu, v, (2 * NT) << sh);
        if (lead && r < 2) out[(int64_t)t * rows + unit * 2 + r] = v / (1.0f + expf(-v)) * u;
    } else if (lead) {
        out[(int64_t)t * rows + unit * 4 + r] = v;
    }
}

// NPL: activation planes of the Q4_K path (2 for bf16 input, 3 otherwise; unused for Q8_0)
template <int QT, bool GATEUP, int NT, int NPL>
__global__ void __launch_bounds__(kThreads, 2) qgemv_kernel(GemvArgs a, int iters, int units_per_warp) {
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

    const int nblk = a.K / Walk<QT>::kBlockWeights;
    const int64_t rb = QT == MOE_Q8_0 && a.q80r ? q80r_row_bytes(a.K) : (int64_t)nblk * Walk<QT>::kBlockBytes;
    const uint8_t* w0 = a.w0 + (int64_t)e * a.expert_stride;
    const uint8_t* w1 = GATEUP ? a.w1 + (int64_t)e * a.expert_stride : nullptr;
    const int n_units = a.rows / (GATEUP ? 2 : 4);
    const int slots = iters * 256;
    // this CTA's weight rows (contiguous: units_per_warp units of every warp) into L2 before staging
    if (threadIdx.x == 0) {
        const int u0 = blockIdx.x * kWarps * units_per_warp;
        const int u1 = min(n_units, u0 + kWarps * units_per_warp);
        const int rpu = GATEUP ? 2 : 4;
        if (u1 > u0 && (rb % 16) == 0) {
            prefetch_rows_l2(w0 + (int64_t)u0 * rpu * rb, (int64_t)(u1 - u0) * rpu * rb);
            if (GATEUP) prefetch_rows_l2(w1 + (int64_t)u0 * rpu * rb, (int64_t)(u1 - u0) * rpu * rb);
        }
    }

    __shared__ int s_rows[NT];
    for (int pb = 0; pb < n_tot; pb += NT) {
        const int nt = min(NT, n_tot - pb);
        if constexpr (QT != MOE_Q8_0) {                     // K-quants and MXFP4: integer planes
            // ---- stage the activation vectors as integer planes (qdot.cuh)
            uint4* X = reinterpret_cast<uint4*>(xs);
            float4* XS = reinterpret_cast<float4*>(X + (size_t)NT * 16 * qd4_groups(a.K));
            if (threadIdx.x < nt) {
                const int i = start + pb + threadIdx.x;
                s_rows[threadIdx.x] = (GATEUP && a.sorted_pairs) ? a.sorted_pairs[i] / a.k : i;
            }
            __syncthreads();
            qd4_stage_par<NPL>(a.vin, a.vin_bf16, false, a.K, nt, s_rows, a.K, X, XS, threadIdx.x, kThreads);
            __syncthreads();
            for (int ui = 0; ui < units_per_warp; ++ui) {
                const int unit = (blockIdx.x * kWarps + warp) * units_per_warp + ui;
                if (unit >= n_units) break;
                const uint8_t* rowp[4];
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
                float acc[4][NT];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
                if constexpr (QT == MOE_Q4_K) qd4_rows4<NT, false, NPL>(rowp, nblk, X, XS, nt, lane, acc);
                else qd56_rows4<QT, NT, NPL>(rowp, nblk, X, XS, nt, lane, acc);
                qd_store_units<NT, GATEUP>(acc, lane, nt, a.out + (int64_t)(start + pb) * a.rows, a.rows, unit);
            }
            __syncthreads();
        } else {
        // ---- stage the activation vectors of pairs start+pb .. +nt in walk order
        for (int t = 0; t < nt; ++t) {
            const int i = start + pb + t;
            int64_t row = i;
            if (GATEUP && a.sorted_pairs) row = a.sorted_pairs[i] / a.k;
            const void* src = a.vin_bf16 ? (const void*)(reinterpret_cast<const __nv_bfloat16*>(a.vin) + row * a.K)
                                         : (const void*)(reinterpret_cast<const float*>(a.vin) + row * a.K);
            qd_stage<QT>(src, a.vin_bf16, false, a.K, iters, xs + (size_t)t * slots, threadIdx.x, kThreads);
        }
        __syncthreads();
        if constexpr (QT == MOE_Q4_K) {
            for (int t = 0; t < nt; ++t)
                qd_stage_sums(xs + (size_t)t * slots, xsum + (size_t)t * iters * 32, iters, threadIdx.x, kThreads);
            __syncthreads();
        }
        for (int ui = 0; ui < units_per_warp; ++ui) {
            const int unit = (blockIdx.x * kWarps + warp) * units_per_warp + ui;
            if (unit >= n_units) break;
            const uint8_t* rowp[4];
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
            float acc[4][NT];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
            qd_rows4<QT, NT>(rowp, nblk, iters, xs, slots, xsum, iters * 32, nt, lane, acc, nullptr, a.q80r);
            qd_store_units<NT, GATEUP>(acc, lane, nt, a.out + (int64_t)(start + pb) * a.rows, a.rows, unit);
        }
        __syncthreads();
        }
    }
}

template <int QT, bool GU, int NT, int NPL>
cudaError_t launch_one(const GemvArgs& a, int iters, int grid_y, cudaStream_t s) {
    const size_t smem = QT != MOE_Q8_0 ? (size_t)NT * qd4_vec_bytes(a.K)
                                       : (size_t)NT * iters * 256 * sizeof(float4) + (size_t)NT * iters * 32 * sizeof(float2);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(qgemv_kernel<QT, GU, NT, NPL>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    // units per warp: enough that the grid is about two waves of two CTAs per SM
    const int n_units = a.rows / (GU ? 2 : 4);
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t target_warps = (int64_t)kWarps * 4 * (sms > 0 ? sms : 152);
    const int upw = (int)std::max<int64_t>(1, ((int64_t)n_units * grid_y + target_warps - 1) / target_warps);
    const int grid_x = (n_units + kWarps * upw - 1) / (kWarps * upw);
    qgemv_kernel<QT, GU, NT, NPL><<<dim3(grid_x, grid_y), kThreads, smem, s>>>(a, iters, upw);
    return cudaGetLastError();
}

template <int QT, bool GU, int NPL>
cudaError_t launch_nt(const GemvArgs& a, int nt, int iters, int grid_y, cudaStream_t s) {
    if constexpr (QT == MOE_Q5_K || QT == MOE_Q6_K || QT == MOE_Q3_K || QT == MOE_MXFP4) {   // codes take registers
        return nt == 1 ? launch_one<QT, GU, 1, NPL>(a, iters, grid_y, s) : launch_one<QT, GU, 2, NPL>(a, iters, grid_y, s);
    } else {
        switch (nt) {
            case 1: return launch_one<QT, GU, 1, NPL>(a, iters, grid_y, s);
            case 2: return launch_one<QT, GU, 2, NPL>(a, iters, grid_y, s);
            case 4: return launch_one<QT, GU, 4, NPL>(a, iters, grid_y, s);
            default: return launch_one<QT, GU, 8, NPL>(a, iters, grid_y, s);
        }
    }
}

}  // namespace

cudaError_t launch_qgemv(const GemvArgs& a, cudaStream_t s) {
    if (a.n_pairs <= 0) return cudaSuccess;
    const int iters = a.qtype == MOE_Q8_0 ? walk_iters<MOE_Q8_0>(a.K) : walk_iters<MOE_Q4_K>(a.K);
    // Tokens per pass: at most the pairs one expert can hold (distinct ids per
    // token: <= tokens), at most 8, and a staged tile of at most ~64 KB.
    const int per_expert_max = a.sorted_pairs ? (a.n_pairs / a.k) : a.n_pairs;
    const size_t per_vec = a.qtype != MOE_Q8_0 ? qd4_vec_bytes(a.K) : (size_t)iters * 4096;
    int nt = 8;
    while (nt > 1 && ((size_t)nt * per_vec > 64 * 1024 || nt / 2 >= per_expert_max)) nt /= 2;
    const int grid_y = a.offsets ? (a.n_pairs < a.E ? a.n_pairs : a.E) : 1;
    auto planes = [&](auto qt) -> cudaError_t {
        constexpr int Q = decltype(qt)::value;
        if (!a.gateup) return launch_nt<Q, false, 3>(a, nt, iters, grid_y, s);   // h is fp32
        return a.vin_bf16 ? launch_nt<Q, true, 2>(a, nt, iters, grid_y, s) : launch_nt<Q, true, 3>(a, nt, iters, grid_y, s);
    };
    if (a.qtype == MOE_Q4_K) return planes(std::integral_constant<int, MOE_Q4_K>{});
    if (a.qtype == MOE_Q5_K) return planes(std::integral_constant<int, MOE_Q5_K>{});
    if (a.qtype == MOE_Q6_K) return planes(std::integral_constant<int, MOE_Q6_K>{});
    if (a.qtype == MOE_Q3_K) return planes(std::integral_constant<int, MOE_Q3_K>{});
    if (a.qtype == MOE_MXFP4) return planes(std::integral_constant<int, MOE_MXFP4>{});
    return a.gateup ? launch_nt<MOE_Q8_0, true, 3>(a, nt, iters, grid_y, s)
                    : launch_nt<MOE_Q8_0, false, 3>(a, nt, iters, grid_y, s);
}

}  // namespace moe
