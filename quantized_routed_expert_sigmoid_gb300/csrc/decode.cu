// decode.cu -- the whole MoE layer at a few tokens in one launch.
//
// The pages run a decode step as one captured CUDA graph ("bloomery README
// 0.3.1", "Why it is fast") with the routed experts on the card.  At T <= 4
// tokens the layer moves ~22 MB (hidden 2048) to ~450 MB (hidden 7168) of
// expert weights, a few microseconds of HBM time, so the fixed cost of a chain
// of small kernels (launch, ramp-up, drain) would dominate.  Here one
// cooperative persistent grid (one CTA per SM) runs every step:
//   phase 0  router logits, experts spread over the CTAs; the activations are
//            staged in shared memory meanwhile          -> grid barrier 1
//   routing  every CTA selects the top-k of the T tokens itself (identical
//            results) and orders the pairs by expert; CTA 0 publishes them
//   phase 1  gate/up + SwiGLU units (2 rows of each matrix of one expert, all
//            its tokens) over all warps of the grid, shared-expert units too;
//            each CTA prefetches into L2 the down rows it will need next
//                                                       -> grid barrier 2
//   phase 2  each CTA owns a slice of the output rows: down rows of every
//            active expert (and the shared expert) against the staged h,
//            then the gate-weighted combine in fixed order, + residual.
// The arithmetic and its order are those of the separate kernels (qdot.cuh,
// route_common.cuh), so results match them bit for bit.  Grid barriers are
// bounded waits; on timeout the kernel records MOE_ERR_TIMEOUT and returns.
#include "internal.cuh"
#include "qdot.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kDW = 8;
constexpr int kDT = kDW * 32;
constexpr int kDMaxT = 4;
constexpr int kDMaxP = 64;
constexpr int kDMaxE = 256;
constexpr uint64_t kBarrierLimitNs = 2000000000ull;

struct DecodeParams {
    RouteCfgDev rc;
    const float* Wr;
    const float* bias;
    const void* x;
    int x_bf16;
    int T, H, I;
    int qtype;
    const uint8_t* wg;
    const uint8_t* wu;
    const uint8_t* wd;
    int64_t stride_gu, stride_d;
    int I_s, s_qtype;
    const uint8_t* sg;
    const uint8_t* su;
    const uint8_t* sd;
    float* logits;
    int32_t* ids;
    float* gw;
    int32_t* sorted;
    int32_t* offsets;
    int32_t* pair_pos;
    float* h;
    float* h_s;
    float* out;
    int accumulate;
    WsHeader* hdr;
    DecodeSync* sync;
    int prefetch_down;
    // shared-memory layout (bytes)
    int off_xs_r, off_xsum_r, off_xs_s, off_xsum_s;      // phase 1 staging (x in both walks)
    int off_hs_r, off_hsum_r, off_hs_s, off_hsum_s;      // phase 2 staging (h, h_s)
    int off_topk, off_y;
    int it_H_r, it_I_r, it_H_s, it_Is_s;                 // walk iterations
};

__device__ __forceinline__ uint64_t dtime() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// All CTAs of the (co-resident) grid meet here.  Returns false on timeout.
__device__ bool grid_barrier(uint32_t* ctr, uint32_t target, volatile int* s_abort) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        const uint64_t t0 = dtime();
        while (ld_acquire(ctr) < target) {
            if (dtime() - t0 > kBarrierLimitNs) { *s_abort = 1; break; }
            __nanosleep(64);
        }
        __threadfence();
    }
    __syncthreads();
    return *s_abort == 0;
}

template <int QT>
__device__ __forceinline__ int64_t row_bytes_q(int K) {
    return (int64_t)(K / Walk<QT>::kBlockWeights) * Walk<QT>::kBlockBytes;
}

// One gate/up unit: rows r0, r0+1 of gate and up of one expert, vectors vidx[0..nt).
template <int QT, int NT>
__device__ __forceinline__ void gateup_unit(const uint8_t* g, const uint8_t* u, int r0, int K, int iters,
                                            const float4* xs, const float2* xsum, const int (&vidx)[NT], int nt,
                                            int lane, float* hout, const int (&orow)[NT], int ostride) {
    const int64_t rb = row_bytes_q<QT>(K);
    const int nblk = K / Walk<QT>::kBlockWeights;
    const uint8_t* rowp[4] = {g + (int64_t)r0 * rb, g + (int64_t)(r0 + 1) * rb, u + (int64_t)r0 * rb,
                              u + (int64_t)(r0 + 1) * rb};
    float acc[4][NT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
    qd_rows4<QT, NT>(rowp, nblk, iters, xs, iters * 256, xsum, iters * 32, nt, lane, acc, vidx);
    qd_warp_reduce<NT>(acc);
    if (lane < 2 * NT) {
        const int t = lane >> 1, ri = lane & 1;
        if (t < nt) {
            const float gv = qd_pick<NT>(acc, ri, t), uv = qd_pick<NT>(acc, 2 + ri, t);
            int o = 0;
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
                if (tt == t) o = orow[tt];
            hout[(int64_t)o * ostride + r0 + ri] = gv / (1.0f + expf(-gv)) * uv;
        }
    }
}

// One down unit: rows n0..n0+3 of one expert's down matrix against vectors vidx[0..nt);
// results into ybuf[ycol[t] * ystride + (n - nbase)].
template <int QT, int NT>
__device__ __forceinline__ void down_unit(const uint8_t* d, int n0, int K, int iters, const float4* hs,
                                          const float2* hsum, const int (&vidx)[NT], int nt, int lane, float* ybuf,
                                          const int (&ycol)[NT], int ystride, int nbase) {
    const int64_t rb = row_bytes_q<QT>(K);
    const int nblk = K / Walk<QT>::kBlockWeights;
    const uint8_t* rowp[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) rowp[r] = d + (int64_t)(n0 + r) * rb;
    float acc[4][NT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
    qd_rows4<QT, NT>(rowp, nblk, iters, hs, iters * 256, hsum, iters * 32, nt, lane, acc, vidx);
    qd_warp_reduce<NT>(acc);
    if (lane < 4 * NT) {
        const int t = lane >> 2, ri = lane & 3;
        if (t < nt) {
            int c = 0;
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
                if (tt == t) c = ycol[tt];
            ybuf[c * ystride + (n0 + ri - nbase)] = qd_pick<NT>(acc, ri, t);
        }
    }
}

template <int QR, int QS, int NT>
__global__ void __launch_bounds__(kDT, 1) decode_layer_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ int32_t s_ids[kDMaxP];
    __shared__ float s_w[kDMaxP];
    __shared__ int32_t s_sorted[kDMaxP], s_ppos[kDMaxP];
    __shared__ int s_act_e[kDMaxP], s_act_start[kDMaxP], s_act_n[kDMaxP];
    __shared__ int s_nact;
    __shared__ float s_lpart[kDW][kDMaxT];
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, c = blockIdx.x;
    const int T = p.T, E = p.rc.E, k = p.rc.k, P = T * k, H = p.H, I = p.I;
    const bool xb = p.x_bf16 != 0;
    const bool has_shared = p.I_s > 0;

    if (*reinterpret_cast<volatile uint32_t*>(&p.sync->magic) != kDecodeMagic) {
        if (c == 0 && tid == 0) p.hdr->status = MOE_ERR_WORKSPACE;
        return;
    }
    if (tid == 0) s_abort = 0;
    if (c == 0 && tid == 0) p.hdr->status = MOE_OK;

    float4* xs_r = reinterpret_cast<float4*>(dsm + p.off_xs_r);
    float2* xsum_r = reinterpret_cast<float2*>(dsm + p.off_xsum_r);
    float4* xs_s = reinterpret_cast<float4*>(dsm + p.off_xs_s);
    float2* xsum_s = reinterpret_cast<float2*>(dsm + p.off_xsum_s);
    const int slots_H_r = p.it_H_r * 256, slots_H_s = p.it_H_s * 256;

    // ------------------------------------------------------------ phase 0: logits
    for (int e = c; e < E; e += G) {
        float acc[kDMaxT] = {0.f, 0.f, 0.f, 0.f};
        const float* wrow = p.Wr + (int64_t)e * H;
        for (int h = tid * 4; h < H; h += kDT * 4) {
            const float4 wv = __ldg(reinterpret_cast<const float4*>(wrow + h));
#pragma unroll
            for (int t = 0; t < kDMaxT; ++t) {
                if (t < T) {
                    const float4 xv = qd_load_vec4(p.x, xb, (int64_t)t * H + h);
                    acc[t] = fmaf(wv.x, xv.x, acc[t]);
                    acc[t] = fmaf(wv.y, xv.y, acc[t]);
                    acc[t] = fmaf(wv.z, xv.z, acc[t]);
                    acc[t] = fmaf(wv.w, xv.w, acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kDMaxT; ++t) {
            float v = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) s_lpart[warp][t] = v;
        }
        __syncthreads();
        if (tid < T) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kDW; ++w) s += s_lpart[w][tid];
            p.logits[(int64_t)tid * E + e] = s;
        }
        __syncthreads();
    }
    // stage x for phase 1 (an input: no dependency on other CTAs)
    for (int t = 0; t < T; ++t) {
        const void* src = xb ? (const void*)(reinterpret_cast<const __nv_bfloat16*>(p.x) + (int64_t)t * H)
                             : (const void*)(reinterpret_cast<const float*>(p.x) + (int64_t)t * H);
        qd_stage<QR>(src, xb, false, H, p.it_H_r, xs_r + (size_t)t * slots_H_r, tid, kDT);
        if (has_shared && QS != QR) qd_stage<QS>(src, xb, false, H, p.it_H_s, xs_s + (size_t)t * slots_H_s, tid, kDT);
    }
    if (!grid_barrier(&p.sync->bar1, (uint32_t)G, &s_abort)) goto timeout;
    if (QR == MOE_Q4_K)
        for (int t = 0; t < T; ++t) qd_stage_sums(xs_r + (size_t)t * slots_H_r, xsum_r + t * p.it_H_r * 32, p.it_H_r, tid, kDT);
    if (has_shared && QS == MOE_Q4_K) {
        const float4* xsrc = QS == QR ? xs_r : xs_s;
        for (int t = 0; t < T; ++t) qd_stage_sums(xsrc + (size_t)t * slots_H_s, xsum_s + t * p.it_H_s * 32, p.it_H_s, tid, kDT);
    }

    // ------------------------------------------------------------ routing (every CTA)
    if (warp < T) {
        float* sel = reinterpret_cast<float*>(dsm + p.off_topk) + warp * 2 * E;
        warp_topk(p.rc, p.logits + (int64_t)warp * E, p.bias, sel, sel + E, s_ids + warp * k, s_w + warp * k);
    }
    __syncthreads();
    if (warp == 0) {
        for (int i = lane; i < P; i += 32) {
            const int ei = s_ids[i];
            int rank = 0;
            for (int j = 0; j < P; ++j) {
                const int ej = s_ids[j];
                rank += (ej < ei || (ej == ei && j < i)) ? 1 : 0;
            }
            s_sorted[rank] = i;
            s_ppos[i] = rank;
        }
        __syncwarp();
        if (lane == 0) {
            int n = 0, prev = -1;
            for (int i = 0; i < P; ++i) {
                const int e = s_ids[s_sorted[i]];
                if (e != prev) { s_act_e[n] = e; s_act_start[n] = i; s_act_n[n] = 0; ++n; prev = e; }
                s_act_n[n - 1] += 1;
            }
            s_nact = n;
        }
    }
    __syncthreads();
    if (c == 0) {                          // publish the routing (debug views, status checks)
        for (int i = tid; i < P; i += kDT) {
            p.ids[i] = s_ids[i];
            p.gw[i] = s_w[i];
            p.sorted[i] = s_sorted[i];
            p.pair_pos[i] = s_ppos[i];
        }
        for (int e = tid; e <= E; e += kDT) {
            int cnt = 0;
            for (int i = 0; i < P; ++i) cnt += s_ids[i] < e ? 1 : 0;
            p.offsets[e] = cnt;
        }
    }
    {
        const int nact = s_nact;
        const int ngroups = H / 4;
        const int g0 = (int)((int64_t)c * ngroups / G), g1 = (int)((int64_t)(c + 1) * ngroups / G);
        const int64_t rbI = row_bytes_q<QR>(I);
        // L2 prefetch of this CTA's phase-2 down rows (contiguous per expert)
        if (p.prefetch_down && warp == kDW - 1 && g1 > g0) {
            const uint32_t bytes = (uint32_t)((g1 - g0) * 4 * rbI) & ~15u;
            for (int a = lane; a < nact; a += 32) {
                const uint8_t* src = p.wd + (int64_t)s_act_e[a] * p.stride_d + (int64_t)g0 * 4 * rbI;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
            }
            if (has_shared && lane == 0) {
                const int64_t rbIs = row_bytes_q<QS>(p.I_s);
                const uint32_t sb = (uint32_t)((g1 - g0) * 4 * rbIs) & ~15u;
                const uint8_t* src = p.sd + (int64_t)g0 * 4 * rbIs;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(sb) : "memory");
            }
        }

        // ------------------------------------------------------------ phase 1: gate/up units
        const int upe = I / 2;
        const int units_r = nact * upe;
        const int units_s = has_shared ? p.I_s / 2 : 0;
        for (int unit = c * kDW + warp; unit < units_r + units_s; unit += G * kDW) {
            if (unit < units_r) {
                const int a = unit / upe, r0 = (unit - a * upe) * 2;
                const int e = s_act_e[a], st = s_act_start[a], n = s_act_n[a];
                int vidx[NT], orow[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int pos = st + min(t, n - 1);
                    vidx[t] = s_sorted[pos] / k;        // token of the pair
                    orow[t] = pos;                      // h row = sorted position
                }
                gateup_unit<QR, NT>(p.wg + (int64_t)e * p.stride_gu, p.wu + (int64_t)e * p.stride_gu, r0, H,
                                        p.it_H_r, xs_r, xsum_r, vidx, n, lane, p.h, orow, I);
            } else {
                const int r0 = (unit - units_r) * 2;
                int vidx[NT], orow[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) { vidx[t] = min(t, T - 1); orow[t] = min(t, T - 1); }
                const float4* xsrc = QS == QR ? xs_r : xs_s;
                gateup_unit<QS, NT>(p.sg, p.su, r0, H, p.it_H_s, xsrc, xsum_s, vidx, T, lane, p.h_s, orow,
                                        p.I_s);
            }
        }
        if (!grid_barrier(&p.sync->bar2, (uint32_t)G, &s_abort)) goto timeout;

        // ------------------------------------------------------------ phase 2: down + combine
        float4* hs_r = reinterpret_cast<float4*>(dsm + p.off_hs_r);
        float2* hsum_r = reinterpret_cast<float2*>(dsm + p.off_hsum_r);
        float4* hs_s = reinterpret_cast<float4*>(dsm + p.off_hs_s);
        float2* hsum_s = reinterpret_cast<float2*>(dsm + p.off_hsum_s);
        const int slots_I_r = p.it_I_r * 256, slots_Is_s = p.it_Is_s * 256;
        qd_stage_many_f32<QR>(p.h, I, P, I, p.it_I_r, hs_r, tid, kDT);
        if (has_shared) qd_stage_many_f32<QS>(p.h_s, p.I_s, T, p.I_s, p.it_Is_s, hs_s, tid, kDT);
        __syncthreads();
        if (QR == MOE_Q4_K)
            for (int i = 0; i < P; ++i) qd_stage_sums(hs_r + (size_t)i * slots_I_r, hsum_r + i * p.it_I_r * 32, p.it_I_r, tid, kDT);
        if (has_shared && QS == MOE_Q4_K)
            for (int t = 0; t < T; ++t) qd_stage_sums(hs_s + (size_t)t * slots_Is_s, hsum_s + t * p.it_Is_s * 32, p.it_Is_s, tid, kDT);
        __syncthreads();
        const int nrows = (g1 - g0) * 4, nbase = g0 * 4;
        float* ybuf = reinterpret_cast<float*>(dsm + p.off_y);        // [P + T][nrows]
        const int nsrc = nact + (has_shared ? 1 : 0);
        for (int unit = warp; unit < nsrc * (g1 - g0); unit += kDW) {
            const int a = unit / (g1 - g0), g = g0 + (unit - a * (g1 - g0));
            if (a < nact) {
                const int st = s_act_start[a], n = s_act_n[a];
                int vidx[NT], ycol[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) { vidx[t] = st + min(t, n - 1); ycol[t] = st + min(t, n - 1); }
                down_unit<QR, NT>(p.wd + (int64_t)s_act_e[a] * p.stride_d, 4 * g, I, p.it_I_r, hs_r, hsum_r,
                                      vidx, n, lane, ybuf, ycol, nrows, nbase);
            } else {
                int vidx[NT], ycol[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) { vidx[t] = min(t, T - 1); ycol[t] = P + min(t, T - 1); }
                down_unit<QS, NT>(p.sd, 4 * g, p.I_s, p.it_Is_s, hs_s, hsum_s, vidx, T, lane, ybuf, ycol, nrows,
                                      nbase);
            }
        }
        __syncthreads();
        for (int idx = tid; idx < T * nrows; idx += kDT) {
            const int t = idx / nrows, nl = idx - t * nrows;
            float acc = 0.f;
            for (int j = 0; j < k; ++j) acc = fmaf(s_w[t * k + j], ybuf[s_ppos[t * k + j] * nrows + nl], acc);
            if (has_shared) acc += ybuf[(P + t) * nrows + nl];
            float* o = p.out + (int64_t)t * H + nbase + nl;
            if (p.accumulate) acc += *o;
            *o = acc;
        }
    }
    // ------------------------------------------------------------ leave the counters at zero
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&p.sync->done, 1u) == (uint32_t)(G - 1)) {
            p.sync->bar1 = 0u;
            p.sync->bar2 = 0u;
            p.sync->done = 0u;
            __threadfence();
        }
    }
    return;
timeout:
    if (tid == 0) atomicCAS(&p.hdr->status, (int)MOE_OK, (int)MOE_ERR_TIMEOUT);
}

__global__ void init_header_kernel(WsHeader* hdr) {
    hdr->status = MOE_OK;
    hdr->ticket = 0u;
    DecodeSync* sync = reinterpret_cast<DecodeSync*>(reinterpret_cast<char*>(hdr) + kDecodeSyncOffset);
    sync->bar1 = 0u;
    sync->bar2 = 0u;
    sync->done = 0u;
    sync->magic = kDecodeMagic;
}

int g_num_sms = 0;

template <int QR, int QS, int NT>
cudaError_t launch_nt(const DecodeParams& p, size_t smem, cudaStream_t s) {
    cudaError_t err = cudaFuncSetAttribute(decode_layer_kernel<QR, QS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g_num_sms);
    cfg.blockDim = dim3(kDT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_layer_kernel<QR, QS, NT>, p);
}

// NT = the largest number of a token batch's pairs one expert can hold (<= T), rounded up.
template <int QR, int QS>
cudaError_t launch_q(const DecodeParams& p, size_t smem, cudaStream_t s) {
    if (p.T == 1) return launch_nt<QR, QS, 1>(p, smem, s);
    if (p.T == 2) return launch_nt<QR, QS, 2>(p, smem, s);
    return launch_nt<QR, QS, 4>(p, smem, s);
}

struct Layout {
    size_t total;
    int off_xs_r, off_xsum_r, off_xs_s, off_xsum_s, off_hs_r, off_hsum_r, off_hs_s, off_hsum_s, off_topk, off_y;
    int it_H_r, it_I_r, it_H_s, it_Is_s;
};

int iters_for(int q, int K) { return q == MOE_Q4_K ? walk_iters<MOE_Q4_K>(K) : walk_iters<MOE_Q8_0>(K); }

Layout layout(const DecodeArgs& a) {
    Layout L{};
    const int T = a.T, P = a.T * a.route.top_k;
    const bool sh = a.I_s > 0;
    L.it_H_r = iters_for(a.qtype, a.H);
    L.it_I_r = iters_for(a.qtype, a.I);
    L.it_H_s = sh ? iters_for(a.s_qtype, a.H) : 0;
    L.it_Is_s = sh ? iters_for(a.s_qtype, a.I_s) : 0;
    // phase 1 and phase 2 staging share one region
    size_t o1 = 0;
    L.off_xs_r = (int)o1; o1 += (size_t)T * L.it_H_r * 256 * 16;
    L.off_xsum_r = (int)o1; o1 += (size_t)T * L.it_H_r * 32 * 8;
    L.off_xs_s = (int)o1; o1 += (sh && a.s_qtype != a.qtype) ? (size_t)T * L.it_H_s * 256 * 16 : 0;
    L.off_xsum_s = (int)o1; o1 += sh ? (size_t)T * L.it_H_s * 32 * 8 : 0;
    size_t o2 = 0;
    L.off_hs_r = (int)o2; o2 += (size_t)P * L.it_I_r * 256 * 16;
    L.off_hsum_r = (int)o2; o2 += (size_t)P * L.it_I_r * 32 * 8;
    L.off_hs_s = (int)o2; o2 += sh ? (size_t)T * L.it_Is_s * 256 * 16 : 0;
    L.off_hsum_s = (int)o2; o2 += sh ? (size_t)T * L.it_Is_s * 32 * 8 : 0;
    size_t o = align_up(o1 > o2 ? o1 : o2, 16);
    L.off_topk = (int)o; o += (size_t)kDMaxT * 2 * a.route.n_experts * 4;
    L.off_y = (int)o;
    const int sms = g_num_sms > 0 ? g_num_sms : 1;
    const int max_rows = ((a.H / 4 + sms - 1) / sms) * 4;
    o += (size_t)(P + T) * max_rows * 4;
    L.total = align_up(o, 16);
    return L;
}

}  // namespace

cudaError_t launch_init_header(WsHeader* hdr, cudaStream_t s) {
    init_header_kernel<<<1, 1, 0, s>>>(hdr);
    return cudaGetLastError();
}

bool decode_fused_supported(const DecodeArgs& a) {
    if (g_num_sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return false;
        int coop = 0;
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        if (!coop) return false;
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int P = a.T * a.route.top_k;
    if (a.T < 1 || a.T > kDMaxT || P > kDMaxP || a.route.n_experts > kDMaxE) return false;
    if (a.H % 4 || a.I % 2 || (a.I_s > 0 && a.I_s % 2)) return false;
    return layout(a).total <= 200 * 1024;
}

cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s) {
    const Layout L = layout(a);
    DecodeParams p{};
    p.rc.mode = (int)a.route.mode;
    p.rc.E = a.route.n_experts;
    p.rc.k = a.route.top_k;
    p.rc.G = a.route.mode == MOE_ROUTE_SIGMOID_GROUP ? a.route.n_groups : 1;
    p.rc.Gk = a.route.mode == MOE_ROUTE_SIGMOID_GROUP ? a.route.topk_groups : 1;
    p.rc.renorm = a.route.renormalize;
    p.rc.scale = a.route.routed_scale;
    p.Wr = a.Wr; p.bias = a.bias; p.x = a.x; p.x_bf16 = a.x_bf16 ? 1 : 0;
    p.T = a.T; p.H = a.H; p.I = a.I;
    p.qtype = a.qtype; p.wg = a.wg; p.wu = a.wu; p.wd = a.wd; p.stride_gu = a.stride_gu; p.stride_d = a.stride_d;
    p.I_s = a.I_s; p.s_qtype = a.s_qtype; p.sg = a.sg; p.su = a.su; p.sd = a.sd;
    p.logits = a.logits; p.ids = a.ids; p.gw = a.gw; p.sorted = a.sorted; p.offsets = a.offsets;
    p.pair_pos = a.pair_pos; p.h = a.h; p.h_s = a.h_s; p.out = a.out; p.accumulate = a.accumulate ? 1 : 0;
    p.hdr = a.hdr;
    p.sync = reinterpret_cast<DecodeSync*>(reinterpret_cast<char*>(a.hdr) + kDecodeSyncOffset);
    // prefetch the down rows into L2 only while they fit comfortably (half of a 128 MB L2)
    const int64_t down_bytes = (int64_t)a.T * a.route.top_k * a.H * (a.qtype == MOE_Q4_K ? a.I / 256 * 144 : a.I / 32 * 34);
    p.prefetch_down = down_bytes < (64ll << 20) ? 1 : 0;
    p.off_xs_r = L.off_xs_r; p.off_xsum_r = L.off_xsum_r; p.off_xs_s = L.off_xs_s; p.off_xsum_s = L.off_xsum_s;
    p.off_hs_r = L.off_hs_r; p.off_hsum_r = L.off_hsum_r; p.off_hs_s = L.off_hs_s; p.off_hsum_s = L.off_hsum_s;
    p.off_topk = L.off_topk; p.off_y = L.off_y;
    p.it_H_r = L.it_H_r; p.it_I_r = L.it_I_r; p.it_H_s = L.it_H_s; p.it_Is_s = L.it_Is_s;
    const int qs = a.I_s > 0 ? a.s_qtype : a.qtype;
    if (a.qtype == MOE_Q4_K) {
        return qs == MOE_Q4_K ? launch_q<MOE_Q4_K, MOE_Q4_K>(p, L.total, s) : launch_q<MOE_Q4_K, MOE_Q8_0>(p, L.total, s);
    }
    return qs == MOE_Q4_K ? launch_q<MOE_Q8_0, MOE_Q4_K>(p, L.total, s) : launch_q<MOE_Q8_0, MOE_Q8_0>(p, L.total, s);
}

}  // namespace moe
