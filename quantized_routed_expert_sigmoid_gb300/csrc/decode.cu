// decode.cu -- the whole MoE layer at a few tokens in one launch.
//
// The pages run a decode step as one captured CUDA graph ("bloomery README
// 0.3.1", "Why it is fast") with the routed experts on the card.  At T <= 4
// tokens a layer moves ~22 MB (hidden 2048) to ~450 MB (hidden 7168) of expert
// weights, a few microseconds of HBM time, so a chain of small kernels would
// spend more time in launches and ramp-up than in moving bytes.  One
// cooperative persistent grid (one CTA per SM) runs every step instead:
//   phase 0  router logits, the E experts spread over the CTAs; the tokens'
//            activations are staged in shared memory meanwhile  -> barrier 1
//   routing  every CTA selects the top-k of the T tokens itself (identical
//            results) and orders the pairs by expert; CTA 0 publishes them
//   phase 1  gate/up + SwiGLU: each CTA takes a contiguous slice of the chosen
//            experts' (gate, up) row pairs, plus shared-expert rows  -> barrier 2
//   phase 2  each CTA owns a slice of the output rows: the down rows of every
//            chosen expert (and of the shared expert) against the staged h,
//            then the gate-weighted combine in fixed order (+ the residual).
// Weight bytes move by TMA: a producer warp streams the CTA's rows, phase 1's
// then phase 2's, with cp.async.bulk into a ring of shared-memory slots
// (mbarrier completion), so the down rows are already arriving while the grid
// waits at barrier 2.  The eight consumer warps synchronise among themselves
// with a named barrier the producer never joins.  The dot products use the
// same walk and summation order as the separate kernels (qdot.cuh), so the
// results are the same bits.  Every wait is bounded; on timeout the kernel
// records MOE_ERR_TIMEOUT and returns.
#include <algorithm>

#include "internal.cuh"
#include "qdot.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kDW = 8;                     // consumer warps
constexpr int kDT = (kDW + 1) * 32;        // + one producer warp
constexpr int kCons = kDW * 32;
constexpr int kDMaxT = 4;
constexpr int kDMaxP = 64;
constexpr int kDMaxE = 256;
constexpr int kMaxSlots = 16;
constexpr uint64_t kWaitNs = 2000000000ull;

struct DecodeParams {
    RouteCfgDev rc;
    const float* Wr;
    const float* bias;
    const void* x;
    int x_bf16;
    int T, H, I;
    const uint8_t* wg;
    const uint8_t* wu;
    const uint8_t* wd;
    int64_t stride_gu, stride_d;
    int I_s;
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
    // shared-memory layout (bytes from the 1024-aligned base)
    int off_xs_r, off_xsum_r, off_xs_s, off_xsum_s;      // phase 1 staging (x, both walks)
    int off_hs_r, off_hsum_r, off_hs_s, off_hsum_s;      // phase 2 staging (h, h_s), same region
    int off_ring, slot_bytes, n_slots;
    int off_topk, off_y;
    int it_H_r, it_I_r, it_H_s, it_Is_s;
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
__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCons) : "memory"); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(sa(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = dtime();
    while (!mbar_test(b, parity)) {
        if (*abort_flag) return false;
        if (dtime() - t0 > kWaitNs) { *abort_flag = 1; return false; }
    }
    return true;
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     sa(dst)),
                 "l"(src), "r"(bytes), "r"(sa(bar))
                 : "memory");
}

// Requests [src, src + bytes) into L2 without waiting (a hint: no completion, no
// fault on the weight tensors it is given).  src and bytes are 16-byte multiples.
__device__ __forceinline__ void prefetch_l2(const uint8_t* src, int64_t bytes) {
    for (int64_t o = 0; o < bytes; o += 65536) {
        const uint32_t n = (uint32_t)(bytes - o < 65536 ? bytes - o : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + o), "r"(n) : "memory");
    }
}

// The consumers of every CTA meet here.  Returns false on timeout.
__device__ bool grid_barrier(uint32_t* ctr, uint32_t target, volatile int* abort_flag) {
    cons_sync();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        const uint64_t t0 = dtime();
        while (ld_acquire(ctr) < target) {
            if (dtime() - t0 > kWaitNs) { *abort_flag = 1; break; }
        }
        __threadfence();
    }
    cons_sync();
    return *abort_flag == 0;
}

template <int QT>
__device__ __forceinline__ int64_t rbytes(int K) {
    return (int64_t)(K / Walk<QT>::kBlockWeights) * Walk<QT>::kBlockBytes;
}

template <int QR, int QS, int NT>
__global__ void __launch_bounds__(kDT, 1) decode_layer_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ uint8_t dsm_raw[];
    uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ int32_t s_ids[kDMaxP];
    __shared__ float s_w[kDMaxP];
    __shared__ int32_t s_sorted[kDMaxP], s_ppos[kDMaxP];
    __shared__ int s_act_e[kDMaxP], s_act_start[kDMaxP], s_act_n[kDMaxP];
    __shared__ int s_nact;
    __shared__ float s_lpart[kDW][kDMaxT];
    __shared__ __align__(8) uint64_t s_full[kMaxSlots], s_empty[kMaxSlots];
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, c = blockIdx.x;
    const int T = p.T, E = p.rc.E, k = p.rc.k, P = T * k, H = p.H, I = p.I;
    const bool xb = p.x_bf16 != 0;
    const bool has_shared = p.I_s > 0;
    const int NS = p.n_slots;

    if (*reinterpret_cast<volatile uint32_t*>(&p.sync->magic) != kDecodeMagic) {
        if (c == 0 && tid == 0) p.hdr->status = MOE_ERR_WORKSPACE;
        return;
    }
    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < NS; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], 1); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (c == 0) p.hdr->status = MOE_OK;
    }
    __syncthreads();
    volatile int* abort_flag = &s_abort;

    float4* xs_r = reinterpret_cast<float4*>(dsm + p.off_xs_r);
    float2* xsum_r = reinterpret_cast<float2*>(dsm + p.off_xsum_r);
    float4* xs_s = reinterpret_cast<float4*>(dsm + p.off_xs_s);
    float2* xsum_s = reinterpret_cast<float2*>(dsm + p.off_xsum_s);
    const int slots_H_r = p.it_H_r * 256, slots_H_s = p.it_H_s * 256;
    uint8_t* ring = dsm + p.off_ring;
    const int SB = p.slot_bytes;
    const int64_t rbH_r = rbytes<QR>(H), rbI_r = rbytes<QR>(I);
    const int64_t rbH_s = has_shared ? rbytes<QS>(H) : 0, rbIs_s = has_shared ? rbytes<QS>(p.I_s) : 0;

    if (warp < kDW) {
        // ------------------------------------------------------------ phase 0: logits
        for (int e = c; e < E; e += G) {
            float acc[kDMaxT] = {0.f, 0.f, 0.f, 0.f};
            const float* wrow = p.Wr + (int64_t)e * H;
            for (int h = tid * 4; h < H; h += kCons * 4) {
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
            cons_sync();
            if (tid < T) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < kDW; ++w) s += s_lpart[w][tid];
                p.logits[(int64_t)tid * E + e] = s;
            }
            cons_sync();
        }
        // stage x for phase 1 (an input: no dependency on other CTAs)
        if (QR == MOE_Q4_K) {
            qd4_stage(p.x, xb, false, H, T, nullptr, H, reinterpret_cast<uint4*>(xs_r),
                      reinterpret_cast<float4*>(xsum_r), tid, kCons);
        } else {
            for (int t = 0; t < T; ++t) {
                const void* src = xb ? (const void*)(reinterpret_cast<const __nv_bfloat16*>(p.x) + (int64_t)t * H)
                                     : (const void*)(reinterpret_cast<const float*>(p.x) + (int64_t)t * H);
                qd_stage<QR>(src, xb, false, H, p.it_H_r, xs_r + (size_t)t * slots_H_r, tid, kCons);
            }
        }
        if (has_shared && QS != QR) {
            if (QS == MOE_Q4_K) {
                qd4_stage(p.x, xb, false, H, T, nullptr, H, reinterpret_cast<uint4*>(xs_s),
                          reinterpret_cast<float4*>(xsum_s), tid, kCons);
            } else {
                for (int t = 0; t < T; ++t) {
                    const void* src = xb ? (const void*)(reinterpret_cast<const __nv_bfloat16*>(p.x) + (int64_t)t * H)
                                         : (const void*)(reinterpret_cast<const float*>(p.x) + (int64_t)t * H);
                    qd_stage<QS>(src, xb, false, H, p.it_H_s, xs_s + (size_t)t * slots_H_s, tid, kCons);
                }
            }
        }
        if (grid_barrier(&p.sync->bar1, (uint32_t)G, abort_flag)) {
            // -------------------------------------------------------- routing (every CTA)
            if (warp < T) {
                float* sel = reinterpret_cast<float*>(dsm + p.off_topk) + warp * 2 * E;
                warp_topk(p.rc, p.logits + (int64_t)warp * E, p.bias, sel, sel + E, s_ids + warp * k, s_w + warp * k);
            }
            cons_sync();
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
                // chosen experts: the first position of every run of equal ids
                const int i0 = lane, i1 = lane + 32;
                const bool f0 = i0 < P && (i0 == 0 || s_ids[s_sorted[i0]] != s_ids[s_sorted[i0 - 1]]);
                const bool f1 = i1 < P && (s_ids[s_sorted[i1]] != s_ids[s_sorted[i1 - 1]]);
                const unsigned first_lo = __ballot_sync(0xffffffffu, f0);
                const unsigned first_hi = __ballot_sync(0xffffffffu, f1);
                const int nact = __popc(first_lo) + __popc(first_hi);
                const unsigned below = (1u << lane) - 1u;
                if (f0) {
                    const int a = __popc(first_lo & below);
                    s_act_e[a] = s_ids[s_sorted[i0]];
                    s_act_start[a] = i0;
                }
                if (f1) {
                    const int a = __popc(first_lo) + __popc(first_hi & below);
                    s_act_e[a] = s_ids[s_sorted[i1]];
                    s_act_start[a] = i1;
                }
                __syncwarp();
                for (int a = lane; a < nact; a += 32)
                    s_act_n[a] = (a + 1 < nact ? s_act_start[a + 1] : P) - s_act_start[a];
                if (lane == 0) s_nact = nact;
            }
        }
    }
    __syncthreads();                                   // routing (or an abort) known to all threads
    if (!*abort_flag) {
        const int nact = s_nact;
        const int half_r = I / 2, half_s = has_shared ? p.I_s / 2 : 0;
        const int Q = nact * half_r + half_s;          // phase-1 row pairs of the whole grid
        const int q0 = (int)((int64_t)c * Q / G);
        const int n1 = (int)((int64_t)(c + 1) * Q / G) - q0;
        const int ngroups = H / 4;
        const int g0 = (int)((int64_t)c * ngroups / G), g1 = (int)((int64_t)(c + 1) * ngroups / G);
        const int ng = g1 - g0;
        const int nsrc = nact + (has_shared ? 1 : 0);
        const int n_units = n1 + nsrc * ng;

        if (warp == kDW) {
            // ======================================================== producer
            if (lane == 0) {
                // The ring holds NS units; the rest of the CTA's slice is requested into L2
                // now, so every weight byte of the layer is in flight at once and the ring's
                // later copies are L2 hits.  Consecutive units of one expert are contiguous
                // rows: one prefetch per run and matrix (pieces of at most 64 KB).
                for (int u = NS; u < n1;) {
                    const int q = q0 + u;
                    const uint8_t *gp, *upp;
                    int64_t rb;
                    int qend, r0;
                    if (q < nact * half_r) {
                        const int a = q / half_r;
                        qend = min(q0 + n1, (a + 1) * half_r);
                        r0 = 2 * (q - a * half_r);
                        gp = p.wg + (int64_t)s_act_e[a] * p.stride_gu;
                        upp = p.wu + (int64_t)s_act_e[a] * p.stride_gu;
                        rb = rbH_r;
                    } else {
                        qend = q0 + n1;
                        r0 = 2 * (q - nact * half_r);
                        gp = p.sg;
                        upp = p.su;
                        rb = rbH_s;
                    }
                    const int64_t nb = 2 * (int64_t)(qend - q) * rb;
                    prefetch_l2(gp + r0 * rb, nb);
                    prefetch_l2(upp + r0 * rb, nb);
                    u = qend - q0;
                }
                for (int u = max(NS, n1); u < n_units;) {
                    const int v = u - n1, a = v / ng, gi = v - a * ng;
                    const uint8_t* d;
                    int64_t rb;
                    if (a < nact) { d = p.wd + (int64_t)s_act_e[a] * p.stride_d; rb = rbI_r; }
                    else { d = p.sd; rb = rbIs_s; }
                    prefetch_l2(d + (int64_t)4 * (g0 + gi) * rb, (int64_t)4 * (ng - gi) * rb);
                    u = n1 + (a + 1) * ng;
                }
                int issued = 0;
                for (int u = 0; u < n_units; ++u) {
                    const int slot = u % NS;
                    if (u >= NS && !mbar_wait(&s_empty[slot], ((u / NS) - 1) & 1, abort_flag)) break;
                    issued = u + 1;
                    uint8_t* dst = ring + (size_t)slot * SB;
                    if (u < n1) {
                        const int q = q0 + u;
                        const uint8_t *gp, *upp;
                        int64_t rb;
                        int r0;
                        if (q < nact * half_r) {
                            const int a = q / half_r;
                            r0 = 2 * (q - a * half_r);
                            gp = p.wg + (int64_t)s_act_e[a] * p.stride_gu;
                            upp = p.wu + (int64_t)s_act_e[a] * p.stride_gu;
                            rb = rbH_r;
                        } else {
                            r0 = 2 * (q - nact * half_r);
                            gp = p.sg;
                            upp = p.su;
                            rb = rbH_s;
                        }
                        mbar_expect(&s_full[slot], (uint32_t)(4 * rb));
                        bulk_copy(dst, gp + r0 * rb, (uint32_t)(2 * rb), &s_full[slot]);
                        bulk_copy(dst + 2 * rb, upp + r0 * rb, (uint32_t)(2 * rb), &s_full[slot]);
                    } else {
                        const int v = u - n1, a = v / ng, g = g0 + (v - a * ng);
                        const uint8_t* d;
                        int64_t rb;
                        if (a < nact) { d = p.wd + (int64_t)s_act_e[a] * p.stride_d; rb = rbI_r; }
                        else { d = p.sd; rb = rbIs_s; }
                        mbar_expect(&s_full[slot], (uint32_t)(4 * rb));
                        bulk_copy(dst, d + (int64_t)4 * g * rb, (uint32_t)(4 * rb), &s_full[slot]);
                    }
                }
                // no copy may still be landing when the CTA exits (consumers waited for all of them
                // unless a timeout cut the run short): wait, bounded, for the last NS issued
                for (int u = issued > NS ? issued - NS : 0; u < issued; ++u) {
                    const uint64_t t0 = dtime();
                    while (!mbar_test(&s_full[u % NS], (u / NS) & 1) && dtime() - t0 < kWaitNs) {
                    }
                }
            }
            __syncwarp();
        } else {
            // ======================================================== consumers
            bool ok = true;
            // ---- phase 1: unit u of this CTA is consumed by warp u % kDW
            for (int u = warp; u < n1; u += kDW) {
                const int slot = u % NS;
                if (!mbar_wait(&s_full[slot], (u / NS) & 1, abort_flag)) { ok = false; break; }
                const uint8_t* base = ring + (size_t)slot * SB;
                const int q = q0 + u;
                float acc[4][NT];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
                int vidx[NT];
                if (q < nact * half_r) {
                    const int a = q / half_r, r0 = 2 * (q - a * half_r);
                    const int st = s_act_start[a], n = s_act_n[a];
                    const uint8_t* rowp[4] = {base, base + rbH_r, base + 2 * rbH_r, base + 3 * rbH_r};
#pragma unroll
                    for (int t = 0; t < NT; ++t) vidx[t] = s_sorted[st + min(t, n - 1)] / k;
                    if (QR == MOE_Q4_K)
                        qd4_rows4<NT, true>(rowp, H / kQ4KWeights, reinterpret_cast<const uint4*>(xs_r),
                                            reinterpret_cast<const float4*>(xsum_r), n, lane, acc, vidx);
                    else
                        qd_rows4<QR, NT, true>(rowp, H / Walk<QR>::kBlockWeights, p.it_H_r, xs_r, slots_H_r, xsum_r,
                                               p.it_H_r * 32, n, lane, acc, vidx);
                    qd_warp_reduce<NT>(acc);
                    if (lane < 2 * NT) {
                        const int t = lane >> 1, ri = lane & 1;
                        if (t < n) {
                            const float gv = qd_pick<NT>(acc, ri, t), uv = qd_pick<NT>(acc, 2 + ri, t);
                            p.h[(int64_t)(st + t) * I + r0 + ri] = gv / (1.0f + expf(-gv)) * uv;
                        }
                    }
                } else {
                    const int r0 = 2 * (q - nact * half_r);
                    const uint8_t* rowp[4] = {base, base + rbH_s, base + 2 * rbH_s, base + 3 * rbH_s};
#pragma unroll
                    for (int t = 0; t < NT; ++t) vidx[t] = min(t, T - 1);
                    const float4* xsrc = QS == QR ? xs_r : xs_s;
                    const float2* xssrc = QS == QR ? xsum_r : xsum_s;
                    if (QS == MOE_Q4_K)
                        qd4_rows4<NT, true>(rowp, H / kQ4KWeights, reinterpret_cast<const uint4*>(xsrc),
                                            reinterpret_cast<const float4*>(xssrc), T, lane, acc, vidx);
                    else
                        qd_rows4<QS, NT, true>(rowp, H / Walk<QS>::kBlockWeights, p.it_H_s, xsrc, slots_H_s, xssrc,
                                               p.it_H_s * 32, T, lane, acc, vidx);
                    qd_warp_reduce<NT>(acc);
                    if (lane < 2 * NT) {
                        const int t = lane >> 1, ri = lane & 1;
                        if (t < T) {
                            const float gv = qd_pick<NT>(acc, ri, t), uv = qd_pick<NT>(acc, 2 + ri, t);
                            p.h_s[(int64_t)t * p.I_s + r0 + ri] = gv / (1.0f + expf(-gv)) * uv;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[slot]);
            }
            // ---- barrier 2: every h written
            if (!grid_barrier(&p.sync->bar2, (uint32_t)G, abort_flag)) ok = false;
            float* ybuf = reinterpret_cast<float*>(dsm + p.off_y);          // [P + T][nrows]
            const int nrows = ng * 4, nbase = g0 * 4;
            if (ok) {
                float4* hs_r = reinterpret_cast<float4*>(dsm + p.off_hs_r);
                float2* hsum_r = reinterpret_cast<float2*>(dsm + p.off_hsum_r);
                float4* hs_s = reinterpret_cast<float4*>(dsm + p.off_hs_s);
                float2* hsum_s = reinterpret_cast<float2*>(dsm + p.off_hsum_s);
                const int slots_I_r = p.it_I_r * 256, slots_Is_s = p.it_Is_s * 256;
                if (QR == MOE_Q4_K)
                    qd4_stage(p.h, false, true, I, P, nullptr, I, reinterpret_cast<uint4*>(hs_r),
                              reinterpret_cast<float4*>(hsum_r), tid, kCons);
                else
                    qd_stage_many_f32<QR>(p.h, I, P, I, p.it_I_r, hs_r, tid, kCons);
                if (has_shared) {
                    if (QS == MOE_Q4_K)
                        qd4_stage(p.h_s, false, true, p.I_s, T, nullptr, p.I_s, reinterpret_cast<uint4*>(hs_s),
                                  reinterpret_cast<float4*>(hsum_s), tid, kCons);
                    else
                        qd_stage_many_f32<QS>(p.h_s, p.I_s, T, p.I_s, p.it_Is_s, hs_s, tid, kCons);
                }
                cons_sync();
                // ---- phase 2: unit u (>= n1) is consumed by warp u % kDW as well
                const int ustart = n1 + ((warp - n1 % kDW) + kDW) % kDW;
                for (int u = ustart; u < n_units; u += kDW) {
                    const int slot = u % NS;
                    if (!mbar_wait(&s_full[slot], (u / NS) & 1, abort_flag)) { ok = false; break; }
                    const uint8_t* base = ring + (size_t)slot * SB;
                    const int v = u - n1, a = v / ng, g = g0 + (v - a * ng);
                    float acc[4][NT];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
                    int vidx[NT], ycol[NT], nt;
                    if (a < nact) {
                        const int st = s_act_start[a];
                        nt = s_act_n[a];
#pragma unroll
                        for (int t = 0; t < NT; ++t) { vidx[t] = st + min(t, nt - 1); ycol[t] = vidx[t]; }
                        const uint8_t* rowp[4] = {base, base + rbI_r, base + 2 * rbI_r, base + 3 * rbI_r};
                        if (QR == MOE_Q4_K)
                            qd4_rows4<NT, true>(rowp, I / kQ4KWeights, reinterpret_cast<const uint4*>(hs_r),
                                                reinterpret_cast<const float4*>(hsum_r), nt, lane, acc, vidx);
                        else
                            qd_rows4<QR, NT, true>(rowp, I / Walk<QR>::kBlockWeights, p.it_I_r, hs_r, slots_I_r,
                                                   hsum_r, p.it_I_r * 32, nt, lane, acc, vidx);
                    } else {
                        nt = T;
#pragma unroll
                        for (int t = 0; t < NT; ++t) { vidx[t] = min(t, T - 1); ycol[t] = P + vidx[t]; }
                        const uint8_t* rowp[4] = {base, base + rbIs_s, base + 2 * rbIs_s, base + 3 * rbIs_s};
                        if (QS == MOE_Q4_K)
                            qd4_rows4<NT, true>(rowp, p.I_s / kQ4KWeights, reinterpret_cast<const uint4*>(hs_s),
                                                reinterpret_cast<const float4*>(hsum_s), nt, lane, acc, vidx);
                        else
                            qd_rows4<QS, NT, true>(rowp, p.I_s / Walk<QS>::kBlockWeights, p.it_Is_s, hs_s, slots_Is_s,
                                                   hsum_s, p.it_Is_s * 32, nt, lane, acc, vidx);
                    }
                    qd_warp_reduce<NT>(acc);
                    if (lane < 4 * NT) {
                        const int t = lane >> 2, ri = lane & 3;
                        if (t < nt) {
                            int col = 0;
#pragma unroll
                            for (int tt = 0; tt < NT; ++tt)
                                if (tt == t) col = ycol[tt];
                            ybuf[col * nrows + (4 * g + ri - nbase)] = qd_pick<NT>(acc, ri, t);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_empty[slot]);
                }
            }
            cons_sync();
            if (ok && !*abort_flag) {
                for (int idx = tid; idx < T * nrows; idx += kCons) {
                    const int t = idx / nrows, nl = idx - t * nrows;
                    float acc = 0.f;
                    for (int j = 0; j < k; ++j) acc = fmaf(s_w[t * k + j], ybuf[s_ppos[t * k + j] * nrows + nl], acc);
                    if (has_shared) acc += ybuf[(P + t) * nrows + nl];
                    float* o = p.out + (int64_t)t * H + nbase + nl;
                    if (p.accumulate) acc += *o;
                    *o = acc;
                }
                if (c == 0) {                  // publish the routing (debug views)
                    for (int i = tid; i < P; i += kCons) {
                        p.ids[i] = s_ids[i];
                        p.gw[i] = s_w[i];
                        p.sorted[i] = s_sorted[i];
                        p.pair_pos[i] = s_ppos[i];
                    }
                    for (int e = tid; e <= E; e += kCons) {
                        int cnt = 0;
                        for (int i = 0; i < P; ++i) cnt += s_ids[i] < e ? 1 : 0;
                        p.offsets[e] = cnt;
                    }
                }
            }
        }
    }
    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) atomicCAS(&p.hdr->status, (int)MOE_OK, (int)MOE_ERR_TIMEOUT);
        return;
    }
    if (tid == 0) {                             // leave the counters at zero for the next launch
        __threadfence();
        if (atomicAdd(&p.sync->done, 1u) == (uint32_t)(G - 1)) {
            p.sync->bar1 = 0u;
            p.sync->bar2 = 0u;
            p.sync->done = 0u;
            __threadfence();
        }
    }
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
    cudaError_t err = cudaFuncSetAttribute(decode_layer_kernel<QR, QS, NT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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

template <int QR, int QS>
cudaError_t launch_q(const DecodeParams& p, size_t smem, cudaStream_t s) {
    if (p.T == 1) return launch_nt<QR, QS, 1>(p, smem, s);
    if (p.T == 2) return launch_nt<QR, QS, 2>(p, smem, s);
    return launch_nt<QR, QS, 4>(p, smem, s);
}

struct Layout {
    size_t total;
    int off_xs_r, off_xsum_r, off_xs_s, off_xsum_s, off_hs_r, off_hsum_r, off_hs_s, off_hsum_s;
    int off_ring, slot_bytes, n_slots, off_topk, off_y;
    int it_H_r, it_I_r, it_H_s, it_Is_s;
};

int iters_for(int q, int K) { return q == MOE_Q4_K ? walk_iters<MOE_Q4_K>(K) : walk_iters<MOE_Q8_0>(K); }
int64_t rbytes_host(int q, int K) { return q == MOE_Q4_K ? (int64_t)K / 256 * 144 : (int64_t)K / 32 * 34; }

Layout layout(const DecodeArgs& a, int n_slots) {
    Layout L{};
    const int T = a.T, P = a.T * a.route.top_k;
    const bool sh = a.I_s > 0;
    L.it_H_r = iters_for(a.qtype, a.H);
    L.it_I_r = iters_for(a.qtype, a.I);
    L.it_H_s = sh ? iters_for(a.s_qtype, a.H) : 0;
    L.it_Is_s = sh ? iters_for(a.s_qtype, a.I_s) : 0;
    // staged vectors: Q4_K as 24-bit integer planes (X: 16 uint4 per 64 values, XS: 1 float4 per 64),
    // Q8_0 as fp32 in walk order (xs) with per-lane half sums (xsum)
    auto xs_bytes = [](int q, int K, int it) { return q == MOE_Q4_K ? (size_t)qd4_groups(K) * 256 : (size_t)it * 4096; };
    auto xsum_bytes = [](int q, int K, int it) { return q == MOE_Q4_K ? (size_t)qd4_groups(K) * 16 : (size_t)it * 256; };
    size_t o1 = 0;                     // phase 1 staging
    L.off_xs_r = (int)o1; o1 += (size_t)T * xs_bytes(a.qtype, a.H, L.it_H_r);
    L.off_xsum_r = (int)o1; o1 += (size_t)T * xsum_bytes(a.qtype, a.H, L.it_H_r);
    L.off_xs_s = (int)o1; o1 += (sh && a.s_qtype != a.qtype) ? (size_t)T * xs_bytes(a.s_qtype, a.H, L.it_H_s) : 0;
    L.off_xsum_s = (int)o1; o1 += (sh && a.s_qtype != a.qtype) ? (size_t)T * xsum_bytes(a.s_qtype, a.H, L.it_H_s) : 0;
    size_t o2 = 0;                     // phase 2 staging (same region)
    L.off_hs_r = (int)o2; o2 += (size_t)P * xs_bytes(a.qtype, a.I, L.it_I_r);
    L.off_hsum_r = (int)o2; o2 += (size_t)P * xsum_bytes(a.qtype, a.I, L.it_I_r);
    L.off_hs_s = (int)o2; o2 += sh ? (size_t)T * xs_bytes(a.s_qtype, a.I_s, L.it_Is_s) : 0;
    L.off_hsum_s = (int)o2; o2 += sh ? (size_t)T * xsum_bytes(a.s_qtype, a.I_s, L.it_Is_s) : 0;
    size_t o = align_up(o1 > o2 ? o1 : o2, 1024);
    int64_t sb = std::max<int64_t>(4 * rbytes_host(a.qtype, a.H), 4 * rbytes_host(a.qtype, a.I));
    if (sh) sb = std::max<int64_t>(sb, std::max(4 * rbytes_host(a.s_qtype, a.H), 4 * rbytes_host(a.s_qtype, a.I_s)));
    L.slot_bytes = (int)align_up((size_t)sb, 128);
    L.n_slots = n_slots;
    L.off_ring = (int)o; o += (size_t)L.slot_bytes * n_slots;
    L.off_topk = (int)o; o += (size_t)kDMaxT * 2 * a.route.n_experts * 4;
    L.off_y = (int)o;
    const int sms = g_num_sms > 0 ? g_num_sms : 1;
    const int max_rows = ((a.H / 4 + sms - 1) / sms) * 4;
    o += (size_t)(P + T) * max_rows * 4;
    L.total = align_up(o, 16) + 1024;  // + alignment slack of the dynamic base
    return L;
}

constexpr size_t kSmemCap = 220 * 1024;   // dynamic; the kernel's static shared memory is ~2.5 KB

Layout best_layout(const DecodeArgs& a) {
    Layout L = layout(a, kMaxSlots);
    for (int ns = kMaxSlots / 2; ns >= 2 && L.total > kSmemCap; ns /= 2) L = layout(a, ns);
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
    // bulk copies move 2 rows (gate/up) or 4 rows (down): 16-byte multiples at 16-byte offsets
    if ((2 * rbytes_host(a.qtype, a.H)) % 16 || (4 * rbytes_host(a.qtype, a.I)) % 16) return false;
    if (a.I_s > 0 && ((2 * rbytes_host(a.s_qtype, a.H)) % 16 || (4 * rbytes_host(a.s_qtype, a.I_s)) % 16))
        return false;
    if ((a.stride_gu % 16) || (a.stride_d % 16)) return false;
    return best_layout(a).total <= kSmemCap;
}

cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s) {
    const Layout L = best_layout(a);
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
    p.wg = a.wg; p.wu = a.wu; p.wd = a.wd; p.stride_gu = a.stride_gu; p.stride_d = a.stride_d;
    p.I_s = a.I_s; p.sg = a.sg; p.su = a.su; p.sd = a.sd;
    p.logits = a.logits; p.ids = a.ids; p.gw = a.gw; p.sorted = a.sorted; p.offsets = a.offsets;
    p.pair_pos = a.pair_pos; p.h = a.h; p.h_s = a.h_s; p.out = a.out; p.accumulate = a.accumulate ? 1 : 0;
    p.hdr = a.hdr;
    p.sync = reinterpret_cast<DecodeSync*>(reinterpret_cast<char*>(a.hdr) + kDecodeSyncOffset);
    p.off_xs_r = L.off_xs_r; p.off_xsum_r = L.off_xsum_r; p.off_xs_s = L.off_xs_s; p.off_xsum_s = L.off_xsum_s;
    p.off_hs_r = L.off_hs_r; p.off_hsum_r = L.off_hsum_r; p.off_hs_s = L.off_hs_s; p.off_hsum_s = L.off_hsum_s;
    p.off_ring = L.off_ring; p.slot_bytes = L.slot_bytes; p.n_slots = L.n_slots;
    p.off_topk = L.off_topk; p.off_y = L.off_y;
    p.it_H_r = L.it_H_r; p.it_I_r = L.it_I_r; p.it_H_s = L.it_H_s; p.it_Is_s = L.it_Is_s;
    const int qs = a.I_s > 0 ? a.s_qtype : a.qtype;
    if (a.qtype == MOE_Q4_K)
        return qs == MOE_Q4_K ? launch_q<MOE_Q4_K, MOE_Q4_K>(p, L.total, s) : launch_q<MOE_Q4_K, MOE_Q8_0>(p, L.total, s);
    return qs == MOE_Q4_K ? launch_q<MOE_Q8_0, MOE_Q4_K>(p, L.total, s) : launch_q<MOE_Q8_0, MOE_Q8_0>(p, L.total, s);
}

}  // namespace moe
