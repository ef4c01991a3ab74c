// decode_chain.cu -- the MoE layer at T <= 8 tokens as three chained launches (as many as
// the gate/up kernel's staged x and its 16 warps' rings fit: T <= 6 at hidden 2048).
//
// The pages run a decode step as one captured CUDA graph with the routed
// experts on the card ("bloomery README 0.3.1", "Why it is fast").  At a few
// tokens a layer reads ~22 MB (hidden 2048) to ~450 MB (hidden 7168) of expert
// weights; what costs time is the chain of dependent steps (router logits ->
// the chosen experts' gate/up -> their down rows), each of which must see the
// previous one complete.  The three kernels are launched with programmatic
// dependent launch: a kernel starts while the one before it still runs, does
// what does not depend on it (router rows into registers, the activations
// staged), then waits (griddepcontrol.wait) for it to complete.
//
//   K1 logits   one CTA per expert row: the T router logits of that expert.
//   K2 gate/up  every CTA selects the top-k of the T tokens itself (identical
//               results everywhere; CTA 0 publishes them), then a persistent
//               grid runs (active expert, row pair) units in rounds of 16 per
//               CTA: a round's 32 gate rows and 32 up rows of one expert arrive
//               as two bulk copies into a two-slot ring in shared memory (one
//               mbarrier per slot), each warp computes h = silu(gate . x) *
//               (up . x) of one row pair, and the CTA stages the round's 32
//               values of h (one sub-block) for K3; the shared expert's rows
//               follow.  Each CTA also requests its share of the chosen down
//               rows into L2.
//   K3 down     one CTA per block of output rows: its down rows of every pair
//               go to shared memory (one bulk copy per pair) while h is
//               staged, then the dot products and the gate-weighted combine in
//               fixed order (+ shared, + residual).
// Dot products use the integer Q4_K walk of qdot.cuh; every reduction has a
// fixed order, so a replay gives the same bits.
#include <algorithm>
#include <type_traits>

#include "internal.cuh"
#include "qdot.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kCMaxT = 8;
constexpr int kCMaxP = 64;
constexpr int kCMaxE = 256;
constexpr int kK1Threads = 128;
constexpr int kK3Threads = 256;
constexpr int kK1MaxVec = 4;               // float4 of a router row per K1 thread: H <= 2048
constexpr int kChunkBlocks = 8;            // ring item: 8 Q4_K blocks (32 groups) of 4 rows
constexpr int kSlotBytes = 4 * kChunkBlocks * kQ4KBytes;
constexpr int kStampCtas = 256, kStampPhases = 8;   // the timing hook's buffer: [3][256][8] uint64
constexpr int kK2MaxWarps = 16;

struct ChainParams {
    RouteCfgDev rc;
    const float* Wr;
    const float* bias;
    const void* x;
    int x_bf16;
    const float* gamma;                     // pre-norm: x is the fp32 residual stream, the layer input
    float eps;                              // is bf16(RMSNorm(x) * gamma) (K1 and K2 compute it)
    int T, H, I;
    const uint8_t* wg;
    const uint8_t* wu;
    const uint8_t* wd;
    int64_t stride_gu, stride_d;
    int I_s, s_q8;                          // shared expert: intermediate, 1 if Q8_0 (else Q4_K)
    int s_q80r;                             // its Q8_0 rows in the repacked layout
    const uint8_t* sg;
    const uint8_t* su;
    const uint8_t* sd;
    float* logits;
    int32_t* ids;
    float* gw;
    int32_t* sorted;
    int32_t* offsets;
    int32_t* pair_pos;
    uint8_t* hq;                            // [P][272 * I/64]: h of each pair (sorted position) as staged planes
    uint8_t* hq_s;                          // [T][272 * I_s/64]: the shared expert's h (Q4_K shared expert)
    float* h_s;                             // [T][I_s] fp32: the shared expert's h (Q8_0 shared expert)
    float* out;
    int accumulate;
    unsigned long long* counts;             // nullable [E]: the running routing histogram
    WsHeader* hdr;
    int it_H_s, it_Is_s;                    // Q8_0 walk iterations of the shared expert
    int k2_warps;                           // K2 warps per CTA (<= kK2MaxWarps)
    int k2_off_xs_s, k2_off_ring;           // K2 dynamic shared-memory offsets (bytes)
    int rows_per_cta;                       // K3 output rows per CTA (multiple of 8)
    int k3_prefetch;                        // K3 copies its down rows to shared memory
    int k3_off_hs_s, k3_off_y, k3_off_w;    // K3 dynamic shared-memory offsets (bytes)
    uint64_t wait_ns;                       // limit of every bounded wait
    int stall;                              // test setting: K2's first wait never completes
    uint64_t* stamps;                       // timing hook (NULL: off): [kernel][CTA][phase] globaltimer
};

// The routing every K2 CTA derives from the logits (shared memory); the top-k scratch is
// sized for the kernel's NT tokens.
template <int NT>
struct CtaRoute {
    int32_t ids[kCMaxP], sorted[kCMaxP], ppos[kCMaxP], tok[kCMaxP];
    float w[kCMaxP];
    int act_e[kCMaxP], act_start[kCMaxP], act_n[kCMaxP];
    int nact;
    float sel[NT][2 * kCMaxE];
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const uint8_t* src, int64_t bytes) {
    for (int64_t o = 0; o < bytes; o += 65536) {
        const uint32_t n = (uint32_t)(bytes - o < 65536 ? bytes - o : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + o), "r"(n) : "memory");
    }
}
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }
// One warp stages the 32 consecutive values v (lane = element) of sub-block sb of a vector
// of G groups into dst as three byte planes: the layout qd4_stage_par gives a staged vector
// with NPL = 3 (X: 16 x G uint4 of planes {hi, mid, lo, 0} of 4 values, then XS: G float4
// {scale lo, scale hi, sum lo, sum hi}).
__device__ __forceinline__ void warp_stage_subblock(float v, uint8_t* dst, int G, int sb, int lane) {
    float m = fabsf(v), sum = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    }
    const float2 sc = qx_scale<3>(m);
    const int x = qx_int<3>(v, sc.x);
    uint32_t w[3];
#pragma unroll
    for (int pl = 0; pl < 3; ++pl) {
        w[pl] = qx_plane<3>(x, pl);
#pragma unroll
        for (int b = 1; b < 4; ++b) w[pl] |= __shfl_down_sync(0xffffffffu, qx_plane<3>(x, pl), b) << (8 * b);
    }
    const int g = sb >> 1, hh = sb & 1;
    if ((lane & 3) == 0) reinterpret_cast<uint4*>(dst)[(hh * 8 + (lane >> 2)) * G + g] = make_uint4(w[0], w[1], w[2], 0u);
    if (lane == 0) {
        float* xs = reinterpret_cast<float*>(dst + (size_t)16 * G * 16) + 4 * g;
        xs[hh] = sc.y;
        xs[2 + hh] = sum;
    }
}
__device__ __forceinline__ float4 ld_nc_v4(const float4* q) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(q));
    return v;
}
__device__ __forceinline__ uint32_t smem_u32(const void* q) { return (uint32_t)__cvta_generic_to_shared(q); }
__device__ __forceinline__ uint64_t gtime() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Timing hook: thread 0 of CTA c records the global time of phase ph of kernel kn.
__device__ __forceinline__ void stamp(const ChainParams& p, int kn, int ph) {
    if (p.stamps && threadIdx.x == 0 && blockIdx.x < kStampCtas)
        p.stamps[((size_t)kn * kStampCtas + blockIdx.x) * kStampPhases + ph] = gtime();
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    // the suspend-time hint lets the warp sleep until the phase completes (or ~0.1 ms pass)
    asm volatile("{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2, %3;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(ok)
                 : "r"(smem_u32(b)), "r"(parity), "r"(100000u)
                 : "memory");
    return ok != 0;
}
// Waits for the phase of parity `parity` to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, uint64_t limit_ns) {
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = gtime();
    while (!mbar_test(b, parity))
        if (gtime() - t0 > limit_ns) return false;
    return true;
}
// A bulk copy global -> shared whose bytes complete the transaction count of bar.
__device__ __forceinline__ void bulk_to_smem(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Every thread of the CTA calls this.  Warp t < T selects token t's experts from the
// logits (read through L2: another grid wrote them); warp 0 then orders the pairs by
// expert (stable) and lists the active experts with their runs of sorted positions.
template <int NT>
__device__ void cta_route(const ChainParams& p, CtaRoute<NT>& R) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int E = p.rc.E, k = p.rc.k, P = p.T * k;
    if (warp < p.T)
        warp_topk(p.rc, p.logits + (int64_t)warp * E, p.bias, R.sel[warp], R.sel[warp] + E, R.ids + warp * k,
                  R.w + warp * k);
    __syncthreads();
    stamp(p, 1, 7);
    if (warp == 0) {
        for (int i = lane; i < P; i += 32) {
            const int ei = R.ids[i];
            int rank = 0;
            for (int j = 0; j < P; ++j) {
                const int ej = R.ids[j];
                rank += (ej < ei || (ej == ei && j < i)) ? 1 : 0;
            }
            R.sorted[rank] = i;
            R.ppos[i] = rank;
        }
        __syncwarp();
        const int i0 = lane, i1 = lane + 32;
        const bool f0 = i0 < P && (i0 == 0 || R.ids[R.sorted[i0]] != R.ids[R.sorted[i0 - 1]]);
        const bool f1 = i1 < P && (R.ids[R.sorted[i1]] != R.ids[R.sorted[i1 - 1]]);
        const unsigned lo = __ballot_sync(0xffffffffu, f0), hi = __ballot_sync(0xffffffffu, f1);
        const unsigned below = (1u << lane) - 1u;
        // the next run's start after position q (or P)
        const unsigned long long runs = ((unsigned long long)hi << 32) | lo;
        auto next_start = [&](int q) {
            const unsigned long long rest = q >= 63 ? 0ull : (runs >> (q + 1)) << (q + 1);
            return rest ? __ffsll((long long)rest) - 1 : P;
        };
        if (f0) {
            const int a = __popc(lo & below);
            R.act_e[a] = R.ids[R.sorted[i0]];
            R.act_start[a] = i0;
            R.act_n[a] = next_start(i0) - i0;
        }
        if (f1) {
            const int a = __popc(lo) + __popc(hi & below);
            R.act_e[a] = R.ids[R.sorted[i1]];
            R.act_start[a] = i1;
            R.act_n[a] = next_start(i1) - i1;
        }
        for (int i = lane; i < P; i += 32) R.tok[i] = R.sorted[i] / k;
        if (lane == 0) R.nact = __popc(lo) + __popc(hi);
    }
    __syncthreads();
}

// ============================================================================ K1: router logits
// The loops run over exactly NT tokens and H/512 <= kK1MaxVec float4 per thread: the kernel
// runs once per layer on every SM, mostly waiting, so short straight code matters.
template <int NT>
__global__ void __launch_bounds__(kK1Threads) chain_logits_kernel(const __grid_constant__ ChainParams p) {
    __shared__ float s_part[kK1Threads / 32][kCMaxT];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e = blockIdx.x, E = p.rc.E, T = p.T, H = p.H;
    const int n4 = H / 4;
    // the router row: a weight, independent of the launches before this one
    // (volatile loads: issued here, ahead of the wait, not moved past it)
    float4 w[kK1MaxVec], gm[kK1MaxVec];
#pragma unroll
    for (int i = 0; i < kK1MaxVec; ++i) {
        const int j = tid + i * kK1Threads;
        w[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        gm[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < n4) w[i] = ld_nc_v4(reinterpret_cast<const float4*>(p.Wr + (int64_t)e * H) + j);
        if (p.gamma && j < n4) gm[i] = ld_nc_v4(reinterpret_cast<const float4*>(p.gamma) + j);
    }
    stamp(p, 0, 0);
    pdl_wait();                                   // x and the workspace belong to the launches before
    pdl_launch_dependents();
    stamp(p, 0, 1);
    if (e == 0 && tid == 0) {
        p.hdr->status = MOE_OK;
        p.hdr->route_ready = 0u;
    }
    const bool xb = p.x_bf16 != 0;
    // pre-norm: the tokens' RMSNorm scales, by all warps
    __shared__ float s_r[kCMaxT], s_rpart[kCMaxT][8];
    if (p.gamma) rms_scales_cta(reinterpret_cast<const float*>(p.x), T, H, p.eps, s_rpart, s_r);
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll
    for (int i = 0; i < kK1MaxVec; ++i) {
        const int j = tid + i * kK1Threads;
        if (j < n4) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (t < T) {
                    float4 xv = qd_load_vec4(p.x, xb, (int64_t)t * H + 4 * j);
                    if (p.gamma) xv = rms_apply4(xv, s_r[t], gm[i]);
                    acc[t] = fmaf(w[i].x, xv.x, acc[t]);
                    acc[t] = fmaf(w[i].y, xv.y, acc[t]);
                    acc[t] = fmaf(w[i].z, xv.z, acc[t]);
                    acc[t] = fmaf(w[i].w, xv.w, acc[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) s_part[warp][t] = v;
    }
    __syncthreads();
    stamp(p, 0, 2);
    if (tid < T) {
        float s = 0.f;
#pragma unroll
        for (int wi = 0; wi < kK1Threads / 32; ++wi) s += s_part[wi][tid];
        p.logits[(int64_t)tid * E + e] = s;
    }
    stamp(p, 0, 3);
}

// ============================================================================ K2: routing + gate/up
// Routed units: (active expert a, row pair rp) = rows 2rp, 2rp+1 of gate and up, split
// into chunks of 32 groups (64 weights each; lane = group in the chunk).  Warp w of the
// grid takes units w, w + W, ...; every chunk of its units streams through the warp's
// two ring slots (each lane copies and later reads only its own 16-byte pieces).
template <int NT, int kSh>
__global__ void __launch_bounds__(kK2MaxWarps * 32, 1) chain_gateup_kernel(const __grid_constant__ ChainParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ CtaRoute<NT> R;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthr = blockDim.x;
    const int T = p.T, H = p.H, I = p.I, k = p.rc.k, E = p.rc.E, P = T * k;
    const int G = qd4_groups(H);
    constexpr bool has_shared = kSh != 0;
    uint4* X = reinterpret_cast<uint4*>(smem);
    float4* XS = reinterpret_cast<float4*>(X + (size_t)T * 16 * G);
    float4* xs_s = reinterpret_cast<float4*>(smem + p.k2_off_xs_s);
    uint8_t* cring = smem + p.k2_off_ring;          // two round slots: [32 gate rows][32 up rows]
    // two ring slots of four quarters (8 gate + 8 up rows each, for warps 4q .. 4q + 3); [8]: the
    // test stall (never arrived on)
    __shared__ __align__(8) uint64_t c_bar[9];
    stamp(p, 1, 0);
    if (tid == 0) {
        for (int i = 0; i < 9; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&c_bar[i])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const bool xb = p.x_bf16 != 0;
    // ---- x is the input of the whole chain: stage it before waiting (with a pre-norm, x is the
    // residual stream that the layer before finished writing before K1 let this kernel start)
    __shared__ float s_r[kCMaxT], s_rpart[kCMaxT][8];
    if (p.gamma) rms_scales_cta(reinterpret_cast<const float*>(p.x), T, H, p.eps, s_rpart, s_r);
    qd4_stage_par<2>(p.x, xb, false, H, T, nullptr, H, X, XS, tid, nthr, p.gamma, s_r);   // bf16 values
    if (kSh == 2) {
        const int slots = p.it_H_s * 256;
        for (int t = 0; t < T; ++t) {
            const void* src = xb ? (const void*)(reinterpret_cast<const __nv_bfloat16*>(p.x) + (int64_t)t * H)
                                 : (const void*)(reinterpret_cast<const float*>(p.x) + (int64_t)t * H);
            qd_stage<MOE_Q8_0>(src, xb, false, H, p.it_H_s, xs_s + (size_t)t * slots, tid, nthr);
        }
    }
    stamp(p, 1, 1);
    pdl_wait();                                   // the logits of K1
    pdl_launch_dependents();
    stamp(p, 1, 2);
    cta_route(p, R);
    stamp(p, 1, 3);
    const int nact = R.nact;
    const int64_t rbH = (int64_t)(H / kQ4KWeights) * kQ4KBytes;
    const int half_I = I / 2;
    const int Ur = nact * half_I;
    const int Us = has_shared ? p.I_s / 2 : 0;
    const int W = gridDim.x * (nthr / 32);
    const int wg = blockIdx.x * (nthr / 32) + warp;
    const int my_units = wg < Ur ? (Ur - wg + W - 1) / W : 0;

    // ---- routed units, one round per 16: round r of this CTA covers the units wg0 + r W ..
    // + 15 (wg0 = 16 * blockIdx.x), i.e. 32 consecutive rows of gate and of up of one expert
    // (half_I is a multiple of 16) -- one staged sub-block of h.  A round arrives in slot r % 2
    // as four quarters, each two bulk copies (8 gate rows, 8 up rows; rows are whole, H <= 2048)
    // on its own mbarrier; warp w computes the row pair of unit wg0 + r W + w as soon as its
    // quarter w / 4 has landed, while the rest of the round still streams in.
    const int n_rounds = my_units;                 // the same for every warp of the CTA
    const uint32_t rows_bytes = (uint32_t)(32 * rbH);
    const uint32_t qbytes = (uint32_t)(8 * rbH);
    auto issue_round = [&](int r) {
        if (tid != 0 || r >= n_rounds) return;
        const int u0 = blockIdx.x * (nthr / 32) + r * W;
        const int a = u0 / half_I, row0 = 2 * (u0 - a * half_I);
        const int64_t off = (int64_t)R.act_e[a] * p.stride_gu + row0 * rbH;
        uint8_t* dst = cring + (r & 1) * 2 * rows_bytes;
        for (int q = 0; q < 4; ++q) {
            uint64_t* bar = &c_bar[(r & 1) * 4 + q];
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(2 * qbytes)
                         : "memory");
            bulk_to_smem(dst + q * qbytes, p.wg + off + q * qbytes, qbytes, bar);
            bulk_to_smem(dst + rows_bytes + q * qbytes, p.wu + off + q * qbytes, qbytes, bar);
        }
    };
    // the CTA's first two rounds go out before anything else
    issue_round(0);
    issue_round(1);
    // ---- this CTA's share of the shared expert's down rows into L2 (the routed down rows are
    // fetched by the down kernel itself, which starts on the SMs this kernel leaves early)
    if constexpr (has_shared) {
        const int rows0 = (int)((int64_t)blockIdx.x * H / gridDim.x), rows1 = (int)((int64_t)(blockIdx.x + 1) * H / gridDim.x);
        if (warp == 0 && lane == 31 && rows1 > rows0) {
            const int64_t rbS = p.s_q8 ? (p.s_q80r ? q80r_row_bytes(p.I_s) : (int64_t)(p.I_s / kQ80Weights) * kQ80Bytes)
                                       : (int64_t)(p.I_s / kQ4KWeights) * kQ4KBytes;
            if ((rbS % 16) == 0) prefetch_l2(p.sd + rows0 * rbS, (int64_t)(rows1 - rows0) * rbS);
        }
    }
    // ---- CTA 0 publishes the routing (the down kernel and the debug views read it)
    if (blockIdx.x == 0) {
        for (int i = tid; i < P; i += nthr) {
            p.ids[i] = R.ids[i];
            p.gw[i] = R.w[i];
            p.sorted[i] = R.sorted[i];
            p.pair_pos[i] = R.ppos[i];
        }
        for (int e = tid; e <= E; e += nthr) {
            int cnt = 0, mine = 0;
            for (int i = 0; i < P; ++i) {
                cnt += R.ids[i] < e ? 1 : 0;
                mine += R.ids[i] == e ? 1 : 0;
            }
            p.offsets[e] = cnt;
            // the running routing histogram (nullable), from the same pass
            if (p.counts && e < E && mine > 0) atomicAdd(&p.counts[e], (unsigned long long)mine);
        }
        __syncthreads();
        if (tid == 0) {                            // the down kernel may read the routing from here on
            __threadfence();
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&p.hdr->route_ready), "r"(1u) : "memory");
        }
    }
    // ---- the rounds.  Every warp runs all of them, so the barrier below is reached uniformly,
    // also after a copy that timed out (the CTA then stops computing and issuing, not looping).
    __shared__ float s_hq[2][kCMaxT][32];
    const int vb = 272 * qd4_groups(I);            // bytes of one staged vector of h
    float acc[4][NT];
    int vidx[NT];
    bool ok = true;
    int issued = min(2, n_rounds);
    for (int r = 0; r < n_rounds; ++r) {
        // (test stall: the first round waits on a barrier that never completes)
        const bool have = ok && (p.stall && r == 0 ? mbar_wait(&c_bar[8], 0u, p.wait_ns)
                                                   : mbar_wait(&c_bar[(r & 1) * 4 + (warp >> 2)], (uint32_t)(r >> 1) & 1u,
                                                               p.wait_ns));
        if (ok && !have) {
            ok = false;
            if (tid == 0) atomicExch(&p.hdr->status, (int)MOE_ERR_TIMEOUT);
        }
        const int u = wg + r * W;
        const int a = u / half_I, r0 = 2 * (u - a * half_I);
        const int st = R.act_start[a], n = R.act_n[a];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[q][t] = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) vidx[t] = R.tok[st + min(t, n - 1)];
        if (have && lane < G) {
            // rows 0, 1 = gate, up of row r0; rows 2, 3 = gate, up of row r0 + 1 (slot rows 2w, 2w + 1)
            const uint8_t* base = cring + (r & 1) * 2 * rows_bytes + (lane >> 2) * kQ4KBytes;
            const uint8_t* rb[4] = {base + (2 * warp) * rbH, base + rows_bytes + (2 * warp) * rbH,
                                    base + (2 * warp + 1) * rbH, base + rows_bytes + (2 * warp + 1) * rbH};
            const int c = lane & 3;
            uint4 hd[4], q0[4], q1[4];
            const bool live[4] = {true, true, true, true};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                hd[q] = *reinterpret_cast<const uint4*>(rb[q]);
                q0[q] = *reinterpret_cast<const uint4*>(rb[q] + 16 + 32 * c);
                q1[q] = *reinterpret_cast<const uint4*>(rb[q] + 32 + 32 * c);
            }
            qd4_group_math<NT, 4, 2>(hd, q0, q1, live, 0, lane, G, X, XS, n, acc, vidx);
        }
        constexpr int sh = qd_red_shift<NT>();
        const float gv = qd_warp_reduce_t<NT>(acc);
        const float uv = __shfl_xor_sync(0xffffffffu, gv, NT << sh);
        {
            const int i = lane >> sh, q = i / NT, t = i - q * NT;
            if ((q & 1) == 0 && (lane & ((1 << sh) - 1)) == 0 && t < n)
                s_hq[r & 1][t][(r0 & 31) + (q >> 1)] = silu_mul(gv, uv);
        }
        __syncthreads();                           // slot r % 2 read by every warp; s_hq complete
        if (ok && r + 2 < n_rounds) {
            issue_round(r + 2);
            issued = r + 3;
        }
        if (warp < n)
            warp_stage_subblock(s_hq[r & 1][warp][lane], p.hq + (size_t)(st + warp) * vb, qd4_groups(I), r0 >> 5, lane);
        if (r == 0) stamp(p, 1, 4);
    }
    stamp(p, 1, 5);
    if (!ok && tid == 0) {
        // let no copy land after the CTA exits: wait (bounded) for the ones still in flight
        for (int i = max(0, issued - 2); i < issued; ++i)      // at most two rounds are in flight
            for (int q = 0; q < 4; ++q) mbar_wait(&c_bar[(i & 1) * 4 + q], (uint32_t)(i >> 1) & 1u, p.wait_ns);
    }
    __syncthreads();
    int round = n_rounds;                          // the shared expert's sub-blocks continue the s_hq parity
    // ---- the shared expert's row pairs (direct loads)
    if constexpr (has_shared) {
    for (int u = wg + my_units * W; u < Ur + Us; u += W) {
        if (u < Ur) continue;
        float sacc[4][NT];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) sacc[r][t] = 0.f;
        const int r0 = 2 * (u - Ur);
        int sv[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) sv[t] = min(t, T - 1);
        if (kSh == 2) {
            const int64_t rbS = p.s_q80r ? q80r_row_bytes(H) : (int64_t)(H / kQ80Weights) * kQ80Bytes;
            const uint8_t* const rowp[4] = {p.sg + r0 * rbS, p.sg + (r0 + 1) * rbS, p.su + r0 * rbS,
                                            p.su + (r0 + 1) * rbS};
            qd_rows4<MOE_Q8_0, NT, false>(rowp, H / kQ80Weights, p.it_H_s, xs_s, p.it_H_s * 256,
                                          reinterpret_cast<const float2*>(xs_s), 0, T, lane, sacc, sv,
                                          p.s_q80r != 0);
        } else {
            const uint8_t* const rowp[4] = {p.sg + r0 * rbH, p.sg + (r0 + 1) * rbH, p.su + r0 * rbH,
                                            p.su + (r0 + 1) * rbH};
            qd4_rows4<NT, false, 2>(rowp, H / kQ4KWeights, X, XS, T, lane, sacc, sv);
        }
        // rows 0, 1 = gate of rows r0, r0 + 1; rows 2, 3 = up of the same rows
        constexpr int sh = qd_red_shift<NT>();
        const float gv = qd_warp_reduce_t<NT>(sacc);
        const float uv = __shfl_xor_sync(0xffffffffu, gv, (2 * NT) << sh);
        const int si = lane >> sh, sr = si / NT, st_ = si - sr * NT;
        const bool s_lead = sr < 2 && (lane & ((1 << sh) - 1)) == 0 && st_ < T;
        if constexpr (kSh == 2) {
            if (s_lead) p.h_s[(int64_t)st_ * p.I_s + r0 + sr] = silu_mul(gv, uv);
        } else {
            if (s_lead) s_hq[round & 1][st_][(r0 & 31) + sr] = silu_mul(gv, uv);
            __syncthreads();
            if (warp < T)
                warp_stage_subblock(s_hq[round & 1][warp][lane], p.hq_s + (size_t)warp * 272 * qd4_groups(p.I_s),
                                    qd4_groups(p.I_s), r0 >> 5, lane);
            ++round;
        }
    }
    }
    if (p.stamps) {                               // (timing hook) the whole CTA is done
        __syncthreads();
        stamp(p, 1, 6);
    }
}

// ============================================================================ K3: down + combine
// CTA c owns output rows [c*R, c*R + R).  Tasks: (pair s, 8 rows) with lane = 4*row + sub
// and sub taking groups sub, sub+4, ...; then the shared expert's rows 4 at a time.
template <int NT, int kSh>
__global__ void __launch_bounds__(kK3Threads) chain_down_kernel(const __grid_constant__ ChainParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int32_t s_e[kCMaxP], s_pos[kCMaxP];
    __shared__ float s_w[kCMaxP];
    __shared__ __align__(8) uint64_t s_wbar, s_hbar;
    __shared__ int s_route_ok;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = p.T, H = p.H, I = p.I, k = p.rc.k, P = T * k;
    const int GI = qd4_groups(I);
    const int R = p.rows_per_cta, n0 = blockIdx.x * R;
    constexpr bool has_shared = kSh != 0;
    const int64_t rbI = (int64_t)(I / kQ4KWeights) * kQ4KBytes;
    const int vb = 272 * GI;                                             // bytes of one staged h vector
    uint8_t* hsm = smem;                                                 // [P][vb]: h of pair s, staged
    float* ybuf = reinterpret_cast<float*>(smem + p.k3_off_y);          // [P + T][R]
    uint8_t* wbuf = smem + p.k3_off_w;                                   // [P][R][rbI] when prefetching
    uint4* SX = reinterpret_cast<uint4*>(smem + p.k3_off_hs_s);          // Q4_K shared expert: [T][16 GS] uint4
    const int GS = kSh == 1 ? qd4_groups(p.I_s) : 1;
    float4* SXS = reinterpret_cast<float4*>(SX + (size_t)T * 16 * GS);   // then [T][GS] float4
    stamp(p, 2, 0);
    // ---- the routing, which CTA 0 of the gate/up kernel publishes ahead of its units: read it
    // (and fetch the down rows it selects) while the gate/up kernel still computes h
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_wbar)) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_hbar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        uint32_t ready = 0u;
        const uint64_t t0 = gtime();
        for (;;) {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(ready) : "l"(&p.hdr->route_ready) : "memory");
            if (ready || gtime() - t0 > p.wait_ns) break;
            __nanosleep(64);
        }
        s_route_ok = ready != 0u;
        if (!ready) atomicExch(&p.hdr->status, (int)MOE_ERR_TIMEOUT);
    }
    __syncthreads();
    const bool route_ok = s_route_ok != 0;
    if (route_ok)
        for (int i = tid; i < P; i += kK3Threads) {
            s_e[i] = __ldcg(p.ids + i);
            s_pos[i] = __ldcg(p.pair_pos + i);
            s_w[i] = __ldcg(p.gw + i);
        }
    __syncthreads();
    stamp(p, 2, 2);
    const int nrows = min(R, H - n0);
    const bool wcopy = route_ok && p.k3_prefetch && nrows > 0;
    if (route_ok && !p.k3_prefetch && nrows > 0 && warp == 0)   // rows read in place later: into L2 now
        for (int s = lane; s < P; s += 32)
            prefetch_l2(p.wd + (int64_t)s_e[s] * p.stride_d + (int64_t)n0 * rbI, (int64_t)nrows * rbI);
    if (wcopy) {
        if (tid == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&s_wbar)),
                         "r"((uint32_t)(P * nrows * rbI))
                         : "memory");
        __syncthreads();
        if (warp == 0)
            for (int s = lane; s < P; s += 32)
                bulk_to_smem(wbuf + (int64_t)s * R * rbI, p.wd + (int64_t)s_e[s] * p.stride_d + (int64_t)n0 * rbI,
                             (uint32_t)(nrows * rbI), &s_wbar);
    }
    pdl_wait();                                   // h of K2
    pdl_launch_dependents();
    stamp(p, 2, 1);
    if (!route_ok) return;
    // ---- every pair's h, which the gate/up kernel wrote already staged (one bulk copy per
    // pair); the CTA's down rows of every pair (rows n0.. of one expert are contiguous: one
    // copy per pair) were requested above, on their own mbarrier
    if (tid == 0) {
        uint32_t total = (uint32_t)P * vb;
        if (kSh == 1) total += (uint32_t)T * 272 * GS;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&s_hbar)), "r"(total)
                     : "memory");
    }
    __syncthreads();
    if (warp == 1) {
        for (int s = lane; s < P; s += 32)
            bulk_to_smem(hsm + (size_t)s * vb, p.hq + (size_t)s_pos[s] * vb, (uint32_t)vb, &s_hbar);
    } else if (warp == 2 && kSh == 1) {
        for (int t = lane; t < T; t += 32) {
            const uint8_t* src = p.hq_s + (size_t)t * 272 * GS;
            bulk_to_smem(SX + (size_t)t * 16 * GS, src, (uint32_t)(256 * GS), &s_hbar);
            bulk_to_smem(SXS + (size_t)t * GS, src + 256 * GS, (uint32_t)(16 * GS), &s_hbar);
        }
    }
    if constexpr (kSh == 2) {                          // Q8_0 shared expert: its h is fp32
        float4* hs = reinterpret_cast<float4*>(smem + p.k3_off_hs_s);
        qd_stage_many_f32<MOE_Q8_0>(p.h_s, p.I_s, T, p.I_s, p.it_Is_s, hs, tid, kK3Threads);
    }
    stamp(p, 2, 3);
    const bool landed = mbar_wait(&s_hbar, 0u, p.wait_ns) && (!wcopy || mbar_wait(&s_wbar, 0u, p.wait_ns));
    if (__syncthreads_or(!landed)) {
        // the copies did not complete in time: report it; let none land after the CTA exits
        if (tid == 0) {
            atomicExch(&p.hdr->status, (int)MOE_ERR_TIMEOUT);
            mbar_wait(&s_hbar, 0u, p.wait_ns);
            if (wcopy) mbar_wait(&s_wbar, 0u, p.wait_ns);
        }
        __syncthreads();
        return;
    }
    stamp(p, 2, 4);
    const int nsub = R / 8;
    const int n_routed = P * nsub;
    const int n_shared = has_shared ? R / 4 : 0;
    for (int task = warp; task < n_routed + n_shared; task += kK3Threads / 32) {
        if (task < n_routed) {
            // each 16-lane half takes 4 of the task's 8 rows; lane = one 64-weight group of all 4
            // rows (groups gl, gl + 16, ...), so each activation load serves 4 rows and the lane
            // has 4 rows' independent integer sums in flight
            const int s = task / nsub, sb = task - s * nsub;
            const int half = lane >> 4, gl = lane & 15;
            const int rl0 = 8 * sb + 4 * half;
            float acc[4][1] = {{0.f}, {0.f}, {0.f}, {0.f}};
            const uint4* Xs = reinterpret_cast<const uint4*>(hsm + (size_t)s * vb);
            const float4* XSs = reinterpret_cast<const float4*>(hsm + (size_t)s * vb + 256 * GI);
            const uint8_t* rowp[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int n = n0 + rl0 + r;
                rowp[r] = n >= H ? nullptr
                          : p.k3_prefetch ? wbuf + ((int64_t)s * R + rl0 + r) * rbI
                                          : p.wd + (int64_t)s_e[s] * p.stride_d + (int64_t)n * rbI;
            }
            if (p.k3_prefetch) {
                for (int g = gl; g < GI; g += 16) qd4_group<1, 4, true, 3>(rowp, 0, g, GI, Xs, XSs, 1, acc, nullptr);
            } else {
                for (int g = gl; g < GI; g += 16) qd4_group<1, 4, false, 3>(rowp, 0, g, GI, Xs, XSs, 1, acc, nullptr);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float v = acc[r][0];
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (gl == 0 && n0 + rl0 + r < H) ybuf[s * R + rl0 + r] = v;
            }
        } else if constexpr (has_shared) {
            const int q = task - n_routed;
            const int nb = n0 + 4 * q;
            float acc[4][NT];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
            int vidx[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) vidx[t] = min(t, T - 1);
            if (kSh == 2) {
                const int64_t rbS = p.s_q80r ? q80r_row_bytes(p.I_s) : (int64_t)(p.I_s / kQ80Weights) * kQ80Bytes;
                const uint8_t* rowp[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) rowp[r] = nb + r < H ? p.sd + (int64_t)(nb + r) * rbS : nullptr;
                const float4* hs = reinterpret_cast<const float4*>(smem + p.k3_off_hs_s);
                qd_rows4<MOE_Q8_0, NT, false>(rowp, p.I_s / kQ80Weights, p.it_Is_s, hs, p.it_Is_s * 256,
                                              reinterpret_cast<const float2*>(hs), 0, T, lane, acc, vidx,
                                              p.s_q80r != 0);
            } else {
                const int64_t rbS = (int64_t)(p.I_s / kQ4KWeights) * kQ4KBytes;
                const uint8_t* rowp[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) rowp[r] = nb + r < H ? p.sd + (int64_t)(nb + r) * rbS : nullptr;
                qd4_rows4<NT, false, 3>(rowp, p.I_s / kQ4KWeights, SX, SXS, T, lane, acc, vidx);
            }
            constexpr int sh = qd_red_shift<NT>();
            const float v = qd_warp_reduce_t<NT>(acc);
            const int i = lane >> sh, ri = i / NT, t = i - ri * NT;
            if ((lane & ((1 << sh) - 1)) == 0 && t < T) ybuf[(P + t) * R + 4 * q + ri] = v;
        }
    }
    __syncthreads();
    stamp(p, 2, 5);
    // ---- combine: out[t][n] = ((sum_j w_tj * y_(t,j)[n]) + shared) (+ old out)
    for (int idx = tid; idx < T * R; idx += kK3Threads) {
        const int t = idx / R, nl = idx - t * R, n = n0 + nl;
        if (n >= H) continue;
        float acc = 0.f;
        for (int j = 0; j < k; ++j) acc = fmaf(s_w[t * k + j], ybuf[(t * k + j) * R + nl], acc);
        if (has_shared) acc += ybuf[(P + t) * R + nl];
        float* o = p.out + (int64_t)t * H + n;
        if (p.accumulate) acc += *o;
        *o = acc;
    }
    if (p.stamps) {                               // (timing hook) the whole CTA is done
        __syncthreads();
        stamp(p, 2, 6);
    }
}

// ============================================================================ host side
struct ChainLayout {
    size_t k2_smem, k3_smem;
    int k2_warps, k2_off_xs_s, k2_off_ring;
    int k3_prefetch, k3_off_hs_s, k3_off_y, k3_off_w;
    int it_H_s, it_Is_s, rows_per_cta;
};

int g_sms = 0;

int sm_count() {
    if (g_sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return 0;
        cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    }
    return g_sms;
}

constexpr size_t kChainSmemCap = 200 * 1024;   // dynamic; the kernels' static shared memory is < 21 KB
constexpr size_t kK3TwoPerSm = 108 * 1024;     // dynamic shared memory of a down CTA that still fits twice

ChainLayout chain_layout(const DecodeArgs& a) {
    ChainLayout L{};
    const int T = a.T, P = a.T * a.route.top_k, H = a.H, I = a.I;
    const bool sh = a.I_s > 0, q8 = sh && a.s_qtype == MOE_Q8_0;
    L.it_H_s = q8 ? walk_iters<MOE_Q8_0>(H) : 0;
    L.it_Is_s = q8 ? walk_iters<MOE_Q8_0>(a.I_s) : 0;
    // K2: staged x, then two ring slots per warp; as many warps as fit (at most 16)
    size_t o = (size_t)T * qd4_vec_bytes(H);
    L.k2_off_xs_s = (int)align_up(o, 16);
    o = L.k2_off_xs_s + (q8 ? (size_t)T * L.it_H_s * 4096 : 0);
    L.k2_off_ring = (int)align_up(o, 128);
    const size_t per_warp = (size_t)2 * kSlotBytes;
    int warps = kK2MaxWarps;
    while (warps > 1 && L.k2_off_ring + warps * per_warp > kChainSmemCap) --warps;
    L.k2_warps = warps;
    L.k2_smem = L.k2_off_ring + warps * per_warp;
    // K3: about two CTAs per SM, 8-row multiples; one CTA per SM with twice the rows when the
    // staged h leaves room for only one (many pairs), so that each SM stages h once
    const int sms = std::max(1, sm_count());
    o = (size_t)P * qd4_vec_bytes(I);
    L.k3_off_hs_s = (int)align_up(o, 16);
    if (sh) o = L.k3_off_hs_s + (q8 ? (size_t)T * L.it_Is_s * 4096 : (size_t)T * qd4_vec_bytes(a.I_s));
    L.k3_off_y = (int)align_up(o, 16);
    int R = (H + 2 * sms - 1) / (2 * sms);
    R = std::max(8, (R + 7) / 8 * 8);
    if (L.k3_off_y + (size_t)(P + T) * R * 4 > kK3TwoPerSm) {
        R = (H + sms - 1) / sms;
        R = std::max(8, (R + 7) / 8 * 8);
    }
    L.rows_per_cta = R;
    o = L.k3_off_y + (size_t)(P + T) * R * 4;
    L.k3_off_w = (int)align_up(o, 16);
    // the down rows are copied into shared memory only while two CTAs still fit an SM (the
    // grid is about two CTAs per SM); otherwise they are read in place, from L2
    const size_t wbytes = (size_t)P * R * (size_t)(I / kQ4KWeights) * kQ4KBytes;
    L.k3_prefetch = L.k3_off_w + wbytes <= kK3TwoPerSm ? 1 : 0;
    L.k3_smem = L.k3_off_w + (L.k3_prefetch ? wbytes : 0);
    return L;
}

template <int NT, int Q8>
cudaError_t launch_chain_nt(const ChainParams& p, const ChainLayout& L, int E, cudaStream_t s, cudaEvent_t evb,
                            cudaEvent_t eva) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    cfg.gridDim = dim3(E);
    cfg.blockDim = dim3(kK1Threads);
    cfg.dynamicSmemBytes = 0;
    if ((err = cudaLaunchKernelEx(&cfg, chain_logits_kernel<NT>, p)) != cudaSuccess) return err;
    if (evb && (err = cudaEventRecord(evb, s)) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(chain_gateup_kernel<NT, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)L.k2_smem)) != cudaSuccess)
        return err;
    cfg.gridDim = dim3(sm_count());
    cfg.blockDim = dim3(L.k2_warps * 32);
    cfg.dynamicSmemBytes = L.k2_smem;
    if ((err = cudaLaunchKernelEx(&cfg, chain_gateup_kernel<NT, Q8>, p)) != cudaSuccess) return err;
    if (eva && (err = cudaEventRecord(eva, s)) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(chain_down_kernel<NT, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)L.k3_smem)) != cudaSuccess)
        return err;
    cfg.gridDim = dim3((p.H + L.rows_per_cta - 1) / L.rows_per_cta);
    cfg.blockDim = dim3(kK3Threads);
    cfg.dynamicSmemBytes = L.k3_smem;
    return cudaLaunchKernelEx(&cfg, chain_down_kernel<NT, Q8>, p);
}

ChainParams chain_params(const DecodeArgs& a, const ChainLayout& L) {
    ChainParams p{};
    p.rc.mode = (int)a.route.mode;
    p.rc.E = a.route.n_experts;
    p.rc.k = a.route.top_k;
    p.rc.G = a.route.mode == MOE_ROUTE_SIGMOID_GROUP ? a.route.n_groups : 1;
    p.rc.Gk = a.route.mode == MOE_ROUTE_SIGMOID_GROUP ? a.route.topk_groups : 1;
    p.rc.renorm = a.route.renormalize;
    p.rc.scale = a.route.routed_scale;
    p.Wr = a.Wr; p.bias = a.bias; p.x = a.x; p.x_bf16 = a.x_bf16 ? 1 : 0;
    p.gamma = a.norm_gamma; p.eps = a.norm_eps;
    p.T = a.T; p.H = a.H; p.I = a.I;
    p.wg = a.wg; p.wu = a.wu; p.wd = a.wd;
    p.stride_gu = a.stride_gu; p.stride_d = a.stride_d;
    p.I_s = a.I_s; p.s_q8 = (a.I_s > 0 && a.s_qtype == MOE_Q8_0) ? 1 : 0;
    p.s_q80r = (p.s_q8 && a.s_q80r) ? 1 : 0;
    p.sg = a.sg; p.su = a.su; p.sd = a.sd;
    p.logits = a.logits; p.ids = a.ids; p.gw = a.gw; p.sorted = a.sorted; p.offsets = a.offsets;
    p.pair_pos = a.pair_pos;
    p.hq = a.hq; p.hq_s = a.hq_s; p.h_s = a.h_s; p.out = a.out; p.accumulate = a.accumulate ? 1 : 0;
    p.hdr = a.hdr; p.counts = a.counts;
    p.it_H_s = L.it_H_s; p.it_Is_s = L.it_Is_s;
    p.k2_warps = L.k2_warps; p.k2_off_xs_s = L.k2_off_xs_s; p.k2_off_ring = L.k2_off_ring;
    p.rows_per_cta = L.rows_per_cta; p.k3_prefetch = L.k3_prefetch;
    p.k3_off_hs_s = L.k3_off_hs_s; p.k3_off_y = L.k3_off_y; p.k3_off_w = L.k3_off_w;
    const WaitCfg wc = wait_cfg();
    p.wait_ns = wc.limit_ns; p.stall = wc.stall;
    p.stamps = static_cast<uint64_t*>(debug_stamps());
    return p;
}

}  // namespace

bool decode_chain_supported(const DecodeArgs& a) {
    if (sm_count() <= 0) return false;
    const int P = a.T * a.route.top_k;
    if (a.T < 1 || a.T > kCMaxT || P > kCMaxP || a.route.n_experts > kCMaxE) return false;
    if (a.qtype != MOE_Q4_K) return false;
    if (!a.x_bf16 && !a.norm_gamma) return false;   // x is staged as bf16 values (two planes)
    if (a.H % kQ4KWeights || a.I % kQ4KWeights || a.H / 4 > kK1MaxVec * kK1Threads) return false;
    // a round of the gate/up kernel copies 32 whole rows of gate and of up: rows of at most
    // kChunkBlocks super-blocks (the ring's slot size), I/2 a multiple of 16
    if (a.H > kChunkBlocks * kQ4KWeights || (a.I / 2) % kK2MaxWarps) return false;
    if (a.I_s > 0) {
        if (a.s_qtype == MOE_Q8_0) {
            if (a.I_s % kQ80Weights || a.H % kQ80Weights || a.I_s % 2) return false;
        } else if (a.s_qtype == MOE_Q4_K) {
            if (a.I_s % kQ4KWeights) return false;
        } else {
            return false;
        }
    }
    if ((a.stride_gu % 16) || (a.stride_d % 16)) return false;
    const ChainLayout L = chain_layout(a);
    return L.k2_warps == kK2MaxWarps && L.k2_smem <= kChainSmemCap && L.k3_smem <= kChainSmemCap;
}

cudaError_t launch_decode_chain(const DecodeArgs& a, cudaStream_t s, cudaEvent_t evb, cudaEvent_t eva) {
    const ChainLayout L = chain_layout(a);
    const ChainParams p = chain_params(a, L);
    const int E = a.route.n_experts;
    const int sh = a.I_s <= 0 ? 0 : p.s_q8 ? 2 : 1;
    auto go = [&](auto nt) -> cudaError_t {
        constexpr int NT = decltype(nt)::value;
        return sh == 0 ? launch_chain_nt<NT, 0>(p, L, E, s, evb, eva) : sh == 1 ? launch_chain_nt<NT, 1>(p, L, E, s, evb, eva)
                                                                       : launch_chain_nt<NT, 2>(p, L, E, s, evb, eva);
    };
    switch (a.T) {
        case 1: return go(std::integral_constant<int, 1>{});
        case 2: return go(std::integral_constant<int, 2>{});
        case 3: case 4: return go(std::integral_constant<int, 4>{});
        default: return go(std::integral_constant<int, 8>{});
    }
}

}  // namespace moe
