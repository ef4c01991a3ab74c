// gemv_seg.cu -- the routed experts' gate/up and down for 5 <= T < 128 tokens.
//
// Between the decode chain (T <= 6 at hidden 2048) and the tensor-core GEMM the layer is still a
// dequant-GEMV bound by the weight bytes, but each chosen expert now serves a few
// tokens.  A persistent grid (one 16-warp CTA per SM) walks the active experts' units,
// once per pass of at most NT of the expert's tokens; CTA c owns a contiguous range of
// these (expert, pass, unit) triples of equal estimated cost, so it meets few segments.
// For each segment it stages the pass's tokens once, then every warp streams its units'
// rows through a two-slot ring in shared memory (bulk copies completing on an mbarrier
// per slot) and computes them against the staged tokens: the weight bytes come from HBM
// once and from L2 on the later passes, with many units in flight per SM.
//   gate/up: unit = rows 2rp, 2rp+1 of gate and up of one expert -> h fp32 [P][I]
//   down:    unit = 8 rows of one expert's down matrix, 4 lanes a row (rows of fewer
//            than 32 activation groups), or 4 rows with one group a lane (the gate/up
//            layout, rows of 32 groups or more)                  -> y fp32 [P][H]
// Pairs are in sorted (expert-major) order; the combine kernel gathers them per token.
// Dot products use the integer Q4_K walk of qdot.cuh in a fixed order.
#include <algorithm>

#include "internal.cuh"
#include "qdot.cuh"

namespace moe {
namespace {

constexpr int kSWarps = 16;
constexpr int kSThreads = kSWarps * 32;
constexpr int kSMaxE = 256;
constexpr int kSChunkBlocks = 8;                       // gate/up item: 8 blocks of 4 rows
constexpr int kSSlotBytes = 4 * kSChunkBlocks * kQ4KBytes;
constexpr int kSDownBlocks = 4;                        // down item: 4 blocks of 8 rows

struct SegParams {
    const void* vin;                 // gate/up: x [T][H] (bf16 or fp32); down: h fp32 [P][I]
    int vin_bf16;
    const int32_t* sorted_pairs;     // gate/up: token of sorted position i = sorted_pairs[i] / k
    const int32_t* offsets;          // [E+1]
    int E, k, K, rows;               // K = input dim, rows = output rows per expert
    const uint8_t* w0;               // gate or down
    const uint8_t* w1;               // up (gate/up)
    int64_t expert_stride;
    float* out;                      // gate/up: h [P][I]; down: y [P][H]
    WsHeader* hdr;
    int nt_max;                      // tokens per staging pass (<= NT)
    uint64_t wait_ns;                // limit of every bounded wait
    int stall;                       // test setting: each warp's first wait never completes
};

__host__ __device__ inline size_t seg_align(size_t v) { return (v + 127) & ~(size_t)127; }
__device__ __forceinline__ uint32_t s_u32(const void* q) { return (uint32_t)__cvta_generic_to_shared(q); }
__device__ __forceinline__ uint64_t s_time() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool s_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2, %3;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(ok)
                 : "r"(s_u32(b)), "r"(parity), "r"(100000u)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool s_wait(uint64_t* b, uint32_t parity, uint64_t limit_ns) {
    if (s_test(b, parity)) return true;
    const uint64_t t0 = s_time();
    while (!s_test(b, parity))
        if (s_time() - t0 > limit_ns) return false;
    return true;
}
__device__ __forceinline__ void s_bulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     s_u32(dst)),
                 "l"(src), "r"(bytes), "r"(s_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void s_expect(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s_u32(b)), "r"(bytes) : "memory");
}

// Work plan.  Expert a (active, ascending id) with n_a tokens is computed in P_a passes of
// at most ntm tokens; its virtual units are its U units once per pass, pass-major, and a
// virtual unit of a pass with nt tokens costs kSegC0 + nt (streaming the unit's weights
// is worth about kSegC0 tokens of arithmetic on it).  CTA c owns the virtual units whose
// start cost lies in [c C / G, (c + 1) C / G), C the total: heavy experts' passes spread
// over several CTAs, light experts' units over few, and every CTA meets few segments.
constexpr int kSegC0 = 4;

struct SegPlan {
    int act_e[kSMaxE], act_st[kSMaxE], act_n[kSMaxE];
    int vb[kSMaxE + 1];              // first virtual unit of active expert a
    long long cb[kSMaxE + 1];        // first cost of active expert a
    int nact, v_lo, v_hi, a_lo;
};

// Virtual unit at cost b (the first one starting at or after it), and its expert.  Warp-wide.
__device__ int seg_locate(const SegPlan& s, int nact, int U, int ntm, long long b, int* a_out) {
    const int lane = threadIdx.x & 31;
    if (b >= s.cb[nact]) { *a_out = nact; return s.vb[nact]; }
    int cnt = 0;
    for (int base = 0; base < nact; base += 32) {
        const int a = base + lane;
        cnt += __popc(__ballot_sync(0xffffffffu, a < nact && s.cb[a] <= b));
    }
    const int a = cnt - 1;
    const int n = s.act_n[a], P = (n + ntm - 1) / ntm;
    const long long r = b - s.cb[a], F = (long long)U * (kSegC0 + ntm);
    const int pass = (int)min((long long)(P - 1), r / F);
    const long long r2 = r - pass * F;
    const int w = kSegC0 + min(ntm, n - pass * ntm);
    *a_out = a;
    return s.vb[a] + pass * U + (int)((r2 + w - 1) / w);
}

__device__ void seg_plan(const int32_t* offsets, int E, int U, int ntm, SegPlan& s) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        int seen = 0, vcarry = 0;
        long long ccarry = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            int o0 = 0, cnt = 0;
            if (e < E) { o0 = __ldcg(offsets + e); cnt = __ldcg(offsets + e + 1) - o0; }
            const unsigned nz = __ballot_sync(0xffffffffu, cnt > 0);
            const int passes = cnt > 0 ? (cnt + ntm - 1) / ntm : 0;
            const long long cost = (long long)U * (kSegC0 * passes + cnt);
            int pv = passes;
            long long pc = cost;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int ov = __shfl_up_sync(0xffffffffu, pv, d);
                const long long oc = __shfl_up_sync(0xffffffffu, pc, d);
                if (lane >= d) { pv += ov; pc += oc; }
            }
            if (cnt > 0) {
                const int a = seen + __popc(nz & ((1u << lane) - 1u));
                s.act_e[a] = e;
                s.act_st[a] = o0;
                s.act_n[a] = cnt;
                s.vb[a] = vcarry + (pv - passes) * U;
                s.cb[a] = ccarry + pc - cost;
            }
            seen += __popc(nz);
            vcarry += U * __shfl_sync(0xffffffffu, pv, 31);
            ccarry += __shfl_sync(0xffffffffu, pc, 31);
        }
        if (lane == 0) { s.vb[seen] = vcarry; s.cb[seen] = ccarry; }
        __syncwarp();
        const long long G = gridDim.x, c = blockIdx.x;
        int a_lo = 0, a_hi = 0;
        const int v_lo = seg_locate(s, seen, U, ntm, ccarry * c / G, &a_lo);
        const int v_hi = c + 1 == G ? vcarry : seg_locate(s, seen, U, ntm, ccarry * (c + 1) / G, &a_hi);
        if (lane == 0) { s.nact = seen; s.v_lo = v_lo; s.v_hi = v_hi; s.a_lo = a_lo; }
    }
    __syncthreads();
}

// ============================================================================ gate/up
// NPL: activation planes (2 for bf16 x, 3 for fp32 x)
template <int NT, int NPL>
__global__ void __launch_bounds__(kSThreads, 1) seg_gateup_kernel(const __grid_constant__ SegParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ SegPlan s_plan;
    __shared__ int s_rows[NT];
    __shared__ __align__(8) uint64_t s_bar[kSWarps][2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.K, I = p.rows, G = qd4_groups(H), half_I = I / 2;
    const int nblk = H / kQ4KWeights, nch = (G + 31) / 32;
    const int64_t rbH = (int64_t)nblk * kQ4KBytes;
    const int rs = nch == 1 ? (int)rbH : kSChunkBlocks * kQ4KBytes;     // row stride in a slot
    uint4* X = reinterpret_cast<uint4*>(smem);
    float4* XS = reinterpret_cast<float4*>(X + (size_t)NT * 16 * G);
    uint8_t* ring = smem + seg_align((size_t)NT * qd4_vec_bytes(H)) + (size_t)warp * 2 * kSSlotBytes;
    __shared__ __align__(8) uint64_t s_never;          // test stall: initialized, never arrived on
    if (lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_u32(&s_bar[warp][0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_u32(&s_bar[warp][1])) : "memory");
        if (warp == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_u32(&s_never)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    seg_plan(p.offsets, p.E, half_I, p.nt_max, s_plan);
    bool ok = true;
    uint32_t gi = 0;                                   // this warp's items so far (slot phases)
    int a = s_plan.a_lo;
    for (int v0 = s_plan.v_lo; v0 < s_plan.v_hi;) {
        while (s_plan.vb[a + 1] <= v0) ++a;
        const int rel = v0 - s_plan.vb[a], pass = rel / half_I, u0 = rel - pass * half_I;
        const int seg_end = min(s_plan.v_hi, s_plan.vb[a] + (pass + 1) * half_I);
        const int len = seg_end - v0;
        const int e = s_plan.act_e[a], st = s_plan.act_st[a], n_a = s_plan.act_n[a];
        const uint8_t* gbase = p.w0 + (int64_t)e * p.expert_stride;
        const uint8_t* ubase = p.w1 + (int64_t)e * p.expert_stride;
        const int my_units = warp < len ? (len - warp + kSWarps - 1) / kSWarps : 0;
        const int n_items = my_units * nch;
        {
            const int pb = pass * p.nt_max, nt = min(p.nt_max, n_a - pb);
            __syncthreads();                               // the previous segment is done with X
            if (tid < nt) s_rows[tid] = __ldcg(p.sorted_pairs + st + pb + tid) / p.k;
            __syncthreads();
            qd4_stage_par<NPL>(p.vin, p.vin_bf16 != 0, false, H, nt, s_rows, H, X, XS, tid, kSThreads);
            __syncthreads();
            int issued = 0, waited = 0;                    // items copied / landed in this pass
            auto issue = [&](int item) {
                if (item >= n_items || !ok) return;
                issued = item + 1;
                if (lane != 0) return;
                const int u = u0 + warp + (item / nch) * kSWarps, ch = item - (item / nch) * nch;
                const int r0 = 2 * u;
                const int b0 = ch * kSChunkBlocks, nb = min(kSChunkBlocks, nblk - b0);
                const uint32_t bytes = (uint32_t)nb * kQ4KBytes;
                const uint32_t slot = (gi + item) & 1u;
                uint8_t* dst = ring + slot * kSSlotBytes;
                uint64_t* bar = &s_bar[warp][slot];
                s_expect(bar, 4 * bytes);
                if (nch == 1) {
                    // whole rows: gate rows r0, r0 + 1 and up rows r0, r0 + 1 are two contiguous runs;
                    // slot rows (gate r0, gate r0 + 1, up r0, up r0 + 1) at rs apart
                    s_bulk(dst, gbase + r0 * rbH, 2 * bytes, bar);
                    s_bulk(dst + 2 * rs, ubase + r0 * rbH, 2 * bytes, bar);
                } else {
                    const uint8_t* rp[4] = {gbase + r0 * rbH, gbase + (r0 + 1) * rbH, ubase + r0 * rbH,
                                            ubase + (r0 + 1) * rbH};
#pragma unroll
                    for (int r = 0; r < 4; ++r) s_bulk(dst + r * rs, rp[r] + (int64_t)b0 * kQ4KBytes, bytes, bar);
                }
            };
            issue(0);
            issue(1);
            float acc[4][NT];
            for (int item = 0; item < n_items; ++item) {
                const uint32_t slot = (gi + item) & 1u, par = ((gi + item) >> 1) & 1u;
                // (test stall: the warp's first wait is on a barrier that never completes)
                uint64_t* wbar = p.stall && gi + item == 0 ? &s_never : &s_bar[warp][slot];
                const bool have = ok && s_wait(wbar, wbar == &s_never ? 0u : par, p.wait_ns);
                if (have) waited = item + 1;
                if (ok && !have) {
                    ok = false;
                    if (lane == 0 && p.hdr) atomicExch(&p.hdr->status, (int)MOE_ERR_TIMEOUT);
                }
                const int u = u0 + warp + (item / nch) * kSWarps, ch = item - (item / nch) * nch;
                if (ch == 0) {
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
                }
                const int g = ch * 32 + lane;
                if (have && g < G) {
                    const uint8_t* blk = ring + slot * kSSlotBytes + (lane >> 2) * kQ4KBytes;
                    const int c = lane & 3;
                    uint4 hd[4], q0[4], q1[4];
                    const bool live[4] = {true, true, true, true};
                    // acc rows 0..3 = gate r0, up r0, gate r0 + 1, up r0 + 1 = slot rows 0, 2, 1, 3
                    constexpr int kSlotRow[4] = {0, 2, 1, 3};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint8_t* rb = blk + kSlotRow[r] * rs;
                        hd[r] = *reinterpret_cast<const uint4*>(rb);
                        q0[r] = *reinterpret_cast<const uint4*>(rb + 16 + 32 * c);
                        q1[r] = *reinterpret_cast<const uint4*>(rb + 32 + 32 * c);
                    }
                    qd4_group_math<NT, 4, NPL>(hd, q0, q1, live, 0, g, G, X, XS, nt, acc, nullptr);
                }
                __syncwarp();
                issue(item + 2);
                if (ch == nch - 1) {
                    // rows 0, 1 = gate, up of row 2u; rows 2, 3 = gate, up of row 2u + 1
                    constexpr int sh = qd_red_shift<NT>();
                    const float gv = qd_warp_reduce_t<NT>(acc);
                    const float uv = __shfl_xor_sync(0xffffffffu, gv, NT << sh);
                    const int i = lane >> sh, r = i / NT, t = i - r * NT;
                    if ((r & 1) == 0 && (lane & ((1 << sh) - 1)) == 0 && t < nt)
                        p.out[(int64_t)(st + pb + t) * I + 2 * u + (r >> 1)] = gv / (1.0f + expf(-gv)) * uv;
                }
            }
            // the items of this pass are all consumed (or, after a timeout, waited for below)
            // after a timeout: wait (bounded) for the copies this warp issued and never saw land
            if (!ok && lane == 0)
                for (int i = waited; i < issued; ++i) s_wait(&s_bar[warp][(gi + i) & 1u], ((gi + i) >> 1) & 1u, p.wait_ns);
            gi += ok ? n_items : 0;
            __syncwarp();
        }
        v0 = seg_end;
    }
}

// ============================================================================ down
// Narrow rows (I/64 groups not a multiple of 32, e.g. I = 768): unit = 8 rows n0.. of one
// expert's down matrix; in every item (at most 4 blocks = 16 groups of the 8 rows) lane = 16 *
// half + gl takes group gl of rows 4 half .. 4 half + 3, so every activation load serves 4 rows;
// the 16 lanes of a half then sum.
// Wide rows (kWide: I/64 a multiple of 32, e.g. I = 2048): the gate/up layout -- unit = 4 rows,
// item = 8 blocks of the 4 rows, lane = group, so every activation load serves 4 rows.
template <int NT, bool kWide>
__global__ void __launch_bounds__(kSThreads, 1) seg_down_kernel(const __grid_constant__ SegParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ SegPlan s_plan;
    __shared__ int s_rows[NT];
    __shared__ __align__(8) uint64_t s_bar[kSWarps][2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kRowsU = kWide ? 4 : 8;           // rows per unit
    constexpr int kBlocksI = kWide ? kSChunkBlocks : kSDownBlocks;   // blocks of each row per item
    const int I = p.K, H = p.rows, GI = qd4_groups(I), upe = H / kRowsU;
    const int nblk = I / kQ4KWeights, ncd = (nblk + kBlocksI - 1) / kBlocksI;
    const int64_t rbI = (int64_t)nblk * kQ4KBytes;
    const int rs = ncd == 1 ? (int)rbI : kBlocksI * kQ4KBytes;     // row stride in a slot
    uint4* X = reinterpret_cast<uint4*>(smem);
    float4* XS = reinterpret_cast<float4*>(X + (size_t)NT * 16 * GI);
    uint8_t* ring = smem + seg_align((size_t)NT * qd4_vec_bytes(I)) + (size_t)warp * 2 * kSSlotBytes;
    __shared__ __align__(8) uint64_t s_never;          // test stall: initialized, never arrived on
    if (lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_u32(&s_bar[warp][0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_u32(&s_bar[warp][1])) : "memory");
        if (warp == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_u32(&s_never)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    seg_plan(p.offsets, p.E, upe, p.nt_max, s_plan);
    const int half = lane >> 4, gl = lane & 15;
    bool ok = true;
    uint32_t gi = 0;
    int a = s_plan.a_lo;
    for (int v0 = s_plan.v_lo; v0 < s_plan.v_hi;) {
        while (s_plan.vb[a + 1] <= v0) ++a;
        const int rel = v0 - s_plan.vb[a], pass = rel / upe, u0 = rel - pass * upe;
        const int seg_end = min(s_plan.v_hi, s_plan.vb[a] + (pass + 1) * upe);
        const int len = seg_end - v0;
        const int e = s_plan.act_e[a], st = s_plan.act_st[a], n_a = s_plan.act_n[a];
        const uint8_t* dbase = p.w0 + (int64_t)e * p.expert_stride;
        const int my_units = warp < len ? (len - warp + kSWarps - 1) / kSWarps : 0;
        const int n_items = my_units * ncd;
        {
            const int pb = pass * p.nt_max, nt = min(p.nt_max, n_a - pb);
            __syncthreads();
            if (tid < nt) s_rows[tid] = st + pb + tid;
            __syncthreads();
            qd4_stage_par<3>(p.vin, false, true, I, nt, s_rows, I, X, XS, tid, kSThreads);
            __syncthreads();
            int issued = 0, waited = 0;                    // items copied / landed in this pass
            auto issue = [&](int item) {
                if (item >= n_items || !ok) return;
                issued = item + 1;
                if (lane != 0) return;
                const int u = u0 + warp + (item / ncd) * kSWarps, ch = item - (item / ncd) * ncd;
                const int n0 = kRowsU * u;
                const int b0 = ch * kBlocksI, nb = min(kBlocksI, nblk - b0);
                const uint32_t slot = (gi + item) & 1u;
                uint8_t* dst = ring + slot * kSSlotBytes;
                uint64_t* bar = &s_bar[warp][slot];
                const uint32_t bytes = (uint32_t)nb * kQ4KBytes;
                s_expect(bar, kRowsU * bytes);
                if (ncd == 1) {                            // whole rows: one contiguous run
                    s_bulk(dst, dbase + (int64_t)n0 * rbI, kRowsU * bytes, bar);
                } else {
                    for (int r = 0; r < kRowsU; ++r)
                        s_bulk(dst + r * rs, dbase + (int64_t)(n0 + r) * rbI + (int64_t)b0 * kQ4KBytes, bytes, bar);
                }
            };
            issue(0);
            issue(1);
            float acc[4][NT];
            for (int item = 0; item < n_items; ++item) {
                const uint32_t slot = (gi + item) & 1u, par = ((gi + item) >> 1) & 1u;
                // (test stall: the warp's first wait is on a barrier that never completes)
                uint64_t* wbar = p.stall && gi + item == 0 ? &s_never : &s_bar[warp][slot];
                const bool have = ok && s_wait(wbar, wbar == &s_never ? 0u : par, p.wait_ns);
                if (have) waited = item + 1;
                if (ok && !have) {
                    ok = false;
                    if (lane == 0 && p.hdr) atomicExch(&p.hdr->status, (int)MOE_ERR_TIMEOUT);
                }
                const int u = u0 + warp + (item / ncd) * kSWarps, ch = item - (item / ncd) * ncd;
                if (ch == 0) {
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
                }
                const int b0 = ch * kBlocksI, nb = min(kBlocksI, nblk - b0);
                if constexpr (kWide) {
                    // lane = group ch * 32 + lane of the 4 rows (block lane / 4, quant group lane % 4)
                    if (have) {
                        const uint8_t* blk = ring + slot * kSSlotBytes + (lane >> 2) * kQ4KBytes;
                        const int c = lane & 3;
                        uint4 hd[4], q0[4], q1[4];
                        const bool live[4] = {true, true, true, true};
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint8_t* rb = blk + r * rs;
                            hd[r] = *reinterpret_cast<const uint4*>(rb);
                            q0[r] = *reinterpret_cast<const uint4*>(rb + 16 + 32 * c);
                            q1[r] = *reinterpret_cast<const uint4*>(rb + 32 + 32 * c);
                        }
                        qd4_group_math<NT, 4, 3>(hd, q0, q1, live, 0, ch * 32 + lane, GI, X, XS, nt, acc, nullptr);
                    }
                } else if (have && gl < 4 * nb) {
                    // rows 4 half .. 4 half + 3, group gl of the item: block gl / 4, quant group gl % 4
                    const uint8_t* blk = ring + slot * kSSlotBytes + (4 * half) * rs + (gl >> 2) * kQ4KBytes;
                    const int c = gl & 3;
                    uint4 hd[4], q0[4], q1[4];
                    const bool live[4] = {true, true, true, true};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint8_t* rb = blk + r * rs;
                        hd[r] = *reinterpret_cast<const uint4*>(rb);
                        q0[r] = *reinterpret_cast<const uint4*>(rb + 16 + 32 * c);
                        q1[r] = *reinterpret_cast<const uint4*>(rb + 32 + 32 * c);
                    }
                    qd4_group_math<NT, 4, 3>(hd, q0, q1, live, 0, b0 * 4 + gl, GI, X, XS, nt, acc, nullptr);
                }
                __syncwarp();
                issue(item + 2);
                if (ch == ncd - 1) {
                    if constexpr (kWide) {
                        constexpr int sh = qd_red_shift<NT>();
                        const float v = qd_warp_reduce_t<NT>(acc);
                        const int i = lane >> sh, r = i / NT, t = i - r * NT;
                        if ((lane & ((1 << sh) - 1)) == 0 && t < nt) p.out[(int64_t)(st + pb + t) * H + 4 * u + r] = v;
                    } else {
                        // the 16 lanes of a half: butterfly over gl, lane gl = 0 writes its 4 rows
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (t >= nt) break;                 // warp-uniform: the pass's tokens only
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                float v = acc[r][t];
#pragma unroll
                                for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                                if (gl == 0) p.out[(int64_t)(st + pb + t) * H + 8 * u + 4 * half + r] = v;
                            }
                        }
                    }
                }
            }
            // after a timeout: wait (bounded) for the copies this warp issued and never saw land
            if (!ok && lane == 0)
                for (int i = waited; i < issued; ++i) s_wait(&s_bar[warp][(gi + i) & 1u], ((gi + i) >> 1) & 1u, p.wait_ns);
            gi += ok ? n_items : 0;
            __syncwarp();
        }
        v0 = seg_end;
    }
}

template <int NT>
size_t seg_smem(int K) { return seg_align((size_t)NT * qd4_vec_bytes(K)) + (size_t)kSWarps * 2 * kSSlotBytes; }

constexpr size_t kSegSmemCap = 216 * 1024;          // + about 7 KB of static shared memory

int seg_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    }
    return n;
}

template <int NT>
cudaError_t seg_launch(bool gateup, const SegParams& p, cudaStream_t s) {
    const size_t smem = seg_smem<NT>(p.K);
    cudaError_t err;
    if (gateup) {
        auto* kern = p.vin_bf16 ? seg_gateup_kernel<NT, 2> : seg_gateup_kernel<NT, 3>;
        if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return err;
        kern<<<seg_sms(), kSThreads, smem, s>>>(p);
    } else {
        if (qd4_groups(p.K) % 32 == 0) {
            if ((err = cudaFuncSetAttribute(seg_down_kernel<NT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)smem)) != cudaSuccess)
                return err;
            seg_down_kernel<NT, true><<<seg_sms(), kSThreads, smem, s>>>(p);
        } else {
            if ((err = cudaFuncSetAttribute(seg_down_kernel<NT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)smem)) != cudaSuccess)
                return err;
            seg_down_kernel<NT, false><<<seg_sms(), kSThreads, smem, s>>>(p);
        }
    }
    return cudaGetLastError();
}

}  // namespace

bool seg_gemv_supported(int qtype, int E, int H, int I) {
    return qtype == MOE_Q4_K && E <= kSMaxE && H % kQ4KWeights == 0 && I % kQ4KWeights == 0 && H % 8 == 0 &&
           seg_smem<1>(H) <= kSegSmemCap && seg_smem<1>(I) <= kSegSmemCap;
}

cudaError_t launch_seg_gemv(bool gateup, const void* vin, bool vin_bf16, const int32_t* sorted_pairs,
                            const int32_t* offsets, int E, int k, int K, int rows, const uint8_t* w0, const uint8_t* w1,
                            int64_t expert_stride, float* out, WsHeader* hdr, int max_tokens, cudaStream_t s) {
    SegParams p{};
    p.vin = vin; p.vin_bf16 = vin_bf16 ? 1 : 0; p.sorted_pairs = sorted_pairs; p.offsets = offsets;
    p.E = E; p.k = k; p.K = K; p.rows = rows; p.w0 = w0; p.w1 = w1; p.expert_stride = expert_stride;
    p.out = out; p.hdr = hdr;
    const WaitCfg wc = wait_cfg();
    p.wait_ns = wc.limit_ns; p.stall = wc.stall;
    // tokens per staging pass: the largest of 8, 4, 2, 1 whose staged vectors fit, and not
    // more than one expert can hold
    const int cap = std::max(1, max_tokens);
    if (seg_smem<8>(K) <= kSegSmemCap && cap > 4) { p.nt_max = 8; return seg_launch<8>(gateup, p, s); }
    if (seg_smem<4>(K) <= kSegSmemCap && cap > 2) { p.nt_max = 4; return seg_launch<4>(gateup, p, s); }
    if (seg_smem<2>(K) <= kSegSmemCap && cap > 1) { p.nt_max = 2; return seg_launch<2>(gateup, p, s); }
    p.nt_max = 1;
    return seg_launch<1>(gateup, p, s);
}

}  // namespace moe
