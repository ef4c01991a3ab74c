// route_common.cuh -- one token's top-k selection and gates, done by one warp.
// Shared by the routing kernel and the fused decode kernel (both compute the
// same definition; see route.cu for it).
#pragma once

#include <math.h>

#include "internal.cuh"

namespace moe {

// (value, id) arg-max across the warp: larger value first, then lower id.
__device__ __forceinline__ void warp_argmax(float& v, int& id) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oid = __shfl_xor_sync(0xffffffffu, id, o);
        if (ov > v || (ov == v && oid < id)) { v = ov; id = oid; }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

struct RouteCfgDev {
    int mode, E, k, G, Gk, renorm;
    float scale;
};

// Sigmoid-group scoring of one token (whole warp): sv[e] = s = 1/(1+exp(-l)), sel[e] = s + b
// for the experts of the topk_groups best groups (a group scored by the sum of its two largest
// sel, ties to the lower group), sel[e] = -inf outside them.  Kept out of line: the chained
// decode kernel inlines only the softmax scoring, the common case there.
static __device__ __noinline__ void warp_scores_sigmoid_group(const RouteCfgDev& c, const float* lrow, const float* bias,
                                                       float* sel, float* sv) {
    const int lane = threadIdx.x & 31;
    const int E = c.E;
    for (int e0 = 0; e0 < E; e0 += 8 * 32) {
        float l[8], b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = e0 + i * 32 + lane;
            l[i] = e < E ? __ldcg(lrow + e) : 0.f;
            b[i] = (bias && e < E) ? __ldg(bias + e) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = e0 + i * 32 + lane;
            if (e < E) {
                const float s = 1.0f / (1.0f + expf(-l[i]));
                sv[e] = s;
                sel[e] = s + b[i];
            }
        }
    }
    __syncwarp();
    const int per = E / c.G;
    float gs = -INFINITY;
    if (lane < c.G) {
        float b1 = -INFINITY, b2 = -INFINITY;
        for (int i = 0; i < per; ++i) {
            const float v = sel[lane * per + i];
            if (v > b1) { b2 = b1; b1 = v; } else if (v > b2) { b2 = v; }
        }
        gs = per >= 2 ? b1 + b2 : b1;
    }
    uint32_t keep = 0u;
    for (int r = 0; r < c.Gk; ++r) {
        float v = (lane < c.G && !((keep >> lane) & 1u)) ? gs : -INFINITY;
        int id = (lane < c.G && !((keep >> lane) & 1u)) ? lane : 0x7fffffff;
        warp_argmax(v, id);
        if (id < 32) keep |= 1u << id;
    }
    for (int e = lane; e < E; e += 32)
        if (!((keep >> (e / per)) & 1u)) sel[e] = -INFINITY;
    __syncwarp();
}

// The whole warp selects token `lrow`'s k experts and writes them in ascending id
// order to ids[0..k) with their gates w[0..k).  sel, sv: 2*E floats of per-warp
// shared memory.  lrow is read through L2 (it may have been written by other CTAs
// of the same grid).
template <int kSlots>
__device__ __forceinline__ void warp_topk_n(const RouteCfgDev& c, const float* lrow, const float* bias, float* sel,
                                            float* sv, int32_t* ids, float* w) {
    const int lane = threadIdx.x & 31;
    const int E = c.E, k = c.k;
    const bool sig = (c.mode == MOE_ROUTE_SIGMOID_GROUP);
    if (sig) {
        warp_scores_sigmoid_group(c, lrow, bias, sel, sv);
    } else {
        // all loads of a chunk are issued before its stores (the shared-memory stores could
        // otherwise alias the global loads and serialise one L2 round trip per element)
        for (int e0 = 0; e0 < E; e0 += 8 * 32) {
            float l[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + i * 32 + lane;
                l[i] = e < E ? __ldcg(lrow + e) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + i * 32 + lane;
                if (e < E) sv[e] = sel[e] = l[i];
            }
        }
        __syncwarp();
    }
    // k rounds of arg-max over sel (larger first, ties to the lower id); lane r keeps the
    // r-th pick.  Scores become order-preserving unsigned keys (-0 folded into +0) held in
    // registers (element lane + 32*i in slot i); a round is a lane-local scan and two warp
    // reductions, and a taken expert's key becomes 0, below every score.
    uint32_t kv[kSlots];                              // E <= 32 * kSlots
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
        const int e = lane + 32 * i;
        uint32_t key = 0u;
        if (e < E) {
            const uint32_t u = __float_as_uint(sel[e] + 0.0f);
            key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
        }
        kv[i] = key;
    }
    int my_id = 0x7fffffff;
#pragma unroll 1                                      // rounds are serial: no gain from copies
    for (int r = 0; r < k; ++r) {
        uint32_t best = 0u;
        int bid = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kSlots; ++i)
            if (kv[i] > best) { best = kv[i]; bid = lane + 32 * i; }   // ascending id: ties keep the lower
        const uint32_t top = __reduce_max_sync(0xffffffffu, best);
        int id = (int)__reduce_min_sync(0xffffffffu, best == top ? (uint32_t)bid : 0x7fffffffu);
        if (id >= E) id = 0;
#pragma unroll
        for (int i = 0; i < kSlots; ++i)
            if (lane + 32 * i == id) kv[i] = 0u;
        if (lane == r) my_id = id;
    }
    const float my_val = lane < k ? sv[my_id] : 0.f;
    float num = 0.f, den;
    if (sig) {
        num = lane < k ? my_val : 0.f;
        den = c.renorm ? warp_sum(num) : 1.0f;
    } else {
        const float m = __shfl_sync(0xffffffffu, my_val, 0);  // the first pick is the largest logit
        num = lane < k ? expf(my_val - m) : 0.f;
        if (c.renorm) {
            den = warp_sum(num);
        } else {
            float part = 0.f;
            for (int e = lane; e < E; e += 32) part += expf(__ldcg(lrow + e) - m);
            den = warp_sum(part);
        }
    }
    int rank = 0;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        const int oid = __shfl_sync(0xffffffffu, my_id, j);
        rank += (oid < my_id) ? 1 : 0;
    }
    if (lane < k) {
        ids[rank] = my_id;
        w[rank] = c.scale * (num / den);
    }
    __syncwarp();
}

// Out-of-line instances for the wider key arrays (E > 128).
static __device__ __noinline__ void warp_topk_256(const RouteCfgDev& c, const float* lrow, const float* bias, float* sel,
                                           float* sv, int32_t* ids, float* w) {
    warp_topk_n<8>(c, lrow, bias, sel, sv, ids, w);
}
static __device__ __noinline__ void warp_topk_1024(const RouteCfgDev& c, const float* lrow, const float* bias, float* sel,
                                            float* sv, int32_t* ids, float* w) {
    warp_topk_n<32>(c, lrow, bias, sel, sv, ids, w);
}

// Same, with the key registers sized for E (E <= 1024); E <= 128 inline.
__device__ __forceinline__ void warp_topk(const RouteCfgDev& c, const float* lrow, const float* bias, float* sel,
                                          float* sv, int32_t* ids, float* w) {
    if (c.E <= 128) warp_topk_n<4>(c, lrow, bias, sel, sv, ids, w);
    else if (c.E <= 256) warp_topk_256(c, lrow, bias, sel, sv, ids, w);
    else warp_topk_1024(c, lrow, bias, sel, sv, ids, w);
}

}  // namespace moe
