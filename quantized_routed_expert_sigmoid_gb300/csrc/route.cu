// route.cu -- router logits and top-k gate selection.
//
// The bloomery pages compare the engine's router top-k ids exactly against
// a CPU reference ("bloomery early V4.1 README", "Oracle sets against
// ik_llama.cpp"); they do not print the routing formula.  This file computes
//   logits[t,e] = sum_h x[t,h] * Wr[e,h]                   (fp32 accumulate)
// and then, per token, either
//   softmax       : top-k of the logits, gates = softmax over the chosen k
//   sigmoid-group : s = sigmoid(l), sel = s + bias, groups of E/G experts
//                   scored by the sum of their two best sel, the best
//                   topk_groups groups kept, top-k sel inside them,
//                   gates = scale * s / sum(s)  (bias excluded from gates).
// Ties go to the lower expert (group) id; ids are written in ascending order.
#include <float.h>
#include <math.h>

#include "internal.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void load4(const void* x, bool bf16, int64_t idx, float v[4]) {
    if (bf16) {
        const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(x) + idx);
        v[0] = __uint_as_float(raw.x << 16);
        v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
        v[2] = __uint_as_float(raw.y << 16);
        v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    } else {
        const float4 f = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + idx);
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
}

// Few tokens: one CTA per (expert, group of TT tokens); the 256 threads stripe
// the hidden dimension and reduce in a fixed order.
constexpr int kSmallTT = 4;

__global__ void __launch_bounds__(256) logits_small_kernel(const void* __restrict__ x, bool x_bf16, int T,
                                                           int H, const float* __restrict__ W, int E,
                                                           float* __restrict__ logits, WsHeader* hdr) {
    if (hdr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        hdr->status = MOE_OK;
        hdr->ticket = 0u;
    }
    const int e = blockIdx.x;
    const int t0 = blockIdx.y * kSmallTT;
    const int nt = min(kSmallTT, T - t0);
    float acc[kSmallTT] = {0.f, 0.f, 0.f, 0.f};
    const float* wrow = W + (int64_t)e * H;
    for (int h = threadIdx.x * 4; h < H; h += 256 * 4) {
        const float4 wv = __ldg(reinterpret_cast<const float4*>(wrow + h));
#pragma unroll
        for (int i = 0; i < kSmallTT; ++i) {
            if (i < nt) {
                float xv[4];
                load4(x, x_bf16, (int64_t)(t0 + i) * H + h, xv);
                acc[i] = fmaf(wv.x, xv[0], acc[i]);
                acc[i] = fmaf(wv.y, xv[1], acc[i]);
                acc[i] = fmaf(wv.z, xv[2], acc[i]);
                acc[i] = fmaf(wv.w, xv[3], acc[i]);
            }
        }
    }
    __shared__ float part[8][kSmallTT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < kSmallTT; ++i) {
        float v = acc[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) part[warp][i] = v;
    }
    __syncthreads();
    if (threadIdx.x < nt) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += part[w][threadIdx.x];
        logits[(int64_t)(t0 + threadIdx.x) * E + e] = s;
    }
}

// Many tokens: a 64x64 (tokens x experts) tile per CTA, 4x4 per thread.
__global__ void __launch_bounds__(256) logits_tiled_kernel(const void* __restrict__ x, bool x_bf16, int T,
                                                           int H, const float* __restrict__ W, int E,
                                                           float* __restrict__ logits, WsHeader* hdr) {
    if (hdr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        hdr->status = MOE_OK;
        hdr->ticket = 0u;
    }
    __shared__ float As[32][64 + 4];
    __shared__ float Bs[32][64 + 4];
    const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int h0 = 0; h0 < H; h0 += 32) {
        // 64 rows x 32 columns of each operand, 8 elements per thread (two float4 loads).
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int idx = threadIdx.x + r * 256;      // 0..511 -> (row, col4)
            const int row = idx >> 3, c4 = (idx & 7) * 4;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (t0 + row < T) load4(x, x_bf16, (int64_t)(t0 + row) * H + h0 + c4, v);
            As[c4 + 0][row] = v[0]; As[c4 + 1][row] = v[1]; As[c4 + 2][row] = v[2]; As[c4 + 3][row] = v[3];
            float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e0 + row < E) wv = __ldg(reinterpret_cast<const float4*>(W + (int64_t)(e0 + row) * H + h0 + c4));
            Bs[c4 + 0][row] = wv.x; Bs[c4 + 1][row] = wv.y; Bs[c4 + 2][row] = wv.z; Bs[c4 + 3][row] = wv.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < 32; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) logits[(int64_t)t * E + e] = acc[i][j];
        }
    }
}

constexpr int kTopkWarps = 4;

// One warp per token.  Shared memory per warp: sel[E] and s[E].
__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(RouteCfgDev c, const float* __restrict__ logits,
                                                               const float* __restrict__ bias, int T,
                                                               int32_t* __restrict__ ids, float* __restrict__ wout,
                                                               WsHeader* hdr) {
    extern __shared__ float sm[];
    if (hdr && blockIdx.x == 0 && threadIdx.x == 0) {
        hdr->status = MOE_OK;
        hdr->ticket = 0u;
    }
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kTopkWarps + warp;
    if (t >= T) return;
    float* sel = sm + (size_t)warp * 2 * c.E;
    warp_topk(c, logits + (int64_t)t * c.E, bias, sel, sel + c.E, ids + (int64_t)t * c.k, wout + (int64_t)t * c.k);
}

}  // namespace

cudaError_t launch_router_logits(const void* x, bool x_bf16, int T, int H, const float* W, int E,
                                 float* logits, WsHeader* clear_hdr, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    if (T < 128) {                                   // one CTA per (expert row, 4 tokens): enough CTAs
        dim3 grid(E, (T + kSmallTT - 1) / kSmallTT);
        logits_small_kernel<<<grid, 256, 0, s>>>(x, x_bf16, T, H, W, E, logits, clear_hdr);
    } else {
        dim3 grid((T + 63) / 64, (E + 63) / 64);
        logits_tiled_kernel<<<grid, 256, 0, s>>>(x, x_bf16, T, H, W, E, logits, clear_hdr);
    }
    return cudaGetLastError();
}

cudaError_t launch_topk(const moe_route_cfg& cfg, const float* logits, const float* bias, int T,
                        int32_t* ids, float* w, WsHeader* clear_hdr, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int E = cfg.n_experts;
    const size_t smem = (size_t)kTopkWarps * 2 * E * sizeof(float);
    // E <= 1024 keeps this at or below 32 KB: no opt-in needed.
    RouteCfgDev c;
    c.mode = (int)cfg.mode;
    c.E = E;
    c.k = cfg.top_k;
    c.G = cfg.mode == MOE_ROUTE_SIGMOID_GROUP ? cfg.n_groups : 1;
    c.Gk = cfg.mode == MOE_ROUTE_SIGMOID_GROUP ? cfg.topk_groups : 1;
    c.renorm = cfg.renormalize;
    c.scale = cfg.routed_scale;
    topk_kernel<<<(T + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, smem, s>>>(c, logits, bias, T, ids, w, clear_hdr);
    return cudaGetLastError();
}

}  // namespace moe
