// combine.cu -- gate-weighted combine of the expert outputs, and the RMSNorm
// that sits between stacked layers.
//
//   out[t,n] = ((sum_{j<k} w[t,j] * y[pair_pos[t*k+j], n]) + shared[t,n]) + old out[t,n]
// in that fixed order (the shared expert unweighted; the old value only when
// accumulating, i.e. as a residual add), and
//   u[t,h] = bf16_rne( x[t,h] / sqrt(mean_h x[t,:]^2 + eps) * gamma[h] ).
// The pages run one captured CUDA graph per decode step ("bloomery README
// 0.3.1", "Why it is fast") and require graph replay to equal eager
// execution bit for bit ("bloomery early V4.1 README", "Bit gates"); both
// kernels are deterministic for that reason.
#include "internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __half* p) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// y fp32 (GEMV paths) or fp16 (tensor-core path); the sum is fp32 either way
template <typename YT>
__global__ void __launch_bounds__(256) combine_kernel(const YT* __restrict__ y, const float* __restrict__ w,
                                                      const int32_t* __restrict__ pair_pos, int k, int H,
                                                      const float* __restrict__ shared, bool accumulate,
                                                      float* __restrict__ out) {
    const int t = blockIdx.x;
    const int n = (blockIdx.y * 256 + threadIdx.x) * 4;
    if (n >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int pp = pair_pos[(int64_t)t * k + j];
        if (pp < 0) continue;
        const float wj = w[(int64_t)t * k + j];
        const float4 v = load4(y + (int64_t)pp * H + n);
        acc.x = fmaf(wj, v.x, acc.x);
        acc.y = fmaf(wj, v.y, acc.y);
        acc.z = fmaf(wj, v.z, acc.z);
        acc.w = fmaf(wj, v.w, acc.w);
    }
    if (shared) {
        const float4 s = *reinterpret_cast<const float4*>(shared + (int64_t)t * H + n);
        acc.x += s.x; acc.y += s.y; acc.z += s.z; acc.w += s.w;
    }
    float4* o = reinterpret_cast<float4*>(out + (int64_t)t * H + n);
    if (accumulate) {
        const float4 old = *o;
        acc.x += old.x; acc.y += old.y; acc.z += old.z; acc.w += old.w;
    }
    *o = acc;
}

__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float* __restrict__ x,
                                                           const float* __restrict__ gamma, int H, float eps,
                                                           __nv_bfloat16* __restrict__ u) {
    const int t = blockIdx.x;
    const float* row = x + (int64_t)t * H;
    float ss = 0.f;
    for (int h = threadIdx.x * 4; h < H; h += 1024) {
        const float4 v = *reinterpret_cast<const float4*>(row + h);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    __shared__ float part[8];
    __shared__ float scale;
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int i = 0; i < 8; ++i) s += part[i];
        scale = 1.0f / sqrtf(s / (float)H + eps);
    }
    __syncthreads();
    const float r = scale;
    for (int h = threadIdx.x * 4; h < H; h += 1024) {
        const float4 v = *reinterpret_cast<const float4*>(row + h);
        const float4 g = *reinterpret_cast<const float4*>(gamma + h);
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x * r * g.x, v.y * r * g.y);
        __nv_bfloat162 b = __floats2bfloat162_rn(v.z * r * g.z, v.w * r * g.w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&a);
        packed.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(u + (int64_t)t * H + h) = packed;
    }
}

}  // namespace

cudaError_t launch_combine(const float* y_pairs, const float* w, const int32_t* pair_pos, int T, int k,
                           int H, const float* shared_out, bool accumulate, float* out, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    dim3 grid(T, (H / 4 + 255) / 256);
    combine_kernel<float><<<grid, 256, 0, s>>>(y_pairs, w, pair_pos, k, H, shared_out, accumulate, out);
    return cudaGetLastError();
}

cudaError_t launch_combine16(const __half* y_pairs, const float* w, const int32_t* pair_pos, int T, int k, int H,
                             const float* shared_out, bool accumulate, float* out, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    dim3 grid(T, (H / 4 + 255) / 256);
    combine_kernel<__half><<<grid, 256, 0, s>>>(y_pairs, w, pair_pos, k, H, shared_out, accumulate, out);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bf16(const float* x, const float* gamma, int T, int H, float eps, void* u,
                                cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    rmsnorm_bf16_kernel<<<T, 256, 0, s>>>(x, gamma, H, eps, reinterpret_cast<__nv_bfloat16*>(u));
    return cudaGetLastError();
}

}  // namespace moe
