// router_tc.cu -- router logits for many tokens on the tensor cores.
//
// l[t, e] = sum_h x[t, h] * W_r[e, h] with x bf16 (exact) and W_r fp32.  W_r is split
// exactly into three bf16 parts, W = hi + mid + lo (hi = bf16(W), mid = bf16(W - hi),
// lo = bf16(W - hi - mid): 24 significant bits together), so every product of a part
// with a bf16 x is exact in fp32 and the three MMAs accumulate the fp32 dot product.
// Tile: M = 128 tokens (A = x rows) x N = 32 experts (B = the three parts' rows), K in
// steps of 64; 128 producer threads stage A and B with cp.async into 128-byte-swizzled
// K-major tiles (6 stages, loads three k-steps ahead, so a stage is refilled three steps
// after the MMAs that read it were issued), one thread issues the 12 MMAs of a k-step (4
// substeps x 3 parts) into one TMEM accumulator, the producers then read it and write l fp32.
// When T/128 x E/32 tiles leave most SMs idle (few tokens, or a long K), K is split over S
// CTAs per tile (grid z); each writes its fp32 partial sums and a second launch adds the S
// partials in split order, so a replay gives the same bits.
#include <algorithm>

#include "internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kRM = 128, kRN = 32, kRK = 64;     // N = 32: T/128 x E/32 CTAs fill the GPU
constexpr int kRStages = 6;                       // loads go 3 k-steps ahead; 3 steps of slack for the MMAs
constexpr int kRProducers = 128;
constexpr int kRThreads = kRProducers + 32;
constexpr int kRAStage = kRM * 128;               // x tile
constexpr int kRBStage = 3 * kRN * 128;           // three parts' tiles
constexpr int kRStageBytes = kRAStage + kRBStage;

struct RouterTcParams {
    const __nv_bfloat16* x;          // [T][H]
    const __nv_bfloat16* w3;         // [3][E][H]: hi, mid, lo
    float* logits;                   // [T][E], or the split's partial sums [S][T][E] when S > 1
    int T, H, E;
    int nsplit;                      // S: K splits per tile (grid z)
    WsHeader* clear_hdr;
    uint64_t wait_ns;                // limit of every bounded wait
};

__global__ void router_split_kernel(const float* __restrict__ W, int64_t n, __nv_bfloat16* __restrict__ w3) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float w = W[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);               // exact
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);             // exact
    w3[i] = hi;
    w3[n + i] = mid;
    w3[2 * n + i] = __float2bfloat16_rn(r2);
}

__global__ void __launch_bounds__(kRThreads, 1) router_tc_kernel(const __grid_constant__ RouterTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t full[kRStages], empty[kRStages], accf;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_s;
    volatile int* abort_flag = &abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kRM, e0 = blockIdx.y * kRN;
    // this CTA's k-steps: kb0 .. kb0 + nk - 1 of the H / 64
    const int nk_all = p.H / kRK, z = blockIdx.z;
    const int kb0 = (int)((int64_t)nk_all * z / p.nsplit);
    const int nk = (int)((int64_t)nk_all * (z + 1) / p.nsplit) - kb0;
    float* const out = p.logits + (size_t)z * p.T * p.E;
    if (tid == 0) {
        for (int i = 0; i < kRStages; ++i) { mbar_init(&full[i], kRProducers); mbar_init(&empty[i], 1); }
        mbar_init(&accf, 1);
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (p.clear_hdr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
            p.clear_hdr->status = MOE_OK;
            p.clear_hdr->ticket = 0u;
        }
    }
    if (warp == kRProducers / 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_slot)),
                     "n"(kRN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = tmem_slot;

    if (warp < kRProducers / 32) {
        // ---- producers: stage k-step kb into stage kb % 4 (rows past T / E are zero-filled)
        auto issue = [&](int kb) {
            uint8_t* st = smem + (kb % kRStages) * kRStageBytes;
            const int ch = tid & 7;
#pragma unroll
            for (int i = 0; i < kRM / 16; ++i) {                   // A: 128 rows x 8 chunks
                const int r = (tid >> 3) + 16 * i, t = t0 + r;
                const bool ok = t < p.T;
                cp_async16(st + swz(r, ch), p.x + (ok ? (int64_t)t * p.H + (kb0 + kb) * kRK + ch * 8 : 0), ok ? 16u : 0u);
            }
#pragma unroll
            for (int i = 0; i < 3 * kRN / 16; ++i) {               // B: 3 parts x kRN rows x 8 chunks
                const int rr = (tid >> 3) + 16 * i, part = rr / kRN, r = rr - part * kRN, e = e0 + r;
                const bool ok = e < p.E;
                const __nv_bfloat16* src =
                    p.w3 + (ok ? ((int64_t)part * p.E + e) * p.H + (kb0 + kb) * kRK + ch * 8 : 0);
                cp_async16(st + kRAStage + part * kRN * 128 + swz(r, ch), src, ok ? 16u : 0u);
            }
        };
        for (int kb = 0; kb < 3; ++kb) {                          // always three groups: the waits count them
            if (kb < nk) issue(kb);
            cp_commit();
        }
        for (int kb = 0; kb < nk; ++kb) {
            if (kb + 3 < nk) {
                // stage (kb + 3) % kRStages was last read by MMA(kb + 3 - kRStages)
                const int prev = kb + 3 - kRStages;
                if (prev >= 0 && !mbar_wait(&empty[(kb + 3) % kRStages], (prev / kRStages) & 1, abort_flag, p.wait_ns)) break;
                issue(kb + 3);
            }
            cp_commit();
            cp_wait<3>();                                          // k-step kb has landed
            fence_async_smem();
            mbar_arrive(&full[kb % kRStages]);
        }
        cp_wait_all();
        // ---- epilogue: lane = token row, 64 expert columns
        if (!*abort_flag && mbar_wait(&accf, 0, abort_flag, p.wait_ns)) {
            tc_after();
            const int t = t0 + warp * 32 + lane;
#pragma unroll
            for (int c16 = 0; c16 < kRN; c16 += 16) {
                uint32_t a[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c16, a);
                tmem_ld_wait();
                if (t < p.T) {
                    float* dst = out + (int64_t)t * p.E + e0 + c16;
                    if (e0 + c16 + 16 <= p.E) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4*>(dst + j) = make_float4(__uint_as_float(a[j]), __uint_as_float(a[j + 1]),
                                                                              __uint_as_float(a[j + 2]), __uint_as_float(a[j + 3]));
                    } else {
                        for (int j = 0; j < 16 && e0 + c16 + j < p.E; ++j) dst[j] = __uint_as_float(a[j]);
                    }
                }
            }
        }
    } else {
        // ---- MMA issuer
        const uint32_t idesc = idesc_mma(kRM, kRN, true);
        bool issued = false;
        for (int kb = 0; kb < nk; ++kb) {
            if (!mbar_wait(&full[kb % kRStages], (kb / kRStages) & 1, abort_flag, p.wait_ns)) break;
            tc_after();
            if (lane == 0) {
                const uint32_t a0 = su32(smem + (kb % kRStages) * kRStageBytes);
                const uint32_t b0 = a0 + kRAStage;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int part = 0; part < 3; ++part)
                        mma_f16(tmem, sdesc(a0 + 32 * kk), sdesc(b0 + part * kRN * 128 + 32 * kk), idesc,
                                (kb | kk | part) != 0);
                mma_commit(&empty[kb % kRStages]);
                if (kb == nk - 1) mma_commit(&accf);
            }
            issued = true;
            __syncwarp();
        }
        if (issued && *abort_flag) {
            // let every issued MMA finish before the accumulator is freed
            if (lane == 0) mma_commit(&accf);
            __syncwarp();
            mbar_wait_for(&accf, 0, p.wait_ns);
        }
    }
    if (*abort_flag && tid == 0 && p.clear_hdr) atomicCAS(&p.clear_hdr->status, (int)MOE_OK, (int)MOE_ERR_TIMEOUT);
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == kRProducers / 32)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kRN) : "memory");
}

// logits = the S partial sums, added in split order (one thread per logit)
__global__ void router_reduce_kernel(const float* __restrict__ partial, int64_t n, int S, float* __restrict__ logits) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = partial[i];
    for (int z = 1; z < S; ++z) v += partial[(size_t)z * n + i];
    logits[i] = v;
}

// Partial sums of a split launch: S * T_pad * E_pad fp32 with S * (T_pad / 128) * (E_pad / 32)
// <= 152 tiles, so at most 152 * 128 * 32 * 4 bytes whatever T and E are.
constexpr size_t kRPartialCap = (size_t)152 * kRM * kRN * sizeof(float);

int router_sms() {
    static int n = 0;
    if (n <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            n = 0;
    }
    return n > 0 ? n : 152;
}

// K splits for a launch of T tokens: doubled while the split tiles still fit the SMs once, each
// split keeps at least four k-steps, and the partial sums fit their buffer.
int router_splits(int T, int H, int E) {
    const int tiles = ((T + kRM - 1) / kRM) * ((E + kRN - 1) / kRN);
    const int sms = std::min(router_sms(), 152);
    int S = 1;
    while (S < 8 && tiles * 2 * S <= sms && H / kRK >= 4 * 2 * S &&
           (size_t)2 * S * T * E * sizeof(float) <= kRPartialCap)
        S *= 2;
    return S;
}

}  // namespace

bool router_tc_supported(int T, int H, int E, bool x_bf16) {
    return x_bf16 && T > 32 && H % kRK == 0 && E % 4 == 0 && E <= 1024;
}

// the three bf16 parts of W, then room for the partial sums of a split launch
size_t router_tc_split_bytes(int H, int E) {
    return align_up((size_t)3 * E * H * sizeof(__nv_bfloat16), 256) + kRPartialCap;
}

cudaError_t launch_router_tc(const void* x, int T, int H, const float* W, int E, float* logits, void* w3,
                             WsHeader* clear_hdr, cudaStream_t s) {
    const int64_t n = (int64_t)E * H;
    __nv_bfloat16* parts = static_cast<__nv_bfloat16*>(w3);
    router_split_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(W, n, parts);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const size_t smem = (size_t)kRStages * kRStageBytes + 1024;
    if ((err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return err;
    const int S = router_splits(T, H, E);
    float* partial = reinterpret_cast<float*>(static_cast<uint8_t*>(w3) + align_up((size_t)3 * n * sizeof(__nv_bfloat16), 256));
    RouterTcParams p{};
    p.x = static_cast<const __nv_bfloat16*>(x);
    p.w3 = parts;
    p.logits = S > 1 ? partial : logits;
    p.T = T; p.H = H; p.E = E;
    p.nsplit = S;
    p.clear_hdr = clear_hdr;
    p.wait_ns = wait_cfg().limit_ns;
    router_tc_kernel<<<dim3((T + kRM - 1) / kRM, (E + kRN - 1) / kRN, S), kRThreads, smem, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess || S == 1) return err;
    const int64_t nl = (int64_t)T * E;
    router_reduce_kernel<<<(unsigned)((nl + 255) / 256), 256, 0, s>>>(partial, nl, S, logits);
    return cudaGetLastError();
}

}  // namespace moe
