// permute.cu -- group the token-expert pairs by expert.
//
// The pages' prompt path runs "each expert over all its tokens at once"
// ("bloomery V4.1 README", feature list, "Batched prompts"); that needs the
// pairs p = t*k + j grouped by their expert.  This file computes
//   offsets[e]        = #{p : id[p] < e}   (E+1 entries, offsets[E] = P)
//   sorted_pairs[...] = p in ascending (expert, p) order (a stable sort)
//   pair_pos[p]       = position of p in sorted_pairs
// in two steps: per-chunk histograms (the last CTA to finish scans them into
// offsets and per-chunk bases), then a stable scatter inside each chunk
// (warp match for the rank inside a warp, per-warp counts for the rank
// across warps).  A single chunk does both steps in one launch.

#include "internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = kPermuteChunk;  // one pair per thread

// Exclusive scan over n <= 1024 values held one per thread (threads >= n hold 0).
// Returns the exclusive prefix; *total receives the sum.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_tot[lane] = wi - w;          // exclusive prefix of the warp totals
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    return inc - v + warp_tot[warp];
}

__device__ __forceinline__ void raise_status(WsHeader* hdr, int code) {
    atomicCAS(&hdr->status, (int)MOE_OK, code);
}

// Shared memory: base[E], wcnt[32][E], plus small scan scratch.
template <bool kFused>
__global__ void __launch_bounds__(kThreads) permute_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                           int nchunks, int32_t* __restrict__ sorted_pairs,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ pair_pos, WsHeader* hdr,
                                                           int32_t* __restrict__ chunk_base, bool scatter,
                                                           unsigned long long* __restrict__ counts) {
    extern __shared__ int smem[];
    int* base = smem;                 // [E]
    int* wcnt = smem + E;             // [32][E]
    __shared__ int warp_tot[32];
    __shared__ int total;
    __shared__ bool is_last;
    const int c = blockIdx.x;
    const int p = c * kThreads + threadIdx.x;
    int e = -2;                       // -2: no pair here, -1: invalid id
    if (p < P) {
        e = ids[p];
        if (e < 0 || e >= E) {
            raise_status(hdr, MOE_ERR_DEVICE_CHECK);
            e = -1;
        }
    }
    if (!scatter) {
        // ---- step 1: histogram of this chunk
        for (int i = threadIdx.x; i < E; i += kThreads) base[i] = 0;
        __syncthreads();
        if (e >= 0) atomicAdd(&base[e], 1);
        __syncthreads();
        if (!kFused) {
            for (int i = threadIdx.x; i < E; i += kThreads) chunk_base[(int64_t)c * E + i] = base[i];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) is_last = (atomicAdd(&hdr->ticket, 1u) == (unsigned)(nchunks - 1));
            __syncthreads();
            if (!is_last) return;
            __threadfence();
        }
        // ---- last CTA: per-expert totals, offsets, per-chunk bases
        int tot = 0;
        if (threadIdx.x < E) {
            if (kFused) {
                tot = base[threadIdx.x];
            } else {
                for (int cc = 0; cc < nchunks; ++cc) {
                    const int64_t at = (int64_t)cc * E + threadIdx.x;
                    const int v = __ldcg(&chunk_base[at]);
                    chunk_base[at] = tot;        // prefix over earlier chunks
                    tot += v;
                }
            }
        }
        // the running routing histogram comes for free: these are the call's per-expert counts
        if (counts && tot > 0) atomicAdd(&counts[threadIdx.x], (unsigned long long)tot);
        // E <= 1024 = blockDim, so one value per thread.
        const int ex = block_exclusive_scan(tot, warp_tot, &total);
        if (threadIdx.x < E) {
            offsets[threadIdx.x] = ex;
            if (kFused) {
                base[threadIdx.x] = ex;
            } else {
                for (int cc = 0; cc < nchunks; ++cc) chunk_base[(int64_t)cc * E + threadIdx.x] += ex;
            }
        }
        if (threadIdx.x == 0) {
            offsets[E] = total;
            if (!kFused) hdr->ticket = 0u;
        }
        if (!kFused) return;
        __syncthreads();
    } else {
        for (int i = threadIdx.x; i < E; i += kThreads) base[i] = chunk_base[(int64_t)c * E + i];
    }
    // ---- step 2: stable scatter of this chunk
    for (int i = threadIdx.x; i < 32 * E; i += kThreads) wcnt[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
        int pos = base[e] + rank;
        for (int w = 0; w < warp; ++w) pos += wcnt[w * E + e];
        sorted_pairs[pos] = p;
        pair_pos[p] = pos;
    } else if (e == -1) {
        pair_pos[p] = -1;
    }
}

size_t smem_bytes(int E) { return (size_t)33 * E * sizeof(int); }

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

size_t permute_scratch_bytes(int T, int k, int E) {
    const int64_t P = (int64_t)T * k;
    const int64_t nchunks = (P + kPermuteChunk - 1) / kPermuteChunk;
    return align_up((size_t)(nchunks > 1 ? nchunks : 1) * E * sizeof(int32_t), 256);
}

cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* sorted_pairs,
                           int32_t* offsets, int32_t* pair_pos, WsHeader* hdr, int32_t* chunk_base,
                           cudaStream_t s, unsigned long long* counts) {
    const int P = T * k;
    if (P == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
    const int nchunks = (P + kPermuteChunk - 1) / kPermuteChunk;
    const size_t sm = smem_bytes(E);
    cudaError_t err;
    if (nchunks == 1) {
        if ((err = set_smem(permute_kernel<true>, sm)) != cudaSuccess) return err;
        permute_kernel<true><<<1, kThreads, sm, s>>>(ids, P, E, 1, sorted_pairs, offsets, pair_pos, hdr,
                                                     chunk_base, false, counts);
        return cudaGetLastError();
    }
    if ((err = set_smem(permute_kernel<false>, sm)) != cudaSuccess) return err;
    permute_kernel<false><<<nchunks, kThreads, sm, s>>>(ids, P, E, nchunks, sorted_pairs, offsets, pair_pos,
                                                        hdr, chunk_base, false, counts);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    permute_kernel<false><<<nchunks, kThreads, sm, s>>>(ids, P, E, nchunks, sorted_pairs, offsets, pair_pos,
                                                        hdr, chunk_base, true, nullptr);
    return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------
// moe_permute_noalloc: the same two-step permute, with its scratch (status
// word, arrival ticket, per-chunk expert bases) in a fixed device array that
// the library owns, so the caller passes only inputs and outputs.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int kNoallocMaxPairs = 65536;                            // T*k limit
constexpr int kNoallocChunks = kNoallocMaxPairs / kPermuteChunk;   // 64 chunks
constexpr size_t kNoallocWords = kHeaderBytes / sizeof(int32_t) + (size_t)kNoallocChunks * kMaxExperts;

// 256 B header + 64 chunks x 1024 experts x 4 B = 262,400 bytes, held by every
// GPU that loads the library until the process exits.
static __device__ __align__(256) int32_t g_permute_scratch[kNoallocWords];

// The device address of g_permute_scratch in the current context.  Host code cannot use the
// symbol itself as an address.  The lookup runs on every call: after the first call in a
// context (which may load the library's device code, so it must not run under stream capture)
// it is a host-side table lookup, and it stays right when the caller switches contexts or a
// context is destroyed and created again, where a cached address would go stale.
cudaError_t scratch_for_current_context(void** out) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (err != cudaSuccess) return err;
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const int32_t* topk_ids, int T, int k, int E, int32_t* sorted_pairs,
                                          int32_t* offsets, int32_t* pair_pos, moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || k < 1 || E < 1 || E > kMaxExperts) return report(MOE_ERR_INVALID_ARG, "bad T/k/E");
    if ((int64_t)T * k > kNoallocMaxPairs)
        return report(MOE_ERR_INVALID_ARG,
                      "moe_permute_noalloc: T*k exceeds its fixed scratch limit of 65536 pairs; "
                      "use moe_permute with a caller workspace");
    if (!offsets) return report(MOE_ERR_INVALID_ARG, "offsets is NULL");
    if (T > 0 && (!topk_ids || !sorted_pairs || !pair_pos)) return report(MOE_ERR_INVALID_ARG, "NULL array");
    void* scratch = nullptr;
    cudaError_t err = scratch_for_current_context(&scratch);
    if (err != cudaSuccess) return report(MOE_ERR_CUDA, "moe_permute_noalloc: scratch lookup failed");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(scratch);
    // status word and arrival ticket must start at zero on every call
    err = cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s);
    if (err != cudaSuccess) return report(MOE_ERR_CUDA, "moe_permute_noalloc: header reset failed");
    int32_t* chunk_base = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(scratch) + kHeaderBytes);
    err = launch_permute(topk_ids, T, k, E, sorted_pairs, offsets, pair_pos, hdr, chunk_base, s);
    if (err != cudaSuccess) return report(MOE_ERR_CUDA, "moe_permute_noalloc: kernel launch failed");
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// moe_expert_counts_add: the running routing histogram for callers of
// moe_permute (moe_layer keeps it inside its own permute).
// ---------------------------------------------------------------------------
namespace moe {
namespace {

__global__ void counts_add_kernel(const int32_t* __restrict__ offsets, int E, unsigned long long* __restrict__ counts) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < E) {
        const int n = offsets[e + 1] - offsets[e];
        if (n > 0) atomicAdd(&counts[e], (unsigned long long)n);
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_expert_counts_add(const int32_t* offsets, int E, unsigned long long* counts,
                                            moe_stream_t stream) {
    using namespace moe;
    if (E < 1 || E > kMaxExperts) return report(MOE_ERR_INVALID_ARG, "bad E");
    if (!offsets || !counts) return report(MOE_ERR_INVALID_ARG, "NULL array");
    counts_add_kernel<<<(E + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(offsets, E, counts);
    if (cudaGetLastError() != cudaSuccess) return report(MOE_ERR_CUDA, "moe_expert_counts_add: kernel launch failed");
    return MOE_OK;
}
