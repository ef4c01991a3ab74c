// internal.cuh -- declarations shared by the kernel translation units of the
// GB300 MoE library.  Nothing here is part of the public C ABI
// (include/moe_gb300.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

// GGUF block geometry.
constexpr int kQ4KBytes = 144;     // fp16 d, fp16 dmin, 12 B scales/mins, 128 B quants
constexpr int kQ4KWeights = 256;
constexpr int kQ80Bytes = 34;      // fp16 d, 32 x int8
constexpr int kQ80Weights = 32;

// MOE_Q8_0_R row: the quants of its K/32 blocks, then their fp16 scales padded to 16 bytes.
__host__ __device__ inline int64_t q80r_row_bytes(int64_t K) {
    const int64_t nb = K / kQ80Weights;
    return 32 * nb + (2 * nb + 15) / 16 * 16;
}
// Bytes of one row of K weights stored as qtype (Q8_0, Q8_0_R or Q4_K).
__host__ __device__ inline int64_t q_row_bytes(int qtype, int64_t K) {
    if (qtype == MOE_Q4_K) return K / kQ4KWeights * kQ4KBytes;
    if (qtype == MOE_Q5_K) return K / 256 * 176;
    if (qtype == MOE_Q6_K) return K / 256 * 210;
    if (qtype == MOE_Q8_0_R) return q80r_row_bytes(K);
    return K / kQ80Weights * kQ80Bytes;
}

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kPermuteChunk = 1024;  // pairs per permute CTA

// Workspace header: a status word (MOE_OK or an error code raised on the
// device) and the arrival ticket of the permute's last-block scan.
struct WsHeader {
    int32_t status;
    uint32_t ticket;
    uint32_t route_ready;    // chained decode: the routing is in the workspace (cleared by the logits kernel)
};
constexpr size_t kHeaderBytes = 256;


inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bounded device-side waits.  Every wait on an mbarrier (bulk copies, TMA, MMA completion)
// gives up after limit_ns, records MOE_ERR_TIMEOUT in the status word, waits (again within
// limit_ns) for the copies its CTA still has in flight and returns.  stall = 1 is a test
// setting: the first wait of the chained, segmented and tensor-core kernels then waits on a
// barrier that nothing completes, so that this path runs.  Set by moe_debug_set_waits.
struct WaitCfg {
    uint64_t limit_ns;
    int stall;
};
constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // 2 s: far above any legitimate wait
WaitCfg wait_cfg();
// Timing hook of the chained decode kernels (moe_debug_set_stamps): a device buffer of
// kStampBytes, or NULL (off).
constexpr size_t kStampBytes = (size_t)3 * 256 * 8 * sizeof(uint64_t);
void* debug_stamps();

// Records `msg` as this host thread's moe_last_error() text and returns `st`.
moe_status report(moe_status st, const char* msg);

// ---------------------------------------------------------------- weights
// Q8_0 [n_rows][K] (34-byte blocks) -> the MOE_Q8_0_R row layout, one launch.
cudaError_t launch_q80_repack(const uint8_t* src, int64_t src_stride, int E, int64_t rows, int64_t K, uint8_t* dst,
                              cudaStream_t s);

// ---------------------------------------------------------------- route
cudaError_t launch_router_logits(const void* x, bool x_bf16, int T, int H, const float* W, int E,
                                 float* logits, WsHeader* clear_hdr, cudaStream_t s);
// Router logits on the tensor cores (router_tc.cu): x bf16, W split into three bf16 parts
// in w3 (router_tc_split_bytes(H, E) of device memory).
bool router_tc_supported(int T, int H, int E, bool x_bf16);
size_t router_tc_split_bytes(int H, int E);
cudaError_t launch_router_tc(const void* x, int T, int H, const float* W, int E, float* logits, void* w3,
                             WsHeader* clear_hdr, cudaStream_t s);
cudaError_t launch_topk(const moe_route_cfg& cfg, const float* logits, const float* bias, int T,
                        int32_t* ids, float* w, WsHeader* clear_hdr, cudaStream_t s);

// ---------------------------------------------------------------- permute
size_t permute_scratch_bytes(int T, int k, int E);
// counts (nullable, [E]): the running routing histogram, += this call's per-expert pair counts
cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* sorted_pairs,
                           int32_t* offsets, int32_t* pair_pos, WsHeader* hdr, int32_t* chunk_base,
                           cudaStream_t s, unsigned long long* counts = nullptr);

// ---------------------------------------------------------------- decode GEMV experts
// One launch computes, for every active expert e and each of its pairs, either
//   GATEUP: h[i, r] = silu(Wg[e][r] . v_i) * (Wu[e][r] . v_i)      (rows r < I)
//   DOWN  : y[i, n] = Wd[e][n] . v_i                               (rows n < H)
// with v_i = x[sorted_pairs[i] / k] (GATEUP) or h[i] (DOWN).
struct GemvArgs {
    int qtype;                  // MOE_Q8_0 / MOE_Q4_K (MOE_Q8_0_R arrives as MOE_Q8_0 with q80r)
    bool q80r;                  // Q8_0 weights in the repacked row layout
    bool gateup;
    const uint8_t* w0;          // gate (GATEUP) or down (DOWN)
    const uint8_t* w1;          // up (GATEUP) or NULL
    int64_t expert_stride;      // bytes between experts
    int rows;                   // output rows per expert
    int K;                      // input length (row length in weights)
    const void* vin;            // x [T][K] (bf16/fp32) or h [P][K] fp32
    bool vin_bf16;
    const int32_t* sorted_pairs;// NULL = identity (one expert, every row in order)
    const int32_t* offsets;     // [E+1] or NULL
    int E, k;
    int n_pairs;                // P (or T for the identity case)
    float* out;                 // h [P][rows] or y [P][rows], fp32
};
cudaError_t launch_qgemv(const GemvArgs& a, cudaStream_t s);
// Routed experts' gate/up (h fp32 [P][I]) or down (y fp32 [P][H]) for a few tokens per
// expert: persistent CTAs over contiguous unit ranges, bulk-copy ring (gemv_seg.cu).
bool seg_gemv_supported(int qtype, int E, int H, int I);
cudaError_t launch_seg_gemv(bool gateup, const void* vin, bool vin_bf16, const int32_t* sorted_pairs,
                            const int32_t* offsets, int E, int k, int K, int rows, const uint8_t* w0, const uint8_t* w1,
                            int64_t expert_stride, float* out, WsHeader* hdr, int max_tokens, cudaStream_t s);

// ---------------------------------------------------------------- combine, norm
cudaError_t launch_combine16(const __half* y_pairs, const float* w, const int32_t* pair_pos, int T, int k, int H,
                             const float* shared_out, bool accumulate, float* out, cudaStream_t s);
cudaError_t launch_combine(const float* y_pairs, const float* w, const int32_t* pair_pos, int T, int k,
                           int H, const float* shared_out, bool accumulate, float* out, cudaStream_t s);
cudaError_t launch_rmsnorm_bf16(const float* x, const float* gamma, int T, int H, float eps, void* u,
                                cudaStream_t s);

// ---------------------------------------------------------------- decode layer (T <= 4)
// The whole layer for a few tokens: shapes, weights and workspace buffers.
struct DecodeArgs {
    moe_route_cfg route;
    const float* Wr;
    const float* bias;
    const void* x;
    bool x_bf16;
    const float* norm_gamma;      // pre-norm inside the chain (x fp32 residual stream), or NULL
    float norm_eps;
    int T, H, I;
    int qtype;
    const uint8_t* wg;
    const uint8_t* wu;
    const uint8_t* wd;
    int64_t stride_gu, stride_d;
    int I_s, s_qtype;             // shared expert (s_qtype MOE_Q8_0_R arrives as MOE_Q8_0 with s_q80r)
    bool s_q80r;
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
    uint8_t* hq;                  // chain: every pair's h, staged (272 * I/64 bytes per pair)
    uint8_t* hq_s;                // chain: the Q4_K shared expert's h, staged (T vectors)
    float* out;
    bool accumulate;
    unsigned long long* counts;   // nullable [E]: += the call's per-expert pair counts
    WsHeader* hdr;
};
// The layer as three launches chained by programmatic dependent launch (decode_chain.cu).
bool decode_chain_supported(const DecodeArgs& a);
// evb / eva (nullable): events recorded around the gate/up launch.
cudaError_t launch_decode_chain(const DecodeArgs& a, cudaStream_t s, cudaEvent_t evb = nullptr,
                                cudaEvent_t eva = nullptr);

// ---------------------------------------------------------------- tensor-core grouped GEMM
// Expert FFN for many tokens per expert on tcgen05: gate/up + SwiGLU into an
// fp16 h, then down into fp32 y (row i = sorted position i, or token i in the
// identity mode used by a shared expert).
struct TcFfnArgs {
    int qtype;                  // MOE_Q4_K or MOE_Q8_0 (gate, up and down share it)
    bool q80r;                  // Q8_0 weights in the repacked row layout
    const uint8_t* wg;
    const uint8_t* wu;
    const uint8_t* wd;
    int64_t stride_gu, stride_d;
    int E, k, H, I, T;
    bool identity;              // one expert over all T tokens in order
    const void* x;              // [T][H] bf16 or fp32
    bool x_bf16;
    bool convert_x;             // write x16 from x first
    const int32_t* sorted_pairs;
    const int32_t* offsets;
    __half* x16;                // [T][H]
    __half* h16;                // [P][I]
    float* y;                   // [P][H] fp32, or
    __half* y16;                // [P][H] fp16 when set (the layer's combine reads it)
    int4* tb_list;              // token-block list (routed mode)
    WsHeader* hdr;
    cudaEvent_t ev_before_gateup, ev_after_gateup;   // optional timing events
};
size_t tc_tile_list_bytes(int T, int k, int E);
bool tc_supported(int qtype, int rows_gu, int K_gu);
cudaError_t launch_tc_expert_ffn(const TcFfnArgs& a, cudaStream_t s);

}  // namespace moe
