/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) routed-expert MoE layer library.
 *
 * The layer: router logits -> softmax or sigmoid(+bias, group-limited) top-k
 * with renormalised gates -> token-to-expert permutation with per-expert
 * offsets -> per-expert SwiGLU FFN over GGUF block-quantized weights (Q4_K,
 * Q8_0) -> gate-weighted combine, plus an optional unweighted shared expert.
 *
 * Where the operation comes from.  The bloomery pages describe an MoE engine
 * whose routed experts run on the card over the stored GGUF quantization
 * ("bloomery README 0.3.1", Status table, "Quant types" row), whose prompt
 * batches run each expert over all its tokens at once ("bloomery V4.1
 * README", feature list, "Batched prompts"), whose decode step is one CUDA
 * graph ("bloomery README 0.3.1", "Why it is fast"), and whose router top-k
 * ids are compared exactly against a CPU reference ("bloomery early V4.1
 * README", "Oracle sets against ik_llama.cpp").  The pages print none of the
 * arithmetic; each call below states the definition it implements.
 *
 * Conventions for every call
 *  - Pointers marked (device) are CUDA device pointers owned by the caller;
 *    (host) pointers are read during the call only.  The library never
 *    allocates device memory and never synchronizes (except the two
 *    *_read_device_status calls): each call enqueues kernels on `stream` and
 *    returns, so every call can be captured in a CUDA graph.
 *  - Arguments are validated on the host before any launch; a rejected call
 *    launches nothing and returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE.  A failed launch returns MOE_ERR_CUDA.  The reason
 *    is readable with moe_last_error() (per host thread).
 *  - Weight, activation, output and workspace pointers must be 16-byte
 *    aligned; int32/fp32 routing arrays need 4-byte alignment.
 *  - Weight matrices are GGUF block rows: [rows][cols / block] blocks, the
 *    blocks running along the input dimension `cols`.  Q8_0: 34 bytes per 32
 *    weights (fp16 d, 32 x int8 q; w = d*q).  Q4_K: 144 bytes per 256
 *    weights (fp16 d, fp16 dmin, 12 bytes of packed 6-bit scales/mins for 8
 *    sub-blocks of 32, 128 bytes of 4-bit q; w = d*sc_j*q - dmin*m_j).
 *    MOE_Q8_0_R: the same Q8_0 values in moe_weights_prepare's row layout.
 *    For gate/up: rows = I, cols = H.  For down: rows = H, cols = I.
 *    Expert e of a stacked tensor starts at data + e * expert_stride_bytes.
 *  - Token-expert pairs: p = t*k + j for token t and its j-th chosen expert.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or mode */
    MOE_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than the size query */
    MOE_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed */
    MOE_ERR_DEVICE_CHECK = 5,  /* a device-side check failed (see *_read_device_status) */
    MOE_ERR_TIMEOUT = 6        /* a bounded device-side wait ran out (see *_read_device_status) */
} moe_status;

/* MOE_Q8_0_R: Q8_0 weights after moe_weights_prepare -- per row of K weights, the int8
 * quants of its K/32 blocks (32 bytes each, in order), then their fp16 scales, padded to
 * a multiple of 16 bytes: 32*(K/32) + roundup16(2*(K/32)) bytes a row.
 * MOE_Q5_K: 176 bytes per 256 weights -- Q4_K's 16-byte header (fp16 d, fp16 dmin, 12 bytes
 * of 6-bit scales and mins), 32 bytes whose byte i holds in bit j the 16s digit of element i
 * of sub-block j, then Q4_K's 128 nibble bytes; q in [0, 31], w = d*sc_j*q - dmin*m_j.
 * MOE_Q6_K: 210 bytes per 256 weights -- 128 bytes of low nibbles, 64 bytes of 2-bit high
 * parts, 16 int8 scales (one per 16 weights), fp16 d; element 128h + 32r + l (r < 4) takes
 * the low (r < 2) or high (r >= 2) nibble of byte 64h + 32(r % 2) + l and bits 2r, 2r + 1 of
 * byte 128 + 32h + l, u = nibble + 16 * those bits, w = d * sc[element / 16] * (u - 32).
 * MOE_Q3_K: 110 bytes per 256 weights -- 32 bytes hmask, 64 bytes of 2-bit low parts, 12
 * bytes of sixteen 6-bit scales stored + 32, fp16 d; element 128h + 32r + l takes bits 2r,
 * 2r + 1 of byte 32 + 32h + l and bit 4h + r of byte l, q = low + 4 * bit - 4 in [-4, 3]; scale
 * j: low nibble of byte 96 + j (j < 8) or high nibble of byte 96 + j - 8, bits 4-5 from bits
 * 2(j / 4).. of byte 104 + j % 4; w = d * (s_j - 32) * q.
 * MOE_MXFP4: 17 bytes per 32 weights (OCP Microscaling) -- an E8M0 scale byte e, then 16 bytes
 * whose byte j holds the FP4 E2M1 element j (low nibble) and j + 16 (high nibble);
 * w = 2^(e - 127) * e2m1 (e = 255 is NaN).  cols must be a multiple of 128.
 * These are the public GGUF layouts; the pages list them among the card-expert types
 * ("bloomery README 0.3.1", Status table, "Quant types" row), and their large model keeps its
 * routed experts as Q3_K gate and up with a Q4_K down ("bloomery README 0.3.11", limits list;
 * desc.down may have another type than gate and up).  They run on the GEMV kernels at every T
 * (moe_layer_path reports MOE_PATH_GEMV). */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_Q8_0 = 2, MOE_Q4_K = 3, MOE_Q8_0_R = 4, MOE_Q5_K = 5,
               MOE_Q6_K = 6, MOE_Q3_K = 7, MOE_MXFP4 = 8 } moe_dtype;

typedef enum { MOE_ROUTE_SOFTMAX = 0, MOE_ROUTE_SIGMOID_GROUP = 1 } moe_route_mode;

/* One quantized weight tensor, possibly a stack of experts. */
typedef struct {
    moe_dtype qtype;             /* MOE_Q8_0, MOE_Q4_K, MOE_Q8_0_R, MOE_Q5_K, MOE_Q6_K, MOE_Q3_K or MOE_MXFP4 */
    const void* data;            /* (device) 16-byte aligned */
    int64_t rows, cols;          /* per expert; cols = input dimension */
    int64_t expert_stride_bytes; /* bytes from expert e to e+1 (multiple of 16) */
} moe_qmat;

typedef struct {
    moe_route_mode mode;
    int n_experts;               /* E, 1..1024 */
    int top_k;                   /* k, 1..min(E, 32) */
    int n_groups;                /* sigmoid mode: G divides E, G <= 32 (softmax: ignored) */
    int topk_groups;             /* sigmoid mode: groups kept, 1..G */
    float routed_scale;          /* gates are multiplied by this (1.0 = none) */
    int renormalize;             /* 1: gates renormalised over the chosen k */
} moe_route_cfg;

/* ---------------------------------------------------------------- weights */

/*
 * moe_weights_prepare -- one-time repack of a stored Q8_0 tensor (n_experts stacked
 * matrices) into MOE_Q8_0_R, the layout the kernels stream with 16-byte loads: a GGUF
 * Q8_0 block is 34 bytes, so its quants never start on a 16-byte boundary.  The values
 * are unchanged (w = d*q of the same bytes); only their place moves.  The pages' large
 * model stores its shared experts in Q8_0 ("bloomery early V4.1 README", model file
 * notes; "bloomery V4.1 README", quant-mix notes); this call lets those be read at the
 * rate of the Q4_K experts.
 *   in_out (host): the tensor to repack (qtype MOE_Q8_0, data device, 16-byte aligned,
 *     rows, cols = K a multiple of 32, expert_stride_bytes >= rows * 34 * K/32 when
 *     n_experts > 1).  On success it is rewritten to describe the repacked tensor:
 *     qtype MOE_Q8_0_R, data = dst, expert_stride_bytes = rows * row bytes.  A MOE_Q4_K
 *     tensor (and a MOE_Q5_K, MOE_Q6_K, MOE_Q3_K or MOE_MXFP4 one) is used as stored: in_out is left unchanged and
 *     nothing is written.
 *   dst (device, 16-byte aligned): at least moe_weights_prepare_size() bytes, owned by
 *     the caller; it must not overlap the source.
 * One kernel on `stream`; the source may be freed once the stream has passed it.
 */
moe_status moe_weights_prepare_size(const moe_qmat* in, int n_experts, size_t* bytes);
moe_status moe_weights_prepare(moe_qmat* in_out, int n_experts, void* dst, size_t dst_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- steps */

/*
 * moe_route -- router logits and top-k gates for T tokens.
 *   logits[t,e] = sum_h x[t,h] * W_router[e,h]          (fp32 accumulate)
 *   softmax mode: the k largest logits (ties: lower id); gates = softmax over
 *     those k (renormalize=1) or softmax over all E at those ids (0).
 *   sigmoid-group mode: s = 1/(1+exp(-l)), sel = s + bias; groups of E/G
 *     consecutive experts scored by the sum of their two largest sel; keep
 *     the topk_groups best groups (ties: lower group); the k best sel inside
 *     them; gates = s_j / sum s (renormalize=1) or s_j; the bias never enters
 *     a gate.  Gates are then multiplied by routed_scale.
 * Chosen ids are written in ascending expert id per token.
 * Pages: the router's top-k ids are integer outputs that an engine must
 * reproduce exactly outside tie bands ("bloomery early V4.1 README", "Oracle
 * sets against ik_llama.cpp"; "bloomery V4.1 README", "Against ik_llama.cpp");
 * the scoring itself is not printed there and is the definition above.
 * x (device) [T][H] in x_type (MOE_F32 or MOE_BF16); W_router (device) fp32
 * [E][H]; bias (device, nullable) fp32 [E]; logits_in (device, nullable)
 * fp32 [T][E] replaces the router product; logits_out (device, nullable) fp32
 * [T][E]; topk_ids (device) int32 [T][k]; topk_w (device) fp32 [T][k].
 * T = 0 is a no-op.
 */
moe_status moe_route(const moe_route_cfg* cfg, const void* x, moe_dtype x_type, int T, int H,
                     const float* W_router, const float* bias, const float* logits_in,
                     float* logits_out, int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/*
 * moe_permute -- group the P = T*k token-expert pairs by expert.
 *   offsets[e] = number of pairs with id < e (E+1 entries, offsets[E] = P);
 *   sorted_pairs lists p in ascending (expert, p) order (stable);
 *   pair_pos[sorted_pairs[i]] = i.
 * topk_ids (device) int32 [T][k], each in [0, E) (an out-of-range id sets the
 * device status word in the workspace to MOE_ERR_DEVICE_CHECK and the pair is
 * dropped); sorted_pairs, pair_pos (device) int32 [P]; offsets (device) int32
 * [E+1]; workspace (device) of moe_permute_workspace_size() bytes.
 * Pages: a prompt batch runs each expert over all of its tokens at once
 * ("bloomery V4.1 README", feature list, "Batched prompts"); this call builds
 * that per-expert work list.  Integer work: the same bits on every run.
 */
moe_status moe_permute_workspace_size(int T, int k, int E, size_t* bytes);
moe_status moe_permute(const int32_t* topk_ids, int T, int k, int E, int32_t* sorted_pairs,
                       int32_t* offsets, int32_t* pair_pos, void* workspace, size_t ws_bytes,
                       moe_stream_t stream);

/*
 * moe_permute_noalloc -- moe_permute for callers that cannot allocate device
 * memory: code running where cudaMalloc is unavailable or forbidden (inside
 * a host callback, under an allocator lock held by an embedding runtime, or
 * in a process whose device memory is fully owned by another framework), or
 * code that must not size and pass a workspace.  The bloomery pages have no
 * counterpart of this call; it is a convenience of this library.
 * Same inputs and outputs as moe_permute, no workspace: the scratch lives in
 * a fixed 262,400-byte array inside the library that every GPU which loads
 * the library keeps until the process exits.  Limit: T*k <= 65536 pairs
 * (larger sizes return MOE_ERR_INVALID_ARG); E <= 1024 as for moe_permute.
 * Every call looks up that array's address in the current context; the first
 * call in a context may load the library's device code, so make it outside
 * any stream capture.
 * Every call on a device shares the array and zeroes its header first, so
 * two calls whose kernels overlap on the GPU (different streams, no ordering)
 * race: order them on one stream or with events.  Out-of-range ids are
 * dropped (pair_pos = -1, offsets[E] < T*k); no status word is kept.
 * Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 */
moe_status moe_permute_noalloc(const int32_t* topk_ids, int T, int k, int E, int32_t* sorted_pairs,
                               int32_t* offsets, int32_t* pair_pos, moe_stream_t stream);

/*
 * moe_expert_counts_add -- the running routing histogram for callers of moe_permute.
 *   Pages: the engine counts its own routing and moves the experts it calls most to the fast
 *   tier between steps ("bloomery README 0.3.1", opening feature list, MoE models larger than
 *   the card; "bloomery V4.1 README", feature list, "Adaptive residency").
 * counts[e] += offsets[e+1] - offsets[e] for e < E, one launch on `stream`.
 *   offsets (device): int32 [E+1], a moe_permute / moe_permute_noalloc result (non-decreasing);
 *   counts (device): uint64 [E], owned by the caller, read and cleared by it between calls.
 *   Atomic adds: calls on several streams may share one counts array.
 * Errors: MOE_ERR_INVALID_ARG for E outside 1..1024 or a NULL array; MOE_ERR_CUDA when the
 * launch fails.  moe_layer keeps the same histogram itself (moe_layer_desc.expert_counts).
 */
moe_status moe_expert_counts_add(const int32_t* offsets, int E, unsigned long long* counts, moe_stream_t stream);

/*
 * moe_expert_ffn -- the SwiGLU experts over the grouped pairs.
 *   for sorted position i with pair p = sorted_pairs[i], token t = p / k,
 *   expert e (offsets[e] <= i < offsets[e+1]):
 *   g = Wg[e] x_t, u = Wu[e] x_t, h = g/(1+exp(-g)) * u, y_pairs[i] = Wd[e] h.
 * gate, up: rows I, cols H; down: rows H, cols I (host structs, device data).
 * x (device) [T][H]; y_pairs (device) fp32 [T*k][H], row i = sorted position
 * i.  With sorted_pairs = NULL and offsets = NULL (then E = 1, k = 1) the
 * expert runs on every token in order, as a shared expert does.
 * fp32 accumulation, fp32 h, for every T.
 * Pages: routed experts run on the card over the file's stored block
 * quantization, Q4_K among the card types ("bloomery README 0.3.1", Status
 * table, "Quant types" row), each expert over its grouped tokens ("bloomery
 * V4.1 README", feature list, "Batched prompts").  The SwiGLU form and the
 * block layouts are not printed on the pages; they are the definitions above
 * and in the conventions at the top of this file.
 */
moe_status moe_expert_ffn_workspace_size(int T, int k, int E, int H, int I, size_t* bytes);
moe_status moe_expert_ffn(const moe_qmat* gate, const moe_qmat* up, const moe_qmat* down, int E,
                          const void* x, moe_dtype x_type, int T, int H, int I,
                          const int32_t* sorted_pairs, const int32_t* offsets, int k,
                          float* y_pairs, void* workspace, size_t ws_bytes, moe_stream_t stream);

/*
 * The two halves of moe_expert_ffn, for callers that keep h or time them:
 * moe_expert_gateup writes h (device, fp32 [T*k][I], row i = sorted
 * position i) = silu(Wg[e] x_t) * (Wu[e] x_t); moe_expert_down writes
 * y_pairs[i] = Wd[e] h[i].  Same arguments and rules as moe_expert_ffn;
 * each is exactly one kernel launch.
 */
moe_status moe_expert_gateup(const moe_qmat* gate, const moe_qmat* up, int E, const void* x, moe_dtype x_type,
                             int T, int H, int I, const int32_t* sorted_pairs, const int32_t* offsets, int k,
                             float* h, moe_stream_t stream);
moe_status moe_expert_down(const moe_qmat* down, int E, const float* h, int T, int H, int I,
                           const int32_t* sorted_pairs, const int32_t* offsets, int k, float* y_pairs,
                           moe_stream_t stream);

/*
 * moe_combine -- out[t,n] = sum_{j<k} topk_w[t,j] * y_pairs[pair_pos[t*k+j], n]
 *                           (+ shared_out[t,n]) (+ old out[t,n] if accumulate),
 * summed in ascending j, then the shared term, then the old value: the same
 * bits on every run.  y_pairs, shared_out (nullable), out: fp32 (device).
 * Pages: no formula for the combine is printed; its fixed summation order
 * serves the requirement that a replay equal the eager run bit for bit
 * ("bloomery early V4.1 README", "Bit gates").
 */
moe_status moe_combine(const float* y_pairs, const float* topk_w, const int32_t* pair_pos, int T,
                       int k, int H, const float* shared_out, int accumulate, float* out,
                       moe_stream_t stream);

/*
 * moe_rmsnorm_bf16 -- u[t,h] = bf16( x[t,h] / sqrt(mean_h x[t,:]^2 + eps) * gamma[h] )
 * (fp32 arithmetic, round to nearest even).  x fp32 [T][H], gamma fp32 [H],
 * u bf16 [T][H] (device).  Used between stacked layers.
 * Pages: none of the normalisation is printed; this is the plain RMSNorm
 * definition, and the bf16 rounding is the layer input's storage type.
 */
moe_status moe_rmsnorm_bf16(const float* x, const float* gamma, int T, int H, float eps, void* u,
                            moe_stream_t stream);

/* ---------------------------------------------------------------- fused layer */

typedef struct {
    moe_route_cfg route;
    int hidden;                   /* H */
    int intermediate;             /* I of a routed expert */
    moe_dtype x_type;             /* MOE_F32 or MOE_BF16 */
    const float* W_router;        /* (device) fp32 [E][H] */
    const float* bias;            /* (device, nullable) fp32 [E] */
    moe_qmat gate, up, down;      /* routed experts, stacked over E */
    int shared_intermediate;      /* I_s, 0 = no shared expert */
    moe_qmat s_gate, s_up, s_down;/* shared expert (single matrices) */
    int accumulate;               /* 1: out += layer(x) (a residual add); 0: out = layer(x) */
    int tc_min_tokens;            /* T at or above this uses the tensor-core path (0 = default 65) */
    int decode_chain_off;         /* 1: never use the chained decode kernels (T <= 8) */
    /* Pre-norm (nullable): x is the fp32 residual stream [T][H] (x_type MOE_F32) and the layer's
     * input is u = bf16(x / sqrt(mean_h x^2 + norm_eps) * norm_gamma), exactly as moe_rmsnorm_bf16
     * computes it; the chained decode kernels compute u themselves (no extra launch), the other
     * paths run moe_rmsnorm_bf16 into the workspace first.  With accumulate = 1 and out == x one
     * call is a whole residual block, out += layer(norm(out)).  norm_gamma: (device) fp32 [H]. */
    const float* norm_gamma;
    float norm_eps;
    /* Routing histogram (nullable): (device) uint64 [E], owned by the caller.  Every moe_layer
     * call adds, for each expert, the number of its T*k pairs routed to that expert, inside
     * the kernels that already order the pairs (no extra launch); the caller reads or clears it
     * between calls.  The pages' engine counts its own routing and moves the experts it calls
     * most to the fast tier ("bloomery README 0.3.1", opening feature list, MoE models larger
     * than the card; "bloomery V4.1 README", feature list, "Adaptive residency"). */
    unsigned long long* expert_counts;
} moe_layer_desc;

typedef struct moe_layer_plan moe_layer_plan;

/* Validates the description once and keeps a host copy of it.  Plans, workspace
 * sizes and path choice are host-side only, so the per-step launches can be
 * recorded once and replayed ("bloomery README 0.3.11", list of why it is fast:
 * one CUDA graph a decode step). */
moe_status moe_layer_plan_create(const moe_layer_desc* desc, moe_layer_plan** plan);
moe_status moe_layer_plan_destroy(moe_layer_plan* plan);
/* Bytes of device workspace moe_layer needs for up to T tokens. */
moe_status moe_layer_workspace_size(const moe_layer_plan* plan, int T, size_t* bytes);
/* Which kernels moe_layer runs for T tokens with this plan (T >= 1):
 *   MOE_PATH_GEMV         route, permute, dequant-GEMV experts and combine as
 *                         separate launches (fp32 accumulation);
 *   MOE_PATH_DECODE_CHAIN the whole layer as three launches chained by
 *                         programmatic dependent launch (router logits; routing
 *                         + gate/up; down + combine), fp32 accumulation;
 *   MOE_PATH_TENSOR       route and permute, then the tcgen05 grouped GEMM
 *                         (fp16 operands, fp32 accumulation) and combine.
 * Host-only; reads nothing on the device. */
#define MOE_PATH_GEMV 0
#define MOE_PATH_DECODE_CHAIN 1
#define MOE_PATH_TENSOR 2
moe_status moe_layer_path(const moe_layer_plan* plan, int T, int* path);
/*
 * moe_layer -- the whole layer: route, permute, experts, combine (+ shared),
 * for T tokens of x (device, [T][H] in desc->x_type) into out (device, fp32
 * [T][H]).  Enqueued on `stream` with no host synchronization and no host
 * read-back, so it can be captured in a CUDA graph; replays give the same
 * bits as eager calls.  The expert path is chosen from T on the host
 * (moe_layer_path tells which): T <= 8 (T*k <= 64, E <= 256, Q4_K routed
 * experts, H <= 2048, the staged x and the gate/up rings within the kernel's
 * shared memory: T <= 6 at H = 2048) the chained decode kernels, T < tc_min_tokens the fp32
 * dequant-GEMV kernels (both fp32 accumulate), larger T the tensor-core
 * grouped GEMM (fp16 operands, fp32 accumulate; the per-pair down outputs
 * are rounded to fp16 before the fp32 combine).  out may alias x when
 * accumulate = 1 (a residual block): x is read before out is written.
 * T = 0 is a no-op that launches nothing (x, out and workspace may be NULL).
 * Pages: one CUDA graph per decode step ("bloomery README 0.3.11", list of why
 * it is fast), prompts as tensor-core GEMMs (same list) over experts grouped by
 * token ("bloomery V4.1 README", feature list, "Batched prompts"), and a graph
 * replay that equals the eager run bit for bit ("bloomery early V4.1 README",
 * "Bit gates").
 */
moe_status moe_layer(const moe_layer_plan* plan, const void* x, int T, float* out, void* workspace,
                     size_t ws_bytes, moe_stream_t stream);
/* moe_layer that also records two caller-owned CUDA events (cudaEvent_t, may
 * be NULL) on `stream` immediately before and after the launch of the routed
 * gate/up kernel, so a caller can time that kernel alone.  Same results as
 * moe_layer; meant for eager calls (not for graph capture). */
moe_status moe_layer_timed(const moe_layer_plan* plan, const void* x, int T, float* out, void* workspace,
                           size_t ws_bytes, moe_stream_t stream, void* ev_before_gateup, void* ev_after_gateup);

/* Device pointers into a moe_layer workspace (any output may be NULL) to
 * the last call's ids int32 [T][k], gates fp32 [T][k] and offsets int32
 * [E+1]. */
moe_status moe_layer_debug_views(const moe_layer_plan* plan, int T, void* workspace,
                                 int32_t** topk_ids, float** topk_w, int32_t** offsets);

/* Copies the device status word of a workspace (MOE_OK or a MOE_ERR_* code
 * raised by a device-side check) to *code and clears it.  Synchronizes the
 * stream first; call it outside graph capture.  Pages: a bad request is
 * refused by name rather than run ("bloomery README 0.3.11", limits list). */
moe_status moe_read_device_status(const moe_layer_plan* plan, int T, void* workspace, int32_t* code,
                                  moe_stream_t stream);
moe_status moe_permute_read_device_status(int T, int k, int E, void* workspace, int32_t* code,
                                          moe_stream_t stream);

/*
 * moe_debug_set_waits -- test hook for the bounded device-side waits; off by
 * default.  Every wait of the library's kernels on a copy or an MMA gives up
 * after limit_ns nanoseconds (0 restores the default of 2 s), records
 * MOE_ERR_TIMEOUT in the workspace status word, waits (within the same limit)
 * for the copies its CTA still has in flight, releases what it holds and
 * returns; the call's outputs are then undefined and moe_read_device_status
 * reports the code.  stall = 1 makes the first wait of the chained decode,
 * segmented GEMV and tensor-core kernels wait on a barrier that nothing
 * completes, so that a test can run this path without a faulty input.
 * Applies to calls launched after it, from any host thread (a graph keeps the
 * setting it was captured with).  The failure reporting follows the pages'
 * refusals by name with named exit codes ("bloomery README 0.3.11").
 */
moe_status moe_debug_set_waits(uint64_t limit_ns, int stall);

/*
 * moe_debug_set_stamps -- timing hook of the chained decode kernels (T <= 8); off by
 * default (buf = NULL).  With a device buffer of at least 3*256*8*8 = 49,152 bytes, every
 * chained call launched afterwards has thread 0 of CTA c (c < 256) of kernel n (0 router
 * logits, 1 routing + gate/up, 2 down + combine) write the GPU's global nanosecond clock
 * at phase ph into buf[(n*256 + c)*8 + ph] (uint64): n = 0: 0 start, 1 after the wait for
 * the previous launch, 2 router dot products done, 3 end; n = 1: 0 start, 1 activations
 * staged, 2 after the wait, 3 routing read, 4 first unit computed, 5 units done, 6 CTA
 * done, 7 top-k written; n = 2: 0 start, 2 routing read and down rows requested (before
 * the wait), 1 after the wait, 3 h copies issued, 4 copies landed, 5 dot products done, 6 CTA
 * done.  Calls overwrite the same slots; a graph keeps the setting it was
 * captured with.  For measuring where a decode layer's time goes; the results are
 * unchanged.  Pages: step times there are quoted with their instrumentation state
 * ("bloomery early V4.1 README", caveats of the depth measurement).
 */
moe_status moe_debug_set_stamps(void* buf, size_t bytes);

/* The reason for the last non-MOE_OK status returned on this host thread
 * (refusals by name: "bloomery README 0.3.11", limits list). */
const char* moe_last_error(void);
/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
