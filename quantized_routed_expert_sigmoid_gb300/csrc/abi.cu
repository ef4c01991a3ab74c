// abi.cu -- the C ABI (include/moe_gb300.h): host-side validation, workspace
// layout, and the order of launches for each call.  No device memory is
// allocated here and no call synchronizes (the two status reads aside).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <new>
#include <vector>

#include "internal.cuh"

using namespace moe;

namespace {

thread_local char g_err[512] = "";

moe_status fail(moe_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

moe_status cuda_fail(cudaError_t err, const char* what) {
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int64_t row_bytes(moe_dtype q, int64_t cols) {
    if (q == MOE_Q3_K) return cols / 256 * 110;
    if (q == MOE_MXFP4) return cols / 32 * 17;
    if (q == MOE_Q4_K || q == MOE_Q8_0 || q == MOE_Q8_0_R || q == MOE_Q5_K || q == MOE_Q6_K) return q_row_bytes(q, cols);
    return -1;
}
// The kernels' view of a weight type: Q8_0 in either layout is MOE_Q8_0, the layout a flag.
int kernel_qtype(moe_dtype q) { return q == MOE_Q8_0_R ? (int)MOE_Q8_0 : (int)q; }

moe_status check_qmat(const moe_qmat* m, const char* name, int64_t rows, int64_t cols, int E) {
    if (!m) return fail(MOE_ERR_INVALID_ARG, "%s: NULL matrix", name);
    if (m->qtype != MOE_Q4_K && m->qtype != MOE_Q8_0 && m->qtype != MOE_Q8_0_R && m->qtype != MOE_Q5_K &&
        m->qtype != MOE_Q6_K && m->qtype != MOE_Q3_K && m->qtype != MOE_MXFP4)
        return fail(MOE_ERR_UNSUPPORTED, "%s: qtype %d (supported: Q8_0, Q8_0_R, Q4_K, Q5_K, Q6_K, Q3_K, MXFP4)", name,
                    (int)m->qtype);
    if (!m->data) return fail(MOE_ERR_INVALID_ARG, "%s: NULL data", name);
    if (!aligned(m->data, 16)) return fail(MOE_ERR_INVALID_ARG, "%s: data not 16-byte aligned", name);
    if (m->rows != rows || m->cols != cols)
        return fail(MOE_ERR_INVALID_ARG, "%s: shape %lldx%lld, expected %lldx%lld", name, (long long)m->rows,
                    (long long)m->cols, (long long)rows, (long long)cols);
    // MXFP4: 17-byte blocks, rows kept to a multiple of 4 bytes (the kernels' aligned word loads)
    const int blk = (m->qtype == MOE_Q8_0 || m->qtype == MOE_Q8_0_R) ? kQ80Weights : m->qtype == MOE_MXFP4 ? 128
                                                                                     : kQ4KWeights;
    if (cols % blk) return fail(MOE_ERR_INVALID_ARG, "%s: cols %lld not a multiple of %d", name, (long long)cols, blk);
    const int64_t need = rows * row_bytes(m->qtype, cols);
    if (E > 1 && (m->expert_stride_bytes < need || m->expert_stride_bytes % 16))
        return fail(MOE_ERR_INVALID_ARG, "%s: expert stride %lld (need >= %lld, multiple of 16)", name,
                    (long long)m->expert_stride_bytes, (long long)need);
    return MOE_OK;
}

moe_status check_route_cfg(const moe_route_cfg* c) {
    if (!c) return fail(MOE_ERR_INVALID_ARG, "route cfg is NULL");
    if (c->n_experts < 1 || c->n_experts > kMaxExperts)
        return fail(MOE_ERR_INVALID_ARG, "n_experts %d outside 1..%d", c->n_experts, kMaxExperts);
    if (c->top_k < 1 || c->top_k > c->n_experts || c->top_k > kMaxTopK)
        return fail(MOE_ERR_INVALID_ARG, "top_k %d outside 1..min(E, %d)", c->top_k, kMaxTopK);
    if (c->mode == MOE_ROUTE_SIGMOID_GROUP) {
        if (c->n_groups < 1 || c->n_groups > 32 || c->n_experts % c->n_groups)
            return fail(MOE_ERR_INVALID_ARG, "n_groups %d must divide E and be <= 32", c->n_groups);
        if (c->topk_groups < 1 || c->topk_groups > c->n_groups)
            return fail(MOE_ERR_INVALID_ARG, "topk_groups %d outside 1..n_groups", c->topk_groups);
        if (c->top_k > c->topk_groups * (c->n_experts / c->n_groups))
            return fail(MOE_ERR_INVALID_ARG, "top_k %d exceeds the experts of the kept groups", c->top_k);
    } else if (c->mode != MOE_ROUTE_SOFTMAX) {
        return fail(MOE_ERR_INVALID_ARG, "unknown routing mode %d", (int)c->mode);
    }
    return MOE_OK;
}

struct FfnWs {
    size_t h, total;
};
FfnWs ffn_ws(int T, int k, int I) {
    FfnWs w;
    w.h = 0;
    w.total = align_up((size_t)T * k * I * sizeof(float), 256);
    return w;
}

}  // namespace

moe_status moe::report(moe_status st, const char* msg) { return fail(st, "%s", msg); }

namespace {
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_wait_stall{0};
}  // namespace

WaitCfg moe::wait_cfg() { return WaitCfg{g_wait_ns.load(), g_wait_stall.load()}; }

namespace {
std::atomic<void*> g_stamps{nullptr};
}  // namespace

void* moe::debug_stamps() { return g_stamps.load(); }

struct moe_layer_plan {
    moe_layer_desc d;
};

namespace {

// Workspace of moe_layer for T tokens (offsets in bytes, all 256-aligned).
struct LayerWs {
    bool tc;                      // tensor-core path for this T
    size_t hdr, logits, ids, w, sorted, pair_pos, offsets, chunk, h, y, sh_h, sh_y, x16, tiles, wsplit, hq, hq_s, u,
        total;
    bool router_tc;               // router logits on the tensor cores
    bool chain;                   // the chained decode kernels
    bool norm_in_chain;           // pre-norm computed by the chain itself (else moe_rmsnorm_bf16 into u)
};

// The layer's input dtype once a pre-norm has run (its output u is bf16).
bool input_bf16(const moe_layer_desc& d) { return d.x_type == MOE_BF16 || d.norm_gamma != nullptr; }

bool use_tc(const moe_layer_desc& d, int T) {
    if (T < d.tc_min_tokens) return false;
    if (!tc_supported(d.gate.qtype, d.intermediate, d.hidden) || !tc_supported(d.down.qtype, d.hidden, d.intermediate))
        return false;
    if (d.gate.qtype != d.down.qtype) return false;
    if (d.shared_intermediate > 0 &&
        (!tc_supported(d.s_gate.qtype, d.shared_intermediate, d.hidden) ||
         !tc_supported(d.s_down.qtype, d.hidden, d.shared_intermediate) || d.s_gate.qtype != d.s_down.qtype))
        return false;
    return true;
}

// The shape-level fields of the chained decode kernels (no buffers yet).
DecodeArgs decode_shape_args(const moe_layer_desc& d, int T) {
    DecodeArgs da{};
    da.route = d.route;
    da.Wr = d.W_router;
    da.x_bf16 = input_bf16(d);    // the values the chain stages (the launch sets the buffers)
    da.bias = d.bias;
    da.T = T; da.H = d.hidden; da.I = d.intermediate;
    da.qtype = kernel_qtype(d.gate.qtype);
    da.wg = static_cast<const uint8_t*>(d.gate.data);
    da.wu = static_cast<const uint8_t*>(d.up.data);
    da.wd = static_cast<const uint8_t*>(d.down.data);
    da.stride_gu = d.gate.expert_stride_bytes;
    da.stride_d = d.down.expert_stride_bytes;
    da.I_s = d.shared_intermediate;
    if (da.I_s > 0) {
        da.s_qtype = kernel_qtype(d.s_gate.qtype);
        da.s_q80r = d.s_gate.qtype == MOE_Q8_0_R;
        da.sg = static_cast<const uint8_t*>(d.s_gate.data);
        da.su = static_cast<const uint8_t*>(d.s_up.data);
        da.sd = static_cast<const uint8_t*>(d.s_down.data);
    }
    da.counts = d.expert_counts;
    return da;
}

// True when moe_layer runs T tokens as the chained decode kernels.
bool decode_chain_applies(const moe_layer_desc& d, int T) {
    if (d.decode_chain_off || use_tc(d, T)) return false;
    const bool same_q = d.gate.qtype == d.up.qtype && d.gate.qtype == d.down.qtype &&
                        (d.shared_intermediate == 0 ||
                         (d.s_gate.qtype == d.s_up.qtype && d.s_gate.qtype == d.s_down.qtype));
    return same_q && decode_chain_supported(decode_shape_args(d, T));
}

LayerWs layer_ws(const moe_layer_desc& d, int T) {
    const int E = d.route.n_experts, k = d.route.top_k, H = d.hidden, I = d.intermediate;
    const size_t P = (size_t)T * k;
    LayerWs w;
    w.tc = use_tc(d, T);
    const size_t hbytes = w.tc ? 2 : 4;   // h is fp16 on the tensor-core path, fp32 on the GEMV path
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    w.hdr = take(kHeaderBytes);
    w.logits = take((size_t)T * E * 4);
    w.ids = take(P * 4);
    w.w = take(P * 4);
    w.sorted = take(P * 4);
    w.pair_pos = take(P * 4);
    w.offsets = take((size_t)(E + 1) * 4);
    w.chunk = take(permute_scratch_bytes(T, k, E));
    w.h = take(P * I * hbytes);
    w.y = take(P * H * 4);
    const int Is = d.shared_intermediate;
    w.sh_h = take(Is > 0 ? (size_t)T * Is * hbytes : 0);
    w.sh_y = take(Is > 0 ? (size_t)T * H * 4 : 0);
    w.x16 = take(w.tc ? (size_t)T * H * 2 : 0);
    w.tiles = take(w.tc ? tc_tile_list_bytes(T, k, E) : 0);
    // tensor-core router logits only on the tensor-core path: their fp32 accumulation inside the
    // MMA is within that path's tolerance, not within the GEMV path's
    w.router_tc = w.tc && router_tc_supported(T, H, E, input_bf16(d));
    w.wsplit = take(w.router_tc ? router_tc_split_bytes(H, E) : 0);
    const bool chain = decode_chain_applies(d, T);
    w.chain = chain;
    // the chain normalizes its own input unless its shared expert is Q8_0 (staged from x apart)
    w.norm_in_chain = chain && d.norm_gamma && !(Is > 0 && kernel_qtype(d.s_gate.qtype) == MOE_Q8_0);
    w.u = take(d.norm_gamma && !w.norm_in_chain ? (size_t)T * H * 2 : 0);
    w.hq = take(chain ? P * (size_t)(I / 64) * 272 : 0);
    w.hq_s = take(chain && Is > 0 ? (size_t)T * (Is / 64) * 272 : 0);
    w.total = o;
    return w;
}

template <typename T>
T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(base) + off);
}

GemvArgs gemv_args(const moe_qmat& m0, const moe_qmat* m1, int E, const void* vin, bool vin_bf16, int rows,
                   int K, const int32_t* sorted, const int32_t* offsets, int k, int n_pairs, float* out) {
    GemvArgs g{};
    g.qtype = kernel_qtype(m0.qtype);
    g.q80r = m0.qtype == MOE_Q8_0_R;
    g.gateup = m1 != nullptr;
    g.w0 = static_cast<const uint8_t*>(m0.data);
    g.w1 = m1 ? static_cast<const uint8_t*>(m1->data) : nullptr;
    g.expert_stride = m0.expert_stride_bytes;
    g.rows = rows;
    g.K = K;
    g.vin = vin;
    g.vin_bf16 = vin_bf16;
    g.sorted_pairs = sorted;
    g.offsets = offsets;
    g.E = E;
    g.k = k;
    g.n_pairs = n_pairs;
    g.out = out;
    return g;
}

moe_status check_ffn_common(int E, int k, int T, int H, int I, const int32_t* sorted_pairs, const int32_t* offsets) {
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", T);
    if (E < 1 || E > kMaxExperts || k < 1 || k > kMaxTopK) return fail(MOE_ERR_INVALID_ARG, "bad E/k");
    if (H < 32 || I < 32) return fail(MOE_ERR_INVALID_ARG, "H/I too small");
    if ((sorted_pairs == nullptr) != (offsets == nullptr))
        return fail(MOE_ERR_INVALID_ARG, "sorted_pairs and offsets must both be set or both be NULL");
    if (!sorted_pairs && (E != 1 || k != 1))
        return fail(MOE_ERR_INVALID_ARG, "the identity mapping needs E = 1 and k = 1");
    return MOE_OK;
}

// Routed gate/up (h fp32 [P][I]) and down (y fp32 [P][H]): the segmented persistent kernels
// when the shape allows them (routed experts with a permutation), else the per-expert GEMV.
cudaError_t routed_gateup(const moe_qmat& gate, const moe_qmat& up, int E, const void* x, bool x_bf16, int T, int H,
                          int I, const int32_t* sorted, const int32_t* offsets, int k, float* h, WsHeader* hdr,
                          cudaStream_t s) {
    if (sorted && offsets && gate.qtype == up.qtype && seg_gemv_supported(gate.qtype, E, H, I))
        return launch_seg_gemv(true, x, x_bf16, sorted, offsets, E, k, H, I, static_cast<const uint8_t*>(gate.data),
                               static_cast<const uint8_t*>(up.data), gate.expert_stride_bytes, h, hdr, T, s);
    return launch_qgemv(gemv_args(gate, &up, E, x, x_bf16, I, H, sorted, offsets, k, T * k, h), s);
}
cudaError_t routed_down(const moe_qmat& down, int E, const float* h, int T, int H, int I, const int32_t* sorted,
                        const int32_t* offsets, int k, float* y, WsHeader* hdr, cudaStream_t s) {
    if (sorted && offsets && seg_gemv_supported(down.qtype, E, H, I))
        return launch_seg_gemv(false, h, false, sorted, offsets, E, k, I, H, static_cast<const uint8_t*>(down.data),
                               nullptr, down.expert_stride_bytes, y, hdr, T, s);
    return launch_qgemv(gemv_args(down, nullptr, E, h, false, H, I, sorted, offsets, k, T * k, y), s);
}

moe_status run_ffn(const moe_qmat& gate, const moe_qmat& up, const moe_qmat& down, int E, const void* x,
                   bool x_bf16, int T, int H, int I, const int32_t* sorted, const int32_t* offsets, int k,
                   float* h, float* y, cudaStream_t s, WsHeader* hdr = nullptr) {
    cudaError_t err = routed_gateup(gate, up, E, x, x_bf16, T, H, I, sorted, offsets, k, h, hdr, s);
    if (err != cudaSuccess) return cuda_fail(err, "gate/up kernel");
    err = routed_down(down, E, h, T, H, I, sorted, offsets, k, y, hdr, s);
    if (err != cudaSuccess) return cuda_fail(err, "down kernel");
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_last_error(void) { return g_err; }

moe_status moe_debug_set_stamps(void* buf, size_t bytes) {
    if (buf && (bytes < kStampBytes || !aligned(buf, 8)))
        return fail(MOE_ERR_INVALID_ARG, "stamp buffer: %zu bytes (need %zu, 8-byte aligned)", bytes, kStampBytes);
    g_stamps.store(buf);
    return MOE_OK;
}

moe_status moe_debug_set_waits(uint64_t limit_ns, int stall) {
    if (stall != 0 && stall != 1) return fail(MOE_ERR_INVALID_ARG, "stall must be 0 or 1");
    g_wait_ns.store(limit_ns == 0 ? kDefaultWaitNs : limit_ns);
    g_wait_stall.store(stall);
    return MOE_OK;
}
const char* moe_version(void) { return "moe_gb300 0.1 (sm_103a)"; }

moe_status moe_weights_prepare_size(const moe_qmat* in, int n_experts, size_t* bytes) {
    if (!in || !bytes) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    if (n_experts < 1) return fail(MOE_ERR_INVALID_ARG, "n_experts = %d < 1", n_experts);
    if (in->qtype == MOE_Q4_K || in->qtype == MOE_Q5_K || in->qtype == MOE_Q6_K || in->qtype == MOE_Q3_K ||
        in->qtype == MOE_MXFP4) {
        *bytes = 0;
        return MOE_OK;
    }
    if (in->qtype != MOE_Q8_0)
        return fail(MOE_ERR_UNSUPPORTED, "moe_weights_prepare: qtype %d (it repacks Q8_0; Q4_K is used as stored)",
                    (int)in->qtype);
    if (in->rows < 1 || in->cols < kQ80Weights || in->cols % kQ80Weights)
        return fail(MOE_ERR_INVALID_ARG, "shape %lldx%lld (cols a positive multiple of 32)", (long long)in->rows,
                    (long long)in->cols);
    *bytes = (size_t)n_experts * (size_t)in->rows * (size_t)q80r_row_bytes(in->cols);
    return MOE_OK;
}

moe_status moe_weights_prepare(moe_qmat* in_out, int n_experts, void* dst, size_t dst_bytes, moe_stream_t stream) {
    size_t need = 0;
    moe_status st = moe_weights_prepare_size(in_out, n_experts, &need);
    if (st) return st;
    if (in_out->qtype == MOE_Q4_K || in_out->qtype == MOE_Q5_K || in_out->qtype == MOE_Q6_K ||
        in_out->qtype == MOE_Q3_K || in_out->qtype == MOE_MXFP4)
        return MOE_OK;
    if ((st = check_qmat(in_out, "in", in_out->rows, in_out->cols, n_experts))) return st;
    if (!dst || !aligned(dst, 16)) return fail(MOE_ERR_INVALID_ARG, "dst NULL or not 16-byte aligned");
    if (dst_bytes < need) return fail(MOE_ERR_WORKSPACE, "dst %zu bytes, need %zu", dst_bytes, need);
    const uintptr_t s0 = (uintptr_t)in_out->data, d0 = (uintptr_t)dst;
    const uintptr_t s1 = s0 + (size_t)(n_experts - 1) * (size_t)in_out->expert_stride_bytes +
                         (size_t)in_out->rows * (size_t)row_bytes(MOE_Q8_0, in_out->cols);
    if (d0 < s1 && s0 < d0 + need) return fail(MOE_ERR_INVALID_ARG, "dst overlaps the source");
    const int64_t rb = q80r_row_bytes(in_out->cols);
    cudaError_t err = launch_q80_repack(static_cast<const uint8_t*>(in_out->data), in_out->expert_stride_bytes,
                                        n_experts, in_out->rows, in_out->cols, static_cast<uint8_t*>(dst),
                                        reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "repack kernel");
    in_out->qtype = MOE_Q8_0_R;
    in_out->data = dst;
    in_out->expert_stride_bytes = in_out->rows * rb;
    return MOE_OK;
}

moe_status moe_route(const moe_route_cfg* cfg, const void* x, moe_dtype x_type, int T, int H,
                     const float* W_router, const float* bias, const float* logits_in, float* logits_out,
                     int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
    moe_status st = check_route_cfg(cfg);
    if (st) return st;
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", T);
    if (T == 0) return MOE_OK;
    if (!topk_ids || !topk_w) return fail(MOE_ERR_INVALID_ARG, "topk_ids / topk_w are NULL");
    if (!aligned(topk_ids, 4) || !aligned(topk_w, 4)) return fail(MOE_ERR_INVALID_ARG, "ids/w not 4-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float* logits = logits_in;
    if (!logits_in) {
        if (!logits_out) return fail(MOE_ERR_INVALID_ARG, "logits_out is needed when logits_in is NULL");
        if (!x || !W_router) return fail(MOE_ERR_INVALID_ARG, "x / W_router are NULL");
        if (x_type != MOE_F32 && x_type != MOE_BF16) return fail(MOE_ERR_UNSUPPORTED, "x_type %d", (int)x_type);
        if (H < 4 || H % 32) return fail(MOE_ERR_INVALID_ARG, "H = %d must be a positive multiple of 32", H);
        if (!aligned(x, 16) || !aligned(W_router, 16) || !aligned(logits_out, 4))
            return fail(MOE_ERR_INVALID_ARG, "x / W_router must be 16-byte aligned");
        cudaError_t err = launch_router_logits(x, x_type == MOE_BF16, T, H, W_router, cfg->n_experts,
                                               logits_out, nullptr, s);
        if (err != cudaSuccess) return cuda_fail(err, "router logits kernel");
        logits = logits_out;
    } else if (logits_out && logits_out != logits_in) {
        cudaError_t err = cudaMemcpyAsync(logits_out, logits_in, sizeof(float) * (size_t)T * cfg->n_experts,
                                          cudaMemcpyDeviceToDevice, s);
        if (err != cudaSuccess) return cuda_fail(err, "logits copy");
    }
    cudaError_t err = launch_topk(*cfg, logits, bias, T, topk_ids, topk_w, nullptr, s);
    if (err != cudaSuccess) return cuda_fail(err, "top-k kernel");
    return MOE_OK;
}

moe_status moe_permute_workspace_size(int T, int k, int E, size_t* bytes) {
    if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
    if (T < 0 || k < 1 || E < 1 || E > kMaxExperts) return fail(MOE_ERR_INVALID_ARG, "bad T/k/E");
    *bytes = kHeaderBytes + permute_scratch_bytes(T, k, E);
    return MOE_OK;
}

moe_status moe_permute(const int32_t* topk_ids, int T, int k, int E, int32_t* sorted_pairs, int32_t* offsets,
                       int32_t* pair_pos, void* workspace, size_t ws_bytes, moe_stream_t stream) {
    size_t need = 0;
    moe_status st = moe_permute_workspace_size(T, k, E, &need);
    if (st) return st;
    if (!offsets) return fail(MOE_ERR_INVALID_ARG, "offsets is NULL");
    if (T > 0 && (!topk_ids || !sorted_pairs || !pair_pos)) return fail(MOE_ERR_INVALID_ARG, "NULL array");
    if ((int64_t)T * k > (int64_t)1 << 30) return fail(MOE_ERR_INVALID_ARG, "T*k too large");
    if (!workspace || ws_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace ? ws_bytes : 0, need);
    if (!aligned(workspace, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    WsHeader* hdr = at<WsHeader>(workspace, 0);
    cudaError_t err = cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s);
    if (err != cudaSuccess) return cuda_fail(err, "workspace header reset");
    err = launch_permute(topk_ids, T, k, E, sorted_pairs, offsets, pair_pos, hdr,
                         at<int32_t>(workspace, kHeaderBytes), s);
    if (err != cudaSuccess) return cuda_fail(err, "permute kernel");
    return MOE_OK;
}

moe_status moe_permute_read_device_status(int T, int k, int E, void* workspace, int32_t* code,
                                          moe_stream_t stream) {
    (void)T; (void)k; (void)E;
    if (!workspace || !code) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = cudaStreamSynchronize(s);
    if (err == cudaSuccess) err = cudaMemcpy(code, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (err == cudaSuccess) err = cudaMemset(workspace, 0, sizeof(int32_t));
    if (err != cudaSuccess) return cuda_fail(err, "status read");
    return MOE_OK;
}

moe_status moe_expert_ffn_workspace_size(int T, int k, int E, int H, int I, size_t* bytes) {
    (void)E; (void)H;
    if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
    if (T < 0 || k < 1 || I < 1) return fail(MOE_ERR_INVALID_ARG, "bad T/k/I");
    *bytes = ffn_ws(T, k, I).total;
    return MOE_OK;
}

moe_status moe_expert_ffn(const moe_qmat* gate, const moe_qmat* up, const moe_qmat* down, int E, const void* x,
                          moe_dtype x_type, int T, int H, int I, const int32_t* sorted_pairs,
                          const int32_t* offsets, int k, float* y_pairs, void* workspace, size_t ws_bytes,
                          moe_stream_t stream) {
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", T);
    if (E < 1 || E > kMaxExperts || k < 1 || k > kMaxTopK) return fail(MOE_ERR_INVALID_ARG, "bad E/k");
    if (H < 32 || I < 32) return fail(MOE_ERR_INVALID_ARG, "H/I too small");
    moe_status st;
    if ((st = check_qmat(gate, "gate", I, H, E)) || (st = check_qmat(up, "up", I, H, E)) ||
        (st = check_qmat(down, "down", H, I, E)))
        return st;
    if (gate->qtype != up->qtype) return fail(MOE_ERR_UNSUPPORTED, "gate and up must share a qtype");
    if (gate->expert_stride_bytes != up->expert_stride_bytes)
        return fail(MOE_ERR_INVALID_ARG, "gate and up must share an expert stride");
    if (x_type != MOE_F32 && x_type != MOE_BF16) return fail(MOE_ERR_UNSUPPORTED, "x_type %d", (int)x_type);
    if ((sorted_pairs == nullptr) != (offsets == nullptr))
        return fail(MOE_ERR_INVALID_ARG, "sorted_pairs and offsets must both be set or both be NULL");
    if (!sorted_pairs && (E != 1 || k != 1))
        return fail(MOE_ERR_INVALID_ARG, "the identity mapping needs E = 1 and k = 1");
    if (T == 0) return MOE_OK;
    if (!x || !y_pairs) return fail(MOE_ERR_INVALID_ARG, "x / y_pairs are NULL");
    if (!aligned(x, 16) || !aligned(y_pairs, 16)) return fail(MOE_ERR_INVALID_ARG, "x / y_pairs not 16-byte aligned");
    const FfnWs w = ffn_ws(T, k, I);
    if (!workspace || ws_bytes < w.total)
        return fail(MOE_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace ? ws_bytes : 0, w.total);
    if (!aligned(workspace, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    return run_ffn(*gate, *up, *down, E, x, x_type == MOE_BF16, T, H, I, sorted_pairs, offsets, k,
                   at<float>(workspace, w.h), y_pairs, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_expert_gateup(const moe_qmat* gate, const moe_qmat* up, int E, const void* x, moe_dtype x_type,
                             int T, int H, int I, const int32_t* sorted_pairs, const int32_t* offsets, int k,
                             float* h, moe_stream_t stream) {
    moe_status st = check_ffn_common(E, k, T, H, I, sorted_pairs, offsets);
    if (st) return st;
    if ((st = check_qmat(gate, "gate", I, H, E)) || (st = check_qmat(up, "up", I, H, E))) return st;
    if (gate->qtype != up->qtype || gate->expert_stride_bytes != up->expert_stride_bytes)
        return fail(MOE_ERR_INVALID_ARG, "gate and up must share qtype and expert stride");
    if (x_type != MOE_F32 && x_type != MOE_BF16) return fail(MOE_ERR_UNSUPPORTED, "x_type %d", (int)x_type);
    if (T == 0) return MOE_OK;
    if (!x || !h || !aligned(x, 16) || !aligned(h, 16)) return fail(MOE_ERR_INVALID_ARG, "x / h NULL or misaligned");
    cudaError_t err = routed_gateup(*gate, *up, E, x, x_type == MOE_BF16, T, H, I, sorted_pairs, offsets, k, h,
                                    nullptr, reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "gate/up kernel");
    return MOE_OK;
}

moe_status moe_expert_down(const moe_qmat* down, int E, const float* h, int T, int H, int I,
                           const int32_t* sorted_pairs, const int32_t* offsets, int k, float* y_pairs,
                           moe_stream_t stream) {
    moe_status st = check_ffn_common(E, k, T, H, I, sorted_pairs, offsets);
    if (st) return st;
    if ((st = check_qmat(down, "down", H, I, E))) return st;
    if (T == 0) return MOE_OK;
    if (!h || !y_pairs || !aligned(h, 16) || !aligned(y_pairs, 16))
        return fail(MOE_ERR_INVALID_ARG, "h / y_pairs NULL or misaligned");
    cudaError_t err = routed_down(*down, E, h, T, H, I, sorted_pairs, offsets, k, y_pairs, nullptr,
                                  reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "down kernel");
    return MOE_OK;
}

moe_status moe_combine(const float* y_pairs, const float* topk_w, const int32_t* pair_pos, int T, int k, int H,
                       const float* shared_out, int accumulate, float* out, moe_stream_t stream) {
    if (T < 0 || k < 1 || H < 4 || H % 4) return fail(MOE_ERR_INVALID_ARG, "bad T/k/H");
    if (T == 0) return MOE_OK;
    if (!y_pairs || !topk_w || !pair_pos || !out) return fail(MOE_ERR_INVALID_ARG, "NULL array");
    if (!aligned(y_pairs, 16) || !aligned(out, 16) || (shared_out && !aligned(shared_out, 16)))
        return fail(MOE_ERR_INVALID_ARG, "y_pairs / shared_out / out not 16-byte aligned");
    cudaError_t err = launch_combine(y_pairs, topk_w, pair_pos, T, k, H, shared_out, accumulate != 0, out,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "combine kernel");
    return MOE_OK;
}

moe_status moe_rmsnorm_bf16(const float* x, const float* gamma, int T, int H, float eps, void* u,
                            moe_stream_t stream) {
    if (T < 0 || H < 4 || H % 4) return fail(MOE_ERR_INVALID_ARG, "bad T/H");
    if (T == 0) return MOE_OK;
    if (!x || !gamma || !u) return fail(MOE_ERR_INVALID_ARG, "NULL array");
    if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(u, 16))
        return fail(MOE_ERR_INVALID_ARG, "x / gamma / u not 16-byte aligned");
    if (!(eps >= 0.0f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
    cudaError_t err = launch_rmsnorm_bf16(x, gamma, T, H, eps, u, reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "rmsnorm kernel");
    return MOE_OK;
}

moe_status moe_layer_plan_create(const moe_layer_desc* desc, moe_layer_plan** plan) {
    if (!desc || !plan) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    *plan = nullptr;
    const moe_layer_desc& d = *desc;
    moe_status st = check_route_cfg(&d.route);
    if (st) return st;
    const int E = d.route.n_experts, H = d.hidden, I = d.intermediate;
    if (H < 32 || H % 32 || I < 32) return fail(MOE_ERR_INVALID_ARG, "hidden %d / intermediate %d", H, I);
    if (d.x_type != MOE_F32 && d.x_type != MOE_BF16) return fail(MOE_ERR_UNSUPPORTED, "x_type %d", (int)d.x_type);
    if (!d.W_router || !aligned(d.W_router, 16)) return fail(MOE_ERR_INVALID_ARG, "W_router NULL or misaligned");
    if (d.route.mode == MOE_ROUTE_SOFTMAX && d.bias)
        return fail(MOE_ERR_INVALID_ARG, "a selection bias needs the sigmoid-group mode");
    if ((st = check_qmat(&d.gate, "gate", I, H, E)) || (st = check_qmat(&d.up, "up", I, H, E)) ||
        (st = check_qmat(&d.down, "down", H, I, E)))
        return st;
    if (d.gate.qtype != d.up.qtype || d.gate.expert_stride_bytes != d.up.expert_stride_bytes)
        return fail(MOE_ERR_INVALID_ARG, "gate and up must share qtype and expert stride");
    if (d.shared_intermediate < 0) return fail(MOE_ERR_INVALID_ARG, "shared_intermediate < 0");
    if (d.norm_gamma) {
        if (d.x_type != MOE_F32) return fail(MOE_ERR_INVALID_ARG, "a pre-norm needs the fp32 residual stream as x");
        if (!aligned(d.norm_gamma, 16)) return fail(MOE_ERR_INVALID_ARG, "norm_gamma not 16-byte aligned");
        if (H % 4) return fail(MOE_ERR_INVALID_ARG, "a pre-norm needs H %% 4 == 0");
        if (!(d.norm_eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "norm_eps < 0");
    }
    if (d.shared_intermediate > 0) {
        const int Is = d.shared_intermediate;
        if ((st = check_qmat(&d.s_gate, "s_gate", Is, H, 1)) || (st = check_qmat(&d.s_up, "s_up", Is, H, 1)) ||
            (st = check_qmat(&d.s_down, "s_down", H, Is, 1)))
            return st;
        if (d.s_gate.qtype != d.s_up.qtype) return fail(MOE_ERR_INVALID_ARG, "s_gate and s_up must share a qtype");
    }
    moe_layer_plan* p = new (std::nothrow) moe_layer_plan;
    if (!p) return fail(MOE_ERR_INVALID_ARG, "out of host memory");
    p->d = d;
    if (p->d.tc_min_tokens <= 0) p->d.tc_min_tokens = 65;      // T > 64: the grouped GEMM
    *plan = p;
    return MOE_OK;
}

moe_status moe_layer_plan_destroy(moe_layer_plan* plan) {
    delete plan;
    return MOE_OK;
}

moe_status moe_layer_workspace_size(const moe_layer_plan* plan, int T, size_t* bytes) {
    if (!plan || !bytes) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T < 0");
    *bytes = layer_ws(plan->d, T).total;
    return MOE_OK;
}

moe_status moe_layer_path(const moe_layer_plan* plan, int T, int* path) {
    if (!plan || !path) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    if (T < 1) return fail(MOE_ERR_INVALID_ARG, "T = %d < 1", T);
    if (use_tc(plan->d, T)) *path = MOE_PATH_TENSOR;
    else if (decode_chain_applies(plan->d, T)) *path = MOE_PATH_DECODE_CHAIN;
    else *path = MOE_PATH_GEMV;
    return MOE_OK;
}

moe_status moe_layer(const moe_layer_plan* plan, const void* x, int T, float* out, void* workspace,
                     size_t ws_bytes, moe_stream_t stream) {
    return moe_layer_timed(plan, x, T, out, workspace, ws_bytes, stream, nullptr, nullptr);
}

moe_status moe_layer_timed(const moe_layer_plan* plan, const void* x, int T, float* out, void* workspace,
                           size_t ws_bytes, moe_stream_t stream, void* ev_before_gateup, void* ev_after_gateup) {
    cudaEvent_t evb = static_cast<cudaEvent_t>(ev_before_gateup);
    cudaEvent_t eva = static_cast<cudaEvent_t>(ev_after_gateup);
    if (!plan) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", T);
    if (T == 0) return MOE_OK;
    if ((int64_t)T * plan->d.route.top_k > (int64_t)1 << 30) return fail(MOE_ERR_INVALID_ARG, "T too large");
    if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "x / out are NULL");
    if (!aligned(x, 16) || !aligned(out, 16)) return fail(MOE_ERR_INVALID_ARG, "x / out not 16-byte aligned");
    const moe_layer_desc& d = plan->d;
    const LayerWs w = layer_ws(d, T);
    if (!workspace || ws_bytes < w.total)
        return fail(MOE_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace ? ws_bytes : 0, w.total);
    if (!aligned(workspace, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int E = d.route.n_experts, k = d.route.top_k, H = d.hidden, I = d.intermediate;
    const void* x_res = x;                         // the call's x (the residual stream with a pre-norm)
    if (d.norm_gamma && !w.norm_in_chain) {
        // pre-norm as its own launch: the layer then reads u
        void* u = at<void>(workspace, w.u);
        cudaError_t e0 = launch_rmsnorm_bf16(static_cast<const float*>(x), d.norm_gamma, T, H, d.norm_eps, u, s);
        if (e0 != cudaSuccess) return cuda_fail(e0, "rmsnorm kernel");
        x = u;
    }
    const bool xb = input_bf16(d);
    WsHeader* hdr = at<WsHeader>(workspace, w.hdr);
    float* logits = at<float>(workspace, w.logits);
    int32_t* ids = at<int32_t>(workspace, w.ids);
    float* gw = at<float>(workspace, w.w);
    int32_t* sorted = at<int32_t>(workspace, w.sorted);
    int32_t* ppos = at<int32_t>(workspace, w.pair_pos);
    int32_t* offs = at<int32_t>(workspace, w.offsets);
    cudaError_t err;
    if (!w.tc && w.chain) {
        DecodeArgs da = decode_shape_args(d, T);
        da.x = w.norm_in_chain ? x_res : x;
        da.x_bf16 = w.norm_in_chain ? false : xb;
        da.norm_gamma = w.norm_in_chain ? d.norm_gamma : nullptr;
        da.norm_eps = d.norm_eps;
        da.logits = logits; da.ids = ids; da.gw = gw; da.sorted = sorted; da.offsets = offs; da.pair_pos = ppos;
        da.h = at<float>(workspace, w.h);
        da.h_s = at<float>(workspace, w.sh_h);
        da.hq = at<uint8_t>(workspace, w.hq);
        da.hq_s = at<uint8_t>(workspace, w.hq_s);
        da.out = out;
        da.accumulate = d.accumulate != 0;
        da.hdr = hdr;
        err = launch_decode_chain(da, s, evb, eva);
        if (err != cudaSuccess) return cuda_fail(err, "decode chain kernels");
        return MOE_OK;
    }
    err = w.router_tc ? launch_router_tc(x, T, H, d.W_router, E, logits, at<void>(workspace, w.wsplit), hdr, s)
                      : launch_router_logits(x, xb, T, H, d.W_router, E, logits, hdr, s);
    if (err != cudaSuccess) return cuda_fail(err, "router logits kernel");
    err = launch_topk(d.route, logits, d.bias, T, ids, gw, nullptr, s);
    if (err != cudaSuccess) return cuda_fail(err, "top-k kernel");
    err = launch_permute(ids, T, k, E, sorted, offs, ppos, hdr, at<int32_t>(workspace, w.chunk), s, d.expert_counts);
    if (err != cudaSuccess) return cuda_fail(err, "permute kernel");
    float* y = at<float>(workspace, w.y);
    const float* shared = nullptr;
    if (w.tc) {
        TcFfnArgs a{};
        a.qtype = kernel_qtype(d.gate.qtype);
        a.q80r = d.gate.qtype == MOE_Q8_0_R;
        a.wg = static_cast<const uint8_t*>(d.gate.data);
        a.wu = static_cast<const uint8_t*>(d.up.data);
        a.wd = static_cast<const uint8_t*>(d.down.data);
        a.stride_gu = d.gate.expert_stride_bytes;
        a.stride_d = d.down.expert_stride_bytes;
        a.E = E; a.k = k; a.H = H; a.I = I; a.T = T;
        a.identity = false;
        a.x = x; a.x_bf16 = xb; a.convert_x = true;
        a.sorted_pairs = sorted; a.offsets = offs;
        a.x16 = at<__half>(workspace, w.x16);
        a.h16 = at<__half>(workspace, w.h);
        a.y = nullptr;
        a.y16 = at<__half>(workspace, w.y);          // fp16 per-pair outputs, read by the combine
        a.tb_list = at<int4>(workspace, w.tiles);
        a.hdr = hdr;
        a.ev_before_gateup = evb;
        a.ev_after_gateup = eva;
        err = launch_tc_expert_ffn(a, s);
        if (err != cudaSuccess) return cuda_fail(err, "tensor-core expert kernels");
        if (d.shared_intermediate > 0) {
            TcFfnArgs b = a;
            b.qtype = kernel_qtype(d.s_gate.qtype);
            b.q80r = d.s_gate.qtype == MOE_Q8_0_R;
            b.wg = static_cast<const uint8_t*>(d.s_gate.data);
            b.wu = static_cast<const uint8_t*>(d.s_up.data);
            b.wd = static_cast<const uint8_t*>(d.s_down.data);
            b.stride_gu = b.stride_d = 0;
            b.E = 1; b.k = 1; b.I = d.shared_intermediate;
            b.identity = true; b.convert_x = false;
            b.sorted_pairs = nullptr; b.offsets = nullptr; b.tb_list = nullptr;
            b.ev_before_gateup = b.ev_after_gateup = nullptr;
            b.h16 = at<__half>(workspace, w.sh_h);
            b.y = at<float>(workspace, w.sh_y);
            b.y16 = nullptr;
            err = launch_tc_expert_ffn(b, s);
            if (err != cudaSuccess) return cuda_fail(err, "tensor-core shared expert kernels");
            shared = b.y;
        }
    } else {
        if (evb && (err = cudaEventRecord(evb, s)) != cudaSuccess) return cuda_fail(err, "event record");
        err = routed_gateup(d.gate, d.up, E, x, xb, T, H, I, sorted, offs, k, at<float>(workspace, w.h), hdr, s);
        if (err != cudaSuccess) return cuda_fail(err, "gate/up kernel");
        if (eva && (err = cudaEventRecord(eva, s)) != cudaSuccess) return cuda_fail(err, "event record");
        err = routed_down(d.down, E, at<float>(workspace, w.h), T, H, I, sorted, offs, k, y, hdr, s);
        if (err != cudaSuccess) return cuda_fail(err, "down kernel");
        moe_status st;
        if (d.shared_intermediate > 0) {
            float* sy = at<float>(workspace, w.sh_y);
            st = run_ffn(d.s_gate, d.s_up, d.s_down, 1, x, xb, T, H, d.shared_intermediate, nullptr, nullptr, 1,
                         at<float>(workspace, w.sh_h), sy, s);
            if (st) return st;
            shared = sy;
        }
    }
    err = w.tc ? launch_combine16(at<__half>(workspace, w.y), gw, ppos, T, k, H, shared, d.accumulate != 0, out, s)
               : launch_combine(y, gw, ppos, T, k, H, shared, d.accumulate != 0, out, s);
    if (err != cudaSuccess) return cuda_fail(err, "combine kernel");
    return MOE_OK;
}

moe_status moe_layer_debug_views(const moe_layer_plan* plan, int T, void* workspace, int32_t** topk_ids,
                                 float** topk_w, int32_t** offsets) {
    if (!plan || !workspace) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    const LayerWs w = layer_ws(plan->d, T);
    if (topk_ids) *topk_ids = at<int32_t>(workspace, w.ids);
    if (topk_w) *topk_w = at<float>(workspace, w.w);
    if (offsets) *offsets = at<int32_t>(workspace, w.offsets);
    return MOE_OK;
}

moe_status moe_read_device_status(const moe_layer_plan* plan, int T, void* workspace, int32_t* code,
                                  moe_stream_t stream) {
    if (!plan || !workspace || !code) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    void* hdr = at<void>(workspace, layer_ws(plan->d, T).hdr);
    return moe_permute_read_device_status(0, 1, 1, hdr, code, stream);
}

}  // extern "C"
