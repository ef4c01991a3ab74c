// ggemm.cu -- grouped expert GEMM on the 5th-generation tensor cores (tcgen05).
//
// At prompt sizes the pages run "each expert over all its tokens at once" on
// tensor cores ("bloomery V4.1 README", "Batched prompts"; "bloomery README
// 0.3.1", "Why it is fast": prompts as tensor-core GEMMs).  Here each expert's
// tokens form a dense GEMM against that expert's GGUF weights:
//   GATEUP: h[i, r] = silu(Wg[e][r] . x_t) * (Wu[e][r] . x_t)     (fp16 out)
//   DOWN  : y[i, n] = Wd[e][n] . h[i]     (fp32 out; fp16 for the layer, whose combine sums in fp32)
// Tile = 128 weight rows (MMA M; gate/up: 128 rows of each) x one token block of the expert
// (MMA N: up to 256 pairs for Q4_K, 128 for Q8_0), K in steps of 64.  Weights are
// dequantized from Q4_K / Q8_0 to fp16 in shared memory (128-byte swizzled K-major tiles);
// token rows arrive in the same layout (gate/up: the producers copy the block's x16 rows,
// found through the pair order, 16 bytes a thread with cp.async; down: one TMA box of
// consecutive h16 rows); one thread issues tcgen05.mma with the
// accumulators in TMEM (fp32); tcgen05.ld reads them back for the epilogue.  Persistent CTAs
// (one per SM) walk a device-built list of token blocks, so the launch needs no host
// knowledge of the per-expert counts.
//
// Warp roles: producer warps (16 for the Q4_K gate/up, else 8) copy the raw blocks with
// cp.async, dequantize them and issue the token rows; gate/up producers also run the
// SwiGLU epilogue (its accumulators fill all 512 TMEM columns); down has 8 epilogue warps
// and two accumulator buffers, so its epilogue overlaps the next tile; the last warp owns
// TMEM and issues the MMAs.  Pipeline per global k-step g: a producer waits until the A
// stage g%2 is free (MMA(g-2) done), waits for raw(g) (and, gate/up, B(g)), dequantizes it,
// arrives on full[g%4] (down: which also counts the TMA bytes of B(g)), then issues raw and
// B of step g + D (D = 2 for gate/up, 3 for down, across tile boundaries); the MMA warp
// waits full[g%4], issues four k-substeps and commits to empty[g%4].  Every wait is bounded
// (globaltimer); on timeout the kernel records MOE_ERR_TIMEOUT, drains its MMAs, waits
// (bounded) on the barriers of the copies still in flight, frees TMEM and returns.
#include <algorithm>
#include <cuda.h>   // CUtensorMap and its enums (the encoder is fetched from the driver at run time)

#include "internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kBNMin = 128;                       // token-block width bound used to size the tile list
// Producer warps: 16 for the Q4_K gate/up (a thread dequantizes half of a row's 64-weight
// k-step, so that enough warps hide the latency of their dependent steps), 8 otherwise (Q4_K
// down: half a k-step per thread already; Q8_0: its raw blocks need the shared memory).
template <int QT, int MODE>
__host__ __device__ constexpr int tc_pw() { return QT == MOE_Q4_K && MODE == 0 ? 16 : 8; }
constexpr int kAStages = 2, kBStages = 4;
// How many k-steps ahead of the dequantization the raw blocks and token rows are issued: 2
// for gate/up (its shared memory is full), 3 for down (its k-steps are half as long, so two
// of them do not cover the latency of a DRAM read); one raw slot per step in flight.
template <int MODE>
__host__ __device__ constexpr int tc_dist() { return MODE == 0 ? 2 : 3; }

enum { kGateUp = 0, kDown = 1 };

// Token-block width (MMA N) per weight type: 256 for Q4_K (each dequantized weight tile
// feeds twice the MMA work), 128 for Q8_0 (its raw blocks need the shared memory).
template <int QT>
__host__ __device__ constexpr int tc_bn() { return QT == MOE_Q4_K ? 256 : 128; }

__device__ __forceinline__ float s8_f(uint32_t word, int b) {    // signed byte b -> float, exact
    return __int_as_float(__byte_perm(word ^ 0x80808080u, 0x4B00u, 0x5440u | (uint32_t)b)) - 8388736.0f;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
// fp16 operands and outputs: a value that rounds to inf (or is NaN) is reported, not hidden.
__device__ __forceinline__ bool half_finite(__half h) { return (__half_as_ushort(h) & 0x7C00u) != 0x7C00u; }
// max that keeps NaN (so that a NaN h is reported like an overflow)
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
// One report per warp: the status word becomes MOE_ERR_DEVICE_CHECK unless it holds an error.
__device__ __forceinline__ void report_out_of_range(bool bad, int lane, WsHeader* hdr) {
    if (__any_sync(0xffffffffu, bad) && lane == 0 && hdr) atomicCAS(&hdr->status, (int)MOE_OK, (int)MOE_ERR_DEVICE_CHECK);
}

// Eight fp16 weights of one Q4_K word into two 16-byte halves of a chunk: the low nibbles of
// bytes b0..b3 are elements 0..3 of sub-block 2c, the high nibbles elements 0..3 of 2c+1.
// A low nibble q placed under the fp16 exponent of 1024 reads as 1024 + q; a high nibble,
// left in place (16q) under the exponent of 64 (one unit in the last place = 1/16), reads as
// 64 + q.  One exact subtraction leaves q, and one fp16 FMA applies the sub-block's scale and
// min: w = s*q - m (rounded once).
struct Q4H2 {
    __half2 s_lo, m_lo, s_hi, m_hi;       // m already negated
};
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
// w -> (lo: elements 0,1 | 2,3 of sub-block 2c) and (hi: the same of 2c+1), as fp16 pairs
__device__ __forceinline__ void q4_word_h2(uint32_t w, const Q4H2& c, uint32_t (&lo)[2], uint32_t (&hi)[2]) {
    const __half2 k1024 = __float2half2_rn(1024.0f), k64 = __float2half2_rn(64.0f);
    const uint32_t t01 = __byte_perm(w, 0u, 0x4140u);        // [b0, 0, b1, 0]
    const uint32_t t23 = __byte_perm(w, 0u, 0x4342u);        // [b2, 0, b3, 0]
    lo[0] = h2u(__hfma2(__hsub2(u2h((t01 & 0x000F000Fu) | 0x64006400u), k1024), c.s_lo, c.m_lo));
    lo[1] = h2u(__hfma2(__hsub2(u2h((t23 & 0x000F000Fu) | 0x64006400u), k1024), c.s_lo, c.m_lo));
    hi[0] = h2u(__hfma2(__hsub2(u2h((t01 & 0x00F000F0u) | 0x54005400u), k64), c.s_hi, c.m_hi));
    hi[1] = h2u(__hfma2(__hsub2(u2h((t23 & 0x00F000F0u) | 0x54005400u), k64), c.s_hi, c.m_hi));
}
// Scales and negated mins of the eight sub-blocks of a Q4_K block header as fp16 pairs:
// sc[c] = (d*sc_2c, d*sc_2c+1) and mn[c] = (-dmin*m_2c, -dmin*m_2c+1) for k-step c of the
// super-block.  The 6-bit codes (public Q4_K packing: codes 0-3 in the low six bits of scale
// bytes 0-3 and 4-7, codes 4-7 from the nibbles of bytes 8-11 and the top two bits of bytes
// 0-7) become exact fp16 integers (1024 + b under the exponent of 1024, minus 1024); each
// product is rounded once, as the exact product rounded to fp16.
struct Q4Scales {
    __half2 sc0, sc1, sc2, sc3, mn0, mn1, mn2, mn3;     // named, so that selecting one stays in registers
};
__device__ __forceinline__ Q4Scales q4k_scales_h2(const uint4& hd) {
    const uint32_t sc_lo = hd.y & 0x3F3F3F3Fu, m_lo = hd.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
    const __half2 d2 = u2h(__byte_perm(hd.x, 0u, 0x1010u));                  // (d, d)
    const __half2 nm2 = u2h(__byte_perm(hd.x, 0u, 0x3232u) ^ 0x80008000u);    // (-dmin, -dmin)
    const __half2 k1024 = __float2half2_rn(1024.0f);
    auto pair = [&](uint32_t v, uint32_t sel) { return __hsub2(u2h(__byte_perm(v, 0x64u, sel)), k1024); };
    Q4Scales r;
    r.sc0 = __hmul2(pair(sc_lo, 0x4140u), d2);
    r.sc1 = __hmul2(pair(sc_lo, 0x4342u), d2);
    r.sc2 = __hmul2(pair(sc_hi, 0x4140u), d2);
    r.sc3 = __hmul2(pair(sc_hi, 0x4342u), d2);
    r.mn0 = __hmul2(pair(m_lo, 0x4140u), nm2);
    r.mn1 = __hmul2(pair(m_lo, 0x4342u), nm2);
    r.mn2 = __hmul2(pair(m_hi, 0x4140u), nm2);
    r.mn3 = __hmul2(pair(m_hi, 0x4342u), nm2);
    return r;
}

// Raw bytes staged per producer thread per k-step.
template <int QT, int MODE>
struct RawCfg {
    static constexpr int kBytes = QT == MOE_Q4_K ? 32 : 80;   // Q4_K: header + up to 16 quant bytes
};

struct TileInfo {
    int e, tok0, ntok, m0, n_inst;
};

struct TcParams {
    CUtensorMap tmap_b;          // DOWN: B rows h16 [P][K] (box 64 x BN, 128-byte swizzle)
    const uint8_t* w0;           // gate (GATEUP) or down (DOWN) weights
    const uint8_t* w1;           // up (GATEUP)
    int64_t expert_stride;
    int rows;                    // weight rows per expert (I for GATEUP, H for DOWN)
    int K;                       // H for GATEUP, I for DOWN
    int k;                       // top-k (token of pair = sorted_pairs[i] / k)
    const int32_t* sorted_pairs; // GATEUP gather map (NULL: identity)
    const __half* x16;           // GATEUP: token rows [T][K] fp16 (copied 16 bytes a thread)
    const int4* tb_list;         // [0].x = number of token blocks, then (e, tok0, ntok, 0); NULL: identity
    int n_identity;              // identity mode: tokens
    int bn;                      // token-block width of the list (tc_bn)
    int b_box_rows;              // DOWN: rows of the B box (BN, or P when fewer)
    __half* h_out;               // GATEUP: [P][rows] fp16
    float* y_out;                // DOWN: [P][rows] fp32, or
    __half* y16_out;             //       [P][rows] fp16 when set
    WsHeader* hdr;
    uint64_t wait_ns;            // limit of every bounded wait
    int stall;                   // test setting: the MMA warp's first wait never completes
};

// The full tile description for tile index t.
__device__ __forceinline__ bool tile_at(const TcParams& p, int n_mb, int t, int n_tb, TileInfo& ti) {
    const int tb = t / n_mb, mb = t - tb * n_mb;
    if (tb >= n_tb) return false;
    if (p.tb_list) {
        const int4 v = p.tb_list[1 + tb];
        ti.e = v.x; ti.tok0 = v.y; ti.ntok = v.z;
    } else {
        ti.e = 0; ti.tok0 = tb * p.bn; ti.ntok = min(p.bn, p.n_identity - ti.tok0);
    }
    ti.m0 = mb * kBM;
    ti.n_inst = (ti.ntok + 15) & ~15;
    return true;
}

// Warp layout: producers, then (DOWN) 8 epilogue warps, then the MMA warp.  DOWN keeps
// two accumulators in TMEM so that its epilogue overlaps the next tile's main loop; GATEUP
// needs all 512 columns for one tile (gate and up, 256 tokens each) and lets the producers
// run its epilogue.
template <int MODE>
__host__ __device__ constexpr int tc_epi_warps() { return MODE == kDown ? 8 : 0; }
template <int QT, int MODE>
__host__ __device__ constexpr int tc_threads() { return 32 * tc_pw<QT, MODE>() + 32 * tc_epi_warps<MODE>() + 32; }

template <int QT, int MODE>
__global__ void __launch_bounds__(tc_threads<QT, MODE>(), 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    constexpr int kAStageBytes = (MODE == kGateUp ? 2 : 1) * kBM * 128;
    constexpr int BN = tc_bn<QT>();
    constexpr int kBStageBytes = BN * 128;
    constexpr int kRawBytes = RawCfg<QT, MODE>::kBytes;
    constexpr int kPW = tc_pw<QT, MODE>();
    constexpr int kNP = kPW * 32;
    constexpr int kMats = MODE == kGateUp ? 2 : 1;
    constexpr int kSplit = kNP / (kBM * kMats);       // threads per (row, matrix) of a k-step
    constexpr int kRawSlotBytes = kNP * kRawBytes;
    constexpr int kDist = tc_dist<MODE>();
    constexpr int kRawSlots = kDist;
    constexpr int kEpiWarps = tc_epi_warps<MODE>();
    constexpr int kMmaWarp = kPW + kEpiWarps;
    constexpr uint32_t kAccCols = (MODE == kGateUp ? 2 : 1) * BN;
    constexpr int kAccBufs = kEpiWarps > 0 ? 2 : 1;
    constexpr uint32_t kTmemCols = kAccCols * kAccBufs;
    static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of two");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = sA + kAStages * kAStageBytes;
    uint8_t* sRaw = sB + kBStages * kBStageBytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sRaw + kRawSlots * kRawSlotBytes);
    uint64_t* full = bar;            // [4]: A dequantized (one arrival per producer warp) + B landed (tx bytes)
    uint64_t* empty = bar + 4;       // [4]
    uint64_t* accf = bar + 8;        // [2]: accumulator buffer complete
    uint64_t* tfree = bar + 10;      // [2]: accumulator buffer read out by the epilogue warps
    uint64_t* drain = bar + 12;      // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 13);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 14);
    uint64_t* never = bar + 15;      // [1]: the test stall (initialized, never arrived on)
    int* max_issued = reinterpret_cast<int*>(bar + 16);   // k-steps the producers issued (abort drain)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) { mbar_init(&full[i], kPW); mbar_init(&empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&accf[i], 1); mbar_init(&tfree[i], kEpiWarps > 0 ? kEpiWarps : 1); }
        mbar_init(drain, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        *max_issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (MODE == kDown) asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tmap_b) : "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *tmem_slot;

    const int n_mb = p.rows / kBM;
    const int n_tb = p.tb_list ? p.tb_list[0].x : (p.n_identity + BN - 1) / BN;
    const int n_tiles = n_tb * n_mb;
    const int nk = p.K / kBK;
    const int nblk_row = QT == MOE_Q4_K ? p.K / kQ4KWeights : p.K / kQ80Weights;
    const int64_t rb = QT == MOE_Q4_K ? (int64_t)nblk_row * kQ4KBytes
                                      : (QT == MOE_Q8_0_R ? q80r_row_bytes(p.K) : (int64_t)nblk_row * kQ80Bytes);

    int n_issued = 0, n_arrived = 0;                // producers: k-steps issued / arrived on full[]
    if (warp < kPW) {
        // ======================= producers (+ GATEUP epilogue) =======================
        const int prow = tid & 127;                 // weight row within the tile
        const int pmat = MODE == kGateUp ? (tid >> 7) & 1 : 0;   // matrix: 0 gate / down, 1 up
        const int part = (tid >> 7) / kMats;        // which 1/kSplit of the row's k-step
        // ---- issue cursor: runs two k-steps ahead of the dequantization, across tile
        // boundaries, so that a tile's first raw blocks and token rows are in flight while the
        // previous tile finishes
        int is_t = blockIdx.x, is_kb = 0;
        TileInfo iti{};
        bool is_valid = false;
        const uint8_t* is_wrow = nullptr;
        // GATEUP: the x16 rows this thread copies for the cursor's tile (NULL past its tokens)
        constexpr int kBRowsPass = kNP / 8, kBPass = BN / kBRowsPass;
        static_assert(kBPass * kBRowsPass == BN, "B rows per producer pass");
        const uint8_t* is_xb[kBPass];
        auto is_tile = [&]() {
            is_valid = is_t < n_tiles && tile_at(p, n_mb, is_t, n_tb, iti);
            if (!is_valid) return;
            is_wrow = (pmat == 1 ? p.w1 : p.w0) + (int64_t)iti.e * p.expert_stride + (int64_t)(iti.m0 + prow) * rb;
            if (MODE == kGateUp) {
                // thread t copies 16-byte chunk t % 8 of columns t / 8 + kBRowsPass * j of the block
#pragma unroll
                for (int j = 0; j < kBPass; ++j) {
                    const int r = (tid >> 3) + kBRowsPass * j;
                    if (r < iti.ntok) {
                        const int i = iti.tok0 + r;
                        const int row = p.sorted_pairs ? p.sorted_pairs[i] / p.k : i;
                        is_xb[j] = reinterpret_cast<const uint8_t*>(p.x16 + (int64_t)row * p.K) + 16 * (tid & 7);
                    } else {
                        is_xb[j] = nullptr;
                    }
                }
            }
        };
        // B of the cursor's k-step into stage `stage`: GATEUP copies the block's x16 rows 16 bytes
        // a thread (cp.async into the 128-byte-swizzled layout, in the same commit group as the
        // raw blocks, so the wait before the dequantization covers both; columns past the block's
        // tokens are not loaded and never stored), DOWN loads its BN consecutive h16 rows in one
        // TMA box that completes on full[stage]
        auto issue_b = [&](int kb, int stage) {
            uint8_t* dst = sB + stage * kBStageBytes;
            uint64_t* fb = &full[stage];
            if (MODE == kGateUp) {
#pragma unroll
                for (int j = 0; j < kBPass; ++j)
                    if (is_xb[j]) cp_async16(dst + swz((tid >> 3) + kBRowsPass * j, tid & 7), is_xb[j] + kb * 128, 16u);
            } else if (tid == 0) {
                mbar_expect_tx(fb, (uint32_t)p.b_box_rows * 128u);
                tma_load_2d(dst, &p.tmap_b, kb * kBK, iti.tok0, fb);
            }
        };
        auto issue_raw = [&](int kb, int slot) {
            uint8_t* dst = sRaw + slot * kRawSlotBytes + tid * kRawBytes;
            if (QT == MOE_Q4_K) {
                const uint8_t* blk = is_wrow + (int64_t)(kb >> 2) * kQ4KBytes;
                if ((kb & 3) == 0) cp_async16(dst, blk, 16u);                 // header, once per super-block
                const uint8_t* qs = blk + 16 + 32 * (kb & 3) + (32 / kSplit) * part;
                if constexpr (kSplit == 2) cp_async16(dst + 16, qs, 16u);
                else cp_async8(dst + 16, qs);
            } else if (QT == MOE_Q8_0_R) {
                // repacked: the k-step's 64 quants (16-byte aligned), then its two scales
                const uint8_t* qsrc = is_wrow + (int64_t)kb * 64;
#pragma unroll
                for (int w = 0; w < 4; ++w) cp_async16(dst + 16 * w, qsrc + 16 * w, 16u);
                cp_async4(dst + 64, is_wrow + (int64_t)nblk_row * 32 + 4 * kb);
            } else {
                const uint8_t* src = is_wrow + (int64_t)kb * 2 * kQ80Bytes;     // two blocks, 68 bytes
#pragma unroll
                for (int w = 0; w < 17; ++w) cp_async4(dst + 4 * w, src + 4 * w);
            }
        };
        // issue global k-step gs (the cursor's) and advance the cursor; always one commit group
        auto issue_next = [&](uint32_t gs) {
            n_issued = (int)gs + 1;
            if (is_valid) {
                issue_raw(is_kb, gs % kRawSlots);
                issue_b(is_kb, gs % kBStages);
                if (++is_kb == nk) {
                    is_kb = 0;
                    is_t += gridDim.x;
                    is_tile();
                }
            }
            cp_commit();
        };
        is_tile();
        for (int i = 0; i < kDist; ++i) issue_next((uint32_t)i);

        uint32_t g = 0;                             // global k-step counter
        int tile_iter = 0;
        Q4Scales qs4{};                             // Q4_K: scales of the current super-block
        for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x, ++tile_iter) {
            TileInfo ti;
            if (!tile_at(p, n_mb, t, n_tb, ti)) break;
            bool ok = true;
            for (int kb = 0; kb < nk; ++kb, ++g) {
                // A stage g%2 was last read by MMA(g-2) (with kDist == 3 already waited for below)
                if (kDist == 2 && g >= 2 &&
                    !mbar_wait(&empty[(g + 2) & 3], ((g - 2) >> 2) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
                cp_wait<kDist - 1>();                // raw(g) has landed (only later steps may be pending)
                // ---- dequantize k-step kb into A stage g%2
                const uint8_t* raw = sRaw + (g % kRawSlots) * kRawSlotBytes + tid * kRawBytes;
                uint8_t* arow = sA + (g % kAStages) * kAStageBytes + pmat * kBM * 128;
                if (QT == MOE_Q4_K) {
                    // the header (read at the super-block's first k-step) gives the scales of all four
                    const int c = kb & 3;
                    if (c == 0) qs4 = q4k_scales_h2(*reinterpret_cast<const uint4*>(raw));
                    const uint32_t scp = c == 0 ? h2u(qs4.sc0) : c == 1 ? h2u(qs4.sc1) : c == 2 ? h2u(qs4.sc2) : h2u(qs4.sc3);
                    const uint32_t mnp = c == 0 ? h2u(qs4.mn0) : c == 1 ? h2u(qs4.mn1) : c == 2 ? h2u(qs4.mn2) : h2u(qs4.mn3);
                    const Q4H2 hc{u2h(__byte_perm(scp, 0u, 0x1010u)), u2h(__byte_perm(mnp, 0u, 0x1010u)),
                                  u2h(__byte_perm(scp, 0u, 0x3232u)), u2h(__byte_perm(mnp, 0u, 0x3232u))};
                    // this thread's quant bytes: elements (32 / kSplit) * part .. of sub-blocks 2c (low
                    // nibbles) and 2c + 1 (high nibbles); each pair of words fills chunk ch (elements
                    // 8ch..8ch+7 of 2c) and chunk 4 + ch (the same elements of 2c + 1)
                    constexpr int kWords = 8 / kSplit;
                    uint32_t qw[kWords];
#pragma unroll
                    for (int w = 0; w < kWords; ++w) qw[w] = reinterpret_cast<const uint32_t*>(raw + 16)[w];
#pragma unroll
                    for (int w2 = 0; w2 < kWords / 2; ++w2) {
                        uint32_t la[2], ha[2], lb[2], hb[2];
                        q4_word_h2(qw[2 * w2], hc, la, ha);
                        q4_word_h2(qw[2 * w2 + 1], hc, lb, hb);
                        const int ch = part * (kWords / 2) + w2;
                        *reinterpret_cast<uint4*>(arow + swz(prow, ch)) = make_uint4(la[0], la[1], lb[0], lb[1]);
                        *reinterpret_cast<uint4*>(arow + swz(prow, 4 + ch)) = make_uint4(ha[0], ha[1], hb[0], hb[1]);
                    }
                } else {
                    // Q8_0: 68 bytes = d0, q0[32], d1, q1[32]; repacked: q0[32], q1[32], d0, d1
                    uint32_t wv[17];
#pragma unroll
                    for (int w = 0; w < 17; ++w) wv[w] = reinterpret_cast<const uint32_t*>(raw)[w];
                    const uint32_t dw0 = QT == MOE_Q8_0_R ? wv[16] & 0xFFFFu : wv[0] & 0xFFFFu;
                    const uint32_t dw1 = QT == MOE_Q8_0_R ? wv[16] >> 16 : wv[8] >> 16;
                    const float d0 = __half2float(__ushort_as_half((unsigned short)dw0));
                    const float d1 = __half2float(__ushort_as_half((unsigned short)dw1));
                    // 8 weights (chunk ch of the k-step) from byte b0 of the 68 with scale d; the byte
                    // offsets stay compile-time constants, so wv stays in registers
                    auto chunk = [&](int ch, int b0, float d) {
                        float v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int off = b0 + i;
                            v[i] = d * s8_f(wv[off >> 2], off & 3);
                        }
                        *reinterpret_cast<uint4*>(arow + swz(prow, ch)) =
                            make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]),
                                       pack_h2(v[6], v[7]));
                    };
                    if (QT == MOE_Q8_0_R) {
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            if (kSplit == 2 && (ch >> 2) != part) continue;   // DOWN: this thread's block only
                            chunk(ch, 8 * ch, ch < 4 ? d0 : d1);
                        }
                    } else {
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            if (kSplit == 2 && (ch >> 2) != part) continue;
                            chunk(ch, ch < 4 ? 2 + 8 * ch : 36 + 8 * (ch - 4), ch < 4 ? d0 : d1);
                        }
                    }
                }
                // every thread makes its own A writes visible to the tensor core's (async) proxy;
                // the warp then arrives once
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[g & 3]);
                n_arrived = (int)g + 1;
                // B stage (g + kDist) % 4 was last read by MMA(g + kDist - 4)
                if (kDist == 3 && g >= 1 &&
                    !mbar_wait(&empty[(g - 1) & 3], ((g - 1) >> 2) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
                issue_next(g + kDist);
            }
            if (!ok) break;
            if constexpr (MODE == kGateUp) {
                // ---- epilogue: wait for the accumulators of this tile, h = SiLU(gate) * up
                if (!mbar_wait(&accf[0], tile_iter & 1, abort_flag, p.wait_ns)) break;
                tc_after();
                // warp w reads TMEM lanes 32 (w % 4).. and every (kPW / 4)-th group of 16 columns;
                // lanes 2i and 2i + 1 trade one value of each column pair, so that each stores two
                // adjacent rows of one column as a half2 (even lane: even column, odd: odd column)
                const int q = warp & 3;
                const int m = q * 32 + lane;
                const bool odd = (lane & 1) != 0;
                __half* hrow = p.h_out + (int64_t)(ti.tok0 + (odd ? 1 : 0)) * p.rows + ti.m0 + (m & ~1);
                float amax = 0.0f;                       // largest |h| of the block's columns (NaN kept)
                for (int c16 = (warp >> 2) * 16; c16 < ti.n_inst; c16 += 16 * (kPW / 4)) {
                    uint32_t a[16], u[16];
                    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c16, a);
                    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(BN + c16), u);
                    tmem_ld_wait();
                    const int nv = ti.ntok - c16;       // columns of this group that hold tokens
                    float h[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float gv = __uint_as_float(a[j]), uv = __uint_as_float(u[j]);
                        h[j] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                        if (j < nv) amax = fmax_nan(amax, fabsf(h[j]));
                    }
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float recv = __shfl_xor_sync(0xffffffffu, odd ? h[j] : h[j + 1], 1);
                        const float keep = odd ? h[j + 1] : h[j];
                        const __half2 hv = odd ? __floats2half2_rn(recv, keep) : __floats2half2_rn(keep, recv);
                        if (j + (odd ? 1 : 0) < nv) *reinterpret_cast<__half2*>(hrow + (int64_t)(c16 + j) * p.rows) = hv;
                    }
                }
                // a value at or beyond 65520 rounds to inf in fp16
                report_out_of_range(!(amax < 65520.0f), lane, p.hdr);
                tc_before();
            }
        }
        cp_wait_all();
        if (lane == 0) atomicMax(max_issued, n_issued);
    } else if (warp < kMmaWarp) {
        // ======================= DOWN epilogue warps =======================
        // epilogue warp e reads TMEM lanes 32q.. (q = warp % 4) and the 64-column chunks
        // e / 4, e / 4 + 2, ... of the accumulator
        const int q = warp & 3;
        const int chunk0 = (warp - kPW) >> 2;
        const int m = q * 32 + lane;
        const bool odd = (lane & 1) != 0;
        int j = 0;
        for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x, ++j) {
            TileInfo ti;
            if (!tile_at(p, n_mb, t, n_tb, ti)) break;
            const int b = j & 1;
            if (!mbar_wait(&accf[b], (j >> 1) & 1, abort_flag, p.wait_ns)) break;
            tc_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * kAccCols;
            // fp16: lanes 2i, 2i+1 swap one value so that each stores rows (m & ~1, m | 1) of one
            // column as a pair (even lane: even column, odd lane: odd column)
            __half* y16row = p.y16_out + (int64_t)(ti.tok0 + (odd ? 1 : 0)) * p.rows + ti.m0 + (m & ~1);
            float* yrow = p.y_out + (int64_t)ti.tok0 * p.rows + ti.m0 + m;
            bool out_of_range = false;                   // a y value beyond the fp16 range
            for (int c64 = 64 * chunk0; c64 < ti.n_inst; c64 += 128) {
                uint32_t a[4][16];
#pragma unroll
                for (int i = 0; i < 4; ++i) tmem_ld16(tb + (uint32_t)(c64 + 16 * i), a[i]);
                tmem_ld_wait();
                if (p.y16_out) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 2) {
                            const float v0 = __uint_as_float(a[i][jj]), v1 = __uint_as_float(a[i][jj + 1]);
                            const float recv = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                            const float keep = odd ? v1 : v0;
                            const __half2 hv = odd ? __floats2half2_rn(recv, keep) : __floats2half2_rn(keep, recv);
                            const int col = c64 + 16 * i + jj;          // this lane stores column col + odd
                            if (col + (odd ? 1 : 0) < ti.ntok) {
                                out_of_range |= !half_finite(__low2half(hv)) || !half_finite(__high2half(hv));
                                *reinterpret_cast<__half2*>(y16row + (int64_t)col * p.rows) = hv;
                            }
                        }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int col = c64 + 16 * i + jj;
                            if (col < ti.ntok) yrow[(int64_t)col * p.rows] = __uint_as_float(a[i][jj]);
                        }
                }
            }
            report_out_of_range(out_of_range, lane, p.hdr);
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfree[b]);
        }
    } else {
        // ======================= MMA issuer =======================
        uint32_t g = 0;
        bool issued = false;
        int j = 0;
        for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x, ++j) {
            TileInfo ti;
            if (!tile_at(p, n_mb, t, n_tb, ti)) break;
            const uint32_t idesc = idesc_mma(kBM, ti.n_inst, false);
            const int b = j % kAccBufs;
            // the accumulator buffer's previous tile has been read out (GATEUP: the producers
            // only reach this tile's first k-step after their epilogue)
            if (kEpiWarps > 0 && j >= kAccBufs) {
                if (!mbar_wait(&tfree[b], ((j / kAccBufs) - 1) & 1, abort_flag, p.wait_ns)) break;
                tc_after();
            }
            const uint32_t acc = tmem + (uint32_t)b * kAccCols;
            bool ok = true;
            for (int kb = 0; kb < nk; ++kb, ++g) {
                uint64_t* fb = p.stall && g == 0 ? never : &full[g & 3];     // (test stall)
                if (!mbar_wait(fb, fb == never ? 0u : (g >> 2) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
                tc_after();
                if (lane == 0) {
                    const uint32_t a0 = su32(sA + (g % kAStages) * kAStageBytes);
                    const uint32_t b0 = su32(sB + (g % kBStages) * kBStageBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = sdesc(b0 + 32 * kk);
                        mma_f16(acc, sdesc(a0 + 32 * kk), bd, idesc, (kb | kk) != 0);
                        if (MODE == kGateUp)
                            mma_f16(acc + BN, sdesc(a0 + kBM * 128 + 32 * kk), bd, idesc, (kb | kk) != 0);
                    }
                    mma_commit(&empty[g & 3]);
                    if (kb == nk - 1) mma_commit(&accf[b]);
                }
                issued = true;
                __syncwarp();
            }
            if (!ok) break;
        }
        // drain: every MMA this thread issued has completed before TMEM is freed
        if (issued) {
            if (lane == 0) mma_commit(drain);
            __syncwarp();
            mbar_wait_for(drain, 0, p.wait_ns);
        }
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (*abort_flag) {
        // every thread has left its loop.  The producers' copies (cp.async) are waited for; the
        // DOWN token rows (TMA) of the last k-steps may still be in flight.  Each producer warp
        // arrives on full[] for the k-steps it has not arrived on, up to the last one any warp
        // issued, so that the phase of each such step completes exactly when its bytes land.
        // Steps older than the last four completed already: a producer issues step s only after
        // the MMAs of step s - 4, which waited for its phase.
        if (warp < kPW && lane == 0)
            for (int s = n_arrived; s < *max_issued; ++s) mbar_arrive(&full[s & 3]);
        __syncthreads();
        if (tid == 0) {
            atomicCAS(&p.hdr->status, (int)MOE_OK, (int)MOE_ERR_TIMEOUT);
            const int last = *max_issued;
            for (int s = max(0, last - 4); s < last; ++s) mbar_wait_for(&full[s & 3], (uint32_t)(s >> 2) & 1u, p.wait_ns);
        }
        tc_before();
        __syncthreads();
        tc_after();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
    }
}

// Token blocks of up to bn pairs per expert: list[0].x = count, then (e, tok0, ntok, 0).
__global__ void __launch_bounds__(1024) tile_list_kernel(const int32_t* __restrict__ offsets, int E, int bn,
                                                         int4* __restrict__ list) {
    __shared__ int warp_tot[32];
    __shared__ int total;
    const int e = threadIdx.x;
    int n = 0, o0 = 0;
    if (e < E) { o0 = offsets[e]; n = offsets[e + 1] - o0; }
    const int nb = (n + bn - 1) / bn;
    // block exclusive scan of nb
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int w = warp_tot[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += v;
        }
        warp_tot[lane] = wi - w;
        if (lane == 31) total = wi;
    }
    __syncthreads();
    const int base = inc - nb + warp_tot[warp];
    for (int b = 0; b < nb; ++b) list[1 + base + b] = make_int4(e, o0 + b * bn, min(bn, n - b * bn), 0);
    if (threadIdx.x == 0) list[0] = make_int4(total, 0, 0, 0);
}

__global__ void to_half_kernel(const void* __restrict__ x, bool bf16, int64_t n, __half* __restrict__ out,
                               WsHeader* hdr) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    bool bad = false;
    if (i < n) {
        float v[4];
        if (bf16) {
            const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(x) + i);
            v[0] = __uint_as_float(raw.x << 16); v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
            v[2] = __uint_as_float(raw.y << 16); v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
        } else {
            const float4 f = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + i);
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        }
        const uint2 h = make_uint2(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]));
        *reinterpret_cast<uint2*>(out + i) = h;
        // x beyond the fp16 range (or not finite) has no fp16 operand: report it
        bad = ((h.x & 0x7C00u) == 0x7C00u) || ((h.x & 0x7C000000u) == 0x7C000000u) ||
              ((h.y & 0x7C00u) == 0x7C00u) || ((h.y & 0x7C000000u) == 0x7C000000u);
    }
    report_out_of_range(bad, threadIdx.x & 31, hdr);
}

template <int QT, int MODE>
size_t tc_smem_bytes() {
    constexpr int a = kAStages * (MODE == kGateUp ? 2 : 1) * kBM * 128;
    constexpr int b = kBStages * tc_bn<QT>() * 128;
    constexpr int r = tc_dist<MODE>() * 32 * tc_pw<QT, MODE>() * RawCfg<QT, MODE>::kBytes;
    return (size_t)a + b + r + 256 + 1024;   // barriers + alignment slack
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// Tensor map of an fp16 matrix [rows][cols] (dense rows): boxes of 64 columns (128 bytes) x
// box_rows rows, 128-byte swizzle, zero fill outside.
cudaError_t make_tmap_f16(CUtensorMap* m, const __half* base, int64_t rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    if (((uintptr_t)base & 15) != 0 || cols % 64 != 0 || rows <= 0 || box_rows <= 0 || box_rows > 256)
        return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * sizeof(__half)};
    const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

template <int QT, int MODE>
cudaError_t launch_tc(const TcParams& p, int max_tiles, cudaStream_t s) {
    const size_t smem = tc_smem_bytes<QT, MODE>();
    cudaError_t err = cudaFuncSetAttribute(tc_gemm_kernel<QT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    const int grid = max(1, min(num_sms(), max_tiles));
    tc_gemm_kernel<QT, MODE><<<grid, tc_threads<QT, MODE>(), smem, s>>>(p);
    return cudaGetLastError();
}

// The weight type as a template: Q4_K, Q8_0 in GGUF blocks, or Q8_0 repacked (MOE_Q8_0_R).
template <int MODE>
cudaError_t launch_tc_q(int qtype, bool q80r, const TcParams& p, int max_tiles, cudaStream_t s) {
    if (qtype == MOE_Q4_K) return launch_tc<MOE_Q4_K, MODE>(p, max_tiles, s);
    return q80r ? launch_tc<MOE_Q8_0_R, MODE>(p, max_tiles, s) : launch_tc<MOE_Q8_0, MODE>(p, max_tiles, s);
}

}  // namespace

size_t tc_tile_list_bytes(int T, int k, int E) {
    const int64_t P = (int64_t)T * k;
    return align_up((size_t)(1 + P / kBNMin + E + 1) * sizeof(int4), 256);
}

bool tc_supported(int qtype, int rows_gu, int K_gu) {
    return (qtype == MOE_Q4_K || qtype == MOE_Q8_0 || qtype == MOE_Q8_0_R) && rows_gu % kBM == 0 && K_gu % kBK == 0 &&
           (qtype != MOE_Q4_K || K_gu % kQ4KWeights == 0);
}

cudaError_t launch_tc_expert_ffn(const TcFfnArgs& a, cudaStream_t s) {
    cudaError_t err;
    const int P = a.identity ? a.T : a.T * a.k;
    if (P <= 0) return cudaSuccess;
    // x -> fp16 copy (once per layer; the caller may share it between routed and shared experts)
    if (a.convert_x) {
        const int64_t n = (int64_t)a.T * a.H;
        to_half_kernel<<<(unsigned)((n / 4 + 255) / 256), 256, 0, s>>>(a.x, a.x_bf16, n, a.x16, a.hdr);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    const int bn = a.qtype == MOE_Q4_K ? tc_bn<MOE_Q4_K>() : tc_bn<MOE_Q8_0>();
    int max_tb;
    if (!a.identity) {
        tile_list_kernel<<<1, 1024, 0, s>>>(a.offsets, a.E, bn, a.tb_list);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        max_tb = P / bn + a.E;
    } else {
        max_tb = (P + bn - 1) / bn;
    }
    TcParams gu{};
    gu.w0 = a.wg; gu.w1 = a.wu; gu.expert_stride = a.stride_gu; gu.rows = a.I; gu.K = a.H; gu.k = a.k;
    if (((uintptr_t)a.x16 & 15) != 0 || a.H % 64 != 0) return cudaErrorInvalidValue;   // 16-byte row copies
    gu.sorted_pairs = a.identity ? nullptr : a.sorted_pairs;
    gu.x16 = a.x16;
    gu.tb_list = a.identity ? nullptr : a.tb_list; gu.n_identity = a.identity ? a.T : 0; gu.bn = bn;
    gu.h_out = a.h16; gu.hdr = a.hdr;
    const WaitCfg wc = wait_cfg();
    gu.wait_ns = wc.limit_ns; gu.stall = wc.stall;
    if (a.ev_before_gateup && (err = cudaEventRecord(a.ev_before_gateup, s)) != cudaSuccess) return err;
    if ((err = launch_tc_q<kGateUp>(a.qtype, a.q80r, gu, max_tb * (a.I / kBM), s)) != cudaSuccess) return err;
    if (a.ev_after_gateup && (err = cudaEventRecord(a.ev_after_gateup, s)) != cudaSuccess) return err;
    TcParams dn{};
    dn.w0 = a.wd; dn.expert_stride = a.stride_d; dn.rows = a.H; dn.K = a.I; dn.k = a.k;
    dn.b_box_rows = std::min(bn, P);
    if ((err = make_tmap_f16(&dn.tmap_b, a.h16, P, a.I, dn.b_box_rows)) != cudaSuccess) return err;
    dn.sorted_pairs = nullptr;
    dn.tb_list = gu.tb_list; dn.n_identity = gu.n_identity; dn.bn = bn;
    dn.y_out = a.y; dn.y16_out = a.y16; dn.hdr = a.hdr;
    dn.wait_ns = wc.limit_ns; dn.stall = wc.stall;
    return launch_tc_q<kDown>(a.qtype, a.q80r, dn, max_tb * (a.H / kBM), s);
}

}  // namespace moe
