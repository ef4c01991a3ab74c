/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the routed-expert MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The product path (the CUDA
 * library under quantized_routed_expert_sigmoid_gb300/) never calls it, and
 * this file shares no code, header, table or helper with that path.
 *
 * What it follows
 * ---------------
 * The bloomery pages describe a mixture-of-experts engine whose card experts
 * run on GGUF block-quantized weights ("bloomery README 0.3.1", Status table,
 * "Quant types" row; "Why it is fast": each expert runs over all its tokens at
 * once, on the stored quantization), and whose router outputs (top-k ids) are
 * compared exactly against a CPU reference while float outputs stay inside
 * rounding bands ("bloomery early V4.1 README", "Oracle sets against
 * ik_llama.cpp").  The pages print none of the arithmetic; every formula below
 * is the plain definition of the layer as specified for this library:
 *
 *   router       l[t,e] = sum_h x[t,h] * Wr[e,h]
 *   softmax      top-k of l (ties: lower id), gates = softmax over the k
 *   sigmoid-grp  s = 1/(1+exp(-l)); sel = s + b; groups of E/G consecutive
 *                experts scored by the sum of their two largest sel; keep the
 *                best G_k groups; top-k sel inside them; gates = scale*s/sum s
 *   permute      counts, exclusive offsets, pairs p = t*k+j sorted by (id, p)
 *   histogram    running per-expert count of routed pairs over many calls
 *   expert FFN   y = Wd * ( silu(Wg x) (.) (Wu x) ),  silu(z) = z/(1+e^-z)
 *   combine      out[t] = sum_j w[t,j] * y[t,j]  (+ shared expert, unweighted)
 *   RMSNorm      u = x / sqrt(mean(x^2) + eps) * gamma
 *
 * Block layouts follow the public GGUF convention, which the pages name but
 * do not print (readings listed in the design notes):
 *   Q8_0: 34 bytes per 32 weights: fp16 d, then 32 int8 q;  w = d*q.
 *   Q4_K: 144 bytes per 256 weights: fp16 d, fp16 dmin, 12 bytes of packed
 *         6-bit (scale, min) for 8 sub-blocks of 32, 128 bytes of 4-bit q;
 *         w = d*sc_j*q - dmin*m_j.
 *   Q5_K: 176 bytes per 256: Q4_K's fields plus 32 bytes of fifth bits;
 *         q in [0, 31], w = d*sc_j*q - dmin*m_j.
 *   Q6_K: 210 bytes per 256: 4-bit low and 2-bit high parts, 16 int8
 *         scales (one per 16 weights), fp16 d last; w = d*sc*(q - 32).
 *   Q3_K: 110 bytes per 256: high-bit mask, 2-bit low parts, 16 packed
 *         6-bit scales stored plus 32, fp16 d last; w = d*(sc - 32)*q with
 *         q = low - 4 where the high bit is clear.
 *   MXFP4: 17 bytes per 32: an E8M0 scale byte, then 16 bytes of E2M1
 *         nibbles (OCP Microscaling formats); w = 2^(e-127) * e2m1(q).
 * Q5_K, Q6_K, Q3_K and MXFP4 are the next expert types the pages list for
 * the card (Q4_K to Q6_K, the Q3_K_M files the large model ships in, and
 * MXFP4).
 *
 * Every value is computed in fp64.  Weight matrices are [rows][K/blk blocks],
 * blocks along the input dimension K; experts are laid out one after another
 * at a fixed byte stride.
 *
 * Parity status of each function (pins live in the test suite):
 *   half_to_double, dequant Q8_0 / Q4_K /
 *   Q5_K / Q6_K / Q3_K / MXFP4            pinned (hand-built blocks; E2M1
 *                                         against the format's value list)
 *   router logits                         pinned (integer closed form)
 *   top-k softmax / sigmoid-group         pinned (brute force, special cases)
 *   permute                               pinned (brute force)
 *   expert counts (routing histogram)     pinned (hand-counted example,
 *                                         brute force, invariants)
 *   expert FFN, layer, combine            pinned (identity-expert closed form,
 *                                         dense-masked equals sparse)
 *   RMSNorm, bf16 rounding, stack         pinned (closed forms)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_Q8_0 2
#define ORACLE_Q4_K 3
#define ORACLE_Q5_K 4
#define ORACLE_Q6_K 5
#define ORACLE_Q3_K 6
#define ORACLE_MXFP4 7

#define ORACLE_ROUTE_SOFTMAX 0
#define ORACLE_ROUTE_SIGMOID_GROUP 1

/* ------------------------------------------------------------------ */
/* IEEE 754 binary16 -> double, from the format's definition:          */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.            */
/* ------------------------------------------------------------------ */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int frac = h & 1023;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                 /* subnormal: f/1024 * 2^-14 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)frac / 1024.0, expo - 15);
    }
    return sign ? -v : v;
}

static uint16_t read_u16_le(const uint8_t* p)
{
    return (uint16_t)(p[0] | ((uint16_t)p[1] << 8));
}

/* ------------------------------------------------------------------ */
/* Dequantization of one row of K weights.                              */
/* ------------------------------------------------------------------ */

/* Q8_0: block b covers weights [32b, 32b+32); w = d * q, q signed 8-bit. */
void oracle_dequant_q8_0_row(const uint8_t* row, int64_t K, double* w)
{
    for (int64_t b = 0; b < K / 32; ++b) {
        const uint8_t* blk = row + b * 34;
        double d = oracle_half_to_double(read_u16_le(blk));
        for (int i = 0; i < 32; ++i) {
            int q = (int)blk[2 + i];
            if (q >= 128) q -= 256;                  /* two's-complement int8 */
            w[b * 32 + i] = d * (double)q;
        }
    }
}

/* Q4_K scale/min of sub-block j from the 12 packed bytes S.
 * j < 4 : low 6 bits of S[j] (scale) and of S[j+4] (min).
 * j >= 4: scale = low nibble of S[j+4] | (top 2 bits of S[j-4]) << 4,
 *         min   = high nibble of S[j+4] | (top 2 bits of S[j])   << 4.   */
static void q4k_scale_min(const uint8_t* S, int j, int* sc, int* m)
{
    if (j < 4) {
        *sc = S[j] & 63;
        *m = S[j + 4] & 63;
    } else {
        *sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4);
        *m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4);
    }
}

/* Q4_K: super-block b covers weights [256b, 256b+256), sub-block j covers
 * [256b+32j, 256b+32j+32).  Quants come in four 32-byte groups c: byte i of
 * group c holds element i of sub-block 2c in its low nibble and element i of
 * sub-block 2c+1 in its high nibble.  w = d*sc_j*q - dmin*m_j.            */
void oracle_dequant_q4_k_row(const uint8_t* row, int64_t K, double* w)
{
    for (int64_t b = 0; b < K / 256; ++b) {
        const uint8_t* blk = row + b * 144;
        double d = oracle_half_to_double(read_u16_le(blk));
        double dmin = oracle_half_to_double(read_u16_le(blk + 2));
        const uint8_t* S = blk + 4;
        const uint8_t* Q = blk + 16;
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            q4k_scale_min(S, j, &sc, &m);
            int c = j / 2;
            for (int i = 0; i < 32; ++i) {
                int byte = Q[32 * c + i];
                int q = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
                w[b * 256 + 32 * j + i] = d * (double)sc * (double)q - dmin * (double)m;
            }
        }
    }
}

/* Q5_K: 176 bytes per 256 weights: d, dmin and the 12 packed (scale, min)
 * bytes exactly as in Q4_K, then 32 bytes of fifth bits, then 128 bytes of
 * low nibbles laid out as the Q4_K quants.  Element i of sub-block j takes
 * bit j of fifth-bit byte i as its 16s digit:
 * q = nibble + 16*bit in [0, 31];  w = d*sc_j*q - dmin*m_j.               */
void oracle_dequant_q5_k_row(const uint8_t* row, int64_t K, double* w)
{
    for (int64_t b = 0; b < K / 256; ++b) {
        const uint8_t* blk = row + b * 176;
        double d = oracle_half_to_double(read_u16_le(blk));
        double dmin = oracle_half_to_double(read_u16_le(blk + 2));
        const uint8_t* S = blk + 4;
        const uint8_t* QH = blk + 16;
        const uint8_t* Q = blk + 48;
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            q4k_scale_min(S, j, &sc, &m);
            int c = j / 2;
            for (int i = 0; i < 32; ++i) {
                int byte = Q[32 * c + i];
                int lo = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
                int hi = (QH[i] >> j) & 1;
                double qv = (double)(lo + 16 * hi);
                w[b * 256 + 32 * j + i] = d * (double)sc * qv - dmin * (double)m;
            }
        }
    }
}

/* Q6_K: 210 bytes per 256 weights: 128 bytes of low nibbles, 64 bytes of
 * two-bit high parts, 16 signed 8-bit scales (one per 16 weights), and the
 * fp16 d last.  The super-block is two halves of 128; in half h, element
 * e = 32r + l (quarter r < 4, l < 32) takes
 *   its low nibble from nibble byte 64h + 32(r % 2) + l
 *     (the low nibble for r < 2, the high nibble for r >= 2),
 *   its high pair from bits 2r, 2r+1 of high-part byte 32h + l;
 * q = nibble + 16*pair - 32 in [-32, 31];  w = d * scale[i/16] * q with
 * i = 128h + e the element's index in the super-block.                   */
void oracle_dequant_q6_k_row(const uint8_t* row, int64_t K, double* w)
{
    for (int64_t b = 0; b < K / 256; ++b) {
        const uint8_t* blk = row + b * 210;
        const uint8_t* QL = blk;
        const uint8_t* QH = blk + 128;
        const uint8_t* SC = blk + 192;
        double d = oracle_half_to_double(read_u16_le(blk + 208));
        for (int i = 0; i < 256; ++i) {
            int h = i / 128, e = i % 128, r = e / 32, l = e % 32;
            int byte = QL[64 * h + 32 * (r % 2) + l];
            int lo = (r < 2) ? (byte & 15) : (byte >> 4);
            int hi = (QH[32 * h + l] >> (2 * r)) & 3;
            int q = lo + 16 * hi - 32;
            int sc = (int)SC[i / 16];
            if (sc >= 128) sc -= 256;                /* two's-complement int8 */
            w[b * 256 + i] = d * (double)sc * (double)q;
        }
    }
}

/* Q3_K scale j (of 16) from the 12 packed bytes S, before the offset of 32:
 * bits 0-3 are the low nibble of S[j] for j < 8 and the high nibble of
 * S[j-8] for j >= 8; bits 4-5 are bits 2(j/4), 2(j/4)+1 of S[8 + j%4].    */
static int q3k_scale(const uint8_t* S, int j)
{
    int lo = (j < 8) ? (S[j] & 15) : (S[j - 8] >> 4);
    int hi = (S[8 + j % 4] >> (2 * (j / 4))) & 3;
    return lo | (hi << 4);
}

/* Q3_K: 110 bytes per 256 weights: 32 bytes of high bits, 64 bytes of
 * two-bit low parts, 12 bytes of packed 6-bit scales (one per 16 weights,
 * stored plus 32), and the fp16 d last.  In half h, element e = 32r + l
 * (r < 4, l < 32) takes bits 2r, 2r+1 of low-part byte 32h + l and bit
 * 4h + r of high-bit byte l; q = low - 4 when that bit is clear, else low,
 * so q is in [-4, 3];  w = d * (scale[i/16] - 32) * q, i = 128h + e.      */
void oracle_dequant_q3_k_row(const uint8_t* row, int64_t K, double* w)
{
    for (int64_t b = 0; b < K / 256; ++b) {
        const uint8_t* blk = row + b * 110;
        const uint8_t* HM = blk;
        const uint8_t* QS = blk + 32;
        const uint8_t* S = blk + 96;
        double d = oracle_half_to_double(read_u16_le(blk + 108));
        for (int i = 0; i < 256; ++i) {
            int h = i / 128, e = i % 128, r = e / 32, l = e % 32;
            int lo = (QS[32 * h + l] >> (2 * r)) & 3;
            int hbit = (HM[l] >> (4 * h + r)) & 1;
            int q = hbit ? lo : lo - 4;
            int sc = q3k_scale(S, i / 16) - 32;
            w[b * 256 + i] = d * (double)sc * (double)q;
        }
    }
}

/* FP4 E2M1 (OCP Microscaling formats): sign bit 3, exponent bits 2-1 with
 * bias 1, mantissa bit 0; exponent 0 is subnormal (m * 0.5), otherwise
 * (1 + m/2) * 2^(exp - 1).  No infinities or NaNs.                      */
double oracle_e2m1_to_double(int nibble)
{
    int sign = (nibble >> 3) & 1;
    int expo = (nibble >> 1) & 3;
    int man = nibble & 1;
    double mag = (expo == 0) ? 0.5 * (double)man : ldexp(1.0 + 0.5 * (double)man, expo - 1);
    return sign ? -mag : mag;
}

/* MXFP4: 17 bytes per 32 weights: one E8M0 scale byte e (2^(e-127); 255 is
 * NaN), then 16 bytes whose byte j holds element j in its low nibble and
 * element j+16 in its high nibble, each an E2M1 value;  w = 2^(e-127) * v. */
void oracle_dequant_mxfp4_row(const uint8_t* row, int64_t K, double* w)
{
    for (int64_t b = 0; b < K / 32; ++b) {
        const uint8_t* blk = row + b * 17;
        int e = blk[0];
        double scale = (e == 255) ? NAN : ldexp(1.0, e - 127);
        for (int j = 0; j < 16; ++j) {
            w[b * 32 + j] = scale * oracle_e2m1_to_double(blk[1 + j] & 15);
            w[b * 32 + j + 16] = scale * oracle_e2m1_to_double(blk[1 + j] >> 4);
        }
    }
}

static int64_t row_bytes(int qtype, int64_t K)
{
    if (qtype == ORACLE_Q8_0) return K / 32 * 34;
    if (qtype == ORACLE_Q4_K) return K / 256 * 144;
    if (qtype == ORACLE_Q5_K) return K / 256 * 176;
    if (qtype == ORACLE_Q6_K) return K / 256 * 210;
    if (qtype == ORACLE_Q3_K) return K / 256 * 110;
    if (qtype == ORACLE_MXFP4) return K / 32 * 17;
    return -1;
}

/* Dequantize `rows` rows of a [rows][K] quantized matrix into w[rows*K]. */
int oracle_dequant_matrix(int qtype, const uint8_t* data, int64_t rows, int64_t K, double* w)
{
    int64_t rb = row_bytes(qtype, K);
    if (rb < 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* src = data + r * rb;
        double* dst = w + r * K;
        switch (qtype) {
        case ORACLE_Q8_0: oracle_dequant_q8_0_row(src, K, dst); break;
        case ORACLE_Q4_K: oracle_dequant_q4_k_row(src, K, dst); break;
        case ORACLE_Q5_K: oracle_dequant_q5_k_row(src, K, dst); break;
        case ORACLE_Q6_K: oracle_dequant_q6_k_row(src, K, dst); break;
        case ORACLE_Q3_K: oracle_dequant_q3_k_row(src, K, dst); break;
        default:          oracle_dequant_mxfp4_row(src, K, dst); break;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Router.                                                             */
/* ------------------------------------------------------------------ */

/* l[t,e] = sum_h x[t,h] * Wr[e,h].  x is [T][H] (already exact doubles of
 * the stored bf16/fp32 activations), Wr is fp32 [E][H].               */
void oracle_router_logits(const double* x, int T, int H, const float* Wr, int E, double* logits)
{
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h) acc += x[(int64_t)t * H + h] * (double)Wr[(int64_t)e * H + h];
            logits[(int64_t)t * E + e] = acc;
        }
}

/* Is candidate a ranked before candidate b?  Larger score first, ties to the
 * lower index.                                                          */
static int ranks_before(double sa, int a, double sb, int b)
{
    if (sa != sb) return sa > sb;
    return a < b;
}

/* Pick the `k` best of the `n` candidates listed in cand[] by score[cand],
 * writing them to out[] in rank order (simple selection, O(n*k)).       */
static void select_best(const double* score, const int* cand, int n, int k, int* out)
{
    char* taken = (char*)calloc((size_t)n, 1);
    for (int r = 0; r < k; ++r) {
        int best = -1;
        for (int i = 0; i < n; ++i) {
            if (taken[i]) continue;
            if (best < 0 || ranks_before(score[cand[i]], cand[i], score[cand[best]], cand[best])) best = i;
        }
        taken[best] = 1;
        out[r] = cand[best];
    }
    free(taken);
}

static void sort_ascending_int(int* v, int n)
{
    for (int i = 1; i < n; ++i) {
        int x = v[i], j = i - 1;
        while (j >= 0 && v[j] > x) { v[j + 1] = v[j]; --j; }
        v[j + 1] = x;
    }
}

/* Softmax routing for one token.  ids come out in ascending expert id.
 * renormalize=1: w_j = exp(l_j) / sum over the k selected (the
 * renormalised top-k softmax);  renormalize=0: w_j = exp(l_j) / sum over
 * all E experts.  `scale` multiplies the gates at the end.              */
static void route_softmax_one(const double* l, int E, int k, int renormalize, double scale,
                              int32_t* ids, double* w)
{
    int* cand = (int*)malloc(sizeof(int) * (size_t)E);
    int* sel = (int*)malloc(sizeof(int) * (size_t)k);
    for (int e = 0; e < E; ++e) cand[e] = e;
    select_best(l, cand, E, k, sel);
    sort_ascending_int(sel, k);
    double m = l[sel[0]];
    for (int j = 1; j < k; ++j) if (l[sel[j]] > m) m = l[sel[j]];
    if (!renormalize) for (int e = 0; e < E; ++e) if (l[e] > m) m = l[e];
    double denom = 0.0;
    if (renormalize) for (int j = 0; j < k; ++j) denom += exp(l[sel[j]] - m);
    else for (int e = 0; e < E; ++e) denom += exp(l[e] - m);
    for (int j = 0; j < k; ++j) {
        ids[j] = sel[j];
        w[j] = scale * exp(l[sel[j]] - m) / denom;
    }
    free(cand);
    free(sel);
}

/* Sigmoid + bias + group-limited routing for one token.
 * s_e = 1/(1+exp(-l_e)), sel_e = s_e + b_e (b may be NULL = 0).
 * Group g = experts [g*E/G, (g+1)*E/G); group score = sum of its two largest
 * sel (all of them if a group has fewer than two).  Keep the topk_groups best
 * groups (ties: lower group id), then the k best sel among their experts.
 * Gates use s, never the bias: w_j = scale * s_j / sum_sel s (renormalize=1)
 * or scale * s_j (renormalize=0).                                        */
static void route_sigmoid_group_one(const double* l, const float* bias, int E, int k, int G, int Gk,
                                    int renormalize, double scale, int32_t* ids, double* w,
                                    double* group_gap, double* sel_gap)
{
    int per = E / G;
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    double* sel = (double*)malloc(sizeof(double) * (size_t)E);
    double* gscore = (double*)malloc(sizeof(double) * (size_t)G);
    int* cand = (int*)malloc(sizeof(int) * (size_t)E);
    int* top = (int*)malloc(sizeof(int) * (size_t)(E + 1));
    for (int e = 0; e < E; ++e) {
        s[e] = 1.0 / (1.0 + exp(-l[e]));
        sel[e] = s[e] + (bias ? (double)bias[e] : 0.0);
    }
    int take = per < 2 ? per : 2;
    for (int g = 0; g < G; ++g) {
        for (int i = 0; i < per; ++i) cand[i] = g * per + i;
        select_best(sel, cand, per, take, top);
        double acc = 0.0;
        for (int i = 0; i < take; ++i) acc += sel[top[i]];
        gscore[g] = acc;
    }
    int* gcand = (int*)malloc(sizeof(int) * (size_t)G);
    int* gkept = (int*)malloc(sizeof(int) * (size_t)(G));
    for (int g = 0; g < G; ++g) gcand[g] = g;
    int gsel = Gk < G ? Gk + 1 : G;            /* one extra to measure the gap */
    select_best(gscore, gcand, G, gsel, gkept);
    if (group_gap) *group_gap = (Gk < G) ? gscore[gkept[Gk - 1]] - gscore[gkept[Gk]] : INFINITY;
    int n = 0;
    for (int r = 0; r < Gk; ++r)
        for (int i = 0; i < per; ++i) cand[n++] = gkept[r] * per + i;
    int ksel = k < n ? k + 1 : n;
    select_best(sel, cand, n, ksel, top);
    if (sel_gap) *sel_gap = (k < n) ? sel[top[k - 1]] - sel[top[k]] : INFINITY;
    sort_ascending_int(top, k);
    double denom = 0.0;
    for (int j = 0; j < k; ++j) denom += s[top[j]];
    for (int j = 0; j < k; ++j) {
        ids[j] = top[j];
        w[j] = renormalize ? scale * s[top[j]] / denom : scale * s[top[j]];
    }
    free(s); free(sel); free(gscore); free(cand); free(top); free(gcand); free(gkept);
}

/* Top-k routing of T tokens from their logits.
 * mode 0 = softmax, 1 = sigmoid + bias + group-limited.
 * gaps (nullable, [T][2]): the selection margins measured in fp64 --
 *   softmax: [0] = l_(k) - l_(k+1), [1] = +inf;
 *   sigmoid: [0] = sel_(k) - sel_(k+1) inside the kept groups,
 *            [1] = groupscore_(Gk) - groupscore_(Gk+1).
 * Returns 0, or -1 on invalid sizes.                                     */
int oracle_route(int mode, const double* logits, const float* bias, int T, int E, int k,
                 int n_groups, int topk_groups, int renormalize, double scale,
                 int32_t* ids, double* w, double* gaps)
{
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    if (mode == ORACLE_ROUTE_SOFTMAX) {
        for (int t = 0; t < T; ++t) {
            const double* l = logits + (int64_t)t * E;
            route_softmax_one(l, E, k, renormalize, scale, ids + (int64_t)t * k, w + (int64_t)t * k);
            if (gaps) {
                int* cand = (int*)malloc(sizeof(int) * (size_t)E);
                int* top = (int*)malloc(sizeof(int) * (size_t)(k + 1));
                for (int e = 0; e < E; ++e) cand[e] = e;
                int ks = k < E ? k + 1 : E;
                select_best(l, cand, E, ks, top);
                gaps[2 * t] = k < E ? l[top[k - 1]] - l[top[k]] : INFINITY;
                gaps[2 * t + 1] = INFINITY;
                free(cand); free(top);
            }
        }
        return 0;
    }
    if (mode == ORACLE_ROUTE_SIGMOID_GROUP) {
        if (n_groups < 1 || E % n_groups || topk_groups < 1 || topk_groups > n_groups) return -1;
        if (k > topk_groups * (E / n_groups)) return -1;
        for (int t = 0; t < T; ++t) {
            double gg, sg;
            route_sigmoid_group_one(logits + (int64_t)t * E, bias, E, k, n_groups, topk_groups,
                                    renormalize, scale, ids + (int64_t)t * k, w + (int64_t)t * k, &gg, &sg);
            if (gaps) { gaps[2 * t] = sg; gaps[2 * t + 1] = gg; }
        }
        return 0;
    }
    return -1;
}

/* ------------------------------------------------------------------ */
/* Permutation: group the T*k token-expert pairs by expert.             */
/* counts[e] = #{p : ids[p] = e}; offsets = exclusive prefix sum (E+1   */
/* entries, offsets[E] = T*k); sorted_pairs lists p = t*k+j in          */
/* ascending (expert, p) order; pair_pos[sorted_pairs[i]] = i.          */
/* ------------------------------------------------------------------ */
int oracle_permute(const int32_t* ids, int T, int k, int E,
                   int32_t* sorted_pairs, int32_t* offsets, int32_t* pair_pos)
{
    int64_t P = (int64_t)T * k;
    int32_t* cursor = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
    for (int64_t p = 0; p < P; ++p) {
        if (ids[p] < 0 || ids[p] >= E) { free(cursor); return -1; }
        cursor[ids[p]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + cursor[e];
    for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t p = 0; p < P; ++p) {
        int32_t i = cursor[ids[p]]++;
        sorted_pairs[i] = (int32_t)p;
        pair_pos[p] = i;
    }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Routing histogram: the engine counts its own routing so that the     */
/* experts it calls most can be moved to the fast tier between steps    */
/* ("bloomery README 0.3.1", opening feature list: MoE models larger    */
/* than the card; "bloomery V4.1 README", feature list, "Adaptive       */
/* residency").  counts[e] += #{p : ids[p] = e} over the P = T*k pairs  */
/* of one call; counts carries over from call to call.                  */
/* ------------------------------------------------------------------ */
int oracle_expert_counts(const int32_t* ids, int64_t P, int E, uint64_t* counts)
{
    for (int64_t p = 0; p < P; ++p)
        if (ids[p] < 0 || ids[p] >= E) return -1;
    for (int e = 0; e < E; ++e) {
        uint64_t n = 0;
        for (int64_t p = 0; p < P; ++p)
            if (ids[p] == e) n += 1;
        counts[e] += n;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* One SwiGLU expert on one token.                                      */
/* gate, up: [I][H] quantized; down: [H][I] quantized.                  */
/* y[H] = down * ( silu(gate*x) (.) (up*x) ).  hout (nullable) gets h.  */
/* ------------------------------------------------------------------ */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* gate and up stored as qtype_gu, down as qtype_d (a file may mix them,
 * e.g. 3-bit gate/up with 4-bit down).                                  */
int oracle_expert_ffn_mixed(int qtype_gu, int qtype_d, const uint8_t* gate, const uint8_t* up,
                            const uint8_t* down, int H, int I, const double* x, double* y,
                            double* hout)
{
    int64_t rb_in = row_bytes(qtype_gu, H), rb_mid = row_bytes(qtype_d, I);
    if (rb_in < 0 || rb_mid < 0) return -1;
    double* wrow = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        oracle_dequant_matrix(qtype_gu, gate + (int64_t)i * rb_in, 1, H, wrow);
        for (int c = 0; c < H; ++c) g += wrow[c] * x[c];
        oracle_dequant_matrix(qtype_gu, up + (int64_t)i * rb_in, 1, H, wrow);
        for (int c = 0; c < H; ++c) u += wrow[c] * x[c];
        h[i] = silu(g) * u;
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        oracle_dequant_matrix(qtype_d, down + (int64_t)n * rb_mid, 1, I, wrow);
        for (int i = 0; i < I; ++i) acc += wrow[i] * h[i];
        y[n] = acc;
    }
    if (hout) memcpy(hout, h, sizeof(double) * (size_t)I);
    free(wrow);
    free(h);
    return 0;
}

int oracle_expert_ffn(int qtype, const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                      int H, int I, const double* x, double* y, double* hout)
{
    return oracle_expert_ffn_mixed(qtype, qtype, gate, up, down, H, I, x, y, hout);
}

/* ------------------------------------------------------------------ */
/* The whole layer.                                                     */
/* ------------------------------------------------------------------ */
typedef struct {
    int mode;              /* ORACLE_ROUTE_* */
    int E, k, n_groups, topk_groups, renormalize;
    double scale;
    int H, I;
    int qtype;             /* routed experts' gate and up */
    const uint8_t* gate;   /* expert e at gate + e*expert_stride_gu */
    const uint8_t* up;
    const uint8_t* down;   /* expert e at down + e*expert_stride_d */
    int64_t expert_stride_gu, expert_stride_d;
    const float* Wr;       /* [E][H] fp32 */
    const float* bias;     /* [E] fp32 or NULL */
    /* optional shared expert (unweighted), NULL gate = none */
    int shared_qtype, I_s;
    const uint8_t* s_gate;
    const uint8_t* s_up;
    const uint8_t* s_down;
    int qtype_down;        /* routed experts' down (may differ from qtype) */
} oracle_layer;

/* out[T][H] = combine of the routed experts (+ shared) for the T tokens.
 * logits_in (nullable) replaces the router GEMV.  ids/w/logits/y_pairs are
 * optional outputs ([T*k], [T*k], [T*E], [T*k][H]).  n_threads > 1 runs the
 * token-expert pairs in parallel (each pair is independent).           */
int oracle_moe_layer(const oracle_layer* L, const double* x, int T, const double* logits_in,
                     double* out, int32_t* ids_out, double* w_out, double* logits_out,
                     double* y_pairs_out, int n_threads)
{
    int E = L->E, k = L->k, H = L->H;
    int64_t P = (int64_t)T * k;
    double* logits = (double*)malloc(sizeof(double) * (size_t)((int64_t)T * E + 1));
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P + 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)(P + 1));
    double* y = (double*)malloc(sizeof(double) * (size_t)(P * H + 1));
    int rc = 0;
    if (logits_in) memcpy(logits, logits_in, sizeof(double) * (size_t)T * E);
    else oracle_router_logits(x, T, H, L->Wr, E, logits);
    rc = oracle_route(L->mode, logits, L->bias, T, E, k, L->n_groups, L->topk_groups,
                      L->renormalize, L->scale, ids, w, NULL);
    if (rc) goto done;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) if (n_threads > 1)
#endif
    for (int64_t p = 0; p < P; ++p) {
        int t = (int)(p / k);
        int e = ids[p];
        oracle_expert_ffn_mixed(L->qtype, L->qtype_down,
                                L->gate + (int64_t)e * L->expert_stride_gu,
                                L->up + (int64_t)e * L->expert_stride_gu,
                                L->down + (int64_t)e * L->expert_stride_d, H, L->I,
                                x + (int64_t)t * H, y + p * H, NULL);
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) if (n_threads > 1)
#endif
    for (int t = 0; t < T; ++t) {
        double* o = out + (int64_t)t * H;
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            const double* yp = y + ((int64_t)t * k + j) * H;
            for (int n = 0; n < H; ++n) o[n] += w[(int64_t)t * k + j] * yp[n];
        }
        if (L->s_gate) {
            double* ys = (double*)malloc(sizeof(double) * (size_t)H);
            oracle_expert_ffn(L->shared_qtype, L->s_gate, L->s_up, L->s_down, H, L->I_s,
                              x + (int64_t)t * H, ys, NULL);
            for (int n = 0; n < H; ++n) o[n] += ys[n];
            free(ys);
        }
    }
    if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)P);
    if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)P);
    if (logits_out) memcpy(logits_out, logits, sizeof(double) * (size_t)T * E);
    if (y_pairs_out) memcpy(y_pairs_out, y, sizeof(double) * (size_t)(P * H));
done:
    free(logits); free(ids); free(w); free(y);
    return rc;
}

/* ------------------------------------------------------------------ */
/* RMSNorm and bf16 rounding (used by the stacked-layer check).         */
/* ------------------------------------------------------------------ */

/* u[t,h] = x[t,h] / sqrt(mean_h(x[t,:]^2) + eps) * gamma[h]. */
void oracle_rmsnorm(const double* x, int T, int H, const float* gamma, double eps, double* u)
{
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int h = 0; h < H; ++h) ss += x[(int64_t)t * H + h] * x[(int64_t)t * H + h];
        double r = 1.0 / sqrt(ss / H + eps);
        for (int h = 0; h < H; ++h) u[(int64_t)t * H + h] = x[(int64_t)t * H + h] * r * (double)gamma[h];
    }
}

/* Round a double to the nearest bfloat16 value (8 significant bits, the
 * exponent range of binary32), ties to even.  Written from the format:
 * keep 8 significant bits of the binary expansion.                      */
double oracle_round_bf16(double v)
{
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    int e;
    double m = frexp(fabs(v), &e);          /* |v| = m * 2^e, m in [0.5, 1) */
    if (e < -125) {                          /* below binary32's normal range: fixed quantum 2^-133 */
        double q = ldexp(1.0, -133);
        double n = fabs(v) / q;
        double r = nearbyint(n);             /* default rounding mode: ties to even */
        double out = r * q;
        return v < 0 ? -out : out;
    }
    double scaled = ldexp(m, 8);             /* 8 significant bits -> integer part */
    double r = nearbyint(scaled);
    double out = ldexp(r, e - 8);
    if (out > 3.3895313892515355e38) out = INFINITY;
    return v < 0 ? -out : out;
}

/* The stacked check: x_{l+1} = x_l + MoE_l( bf16( RMSNorm_l(x_l) ) ).
 * layers[l] describes layer l, gammas[l] its RMSNorm weight.  x is updated
 * in place ([T][H]).  ids_out (nullable) gets [n_layers][T*k] and gaps_out
 * (nullable) [n_layers][T][2] (the routing margins of each layer).      */
int oracle_moe_stack(const oracle_layer* layers, const float* const* gammas, int n_layers,
                     double eps, double* x, int T, int32_t* ids_out, double* gaps_out, int n_threads)
{
    int H = layers[0].H;
    double* u = (double*)malloc(sizeof(double) * (size_t)T * H);
    double* y = (double*)malloc(sizeof(double) * (size_t)T * H);
    int rc = 0;
    for (int l = 0; l < n_layers && !rc; ++l) {
        const oracle_layer* L = &layers[l];
        oracle_rmsnorm(x, T, H, gammas[l], eps, u);
        for (int64_t i = 0; i < (int64_t)T * H; ++i) u[i] = oracle_round_bf16(u[i]);
        if (gaps_out) {
            double* lg = (double*)malloc(sizeof(double) * (size_t)T * L->E);
            int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * L->k);
            double* w = (double*)malloc(sizeof(double) * (size_t)T * L->k);
            oracle_router_logits(u, T, H, L->Wr, L->E, lg);
            rc = oracle_route(L->mode, lg, L->bias, T, L->E, L->k, L->n_groups, L->topk_groups,
                              L->renormalize, L->scale, ids, w, gaps_out + (int64_t)l * T * 2);
            free(lg); free(ids); free(w);
            if (rc) break;
        }
        rc = oracle_moe_layer(L, u, T, NULL, y, ids_out ? ids_out + (int64_t)l * T * L->k : NULL,
                              NULL, NULL, NULL, n_threads);
        for (int64_t i = 0; i < (int64_t)T * H; ++i) x[i] += y[i];
    }
    free(u);
    free(y);
    return rc;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
