// prepare.cu -- one-time weight preparation: Q8_0 blocks into the MOE_Q8_0_R row layout.
//
// A GGUF Q8_0 block is 34 bytes (fp16 d, 32 int8 q), so the quants of a block start on a
// 2-byte boundary only and a kernel reading them in place needs 2-byte loads.  The
// repacked row keeps the same values: the 32-byte quant runs of its blocks in order (every
// run 16-byte aligned), then the blocks' fp16 scales, padded to a multiple of 16 bytes.
// The pages' large model keeps its shared experts in Q8_0 ("bloomery early V4.1 README",
// model file notes); repacked, they stream with 16-byte loads like the Q4_K experts.
#include "internal.cuh"

namespace moe {
namespace {

// One thread per Q8_0 block: its 17 halfwords in, 32 quant bytes and the scale out.
__global__ void q80_repack_kernel(const uint8_t* __restrict__ src, int64_t src_stride, int64_t rows, int64_t nb,
                                  int64_t total, uint8_t* __restrict__ dst, int64_t dst_row) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t b = i % nb, r = (i / nb) % rows, e = i / (nb * rows);
    const uint8_t* blk = src + e * src_stride + r * nb * kQ80Bytes + b * kQ80Bytes;   // 2-byte aligned
    const unsigned short* h = reinterpret_cast<const unsigned short*>(blk);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = (uint32_t)__ldg(h + 1 + 2 * j) | ((uint32_t)__ldg(h + 2 + 2 * j) << 16);
    uint8_t* row = dst + (e * rows + r) * dst_row;
    *reinterpret_cast<uint4*>(row + 32 * b) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(row + 32 * b + 16) = make_uint4(w[4], w[5], w[6], w[7]);
    *reinterpret_cast<unsigned short*>(row + 32 * nb + 2 * b) = __ldg(h);
    if (b == 0)                                       // the row's padding after the scales
        for (int64_t o = 32 * nb + 2 * nb; o < dst_row; ++o) row[o] = 0;
}

}  // namespace

cudaError_t launch_q80_repack(const uint8_t* src, int64_t src_stride, int E, int64_t rows, int64_t K, uint8_t* dst,
                              cudaStream_t s) {
    const int64_t nb = K / kQ80Weights;
    const int64_t total = (int64_t)E * rows * nb;
    if (total <= 0) return cudaSuccess;
    const int threads = 256;
    q80_repack_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, s>>>(src, src_stride, rows, nb, total,
                                                                                      dst, q80r_row_bytes(K));
    return cudaGetLastError();
}

}  // namespace moe
