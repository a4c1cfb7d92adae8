// isums_tc.cu -- test hook: the per-block integer sums as the tensor-core
// path forms them (minfer README M16: the batched path forms the same
// per-block integer sums as the one-token path).
//
// One warp per (16-row slab, block).  Lane (g, j) takes weight word j of rows
// g and g + 8 and builds the B registers of token min(g, T - 1) with the
// GEMV kernel's own conversions: from the f16 operand words
// (f16_block_words, small activation images) or from the biased int8 words
// (mma_b_from_biased, large images).  The folded offset of tokens 2j and
// 2j + 1 starts the accumulator, and mma_block_sums -- the GEMV kernel's two
// MMAs -- leaves isum * 2^-24 in each output slot, exact; the hook writes
// isum.
#include "gemv_kernel.cuh"
#include "qgemv_launch.h"

namespace qg {

__global__ void __launch_bounds__(256) isums_tc_kernel(const uint8_t *__restrict__ W, bool packed,
                                                       const uint8_t *__restrict__ xq, int32_t *__restrict__ isums,
                                                       long long N, int K, int T, bool f16_image)
{
    const int nb = K / QK;
    const long long nslabs = (N + SLAB_ROWS - 1) / SLAB_ROWS;
    const long long nfull = N / SLAB_ROWS;
    const int lane = threadIdx.x & 31, g = lane >> 2, j = lane & 3;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         w < nslabs * nb; w += warps) {
        const long long slab = w / nb;
        const int b = static_cast<int>(w - slab * nb);
        unsigned wr[2] = {0u, 0u};  // weight word j of rows g, g + 8
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long row = slab * SLAB_ROWS + g + 8 * h;
            if (row >= N) continue;
            if (packed && slab < nfull) {
                long long nib_off, sc_off;
                packed_offsets(row, b, nb, nib_off, sc_off);
                wr[h] = *reinterpret_cast<const unsigned *>(W + nib_off + 4 * j);
            } else {
                const unsigned short *p =
                    reinterpret_cast<const unsigned short *>(W + (row * nb + b) * Q4_BYTES + 2 + 4 * j);
                wr[h] = static_cast<unsigned>(p[0]) | (static_cast<unsigned>(p[1]) << 16);
            }
        }
        // B operand: token min(g, T - 1) (columns past T reach only their own outputs)
        const int tg = g < T ? g : T - 1;
        const uint4 *qp = reinterpret_cast<const uint4 *>(xq + static_cast<long long>(tg) * K + b * QK);
        const uint4 qa = qp[0], qb = qp[1];
        unsigned bl0, bl1, bh0, bh1;
        if (f16_image) {
            unsigned wd[16];
            f16_block_words(qa, qb, wd);
            bl0 = wd[j];
            bl1 = wd[4 + j];
            bh0 = wd[8 + j];
            bh1 = wd[12 + j];
        } else {
            const unsigned flip = 0x80808080u;  // the int8 image holds q xor 0x80
            const unsigned qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
            mma_b_from_biased(qw[j] ^ flip, qw[4 + j] ^ flip, bl0, bl1, bh0, bh1);
        }
        // accumulator start: the folded offset of tokens 2j and 2j + 1 (0 past T)
        float C[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = 2 * j + u;
            C[u] = 0.0f;
            if (t < T) {
                const uint4 *tp = reinterpret_cast<const uint4 *>(xq + static_cast<long long>(t) * K + b * QK);
                const uint4 ta = tp[0], tb = tp[1];
                const int ones = 0x01010101;
                int sq = 0;
                sq = dp4a_ss((int)ta.x, ones, sq);
                sq = dp4a_ss((int)ta.y, ones, sq);
                sq = dp4a_ss((int)ta.z, ones, sq);
                sq = dp4a_ss((int)ta.w, ones, sq);
                sq = dp4a_ss((int)tb.x, ones, sq);
                sq = dp4a_ss((int)tb.y, ones, sq);
                sq = dp4a_ss((int)tb.z, ones, sq);
                sq = dp4a_ss((int)tb.w, ones, sq);
                C[u] = mma_fold_const(sq);
            }
        }
        float d[4];
        mma_block_sums(wr[0], wr[1], bl0, bl1, bh0, bh1, make_float4(C[0], C[1], C[0], C[1]), d);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const long long row = slab * SLAB_ROWS + g + 8 * (k >> 1);
            const int t = 2 * j + (k & 1);
            if (row < N && t < T)
                isums[(static_cast<long long>(t) * N + row) * nb + b] = __float2int_rn(__fmul_rn(d[k], MMA_UNSCALE));
        }
    }
}

cudaError_t launch_isums_tc(const void *W, bool packed, const void *xq, int32_t *isums, long long N, long long K,
                            int T, bool f16_image, cudaStream_t st)
{
    const long long warps = ((N + SLAB_ROWS - 1) / SLAB_ROWS) * (K / QK);
    long long grid = (warps + 7) / 8;
    if (grid > 65535) grid = 65535;
    isums_tc_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<const uint8_t *>(W), packed,
                                                               static_cast<const uint8_t *>(xq), isums, N,
                                                               static_cast<int>(K), T, f16_image);
    return cudaGetLastError();
}

}  // namespace qg
