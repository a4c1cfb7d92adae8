// kernels_misc.cu -- activation quantiser, weight pack / unpack and the
// block-sum test hook.
#include "qgemv_launch.h"

namespace qg {

// ------------------------------------------------------------ Q8_0 quantiser
//
// One warp per block of 32 activations (minfer README "How it works": int8
// activations; colibri qwen36 docs, dense int8 IDOT GEMV: scale amax/127):
// amax by a shuffle tree of fmaxf (exact), d = amax / 127 (IEEE division),
// 1/d from the fp32 d (0 when d = 0), q = roundf(x * (1/d)) -- roundf rounds
// halfway cases away from zero -- and d stored as fp16, round to nearest even.
// One warp quantises block `rem` (row r = rem / nb, block b = rem % nb) of
// a planar buffer `dst` of R rows of K.
__device__ __forceinline__ void quantize_block_warp(const float *__restrict__ x, uint8_t *__restrict__ dst, int R,
                                                    int K, long long rem, long long xq_bytes, int lane)
{
    const int nb = K / QK;
    const int r = static_cast<int>(rem / nb), b = static_cast<int>(rem - static_cast<long long>(r) * nb);
    const float v = __ldg(x + static_cast<long long>(r) * K + b * QK + lane);
    float amax = fabsf(v);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    float d, id;
    q8_scale(amax, d, id);
    dst[static_cast<long long>(r) * K + b * QK + lane] = static_cast<uint8_t>(static_cast<int8_t>(q8_code(v, id)));
    if (lane == 0) {
        const unsigned short dh = q8_half(d);
        reinterpret_cast<unsigned short *>(dst + static_cast<long long>(R) * K)[rem] = dh;
    }
    if (rem == 0) {  // zero the padding after the scales
        const long long used = static_cast<long long>(R) * K + 2ll * R * nb;
        if (used + lane < xq_bytes) dst[used + lane] = 0;
    }
}

__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float *__restrict__ x, uint8_t *__restrict__ xq,
                                                            int R, int K, long long nblocks, long long xq_bytes)
{
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long per_batch = static_cast<long long>(R) * (K / QK);
    for (long long gb = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; gb < nblocks;
         gb += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
        const long long bi = gb / per_batch;
        quantize_block_warp(x + bi * per_batch * QK, xq + bi * xq_bytes, R, K, gb - bi * per_batch, xq_bytes, lane);
    }
}

cudaError_t launch_quantize(const float *x, void *xq, int R, long long K, int batch, cudaStream_t st)
{
    const long long nblocks = static_cast<long long>(batch) * R * (K / QK);
    const long long xqb = static_cast<long long>(xq_bytes_host(R, K));
    long long grid = (nblocks + 7) / 8;
    if (grid > 65535) grid = 65535;
    quantize_q8_0_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(x, static_cast<uint8_t *>(xq), R,
                                                                    static_cast<int>(K), nblocks, xqb);
    return cudaGetLastError();
}


// ------------------------------------------------------------ pack / unpack
//
// Packed layout (see include/qgemv.h): slab s of rows [16s, 16s+16) holds
// quads q of nbq = min(4, nb - 4q) blocks at s * 288 * nb + 1152 * q:
// nibbles [r][chunk][16 bytes] with block jq in chunk quad_chunk(jq, r, nbq),
// then fp16 scales [r % 8][jq][r / 8].  Rows past
// the last full slab keep their GGML position, so the byte offset of their
// blocks is the same in both layouts.

__device__ __forceinline__ void packed_offsets(long long row, int b, int nb, long long &nib_off, long long &sc_off)
{
    const long long s = row / SLAB_ROWS;
    const int r = static_cast<int>(row - s * SLAB_ROWS);
    const int q = b / QUAD, jq = b - q * QUAD;
    const int nbq = min(QUAD, nb - q * QUAD);
    const long long base = s * static_cast<long long>(SLAB_COL_BYTES) * nb + static_cast<long long>(q) * QUAD_BYTES;
    nib_off = base + (r * nbq + quad_chunk(jq, r, nbq)) * 16;
    sc_off = base + 256 * nbq + ((r % 8) * nbq + jq) * 4 + (r / 8) * 2;
}

__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                                   long long N, int nb, bool to_packed)
{
    const long long nfull = N / SLAB_ROWS;
    const long long total = N * nb;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = i / nb;
        const int b = static_cast<int>(i - row * nb);
        const long long g_off = i * Q4_BYTES;
        if (row >= nfull * SLAB_ROWS) {  // tail rows: same offset in both layouts
            const unsigned short *s16 = reinterpret_cast<const unsigned short *>(src + g_off);
            unsigned short *d16 = reinterpret_cast<unsigned short *>(dst + g_off);
#pragma unroll
            for (int k = 0; k < 9; ++k) d16[k] = s16[k];
            continue;
        }
        long long nib_off, sc_off;
        packed_offsets(row, b, nb, nib_off, sc_off);
        if (to_packed) {
            uint4 nib;
            unsigned d;
            load_ggml_block(src + g_off, nib, d);
            *reinterpret_cast<uint4 *>(dst + nib_off) = nib;
            *reinterpret_cast<unsigned short *>(dst + sc_off) = static_cast<unsigned short>(d);
        } else {
            const uint4 nib = *reinterpret_cast<const uint4 *>(src + nib_off);
            const unsigned short d = *reinterpret_cast<const unsigned short *>(src + sc_off);
            unsigned short *d16 = reinterpret_cast<unsigned short *>(dst + g_off);
            d16[0] = d;
            const unsigned w[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                d16[1 + 2 * k] = static_cast<unsigned short>(w[k] & 0xFFFFu);
                d16[2 + 2 * k] = static_cast<unsigned short>(w[k] >> 16);
            }
        }
    }
}

cudaError_t launch_pack(const void *src, void *dst, long long N, long long K, bool to_packed, cudaStream_t st)
{
    const long long total = N * (K / QK);
    long long grid = (total + 255) / 256;
    if (grid > 65535) grid = 65535;
    pack_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<const uint8_t *>(src),
                                                           static_cast<uint8_t *>(dst), N,
                                                           static_cast<int>(K / QK), to_packed);
    return cudaGetLastError();
}

// ------------------------------------------------------------ block sums (test hook)
//
// Same unpack, dp4a chains and folded offset as the GEMV kernel
// (block_dot16_magic / block_fold16_const), minus the magic bias, over 16.
__global__ void __launch_bounds__(256) isums_kernel(const uint8_t *__restrict__ W, bool packed,
                                                    const uint8_t *__restrict__ xq, int32_t *__restrict__ isums,
                                                    long long N, int K, int T)
{
    const int nb = K / QK;
    const long long nfull = N / SLAB_ROWS;
    const long long total = static_cast<long long>(T) * N * nb;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long t = i / (N * nb);
        const long long rem = i - t * N * nb;
        const long long row = rem / nb;
        const int b = static_cast<int>(rem - row * nb);
        uint4 nib;
        if (packed && row < nfull * SLAB_ROWS) {
            long long nib_off, sc_off;
            packed_offsets(row, b, nb, nib_off, sc_off);
            nib = *reinterpret_cast<const uint4 *>(W + nib_off);
        } else {
            unsigned d;
            load_ggml_block(W + (row * nb + b) * Q4_BYTES, nib, d);
        }
        const uint4 *xp = reinterpret_cast<const uint4 *>(xq + t * K + static_cast<long long>(b) * QK);
        const uint4 qa = xp[0], qb = xp[1];
        isums[i] = (block_dot16_magic(nib, qa, qb, block_fold16_const(qa, qb)) - MAGIC_I) >> 4;
    }
}

cudaError_t launch_isums(const void *W, bool packed, const void *xq, int32_t *isums, long long N, long long K, int T,
                         cudaStream_t st)
{
    const long long total = static_cast<long long>(T) * N * (K / QK);
    long long grid = (total + 255) / 256;
    if (grid > 65535) grid = 65535;
    isums_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<const uint8_t *>(W), packed,
                                                            static_cast<const uint8_t *>(xq), isums, N,
                                                            static_cast<int>(K), T);
    return cudaGetLastError();
}

// ------------------------------------------------------------ FFN step
//
// h = SiLU(g) * u, quantised to planar Q8_0 for the down projection (minfer
// README M15: the FFN between the GEMVs of a decode step).  exp by Cody and
// Waite's method (W. J. Cody, W. Waite, "Software Manual for the Elementary
// Functions", 1980): x = k ln2 + r, k = rint(x log2 e), ln 2 split into a
// head whose products with k are exact and a tail; exp(r) by its Taylor
// series to r^7/7! in Horner form; the exact scale 2^k.  x is clamped to
// [-87, 88].  Every operation is an explicitly rounded fp32 one, in the
// order written, so the values (and so the codes) are a fixed function of
// g and u.
__device__ __forceinline__ float ffn_exp(float x)
{
    x = fminf(fmaxf(x, -87.0f), 88.0f);
    const float k = rintf(__fmul_rn(x, 1.44269504088896340736f));
    float r = __fmaf_rn(-k, 0.693145751953125f, x);   // ln 2 head: 13 significant bits
    r = __fmaf_rn(-k, 1.42860682030941723212e-6f, r);  // ln 2 - head
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float((static_cast<int>(k) + 127) << 23));
}

__device__ __forceinline__ float ffn_silu(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, ffn_exp(-g))); }

// One warp per block of 32: h for lane j, the block maximum by shuffles, then
// the Q8_0 steps of the activation quantiser.  hq: T rows of F codes, then
// [T][F/32] fp16 scales, zero-padded like qgemv_quantize_q8_0's output.
__global__ void __launch_bounds__(256) silu_mul_q8_kernel(const float *__restrict__ g, const float *__restrict__ u,
                                                          uint8_t *__restrict__ hq, int T, int F, long long nblocks,
                                                          long long hq_bytes)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int nb = F / QK;
    for (long long blk = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5; blk < nblocks;
         blk += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
        const int t = static_cast<int>(blk / nb), b = static_cast<int>(blk - static_cast<long long>(t) * nb);
        const long long e = static_cast<long long>(t) * F + b * QK + lane;
        const float h = __fmul_rn(ffn_silu(__ldg(g + e)), __ldg(u + e));
        float amax = fabsf(h);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
        float d, id;
        q8_scale(amax, d, id);
        hq[e] = static_cast<uint8_t>(static_cast<int8_t>(q8_code(h, id)));
        if (lane == 0) reinterpret_cast<unsigned short *>(hq + static_cast<long long>(T) * F)[blk] = q8_half(d);
        if (blk == 0) {  // zero the padding after the scales
            const long long used = static_cast<long long>(T) * F + 2ll * T * nb;
            if (used + lane < hq_bytes) hq[used + lane] = 0;
        }
    }
}

cudaError_t launch_silu_mul_q8(const float *g, const float *u, void *hq, int T, long long F, bool pdl, cudaStream_t st)
{
    const long long nblocks = static_cast<long long>(T) * (F / QK);
    long long grid = (nblocks + 7) / 8;
    if (grid > 65535) grid = 65535;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, silu_mul_q8_kernel, g, u, static_cast<uint8_t *>(hq), T, static_cast<int>(F),
                              nblocks, static_cast<long long>(xq_bytes_host(T, F)));
}

// The lossless verify rule (minfer README M17): tokens[0] is the step's
// current token, tokens[1..T-1] its drafts, pred[t] the greedy prediction
// after tokens[0..t] (at pred[t * pred_stride]).  The step commits pred[0] and each later prediction
// while every draft so far equalled the prediction before it: n = 1 + the
// length of the leading run of t with tokens[t + 1] == pred[t].  One warp.
__global__ void __launch_bounds__(32) verify_commit_kernel(const long long *__restrict__ tokens,
                                                           const long long *__restrict__ pred, int pred_stride,
                                                           int T, int32_t *__restrict__ n_commit)
{
    const int t = threadIdx.x;
    const bool match = t + 1 < T && tokens[t + 1] == pred[static_cast<long long>(t) * pred_stride];
    const unsigned m = __ballot_sync(0xFFFFFFFFu, match);
    if (t == 0) *n_commit = __ffs(~m);  // bit T-1 of m is clear, so n <= T
}

cudaError_t launch_verify_commit(const long long *tokens, const long long *pred, int pred_stride, int T,
                                 int32_t *n_commit, cudaStream_t st)
{
    verify_commit_kernel<<<1, 32, 0, st>>>(tokens, pred, pred_stride, T, n_commit);
    return cudaGetLastError();
}

}  // namespace qg
