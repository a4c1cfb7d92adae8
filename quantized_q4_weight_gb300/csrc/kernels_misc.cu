// kernels_misc.cu -- activation quantiser, weight pack / unpack and the
// block-sum test hook.
#include <cstring>

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

// A whole sequence's activations in one launch: item i's T rows of K[i]
// fp32 values into its planar buffer, the same bytes as launch_quantize.
struct QuantList {
    int n, T;
    const float *x[MAXG_SEQ];
    uint8_t *xq[MAXG_SEQ];
    int K[MAXG_SEQ];
    long long block_begin[MAXG_SEQ + 1];  // prefix of T * K[i] / 32
};

__global__ void __launch_bounds__(256) quantize_list_kernel(const __grid_constant__ QuantList L)
{
    // The grid is small enough to be resident at once, so a dependent
    // kernel launched early cannot take the SMs this one still needs.
    pdl_launch_dependents();
    pdl_wait();
    const long long total = L.block_begin[L.n];
    for (long long gb = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; gb < total;
         gb += static_cast<long long>(gridDim.x) * blockDim.x) {
        int lo = 0, hi = L.n;  // the item holding block gb: block_begin[lo] <= gb < block_begin[lo + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (L.block_begin[mid] <= gb) lo = mid;
            else hi = mid;
        }
        const int K = L.K[lo], nb = K / QK, T = L.T;
        const long long rem = gb - L.block_begin[lo];
        const int r = static_cast<int>(rem / nb), b = static_cast<int>(rem - static_cast<long long>(r) * nb);
        const float *x = L.x[lo] + static_cast<long long>(r) * K + b * QK;
        uint4 qa, qb;
        unsigned short dh;
        q8_block_thread(x, (reinterpret_cast<uintptr_t>(x) & 15) == 0, qa, qb, dh);
        uint8_t *dst = L.xq[lo];
        uint4 *dq = reinterpret_cast<uint4 *>(dst + static_cast<long long>(r) * K + b * QK);
        dq[0] = qa;
        dq[1] = qb;
        reinterpret_cast<unsigned short *>(dst + static_cast<long long>(T) * K)[rem] = dh;
        if (rem == 0) {  // zero the padding after the scales
            const long long used = static_cast<long long>(T) * K + 2ll * T * nb;
            const long long xqb = static_cast<long long>(T) * K + ((2ll * T * nb + 15) & ~15ll);
            for (long long p = used; p < xqb; ++p) dst[p] = 0;
        }
    }
}

cudaError_t launch_quantize_list(const float *const *x, uint8_t *const *xq, const long long *K, int n, int T,
                                 int max_ctas, cudaStream_t st)
{
    if (n < 1 || n > MAXG_SEQ || max_ctas < 1) return cudaErrorInvalidValue;
    QuantList L;
    memset(&L, 0, sizeof(L));
    L.n = n;
    L.T = T;
    for (int i = 0; i < n; ++i) {
        L.x[i] = x[i];
        L.xq[i] = xq[i];
        L.K[i] = static_cast<int>(K[i]);
        L.block_begin[i + 1] = L.block_begin[i] + static_cast<long long>(T) * (K[i] / QK);
    }
    long long grid = (L.block_begin[n] + 255) / 256;  // one thread per block of 32 values
    if (grid > max_ctas) grid = max_ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_list_kernel, L);
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
// h = SiLU(g) * u quantised to planar Q8_0 for the down projection: the
// steps of ffn_exp / ffn_silu (qgemv_internal.cuh), then the Q8_0 steps.

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

// Weights requantised to GGML Q4_0 blocks at load (minfer README M14 and
// M18: heads requantised to q4_0 when the model is loaded).  The encoder is
// GGML's q4_0 one: m = the block's first element of largest magnitude (+0
// for a block of zeros), d = m / -8 in fp32 (m becomes code 0), 1/d from
// that d (0 when d = 0), code min(15, floor(x * (1/d) + 8.5)) with the
// multiply and the add each rounded to nearest, d stored as fp16.  From Q8_0
// blocks the values are q * d8 (exact in fp32).
//
// The conversion units (int <-> float, floor) run at a quarter of the FP32
// rate, and three per element made the Q8_0 encoder bound by them.  Both
// conversions are done in the FP32 pipe instead, exactly:
//  - int8 q -> float: the float with bits 0x4B000000 | (q + 128) is
//    2^23 + q + 128, so subtracting 2^23 + 128 leaves q;
//  - floor(s) for 0 <= s <= 15: 2^23 + s rounded toward minus infinity is
//    2^23 + floor(s) (the spacing of floats at 2^23 is 1), whose low four
//    bits are floor(s).
__device__ __forceinline__ float q8_code_to_float(unsigned byte)
{
    return __fsub_rn(__uint_as_float(0x4B000000u | (byte ^ 0x80u)), 8388736.0f);
}

// One block of 32 values -> its 18 bytes as nine two-byte words: d, then
// byte j = code j | code j+16 << 4.
__device__ __forceinline__ void q4_encode_block(const float (&x)[QK], unsigned short (&o)[9])
{
    float amax = 0.0f, m = 0.0f;
#pragma unroll
    for (int j = 0; j < QK; ++j) {
        const float a = fabsf(x[j]);
        if (a > amax) {
            amax = a;
            m = x[j];
        }
    }
    const float d = __fdiv_rn(m, -8.0f);
    const float id = d != 0.0f ? __frcp_rn(d) : 0.0f;
    int c[QK];
#pragma unroll
    for (int j = 0; j < QK; ++j) {
        // min(15, floor(s)) with s first clamped to [0, 15]: an infinite s
        // (1/d overflows for an fp32-subnormal d) gives 15 or 0, a NaN
        // (0 * inf) gives 0 (fmaxf returns the number)
        const float sj = __fadd_rn(__fmul_rn(x[j], id), 8.5f);
        const float cl = fminf(fmaxf(sj, 0.0f), 15.0f);
        c[j] = static_cast<int>(__float_as_uint(__fadd_rd(cl, 8388608.0f)) & 0xFu);
    }
    o[0] = __half_as_ushort(__float2half_rn(d));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        o[1 + i] = static_cast<unsigned short>((c[2 * i] | (c[2 * i + 16] << 4)) |
                                               ((c[2 * i + 1] | (c[2 * i + 17] << 4)) << 8));
}

// One thread per block, all of its loads issued before any use, blocks in a
// grid-stride loop (unaligned sources, and the blocks after the last whole
// chunk of the staged kernel below).  VEC: the fp32 source is 16-byte
// aligned (float4 loads).
template <bool FROM_Q8, bool VEC>
__global__ void __launch_bounds__(256) requant_q4_0_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst,
                                                           long long nblocks)
{
    const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long blk = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; blk < nblocks; blk += step) {
        float x[QK];
        if constexpr (FROM_Q8) {
            // 34 bytes at an even offset: 17 two-byte loads
            const unsigned short *s =
                reinterpret_cast<const unsigned short *>(static_cast<const uint8_t *>(src) + blk * 34);
            unsigned short h[17];
#pragma unroll
            for (int i = 0; i < 17; ++i) h[i] = __ldg(s + i);
            const float d8 = __half2float(__ushort_as_half(h[0]));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                x[2 * i] = __fmul_rn(q8_code_to_float(h[1 + i] & 0xFFu), d8);
                x[2 * i + 1] = __fmul_rn(q8_code_to_float(h[1 + i] >> 8), d8);
            }
        } else if constexpr (VEC) {
            const float4 *s = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + blk * QK);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 v = __ldg(s + i);
                x[4 * i] = v.x;
                x[4 * i + 1] = v.y;
                x[4 * i + 2] = v.z;
                x[4 * i + 3] = v.w;
            }
        } else {
            const float *s = static_cast<const float *>(src) + blk * QK;
#pragma unroll
            for (int j = 0; j < QK; ++j) x[j] = __ldg(s + j);
        }
        unsigned short o[9];
        q4_encode_block(x, o);
        unsigned short *out = reinterpret_cast<unsigned short *>(dst + blk * 18);
#pragma unroll
        for (int i = 0; i < 9; ++i) out[i] = o[i];
    }
}

// The same encoder over chunks of 256 blocks staged through shared memory,
// so that global memory sees only coalesced 16-byte loads and stores (source
// and destination 16-byte aligned; whole chunks only).  fp32 chunks are
// stored transposed, element j of block b at word j * 257 + b: the staging
// stores of one 16-byte load and the per-thread reads of one element then
// fall in distinct banks.  Q8_0 chunks stay as they are (34-byte blocks,
// read as two-byte words: at most two threads per bank).
constexpr int RQ_CHUNK = 256;

// Q8_0 chunks: two staging buffers filled by cp.async, the next chunk's
// copies issued before the current chunk is encoded (a grid of a few CTAs
// per SM walks the chunks), so that the copies overlap the encoder.
__device__ __forceinline__ void rq_issue_q8_chunk(uint8_t *s, const uint8_t *g, int tid)
{
    for (int i = tid; i < 34 * RQ_CHUNK / 16; i += RQ_CHUNK)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(s + 16 * i)), "l"(g + 16 * i)
                     : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void rq_encode_q8_chunk(const uint8_t *s_in, uint8_t *s_out, int tid)
{
    float x[QK];
    const unsigned short *h = reinterpret_cast<const unsigned short *>(s_in + tid * 34);
    const float d8 = __half2float(__ushort_as_half(h[0]));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const unsigned w = h[1 + i];
        x[2 * i] = __fmul_rn(q8_code_to_float(w & 0xFFu), d8);
        x[2 * i + 1] = __fmul_rn(q8_code_to_float(w >> 8), d8);
    }
    unsigned short o[9];
    q4_encode_block(x, o);
    unsigned short *so = reinterpret_cast<unsigned short *>(s_out + tid * 18);
#pragma unroll
    for (int i = 0; i < 9; ++i) so[i] = o[i];
}

__global__ void __launch_bounds__(RQ_CHUNK) requant_q4_0_staged_q8(const uint8_t *__restrict__ src,
                                                                   uint8_t *__restrict__ dst, long long nchunks)
{
    __shared__ __align__(16) uint8_t s_in[2][34 * RQ_CHUNK];
    __shared__ __align__(16) uint8_t s_out[18 * RQ_CHUNK];
    const int tid = threadIdx.x;
    long long ch = blockIdx.x;
    int buf = 0;
    if (ch < nchunks) rq_issue_q8_chunk(s_in[0], src + ch * (34ll * RQ_CHUNK), tid);
    for (; ch < nchunks; ch += gridDim.x) {
        const long long nx = ch + gridDim.x;
        if (nx < nchunks) {
            // s_in[buf ^ 1] was last read before the previous chunk's second barrier
            rq_issue_q8_chunk(s_in[buf ^ 1], src + nx * (34ll * RQ_CHUNK), tid);
            asm volatile("cp.async.wait_group 1;" ::: "memory");  // this chunk's group is complete
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        rq_encode_q8_chunk(s_in[buf], s_out, tid);
        __syncthreads();
        int4 *go = reinterpret_cast<int4 *>(dst + ch * (18ll * RQ_CHUNK));
        for (int i = tid; i < 18 * RQ_CHUNK / 16; i += RQ_CHUNK) go[i] = reinterpret_cast<const int4 *>(s_out)[i];
        buf ^= 1;
        // s_out is written again only after the next chunk's first barrier
    }
}

template <bool FROM_Q8>
__global__ void __launch_bounds__(RQ_CHUNK) requant_q4_0_staged(const uint8_t *__restrict__ src,
                                                                uint8_t *__restrict__ dst, long long nchunks)
{
    constexpr int IN_BYTES = FROM_Q8 ? 34 * RQ_CHUNK : QK * 257 * 4;  // staging area
    constexpr int IN_LOADS = (FROM_Q8 ? 34 : 128) * RQ_CHUNK / 16;     // 16-byte loads per chunk
    constexpr int OUT_STORES = 18 * RQ_CHUNK / 16;
    __shared__ __align__(16) uint8_t s_in[IN_BYTES];
    __shared__ __align__(16) uint8_t s_out[18 * RQ_CHUNK];
    const int tid = threadIdx.x;
    for (long long ch = blockIdx.x; ch < nchunks; ch += gridDim.x) {
        const int4 *g = reinterpret_cast<const int4 *>(src + ch * (IN_LOADS * 16ll));
        if constexpr (FROM_Q8) {
            for (int i = tid; i < IN_LOADS; i += RQ_CHUNK) reinterpret_cast<int4 *>(s_in)[i] = __ldg(g + i);
        } else {
            float *t = reinterpret_cast<float *>(s_in);
            for (int i = tid; i < IN_LOADS; i += RQ_CHUNK) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(g) + i);
                const int b = i >> 3, j = (i & 7) * 4;  // block, first element
                t[j * 257 + b] = v.x;
                t[(j + 1) * 257 + b] = v.y;
                t[(j + 2) * 257 + b] = v.z;
                t[(j + 3) * 257 + b] = v.w;
            }
        }
        __syncthreads();
        float x[QK];
        if constexpr (FROM_Q8) {
            const unsigned short *h = reinterpret_cast<const unsigned short *>(s_in + tid * 34);
            const float d8 = __half2float(__ushort_as_half(h[0]));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const unsigned w = h[1 + i];
                x[2 * i] = __fmul_rn(q8_code_to_float(w & 0xFFu), d8);
                x[2 * i + 1] = __fmul_rn(q8_code_to_float(w >> 8), d8);
            }
        } else {
            const float *t = reinterpret_cast<const float *>(s_in);
#pragma unroll
            for (int j = 0; j < QK; ++j) x[j] = t[j * 257 + tid];
        }
        unsigned short o[9];
        q4_encode_block(x, o);
        unsigned short *so = reinterpret_cast<unsigned short *>(s_out + tid * 18);
#pragma unroll
        for (int i = 0; i < 9; ++i) so[i] = o[i];
        __syncthreads();
        int4 *go = reinterpret_cast<int4 *>(dst + ch * (OUT_STORES * 16ll));
        for (int i = tid; i < OUT_STORES; i += RQ_CHUNK) go[i] = reinterpret_cast<const int4 *>(s_out)[i];
        // the next chunk's staging stores wait for these reads at its first barrier;
        // its s_out writes come after that barrier too
    }
}

cudaError_t launch_requant_q4_0(const void *src, bool from_q8, void *dst, long long nblocks, cudaStream_t st)
{
    const uint8_t *s8 = static_cast<const uint8_t *>(src);
    uint8_t *o = static_cast<uint8_t *>(dst);
    const bool aligned16 = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
    long long done = 0;
    if (aligned16 && nblocks >= RQ_CHUNK) {
        const long long nchunks = nblocks / RQ_CHUNK;
        // fp32: 5 resident CTAs per SM (37 KB of shared memory each), many waves; Q8_0:
        // four CTAs per SM of the 152-SM grid walk the chunks with the next one in flight
        long long grid = nchunks < 152ll * 8 * 16 ? nchunks : 152ll * 8 * 16;
        if (from_q8)
            requant_q4_0_staged_q8<<<static_cast<unsigned>(nchunks < 152ll * 4 ? nchunks : 152ll * 4), RQ_CHUNK, 0,
                                     st>>>(s8, o, nchunks);
        else
            requant_q4_0_staged<false><<<static_cast<unsigned>(grid), RQ_CHUNK, 0, st>>>(s8, o, nchunks);
        done = nchunks * RQ_CHUNK;
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess || done == nblocks) return e;
    }
    // the rest (or everything, unaligned): one thread per block
    const long long rest = nblocks - done;
    const void *s = s8 + done * (from_q8 ? 34 : 128);
    o += done * 18;
    long long grid = (rest + 255) / 256;
    if (grid > (1 << 20)) grid = 1 << 20;
    const dim3 g(static_cast<unsigned>(grid));
    if (from_q8)
        requant_q4_0_kernel<true, false><<<g, 256, 0, st>>>(s, o, rest);
    else if ((reinterpret_cast<uintptr_t>(s) & 15) == 0)
        requant_q4_0_kernel<false, true><<<g, 256, 0, st>>>(s, o, rest);
    else
        requant_q4_0_kernel<false, false><<<g, 256, 0, st>>>(s, o, rest);
    return cudaGetLastError();
}

}  // namespace qg
