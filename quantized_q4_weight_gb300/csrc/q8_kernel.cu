// q8_kernel.cu -- the Q8_0-weight decode GEMV y = W.x (minfer README "How it
// works": gemv_q8_dp4a; M14: the lm_head held as Q8_0).  A weight block is a
// Q8_0 block, fp16 d then 32 int8 q, and the weight is q * d.  Activations
// are the same planar Q8_0 as the Q4_0 path's.
//
// Device layout (qgemv_pack_q8_0; same byte count as GGML's [N][nb][34]):
// slabs of 16 rows, each a run of stages of 8 blocks (256 weights per row).
// A full stage is 4352 bytes: [16 rows][16 chunks of 16 bytes] of int8 q,
// chunk c of row r stored at position c ^ (r & 7), then the fp16 scales as
// [16 rows][2 parities][4].  A partial last stage of nbs < 8 blocks is
// [16][nbs][32] q then [16][nbs] scales, unswizzled.  The N % 16 tail rows
// stay in GGML layout after the slabs.
//
// Lane (r, h) = (lane & 15, lane >> 4) computes row r over the blocks 2i + h
// of each stage.  Fixed fp32 order, a function of K alone: the lane's sum of
// its blocks in increasing order (from zero), then the two parities added
// (h = 0 plus h = 1), then the stage sums folded in stage order.  The block
// sum isum = sum w q is exact in int32 (8 dp4a), and (d_w d_x) is exact in
// fp32, so each term is one fused multiply-add.
#include <atomic>

#include "qgemv_launch.h"

namespace qg {

constexpr int Q8_STAGE_BLOCKS = 8;
constexpr int Q8_BLOCK_BYTES = 34;
constexpr int Q8_STAGE_BYTES = SLAB_ROWS * Q8_STAGE_BLOCKS * Q8_BLOCK_BYTES;  // 4352

// ------------------------------------------------------------------ packing

// Byte offset, within a slab, of block b of row r (q bytes) and of its scale.
__host__ __device__ inline void q8_pack_offsets(int r, int b, int nb, long long &q_off, long long &d_off)
{
    const int st = b / Q8_STAGE_BLOCKS, bs = b - st * Q8_STAGE_BLOCKS;
    const int nbs = min(Q8_STAGE_BLOCKS, nb - st * Q8_STAGE_BLOCKS);
    const long long base = static_cast<long long>(st) * Q8_STAGE_BYTES;
    if (nbs == Q8_STAGE_BLOCKS) {
        q_off = base + r * 256;  // chunk-level swizzle applied per 16-byte chunk by the caller
        d_off = base + 4096 + (r * 2 + (bs & 1)) * 8 + (bs >> 1) * 2;
    } else {
        q_off = base + (r * nbs + bs) * 32;
        d_off = base + SLAB_ROWS * nbs * 32 + (r * nbs + bs) * 2;
    }
}

// One thread per (row, block): moves the block's 34 bytes between GGML and
// the packed layout (to_packed) or back.
__global__ void q8_pack_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, long long N, int nb,
                               bool to_packed)
{
    const long long nslabs = N / SLAB_ROWS;
    const long long slab_bytes = static_cast<long long>(SLAB_ROWS) * nb * Q8_BLOCK_BYTES;
    const long long total = N * nb;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = i / nb;
        const int b = static_cast<int>(i - row * nb);
        const long long g = i * Q8_BLOCK_BYTES;  // GGML offset
        if (row >= nslabs * SLAB_ROWS) {          // tail rows: same place in both layouts
            for (int k = 0; k < Q8_BLOCK_BYTES; ++k) dst[g + k] = src[g + k];
            continue;
        }
        const int r = static_cast<int>(row % SLAB_ROWS);
        long long q_off, d_off;
        q8_pack_offsets(r, b, nb, q_off, d_off);
        const long long sb = (row / SLAB_ROWS) * slab_bytes;
        const int st = b / Q8_STAGE_BLOCKS, bs = b - st * Q8_STAGE_BLOCKS;
        const bool full = nb - st * Q8_STAGE_BLOCKS >= Q8_STAGE_BLOCKS;
        long long qpos[2];
        for (int h = 0; h < 2; ++h) {
            const int c = 2 * bs + h;  // 16-byte chunk of the row within the stage
            qpos[h] = sb + (full ? q_off + 16 * (c ^ (r & 7)) : q_off + 16 * h);
        }
        if (to_packed) {
            dst[sb + d_off] = src[g];
            dst[sb + d_off + 1] = src[g + 1];
            for (int k = 0; k < 32; ++k) dst[qpos[k >> 4] + (k & 15)] = src[g + 2 + k];
        } else {
            dst[g] = src[sb + d_off];
            dst[g + 1] = src[sb + d_off + 1];
            for (int k = 0; k < 32; ++k) dst[g + 2 + k] = src[qpos[k >> 4] + (k & 15)];
        }
    }
}

cudaError_t launch_q8_pack(const void *src, void *dst, long long N, long long K, bool to_packed, cudaStream_t st)
{
    const long long total = N * (K / QK);
    long long grid = (total + 255) / 256;
    if (grid > 65535) grid = 65535;
    if (grid < 1) grid = 1;
    q8_pack_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<const uint8_t *>(src),
                                                                static_cast<uint8_t *>(dst), N,
                                                                static_cast<int>(K / QK), to_packed);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ GEMV

// Launch parameters of the Q8_0-weight GEMV (host-computed plan).
struct Q8Params {
    const uint8_t *W;   // packed weights
    const uint8_t *xq;  // planar Q8_0: [T][K] int8, then [T][nb] fp16
    float *y;           // [T][N]
    float *part;        // [nslabs][nstage][T][16] stage sums of slabs split over warps
    unsigned *cnt;      // [nslabs] arrival counters (left at zero)
    unsigned *status;   // per-device status word
    long long N;
    int K, nb, nstage, nslabs, tail_rows;
    int chunks;         // warps (items) per slab: stage ranges of one slab
    int items;          // nslabs * chunks (+ 1 for the tail rows)
    int nwarps, ring_depth;
    int off_dx, off_bar, off_ring;  // dynamic shared memory: [x codes][dx][barriers][rings]
};

__device__ __forceinline__ int dp4a_ss8(const uint4 &w0, const uint4 &w1, const uint4 &x0, const uint4 &x1)
{
    int s = 0;
    s = dp4a_ss(static_cast<int>(w0.x), static_cast<int>(x0.x), s);
    s = dp4a_ss(static_cast<int>(w0.y), static_cast<int>(x0.y), s);
    s = dp4a_ss(static_cast<int>(w0.z), static_cast<int>(x0.z), s);
    s = dp4a_ss(static_cast<int>(w0.w), static_cast<int>(x0.w), s);
    s = dp4a_ss(static_cast<int>(w1.x), static_cast<int>(x1.x), s);
    s = dp4a_ss(static_cast<int>(w1.y), static_cast<int>(x1.y), s);
    s = dp4a_ss(static_cast<int>(w1.z), static_cast<int>(x1.z), s);
    s = dp4a_ss(static_cast<int>(w1.w), static_cast<int>(x1.w), s);
    return s;  // |s| <= 32 * 128 * 127 < 2^20
}

// The lane's terms of one block for every token: acc[t] += (d_w d_x) isum.
// isum enters fp32 exactly through the magic-number form (|isum| < 2^22).
template <int T>
__device__ __forceinline__ void q8_block_terms(const uint4 &w0, const uint4 &w1, float dw, uint32_t xa, int xs,
                                               const float *dxp, int dx_tstride, float (&acc)[T])
{
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const uint4 x0 = lds128(xa + t * xs), x1 = lds128(xa + t * xs + 16);
        const int isum = dp4a_ss8(w0, w1, x0, x1);
        const float f = __fsub_rn(__int_as_float(MAGIC_I + isum), MAGIC_F);
        acc[t] = __fmaf_rn(__fmul_rn(dw, dxp[t * dx_tstride]), f, acc[t]);
    }
}

// Stage sums of one stage for this lane's row: blocks 2i + h in increasing
// order from +0, then the two parities added.  sa: the stage in shared memory.
template <int T>
__device__ __forceinline__ void q8_stage_sums(uint32_t sa, int st, int nbs, int r, int h, uint32_t ximg, int xs,
                                              const float *dxi, int nstage, float (&ss)[T])
{
    float acc[T];
#pragma unroll
    for (int t = 0; t < T; ++t) acc[t] = 0.0f;
    const float *dxp = dxi + (st * 2 + h) * 4;  // [t][stage][h][4]
    const int dxt = nstage * 8;
    if (nbs == Q8_STAGE_BLOCKS) {
        unsigned dws[2];
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(dws[0]), "=r"(dws[1]) : "r"(sa + 4096 + (r * 2 + h) * 8));
        const uint32_t row = sa + r * 256;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c0 = 4 * i + 2 * h;  // the block's two 16-byte chunks
            const uint4 w0 = lds128(row + 16 * (c0 ^ (r & 7))), w1 = lds128(row + 16 * ((c0 + 1) ^ (r & 7)));
            const unsigned short d16 = static_cast<unsigned short>((i & 1) ? dws[i >> 1] >> 16 : dws[i >> 1] & 0xFFFFu);
            const int b = st * Q8_STAGE_BLOCKS + 2 * i + h;
            q8_block_terms<T>(w0, w1, h2f(d16), ximg + b * QK, xs, dxp + i, dxt, acc);
        }
    } else {
        for (int i = 0; 2 * i + h < nbs; ++i) {
            const int bs = 2 * i + h;
            const uint32_t q = sa + (r * nbs + bs) * 32;
            const uint4 w0 = lds128(q), w1 = lds128(q + 16);
            unsigned short d16;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(d16) : "r"(sa + SLAB_ROWS * nbs * 32 + (r * nbs + bs) * 2));
            const int b = st * Q8_STAGE_BLOCKS + bs;
            q8_block_terms<T>(w0, w1, h2f(d16), ximg + b * QK, xs, dxp + i, dxt, acc);
        }
    }
#pragma unroll
    for (int t = 0; t < T; ++t) ss[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xFFFFFFFFu, acc[t], 16));
}

// One GGML block (34 bytes, 2-byte aligned) from global memory: scale and codes.
__device__ __forceinline__ void q8_ggml_block(const uint8_t *p, unsigned short &d, uint4 &w0, uint4 &w1)
{
    const unsigned short *h = reinterpret_cast<const unsigned short *>(p);
    d = __ldg(h);
    unsigned w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        w[k] = static_cast<unsigned>(__ldg(h + 1 + 2 * k)) | (static_cast<unsigned>(__ldg(h + 2 + 2 * k)) << 16);
    w0 = make_uint4(w[0], w[1], w[2], w[3]);
    w1 = make_uint4(w[4], w[5], w[6], w[7]);
}

template <int T>
__global__ void __launch_bounds__(NWARPS_MAX * 32, 1) q8_gemv_kernel(const __grid_constant__ Q8Params P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = lane & 15, h = lane >> 4;
    const int nw = P.nwarps, D = P.ring_depth, nthreads = nw * 32;
    const int xs = P.K;
    const uint32_t ximg = smem_addr(smem);
    float *dxi = reinterpret_cast<float *>(smem + P.off_dx);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + P.off_bar) + warp * D;
    uint8_t *ring = smem + P.off_ring + static_cast<size_t>(warp) * D * Q8_STAGE_BYTES;
    volatile int *abort_flag = &s_abort;
    const long long slab_bytes = static_cast<long long>(SLAB_ROWS) * P.nb * Q8_BLOCK_BYTES;
    const int last_nbs = P.nb - (P.nstage - 1) * Q8_STAGE_BLOCKS;
    const int G = gridDim.x * nw, gw = blockIdx.x * nw + warp;
    const int slab_items = P.nslabs * P.chunks;

    if (tid == 0) s_abort = 0;
    if (lane == 0)
        for (int d = 0; d < D; ++d) mbar_init(&bar[d], 1);
    fence_mbar_init();
    __syncthreads();
    pdl_launch_dependents();

    // the TMA walker over this warp's stages: items gw, gw + G, ... (slab items only)
    int c_it = gw, c_st = 0, c_end = 0;
    auto c_enter = [&](int it) {
        c_it = it;
        if (it < slab_items) {
            const int sl = it / P.chunks, c = it - sl * P.chunks;
            c_st = P.nstage * c / P.chunks;
            c_end = P.nstage * (c + 1) / P.chunks;
        }
    };
    c_enter(gw);
    auto c_valid = [&]() { return c_it < slab_items; };
    auto c_step = [&]() {
        if (++c_st >= c_end) c_enter(c_it + G);
    };
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int slot) {
        if (lane == 0) {
            const int sl = c_it / P.chunks;
            const unsigned bytes = c_st == P.nstage - 1 ? static_cast<unsigned>(SLAB_ROWS * last_nbs * Q8_BLOCK_BYTES)
                                                        : static_cast<unsigned>(Q8_STAGE_BYTES);
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[slot], bytes);
            bulk_g2s(ring + slot * Q8_STAGE_BYTES,
                     P.W + sl * slab_bytes + static_cast<long long>(c_st) * Q8_STAGE_BYTES, bytes, &bar[slot], pol);
        }
    };
    int issued = 0;
    for (int d = 0; d < D && c_valid(); ++d) {
        issue(d);
        ++issued;
        c_step();
    }

    // activations after the preceding kernel: codes as copied, scales as fp32
    // in [t][stage][parity][4] order
    pdl_wait();
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(P.xq);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        for (int i = tid; i < T * P.K / 16; i += nthreads) dst[i] = __ldcg(src + i);
        const unsigned short *xd = reinterpret_cast<const unsigned short *>(P.xq + static_cast<long long>(T) * P.K);
        for (int i = tid; i < T * P.nb; i += nthreads) {
            const int t = i / P.nb, b = i - t * P.nb;
            const int st = b / Q8_STAGE_BLOCKS, bs = b - st * Q8_STAGE_BLOCKS;
            dxi[((t * P.nstage + st) * 2 + (bs & 1)) * 4 + (bs >> 1)] = h2f(__ldcg(xd + i));
        }
    }
    __syncthreads();

    int slot = 0, consumed = 0;
    unsigned phase = 0;
    bool ok = true;
    for (int it = gw; it < P.items; it += G) {
        float ss[T], tot[T];
#pragma unroll
        for (int t = 0; t < T; ++t) tot[t] = 0.0f;
        if (it >= slab_items) {
            // the N % 16 tail rows, in GGML layout: direct loads, the same order
            const long long row = static_cast<long long>(P.nslabs) * SLAB_ROWS + r;
            const bool live = r < P.tail_rows;
            for (int st = 0; st < P.nstage; ++st) {
                float acc[T];
#pragma unroll
                for (int t = 0; t < T; ++t) acc[t] = 0.0f;
                const float *dxp = dxi + (st * 2 + h) * 4;
                for (int i = 0; i < 4; ++i) {
                    const int b = st * Q8_STAGE_BLOCKS + 2 * i + h;
                    if (live && b < P.nb) {
                        unsigned short d16;
                        uint4 w0, w1;
                        q8_ggml_block(P.W + (row * P.nb + b) * Q8_BLOCK_BYTES, d16, w0, w1);
                        q8_block_terms<T>(w0, w1, h2f(d16), ximg + b * QK, xs, dxp + i, P.nstage * 8, acc);
                    }
                }
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    ss[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xFFFFFFFFu, acc[t], 16));
                    tot[t] = st == 0 ? ss[t] : __fadd_rn(tot[t], ss[t]);
                }
            }
            if (live && h == 0)
#pragma unroll
                for (int t = 0; t < T; ++t) P.y[static_cast<long long>(t) * P.N + row] = tot[t];
            continue;
        }
        const int sl = it / P.chunks, c = it - sl * P.chunks;
        const int a = P.nstage * c / P.chunks, e = P.nstage * (c + 1) / P.chunks;
        const bool split = P.chunks > 1;
        for (int st = a; st < e; ++st) {
            if (ok) ok = mbar_wait_bounded(&bar[slot], phase, abort_flag, P.status, WAIT_LIMIT_NS);
            if (ok) {
                const int nbs = st == P.nstage - 1 ? last_nbs : Q8_STAGE_BLOCKS;
                q8_stage_sums<T>(smem_addr(ring + slot * Q8_STAGE_BYTES), st, nbs, r, h, ximg, xs, dxi, P.nstage, ss);
            } else {
#pragma unroll
                for (int t = 0; t < T; ++t) ss[t] = 0.0f;
            }
            __syncwarp();
            ++consumed;
            if (c_valid() && ok) {  // refill the slot just consumed
                issue(slot);
                ++issued;
                c_step();
            }
            if (++slot == D) {
                slot = 0;
                phase ^= 1u;
            }
            if (split) {
                if (h == 0)
#pragma unroll
                    for (int t = 0; t < T; ++t)
                        P.part[((static_cast<long long>(sl) * P.nstage + st) * T + t) * SLAB_ROWS + r] = ss[t];
            } else {
#pragma unroll
                for (int t = 0; t < T; ++t) tot[t] = st == a ? ss[t] : __fadd_rn(tot[t], ss[t]);
            }
        }
        const long long row = static_cast<long long>(sl) * SLAB_ROWS + r;
        if (!split) {
            if (h == 0)
#pragma unroll
                for (int t = 0; t < T; ++t) P.y[static_cast<long long>(t) * P.N + row] = tot[t];
            continue;
        }
        // the last of the slab's warps folds every stage sum in stage order
        __threadfence();
        __syncwarp();
        unsigned old = 0;
        if (lane == 0) old = atomicAdd(P.cnt + sl, 1u);
        old = __shfl_sync(0xFFFFFFFFu, old, 0);
        if (old == static_cast<unsigned>(P.chunks - 1)) {
            __threadfence();
            if (h == 0)
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const float *pb = P.part + (static_cast<long long>(sl) * P.nstage * T + t) * SLAB_ROWS + r;
                    const float v = ordered_sum_ldcg(pb, P.nstage, static_cast<long long>(T) * SLAB_ROWS);
                    P.y[static_cast<long long>(t) * P.N + row] = v;
                }
            __syncwarp();
            if (lane == 0) P.cnt[sl] = 0u;
        }
    }
    // copies still in flight (only after an abort): wait for them, bounded
    while (consumed < issued) {
        mbar_drain(&bar[slot], phase);
        ++consumed;
        if (++slot == D) {
            slot = 0;
            phase ^= 1u;
        }
    }
}

template <int T>
cudaError_t launch_q8_t(const Q8Params &P, int grid, size_t smem, cudaStream_t st)
{
    auto kern = q8_gemv_kernel<T>;
    static std::atomic<unsigned long long> raised{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(raised.load(std::memory_order_acquire) & bit)) {
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        raised.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(P.nwarps * 32));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

// Plan (workspace, shared memory, launch shape) and, when do_launch, launch.
cudaError_t launch_q8(const void *W, const void *xq, float *y, long long N, long long K, int T, void *ws,
                      long long ws_bytes, bool do_launch, int sms, int smem_budget, unsigned *status,
                      cudaStream_t st, long long *ws_need, int *unsupported)
{
    Q8Params P = {};
    P.W = static_cast<const uint8_t *>(W);
    P.xq = static_cast<const uint8_t *>(xq);
    P.y = y;
    P.status = status;
    P.N = N;
    P.K = static_cast<int>(K);
    P.nb = P.K / QK;
    P.nstage = (P.nb + Q8_STAGE_BLOCKS - 1) / Q8_STAGE_BLOCKS;
    P.nslabs = static_cast<int>(N / SLAB_ROWS);
    P.tail_rows = static_cast<int>(N % SLAB_ROWS);
    const int grid = sms;
    // warps per slab: spread few slabs over the launch's warps by stage ranges
    long long ch = P.nslabs > 0 ? (static_cast<long long>(grid) * NWARPS_MAX + P.nslabs - 1) / P.nslabs : 1;
    if (ch > P.nstage) ch = P.nstage;
    if (ch < 1) ch = 1;
    P.chunks = static_cast<int>(ch);
    P.items = P.nslabs * P.chunks + (P.tail_rows > 0 ? 1 : 0);
    long long need = 0;
    if (P.chunks > 1) {
        need = 256 + (4ll * P.nslabs + 255) / 256 * 256 + 4ll * P.nslabs * P.nstage * T * SLAB_ROWS;
    }
    *ws_need = need;
    *unsupported = 0;
    // shared memory: codes, dx, barriers, rings; the widest shape that fits
    const long long xbytes = (static_cast<long long>(T) * K + 127) / 128 * 128;
    const long long dxbytes = (static_cast<long long>(T) * P.nstage * 32 + 127) / 128 * 128;
    const int shapes[4][2] = {{16, 2}, {16, 1}, {8, 2}, {8, 1}};
    int nw = 0, D = 0;
    long long smem = 0;
    for (const auto &c : shapes) {
        const long long bars = (8ll * c[0] * c[1] + 127) / 128 * 128;
        const long long total = xbytes + dxbytes + bars + static_cast<long long>(c[0]) * c[1] * Q8_STAGE_BYTES;
        if (total <= smem_budget) {
            nw = c[0];
            D = c[1];
            smem = total;
            P.off_dx = static_cast<int>(xbytes);
            P.off_bar = static_cast<int>(xbytes + dxbytes);
            P.off_ring = static_cast<int>(xbytes + dxbytes + bars);
            break;
        }
    }
    if (nw == 0) {
        *unsupported = 1;
        return cudaSuccess;
    }
    if (!do_launch) return cudaSuccess;
    if (need > 0 && (ws == nullptr || ws_bytes < need)) {
        *unsupported = 2;
        return cudaSuccess;
    }
    P.nwarps = nw;
    P.ring_depth = D;
    if (P.chunks > 1) {
        uint8_t *w = static_cast<uint8_t *>(ws);
        P.cnt = reinterpret_cast<unsigned *>(w + 256);
        P.part = reinterpret_cast<float *>(w + 256 + (4ll * P.nslabs + 255) / 256 * 256);
    }
    switch (T) {
    case 1: return launch_q8_t<1>(P, grid, static_cast<size_t>(smem), st);
    case 2: return launch_q8_t<2>(P, grid, static_cast<size_t>(smem), st);
    case 3: return launch_q8_t<3>(P, grid, static_cast<size_t>(smem), st);
    case 4: return launch_q8_t<4>(P, grid, static_cast<size_t>(smem), st);
    case 5: return launch_q8_t<5>(P, grid, static_cast<size_t>(smem), st);
    case 6: return launch_q8_t<6>(P, grid, static_cast<size_t>(smem), st);
    case 7: return launch_q8_t<7>(P, grid, static_cast<size_t>(smem), st);
    case 8: return launch_q8_t<8>(P, grid, static_cast<size_t>(smem), st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
