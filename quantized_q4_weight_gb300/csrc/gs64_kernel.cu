// gs64_kernel.cu -- the grouped int4 GEMV with per-vector int8 activations
// (colibri qwen36 docs: the gs64 container, one scale per 64-weight group,
// its nibbles repacked once into a planar layout where one AND gives a
// group's first 32 elements in order and one shift the other 32; the dense
// int8 IDOT GEMV: the activation quantised to int8 once per call, one scale
// amax / 127, exact int32 sums scaled afterwards).
//
// Format (the reading this library takes where the pages leave it open):
//   - a group is 64 weights of one row in 32 bytes: byte j (j < 32) holds
//     element j in its low nibble and element j + 32 in its high nibble; the
//     weight is (n - 8) * s with one fp32 scale s per group (4.5 bits per
//     weight, as the pages count the container);
//   - the activation row of K values has one fp32 scale s_x = amax / 127 and
//     int8 codes q = round-half-away(x * (1 / s_x)) (all zero when amax = 0);
//   - y = s_x * sum_g s_g * isum_g, isum_g = sum_e (n_e - 8) q_e exact in int32.
//
// Device layout (qgemv_pack_gs64, 36 bytes per group as in the row planes):
// slabs of 16 rows, each a run of stages of 8 groups (512 weights per row).
// A full stage is 4608 bytes: [16 rows][16 chunks of 16 bytes] of nibbles,
// chunk c of row r (group c / 2, half c % 2) at position c ^ (r & 7), then the
// fp32 scales as [16 rows][2 parities][4].  A partial last stage of ngs < 8
// groups is [16][ngs][32] nibbles then [16][ngs] scales, unswizzled.  The
// N % 16 tail rows follow the slabs, each as its [ng][32] nibbles then its
// [ng] scales.
//
// Lane (r, h) = (lane & 15, lane >> 4) computes row r over the groups 2i + h
// of each stage.  Fixed fp32 order, a function of K alone: per stage the
// lane's groups in increasing order from +0, each term one fused
// multiply-add s_g * (16 isum_g); the two parities added; the stage sums
// added in stage order; the total times 1/16, then times s_x.  16 isum is
// exact in fp32 (|16 isum| <= 16 * 64 * 8 * 127 < 2^21).
#include <atomic>

#include "qgemv_launch.h"

namespace qg {

constexpr int G64_W = 64;             // weights per group
constexpr int G64_NIB = 32;           // nibble bytes per group
constexpr int G64_BYTES = 36;         // nibbles + fp32 scale
constexpr int G64_STAGE_GROUPS = 8;
constexpr int G64_STAGE_BYTES = SLAB_ROWS * G64_STAGE_GROUPS * G64_BYTES;  // 4608

// ------------------------------------------------------------------ packing

// Byte offsets, within its slab, of group g of row r: the nibble chunk k
// (k = 0, 1: bytes 16k..16k+15) and the scale.
__host__ __device__ inline void g64_offsets(int r, int g, int k, int ng, long long &n_off, long long &s_off)
{
    const int st = g / G64_STAGE_GROUPS, gs = g - st * G64_STAGE_GROUPS;
    const int ngs = ng - st * G64_STAGE_GROUPS < G64_STAGE_GROUPS ? ng - st * G64_STAGE_GROUPS : G64_STAGE_GROUPS;
    const long long base = static_cast<long long>(st) * G64_STAGE_BYTES;
    if (ngs == G64_STAGE_GROUPS) {
        const int c = 2 * gs + k;
        n_off = base + r * 256 + 16 * (c ^ (r & 7));
        s_off = base + 4096 + (r * 2 + (gs & 1)) * 16 + (gs >> 1) * 4;
    } else {
        n_off = base + (r * ngs + gs) * G64_NIB + 16 * k;
        s_off = base + SLAB_ROWS * ngs * G64_NIB + (r * ngs + gs) * 4;
    }
}

// One thread per (row, group): moves the group's 32 nibble bytes and its
// scale between the row planes (wq [N][ng][32], ws [N][ng]) and the packed
// layout (to_packed), or back.
__global__ void g64_pack_kernel(uint8_t *__restrict__ wq, float *__restrict__ wsc, uint8_t *__restrict__ packed,
                                long long N, int ng, bool to_packed)
{
    const long long nslabs = N / SLAB_ROWS;
    const long long slab_bytes = static_cast<long long>(SLAB_ROWS) * ng * G64_BYTES;
    const long long total = N * ng;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = i / ng;
        const int g = static_cast<int>(i - row * ng);
        uint8_t *plane = wq + i * G64_NIB;
        long long n_off[2], s_off;
        if (row >= nslabs * SLAB_ROWS) {  // tail rows: [ng][32] nibbles, then [ng] scales
            const long long tb = nslabs * slab_bytes + (row - nslabs * SLAB_ROWS) * ng * G64_BYTES;
            n_off[0] = tb + static_cast<long long>(g) * G64_NIB;
            n_off[1] = n_off[0] + 16;
            s_off = tb + static_cast<long long>(ng) * G64_NIB + 4ll * g;
        } else {
            const long long sb = (row / SLAB_ROWS) * slab_bytes;
            const int r = static_cast<int>(row % SLAB_ROWS);
            long long s1;
            g64_offsets(r, g, 0, ng, n_off[0], s_off);
            g64_offsets(r, g, 1, ng, n_off[1], s1);
            n_off[0] += sb;
            n_off[1] += sb;
            s_off += sb;
        }
        unsigned *ps = reinterpret_cast<unsigned *>(packed + s_off);  // 4-byte aligned in both forms
        unsigned *ss = reinterpret_cast<unsigned *>(wsc + i);
        if (to_packed) {
            for (int k = 0; k < 32; ++k) packed[n_off[k >> 4] + (k & 15)] = plane[k];
            *ps = *ss;
        } else {
            for (int k = 0; k < 32; ++k) plane[k] = packed[n_off[k >> 4] + (k & 15)];
            *ss = *ps;
        }
    }
}

cudaError_t launch_gs64_pack(void *wq, float *wsc, void *packed, long long N, long long K, bool to_packed,
                             cudaStream_t st)
{
    const long long total = N * (K / G64_W);
    long long grid = (total + 255) / 256;
    if (grid > 65535) grid = 65535;
    if (grid < 1) grid = 1;
    g64_pack_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<uint8_t *>(wq), wsc,
                                                                  static_cast<uint8_t *>(packed), N,
                                                                  static_cast<int>(K / G64_W), to_packed);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ quantiser

// One CTA per activation row: s = amax / 127 over the whole row (fp32, IEEE
// division), 1/s from it (0 when s = 0), q = roundf(x * (1/s)) -- the Q8_0
// quantiser's steps over a row instead of a 32-value block.
__global__ void __launch_bounds__(1024) quantize_vec_i8_kernel(const float *__restrict__ x, int8_t *__restrict__ q,
                                                               float *__restrict__ s, long long K)
{
    __shared__ float s_max[32];
    __shared__ float s_id;
    const float *xr = x + static_cast<long long>(blockIdx.x) * K;
    int8_t *qr = q + static_cast<long long>(blockIdx.x) * K;
    float amax = 0.0f;
    for (long long k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(__ldg(xr + k)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float m = threadIdx.x < (blockDim.x >> 5) ? s_max[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (threadIdx.x == 0) {
            float d, id;
            q8_scale(m, d, id);  // the maximum is exact in any order
            s[blockIdx.x] = d;
            s_id = id;
        }
    }
    __syncthreads();
    const float id = s_id;
    for (long long k = threadIdx.x; k < K; k += blockDim.x) qr[k] = static_cast<int8_t>(q8_code(__ldg(xr + k), id));
}

cudaError_t launch_quantize_vec_i8(const float *x, int8_t *q, float *s, int R, long long K, cudaStream_t st)
{
    quantize_vec_i8_kernel<<<static_cast<unsigned>(R), 1024, 0, st>>>(x, q, s, K);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ GEMV

struct G64Params {
    const uint8_t *W;   // packed weights
    const int8_t *q;    // activation codes [T][K]
    const float *sx;    // activation scales [T]
    const float *xf;    // or fp32 activations [T][K], quantised in the kernel (q, sx unused)
    float *y;           // [T][N]
    float *part;        // [nslabs][nstage][T][16] stage sums of slabs split over warps
    unsigned *cnt;      // [nslabs] arrival counters (left at zero)
    unsigned *status;   // per-device status word
    long long N;
    int K, ng, nstage, nslabs, tail_rows;
    int chunks;         // warps (items) per slab: stage ranges of one slab
    int items;          // nslabs * chunks (+ 1 for the tail rows)
    int nwarps, ring_depth;
    int off_c, off_bar, off_ring;  // dynamic shared memory: [codes][folded constants][barriers][rings]
};

// The lane's term of one group for every token: acc[t] += s_g * (16 isum).
// n0: bytes 0..15 of the group (elements 0..15 low, 32..47 high), n1: bytes
// 16..31 (elements 16..31 low, 48..63 high).  The low nibbles are masked in
// place, the high ones without a shift (that chain sums 16 n q); the two
// meet in one shift-add with the folded constant MAGIC - 128 sum(q).
template <int T>
__device__ __forceinline__ void g64_group_terms(const uint4 &n0, const uint4 &n1, float sg, uint32_t xa, int xs,
                                                const int *cg, int cg_tstride, float (&acc)[T])
{
    const unsigned lo_m = 0x0F0F0F0Fu, hi_m = 0xF0F0F0F0u;
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const uint32_t a = xa + t * xs;
        const uint4 q0 = lds128(a), q1 = lds128(a + 16), q2 = lds128(a + 32), q3 = lds128(a + 48);
        int lo = 0, hi = cg[t * cg_tstride];
        lo = dp4a_us(n0.x & lo_m, (int)q0.x, lo);
        hi = dp4a_us(n0.x & hi_m, (int)q2.x, hi);
        lo = dp4a_us(n0.y & lo_m, (int)q0.y, lo);
        hi = dp4a_us(n0.y & hi_m, (int)q2.y, hi);
        lo = dp4a_us(n0.z & lo_m, (int)q0.z, lo);
        hi = dp4a_us(n0.z & hi_m, (int)q2.z, hi);
        lo = dp4a_us(n0.w & lo_m, (int)q0.w, lo);
        hi = dp4a_us(n0.w & hi_m, (int)q2.w, hi);
        lo = dp4a_us(n1.x & lo_m, (int)q1.x, lo);
        hi = dp4a_us(n1.x & hi_m, (int)q3.x, hi);
        lo = dp4a_us(n1.y & lo_m, (int)q1.y, lo);
        hi = dp4a_us(n1.y & hi_m, (int)q3.y, hi);
        lo = dp4a_us(n1.z & lo_m, (int)q1.z, lo);
        hi = dp4a_us(n1.z & hi_m, (int)q3.z, hi);
        lo = dp4a_us(n1.w & lo_m, (int)q1.w, lo);
        hi = dp4a_us(n1.w & hi_m, (int)q3.w, hi);
        acc[t] = __fmaf_rn(sg, magic_to_float((lo << 4) + hi), acc[t]);  // MAGIC + 16 isum, exact
    }
}

// Stage sums of one stage for this lane's row (groups 2i + h in increasing
// order from +0, then the two parities added).  sa: the stage in shared memory.
template <int T>
__device__ __forceinline__ void g64_stage_sums(uint32_t sa, int st, int ngs, int r, int h, uint32_t ximg, int xs,
                                               const int *cimg, int ng, float (&ss)[T])
{
    float acc[T];
#pragma unroll
    for (int t = 0; t < T; ++t) acc[t] = 0.0f;
    if (ngs == G64_STAGE_GROUPS) {
        const uint4 sc = lds128(sa + 4096 + (r * 2 + h) * 16);
        const float sgs[4] = {__uint_as_float(sc.x), __uint_as_float(sc.y), __uint_as_float(sc.z),
                              __uint_as_float(sc.w)};
        const uint32_t row = sa + r * 256;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c0 = 4 * i + 2 * h;  // the group's two 16-byte chunks
            const uint4 n0 = lds128(row + 16 * (c0 ^ (r & 7))), n1 = lds128(row + 16 * ((c0 + 1) ^ (r & 7)));
            const int g = st * G64_STAGE_GROUPS + 2 * i + h;
            g64_group_terms<T>(n0, n1, sgs[i], ximg + g * G64_W, xs, cimg + g, ng, acc);
        }
    } else {
        for (int i = 0; 2 * i + h < ngs; ++i) {
            const int gs = 2 * i + h;
            const uint32_t nb = sa + (r * ngs + gs) * G64_NIB;
            const uint4 n0 = lds128(nb), n1 = lds128(nb + 16);
            float sg;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sg) : "r"(sa + SLAB_ROWS * ngs * G64_NIB + (r * ngs + gs) * 4));
            const int g = st * G64_STAGE_GROUPS + gs;
            g64_group_terms<T>(n0, n1, sg, ximg + g * G64_W, xs, cimg + g, ng, acc);
        }
    }
#pragma unroll
    for (int t = 0; t < T; ++t) ss[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xFFFFFFFFu, acc[t], 16));
}

// 16 nibble bytes from global memory at a 4-byte aligned address.
__device__ __forceinline__ uint4 ldg_u4_a4(const uint8_t *p)
{
    const unsigned *w = reinterpret_cast<const unsigned *>(p);
    return make_uint4(__ldg(w), __ldg(w + 1), __ldg(w + 2), __ldg(w + 3));
}

// The activation rows x[T][K] (fp32) quantised by this CTA into the code
// image [T][K] and s_sx[T]: the steps of quantize_vec_i8_kernel (s =
// amax / 127 over the row, 1/s from it, codes round-half-away(x * (1/s))).
// The maximum is exact in any order, so codes and scales equal that
// kernel's.  K % 64 == 0.
template <int T>
__device__ __forceinline__ void g64_quantize_rows(const float *x, int K, uint8_t *img, float *s_sx, int tid,
                                                  int nthreads)
{
    __shared__ float s_red[T][NWARPS_MAX];
    __shared__ float s_id[T];
    const int warp = tid >> 5, lane = tid & 31, nw = nthreads >> 5;
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    auto load4 = [&](long long i) -> float4 {
        if (vec) return __ldcg(reinterpret_cast<const float4 *>(x + i));
        return make_float4(__ldcg(x + i), __ldcg(x + i + 1), __ldcg(x + i + 2), __ldcg(x + i + 3));
    };
#pragma unroll
    for (int t = 0; t < T; ++t) {
        float m = 0.0f;
        for (int k = 4 * tid; k < K; k += 4 * nthreads) {
            const float4 v = load4(static_cast<long long>(t) * K + k);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) s_red[t][warp] = m;
    }
    __syncthreads();
    if (tid < T) {
        float m = 0.0f;
        for (int w = 0; w < nw; ++w) m = fmaxf(m, s_red[tid][w]);
        float d, id;
        q8_scale(m, d, id);
        s_sx[tid] = d;
        s_id[tid] = id;
    }
    __syncthreads();
    for (int i = 4 * tid; i < T * K; i += 4 * nthreads) {
        const float id = s_id[i / K];
        const float4 v = load4(i);
        *reinterpret_cast<unsigned *>(img + i) =
            (static_cast<unsigned>(q8_code(v.x, id)) & 0xFFu) | ((static_cast<unsigned>(q8_code(v.y, id)) & 0xFFu) << 8) |
            ((static_cast<unsigned>(q8_code(v.z, id)) & 0xFFu) << 16) |
            ((static_cast<unsigned>(q8_code(v.w, id)) & 0xFFu) << 24);
    }
}

// y = (total / 16) * s_x: the output of one row and token.
__device__ __forceinline__ float g64_output(float total, float sx) { return __fmul_rn(__fmul_rn(total, 0.0625f), sx); }

template <int T>
__global__ void __launch_bounds__(NWARPS_MAX * 32, 1) gs64_gemv_kernel(const __grid_constant__ G64Params P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    __shared__ float s_sx[T];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = lane & 15, h = lane >> 4;
    const int nw = P.nwarps, D = P.ring_depth, nthreads = nw * 32;
    const int xs = P.K;
    const uint32_t ximg = smem_addr(smem);
    int *cimg = reinterpret_cast<int *>(smem + P.off_c);  // [T][ng] folded constants
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + P.off_bar) + warp * D;
    uint8_t *ring = smem + P.off_ring + static_cast<size_t>(warp) * D * G64_STAGE_BYTES;
    volatile int *abort_flag = &s_abort;
    const long long slab_bytes = static_cast<long long>(SLAB_ROWS) * P.ng * G64_BYTES;
    const int last_ngs = P.ng - (P.nstage - 1) * G64_STAGE_GROUPS;
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
            const unsigned bytes = c_st == P.nstage - 1
                                       ? static_cast<unsigned>(SLAB_ROWS * last_ngs * G64_BYTES)
                                       : static_cast<unsigned>(G64_STAGE_BYTES);
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[slot], bytes);
            bulk_g2s(ring + slot * G64_STAGE_BYTES,
                     P.W + sl * slab_bytes + static_cast<long long>(c_st) * G64_STAGE_BYTES, bytes, &bar[slot], pol);
        }
    };
    int issued = 0;
    for (int d = 0; d < D && c_valid(); ++d) {
        issue(d);
        ++issued;
        c_step();
    }

    // activations after the preceding kernel: the codes as given, then per
    // token and group the folded constant MAGIC - 128 sum(q)
    pdl_wait();
    if (P.xf != nullptr) {
        g64_quantize_rows<T>(P.xf, P.K, smem, s_sx, tid, nthreads);
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(P.q);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        for (int i = tid; i < T * P.K / 16; i += nthreads) dst[i] = __ldcg(src + i);
        if (tid < T) s_sx[tid] = __ldcg(P.sx + tid);
    }
    __syncthreads();
    for (int i = tid; i < T * P.ng; i += nthreads) {
        const uint4 *g = reinterpret_cast<const uint4 *>(smem + static_cast<long long>(i) * G64_W);
        const int ones = 0x01010101;
        int s = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 v = g[k];
            s = dp4a_ss((int)v.x, ones, s);
            s = dp4a_ss((int)v.y, ones, s);
            s = dp4a_ss((int)v.z, ones, s);
            s = dp4a_ss((int)v.w, ones, s);
        }
        cimg[i] = MAGIC_I - 128 * s;  // [t][g]: i = t * ng + g (the codes are [t][K])
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
            // the N % 16 tail rows: direct loads, the same order
            const long long row = static_cast<long long>(P.nslabs) * SLAB_ROWS + r;
            const bool live = r < P.tail_rows;
            const uint8_t *tb = P.W + static_cast<long long>(P.nslabs) * slab_bytes +
                                static_cast<long long>(live ? r : 0) * P.ng * G64_BYTES;
            const float *tsc = reinterpret_cast<const float *>(tb + static_cast<long long>(P.ng) * G64_NIB);
            for (int st = 0; st < P.nstage; ++st) {
                float acc[T];
#pragma unroll
                for (int t = 0; t < T; ++t) acc[t] = 0.0f;
                for (int i = 0; i < 4; ++i) {
                    const int g = st * G64_STAGE_GROUPS + 2 * i + h;
                    if (live && g < P.ng) {
                        const uint8_t *gp = tb + static_cast<long long>(g) * G64_NIB;
                        g64_group_terms<T>(ldg_u4_a4(gp), ldg_u4_a4(gp + 16), __ldg(tsc + g), ximg + g * G64_W, xs,
                                           cimg + g, P.ng, acc);
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
                for (int t = 0; t < T; ++t) P.y[static_cast<long long>(t) * P.N + row] = g64_output(tot[t], s_sx[t]);
            continue;
        }
        const int sl = it / P.chunks, c = it - sl * P.chunks;
        const int a = P.nstage * c / P.chunks, e = P.nstage * (c + 1) / P.chunks;
        const bool split = P.chunks > 1;
        for (int st = a; st < e; ++st) {
            if (ok) ok = mbar_wait_bounded(&bar[slot], phase, abort_flag, P.status, WAIT_LIMIT_NS);
            if (ok) {
                const int ngs = st == P.nstage - 1 ? last_ngs : G64_STAGE_GROUPS;
                g64_stage_sums<T>(smem_addr(ring + slot * G64_STAGE_BYTES), st, ngs, r, h, ximg, xs, cimg, P.ng, ss);
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
                for (int t = 0; t < T; ++t) P.y[static_cast<long long>(t) * P.N + row] = g64_output(tot[t], s_sx[t]);
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
                    P.y[static_cast<long long>(t) * P.N + row] = g64_output(v, s_sx[t]);
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
cudaError_t launch_gs64_t(const G64Params &P, int grid, size_t smem, cudaStream_t st)
{
    auto kern = gs64_gemv_kernel<T>;
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

cudaError_t launch_gs64(const void *W, const int8_t *q, const float *sx, const float *xf, float *y, long long N,
                        long long K, int T, void *ws, long long ws_bytes, bool do_launch, int sms, int smem_budget,
                        unsigned *status, cudaStream_t st, long long *ws_need, int *unsupported)
{
    G64Params P = {};
    P.W = static_cast<const uint8_t *>(W);
    P.q = q;
    P.sx = sx;
    P.xf = xf;
    P.y = y;
    P.status = status;
    P.N = N;
    P.K = static_cast<int>(K);
    P.ng = P.K / G64_W;
    P.nstage = (P.ng + G64_STAGE_GROUPS - 1) / G64_STAGE_GROUPS;
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
    if (P.chunks > 1) need = 256 + (4ll * P.nslabs + 255) / 256 * 256 + 4ll * P.nslabs * P.nstage * T * SLAB_ROWS;
    *ws_need = need;
    *unsupported = 0;
    // shared memory: codes, constants, barriers, rings; the widest shape that fits
    const long long xbytes = (static_cast<long long>(T) * K + 127) / 128 * 128;
    const long long cbytes = (4ll * T * P.ng + 127) / 128 * 128;
    const int shapes[4][2] = {{16, 2}, {16, 1}, {8, 2}, {8, 1}};
    int nw = 0, D = 0;
    long long smem = 0;
    for (const auto &c : shapes) {
        const long long bars = (8ll * c[0] * c[1] + 127) / 128 * 128;
        const long long total = xbytes + cbytes + bars + static_cast<long long>(c[0]) * c[1] * G64_STAGE_BYTES;
        if (total <= smem_budget) {
            nw = c[0];
            D = c[1];
            smem = total;
            P.off_c = static_cast<int>(xbytes);
            P.off_bar = static_cast<int>(xbytes + cbytes);
            P.off_ring = static_cast<int>(xbytes + cbytes + bars);
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
    case 1: return launch_gs64_t<1>(P, grid, static_cast<size_t>(smem), st);
    case 2: return launch_gs64_t<2>(P, grid, static_cast<size_t>(smem), st);
    case 3: return launch_gs64_t<3>(P, grid, static_cast<size_t>(smem), st);
    case 4: return launch_gs64_t<4>(P, grid, static_cast<size_t>(smem), st);
    case 5: return launch_gs64_t<5>(P, grid, static_cast<size_t>(smem), st);
    case 6: return launch_gs64_t<6>(P, grid, static_cast<size_t>(smem), st);
    case 7: return launch_gs64_t<7>(P, grid, static_cast<size_t>(smem), st);
    case 8: return launch_gs64_t<8>(P, grid, static_cast<size_t>(smem), st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
